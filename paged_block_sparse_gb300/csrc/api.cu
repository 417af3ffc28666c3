// The C ABI of libpbs (include/pbs.h): argument validation, scale folding, tensor-map encoding,
// launch-shape choice and dispatch to the kernels. Nothing here allocates device memory.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/pbs.h"
#include "pbs_internal.h"

namespace {

using pbs::AttendArgs;
using pbs::InsertArgs;
using pbs::TableArgs;

constexpr int kBlockPages = 8;
constexpr int kPageRows = 16;
constexpr int kHeadDim = 128;
constexpr int kMaxTopk = 64;
constexpr int kNvfp4SlotBytes = 1152;

bool aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

int page_content_bytes(int kv_dtype, int num_kv_heads) {
  switch (kv_dtype) {
    case PBS_KV_BF16: return num_kv_heads * kPageRows * 2 * kHeadDim * 2;
    case PBS_KV_FP8_E4M3: return num_kv_heads * kPageRows * 2 * kHeadDim;
    case PBS_KV_NVFP4: return num_kv_heads * 2 * kNvfp4SlotBytes;
    default: return -1;
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Page rows of one kv head as a 4-D tensor {row elements, 16 rows, kv heads, pages}. A box is
// 128 bytes of 16 consecutive rows of one (page, head), stored 128B-swizzled in shared memory.
int encode_cache_map(CUtensorMap* map, const void* cache, int kv_dtype, int num_kv_heads, int64_t num_pages,
                     int64_t page_stride_bytes) {
  std::memset(map, 0, sizeof(*map));
  if (kv_dtype == PBS_KV_NVFP4) return PBS_OK;  // read with untiled bulk copies
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return PBS_ERR_CUDA;
  const int eb = kv_dtype == PBS_KV_BF16 ? 2 : 1;
  const cuuint64_t row_elems = 2 * kHeadDim;
  const cuuint64_t dims[4] = {row_elems, kPageRows, static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(num_pages)};
  const cuuint64_t strides[3] = {row_elems * eb, row_elems * eb * kPageRows, static_cast<cuuint64_t>(page_stride_bytes)};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / eb), kPageRows, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = enc(map, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
                         const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PBS_OK : PBS_ERR_CUDA;
}

// A packed cache (pages back to back: page stride = Hkv * 16 rows * row bytes) as one box per
// (page, kv head): a 5-D map {row bytes' first 128 B, 8 rows, q, 2 row halves, page * Hkv + head}
// whose box lands as [row half][q][8 rows][128 B], q = the four 64-element quarters of a bf16 row
// (K lo, K hi, V lo, V hi) or the two halves of an fp8 row (K, V): 128B-swizzle atoms of 8 rows.
// Every address stays inside its own (page, head) chunk.
// With quarters_per_box = 2 (bf16 only) a box holds either the K or the V half of every row
// (quarter coordinate 0 or 2), landing as [row half][2][8 rows][128 B].
int encode_cache_map_packed(CUtensorMap* map, const void* cache, int kv_dtype, int num_kv_heads, int64_t num_pages,
                            int64_t page_stride_bytes, int quarters_per_box = 0) {
  std::memset(map, 0, sizeof(*map));
  if (kv_dtype != PBS_KV_BF16 && kv_dtype != PBS_KV_FP8_E4M3) return PBS_ERR_UNSUPPORTED;
  if (page_stride_bytes != page_content_bytes(kv_dtype, num_kv_heads)) return PBS_ERR_UNSUPPORTED;
  if (num_pages * num_kv_heads > 0x7fffffffLL) return PBS_ERR_UNSUPPORTED;
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return PBS_ERR_CUDA;
  const bool bf = kv_dtype == PBS_KV_BF16;
  const cuuint64_t row = bf ? 512 : 256;  // bytes per page row of one head
  const cuuint64_t nq = bf ? 4 : 2;
  const cuuint64_t dims[5] = {bf ? 64u : 128u, 8, nq, 2, static_cast<cuuint64_t>(num_pages) * num_kv_heads};
  const cuuint64_t strides[4] = {row, 128, 8 * row, 16 * row};
  if (quarters_per_box != 0 && (!bf || quarters_per_box != 2)) return PBS_ERR_UNSUPPORTED;
  const cuuint32_t qbox = quarters_per_box != 0 ? static_cast<cuuint32_t>(quarters_per_box) : static_cast<cuuint32_t>(nq);
  const cuuint32_t box[5] = {bf ? 64u : 128u, 8, qbox, 2, 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = enc(map, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 5,
                         const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PBS_OK : PBS_ERR_CUDA;
}

// A packed bf16 cache as one box per 128-key block of one kv head: a 5-D map {the first 64
// elements of a page row, 16 rows, kv head, page, row quarter} (strides: row, one head's 16 rows,
// the page, 128 B) whose box {64, 16, 1, 8, 2} starts at the block's first page and at quarter
// 0 (K) or 2 (V). It lands as [quarter][8 pages][16 rows][128 B]: key k of the block at k * 128 B,
// the block's dims 64..127 16 KiB further, in 128B-swizzle atoms of 8 keys. The block's 8 pages
// are consecutive (block_page_stride >= 8); pages past the cache read as zeros.
int encode_cache_map_block(CUtensorMap* map, const void* cache, int num_kv_heads, int64_t num_pages,
                           int64_t page_stride_bytes) {
  std::memset(map, 0, sizeof(*map));
  if (page_stride_bytes != page_content_bytes(PBS_KV_BF16, num_kv_heads)) return PBS_ERR_UNSUPPORTED;
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return PBS_ERR_CUDA;
  const cuuint64_t row = 2 * kHeadDim * 2;  // K and V of one row of one head, bf16
  const cuuint64_t dims[5] = {kHeadDim / 2, kPageRows, static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(num_pages), 4};
  const cuuint64_t strides[4] = {row, row * kPageRows, static_cast<cuuint64_t>(page_stride_bytes), 128};
  const cuuint32_t box[5] = {kHeadDim / 2, kPageRows, 1, 8, 2};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(cache), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PBS_OK : PBS_ERR_CUDA;
}

// The tensor map the token-centric kernel reads: the packed one when the cache allows it and the
// caller did not ask for the per-quarter map.
int encode_attend_map(CUtensorMap* map, const void* cache, int kv_dtype, int num_kv_heads, int64_t num_pages,
                      int64_t page_stride_bytes, bool quarter_map, int32_t* packed) {
  *packed = 0;
  if (!quarter_map &&
      encode_cache_map_packed(map, cache, kv_dtype, num_kv_heads, num_pages, page_stride_bytes) == PBS_OK) {
    *packed = 1;
    return PBS_OK;
  }
  return encode_cache_map(map, cache, kv_dtype, num_kv_heads, num_pages, page_stride_bytes);
}

// Queries as a 3-D tensor {head_dim, heads, tokens}; a box is (128 / G) tokens x G heads x 64
// dims (G = 8 or 16 query heads per kv head), laid out in shared memory as the 128-row K-major
// operand of the prefill MMA (row = token * G + head).
int encode_q_map(CUtensorMap* map, const void* q, int num_heads, int group, int total_q, int64_t q_row_stride,
                 int64_t q_head_stride, int box_tokens = 0) {
  std::memset(map, 0, sizeof(*map));
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return PBS_ERR_CUDA;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(num_heads),
                              static_cast<cuuint64_t>(total_q)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(q_head_stride) * 2, static_cast<cuuint64_t>(q_row_stride) * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group),
                             static_cast<cuuint32_t>(box_tokens > 0 ? box_tokens : 128 / group)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PBS_OK : PBS_ERR_CUDA;
}

// The query rows of one token and one kv head as a single tensor copy (the gathered-row kernel):
// a 5-D view {64 dims, 8 heads, dim half, head octet, token} of q ([tokens, heads, 128] with the
// caller's strides) with a {64, 8, 2, group / 8, 1} box. Shared memory then holds the token's
// rows as [octet][half][8 heads][128 B] (128B swizzle): 1 KiB atoms, K halves 1 KiB apart and
// consecutive 8-row atoms of the M dimension 2 KiB apart.
int encode_q_map_tokens(CUtensorMap* map, const void* q, int num_heads, int group, int total_q, int64_t q_row_stride,
                        int64_t q_head_stride) {
  std::memset(map, 0, sizeof(*map));
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return PBS_ERR_CUDA;
  if (num_heads % 8 != 0 || group % 8 != 0) return PBS_ERR_UNSUPPORTED;
  const cuuint64_t dims[5] = {64, 8, 2, static_cast<cuuint64_t>(num_heads / 8), static_cast<cuuint64_t>(total_q)};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(q_head_stride) * 2, 128,
                                 static_cast<cuuint64_t>(q_head_stride) * 2 * 8, static_cast<cuuint64_t>(q_row_stride) * 2};
  const cuuint32_t box[5] = {64, 8, 2, static_cast<cuuint32_t>(group / 8), 1};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(q), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PBS_OK : PBS_ERR_CUDA;
}

// Which prefill kernel runs: the caller's choice (pbs_attend_options.prefill_kernel) when given,
// else by the page table's width (the only bound on the contexts that the host sees without a
// device read) and the GQA ratio:
//
// The tile kernel streams the union of its 16 tokens' selections to all of them, so its waste
// grows with the context a token chooses from: a token at block s selects k of s + 1 blocks,
// and the union nears min(s + 1, 16 k). The gathered-row kernel's MMA rows are the tokens that
// selected a block, so its work does not grow with the context, but every (token, block) pair
// costs a partial output written and merged through the workspace; it hands the dense leading
// tiles of every request (tokens before position 128 k, which select every block they see) to
// the tile kernel. With its workspace the gathered-row kernel is taken at GQA 8, and at GQA 16
// for page tables wider than kTileMaxBlocksPerTopk * k blocks; otherwise the tile kernel (fp8 /
// NVFP4 with its images; bf16 only up to that width) or the token-centric kernel. Measured (64
// query heads, top-k 16): the varlen prompts of 2k-8k tokens (64-block table) take 2.37 ms on
// the tile kernel, 2.22 on the gathered rows (2.10 / 2.45 at GQA 16); 2 x 4096 NVFP4 tokens
// after 16k / 32k of context take 4.71 and 1.59 ms; bf16 on the tile kernel gives 462 / 312 / 114
// TFLOP/s for contexts 0 / 2k-4k / 16k-32k, the token-centric kernel about 139 throughout.
constexpr int kTileMaxBlocksPerTopk = 8;

// The caller's options, checked (a null pointer reads as all zero).
struct Options {
  int prefill_kernel = PBS_PREFILL_AUTO;
  int splits = 0;
  bool quarter_map = false;
};

int read_options(const pbs_attend_options* o, Options* out) {
  *out = Options();
  if (o == nullptr) return PBS_OK;
  if (o->prefill_kernel < PBS_PREFILL_AUTO || o->prefill_kernel > PBS_PREFILL_GATHER) return PBS_ERR_ARG;
  if (o->splits != 0 && o->splits != 1 && o->splits != 2 && o->splits != 4 && o->splits != 8) return PBS_ERR_ARG;
  if (o->cache_map != 0 && o->cache_map != 1) return PBS_ERR_ARG;
  if (o->reserved != 0) return PBS_ERR_ARG;
  out->prefill_kernel = o->prefill_kernel;
  out->splits = o->splits;
  out->quarter_map = o->cache_map == 1;
  return PBS_OK;
}

// Sets *kernel (PBS_PREFILL_TOKEN / _TILE / _GATHER) for a prefill call whose AttendArgs (map
// already encoded, table attached) are `a`, given the caller's workspace size and option;
// PBS_ERR_UNSUPPORTED when the option asks for a kernel that cannot run the call. The one rule
// behind both the call and pbs_prefill_kernel_choice.
int choose_prefill_kernel(const AttendArgs& a, size_t workspace_bytes, int forced, int* kernel) {
  // the tile kernel reads a packed bf16 cache through its block map, an fp8 / NVFP4 cache through
  // the images its conversion kernel writes into the workspace
  const size_t tile_ws = pbs::prefill_tc_workspace_bytes(a.num_reqs, a.num_kv_heads, a.max_blocks, a.kv_dtype);
  const bool tile_fits = (a.kv_dtype != PBS_KV_BF16 || a.packed_map != 0) &&
                         pbs::prefill_tc_supported(a, tile_ws != 0 && workspace_bytes >= tile_ws);
  const bool gather_fits = (a.kv_dtype != PBS_KV_BF16 || a.packed_map != 0) && pbs::prefill_gather_supported(a) &&
                           a.num_rows < (1 << 25) &&
                           pbs::gather_segment_tokens(a.num_rows, a.num_reqs, a.num_heads, a.num_kv_heads, a.k,
                                                      a.max_blocks, workspace_bytes) > 0;
  if ((forced == PBS_PREFILL_TILE && !tile_fits) || (forced == PBS_PREFILL_GATHER && !gather_fits))
    return PBS_ERR_UNSUPPORTED;
  // fp8 / NVFP4: the token-centric kernel dequantises every gathered row per token, the tile kernel
  // once per block; measured faster at every page-table width (prefill prompts 3.3x / 3.6x,
  // contexts of 16k / 32k keys 1.04x)
  const bool wide = a.max_blocks > kTileMaxBlocksPerTopk * a.k;
  if (forced != PBS_PREFILL_AUTO) *kernel = forced;
  else if (gather_fits && (wide || a.group == 8)) *kernel = PBS_PREFILL_GATHER;
  else if (tile_fits && (a.kv_dtype != PBS_KV_BF16 || !wide)) *kernel = PBS_PREFILL_TILE;
  else *kernel = PBS_PREFILL_TOKEN;
  return PBS_OK;
}

// CTAs per (row, kv head). Splitting a row across a cluster costs a cluster barrier, a DSMEM
// merge and one more CTA start-up (a chain of dependent loads: top-k, page table, first page)
// per split; measured on the 64-request decode workload (512 row x head units, 2 CTAs per SM)
// one CTA per unit streams at 75% of HBM peak against 61% / 57% / 43% for 2 / 4 / 8 splits.
// So rows are split only while the units alone cannot fill every SM twice, and only while
// each split keeps at least four 128-key slots. The caller's option (1, 2, 4 or 8) overrides.
//
// With a workspace the splits merge through it instead (no cluster, no waiting: the last chunk
// of a row merges), so any split count up to 8 schedules freely; a row is cut into chunks while
// the chunks still fit one wave of resident CTAs (4 per SM), keeping at least two 128-key slots
// per chunk. More than one wave loses more to per-CTA start-up than it gains in balance.
int num_sms() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

int choose_splits(int64_t units, int k, bool workspace, int forced) {
  if (forced != 0) return forced;
  const int64_t sms = num_sms();
  int s = 1;
  if (workspace) {
    while (s < pbs::kMaxSplits && units * (2 * s) <= 4 * sms && 2 * (2 * s) <= k) s *= 2;
  } else {
    while (s < 8 && units * s < 2 * sms && 4 * (2 * s) <= k) s *= 2;
  }
  return s;
}

// Optional log-sum-exp output: [rows, num_heads] fp32 with a unit head stride.
int attach_lse(AttendArgs* a, float* lse, int64_t lse_row_stride) {
  a->lse = lse;
  a->lse_row_stride = lse_row_stride;
  if (lse == nullptr) return PBS_OK;
  if (!aligned(lse, 4)) return PBS_ERR_ALIGN;
  if (lse_row_stride < a->num_heads) return PBS_ERR_SHAPE;
  return PBS_OK;
}

// A workspace (optional) lets splits merge through global memory. It must hold
// attend_workspace_bytes(units) bytes, 16-byte aligned. Partials fill it from the front, the
// per-unit tickets sit at its very end: a call of any size that fits the buffer writes partials
// only below the ticket words of every other call that fits it, so one zeroing of the buffer
// serves calls of all sizes (each completed call leaves its tickets zero).
int attach_workspace(AttendArgs* a, int64_t units, void* workspace, size_t workspace_bytes) {
  a->split_ws = nullptr;
  a->split_tickets = nullptr;
  if (workspace == nullptr) return workspace_bytes == 0 ? PBS_OK : PBS_ERR_ARG;
  if (!aligned(workspace, 16)) return PBS_ERR_ALIGN;
  if (workspace_bytes < pbs::attend_workspace_bytes(units)) return PBS_ERR_SHAPE;
  a->split_ws = static_cast<float*>(workspace);
  a->split_tickets = static_cast<int32_t*>(workspace) + (workspace_bytes / sizeof(int32_t) - static_cast<size_t>(units));
  return PBS_OK;
}

int check_common_table(const int32_t* topk, int64_t topk_row_stride, int32_t topk_k, const int32_t* page_table,
                       int64_t pt_row_stride, int32_t max_blocks, int32_t block_page_stride, bool topk_optional = false) {
  if ((topk == nullptr && !topk_optional) || page_table == nullptr) return PBS_ERR_ARG;
  if (topk_k <= 0 || max_blocks <= 0) return PBS_ERR_ARG;
  if (topk_k > kMaxTopk) return PBS_ERR_UNSUPPORTED;
  if (topk_row_stride < topk_k || pt_row_stride < max_blocks) return PBS_ERR_SHAPE;
  if (block_page_stride < kBlockPages) return PBS_ERR_SHAPE;
  return PBS_OK;
}

int check_attend(const void* q, int64_t q_row_stride, int64_t q_head_stride, const void* kv_cache,
                 int64_t page_stride_bytes, int64_t num_pages, int32_t kv_dtype, int32_t num_heads,
                 int32_t num_kv_heads, int32_t head_dim, float softmax_scale, float k_scale, float v_scale,
                 const void* out, int64_t out_row_stride, int64_t out_head_stride) {
  if (q == nullptr || kv_cache == nullptr || out == nullptr) return PBS_ERR_ARG;
  if (kv_dtype != PBS_KV_BF16 && kv_dtype != PBS_KV_FP8_E4M3 && kv_dtype != PBS_KV_NVFP4) return PBS_ERR_ARG;
  if (!std::isfinite(softmax_scale) || !std::isfinite(k_scale) || !std::isfinite(v_scale)) return PBS_ERR_ARG;
  if (num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return PBS_ERR_ARG;
  if (num_heads % num_kv_heads != 0) return PBS_ERR_SHAPE;
  if (head_dim != kHeadDim) return PBS_ERR_UNSUPPORTED;
  const int G = num_heads / num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return PBS_ERR_UNSUPPORTED;
  if (num_kv_heads > 65535) return PBS_ERR_UNSUPPORTED;
  if (q_row_stride < 0 || q_head_stride < 0 || out_row_stride < 0 || out_head_stride < 0) return PBS_ERR_SHAPE;
  if (num_pages <= 0 || num_pages > 0x7fffffffLL) return PBS_ERR_SHAPE;
  if (page_stride_bytes < page_content_bytes(kv_dtype, num_kv_heads)) return PBS_ERR_SHAPE;
  if (!aligned(kv_cache, 16) || page_stride_bytes % 16 != 0) return PBS_ERR_ALIGN;
  if (!aligned(q, 4) || q_row_stride % 2 != 0 || q_head_stride % 2 != 0) return PBS_ERR_ALIGN;
  if (!aligned(out, 2)) return PBS_ERR_ALIGN;
  return PBS_OK;
}

// An optional prebuilt table ([rows, >= k * 8] page ids and per-row ctx): both or neither.
int attach_table(AttendArgs* a, const int32_t* sparse_bt, int64_t sbt_row_stride, const int32_t* sparse_ctx) {
  a->sparse_bt = nullptr;
  a->sbt_row_stride = 0;
  a->sparse_ctx = nullptr;
  if (sparse_bt == nullptr && sparse_ctx == nullptr) return PBS_OK;
  if (sparse_bt == nullptr || sparse_ctx == nullptr) return PBS_ERR_ARG;
  if (sbt_row_stride < static_cast<int64_t>(a->k) * kBlockPages) return PBS_ERR_SHAPE;
  if (!aligned(sparse_bt, 4) || !aligned(sparse_ctx, 4)) return PBS_ERR_ALIGN;
  a->sparse_bt = sparse_bt;
  a->sbt_row_stride = sbt_row_stride;
  a->sparse_ctx = sparse_ctx;
  return PBS_OK;
}

AttendArgs make_attend_args(const void* q, int64_t q_row_stride, int64_t q_head_stride, const void* kv_cache,
                            int64_t page_stride_bytes, int64_t num_pages, int32_t kv_dtype, int32_t num_heads,
                            int32_t num_kv_heads, const int32_t* topk, int64_t topk_row_stride, int32_t topk_k,
                            const int32_t* page_table, int64_t pt_row_stride, int32_t max_blocks,
                            const int32_t* seq_lens, int32_t block_page_stride, float softmax_scale,
                            float k_scale, float v_scale, void* out, int64_t out_row_stride,
                            int64_t out_head_stride, int32_t* err_word) {
  AttendArgs a = {};
  a.q = static_cast<const uint16_t*>(q);
  a.q_row_stride = q_row_stride;
  a.q_head_stride = q_head_stride;
  a.kv_cache = static_cast<const uint8_t*>(kv_cache);
  a.page_stride_bytes = page_stride_bytes;
  a.num_pages = num_pages;
  a.kv_dtype = kv_dtype;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = num_heads / num_kv_heads;
  a.sub_groups = a.group > 8 ? a.group / 8 : 1;
  a.topk = topk;
  a.topk_row_stride = topk_row_stride;
  a.k = topk_k;
  a.page_table = page_table;
  a.pt_row_stride = pt_row_stride;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.block_page_stride = block_page_stride;
  // k_scale folds into the logits, v_scale into the output (vLLM page
  // vllm.models.minimax_m3.nvidia.sparse_attention_flashinfer, forward); log2(e) moves the
  // softmax to base 2.
  a.scale_log2 = static_cast<float>(static_cast<double>(softmax_scale) * k_scale * 1.4426950408889634);
  a.v_scale = v_scale;
  a.out = static_cast<uint16_t*>(out);
  a.out_row_stride = out_row_stride;
  a.out_head_stride = out_head_stride;
  a.err_word = err_word;
  return a;
}

}  // namespace

// ---- fixed scratch of pbs_sparse_decode_attention_noalloc ------------------------------------
// Some callers cannot allocate device memory while serving a step: an engine that fixes its
// memory plan at start-up and treats any later allocation as an error, or one sharing the GPU
// with a framework that owns the allocator. For them the split partials and arrival tickets
// live in this file-scope device array instead of a caller workspace. Layout: partials from
// the front (kWsPartialBytes each, at most kNoAllocMaxPartials), tickets in the last
// kNoAllocTicketBytes. The tickets must start at zero: a static device array is zero when the
// module loads, and every completed call leaves the tickets it used at zero. The partials need
// no initial value. All calls on one device share the array, so two calls whose kernels could
// overlap (different streams, or host threads without ordering) race on it.
namespace {
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
constexpr size_t kNoAllocTicketBytes = size_t(16) << 10;
constexpr int64_t kNoAllocMaxUnits = static_cast<int64_t>(kNoAllocTicketBytes / sizeof(int32_t));
constexpr int64_t kNoAllocMaxPartials =
    static_cast<int64_t>((kNoAllocScratchBytes - kNoAllocTicketBytes) / pbs::kWsPartialBytes);
static_assert(kNoAllocMaxPartials == 1004, "the status text states this limit");
}  // namespace

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};
CUcontext g_noalloc_ctx[kNoAllocMaxDevices] = {};

// The driver's cuCtxGetCurrent, reached through the runtime's entry-point query (the library
// links no driver library).
PFN_cuCtxGetCurrent_v4000 ctx_getter() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  return fn;
}

// Device address of the scratch on the current device, looked up once per device and context
// (the lookup may load this library's device module, which is why the first call should come
// before any stream capture begins). A new context on the device (after a reset the module, and
// the array with it, is loaded again) triggers a new lookup, so a stale address is never used.
int noalloc_scratch(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return PBS_ERR_CUDA;
  auto get_ctx = ctx_getter();
  if (get_ctx == nullptr) return PBS_ERR_CUDA;
  // null until the runtime has made the device's context current (the lookup below does)
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return PBS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr || ctx == nullptr || g_noalloc_ctx[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return PBS_ERR_CUDA;
    if (get_ctx(&ctx) != CUDA_SUCCESS) return PBS_ERR_CUDA;
    g_noalloc_addr[dev] = p;
    g_noalloc_ctx[dev] = ctx;
  }
  *addr = g_noalloc_addr[dev];
  return PBS_OK;
}
}  // namespace

extern "C" {

const char* pbs_status_string(int status) {
  switch (status) {
    case PBS_OK: return "ok";
    case PBS_ERR_ARG: return "invalid argument (null pointer, bad enum or non-positive size)";
    case PBS_ERR_SHAPE: return "inconsistent shapes or strides";
    case PBS_ERR_UNSUPPORTED: return "unsupported configuration (head_dim must be 128, GQA ratio 1/2/4/8/16, top-k <= 64)";
    case PBS_ERR_ALIGN: return "misaligned pointer or stride (cache 16 B, q 4 B, out 2 B)";
    case PBS_ERR_CUDA: return "CUDA error (launch, tensor-map encoding or driver entry point)";
    case PBS_ERR_SCRATCH:
      return "request needs more than the fixed no-allocation scratch (4 MiB: at most 1004 split partials "
             "= rows x head groups x splits, and 4096 rows x head groups when split)";
    default: return "unknown status";
  }
}

int pbs_abi_version(void) { return 9; }

size_t pbs_attend_workspace_bytes(int64_t num_rows, int32_t num_heads, int32_t num_kv_heads) {
  if (num_rows <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return 0;
  return pbs::attend_workspace_bytes(pbs::attend_units(num_rows, num_kv_heads, num_heads / num_kv_heads));
}

int pbs_build_sparse_block_table_decode(const int32_t* topk, int64_t topk_row_stride, int32_t num_rows,
                                        int32_t topk_k, const int32_t* page_table, int64_t pt_row_stride,
                                        int32_t max_blocks, const int32_t* seq_lens, int32_t batch,
                                        int32_t decode_query_len, int32_t block_page_stride, int32_t* sparse_bt,
                                        int64_t sbt_row_stride, int32_t* sparse_ctx, int32_t* err_word,
                                        pbs_stream_t stream) {
  if (num_rows < 0 || batch < 0 || decode_query_len <= 0) return PBS_ERR_ARG;
  if (static_cast<int64_t>(batch) * decode_query_len != num_rows) return PBS_ERR_SHAPE;
  if (num_rows == 0) return PBS_OK;
  int st = check_common_table(topk, topk_row_stride, topk_k, page_table, pt_row_stride, max_blocks, block_page_stride);
  if (st != PBS_OK) return st;
  if (seq_lens == nullptr || sparse_bt == nullptr || sparse_ctx == nullptr) return PBS_ERR_ARG;
  if (sbt_row_stride < static_cast<int64_t>(topk_k) * kBlockPages) return PBS_ERR_SHAPE;
  TableArgs a = {};
  a.topk = topk;
  a.topk_row_stride = topk_row_stride;
  a.num_rows = num_rows;
  a.k = topk_k;
  a.page_table = page_table;
  a.pt_row_stride = pt_row_stride;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.decode_query_len = decode_query_len;
  a.block_page_stride = block_page_stride;
  a.sparse_bt = sparse_bt;
  a.sbt_row_stride = sbt_row_stride;
  a.sparse_ctx = sparse_ctx;
  a.err_word = err_word;
  return pbs::launch_build_table(a, false, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PBS_OK
                                                                                                  : PBS_ERR_CUDA;
}

int pbs_build_sparse_block_table_prefill(const int32_t* topk, int64_t topk_row_stride, int32_t total_q,
                                         int32_t topk_k, const int32_t* page_table, int64_t pt_row_stride,
                                         int32_t max_blocks, const int32_t* cu_seqlens_q, const int32_t* seq_lens,
                                         int32_t num_reqs, int32_t block_page_stride, int32_t* sparse_bt,
                                         int64_t sbt_row_stride, int32_t* sparse_ctx, int32_t* err_word,
                                         pbs_stream_t stream) {
  if (total_q < 0 || num_reqs < 0) return PBS_ERR_ARG;
  if (total_q == 0) return PBS_OK;
  if (num_reqs == 0) return PBS_ERR_SHAPE;
  int st = check_common_table(topk, topk_row_stride, topk_k, page_table, pt_row_stride, max_blocks, block_page_stride);
  if (st != PBS_OK) return st;
  if (cu_seqlens_q == nullptr || seq_lens == nullptr || sparse_bt == nullptr || sparse_ctx == nullptr)
    return PBS_ERR_ARG;
  if (sbt_row_stride < static_cast<int64_t>(topk_k) * kBlockPages) return PBS_ERR_SHAPE;
  TableArgs a = {};
  a.topk = topk;
  a.topk_row_stride = topk_row_stride;
  a.num_rows = total_q;
  a.k = topk_k;
  a.page_table = page_table;
  a.pt_row_stride = pt_row_stride;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.cu_seqlens_q = cu_seqlens_q;
  a.num_reqs = num_reqs;
  a.block_page_stride = block_page_stride;
  a.sparse_bt = sparse_bt;
  a.sbt_row_stride = sbt_row_stride;
  a.sparse_ctx = sparse_ctx;
  a.err_word = err_word;
  return pbs::launch_build_table(a, true, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PBS_OK
                                                                                                 : PBS_ERR_CUDA;
}

int pbs_sparse_decode_attention(const void* q, int64_t q_row_stride, int64_t q_head_stride, const void* kv_cache,
                                int64_t page_stride_bytes, int64_t num_pages, int32_t kv_dtype, int32_t num_heads,
                                int32_t num_kv_heads, int32_t head_dim, const int32_t* topk, int64_t topk_row_stride,
                                int32_t topk_k, const int32_t* page_table, int64_t pt_row_stride, int32_t max_blocks,
                                const int32_t* seq_lens, int32_t batch, int32_t decode_query_len,
                                int32_t block_page_stride, const int32_t* sparse_bt, int64_t sbt_row_stride,
                                const int32_t* sparse_ctx, float softmax_scale, float k_scale, float v_scale,
                                void* out, int64_t out_row_stride, int64_t out_head_stride, float* lse,
                                int64_t lse_row_stride, void* workspace, size_t workspace_bytes,
                                const pbs_attend_options* options, int32_t* err_word, pbs_stream_t stream) {
  if (batch < 0 || decode_query_len <= 0) return PBS_ERR_ARG;
  const int64_t rows = static_cast<int64_t>(batch) * decode_query_len;
  if (rows == 0) return PBS_OK;
  if (rows > 0x7fffffffLL / 8) return PBS_ERR_UNSUPPORTED;
  Options opt;
  int st = read_options(options, &opt);
  if (st != PBS_OK) return st;
  st = check_attend(q, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages, kv_dtype, num_heads,
                    num_kv_heads, head_dim, softmax_scale, k_scale, v_scale, out, out_row_stride, out_head_stride);
  if (st != PBS_OK) return st;
  st = check_common_table(topk, topk_row_stride, topk_k, page_table, pt_row_stride, max_blocks, block_page_stride,
                          sparse_bt != nullptr);
  if (st != PBS_OK) return st;
  if (seq_lens == nullptr) return PBS_ERR_ARG;
  AttendArgs a = make_attend_args(q, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages, kv_dtype,
                                  num_heads, num_kv_heads, topk, topk_row_stride, topk_k, page_table, pt_row_stride,
                                  max_blocks, seq_lens, block_page_stride, softmax_scale, k_scale, v_scale, out,
                                  out_row_stride, out_head_stride, err_word);
  a.decode_query_len = decode_query_len;
  a.num_rows = static_cast<int32_t>(rows);
  st = attach_table(&a, sparse_bt, sbt_row_stride, sparse_ctx);
  if (st != PBS_OK) return st;
  st = attach_lse(&a, lse, lse_row_stride);
  if (st != PBS_OK) return st;
  const int64_t units = pbs::attend_units(rows, num_kv_heads, a.group);
  st = attach_workspace(&a, units, workspace, workspace_bytes);
  if (st != PBS_OK) return st;
  a.splits = choose_splits(units, topk_k, a.split_ws != nullptr, opt.splits);
  CUtensorMap map;
  st = encode_attend_map(&map, kv_cache, kv_dtype, num_kv_heads, num_pages, page_stride_bytes, opt.quarter_map,
                         &a.packed_map);
  if (st != PBS_OK) return st;
  return pbs::launch_attend(a, pbs::kModeDecode, map, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PBS_OK
                                                                                                  : PBS_ERR_CUDA;
}

int pbs_sparse_decode_attention_noalloc(const void* q, int64_t q_row_stride, int64_t q_head_stride,
                                        const void* kv_cache, int64_t page_stride_bytes, int64_t num_pages,
                                        int32_t kv_dtype, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                        const int32_t* topk, int64_t topk_row_stride, int32_t topk_k,
                                        const int32_t* page_table, int64_t pt_row_stride, int32_t max_blocks,
                                        const int32_t* seq_lens, int32_t batch, int32_t decode_query_len,
                                        int32_t block_page_stride, float softmax_scale, float k_scale,
                                        float v_scale, void* out, int64_t out_row_stride, int64_t out_head_stride,
                                        const pbs_attend_options* options, int32_t* err_word, pbs_stream_t stream) {
  if (batch < 0 || decode_query_len <= 0) return PBS_ERR_ARG;
  const int64_t rows = static_cast<int64_t>(batch) * decode_query_len;
  if (rows == 0) return PBS_OK;
  if (rows > 0x7fffffffLL / 8) return PBS_ERR_UNSUPPORTED;
  Options opt;
  int st = read_options(options, &opt);
  if (st != PBS_OK) return st;
  st = check_attend(q, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages, kv_dtype, num_heads,
                        num_kv_heads, head_dim, softmax_scale, k_scale, v_scale, out, out_row_stride,
                        out_head_stride);
  if (st != PBS_OK) return st;
  st = check_common_table(topk, topk_row_stride, topk_k, page_table, pt_row_stride, max_blocks, block_page_stride);
  if (st != PBS_OK) return st;
  if (seq_lens == nullptr) return PBS_ERR_ARG;
  AttendArgs a = make_attend_args(q, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages, kv_dtype,
                                  num_heads, num_kv_heads, topk, topk_row_stride, topk_k, page_table, pt_row_stride,
                                  max_blocks, seq_lens, block_page_stride, softmax_scale, k_scale, v_scale, out,
                                  out_row_stride, out_head_stride, err_word);
  a.decode_query_len = decode_query_len;
  a.num_rows = static_cast<int32_t>(rows);
  // resolved on every call (cached after the first one on a device), split or not, so the
  // one-time lookup always happens on a device's first call
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != PBS_OK) return st;
  const int64_t units = pbs::attend_units(rows, num_kv_heads, a.group);
  a.splits = choose_splits(units, topk_k, true, opt.splits);
  a.split_ws = nullptr;
  a.split_tickets = nullptr;
  if (a.splits > 1) {
    // split rows merge through the fixed scratch: refuse what it cannot hold
    if (units > kNoAllocMaxUnits || units * a.splits > kNoAllocMaxPartials) return PBS_ERR_SCRATCH;
    a.split_ws = static_cast<float*>(scratch);
    a.split_tickets = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(scratch) + kNoAllocScratchBytes) - units;
  }
  CUtensorMap map;
  st = encode_attend_map(&map, kv_cache, kv_dtype, num_kv_heads, num_pages, page_stride_bytes, false, &a.packed_map);
  if (st != PBS_OK) return st;
  return pbs::launch_attend(a, pbs::kModeDecode, map, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PBS_OK
                                                                                                  : PBS_ERR_CUDA;
}

int pbs_sparse_prefill_attention(const void* q, int64_t q_row_stride, int64_t q_head_stride, const void* kv_cache,
                                 int64_t page_stride_bytes, int64_t num_pages, int32_t kv_dtype, int32_t num_heads,
                                 int32_t num_kv_heads, int32_t head_dim, const int32_t* topk, int64_t topk_row_stride,
                                 int32_t topk_k, const int32_t* page_table, int64_t pt_row_stride, int32_t max_blocks,
                                 const int32_t* cu_seqlens_q, const int32_t* seq_lens, int32_t num_reqs,
                                 int32_t total_q, int32_t block_page_stride, const int32_t* sparse_bt,
                                 int64_t sbt_row_stride, const int32_t* sparse_ctx, float softmax_scale,
                                 float k_scale, float v_scale, void* out, int64_t out_row_stride,
                                 int64_t out_head_stride, float* lse, int64_t lse_row_stride, void* workspace,
                                 size_t workspace_bytes, const pbs_attend_options* options, int32_t* err_word,
                                 pbs_stream_t stream) {
  if (total_q < 0 || num_reqs < 0) return PBS_ERR_ARG;
  if (total_q == 0) return PBS_OK;
  if (num_reqs == 0) return PBS_ERR_SHAPE;
  if (total_q > 0x7fffffff / 8) return PBS_ERR_UNSUPPORTED;
  Options opt;
  int st = read_options(options, &opt);
  if (st != PBS_OK) return st;
  st = check_attend(q, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages, kv_dtype, num_heads,
                    num_kv_heads, head_dim, softmax_scale, k_scale, v_scale, out, out_row_stride, out_head_stride);
  if (st != PBS_OK) return st;
  st = check_common_table(topk, topk_row_stride, topk_k, page_table, pt_row_stride, max_blocks, block_page_stride,
                          sparse_bt != nullptr);
  if (st != PBS_OK) return st;
  if (cu_seqlens_q == nullptr || seq_lens == nullptr) return PBS_ERR_ARG;
  AttendArgs a = make_attend_args(q, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages, kv_dtype,
                                  num_heads, num_kv_heads, topk, topk_row_stride, topk_k, page_table, pt_row_stride,
                                  max_blocks, seq_lens, block_page_stride, softmax_scale, k_scale, v_scale, out,
                                  out_row_stride, out_head_stride, err_word);
  a.cu_seqlens_q = cu_seqlens_q;
  a.num_reqs = num_reqs;
  a.num_rows = total_q;
  st = attach_table(&a, sparse_bt, sbt_row_stride, sparse_ctx);
  if (st != PBS_OK) return st;
  st = attach_lse(&a, lse, lse_row_stride);
  if (st != PBS_OK) return st;
  if (workspace == nullptr && workspace_bytes != 0) return PBS_ERR_ARG;
  CUtensorMap map;
  st = encode_attend_map(&map, kv_cache, kv_dtype, num_kv_heads, num_pages, page_stride_bytes, false, &a.packed_map);
  if (st != PBS_OK) return st;
  // the gathered-row kernel lays its arrays out from a 256-byte aligned workspace base
  int kernel = PBS_PREFILL_TOKEN;
  st = choose_prefill_kernel(a, workspace != nullptr && aligned(workspace, 256) ? workspace_bytes : 0,
                             opt.prefill_kernel, &kernel);
  if (st != PBS_OK) return st;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (kernel == PBS_PREFILL_TOKEN) {
    if (opt.quarter_map) {  // the per-quarter map on request (it applies to this kernel only)
      st = encode_attend_map(&map, kv_cache, kv_dtype, num_kv_heads, num_pages, page_stride_bytes, true,
                             &a.packed_map);
      if (st != PBS_OK) return st;
    }
    // the workspace, when it holds the split partials, merges split rows
    const int64_t units = pbs::attend_units(total_q, num_kv_heads, a.group);
    if (workspace != nullptr && workspace_bytes >= pbs::attend_workspace_bytes(units)) {
      st = attach_workspace(&a, units, workspace, workspace_bytes);
      if (st != PBS_OK) return st;
      // a prefill workspace may hold anything (the tcgen05 kernels' data): clear the tickets
      if (cudaMemsetAsync(a.split_tickets, 0, static_cast<size_t>(units) * sizeof(int32_t), cs) != cudaSuccess)
        return PBS_ERR_CUDA;
    }
    a.splits = choose_splits(units, topk_k, a.split_ws != nullptr, opt.splits);
    e = pbs::launch_attend(a, pbs::kModePrefill, map, cs);
  } else {
    // both tcgen05 kernels read a bf16 K through one box per (block, head) half row, and V (and
    // fp8 / NVFP4 K) from converted images (the map is then unused)
    CUtensorMap half_map;
    std::memset(&half_map, 0, sizeof(half_map));
    if (kv_dtype == PBS_KV_BF16)
      st = encode_cache_map_block(&half_map, kv_cache, num_kv_heads, num_pages, page_stride_bytes);
    if (st != PBS_OK) return st;
    CUtensorMap qmap, tile_qmap;
    st = kernel == PBS_PREFILL_GATHER
             ? encode_q_map_tokens(&qmap, q, num_heads, a.group, total_q, q_row_stride, q_head_stride)
             : encode_q_map(&qmap, q, num_heads, a.group, total_q, q_row_stride, q_head_stride);
    if (st != PBS_OK) return st;
    // the gathered-row kernel hands the call's leading tiles to the tile kernel
    const bool tile_part = kernel == PBS_PREFILL_GATHER &&
                           encode_q_map(&tile_qmap, q, num_heads, a.group, total_q, q_row_stride, q_head_stride) ==
                               PBS_OK;
    if (kernel == PBS_PREFILL_TILE && workspace != nullptr && aligned(workspace, 256) && num_reqs <= 65535) {
      // with room for the converted V of every (request, block, kv head), the tile kernel applies
      // P in fp16 with one MMA per 16 keys instead of bf16 hi + lo; fp8 / NVFP4 K comes from
      // converted bf16 images after them (the kernel choice made sure the workspace holds them)
      const size_t need = pbs::prefill_tc_workspace_bytes(num_reqs, num_kv_heads, max_blocks, kv_dtype);
      if (need != 0 && workspace_bytes >= need) {
        const int64_t n = static_cast<int64_t>(num_reqs) * max_blocks * num_kv_heads;
        a.vconv = static_cast<uint8_t*>(workspace);
        a.vconv_exp = reinterpret_cast<int32_t*>(a.vconv + n * pbs::kTileVBytes);
        if (kv_dtype != PBS_KV_BF16)
          a.kconv = a.vconv + n * pbs::kTileVBytes + ((n * 4 + 255) / 256) * 256;
      }
    }
    e = kernel == PBS_PREFILL_GATHER
            ? pbs::launch_prefill_gather(a, half_map, qmap, tile_part ? &tile_qmap : nullptr, workspace,
                                         workspace_bytes, cs)
            : pbs::launch_prefill_tc(a, half_map, qmap, cs);
  }
  return e == cudaSuccess ? PBS_OK : PBS_ERR_CUDA;
}

int pbs_prefill_kernel_choice(int32_t total_q, int32_t num_reqs, int32_t kv_dtype, int64_t page_stride_bytes,
                              int32_t num_heads, int32_t num_kv_heads, int32_t topk_k, int32_t max_blocks,
                              int32_t with_table, size_t workspace_bytes, const pbs_attend_options* options) {
  Options opt;
  int st = read_options(options, &opt);
  if (st != PBS_OK) return -st;
  if (total_q <= 0 || num_reqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
      topk_k <= 0 || topk_k > kMaxTopk || max_blocks <= 0 || page_content_bytes(kv_dtype, num_kv_heads) < 0)
    return -PBS_ERR_ARG;
  // the shape as a call would see it, with 16-byte aligned q / out rows and a cache small enough
  // for the packed map
  AttendArgs a = {};
  a.kv_dtype = kv_dtype;
  a.num_heads = num_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = num_heads / num_kv_heads;
  a.k = topk_k;
  a.max_blocks = max_blocks;
  a.num_rows = total_q;
  a.num_reqs = num_reqs;
  a.page_stride_bytes = page_stride_bytes;
  a.num_pages = 1;
  a.q_row_stride = a.q_head_stride = a.out_row_stride = a.out_head_stride = 8;
  static const int32_t dummy_table = 0;
  a.sparse_bt = with_table ? &dummy_table : nullptr;
  a.packed_map = (kv_dtype == PBS_KV_BF16 || kv_dtype == PBS_KV_FP8_E4M3) &&
                 page_stride_bytes == page_content_bytes(kv_dtype, num_kv_heads);
  int kernel = PBS_PREFILL_TOKEN;
  st = choose_prefill_kernel(a, workspace_bytes, opt.prefill_kernel, &kernel);
  return st == PBS_OK ? kernel : -st;
}

size_t pbs_prefill_tile_workspace_bytes(int32_t num_reqs, int32_t num_kv_heads, int32_t max_blocks, int32_t kv_dtype) {
  return pbs::prefill_tc_workspace_bytes(num_reqs, num_kv_heads, max_blocks, kv_dtype);
}

size_t pbs_prefill_workspace_bytes(int32_t total_q, int32_t num_reqs, int32_t num_heads, int32_t num_kv_heads,
                                   int32_t topk_k, int32_t max_blocks) {
  if (total_q <= 0 || num_reqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
      topk_k <= 0 || topk_k > kMaxTopk || max_blocks <= 0)
    return 0;
  const int64_t seg = std::min<int64_t>(total_q, pbs::kGatherMaxSegment);
  return pbs::gather_workspace_bytes(seg, num_reqs, num_heads, num_kv_heads, topk_k, max_blocks);
}

int pbs_sparse_mixed_attention(const void* q, int64_t q_row_stride, int64_t q_head_stride, const void* kv_cache,
                               int64_t page_stride_bytes, int64_t num_pages, int32_t kv_dtype, int32_t num_heads,
                               int32_t num_kv_heads, int32_t head_dim, const int32_t* topk, int64_t topk_row_stride,
                               int32_t topk_k, const int32_t* dec_page_table, int64_t dec_pt_row_stride,
                               int32_t dec_max_blocks, const int32_t* dec_seq_lens, int32_t batch,
                               int32_t decode_query_len, const int32_t* pre_page_table, int64_t pre_pt_row_stride,
                               int32_t pre_max_blocks, const int32_t* cu_seqlens_q, const int32_t* pre_seq_lens,
                               int32_t num_reqs, int32_t total_q, int32_t block_page_stride,
                               const int32_t* sparse_bt, int64_t sbt_row_stride, const int32_t* sparse_ctx,
                               float softmax_scale, float k_scale, float v_scale, void* out, int64_t out_row_stride,
                               int64_t out_head_stride, float* lse, int64_t lse_row_stride, void* workspace,
                               size_t workspace_bytes, const pbs_attend_options* options, int32_t* err_word,
                               pbs_stream_t stream) {
  if (batch < 0 || decode_query_len <= 0 || total_q < 0 || num_reqs < 0) return PBS_ERR_ARG;
  if (workspace == nullptr && workspace_bytes != 0) return PBS_ERR_ARG;
  const int64_t nd = static_cast<int64_t>(batch) * decode_query_len;
  // one part only: the plain entry points
  if (total_q == 0)
    return pbs_sparse_decode_attention(q, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages,
                                       kv_dtype, num_heads, num_kv_heads, head_dim, topk, topk_row_stride, topk_k,
                                       dec_page_table, dec_pt_row_stride, dec_max_blocks, dec_seq_lens, batch,
                                       decode_query_len, block_page_stride, sparse_bt, sbt_row_stride, sparse_ctx,
                                       softmax_scale, k_scale, v_scale, out, out_row_stride, out_head_stride, lse,
                                       lse_row_stride, nullptr, 0, options, err_word, stream);
  if (nd == 0)
    return pbs_sparse_prefill_attention(q, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages,
                                        kv_dtype, num_heads, num_kv_heads, head_dim, topk, topk_row_stride, topk_k,
                                        pre_page_table, pre_pt_row_stride, pre_max_blocks, cu_seqlens_q, pre_seq_lens,
                                        num_reqs, total_q, block_page_stride, sparse_bt, sbt_row_stride, sparse_ctx,
                                        softmax_scale, k_scale, v_scale, out, out_row_stride, out_head_stride, lse,
                                        lse_row_stride, workspace, workspace_bytes, options, err_word, stream);
  if (num_reqs == 0) return PBS_ERR_SHAPE;
  if (nd + total_q > 0x7fffffffLL / 8) return PBS_ERR_UNSUPPORTED;
  Options opt;
  int st = read_options(options, &opt);
  if (st != PBS_OK) return st;
  st = check_attend(q, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages, kv_dtype, num_heads,
                    num_kv_heads, head_dim, softmax_scale, k_scale, v_scale, out, out_row_stride, out_head_stride);
  if (st != PBS_OK) return st;
  st = check_common_table(topk, topk_row_stride, topk_k, dec_page_table, dec_pt_row_stride, dec_max_blocks,
                          block_page_stride, sparse_bt != nullptr);
  if (st != PBS_OK) return st;
  st = check_common_table(topk, topk_row_stride, topk_k, pre_page_table, pre_pt_row_stride, pre_max_blocks,
                          block_page_stride, sparse_bt != nullptr);
  if (st != PBS_OK) return st;
  if (dec_seq_lens == nullptr || cu_seqlens_q == nullptr || pre_seq_lens == nullptr) return PBS_ERR_ARG;

  // the prefill part as its own call would see: rows from nd on
  const void* q_pre = static_cast<const uint8_t*>(q) + nd * q_row_stride * 2;
  const int32_t* topk_pre = topk != nullptr ? topk + nd * topk_row_stride : nullptr;
  const int32_t* sbt_pre = sparse_bt != nullptr ? sparse_bt + nd * sbt_row_stride : nullptr;
  const int32_t* ctx_pre = sparse_ctx != nullptr ? sparse_ctx + nd : nullptr;
  void* out_pre = static_cast<uint8_t*>(out) + nd * out_row_stride * 2;
  float* lse_pre = lse != nullptr ? lse + nd * lse_row_stride : nullptr;
  AttendArgs p = make_attend_args(q_pre, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages,
                                  kv_dtype, num_heads, num_kv_heads, topk_pre, topk_row_stride, topk_k,
                                  pre_page_table, pre_pt_row_stride, pre_max_blocks, pre_seq_lens,
                                  block_page_stride, softmax_scale, k_scale, v_scale, out_pre, out_row_stride,
                                  out_head_stride, err_word);
  p.cu_seqlens_q = cu_seqlens_q;
  p.num_reqs = num_reqs;
  p.num_rows = total_q;
  st = attach_table(&p, sbt_pre, sbt_row_stride, ctx_pre);
  if (st != PBS_OK) return st;
  CUtensorMap map;
  st = encode_attend_map(&map, kv_cache, kv_dtype, num_kv_heads, num_pages, page_stride_bytes, false, &p.packed_map);
  if (st != PBS_OK) return st;
  int kernel = PBS_PREFILL_TOKEN;
  st = choose_prefill_kernel(p, workspace != nullptr && aligned(workspace, 256) ? workspace_bytes : 0,
                             opt.prefill_kernel, &kernel);
  if (st != PBS_OK) return st;
  if (kernel != PBS_PREFILL_TOKEN) {
    // the prefill part runs on a tcgen05 kernel: two launches, decode first
    st = pbs_sparse_decode_attention(q, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages,
                                     kv_dtype, num_heads, num_kv_heads, head_dim, topk, topk_row_stride, topk_k,
                                     dec_page_table, dec_pt_row_stride, dec_max_blocks, dec_seq_lens, batch,
                                     decode_query_len, block_page_stride, sparse_bt, sbt_row_stride, sparse_ctx,
                                     softmax_scale, k_scale, v_scale, out, out_row_stride, out_head_stride, lse,
                                     lse_row_stride, nullptr, 0, options, err_word, stream);
    if (st != PBS_OK) return st;
    return pbs_sparse_prefill_attention(q_pre, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages,
                                        kv_dtype, num_heads, num_kv_heads, head_dim, topk_pre, topk_row_stride,
                                        topk_k, pre_page_table, pre_pt_row_stride, pre_max_blocks, cu_seqlens_q,
                                        pre_seq_lens, num_reqs, total_q, block_page_stride, sbt_pre, sbt_row_stride,
                                        ctx_pre, softmax_scale, k_scale, v_scale, out_pre, out_row_stride,
                                        out_head_stride, lse_pre, lse_row_stride, workspace, workspace_bytes, options,
                                        err_word, stream);
  }
  // both parts on the token-centric kernel: one launch, each CTA picks its part by row
  if (opt.quarter_map) {
    st = encode_attend_map(&map, kv_cache, kv_dtype, num_kv_heads, num_pages, page_stride_bytes, true, &p.packed_map);
    if (st != PBS_OK) return st;
  }
  AttendArgs a = make_attend_args(q, q_row_stride, q_head_stride, kv_cache, page_stride_bytes, num_pages, kv_dtype,
                                  num_heads, num_kv_heads, topk, topk_row_stride, topk_k, dec_page_table,
                                  dec_pt_row_stride, dec_max_blocks, dec_seq_lens, block_page_stride, softmax_scale,
                                  k_scale, v_scale, out, out_row_stride, out_head_stride, err_word);
  a.decode_query_len = decode_query_len;
  a.num_dec_rows = static_cast<int32_t>(nd);
  a.cu_seqlens_q = cu_seqlens_q;
  a.num_reqs = num_reqs;
  a.pre_page_table = pre_page_table;
  a.pre_pt_row_stride = pre_pt_row_stride;
  a.pre_max_blocks = pre_max_blocks;
  a.pre_seq_lens = pre_seq_lens;
  a.num_rows = static_cast<int32_t>(nd + total_q);
  a.packed_map = p.packed_map;
  st = attach_table(&a, sparse_bt, sbt_row_stride, sparse_ctx);
  if (st != PBS_OK) return st;
  st = attach_lse(&a, lse, lse_row_stride);
  if (st != PBS_OK) return st;
  a.splits = choose_splits(pbs::attend_units(nd + total_q, num_kv_heads, a.group), topk_k, false, opt.splits);
  return pbs::launch_attend(a, pbs::kModeMixed, map, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PBS_OK
             : PBS_ERR_CUDA;
}

int pbs_insert_index_cache(const void* index_k, int64_t k_stride0, int64_t k_stride1, int32_t num_tokens, int32_t dim,
                           void* index_cache, int64_t c_stride0, int64_t c_stride1, int32_t num_blocks,
                           int32_t block_tokens, const int64_t* slot_mapping, int64_t slot_stride, int32_t elem_bytes,
                           int32_t* err_word, pbs_stream_t stream) {
  if (num_tokens < 0 || dim < 0 || num_blocks < 0 || block_tokens < 0) return PBS_ERR_ARG;
  if (num_tokens == 0 || dim == 0 || num_blocks == 0 || block_tokens == 0) return PBS_OK;  // empty: nothing to do
  if (index_k == nullptr || index_cache == nullptr || slot_mapping == nullptr) return PBS_ERR_ARG;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4) return PBS_ERR_ARG;
  if (k_stride0 < 0 || k_stride1 < 0 || c_stride0 < 0 || c_stride1 < 0 || slot_stride < 0) return PBS_ERR_SHAPE;
  if (!aligned(index_k, elem_bytes) || !aligned(index_cache, elem_bytes) || !aligned(slot_mapping, 8))
    return PBS_ERR_ALIGN;
  InsertArgs a = {};
  a.index_k = static_cast<const uint8_t*>(index_k);
  a.k_stride0 = k_stride0;
  a.k_stride1 = k_stride1;
  a.num_tokens = num_tokens;
  a.dim = dim;
  a.index_cache = static_cast<uint8_t*>(index_cache);
  a.c_stride0 = c_stride0;
  a.c_stride1 = c_stride1;
  a.num_blocks = num_blocks;
  a.block_tokens = block_tokens;
  a.slot_mapping = slot_mapping;
  a.slot_stride = slot_stride;
  a.elem_bytes = elem_bytes;
  a.err_word = err_word;
  return pbs::launch_insert_index_cache(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PBS_OK
                                                                                                  : PBS_ERR_CUDA;
}

}  // extern "C"
