// Host-side argument blocks and kernel launchers of libpbs (internal; not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace pbs {

struct TableArgs {
  const int32_t* topk;
  int64_t topk_row_stride;
  int32_t num_rows;
  int32_t k;
  const int32_t* page_table;
  int64_t pt_row_stride;
  int32_t max_blocks;
  const int32_t* seq_lens;
  int32_t decode_query_len;   // decode
  const int32_t* cu_seqlens_q;  // prefill
  int32_t num_reqs;             // prefill
  int32_t block_page_stride;
  int32_t* sparse_bt;
  int64_t sbt_row_stride;
  int32_t* sparse_ctx;
  int32_t* err_word;
};

cudaError_t launch_build_table(const TableArgs& a, bool prefill, cudaStream_t stream);

// Token-centric sparse attend (one query row per cluster of split CTAs, one kv head per cluster).
struct AttendArgs {
  const uint16_t* q;          // bf16 bits
  int64_t q_row_stride;
  int64_t q_head_stride;
  const uint8_t* kv_cache;
  int64_t page_stride_bytes;
  int64_t num_pages;
  int32_t kv_dtype;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t group;              // num_heads / num_kv_heads (1, 2, 4, 8 or 16)
  int32_t sub_groups;         // query-head groups of at most 8 per kv head (2 when group is 16)
  const int32_t* topk;
  int64_t topk_row_stride;
  int32_t k;
  const int32_t* page_table;
  int64_t pt_row_stride;
  int32_t max_blocks;
  const int32_t* seq_lens;
  int32_t decode_query_len;   // decode mode
  const int32_t* cu_seqlens_q;  // prefill mode
  int32_t num_reqs;
  // mixed mode: rows [0, num_dec_rows) are decode rows (page_table, seq_lens, decode_query_len
  // above), the rest prefill tokens with their own page table and sequence lengths
  int32_t num_dec_rows;
  const int32_t* pre_page_table;
  int64_t pre_pt_row_stride;
  int32_t pre_max_blocks;
  const int32_t* pre_seq_lens;
  int32_t num_rows;
  int32_t block_page_stride;
  // optional prebuilt table ([rows, >= k * 8] page ids, row stride sbt_row_stride; ctx per row):
  // non-null, the kernels attend it instead of compacting each row from top-k
  const int32_t* sparse_bt;
  int64_t sbt_row_stride;
  const int32_t* sparse_ctx;
  float scale_log2;           // softmax_scale * k_scale * log2(e)
  float v_scale;
  uint16_t* out;              // bf16 bits
  int64_t out_row_stride;
  int64_t out_head_stride;
  float* lse;                 // optional [rows, num_heads] natural-log log-sum-exp of the logits
  int64_t lse_row_stride;
  int32_t* err_word;
  int32_t splits;             // CTAs per (row, head group) = cluster size
  int32_t packed_map;         // tmap is the 5-D one-box-per-(page, head) map of a packed cache
  float* split_ws;            // non-null: splits merge through this workspace, not a cluster
  int32_t* split_tickets;     // one arrival counter per (row, head group), zero between calls
  // prefill tile kernel: V of every (request, block, kv head) converted to fp16 as a 32 KiB
  // shared-memory image, and its exponents (null: the kernel applies bf16 P as hi + lo); for fp8
  // / NVFP4 caches also K as bf16 images
  uint8_t* vconv;
  int32_t* vconv_exp;
  uint8_t* kconv;
  // prefill split between the two tcgen05 kernels (0: none): the tile kernel takes each
  // request's leading tiles of tokens before this position (1.5 x 128 k: such a token selects at
  // least two thirds of the blocks it sees, so its tile wastes few rows), the gathered-row kernel
  // every other token
  int32_t tile_pos_limit;
};

// Leading tiles of a request (q_len tokens after ctx0 tokens of context) whose last token lies
// before `limit`; with limit <= 0, all of its ceil(q_len / tok) tiles.
__host__ __device__ inline int leading_tiles(int q_len, int ctx0, int limit, int tok) {
  const int tiles = (q_len + tok - 1) / tok;
  if (limit <= 0 || ctx0 + q_len <= limit) return tiles;
  return ctx0 >= limit ? 0 : (limit - ctx0) / tok;
}

// ln 2: a base-2 log-sum-exp (what the kernels track) times this is the natural-log one.
constexpr float kLn2 = 0.693147180559945309f;

// Work units of the token-centric attend: (row, head group) pairs, a head group being the query
// heads of one kv head (two groups of 8 when a kv head serves 16).
inline int64_t attend_units(int64_t rows, int num_kv_heads, int group) {
  return rows * num_kv_heads * (group > 8 ? group / 8 : 1);
}

// Workspace of the split decode / token-centric prefill: per (unit, chunk) a partial (1040
// floats) from the front, one int32 ticket per unit at the end of the caller's buffer. Sized for
// up to kMaxSplits chunks.
constexpr int kMaxSplits = 8;
constexpr size_t kWsPartialBytes = (8 * 128 + 16) * sizeof(float);
inline size_t attend_workspace_bytes(int64_t units) {
  return static_cast<size_t>(units) * kMaxSplits * kWsPartialBytes + static_cast<size_t>(units) * sizeof(int32_t);
}

// Launch the attend; `tmap` is a tensor map over the cache rows for the bf16/fp8 formats
// (unused for NVFP4): 4-D (one box per quarter / half row) or, with a.packed_map, 5-D (one box
// per page and head). `mode`: kModeDecode, kModePrefill or kModeMixed (decode rows then prefill
// tokens in one launch). Returns the launch status.
constexpr int kModeDecode = 0;
constexpr int kModePrefill = 1;
constexpr int kModeMixed = 2;
cudaError_t launch_attend(const AttendArgs& a, int mode, const CUtensorMap& tmap, cudaStream_t stream);

// Prefill attend on tcgen05 tensor cores (GQA 8 or 16, top-k <= 16, page tables up to 65535
// blocks, 16-byte aligned q/out rows): a packed bf16 cache, or (with the workspace) an fp8 /
// NVFP4 cache through converted images. `kv_map` is the per-block map of a packed bf16 cache (one
// {64, 16, 1, 8, 2} box per 128-key block of one kv head; unused for fp8 / NVFP4); `q_map` a 3-D
// tensor map {head_dim, heads, tokens} with a {64, G, 128 / G} box.
bool prefill_tc_supported(const AttendArgs& a, bool with_workspace);
// Bytes of the tile kernel's workspace (0: arguments out of range): one 32 KiB fp16 V image
// (kTileVBytes) per (request, block, kv head), then one int32 exponent each (rounded up to 256
// bytes), then for fp8 / NVFP4 one 32 KiB bf16 K image each.
constexpr int64_t kTileVBytes = 32768;
size_t prefill_tc_workspace_bytes(int64_t num_reqs, int64_t num_kv_heads, int64_t max_blocks, int kv_dtype);
cudaError_t launch_prefill_tc(const AttendArgs& a, const CUtensorMap& kv_map, const CUtensorMap& q_map,
                              cudaStream_t stream);

// Prefill attend by key block (tcgen05; bf16 packed cache, or fp8 / NVFP4 through converted
// images; GQA 8 or 16): the tile kernel's conversion kernels write the V (and fp8 / NVFP4 K)
// images, an index kernel buckets each 256-token window's tokens by selected block, a
// persistent kernel attends every (block, kv head) bucket 16 gathered tokens at a time and
// stores one partial per (token, block), and a merge kernel combines each token's partials.
// Workspace (caller-owned): the images, then per segment of tokens the fp16 partials and their
// (log2-sum-exp, exponent) pairs, per-token partial counts and the buckets. A call is processed
// in segments of at most `gather_segment_tokens` tokens, one index + attend + merge launch each.
constexpr int kGatherWinTok = 512;      // tokens per window (request-relative)
constexpr int kGatherMaxBlocks = 8192;  // page-table width the index kernel's histogram covers
constexpr int64_t kGatherMaxSegment = int64_t(1) << 19;

struct GatherWs {
  uint16_t* part;      // fp16 [seg][Hkv][k][G][128]: per-(token, block) output / l * 2^-e
  float2* ml;          // [seg][Hkv][k][G]: (log2-sum-exp of the block's logits, e)
  int32_t* nparts;     // [seg]: partials of each token (its distinct valid blocks)
  int32_t* pairs;      // bucket entries: segment token << 12 | (partials - 1) << 6 | partial slot
  int4* chunks;        // [windows][ccap]: (block | kv head << 13, first entry, tokens, physical block)
  int32_t* wins;       // [windows][8]: request, first token, context, seq_len, chunks
  int32_t T0, T1;      // segment [T0, T1) of the call's tokens
  int32_t num_win;     // windows of the segment (upper bound; surplus ones are empty)
  int32_t ccap;        // chunk records per window
  int32_t tok_per_chunk;
};

bool prefill_gather_supported(const AttendArgs& a);
size_t gather_workspace_bytes(int64_t seg_tokens, int num_reqs, int num_heads, int num_kv_heads, int k,
                              int max_blocks);
// Tokens per segment a workspace of `ws_bytes` allows (0: not even one window).
int64_t gather_segment_tokens(int64_t total_q, int num_reqs, int num_heads, int num_kv_heads, int k, int max_blocks,
                              size_t ws_bytes);
// `kv_map`: the per-block map of a packed bf16 cache (as for the tile kernel; unused for fp8 /
// NVFP4); `q_map`: {128, heads, tokens} with a {64, G, 1} box.
// `tile_q_map`: the tile kernel's Q map, with which the tile kernel takes the call's leading tiles
// when it can run the call (AttendArgs::tile_pos_limit); null: the gathered-row kernel takes all.
cudaError_t launch_prefill_gather(const AttendArgs& a, const CUtensorMap& kv_map, const CUtensorMap& q_map,
                                  const CUtensorMap* tile_q_map, void* ws, size_t ws_bytes, cudaStream_t stream);
// The conversion kernels of both tcgen05 prefill kernels: V (and for fp8 / NVFP4 caches K) of
// every (request, block, kv head) into a.vconv / a.vconv_exp (/ a.kconv).
cudaError_t launch_convert_images(const AttendArgs& a, cudaStream_t stream);
// The tile kernel's attend alone, on images already converted (a.vconv set).
cudaError_t launch_prefill_tc_attend(const AttendArgs& a, const CUtensorMap& kv_map, const CUtensorMap& q_map,
                                     cudaStream_t stream);

// Index-cache insert.
struct InsertArgs {
  const uint8_t* index_k;
  int64_t k_stride0, k_stride1;  // elements
  int32_t num_tokens, dim;
  uint8_t* index_cache;
  int64_t c_stride0, c_stride1;  // elements
  int32_t num_blocks, block_tokens;
  const int64_t* slot_mapping;
  int64_t slot_stride;
  int32_t elem_bytes;
  int32_t* err_word;
};

cudaError_t launch_insert_index_cache(const InsertArgs& a, cudaStream_t stream);

}  // namespace pbs
