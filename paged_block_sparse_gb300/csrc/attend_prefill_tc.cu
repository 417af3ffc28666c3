// Prefill attend on the 5th-generation tensor cores (tcgen05 + TMEM), bf16 KV cache, GQA 8 or 16.
//
// What it computes (vLLM page vllm.models.minimax_m3.nvidia.sparse_attention_flashinfer, forward:
// the varlen msa_sparse_attention call; row rule of vllm.models.minimax_m3.amd.ops.sparse_pa,
// _write_sparse_block_table_row_from_values): for every prefill token and query head h of kv
// head g, out = v_scale * softmax(softmax_scale * k_scale * q_h K^T) V over the keys of the
// 128-token blocks the token's top-k selects (block b valid iff 0 <= b <= pos/128; the own
// block truncated at pos).
//
// GB300 design
// ------------
// * A tile is 16 consecutive tokens of one request and one kv head x 8 query heads, or 8 tokens
//   x 16 heads, = 128 rows, one MMA M-tile. The tile's selected blocks are merged into a sorted
//   union; every union block is streamed once and each row is masked by its own token's
//   selection.
// * Persistent: one CTA per SM walks a list of tiles, longest first. Warp 2 (scheduler) writes
//   the description of the tile after next (request, tokens, per-token 128-bit block sets, the
//   union) into one of two shared-memory slots and loads each tile's Q (3-D tensor map). The
//   rings, the S buffers and the MMA order run on across tiles.
// * Warps 0 and 3: TMA producers. Warp 0 streams the K of each union block, warp 3 its V, each
//   through its own 3-stage ring, one 32 KiB copy per block: K (and V without a workspace)
//   through a 5-D map {64 elements, 16 rows, kv head, page, row quarter} over the packed cache,
//   128B swizzle; with a workspace, V as the block's fp16 image that convert_v_kernel wrote
//   there. A stage is [64-dim quarter][128 keys][128 B]: 8-key groups 1 KiB apart, the block's
//   second 64 dims 16 KiB further. Warp 1: one thread issues the tcgen05 MMAs, S two blocks
//   ahead of PV. Warps 4-11: softmax and epilogue, two warps per TMEM lane quadrant.
// * TMEM (512 columns): S triple buffer (3 x 128, fp32) and the O accumulator (128, fp32). Each
//   softmax part rewrites its own 64 S columns with P once all 64 S values are in its registers:
//   fp16 P in the first 32 (converted-V path), or bf16 hi in the first 32 and lo in the last 32.
// * S = Q K^T: A = Q (K-major smem), B = K tile (K-major smem), bf16. O += P V: A = P read from
//   TMEM, B = V tile (MN-major smem). Converted-V path: V * 2^-e per block in fp16 (exact), P as
//   P * 2^(e - E) in fp16 against a per-tile reference E, one MMA per 16 keys. Otherwise P is
//   split into bf16 hi + lo halves, two MMAs. Either way the result stays within 2e-3 relative
//   RMS of the fp64 attend (bf16 P alone would not).
// * The MMAs of one thread execute in issue order, so S(i) may reuse the buffer whose P(i-3)
//   was read by PV(i-3), issued before it; the softmax of block i waits only for S(i), and for
//   PV(i-1) when it has to rescale O. K stages are released when S has read them, V stages when
//   PV has, so K is fetched up to three blocks ahead of S.
// * Online softmax in base 2 with lazy rescaling: the O row is rescaled only when the running
//   maximum grows by more than 2^8, so most blocks never touch O from the CUDA cores.
// * A token's top-k row is a set of blocks: an id listed twice counts once, as in the table
//   builders and the token-centric kernel.
#include <algorithm>

#include "pbs_device.cuh"
#include "pbs_internal.h"
#include "tc_device.cuh"

namespace pbs {
namespace {

// A tile is 128 rows = the MMA M: kTok tokens x kG query heads of one kv head, kG = 8 (16
// tokens) or 16 (8 tokens). Rows are token-major: row = token * kG + head.
constexpr int kRows = 128;
constexpr int kTokMax = 16;
constexpr int kSplit = 2;                        // softmax warps per TMEM lane quadrant
constexpr int kW = 128 / kSplit;                 // S columns (keys) per softmax thread
constexpr int kSoftWarps = 4 * kSplit;
constexpr int kThreadsTc = 32 * (4 + kSoftWarps);
constexpr int kQBytes = kRows * kHeadDim * 2;          // 32 KiB
constexpr int kHalf = 128 * 128;                       // one 64-dim half of a 128 x 128 bf16 tile
constexpr int kTileBytes = 2 * kHalf;                  // 32 KiB: a block's K, or its V
constexpr int kStagesTc = 3;                           // stages of the K ring and of the V ring
constexpr int kSBuf = 3;                               // S buffers in TMEM (S runs 2 blocks ahead of PV)
constexpr int kBigBytes = kQBytes + 2 * kStagesTc * kTileBytes;  // 224 KiB
// Union entries per tile descriptor. A tile's union (at most 16 tokens x top-k 16 = 256 distinct
// blocks) spans one or two descriptors; block ids travel as 16 bits, so page tables may be up to
// kTcMaxBlocks blocks wide.
constexpr int kMaxUnion = 128;
constexpr int kTcMaxBlocks = 65535;
constexpr int kTcMaxTopk = 16;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (factor 256)
// fp16-V path: P' = P * 2^(e_b - E) in fp16. P <= 2^8 under the lazy rescale, so e_b - E <= 7 keeps
// P' below 2^15; below -8 the block's largest weights would leave fp16's normal range. Outside
// that window E moves to e_b and O is rescaled by the power of two.
constexpr int kExpUp = 7, kExpDown = -8;

// One descriptor, written by the scheduler warp for the other roles (two slots, used
// alternately): a tile's tokens and up to kMaxUnion entries of its sorted union of selected
// blocks. A tile whose union is longer continues in the next descriptor (`more` here, `cont`
// there): same tokens, O and the softmax state carry on, Q stays loaded.
struct TileDesc {
  int32_t end;  // no tile: the CTA's list is done
  int32_t req, g, t0, n_tok, c0, ctx0, pos_last;  // request, kv head, first token row, tokens, ...
  int32_t n_union;                   // entries in this descriptor
  int32_t bad_mask;                  // tokens whose row could not be read (the row attends nothing)
  int32_t cont;                      // continues the previous descriptor's tile
  int32_t more;                      // the tile continues in the next descriptor
  int32_t by_block;                  // masks are indexed by block id (all of the tile's blocks < 128)
  int32_t own[kTokMax];              // own block of each token (-1: none)
  int16_t lim[kTokMax];              // keys of the own block the token sees
  uint16_t union_blk[kMaxUnion];     // the entries' blocks, increasing
  // bit x of masks[t]: token t selected the block of entry x of this descriptor (by_block 0) or
  // block x (by_block 1)
  uint32_t masks[kTokMax][kMaxUnion / 32];
  int8_t vexp[kMaxUnion];            // fp16-V path: the entry's V image is V * 2^-vexp
};

// Roles that read a tile slot and release it: the two TMA warps, the MMA thread, the softmax warps.
constexpr uint32_t kTileUsers = 3 + kSoftWarps;

struct TcCtl {
  uint64_t q_full;
  uint64_t q_empty;  // the S MMAs of the tile whose Q sits in shared memory have completed
  // K and V stream through separate rings: a K stage is free once S has read it, a V stage once
  // PV has, so K can be loaded three blocks ahead of S while S runs two blocks ahead of PV
  uint64_t k_full[kStagesTc];
  uint64_t k_empty[kStagesTc];
  uint64_t v_full[kStagesTc];
  uint64_t v_empty[kStagesTc];
  uint64_t s_full[kSBuf];
  // per S buffer (block i of the CTA's block sequence uses buffer i % 3): P(i) written, PV(i)
  // done. A barrier cannot be lapped: block i + 3 needs S(i + 3), which the MMA thread issues only
  // after PV(i).
  uint64_t p_full[kSBuf];
  uint64_t pv_done[kSBuf];
  uint64_t tile_full[2];
  uint64_t tile_empty[2];
  uint32_t tmem_base;
  int32_t abort;
  TileDesc tile[2];
  float xchg[kSplit][kRows];  // per-row partial maxima / sums exchanged within a lane quadrant
};

constexpr size_t kTcSmem = 232448;  // the per-block opt-in maximum of sm_100-family GPUs
// The big buffers start at the (1024-aligned) dynamic shared memory base; the control block
// follows them.
static_assert(kBigBytes + sizeof(TcCtl) <= kTcSmem, "shared memory layout exceeds 227 KiB");

#ifdef PBS_TRACE
// Trace build only: one CTA records SM-clock timestamps of its pipeline events.
constexpr int kTraceBlocks = 64;
enum TraceEv { kEvStart, kEvSetup, kEvEpi, kEvEnd, kEvProdIssue0, kEvProdIssue1 = kEvProdIssue0 + kTraceBlocks,
               kEvS = kEvProdIssue1 + kTraceBlocks, kEvPV = kEvS + kTraceBlocks,
               kEvSoftIn = kEvPV + kTraceBlocks, kEvSoftMax = kEvSoftIn + kTraceBlocks,
               kEvSoftOut = kEvSoftMax + kTraceBlocks, kEvDesc = kEvSoftOut + kTraceBlocks,
               kEvQ = kEvDesc + kTraceBlocks, kEvTileIn = kEvQ + kTraceBlocks, kEvTileOut = kEvTileIn + kTraceBlocks,
               kEvDesc0 = kEvTileOut + kTraceBlocks, kEvCount = kEvDesc0 + kTraceBlocks };
__device__ long long g_trace[kEvCount + 4];
__device__ int g_trace_cta;
__device__ int g_trace_b0;  // first block of the CTA's sequence the per-block events record
#define TRACE(ev) do { if (blockIdx.x == static_cast<unsigned>(g_trace_cta) && (ev) < kEvCount) \
                         g_trace[(ev)] = clock64(); } while (0)
#define TRACEB(ev, i) do { if ((i) - g_trace_b0 >= 0 && (i) - g_trace_b0 < kTraceBlocks) TRACE((ev) + (i) - g_trace_b0); } while (0)
#define TRACET(ev, i) do { if ((i) < kTraceBlocks) TRACE((ev) + (i)); } while (0)
#else
#define TRACE(ev) do { } while (0)
#define TRACEB(ev, i) do { } while (0)
#define TRACET(ev, i) do { } while (0)
#endif

// p = 2^(s * sl2 - m) for the first `nval` of this thread's kW key columns (0 beyond), written
// to TMEM as bf16 hi (over the thread's own S columns) and lo; returns the sum of p and the
// maximum of the valid s. `prefix` = some lane of the warp has a partly valid range (the own
// block), so keys are masked one by one; otherwise every lane has all or none of its keys
// valid, and a lane with none gets m = +inf (p = 0) and maximum -inf. The caller skips warps in
// which no lane has a valid key, so on the unmasked path every column holds a written key row.
template <bool kPrefix>
__device__ __forceinline__ float write_p(const uint32_t (&v)[kW], int nval, float sl2, float m, uint32_t t_hi,
                                         uint32_t t_lo, float& smax) {
  float psum0 = 0.f, psum1 = 0.f, mx = -INFINITY;
  const float mu = (!kPrefix && nval == 0) ? INFINITY : m;
#pragma unroll
  for (int c = 0; c < kW / 32; ++c) {
    uint32_t hi[16], lo[16];
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const int k = 32 * c + j;
      float s0 = __uint_as_float(v[k]), s1 = __uint_as_float(v[k + 1]);
      float p0, p1;
      if (kPrefix) {
        // columns past the valid range may hold anything (rows beyond the last token): select
        // on the results, never compute with them
        s0 = k < nval ? s0 : -INFINITY;
        s1 = k + 1 < nval ? s1 : -INFINITY;
        p0 = k < nval ? ex2(fmaf(s0, sl2, -mu)) : 0.f;
        p1 = k + 1 < nval ? ex2(fmaf(s1, sl2, -mu)) : 0.f;
      } else {
        p0 = ex2(fmaf(s0, sl2, -mu));
        p1 = ex2(fmaf(s1, sl2, -mu));
      }
      mx = fmaxf(mx, fmaxf(s0, s1));
      psum0 += p0;
      psum1 += p1;
      const uint32_t hh = pack_bf16(p0, p1);
      hi[j >> 1] = hh;
      lo[j >> 1] = pack_bf16(p0 - bf16_lo(hh), p1 - bf16_hi(hh));
    }
    tc::st16(t_hi + 16 * c, hi);
    tc::st16(t_lo + 16 * c, lo);
  }
  smax = (!kPrefix && nval == 0) ? -INFINITY : mx;
  return psum0 + psum1;
}

__device__ __forceinline__ void zero_p(uint32_t t_hi, uint32_t t_lo) {
  uint32_t z[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) z[j] = 0u;
#pragma unroll
  for (int c = 0; c < kW / 32; ++c) {
    tc::st16(t_hi + 16 * c, z);
    tc::st16(t_lo + 16 * c, z);
  }
}

// fp16-V path: p = 2^(s * sl2 - m) for the thread's kW keys as fp16 pairs over the first kW / 2
// of its own S columns; otherwise as write_p.
template <bool kPrefix>
__device__ __forceinline__ float write_p16(const uint32_t (&v)[kW], int nval, float sl2, float m, uint32_t t_p,
                                           float& smax) {
  float psum0 = 0.f, psum1 = 0.f, mx = -INFINITY;
  const float mu = (!kPrefix && nval == 0) ? INFINITY : m;
#pragma unroll
  for (int c = 0; c < kW / 32; ++c) {
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const int k = 32 * c + j;
      float s0 = __uint_as_float(v[k]), s1 = __uint_as_float(v[k + 1]);
      float p0, p1;
      if (kPrefix) {
        s0 = k < nval ? s0 : -INFINITY;
        s1 = k + 1 < nval ? s1 : -INFINITY;
        p0 = k < nval ? ex2(fmaf(s0, sl2, -mu)) : 0.f;
        p1 = k + 1 < nval ? ex2(fmaf(s1, sl2, -mu)) : 0.f;
      } else {
        p0 = ex2(fmaf(s0, sl2, -mu));
        p1 = ex2(fmaf(s1, sl2, -mu));
      }
      mx = fmaxf(mx, fmaxf(s0, s1));
      psum0 += p0;
      psum1 += p1;
      pk[j >> 1] = pack_f16(p0, p1);
    }
    tc::st16(t_p + 16 * c, pk);
  }
  smax = (!kPrefix && nval == 0) ? -INFINITY : mx;
  return psum0 + psum1;
}

__device__ __forceinline__ void zero_p16(uint32_t t_p) {
  uint32_t z[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) z[j] = 0u;
#pragma unroll
  for (int c = 0; c < kW / 32; ++c) tc::st16(t_p + 16 * c, z);
}

// 2^n as a float, exact for -126 <= n <= 127.
__device__ __forceinline__ float exp2i(int n) { return __uint_as_float(static_cast<uint32_t>(127 + n) << 23); }

// O columns [col, col + kW) of this warp's 32 rows times f.
__device__ __forceinline__ void scale_o(uint32_t t_o, float f) {
#pragma unroll
  for (int c = 0; c < kW / 32; ++c) {
    uint32_t o[32];
    tc::ld32(t_o + 32 * c, o);
    tc::wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
    tc::st32(t_o + 32 * c, o);
  }
}

__device__ __forceinline__ void quad_bar(int quad) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + quad), "r"(32 * kSplit) : "memory");
}

// The quadrant's warps meet at their named barrier and agree whether any thread passed true.
__device__ __forceinline__ bool quad_any(int quad, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(1 + quad), "r"(32 * kSplit)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_5d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1, int c2, int c3,
                                            int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Waits in this kernel last microseconds; give up after 100 ms.
constexpr unsigned long long kTcWaitNs = 100000000ull;

// Bounded wait that records a timeout and raises the CTA's abort flag.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, TcCtl* ctl, int32_t* err) {
  if (mbar_wait_bounded(bar, parity, kTcWaitNs)) return true;
  set_err(err, PBS_DEVERR_TIMEOUT);
  atomicExch(&ctl->abort, 1);
  return false;
}

// Same, for a whole warp that must stay converged (the softmax warps issue warp-collective
// tcgen05.ld / st): every lane waits, and the warp agrees on the result.
__device__ __forceinline__ bool warp_wait_or_abort(uint64_t* bar, uint32_t parity, TcCtl* ctl, int32_t* err) {
  const bool ok = wait_or_abort(bar, parity, ctl, err);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool aborted(TcCtl* ctl) { return *reinterpret_cast<volatile int32_t*>(&ctl->abort) != 0; }

// fp16-V path, before the attend: the V of block b of request r and kv head g (CTA (b, r, g))
// as the 32 KiB shared-memory image a V stage holds ([64-dim quarter][128 keys][128 B], 128B
// swizzle: 16-byte chunk c of key k at chunk c ^ (k % 8)), in fp16 as V * 2^-e with e putting
// the block's max |V| at 2^14..2^15 (exact: bf16 has 8 significant bits and fp16 keeps 28
// binades below its maximum normal). Keys past the request's last token, or on pages past the
// cache, become zeros. Thread t converts key t.
__global__ void __launch_bounds__(128) convert_v_kernel(const AttendArgs a) {
  const int b = blockIdx.x, r = blockIdx.y, g = blockIdx.z, t = threadIdx.x;
  const int seq_len = __ldg(a.seq_lens + r);
  if (b * kSparseBlock >= seq_len) return;  // no token of the request sees this block
  const int nv = min(kSparseBlock, seq_len - b * kSparseBlock);
  const int64_t page = static_cast<int64_t>(__ldg(a.page_table + static_cast<int64_t>(r) * a.pt_row_stride + b)) *
                           a.block_page_stride + t / kPageRows;
  const bool in_cache = page >= 0 && page < a.num_pages;
  if (t < nv && !in_cache) set_err(a.err_word, PBS_DEVERR_PAGE_OOB);
  uint32_t x[16][4];
  uint32_t mx2 = 0u;
  if (t < nv && in_cache) {
    // the V half (bytes 256..511) of the key's 512-byte row of this kv head
    const uint4* src = reinterpret_cast<const uint4*>(a.kv_cache + page * a.page_stride_bytes + g * 8192 +
                                                      (t % kPageRows) * 512 + 256);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 u = __ldg(src + c);
      x[c][0] = u.x;
      x[c][1] = u.y;
      x[c][2] = u.z;
      x[c][3] = u.w;
    }
  } else {
#pragma unroll
    for (int c = 0; c < 16; ++c) x[c][0] = x[c][1] = x[c][2] = x[c][3] = 0u;
  }
  // |bf16| bit patterns compare like the magnitudes
#pragma unroll
  for (int c = 0; c < 16; ++c)
#pragma unroll
    for (int q = 0; q < 4; ++q) mx2 = max(mx2, max((x[c][q] & 0x7fff7fffu) >> 16, x[c][q] & 0x7fffu));
  __shared__ uint32_t wmax[4];
  uint32_t mx = __reduce_max_sync(0xffffffffu, mx2);
  if ((t & 31) == 0) wmax[t >> 5] = mx;
  __syncthreads();
  mx = max(max(wmax[0], wmax[1]), max(wmax[2], wmax[3]));
  const float vm = __uint_as_float(mx << 16);
  int e = 0;
  if (vm > 0.f) e = static_cast<int>((__float_as_uint(vm) >> 23) & 0xffu) - 127 - 14;
  e = max(-100, min(100, e));
  const float sc = exp2i(-e);
  uint8_t* dst = a.vconv + ((static_cast<int64_t>(r) * a.max_blocks + b) * a.num_kv_heads + g) * kTileBytes;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const int q = c >> 3, c8 = c & 7;
    *reinterpret_cast<uint4*>(dst + q * kHalf + t * 128 + ((c8 ^ (t & 7)) << 4)) =
        make_uint4(pack_f16(bf16_lo(x[c][0]) * sc, bf16_hi(x[c][0]) * sc),
                   pack_f16(bf16_lo(x[c][1]) * sc, bf16_hi(x[c][1]) * sc),
                   pack_f16(bf16_lo(x[c][2]) * sc, bf16_hi(x[c][2]) * sc),
                   pack_f16(bf16_lo(x[c][3]) * sc, bf16_hi(x[c][3]) * sc));
  }
  if (t == 0) a.vconv_exp[(static_cast<int64_t>(r) * a.max_blocks + b) * a.num_kv_heads + g] = e;
}

// fp8 / NVFP4 caches, before the attend: K and V of block b of request r and kv head g (CTA
// (b, r, g)) as the images the tile kernel's stages hold, K as bf16 (an e4m3 value, or an e2m1
// code times its e4m3 block scale, has at most 6 significant bits and fits bf16's range: exact)
// and V as fp16 times 2^-e like convert_v_kernel (exact: the values fit fp16's normal range once
// the block's maximum sits at 2^14..2^15). The per-tensor scales stay folded as for bf16. Keys
// past the request's last token, or on pages past the cache, become zeros. Thread t converts key
// t, 8 elements (one 16-byte image chunk) at a time.
// The lower / upper half of an f16x2 word as float (exact).
__device__ __forceinline__ float f16x2_lo(uint32_t x) {
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}" : "=f"(f) : "r"(x));
  return f;
}
__device__ __forceinline__ float f16x2_hi(uint32_t x) {
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, hi;\n\t}" : "=f"(f) : "r"(x));
  return f;
}

// One side (K or V) of one key as stored: fp8 128 bytes; NVFP4 64 bytes of e2m1 codes (element
// 2i in the low nibble of byte i) and 8 e4m3 block scales (scale j covers elements 16j .. 16j + 15).
// Loaded with 16-byte (codes) and 8-byte (scales) vector loads.
template <int FMT>
struct KeySide {
  uint4 w[FMT == PBS_KV_FP8_E4M3 ? 8 : 4];
  uint2 sc;
};

template <int FMT>
__device__ __forceinline__ void load_side(const uint8_t* side, int row, KeySide<FMT>& k) {
  if (FMT == PBS_KV_FP8_E4M3) {
#pragma unroll
    for (int i = 0; i < 8; ++i) k.w[i] = __ldg(reinterpret_cast<const uint4*>(side) + i);
    k.sc = make_uint2(0u, 0u);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) k.w[i] = __ldg(reinterpret_cast<const uint4*>(side + row * 64) + i);
    k.sc = __ldg(reinterpret_cast<const uint2*>(side + 1024 + row * 8));
  }
}

__device__ __forceinline__ uint32_t word4(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Elements 8c .. 8c + 7 of a key side, dequantised to float (exact). c must be a compile-time
// constant after unrolling.
template <int FMT>
__device__ __forceinline__ void dequant8(const KeySide<FMT>& k, int c, float (&v)[8]) {
  if (FMT == PBS_KV_FP8_E4M3) {
    const uint4& q = k.w[c >> 1];
    const uint32_t lo = word4(q, 2 * (c & 1)), hi = word4(q, 2 * (c & 1) + 1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t h2 = e4m3x2_to_f16x2(((i < 2 ? lo : hi) >> (16 * (i & 1))) & 0xffffu);
      v[2 * i] = f16x2_lo(h2);
      v[2 * i + 1] = f16x2_hi(h2);
    }
  } else {
    const uint32_t w = word4(k.w[c >> 2], c & 3);
    const uint32_t sb = ((c >> 1) < 4 ? k.sc.x : k.sc.y) >> (8 * ((c >> 1) & 3));
    const float sc = f16x2_lo(e4m3x2_to_f16x2(sb & 0xffu));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t h2 = e2m1x2_to_f16x2((w >> (8 * i)) & 0xffu);
      v[2 * i] = f16x2_lo(h2) * sc;
      v[2 * i + 1] = f16x2_hi(h2) * sc;
    }
  }
}

template <int FMT>
__global__ void __launch_bounds__(128) convert_kv_kernel(const AttendArgs a) {
  const int b = blockIdx.x, r = blockIdx.y, g = blockIdx.z, t = threadIdx.x;
  const int seq_len = __ldg(a.seq_lens + r);
  if (b * kSparseBlock >= seq_len) return;  // no token of the request sees this block
  const int nv = min(kSparseBlock, seq_len - b * kSparseBlock);
  const int64_t page = static_cast<int64_t>(__ldg(a.page_table + static_cast<int64_t>(r) * a.pt_row_stride + b)) *
                           a.block_page_stride + t / kPageRows;
  const bool in_cache = page >= 0 && page < a.num_pages;
  if (t < nv && !in_cache) set_err(a.err_word, PBS_DEVERR_PAGE_OOB);
  const bool live = t < nv && in_cache;
  const int row = t % kPageRows;
  const uint8_t* base = a.kv_cache + (live ? page : 0) * a.page_stride_bytes;
  // fp8: [Hkv][16 rows][K 128 B | V 128 B]; NVFP4: [2 Hkv slots of 1152 B], slot 2g = K, 2g + 1 = V
  const uint8_t* kside = FMT == PBS_KV_FP8_E4M3 ? base + g * 4096 + row * 256 : base + (2 * g) * 1152;
  const uint8_t* vside = FMT == PBS_KV_FP8_E4M3 ? kside + 128 : kside + 1152;
  KeySide<FMT> ks, vs;
  if (live) {
    load_side<FMT>(kside, row, ks);
    load_side<FMT>(vside, row, vs);
  }
  const int64_t image = (static_cast<int64_t>(r) * a.max_blocks + b) * a.num_kv_heads + g;
  // K: bf16 image
  uint8_t* kdst = a.kconv + image * kTileBytes;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    float v[8];
    if (live) dequant8<FMT>(ks, c, v);
    else
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    const int q = c >> 3, c8 = c & 7;
    *reinterpret_cast<uint4*>(kdst + q * kHalf + t * 128 + ((c8 ^ (t & 7)) << 4)) =
        make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
  }
  // V: the block's maximum |V|, then fp16 V * 2^-e
  float mx = 0.f;
  if (live) {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      float v[8];
      dequant8<FMT>(vs, c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(v[i]));
    }
  }
  __shared__ float wmax[4];
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  if ((t & 31) == 0) wmax[t >> 5] = mx;
  __syncthreads();
  mx = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
  int e = 0;
  if (mx > 0.f) e = static_cast<int>((__float_as_uint(mx) >> 23) & 0xffu) - 127 - 14;
  e = max(-100, min(100, e));
  const float sc = exp2i(-e);
  uint8_t* vdst = a.vconv + image * kTileBytes;
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    float v[8];
    if (live) dequant8<FMT>(vs, c, v);
    else
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    const int q = c >> 3, c8 = c & 7;
    *reinterpret_cast<uint4*>(vdst + q * kHalf + t * 128 + ((c8 ^ (t & 7)) << 4)) =
        make_uint4(pack_f16(v[0] * sc, v[1] * sc), pack_f16(v[2] * sc, v[3] * sc), pack_f16(v[4] * sc, v[5] * sc),
                   pack_f16(v[6] * sc, v[7] * sc));
  }
  if (t == 0) a.vconv_exp[image] = e;
}

// ---- the scheduler warp's tile union --------------------------------------------------------
// A tile's (token, selected block) pairs as 256 keys block << 16 | 1 << token, held 8 per lane
// (element e = 32 r + lane), sorted by a bitonic network; runs of one block are then ORed into
// their first element (the run's head), which also gets the block's index in the tile's union.
constexpr uint32_t kNoKey = 0xffffffffu;

// Compare-exchange of elements (r, lane) and (r ^ RJ, lane) of one lane (a stage of distance
// 32 RJ), ascending where bit k of the element index is clear.
template <int RJ>
__device__ __forceinline__ void bitonic_in_lane(uint32_t (&key)[8], int lane, int k) {
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    if (r & RJ) continue;
    const bool up = ((32 * r + lane) & k) == 0;
    const uint32_t x = key[r], y = key[r | RJ];
    const bool sw = up ? (x > y) : (x < y);
    key[r] = sw ? y : x;
    key[r | RJ] = sw ? x : y;
  }
}

// Bitonic sort of the 256 keys, ascending (element e = 32 r + lane). The stages run as loops, so
// the scheduler's code stays small next to the pipeline's hot loops.
__device__ __forceinline__ void sort_keys(uint32_t (&key)[8], int lane) {
#pragma unroll 1
  for (int k = 2; k <= 256; k <<= 1) {
#pragma unroll 1
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 32) {
        if (j == 32) bitonic_in_lane<1>(key, lane, k);
        else if (j == 64) bitonic_in_lane<2>(key, lane, k);
        else bitonic_in_lane<4>(key, lane, k);
      } else {
        const bool lower = (lane & j) == 0;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const bool up = ((32 * r + lane) & k) == 0;
          const uint32_t other = __shfl_xor_sync(0xffffffffu, key[r], j);
          key[r] = (lower == up) ? min(key[r], other) : max(key[r], other);
        }
      }
    }
  }
}

// acc[e] |= acc[e + d] for every element whose element e + d holds the same block (sorted keys:
// then so does every element between them); after d = 1, 2, ..., 128 each element holds the OR of
// its run's tail.
template <int RD>
__device__ __forceinline__ void run_or_in_lane(const uint32_t (&key)[8], uint32_t (&acc)[8]) {
#pragma unroll
  for (int r = 0; r < 8 - RD; ++r) {
    // ascending r: acc[r + RD] is still the value before this step
    const bool same = key[r] != kNoKey && key[r + RD] != kNoKey && (key[r + RD] >> 16) == (key[r] >> 16);
    acc[r] |= same ? acc[r + RD] : 0u;
  }
}

__device__ __forceinline__ void run_or(const uint32_t (&key)[8], uint32_t (&acc)[8], int lane) {
#pragma unroll 1
  for (int d = 1; d < 32; d <<= 1) {
    const int src = (lane + d) & 31;
    const bool same_reg = lane + d < 32;
    uint32_t nacc[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const uint32_t k0 = __shfl_sync(0xffffffffu, key[r], src), a0 = __shfl_sync(0xffffffffu, acc[r], src);
      const uint32_t k1 = __shfl_sync(0xffffffffu, key[(r + 1) & 7], src);
      const uint32_t a1 = __shfl_sync(0xffffffffu, acc[(r + 1) & 7], src);
      const uint32_t ok_key = same_reg ? k0 : (r + 1 < 8 ? k1 : kNoKey);
      const uint32_t ok_acc = same_reg ? a0 : a1;
      const bool same = key[r] != kNoKey && ok_key != kNoKey && (ok_key >> 16) == (key[r] >> 16);
      nacc[r] = acc[r] | (same ? ok_acc : 0u);
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) acc[r] = nacc[r];
  }
  run_or_in_lane<1>(key, acc);
  run_or_in_lane<2>(key, acc);
  run_or_in_lane<4>(key, acc);
}

struct TileUnion {
  uint32_t key[8];  // sorted keys; at a head, the low 16 bits hold the OR of the run's token bits
  int32_t u[8];     // union index of a head element
  uint32_t heads;   // bit r: element (r, lane) heads its block's run
  int32_t n;        // distinct blocks of the tile
  bool direct;      // the tile's only descriptor is already written (blocks below 128: masks)
};

// The tile's request and tokens (flat tile f of the CTA's list: kv head f % Hkv of request tile
// tiles - 1 - f / Hkv, request tiles numbered request by request, so the list starts at the
// last request's last tiles, whose tokens see the most blocks), each token's own block and
// visible keys of it, and the sorted union of the tokens' selections. Lane t < kTok owns token
// t's row; the rest of the warp helps with the loads, the sort and the scans.
template <int kTok, bool kF16V>
__device__ __forceinline__ void build_tile(const AttendArgs& a, int f, int total_tiles, int lane, TileDesc* d,
                                           TileUnion& un) {
  const int g = f % a.num_kv_heads;
  const int rt = total_tiles - 1 - f / a.num_kv_heads;
  int r = -1, t0 = 0, n = 0, c0 = 0, ctx0 = 0, seq_len = 0;
  int base_tiles = 0;
  for (int r0 = 0; r0 < a.num_reqs && r < 0; r0 += 32) {
    const int rr = r0 + lane;
    // every lane loads its request's bounds and length at once (one round trip)
    int q_len = 0, cb = 0, sl = 0;
    if (rr < a.num_reqs) {
      cb = __ldg(a.cu_seqlens_q + rr);
      q_len = __ldg(a.cu_seqlens_q + rr + 1) - cb;
      sl = __ldg(a.seq_lens + rr);
    }
    const int tiles = rr < a.num_reqs ? leading_tiles(q_len, sl - q_len, a.tile_pos_limit, kTok) : 0;
    int incl = tiles;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    const int excl = incl - tiles + base_tiles;
    const uint32_t hit = __ballot_sync(0xffffffffu, rt >= excl && rt < excl + tiles);
    if (hit) {
      const int src = __ffs(hit) - 1;
      r = r0 + src;
      const int tile = rt - __shfl_sync(0xffffffffu, excl, src);
      const int ql = __shfl_sync(0xffffffffu, q_len, src);
      c0 = __shfl_sync(0xffffffffu, cb, src);
      seq_len = __shfl_sync(0xffffffffu, sl, src);
      ctx0 = seq_len - ql;
      t0 = c0 + tile * kTok;
      n = min(kTok, ql - tile * kTok);
    }
    base_tiles += __shfl_sync(0xffffffffu, incl, 31);
  }
  if (r < 0) n = 0;
  // lane t < n: token t's selected blocks (ids[j], -1 where none), its own block and the keys of
  // it the token sees
  int ids[kTcMaxTopk];
  int own = -1, lim = 0;
  bool bad = false;
#pragma unroll
  for (int j = 0; j < kTcMaxTopk; ++j) ids[j] = -1;
  if (a.sparse_bt == nullptr) {
    if (lane < n) {
      const int pos = ctx0 + (t0 + lane - c0);
      const int causal_len = pos + 1 > 0 ? pos + 1 : 0;
      own = causal_len > 0 ? pos / kSparseBlock : -1;
      lim = own >= 0 ? causal_len - own * kSparseBlock : 0;
      const int32_t* row = a.topk + static_cast<int64_t>(t0 + lane) * a.topk_row_stride;
#pragma unroll
      for (int j = 0; j < kTcMaxTopk; ++j) {
        const int b = j < a.k ? __ldg(row + j) : -1;
        if (b >= 0 && b <= own) {
          if (b >= a.max_blocks) bad = true;
          else ids[j] = b;  // a repeated id gives the same key twice: the run OR merges it
        }
      }
      // a row with an out-of-range id contributes nothing (its output is zero, the error recorded)
      if (bad) set_err(a.err_word, PBS_DEVERR_BLOCK_OOB);
    }
  } else {
    // Prebuilt table: slot j of the token's row lists the pages of one block; the block is found
    // by walking the request's page-table row (a slot's first page is page_table[r][b] *
    // block_page_stride). Keys of slot j: min(128, ctx - 128 j), so only the last slot can be
    // partial; it plays the own block's part (lim keys).
    int first[kTcMaxTopk];
    int n_slots = 0, tctx = 0;
    if (lane < n) {
      tctx = __ldg(a.sparse_ctx + t0 + lane);
      if (tctx < 0 || tctx > a.k * kSparseBlock) {
        bad = true;
        tctx = 0;
      }
      n_slots = (tctx + kSparseBlock - 1) / kSparseBlock;
    }
    const int32_t* trow = a.sparse_bt + static_cast<int64_t>(t0 + min(lane, max(n - 1, 0))) * a.sbt_row_stride;
#pragma unroll
    for (int j = 0; j < kTcMaxTopk; ++j) first[j] = j < n_slots ? __ldg(trow + j * kPagesPerBlock) : -1;
    // the last block any of the tile's tokens can see bounds the walk
    const int pos_max = ctx0 + (t0 + max(n, 1) - 1 - c0);
    const int walk = min(a.max_blocks, pos_max >= 0 ? pos_max / kSparseBlock + 1 : 0);
    const int32_t* pt_row = a.page_table + static_cast<int64_t>(max(r, 0)) * a.pt_row_stride;
    for (int b0 = 0; b0 < walk; b0 += 32) {
      const int bb = b0 + lane;
      const int64_t base64 = bb < walk ? static_cast<int64_t>(__ldg(pt_row + bb)) * a.block_page_stride : -1;
      const int base = base64 >= 0 && base64 <= 0x7fffffffLL ? static_cast<int>(base64) : -2;
      const int nj = min(32, walk - b0);
      for (int j = 0; j < nj; ++j) {
        const int x = __shfl_sync(0xffffffffu, base, j);
#pragma unroll
        for (int sl = 0; sl < kTcMaxTopk; ++sl)
          if (ids[sl] < 0 && first[sl] == x) ids[sl] = b0 + j;
      }
    }
    if (lane < n && !bad) {
      uint32_t seen[4] = {0u, 0u, 0u, 0u};  // blocks of this row so far, hashed to 128 bits
#pragma unroll
      for (int sl = 0; sl < kTcMaxTopk; ++sl) {
        if (sl < n_slots) {
          // a slot that names no block of the request makes the row unreadable
          const int b = ids[sl];
          bad |= b < 0;
          if (b >= 0) {
            // a block in two slots is no table the builders write (a row is a set of blocks)
            const uint32_t bit = 1u << (b & 31);
            const int w = (b >> 5) & 3;
            for (int sl2 = 0; sl2 < sl; ++sl2) bad |= ids[sl2] == b && (seen[w] & bit) != 0;
            seen[w] |= bit;
          }
          if (sl == n_slots - 1) {
            own = b;
            lim = tctx - sl * kSparseBlock;
          }
        } else {
          ids[sl] = -1;
        }
      }
      // every page a slot's keys reach must be the block's own page (the kernel copies the block)
      for (int sl = 0; sl < n_slots && !bad; ++sl) {
        const int fp = __ldg(trow + sl * kPagesPerBlock);
        const int keys = min(kSparseBlock, tctx - sl * kSparseBlock);
        for (int j = 1; j < (keys + kPageRows - 1) / kPageRows; ++j) bad |= __ldg(trow + sl * kPagesPerBlock + j) != fp + j;
      }
    }
    if (lane >= n) {
#pragma unroll
      for (int j = 0; j < kTcMaxTopk; ++j) ids[j] = -1;
    }
    if (lane < n && bad) set_err(a.err_word, PBS_DEVERR_TABLE);
  }
  if (bad) {
#pragma unroll
    for (int j = 0; j < kTcMaxTopk; ++j) ids[j] = -1;
  }
  const uint32_t bad_mask = __ballot_sync(0xffffffffu, bad && lane < n);
  // the last block any token of the tile can see
  const int pos_max = ctx0 + (t0 + max(n, 1) - 1 - c0);
  const int own_max = pos_max >= 0 ? pos_max / kSparseBlock : -1;
  un.heads = 0u;
  const uint32_t lt = lanemask_lt();
  un.direct = false;
  if (own_max < 128) {
    // every selected block is below 128: each token's blocks as a 128-bit set (a repeated id sets
    // the same bit) that the softmax warps test per block, and the union, the OR of the sets,
    // listed in increasing order straight into the tile's only descriptor
    uint32_t m0 = 0u, m1 = 0u, m2 = 0u, m3 = 0u;
#pragma unroll
    for (int j = 0; j < kTcMaxTopk; ++j) {
      const int b = ids[j];
      if (b >= 0) {
        const uint32_t bit = 1u << (b & 31);
        m0 |= (b >> 5) == 0 ? bit : 0u;
        m1 |= (b >> 5) == 1 ? bit : 0u;
        m2 |= (b >> 5) == 2 ? bit : 0u;
        m3 |= (b >> 5) == 3 ? bit : 0u;
      }
    }
    if (lane < kTok) {
      d->masks[lane][0] = m0;
      d->masks[lane][1] = m1;
      d->masks[lane][2] = m2;
      d->masks[lane][3] = m3;
    }
    int nu = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint32_t word = __reduce_or_sync(0xffffffffu, w == 0 ? m0 : w == 1 ? m1 : w == 2 ? m2 : m3);
      if ((word >> lane) & 1u) {
        const int u = nu + __popc(word & lt), b = 32 * w + lane;
        d->union_blk[u] = static_cast<uint16_t>(b);
        if (kF16V)
          d->vexp[u] = static_cast<int8_t>(
              __ldg(a.vconv_exp + (static_cast<int64_t>(r) * a.max_blocks + b) * a.num_kv_heads + g));
      }
      nu += __popc(word);
    }
    un.n = nu;
    un.direct = true;
  } else {
    // keys: lane l holds token l % kTok's ids j = l / kTok + (32 / kTok) r; sorted, then each run
    // of one block ORed into its head
    constexpr int kLpt = 32 / kTok;
    const int tl = lane % kTok;
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) un.key[rr] = kNoKey;
#pragma unroll
    for (int j = 0; j < kTcMaxTopk; ++j) {
      const int v = __shfl_sync(0xffffffffu, ids[j], tl);
      if (j % kLpt == lane / kTok && j / kLpt < 8)
        un.key[j / kLpt] = v >= 0 ? (static_cast<uint32_t>(v) << 16) | (1u << tl) : kNoKey;
    }
    sort_keys(un.key, lane);
    uint32_t acc[8];
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) acc[rr] = un.key[rr] & 0xffffu;
    run_or(un.key, acc, lane);
    // heads (the first element of each block's run) and their union indices
    int before = 0;
#pragma unroll
    for (int rr = 0; rr < 8; ++rr) {
      const uint32_t up = __shfl_up_sync(0xffffffffu, un.key[rr], 1);
      const uint32_t prev_last = __shfl_sync(0xffffffffu, un.key[(rr + 7) & 7], 31);
      const uint32_t prev = lane > 0 ? up : (rr > 0 ? prev_last : kNoKey);
      const bool head = un.key[rr] != kNoKey && (prev == kNoKey || (prev >> 16) != (un.key[rr] >> 16));
      const uint32_t hb = __ballot_sync(0xffffffffu, head);
      un.u[rr] = before + __popc(hb & lt);
      before += __popc(hb);
      if (head) {
        un.heads |= 1u << rr;
        un.key[rr] = (un.key[rr] & 0xffff0000u) | (acc[rr] & 0xffffu);
      }
    }
    un.n = before;
  }
  // the descriptor fields every part of the tile shares
  if (lane < kTok) {
    d->own[lane] = own;
    d->lim[lane] = static_cast<int16_t>(lim);
  }
  if (lane == 0) {
    d->end = 0;
    d->req = r;
    d->g = g;
    d->t0 = t0;
    d->n_tok = n;
    d->c0 = c0;
    d->ctx0 = ctx0;
    d->pos_last = seq_len - 1;
    d->bad_mask = static_cast<int32_t>(bad_mask);
  }
}

// Part `part` of a tile's union (entries kMaxUnion * part ..) into descriptor d; copies the shared
// fields from the tile's first descriptor `d0` when the part is a continuation.
template <bool kF16V>
__device__ __forceinline__ void write_tile_part(const AttendArgs& a, const TileUnion& un, int part, TileDesc* d,
                                                const TileDesc* d0, int lane) {
  const int u0 = part * kMaxUnion;
  const int nu = min(kMaxUnion, max(un.n - u0, 0));
  if (un.direct) {  // the block-mask path wrote the tile's only descriptor
    if (lane == 0) {
      d->n_union = d->req < 0 ? 0 : nu;
      d->cont = 0;
      d->more = 0;
      d->by_block = 1;
    }
    return;
  }
  // token masks over this part's entries: cleared, then each head ORs in its tokens' bits
  for (int i = lane; i < kTokMax * (kMaxUnion / 32); i += 32) (&d->masks[0][0])[i] = 0u;
  __syncwarp();
  if (part > 0) {
    // the tile's shared fields, from the descriptor its first part went to
    if (lane < kTokMax) {
      d->own[lane] = d0->own[lane];
      d->lim[lane] = d0->lim[lane];
    }
    if (lane == 0) {
      d->end = 0;
      d->req = d0->req;
      d->g = d0->g;
      d->t0 = d0->t0;
      d->n_tok = d0->n_tok;
      d->c0 = d0->c0;
      d->ctx0 = d0->ctx0;
      d->pos_last = d0->pos_last;
      d->bad_mask = d0->bad_mask;
    }
  }
  const int req = part > 0 ? d0->req : d->req, g = part > 0 ? d0->g : d->g;
#pragma unroll
  for (int rr = 0; rr < 8; ++rr) {
    const int u = un.u[rr] - u0;
    if (((un.heads >> rr) & 1u) && u >= 0 && u < kMaxUnion) {
      const int b = static_cast<int>(un.key[rr] >> 16);
      d->union_blk[u] = static_cast<uint16_t>(b);
      for (uint32_t toks = un.key[rr] & 0xffffu; toks != 0u; toks &= toks - 1u)
        atomicOr(&d->masks[__ffs(toks) - 1][u >> 5], 1u << (u & 31));
      if (kF16V)
        d->vexp[u] = static_cast<int8_t>(
            __ldg(a.vconv_exp + (static_cast<int64_t>(req) * a.max_blocks + b) * a.num_kv_heads + g));
    }
  }
  if (lane == 0) {
    d->n_union = req < 0 ? 0 : nu;
    d->cont = part > 0;
    d->more = u0 + kMaxUnion < un.n;
    d->by_block = 0;
  }
}

// One CTA per SM walks its list of tiles (one flat tile per round of gridDim.x). The K / V
// rings, the S buffers and the MMA order run on across tile boundaries (block counters count
// the CTA's whole block sequence), so the next tile's S runs while the softmax warps finish the
// previous tile, and its description, Q tile and first K / V blocks are ready before they do.
template <int kG, bool kF16V>
__global__ void __launch_bounds__(kThreadsTc, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                      const AttendArgs a) {
  constexpr int kTok = kRows / kG;  // tokens per tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* big = smem_raw;
  TcCtl* ctl = reinterpret_cast<TcCtl*>(smem_raw + kBigBytes);
  // the 128B-swizzled operands need 1024-byte alignment; the dynamic base provides it
  if ((smem_u32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_err(a.err_word, PBS_DEVERR_TIMEOUT);
    return;
  }
  uint8_t* q_s = big;
  // stage st of each ring at + st * kTileBytes; a stage is [64-dim quarter][128 keys][128 B], so
  // 8-key groups are 1 KiB apart and the two quarters of a key 16 KiB apart
  uint8_t* k_s = big + kQBytes;
  uint8_t* v_s = k_s + kStagesTc * kTileBytes;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    TRACE(kEvStart);
    ctl->abort = 0;
    mbar_init(&ctl->q_full, 1);
    mbar_init(&ctl->q_empty, 1);
    for (int i = 0; i < kStagesTc; ++i) {
      mbar_init(&ctl->k_full[i], 1);
      mbar_init(&ctl->k_empty[i], 1);
      mbar_init(&ctl->v_full[i], 1);
      mbar_init(&ctl->v_empty[i], 1);
    }
    for (int i = 0; i < kSBuf; ++i) {
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->p_full[i], kSoftWarps);
      mbar_init(&ctl->pv_done[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->tile_full[i], 1);
      mbar_init(&ctl->tile_empty[i], kTileUsers);
    }
    fence_mbar_init();
  }
  if (warp == 2) tc::alloc(&ctl->tmem_base, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  const uint32_t tm_s0 = tmem, tm_o = tmem + kSBuf * 128;

  if (warp == 2) {
    // ------------------------------------------------------------------ tile scheduler
    // request tiles in the batch (lane-parallel over requests)
    int total = 0;
    for (int r0 = 0; r0 < a.num_reqs; r0 += 32) {
      const int rr = r0 + lane;
      int tiles = 0;
      if (rr < a.num_reqs) {
        const int q_len = __ldg(a.cu_seqlens_q + rr + 1) - __ldg(a.cu_seqlens_q + rr);
        tiles = leading_tiles(q_len, __ldg(a.seq_lens + rr) - q_len, a.tile_pos_limit, kTok);
      }
      total += __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(tiles));
    }
    const int flat = total * a.num_kv_heads;
    int k = 0;   // descriptors written (slot k & 1)
    int nq = 0;  // Q tiles loaded
    bool done = false;
    for (int kt = 0; !done; ++kt) {
      // round kt of the list: its gridDim.x tiles dealt in alternating directions, so a CTA that
      // took a longer tile of one round takes a shorter one of the next (costs fall along the list)
      const int f = kt * static_cast<int>(gridDim.x) +
                    ((kt & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x)
                              : static_cast<int>(blockIdx.x));
      TileUnion un;
      un.n = 0;
      TileDesc* d0 = nullptr;
      for (int part = 0;; ++part, ++k) {
        const int sl = k & 1;
        TileDesc* d = &ctl->tile[sl];
        // the slot's previous descriptor (k - 2) has been released by every role
        bool go = true;
        if (lane == 0 && k >= 2) go = wait_or_abort(&ctl->tile_empty[sl], ((k >> 1) - 1) & 1, ctl, a.err_word);
        go = __shfl_sync(0xffffffffu, go, 0);
        // once any CTA has given up on a wait, the rest of the grid does no work
        if (lane == 0)
          go = go && !aborted(ctl) &&
               !(a.err_word != nullptr && (*reinterpret_cast<volatile int32_t*>(a.err_word) & PBS_DEVERR_TIMEOUT) != 0);
        go = __shfl_sync(0xffffffffu, go, 0);
        const bool last = !go || f >= flat;
        if (lane == 0) TRACET(kEvDesc0, k);
        if (!last) {
          if (part == 0) {
            build_tile<kTok, kF16V>(a, f, total, lane, d, un);
            d0 = d;
          }
          __syncwarp();
          write_tile_part<kF16V>(a, un, part, d, d0, lane);
        }
        if (lane == 0 && last) d->end = 1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->tile_full[sl]);
        if (lane == 0) TRACET(kEvDesc, k);
        if (last) {
          done = true;
          break;
        }
        if (part == 0) {
          // the tile's Q, once the previous tile's S MMAs have read theirs
          if (lane == 0 && (nq == 0 || wait_or_abort(&ctl->q_empty, (nq - 1) & 1, ctl, a.err_word))) {
            mbar_arrive_expect_tx(&ctl->q_full, kQBytes);
            tma_load_3d(q_s, &q_map, &ctl->q_full, 0, d->g * kG, d->t0);
            tma_load_3d(q_s + kHalf, &q_map, &ctl->q_full, 64, d->g * kG, d->t0);
            TRACET(kEvQ, kt);
          }
          ++nq;
          __syncwarp();
        }
        if ((part + 1) * kMaxUnion >= un.n) {
          ++k;
          break;
        }
      }
    }
  } else if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------------ TMA producers
    // Warp 0 streams the K of each tile's union blocks, warp 3 their V: one 32 KiB copy per block
    // (quarter coordinate 0 for K, 2 for V, from the block's first page; on the fp16-V path V is
    // the block's converted image, one bulk copy).
    const bool is_k = warp == 0;
    // K from the cache through the block map (bf16 caches), or from its converted bf16 image
    const bool k_image = a.kconv != nullptr;
    if (is_k && lane == 0) {
      if (!k_image) asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kv_map)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&q_map)) : "memory");
    }
    uint64_t* full = is_k ? ctl->k_full : ctl->v_full;
    uint64_t* empty = is_k ? ctl->k_empty : ctl->v_empty;
    uint8_t* ring = is_k ? k_s : v_s;
    const int quarter = is_k ? 0 : 2;
    int gb = 0;  // blocks this warp has issued, over the CTA's tiles
    bool go = true;
    for (int k = 0; go; ++k) {
      const int sl = k & 1;
      if (lane == 0) go = wait_or_abort(&ctl->tile_full[sl], (k >> 1) & 1, ctl, a.err_word);
      go = __shfl_sync(0xffffffffu, go, 0);
      if (!go) break;
      const TileDesc* d = &ctl->tile[sl];
      if (d->end) break;
      const int nU = d->n_union, g = d->g;
      const int32_t* bt_row = a.page_table + static_cast<int64_t>(d->req) * a.pt_row_stride;
      int phys_lane = 0;
      for (int i = 0; go && i < nU; ++i, ++gb) {
        const int st = gb % kStagesTc;
        if ((i & 31) == 0) phys_lane = i + lane < nU && !(k_image && is_k) && !(kF16V && !is_k)
                                         ? __ldg(bt_row + d->union_blk[i + lane]) : 0;
        const int phys = __shfl_sync(0xffffffffu, phys_lane, i & 31);
        if (lane == 0 && gb >= kStagesTc) go = wait_or_abort(&empty[st], ((gb / kStagesTc) - 1) & 1, ctl, a.err_word);
        if (lane == 0) go = go && !aborted(ctl);
        go = __shfl_sync(0xffffffffu, go, 0);
        if (!go) break;
        const int64_t base = static_cast<int64_t>(phys) * a.block_page_stride;
        // (with converted images the conversion kernel checked the pages)
        if (is_k && !k_image && lane == 0 && (base < 0 || base + (kPagesPerBlock - 1) >= a.num_pages))
          set_err(a.err_word, PBS_DEVERR_PAGE_OOB);
        if (is_k) TRACEB(kEvProdIssue0, gb);
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[st], kTileBytes);
          const int64_t image = (static_cast<int64_t>(d->req) * a.max_blocks + d->union_blk[i]) * a.num_kv_heads + g;
          if (kF16V && !is_k)
            bulk_load(ring + st * kTileBytes, a.vconv + image * kTileBytes, kTileBytes, &full[st]);
          else if (is_k && k_image)
            bulk_load(ring + st * kTileBytes, a.kconv + image * kTileBytes, kTileBytes, &full[st]);
          else  // out-of-range pages read as zeros (TMA bounds)
            tma_load_5d(ring + st * kTileBytes, &kv_map, &full[st], 0, 0, g, static_cast<int>(base), quarter);
        }
        if (is_k) TRACEB(kEvProdIssue1, gb);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->tile_empty[sl]);
    }
    // every copy issued must land before the CTA exits
    if (lane == 0)
      for (int i = max(0, gb - kStagesTc); i < gb; ++i)
        if (!mbar_wait_bounded(&full[i % kStagesTc], (i / kStagesTc) & 1, kTcWaitNs)) set_err(a.err_word, PBS_DEVERR_TIMEOUT);
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = tc::idesc_f16(128, 128, true, false, false);
      constexpr uint32_t kIdescPV = tc::idesc_f16(128, 128, !kF16V, false, true);  // bf16, or fp16 P and V
      const uint32_t q_addr = smem_u32(q_s);
      int gs = 0, gp = 0;      // next block for S, for PV, over the CTA's tiles
      uint32_t first = 0u;     // bit (i & 31): block i is its tile's first (its PV starts O afresh)
      bool ok = true;
      // O += P(j) V(j): in S buffer j % 3 each softmax part's 64 columns hold P hi (bf16, two keys
      // per column) in their first 32 and P lo in their last 32; on the fp16-V path the first 32
      // hold P as fp16 pairs and one MMA per 16 keys does
      auto issue_pv = [&](int j) -> bool {
        const int st = j % kStagesTc, sb = j % kSBuf;
        if (!wait_or_abort(&ctl->p_full[sb], (j / kSBuf) & 1, ctl, a.err_word)) return false;
        if (!wait_or_abort(&ctl->v_full[st], (j / kStagesTc) & 1, ctl, a.err_word)) return false;
        tc::fence_after_sync();
        const uint32_t v_addr = smem_u32(v_s + st * kTileBytes);
        const bool fresh = (first >> (j & 31)) & 1u;
#pragma unroll
        for (int part = 0; part < (kF16V ? 1 : 2); ++part) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            // keys 16ks..16ks+15 belong to softmax part `owner`
            const int owner = (16 * ks) / kW;
            const uint32_t pa = tm_s0 + sb * 128 + owner * kW + part * (kW / 2) + (16 * ks - owner * kW) / 2;
            // keys 16ks..16ks+15 = two 8-key groups (1 KiB apart) from key group 2ks; dims in
            // two 64-wide MN atoms 16 KiB apart
            tc::mma_ts(tm_o, pa, tc::smem_desc_sw128(v_addr + ks * 2048, kHalf, 1024), kIdescPV,
                       !(fresh && part == 0 && ks == 0));
          }
        }
        tc::commit(&ctl->pv_done[sb]);
        TRACEB(kEvPV, j);
        tc::commit(&ctl->v_empty[st]);
        return true;
      };
      int nq = 0;  // Q tiles consumed
      for (int k = 0; ok; ++k) {
        const int sl = k & 1;
        // The previous descriptor's last PVs go first, before waiting for this one: a tile's
        // epilogue, on the softmax warps' path, waits for them (and descriptor k waits for
        // descriptor k - 2's release), while this descriptor's first S runs during that epilogue.
        while (ok && gp < gs) {
          if (!issue_pv(gp)) ok = false;
          ++gp;
        }
        if (!ok || !wait_or_abort(&ctl->tile_full[sl], (k >> 1) & 1, ctl, a.err_word)) break;
        const TileDesc* d = &ctl->tile[sl];
        if (d->end) break;
        const int nU = d->n_union;
        const bool cont = d->cont != 0, more = d->more != 0;
        // a continuation uses the Q its tile's first descriptor loaded
        if (!cont) {
          if (!wait_or_abort(&ctl->q_full, nq & 1, ctl, a.err_word)) break;
          ++nq;
        }
        tc::fence_after_sync();
        // issue order S(0), S(1), S(2), PV(0), S(3), PV(1), ... over the CTA's block sequence: S
        // runs two blocks ahead of PV, so the softmax of block i + 1 finds S(i + 1) done while
        // PV(i - 1) is still queued. S(i) reuses buffer i % 3, whose last reader PV(i - 3) was
        // issued before it.
        for (int i = 0; i < nU; ++i, ++gs) {
          const int st = gs % kStagesTc, sb = gs % kSBuf;
          if (!wait_or_abort(&ctl->k_full[st], (gs / kStagesTc) & 1, ctl, a.err_word)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t k_addr = smem_u32(k_s + st * kTileBytes);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            // dims 16ks..: Q half ks/4 and K quarter ks/4 (each 16 KiB apart, 8-row groups 1 KiB
            // apart)
            tc::mma_ss(tm_s0 + sb * 128,
                       tc::smem_desc_sw128(q_addr + (ks >> 2) * kHalf + (ks & 3) * 32, 16, 1024),
                       tc::smem_desc_sw128(k_addr + (ks >> 2) * kHalf + (ks & 3) * 32, 16, 1024), kIdescS,
                       ks > 0);
          }
          tc::commit(&ctl->s_full[sb]);
          tc::commit(&ctl->k_empty[st]);  // the K stage is free once S(i) has read it
          TRACEB(kEvS, gs);
          first = (i == 0 && !cont) ? (first | (1u << (gs & 31))) : (first & ~(1u << (gs & 31)));
          if (gs - gp >= 2) {
            if (!issue_pv(gp)) {
              ok = false;
              break;
            }
            ++gp;
          }
        }
        // the tile's Q is free once the S MMAs of its last descriptor have completed
        if (!more) tc::commit(&ctl->q_empty);
        mbar_arrive(&ctl->tile_empty[sl]);
      }
      while (ok && gp < gs) {
        if (!issue_pv(gp)) break;
        ++gp;
      }
      // every MMA issued must complete before TMEM is released
      if (gp > 0) mbar_wait_bounded(&ctl->pv_done[(gp - 1) % kSBuf], ((gp - 1) / kSBuf) & 1, kTcWaitNs);
      if (gs > gp) mbar_wait_bounded(&ctl->s_full[(gs - 1) % kSBuf], ((gs - 1) / kSBuf) & 1, kTcWaitNs);
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    // kSplit warps share each 32-lane quadrant of TMEM; warp part p owns S / O columns
    // [p*kW, p*kW + kW) of its 32 rows. Row maxima and sums are combined through shared memory.
    const int sw = warp - 4, quad = sw & 3, part = sw >> 2;
    const int row = quad * 32 + lane;  // = TMEM lane
    const int col0 = part * kW;
    const int tt = row / kG, h = row % kG;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = a.scale_log2;
    int gb = 0;  // blocks of the CTA's sequence this warp has processed
    // a tile's softmax state, kept across its descriptors
    float m_ref = -INFINITY, l = 0.f;  // l: this part's share of the row sum
    bool started = false;              // the row has had an active block (same in every part)
    int E = 0;                         // fp16-V path: O holds sum(P V) * 2^-E (set by the first block)
    bool ok = true;
    for (int k = 0;; ++k) {
      const int sl = k & 1;
      const bool got = warp_wait_or_abort(&ctl->tile_full[sl], (k >> 1) & 1, ctl, a.err_word);
      const TileDesc* d = &ctl->tile[sl];
      // both warps of the quadrant leave together (they meet at named barriers below)
      if (quad_any(quad, !got || d->end != 0 || aborted(ctl))) break;
      const int nU = d->n_union, n_tok = d->n_tok, t0 = d->t0, g = d->g;
      const bool cont = d->cont != 0, more = d->more != 0, by_block = d->by_block != 0;
      if (sw == 0 && lane == 0) TRACET(kEvTileIn, k);
      const bool live = tt < n_tok && !((d->bad_mask >> tt) & 1);
      const int own_t = d->own[tt], lim_t = d->lim[tt];
      const int pos_last = d->pos_last;
      const int last_blk = pos_last / kSparseBlock;
      const int last_rows = pos_last - last_blk * kSparseBlock + 1;  // valid rows of the request's last block
      // a continuation descriptor carries on the tile's softmax state and O
      if (!cont) {
        m_ref = -INFINITY;
        l = 0.f;
        started = false;
        E = 0;
        ok = true;
      }
      // A wait that gives up clears `ok`; the warp then stops waiting but keeps stepping through
      // the blocks, so the two warps of a quadrant always meet at the same named barriers.
      for (int i = 0; i < nU; ++i, ++gb) {
        const int sb = gb % kSBuf, st = gb % kStagesTc;
        const int b = d->union_blk[i];
        const int x = by_block ? b : i;
        const bool active = live && ((d->masks[tt][x >> 5] >> (x & 31)) & 1u);
        const int lim = b == own_t ? lim_t : kSparseBlock;
        if (ok && !warp_wait_or_abort(&ctl->s_full[sb], (gb / kSBuf) & 1, ctl, a.err_word)) ok = false;
        tc::fence_after_sync();
        if (sw == 0 && lane == 0) TRACEB(kEvSoftIn, gb);
        // fp16-V path: this block's P' = P * 2^de; E is CTA-uniform, so every warp moves it (and
        // rescales its O columns) at the same block
        int de = 0;
        if (kF16V) {
          const int eb = d->vexp[i];
          if (i == 0 && !cont) E = eb;
          if (eb - E > kExpUp || eb - E < kExpDown) {
            // O holds this tile's PV(i-1) once that completes (S(i) done implies PV(i-2) done)
            if (ok && !warp_wait_or_abort(&ctl->pv_done[(gb - 1) % kSBuf], ((gb - 1) / kSBuf) & 1, ctl, a.err_word))
              ok = false;
            tc::fence_after_sync();
            scale_o(tm_o + lane_off + col0, exp2i(E - eb));
            tc::wait_st();
            E = eb;
          }
          de = eb - E;
        }
        const float unshift = exp2i(-de);  // psum' * 2^-de = psum
        // rows past the request's last token in its last block may hold anything: zero that V
        // (the converted images already hold zeros there)
        if (!kF16V && b == last_blk && last_rows < kSparseBlock) {
          if (ok && !warp_wait_or_abort(&ctl->v_full[st], (gb / kStagesTc) & 1, ctl, a.err_word)) ok = false;
          const uint32_t v_base = smem_u32(v_s + st * kTileBytes);
          for (int e = sw * 32 + lane; e < (kSparseBlock - last_rows) * 16; e += 32 * kSoftWarps) {
            const int key = last_rows + (e >> 4), vq = (e >> 3) & 1, chunk = e & 7;
            // key k of quarter vq at vq * 16 KiB + k * 128 B
            sts128(v_base + vq * kHalf + key * 128 + chunk * 16, 0, 0, 0, 0);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        const uint32_t ts = tm_s0 + sb * 128 + lane_off;
        // tcgen05.ld / st are warp-collective: every lane of the warp issues them; rows that do not
        // take part in this block are masked arithmetically (their P row becomes zero). Activity
        // depends only on the row, so the kSplit warps of a quadrant always agree and take the same
        // branches around the named barriers below.
        if (__any_sync(0xffffffffu, active)) {
          const int nval = active ? min(max(lim - col0, 0), kW) : 0;  // valid keys among my columns
          // a part whose columns hold no valid key (they may lie past the last token) writes zeros
          const bool any_valid = __any_sync(0xffffffffu, nval > 0);
          uint32_t v[kW];
          bool prefix = false;
          float pm = -INFINITY, psum = 0.f;
          if (any_valid) {
#pragma unroll
            for (int c = 0; c < kW / 32; ++c) tc::ld32(ts + col0 + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&v[32 * c]));
            tc::wait_ld();
            prefix = __any_sync(0xffffffffu, nval != 0 && nval != kW);
            // P with the running reference (the common case), and this part's maximum
            if (kF16V)
              psum = prefix ? write_p16<true>(v, nval, sl2, m_ref - de, ts + col0, pm)
                            : write_p16<false>(v, nval, sl2, m_ref - de, ts + col0, pm);
            else
              psum = prefix ? write_p<true>(v, nval, sl2, m_ref, ts + col0, ts + col0 + kW / 2, pm)
                            : write_p<false>(v, nval, sl2, m_ref, ts + col0, ts + col0 + kW / 2, pm);
          } else if (kF16V) {
            zero_p16(ts + col0);
          } else {
            zero_p(ts + col0, ts + col0 + kW / 2);
          }
          ctl->xchg[part][row] = pm;
          quad_bar(quad);
          float mx = pm;
#pragma unroll
          for (int q = 0; q < kSplit; ++q) mx = fmaxf(mx, ctl->xchg[q][row]);
          quad_bar(quad);  // every part has read before the next block overwrites
          if (sw == 0 && lane == 0) TRACEB(kEvSoftMax, gb);
          mx *= sl2;
          // the reference moves only when the row maximum passes it by 2^8 (or on the row's first
          // block); then O is rescaled and this block's P recomputed
          const bool grow = active && (m_ref == -INFINITY || mx > m_ref + kRescaleLog2);
          if (__any_sync(0xffffffffu, grow)) {
            const float m_new = grow ? fmaxf(mx, m_ref) : m_ref;
            // O's dim columns hold contributions of every key part once the row has started
            const bool resc = grow && started;
            const float alpha = resc ? ex2(m_ref - m_new) : 1.f;
            if (__any_sync(0xffffffffu, resc)) {
              // O holds this tile's PV(i-1) once that completes (S(i) done implies PV(i-2) done)
              if (ok && !warp_wait_or_abort(&ctl->pv_done[(gb - 1) % kSBuf], ((gb - 1) / kSBuf) & 1, ctl, a.err_word))
                ok = false;
              tc::fence_after_sync();
              scale_o(tm_o + lane_off + col0, alpha);
            }
            l *= alpha;
            m_ref = m_new;
            if (any_valid) {
              float unused;
              if (kF16V)
                psum = prefix ? write_p16<true>(v, nval, sl2, m_ref - de, ts + col0, unused)
                              : write_p16<false>(v, nval, sl2, m_ref - de, ts + col0, unused);
              else
                psum = prefix ? write_p<true>(v, nval, sl2, m_ref, ts + col0, ts + col0 + kW / 2, unused)
                              : write_p<false>(v, nval, sl2, m_ref, ts + col0, ts + col0 + kW / 2, unused);
            }
          }
          l += psum * unshift;
          started = started || active;
        } else if (kF16V) {
          zero_p16(ts + col0);
        } else {
          zero_p(ts + col0, ts + col0 + kW / 2);
        }
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full[sb]);
        if (sw == 0 && lane == 0) TRACEB(kEvSoftOut, gb);
      }
      if (sw == 0 && lane == 0) TRACE(kEvEpi);
      // ---- epilogue, at the tile's last descriptor: O / l -> bf16 (row sum combined over the parts
      // of the quadrant). The next tile's first PV, which starts O afresh, waits for this warp's
      // arrival on its P.
      if (!more) {
        if (ok && nU > 0 && !warp_wait_or_abort(&ctl->pv_done[(gb - 1) % kSBuf], ((gb - 1) / kSBuf) & 1, ctl, a.err_word))
          ok = false;
        tc::fence_after_sync();
        ctl->xchg[part][row] = l;
        quad_bar(quad);
        float lsum = 0.f;
#pragma unroll
        for (int q = 0; q < kSplit; ++q) lsum += ctl->xchg[q][row];
        quad_bar(quad);  // every part has read before the next tile's first block overwrites
        {
          // warp-collective TMEM reads for every lane; only rows of real tokens are stored
          uint16_t* out = a.out + static_cast<int64_t>(t0 + tt) * a.out_row_stride +
                          static_cast<int64_t>(g * kG + h) * a.out_head_stride + col0;
          const float inv = (live && lsum > 0.f && ok) ? a.v_scale * (kF16V ? exp2i(E) : 1.f) / lsum : 0.f;
          // p = 2^(t - m_ref), so the row's base-2 log-sum-exp is m_ref + log2(sum p)
          if (a.lse != nullptr && part == 0 && tt < n_tok)
            a.lse[static_cast<int64_t>(t0 + tt) * a.lse_row_stride + g * kG + h] =
                (live && lsum > 0.f && ok) ? (m_ref + log2f(lsum)) * kLn2 : -INFINITY;
#pragma unroll
          for (int c = 0; c < kW / 32; ++c) {
            uint32_t v[32];
            if (nU > 0) {
              tc::ld32(tm_o + lane_off + col0 + 32 * c, v);
              tc::wait_ld();
            }
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float o0 = nU > 0 ? __uint_as_float(v[j]) * inv : 0.f;
              const float o1 = nU > 0 ? __uint_as_float(v[j + 1]) * inv : 0.f;
              w[j >> 1] = pack_bf16(o0, o1);
            }
            if (tt < n_tok) {
              uint4* dst = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4)
                dst[q4] = make_uint4(w[4 * q4], w[4 * q4 + 1], w[4 * q4 + 2], w[4 * q4 + 3]);
            }
          }
        }
      }
      // O has been read: the next tile's PVs may overwrite it (they wait for this warp's P)
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->tile_empty[sl]);
      if (sw == 0 && lane == 0) TRACET(kEvTileOut, k);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc::fence_after_sync();
    tc::dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) TRACE(kEvEnd);
}

}  // namespace

#ifdef PBS_TRACE
}  // namespace pbs
// Trace build only: choose the traced CTA, and copy the timestamps out (host buffer of
// kEvCount int64). Not part of the C ABI.
extern "C" __attribute__((visibility("default"))) int pbs_debug_trace_set(int cta) {
  return cudaMemcpyToSymbol(pbs::g_trace_cta, &cta, sizeof(int)) == cudaSuccess ? 0 : 5;
}
extern "C" __attribute__((visibility("default"))) int pbs_debug_trace_window(int b0) {
  return cudaMemcpyToSymbol(pbs::g_trace_b0, &b0, sizeof(int)) == cudaSuccess ? 0 : 5;
}
extern "C" __attribute__((visibility("default"))) int pbs_debug_trace_get(long long* host, int n) {
  if (n > pbs::kEvCount) n = pbs::kEvCount;
  return cudaMemcpyFromSymbol(host, pbs::g_trace, sizeof(long long) * n) == cudaSuccess ? 0 : 5;
}
namespace pbs {
#endif

cudaError_t launch_convert_images(const AttendArgs& a, cudaStream_t stream) {
  const dim3 cgrid(static_cast<unsigned>(a.max_blocks), static_cast<unsigned>(a.num_reqs),
                   static_cast<unsigned>(a.num_kv_heads));
  if (a.kv_dtype == PBS_KV_FP8_E4M3) convert_kv_kernel<PBS_KV_FP8_E4M3><<<cgrid, 128, 0, stream>>>(a);
  else if (a.kv_dtype == PBS_KV_NVFP4) convert_kv_kernel<PBS_KV_NVFP4><<<cgrid, 128, 0, stream>>>(a);
  else convert_v_kernel<<<cgrid, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

bool prefill_tc_supported(const AttendArgs& a, bool with_workspace) {
  // bf16: K (and V without a workspace) through the block map of a packed cache; fp8 / NVFP4: K
  // and V from images the conversion kernel writes into the workspace
  const bool cache_ok = a.kv_dtype == PBS_KV_BF16 ? a.page_stride_bytes == static_cast<int64_t>(a.num_kv_heads) * 8192
                                                  : with_workspace;
  return cache_ok && (a.group == 8 || a.group == 16) && a.k <= kTcMaxTopk && a.max_blocks <= kTcMaxBlocks &&
         a.num_pages * a.num_kv_heads <= 0x7fffffffLL && a.num_reqs <= 65535 &&
         a.out_head_stride % 8 == 0 && a.out_row_stride % 8 == 0 &&
         reinterpret_cast<uintptr_t>(a.out) % 16 == 0 && a.q_head_stride % 8 == 0 && a.q_row_stride % 8 == 0 &&
         reinterpret_cast<uintptr_t>(a.q) % 16 == 0;
}

template <int kG, bool kF16V>
cudaError_t launch_tc(const AttendArgs& a, const CUtensorMap& kv_map, const CUtensorMap& q_map, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<kG, kF16V>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kTcSmem));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (kF16V) {
    // the images the attend streams: V (bf16 caches; K comes through the block map), or K and V
    e = launch_convert_images(a, stream);
    if (e != cudaSuccess) return e;
  }
  // one CTA per SM; at most one per tile (an upper bound: tiles are counted on the device)
  const int64_t tiles = (static_cast<int64_t>(a.num_rows) / (kRows / kG) + a.num_reqs + 1) * a.num_kv_heads;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(std::max(sms, 1), tiles));
  prefill_tc_kernel<kG, kF16V><<<grid, kThreadsTc, kTcSmem, stream>>>(kv_map, q_map, a);
  return cudaGetLastError();
}

template <int kG>
cudaError_t launch_tc_attend(const AttendArgs& a, const CUtensorMap& kv_map, const CUtensorMap& q_map,
                             cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<kG, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kTcSmem));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (static_cast<int64_t>(a.num_rows) / (kRows / kG) + a.num_reqs + 1) * a.num_kv_heads;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(std::max(sms, 1), tiles));
  prefill_tc_kernel<kG, true><<<grid, kThreadsTc, kTcSmem, stream>>>(kv_map, q_map, a);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tc_attend(const AttendArgs& a, const CUtensorMap& kv_map, const CUtensorMap& q_map,
                                     cudaStream_t stream) {
  if (a.vconv == nullptr || (a.kv_dtype != PBS_KV_BF16 && a.kconv == nullptr)) return cudaErrorInvalidValue;
  return a.group == 16 ? launch_tc_attend<16>(a, kv_map, q_map, stream) : launch_tc_attend<8>(a, kv_map, q_map, stream);
}

cudaError_t launch_prefill_tc(const AttendArgs& a, const CUtensorMap& kv_map, const CUtensorMap& q_map,
                              cudaStream_t stream) {
  // fp8 / NVFP4 caches are read only through the converted images
  if (a.kv_dtype != PBS_KV_BF16 && (a.vconv == nullptr || a.kconv == nullptr)) return cudaErrorInvalidValue;
  if (a.vconv != nullptr)
    return a.group == 16 ? launch_tc<16, true>(a, kv_map, q_map, stream) : launch_tc<8, true>(a, kv_map, q_map, stream);
  return a.group == 16 ? launch_tc<16, false>(a, kv_map, q_map, stream) : launch_tc<8, false>(a, kv_map, q_map, stream);
}

size_t prefill_tc_workspace_bytes(int64_t num_reqs, int64_t num_kv_heads, int64_t max_blocks, int kv_dtype) {
  if (num_reqs <= 0 || num_reqs > 65535 || num_kv_heads <= 0 || max_blocks <= 0 || max_blocks > kTcMaxBlocks) return 0;
  if (kv_dtype != PBS_KV_BF16 && kv_dtype != PBS_KV_FP8_E4M3 && kv_dtype != PBS_KV_NVFP4) return 0;
  const int64_t n = num_reqs * max_blocks * num_kv_heads;
  // V images, their exponents, then (fp8 / NVFP4) the K images
  int64_t bytes = n * kTileBytes + ((n * 4 + 255) / 256) * 256;
  if (kv_dtype != PBS_KV_BF16) bytes += n * kTileBytes;
  return static_cast<size_t>(bytes);
}

}  // namespace pbs
