// Prefill attend by key block ("gathered rows") on the 5th-generation tensor cores (tcgen05 +
// TMEM), bf16 KV cache, GQA 8 or 16.
//
// What it computes (vLLM page vllm.models.minimax_m3.nvidia.sparse_attention_flashinfer, forward:
// the varlen msa_sparse_attention call; row rule of vllm.models.minimax_m3.amd.ops.sparse_pa,
// _write_sparse_block_table_row_from_values): for every prefill token and query head h of kv
// head g, out = v_scale * softmax(softmax_scale * k_scale * q_h K^T) V over the keys of the
// 128-token blocks the token's top-k selects (block b valid iff 0 <= b <= pos/128; the own
// block truncated at pos). Duplicate ids in a token's list count once.
//
// GB300 design
// ------------
// A tile of consecutive tokens shares few of its selected blocks when the selections are
// spread over a long context, so a tile that streams the union of its tokens' blocks wastes
// most of its MMA rows. Here the work is inverted: a work item is one (key block b, kv head g)
// of a window of 256 consecutive tokens of one request, and its MMA rows are the window's
// tokens that selected b, gathered 16 at a time (x 8 query heads = the 128-row M tile; 8 tokens
// x 16 heads at GQA 16). Every row of every tile does useful work except in a bucket's last
// chunk.
//
// * Index kernel (one CTA per window): each token's distinct valid blocks, sorted, give the
//   token's partial slots; tokens are bucketed by block (shared-memory histogram, block scan,
//   scatter). Tokens with no valid block get zero output here.
// * Attend kernel (persistent, one CTA per SM): windows are taken in order and the items of a
//   window from a per-window counter, so the partial results of a window are written and
//   merged while they sit in L2. Per item, warp 0 loads K_b and V_b of head g (one 4 KiB tensor
//   copy per page and half row, 128B swizzle) into one of two K/V buffers, then per chunk writes
//   a descriptor (tokens, partial slots, own-block key limits) into a 4-deep ring and gathers
//   the chunk's Q rows (one {64 dims, G heads, 1 token} tensor copy per token and half). Warp 1
//   (one thread) issues S(c) = Q K^T into TMEM buffer c % 2, then PV(c-1), so the softmax of
//   chunk c overlaps PV(c-1) and S(c+1). Warps 4-7 and 8-11 are two softmax warpgroups taking
//   chunks alternately; a thread owns one row (TMEM lane). Warps 2 and 3 count and merge the
//   chunks' partials (chunks alternately), off the softmax warps' path.
// * Softmax of one chunk (one key block): the row maximum over the block's valid keys (first
//   pass over the S row in TMEM), then P = 2^(s * scale * log2 e - m) written back over S as bf16
//   hi + lo (32 keys at a time into the same 32 columns), so the PV product (two MMAs, A = P from
//   TMEM) keeps the output within 2e-3 relative RMS of the fp64 attend.
// * Epilogue: the row's partial output O / l, scaled by a power of two so that its largest
//   element lies in [2^14, 2^15), is stored as fp16 together with (log2-sum-exp, exponent).
//   The stores are fenced one softmax phase later (by then they have landed), and the chunk goes
//   to its merge warp: one atomic ticket per (token, kv head) counts the finished partials, and
//   the chunk that completes a token merges its partials (fp32, log-sum-exp weights), writes the
//   bf16 output and the log-sum-exp, and drops the merged partial lines from L2 without writing
//   them back.
// * TMEM (512 columns): S / P double buffer (2 x 128) and O double buffer (2 x 128).
#include <algorithm>

#include <cuda_fp16.h>

#include "pbs_device.cuh"
#include "pbs_internal.h"
#include "tc_device.cuh"

namespace pbs {
namespace {

constexpr int kGRows = 128;                     // MMA M: tokens x query heads of a chunk
constexpr int kGThreads = 384;                  // 12 warps
constexpr int kDescRing = 8;                    // chunk descriptors in flight
constexpr int kGQBytes = kGRows * kHeadDim * 2;  // 32 KiB Q tile
constexpr int kGHalf = kGQBytes / 2;            // one 64-dim half of the Q tile
constexpr int kGTile = 32768;                   // a block's K (or V) for one kv head
constexpr int kRingBytes = 10240;               // merge ring of one merge warp: 5 x 2 KiB or 2 x 4 KiB
constexpr int kMaxSlots = 5;
constexpr int kTaskQ = 32;                      // completed tokens waiting for their merge, per merge warp
constexpr int kGSmemBig = 2 * kGQBytes + 4 * kGTile + 2 * kRingBytes;  // Q x 2, K x 2, V x 2, 2 rings
constexpr unsigned long long kGWaitNs = 100000000ull;  // waits here last microseconds: 100 ms cap
constexpr int kIdxThreads = 256;
constexpr int kGatherMaxSms = 1024;

struct ChunkDesc {
  int32_t end;    // 1: no more work for this CTA
  int32_t b;      // key block
  int32_t g;      // kv head
  int32_t ybuf;   // K/V buffer of the item
  int32_t n_tok;  // tokens in this chunk
  int32_t item;   // the CTA's item number (phase of the K/V buffer barriers)
  int32_t pad[2];
  int32_t tr[16];    // segment-relative token index
  int32_t slot[16];  // the token's partial slot for block b
  int32_t lim[16];   // keys of block b the token sees (128, or pos - 128 b + 1 for its own block)
  int32_t nsel[16];  // the token's number of partials
};

struct GCtl {
  uint64_t desc_full[kDescRing];
  uint64_t desc_empty[kDescRing];  // 1 (MMA thread) + 1 (merge warp) arrivals
  uint64_t part_done[kDescRing];   // the chunk's partials are stored and fenced: 4 softmax warps
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[2], v_full[2], v_land[2], kv_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t o_free[2];    // O buffer X has been read (softmax warps -> MMA)
  // item n's V is in fp16 (merge warp n % 2 -> MMA and softmax warps), one barrier per n % 4:
  // item n + 4 needs the K/V buffer of item n + 2, freed only after every PV of item n + 2,
  // which comes after the epilogues of item n
  uint64_t vx_ready[4];
  uint64_t ring_full[2][kMaxSlots];
  uint64_t mma_fin;
  uint32_t tmem_base;
  int32_t abort;
  ChunkDesc desc[kDescRing];
  int32_t ents[128];  // bucket entries of the producer's current batch
  alignas(16) int4 tq[2][kTaskQ];                     // merge tasks: (token, kv head, partials, 0)
  float lsum[4][2][kGRows];                             // chunk c & 3, key half, row: partial sum
  float xchg[2][2][kGRows];                            // row maxima of the two key halves
  int32_t vexp[4];                                     // item n's V buffer holds V * 2^-vexp[n % 4]
  int32_t items_total;                                 // items of this CTA (written before the end)
  alignas(16) float2 ring_ml[2][kMaxSlots][16];       // (lse, exponent) of each ring slot's heads
};

// A batch of up to 8 consecutive chunks of one window (producer).
struct Batch {
  int w, base, nb, r, c0, ctx0, seq_len;
};

constexpr size_t kGSmem = kGSmemBig + sizeof(GCtl) + 1024;
static_assert(kGSmem <= 232448, "shared memory layout exceeds 227 KiB");

#ifdef PBS_TRACE
// Trace build only: one CTA records SM-clock timestamps of the first kGtChunks chunks' pipeline
// events (producer, MMA, softmax, epilogue, merge) and the number of merges per chunk.
constexpr int kGtChunks = 64;
enum GTraceEv { kGtStart, kGtEnd, kGtProd = 2, kGtS = kGtProd + kGtChunks, kGtPV = kGtS + kGtChunks,
                kGtSm0 = kGtPV + kGtChunks, kGtSm1 = kGtSm0 + kGtChunks, kGtE0 = kGtSm1 + kGtChunks,
                kGtE1 = kGtE0 + kGtChunks, kGtM0 = kGtE1 + kGtChunks, kGtM1 = kGtM0 + kGtChunks,
                kGtM2 = kGtM1 + kGtChunks, kGtNM = kGtM2 + kGtChunks, kGtCount = kGtNM + kGtChunks };
__device__ long long g_gtrace[kGtCount];
__device__ int g_gtrace_cta;
#define GTRACE(ev, c) do { if (blockIdx.x == static_cast<unsigned>(g_gtrace_cta) && (c) < kGtChunks) \
                             g_gtrace[(ev) + (c)] = clock64(); } while (0)
#define GTRACE_VAL(ev, c, v) do { if (blockIdx.x == static_cast<unsigned>(g_gtrace_cta) && (c) < kGtChunks) \
                                    g_gtrace[(ev) + (c)] = (v); } while (0)
#else
#define GTRACE(ev, c) do { } while (0)
#define GTRACE_VAL(ev, c, v) do { } while (0)
#endif

__device__ __forceinline__ bool g_aborted(GCtl* ctl) { return *reinterpret_cast<volatile int32_t*>(&ctl->abort) != 0; }

__device__ __forceinline__ bool g_wait(uint64_t* bar, uint32_t parity, GCtl* ctl, int32_t* err) {
  if (mbar_wait_bounded(bar, parity, kGWaitNs)) return true;
  set_err(err, PBS_DEVERR_TIMEOUT);
  atomicExch(&ctl->abort, 1);
  return false;
}

__device__ __forceinline__ bool g_warp_wait(uint64_t* bar, uint32_t parity, GCtl* ctl, int32_t* err) {
  const bool ok = g_wait(bar, parity, ctl, err);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void g_tma_3d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void g_tma_5d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1, int c2, int c3,
                                         int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

__device__ __forceinline__ void g_sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Drop a 128-byte line from L2 without writing it back (its contents become undefined).
__device__ __forceinline__ void discard_l2(const void* p) {
  asm volatile("discard.global.L2 [%0], 128;" ::"l"(p) : "memory");
}

__device__ __forceinline__ float f16_lo(uint32_t x) { return __half2float(__ushort_as_half(static_cast<unsigned short>(x & 0xffffu))); }
__device__ __forceinline__ float f16_hi(uint32_t x) { return __half2float(__ushort_as_half(static_cast<unsigned short>(x >> 16))); }

// Window of the segment [T0, T1) with index `wi`: windows are numbered request by request, each
// request's tokens cut at multiples of kGatherWinTok from its first token. Warp-collective.
// Returns false when wi is past the last window.
struct WinInfo {
  int r, ta, tb, c0, ctx0, seq_len;
};
__device__ __forceinline__ bool find_window(const AttendArgs& a, const GatherWs& w, int wi, WinInfo& out) {
  const int lane = threadIdx.x & 31;
  int base = 0;
  bool found = false;
  for (int r0 = 0; r0 < a.num_reqs && !found; r0 += 32) {
    const int rr = r0 + lane;
    int c0 = 0, c1 = 0, sl = 0;
    if (rr < a.num_reqs) {
      c0 = __ldg(a.cu_seqlens_q + rr);
      c1 = __ldg(a.cu_seqlens_q + rr + 1);
      sl = __ldg(a.seq_lens + rr);
    }
    const int lo = max(c0, w.T0), hi = min(c1, w.T1);
    const int nw = lo < hi ? (hi - 1 - c0) / kGatherWinTok - (lo - c0) / kGatherWinTok + 1 : 0;
    int incl = nw;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    const int excl = incl - nw + base;
    const uint32_t hit = __ballot_sync(0xffffffffu, wi >= excl && wi < excl + nw);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const int ex = __shfl_sync(0xffffffffu, excl, src);
      const int sc0 = __shfl_sync(0xffffffffu, c0, src);
      const int sc1 = __shfl_sync(0xffffffffu, c1, src);
      const int ssl = __shfl_sync(0xffffffffu, sl, src);
      const int slo = max(sc0, w.T0), shi = min(sc1, w.T1);
      const int wrel = (slo - sc0) / kGatherWinTok + (wi - ex);
      out.r = r0 + src;
      out.c0 = sc0;
      out.ctx0 = ssl - (sc1 - sc0);
      out.seq_len = ssl;
      out.ta = max(sc0 + wrel * kGatherWinTok, slo);
      out.tb = min(sc0 + (wrel + 1) * kGatherWinTok, shi);
      found = true;
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  return found;
}

// ------------------------------------------------------------------------------------------
// index kernel: one CTA per window
// ------------------------------------------------------------------------------------------
// Dynamic shared memory: cnt[max_blocks], cur[max_blocks], pairs_s[kGatherWinTok * k].
// Output per window: the chunk records in processing order (buckets by decreasing block id;
// within a bucket kv head by kv head, 16 (or 8) tokens per chunk), the bucket entries they point
// at, and the window record {request, first token, context, seq_len, chunks}.
__global__ void __launch_bounds__(kIdxThreads) gather_index_kernel(const AttendArgs a, const GatherWs w) {
  extern __shared__ int32_t ish[];
  int32_t* cnt = ish;
  int32_t* cur = ish + a.max_blocks;
  int32_t* pairs_s = cur + a.max_blocks;
  __shared__ int s_win[6];
  __shared__ int s_found, s_np, s_nblk;
  __shared__ int s_wsum[kIdxThreads / 32], s_wch[kIdxThreads / 32];
  __shared__ int s_tn[kGatherWinTok];  // partial count of each window token
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wi = blockIdx.x;
  const int kTok = w.tok_per_chunk;
  int32_t* wrec = w.wins + static_cast<int64_t>(wi) * 8;
  if (warp == 0) {
    WinInfo info;
    const bool f = find_window(a, w, wi, info);
    if (lane == 0) {
      s_found = f ? 1 : 0;
      s_np = 0;
      if (f) {
        s_win[0] = info.r;
        s_win[1] = info.ta;
        s_win[2] = info.tb;
        s_win[3] = info.c0;
        s_win[4] = info.ctx0;
        s_win[5] = info.seq_len;
        // blocks any token of the window may select: up to the last token's own block
        const int pos_last = info.ctx0 + (info.tb - 1 - info.c0);
        s_nblk = pos_last >= 0 ? min(pos_last / kSparseBlock + 1, a.max_blocks) : 0;
      } else {
        s_nblk = 0;
      }
    }
  }
  __syncthreads();
  if (!s_found) {
    if (threadIdx.x == 0) {
      wrec[0] = -1;
      wrec[4] = 0;
    }
    return;
  }
  const int r = s_win[0], ta = s_win[1], tb = s_win[2], c0 = s_win[3], ctx0 = s_win[4];
  const int nblk = s_nblk;
  for (int i = threadIdx.x; i < nblk; i += kIdxThreads) cnt[i] = 0;
  __syncthreads();

  // ---- each token's distinct valid blocks, sorted; count per block -------------------------
  const int n = tb - ta;
  for (int tt = warp; tt < n; tt += kIdxThreads / 32) {
    const int t = ta + tt;
    const int tr = t - w.T0;
    const int pos = ctx0 + (t - c0);
    const int causal_len = pos + 1 > 0 ? pos + 1 : 0;
    const int own = causal_len > 0 ? pos / kSparseBlock : -1;
    const int32_t* row = a.topk + static_cast<int64_t>(t) * a.topk_row_stride;
    const int b0 = lane < a.k ? __ldg(row + lane) : -1;
    const int b1 = lane + 32 < a.k ? __ldg(row + lane + 32) : -1;
    bool v0 = lane < a.k && causal_len > 0 && b0 >= 0 && b0 <= own;
    bool v1 = lane + 32 < a.k && causal_len > 0 && b1 >= 0 && b1 <= own;
    const bool oob = (v0 && b0 >= a.max_blocks) || (v1 && b1 >= a.max_blocks);
    const bool bad = __any_sync(0xffffffffu, oob);
    int n_t = 0;
    if (bad) {
      if (lane == 0) set_err(a.err_word, PBS_DEVERR_BLOCK_OOB);
    } else {
      // keep the first occurrence of every value (entries j = lane and j = lane + 32)
      const uint32_t vm0 = __ballot_sync(0xffffffffu, v0), vm1 = __ballot_sync(0xffffffffu, v1);
      bool k0 = v0, k1 = v1;
      const int kk = a.k;
      for (int j = 0; j < kk; ++j) {
        const int bj = j < 32 ? __shfl_sync(0xffffffffu, b0, j) : __shfl_sync(0xffffffffu, b1, j - 32);
        const bool vj = ((j < 32 ? vm0 >> j : vm1 >> (j - 32)) & 1u) != 0;
        if (vj) {
          if (j < lane && bj == b0) k0 = false;
          if (j < lane + 32 && bj == b1) k1 = false;
        }
      }
      const uint32_t km0 = __ballot_sync(0xffffffffu, k0), km1 = __ballot_sync(0xffffffffu, k1);
      n_t = __popc(km0) + __popc(km1);
      // slot = rank of the value among the kept ones (sorted order)
      int r0 = 0, r1 = 0;
      for (int j = 0; j < kk; ++j) {
        const int bj = j < 32 ? __shfl_sync(0xffffffffu, b0, j) : __shfl_sync(0xffffffffu, b1, j - 32);
        const bool kj = ((j < 32 ? km0 >> j : km1 >> (j - 32)) & 1u) != 0;
        if (kj) {
          r0 += bj < b0 ? 1 : 0;
          r1 += bj < b1 ? 1 : 0;
        }
      }
      if (k0) {
        atomicAdd(&cnt[b0], 1);
        const int at = atomicAdd(&s_np, 1);
        pairs_s[at] = (b0 << 14) | (tt << 6) | r0;
      }
      if (k1) {
        atomicAdd(&cnt[b1], 1);
        const int at = atomicAdd(&s_np, 1);
        pairs_s[at] = (b1 << 14) | (tt << 6) | r1;
      }
    }
    if (lane == 0) s_tn[tt] = n_t;
    for (int g = lane; g < a.num_kv_heads; g += 32) {
      const int64_t x = static_cast<int64_t>(tr) * a.num_kv_heads + g;
      w.tickets[x] = 0;
      // the merge task of (token, head): ready at once when there is nothing to merge
      w.inbox[(x % w.n_mw) * w.inbox_cap + x / w.n_mw] = make_int4(tr, g, n_t, n_t == 0 ? 1 : 0);
    }
    if (n_t == 0) {
      // nothing to attend (no valid block, or a block past the page table): zero output
      uint16_t* orow = a.out + static_cast<int64_t>(t) * a.out_row_stride;
      for (int h = 0; h < a.num_heads; ++h) {
        if (lane < 16)
          *reinterpret_cast<uint4*>(orow + static_cast<int64_t>(h) * a.out_head_stride + lane * 8) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      if (a.lse != nullptr)
        for (int h = lane; h < a.num_heads; h += 32)
          a.lse[static_cast<int64_t>(t) * a.lse_row_stride + h] = -INFINITY;
    }
  }
  __syncthreads();

  // ---- scans of the entry counts and the chunk counts over the blocks -------------------------
  const int per = (nblk + kIdxThreads - 1) / kIdxThreads;
  const int lo = min(static_cast<int>(threadIdx.x) * per, nblk), hi = min(lo + per, nblk);
  int s = 0, ch = 0;
  for (int i = lo; i < hi; ++i) {
    s += cnt[i];
    ch += (cnt[i] + kTok - 1) / kTok;
  }
  int is = s, ich = ch;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int vs = __shfl_up_sync(0xffffffffu, is, off), vc = __shfl_up_sync(0xffffffffu, ich, off);
    if (lane >= off) {
      is += vs;
      ich += vc;
    }
  }
  if (lane == 31) {
    s_wsum[warp] = is;
    s_wch[warp] = ich;
  }
  __syncthreads();
  int ws = 0, wc = 0, tch = 0;
  for (int i = 0; i < kIdxThreads / 32; ++i) {
    if (i < warp) {
      ws += s_wsum[i];
      wc += s_wch[i];
    }
    tch += s_wch[i];
  }
  int off_s = ws + is - s, off_ch = wc + ich - ch;  // exclusive prefixes at this thread's first block
  const int64_t pair_base = static_cast<int64_t>(wi) * kGatherWinTok * a.k;
  int4* crow = w.chunks + static_cast<int64_t>(wi) * w.ccap;
  const int hkv = a.num_kv_heads;
  for (int i = lo; i < hi; ++i) {
    const int c = cnt[i];
    cur[i] = off_s;
    if (c > 0) {
      const int nch = (c + kTok - 1) / kTok;
      // buckets with larger block ids come first; inside a bucket kv head by kv head
      const int first = (tch - off_ch - nch) * hkv;
      const int phys = __ldg(a.page_table + static_cast<int64_t>(r) * a.pt_row_stride + i);
      for (int g = 0; g < hkv; ++g)
        for (int sl = 0; sl < nch; ++sl)
          crow[first + g * nch + sl] =
              make_int4(i | (g << 13), static_cast<int>(pair_base + off_s + sl * kTok), min(kTok, c - sl * kTok), phys);
      off_ch += nch;
    }
    off_s += c;
  }
  __syncthreads();

  // ---- scatter the entries into their buckets: token << 12 | (partials - 1) << 6 | slot -------
  const int np = s_np;
  for (int p = threadIdx.x; p < np; p += kIdxThreads) {
    const int v = pairs_s[p];
    const int b = v >> 14, tt = (v >> 6) & 255, rank = v & 63;
    const int at = atomicAdd(&cur[b], 1);
    w.pairs[pair_base + at] = ((ta + tt - w.T0) << 12) | ((s_tn[tt] - 1) << 6) | rank;
  }
  if (threadIdx.x == 0) {
    wrec[0] = r;
    wrec[1] = c0;
    wrec[2] = ctx0;
    wrec[3] = s_win[5];
    wrec[4] = tch * hkv;  // chunk records
  }
}

// ------------------------------------------------------------------------------------------
// attend kernel: persistent, one CTA per SM
// ------------------------------------------------------------------------------------------

template <int kG>
__global__ void __launch_bounds__(kGThreads, 1)
    gather_attend_kernel(const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map,
                         const AttendArgs a, const GatherWs w) {
  constexpr int kTok = kGRows / kG;  // tokens per chunk
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // the 128B-swizzled operands need 1024-byte alignment
  uint8_t* big = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = big;                   // 2 x 32 KiB: [half][rows][128 B]
  uint8_t* k_s = big + 2 * kGQBytes;    // 2 x 32 KiB: [page][row half][quarter][8 rows][128 B]
  uint8_t* v_s = k_s + 2 * kGTile;      // 2 x 32 KiB
  uint8_t* ring_s = v_s + 2 * kGTile;    // 2 x kRingBytes: partial rows being merged
  GCtl* ctl = reinterpret_cast<GCtl*>(ring_s + 2 * kRingBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDescRing; ++i) {
      mbar_init(&ctl->desc_full[i], 1);
      mbar_init(&ctl->desc_empty[i], 2);
      mbar_init(&ctl->part_done[i], 8);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->q_full[i], 1);
      mbar_init(&ctl->q_empty[i], 1);
      mbar_init(&ctl->k_full[i], 1);
      mbar_init(&ctl->v_full[i], 1);
      mbar_init(&ctl->v_land[i], 1);
      mbar_init(&ctl->kv_empty[i], 1);
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->p_full[i], 8);
      mbar_init(&ctl->pv_done[i], 1);
      mbar_init(&ctl->o_free[i], 8);
      mbar_init(&ctl->vx_ready[2 * i], 1);
      mbar_init(&ctl->vx_ready[2 * i + 1], 1);
      for (int j = 0; j < kMaxSlots; ++j) mbar_init(&ctl->ring_full[i][j], 1);
    }

    mbar_init(&ctl->mma_fin, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 2) tc::alloc(&ctl->tmem_base, 512);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  if (threadIdx.x == 0) GTRACE(kGtStart, 0);

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    // Windows in order; CTA i takes chunks [i C / G, (i + 1) C / G) of a window with C chunks,
    // so every window is spread over the whole grid and its partials are merged while in L2.
    // Chunks go in batches of up to 8: the records of batch n + 2 and the bucket entries of
    // batch n + 1 are in flight while batch n is issued.
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kv_map)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&q_map)) : "memory");
    }
    const int cta = blockIdx.x, grid = gridDim.x;
    // window records of windows [wc0, wc0 + 32), one per lane
    int wc0 = -64, wr_r = 0, wr_c0 = 0, wr_ctx0 = 0, wr_sl = 0, wr_C = 0;
    int cw = 0, cbase = 0, chi = -1;  // cursor: window, next chunk of its slice, slice end (-1: not entered)
    auto next_batch = [&](Batch& B) {
      B.nb = 0;
      while (cw < w.num_win) {
        if (cw >= wc0 + 32 || cw < wc0) {
          wc0 = cw & ~31;
          const int wl = wc0 + lane;
          if (wl < w.num_win) {
            const int32_t* wrp = w.wins + static_cast<int64_t>(wl) * 8;
            wr_r = __ldg(wrp + 0);
            wr_c0 = __ldg(wrp + 1);
            wr_ctx0 = __ldg(wrp + 2);
            wr_sl = __ldg(wrp + 3);
            wr_C = __ldg(wrp + 4);
          } else {
            wr_C = 0;
          }
        }
        const int src = cw - wc0;
        const int C = __shfl_sync(0xffffffffu, wr_C, src);
        if (chi < 0) {
          cbase = static_cast<int>(static_cast<int64_t>(cta) * C / grid);
          chi = static_cast<int>(static_cast<int64_t>(cta + 1) * C / grid);
        }
        if (cbase < chi) {
          B.w = cw;
          B.base = cbase;
          B.nb = min(8, chi - cbase);
          B.r = __shfl_sync(0xffffffffu, wr_r, src);
          B.c0 = __shfl_sync(0xffffffffu, wr_c0, src);
          B.ctx0 = __shfl_sync(0xffffffffu, wr_ctx0, src);
          B.seq_len = __shfl_sync(0xffffffffu, wr_sl, src);
          cbase += B.nb;
          return;
        }
        ++cw;
        chi = -1;
      }
    };
    auto load_recs = [&](const Batch& B) {
      int4 v = make_int4(0, 0, 0, 0);
      if (lane < B.nb) v = __ldg(w.chunks + static_cast<int64_t>(B.w) * w.ccap + B.base + lane);
      return v;
    };
    // bucket entries of a batch: entry e = chunk e / kTok, token e % kTok; four per lane
    auto load_ents = [&](const Batch& B, const int4& rec, int (&e)[4]) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int idx = lane + 32 * q;
        const int j = idx / kTok, l = idx % kTok;
        const int poff = __shfl_sync(0xffffffffu, rec.y, j & 7);
        const int ntk = __shfl_sync(0xffffffffu, rec.z, j & 7);
        e[q] = (j < B.nb && l < ntk) ? __ldg(w.pairs + poff + l) : 0;
      }
    };
    int* ent_s = ctl->ents;
    int n_item = -1, c = 0;
    int item_r = -1, item_b = -1, item_g = -1;
    // uses of each buffer so far (their barrier phases); scalars, so they stay in registers
    int q_n0 = 0, q_n1 = 0, kv_n0 = 0, kv_n1 = 0, land_n0 = 0, land_n1 = 0;
    bool ok = true;
    Batch B0, B1, B2;
    next_batch(B0);
    int4 rec0 = load_recs(B0);
    next_batch(B1);
    int4 rec1 = load_recs(B1);
    int e_cur[4];
    load_ents(B0, rec0, e_cur);
    while (ok && B0.nb > 0) {
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q) ent_s[lane + 32 * q] = e_cur[q];
      __syncwarp();
      next_batch(B2);
      const int4 rec2 = load_recs(B2);
      load_ents(B1, rec1, e_cur);
      for (int jc = 0; jc < B0.nb && ok; ++jc, ++c) {
        const int rx = __shfl_sync(0xffffffffu, rec0.x, jc);
        const int b = rx & 8191, g = rx >> 13;
        const int n_tok = __shfl_sync(0xffffffffu, rec0.z, jc);
        const int phys = __shfl_sync(0xffffffffu, rec0.w, jc);
        // ---- a new (request, block, kv head): K and V into the next buffer
        if (B0.r != item_r || b != item_b || g != item_g) {
          ++n_item;
          item_r = B0.r;
          item_b = b;
          item_g = g;
          const int Y = n_item & 1;
          if (n_item >= 2) {
            bool go = true;
            if (lane == 0) go = g_wait(&ctl->kv_empty[Y], ((n_item >> 1) - 1) & 1, ctl, a.err_word);
            if (!__shfl_sync(0xffffffffu, go, 0)) {
              ok = false;
              break;
            }
          }
          const int64_t pbase = static_cast<int64_t>(phys) * a.block_page_stride;
          if (lane == 0 && (pbase < 0 || pbase + (kPagesPerBlock - 1) >= a.num_pages))
            set_err(a.err_word, PBS_DEVERR_PAGE_OOB);
          const int last_rows = B0.seq_len - 1 - b * kSparseBlock + 1;  // rows of block b holding written tokens
          const bool tail = last_rows < kSparseBlock;
          uint64_t* vbar = tail ? &ctl->v_land[Y] : &ctl->v_full[Y];
          if (lane == 0) {
            mbar_arrive_expect_tx(&ctl->k_full[Y], kGTile);
            mbar_arrive_expect_tx(vbar, kGTile);
          }
          __syncwarp();
          // out-of-range pages read as zeros (tensor-map bounds)
          if (lane < 2 * kPagesPerBlock) {
            const int pg = lane & 7;
            const bool isv = lane >= kPagesPerBlock;
            g_tma_5d((isv ? v_s : k_s) + Y * kGTile + pg * 4096, &kv_map, isv ? vbar : &ctl->k_full[Y], 0, 0,
                     isv ? 2 : 0, 0, static_cast<int>((pbase + pg) * a.num_kv_heads + g));
          }
          if (Y == 0) ++kv_n0; else ++kv_n1;
          if (tail) {
            // rows past the request's last token may hold anything (unwritten cache rows): zero
            // them in V before any PV reads the buffer
            const int ln = Y == 0 ? ++land_n0 : ++land_n1;
            bool go = true;
            if (lane == 0) go = g_wait(&ctl->v_land[Y], (ln - 1) & 1, ctl, a.err_word);
            if (!__shfl_sync(0xffffffffu, go, 0)) {
              ok = false;
              break;
            }
            const uint32_t vb = smem_u32(v_s + Y * kGTile);
            const int first = max(last_rows, 0);
            for (int e = lane; e < (kSparseBlock - first) * 16; e += 32) {
              const int key = first + (e >> 4), vq = (e >> 3) & 1, chn = e & 7;
              g_sts128(vb + (key >> 3) * 2048 + vq * 1024 + (key & 7) * 128 + chn * 16, 0, 0, 0, 0);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->v_full[Y]);
          }
        }
        // ---- the chunk's descriptor
        const int ds = c % kDescRing;
        if (c >= kDescRing) {
          bool go = true;
          if (lane == 0) go = g_wait(&ctl->desc_empty[ds], ((c / kDescRing) - 1) & 1, ctl, a.err_word);
          if (!__shfl_sync(0xffffffffu, go, 0)) {
            ok = false;
            break;
          }
        }
        ChunkDesc* d = &ctl->desc[ds];
        int t_lane = 0;
        if (lane < n_tok) {
          const int en = ent_s[jc * kTok + lane];
          const int tr = en >> 12;
          const int t = w.T0 + tr;
          const int pos = B0.ctx0 + (t - B0.c0);
          d->tr[lane] = tr;
          d->slot[lane] = en & 63;
          d->nsel[lane] = ((en >> 6) & 63) + 1;
          d->lim[lane] = pos / kSparseBlock == b ? pos - b * kSparseBlock + 1 : kSparseBlock;
          t_lane = t;
        }
        if (lane == 0) {
          d->end = 0;
          d->b = b;
          d->g = g;
          d->ybuf = n_item & 1;
          d->n_tok = n_tok;
          d->item = n_item;
        }
        // ---- gather the chunk's Q rows: token j, half hf -> rows j*G.., dims 64 hf..
        const int qb = c & 1;
        if (c >= 2) {
          bool go = true;
          if (lane == 0) go = g_wait(&ctl->q_empty[qb], ((c >> 1) - 1) & 1, ctl, a.err_word);
          if (!__shfl_sync(0xffffffffu, go, 0)) {
            ok = false;
            break;
          }
        }
        if (lane == 0) mbar_arrive_expect_tx(&ctl->q_full[qb], n_tok * 2 * kG * 128);
        __syncwarp();
        {
          const int j = lane % kTok, hf = lane / kTok;
          const int tj = __shfl_sync(0xffffffffu, t_lane, j);
          if (lane < 2 * kTok && j < n_tok)
            g_tma_3d(q_s + qb * kGQBytes + hf * kGHalf + j * kG * 128, &q_map, &ctl->q_full[qb], hf * 64, g * kG, tj);
        }
        if (qb == 0) ++q_n0; else ++q_n1;
        __threadfence_block();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&ctl->desc_full[ds]);
          GTRACE(kGtProd, c);
        }
      }
      B0 = B1;
      rec0 = rec1;
      B1 = B2;
      rec1 = rec2;
    }
    // ---- end marks: chunks c and c + 1 (each merge warp takes every other chunk)
    if (lane == 0) ctl->items_total = n_item + 1;
    for (int e = 0; e < 2 && ok; ++e, ++c) {
      const int ds = c % kDescRing;
      if (c >= kDescRing) {
        bool go = true;
        if (lane == 0) go = g_wait(&ctl->desc_empty[ds], ((c / kDescRing) - 1) & 1, ctl, a.err_word);
        if (!__shfl_sync(0xffffffffu, go, 0)) break;
      }
      if (lane == 0) {
        ctl->desc[ds].end = 1;
        __threadfence_block();
        mbar_arrive(&ctl->desc_full[ds]);
      }
      __syncwarp();
    }
    // every copy issued must land before the CTA exits
    if (lane == 0) {
      if (q_n0 > 0) mbar_wait_bounded(&ctl->q_full[0], (q_n0 - 1) & 1, kGWaitNs);
      if (q_n1 > 0) mbar_wait_bounded(&ctl->q_full[1], (q_n1 - 1) & 1, kGWaitNs);
      if (kv_n0 > 0) mbar_wait_bounded(&ctl->k_full[0], (kv_n0 - 1) & 1, kGWaitNs);
      if (kv_n1 > 0) mbar_wait_bounded(&ctl->k_full[1], (kv_n1 - 1) & 1, kGWaitNs);
      if (kv_n0 > 0) mbar_wait_bounded(&ctl->v_full[0], (kv_n0 - 1) & 1, kGWaitNs);
      if (kv_n1 > 0) mbar_wait_bounded(&ctl->v_full[1], (kv_n1 - 1) & 1, kGWaitNs);
      if (land_n0 > 0) mbar_wait_bounded(&ctl->v_land[0], (land_n0 - 1) & 1, kGWaitNs);
      if (land_n1 > 0) mbar_wait_bounded(&ctl->v_land[1], (land_n1 - 1) & 1, kGWaitNs);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = tc::idesc_f16(128, 128, true, false, false);
      constexpr uint32_t kIdescPV = tc::idesc_f16(128, 128, false, false, true);  // fp16 P, fp16 V
      int prev_y = 0, prev_item = 0;
      for (int c = 0;; ++c) {
        const int ds = c % kDescRing;
        if (!g_wait(&ctl->desc_full[ds], (c / kDescRing) & 1, ctl, a.err_word)) break;
        const ChunkDesc* d = &ctl->desc[ds];
        const int end = d->end;
        const int Y = d->ybuf, item = d->item;
        if (!end) {
          const int X = c & 1;
          // the K buffer of item n completes once per use: phase (n / 2) & 1
          if (!g_wait(&ctl->k_full[Y], (item >> 1) & 1, ctl, a.err_word)) break;
          if (!g_wait(&ctl->q_full[X], (c >> 1) & 1, ctl, a.err_word)) break;
          tc::fence_after_sync();
          const uint32_t q_addr = smem_u32(q_s + X * kGQBytes);
          const uint32_t k_addr = smem_u32(k_s + Y * kGTile);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_ss(tmem + X * 128, tc::smem_desc_sw128(q_addr + (ks >> 2) * kGHalf + (ks & 3) * 32, 16, 1024),
                       tc::smem_desc_sw128(k_addr + (ks >> 2) * 1024 + (ks & 3) * 32, 16, 2048), kIdescS, ks > 0);
          tc::commit(&ctl->s_full[X]);
          tc::commit(&ctl->q_empty[X]);
          GTRACE(kGtS, c);
        }
        if (c >= 1) {
          // PV of the previous chunk: O(X') = P V, P (fp16, two keys per column) in columns
          // 0..63 of S buffer X', V the fp16 copy of the item's V
          const int cp = c - 1, Xp = cp & 1;
          if (!g_wait(&ctl->p_full[Xp], (cp >> 1) & 1, ctl, a.err_word)) break;
          if (!g_wait(&ctl->vx_ready[prev_item & 3], (prev_item >> 2) & 1, ctl, a.err_word)) break;
          // O buffer X' was read by the epilogue of chunk cp - 2
          if (cp >= 2 && !g_wait(&ctl->o_free[Xp], ((cp >> 1) - 1) & 1, ctl, a.err_word)) break;
          tc::fence_after_sync();
          const uint32_t v_addr = smem_u32(v_s + prev_y * kGTile);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc::mma_ts(tmem + 256 + Xp * 128, tmem + Xp * 128 + ks * 8,
                       tc::smem_desc_sw128(v_addr + ks * 4096, 1024, 2048), kIdescPV, ks > 0);
          tc::commit(&ctl->pv_done[Xp]);
          GTRACE(kGtPV, cp);
          // the previous chunk was its item's last: its K/V buffer is free once this PV completes
          if (end || item != prev_item) tc::commit(&ctl->kv_empty[prev_y]);
          mbar_arrive(&ctl->desc_empty[cp % kDescRing]);
        }
        if (end) break;
        prev_y = Y;
        prev_item = item;
      }
      // every MMA issued must complete before TMEM is released
      tc::commit(&ctl->mma_fin);
      mbar_wait_bounded(&ctl->mma_fin, 0, kGWaitNs);
    }
  } else if (warp == 2 || warp == 3) {
    // ---------------------------------------------------------------- merge warps
    // Warp 2 takes chunks 0, 2, ..., warp 3 chunks 1, 3, ...: once a chunk's partials are stored
    // and fenced it releases the descriptor and counts one ticket per (token, kv head); a token
    // whose count reaches its partial total is queued. Queued tokens' partials (and their
    // (lse, exponent) pairs) stream through a ring of bulk copies and are merged with a running
    // maximum, so loads for later partials are in flight while earlier ones are summed. The loop
    // never blocks on one event while another could make progress.
    const int m = warp - 2;
    constexpr int kSlotBytes = kG * kHeadDim * 2;  // one partial of one (token, kv head)
    constexpr int kSlots = kRingBytes / kSlotBytes;
    static_assert(kSlots <= kMaxSlots, "ring slots");
    constexpr int kLanesPerHead = 32 / kG;
    constexpr int kE = kHeadDim / kLanesPerHead;  // dims per lane: 32 or 64
    uint8_t* ring = ring_s + m * kRingBytes;
    float2* rml = &ctl->ring_ml[m][0][0];
    uint64_t* rfull = ctl->ring_full[m];
    int4* tq = ctl->tq[m];
    const int h = lane / kLanesPerHead, d0 = (lane % kLanesPerHead) * kE;
    const int hkv = a.num_kv_heads;
    // this warp's inbox: the tasks x = token * Hkv + head with x % n_mw == me, in order of x
    const int me = static_cast<int>(blockIdx.x) * 2 + m;
    const int64_t n_x = static_cast<int64_t>(w.T1 - w.T0) * hkv;
    const int expected = static_cast<int>(n_x / w.n_mw + (n_x % w.n_mw > me ? 1 : 0));
    const int4* inbox = w.inbox + static_cast<int64_t>(me) * w.inbox_cap;
    int head = 0;
    int conv_n = m;  // next item whose V this warp converts (items m, m + 2, ... use V buffer m)
    int c = m;
    bool end_seen = false, have_atom = false;
    int at_old = 0, at_tr = 0, at_nsel = 0, at_g = 0, at_n = 0;
    int tq_tail = 0;                          // tokens queued
    int iss_task = 0, iss_j = 0, ri_iss = 0;  // next partial to load (task, slot, ring sequence)
    int con_task = 0, con_j = 0, ri_con = 0;  // next partial to merge
    float acc[kE];
#pragma unroll
    for (int i = 0; i < kE; ++i) acc[i] = 0.f;
    float L = -INFINITY, den = 0.f;
    unsigned long long idle_t0 = 0;
    bool failed = false;
    while (true) {
      bool progress = false;
      // (0) the V of this warp's next item, once it has landed: converted in place to fp16 as
      // V * 2^-e, e putting max |V| at 2^14..2^15 (exact: bf16 has 8 significant bits, fp16 keeps
      // 29 binades below that maximum), for the single fp16 PV MMA
      {
        bool landed = false;
        if (lane == 0) landed = mbar_try_wait(&ctl->v_full[m], (conv_n >> 1) & 1);
        landed = __shfl_sync(0xffffffffu, landed, 0);
        if (landed) landed = __all_sync(0xffffffffu, mbar_wait_bounded(&ctl->v_full[m], (conv_n >> 1) & 1, kGWaitNs));
        if (landed) {
          const uint32_t vb = smem_u32(v_s + m * kGTile);
          uint32_t mxv = 0;
#pragma unroll 8
          for (int q = 0; q < kGTile / 16 / 32; ++q) {
            uint32_t x0, x1, x2, x3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                         : "r"(vb + (lane + 32 * q) * 16));
            // |bf16| bit patterns compare like the magnitudes
            mxv = max(mxv, max(max(x0 & 0x7fff7fffu, x1 & 0x7fff7fffu), max(x2 & 0x7fff7fffu, x3 & 0x7fff7fffu)) >> 16);
            mxv = max(mxv, max(max(x0 & 0x7fffu, x1 & 0x7fffu), max(x2 & 0x7fffu, x3 & 0x7fffu)));
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mxv = max(mxv, __shfl_xor_sync(0xffffffffu, mxv, off));
          const float vm = __uint_as_float(mxv << 16);
          int e = 0;
          if (vm > 0.f) e = static_cast<int>((__float_as_uint(vm) >> 23) & 0xffu) - 127 - 14;
          e = max(-100, min(100, e));
          const float sc = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
#pragma unroll 8
          for (int q = 0; q < kGTile / 16 / 32; ++q) {
            const uint32_t ad = vb + (lane + 32 * q) * 16;
            uint32_t x0, x1, x2, x3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3) : "r"(ad));
            g_sts128(ad, pack_f16(bf16_lo(x0) * sc, bf16_hi(x0) * sc), pack_f16(bf16_lo(x1) * sc, bf16_hi(x1) * sc),
                     pack_f16(bf16_lo(x2) * sc, bf16_hi(x2) * sc), pack_f16(bf16_lo(x3) * sc, bf16_hi(x3) * sc));
          }
          // the tensor core reads the copy through the async proxy
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          if (lane == 0) ctl->vexp[conv_n & 3] = e;
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->vx_ready[conv_n & 3]);
          conv_n += 2;
          progress = true;
        }
      }
      // the tickets of the last chunk taken (their atomics were issued one step earlier, so the
      // round trip is mostly over): a token that is now complete is announced to its merge warp
      // (the fence orders every partial the ticket counted before the flag)
      auto resolve_tickets = [&]() {
        const bool done = lane < at_n && at_old + 1 == at_nsel;
        const uint32_t dm = __ballot_sync(0xffffffffu, done);
        if (dm) {
          __threadfence();
          if (done) {
            const int64_t x = static_cast<int64_t>(at_tr) * hkv + at_g;
            int* flag = reinterpret_cast<int*>(w.inbox + (x % w.n_mw) * w.inbox_cap + x / w.n_mw) + 3;
            asm volatile("st.volatile.global.s32 [%0], %1;" ::"l"(flag), "r"(1) : "memory");
          }
        }
        have_atom = false;
      };
      // (1) the next chunk, once its partials are fenced
      if (!end_seen) {
        const int ds = c % kDescRing;
        const uint32_t ph = (c / kDescRing) & 1;
        bool got = false;
        if (lane == 0) got = mbar_try_wait(&ctl->desc_full[ds], ph);
        got = __shfl_sync(0xffffffffu, got, 0);
        // once lane 0 has seen the phase complete, every lane waits on it (returns at once) so
        // that each lane's reads of the descriptor are ordered after it
        if (got) got = __all_sync(0xffffffffu, mbar_wait_bounded(&ctl->desc_full[ds], ph, kGWaitNs));
        if (got) {
          const ChunkDesc* d = &ctl->desc[ds];
          if (d->end) {
            end_seen = true;
            progress = true;
          } else {
            bool pd = false;
            if (lane == 0) pd = mbar_try_wait(&ctl->part_done[ds], ph);
            pd = __shfl_sync(0xffffffffu, pd, 0);
            if (pd) pd = __all_sync(0xffffffffu, mbar_wait_bounded(&ctl->part_done[ds], ph, kGWaitNs));
            if (pd) {
              if (have_atom) resolve_tickets();
              if (lane == 0) GTRACE(kGtM0, c);
              at_g = d->g;
              at_n = d->n_tok;
              at_tr = lane < at_n ? d->tr[lane] : 0;
              at_nsel = lane < at_n ? d->nsel[lane] : 0;
              __syncwarp();
              if (lane == 0) mbar_arrive(&ctl->desc_empty[ds]);
              // the softmax warps fenced the partials before announcing them
              at_old = lane < at_n ? atomicAdd(w.tickets + static_cast<int64_t>(at_tr) * hkv + at_g, 1) : -2;
              have_atom = true;
              c += 2;
              progress = true;
            }
          }
        }
      }
      if (end_seen && have_atom) {
        resolve_tickets();
        progress = true;
      }
      // (2) bulk loads of queued partials while the ring has room
      while (ri_iss - ri_con < kSlots && iss_task < tq_tail) {
        const int4 t = tq[iss_task % kTaskQ];
        const int slot = ri_iss % kSlots;
        const int64_t pidx = (static_cast<int64_t>(t.x) * hkv + t.y) * a.k + iss_j;
        if (lane == 0) {
          mbar_arrive_expect_tx(&rfull[slot], kSlotBytes + kG * 8);
          bulk_load(ring + slot * kSlotBytes, w.part + pidx * kG * kHeadDim, kSlotBytes, &rfull[slot]);
          bulk_load(rml + slot * 16, w.ml + pidx * kG, kG * 8, &rfull[slot]);
        }
        if (++iss_j == t.z) {
          iss_j = 0;
          ++iss_task;
        }
        ++ri_iss;
        progress = true;
      }
      // (3) merge every landed partial
      while (ri_con < ri_iss) {
        const int slot = ri_con % kSlots;
        bool rdy = false;
        if (lane == 0) rdy = mbar_try_wait(&rfull[slot], (ri_con / kSlots) & 1);
        rdy = __shfl_sync(0xffffffffu, rdy, 0);
        if (rdy) rdy = __all_sync(0xffffffffu, mbar_wait_bounded(&rfull[slot], (ri_con / kSlots) & 1, kGWaitNs));
        if (rdy) {
          const float2 me = rml[slot * 16 + h];
          if (me.x > L) {
            const float sc = ex2(L - me.x);  // 0 while nothing is accumulated
            den *= sc;
#pragma unroll
            for (int i = 0; i < kE; ++i) acc[i] *= sc;
            L = me.x;
          }
          den += ex2(me.x - L);
          const float f = ex2(me.x - L + me.y);
          const uint32_t src = smem_u32(ring + slot * kSlotBytes + (h * kHeadDim + d0) * 2);
#pragma unroll
          for (int q = 0; q < kE / 8; ++q) {
            uint32_t x0, x1, x2, x3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                         : "r"(src + 16 * q));
            acc[8 * q + 0] = fmaf(f, f16_lo(x0), acc[8 * q + 0]);
            acc[8 * q + 1] = fmaf(f, f16_hi(x0), acc[8 * q + 1]);
            acc[8 * q + 2] = fmaf(f, f16_lo(x1), acc[8 * q + 2]);
            acc[8 * q + 3] = fmaf(f, f16_hi(x1), acc[8 * q + 3]);
            acc[8 * q + 4] = fmaf(f, f16_lo(x2), acc[8 * q + 4]);
            acc[8 * q + 5] = fmaf(f, f16_hi(x2), acc[8 * q + 5]);
            acc[8 * q + 6] = fmaf(f, f16_lo(x3), acc[8 * q + 6]);
            acc[8 * q + 7] = fmaf(f, f16_hi(x3), acc[8 * q + 7]);
          }
          // the slot's generic reads precede the next bulk write into it
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          ++ri_con;
          const int4 t = tq[con_task % kTaskQ];
          if (++con_j == t.z) {
            // the token is complete: output rows and log-sum-exp, then drop its partial lines
            const int tt = w.T0 + t.x;
            const float inv = a.v_scale / den;
            uint16_t* dst = a.out + static_cast<int64_t>(tt) * a.out_row_stride +
                            static_cast<int64_t>(t.y * kG + h) * a.out_head_stride + d0;
#pragma unroll
            for (int q = 0; q < kE / 8; ++q)
              *reinterpret_cast<uint4*>(dst + 8 * q) = make_uint4(
                  pack_bf16(acc[8 * q] * inv, acc[8 * q + 1] * inv), pack_bf16(acc[8 * q + 2] * inv, acc[8 * q + 3] * inv),
                  pack_bf16(acc[8 * q + 4] * inv, acc[8 * q + 5] * inv), pack_bf16(acc[8 * q + 6] * inv, acc[8 * q + 7] * inv));
            if (a.lse != nullptr && (lane % kLanesPerHead) == 0)
              a.lse[static_cast<int64_t>(tt) * a.lse_row_stride + t.y * kG + h] = (L + log2f(den)) * kLn2;
            if ((d0 & 63) == 0) {
              const uint16_t* pp = w.part + ((static_cast<int64_t>(t.x) * hkv + t.y) * a.k * kG + h) * kHeadDim + d0;
              for (int j = 0; j < t.z; ++j) discard_l2(pp + static_cast<int64_t>(j) * kG * kHeadDim);
            }
#pragma unroll
            for (int i = 0; i < kE; ++i) acc[i] = 0.f;
            L = -INFINITY;
            den = 0.f;
            con_j = 0;
            ++con_task;
          }
          progress = true;
        } else {
          break;
        }
      }
      // (5) this warp's inbox: the leading run of ready tasks joins the merge queue
      if (head < expected && tq_tail - con_task < 4) {
        const int room = kTaskQ - (tq_tail - con_task);
        const int p = head + lane;
        int flag = 0;
        if (lane < room && p < expected)
          asm volatile("ld.volatile.global.s32 %0, [%1];" : "=r"(flag) : "l"(reinterpret_cast<const int*>(inbox + p) + 3));
        const uint32_t ready = __ballot_sync(0xffffffffu, flag != 0);
        const int run = ready == 0xffffffffu ? 32 : __ffs(~ready) - 1;
        if (run > 0) {
          // acquire the partials the flags announce, for the generic and the bulk-copy proxy
          __threadfence();
          asm volatile("fence.proxy.async.global;" ::: "memory");
          int4 e = make_int4(0, 0, 0, 0);
          if (lane < run) e = __ldcg(inbox + p);
          const bool real = lane < run && e.z > 0;  // tasks with nothing to merge are dropped
          const uint32_t rm = __ballot_sync(0xffffffffu, real);
          if (real) tq[(tq_tail + __popc(rm & lanemask_lt())) % kTaskQ] = make_int4(e.x, e.y, e.z, 0);
          tq_tail += __popc(rm);
          head += run;
          __syncwarp();
          progress = true;
        }
      }
      if (end_seen && !have_atom && head == expected && con_task == tq_tail && ri_con == ri_iss &&
          conv_n >= *reinterpret_cast<volatile int32_t*>(&ctl->items_total))
        break;
      if (progress) {
        idle_t0 = 0;
      } else {
        __nanosleep(64);
        const unsigned long long now = global_timer_ns();
        if (idle_t0 == 0) {
          idle_t0 = now;
        } else if (now - idle_t0 > kGWaitNs) {
          failed = true;
          break;
        }
      }
    }
    if (failed && lane == 0) {
      set_err(a.err_word, PBS_DEVERR_TIMEOUT);
      atomicExch(&ctl->abort, 1);
    }
    // copies still in flight (only after a give-up) must land before the CTA exits
    if (lane == 0)
      for (int r = ri_con; r < ri_iss; ++r) mbar_wait_bounded(&rfull[r % kSlots], (r / kSlots) & 1, kGWaitNs);
  } else {
    // ---------------------------------------------------------------- softmax + epilogue
    // Warps 4-11 take every chunk in turn, two warps per 32-lane TMEM quadrant: warp part p owns
    // key columns [64 p, 64 p + 64) of S and head-dim columns [64 p, 64 p + 64) of O. The two
    // parts' row maxima meet in shared memory;
    // P (fp16, two keys per column) goes to columns 32 p .. 32 p + 31 of the same S buffer once
    // both parts have read their S columns. Then the partial of chunk c - 1 (O / l as fp16 with
    // its item's V exponent) is stored while PV(c) runs.
    const int sw = warp - 4, quad = sw & 3, part = sw >> 2;
    const int row = quad * 32 + lane;  // TMEM lane
    const int j = row / kG, h = row % kG;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = a.scale_log2;
    float m_prev = 0.f, l_prev = 0.f;  // chunk c - 1: row maximum (log2 units), this part's sum
    int pending = -1;                  // chunk whose partial stores are not yet fenced
    const ChunkDesc* dprev = nullptr;
    for (int c = 0;; ++c) {
      const int ds = c % kDescRing, X = c & 1;
      if (!g_warp_wait(&ctl->desc_full[ds], (c / kDescRing) & 1, ctl, a.err_word)) break;
      const ChunkDesc* d = &ctl->desc[ds];
      const bool end = d->end != 0;
      uint32_t v[64];
      if (!end) {
        if (!g_warp_wait(&ctl->s_full[X], (c >> 1) & 1, ctl, a.err_word)) break;
        tc::fence_after_sync();
        if (sw == 0 && lane == 0) GTRACE(kGtSm0, c);
        const uint32_t ts = tmem + X * 128 + lane_off + 64 * part;
        tc::ld32(ts, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tc::ld32(ts + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      }
      tc::wait_ld();
      // ---- softmax of chunk c
      const int lim = !end && j < d->n_tok ? d->lim[j] : 0;
      const int nval = min(max(lim - 64 * part, 0), 64);  // valid keys among my columns
      const bool full = __all_sync(0xffffffffu, nval == 64);
      float mx = -INFINITY;
      if (!end) {
        if (full) {
#pragma unroll
          for (int i = 0; i < 64; i += 2) mx = fmaxf(mx, fmaxf(__uint_as_float(v[i]), __uint_as_float(v[i + 1])));
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) mx = i < nval ? fmaxf(mx, __uint_as_float(v[i])) : mx;
        }
        ctl->xchg[c & 1][part][row] = mx;
      }
      // both parts have read their S columns and posted their maxima (and finished chunk c - 1)
      asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory");
      float m = 0.f, lp = 0.f;
      if (!end) {
        mx = fmaxf(mx, ctl->xchg[c & 1][part ^ 1][row]);
        m = lim > 0 ? mx * sl2 : 0.f;
        float l0 = 0.f, l1 = 0.f;
        uint32_t pk[32];
        if (full) {
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            const float p0 = ex2(fmaf(__uint_as_float(v[i]), sl2, -m));
            const float p1 = ex2(fmaf(__uint_as_float(v[i + 1]), sl2, -m));
            l0 += p0;
            l1 += p1;
            pk[i >> 1] = pack_f16(p0, p1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 64; i += 2) {
            const float p0 = i < nval ? ex2(fmaf(__uint_as_float(v[i]), sl2, -m)) : 0.f;
            const float p1 = i + 1 < nval ? ex2(fmaf(__uint_as_float(v[i + 1]), sl2, -m)) : 0.f;
            l0 += p0;
            l1 += p1;
            pk[i >> 1] = pack_f16(p0, p1);
          }
        }
        tc::st32(tmem + X * 128 + lane_off + 32 * part, pk);
        lp = l0 + l1;
        // four slots: the partner reads slot c & 3 after the next chunk's quad barrier
        ctl->lsum[c & 3][part][row] = lp;
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full[X]);
        if (sw == 0 && lane == 0) GTRACE(kGtSm1, c);
      }
      // ---- partial of chunk c - 1
      if (c >= 1) {
        // the chunk before it, stored an iteration ago, is fenced and handed to its merge warp
        if (pending >= 0) {
          __threadfence();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->part_done[pending % kDescRing]);
          pending = -1;
        }
        if (sw == 0 && lane == 0) GTRACE(kGtE0, c - 1);
        // O(c - 1), read once P(c) is out (so PV(c) is not held up, and S and O never share the
        // registers)
        uint32_t o[64];
        if (!g_warp_wait(&ctl->pv_done[X ^ 1], ((c - 1) >> 1) & 1, ctl, a.err_word)) break;
        tc::fence_after_sync();
        const uint32_t to = tmem + 256 + (X ^ 1) * 128 + lane_off + 64 * part;
        tc::ld32(to, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
        tc::ld32(to + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
        tc::wait_ld();
        // O buffer (c - 1) % 2 is read: PV(c + 1) may overwrite it
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->o_free[X ^ 1]);
        const int itp = dprev->item;
        if (!g_warp_wait(&ctl->vx_ready[itp & 3], (itp >> 2) & 1, ctl, a.err_word)) break;
        const int e = ctl->vexp[itp & 3];
        const float lt = l_prev + ctl->lsum[(c - 1) & 3][part ^ 1][row];
        const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
        const bool valid = j < dprev->n_tok;
        if (valid) {
          const int64_t prow =
              ((static_cast<int64_t>(dprev->tr[j]) * a.num_kv_heads + dprev->g) * a.k + dprev->slot[j]) * kG + h;
          uint16_t* dst = w.part + prow * kHeadDim + 64 * part;
#pragma unroll
          for (int q8 = 0; q8 < 8; ++q8) {
            const uint32_t* f = &o[8 * q8];
            *reinterpret_cast<uint4*>(dst + 8 * q8) = make_uint4(
                pack_f16(__uint_as_float(f[0]) * inv_l, __uint_as_float(f[1]) * inv_l),
                pack_f16(__uint_as_float(f[2]) * inv_l, __uint_as_float(f[3]) * inv_l),
                pack_f16(__uint_as_float(f[4]) * inv_l, __uint_as_float(f[5]) * inv_l),
                pack_f16(__uint_as_float(f[6]) * inv_l, __uint_as_float(f[7]) * inv_l));
          }
          if (part == 0) *reinterpret_cast<float2*>(w.ml + prow) = make_float2(m_prev + log2f(lt), static_cast<float>(e));
        }
        if (sw == 0 && lane == 0) GTRACE(kGtE1, c - 1);
        pending = c - 1;
      }
      if (end) break;
      m_prev = m;
      l_prev = lp;
      dprev = d;
    }
    if (pending >= 0) {
      __threadfence();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->part_done[pending % kDescRing]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 2) {
    tc::fence_after_sync();
    tc::dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) GTRACE(kGtEnd, 0);
}

}  // namespace

#ifdef PBS_TRACE
}  // namespace pbs
// Trace build only: choose the traced CTA, and copy the timestamps out (host buffer of
// kGtCount int64). Not part of the C ABI.
extern "C" __attribute__((visibility("default"))) int pbs_debug_gtrace_set(int cta) {
  return cudaMemcpyToSymbol(pbs::g_gtrace_cta, &cta, sizeof(int)) == cudaSuccess ? 0 : 5;
}
extern "C" __attribute__((visibility("default"))) int pbs_debug_gtrace_get(long long* host, int n) {
  if (n > pbs::kGtCount) n = pbs::kGtCount;
  return cudaMemcpyFromSymbol(host, pbs::g_gtrace, sizeof(long long) * n) == cudaSuccess ? 0 : 5;
}
namespace pbs {
#endif

bool prefill_gather_supported(const AttendArgs& a) {
  // buckets are built from top-k ids; a prebuilt table carries page ids only
  return a.sparse_bt == nullptr && a.kv_dtype == PBS_KV_BF16 && (a.group == 8 || a.group == 16) && a.max_blocks <= kGatherMaxBlocks &&
         a.page_stride_bytes == static_cast<int64_t>(a.num_kv_heads) * 8192 &&
         a.num_pages * a.num_kv_heads <= 0x7fffffffLL && a.out_head_stride % 8 == 0 && a.out_row_stride % 8 == 0 &&
         reinterpret_cast<uintptr_t>(a.out) % 16 == 0 && a.q_head_stride % 8 == 0 && a.q_row_stride % 8 == 0 &&
         reinterpret_cast<uintptr_t>(a.q) % 16 == 0;
}

namespace {
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct GatherLayout {
  size_t part, ml, tickets, pairs, chunks, wins, inbox, total;
  int num_win, ccap;
};

GatherLayout gather_layout(int64_t seg_tokens, int num_reqs, int num_heads, int num_kv_heads, int k, int max_blocks) {
  GatherLayout L = {};
  const int group = num_heads / num_kv_heads;
  const int tok = kGRows / (group > 8 ? group : 8);
  L.num_win = static_cast<int>(seg_tokens / kGatherWinTok + 2 * static_cast<int64_t>(num_reqs) + 1);
  // chunks of one kv head in a window: sum over its buckets of ceil(tokens / tok) <= (entries +
  // buckets * (tok - 1)) / tok, with entries <= 256 k and buckets <= min(max_blocks, entries)
  const int64_t entries = static_cast<int64_t>(kGatherWinTok) * k;
  const int64_t buckets = std::min<int64_t>(max_blocks, entries);
  L.ccap = static_cast<int>(((entries + buckets * (tok - 1)) / tok + 1) * num_kv_heads);
  size_t off = 0;
  L.part = off;
  off = align256(off + static_cast<size_t>(seg_tokens) * num_heads * k * kHeadDim * 2);
  L.ml = off;
  off = align256(off + static_cast<size_t>(seg_tokens) * num_heads * k * 8);
  L.tickets = off;
  off = align256(off + static_cast<size_t>(seg_tokens) * num_kv_heads * 4);
  L.pairs = off;
  off = align256(off + static_cast<size_t>(L.num_win) * kGatherWinTok * k * 4);
  L.chunks = off;
  off = align256(off + static_cast<size_t>(L.num_win) * L.ccap * 16);
  L.wins = off;
  off = align256(off + static_cast<size_t>(L.num_win) * 8 * 4);
  // merge tasks: one per (token, kv head), plus one task of rounding per merge warp
  L.inbox = off;
  off = align256(off + (static_cast<size_t>(seg_tokens) * num_kv_heads + 2 * kGatherMaxSms) * 16);
  L.total = off;
  return L;
}
}  // namespace

size_t gather_workspace_bytes(int64_t seg_tokens, int num_reqs, int num_heads, int num_kv_heads, int k,
                              int max_blocks) {
  return gather_layout(seg_tokens, num_reqs, num_heads, num_kv_heads, k, max_blocks).total;
}

int64_t gather_segment_tokens(int64_t total_q, int num_reqs, int num_heads, int num_kv_heads, int k, int max_blocks,
                              size_t ws_bytes) {
  if (total_q <= kGatherMaxSegment &&
      gather_workspace_bytes(total_q, num_reqs, num_heads, num_kv_heads, k, max_blocks) <= ws_bytes)
    return total_q;
  // the largest multiple of the window that fits
  int64_t lo = 0, hi = std::min(total_q, kGatherMaxSegment) / kGatherWinTok;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) / 2;
    if (gather_workspace_bytes(mid * kGatherWinTok, num_reqs, num_heads, num_kv_heads, k, max_blocks) <= ws_bytes)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo * kGatherWinTok;
}

template <int kG>
cudaError_t launch_gather_g(const AttendArgs& a, const CUtensorMap& kv_map, const CUtensorMap& q_map, void* ws,
                            size_t ws_bytes, cudaStream_t stream) {
  const int64_t seg = gather_segment_tokens(a.num_rows, a.num_reqs, a.num_heads, a.num_kv_heads, a.k, a.max_blocks,
                                            ws_bytes);
  if (seg <= 0) return cudaErrorInvalidValue;
  const GatherLayout L = gather_layout(seg, a.num_reqs, a.num_heads, a.num_kv_heads, a.k, a.max_blocks);
  uint8_t* base = static_cast<uint8_t*>(ws);
  GatherWs w = {};
  w.part = reinterpret_cast<uint16_t*>(base + L.part);
  w.ml = reinterpret_cast<float2*>(base + L.ml);
  w.tickets = reinterpret_cast<int32_t*>(base + L.tickets);
  w.pairs = reinterpret_cast<int32_t*>(base + L.pairs);
  w.chunks = reinterpret_cast<int4*>(base + L.chunks);
  w.wins = reinterpret_cast<int32_t*>(base + L.wins);
  w.ccap = L.ccap;
  w.tok_per_chunk = kGRows / kG;
  w.inbox = reinterpret_cast<int4*>(base + L.inbox);

  const size_t idx_smem = static_cast<size_t>(2 * a.max_blocks + kGatherWinTok * a.k) * 4;
  cudaError_t e = cudaFuncSetAttribute(gather_index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(idx_smem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gather_attend_kernel<kG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kGSmem));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  sms = std::min(sms, kGatherMaxSms);
  // merge warps wait for tasks other CTAs announce, so every CTA must be resident: a
  // cooperative launch of one CTA per SM guarantees that
  w.n_mw = 2 * sms;
  for (int64_t t0 = 0; t0 < a.num_rows; t0 += seg) {
    w.T0 = static_cast<int32_t>(t0);
    w.T1 = static_cast<int32_t>(std::min<int64_t>(a.num_rows, t0 + seg));
    w.num_win = static_cast<int32_t>((w.T1 - w.T0) / kGatherWinTok + 2 * static_cast<int64_t>(a.num_reqs) + 1);
    w.inbox_cap = static_cast<int32_t>((static_cast<int64_t>(w.T1 - w.T0) * a.num_kv_heads + w.n_mw - 1) / w.n_mw);
    gather_index_kernel<<<w.num_win, kIdxThreads, idx_smem, stream>>>(a, w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms));
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = kGSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, gather_attend_kernel<kG>, kv_map, q_map, a, w);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_prefill_gather(const AttendArgs& a, const CUtensorMap& kv_map, const CUtensorMap& q_map, void* ws,
                                  size_t ws_bytes, cudaStream_t stream) {
  return a.group == 16 ? launch_gather_g<16>(a, kv_map, q_map, ws, ws_bytes, stream)
                       : launch_gather_g<8>(a, kv_map, q_map, ws, ws_bytes, stream);
}

}  // namespace pbs
