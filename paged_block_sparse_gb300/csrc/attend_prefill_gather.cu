// Prefill attend by key block ("gathered rows") on the 5th-generation tensor cores (tcgen05 +
// TMEM): bf16, fp8-e4m3 and NVFP4 caches, GQA 8 or 16.
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
// of a window of 512 consecutive tokens of one request, and its MMA rows are the window's
// tokens that selected b, gathered 16 at a time (x 8 query heads = the 128-row M tile; 8 tokens
// x 16 heads at GQA 16). Every row of every tile does useful work except in a bucket's last
// chunk.
//
// * Images (before the attend; the tile kernel's conversion kernels): the V of every (request,
//   block, kv head) as fp16 V * 2^-e in the 128B-swizzled layout of a shared-memory stage, and
//   for fp8 / NVFP4 caches K as bf16 likewise (exact). A bf16 K comes straight from the packed
//   cache through the per-block tensor map.
// * Index kernel (one CTA per window): each token's distinct valid blocks, sorted, give the
//   token's partial slots and count; tokens are bucketed by block (shared-memory histogram,
//   block scan, scatter). Tokens with no valid block get zero output here.
// * Attend kernel (persistent, one CTA per SM): windows are taken in order and CTA i takes chunks
//   [i C / G, (i + 1) C / G) of a window with C chunks, so every CTA works on the same few
//   windows at a time and their Q rows and K / V images stay in L2. Warp 0 loads the K of a
//   (block, kv head) item (one 32 KiB copy) into one of two buffers, writes each chunk's
//   descriptor (tokens, partial slots, own-block key limits, the V image's exponent) into an
//   8-deep ring and gathers the chunk's Q rows (one tensor copy per token: its G heads, both
//   64-dim halves); warp 3 loads each item's V image into one of two buffers. Warp 1 (one
//   thread) issues S(c) = Q K^T into TMEM buffer c % 2 and PV(c - 1), in whichever order their
//   operands arrive, so the softmax of chunk c overlaps PV(c - 1) and S(c + 1). Warps 4-11 (two
//   per TMEM lane quadrant, 64 keys each) take the softmax of chunk c, writing P as fp16 over S,
//   then store chunk c - 1's partial while PV(c) runs.
// * With the tile kernel's Q map, each request's leading tiles (tokens before position
//   1.5 x 128 k, `leading_tiles`) go to the tile kernel on the same images, and the index kernel
//   skips their tokens.
// * Softmax of one chunk (one key block): the row maximum over the block's valid keys (row
//   maxima of the two key halves meet in shared memory), P = 2^(s * scale * log2 e - m) <= 1 as
//   fp16 (one PV MMA per 16 keys against the fp16 V image). The partial is O / l (the image's
//   V * 2^-e keeps it below 2^15) as fp16 with (log2-sum-exp, e).
// * Merge kernel (one warp per (token, kv head)): the token's partials weighted by 2^(lse - max),
//   the bf16 output and the log-sum-exp.
// * TMEM (512 columns): S / P double buffer (2 x 128) and O double buffer (2 x 128).
#include <algorithm>

#include "pbs_device.cuh"
#include "pbs_internal.h"
#include "tc_device.cuh"

namespace pbs {
namespace {

constexpr int kGRows = 128;                     // MMA M: tokens x query heads of a chunk
constexpr int kGThreads = 384;                  // 12 warps
constexpr int kDescRing = 8;                    // chunk descriptors in flight
constexpr int kGQBytes = kGRows * kHeadDim * 2;  // 32 KiB Q tile
constexpr int kGHalf = kGQBytes / 2;            // one 64-dim half of a Q, K or V tile: [128 rows][128 B]
constexpr int kGTile = 32768;                   // a block's K (or V) for one kv head
constexpr int kGSmemBig = 2 * kGQBytes + 4 * kGTile;  // Q x 2, K x 2, V x 2
constexpr unsigned long long kGWaitNs = 100000000ull;  // waits here last microseconds: 100 ms cap
constexpr int kIdxThreads = 1024;                // index kernel: 32 warps, 8 tokens of a window each
constexpr int kSoftWarpsG = 8;                  // softmax warps (4 - 11)
constexpr int kMergeWarps = 8;                  // warps per merge CTA

struct ChunkDesc {
  int32_t end;    // 1: no more work for this CTA
  int32_t b;      // key block
  int32_t g;      // kv head
  int32_t ybuf;   // K/V buffer of the item
  int32_t n_tok;  // tokens in this chunk
  int32_t item;   // the CTA's item number (phase of the K/V buffer barriers)
  int32_t req;    // request (the item's images are those of (req, b, g))
  int32_t vexp;   // the item's V image holds V * 2^-vexp
  int32_t tr[16];    // segment-relative token index
  int32_t slot[16];  // the token's partial slot for block b
  int32_t lim[16];   // keys of block b the token sees (128, or pos - 128 b + 1 for its own block)
};

struct GCtl {
  uint64_t desc_full[kDescRing];
  // released by the MMA thread (PV issued), the V producer and the softmax warps (partial stored)
  uint64_t desc_empty[kDescRing];
  uint64_t q_full[2], q_empty[2];
  // K buffer Y is free once the S of its item's last chunk has completed, V buffer Y once its PV
  // has: each is reloaded two items later, so both are fetched about two chunks ahead
  uint64_t k_full[2], k_empty[2], v_full[2], v_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t o_free[2];  // O buffer X has been read (softmax warps -> MMA)
  uint64_t mma_fin;
  uint32_t tmem_base;
  int32_t abort;
  ChunkDesc desc[kDescRing];
  int32_t ents[128];         // bucket entries of the producer's current batch
  float lsum[4][2][kGRows];  // chunk c & 3, key half, row: partial sum
  float xchg[2][2][kGRows];  // row maxima of the two key halves
};

// A batch of up to 8 consecutive chunks of one window (producer).
struct Batch {
  int w, base, nb, r, c0, ctx0, seq_len;
};

constexpr size_t kGSmem = kGSmemBig + sizeof(GCtl) + 1024;
static_assert(kGSmem <= 232448, "shared memory layout exceeds 227 KiB");

#ifdef PBS_TRACE
// Trace build only: one CTA records SM-clock timestamps of the first kGtChunks chunks' pipeline
// events.
constexpr int kGtChunks = 64;
enum GTraceEv { kGtStart, kGtEnd, kGtProd = 2, kGtK = kGtProd + kGtChunks, kGtV = kGtK + kGtChunks,
                kGtS = kGtV + kGtChunks, kGtPV = kGtS + kGtChunks, kGtSm0 = kGtPV + kGtChunks,
                kGtSm1 = kGtSm0 + kGtChunks, kGtE0 = kGtSm1 + kGtChunks, kGtE1 = kGtE0 + kGtChunks,
                kGtCount = kGtE1 + kGtChunks };
__device__ long long g_gtrace[kGtCount];
__device__ int g_gtrace_cta;
// the traced CTA is read once per thread, so an event costs one clock read and one store
#define GTRACE_INIT const bool gt_on_ = blockIdx.x == static_cast<unsigned>(g_gtrace_cta)
#define GTRACE(ev, c) do { if (gt_on_ && (c) < kGtChunks) g_gtrace[(ev) + (c)] = clock64(); } while (0)
#else
#define GTRACE_INIT do { } while (0)
#define GTRACE(ev, c) do { } while (0)
#endif

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

__device__ __forceinline__ void g_tma_5d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1, int c2, int c3,
                                         int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

// 32 bytes to global memory in one store (32-byte aligned address).
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]),
               "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The lower / upper half of an f16x2 word as float (exact).
__device__ __forceinline__ float g_f16_lo(uint32_t x) {
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}" : "=f"(f) : "r"(x));
  return f;
}
__device__ __forceinline__ float g_f16_hi(uint32_t x) {
  float f;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, hi;\n\t}" : "=f"(f) : "r"(x));
  return f;
}

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
  // tokens of the request's leading tiles belong to the tile kernel (AttendArgs::tile_pos_limit)
  const int dense_tiles = a.tile_pos_limit > 0 ? leading_tiles(s_win[5] - ctx0, ctx0, a.tile_pos_limit, kTok) : 0;
  for (int tt = warp; tt < n; tt += kIdxThreads / 32) {
    const int t = ta + tt;
    const int tr = t - w.T0;
    if ((t - c0) / kTok < dense_tiles) {
      if (lane == 0) {
        s_tn[tt] = 0;
        w.nparts[tr] = 0;
      }
      continue;
    }
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
      if (kk <= 32) {
        // one entry per lane: the lanes holding one value form one match group, its lowest keeps it
        const uint32_t grp = __match_any_sync(0xffffffffu, v0 ? b0 : -1 - lane);
        k0 = v0 && __ffs(grp) - 1 == lane;
      } else {
        for (int j = 0; j < kk; ++j) {
          const int bj = j < 32 ? __shfl_sync(0xffffffffu, b0, j) : __shfl_sync(0xffffffffu, b1, j - 32);
          const bool vj = ((j < 32 ? vm0 >> j : vm1 >> (j - 32)) & 1u) != 0;
          if (vj) {
            if (j < lane && bj == b0) k0 = false;
            if (j < lane + 32 && bj == b1) k1 = false;
          }
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
      // the token's pairs take n_t consecutive entries (one atomic per token, not per pair)
      int base = 0;
      if (lane == 0) base = atomicAdd(&s_np, n_t);
      base = __shfl_sync(0xffffffffu, base, 0);
      const uint32_t lt = lanemask_lt();
      if (k0) {
        atomicAdd(&cnt[b0], 1);
        pairs_s[base + __popc(km0 & lt)] = (b0 << 16) | (tt << 6) | r0;
      }
      if (k1) {
        atomicAdd(&cnt[b1], 1);
        pairs_s[base + __popc(km0) + __popc(km1 & lt)] = (b1 << 16) | (tt << 6) | r1;
      }
    }
    if (lane == 0) {
      s_tn[tt] = n_t;
      w.nparts[tr] = n_t;  // the merge kernel's partial count for this token
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
  // lanes of a warp that fill the same bucket take consecutive places with one atomic
  const int np = s_np;
  for (int p0 = 0; p0 < np; p0 += kIdxThreads) {
    const int p = p0 + threadIdx.x;
    const bool act = p < np;
    const int v = act ? pairs_s[p] : 0;
    const int b = act ? v >> 16 : -1 - lane;  // idle lanes in groups of their own
    const uint32_t grp = __match_any_sync(0xffffffffu, b);
    const int leader = __ffs(grp) - 1;
    int at = 0;
    if (act && lane == leader) at = atomicAdd(&cur[b], __popc(grp));
    at = __shfl_sync(0xffffffffu, at, leader) + __popc(grp & lanemask_lt());
    if (act) {
      const int tt = (v >> 6) & 1023, rank = v & 63;
      w.pairs[pair_base + at] = ((ta + tt - w.T0) << 12) | ((s_tn[tt] - 1) << 6) | rank;
    }
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
  uint8_t* q_s = big;                 // 2 x 32 KiB: [row atom][half][8 rows][128 B]
  uint8_t* k_s = big + 2 * kGQBytes;  // 2 x 32 KiB: [half][128 keys][128 B]
  uint8_t* v_s = k_s + 2 * kGTile;    // 2 x 32 KiB: [half][128 keys][128 B] (fp16 image)
  GCtl* ctl = reinterpret_cast<GCtl*>(v_s + 2 * kGTile);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  GTRACE_INIT;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kDescRing; ++i) {
      mbar_init(&ctl->desc_full[i], 1);
      mbar_init(&ctl->desc_empty[i], 2 + kSoftWarpsG);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->q_full[i], 1);
      mbar_init(&ctl->q_empty[i], 1);
      mbar_init(&ctl->k_full[i], 1);
      mbar_init(&ctl->k_empty[i], 1);
      mbar_init(&ctl->v_full[i], 1);
      mbar_init(&ctl->v_empty[i], 1);
      mbar_init(&ctl->s_full[i], 1);
      mbar_init(&ctl->p_full[i], kSoftWarpsG);
      mbar_init(&ctl->pv_done[i], 1);
      mbar_init(&ctl->o_free[i], kSoftWarpsG);
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
    // ---------------------------------------------------------------- producer (Q, K, descriptors)
    // Windows in order; CTA i takes chunks [i C / G, (i + 1) C / G) of a window with C chunks.
    // Chunks go in batches of up to 8: the records of batch n + 2 and the bucket entries of
    // batch n + 1 are in flight while batch n is issued.
    if (lane == 0) {
      if (a.kconv == nullptr)
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
    // the V image exponent of each chunk of a batch whose records are in hand, one per lane
    auto load_exps = [&](const Batch& B, const int4& rec) {
      int e = 0;
      if (lane < B.nb)
        e = __ldg(a.vconv_exp + (static_cast<int64_t>(B.r) * a.max_blocks + (rec.x & 8191)) * a.num_kv_heads +
                  (rec.x >> 13));
      return e;
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
    int q_n0 = 0, q_n1 = 0, kv_n0 = 0, kv_n1 = 0;
    bool ok = true;
    Batch B0, B1, B2;
    next_batch(B0);
    int4 rec0 = load_recs(B0);
    int x0 = load_exps(B0, rec0);
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
      const int x1 = load_exps(B1, rec1);
      for (int jc = 0; jc < B0.nb && ok; ++jc, ++c) {
        const int rx = __shfl_sync(0xffffffffu, rec0.x, jc);
        const int b = rx & 8191, g = rx >> 13;
        const int n_tok = __shfl_sync(0xffffffffu, rec0.z, jc);
        const int phys = __shfl_sync(0xffffffffu, rec0.w, jc);
        const int vexp = __shfl_sync(0xffffffffu, x0, jc);
        // ---- a new (request, block, kv head): its K into the next K buffer (warp 3 loads V)
        if (B0.r != item_r || b != item_b || g != item_g) {
          ++n_item;
          item_r = B0.r;
          item_b = b;
          item_g = g;
          const int Y = n_item & 1;
          if (n_item >= 2) {
            bool go = true;
            if (lane == 0) go = g_wait(&ctl->k_empty[Y], ((n_item >> 1) - 1) & 1, ctl, a.err_word);
            if (!__shfl_sync(0xffffffffu, go, 0)) {
              ok = false;
              break;
            }
          }
          if (lane == 0) {
            mbar_arrive_expect_tx(&ctl->k_full[Y], kGTile);
            if (a.kconv != nullptr) {
              const int64_t image = (static_cast<int64_t>(B0.r) * a.max_blocks + b) * a.num_kv_heads + g;
              bulk_load(k_s + Y * kGTile, a.kconv + image * kGTile, kGTile, &ctl->k_full[Y]);
            } else {
              // one {64, 16 rows, head, 8 pages, K half} box; pages past the cache read as zeros
              const int64_t pbase = static_cast<int64_t>(phys) * a.block_page_stride;
              if (pbase < 0 || pbase + (kPagesPerBlock - 1) >= a.num_pages) set_err(a.err_word, PBS_DEVERR_PAGE_OOB);
              g_tma_5d(k_s + Y * kGTile, &kv_map, &ctl->k_full[Y], 0, 0, g, static_cast<int>(pbase), 0);
            }
          }
          if (Y == 0) ++kv_n0; else ++kv_n1;
          if (lane == 0) GTRACE(kGtK, c);
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
          d->req = B0.r;
          d->vexp = vexp;
        }
        // ---- gather the chunk's Q rows: token j -> its G rows, one {64, 8, 2, G / 8, 1} copy
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
        if (lane < n_tok)
          g_tma_5d(q_s + qb * kGQBytes + lane * kG * 256, &q_map, &ctl->q_full[qb], 0, 0, 0, g * (kG / 8), t_lane);
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
      x0 = x1;
      B1 = B2;
      rec1 = rec2;
    }
    // ---- end mark
    if (ok) {
      const int ds = c % kDescRing;
      bool go = true;
      if (c >= kDescRing && lane == 0) go = g_wait(&ctl->desc_empty[ds], ((c / kDescRing) - 1) & 1, ctl, a.err_word);
      if (__shfl_sync(0xffffffffu, go, 0) && lane == 0) {
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
    }
  } else if (warp == 3) {
    // ---------------------------------------------------------------- V producer
    // Follows the descriptors: the first chunk of every item loads the item's fp16 V image into
    // V buffer item % 2 once the PV of the item two before has completed.
    int v_n0 = 0, v_n1 = 0, prev_item = -1;
    for (int c = 0;; ++c) {
      const int ds = c % kDescRing;
      if (!g_warp_wait(&ctl->desc_full[ds], (c / kDescRing) & 1, ctl, a.err_word)) break;
      const ChunkDesc* d = &ctl->desc[ds];
      if (d->end) break;
      const int item = d->item, Y = d->ybuf;
      if (item != prev_item) {
        prev_item = item;
        if (item >= 2 && !g_warp_wait(&ctl->v_empty[Y], ((item >> 1) - 1) & 1, ctl, a.err_word)) break;
        if (lane == 0) {
          const int64_t image = (static_cast<int64_t>(d->req) * a.max_blocks + d->b) * a.num_kv_heads + d->g;
          mbar_arrive_expect_tx(&ctl->v_full[Y], kGTile);
          bulk_load(v_s + Y * kGTile, a.vconv + image * kGTile, kGTile, &ctl->v_full[Y]);
          GTRACE(kGtV, c);
        }
        if (Y == 0) ++v_n0; else ++v_n1;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->desc_empty[ds]);
    }
    if (lane == 0) {
      if (v_n0 > 0) mbar_wait_bounded(&ctl->v_full[0], (v_n0 - 1) & 1, kGWaitNs);
      if (v_n1 > 0) mbar_wait_bounded(&ctl->v_full[1], (v_n1 - 1) & 1, kGWaitNs);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = tc::idesc_f16(128, 128, true, false, false);
      constexpr uint32_t kIdescPV = tc::idesc_f16(128, 128, false, false, true);  // fp16 P, fp16 V
      int prev_y = 0, prev_item = 0;
      bool ok = true;
      for (int c = 0; ok; ++c) {
        const int ds = c % kDescRing;
        if (!g_wait(&ctl->desc_full[ds], (c / kDescRing) & 1, ctl, a.err_word)) break;
        const ChunkDesc* d = &ctl->desc[ds];
        const int end = d->end;
        const int Y = d->ybuf, item = d->item;
        const bool new_item = c >= 1 && (end || item != prev_item);
        // chunk c starts a new item (or there is none): the S of the previous item's last chunk,
        // issued before, is the last reader of its K buffer
        if (new_item) tc::commit(&ctl->k_empty[prev_y]);
        // S(c) and PV(c - 1), whichever has its operands first: S(c) waits for the chunk's Q and K,
        // PV(c - 1) for P(c - 1), its V and a free O buffer, and neither holds up the other. S(c)
        // reuses the S buffer of chunk c - 2, whose PV was issued in the previous iteration.
        bool s_todo = !end, pv_todo = c >= 1;
        const int X = c & 1, cp = c - 1, Xp = cp & 1;
        const unsigned long long t0 = global_timer_ns();
        while (s_todo || pv_todo) {
          bool progressed = false;
          if (pv_todo && mbar_test(&ctl->p_full[Xp], (cp >> 1) & 1) &&
              mbar_test(&ctl->v_full[prev_y], (prev_item >> 1) & 1) &&
              (cp < 2 || mbar_test(&ctl->o_free[Xp], ((cp >> 1) - 1) & 1))) {
            // O(X') = P V: P (fp16, two keys per column) in columns 0..63 of S buffer X', V the
            // item's fp16 image (keys 16ks.. = two 8-key groups 1 KiB apart; dims in two 64-wide
            // MN atoms 16 KiB apart)
            tc::fence_after_sync();
            const uint32_t v_addr = smem_u32(v_s + prev_y * kGTile);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              tc::mma_ts(tmem + 256 + Xp * 128, tmem + Xp * 128 + ks * 8,
                         tc::smem_desc_sw128(v_addr + ks * 2048, kGHalf, 1024), kIdescPV, ks > 0);
            tc::commit(&ctl->pv_done[Xp]);
            GTRACE(kGtPV, cp);
            // the previous chunk was its item's last: its V buffer is free once this PV completes
            if (new_item) tc::commit(&ctl->v_empty[prev_y]);
            mbar_arrive(&ctl->desc_empty[cp % kDescRing]);
            pv_todo = false;
            progressed = true;
          }
          // the K buffer of item n completes once per use: phase (n / 2) & 1
          if (s_todo && mbar_test(&ctl->k_full[Y], (item >> 1) & 1) && mbar_test(&ctl->q_full[X], (c >> 1) & 1)) {
            tc::fence_after_sync();
            const uint32_t q_addr = smem_u32(q_s + X * kGQBytes);
            const uint32_t k_addr = smem_u32(k_s + Y * kGTile);
            // dims 16ks..: Q half ks/4 1 KiB into each 2 KiB pair of 8-row atoms; K half ks/4 16
            // KiB apart, its 8-key groups 1 KiB apart
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              tc::mma_ss(tmem + X * 128, tc::smem_desc_sw128(q_addr + (ks >> 2) * 1024 + (ks & 3) * 32, 16, 2048),
                         tc::smem_desc_sw128(k_addr + (ks >> 2) * kGHalf + (ks & 3) * 32, 16, 1024), kIdescS,
                         ks > 0);
            tc::commit(&ctl->s_full[X]);
            tc::commit(&ctl->q_empty[X]);
            GTRACE(kGtS, c);
            s_todo = false;
            progressed = true;
          }
          if (!progressed) {
            if (global_timer_ns() - t0 > kGWaitNs) {
              set_err(a.err_word, PBS_DEVERR_TIMEOUT);
              atomicExch(&ctl->abort, 1);
              ok = false;
              break;
            }
            __nanosleep(20);
          }
        }
        if (end) break;
        prev_y = Y;
        prev_item = item;
      }
      // every MMA issued must complete before TMEM is released
      tc::commit(&ctl->mma_fin);
      mbar_wait_bounded(&ctl->mma_fin, 0, kGWaitNs);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax + partials
    // Warps 4-11 take every chunk in turn, two warps per 32-lane TMEM quadrant: warp part p owns
    // key columns [64 p, 64 p + 64) of S and head-dim columns [64 p, 64 p + 64) of O. The two
    // parts' row maxima meet in shared memory; P (fp16, two keys per column) goes to columns
    // 32 p .. 32 p + 31 of the same S buffer once both parts have read their S columns. Then the
    // partial of chunk c - 1 (O / l as fp16, with (log2-sum-exp, V exponent)) is stored while
    // PV(c) runs.
    const int sw = warp - 4, quad = sw & 3, part = sw >> 2;
    const int row = quad * 32 + lane;  // TMEM lane
    const int j = row / kG, h = row % kG;
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sl2 = a.scale_log2;
    float m_prev = 0.f, l_prev = 0.f;  // chunk c - 1: row maximum (log2 units), this part's sum
    int e_prev = 0;                    // chunk c - 1: its V image holds V * 2^-e
    const ChunkDesc* dprev = nullptr;
    for (int c = 0;; ++c) {
      const int ds = c % kDescRing, X = c & 1;
      if (!g_warp_wait(&ctl->desc_full[ds], (c / kDescRing) & 1, ctl, a.err_word)) break;
      const ChunkDesc* d = &ctl->desc[ds];
      const bool end = d->end != 0;
      uint32_t v[64];
      // the exponent of this chunk's V image, for its partial one iteration later
      const int e_cur = end ? 0 : d->vexp;
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
        // four slots: the partner reads slot c & 3 in the next iteration
        ctl->lsum[c & 3][part][row] = lp;
        tc::wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full[X]);
        if (sw == 0 && lane == 0) GTRACE(kGtSm1, c);
      }
      // ---- partial of chunk c - 1
      if (c >= 1) {
        // O(c - 1), read once P(c) is out (so PV(c) is not held up, and S and O never share the
        // registers)
        uint32_t o[64];
        if (!g_warp_wait(&ctl->pv_done[X ^ 1], ((c - 1) >> 1) & 1, ctl, a.err_word)) break;
        tc::fence_after_sync();
        if (sw == 0 && lane == 0) GTRACE(kGtE0, c - 1);
        const uint32_t to = tmem + 256 + (X ^ 1) * 128 + lane_off + 64 * part;
        tc::ld32(to, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
        tc::ld32(to + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
        tc::wait_ld();
        // O buffer (c - 1) % 2 is read: PV(c + 1) may overwrite it
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->o_free[X ^ 1]);
        const float lt = l_prev + ctl->lsum[(c - 1) & 3][part ^ 1][row];
        const float inv_l = lt > 0.f ? 1.f / lt : 0.f;
        if (j < dprev->n_tok) {
          const int64_t prow =
              ((static_cast<int64_t>(dprev->tr[j]) * a.num_kv_heads + dprev->g) * a.k + dprev->slot[j]) * kG + h;
          // 128 bytes of the row as four 32-byte stores: every store fills whole sectors
          uint16_t* dst = w.part + prow * kHeadDim + 64 * part;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t* f = &o[16 * q];
            uint32_t wv[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              wv[i] = pack_f16(__uint_as_float(f[2 * i]) * inv_l, __uint_as_float(f[2 * i + 1]) * inv_l);
            st_global_v8(dst + 16 * q, wv);
          }
          if (part == 0)
            w.ml[prow] = make_float2(m_prev + log2f(lt), static_cast<float>(e_prev));
        }
        // this warp is done with descriptor c - 1
        if (sw == 0 && lane == 0) GTRACE(kGtE1, c - 1);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->desc_empty[(c - 1) % kDescRing]);
      }
      if (end) break;
      m_prev = m;
      l_prev = lp;
      e_prev = e_cur;
      dprev = d;
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

// ------------------------------------------------------------------------------------------
// merge kernel: one warp per (segment token, kv head)
// ------------------------------------------------------------------------------------------
// The token's n partials P_s (O_s / l_s stored as fp16 times 2^-e_s) and their base-2
// log-sum-exps L_s combine to out = v_scale * sum_s 2^(L_s - M) 2^e_s P_s / sum_s 2^(L_s - M)
// with M = max_s L_s; the row's log-sum-exp is M + log2(sum_s 2^(L_s - M)) (times ln 2).
template <int kG>
__global__ void __launch_bounds__(kMergeWarps * 32) gather_merge_kernel(const AttendArgs a, const GatherWs w) {
  constexpr int kLanesPerHead = 32 / kG;        // 4 (GQA 8) or 2 (GQA 16)
  constexpr int kE = kHeadDim / kLanesPerHead;  // dims per lane: 32 or 64
  const int lane = threadIdx.x & 31;
  const int hkv = a.num_kv_heads;
  const int64_t x = static_cast<int64_t>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  if (x >= static_cast<int64_t>(w.T1 - w.T0) * hkv) return;
  const int tr = static_cast<int>(x / hkv), g = static_cast<int>(x % hkv);
  const int n = __ldg(w.nparts + tr);
  if (n <= 0) return;  // the index kernel wrote this token's zero output
  const int h = lane / kLanesPerHead, d0 = (lane % kLanesPerHead) * kE;
  const int64_t prow0 = x * a.k * kG + h;  // partial row of slot s: prow0 + s * kG
  // M: the lanes of head h share the n log-sum-exps (n <= 64), then meet by shuffles
  const int sub = lane % kLanesPerHead;
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < 64 / kLanesPerHead; ++i) {
    const int s = sub + i * kLanesPerHead;
    if (s < n) M = fmaxf(M, __ldg(&w.ml[prow0 + static_cast<int64_t>(s) * kG].x));
  }
#pragma unroll
  for (int off = 1; off < kLanesPerHead; off <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float L = 0.f;
  float acc[kE];
#pragma unroll
  for (int i = 0; i < kE; ++i) acc[i] = 0.f;
  // partials in groups whose loads are all in flight together
  constexpr int kGrp = kG == 8 ? 4 : 2;
  for (int s0 = 0; s0 < n; s0 += kGrp) {
    float2 mlv[kGrp];
    uint4 u4[kGrp][kE / 8];
#pragma unroll
    for (int s1 = 0; s1 < kGrp; ++s1)
      if (s0 + s1 < n) {
        const int64_t prow = prow0 + static_cast<int64_t>(s0 + s1) * kG;
        mlv[s1] = __ldg(&w.ml[prow]);
        const uint4* src = reinterpret_cast<const uint4*>(w.part + prow * kHeadDim + d0);
#pragma unroll
        for (int q = 0; q < kE / 8; ++q) u4[s1][q] = __ldg(src + q);
      }
#pragma unroll
    for (int s1 = 0; s1 < kGrp; ++s1)
      if (s0 + s1 < n) {
        const float wl = exp2f(mlv[s1].x - M);
        L += wl;
        const float f = wl * exp2f(mlv[s1].y);
#pragma unroll
        for (int q = 0; q < kE / 8; ++q) {
          const uint32_t wd[4] = {u4[s1][q].x, u4[s1][q].y, u4[s1][q].z, u4[s1][q].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            acc[8 * q + 2 * i] = fmaf(f, g_f16_lo(wd[i]), acc[8 * q + 2 * i]);
            acc[8 * q + 2 * i + 1] = fmaf(f, g_f16_hi(wd[i]), acc[8 * q + 2 * i + 1]);
          }
        }
      }
  }
  const float inv = a.v_scale / L;
  const int64_t t = static_cast<int64_t>(w.T0) + tr;
  uint16_t* dst = a.out + t * a.out_row_stride + static_cast<int64_t>(g * kG + h) * a.out_head_stride + d0;
#pragma unroll
  for (int q = 0; q < kE / 8; ++q)
    *reinterpret_cast<uint4*>(dst + 8 * q) =
        make_uint4(pack_bf16(acc[8 * q] * inv, acc[8 * q + 1] * inv), pack_bf16(acc[8 * q + 2] * inv, acc[8 * q + 3] * inv),
                   pack_bf16(acc[8 * q + 4] * inv, acc[8 * q + 5] * inv), pack_bf16(acc[8 * q + 6] * inv, acc[8 * q + 7] * inv));
  if (a.lse != nullptr && lane % kLanesPerHead == 0)
    a.lse[t * a.lse_row_stride + g * kG + h] = (M + log2f(L)) * kLn2;
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
  // buckets are built from top-k ids (a prebuilt table carries page ids only); a bf16 K comes
  // through the per-block map of a packed cache, fp8 / NVFP4 K and V from converted images
  const bool cache_ok =
      a.kv_dtype != PBS_KV_BF16 || a.page_stride_bytes == static_cast<int64_t>(a.num_kv_heads) * 8192;
  return a.sparse_bt == nullptr && cache_ok && (a.group == 8 || a.group == 16) && a.max_blocks <= kGatherMaxBlocks &&
         a.num_reqs <= 65535 && a.num_pages * a.num_kv_heads <= 0x7fffffffLL && a.out_head_stride % 8 == 0 &&
         a.out_row_stride % 8 == 0 && reinterpret_cast<uintptr_t>(a.out) % 16 == 0 && a.q_head_stride % 8 == 0 &&
         a.q_row_stride % 8 == 0 && reinterpret_cast<uintptr_t>(a.q) % 16 == 0;
}

namespace {
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The workspace: the conversion kernels' images (V and its exponents, then K, for every (request,
// block, kv head); the K images are used by fp8 / NVFP4 caches only), then per segment the
// partials, their (log2-sum-exp, exponent) pairs, each token's partial count, the bucket entries,
// the chunk records and the window records.
struct GatherLayout {
  size_t images, part, ml, nparts, pairs, chunks, wins, total;
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
  L.images = off;
  off = align256(off + prefill_tc_workspace_bytes(num_reqs, num_kv_heads, max_blocks, PBS_KV_FP8_E4M3));
  L.part = off;
  off = align256(off + static_cast<size_t>(seg_tokens) * num_heads * k * kHeadDim * 2);
  L.ml = off;
  off = align256(off + static_cast<size_t>(seg_tokens) * num_heads * k * 8);
  L.nparts = off;
  off = align256(off + static_cast<size_t>(seg_tokens) * 4);
  L.pairs = off;
  off = align256(off + static_cast<size_t>(L.num_win) * kGatherWinTok * k * 4);
  L.chunks = off;
  off = align256(off + static_cast<size_t>(L.num_win) * L.ccap * 16);
  L.wins = off;
  off = align256(off + static_cast<size_t>(L.num_win) * 8 * 4);
  L.total = off;
  return L;
}
}  // namespace

size_t gather_workspace_bytes(int64_t seg_tokens, int num_reqs, int num_heads, int num_kv_heads, int k,
                              int max_blocks) {
  if (prefill_tc_workspace_bytes(num_reqs, num_kv_heads, max_blocks, PBS_KV_FP8_E4M3) == 0) return 0;
  return gather_layout(seg_tokens, num_reqs, num_heads, num_kv_heads, k, max_blocks).total;
}

int64_t gather_segment_tokens(int64_t total_q, int num_reqs, int num_heads, int num_kv_heads, int k, int max_blocks,
                              size_t ws_bytes) {
  if (gather_workspace_bytes(kGatherWinTok, num_reqs, num_heads, num_kv_heads, k, max_blocks) == 0) return 0;
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
cudaError_t launch_gather_g(const AttendArgs& args, const CUtensorMap& kv_map, const CUtensorMap& q_map,
                            const CUtensorMap* tile_q_map, void* ws, size_t ws_bytes, cudaStream_t stream) {
  const int64_t seg = gather_segment_tokens(args.num_rows, args.num_reqs, args.num_heads, args.num_kv_heads, args.k,
                                            args.max_blocks, ws_bytes);
  if (seg <= 0) return cudaErrorInvalidValue;
  const GatherLayout L = gather_layout(seg, args.num_reqs, args.num_heads, args.num_kv_heads, args.k, args.max_blocks);
  uint8_t* base = static_cast<uint8_t*>(ws);
  // the images: V (fp16) and its exponents for every cache format, K (bf16) for fp8 / NVFP4
  AttendArgs a = args;
  const int64_t n_img = static_cast<int64_t>(a.num_reqs) * a.max_blocks * a.num_kv_heads;
  a.vconv = base + L.images;
  a.vconv_exp = reinterpret_cast<int32_t*>(a.vconv + n_img * kTileVBytes);
  a.kconv = a.kv_dtype == PBS_KV_BF16 ? nullptr : a.vconv + n_img * kTileVBytes + ((n_img * 4 + 255) / 256) * 256;
  cudaError_t e = launch_convert_images(a, stream);
  if (e != cudaSuccess) return e;
  // Tokens before position 128 k may select every block they see, and up to 1.5 x 128 k at least
  // two thirds of them, so a 16-token tile there wastes few MMA rows: the tile kernel takes each
  // request's leading tiles up to that position on the same images (no partials), this kernel
  // the rest. (Measured on the varlen prompts: limits of 1, 1.5, 2 and 3 x 128 k gave 2.10,
  // 2.03, 2.04 and 2.18 ms.)
  a.tile_pos_limit = 0;
  if (tile_q_map != nullptr && a.k <= 16 && prefill_tc_supported(a, true)) {
    a.tile_pos_limit = 3 * a.k * kSparseBlock / 2;
    e = launch_prefill_tc_attend(a, kv_map, *tile_q_map, stream);
    if (e != cudaSuccess) return e;
  }

  GatherWs w = {};
  w.part = reinterpret_cast<uint16_t*>(base + L.part);
  w.ml = reinterpret_cast<float2*>(base + L.ml);
  w.nparts = reinterpret_cast<int32_t*>(base + L.nparts);
  w.pairs = reinterpret_cast<int32_t*>(base + L.pairs);
  w.chunks = reinterpret_cast<int4*>(base + L.chunks);
  w.wins = reinterpret_cast<int32_t*>(base + L.wins);
  w.ccap = L.ccap;
  w.tok_per_chunk = kGRows / kG;

  const size_t idx_smem = static_cast<size_t>(2 * a.max_blocks + kGatherWinTok * a.k) * 4;
  e = cudaFuncSetAttribute(gather_index_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(idx_smem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gather_attend_kernel<kG>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kGSmem));
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  for (int64_t t0 = 0; t0 < a.num_rows; t0 += seg) {
    w.T0 = static_cast<int32_t>(t0);
    w.T1 = static_cast<int32_t>(std::min<int64_t>(a.num_rows, t0 + seg));
    w.num_win = static_cast<int32_t>((w.T1 - w.T0) / kGatherWinTok + 2 * static_cast<int64_t>(a.num_reqs) + 1);
    gather_index_kernel<<<w.num_win, kIdxThreads, idx_smem, stream>>>(a, w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    gather_attend_kernel<kG><<<static_cast<unsigned>(std::max(sms, 1)), kGThreads, kGSmem, stream>>>(kv_map, q_map,
                                                                                                      a, w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t units = static_cast<int64_t>(w.T1 - w.T0) * a.num_kv_heads;
    gather_merge_kernel<kG><<<static_cast<unsigned>((units + kMergeWarps - 1) / kMergeWarps), kMergeWarps * 32, 0,
                              stream>>>(a, w);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_prefill_gather(const AttendArgs& a, const CUtensorMap& kv_map, const CUtensorMap& q_map,
                                  const CUtensorMap* tile_q_map, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return a.group == 16 ? launch_gather_g<16>(a, kv_map, q_map, tile_q_map, ws, ws_bytes, stream)
                       : launch_gather_g<8>(a, kv_map, q_map, tile_q_map, ws, ws_bytes, stream);
}

}  // namespace pbs
