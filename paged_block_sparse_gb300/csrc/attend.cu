// Token-centric paged block-sparse attend (decode rows and prefill tokens).
//
// What it computes (vLLM pages vllm.models.minimax_m3.nvidia.sparse_attention_flashinfer, forward,
// and vllm.models.minimax_m3.amd.sparse_attention_nvfp4, forward): for each query row and kv head g,
// out[h] = v_scale * softmax(softmax_scale * k_scale * q_h K^T) V over the keys of the row's
// compacted sparse block table (built in-kernel by compact_row, the rule of
// vllm.models.minimax_m3.amd.ops.sparse_pa, _write_sparse_block_table_row_from_values), for the G
// query heads h of group g.
//
// GB300 design
// ------------
// * One cluster of S CTAs per (row, kv head); CTA s takes a contiguous range of the row's
//   128-key slots. The S partial (max, sum, O) triples are merged through distributed shared
//   memory after a cluster barrier, so no global scratch and no second launch are needed.
// * Per CTA: 1 producer warp issues one page (16 rows x one kv head) per pipeline stage with TMA
//   (cp.async.bulk.tensor, 128-byte swizzle, mbarrier completion); 4 consumer warps take pages
//   round-robin. bf16/fp8 pages come through a 4-D tensor map; NVFP4 slots (K|V of the head,
//   2304 contiguous bytes) through an untiled bulk copy.
// * The contraction is tiny (8 heads x 16 keys x 128 dims per page), so it runs on mma.sync with
//   keys as the M dimension (no padding of the 8 heads): S^T = K Q^T, then P^T is transposed in
//   registers (movmatrix) into the B operand of O^T = V^T P^T. The kernel is HBM-bound; the
//   tensor path only keeps the arithmetic off the critical path.
// * bf16 K/V: bf16 MMAs, P split into bf16 hi + lo parts (keeps the attend within a 2e-3
//   relative RMS of the fp64 result). fp8 / NVFP4 K/V: dequantised exactly to fp16 in
//   registers, fp16 MMAs with fp16 P.
// * Online softmax in the log2 domain, fp32 state; k_scale folds into the softmax scale and
//   v_scale into the output (exact, since logits are linear in K and the output in V).
#include <cooperative_groups.h>

#include "pbs_device.cuh"
#include "pbs_internal.h"

namespace cg = cooperative_groups;

namespace pbs {
namespace {

// 3 consumer warps + 1 producer (128 threads, <= 128 registers) and the merge buffer aliased
// onto the drained stages keep a CTA near 50 KB, so 4 CTAs fit on an SM and a 64-request batch
// (512 row x kv-head CTAs) runs in a single wave.
constexpr int kConsumerWarps = 3;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
// A consumer warp takes kPagesPerIter<FMT> consecutive pages per iteration: one for bf16 (the
// kernel is HBM-bound there), two for fp8 / NVFP4, whose per-page work (dequantisation, two
// dependent MMA chains, a softmax round) is the limit: two pages give each warp two independent
// chains and one softmax round per 32 keys. Page p goes to stage p % kStages<FMT> and to
// consumer warp (p / kPagesPerIter) % kConsumerWarps. With the stage count a multiple of
// kPagesPerIter * kConsumerWarps every stage is always consumed by the same warp, one phase
// after the other, so a parity wait can never be answered by a phase two steps behind (with 6
// stages and 4 single-page warps a warp would skip every other phase of a stage and could pass
// its wait early). fp8 / NVFP4 pages are smaller, so twice the stages keep as many bytes in
// flight.
template <int FMT>
constexpr int kPagesPerIter = FMT == PBS_KV_BF16 ? 1 : 2;
template <int FMT>
constexpr int kStagesF = FMT == PBS_KV_BF16 ? 6 : 12;
// fp8 / NVFP4 softmax: the running reference moves only by more than 2^8 (log2 domain)
constexpr float kLazyRescaleLog2 = 8.0f;
constexpr int kMaxStages = 12;
static_assert(kStagesF<PBS_KV_BF16> % (kPagesPerIter<PBS_KV_BF16> * kConsumerWarps) == 0 &&
                  kStagesF<PBS_KV_FP8_E4M3> % (kPagesPerIter<PBS_KV_FP8_E4M3> * kConsumerWarps) == 0 &&
                  kStagesF<PBS_KV_NVFP4> % (kPagesPerIter<PBS_KV_NVFP4> * kConsumerWarps) == 0,
              "each stage must belong to one consumer warp");
constexpr int kTileHeads = 8;  // the n8 tile of the MMA: up to 8 query heads per kv head

template <int FMT>
struct StageBytes;
template <>
struct StageBytes<PBS_KV_BF16> {  // [4 quarter rows][16 rows][128 B], 128B-swizzled
  static constexpr int v = 8192;
};
template <>
struct StageBytes<PBS_KV_FP8_E4M3> {  // [2 halves][16 rows][128 B], 128B-swizzled
  static constexpr int v = 4096;
};
template <>
struct StageBytes<PBS_KV_NVFP4> {  // K slot (1152 B) then V slot (1152 B), as stored
  static constexpr int v = 2304;
};
constexpr int kNvfp4Slot = 1152;
// Workspace partial of one chunk: O [8 heads][128] then m[8], l[8] (floats).
constexpr int kWsPartial = 8 * 128 + 16;

// Byte offset of the 128-byte line holding page row r (0..15), quarter q of a bf16 row (K lo,
// K hi, V lo, V hi) or half q of an fp8 row (K, V), inside a stage. Unpacked caches arrive as
// one box per quarter ([q][16 rows][128 B]); packed caches (page stride = Hkv * rows * row bytes)
// as one box per (page, head) from a 5-D map ([row half][q][8 rows][128 B]). The 128B swizzle
// XORs the 16-byte chunk index with r % 8 in both.
template <int FMT, bool PACKED>
__device__ __forceinline__ uint32_t line_off(int r, int q) {
  if (!PACKED) return q * 2048 + r * 128;
  if (FMT == PBS_KV_BF16) return (r >> 3) * 4096 + q * 1024 + (r & 7) * 128;
  return (r >> 3) * 2048 + q * 1024 + (r & 7) * 128;
}

struct Merge {
  float o[kConsumerWarps][kTileHeads][kHeadDim];
  float m[kConsumerWarps][kTileHeads];
  float l[kConsumerWarps][kTileHeads];
  float cta_m[kTileHeads];
  float cta_l[kTileHeads];
};

struct Ctl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int32_t slot_base[kMaxTopk];
  int32_t page_id[kMaxTopk * kPagesPerBlock];  // page of the row's 16-key group n (n < ceil(ctx / 16))
  int32_t ctx;
  int32_t abort;
  int32_t last;  // this chunk arrived last for its (row, kv head)
};

// The merge buffer reuses the stage ring once every page has been consumed.
template <int FMT>
constexpr size_t ring_bytes() {
  return size_t(kStagesF<FMT>) * StageBytes<FMT>::v > sizeof(Merge) ? size_t(kStagesF<FMT>) * StageBytes<FMT>::v
                                                               : ((sizeof(Merge) + 1023) / 1024) * 1024;
}
template <int FMT>
constexpr size_t smem_bytes() {
  return 1024 + ring_bytes<FMT>() + sizeof(Ctl);
}

__device__ __forceinline__ void tma_load_5d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1, int c2, int c3,
                                            int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.b16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts128_zero(uint32_t addr) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Zero the V rows [nv, 16) of a stage, so that masked keys cannot inject NaN/Inf from
// uninitialised cache rows into P*V (P is 0 there, but 0 * NaN is NaN).
template <int FMT, bool PACKED>
__device__ __forceinline__ void zero_v_tail(uint32_t st, int nv, int lane) {
  if (FMT == PBS_KV_BF16) {
    // quarters 2 and 3, 8 chunks of 16 B per row each
    for (int i = lane; i < (16 - nv) * 16; i += 32) {
      const int r = nv + (i >> 4), q = 2 + ((i >> 3) & 1), c = i & 7;
      sts128_zero(st + line_off<FMT, PACKED>(r, q) + c * 16);
    }
  } else if (FMT == PBS_KV_FP8_E4M3) {
    for (int i = lane; i < (16 - nv) * 8; i += 32) {
      const int r = nv + (i >> 3), c = i & 7;
      sts128_zero(st + line_off<FMT, PACKED>(r, 1) + c * 16);
    }
  } else {
    // V codes: 4 chunks of 16 B per row; V scales: 8 B per row
    for (int i = lane; i < (16 - nv) * 4; i += 32) {
      const int r = nv + (i >> 2), c = i & 3;
      sts128_zero(st + kNvfp4Slot + r * 64 + c * 16);
    }
    for (int r = nv + lane; r < 16; r += 32) {
      asm volatile("st.shared.v2.b32 [%0], {%1, %1};" ::"r"(st + kNvfp4Slot + 1024 + r * 8), "r"(0) : "memory");
    }
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
}

// S^T = K Q^T for the 16 keys of each of NP page stages (addresses st[0..NP)), the first n_live
// of which hold pages: keys as the MMA's M, the (up to) 8 query heads as its N; lane holds keys
// hh, hh + 8 (hh = lane / 4) of heads 2c, 2c + 1 (c = lane % 4) in s[i][0..3]. The stages' MMA
// chains are interleaved step by step, so each MMA's wait on its accumulator overlaps the other
// chain. qf: the warp's Q fragments (bf16, or converted to f16).
template <int FMT, bool PACKED, int NP>
__device__ __forceinline__ void page_scores(const uint32_t (&st)[NP], int n_live, const uint32_t (&qf)[8][2], int lane,
                                            float (&s)[NP][4]) {
  const int hh = lane >> 2, c = lane & 3;
#pragma unroll
  for (int i = 0; i < NP; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
  if (FMT == PBS_KV_BF16) {
    const int key = (lane & 7) + ((lane >> 3) & 1) * 8;
    const int hi = lane >> 4;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int chunk = 2 * (j & 3) + hi;
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        if (i >= n_live) continue;
        uint32_t af[4];
        ldsm_x4(st[i] + line_off<FMT, PACKED>(key, j >> 2) + ((chunk ^ (key & 7)) << 4), af);
        mma_bf16(s[i], af, qf[j][0], qf[j][1]);
      }
    }
  } else if (FMT == PBS_KV_FP8_E4M3) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        if (i >= n_live) continue;
        const uint32_t w0 = lds32(st[i] + line_off<FMT, PACKED>(hh, 0) + ((j ^ hh) << 4) + 4 * c);
        const uint32_t w1 = lds32(st[i] + line_off<FMT, PACKED>(hh + 8, 0) + ((j ^ hh) << 4) + 4 * c);
        uint32_t af[4] = {e4m3x2_to_f16x2(w0), e4m3x2_to_f16x2(w1), e4m3x2_to_f16x2(w0 >> 16),
                          e4m3x2_to_f16x2(w1 >> 16)};
        mma_f16(s[i], af, qf[j][0], qf[j][1]);
      }
    }
  } else {
    uint4 k0[NP], k1[NP];
    uint32_t s0lo[NP], s0hi[NP], s1lo[NP], s1hi[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      if (i >= n_live) continue;
      k0[i] = lds128(st[i] + hh * 64 + 16 * c);
      k1[i] = lds128(st[i] + (hh + 8) * 64 + 16 * c);
      const uint32_t sc0 = e4m3x2_to_f16x2(lds16(st[i] + 1024 + hh * 8 + 2 * c));
      const uint32_t sc1 = e4m3x2_to_f16x2(lds16(st[i] + 1024 + (hh + 8) * 8 + 2 * c));
      s0lo[i] = prmt(sc0, sc0, 0x1010);
      s0hi[i] = prmt(sc0, sc0, 0x3232);
      s1lo[i] = prmt(sc1, sc1, 0x1010);
      s1hi[i] = prmt(sc1, sc1, 0x3232);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int i = 0; i < NP; ++i) {
        if (i >= n_live) continue;
        const uint32_t w0 = word_of(k0[i], j >> 1) >> (16 * (j & 1));
        const uint32_t w1 = word_of(k1[i], j >> 1) >> (16 * (j & 1));
        const uint32_t sa = j < 4 ? s0lo[i] : s0hi[i], sb = j < 4 ? s1lo[i] : s1hi[i];
        uint32_t af[4] = {hmul2(e2m1x2_to_f16x2(w0), sa), hmul2(e2m1x2_to_f16x2(w1), sb),
                          hmul2(e2m1x2_to_f16x2(w0 >> 8), sa), hmul2(e2m1x2_to_f16x2(w1 >> 8), sb)};
        mma_f16(s[i], af, qf[j][0], qf[j][1]);
      }
    }
  }
}

// O^T += V^T P^T for one page stage, given this lane's probabilities p0..p3 (keys hh, hh + 8 of
// heads 2c, 2c + 1, laid out as page_scores returns them). bf16 V: P split into bf16 hi + lo
// (two MMAs); fp8 / NVFP4 V: dequantised to f16, P in f16.
template <int FMT, bool PACKED>
__device__ __forceinline__ void page_pv(uint32_t st, float p0, float p1, float p2, float p3, int lane,
                                        float (&o)[8][4]) {
  const int hh = lane >> 2, c = lane & 3;
  if (FMT == PBS_KV_BF16) {
    const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
    const uint32_t l01 = pack_bf16(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
    const uint32_t l23 = pack_bf16(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
    const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
    const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);
    const int mi = lane >> 3;
    const int key = (lane & 7) + 8 * (mi >> 1);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int chunk = 2 * (i & 3) + (mi & 1);
      uint32_t vf[4];
      ldsm_x4_trans(st + line_off<FMT, PACKED>(key, 2 + (i >> 2)) + ((chunk ^ (key & 7)) << 4), vf);
      mma_bf16(o[i], vf, bh0, bh1);
      mma_bf16(o[i], vf, bl0, bl1);
    }
  } else {
    const uint32_t b0 = movmatrix_trans(pack_f16(p0, p1)), b1 = movmatrix_trans(pack_f16(p2, p3));
    if (FMT == PBS_KV_FP8_E4M3) {
      const uint4 va = lds128(st + line_off<FMT, PACKED>(2 * c, 1) + ((hh ^ ((2 * c) & 7)) << 4));
      const uint4 vbb = lds128(st + line_off<FMT, PACKED>(2 * c + 1, 1) + ((hh ^ ((2 * c + 1) & 7)) << 4));
      const uint4 vc = lds128(st + line_off<FMT, PACKED>(2 * c + 8, 1) + ((hh ^ ((2 * c + 8) & 7)) << 4));
      const uint4 vd = lds128(st + line_off<FMT, PACKED>(2 * c + 9, 1) + ((hh ^ ((2 * c + 9) & 7)) << 4));
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
        const uint32_t x = prmt(word_of(va, i >> 1), word_of(vbb, i >> 1), sel);
        const uint32_t y = prmt(word_of(vc, i >> 1), word_of(vd, i >> 1), sel);
        uint32_t af[4] = {e4m3x2_to_f16x2(x), e4m3x2_to_f16x2(x >> 16), e4m3x2_to_f16x2(y),
                          e4m3x2_to_f16x2(y >> 16)};
        mma_f16(o[i], af, b0, b1);
      }
    } else {
      const uint32_t vc0 = st + kNvfp4Slot, vs0 = st + kNvfp4Slot + 1024;
      const uint2 wa = lds64(vc0 + (2 * c) * 64 + 8 * hh);
      const uint2 wb = lds64(vc0 + (2 * c + 1) * 64 + 8 * hh);
      const uint2 wc = lds64(vc0 + (2 * c + 8) * 64 + 8 * hh);
      const uint2 wd = lds64(vc0 + (2 * c + 9) * 64 + 8 * hh);
      const uint32_t sab = e4m3x2_to_f16x2(lds8(vs0 + (2 * c) * 8 + hh) | (lds8(vs0 + (2 * c + 1) * 8 + hh) << 8));
      const uint32_t scd = e4m3x2_to_f16x2(lds8(vs0 + (2 * c + 8) * 8 + hh) | (lds8(vs0 + (2 * c + 9) * 8 + hh) << 8));
#pragma unroll
      for (int wh = 0; wh < 2; ++wh) {
        const uint32_t A = wh ? wa.y : wa.x, B = wh ? wb.y : wb.x;
        const uint32_t C = wh ? wc.y : wc.x, D = wh ? wd.y : wd.x;
        const uint32_t lo_ab = (A & 0x0F0F0F0Fu) | ((B & 0x0F0F0F0Fu) << 4);
        const uint32_t hi_ab = ((A >> 4) & 0x0F0F0F0Fu) | (B & 0xF0F0F0F0u);
        const uint32_t lo_cd = (C & 0x0F0F0F0Fu) | ((D & 0x0F0F0F0Fu) << 4);
        const uint32_t hi_cd = ((C >> 4) & 0x0F0F0F0Fu) | (D & 0xF0F0F0F0u);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          const int i = 4 * wh + b;
          uint32_t af[4] = {hmul2(e2m1x2_to_f16x2(lo_ab >> (8 * b)), sab),
                            hmul2(e2m1x2_to_f16x2(hi_ab >> (8 * b)), sab),
                            hmul2(e2m1x2_to_f16x2(lo_cd >> (8 * b)), scd),
                            hmul2(e2m1x2_to_f16x2(hi_cd >> (8 * b)), scd)};
          mma_f16(o[i], af, b0, b1);
        }
      }
    }
  }
}

#ifdef PBS_TRACE
// Trace build only: per CTA {SM id, start, first page landed, end} in global-timer ns.
constexpr int kDTraceCtas = 8192;
__device__ unsigned long long g_dtrace[kDTraceCtas][4];
#define DTRACE(k, v) do { const unsigned _c = blockIdx.y * gridDim.x + blockIdx.x; \
                          if (_c < kDTraceCtas) g_dtrace[_c][(k)] = (v); } while (0)
#else
#define DTRACE(k, v) do { } while (0)
#endif

template <int FMT, int MODE, bool PACKED>
__global__ void __launch_bounds__(kThreads, 4) attend_kernel(const __grid_constant__ CUtensorMap tmap,
                                                             const AttendArgs a) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int kStage = StageBytes<FMT>::v;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_u32 & 1023u)) & 1023u);
  uint8_t* stages = smem;
  Merge* mg = reinterpret_cast<Merge*>(smem);  // valid only after the pipeline has drained
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + ring_bytes<FMT>());

  const int S = a.splits;
  const int split = blockIdx.x % S;
  const int row = blockIdx.x / S;
  // head group gv = kv head g's query heads gv * G .. gv * G + G - 1 (G <= 8 heads per CTA)
  const int gv = blockIdx.y;
  const int g = gv / a.sub_groups;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = a.group / a.sub_groups;

  if (threadIdx.x == 0) {
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    DTRACE(0, smid);
    DTRACE(1, global_timer_ns());
    for (int i = 0; i < kStagesF<FMT>; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->empty[i], 1);
    }
    ctl->abort = 0;
    fence_mbar_init();
  }

  // the row's position, and the page table its request reads
  int req, abs_pos;
  const int32_t* pt = a.page_table;
  int64_t pt_stride = a.pt_row_stride;
  int max_blocks = a.max_blocks;
  if (MODE == kModePrefill) {
    prefill_position(row, a.cu_seqlens_q, a.num_reqs, a.seq_lens, req, abs_pos);
  } else if (MODE == kModeDecode || row < a.num_dec_rows) {
    decode_position(row, a.decode_query_len, a.seq_lens, req, abs_pos);
  } else {
    prefill_position(row - a.num_dec_rows, a.cu_seqlens_q, a.num_reqs, a.pre_seq_lens, req, abs_pos);
    pt = a.pre_page_table;
    pt_stride = a.pre_pt_row_stride;
    max_blocks = a.pre_max_blocks;
  }

  // ---- producer warp: the row's table (compacted here, or a prebuilt one); consumers: Q --------
  uint32_t qf[8][2];
  if (warp == kConsumerWarps) {
    int ctx;
    bool row_bad = false;  // block id past the page table, or an unreadable prebuilt row
    if (a.sparse_bt == nullptr) {
      const RowCompaction rc = compact_row(a.topk + static_cast<int64_t>(row) * a.topk_row_stride, a.k, abs_pos,
                                           pt + static_cast<int64_t>(req) * pt_stride, max_blocks,
                                           a.block_page_stride, ctl->slot_base);
      ctx = rc.ctx;
      row_bad = rc.bad;
      // slot s holds the 8 consecutive pages from slot_base[s]
      for (int n = lane; n < rc.n_written * kPagesPerBlock; n += 32)
        ctl->page_id[n] = ctl->slot_base[n / kPagesPerBlock] + (n % kPagesPerBlock);
    } else {
      // prebuilt: the row's ctx and page ids as the [sparse_pa] builders wrote them
      ctx = __ldg(a.sparse_ctx + row);
      row_bad = ctx < 0 || ctx > a.k * kSparseBlock;
      if (row_bad) ctx = 0;
      const int32_t* trow = a.sparse_bt + static_cast<int64_t>(row) * a.sbt_row_stride;
      for (int n = lane; n < (ctx + kPageRows - 1) / kPageRows; n += 32) ctl->page_id[n] = __ldg(trow + n);
    }
    __syncwarp();
    // every page the row reads must lie in the cache
    bool page_bad = false;
    for (int n = lane; n < (ctx + kPageRows - 1) / kPageRows; n += 32) {
      const int id = ctl->page_id[n];
      page_bad |= id < 0 || id >= a.num_pages;
    }
    page_bad = __any_sync(0xffffffffu, page_bad);
    if (lane == 0) {
      if (row_bad && split == 0 && gv == 0)
        set_err(a.err_word, a.sparse_bt == nullptr ? PBS_DEVERR_BLOCK_OOB : PBS_DEVERR_TABLE);
      if (page_bad && split == 0 && gv == 0) set_err(a.err_word, PBS_DEVERR_PAGE_OOB);
      ctl->ctx = page_bad ? 0 : ctx;
    }
  } else {
    const int hh = lane >> 2, c = lane & 3;
    const bool live = hh < G;
    const uint16_t* qh =
        a.q + static_cast<int64_t>(row) * a.q_row_stride + static_cast<int64_t>(gv * G + (live ? hh : 0)) * a.q_head_stride;
    const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qh);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      int d0, d1;
      if (FMT == PBS_KV_BF16) {
        d0 = 16 * j + 2 * c;
        d1 = d0 + 8;
      } else if (FMT == PBS_KV_FP8_E4M3) {
        d0 = 16 * j + 4 * c;
        d1 = d0 + 2;
      } else {
        d0 = 32 * c + 4 * j;
        d1 = d0 + 2;
      }
      uint32_t w0 = live ? __ldg(q32 + (d0 >> 1)) : 0u;
      uint32_t w1 = live ? __ldg(q32 + (d1 >> 1)) : 0u;
      if (FMT != PBS_KV_BF16) {
        w0 = bf16x2_to_f16x2(w0);
        w1 = bf16x2_to_f16x2(w1);
      }
      qf[j][0] = w0;
      qf[j][1] = w1;
    }
  }
  __syncthreads();

  const int ctx = ctl->ctx;
  const int n_slots = (ctx + kSparseBlock - 1) / kSparseBlock;
  const int per = (n_slots + S - 1) / S;
  const int slot0 = min(split * per, n_slots), slot1 = min(slot0 + per, n_slots);
  const int key0 = slot0 * kSparseBlock;
  const int key1 = min(slot1 * kSparseBlock, ctx);
  const int npages = key1 > key0 ? (key1 - key0 + kPageRows - 1) / kPageRows : 0;

  // a consumer warp's partial (max, sum, O) waits in registers until the ring has drained
  float part_m[2] = {-INFINITY, -INFINITY}, part_l[2] = {0.f, 0.f}, part_o[8][4] = {};
  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      for (int p = 0; p < npages; ++p) {
        const int stage = p % kStagesF<FMT>;
        if (p >= kStagesF<FMT>) {
          if (!mbar_wait_bounded(&ctl->empty[stage], ((p / kStagesF<FMT>) - 1) & 1)) {
            set_err(a.err_word, PBS_DEVERR_TIMEOUT);
            atomicExch(&ctl->abort, 1);
            break;
          }
        }
        if (*reinterpret_cast<volatile int32_t*>(&ctl->abort)) break;
        const int kp = (key0 >> 4) + p;
        const int page = ctl->page_id[kp];
        uint8_t* dst = stages + stage * kStage;
#ifdef PBS_CHECKED
        // checked build: every copy's source and destination are validated before issue
        {
          int bad = 0;
          if (kp >= kMaxTopk * kPagesPerBlock || kp < 0) bad |= 1 << 16;
          if (page < 0 || page >= a.num_pages) bad |= 1 << 17;
          if (g < 0 || g >= a.num_kv_heads) bad |= 1 << 18;
          if ((smem_u32(dst) & 1023u) != 0 || dst + kStage > reinterpret_cast<uint8_t*>(mg)) bad |= 1 << 19;
          if ((reinterpret_cast<uintptr_t>(&tmap) & 63u) != 0) bad |= 1 << 20;
          if (bad) {
            set_err(a.err_word, bad);
            mbar_arrive(&ctl->full[stage]);  // complete the phase without data
            issued = p + 1;
            continue;
          }
        }
#endif
        mbar_arrive_expect_tx(&ctl->full[stage], kStage);
        if (FMT != PBS_KV_NVFP4 && PACKED) {
          // one box per (page, head): coordinate page * Hkv + head on the 5-D map
          tma_load_5d(dst, &tmap, &ctl->full[stage], 0, 0, 0, 0, page * a.num_kv_heads + g);
        } else if (FMT == PBS_KV_BF16) {
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) tma_load_4d(dst + qq * 2048, &tmap, &ctl->full[stage], 64 * qq, 0, g, page);
        } else if (FMT == PBS_KV_FP8_E4M3) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) tma_load_4d(dst + hh * 2048, &tmap, &ctl->full[stage], 128 * hh, 0, g, page);
        } else {
          const uint8_t* src = a.kv_cache + static_cast<int64_t>(page) * a.page_stride_bytes +
                               static_cast<int64_t>(g) * (2 * kNvfp4Slot);
          bulk_load(dst, src, kStage, &ctl->full[stage]);
        }
        issued = p + 1;
      }
      // every copy this CTA issued must land before its shared memory goes away
      for (int p = max(0, issued - kStagesF<FMT>); p < issued; ++p) {
        if (!mbar_wait_bounded(&ctl->full[p % kStagesF<FMT>], (p / kStagesF<FMT>) & 1)) {
          set_err(a.err_word, PBS_DEVERR_TIMEOUT);
          break;
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    constexpr int kPP = kPagesPerIter<FMT>;
    constexpr int kNS = kStagesF<FMT>;
    const int hh = lane >> 2;
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const float sl2 = a.scale_log2;

    for (int p0 = warp * kPP; p0 < npages; p0 += kPP * kConsumerWarps) {
      // the iteration's pages p0 .. p0 + kPP - 1 that exist (a row's last iteration may have fewer)
      const int n_live = kPP == 1 ? 1 : min(kPP, npages - p0);  // p0 < npages: one page at least
      uint32_t st[kPP];
      int nv[kPP];
      bool ok = true;
#pragma unroll
      for (int i = 0; i < kPP; ++i) {
        const int p = p0 + i;
        st[i] = smem_u32(stages + (p % kNS) * kStage);
        nv[i] = 0;
        if (i >= n_live) continue;
        if (!mbar_wait_bounded(&ctl->full[p % kNS], (p / kNS) & 1)) {
          set_err(a.err_word, PBS_DEVERR_TIMEOUT);
          atomicExch(&ctl->abort, 1);
          ok = false;
          break;
        }
        if (p == 0 && lane == 0) DTRACE(2, global_timer_ns());
        nv[i] = min(kPageRows, key1 - (key0 + p * kPageRows));
        if (nv[i] < kPageRows) zero_v_tail<FMT, PACKED>(st[i], nv[i], lane);
      }
      if (!ok) break;
      // ---- S^T = K Q^T (16 keys x 8 heads per page)
      float sc[kPP][4];
      page_scores<FMT, PACKED, kPP>(st, n_live, qf, lane, sc);
      float t[kPP][4];
#pragma unroll
      for (int i = 0; i < kPP; ++i) {
        // keys past the range (or a page that does not exist: nv 0) take no weight
        const bool ok_lo = hh < nv[i], ok_hi = hh + 8 < nv[i];
        t[i][0] = ok_lo ? sc[i][0] * sl2 : -INFINITY;
        t[i][1] = ok_lo ? sc[i][1] * sl2 : -INFINITY;
        t[i][2] = ok_hi ? sc[i][2] * sl2 : -INFINITY;
        t[i][3] = ok_hi ? sc[i][3] * sl2 : -INFINITY;
      }

      // ---- online softmax (log2 domain) over the iteration's keys
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int i = 0; i < kPP; ++i) {
        mx0 = fmaxf(mx0, fmaxf(t[i][0], t[i][2]));
        mx1 = fmaxf(mx1, fmaxf(t[i][1], t[i][3]));
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
      }
      float mu0, mu1, al0, al1;
      if (kPP == 1) {
        // exact running maximum (bf16 P, split into hi + lo, keeps full precision either way)
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        mu0 = mn0 == -INFINITY ? 0.f : mn0;
        mu1 = mn1 == -INFINITY ? 0.f : mn1;
        al0 = ex2(m0 - mu0);
        al1 = ex2(m1 - mu1);
        m0 = mn0;
        m1 = mn1;
      } else {
        // lazy reference (f16 P): m moves, and O and l are rescaled, only when the iteration's
        // maximum passes it by 2^8, so P stays below 2^8 and most iterations skip the rescale
        const bool g0 = mx0 > m0 + kLazyRescaleLog2, g1 = mx1 > m1 + kLazyRescaleLog2;
        al0 = g0 ? ex2(m0 - mx0) : 1.f;
        al1 = g1 ? ex2(m1 - mx1) : 1.f;
        m0 = g0 ? mx0 : m0;
        m1 = g1 ? mx1 : m1;
        mu0 = m0 == -INFINITY ? 0.f : m0;
        mu1 = m1 == -INFINITY ? 0.f : m1;
      }
      float pr[kPP][4];
      float add0 = 0.f, add1 = 0.f;
#pragma unroll
      for (int i = 0; i < kPP; ++i) {
        pr[i][0] = ex2(t[i][0] - mu0);
        pr[i][1] = ex2(t[i][1] - mu1);
        pr[i][2] = ex2(t[i][2] - mu0);
        pr[i][3] = ex2(t[i][3] - mu1);
        add0 += pr[i][0] + pr[i][2];
        add1 += pr[i][1] + pr[i][3];
      }
      l0 = l0 * al0 + add0;
      l1 = l1 * al1 + add1;
      if (kPP == 1 || __any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          o[i][0] *= al0;
          o[i][1] *= al1;
          o[i][2] *= al0;
          o[i][3] *= al1;
        }
      }

      // ---- O^T += V^T P^T, page by page (a page that does not exist holds no V to read)
#pragma unroll
      for (int i = 0; i < kPP; ++i)
        if (i < n_live) page_pv<FMT, PACKED>(st[i], pr[i][0], pr[i][1], pr[i][2], pr[i][3], lane, o);
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kPP; ++i)
          if (i < n_live) mbar_arrive(&ctl->empty[(p0 + i) % kNS]);
      }
    }

    // ---- this warp's row sums; the partials go to shared memory once the ring is drained
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    part_m[0] = m0;
    part_m[1] = m1;
    part_l[0] = l0;
    part_l[1] = l1;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) part_o[i][j] = o[i][j];
  }
  // every warp has finished with the stage ring (and the producer has drained its copies)
  __syncthreads();
  if (warp < kConsumerWarps) {
    const int hh = lane >> 2, c = lane & 3;
    const float m0 = part_m[0], m1 = part_m[1], l0 = part_l[0], l1 = part_l[1];
    const float(&o)[8][4] = part_o;
    float(*ow)[kHeadDim] = mg->o[warp];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      int d0, d1;
      if (FMT == PBS_KV_BF16) {
        d0 = 16 * i + hh;
        d1 = d0 + 8;
      } else {
        d0 = 16 * hh + 2 * i;
        d1 = d0 + 1;
      }
      ow[2 * c][d0] = o[i][0];
      ow[2 * c + 1][d0] = o[i][1];
      ow[2 * c][d1] = o[i][2];
      ow[2 * c + 1][d1] = o[i][3];
    }
    if (hh == 0) {
      mg->m[warp][2 * c] = m0;
      mg->m[warp][2 * c + 1] = m1;
      mg->l[warp][2 * c] = l0;
      mg->l[warp][2 * c + 1] = l1;
    }
  }
  __syncthreads();

  // ---- merge the consumer warps (and write the output when the row has a single split)
  const int E = G * kHeadDim;
  uint16_t* out_row = a.out + static_cast<int64_t>(row) * a.out_row_stride;
  if (threadIdx.x < kConsumerWarps * 32) {
    for (int e = threadIdx.x; e < E; e += kConsumerWarps * 32) {
      const int h = e >> 7, d = e & (kHeadDim - 1);
      float M = mg->m[0][h];
#pragma unroll
      for (int w = 1; w < kConsumerWarps; ++w) M = fmaxf(M, mg->m[w][h]);
      float O = 0.f, L = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float f = ex2(mg->m[w][h] - M);
          O += f * mg->o[w][h][d];
          L += f * mg->l[w][h];
        }
      }
      if (S == 1) {
        const float r = L > 0.f ? a.v_scale * O / L : 0.f;
        out_row[static_cast<int64_t>(gv * G + h) * a.out_head_stride + d] = f32_to_bf16_bits(r);
        if (a.lse != nullptr && d == 0)
          a.lse[static_cast<int64_t>(row) * a.lse_row_stride + gv * G + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
      } else if (a.split_ws != nullptr) {
        const int64_t pi = (static_cast<int64_t>(row) * gridDim.y + gv) * S + split;
        a.split_ws[pi * kWsPartial + h * kHeadDim + d] = O;
        if (d == 0) {
          a.split_ws[pi * kWsPartial + kTileHeads * kHeadDim + h] = M;
          a.split_ws[pi * kWsPartial + kTileHeads * kHeadDim + kTileHeads + h] = L;
        }
      } else {
        mg->o[0][h][d] = O;
        if (d == 0) {
          mg->cta_m[h] = M;
          mg->cta_l[h] = L;
        }
      }
    }
  }
  if (S > 1 && a.split_ws != nullptr) {
    // Split through the workspace: publish this chunk's partial, take a ticket; the last chunk
    // of the (row, kv head) merges all partials and clears the ticket for the next call.
    // No chunk waits for another, so early finishers free their SM slot at once.
    const int64_t unit = static_cast<int64_t>(row) * gridDim.y + gv;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) ctl->last = atomicAdd(a.split_tickets + unit, 1) == S - 1;
    __syncthreads();
    if (ctl->last) {
      __threadfence();
      const float* base = a.split_ws + unit * S * kWsPartial;
      for (int e = threadIdx.x; e < E; e += kThreads) {
        const int h = e >> 7, d = e & (kHeadDim - 1);
        float M = -INFINITY;
        for (int r = 0; r < S; ++r) M = fmaxf(M, __ldcg(base + r * kWsPartial + kTileHeads * kHeadDim + h));
        float O = 0.f, L = 0.f;
        if (M != -INFINITY) {
          for (int r = 0; r < S; ++r) {
            const float f = ex2(__ldcg(base + r * kWsPartial + kTileHeads * kHeadDim + h) - M);
            O += f * __ldcg(base + r * kWsPartial + h * kHeadDim + d);
            L += f * __ldcg(base + r * kWsPartial + kTileHeads * kHeadDim + kTileHeads + h);
          }
        }
        const float res = L > 0.f ? a.v_scale * O / L : 0.f;
        out_row[static_cast<int64_t>(gv * G + h) * a.out_head_stride + d] = f32_to_bf16_bits(res);
        if (a.lse != nullptr && d == 0)
          a.lse[static_cast<int64_t>(row) * a.lse_row_stride + gv * G + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
      }
      if (threadIdx.x == 0) a.split_tickets[unit] = 0;
    }
  } else if (S > 1) {
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int rank = static_cast<int>(cluster.block_rank());
    const int e0 = (E * rank) / S, e1 = (E * (rank + 1)) / S;
    for (int e = e0 + threadIdx.x; e < e1; e += kThreads) {
      const int h = e >> 7, d = e & (kHeadDim - 1);
      float M = -INFINITY;
      for (int r = 0; r < S; ++r) M = fmaxf(M, cluster.map_shared_rank(mg, r)->cta_m[h]);
      float O = 0.f, L = 0.f;
      if (M != -INFINITY) {
        for (int r = 0; r < S; ++r) {
          const Merge* rm = cluster.map_shared_rank(mg, r);
          const float f = ex2(rm->cta_m[h] - M);
          O += f * rm->o[0][h][d];
          L += f * rm->cta_l[h];
        }
      }
      const float res = L > 0.f ? a.v_scale * O / L : 0.f;
      out_row[static_cast<int64_t>(gv * G + h) * a.out_head_stride + d] = f32_to_bf16_bits(res);
      if (a.lse != nullptr && d == 0)
        a.lse[static_cast<int64_t>(row) * a.lse_row_stride + gv * G + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
    cluster.sync();  // peers may still be reading this CTA's partial
  }
  if (threadIdx.x == 0) DTRACE(3, global_timer_ns());
}

template <int FMT, int MODE, bool PACKED>
cudaError_t launch_one(const AttendArgs& a, const CUtensorMap& tmap, cudaStream_t stream) {
  constexpr size_t smem = smem_bytes<FMT>();
  auto kern = attend_kernel<FMT, MODE, PACKED>;
  // dynamic shared memory above 48 KB must be opted into (per device; cheap to repeat)
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.num_rows) * static_cast<unsigned>(a.splits),
                     static_cast<unsigned>(a.num_kv_heads * a.sub_groups), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = a.split_ws != nullptr ? 1u : static_cast<unsigned>(a.splits);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmap, a);
}

}  // namespace

#ifdef PBS_TRACE
}  // namespace pbs
// Trace build only: copy the per-CTA decode timeline out (host buffer of n x 4 uint64).
extern "C" __attribute__((visibility("default"))) int pbs_debug_dtrace_get(unsigned long long* host, int n) {
  if (n > pbs::kDTraceCtas) n = pbs::kDTraceCtas;
  return cudaMemcpyFromSymbol(host, pbs::g_dtrace, sizeof(unsigned long long) * 4 * n) == cudaSuccess ? 0 : 5;
}
namespace pbs {
#endif

template <int FMT, bool PACKED>
cudaError_t launch_mode(const AttendArgs& a, int mode, const CUtensorMap& tmap, cudaStream_t stream) {
  switch (mode) {
    case kModeDecode: return launch_one<FMT, kModeDecode, PACKED>(a, tmap, stream);
    case kModePrefill: return launch_one<FMT, kModePrefill, PACKED>(a, tmap, stream);
    case kModeMixed: return launch_one<FMT, kModeMixed, PACKED>(a, tmap, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attend(const AttendArgs& a, int mode, const CUtensorMap& tmap, cudaStream_t stream) {
  const bool packed = a.packed_map != 0;
  switch (a.kv_dtype) {
    case PBS_KV_BF16:
      return packed ? launch_mode<PBS_KV_BF16, true>(a, mode, tmap, stream)
                    : launch_mode<PBS_KV_BF16, false>(a, mode, tmap, stream);
    case PBS_KV_FP8_E4M3:
      return packed ? launch_mode<PBS_KV_FP8_E4M3, true>(a, mode, tmap, stream)
                    : launch_mode<PBS_KV_FP8_E4M3, false>(a, mode, tmap, stream);
    case PBS_KV_NVFP4:
      return launch_mode<PBS_KV_NVFP4, false>(a, mode, tmap, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace pbs
