// Device-side building blocks shared by the kernels of libpbs: method constants, inline-PTX
// wrappers (mbarrier, bulk/tensor copies, ldmatrix, mma.sync, movmatrix, conversions) and the
// warp-level compaction of one query row's top-k list into its sparse block table.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/pbs.h"

namespace pbs {

// Method constants (vLLM page vllm.models.minimax_m3.amd.ops.sparse_pa, row writer): a logical
// sparse block is 128 tokens, a physical page holds 16 token rows, a block spans 8 pages.
constexpr int kSparseBlock = 128;
constexpr int kPageRows = 16;
constexpr int kPagesPerBlock = kSparseBlock / kPageRows;
constexpr int kMaxTopk = 64;
constexpr int kHeadDim = 128;

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ------------------------------------------------------------------------------------------
// small PTX wrappers
// ------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false after `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// 4-D tiled tensor copy global -> shared, completion counted on an mbarrier.
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Untiled bulk copy global -> shared (both addresses and size multiples of 16 bytes).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pack two floats: `lo` goes to the lower 16 bits (the first element of the pair).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// Two e4m3 bytes (low 16 bits of x) -> f16x2, byte 0 to the lower half. Exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t x) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(r) : "r"(x));
  return r;
}

// One byte of two e2m1 codes (low 8 bits of x) -> f16x2, low nibble to the lower half. Exact.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t x) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b0;\n\t}"
      : "=r"(r)
      : "r"(x));
  return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// bf16x2 -> f16x2 (rounds to nearest; exact for |x| in the f16 normal range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x) { return pack_f16(bf16_lo(x), bf16_hi(x)); }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ void set_err(int32_t* err_word, int32_t bits) {
  if (err_word != nullptr) atomicOr(err_word, bits);
}

// ------------------------------------------------------------------------------------------
// query positions
// ------------------------------------------------------------------------------------------

// Decode row -> (request, absolute position); queries are right-aligned to seq_len
// (vLLM page vllm.models.minimax_m3.nvidia.sparse_attention_flashinfer, forward: default q_offset).
__device__ __forceinline__ void decode_position(int row, int dql, const int32_t* seq_lens, int& req,
                                                int& abs_pos) {
  req = row / dql;
  abs_pos = __ldg(seq_lens + req) - dql + (row - req * dql);
}

// Prefill token -> (request, absolute position): request r holds tokens cu[r] .. cu[r+1]-1,
// preceded by seq_len - q_len context tokens (vLLM page
// vllm.models.minimax_m3.amd.sparse_attention_nvfp4, metadata builder).
__device__ __forceinline__ void prefill_position(int t, const int32_t* cu, int num_reqs, const int32_t* seq_lens,
                                                 int& req, int& abs_pos) {
  // last r with cu[r] <= t (upper bound - 1); empty requests are skipped naturally
  int lo = 0, hi = num_reqs;  // answer in [0, num_reqs)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
  }
  req = lo;
  const int c0 = __ldg(cu + lo), c1 = __ldg(cu + lo + 1);
  abs_pos = __ldg(seq_lens + lo) - (c1 - c0) + (t - c0);
}

// ------------------------------------------------------------------------------------------
// one row of the sparse block table (warp-cooperative)
// ------------------------------------------------------------------------------------------

struct RowCompaction {
  int ctx;        // attended keys
  int n_written;  // slots holding a block: n_full + (own block present)
  bool bad;       // a valid block id was >= max_blocks
};

// Compacts one query row's top-k list (vLLM page vllm.models.minimax_m3.amd.ops.sparse_pa,
// _write_sparse_block_table_row_from_values): a block b is valid iff the causal length
// max(abs_pos+1, 0) is positive and 0 <= b <= abs_pos/128; valid blocks before the own block
// are numbered in top-k order (ballot + popc prefix), the own block takes slot n_full. A row
// is a set of blocks: an entry whose id an earlier entry already holds is dropped (the writer
// files every copy of the own block under one slot and counts its keys once; repeated full
// blocks are read the same way). Slot s's first page id (page_table[b] * block_page_stride)
// goes to slot_base[s] (shared memory, kMaxTopk entries). All 32 lanes must call this; the
// result is warp-uniform.
__device__ __forceinline__ RowCompaction compact_row(const int32_t* __restrict__ topk_row, int k, int abs_pos,
                                                     const int32_t* __restrict__ bt_row, int max_blocks,
                                                     int block_page_stride, int32_t* slot_base) {
  const int lane = threadIdx.x & 31;
  const int causal_len = abs_pos + 1 > 0 ? abs_pos + 1 : 0;
  const int own = causal_len > 0 ? abs_pos / kSparseBlock : -1;
  int b[2];
  bool valid[2], full[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = lane + 32 * h;
    b[h] = e < k ? __ldg(topk_row + e) : -1;
  }
  // entry lane (lane + 32) repeats an earlier one: a lower lane of its half holds the same id,
  // or (second half) any lane of the first half does
  const uint32_t lt = lanemask_lt();
  bool rep[2];
  rep[0] = (__match_any_sync(0xffffffffu, b[0]) & lt) != 0;
  rep[1] = false;
  if (k > 32) {  // warp-uniform
    bool r1 = (__match_any_sync(0xffffffffu, b[1]) & lt) != 0;
    for (int j = 0; j < 32; ++j) r1 |= __shfl_sync(0xffffffffu, b[0], j) == b[1];
    rep[1] = r1;
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int e = lane + 32 * h;
    valid[h] = e < k && !rep[h] && causal_len > 0 && b[h] >= 0 && b[h] <= own;
    full[h] = valid[h] && b[h] < own;
  }
  const uint32_t f0 = __ballot_sync(0xffffffffu, full[0]), f1 = __ballot_sync(0xffffffffu, full[1]);
  const uint32_t v0 = __ballot_sync(0xffffffffu, valid[0]), v1 = __ballot_sync(0xffffffffu, valid[1]);
  const int n_full = __popc(f0) + __popc(f1);
  const int n_valid = __popc(v0) + __popc(v1);
  const bool has_tail = n_valid > n_full;
  bool oob = false;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (!valid[h]) continue;
    const int slot = full[h] ? (h == 0 ? __popc(f0 & lt) : __popc(f0) + __popc(f1 & lt)) : n_full;
    if (b[h] >= max_blocks) {
      oob = true;
      continue;
    }
    slot_base[slot] = __ldg(bt_row + b[h]) * block_page_stride;
  }
  RowCompaction rc;
  rc.bad = __any_sync(0xffffffffu, oob);
  rc.n_written = n_full + (has_tail ? 1 : 0);
  if (has_tail) {
    rc.ctx = n_full * kSparseBlock + (causal_len - own * kSparseBlock);
  } else {
    const int c = n_valid * kSparseBlock;
    rc.ctx = c < causal_len ? c : causal_len;
  }
  if (rc.bad) {
    rc.ctx = 0;
    rc.n_written = 0;
  }
  __syncwarp();
  return rc;
}

}  // namespace pbs
