// Index-cache insert: scatter index keys [N, D] into the key-only side cache [B, T, D]
// (vLLM page vllm.models.minimax_m3.amd.ops.sparse_pa, minimax_m3_insert_index_cache).
//
// A pure HBM copy: one warp per source row, 16-byte vector loads/stores when the row bytes,
// both row starts and the strides allow it, element copies otherwise.
#include "pbs_device.cuh"
#include "pbs_internal.h"

namespace pbs {
namespace {

constexpr int kWarps = 8;

template <bool kVec>
__global__ void __launch_bounds__(kWarps * 32) insert_kernel(InsertArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * kWarps + warp;
  if (n >= a.num_tokens) return;
  const int64_t slot = a.slot_mapping[static_cast<int64_t>(n) * a.slot_stride];
  if (slot < 0) return;  // padding
  const int64_t cap = static_cast<int64_t>(a.num_blocks) * a.block_tokens;
  if (slot >= cap) {
    if (lane == 0) set_err(a.err_word, PBS_DEVERR_SLOT_OOB);
    return;
  }
  const int64_t blk = slot / a.block_tokens, t = slot % a.block_tokens;
  const int eb = a.elem_bytes;
  const uint8_t* src = a.index_k + static_cast<int64_t>(n) * a.k_stride0 * eb;
  uint8_t* dst = a.index_cache + (blk * a.c_stride0 + t * a.c_stride1) * eb;
  if (kVec) {
    const int chunks = a.dim * eb / 16;
    for (int c = lane; c < chunks; c += 32)
      reinterpret_cast<uint4*>(dst)[c] = reinterpret_cast<const uint4*>(src)[c];
  } else {
    for (int d = lane; d < a.dim; d += 32) {
      const uint8_t* s = src + static_cast<int64_t>(d) * a.k_stride1 * eb;
      uint8_t* o = dst + static_cast<int64_t>(d) * eb;
      if (eb == 4) *reinterpret_cast<uint32_t*>(o) = *reinterpret_cast<const uint32_t*>(s);
      else if (eb == 2) *reinterpret_cast<uint16_t*>(o) = *reinterpret_cast<const uint16_t*>(s);
      else *o = *s;
    }
  }
}

}  // namespace

cudaError_t launch_insert_index_cache(const InsertArgs& a, cudaStream_t stream) {
  const int64_t eb = a.elem_bytes;
  const bool vec = a.k_stride1 == 1 && (a.dim * eb) % 16 == 0 && (a.k_stride0 * eb) % 16 == 0 &&
                   (a.c_stride0 * eb) % 16 == 0 && (a.c_stride1 * eb) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(a.index_k) % 16 == 0 &&
                   reinterpret_cast<uintptr_t>(a.index_cache) % 16 == 0;
  const dim3 grid((a.num_tokens + kWarps - 1) / kWarps), block(kWarps * 32);
  if (vec) insert_kernel<true><<<grid, block, 0, stream>>>(a);
  else insert_kernel<false><<<grid, block, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pbs
