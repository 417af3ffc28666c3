// Sparse block table build (decode and prefill): one warp per query row.
//
// vLLM page vllm.models.minimax_m3.amd.ops.sparse_pa: _write_sparse_block_table_row_from_values
// and the minimax_m3_build_sparse_block_table_decode / _prefill launchers. Positions: decode rows
// right-aligned (vllm.models.minimax_m3.nvidia.sparse_attention_flashinfer, forward); prefill tokens
// at context + offset (vllm.models.minimax_m3.amd.sparse_attention_nvfp4, metadata builder).
//
// GB300 mapping: the compaction is a ballot + popc prefix over the (<= 64) ids of a row, the
// block bases are staged in shared memory and the row (topk*8 int32) is written as 16-byte
// vector stores, so each warp writes its row in one or two coalesced sweeps.
#include "pbs_device.cuh"
#include "pbs_internal.h"

namespace pbs {

namespace {

constexpr int kRowsPerCta = 8;

template <bool kPrefill, bool kVec>
__global__ void __launch_bounds__(kRowsPerCta * 32) build_table_kernel(TableArgs a) {
  __shared__ int32_t bases[kRowsPerCta][kMaxTopk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerCta + warp;
  if (row >= a.num_rows) return;  // warp-uniform
  int req, abs_pos;
  if (kPrefill) prefill_position(row, a.cu_seqlens_q, a.num_reqs, a.seq_lens, req, abs_pos);
  else decode_position(row, a.decode_query_len, a.seq_lens, req, abs_pos);
  const RowCompaction rc =
      compact_row(a.topk + static_cast<int64_t>(row) * a.topk_row_stride, a.k, abs_pos,
                  a.page_table + static_cast<int64_t>(req) * a.pt_row_stride, a.max_blocks,
                  a.block_page_stride, bases[warp]);
  if (rc.bad && lane == 0) set_err(a.err_word, PBS_DEVERR_BLOCK_OOB);
  int32_t* out = a.sparse_bt + static_cast<int64_t>(row) * a.sbt_row_stride;
  const int width = a.k * kPagesPerBlock;
  if (kVec) {
    // chunk c holds ids 4c..4c+3: slot c/2, pages 4*(c%2)..+3
    for (int c = lane; c < width / 4; c += 32) {
      const int slot = c >> 1;
      int4 v = make_int4(0, 0, 0, 0);
      if (slot < rc.n_written) {
        const int base = bases[warp][slot] + 4 * (c & 1);
        v = make_int4(base, base + 1, base + 2, base + 3);
      }
      reinterpret_cast<int4*>(out)[c] = v;
    }
  } else {
    for (int i = lane; i < width; i += 32) {
      const int slot = i / kPagesPerBlock;
      out[i] = slot < rc.n_written ? bases[warp][slot] + (i % kPagesPerBlock) : 0;
    }
  }
  if (lane == 0) a.sparse_ctx[row] = rc.ctx;
}

}  // namespace

cudaError_t launch_build_table(const TableArgs& a, bool prefill, cudaStream_t stream) {
  const bool vec = (reinterpret_cast<uintptr_t>(a.sparse_bt) % 16 == 0) && (a.sbt_row_stride % 4 == 0);
  const dim3 grid((a.num_rows + kRowsPerCta - 1) / kRowsPerCta), block(kRowsPerCta * 32);
  if (prefill) {
    if (vec) build_table_kernel<true, true><<<grid, block, 0, stream>>>(a);
    else build_table_kernel<true, false><<<grid, block, 0, stream>>>(a);
  } else {
    if (vec) build_table_kernel<false, true><<<grid, block, 0, stream>>>(a);
    else build_table_kernel<false, false><<<grid, block, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace pbs
