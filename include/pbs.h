/*
 * pbs.h — C ABI of the paged block-sparse attend (MiniMax-M3 style) for GB300 (sm_103a).
 *
 * The library computes, for every query token, attention over only the keys of
 * the 128-token blocks its top-k list selects, read from a paged KV cache:
 *
 *   1. query position  (decode rows right-aligned to seq_len; prefill tokens
 *      at context_len + offset in their request),
 *   2. sparse block table build: causal filter, compaction, page-16 ids and
 *      the attended context length,
 *   3. gather + dequantise of the selected K/V rows (bf16, fp8-e4m3, NVFP4),
 *   4. softmax(scale * q K^T) V per query head with GQA sharing,
 *   5. index-cache insert (a side path that scatters index keys).
 *
 * Sources (vLLM API pages):
 *   [flashinfer] vllm.models.minimax_m3.nvidia.sparse_attention_flashinfer,
 *                MiniMaxM3SparseFlashInferImpl.forward
 *   [nvfp4]      vllm.models.minimax_m3.amd.sparse_attention_nvfp4,
 *                customize_spec / MiniMaxM3SparseRocmNvfp4Impl.forward / metadata builder
 *   [sparse_pa]  vllm.models.minimax_m3.amd.ops.sparse_pa,
 *                _write_sparse_block_table_row_from_values,
 *                minimax_m3_build_sparse_block_table_decode / _prefill,
 *                minimax_m3_insert_index_cache, minimax_m3_sparse_block_page_stride
 *
 * Conventions for every entry point
 * ---------------------------------
 * - All pointers are DEVICE pointers owned by the caller, unless stated otherwise.
 *   The library allocates no memory and keeps no state between calls (an optional caller-owned
 *   workspace carries split partials within a call), except the fixed device scratch of
 *   pbs_sparse_decode_attention_noalloc, whose tickets are zero between calls.
 * - Work is enqueued on `stream` (NULL = legacy default stream) and is
 *   asynchronous; the return value only reports what the host could check
 *   plus launch errors. Faults found by the kernels themselves are OR-ed into
 *   `*err_word` (device int32, may be NULL) as PBS_DEVERR_* bits; the caller
 *   zeroes it and reads it back when it wants to know.
 * - Strides are in ELEMENTS of the pointed-to type except where the name ends
 *   in `_bytes`.
 * - Empty work (zero rows) returns PBS_OK without launching anything, as the
 *   index-cache insert on [sparse_pa] returns early on empty tensors.
 * - Constants fixed by the method: SPARSE_BLOCK_SIZE = 128 tokens per logical
 *   block, 16 token rows per physical page, PAGES_PER_BLOCK = 8 pages per block.
 *   A page-table entry is a physical BLOCK id b; its pages are
 *   b * block_page_stride + j, j = 0..7 ([sparse_pa] row writer;
 *   block_page_stride is 8 when K and V of a block share its pages, 16 when a
 *   block holds separate K and V sides, [sparse_pa] minimax_m3_sparse_block_page_stride).
 */
#ifndef PBS_H
#define PBS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PBS_API __attribute__((visibility("default")))
#else
#define PBS_API
#endif

/* Same object as cudaStream_t; kept opaque so this header needs no CUDA headers. */
typedef struct CUstream_st* pbs_stream_t;

/* ---- status codes (return values) ------------------------------------------------------ */
#define PBS_OK              0
#define PBS_ERR_ARG         1   /* null pointer where data is needed, bad enum, negative size */
#define PBS_ERR_SHAPE       2   /* inconsistent sizes/strides ([sparse_pa] asserts and ValueErrors) */
#define PBS_ERR_UNSUPPORTED 3   /* valid but not implemented here (head_dim != 128, GQA ratio, top-k > 64) */
#define PBS_ERR_ALIGN       4   /* a pointer or stride breaks the 16-byte alignment the copy engine needs */
#define PBS_ERR_CUDA        5   /* a CUDA runtime/driver call or a launch failed */
#define PBS_ERR_SCRATCH     6   /* pbs_sparse_decode_attention_noalloc: request beyond its fixed scratch */

/* ---- device error bits (OR-ed into *err_word by the kernels) ----------------------------- */
#define PBS_DEVERR_BLOCK_OOB  1  /* a selected, causally valid block id >= max_blocks (row written as empty) */
#define PBS_DEVERR_PAGE_OOB   2  /* a physical page id >= num_pages (row attends nothing) */
#define PBS_DEVERR_SLOT_OOB   4  /* an index-cache slot >= num_blocks * block_tokens (row skipped) */
#define PBS_DEVERR_TIMEOUT    8  /* a bounded wait on a copy gave up (output of that row is undefined) */
#define PBS_DEVERR_TABLE     16  /* a prebuilt table row the kernel cannot read: ctx outside
                                    [0, topk_k * 128], or (prefill tile kernel) a slot whose page ids
                                    are not page_table[r][b] * block_page_stride + j of a block b of
                                    the row's request (the row attends nothing) */

/* ---- KV cache formats -------------------------------------------------------------------- */
#define PBS_KV_BF16      0  /* page = [Hkv][16 rows][K(head_dim) | V(head_dim)] bf16 ([flashinfer]: K|V
                               interleaved per row, head-major LBHNC; K = [..., :D], V = [..., D:]) */
#define PBS_KV_FP8_E4M3  1  /* same layout, one e4m3 byte per element ([flashinfer] fp8 view) */
#define PBS_KV_NVFP4     2  /* page = [2*Hkv slots][1152 B]; slot 2g = K of kv head g, 2g+1 = V
                               ([nvfp4] customize_spec: two slots per head of packed data + block
                               scales). A slot is 16 rows x 64 B of e2m1 codes (element 2i in the
                               low nibble of byte i) then 16 rows x 8 B of e4m3 scales (scale j
                               covers elements 16j..16j+15). head_dim must be 128. */

/* ---- attend options ---------------------------------------------------------------------- */
/* Prefill kernels (pbs_attend_options.prefill_kernel and the return value of
 * pbs_prefill_kernel_choice). */
#define PBS_PREFILL_AUTO    0  /* the library's rule (see pbs_prefill_kernel_choice) */
#define PBS_PREFILL_TOKEN   1  /* token-centric kernel: any shape, mma.sync, one row per CTA group */
#define PBS_PREFILL_TILE    2  /* tcgen05 tile kernel: GQA 8 or 16, top-k <= 16, page table <= 65535
                                  blocks, 16-byte aligned q / out rows; a packed bf16 cache, or an
                                  fp8 / NVFP4 cache with its workspace (pbs_prefill_tile_workspace_bytes) */
#define PBS_PREFILL_GATHER  3  /* tcgen05 gathered-row kernel: GQA 8 or 16, top-k <= 64, page table
                                  <= 8192 blocks, a packed bf16 cache or an fp8 / NVFP4 cache, 16-byte
                                  aligned q / out rows; needs its workspace
                                  (pbs_prefill_workspace_bytes); no prebuilt table */

/*
 * Optional tuning of one attend call (a NULL pointer or an all-zero struct = the library's own
 * choices). No counterpart on the pages; there are no global switches: every choice the caller
 * can override is an argument of the call.
 *   prefill_kernel  PBS_PREFILL_*: run this prefill kernel; PBS_ERR_UNSUPPORTED when it cannot
 *                   take the call. Decode calls ignore it.
 *   splits          0, or 1 / 2 / 4 / 8: CTAs per (row, head group) of the decode and token-centric
 *                   prefill kernel (the library otherwise splits rows only while they cannot fill
 *                   the GPU); any other value is PBS_ERR_ARG.
 *   cache_map       0, or 1: read a packed bf16 / fp8 cache through the per-row-quarter tensor map
 *                   instead of the one-box-per-page map (token-centric kernel; testing).
 *   reserved        must be 0.
 */
typedef struct pbs_attend_options {
  int32_t prefill_kernel;
  int32_t splits;
  int32_t cache_map;
  int32_t reserved;
} pbs_attend_options;

/* Text for a status code (static storage; never NULL). */
PBS_API const char* pbs_status_string(int status);

/* ABI version, bumped on any incompatible change. */
PBS_API int pbs_abi_version(void);

/*
 * Bytes of the optional workspace of pbs_sparse_decode_attention / pbs_sparse_prefill_attention
 * for `num_rows` query rows (decode rows or prefill tokens), `num_heads` query heads and
 * `num_kv_heads` kv heads (0 for an invalid combination).
 * No counterpart on the pages: with a workspace, a row x kv-head split into chunks merges
 * through it (the last chunk to finish merges the others' partials) instead of through a
 * thread-block cluster, with no co-scheduling needed between the chunks. The caller
 * owns it (16-byte aligned) and zeroes it once before first use. Partials are written from its
 * front, one int32 arrival ticket per (row, kv head) sits in its last bytes; every completed call
 * leaves its tickets zero again, so the buffer serves any later call that fits it without
 * re-zeroing (after a PBS_DEVERR_TIMEOUT, zero it again). Calls that share one workspace must
 * not run concurrently.
 */
PBS_API size_t pbs_attend_workspace_bytes(int64_t num_rows, int32_t num_heads, int32_t num_kv_heads);

/*
 * Sparse block table, decode ([sparse_pa] minimax_m3_build_sparse_block_table_decode and
 * _write_sparse_block_table_row_from_values; positions right-aligned per [flashinfer] forward).
 *
 *   topk        [num_rows, topk_k] int32 logical block ids, -1 padded; row r at topk + r*topk_row_stride
 *   page_table  [batch, max_blocks] int32 physical block ids, row stride pt_row_stride
 *   seq_lens    [batch] int32
 *   num_rows    must equal batch * decode_query_len (PBS_ERR_SHAPE otherwise, as the page asserts);
 *               row r belongs to request r / decode_query_len at
 *               abs_pos = seq_lens[b] - decode_query_len + r % decode_query_len
 *   sparse_bt   out [num_rows, topk_k * 8] int32 page-16 ids, row stride sbt_row_stride >= topk_k*8
 *   sparse_ctx  out [num_rows] int32 attended keys per row
 * Per row: a block b is valid iff abs_pos >= 0 and 0 <= b <= abs_pos / 128. Valid blocks
 * below the own block are packed in top-k order, then the own block; each takes 8 ids
 * page_table[b]*block_page_stride + j; the rest of the row is 0. ctx = 128*n_full +
 * (abs_pos + 1 - 128*own) with the own block present, else min(128*n_valid, abs_pos + 1).
 * 1 <= topk_k <= 64.
 */
PBS_API int pbs_build_sparse_block_table_decode(
    const int32_t* topk, int64_t topk_row_stride, int32_t num_rows, int32_t topk_k,
    const int32_t* page_table, int64_t pt_row_stride, int32_t max_blocks,
    const int32_t* seq_lens, int32_t batch, int32_t decode_query_len, int32_t block_page_stride,
    int32_t* sparse_bt, int64_t sbt_row_stride, int32_t* sparse_ctx,
    int32_t* err_word, pbs_stream_t stream);

/*
 * Sparse block table, prefill ([sparse_pa] minimax_m3_build_sparse_block_table_prefill; the
 * per-token request id and position of [nvfp4]'s metadata builder are derived here).
 *
 *   cu_seqlens_q [num_reqs + 1] int32, non-decreasing, cu_seqlens_q[0] = 0, cu_seqlens_q[num_reqs] = total_q
 *   seq_lens     [num_reqs] int32 (context + query tokens)
 * Token t of request r (cu_seqlens_q[r] <= t < cu_seqlens_q[r+1]) sits at
 * abs_pos = seq_lens[r] - (cu_seqlens_q[r+1] - cu_seqlens_q[r]) + (t - cu_seqlens_q[r]).
 * Other arguments and the row rule as for the decode table.
 */
PBS_API int pbs_build_sparse_block_table_prefill(
    const int32_t* topk, int64_t topk_row_stride, int32_t total_q, int32_t topk_k,
    const int32_t* page_table, int64_t pt_row_stride, int32_t max_blocks,
    const int32_t* cu_seqlens_q, const int32_t* seq_lens, int32_t num_reqs, int32_t block_page_stride,
    int32_t* sparse_bt, int64_t sbt_row_stride, int32_t* sparse_ctx,
    int32_t* err_word, pbs_stream_t stream);

/*
 * Sparse decode attention ([flashinfer] msa_sparse_decode_attention call in forward;
 * [nvfp4] minimax_m3_nvfp4_sparse_decode_fly call). Builds each row's table itself
 * (same rule as pbs_build_sparse_block_table_decode) and attends over it, or attends a
 * prebuilt table.
 *
 *   q           [num_rows, num_heads, head_dim] bf16; element (r, h, d) at
 *               q + r*q_row_stride + h*q_head_stride + d
 *   kv_cache    base of page 0 in the format `kv_dtype`; page p starts at
 *               kv_cache + p*page_stride_bytes (16-byte aligned, as is the base)
 *   num_pages   pages addressable from kv_cache (page ids >= num_pages set PBS_DEVERR_PAGE_OOB)
 *   num_heads / num_kv_heads: GQA ratio G = num_heads / num_kv_heads; query head h reads kv head h / G.
 *               Supported: head_dim 128, G in {1, 2, 4, 8, 16}.
 *   softmax_scale, k_scale, v_scale: fp32. The stored K is multiplied by k_scale and V by v_scale
 *               (for NVFP4 these are the per-tensor global scales). As on [flashinfer] forward the
 *               kernel folds k_scale into the softmax scale and v_scale into the output.
 *   out         [num_rows, num_heads, head_dim] bf16, strides out_row_stride / out_head_stride.
 *               A row that attends no key gets zeros.
 *   lse         optional (NULL: not written) [num_rows, num_heads] fp32, row stride lse_row_stride
 *               (>= num_heads, else PBS_ERR_SHAPE), head stride 1: the natural-log log-sum-exp of
 *               each head's scaled logits, ln sum_n exp(softmax_scale * k_scale * q_h . k_n), over
 *               the row's attended keys; -inf for a row with none. Not on the pages: it lets a
 *               caller merge this attend with another over disjoint keys.
 *   sparse_bt, sbt_row_stride, sparse_ctx: optional prebuilt table (both NULL: the kernel
 *               compacts each row from topk and page_table itself). Given, row r attends keys
 *               n < sparse_ctx[r] at page sparse_bt[r * sbt_row_stride + n / 16], row n % 16,
 *               exactly as [sparse_pa] tables are read; topk is then not read (it may be NULL)
 *               and page_table only by the prefill tile kernel. This is the table
 *               pbs_build_sparse_block_table_decode / _prefill write, which the pages build once
 *               per step and share across sparse layers ([sparse_pa]
 *               minimax_m3_rebase_block_table_to_page16: every sparse layer resolves its
 *               selection through the same table). sbt_row_stride >= topk_k * 8 and both
 *               pointers 4-byte aligned, else PBS_ERR_SHAPE / PBS_ERR_ALIGN; one of the two
 *               NULL -> PBS_ERR_ARG. A ctx outside [0, topk_k * 128] sets PBS_DEVERR_TABLE and a
 *               page id >= num_pages PBS_DEVERR_PAGE_OOB; such a row attends nothing.
 *   workspace   optional (NULL, 0): see pbs_attend_workspace_bytes; too small -> PBS_ERR_SHAPE.
 *   options     optional (NULL): see pbs_attend_options.
 */
PBS_API int pbs_sparse_decode_attention(
    const void* q, int64_t q_row_stride, int64_t q_head_stride,
    const void* kv_cache, int64_t page_stride_bytes, int64_t num_pages, int32_t kv_dtype,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    const int32_t* topk, int64_t topk_row_stride, int32_t topk_k,
    const int32_t* page_table, int64_t pt_row_stride, int32_t max_blocks,
    const int32_t* seq_lens, int32_t batch, int32_t decode_query_len, int32_t block_page_stride,
    const int32_t* sparse_bt, int64_t sbt_row_stride, const int32_t* sparse_ctx,
    float softmax_scale, float k_scale, float v_scale,
    void* out, int64_t out_row_stride, int64_t out_head_stride,
    float* lse, int64_t lse_row_stride,
    void* workspace, size_t workspace_bytes,
    const pbs_attend_options* options,
    int32_t* err_word, pbs_stream_t stream);

/*
 * Sparse decode attention without caller memory: pbs_sparse_decode_attention with the split
 * partials and arrival tickets in a fixed 4 MiB device array inside this library instead of a
 * workspace. No counterpart on the pages; it exists for callers that may not allocate device
 * memory once serving has started (a fixed memory plan, or an allocator owned by another
 * framework) and still want split rows merged without a thread-block cluster. The call itself
 * never allocates (no cudaMalloc, no allocating library routine).
 *
 * Limits: when the call splits rows (it does so only while the chunks fit one wave of CTAs),
 * rows x head groups must be <= 4096 and rows x head groups x splits <= 1004 (a head group is a
 * kv head's query heads, or 8 of them when it serves 16), else PBS_ERR_SCRATCH
 * and nothing is launched. Unsplit calls have no limit.
 * Setup: the first call on each device looks up the array's device address with the device
 * current (a CUDA runtime call that may load the library's device module); make that first
 * call before any stream capture begins. A failed lookup returns PBS_ERR_CUDA. The address is
 * kept with the device's current context and looked up again when that context changes (after
 * a device reset, for instance, which also reloads the array, zeroed).
 * State: the tickets start at zero (static device memory is zero at module load) and every
 * completed call leaves them zero. All calls on one device share the array: calls whose
 * kernels could run at the same time (other streams, unordered host threads) race on it and
 * must be serialised by the caller, e.g. by issuing them on one stream.
 * options: optional (NULL); its `splits` forces the split count as for the other entries (the
 * limits above still apply), the other fields are ignored.
 * Arguments, layouts and error behaviour otherwise as in pbs_sparse_decode_attention.
 */
PBS_API int pbs_sparse_decode_attention_noalloc(
    const void* q, int64_t q_row_stride, int64_t q_head_stride,
    const void* kv_cache, int64_t page_stride_bytes, int64_t num_pages, int32_t kv_dtype,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    const int32_t* topk, int64_t topk_row_stride, int32_t topk_k,
    const int32_t* page_table, int64_t pt_row_stride, int32_t max_blocks,
    const int32_t* seq_lens, int32_t batch, int32_t decode_query_len, int32_t block_page_stride,
    float softmax_scale, float k_scale, float v_scale,
    void* out, int64_t out_row_stride, int64_t out_head_stride,
    const pbs_attend_options* options,
    int32_t* err_word, pbs_stream_t stream);

/*
 * Sparse prefill attention, varlen ([flashinfer] msa_sparse_attention call with cu_seqlens_q;
 * [nvfp4] minimax_m3_nvfp4_sparse_prefill call). Token positions as in
 * pbs_build_sparse_block_table_prefill; everything else as in pbs_sparse_decode_attention
 * (including the optional prebuilt table: the token-centric kernel reads its page ids as they
 * are; the tile kernel, which streams whole 128-key blocks shared by a tile's tokens, maps each
 * slot back to the block of the request's page table whose 8 pages it lists, so a slot must
 * hold page_table[r][b] * block_page_stride + j, j < 8, as the builders write it), except the
 * workspace:
 *   workspace   optional (NULL, 0), caller-owned device memory, contents need no initial value.
 *               With a 256-byte aligned workspace of at least
 *               pbs_prefill_workspace_bytes(512, num_reqs, num_heads, num_kv_heads, topk_k,
 *               max_blocks) bytes, calls the gathered-row kernel takes (see PBS_PREFILL_GATHER and
 *               pbs_prefill_kernel_choice) run on it: the converted K / V images, per-block partial
 *               outputs and the per-window token buckets live in the workspace, and the call is
 *               processed in as many token segments as its size requires
 *               (pbs_prefill_workspace_bytes(total_q, ...) bytes: one segment).
 *               Otherwise the tcgen05 tile kernel or the token-centric kernel runs. The tile
 *               kernel, given a 256-byte aligned workspace of at least
 *               pbs_prefill_tile_workspace_bytes(num_reqs, num_kv_heads, max_blocks, kv_dtype)
 *               bytes, first converts the V of every (request, block, kv head) the call can read
 *               to fp16 there (V * 2^-e per block, exact), and for fp8 / NVFP4 caches K to bf16,
 *               and then applies P in fp16, one MMA per 16 keys; without it (bf16 caches only) it
 *               applies bf16 P as hi + lo parts (two MMAs, same accuracy). The
 *               token-centric kernel merges split rows through the workspace when it holds
 *               pbs_attend_workspace_bytes (its tickets are cleared by the call, so here the
 *               workspace needs no zeroing) and ignores a smaller one. Calls that share one
 *               workspace must not run concurrently.
 */
PBS_API int pbs_sparse_prefill_attention(
    const void* q, int64_t q_row_stride, int64_t q_head_stride,
    const void* kv_cache, int64_t page_stride_bytes, int64_t num_pages, int32_t kv_dtype,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    const int32_t* topk, int64_t topk_row_stride, int32_t topk_k,
    const int32_t* page_table, int64_t pt_row_stride, int32_t max_blocks,
    const int32_t* cu_seqlens_q, const int32_t* seq_lens, int32_t num_reqs, int32_t total_q,
    int32_t block_page_stride,
    const int32_t* sparse_bt, int64_t sbt_row_stride, const int32_t* sparse_ctx,
    float softmax_scale, float k_scale, float v_scale,
    void* out, int64_t out_row_stride, int64_t out_head_stride,
    float* lse, int64_t lse_row_stride,
    void* workspace, size_t workspace_bytes,
    const pbs_attend_options* options,
    int32_t* err_word, pbs_stream_t stream);

/*
 * Which prefill kernel pbs_sparse_prefill_attention runs for a call of this shape: returns
 * PBS_PREFILL_TOKEN, _TILE or _GATHER, or minus a PBS_ERR_* status (-PBS_ERR_UNSUPPORTED when
 * options ask for a kernel that cannot take the call, -PBS_ERR_ARG for bad arguments). No
 * counterpart on the pages; a caller uses it to size the workspace the chosen kernel wants.
 * The rule: options->prefill_kernel when set; else the tile kernel while it can take the call
 * (PBS_PREFILL_TILE above) and, for a bf16 cache, the page table is at most 8 x topk_k blocks wide
 * (a tile streams the union of its tokens' selections, which grows with the context they choose
 * from); else the token-centric kernel. fp8 / NVFP4 calls with the tile kernel's workspace take
 * it at any width (the token-centric kernel dequantises every gathered row per token). The answer assumes 16-byte aligned q and out rows; a call whose rows are
 * not takes the token-centric kernel (or PBS_ERR_UNSUPPORTED when a tcgen05 kernel was asked for).
 *   with_table       non-zero: the call passes a prebuilt table
 *   workspace_bytes  the workspace the call will pass (0 for none), 256-byte aligned
 */
PBS_API int pbs_prefill_kernel_choice(int32_t total_q, int32_t num_reqs, int32_t kv_dtype, int64_t page_stride_bytes,
                                      int32_t num_heads, int32_t num_kv_heads, int32_t topk_k, int32_t max_blocks,
                                      int32_t with_table, size_t workspace_bytes,
                                      const pbs_attend_options* options);

/*
 * Bytes of the workspace with which pbs_sparse_prefill_attention runs a call of `total_q`
 * tokens (at most 2^19 per segment) over `num_reqs` requests on its gathered-row kernel in one
 * segment; 0 for invalid arguments. No counterpart on the pages. With total_q = 512 (one window
 * of the kernel's token buckets) it is the smallest workspace that kernel accepts. For Hq query
 * heads and top-k k the size is about total_q * Hq * k * 264 bytes (fp16 partial outputs and
 * their log-sum-exp pairs), plus the buckets and 64 KiB per (request, block, kv head) of K and
 * V images (as pbs_prefill_tile_workspace_bytes for an fp8 cache).
 */
PBS_API size_t pbs_prefill_workspace_bytes(int32_t total_q, int32_t num_reqs, int32_t num_heads,
                                           int32_t num_kv_heads, int32_t topk_k, int32_t max_blocks);

/*
 * Bytes of the workspace with which pbs_sparse_prefill_attention's tcgen05 tile kernel runs on a
 * cache of format kv_dtype: num_reqs * max_blocks * num_kv_heads converted V blocks of 32 KiB
 * (fp16), one int32 exponent each (rounded up to 256 bytes), and for fp8 / NVFP4 as many converted
 * K blocks of 32 KiB (bf16, exact). With it a bf16 call applies P in fp16 (one MMA per 16 keys);
 * an fp8 / NVFP4 call needs it to run on the tile kernel at all. 0 for invalid arguments,
 * num_reqs > 65535 or max_blocks > 65535. No counterpart on the pages.
 */
PBS_API size_t pbs_prefill_tile_workspace_bytes(int32_t num_reqs, int32_t num_kv_heads, int32_t max_blocks,
                                                int32_t kv_dtype);

/*
 * Mixed batch in one call ([flashinfer] forward with both parts: decode rows q[:nd], prefill
 * tokens q[nd:], one token-major top-k buffer for all of them). Rows [0, nd), nd = batch *
 * decode_query_len, are decode rows read with dec_page_table / dec_seq_lens / decode_query_len
 * as in pbs_sparse_decode_attention; rows [nd, nd + total_q) are prefill tokens read with
 * pre_page_table / cu_seqlens_q / pre_seq_lens as in pbs_sparse_prefill_attention. q, topk,
 * out, lse and the optional prebuilt table (sparse_bt / sparse_ctx rows, as in the two calls)
 * are indexed by that row over both parts. Where the prefill part takes a tcgen05 kernel this
 * issues the two calls on `stream`, decode first (what the page's forward does), and passes the
 * optional workspace (NULL, 0) to the prefill call exactly as pbs_sparse_prefill_attention takes
 * it (the tile kernel's images; fp8 / NVFP4 prefill parts need it to run on the tile kernel);
 * otherwise it is one launch of the token-centric kernel, whose CTAs take their part by row, so
 * the decode rows run beside the prefill tokens, and the workspace is not used. The kernel choice
 * for the prefill part is pbs_prefill_kernel_choice's for its shape and this workspace. Errors as
 * in the two calls; with no rows in one part it is that part's call.
 */
PBS_API int pbs_sparse_mixed_attention(
    const void* q, int64_t q_row_stride, int64_t q_head_stride,
    const void* kv_cache, int64_t page_stride_bytes, int64_t num_pages, int32_t kv_dtype,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    const int32_t* topk, int64_t topk_row_stride, int32_t topk_k,
    const int32_t* dec_page_table, int64_t dec_pt_row_stride, int32_t dec_max_blocks,
    const int32_t* dec_seq_lens, int32_t batch, int32_t decode_query_len,
    const int32_t* pre_page_table, int64_t pre_pt_row_stride, int32_t pre_max_blocks,
    const int32_t* cu_seqlens_q, const int32_t* pre_seq_lens, int32_t num_reqs, int32_t total_q,
    int32_t block_page_stride,
    const int32_t* sparse_bt, int64_t sbt_row_stride, const int32_t* sparse_ctx,
    float softmax_scale, float k_scale, float v_scale,
    void* out, int64_t out_row_stride, int64_t out_head_stride,
    float* lse, int64_t lse_row_stride,
    void* workspace, size_t workspace_bytes,
    const pbs_attend_options* options,
    int32_t* err_word, pbs_stream_t stream);

/*
 * Index-cache insert ([sparse_pa] minimax_m3_insert_index_cache): for n < num_tokens,
 * index_cache[slot / block_tokens, slot % block_tokens, :] = index_k[n, :] with
 * slot = slot_mapping[n * slot_stride]. A negative slot is padding and is skipped; a slot
 * >= num_blocks*block_tokens sets PBS_DEVERR_SLOT_OOB and is skipped. Slots must be distinct
 * (two rows writing one slot leave either row there).
 *
 *   index_k      [num_tokens, dim] elements of elem_bytes (1, 2 or 4) with strides k_stride0, k_stride1
 *   index_cache  [num_blocks, block_tokens, dim], strides c_stride0, c_stride1, and a
 *                contiguous last dimension (PBS_ERR_SHAPE otherwise, as the page raises)
 *   slot_mapping [num_tokens] int64
 */
PBS_API int pbs_insert_index_cache(
    const void* index_k, int64_t k_stride0, int64_t k_stride1, int32_t num_tokens, int32_t dim,
    void* index_cache, int64_t c_stride0, int64_t c_stride1, int32_t num_blocks, int32_t block_tokens,
    const int64_t* slot_mapping, int64_t slot_stride, int32_t elem_bytes,
    int32_t* err_word, pbs_stream_t stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif /* PBS_H */
