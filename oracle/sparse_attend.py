"""Oracle for the MiniMax-M3 paged block-sparse attend: plain, slow, CPU, float64.

TEST INFRASTRUCTURE ONLY. The product (``paged_block_sparse_gb300``) never
imports, calls or links this package; only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline leg may. It shares
no code with the CUDA path: only the seeded input generators (``workloads``)
feed both.

What is computed, and where the pages define it
-----------------------------------------------
Sources are three vLLM API pages:

* [flashinfer] ``vllm.models.minimax_m3.nvidia.sparse_attention_flashinfer``,
  ``MiniMaxM3SparseFlashInferImpl.forward``;
* [nvfp4] ``vllm.models.minimax_m3.amd.sparse_attention_nvfp4``,
  ``MiniMaxM3SparseRocmNvfp4Impl.forward`` and its metadata builder;
* [sparse_pa] ``vllm.models.minimax_m3.amd.ops.sparse_pa``,
  ``_write_sparse_block_table_row_from_values``,
  ``minimax_m3_build_sparse_block_table_decode`` / ``_prefill``,
  ``minimax_m3_insert_index_cache``, ``minimax_m3_sparse_block_page_stride``.

1. Query positions. Decode queries are right-aligned to the request's
   sequence length ([flashinfer] forward: "the default q_offset, which
   right-aligns tokens"); row b*dql+i sits at seq_len[b]-dql+i. Prefill token
   t of request r sits at context_len[r] + (t - cu_seqlens_q[r]) with
   context_len = seq_len - query_len ([nvfp4] metadata builder, per-token
   request id and absolute position).
2. Sparse block table ([sparse_pa] row writer): a selected logical 128-token
   block b is valid iff the row's causal length max(p+1, 0) is positive and
   0 <= b <= p // 128. A block id listed more than once in a row is one
   selection (only its first entry counts). Valid blocks before the query's
   own block are "full" and are packed in top-k order; a valid block equal to
   the own block is the "tail" and goes right after the full ones. Each packed block expands to
   PAGES_PER_BLOCK page-16 ids  page_table[b]*block_page_stride + j. The row
   is zero past the used slots, and the context length is
   128*n_full + (p+1 - 128*(p//128)) when a tail is present, else
   min(128*n_valid, p+1).
3. Attend ([flashinfer] forward, [nvfp4] forward): per query head h of kv
   group g = h // (Hq/Hkv), out = softmax(scale * q_h K^T) V over the keys the
   row attends: every position of each valid full block and positions
   128*(p//128) .. p of the own block when it is selected. K and V are the
   stored values times k_scale / v_scale; the pages fold k_scale into the
   softmax scale and v_scale into the output (exact, since logits are linear
   in K and the output in V); the oracle applies them to the values instead.
4. Index-cache insert ([sparse_pa] insert): cache[slot // T, slot % T, :] =
   index_k[n, :].
5. Log-sum-exp of a row's logits (not on the pages; an optional output of the
   attends so that partial attends over disjoint key sets can be merged):
   lse_h = ln sum_n exp(scale * q_h . k_n) over the same keys as step 3, with
   the same scales; -inf for a row with no attended key.

Readings where the pages are silent (each listed in the design notes too):
SPARSE_BLOCK_SIZE = 128, page rows = 16, PAGES_PER_BLOCK = 8; a page-table
entry is a physical *block* id; rows with no attended key give a zero output.
Repeated ids in one top-k row: a top-k row is read as a SET of blocks. The
row writer itself treats a repeated own block that way (every copy lands on
slot n_full and ctx counts its keys once, through n_full); the same rule for
a repeated full block makes the table, ctx and the attend agree, so the
table of a row equals the row writer applied to the row with its later
repeats removed, and the attend reads every selected block once.
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_bits_to_float, e4m3_to_float, nvfp4_slot_rows

SPARSE_BLOCK_SIZE = 128
PAGE_ROWS = 16
PAGES_PER_BLOCK = SPARSE_BLOCK_SIZE // PAGE_ROWS


# ------------------------------------------------------------------------------------------
# 1. query positions
# ------------------------------------------------------------------------------------------

def decode_query_positions(seq_lens, decode_query_len: int):
    """(request index, absolute position) of each decode row, queries right-aligned."""
    req, pos = [], []
    for b, L in enumerate(np.asarray(seq_lens).tolist()):
        for i in range(decode_query_len):
            req.append(b)
            pos.append(L - decode_query_len + i)
    return np.array(req, dtype=np.int64), np.array(pos, dtype=np.int64)


def prefill_query_positions(cu_seqlens_q, seq_lens):
    """(request index, absolute position) of each prefill token."""
    cu = np.asarray(cu_seqlens_q).tolist()
    sl = np.asarray(seq_lens).tolist()
    req, pos = [], []
    for r in range(len(sl)):
        q_len = cu[r + 1] - cu[r]
        context = sl[r] - q_len
        for j in range(q_len):
            req.append(r)
            pos.append(context + j)
    return np.array(req, dtype=np.int64), np.array(pos, dtype=np.int64)


# ------------------------------------------------------------------------------------------
# 2. sparse block table
# ------------------------------------------------------------------------------------------

def sparse_block_table_row(topk_row, bt_row, abs_pos: int, block_page_stride: int = PAGES_PER_BLOCK):
    """One query's compacted page-16 table row and attended context length."""
    k = len(topk_row)
    causal_len = max(abs_pos + 1, 0)
    own = abs_pos // SPARSE_BLOCK_SIZE
    full, tail = [], []
    seen = set()
    for b in (int(x) for x in topk_row):
        # a block listed again is the same selection: only its first entry is kept
        if b in seen:
            continue
        seen.add(b)
        if causal_len == 0 or b < 0 or b > own:
            continue
        if b == own:
            tail.append(b)
        else:
            full.append(b)
    row = [0] * (k * PAGES_PER_BLOCK)

    def place(slot, b):
        if b >= len(bt_row):
            raise IndexError(f"block {b} is past the page table row ({len(bt_row)} entries)")
        base = int(bt_row[b]) * block_page_stride
        for j in range(PAGES_PER_BLOCK):
            row[slot * PAGES_PER_BLOCK + j] = base + j

    for slot, b in enumerate(full):
        place(slot, b)
    for b in tail:                      # at most one: the own block, after the full ones
        place(len(full), b)
    n_valid = len(full) + len(tail)
    if tail:
        ctx = SPARSE_BLOCK_SIZE * len(full) + (causal_len - SPARSE_BLOCK_SIZE * own)
    else:
        ctx = min(SPARSE_BLOCK_SIZE * n_valid, causal_len)
    return np.array(row, dtype=np.int64), int(ctx)


def _build_rows(topk, page_table, req, pos, block_page_stride):
    tk = np.asarray(topk).reshape(-1, np.asarray(topk).shape[-1])
    pt = np.asarray(page_table)
    n, k = tk.shape
    sbt = np.zeros((n, k * PAGES_PER_BLOCK), dtype=np.int64)
    ctx = np.zeros(n, dtype=np.int64)
    for q in range(n):
        sbt[q], ctx[q] = sparse_block_table_row(tk[q], pt[req[q]], int(pos[q]), block_page_stride)
    return sbt, ctx


def build_sparse_block_table_decode(topk, page_table, seq_lens, decode_query_len: int = 1,
                                    block_page_stride: int = PAGES_PER_BLOCK):
    """[flashinfer]/[sparse_pa] decode: one table row per decode query row."""
    req, pos = decode_query_positions(seq_lens, decode_query_len)
    n = np.asarray(topk).shape[-2]
    if n != len(req):
        raise ValueError(f"decode top-k rows must equal batch * decode_query_len: {n} != {len(req)}")
    return _build_rows(topk, page_table, req, pos, block_page_stride)


def build_sparse_block_table_prefill(topk, page_table, cu_seqlens_q, seq_lens,
                                     block_page_stride: int = PAGES_PER_BLOCK):
    """[sparse_pa] prefill: one table row per prefill token."""
    req, pos = prefill_query_positions(cu_seqlens_q, seq_lens)
    return _build_rows(topk, page_table, req, pos, block_page_stride)


# ------------------------------------------------------------------------------------------
# 3. attend
# ------------------------------------------------------------------------------------------

def attended_positions(topk_row, abs_pos: int) -> np.ndarray:
    """Logical key positions a query attends: each selected block once, however often listed."""
    if abs_pos < 0:
        return np.zeros(0, dtype=np.int64)
    own = abs_pos // SPARSE_BLOCK_SIZE
    chosen = sorted({int(b) for b in topk_row if 0 <= int(b) <= own})
    keys = []
    for b in chosen:
        last = abs_pos if b == own else SPARSE_BLOCK_SIZE * (b + 1) - 1
        keys.extend(range(SPARSE_BLOCK_SIZE * b, last + 1))
    return np.array(keys, dtype=np.int64)


def gather_kv(cache, kv_dtype: str, num_kv_heads: int, head_dim: int, bt_row, positions,
              block_page_stride: int = PAGES_PER_BLOCK):
    """Stored K and V (float64, before k_scale/v_scale) of logical key positions.

    A position x lives on page page_table[x // 128] * block_page_stride +
    (x % 128) // 16, row x % 16. ``cache[ids]`` must return the raw bytes of the
    listed pages, shape [len(ids), page_bytes]. Returns K, V of shape
    [num_kv_heads, len(positions), head_dim].
    """
    x = np.asarray(positions, dtype=np.int64)
    Hkv, D = num_kv_heads, head_dim
    if x.size == 0:
        z = np.zeros((Hkv, 0, D))
        return z, z.copy()
    bt = np.asarray(bt_row, dtype=np.int64)
    pages = bt[x // SPARSE_BLOCK_SIZE] * block_page_stride + (x % SPARSE_BLOCK_SIZE) // PAGE_ROWS
    rows = x % PAGE_ROWS
    uniq, inv = np.unique(pages, return_inverse=True)
    raw = np.asarray(cache[uniq], dtype=np.uint8)            # [u, page_bytes]
    if kv_dtype == "bf16":
        pg = raw.view(np.uint16).reshape(len(uniq), Hkv, PAGE_ROWS, 2 * D)
        sel = pg[inv, :, rows, :]                               # [n, Hkv, 2D]
        vals = bf16_bits_to_float(sel)
        K, V = vals[..., :D], vals[..., D:]
    elif kv_dtype == "fp8_e4m3":
        pg = raw.reshape(len(uniq), Hkv, PAGE_ROWS, 2 * D)
        vals = e4m3_to_float(pg[inv, :, rows, :])
        K, V = vals[..., :D], vals[..., D:]
    elif kv_dtype == "nvfp4":
        if D != 128:
            raise ValueError("the NVFP4 slot layout holds head_dim 128")
        pg = raw.reshape(len(uniq), 2 * Hkv, -1)
        K = np.empty((len(x), Hkv, D))
        V = np.empty((len(x), Hkv, D))
        for u in range(len(uniq)):
            sel = np.nonzero(inv == u)[0]
            for g in range(Hkv):
                K[sel, g] = nvfp4_slot_rows(pg[u, 2 * g], rows[sel])
                V[sel, g] = nvfp4_slot_rows(pg[u, 2 * g + 1], rows[sel])
    else:
        raise ValueError(f"unknown kv dtype {kv_dtype!r}")
    return np.ascontiguousarray(K.transpose(1, 0, 2)), np.ascontiguousarray(V.transpose(1, 0, 2))


def attend(q_heads, K, V, softmax_scale: float, k_scale: float = 1.0, v_scale: float = 1.0):
    """Plain GQA attention of one query row over its gathered keys.

    q_heads [Hq, D]; K, V [Hkv, n, D] stored values. Head h reads kv head
    h // (Hq // Hkv). The scales multiply the stored values. Returns [Hq, D];
    zero when n == 0.
    """
    q = np.asarray(q_heads, dtype=np.float64)
    Hq, D = q.shape
    Hkv, n, _ = K.shape
    G = Hq // Hkv
    out = np.zeros((Hq, D))
    if n == 0:
        return out
    Kd = K * k_scale
    Vd = V * v_scale
    for h in range(Hq):
        g = h // G
        logits = softmax_scale * (Kd[g] @ q[h])                # [n]
        w = np.exp(logits - logits.max())
        out[h] = (w @ Vd[g]) / w.sum()
    return out


def attend_lse(q_heads, K, softmax_scale: float, k_scale: float = 1.0):
    """Natural-log log-sum-exp of each head's logits (step 5): [Hq], -inf when n == 0."""
    q = np.asarray(q_heads, dtype=np.float64)
    Hq, _ = q.shape
    Hkv, n, _ = K.shape
    G = Hq // Hkv
    lse = np.full(Hq, -np.inf)
    if n == 0:
        return lse
    Kd = K * k_scale
    for h in range(Hq):
        logits = softmax_scale * (Kd[h // G] @ q[h])
        m = logits.max()
        lse[h] = m + np.log(np.exp(logits - m).sum())
    return lse


def _attend_rows(q, cache, kv_dtype, num_kv_heads, topk, page_table, req, pos, softmax_scale,
                 k_scale, v_scale, block_page_stride, rows, return_lse=False):
    qa = np.asarray(q, dtype=np.float64)
    tk = np.asarray(topk).reshape(-1, np.asarray(topk).shape[-1])
    pt = np.asarray(page_table)
    n, Hq, D = qa.shape
    rows = range(n) if rows is None else rows
    out, lse = {}, {}
    for r in rows:
        keys = attended_positions(tk[r], int(pos[r]))
        K, V = gather_kv(cache, kv_dtype, num_kv_heads, D, pt[req[r]], keys, block_page_stride)
        out[r] = attend(qa[r], K, V, softmax_scale, k_scale, v_scale)
        if return_lse:
            lse[r] = attend_lse(qa[r], K, softmax_scale, k_scale)
    return (out, lse) if return_lse else out


def sparse_decode_attention(q, cache, kv_dtype: str, num_kv_heads: int, topk, page_table, seq_lens,
                            decode_query_len: int, softmax_scale: float, k_scale: float = 1.0,
                            v_scale: float = 1.0, block_page_stride: int = PAGES_PER_BLOCK, rows=None,
                            return_lse: bool = False):
    """Decode attend; returns {row: out[Hq, D]} for the requested rows (all by default), and
    {row: lse[Hq]} as well with ``return_lse``."""
    req, pos = decode_query_positions(seq_lens, decode_query_len)
    return _attend_rows(q, cache, kv_dtype, num_kv_heads, topk, page_table, req, pos, softmax_scale,
                        k_scale, v_scale, block_page_stride, rows, return_lse)


def sparse_prefill_attention(q, cache, kv_dtype: str, num_kv_heads: int, topk, page_table,
                             cu_seqlens_q, seq_lens, softmax_scale: float, k_scale: float = 1.0,
                             v_scale: float = 1.0, block_page_stride: int = PAGES_PER_BLOCK, rows=None,
                             return_lse: bool = False):
    """Prefill attend (varlen); returns {token: out[Hq, D]} (and {token: lse[Hq]})."""
    req, pos = prefill_query_positions(cu_seqlens_q, seq_lens)
    return _attend_rows(q, cache, kv_dtype, num_kv_heads, topk, page_table, req, pos, softmax_scale,
                        k_scale, v_scale, block_page_stride, rows, return_lse)


# ------------------------------------------------------------------------------------------
# 4. index-cache insert
# ------------------------------------------------------------------------------------------

def insert_index_cache(index_k, index_cache, slot_mapping):
    """Return a copy of index_cache [B, T, D] with row n of index_k written at slot_mapping[n].

    A negative slot is padding and writes nothing (a reading: the page does
    not say what a negative slot means).
    """
    cache = np.array(index_cache, copy=True)
    B, T, D = cache.shape
    for n, slot in enumerate(np.asarray(slot_mapping).tolist()):
        if slot < 0:
            continue
        cache[slot // T, slot % T, :] = np.asarray(index_k)[n, :]
    return cache
