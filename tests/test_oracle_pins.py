"""Pins for the CPU oracle: values the pages fix, closed forms, invariants and
library special cases that do not go through the oracle's own code.

Each test names the passage it follows (vLLM API pages
``vllm.models.minimax_m3.amd.ops.sparse_pa`` [sparse_pa],
``vllm.models.minimax_m3.nvidia.sparse_attention_flashinfer`` [flashinfer],
``vllm.models.minimax_m3.amd.sparse_attention_nvfp4`` [nvfp4]).
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------------------------
# sparse block table: hand-worked rows, closed form, brute force
# ---------------------------------------------------------------------------------------------

@pytest.mark.parametrize("case", _load("sparse_table_rows.json")["cases"], ids=lambda c: c["name"])
def test_table_row_golden(case):
    """[sparse_pa] row writer, worked by hand."""
    row, ctx = oracle.sparse_block_table_row(case["topk"], case["bt_row"], case["abs_pos"],
                                             case["block_page_stride"])
    want = case["row_prefix"] + [0] * (case["width"] - len(case["row_prefix"]))
    assert row.tolist() == want
    assert ctx == case["ctx"]


def test_query_positions_golden():
    g = _load("query_positions.json")
    for c in g["decode"]:
        req, pos = oracle.decode_query_positions(c["seq_lens"], c["decode_query_len"])
        assert req.tolist() == c["req"] and pos.tolist() == c["pos"]
    for c in g["prefill"]:
        req, pos = oracle.prefill_query_positions(c["cu_seqlens_q"], c["seq_lens"])
        assert req.tolist() == c["req"] and pos.tolist() == c["pos"]


def _random_rows(rng, n, k, max_pos, distinct=True):
    rows, poss = [], []
    for _ in range(n):
        p = int(rng.integers(-3, max_pos))
        own = max(p, 0) // 128
        cand = np.arange(0, own + 4)           # includes future blocks to exercise the filter
        pick = rng.choice(cand, size=min(k, len(cand)), replace=not distinct)
        row = list(pick) + [-1] * (k - len(pick))
        rng.shuffle(row)
        rows.append(row)
        poss.append(p)
    return rows, poss


def test_ctx_closed_form():
    """ctx = 128 * #{valid b < own} + [own selected] * (p - 128*own + 1) for distinct ids."""
    rng = np.random.default_rng(1)
    bt = np.arange(40)[::-1].copy()
    rows, poss = _random_rows(rng, 400, 6, 4000)
    for row, p in zip(rows, poss):
        _, ctx = oracle.sparse_block_table_row(row, bt, p)
        if p < 0:
            assert ctx == 0
            continue
        own = p // 128
        n_full = sum(1 for b in row if 0 <= b < own)
        has_own = own in row
        assert ctx == 128 * n_full + (p - 128 * own + 1 if has_own else 0)


def test_table_walk_equals_direct_mapping():
    """Brute force: keys 0..ctx-1 read through the compacted table are exactly the
    attended positions mapped page by page ([sparse_pa] row writer vs the attend's key set)."""
    rng = np.random.default_rng(2)
    bt = rng.permutation(40)
    for bps in (8, 16):
        rows, poss = _random_rows(rng, 300, 5, 4500)
        for row, p in zip(rows, poss):
            sbt, ctx = oracle.sparse_block_table_row(row, bt, p, bps)
            walked = sorted((int(sbt[n // 16]), n % 16) for n in range(ctx))
            direct = sorted((int(bt[x // 128]) * bps + (x % 128) // 16, x % 16)
                            for x in oracle.attended_positions(row, p))
            assert walked == direct


def test_table_walk_with_repeated_ids_reads_each_block_once():
    """Brute force on rows whose ids repeat (drawn with replacement): walking keys 0..ctx-1
    through the table visits every attended (page, row) exactly once, and ctx is the closed
    form counted over the row's distinct blocks (the writer's own treatment of a repeated own
    block, one slot and its keys counted once, applied to every block)."""
    rng = np.random.default_rng(7)
    bt = rng.permutation(40)
    rows, poss = _random_rows(rng, 400, 8, 4500, distinct=False)
    assert sum(len(set(r) - {-1}) < len([b for b in r if b >= 0]) for r in rows) > 100
    for row, p in zip(rows, poss):
        sbt, ctx = oracle.sparse_block_table_row(row, bt, p)
        walked = [(int(sbt[n // 16]), n % 16) for n in range(ctx)]
        assert len(walked) == len(set(walked))
        direct = sorted((int(bt[x // 128]) * 8 + (x % 128) // 16, x % 16) for x in oracle.attended_positions(row, p))
        assert sorted(walked) == direct
        if p >= 0:
            own = p // 128
            distinct = {b for b in row if 0 <= b <= own}
            n_full = len(distinct - {own})
            assert ctx == 128 * n_full + (p - 128 * own + 1 if own in distinct else 0)


def test_table_repeats_equal_row_without_them():
    """A repeated id is one selection: replacing every later copy of an id by -1 leaves the row
    and ctx unchanged, bit for bit (written for any mix of full and own-block repeats)."""
    rng = np.random.default_rng(8)
    bt = rng.permutation(40)
    rows, poss = _random_rows(rng, 300, 7, 4500, distinct=False)
    for row, p in zip(rows, poss):
        seen, stripped = set(), []
        for b in row:
            stripped.append(-1 if b in seen else b)
            seen.add(b)
        a, ca = oracle.sparse_block_table_row(row, bt, p)
        b_, cb = oracle.sparse_block_table_row(stripped, bt, p)
        assert ca == cb and np.array_equal(a, b_)


def test_table_order_and_padding_invariance():
    """Permuting a row's ids or moving its -1s keeps ctx and the set of 8-page groups."""
    rng = np.random.default_rng(3)
    bt = rng.permutation(40)
    rows, poss = _random_rows(rng, 200, 6, 4500)
    for row, p in zip(rows, poss):
        a, ca = oracle.sparse_block_table_row(row, bt, p)
        row2 = list(row)
        rng.shuffle(row2)
        b, cb = oracle.sparse_block_table_row(row2, bt, p)
        assert ca == cb
        ga = sorted(tuple(a[i:i + 8]) for i in range(0, len(a), 8))
        gb = sorted(tuple(b[i:i + 8]) for i in range(0, len(b), 8))
        assert ga == gb


def test_decode_table_row_count_contract():
    """[sparse_pa] decode builder: rows must equal batch * decode_query_len."""
    with pytest.raises(ValueError):
        oracle.build_sparse_block_table_decode(np.zeros((1, 3, 4), np.int32), np.zeros((2, 4), np.int32),
                                               [100, 100], decode_query_len=1)


# ---------------------------------------------------------------------------------------------
# element formats
# ---------------------------------------------------------------------------------------------

def test_e2m1_and_e4m3_golden():
    g = _load("element_formats.json")
    v = oracle.e2m1_to_float(np.array(g["e2m1"]["codes"], np.uint8))
    assert v.tolist() == g["e2m1"]["values"]
    assert np.signbit(v[8])
    v = oracle.e4m3_to_float(np.array(g["e4m3"]["codes"], np.uint8))
    assert v.tolist() == g["e4m3"]["values"]
    assert np.isnan(oracle.e4m3_to_float(np.array(g["e4m3"]["nan_codes"], np.uint8))).all()


def test_e4m3_matches_torch_for_all_codes():
    """Library special case: torch's float8_e4m3fn decodes every code the same way."""
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_float(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(lib)
    assert np.array_equal(ours[~both_nan], lib[~both_nan])
    assert np.array_equal(np.isnan(ours), np.isnan(lib))


def test_bf16_decode_matches_torch():
    x = torch.randn(4096, dtype=torch.float32).to(torch.bfloat16)
    ours = oracle.bf16_bits_to_float(x.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(ours, x.to(torch.float64).numpy())


def test_nvfp4_slot_layout_hand_built():
    """Slot = 16 rows x 64 B codes (element 2i low nibble) then 16 rows x 8 B e4m3 scales."""
    slot = np.zeros(1152, np.uint8)
    slot[0] = 0x21                       # row 0: elem 0 = code 1 (0.5), elem 1 = code 2 (1.0)
    slot[8] = 0xF7                       # row 0: elem 16 = code 7 (6.0), elem 17 = code 15 (-6.0)
    slot[64 * 3 + 63] = 0x5D             # row 3: elem 126 = code 13 (-3.0), elem 127 = code 5 (3.0)
    slot[1024 + 0] = 0x38                # row 0 scale 0 = 1.0 (elements 0..15)
    slot[1024 + 1] = 0x40                # row 0 scale 1 = 2.0 (elements 16..31)
    slot[1024 + 3 * 8 + 7] = 0x30        # row 3 scale 7 = 0.5 (elements 112..127)
    r = oracle.nvfp4_slot_rows(slot, np.array([0, 3]))
    assert r.shape == (2, 128)
    assert r[0, 0] == 0.5 and r[0, 1] == 1.0 and r[0, 16] == 12.0 and r[0, 17] == -12.0
    assert r[1, 126] == -1.5 and r[1, 127] == 1.5
    assert np.count_nonzero(r) == 6


# ---------------------------------------------------------------------------------------------
# attend: dense special case against torch SDPA, closed forms, invariants
# ---------------------------------------------------------------------------------------------

def _paged_cache_from_logical(K, V, kv_dtype, rng, nblocks_pool=None):
    """Scatter logical K/V [Hkv, L, D] (already in stored form) into a shuffled paged cache.

    Returns (cache uint8 [pages, page_bytes], bt_row). The physical page of
    logical position x is bt[x // 128] * 8 + (x % 128) // 16, row x % 16.
    """
    Hkv, L, D = K.shape
    nb = math.ceil(L / 128)
    pool = nblocks_pool or nb + 3
    bt = rng.permutation(pool)[:nb]
    if kv_dtype == "bf16":
        elem = np.uint16
    else:
        elem = np.uint8
    pages = np.zeros((pool * 8, Hkv, 16, 2 * D), dtype=elem)
    for x in range(L):
        pg = bt[x // 128] * 8 + (x % 128) // 16
        pages[pg, :, x % 16, :D] = K[:, x, :]
        pages[pg, :, x % 16, D:] = V[:, x, :]
    return pages.reshape(pool * 8, -1).view(np.uint8), bt


def _sdpa_reference(q, K, V, scale, positions):
    """torch SDPA (float64, CPU) with an explicit causal mask: query at position p sees 0..p."""
    Hq = q.shape[1]
    Hkv, L, D = K.shape
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]            # [1, Hq, n, D]
    kt = torch.from_numpy(K)[None]
    vt = torch.from_numpy(V)[None]
    mask = torch.from_numpy(np.arange(L)[None, :] <= np.asarray(positions)[:, None])
    out = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale, enable_gqa=True)
    return out[0].permute(1, 0, 2).numpy()                     # [n, Hq, D]


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (8, 2), (4, 4)])
def test_dense_topk_equals_causal_attention(kv_dtype, Hq, Hkv):
    """Top-k listing every block 0..own: the attend is plain causal attention
    ([flashinfer] forward: causal=True; GQA head h reads kv head h // (Hq/Hkv)).
    Reference: torch scaled_dot_product_attention on the unpaged sequence."""
    rng = np.random.default_rng(4)
    L, D = 300, 128
    if kv_dtype == "bf16":
        Kb = torch.randn(Hkv, L, D).to(torch.bfloat16)
        Vb = torch.randn(Hkv, L, D).to(torch.bfloat16)
        Kst, Vst = (t.view(torch.int16).numpy().view(np.uint16) for t in (Kb, Vb))
        Kf, Vf = Kb.double().numpy(), Vb.double().numpy()
        ks, vs = 1.0, 1.0
    else:
        Kb = torch.randn(Hkv, L, D).to(torch.float8_e4m3fn)
        Vb = torch.randn(Hkv, L, D).to(torch.float8_e4m3fn)
        Kst, Vst = (t.view(torch.uint8).numpy() for t in (Kb, Vb))
        Kf, Vf = Kb.double().numpy(), Vb.double().numpy()
        ks, vs = 1.5, 0.625
    cache, bt = _paged_cache_from_logical(Kst, Vst, kv_dtype, rng)
    positions = np.array([0, 1, 77, 127, 128, 129, 200, 255, 256, 299])
    nb = math.ceil(L / 128)
    topk = np.full((1, len(positions), nb + 1), -1, np.int32)
    for i, p in enumerate(positions):
        own = p // 128
        ids = rng.permutation(own + 1)
        topk[0, i, :own + 1] = ids
    q = torch.randn(len(positions), Hq, D).to(torch.bfloat16).double().numpy()
    scale = 1.0 / math.sqrt(D)
    cu = [0, len(positions)]
    # every position is its own one-token "request" that shares the same pages
    outs = []
    for i, p in enumerate(positions):
        o = oracle.sparse_prefill_attention(q[i:i + 1], cache, kv_dtype, Hkv, topk[:, i:i + 1], bt[None],
                                            [0, 1], [p + 1], scale, ks, vs)
        outs.append(o[0])
    ours = np.stack(outs)
    ref = _sdpa_reference(q, Kf * ks, Vf * vs, scale, positions)
    np.testing.assert_allclose(ours, ref, rtol=0, atol=1e-12)


def test_partials_over_disjoint_key_sets_combine_by_lse():
    """Attention over a key set split into disjoint parts: each part's output weighted by
    exp(lse_part - lse_all), summed, is the output over the whole set, and lse_all is the
    log-sum-exp of the parts' lse (the identity behind per-block partials merged by their
    log-sum-exp; a dropped or mis-signed term in either oracle function breaks it)."""
    rng = np.random.default_rng(31)
    Hq, Hkv, n, D = 8, 2, 300, 64
    q = rng.standard_normal((Hq, D))
    K = rng.standard_normal((Hkv, n, D))
    V = rng.standard_normal((Hkv, n, D))
    scale, ks, vs = 0.11, 1.5, 0.75
    full = oracle.attend(q, K, V, scale, ks, vs)
    lse_full = oracle.attend_lse(q, K, scale, ks)
    cuts = [0, 1, 128, 131, 300]  # parts of 1, 127, 3 and 169 keys
    outs, lses = [], []
    for a, b in zip(cuts[:-1], cuts[1:]):
        outs.append(oracle.attend(q, K[:, a:b], V[:, a:b], scale, ks, vs))
        lses.append(oracle.attend_lse(q, K[:, a:b], scale, ks))
    lses = np.stack(lses)                      # [parts, Hq]
    m = lses.max(axis=0)
    lse_comb = m + np.log(np.exp(lses - m).sum(axis=0))
    np.testing.assert_allclose(lse_comb, lse_full, rtol=0, atol=1e-12)
    comb = sum(np.exp(l - lse_full)[:, None] * o for l, o in zip(lses, outs))
    np.testing.assert_allclose(comb, full, rtol=0, atol=1e-12)


def test_dense_lse_equals_torch_logsumexp():
    """Log-sum-exp output, dense top-k: equals torch.logsumexp of the causal logits computed on
    the unpaged sequence (a library routine on an independent path from the paged gather)."""
    rng = np.random.default_rng(14)
    Hq, Hkv, L, D = 8, 2, 300, 128
    Kb = torch.randn(Hkv, L, D).to(torch.bfloat16)
    Vb = torch.randn(Hkv, L, D).to(torch.bfloat16)
    Kst, Vst = (t.view(torch.int16).numpy().view(np.uint16) for t in (Kb, Vb))
    cache, bt = _paged_cache_from_logical(Kst, Vst, "bf16", rng)
    positions = np.array([0, 1, 127, 128, 200, 299])
    topk = np.full((1, len(positions), 4), -1, np.int32)
    for i, p in enumerate(positions):
        topk[0, i, :p // 128 + 1] = rng.permutation(p // 128 + 1)
    q = torch.randn(len(positions), Hq, D).to(torch.bfloat16).double()
    scale, ks = 0.07, 1.25
    logits = torch.einsum("nhd,hld->nhl", q, Kb.double().repeat_interleave(Hq // Hkv, 0) * ks) * scale
    mask = torch.from_numpy(np.arange(L)[None, :] <= positions[:, None])[:, None, :]
    ref = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=-1).numpy()
    for i, p in enumerate(positions):
        _, lse = oracle.sparse_prefill_attention(q[i:i + 1].numpy(), cache, "bf16", Hkv, topk[:, i:i + 1], bt[None],
                                                 [0, 1], [p + 1], scale, ks, 1.0, return_lse=True)
        np.testing.assert_allclose(lse[0], ref[i], rtol=0, atol=1e-11)


def test_lse_with_equal_keys_is_logit_plus_log_ctx():
    """Closed form: when every cached key is the same vector k, every logit is scale*q.k, so
    lse = scale*q.k + ln(ctx) with ctx the row's attended-key count from the table's closed form
    (random top-k with padding and future ids); an empty row gives -inf."""
    rng = np.random.default_rng(15)
    Hq, Hkv, L, D = 4, 1, 1000, 128
    k = torch.randn(D).to(torch.bfloat16)
    Kst = k.view(torch.int16).numpy().view(np.uint16)[None, None, :].repeat(L, 1)
    Vst = torch.randn(Hkv, L, D).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    cache, bt = _paged_cache_from_logical(Kst, Vst, "bf16", rng)
    q = torch.randn(1, Hq, D).to(torch.bfloat16).double().numpy()
    scale = 0.09
    for p in [-1, 0, 130, 511, 999]:
        row = rng.permutation(np.arange(-1, 9))[:6].astype(np.int32)
        _, ctx = oracle.sparse_block_table_row(row, bt, p)
        _, lse = oracle.sparse_prefill_attention(q, cache, "bf16", Hkv, row[None, None, :], bt[None], [0, 1], [p + 1],
                                                 scale, return_lse=True)
        if ctx == 0:
            assert np.all(np.isneginf(lse[0]))
        else:
            want = scale * (q[0] @ k.double().numpy()) + math.log(ctx)
            np.testing.assert_allclose(lse[0], want, rtol=0, atol=1e-11)


def test_dense_ctx_is_position_plus_one():
    rng = np.random.default_rng(5)
    bt = rng.permutation(10)
    for p in [0, 5, 127, 128, 500, 1279]:
        own = p // 128
        _, ctx = oracle.sparse_block_table_row(list(range(own + 1)), bt, p)
        assert ctx == p + 1


def test_position_zero_returns_first_value():
    """Closed form: a query at position 0 attends only key 0, so out = v_scale * v_0."""
    b = workloads.small(kv_dtype="fp8_e4m3", num_heads=4, num_kv_heads=2, topk=3, pre_q_lens=[5], seed=3)
    q = b.pre.q.double().numpy()
    out = oracle.sparse_prefill_attention(q, b.cache.numpy(), "fp8_e4m3", 2, b.pre.topk.numpy(),
                                          b.pre.page_table.numpy(), b.pre.cu_seqlens_q.numpy(),
                                          b.pre.seq_lens.numpy(), b.softmax_scale, b.k_scale, b.v_scale, rows=[0])[0]
    pg = int(b.pre.page_table[0, 0]) * 8
    raw = b.cache[pg].view(torch.float8_e4m3fn).reshape(2, 16, 256)[:, 0, 128:].double().numpy()
    for h in range(4):
        np.testing.assert_allclose(out[h], b.v_scale * raw[h // 2], rtol=0, atol=1e-12)


def test_zero_query_is_mean_of_values():
    """Closed form: q = 0 gives uniform weights, so out = mean of the attended V rows."""
    rng = np.random.default_rng(6)
    Hkv, L, D = 2, 400, 128
    Vb = torch.randn(Hkv, L, D).to(torch.bfloat16)
    Kb = torch.randn(Hkv, L, D).to(torch.bfloat16)
    cache, bt = _paged_cache_from_logical(Kb.view(torch.int16).numpy().view(np.uint16),
                                          Vb.view(torch.int16).numpy().view(np.uint16), "bf16", rng)
    p = 390                                # own block 3; select blocks 0 and 3 -> keys 0..127, 384..390
    topk = np.array([[[3, -1, 0]]], np.int32)
    out = oracle.sparse_prefill_attention(np.zeros((1, 4, D)), cache, "bf16", Hkv, topk, bt[None], [0, 1], [p + 1],
                                          0.1, 1.0, 2.0)[0]
    keys = list(range(0, 128)) + list(range(384, 391))
    want = 2.0 * Vb.double().numpy()[:, keys, :].mean(axis=1)
    for h in range(4):
        np.testing.assert_allclose(out[h], want[h // 2], rtol=0, atol=1e-12)


def test_zero_query_with_repeated_blocks_is_mean_over_distinct_keys():
    """Closed form with repeated ids: q = 0 gives uniform weights over the attended keys, and a
    block listed twice (full block 1, own block 3) contributes its keys once, so out is the
    plain mean of V over blocks 0, 1 and keys 384..390 (computed here from the unpaged values)."""
    rng = np.random.default_rng(16)
    Hkv, L, D = 2, 400, 128
    Vb = torch.randn(Hkv, L, D).to(torch.bfloat16)
    Kb = torch.randn(Hkv, L, D).to(torch.bfloat16)
    cache, bt = _paged_cache_from_logical(Kb.view(torch.int16).numpy().view(np.uint16),
                                          Vb.view(torch.int16).numpy().view(np.uint16), "bf16", rng)
    p = 390
    topk = np.array([[[1, 3, 0, 1, 3, -1]]], np.int32)
    out = oracle.sparse_prefill_attention(np.zeros((1, 4, D)), cache, "bf16", Hkv, topk, bt[None], [0, 1], [p + 1],
                                          0.1, 1.0, 1.0)[0]
    keys = list(range(0, 256)) + list(range(384, 391))
    want = Vb.double().numpy()[:, keys, :].mean(axis=1)
    for h in range(4):
        np.testing.assert_allclose(out[h], want[h // 2], rtol=0, atol=1e-12)


def test_gqa_head_equals_single_head_run():
    """With G = Hq/Hkv, head h of a GQA run equals a 1-q-head, 1-kv-head run on (q_h, kv head h//G)."""
    b = workloads.small(num_heads=8, num_kv_heads=2, topk=4, pre_q_lens=[300], seed=9)
    cache = b.cache.numpy()
    q = b.pre.q.double().numpy()
    full = oracle.sparse_prefill_attention(q, cache, "bf16", 2, b.pre.topk.numpy(), b.pre.page_table.numpy(),
                                           b.pre.cu_seqlens_q.numpy(), b.pre.seq_lens.numpy(),
                                           b.softmax_scale, rows=[10, 150, 299])
    # single kv head view: keep only kv head g of each page
    pages = b.cache.view(torch.bfloat16).reshape(b.num_pages, 2, 16, 256)
    for h in (0, 3, 4, 7):
        g = h // 4
        one = pages[:, g:g + 1].contiguous().view(torch.uint8).reshape(b.num_pages, -1).numpy()
        single = oracle.sparse_prefill_attention(q[:, h:h + 1], one, "bf16", 1, b.pre.topk.numpy(),
                                                 b.pre.page_table.numpy(), b.pre.cu_seqlens_q.numpy(),
                                                 b.pre.seq_lens.numpy(), b.softmax_scale, rows=[10, 150, 299])
        for r in (10, 150, 299):
            np.testing.assert_allclose(full[r][h], single[r][0], rtol=0, atol=1e-13)


def test_scale_fold_identity():
    """[flashinfer] forward: folding k_scale into the softmax scale and v_scale into the
    output is exact, i.e. attend(scale, ks, vs) = vs * attend(scale * ks, 1, 1)."""
    b = workloads.small(kv_dtype="fp8_e4m3", num_heads=8, num_kv_heads=2, topk=4, pre_q_lens=[260], seed=10)
    args = (b.pre.q.double().numpy(), b.cache.numpy(), "fp8_e4m3", 2, b.pre.topk.numpy(),
            b.pre.page_table.numpy(), b.pre.cu_seqlens_q.numpy(), b.pre.seq_lens.numpy())
    a = oracle.sparse_prefill_attention(*args, b.softmax_scale, b.k_scale, b.v_scale, rows=[3, 259])
    f = oracle.sparse_prefill_attention(*args, b.softmax_scale * b.k_scale, 1.0, 1.0, rows=[3, 259])
    for r in (3, 259):
        np.testing.assert_allclose(a[r], b.v_scale * f[r], rtol=1e-12, atol=1e-12)


def test_attend_order_and_padding_invariance():
    b = workloads.small(num_heads=4, num_kv_heads=1, topk=5, pre_q_lens=[700], seed=11)
    tk = b.pre.topk.numpy().copy()
    rng = np.random.default_rng(0)
    tk2 = tk.copy()
    for r in range(tk.shape[1]):
        rng.shuffle(tk2[0, r])
    args = lambda t: (b.pre.q.double().numpy(), b.cache.numpy(), "bf16", 1, t, b.pre.page_table.numpy(),
                      b.pre.cu_seqlens_q.numpy(), b.pre.seq_lens.numpy(), b.softmax_scale)
    rows = [0, 130, 500, 699]
    a = oracle.sparse_prefill_attention(*args(tk), rows=rows)
    c = oracle.sparse_prefill_attention(*args(tk2), rows=rows)
    for r in rows:
        np.testing.assert_array_equal(a[r], c[r])


def test_empty_row_gives_zero():
    """Reading: a row with no attended key (padded, or every id filtered) outputs zeros."""
    b = workloads.small(num_heads=4, num_kv_heads=1, topk=3, dec_seq_lens=[0, 300], seed=12)
    out = oracle.sparse_decode_attention(b.dec.q.double().numpy(), b.cache.numpy(), "bf16", 1, b.dec.topk.numpy(),
                                         b.dec.page_table.numpy(), b.dec.seq_lens.numpy(), 1, b.softmax_scale)
    assert np.all(out[0] == 0.0)
    assert np.abs(out[1]).sum() > 0


def test_tiny_decode_equals_prefill_last_row():
    """Tiny workload: the decode row (seq 1024, right-aligned at 1023) with prefill token
    1023's top-k has the same table, context length and output as that prefill row."""
    b = workloads.tiny()
    cache = b.cache.numpy()
    d_sbt, d_ctx = oracle.build_sparse_block_table_decode(b.dec.topk.numpy(), b.dec.page_table.numpy(),
                                                          b.dec.seq_lens.numpy(), 1)
    p_sbt, p_ctx = oracle.build_sparse_block_table_prefill(b.pre.topk.numpy(), b.pre.page_table.numpy(),
                                                           b.pre.cu_seqlens_q.numpy(), b.pre.seq_lens.numpy())
    assert np.array_equal(d_sbt[0], p_sbt[1023]) and d_ctx[0] == p_ctx[1023]
    d = oracle.sparse_decode_attention(b.dec.q.double().numpy(), cache, "bf16", 1, b.dec.topk.numpy(),
                                       b.dec.page_table.numpy(), b.dec.seq_lens.numpy(), 1, b.softmax_scale)[0]
    p = oracle.sparse_prefill_attention(b.pre.q.double().numpy(), cache, "bf16", 1, b.pre.topk.numpy(),
                                        b.pre.page_table.numpy(), b.pre.cu_seqlens_q.numpy(),
                                        b.pre.seq_lens.numpy(), b.softmax_scale, rows=[1023])[1023]
    np.testing.assert_array_equal(d, p)


# ---------------------------------------------------------------------------------------------
# index-cache insert
# ---------------------------------------------------------------------------------------------

def test_insert_index_cache_hand_example():
    """[sparse_pa] insert: cache[slot // T, slot % T, :] = index_k[n, :] (negative slot skipped)."""
    k = np.array([[1, 2], [3, 4], [5, 6]], np.float32)
    c = np.zeros((2, 2, 2), np.float32)
    out = oracle.insert_index_cache(k, c, [3, -1, 0])
    want = np.zeros((2, 2, 2), np.float32)
    want[1, 1] = [1, 2]
    want[0, 0] = [5, 6]
    assert np.array_equal(out, want)
    assert np.all(c == 0)


def test_nvfp4_gather_reads_k_and_v_slots_of_the_right_head():
    """Reading of [nvfp4] customize_spec (two slots per kv head): slot 2g = K_g, slot 2g+1 = V_g."""
    Hkv = 2
    page = np.zeros((2 * Hkv, 1152), np.uint8)
    for slot in range(2 * Hkv):
        page[slot, 5 * 64 + 0] = slot + 1          # row 5, element 0 = code slot+1
        page[slot, 1024 + 5 * 8 + 0] = 0x38        # row 5 scale 0 = 1.0
    cache = np.zeros((32, 2 * Hkv * 1152), np.uint8)
    cache[8 * 3 + 0] = page.reshape(-1)            # logical block 0 -> physical block 3, page 0
    K, V = oracle.gather_kv(cache, "nvfp4", Hkv, 128, [3], [5])
    e = oracle.e2m1_to_float(np.arange(1, 5, dtype=np.uint8))
    assert K[0, 0, 0] == e[0] and V[0, 0, 0] == e[1] and K[1, 0, 0] == e[2] and V[1, 0, 0] == e[3]
