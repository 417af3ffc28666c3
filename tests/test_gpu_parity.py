"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tables and context lengths must match bit for bit; attention outputs within max-abs 1e-2 /
relative-RMS 2e-3 (bf16 KV) or 5e-2 / 1e-2 (fp8 / NVFP4 KV, against the oracle on the same
dequantised values)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_close, cache_source, np_i32, oracle_decode, oracle_prefill, q64

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def pbs():
    from paged_block_sparse_gb300 import _build
    _build.build()
    import paged_block_sparse_gb300 as m
    return m


def _err():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def gpu_tables(pbs, b, part):
    err = _err()
    if part == "dec":
        d = b.dec
        sbt, ctx = pbs.build_sparse_block_table_decode(d.topk, d.page_table, d.seq_lens, d.decode_query_len,
                                                       b.block_page_stride, err_word=err)
    else:
        p = b.pre
        sbt, ctx = pbs.build_sparse_block_table_prefill(p.topk, p.page_table, p.cu_seqlens_q, p.seq_lens,
                                                        b.block_page_stride, err_word=err)
    torch.cuda.synchronize()
    return np_i32(sbt), np_i32(ctx), int(err.item())


def oracle_tables(b, part):
    if part == "dec":
        d = b.dec
        return oracle.build_sparse_block_table_decode(np_i32(d.topk), np_i32(d.page_table), np_i32(d.seq_lens),
                                                      d.decode_query_len, b.block_page_stride)
    p = b.pre
    return oracle.build_sparse_block_table_prefill(np_i32(p.topk), np_i32(p.page_table), np_i32(p.cu_seqlens_q),
                                                   np_i32(p.seq_lens), b.block_page_stride)


def gpu_attend(pbs, b, part, err=None, workspace="default", kernel=None, splits=None, cache_map=None,
               sparse_table=None):
    """The binding's call for one part; workspace "default" leaves the binding's own default
    (decode: none; prefill: the workspace the chosen kernel wants). kernel / splits / cache_map are
    the call's options; sparse_table an optional prebuilt (sparse_bt, sparse_ctx)."""
    kw = {} if isinstance(workspace, str) and workspace == "default" else {"workspace": workspace}
    kw.update(splits=splits, cache_map=cache_map, sparse_table=sparse_table)
    if part == "dec":
        d = b.dec
        out = pbs.sparse_decode_attention(d.q, b.cache, b.kv_dtype, b.num_kv_heads, d.topk, d.page_table,
                                          d.seq_lens, d.decode_query_len, b.softmax_scale, b.k_scale, b.v_scale,
                                          b.block_page_stride, err_word=err, **kw)
    else:
        p = b.pre
        out = pbs.sparse_prefill_attention(p.q, b.cache, b.kv_dtype, b.num_kv_heads, p.topk, p.page_table,
                                           p.cu_seqlens_q, p.seq_lens, b.softmax_scale, b.k_scale, b.v_scale,
                                           b.block_page_stride, err_word=err, kernel=kernel, **kw)
    torch.cuda.synchronize()
    return out.to(torch.float64).cpu().numpy()


# ------------------------------------------------------------------------------------------
# sparse block tables: bit-exact
# ------------------------------------------------------------------------------------------

def test_tables_tiny(pbs):
    b = workloads.tiny(device=DEV)
    for part in ("dec", "pre"):
        sbt, ctx, err = gpu_tables(pbs, b, part)
        o_sbt, o_ctx = oracle_tables(b, part)
        assert err == 0
        assert np.array_equal(sbt, o_sbt) and np.array_equal(ctx, o_ctx)


@pytest.mark.parametrize("case", [
    dict(dec_seq_lens=[0, 1, 127, 128, 129, 5000], topk=1),
    dict(dec_seq_lens=[300, 4000, 9000], decode_query_len=3, topk=7),
    dict(dec_seq_lens=[20000, 1500], topk=33),
    dict(dec_seq_lens=[70000, 30, 2000], topk=64),
    dict(pre_q_lens=[700, 0, 300, 1], pre_ctx_lens=[0, 5, 200, 4095], topk=16, future_prob=0.3),
])
def test_tables_small_variants(pbs, case):
    b = workloads.small(device=DEV, seed=21, **case)
    for part in ("dec", "pre"):
        if (part == "dec" and b.dec is None) or (part == "pre" and b.pre is None):
            continue
        sbt, ctx, err = gpu_tables(pbs, b, part)
        o_sbt, o_ctx = oracle_tables(b, part)
        assert err == 0
        assert np.array_equal(sbt, o_sbt), "sparse block table differs"
        assert np.array_equal(ctx, o_ctx), "context lengths differ"


def test_tables_duplicates_strides_and_side_packed(pbs):
    """Repeated ids (a row is a set of blocks: later repeats dropped, as the oracle reads it); a
    strided top-k view and block stride 16."""
    rng = np.random.default_rng(5)
    rows, k = 300, 12
    seq = rng.integers(1, 6000, size=rows).astype(np.int32)
    pos = seq - 1
    own = pos // 128
    topk = np.full((rows, k + 5), -7, np.int32)             # wider buffer: row stride k+5
    for r in range(rows):
        ids = rng.integers(-1, own[r] + 3, size=k)
        if r % 3 == 0:
            ids[1] = ids[0]                                  # duplicate
        if r % 5 == 0:
            ids[2] = own[r]
            ids[3] = own[r]                                  # duplicate own block
        topk[r, :k] = ids
    pt = rng.permutation(rows * 50).astype(np.int32).reshape(rows, 50)[:, :48]
    t_topk = torch.from_numpy(topk).to(DEV)[:, :k]
    t_pt = torch.from_numpy(np.ascontiguousarray(pt)).to(DEV)
    for bps in (8, 16):
        err = _err()
        sbt, ctx = pbs.build_sparse_block_table_decode(t_topk, t_pt, torch.from_numpy(seq).to(DEV), 1, bps,
                                                       err_word=err)
        o_sbt, o_ctx = oracle.build_sparse_block_table_decode(topk[:, :k], pt, seq, 1, bps)
        assert int(err.item()) == 0
        assert np.array_equal(np_i32(sbt), o_sbt) and np.array_equal(np_i32(ctx), o_ctx)


def test_table_block_past_page_table_sets_error(pbs):
    topk = torch.tensor([[[0, 3, -1]]], dtype=torch.int32, device=DEV)   # block 3 is causal but past the table
    pt = torch.tensor([[5, 6]], dtype=torch.int32, device=DEV)
    err = _err()
    sbt, ctx = pbs.build_sparse_block_table_decode(topk, pt, torch.tensor([500], dtype=torch.int32, device=DEV),
                                                   err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & pbs.DEVERR["block_oob"]
    assert int(ctx.item()) == 0 and int(sbt.abs().sum().item()) == 0


# ------------------------------------------------------------------------------------------
# attention
# ------------------------------------------------------------------------------------------

def test_attend_tiny_bf16(pbs):
    b = workloads.tiny(device=DEV)
    got = gpu_attend(pbs, b, "dec")
    want = oracle_decode(b)
    assert_close({0: got[0]}, want, "bf16", "tiny decode")
    got = gpu_attend(pbs, b, "pre")
    want = oracle_prefill(b)
    assert_close(dict(enumerate(got)), want, "bf16", "tiny prefill")


@pytest.mark.parametrize("workspace", [None, "auto"])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "nvfp4"])
@pytest.mark.parametrize("heads", [(64, 8), (32, 2), (16, 4), (8, 4), (4, 4)])
def test_attend_small_decode(pbs, kv_dtype, heads, workspace):
    hq, hkv = heads
    b = workloads.small(device=DEV, kv_dtype=kv_dtype, num_heads=hq, num_kv_heads=hkv, topk=9,
                        dec_seq_lens=[1, 129, 2000, 5000, 1170], decode_query_len=2, seed=31)
    got = gpu_attend(pbs, b, "dec", workspace=workspace)
    want = oracle_decode(b)
    assert_close(dict(enumerate(got)), want, kv_dtype, f"decode {kv_dtype} {heads}")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "nvfp4"])
def test_attend_small_prefill(pbs, kv_dtype):
    b = workloads.small(device=DEV, kv_dtype=kv_dtype, num_heads=64, num_kv_heads=8, topk=8,
                        pre_q_lens=[300, 1, 260], pre_ctx_lens=[0, 700, 1000], future_prob=0.3, seed=32)
    got = gpu_attend(pbs, b, "pre")
    want = oracle_prefill(b)
    assert_close(dict(enumerate(got)), want, kv_dtype, f"prefill {kv_dtype}")


@pytest.mark.parametrize("workspace", [None, "auto"])
@pytest.mark.parametrize("splits", ["1", "2", "4", "8"])
def test_attend_split_counts_agree(pbs, splits, workspace):
    """Every split count gives the oracle's answer, merged through a cluster's shared memory
    (no workspace) or through the workspace by the last chunk to finish."""
    b = workloads.small(device=DEV, num_heads=64, num_kv_heads=8, topk=16, dec_seq_lens=[3000, 9000, 700],
                        seed=33)
    got = gpu_attend(pbs, b, "dec", workspace=workspace, splits=int(splits))
    assert_close(dict(enumerate(got)), oracle_decode(b), "bf16", f"splits={splits} workspace={workspace}")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "nvfp4"])
def test_attend_workspace_leaves_tickets_zero(pbs, kv_dtype):
    """Two calls in a row on one caller workspace: both match the oracle, and each leaves the
    per-(row, kv head) arrival counters at zero for the next call."""
    b = workloads.small(device=DEV, kv_dtype=kv_dtype, num_heads=16, num_kv_heads=4, topk=16,
                        dec_seq_lens=[1, 2100, 7000, 0, 4000], decode_query_len=2, seed=38)
    rows, hkv = b.dec.q.shape[0], b.num_kv_heads
    nbytes = pbs.attend_workspace_bytes(rows, b.num_heads, hkv)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    want = oracle_decode(b)
    for call in range(2):
        got = gpu_attend(pbs, b, "dec", workspace=ws, splits=8)
        assert_close(dict(enumerate(got)), want, kv_dtype, f"workspace call {call}")
        assert int(ws[nbytes - rows * hkv * 4:].view(torch.int32).abs().sum()) == 0
    # a smaller call on the same buffer (its tickets sit in the same tail) still matches
    sub = workloads.small(device=DEV, kv_dtype=kv_dtype, num_heads=16, num_kv_heads=4, topk=16,
                          dec_seq_lens=[5000], decode_query_len=1, seed=40)
    got = gpu_attend(pbs, sub, "dec", workspace=ws, splits=8)
    assert_close(dict(enumerate(got)), oracle_decode(sub), kv_dtype, "smaller call after")
    assert int(ws[nbytes - rows * hkv * 4:].view(torch.int32).abs().sum()) == 0
    got = gpu_attend(pbs, b, "dec", workspace=ws, splits=8)
    assert_close(dict(enumerate(got)), want, kv_dtype, "larger call again")


def test_prefill_token_kernel_workspace_splits(pbs):
    """The token-centric prefill kernel with its splits merged through the workspace."""
    b = workloads.small(device=DEV, kv_dtype="fp8_e4m3", num_heads=64, num_kv_heads=8, topk=16,
                        pre_q_lens=[200, 1, 90], pre_ctx_lens=[3000, 700, 5000], future_prob=0.3, seed=39)
    ws = pbs.attend_workspace(b.pre.q.shape[0], b.num_heads, b.num_kv_heads, DEV)
    got = gpu_attend(pbs, b, "pre", workspace=ws, kernel="token", splits=4)
    assert_close(dict(enumerate(got)), oracle_prefill(b), "fp8_e4m3", "prefill workspace splits")


# log-sum-exp output: |lse - oracle| within this bound (logits are fp32 dot products of the
# stored values; ex2 / log2 round-off is far below it)
LSE_TOL = 2e-3


def _oracle_lse(b, part):
    if part == "dec":
        d = b.dec
        return oracle.sparse_decode_attention(q64(d.q), cache_source(b), b.kv_dtype, b.num_kv_heads, np_i32(d.topk),
                                              np_i32(d.page_table), np_i32(d.seq_lens), d.decode_query_len,
                                              b.softmax_scale, b.k_scale, b.v_scale, b.block_page_stride,
                                              return_lse=True)[1]
    p = b.pre
    return oracle.sparse_prefill_attention(q64(p.q), cache_source(b), b.kv_dtype, b.num_kv_heads, np_i32(p.topk),
                                           np_i32(p.page_table), np_i32(p.cu_seqlens_q), np_i32(p.seq_lens),
                                           b.softmax_scale, b.k_scale, b.v_scale, b.block_page_stride,
                                           return_lse=True)[1]


def _check_lse(got, want, what):
    got = got.double().cpu().numpy()
    for r, w in want.items():
        fin = np.isfinite(w)
        assert np.array_equal(np.isfinite(got[r]), fin), f"{what}: row {r} empty-row pattern"
        assert np.all(np.isneginf(got[r][~fin])), f"{what}: row {r} empty heads not -inf"
        if fin.any():
            err = float(np.abs(got[r][fin] - w[fin]).max())
            assert err <= LSE_TOL, f"{what}: row {r} lse error {err:.3g}"


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "nvfp4"])
@pytest.mark.parametrize("split", ["1", "4", "4ws"])
@pytest.mark.parametrize("heads", [(64, 8), (32, 2)])
def test_attend_lse_decode(pbs, kv_dtype, split, heads):
    """The optional log-sum-exp of every row and head, through each merge path."""
    b = workloads.small(device=DEV, kv_dtype=kv_dtype, num_heads=heads[0], num_kv_heads=heads[1], topk=16,
                        dec_seq_lens=[0, 129, 2000, 9000, 1170], decode_query_len=2, seed=60)
    d = b.dec
    out, lse = pbs.sparse_decode_attention(d.q, b.cache, kv_dtype, b.num_kv_heads, d.topk, d.page_table, d.seq_lens,
                                           d.decode_query_len, b.softmax_scale, b.k_scale, b.v_scale,
                                           workspace="auto" if split.endswith("ws") else None, return_lse=True,
                                           splits=int(split[0]))
    torch.cuda.synchronize()
    _check_lse(lse, _oracle_lse(b, "dec"), f"decode lse {kv_dtype} S={split} {heads}")
    assert_close(dict(enumerate(out.double().cpu().numpy())), oracle_decode(b), kv_dtype, "decode out with lse")


@pytest.mark.parametrize("kernel", ["tile", "token", "gather"])
@pytest.mark.parametrize("heads", [(64, 8), (32, 2)])
def test_attend_lse_prefill(pbs, kernel, heads):
    b = workloads.small(device=DEV, num_heads=heads[0], num_kv_heads=heads[1], topk=8, pre_q_lens=[37, 200, 1],
                        pre_ctx_lens=[0, 700, 3000], future_prob=0.3, seed=61)
    p = b.pre
    out, lse = pbs.sparse_prefill_attention(p.q, b.cache, "bf16", b.num_kv_heads, p.topk, p.page_table,
                                            p.cu_seqlens_q, p.seq_lens, b.softmax_scale, return_lse=True,
                                            workspace="auto" if kernel == "gather" else None, kernel=kernel)
    torch.cuda.synchronize()
    _check_lse(lse, _oracle_lse(b, "pre"), f"prefill lse {kernel} {heads}")


def test_attend_empty_rows_are_zero(pbs):
    b = workloads.small(device=DEV, num_heads=8, num_kv_heads=1, topk=4, dec_seq_lens=[0, 300, 0], seed=34)
    got = gpu_attend(pbs, b, "dec")
    assert np.all(got[0] == 0) and np.all(got[2] == 0)
    assert_close({1: got[1]}, oracle_decode(b, rows=[1]), "bf16", "row 1")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "nvfp4"])
def test_attend_ignores_nan_past_the_context(pbs, kv_dtype):
    """Cache rows past a query's position (unwritten in a live cache) may hold NaN; they are masked."""
    b = workloads.small(device=DEV, kv_dtype=kv_dtype, num_heads=8, num_kv_heads=2, topk=4,
                        dec_seq_lens=[200, 1000, 77], seed=35)
    d = b.dec
    pt = np_i32(d.page_table)
    for r, L in enumerate(np_i32(d.seq_lens)):
        for x in range(L, ((L + 127) // 128) * 128):
            page = int(pt[r, x // 128]) * 8 + (x % 128) // 16
            row = x % 16
            if kv_dtype == "nvfp4":
                pg = b.cache[page].view(2 * b.num_kv_heads, 1152)
                pg[:, row * 64:(row + 1) * 64] = 0xFF                # e2m1 -6 codes
                pg[:, 1024 + row * 8:1024 + (row + 1) * 8] = 0x7F    # e4m3 NaN scales
            else:
                view = b.cache[page].view(b.num_kv_heads, 16, -1)
                view[:, row, :] = 0xFF                               # NaN in bf16 and e4m3
    got = gpu_attend(pbs, b, "dec")
    assert_close(dict(enumerate(got)), oracle_decode(b), kv_dtype, "NaN past context")


def test_attend_page_past_cache_sets_error(pbs):
    b = workloads.small(device=DEV, num_heads=8, num_kv_heads=1, topk=4, dec_seq_lens=[300, 300], seed=36)
    d = b.dec
    pt = d.page_table.clone()
    pt[0, 0] = b.num_pages // 8 + 10                                # block beyond the cache
    err = _err()
    out = pbs.sparse_decode_attention(d.q, b.cache, "bf16", 1, d.topk, pt, d.seq_lens, 1, b.softmax_scale,
                                      err_word=err)
    torch.cuda.synchronize()
    tk = np_i32(d.topk)[0, 0]
    if 0 in tk:
        assert int(err.item()) & 2
        assert float(out[0].abs().sum()) == 0.0
    assert_close({1: out[1].double().cpu().numpy()}, oracle_decode(b, rows=[1]), "bf16", "row 1")


def test_strided_q_and_out(pbs):
    b = workloads.small(device=DEV, num_heads=16, num_kv_heads=2, topk=5, dec_seq_lens=[900, 1300], seed=37)
    d = b.dec
    big = torch.zeros(d.q.shape[0], 20, 128 + 64, dtype=torch.bfloat16, device=DEV)
    big[:, 2:18, 32:160] = d.q
    qv = big[:, 2:18, 32:160]
    outbig = torch.full((d.q.shape[0], 24, 256), 7.0, dtype=torch.bfloat16, device=DEV)
    ov = outbig[:, 4:20, 64:192]
    pbs.sparse_decode_attention(qv, b.cache, "bf16", 2, d.topk, d.page_table, d.seq_lens, 1, b.softmax_scale,
                                out=ov)
    torch.cuda.synchronize()
    assert_close(dict(enumerate(ov.double().cpu().numpy())), oracle_decode(b), "bf16", "strided")
    assert float(outbig[:, :4].double().sub(7).abs().sum()) == 0.0       # nothing written outside the view


# ------------------------------------------------------------------------------------------
# index-cache insert
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_insert_index_cache(pbs, dtype):
    g = torch.Generator(device=DEV)
    g.manual_seed(5)
    N, B, T, D = 4096, 300, 16, 128
    k = torch.randn(N, D, generator=g, device=DEV).to(dtype)
    cache = torch.randn(B, T, D, generator=g, device=DEV).to(dtype)
    slots = torch.randperm(B * T, generator=g, device=DEV)[:N].to(torch.int64)
    slots[::97] = -1
    want = oracle.insert_index_cache(k.float().cpu().numpy(), cache.float().cpu().numpy(), slots.cpu().numpy())
    err = _err()
    pbs.insert_index_cache(k, cache, slots, err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(cache.float().cpu().numpy(), want)


def test_insert_index_cache_slot_past_cache(pbs):
    k = torch.ones(2, 128, dtype=torch.bfloat16, device=DEV)
    cache = torch.zeros(2, 4, 128, dtype=torch.bfloat16, device=DEV)
    err = _err()
    pbs.insert_index_cache(k, cache, torch.tensor([1, 8], dtype=torch.int64, device=DEV), err_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 4
    assert float(cache[0, 1].sum()) == 128.0 and float(cache.sum()) == 128.0


# ------------------------------------------------------------------------------------------
# prefill: tcgen05 tile kernel and token-centric kernel
# ------------------------------------------------------------------------------------------

PREFILL_CASES = [
    dict(pre_q_lens=[37, 16, 1, 200], pre_ctx_lens=[0, 100, 5, 3000], topk=16),
    dict(pre_q_lens=[3] * 40, pre_ctx_lens=[i * 50 for i in range(40)], topk=8),   # > 32 requests
    dict(pre_q_lens=[500], pre_ctx_lens=[7], topk=12, future_prob=0.5),
    dict(pre_q_lens=[130, 260], pre_ctx_lens=[0, 0], topk=2),
    dict(pre_q_lens=[20, 0, 33, 0], pre_ctx_lens=[100, 500, 1300, 0], topk=8),   # requests without tokens
]


@pytest.mark.parametrize("heads", [(64, 8), (32, 2)])
@pytest.mark.parametrize("kernel", ["tile", "tile_hilo", "token", "gather"])
@pytest.mark.parametrize("ci", range(len(PREFILL_CASES)))
def test_prefill_kernels_agree_with_oracle(pbs, kernel, ci, heads):
    """Every prefill kernel, GQA 8 (tile = 16 tokens x 8 heads) and GQA 16 (8 tokens x 16 heads);
    tile_hilo: the tile kernel without a workspace (bf16 P as hi + lo instead of converted fp16 V)."""
    b = workloads.small(device=DEV, num_heads=heads[0], num_kv_heads=heads[1], seed=41 + ci, **PREFILL_CASES[ci])
    err = _err()
    got = gpu_attend(pbs, b, "pre", err, workspace=None if kernel == "tile_hilo" else "default",
                     kernel="tile" if kernel == "tile_hilo" else kernel)
    assert int(err.item()) == 0
    assert_close(dict(enumerate(got)), oracle_prefill(b), "bf16", f"prefill {kernel} case {ci}")


def _with_repeats(topk):
    """A copy of a top-k buffer [1, rows, k] in which rows repeat ids: slot 1 copies slot 0 in every
    row, and in every third row the last slot copies the row's largest id (often the own block)."""
    tk = topk.clone()
    tk[0, :, 1] = tk[0, :, 0]
    rows = torch.arange(0, tk.shape[1], 3, device=tk.device)
    tk[0, rows, -1] = tk[0, rows].max(dim=1).values
    return tk


@pytest.mark.parametrize("entry", ["dec", "dec_ws", "dec_split8", "dec_split8_ws", "tile", "tile_hilo", "token",
                                   "gather", "mixed"])
def test_repeated_ids_read_once_by_every_kernel(pbs, entry):
    """A top-k row is a set of blocks: rows with repeated full and own-block ids give the oracle's
    answer (each selected block read once) on every kernel and merge path, and the table builders
    write the oracle's table for them."""
    b = workloads.small(device=DEV, num_heads=64, num_kv_heads=8, topk=6, dec_seq_lens=[3000, 700, 9000, 129],
                        decode_query_len=2, pre_q_lens=[300, 40], pre_ctx_lens=[400, 2000], future_prob=0.2, seed=45)
    b.dec.topk = _with_repeats(b.dec.topk)
    b.pre.topk = _with_repeats(b.pre.topk)
    assert int((b.pre.topk[0, :, 0] >= 0).sum()) > 0
    err = _err()
    if entry.startswith("dec"):
        for part in ("dec", "pre"):
            sbt, ctx, terr = gpu_tables(pbs, b, part)
            o_sbt, o_ctx = oracle_tables(b, part)
            assert terr == 0 and np.array_equal(sbt, o_sbt) and np.array_equal(ctx, o_ctx)
        ws = "auto" if entry.endswith("_ws") else None
        got = gpu_attend(pbs, b, "dec", err, workspace=ws, splits=8 if "split8" in entry else None)
        want = oracle_decode(b)
    elif entry == "mixed":
        d, p = b.dec, b.pre
        out = pbs.sparse_mixed_attention(torch.cat([d.q, p.q]), b.cache, "bf16", 8, torch.cat([d.topk[0], p.topk[0]]),
                                         d.page_table, d.seq_lens, d.decode_query_len, p.page_table, p.cu_seqlens_q,
                                         p.seq_lens, b.softmax_scale, err_word=err)
        torch.cuda.synchronize()
        got = out.double().cpu().numpy()
        want = {**oracle_decode(b), **{d.q.shape[0] + r: v for r, v in oracle_prefill(b).items()}}
    else:
        kernel = "tile" if entry == "tile_hilo" else entry
        got = gpu_attend(pbs, b, "pre", err, workspace=None if entry == "tile_hilo" else "default", kernel=kernel)
        want = oracle_prefill(b)
    assert int(err.item()) == 0
    assert_close(dict(enumerate(got)), want, "bf16", f"repeated ids {entry}")


@pytest.mark.parametrize("workspace", ["default", None])
def test_prefill_tc_widest_page_table(pbs, workspace):
    """Contexts reaching block 127: the tile kernel's 128-bit block sets filled to the last bit."""
    b = workloads.small(device=DEV, num_heads=64, num_kv_heads=8, topk=16, pre_q_lens=[40, 17],
                        pre_ctx_lens=[16344, 9000], future_prob=0.2, seed=48)
    p = b.pre
    assert p.page_table.shape[1] <= 128 and int(p.seq_lens.max()) > 127 * 128
    err = _err()
    got = gpu_attend(pbs, b, "pre", err, workspace=workspace, kernel="tile")
    assert int(err.item()) == 0
    assert_close(dict(enumerate(got)), oracle_prefill(b), "bf16", "prefill widest table")


@pytest.mark.parametrize("workspace", ["default", None])
def test_prefill_tc_v_scales_across_blocks(pbs, workspace):
    """V blocks whose magnitudes differ by up to 2^40: on the converted-V path the tile kernel moves
    its exponent reference and rescales O by powers of two; outputs compared row-normalised."""
    b = workloads.small(device=DEV, num_heads=64, num_kv_heads=8, topk=8, pre_q_lens=[300, 40],
                        pre_ctx_lens=[900, 2000], seed=47)
    p = b.pre
    pt = np_i32(p.page_table)
    rng = np.random.default_rng(3)
    for r, L in enumerate(np_i32(p.seq_lens)):
        for blk in range((int(L) + 127) // 128):
            f = 2.0 ** int(rng.integers(-20, 21))
            for pg in range(8):
                page = int(pt[r, blk]) * b.block_page_stride + pg
                b.cache[page].view(b.num_kv_heads, 16, -1)[:, :, 256:].view(torch.bfloat16).mul_(f)
    err = _err()
    got = gpu_attend(pbs, b, "pre", err, workspace=workspace, kernel="tile")
    assert int(err.item()) == 0
    want = oracle_prefill(b)
    norm = {r: np.abs(want[r]).max() for r in want}
    assert_close({r: got[r] / norm[r] for r in want}, {r: want[r] / norm[r] for r in want}, "bf16",
                 "prefill V scales")


@pytest.mark.parametrize("kernel", ["tile", "gather"])
def test_prefill_tc_ignores_nan_past_last_token(pbs, kernel):
    b = workloads.small(device=DEV, num_heads=64, num_kv_heads=8, topk=8, pre_q_lens=[77, 200], pre_ctx_lens=[0, 50],
                        seed=46)
    p = b.pre
    pt = np_i32(p.page_table)
    for r, L in enumerate(np_i32(p.seq_lens)):
        for x in range(L, ((L + 127) // 128) * 128):
            page = int(pt[r, x // 128]) * 8 + (x % 128) // 16
            b.cache[page].view(b.num_kv_heads, 16, -1)[:, x % 16, :] = 0xFF
    err = _err()
    got = gpu_attend(pbs, b, "pre", err, kernel=kernel)
    assert int(err.item()) == 0
    assert_close(dict(enumerate(got)), oracle_prefill(b), "bf16", "prefill NaN past the end")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_attend_per_quarter_map(pbs, kv_dtype):
    """The token-centric kernel on the per-quarter (4-D) cache map as well as the packed one."""
    b = workloads.small(device=DEV, kv_dtype=kv_dtype, num_heads=64, num_kv_heads=8, topk=9,
                        dec_seq_lens=[129, 2000, 5000], decode_query_len=2, pre_q_lens=[50, 200],
                        pre_ctx_lens=[900, 0], seed=51)
    assert_close(dict(enumerate(gpu_attend(pbs, b, "dec", cache_map="quarter"))), oracle_decode(b), kv_dtype,
                 "decode 4-D map")
    assert_close(dict(enumerate(gpu_attend(pbs, b, "pre", kernel="token", cache_map="quarter"))), oracle_prefill(b),
                 kv_dtype, "prefill 4-D map")


@pytest.mark.parametrize("kv_dtype,prefill_kernel", [("bf16", "tile"), ("bf16", "token"), ("fp8_e4m3", None),
                                                     ("fp8_e4m3", "token"), ("nvfp4", None), ("nvfp4", "token")])
def test_mixed_batch_in_one_call(pbs, kv_dtype, prefill_kernel):
    """Decode rows then prefill tokens through pbs_sparse_mixed_attention: one fused launch of the
    token-centric kernel, or decode + tile kernel when the prefill part takes the tile kernel (the
    default here, with the binding's workspace: fp8 / NVFP4 parts through converted K / V images);
    outputs and log-sum-exp against the oracle's decode and prefill attends."""
    b = workloads.small(device=DEV, kv_dtype=kv_dtype, num_heads=64, num_kv_heads=8, topk=12,
                        dec_seq_lens=[2500, 0, 9000], decode_query_len=2, pre_q_lens=[150, 1, 60],
                        pre_ctx_lens=[0, 900, 2000], future_prob=0.3, seed=54)
    d, p = b.dec, b.pre
    nd = d.q.shape[0]
    q = torch.cat([d.q, p.q])
    topk = torch.cat([d.topk[0], p.topk[0]])
    out, lse = pbs.sparse_mixed_attention(q, b.cache, kv_dtype, b.num_kv_heads, topk, d.page_table, d.seq_lens,
                                          d.decode_query_len, p.page_table, p.cu_seqlens_q, p.seq_lens,
                                          b.softmax_scale, b.k_scale, b.v_scale, return_lse=True, kernel=prefill_kernel)
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    assert_close(dict(enumerate(got[:nd])), oracle_decode(b), kv_dtype, "mixed: decode rows")
    assert_close(dict(enumerate(got[nd:])), oracle_prefill(b), kv_dtype, "mixed: prefill rows")
    _check_lse(lse[:nd], _oracle_lse(b, "dec"), "mixed lse decode")
    _check_lse(lse[nd:], _oracle_lse(b, "pre"), "mixed lse prefill")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "nvfp4"])
def test_attend_topk_64_and_padded_topk_rows(pbs, kv_dtype):
    """The largest top-k the boundary accepts (64), four query rows per decode request, and top-k
    rows read through a padded row stride (a [rows, 80] buffer viewed as [rows, 64])."""
    b = workloads.small(device=DEV, kv_dtype=kv_dtype, num_heads=16, num_kv_heads=2, topk=64,
                        dec_seq_lens=[9000, 300, 20000], decode_query_len=4, pre_q_lens=[100, 30],
                        pre_ctx_lens=[12000, 0], future_prob=0.3, seed=55)
    for part in ("dec", "pre"):
        src = b.dec if part == "dec" else b.pre
        padded = torch.full((src.topk.shape[1], 80), -1, dtype=torch.int32, device=DEV)
        padded[:, :64] = src.topk[0]
        src.topk = padded[:, :64]
        got = gpu_attend(pbs, b, part)
        want = oracle_decode(b) if part == "dec" else oracle_prefill(b)
        assert_close(dict(enumerate(got)), want, kv_dtype, f"top-k 64 {part}")


@pytest.mark.parametrize("part", ["dec", "tile", "token", "gather"])
def test_attend_side_packed_blocks(pbs, part):
    """block_page_stride 16 ([sparse_pa] minimax_m3_sparse_block_page_stride with packed sides):
    block b's pages are 16 b + j, j < 8; the other 8 pages of each block hold NaN and must not be
    read."""
    b = workloads.small(device=DEV, num_heads=64, num_kv_heads=8, topk=8, dec_seq_lens=[3000, 700],
                        pre_q_lens=[200, 40], pre_ctx_lens=[900, 0], future_prob=0.3, seed=53)
    nblk = b.num_pages // 8
    wide = torch.full((nblk * 16, b.page_bytes), 0xFF, dtype=torch.uint8, device=DEV)
    wide.view(nblk, 16, -1)[:, :8] = b.cache.view(nblk, 8, -1)
    b.cache = wide
    b.block_page_stride = 16
    err = _err()
    got = gpu_attend(pbs, b, "dec" if part == "dec" else "pre", err, kernel=None if part == "dec" else part)
    assert int(err.item()) == 0
    want = oracle_decode(b) if part == "dec" else oracle_prefill(b)
    assert_close(dict(enumerate(got)), want, "bf16", f"side-packed {part}")


def test_attend_strided_pages(pbs):
    """A cache whose pages are not back to back (page stride > content) uses the 4-D map."""
    b = workloads.small(device=DEV, num_heads=16, num_kv_heads=2, topk=6, dec_seq_lens=[700, 1500], seed=52)
    wide = torch.zeros(b.num_pages, b.page_bytes + 4096, dtype=torch.uint8, device=DEV)
    wide[:, :b.page_bytes] = b.cache
    view = wide[:, :b.page_bytes]
    d = b.dec
    out = pbs.sparse_decode_attention(d.q, view, "bf16", 2, d.topk, d.page_table, d.seq_lens, 1, b.softmax_scale)
    torch.cuda.synchronize()
    assert_close(dict(enumerate(out.double().cpu().numpy())), oracle_decode(b), "bf16", "strided pages")


def test_prefill_gather_segments_and_reuse(pbs):
    """The gathered-row kernel on a workspace that holds one 512-token segment runs the call in
    segments; each token's partials and merge do not depend on the segment, so the output is
    bit-identical to the one-segment run on a larger workspace, and a second call on the same
    (now stale) workspace gives the same bits again."""
    b = workloads.small(device=DEV, num_heads=64, num_kv_heads=8, topk=16, pre_q_lens=[700, 3, 300, 260],
                        pre_ctx_lens=[1500, 0, 6000, 128], future_prob=0.3, seed=70)
    p = b.pre
    nreq, k, mb = p.seq_lens.shape[0], p.topk.shape[-1], p.page_table.shape[1]
    small = pbs.prefill_workspace_bytes(512, nreq, 64, 8, k, mb)
    full = pbs.prefill_workspace_bytes(p.q.shape[0], nreq, 64, 8, k, mb)
    assert 0 < small < full
    outs = []
    for nbytes in (full, small, small):
        ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device=DEV)   # stale contents: all NaN
        err = _err()
        outs.append(gpu_attend(pbs, b, "pre", err, workspace=ws, kernel="gather"))
        assert int(err.item()) == 0
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])
    assert_close(dict(enumerate(outs[0])), oracle_prefill(b), "bf16", "gather segments")


# ------------------------------------------------------------------------------------------
# prebuilt sparse tables: built once, shared by the attends of several layers
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("entry", ["dec", "dec_ws", "dec_split4", "pre_token", "pre_tile", "pre_tile_hilo", "mixed"])
def test_prebuilt_table_shared_by_two_layers(pbs, entry):
    """The tables are built once with the builders ([sparse_pa] minimax_m3_build_sparse_block_table_*)
    and fed to the attends of two "layers" (different queries, one selection). Each table-fed call
    matches the oracle and is bit-identical to the same kernel compacting from top-k itself."""
    b = workloads.small(device=DEV, num_heads=64, num_kv_heads=8, topk=8, dec_seq_lens=[3000, 700, 9000, 0],
                        decode_query_len=2, pre_q_lens=[300, 40, 17], pre_ctx_lens=[400, 2000, 0], future_prob=0.3,
                        seed=80)
    d, p = b.dec, b.pre
    sbt_d, ctx_d = pbs.build_sparse_block_table_decode(d.topk, d.page_table, d.seq_lens, d.decode_query_len)
    sbt_p, ctx_p = pbs.build_sparse_block_table_prefill(p.topk, p.page_table, p.cu_seqlens_q, p.seq_lens)
    g = torch.Generator(device=DEV)
    g.manual_seed(81)
    for layer in range(2):
        if layer == 1:  # the next layer: new queries, the same selection and tables
            d.q = torch.randn(d.q.shape, generator=g, device=DEV).to(torch.bfloat16)
            p.q = torch.randn(p.q.shape, generator=g, device=DEV).to(torch.bfloat16)
        err = _err()
        if entry == "mixed":
            nd = d.q.shape[0]
            args = (torch.cat([d.q, p.q]), b.cache, "bf16", 8, torch.cat([d.topk[0], p.topk[0]]), d.page_table,
                    d.seq_lens, d.decode_query_len, p.page_table, p.cu_seqlens_q, p.seq_lens, b.softmax_scale)
            # the prefill part on the tile kernel in both calls (the gathered rows read top-k only)
            fused = pbs.sparse_mixed_attention(*args, kernel="tile")
            tabled = pbs.sparse_mixed_attention(*args, err_word=err, kernel="tile",
                                                sparse_table=(torch.cat([sbt_d, sbt_p]), torch.cat([ctx_d, ctx_p])))
            torch.cuda.synchronize()
            fused, tabled = fused.double().cpu().numpy(), tabled.double().cpu().numpy()
            want = {**oracle_decode(b), **{nd + r: v for r, v in oracle_prefill(b).items()}}
        elif entry.startswith("dec"):
            kw = dict(workspace="auto" if entry == "dec_ws" else None, splits=4 if entry == "dec_split4" else None)
            fused = gpu_attend(pbs, b, "dec", **kw)
            tabled = gpu_attend(pbs, b, "dec", err, sparse_table=(sbt_d, ctx_d), **kw)
            want = oracle_decode(b)
        else:
            kernel = "token" if entry == "pre_token" else "tile"
            ws = None if entry == "pre_tile_hilo" else "default"
            fused = gpu_attend(pbs, b, "pre", workspace=ws, kernel=kernel)
            tabled = gpu_attend(pbs, b, "pre", err, workspace=ws, kernel=kernel, sparse_table=(sbt_p, ctx_p))
            want = oracle_prefill(b)
        assert int(err.item()) == 0
        assert np.array_equal(fused, tabled), f"{entry} layer {layer}: table-fed call differs from the fused one"
        assert_close(dict(enumerate(tabled)), want, "bf16", f"prebuilt table {entry} layer {layer}")


@pytest.mark.parametrize("kernel", ["dec", "token", "tile"])
def test_prebuilt_table_unreadable_rows(pbs, kernel):
    """A ctx past top-k x 128 (every kernel), or a slot that names no block of the request's page table
    (the tile kernel, which streams whole blocks), sets PBS_DEVERR_TABLE and the row attends nothing;
    the other rows are unaffected."""
    b = workloads.small(device=DEV, num_heads=64, num_kv_heads=8, topk=4, dec_seq_lens=[900, 1500],
                        pre_q_lens=[20], pre_ctx_lens=[700], seed=82)
    part = "dec" if kernel == "dec" else "pre"
    src = b.dec if part == "dec" else b.pre
    if part == "dec":
        sbt, ctx = pbs.build_sparse_block_table_decode(src.topk, src.page_table, src.seq_lens, 1)
    else:
        sbt, ctx = pbs.build_sparse_block_table_prefill(src.topk, src.page_table, src.cu_seqlens_q, src.seq_lens)
    ctx[0] = 4 * 128 + 1
    if kernel == "tile":
        sbt[1, 0] += 1                     # slot 0 of row 1 no longer starts a block
    err = _err()
    got = gpu_attend(pbs, b, part, err, kernel=None if kernel == "dec" else kernel, sparse_table=(sbt, ctx))
    assert int(err.item()) & pbs.DEVERR["table"]
    assert np.all(got[0] == 0)
    bad = {0, 1} if kernel == "tile" else {0}
    if kernel == "tile":
        assert np.all(got[1] == 0)
    want = oracle_decode(b) if part == "dec" else oracle_prefill(b)
    assert_close({r: got[r] for r in want if r not in bad}, {r: v for r, v in want.items() if r not in bad}, "bf16",
                 "rows beside the unreadable ones")


# ------------------------------------------------------------------------------------------
# tile kernel: fp8 / NVFP4 caches through converted images; long contexts; two-part unions
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("kernel", ["tile", "gather"])
@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3", "nvfp4"])
@pytest.mark.parametrize("heads", [(64, 8), (32, 2)])
@pytest.mark.parametrize("ci", range(len(PREFILL_CASES)))
def test_prefill_tc_kernels_fp8_nvfp4(pbs, kv_dtype, heads, ci, kernel):
    """fp8 and NVFP4 caches on both tcgen05 prefill kernels: K converted to bf16 and V to fp16
    images once per (request, block, kv head), both exact, then the same pipelines as bf16."""
    b = workloads.small(device=DEV, kv_dtype=kv_dtype, num_heads=heads[0], num_kv_heads=heads[1], seed=141 + ci,
                        **PREFILL_CASES[ci])
    err = _err()
    got = gpu_attend(pbs, b, "pre", err, kernel=kernel)
    assert int(err.item()) == 0
    assert_close(dict(enumerate(got)), oracle_prefill(b), kv_dtype, f"{kernel} {kv_dtype} case {ci}")


def _largest_tile_union(b, tok):
    """Distinct valid blocks of the first `tok` tokens of each request (one tile each)."""
    p = b.pre
    tk = np_i32(p.topk)[0]
    cu = np_i32(p.cu_seqlens_q)
    sl = np_i32(p.seq_lens)
    best = 0
    for r in range(len(sl)):
        ctx = int(sl[r]) - int(cu[r + 1] - cu[r])
        blocks = set()
        for t in range(int(cu[r]), min(int(cu[r]) + tok, int(cu[r + 1]))):
            pos = ctx + t - int(cu[r])
            blocks.update(int(x) for x in tk[t] if 0 <= x <= pos // 128)
        best = max(best, len(blocks))
    return best


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "nvfp4"])
@pytest.mark.parametrize("heads", [(64, 8), (32, 2)])
def test_prefill_tile_long_context_two_part_unions(pbs, kv_dtype, heads):
    """Page tables far wider than 128 blocks (contexts of 30k-41k keys) and tiles whose union of
    selected blocks exceeds one descriptor's 128 entries, so a tile continues in a second descriptor
    (O and the softmax state carried over); with and without the workspace (bf16), and fed the
    prebuilt table (bit-identical to the self-compacting call)."""
    b = workloads.small(device=DEV, kv_dtype=kv_dtype, num_heads=heads[0], num_kv_heads=heads[1], topk=16,
                        pre_q_lens=[40, 17, 3], pre_ctx_lens=[30000, 41000, 2000], future_prob=0.05, seed=150)
    p = b.pre
    assert p.page_table.shape[1] > 128
    tok = 16 if heads == (64, 8) else 8
    if tok == 16:
        assert _largest_tile_union(b, tok) > 128
    want = oracle_prefill(b)
    for ws in (("default", None) if kv_dtype == "bf16" else ("default",)):
        err = _err()
        got = gpu_attend(pbs, b, "pre", err, workspace=ws, kernel="tile")
        assert int(err.item()) == 0
        assert_close(dict(enumerate(got)), want, kv_dtype, f"tile long context {kv_dtype} workspace={ws}")
        tbl = pbs.build_sparse_block_table_prefill(p.topk, p.page_table, p.cu_seqlens_q, p.seq_lens)
        tabled = gpu_attend(pbs, b, "pre", err, workspace=ws, kernel="tile", sparse_table=tbl)
        assert int(err.item()) == 0
        assert np.array_equal(got, tabled), "table-fed tile call differs from the fused one"
    # the gathered-row kernel on the same long contexts (its buckets hold a few tokens each)
    err = _err()
    got = gpu_attend(pbs, b, "pre", err, kernel="gather")
    assert int(err.item()) == 0
    assert_close(dict(enumerate(got)), want, kv_dtype, f"gather long context {kv_dtype}")
