"""Parity at the full workload sizes, in the launch configuration bench.py times: every row of the
sparse block tables bit-exact, attention on seeded samples of rows (the oracle computes them one
by one; pages are copied to the host on demand)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import assert_close, np_i32, oracle_decode, oracle_prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pbs():
    from paged_block_sparse_gb300 import _build
    _build.build()
    import paged_block_sparse_gb300 as m
    return m


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    picks = set(rng.choice(n, size=min(k, n), replace=False).tolist())
    picks.update({0, n - 1})
    return sorted(picks)


def _check_tables(pbs, b):
    if b.dec is not None:
        d = b.dec
        sbt, ctx = pbs.build_sparse_block_table_decode(d.topk, d.page_table, d.seq_lens, d.decode_query_len)
        o_sbt, o_ctx = oracle.build_sparse_block_table_decode(np_i32(d.topk), np_i32(d.page_table),
                                                              np_i32(d.seq_lens), d.decode_query_len)
        assert np.array_equal(np_i32(sbt), o_sbt) and np.array_equal(np_i32(ctx), o_ctx)
    if b.pre is not None:
        p = b.pre
        sbt, ctx = pbs.build_sparse_block_table_prefill(p.topk, p.page_table, p.cu_seqlens_q, p.seq_lens)
        o_sbt, o_ctx = oracle.build_sparse_block_table_prefill(np_i32(p.topk), np_i32(p.page_table),
                                                               np_i32(p.cu_seqlens_q), np_i32(p.seq_lens))
        assert np.array_equal(np_i32(sbt), o_sbt) and np.array_equal(np_i32(ctx), o_ctx)


def _decode_parity(pbs, b, nrows, seed):
    d = b.dec
    out = pbs.sparse_decode_attention(d.q, b.cache, b.kv_dtype, b.num_kv_heads, d.topk, d.page_table, d.seq_lens,
                                      d.decode_query_len, b.softmax_scale, b.k_scale, b.v_scale)
    torch.cuda.synchronize()
    rows = _sample(d.q.shape[0], nrows, seed)
    want = oracle_decode(b, rows=rows)
    got = {r: out[r].double().cpu().numpy() for r in rows}
    return assert_close(got, want, b.kv_dtype, b.name)


def _prefill_parity(pbs, b, nrows, seed, workspace="auto", kernel=None):
    p = b.pre
    out = pbs.sparse_prefill_attention(p.q, b.cache, b.kv_dtype, b.num_kv_heads, p.topk, p.page_table,
                                       p.cu_seqlens_q, p.seq_lens, b.softmax_scale, b.k_scale, b.v_scale,
                                       workspace=workspace, kernel=kernel)
    torch.cuda.synchronize()
    rows = _sample(p.q.shape[0], nrows, seed)
    want = oracle_prefill(b, rows=rows)
    got = {r: out[r].double().cpu().numpy() for r in rows}
    return assert_close(got, want, b.kv_dtype, b.name)


def test_decode_b64_bf16(pbs):
    b = workloads.decode(device="cuda")
    _check_tables(pbs, b)
    _decode_parity(pbs, b, 24, 1)


def test_prefill_varlen_bf16(pbs):
    b = workloads.prefill(device="cuda")
    _check_tables(pbs, b)
    _prefill_parity(pbs, b, 48, 2)


def test_prefill_varlen_bf16_gathered(pbs):
    """The gathered-row prefill kernel at full size (several token segments on the default
    2 GiB workspace), sampled rows against the oracle."""
    b = workloads.prefill(device="cuda")
    _prefill_parity(pbs, b, 48, 6, kernel="gather")


def test_mtp_fp8(pbs):
    b = workloads.mtp_fp8(device="cuda")
    _check_tables(pbs, b)
    _decode_parity(pbs, b, 16, 3)
    del b
    torch.cuda.empty_cache()


def test_mixed_nvfp4(pbs):
    b = workloads.mixed_nvfp4(device="cuda")
    _check_tables(pbs, b)
    _decode_parity(pbs, b, 12, 4)
    # the prefill part as the binding runs it by default: the tcgen05 tile kernel (NVFP4 K / V
    # converted to bf16 / fp16 images; contexts of 16k and 32k keys: page tables of 160 and 288
    # blocks), and on the token-centric kernel
    _prefill_parity(pbs, b, 24, 5)
    _prefill_parity(pbs, b, 24, 8, kernel="token")
    del b
    torch.cuda.empty_cache()
