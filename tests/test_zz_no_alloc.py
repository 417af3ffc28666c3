"""The no-allocation decode entry (pbs_sparse_decode_attention_noalloc): the split attend with its
partials and arrival tickets in the library's fixed device scratch instead of a caller workspace.

Its output is checked against the workspace entry point (the same kernel with the same split
count) and against the fp64 oracle, within the parity tolerances, on two calls in a row: the
second call only works if the first one left the scratch's tickets at zero. Cases cover GQA 8,
GQA 16 (two head groups per kv head, so units sit at row * 16 + head group) and two right-aligned
query rows per request. The file is named to be collected last, and its tests depend on no state
that earlier tests leave behind."""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from helpers import TOL, assert_close, oracle_decode

DEV = "cuda"


@pytest.fixture(scope="module")
def pbs():
    from paged_block_sparse_gb300 import _build
    _build.build()
    import paged_block_sparse_gb300 as m
    return m


def _errors(got: np.ndarray, want: np.ndarray):
    diff = got - want
    return float(np.abs(diff).max()), float(np.sqrt((diff ** 2).mean() / max((want ** 2).mean(), 1e-300)))


# (query heads, kv heads, decode_query_len, sequence lengths): each has 48 (row, head group)
# units with top-k 16, so the call splits each row 8 ways (384 partials, under the 1004 limit)
CASES = [
    (64, 8, 1, [9000, 2048, 31000, 130, 16500, 5000]),     # GQA 8
    (64, 4, 1, [9000, 2048, 31000, 130, 16500, 5000]),     # GQA 16: two head groups of 8 per kv head
    (64, 8, 2, [9000, 31000, 130]),                        # two right-aligned rows per request
]


@pytest.mark.gpu
@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3", "nvfp4"])
def test_noalloc_matches_workspace_entry_twice(pbs, kv_dtype, case):
    hq, hkv, dql, seqs = CASES[case]
    b = workloads.small(device=DEV, kv_dtype=kv_dtype, num_heads=hq, num_kv_heads=hkv, topk=16,
                        dec_seq_lens=seqs, decode_query_len=dql, seed=51 + case)
    d = b.dec
    args = (d.q, b.cache, kv_dtype, b.num_kv_heads, d.topk, d.page_table, d.seq_lens, d.decode_query_len,
            b.softmax_scale)
    ws = torch.zeros(pbs.attend_workspace_bytes(d.q.shape[0], b.num_heads, b.num_kv_heads), dtype=torch.uint8,
                     device=DEV)
    want = pbs.sparse_decode_attention(*args, b.k_scale, b.v_scale, workspace=ws)
    torch.cuda.synchronize()
    want = want.double().cpu().numpy()
    oracle_rows = oracle_decode(b)
    tmax, trel = TOL[kv_dtype]
    out = torch.empty_like(d.q)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for call in range(2):
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        before = (torch.cuda.memory_allocated(), torch.cuda.memory_reserved())
        pbs.sparse_decode_attention_noalloc(*args, out=out, k_scale=b.k_scale, v_scale=b.v_scale, err_word=err)
        torch.cuda.synchronize()
        assert (torch.cuda.memory_allocated(), torch.cuda.memory_reserved()) == before
        got = out.double().cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}: rows left unwritten"
        mx, rel = _errors(got, want)
        assert mx <= tmax and rel <= trel, f"call {call}: max-abs {mx:.3g} rel-rms {rel:.3g}"
        assert_close(dict(enumerate(got)), oracle_rows, kv_dtype, f"no-allocation call {call} against the oracle")
    assert int(err.item()) == 0


@pytest.mark.gpu
def test_noalloc_refuses_what_the_scratch_cannot_hold(pbs):
    # 20 rows x 8 kv heads forced to 8 splits = 1280 partials > 1004: refused before any launch
    b = workloads.small(device=DEV, num_heads=64, num_kv_heads=8, topk=16, dec_seq_lens=[4000] * 20, seed=52)
    d = b.dec
    out = torch.zeros_like(d.q)
    with pytest.raises(pbs.PbsError) as e:
        pbs.sparse_decode_attention_noalloc(d.q, b.cache, "bf16", 8, d.topk, d.page_table, d.seq_lens, 1,
                                            b.softmax_scale, out=out, splits=8)
    assert e.value.status == 6
    torch.cuda.synchronize()
    assert float(out.abs().sum()) == 0.0


def test_noalloc_binding_requires_out():
    import paged_block_sparse_gb300 as pbs
    with pytest.raises(ValueError):
        pbs.sparse_decode_attention_noalloc(None, None, "bf16", 8, None, None, None, 1, 0.1, out=None)


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-check tests use fake device addresses")
def test_noalloc_host_checks(pbs):
    """Argument checks run before the scratch lookup, so they need no GPU."""
    L = pbs.lib()
    A, N = ctypes.c_void_p(0x10000), ctypes.c_void_p(0)

    def call(**kw):
        a = dict(q=A, hd=128, batch=4, hq=64, hkv=8)
        a.update(kw)
        return L.pbs_sparse_decode_attention_noalloc(a["q"], 1024, 128, A, 65536, 100, 0, a["hq"], a["hkv"], a["hd"],
                                                     A, 16, 16, A, 64, 64, A, a["batch"], 1, 8, 0.088, 1.0, 1.0,
                                                     A, 8192, 128, N, N, N)

    assert call(hd=64) == 3
    assert call(q=N) == 1
    assert call(hq=60) == 2
    assert call(batch=0) == 0
    assert pbs.status_string(6).startswith("request needs more than the fixed no-allocation scratch")
