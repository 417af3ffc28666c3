"""Test plumbing shared by the parity tests: page readers for the oracle, oracle calls on a
workloads.Batch, and the error metrics. Holds none of the attend's arithmetic."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# max-abs / relative-RMS bars on bf16 outputs against the fp64 oracle (bf16 KV), and for fp8 /
# NVFP4 KV against the oracle run on the same dequantised values.
TOL = {"bf16": (1e-2, 2e-3), "fp8_e4m3": (5e-2, 1e-2), "nvfp4": (5e-2, 1e-2)}


class DevicePages:
    """cache[ids] for the oracle, copying only the requested pages from a device tensor."""

    def __init__(self, cache: torch.Tensor):
        self.cache = cache

    def __getitem__(self, ids):
        idx = torch.from_numpy(np.asarray(ids, dtype=np.int64)).to(self.cache.device)
        return self.cache.index_select(0, idx).cpu().numpy()


def np_i32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def q64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().to(torch.float64).numpy()


def cache_source(b):
    return DevicePages(b.cache) if b.cache.is_cuda else b.cache.numpy()


def oracle_decode(b, rows=None):
    d = b.dec
    return oracle.sparse_decode_attention(q64(d.q), cache_source(b), b.kv_dtype, b.num_kv_heads, np_i32(d.topk),
                                          np_i32(d.page_table), np_i32(d.seq_lens), d.decode_query_len,
                                          b.softmax_scale, b.k_scale, b.v_scale, b.block_page_stride, rows=rows)


def oracle_prefill(b, rows=None):
    p = b.pre
    return oracle.sparse_prefill_attention(q64(p.q), cache_source(b), b.kv_dtype, b.num_kv_heads, np_i32(p.topk),
                                           np_i32(p.page_table), np_i32(p.cu_seqlens_q), np_i32(p.seq_lens),
                                           b.softmax_scale, b.k_scale, b.v_scale, b.block_page_stride, rows=rows)


def errors(got: np.ndarray, want: np.ndarray):
    """(max-abs error, relative RMS error) over all elements."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    diff = got - want
    denom = np.sqrt(np.sum(want * want))
    rel = float(np.sqrt(np.sum(diff * diff)) / denom) if denom > 0 else float(np.sqrt(np.sum(diff * diff)))
    return float(np.max(np.abs(diff))) if diff.size else 0.0, rel


def assert_close(got_rows: dict, want_rows: dict, kv_dtype: str, what: str = ""):
    rows = sorted(want_rows)
    got = np.stack([got_rows[r] for r in rows])
    want = np.stack([want_rows[r] for r in rows])
    mx, rel = errors(got, want)
    tmax, trel = TOL[kv_dtype]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert mx <= tmax and rel <= trel, f"{what}: max-abs {mx:.3e} (bar {tmax}), rel-RMS {rel:.3e} (bar {trel})"
    return mx, rel
