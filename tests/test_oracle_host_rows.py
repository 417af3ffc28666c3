"""The host-core timing driver of the oracle (oracle/host_rows.py): its spawn-started workers
load their rows and pages, run the oracle for a time budget and report, and the pool closes."""
import numpy as np
import torch

import workloads
from oracle.host_rows import DecodeRowPool, host_cores


def _row_pages(b):
    d = b.dec
    tk = d.topk.numpy()
    pt = d.page_table.numpy()
    out = []
    for r in range(d.q.shape[0]):
        req = r // d.decode_query_len
        blocks = sorted({int(x) for x in tk[0, r] if 0 <= x < pt.shape[1]})
        pages = [int(pt[req, x]) * b.block_page_stride + j for x in blocks for j in range(8)]
        out.append({pg: b.cache[pg].numpy() for pg in pages})
    return out


def test_pool_runs_the_oracle_on_two_workers():
    b = workloads.small(num_heads=16, num_kv_heads=2, topk=4, dec_seq_lens=[700, 3000, 1500],
                        decode_query_len=2, pre_q_lens=[], pre_ctx_lens=[], seed=3)
    d = b.dec
    assert host_cores() >= 1
    with DecodeRowPool(2, _row_pages(b), q=d.q.to(torch.float64).numpy(), kv_dtype=b.kv_dtype,
                       num_kv_heads=b.num_kv_heads, topk=d.topk.numpy(), page_table=d.page_table.numpy(),
                       seq_lens=d.seq_lens.numpy(), decode_query_len=d.decode_query_len,
                       softmax_scale=b.softmax_scale, k_scale=b.k_scale, v_scale=b.v_scale,
                       block_page_stride=b.block_page_stride, timeout_s=120.0) as pool:
        assert pool.workers == 2
        for _ in range(2):
            rate, done, t = pool.run(0.2)
            assert done >= 2 and t >= 0.2 and np.isfinite(rate) and rate > 0
    assert pool.procs == []
