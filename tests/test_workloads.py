"""Sanity of the seeded generators (shapes, top-k draw rules, page-table injectivity)."""
import numpy as np
import torch

import workloads


def test_tiny_shapes_and_rules():
    b = workloads.tiny()
    assert b.cache.shape == (64, 1 * 16 * 256 * 2)
    tk = b.pre.topk[0].numpy()
    assert tk.shape == (1024, 4)
    for t in range(1024):
        own = t // 128
        ids = [x for x in tk[t] if x >= 0]
        assert own in ids and len(set(ids)) == len(ids) and max(ids) <= own
        assert len(ids) == min(4, own + 1)
    assert sorted(b.pre.page_table[0].tolist()) == list(range(8))
    assert torch.equal(b.dec.topk[0, 0], b.pre.topk[0, 1023])


def test_prefill_rules_small():
    b = workloads.small(pre_q_lens=[700, 300], pre_ctx_lens=[0, 200], topk=8, future_prob=0.3)
    tk = b.pre.topk[0].numpy()
    cu = b.pre.cu_seqlens_q.tolist()
    assert cu == [0, 700, 1000]
    assert b.pre.seq_lens.tolist() == [700, 500]
    fut = 0
    for t in range(tk.shape[0]):
        r = 0 if t < 700 else 1
        pos = t if r == 0 else 200 + (t - 700)
        own = pos // 128
        assert own in tk[t]
        fut += int((tk[t] > own).sum())
    assert fut > 0


def test_page_tables_injective():
    b = workloads.small(dec_seq_lens=[1000, 3000], pre_q_lens=[500], topk=4)
    ids = []
    for pt, lens in ((b.dec.page_table, b.dec.seq_lens), (b.pre.page_table, b.pre.seq_lens)):
        for r in range(pt.shape[0]):
            nb = -(-int(lens[r]) // 128)
            ids += pt[r, :nb].tolist()
    assert len(ids) == len(set(ids))
    assert max(ids) * 8 + 7 < b.num_pages


def test_nvfp4_codes_roundtrip_range():
    b = workloads.small(kv_dtype="nvfp4", num_kv_heads=1, num_heads=2, dec_seq_lens=[128], topk=2)
    pg = b.cache.numpy().reshape(b.num_pages, 2, 1152)
    scales = pg[:, :, 1024:].view(np.uint8)
    assert not np.any((scales & 0x7F) == 0x7F)      # no NaN scales
    assert b.k_scale > 0 and b.v_scale > 0
