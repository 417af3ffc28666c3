"""Row-parallel timing driver for the oracle on the host's cores.

TEST INFRASTRUCTURE ONLY: the cpu_baseline leg and the reference arm of ``bench.py`` use it to
time :func:`oracle.sparse_decode_attention` on every host core. Nothing here changes what the
oracle computes: each worker process (started with the ``spawn`` method, one numpy thread each)
receives its share of the decode rows and the cache pages those rows read, then calls the
oracle on them one row at a time for the time budget it is given, and reports how many rows it
finished in how long. The rates of workers that ran side by side add up to the host's rate.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import time

import numpy as np


class _Pages:
    """The slice of the paged cache a worker holds: page id -> page contents."""

    def __init__(self, host):
        self.host = host

    def __getitem__(self, ids):
        return np.stack([self.host[int(i)] for i in ids])


def _worker(conn, call):
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    from .sparse_attend import sparse_decode_attention
    rows, host = call.pop("rows"), call.pop("host")
    pages = _Pages(host)
    conn.send("ready")
    while True:
        msg = conn.recv()
        if msg is None:
            break
        budget_s = float(msg)
        done, t0 = 0, time.perf_counter()
        while True:
            for r in rows:
                sparse_decode_attention(call["q"], pages, call["kv_dtype"], call["num_kv_heads"], call["topk"],
                                        call["page_table"], call["seq_lens"], call["decode_query_len"],
                                        call["softmax_scale"], call["k_scale"], call["v_scale"],
                                        call["block_page_stride"], rows=[r])
                done += 1
                if time.perf_counter() - t0 >= budget_s:
                    break
            else:
                continue
            break
        conn.send((done, time.perf_counter() - t0))


def host_cores() -> int:
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class DecodeRowPool:
    """``workers`` processes, each holding decode rows ``w, w + workers, ...`` of the batch and
    the pages they read (``row_pages[r]``: page id -> contents). ``run(budget_s)`` returns the
    host's rows per second (the sum of the workers' rates), the rows finished and the longest
    worker time."""

    def __init__(self, workers, row_pages, *, q, kv_dtype, num_kv_heads, topk, page_table, seq_lens,
                 decode_query_len, softmax_scale, k_scale, v_scale, block_page_stride, timeout_s=300.0):
        ctx = mp.get_context("spawn")
        self.timeout_s = timeout_s
        self.procs, self.conns = [], []
        n = len(row_pages)
        self.workers = max(1, min(int(workers), n))
        try:
            for w in range(self.workers):
                rows = list(range(w, n, self.workers))
                host = {}
                for r in rows:
                    host.update(row_pages[r])
                call = dict(rows=rows, host=host, q=q, kv_dtype=kv_dtype, num_kv_heads=num_kv_heads, topk=topk,
                            page_table=page_table, seq_lens=seq_lens, decode_query_len=decode_query_len,
                            softmax_scale=softmax_scale, k_scale=k_scale, v_scale=v_scale,
                            block_page_stride=block_page_stride)
                parent, child = ctx.Pipe()
                p = ctx.Process(target=_worker, args=(child, call), daemon=True)
                p.start()
                child.close()
                self.procs.append(p)
                self.conns.append(parent)
            for c in self.conns:
                if not c.poll(self.timeout_s):
                    raise TimeoutError("oracle worker did not start")
                if c.recv() != "ready":
                    raise RuntimeError("oracle worker failed to start")
        except BaseException:
            self.close()
            raise

    def run(self, budget_s: float):
        for c in self.conns:
            c.send(float(budget_s))
        res = []
        for c in self.conns:
            if not c.poll(budget_s + self.timeout_s):
                raise TimeoutError("oracle worker did not report")
            res.append(c.recv())
        rate = sum(d / t for d, t in res if t > 0)
        return rate, sum(d for d, _ in res), max(t for _, t in res)

    def close(self):
        for c in self.conns:
            try:
                c.send(None)
            except (BrokenPipeError, OSError):
                pass
        for p in self.procs:
            p.join(timeout=10)
            if p.is_alive():
                p.terminate()
                p.join(timeout=10)
        self.procs, self.conns = [], []

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
