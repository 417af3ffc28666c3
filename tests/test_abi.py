"""The C ABI library: it loads, exports every function include/pbs.h declares, and its host-side
checks reject bad arguments before anything is launched (no GPU needed: every call below fails a
check that runs before the first CUDA call)."""
import ctypes
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pbs.h")


@pytest.fixture(scope="module")
def L():
    from paged_block_sparse_gb300 import _build
    _build.build()
    import paged_block_sparse_gb300 as pbs
    return pbs.lib()


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"PBS_API\s+[\w\s\*]+?\b(pbs_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("pbs_build_sparse_block_table_decode", "pbs_build_sparse_block_table_prefill",
                 "pbs_sparse_decode_attention", "pbs_sparse_prefill_attention", "pbs_insert_index_cache",
                 "pbs_status_string", "pbs_abi_version"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"libpbs.so does not export {name}"


def test_status_strings(L):
    import paged_block_sparse_gb300 as pbs
    assert pbs.abi_version() == 9
    texts = {pbs.status_string(s) for s in range(6)}
    assert len(texts) == 6 and "ok" in texts
    assert pbs.status_string(99) == "unknown status"


# Fake device addresses: never dereferenced, because each call below fails a host check first.
A = ctypes.c_void_p(0x10000)
N = ctypes.c_void_p(0)
S = ctypes.c_void_p(0)


def _decode_table(L, **kw):
    args = dict(topk=A, trs=4, rows=2, k=4, pt=A, pts=8, mb=8, sl=A, batch=2, dql=1, bps=8, sbt=A, sbts=32,
                ctx=A)
    args.update(kw)
    return L.pbs_build_sparse_block_table_decode(args["topk"], args["trs"], args["rows"], args["k"], args["pt"],
                                                 args["pts"], args["mb"], args["sl"], args["batch"], args["dql"],
                                                 args["bps"], args["sbt"], args["sbts"], args["ctx"], N, S)


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-check tests use fake device addresses")
def test_table_host_checks(L):
    assert _decode_table(L, rows=3) == 2                  # rows != batch * dql (the page's assert)
    assert _decode_table(L, topk=N) == 1
    assert _decode_table(L, k=65, trs=65) == 3            # top-k wider than 64
    assert _decode_table(L, k=0) == 1
    assert _decode_table(L, trs=3) == 2                   # row stride < k
    assert _decode_table(L, sbts=31) == 2                 # table row narrower than k*8
    assert _decode_table(L, bps=4) == 2                   # a block spans at least 8 pages
    assert _decode_table(L, rows=0, batch=0) == 0         # empty: nothing launched
    assert _decode_table(L, dql=0) == 1
    st = L.pbs_build_sparse_block_table_prefill(A, 4, 5, 4, A, 8, 8, A, A, 0, 8, A, 32, A, N, S)
    assert st == 2                                        # tokens but no request


class _Opts(ctypes.Structure):
    _fields_ = [("prefill_kernel", ctypes.c_int32), ("splits", ctypes.c_int32), ("cache_map", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


def _decode_attend(L, **kw):
    a = dict(q=A, qrs=1024, qhs=128, kv=A, psb=65536, npages=100, dt=0, hq=64, hkv=8, hd=128, topk=A, trs=16,
             k=16, pt=A, pts=64, mb=64, sl=A, batch=4, dql=1, bps=8, sbt=N, sbts=0, sctx=N, sc=0.088, ks=1.0, vs=1.0,
             out=A, ors=8192, ohs=128, lse=N, lses=0, ws=N, wsb=0, opt=N)
    a.update(kw)
    return L.pbs_sparse_decode_attention(a["q"], a["qrs"], a["qhs"], a["kv"], a["psb"], a["npages"], a["dt"],
                                         a["hq"], a["hkv"], a["hd"], a["topk"], a["trs"], a["k"], a["pt"], a["pts"],
                                         a["mb"], a["sl"], a["batch"], a["dql"], a["bps"], a["sbt"], a["sbts"],
                                         a["sctx"], a["sc"], a["ks"], a["vs"], a["out"], a["ors"], a["ohs"], a["lse"],
                                         a["lses"], a["ws"], a["wsb"], a["opt"], N, S)


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-check tests use fake device addresses")
def test_attend_host_checks(L):
    assert _decode_attend(L, hd=64) == 3                  # head_dim must be 128
    assert _decode_attend(L, hq=48, hkv=8) == 3           # G = 6 unsupported
    assert _decode_attend(L, hq=256, hkv=8) == 3          # G = 32 unsupported
    assert _decode_attend(L, hq=60, hkv=8) == 2           # heads not a multiple of kv heads
    assert _decode_attend(L, dt=7) == 1
    assert _decode_attend(L, q=N) == 1
    assert _decode_attend(L, kv=ctypes.c_void_p(0x10008)) == 4   # cache not 16-byte aligned
    assert _decode_attend(L, psb=65536 + 8) == 4                # page stride not a multiple of 16
    assert _decode_attend(L, psb=4096) == 2                     # page stride below one page
    assert _decode_attend(L, qhs=127) == 4
    assert _decode_attend(L, sc=float("nan")) == 1
    assert _decode_attend(L, batch=0) == 0
    assert _decode_attend(L, npages=0) == 2
    assert _decode_attend(L, k=80, trs=80) == 3
    assert _decode_attend(L, lse=ctypes.c_void_p(0x10002), lses=64) == 4   # lse not 4-byte aligned
    assert _decode_attend(L, lse=A, lses=63) == 2                         # lse row narrower than Hq
    need = L.pbs_attend_workspace_bytes(4, 64, 8)
    assert need == 4 * 8 * (8 * 1040 * 4 + 4)              # 8 split partials + 1 ticket per (row, kv head)
    assert L.pbs_attend_workspace_bytes(4, 128, 8) == 2 * need   # GQA 16: two head groups per kv head
    assert L.pbs_attend_workspace_bytes(0, 64, 8) == 0
    assert L.pbs_attend_workspace_bytes(4, 60, 8) == 0
    assert _decode_attend(L, ws=N, wsb=16) == 1            # bytes without a pointer
    assert _decode_attend(L, ws=ctypes.c_void_p(0x10008), wsb=need) == 4
    assert _decode_attend(L, ws=A, wsb=need - 1) == 2      # too small for the rows
    # prebuilt table: both pointers or neither, rows at least top-k x 8 wide, 4-byte aligned
    assert _decode_attend(L, sbt=A, sbts=128) == 1          # table without its ctx
    assert _decode_attend(L, sctx=A) == 1                   # ctx without its table
    assert _decode_attend(L, sbt=A, sbts=127, sctx=A) == 2
    assert _decode_attend(L, sbt=ctypes.c_void_p(0x10002), sbts=128, sctx=A) == 4
    assert _decode_attend(L, topk=N) == 1                   # no table: top-k is needed
    # options: every field checked
    for bad in (_Opts(4, 0, 0, 0), _Opts(0, 3, 0, 0), _Opts(0, 16, 0, 0), _Opts(0, 0, 2, 0), _Opts(0, 0, 0, 1)):
        assert _decode_attend(L, opt=ctypes.byref(bad)) == 1


def test_prefill_workspace_bytes(L):
    f = L.pbs_prefill_workspace_bytes
    f.restype = ctypes.c_size_t
    one = f(256, 1, 64, 8, 16, 64)
    # fp16 partials + (lse, exponent) pairs per (token, query head, top-k slot), plus the buckets
    assert one >= 256 * 64 * 16 * (2 * 128 + 8)
    assert f(512, 1, 64, 8, 16, 64) > one and f(256, 1, 64, 8, 32, 64) > one
    assert f(1 << 21, 1, 64, 8, 16, 64) == f(1 << 19, 1, 64, 8, 16, 64)   # one segment holds at most 2^19 tokens
    for bad in ((0, 1, 64, 8, 16, 64), (256, 0, 64, 8, 16, 64), (256, 1, 60, 8, 16, 64), (256, 1, 64, 8, 65, 64),
                (256, 1, 64, 8, 16, 0)):
        assert f(*bad) == 0


def test_prefill_tile_workspace_bytes(L):
    f = L.pbs_prefill_tile_workspace_bytes
    f.restype = ctypes.c_size_t
    # one 32 KiB fp16 V image per (request, block, kv head), then the int32 exponents (256-aligned);
    # fp8 / NVFP4 add a 32 KiB bf16 K image each
    assert f(4, 8, 64, 0) == 4 * 64 * 8 * 32768 + 8192
    assert f(1, 1, 1, 0) == 32768 + 256
    assert f(4, 8, 64, 1) == f(4, 8, 64, 2) == f(4, 8, 64, 0) + 4 * 64 * 8 * 32768
    assert f(3, 2, 300, 0) > f(3, 2, 64, 0)                   # page tables wider than 128 blocks
    for bad in ((0, 8, 64, 0), (4, 0, 64, 0), (4, 8, 0, 0), (4, 8, 65536, 0), (65536, 8, 64, 0), (4, 8, 64, 3)):
        assert f(*bad) == 0
    import paged_block_sparse_gb300 as pbs
    assert pbs.prefill_tile_workspace_bytes(4, 8, 64) == f(4, 8, 64, 0)
    assert pbs.prefill_tile_workspace_bytes(4, 8, 64, "nvfp4") == f(4, 8, 64, 2)


def _mixed_attend(L, **kw):
    args = dict(batch=2, dql=1, nreqs=1, tq=4, ws=N, wsb=0, dmb=8, pmb=8)
    args.update(kw)
    return L.pbs_sparse_mixed_attention(A, 8192, 128, A, 65536, 64, 0, 64, 8, 128, A, 16, 16, A, 8, args["dmb"],
                                        A, args["batch"], args["dql"], A, 8, args["pmb"], A, A, args["nreqs"],
                                        args["tq"], 8, N, 0, N, 0.125, 1.0, 1.0, A, 8192, 128, N, 0, args["ws"],
                                        args["wsb"], N, N, S)


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-check tests use fake device addresses")
def test_mixed_host_checks(L):
    assert _mixed_attend(L, batch=-1) == 1
    assert _mixed_attend(L, dql=0) == 1
    assert _mixed_attend(L, ws=N, wsb=16) == 1             # workspace bytes without a pointer
    assert _mixed_attend(L, batch=0, tq=0) == 0            # nothing to attend
    assert _mixed_attend(L, nreqs=0) == 2                  # prefill tokens without a request


@pytest.mark.skipif(torch.cuda.is_available(), reason="host-check tests use fake device addresses")
def test_insert_host_checks(L):
    f = L.pbs_insert_index_cache
    assert f(A, 128, 1, 0, 128, A, 2048, 128, 4, 16, A, 1, 2, N, S) == 0   # empty: early return
    assert f(N, 128, 1, 4, 128, A, 2048, 128, 4, 16, A, 1, 2, N, S) == 1
    assert f(A, 128, 1, 4, 128, A, 2048, 128, 4, 16, A, 1, 3, N, S) == 1   # bad element size
    assert f(A, 128, 1, 4, 128, ctypes.c_void_p(0x10001), 2048, 128, 4, 16, A, 1, 2, N, S) == 4


def test_binding_refuses_host_tensors():
    import paged_block_sparse_gb300 as pbs
    with pytest.raises(ValueError):
        pbs.build_sparse_block_table_decode(torch.zeros(1, 2, 4, dtype=torch.int32),
                                            torch.zeros(2, 4, dtype=torch.int32), torch.zeros(2, dtype=torch.int32))


def test_binding_insert_shape_checks():
    """[sparse_pa] minimax_m3_insert_index_cache raises ValueError on rank/dim/length/stride."""
    import paged_block_sparse_gb300 as pbs
    k = torch.zeros(4, 8)
    with pytest.raises(ValueError):
        pbs.insert_index_cache(k, torch.zeros(2, 4, 7), torch.zeros(4, dtype=torch.int64))
    with pytest.raises(ValueError):
        pbs.insert_index_cache(k, torch.zeros(2, 4, 8), torch.zeros(3, dtype=torch.int64))
    with pytest.raises(ValueError):
        pbs.insert_index_cache(k, torch.zeros(2, 8, 4).transpose(1, 2), torch.zeros(4, dtype=torch.int64))
    pbs.insert_index_cache(torch.zeros(0, 8), torch.zeros(2, 4, 8), torch.zeros(0, dtype=torch.int64))


def test_prefill_kernel_choice_rule():
    """The library's prefill dispatch, asked through pbs_prefill_kernel_choice (the binding sizes its
    workspace from the same answer, so there is one rule)."""
    import paged_block_sparse_gb300 as pbs
    packed = 8 * 8192

    def run(kv, hq, hkv, k, mb, psb, kernel=None, table=False, ws=0, total_q=4096):
        try:
            return pbs.prefill_kernel_choice(total_q, 4, kv, psb, hq, hkv, k, mb, table, ws, kernel)
        except pbs.PbsError as e:
            return e.status
    assert run("bf16", 64, 8, 16, 64, packed) == "tile"
    assert run("bf16", 64, 4, 16, 128, 4 * 8192) == "tile"          # GQA 16, table 8 x top-k wide
    assert run("bf16", 64, 8, 16, 129, packed) == "token"            # wider than 8 x top-k
    assert run("bf16", 64, 8, 8, 65, packed) == "token"              # 8 x top-k = 64 blocks
    assert run("bf16", 64, 8, 8, 65, packed, "tile") == "tile"       # asked for: wider page tables too
    assert run("bf16", 64, 8, 8, 4000, packed, "tile") == "tile"
    assert run("bf16", 64, 8, 8, 65536, packed, "tile") == 3         # block ids travel as 16 bits
    assert run("bf16", 64, 8, 17, 64, packed, "tile") == 3           # top-k above 16
    assert run("bf16", 64, 8, 16, 64, packed, "token") == "token"
    # fp8 / NVFP4 caches take the tile kernel only with its workspace (K and V images)
    assert run("fp8_e4m3", 64, 8, 16, 64, 8 * 4096) == "token"
    big = 1 << 62
    assert run("fp8_e4m3", 64, 8, 16, 64, 8 * 4096, ws=big) == "gather"   # GQA 8: the gathered rows first
    assert run("nvfp4", 64, 8, 16, 64, 8 * 2304, ws=big) == "gather"
    assert run("fp8_e4m3", 64, 8, 16, 64, 8 * 4096, ws=pbs.prefill_tile_workspace_bytes(4, 8, 64, "fp8_e4m3")) == "tile"
    assert run("nvfp4", 64, 8, 16, 64, 8 * 2304, ws=pbs.prefill_tile_workspace_bytes(4, 8, 64, "nvfp4")) == "tile"
    assert run("nvfp4", 64, 8, 16, 64, 8 * 2304, "tile") == 3        # asked for without the workspace
    # page tables wider than 8 x top-k: the gathered-row kernel when its workspace is given
    assert run("nvfp4", 64, 8, 16, 400, 8 * 2304, ws=big) == "gather"
    assert run("bf16", 64, 8, 16, 400, packed, ws=big) == "gather"
    assert run("bf16", 64, 8, 16, 400, packed) == "token"
    tile_need = pbs.prefill_tile_workspace_bytes(4, 8, 400, "nvfp4")
    assert run("nvfp4", 64, 8, 16, 400, 8 * 2304, ws=tile_need) == "tile"   # room for the images only
    gneed = pbs.prefill_workspace_bytes(512, 4, 64, 8, 16, 400)
    assert run("bf16", 64, 8, 16, 400, packed, ws=gneed) == "gather"
    assert run("bf16", 64, 8, 16, 400, packed, ws=gneed - 256) == "token"
    assert run("bf16", 64, 8, 16, 400, packed, ws=big, table=True) == "token"  # the gathered rows need top-k
    need = pbs.prefill_tile_workspace_bytes(4, 8, 64, "fp8_e4m3")
    assert run("fp8_e4m3", 64, 8, 16, 64, 8 * 4096, "tile", ws=need) == "tile"
    assert run("fp8_e4m3", 64, 8, 16, 64, 8 * 4096, "tile", ws=need - 256) == 3
    assert run("bf16", 32, 8, 16, 64, packed) == "token"             # GQA 4
    assert run("bf16", 64, 8, 17, 64, packed) == "token"             # top-k above 16
    assert run("bf16", 64, 8, 16, 64, packed + 16) == "token"        # pages strided inside a larger allocation
    assert run("bf16", 64, 8, 16, 64, packed, table=True) == "tile"  # a prebuilt table: the tile kernel reads it
    # the gathered-row kernel on request, with a workspace of at least one 512-token window
    need = pbs.prefill_workspace_bytes(512, 4, 64, 8, 16, 64)
    assert run("bf16", 64, 8, 16, 64, packed, "gather", ws=need) == "gather"
    assert run("bf16", 64, 8, 16, 64, packed, "gather", ws=need - 256) == 3
    assert run("bf16", 64, 8, 16, 64, packed, "gather", ws=need, table=True) == 3   # it reads top-k only
    assert run("bf16", 64, 8, 16, 64, packed, ws=need) == "gather"   # GQA 8 with its workspace
    assert run("bf16", 64, 4, 16, 64, 4 * 8192, ws=big) == "tile"    # GQA 16: only for wider page tables
    assert run("bf16", 64, 4, 16, 400, 4 * 8192, ws=big) == "gather"
    assert run("bf16", 60, 8, 16, 64, packed) == 1
