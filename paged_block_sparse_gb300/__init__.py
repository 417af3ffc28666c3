"""paged_block_sparse_gb300 — MiniMax-M3 paged block-sparse attend on GB300 (sm_103a).

A thin ctypes binding over ``libpbs.so`` (C ABI in ``include/pbs.h``). Every function here only
marshals torch tensors into pointers, strides and sizes, passes the current CUDA stream and
turns a non-zero status into :class:`PbsError`; all computation runs in the library's CUDA
kernels. There is no CPU fallback: without the built library every call raises.

Sources (vLLM API pages): ``vllm.models.minimax_m3.nvidia.sparse_attention_flashinfer``
(forward), ``vllm.models.minimax_m3.amd.sparse_attention_nvfp4`` (forward, customize_spec) and
``vllm.models.minimax_m3.amd.ops.sparse_pa`` (table builders, row writer, index-cache insert).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "PbsError", "KV_DTYPES", "SPARSE_BLOCK_SIZE", "PAGES_PER_BLOCK", "PAGE_ROWS", "library_path", "lib",
    "abi_version", "status_string", "build_sparse_block_table_decode", "build_sparse_block_table_prefill",
    "sparse_decode_attention", "sparse_prefill_attention", "insert_index_cache", "DEVERR",
    "attend_workspace_bytes", "attend_workspace", "sparse_decode_attention_noalloc", "sparse_mixed_attention",
    "prefill_workspace_bytes", "prefill_workspace", "prefill_tile_workspace_bytes", "prefill_tile_workspace",
    "prefill_kernel_choice", "PREFILL_KERNELS",
]

SPARSE_BLOCK_SIZE = 128
PAGE_ROWS = 16
PAGES_PER_BLOCK = 8
KV_DTYPES = {"bf16": 0, "fp8_e4m3": 1, "nvfp4": 2}
DEVERR = {"block_oob": 1, "page_oob": 2, "slot_oob": 4, "timeout": 8, "table": 16}
# prefill kernels (pbs_attend_options.prefill_kernel / pbs_prefill_kernel_choice)
PREFILL_KERNELS = {"auto": 0, "token": 1, "tile": 2, "gather": 3}
_PREFILL_NAMES = {v: k for k, v in PREFILL_KERNELS.items()}


class _Options(ctypes.Structure):
    """pbs_attend_options (include/pbs.h)."""
    _fields_ = [("prefill_kernel", ctypes.c_int32), ("splits", ctypes.c_int32), ("cache_map", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None


class PbsError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status}: {status_string(status) if _lib else '?'}")


def library_path() -> str:
    return os.environ.get("PBS_LIBRARY", os.path.join(_HERE, "libpbs.so"))


def lib() -> ctypes.CDLL:
    """The loaded libpbs.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libpbs.so is not built ({path} missing); run "
                           "`python -m paged_block_sparse_gb300._build` (needs nvcc for sm_103a)")
    L = ctypes.CDLL(path)
    i32, i64, f32, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
    L.pbs_status_string.restype = ctypes.c_char_p
    L.pbs_status_string.argtypes = [ctypes.c_int]
    L.pbs_abi_version.restype = ctypes.c_int
    L.pbs_abi_version.argtypes = []
    L.pbs_attend_workspace_bytes.restype = ctypes.c_size_t
    L.pbs_attend_workspace_bytes.argtypes = [i64, i32, i32]
    L.pbs_prefill_workspace_bytes.restype = ctypes.c_size_t
    L.pbs_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    L.pbs_prefill_tile_workspace_bytes.restype = ctypes.c_size_t
    L.pbs_prefill_tile_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.pbs_prefill_kernel_choice.restype = ctypes.c_int
    L.pbs_prefill_kernel_choice.argtypes = [i32, i32, i32, i64, i32, i32, i32, i32, i32, ctypes.c_size_t, vp]
    table_common = [vp, i64, i32, i32, vp, i64, i32]
    L.pbs_build_sparse_block_table_decode.restype = ctypes.c_int
    L.pbs_build_sparse_block_table_decode.argtypes = table_common + [vp, i32, i32, i32, vp, i64, vp, vp, vp]
    L.pbs_build_sparse_block_table_prefill.restype = ctypes.c_int
    L.pbs_build_sparse_block_table_prefill.argtypes = table_common + [vp, vp, i32, i32, vp, i64, vp, vp, vp]
    attend_head = [vp, i64, i64, vp, i64, i64, i32, i32, i32, i32, vp, i64, i32, vp, i64, i32]
    table = [vp, i64, vp]
    L.pbs_sparse_decode_attention.restype = ctypes.c_int
    L.pbs_sparse_decode_attention.argtypes = attend_head + [vp, i32, i32, i32] + table + [
        f32, f32, f32, vp, i64, i64, vp, i64, vp, ctypes.c_size_t, vp, vp, vp]
    L.pbs_sparse_decode_attention_noalloc.restype = ctypes.c_int
    L.pbs_sparse_decode_attention_noalloc.argtypes = attend_head + [vp, i32, i32, i32, f32, f32, f32, vp, i64, i64,
                                                                    vp, vp, vp]
    L.pbs_sparse_prefill_attention.restype = ctypes.c_int
    L.pbs_sparse_prefill_attention.argtypes = attend_head + [vp, vp, i32, i32, i32] + table + [
        f32, f32, f32, vp, i64, i64, vp, i64, vp, ctypes.c_size_t, vp, vp, vp]
    L.pbs_sparse_mixed_attention.restype = ctypes.c_int
    L.pbs_sparse_mixed_attention.argtypes = attend_head[:13] + [vp, i64, i32, vp, i32, i32, vp, i64, i32, vp, vp, i32,
                                                                i32, i32] + table + [
        f32, f32, f32, vp, i64, i64, vp, i64, vp, ctypes.c_size_t, vp, vp, vp]
    L.pbs_insert_index_cache.restype = ctypes.c_int
    L.pbs_insert_index_cache.argtypes = [vp, i64, i64, i32, i32, vp, i64, i64, i32, i32, vp, i64, i32, vp, vp]
    del sz
    _lib = L
    return L


def abi_version() -> int:
    return int(lib().pbs_abi_version())


def status_string(status: int) -> str:
    return lib().pbs_status_string(int(status)).decode()


# --------------------------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------------------------

def _dev(t: torch.Tensor, name: str, dtype=None, min_dim=1) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library reads device memory only)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() < min_dim:
        raise ValueError(f"{name} must have at least {min_dim} dims")
    return t


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(status: int, where: str):
    if status != 0:
        raise PbsError(status, where)


def _rows2d(t: torch.Tensor, name: str) -> torch.Tensor:
    """[1, R, k] or [R, k] int32 with unit last stride -> [R, k] view."""
    _dev(t, name, torch.int32, 2)
    if t.dim() == 3:
        if t.shape[0] != 1:
            raise ValueError(f"{name} must be [1, rows, topk] or [rows, topk]")
        t = t[0]
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must have a contiguous last dimension")
    return t


def _table2d(t: torch.Tensor, name: str) -> torch.Tensor:
    _dev(t, name, torch.int32, 2)
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1):
        raise ValueError(f"{name} must be [rows, cols] with a contiguous last dimension")
    return t


def _options(kernel=None, splits=None, cache_map=None):
    """A pbs_attend_options pointer for the call (None: the library's own choices).

    kernel: None / "auto" / "token" / "tile" / "gather" (prefill); splits: None or 1, 2, 4, 8;
    cache_map: None or "quarter" (the token-centric kernel's per-row-quarter cache map)."""
    if kernel in (None, "auto") and splits is None and cache_map is None:
        return None
    if kernel not in (None, *PREFILL_KERNELS):
        raise ValueError(f"kernel must be one of {sorted(PREFILL_KERNELS)}")
    if cache_map not in (None, "quarter"):
        raise ValueError('cache_map must be None or "quarter"')
    o = _Options(PREFILL_KERNELS[kernel or "auto"], int(splits or 0), 1 if cache_map == "quarter" else 0, 0)
    return ctypes.byref(o)


def _table_args(sparse_table, rows):
    """(sparse_bt pointer, row stride, sparse_ctx pointer) of an optional prebuilt table
    ``(sparse_bt [rows, >= topk*8] int32, sparse_ctx [rows] int32)`` as the builders return it."""
    if sparse_table is None:
        return ctypes.c_void_p(0), 0, ctypes.c_void_p(0)
    sbt, ctx = sparse_table
    _table2d(sbt, "sparse_bt")
    _dev(ctx, "sparse_ctx", torch.int32)
    if sbt.shape[0] != rows or ctx.shape[0] != rows or ctx.dim() != 1 or (rows > 1 and ctx.stride(0) != 1):
        raise ValueError(f"sparse_table must be ([{rows}, >= topk*8], [{rows}]) int32 with contiguous rows")
    return _ptr(sbt), sbt.stride(0), _ptr(ctx)


def _cache_geometry(kv_cache: torch.Tensor):
    _dev(kv_cache, "kv_cache")
    page_stride_bytes = kv_cache.stride(0) * kv_cache.element_size()
    return int(kv_cache.shape[0]), int(page_stride_bytes)


# --------------------------------------------------------------------------------------------
# entry points
# --------------------------------------------------------------------------------------------

def build_sparse_block_table_decode(topk, page_table, seq_lens, decode_query_len: int = 1,
                                    block_page_stride: int = PAGES_PER_BLOCK, sparse_bt=None, sparse_ctx=None,
                                    err_word=None, stream=None):
    """Decode sparse block table (vLLM sparse_pa minimax_m3_build_sparse_block_table_decode).

    Returns (sparse_bt [rows, topk*8] int32, sparse_ctx [rows] int32)."""
    tk = _rows2d(topk, "topk")
    pt = _table2d(page_table, "page_table")
    sl = _dev(seq_lens, "seq_lens", torch.int32)
    rows, k = tk.shape
    if sparse_bt is None:
        sparse_bt = torch.empty(rows, k * PAGES_PER_BLOCK, dtype=torch.int32, device=tk.device)
    if sparse_ctx is None:
        sparse_ctx = torch.empty(rows, dtype=torch.int32, device=tk.device)
    _dev(sparse_bt, "sparse_bt", torch.int32, 2)
    _dev(sparse_ctx, "sparse_ctx", torch.int32)
    st = lib().pbs_build_sparse_block_table_decode(
        _ptr(tk), tk.stride(0), rows, k, _ptr(pt), pt.stride(0), pt.shape[1], _ptr(sl), sl.shape[0],
        int(decode_query_len), int(block_page_stride), _ptr(sparse_bt), sparse_bt.stride(0), _ptr(sparse_ctx),
        _ptr(err_word), _stream(stream, tk.device))
    _check(st, "pbs_build_sparse_block_table_decode")
    return sparse_bt, sparse_ctx


def build_sparse_block_table_prefill(topk, page_table, cu_seqlens_q, seq_lens,
                                     block_page_stride: int = PAGES_PER_BLOCK, sparse_bt=None, sparse_ctx=None,
                                     err_word=None, stream=None):
    """Prefill sparse block table (vLLM sparse_pa minimax_m3_build_sparse_block_table_prefill)."""
    tk = _rows2d(topk, "topk")
    pt = _table2d(page_table, "page_table")
    cu = _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    sl = _dev(seq_lens, "seq_lens", torch.int32)
    rows, k = tk.shape
    if sparse_bt is None:
        sparse_bt = torch.empty(rows, k * PAGES_PER_BLOCK, dtype=torch.int32, device=tk.device)
    if sparse_ctx is None:
        sparse_ctx = torch.empty(rows, dtype=torch.int32, device=tk.device)
    _dev(sparse_bt, "sparse_bt", torch.int32, 2)
    _dev(sparse_ctx, "sparse_ctx", torch.int32)
    st = lib().pbs_build_sparse_block_table_prefill(
        _ptr(tk), tk.stride(0), rows, k, _ptr(pt), pt.stride(0), pt.shape[1], _ptr(cu), _ptr(sl), sl.shape[0],
        int(block_page_stride), _ptr(sparse_bt), sparse_bt.stride(0), _ptr(sparse_ctx), _ptr(err_word),
        _stream(stream, tk.device))
    _check(st, "pbs_build_sparse_block_table_prefill")
    return sparse_bt, sparse_ctx


def _attend_prologue(q, kv_cache, kv_dtype, num_kv_heads, topk, page_table, out):
    _dev(q, "q", torch.bfloat16, 3)
    if q.stride(2) != 1:
        raise ValueError("q must have a contiguous head_dim")
    if kv_dtype not in KV_DTYPES:
        raise ValueError(f"kv_dtype must be one of {sorted(KV_DTYPES)}")
    num_pages, page_stride_bytes = _cache_geometry(kv_cache)
    tk = _rows2d(topk, "topk")
    pt = _table2d(page_table, "page_table")
    if tk.shape[0] != q.shape[0]:
        raise ValueError(f"topk has {tk.shape[0]} rows but q has {q.shape[0]}")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    _dev(out, "out", torch.bfloat16, 3)
    if out.shape != q.shape or out.stride(2) != 1:
        raise ValueError("out must match q's shape with a contiguous head_dim")
    return num_pages, page_stride_bytes, tk, pt, out


def attend_workspace_bytes(num_rows: int, num_heads: int, num_kv_heads: int) -> int:
    """Bytes of the optional split-merge workspace for ``num_rows`` query rows."""
    return int(lib().pbs_attend_workspace_bytes(int(num_rows), int(num_heads), int(num_kv_heads)))


_workspaces: dict = {}


def attend_workspace(num_rows: int, num_heads: int, num_kv_heads: int, device, stream=None) -> torch.Tensor:
    """A zeroed workspace for the attends, cached per (device, stream) and grown on demand.

    Calls that share one workspace must not overlap, so the cache is keyed by stream: calls on
    one stream run in order. Every completed call leaves the workspace's ticket words zero."""
    device = torch.device(device)
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (device.index, s.cuda_stream)
    need = attend_workspace_bytes(num_rows, num_heads, num_kv_heads)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        with torch.cuda.stream(s):
            ws = torch.zeros(max(need, 1 << 20), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def _workspace_args(workspace, rows, num_heads, num_kv_heads, device, stream):
    """(pointer, bytes) for the C call: "auto" takes the cached workspace, None passes none."""
    if workspace is None:
        return None, 0
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError('workspace must be "auto", None or a uint8 CUDA tensor')
        workspace = attend_workspace(rows, num_heads, num_kv_heads, device, stream)
    _dev(workspace, "workspace", torch.uint8)
    if not workspace.is_contiguous():
        raise ValueError("workspace must be contiguous")
    return _ptr(workspace), workspace.numel()


def prefill_workspace_bytes(total_q: int, num_reqs: int, num_heads: int, num_kv_heads: int, topk: int,
                            max_blocks: int) -> int:
    """Bytes with which the prefill attend runs ``total_q`` tokens on its gathered-row kernel in
    one segment (``total_q = 512``, one window: the smallest workspace that kernel takes)."""
    return int(lib().pbs_prefill_workspace_bytes(int(total_q), int(num_reqs), int(num_heads), int(num_kv_heads),
                                                 int(topk), int(max_blocks)))


def prefill_tile_workspace_bytes(num_reqs: int, num_kv_heads: int, max_blocks: int, kv_dtype: str = "bf16") -> int:
    """Bytes with which the prefill attend's tcgen05 tile kernel converts V to fp16 (and, for fp8 /
    NVFP4 caches, K to bf16) once per (request, block, kv head) and applies P in fp16 (0: the tile
    kernel cannot take this shape)."""
    return int(lib().pbs_prefill_tile_workspace_bytes(int(num_reqs), int(num_kv_heads), int(max_blocks),
                                                      KV_DTYPES[kv_dtype]))


# the tile kernel's converted-V workspace is allocated by default up to this size
TILE_WORKSPACE_CAP = 1 << 30
# "the call will pass whatever workspace the chosen kernel asks for" (pbs_prefill_kernel_choice)
_ANY_WORKSPACE = (1 << 63) - 1
_tile_workspaces: dict = {}


def prefill_tile_workspace(num_reqs: int, num_kv_heads: int, max_blocks: int, device, stream=None,
                           kv_dtype: str = "bf16"):
    """The tile kernel's workspace (converted V, and K for fp8 / NVFP4), cached per (device, stream)
    and grown on demand; None when the shape does not take it or it would exceed
    ``TILE_WORKSPACE_CAP`` (a bf16 call then applies P as hi + lo parts, an fp8 / NVFP4 call runs
    on the token-centric kernel). Needs no initial value."""
    need = prefill_tile_workspace_bytes(num_reqs, num_kv_heads, max_blocks, kv_dtype)
    if need == 0 or need > TILE_WORKSPACE_CAP:
        return None
    device = torch.device(device)
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (device.index, s.cuda_stream)
    ws = _tile_workspaces.get(key)
    if ws is None or ws.numel() < need:
        _tile_workspaces[key] = ws = None
        ws = torch.empty(need, dtype=torch.uint8, device=device)
        _tile_workspaces[key] = ws
    return ws


def prefill_kernel_choice(total_q: int, num_reqs: int, kv_dtype: str, page_stride_bytes: int, num_heads: int,
                          num_kv_heads: int, topk: int, max_blocks: int, with_table: bool = False,
                          workspace_bytes: int = 0, kernel=None) -> str:
    """The prefill kernel the library runs for a call of this shape ("token", "tile" or "gather"),
    asked from the library itself (pbs_prefill_kernel_choice): the binding sizes the workspace the
    chosen kernel wants from it."""
    r = int(lib().pbs_prefill_kernel_choice(int(total_q), int(num_reqs), KV_DTYPES[kv_dtype], int(page_stride_bytes),
                                            int(num_heads), int(num_kv_heads), int(topk), int(max_blocks),
                                            1 if with_table else 0, int(workspace_bytes), _options(kernel)))
    if r < 0:
        raise PbsError(-r, "pbs_prefill_kernel_choice")
    return _PREFILL_NAMES[r]


# the default prefill workspace is capped; larger calls run in several token segments
PREFILL_WORKSPACE_CAP = 8 << 30
_prefill_workspaces: dict = {}


def prefill_workspace(total_q: int, num_reqs: int, num_heads: int, num_kv_heads: int, topk: int, max_blocks: int,
                      device, stream=None) -> torch.Tensor:
    """A workspace for the prefill attend's gathered-row kernel, cached per (device, stream) and
    grown on demand: one segment for the whole call when that fits ``PREFILL_WORKSPACE_CAP``,
    else the cap (the call then runs in segments). Needs no initial value."""
    device = torch.device(device)
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (device.index, s.cuda_stream)
    full = prefill_workspace_bytes(total_q, num_reqs, num_heads, num_kv_heads, topk, max_blocks)
    least = prefill_workspace_bytes(min(total_q, 512), num_reqs, num_heads, num_kv_heads, topk, max_blocks)
    need = max(min(full, PREFILL_WORKSPACE_CAP), least)
    ws = _prefill_workspaces.get(key)
    if ws is None or ws.numel() < need:
        _prefill_workspaces.pop(key, None)
        with torch.cuda.stream(s):
            ws = torch.empty(need, dtype=torch.uint8, device=device)
        _prefill_workspaces[key] = ws
    return ws


def _prefill_auto_workspace(total_q, num_reqs, kv_dtype, psb, num_heads, num_kv_heads, topk, max_blocks, with_table,
                            kernel, device, stream):
    """The workspace the library's choice of prefill kernel for this shape wants (given any
    workspace): the gathered-row kernel's, the tile kernel's images, or none."""
    chosen = prefill_kernel_choice(total_q, num_reqs, kv_dtype, psb, num_heads, num_kv_heads, topk, max_blocks,
                                   with_table, _ANY_WORKSPACE, kernel)
    if chosen == "gather":
        return prefill_workspace(total_q, num_reqs, num_heads, num_kv_heads, topk, max_blocks, device, stream)
    if chosen == "tile":
        return prefill_tile_workspace(num_reqs, num_kv_heads, max_blocks, device, stream, kv_dtype)
    return None  # the token-centric kernel merges its splits in a cluster


def _lse_arg(lse, return_lse, q):
    """(tensor or None) for the optional log-sum-exp output [rows, Hq] fp32."""
    if lse is None and not return_lse:
        return None
    if lse is None:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    _dev(lse, "lse", torch.float32, 2)
    if lse.shape[0] != q.shape[0] or lse.shape[1] != q.shape[1] or lse.stride(1) != 1:
        raise ValueError("lse must be [rows, Hq] float32 with a contiguous last dimension")
    return lse


def sparse_decode_attention(q, kv_cache, kv_dtype: str, num_kv_heads: int, topk, page_table, seq_lens,
                            decode_query_len: int, softmax_scale: float, k_scale: float = 1.0, v_scale: float = 1.0,
                            block_page_stride: int = PAGES_PER_BLOCK, out=None, err_word=None, stream=None,
                            workspace=None, lse=None, return_lse: bool = False, sparse_table=None, splits=None,
                            cache_map=None):
    """Sparse decode attend (vLLM flashinfer msa_sparse_decode_attention / nvfp4 decode call).

    q [rows, Hq, 128] bf16 with rows = batch * decode_query_len; kv_cache [num_pages, ...] in the
    ``kv_dtype`` page layout; returns out [rows, Hq, 128] bf16. ``workspace``: None (the default:
    splits merge inside a thread-block cluster, the faster path on GB300), "auto" (a cached
    per-stream buffer) or a zeroed uint8 tensor of at least
    ``attend_workspace_bytes(rows, Hq, num_kv_heads)`` bytes; with one, splits merge through it.
    With ``return_lse`` (or an ``lse`` tensor [rows, Hq] fp32) the natural-log log-sum-exp of each
    head's scaled logits is written too and ``(out, lse)`` is returned. ``sparse_table``: an
    optional prebuilt ``(sparse_bt, sparse_ctx)`` pair (what :func:`build_sparse_block_table_decode`
    returns, built once and shared by every sparse layer of a step): the kernel attends it
    instead of compacting each row from ``topk``. ``splits`` / ``cache_map``: see
    ``pbs_attend_options``."""
    num_pages, psb, tk, pt, out = _attend_prologue(q, kv_cache, kv_dtype, num_kv_heads, topk, page_table, out)
    sl = _dev(seq_lens, "seq_lens", torch.int32)
    wp, wb = _workspace_args(workspace, q.shape[0], q.shape[1], num_kv_heads, q.device, stream)
    lse = _lse_arg(lse, return_lse, q)
    tb, ts, tc = _table_args(sparse_table, q.shape[0])
    st = lib().pbs_sparse_decode_attention(
        _ptr(q), q.stride(0), q.stride(1), _ptr(kv_cache), psb, num_pages, KV_DTYPES[kv_dtype], q.shape[1],
        int(num_kv_heads), q.shape[2], _ptr(tk), tk.stride(0), tk.shape[1], _ptr(pt), pt.stride(0), pt.shape[1],
        _ptr(sl), sl.shape[0], int(decode_query_len), int(block_page_stride), tb, ts, tc, float(softmax_scale),
        float(k_scale), float(v_scale), _ptr(out), out.stride(0), out.stride(1), _ptr(lse),
        lse.stride(0) if lse is not None else 0, wp, wb, _options(None, splits, cache_map), _ptr(err_word),
        _stream(stream, q.device))
    _check(st, "pbs_sparse_decode_attention")
    return (out, lse) if lse is not None else out


def sparse_decode_attention_noalloc(q, kv_cache, kv_dtype: str, num_kv_heads: int, topk, page_table, seq_lens,
                                    decode_query_len: int, softmax_scale: float, out, k_scale: float = 1.0,
                                    v_scale: float = 1.0, block_page_stride: int = PAGES_PER_BLOCK, err_word=None,
                                    stream=None, splits=None):
    """:func:`sparse_decode_attention` for callers that may not allocate device memory: split
    partials go to a fixed 4 MiB scratch inside the library, and ``out`` must be given (this
    wrapper allocates nothing either). Calls that could overlap on one device (other streams,
    unordered threads) race on the scratch; the first call on a device does a one-time address
    lookup and should come before any stream capture. ``splits`` forces the split count."""
    if out is None:
        raise ValueError("out is required: the no-allocation entry allocates nothing")
    num_pages, psb, tk, pt, out = _attend_prologue(q, kv_cache, kv_dtype, num_kv_heads, topk, page_table, out)
    sl = _dev(seq_lens, "seq_lens", torch.int32)
    st = lib().pbs_sparse_decode_attention_noalloc(
        _ptr(q), q.stride(0), q.stride(1), _ptr(kv_cache), psb, num_pages, KV_DTYPES[kv_dtype], q.shape[1],
        int(num_kv_heads), q.shape[2], _ptr(tk), tk.stride(0), tk.shape[1], _ptr(pt), pt.stride(0), pt.shape[1],
        _ptr(sl), sl.shape[0], int(decode_query_len), int(block_page_stride), float(softmax_scale),
        float(k_scale), float(v_scale), _ptr(out), out.stride(0), out.stride(1), _options(None, splits),
        _ptr(err_word), _stream(stream, q.device))
    _check(st, "pbs_sparse_decode_attention_noalloc")
    return out


def sparse_prefill_attention(q, kv_cache, kv_dtype: str, num_kv_heads: int, topk, page_table, cu_seqlens_q,
                             seq_lens, softmax_scale: float, k_scale: float = 1.0, v_scale: float = 1.0,
                             block_page_stride: int = PAGES_PER_BLOCK, out=None, err_word=None, stream=None,
                             workspace="auto", lse=None, return_lse: bool = False, sparse_table=None, kernel=None,
                             splits=None, cache_map=None):
    """Sparse prefill attend, varlen (vLLM flashinfer msa_sparse_attention / nvfp4 prefill call).

    ``workspace``: "auto" (the default: a cached per-stream buffer sized for the kernel the library
    picks, :func:`prefill_kernel_choice`: the gathered-row kernel's :func:`prefill_workspace`, the
    tile kernel's converted-V :func:`prefill_tile_workspace`, none for the token-centric kernel),
    None (no scratch: the tile kernel applies bf16 P as hi + lo parts) or a uint8 CUDA tensor (see
    ``pbs_sparse_prefill_attention`` in include/pbs.h for how each kernel uses it). ``lse`` and
    ``return_lse`` as in :func:`sparse_decode_attention`; ``sparse_table`` the optional prebuilt
    ``(sparse_bt, sparse_ctx)`` of :func:`build_sparse_block_table_prefill`; ``kernel`` ("token",
    "tile", "gather"), ``splits`` and ``cache_map``: see ``pbs_attend_options``."""
    num_pages, psb, tk, pt, out = _attend_prologue(q, kv_cache, kv_dtype, num_kv_heads, topk, page_table, out)
    cu = _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    sl = _dev(seq_lens, "seq_lens", torch.int32)
    if isinstance(workspace, str) and workspace == "auto":
        workspace = _prefill_auto_workspace(q.shape[0], sl.shape[0], kv_dtype, psb, q.shape[1], num_kv_heads,
                                            tk.shape[1], pt.shape[1], sparse_table is not None, kernel, q.device,
                                            stream)
    wp, wb = _workspace_args(workspace, q.shape[0], q.shape[1], num_kv_heads, q.device, stream)
    lse = _lse_arg(lse, return_lse, q)
    tb, ts, tc = _table_args(sparse_table, q.shape[0])
    st = lib().pbs_sparse_prefill_attention(
        _ptr(q), q.stride(0), q.stride(1), _ptr(kv_cache), psb, num_pages, KV_DTYPES[kv_dtype], q.shape[1],
        int(num_kv_heads), q.shape[2], _ptr(tk), tk.stride(0), tk.shape[1], _ptr(pt), pt.stride(0), pt.shape[1],
        _ptr(cu), _ptr(sl), sl.shape[0], q.shape[0], int(block_page_stride), tb, ts, tc, float(softmax_scale),
        float(k_scale), float(v_scale), _ptr(out), out.stride(0), out.stride(1), _ptr(lse),
        lse.stride(0) if lse is not None else 0, wp, wb, _options(kernel, splits, cache_map), _ptr(err_word),
        _stream(stream, q.device))
    _check(st, "pbs_sparse_prefill_attention")
    return (out, lse) if lse is not None else out


def sparse_mixed_attention(q, kv_cache, kv_dtype: str, num_kv_heads: int, topk, dec_page_table, dec_seq_lens,
                           decode_query_len: int, pre_page_table, cu_seqlens_q, pre_seq_lens, softmax_scale: float,
                           k_scale: float = 1.0, v_scale: float = 1.0, block_page_stride: int = PAGES_PER_BLOCK,
                           out=None, err_word=None, stream=None, lse=None, return_lse: bool = False,
                           sparse_table=None, kernel=None, splits=None, cache_map=None, workspace="auto"):
    """Decode rows then prefill tokens in one call (vLLM flashinfer forward with both parts):
    q [nd + total_q, Hq, 128] with nd = len(dec_seq_lens) * decode_query_len; topk (and the
    optional prebuilt ``sparse_table``) one row per q row. ``workspace`` is the prefill part's, as in
    :func:`sparse_prefill_attention` ("auto": sized for the kernel the library picks for that part;
    None: none, so fp8 / NVFP4 prefill parts stay on the token-centric kernel). Returns out (and
    lse)."""
    num_pages, psb, tk, pt_d, out = _attend_prologue(q, kv_cache, kv_dtype, num_kv_heads, topk, dec_page_table, out)
    pt_p = _table2d(pre_page_table, "pre_page_table")
    sl_d = _dev(dec_seq_lens, "dec_seq_lens", torch.int32)
    cu = _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    sl_p = _dev(pre_seq_lens, "pre_seq_lens", torch.int32)
    nd = sl_d.shape[0] * int(decode_query_len)
    total_q = q.shape[0] - nd
    if total_q < 0:
        raise ValueError(f"q has {q.shape[0]} rows, fewer than the {nd} decode rows")
    if isinstance(workspace, str) and workspace == "auto":
        workspace = None
        if total_q > 0 and nd > 0:
            workspace = _prefill_auto_workspace(total_q, sl_p.shape[0], kv_dtype, psb, q.shape[1], num_kv_heads,
                                                tk.shape[1], pt_p.shape[1], sparse_table is not None, kernel,
                                                q.device, stream)
    wp, wb = _workspace_args(workspace, total_q, q.shape[1], num_kv_heads, q.device, stream)
    lse = _lse_arg(lse, return_lse, q)
    tb, ts, tc = _table_args(sparse_table, q.shape[0])
    st = lib().pbs_sparse_mixed_attention(
        _ptr(q), q.stride(0), q.stride(1), _ptr(kv_cache), psb, num_pages, KV_DTYPES[kv_dtype], q.shape[1],
        int(num_kv_heads), q.shape[2], _ptr(tk), tk.stride(0), tk.shape[1], _ptr(pt_d), pt_d.stride(0),
        pt_d.shape[1], _ptr(sl_d), sl_d.shape[0], int(decode_query_len), _ptr(pt_p), pt_p.stride(0), pt_p.shape[1],
        _ptr(cu), _ptr(sl_p), sl_p.shape[0], total_q, int(block_page_stride), tb, ts, tc, float(softmax_scale),
        float(k_scale), float(v_scale), _ptr(out), out.stride(0), out.stride(1), _ptr(lse),
        lse.stride(0) if lse is not None else 0, wp, wb, _options(kernel, splits, cache_map), _ptr(err_word),
        _stream(stream, q.device))
    _check(st, "pbs_sparse_mixed_attention")
    return (out, lse) if lse is not None else out


def insert_index_cache(index_k, index_cache, index_slot_mapping, err_word=None, stream=None) -> None:
    """Scatter index keys [N, D] into the key-only side cache [B, T, D] (vLLM sparse_pa
    minimax_m3_insert_index_cache), with the page's argument checks."""
    if index_k.numel() == 0 or index_cache.numel() == 0:
        return
    if index_k.dim() != 2 or index_cache.dim() != 3:
        raise ValueError("index cache insert expects [N,D] and [B,T,D]")
    if index_k.shape[1] != index_cache.shape[2]:
        raise ValueError("index key dim must match index cache head dim")
    if index_slot_mapping.dim() != 1 or index_slot_mapping.shape[0] != index_k.shape[0]:
        raise ValueError("index slot mapping must be a length-N vector")
    if index_cache.stride(2) != 1:
        raise ValueError("index cache requires contiguous head dimension")
    _dev(index_k, "index_k")
    _dev(index_cache, "index_cache")
    _dev(index_slot_mapping, "index_slot_mapping", torch.int64)
    if index_k.dtype != index_cache.dtype:
        raise TypeError("index_k and index_cache must share a dtype")
    st = lib().pbs_insert_index_cache(
        _ptr(index_k), index_k.stride(0), index_k.stride(1), index_k.shape[0], index_k.shape[1], _ptr(index_cache),
        index_cache.stride(0), index_cache.stride(1), index_cache.shape[0], index_cache.shape[1],
        _ptr(index_slot_mapping), index_slot_mapping.stride(0), index_k.element_size(), _ptr(err_word),
        _stream(stream, index_k.device))
    _check(st, "pbs_insert_index_cache")
