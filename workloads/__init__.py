"""Seeded synthetic inputs for the paged block-sparse attend.

This module only *draws* data: queries, KV-cache bytes, per-token top-k block
lists, page tables and sequence lengths, in the shapes and layouts that the
attend consumes. It holds none of the attend's arithmetic (no causal filter,
no compaction, no softmax); the CUDA path and the CPU oracle both take what it
returns. The NVFP4 and fp8 encoders here only synthesise stored cache bytes.

Workloads (sizes follow the MiniMax-M3 sparse attend as the vLLM pages
``vllm.models.minimax_m3.nvidia.sparse_attention_flashinfer`` and
``vllm.models.minimax_m3.amd.ops.sparse_pa`` describe it: 128-token sparse
blocks, page-16 physical pages, a per-token top-k of logical block ids padded
with -1):

* ``tiny``      1 request of 1024 tokens, 8 q heads / 1 kv head, top-k 4,
                prefill of all 1024 tokens plus one decode token.
* ``decode``    64 requests, seq 16k..32k, 64/8 heads, top-k 16, bf16.
* ``prefill``   4 prompts {2048, 4096, 8192, 8192}, 64/8 heads, top-k 16,
                30% of the non-self slots point past the query's own block.
* ``mtp_fp8``   128 requests, seq 64k..128k, 2 queries per request,
                top-k 32, fp8-e4m3 cache with per-tensor scales in [0.5, 2].
* ``mixed_nvfp4`` 32 decode requests (8k..64k) plus 2 prefill chunks of 4096
                at contexts 16k and 32k, NVFP4 cache, top-k 16.
* ``prefill_g16`` the prefill prompts with GQA 16 (64 q heads on 4 kv heads).
* ``small``     parameterised small cases for parity tests.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

# Layout constants of the synthetic data (the attend's own copies live with
# the kernels and with the oracle; these only size the generated tensors).
BLOCK_TOKENS = 128          # tokens per logical sparse block
PAGE_ROWS = 16              # tokens per physical page
PAGES_PER_BLOCK = BLOCK_TOKENS // PAGE_ROWS
NVFP4_SLOT_BYTES = PAGE_ROWS * 64 + PAGE_ROWS * 8   # codes then e4m3 scales, per (page, K or V of a head)

KV_DTYPES = ("bf16", "fp8_e4m3", "nvfp4")


def page_bytes_for(kv_dtype: str, num_kv_heads: int, head_dim: int) -> int:
    """Bytes of one physical page (all kv heads) in the given cache format."""
    if kv_dtype == "bf16":
        return num_kv_heads * PAGE_ROWS * 2 * head_dim * 2
    if kv_dtype == "fp8_e4m3":
        return num_kv_heads * PAGE_ROWS * 2 * head_dim
    if kv_dtype == "nvfp4":
        assert head_dim == 128
        return 2 * num_kv_heads * NVFP4_SLOT_BYTES
    raise ValueError(kv_dtype)


@dataclass
class DecodePart:
    q: torch.Tensor            # [nd, Hq, D] bf16, nd = batch * decode_query_len
    topk: torch.Tensor         # [1, nd, k] int32 logical block ids, -1 padded
    page_table: torch.Tensor   # [batch, max_blocks] int32 physical block ids
    seq_lens: torch.Tensor     # [batch] int32
    decode_query_len: int


@dataclass
class PrefillPart:
    q: torch.Tensor            # [total_q, Hq, D] bf16
    topk: torch.Tensor         # [1, total_q, k] int32
    page_table: torch.Tensor   # [num_reqs, max_blocks] int32
    cu_seqlens_q: torch.Tensor  # [num_reqs + 1] int32
    seq_lens: torch.Tensor     # [num_reqs] int32 (context + query tokens)


@dataclass
class Batch:
    name: str
    kv_dtype: str
    num_heads: int
    num_kv_heads: int
    head_dim: int
    topk: int
    cache: torch.Tensor        # uint8 [num_pages, page_bytes]
    block_page_stride: int
    softmax_scale: float
    k_scale: float
    v_scale: float
    dec: DecodePart | None = None
    pre: PrefillPart | None = None
    meta: dict = field(default_factory=dict)

    @property
    def num_pages(self) -> int:
        return int(self.cache.shape[0])

    @property
    def page_bytes(self) -> int:
        return int(self.cache.shape[1])

    def to(self, device) -> "Batch":
        def mv(part):
            if part is None:
                return None
            return type(part)(**{k: (v.to(device) if isinstance(v, torch.Tensor) else v)
                                 for k, v in part.__dict__.items()})
        return Batch(self.name, self.kv_dtype, self.num_heads, self.num_kv_heads, self.head_dim,
                     self.topk, self.cache.to(device), self.block_page_stride, self.softmax_scale,
                     self.k_scale, self.v_scale, mv(self.dec), mv(self.pre), dict(self.meta))


# --------------------------------------------------------------------------------------------
# top-k draws
# --------------------------------------------------------------------------------------------

def draw_topk(abs_pos: torch.Tensor, k: int, gen: torch.Generator, future_prob: float = 0.0,
              blocks_in_request: torch.Tensor | None = None) -> torch.Tensor:
    """Per query row: its own block plus k-1 other slots, shuffled.

    Slot j (j = 0..k-2) holds the j-th id of a seeded random permutation of
    the row's past blocks [0, s) with s = abs_pos // 128, or -1 once j >= s.
    With probability ``future_prob`` a slot is instead replaced by a future
    id drawn uniformly from [s+1, s+nb] (nb = blocks of the row's request).
    The k slots are then shuffled. Rows with abs_pos < 0 get all -1.
    """
    n = abs_pos.numel()
    pos = abs_pos.to(torch.int64).cpu()
    s = torch.div(pos.clamp(min=0), BLOCK_TOKENS, rounding_mode="floor")
    if n == 0:
        return torch.empty(1, 0, k, dtype=torch.int32)
    smax = max(int(s.max()), 1)
    keys = torch.rand(n, smax, generator=gen)
    cand = torch.arange(smax).expand(n, smax)
    keys = torch.where(cand < s[:, None], keys, torch.full_like(keys, 2.0))
    order = keys.argsort(dim=1)
    m = k - 1
    if order.shape[1] < m:
        order = torch.cat([order, torch.full((n, m - order.shape[1]), smax, dtype=order.dtype)], 1)
    past = order[:, :m].clone()
    past[past >= s[:, None]] = -1
    if future_prob > 0.0:
        assert blocks_in_request is not None
        fut = torch.rand(n, m, generator=gen) < future_prob
        nb = blocks_in_request.to(torch.int64).cpu()[:, None].clamp(min=1)
        fid = s[:, None] + 1 + (torch.rand(n, m, generator=gen) * nb).floor().to(torch.int64).clamp(max=nb - 1)
        past = torch.where(fut, fid, past)
    rows = torch.cat([s[:, None], past], 1)
    perm = torch.rand(n, k, generator=gen).argsort(dim=1)
    rows = torch.gather(rows, 1, perm)
    rows[pos < 0] = -1
    return rows.to(torch.int32).reshape(1, n, k)


# --------------------------------------------------------------------------------------------
# page tables
# --------------------------------------------------------------------------------------------

def allocate_blocks(seq_groups: list[list[int]], gen: torch.Generator, slack: float = 0.05,
                    exact_pool: bool = False):
    """Random injective map of every request's logical blocks into one pool.

    ``seq_groups`` is a list of groups (e.g. decode requests, prefill requests);
    returns one page table per group (int32 [R, max_blocks], unused entries 0)
    and the pool size in physical blocks.
    """
    need = [[math.ceil(s / BLOCK_TOKENS) for s in g] for g in seq_groups]
    total = sum(sum(g) for g in need)
    pool = total if exact_pool else max(total, math.ceil(total * (1.0 + slack)))
    perm = torch.randperm(max(pool, 1), generator=gen)[:total]
    tables, at = [], 0
    for g in need:
        width = max(g) if g else 1
        width = max(width, 1)
        t = torch.zeros(len(g), width, dtype=torch.int32)
        for r, nb in enumerate(g):
            t[r, :nb] = perm[at:at + nb].to(torch.int32)
            at += nb
        tables.append(t)
    return tables, max(pool, 1)


# --------------------------------------------------------------------------------------------
# cache synthesis
# --------------------------------------------------------------------------------------------

def _e2m1_encode(x: torch.Tensor) -> torch.Tensor:
    """Round x (already clamped to [-6, 6]) to the nearest e2m1 value, ties to the even code.

    The magnitude code counts the midpoints between neighbouring magnitudes
    (0, 0.5, 1, 1.5, 2, 3, 4, 6) that |x| passes; a midpoint that lies below an
    even code is inclusive, one below an odd code exclusive.
    """
    a = x.abs().float()
    code = ((a > 0.25).to(torch.uint8) + (a >= 0.75).to(torch.uint8) + (a > 1.25).to(torch.uint8)
            + (a >= 1.75).to(torch.uint8) + (a > 2.5).to(torch.uint8) + (a >= 3.5).to(torch.uint8)
            + (a > 5.0).to(torch.uint8))
    sign = ((x < 0) & (code != 0)).to(torch.uint8) << 3
    return code | sign


def _nvfp4_quantise(x: torch.Tensor, gs: float):
    """x [..., 128] float -> (codes uint8 [..., 64], scales uint8 [..., 8]).

    Per 16 elements: sc = e4m3(amax16 / (6 * gs)); code = e2m1(x / (sc * gs)).
    Element 2i goes to the low nibble of byte i.
    """
    shp = x.shape[:-1]
    xb = x.float().reshape(*shp, 8, 16)
    amax = xb.abs().amax(dim=-1)
    sc = (amax / (6.0 * gs)).to(torch.float8_e4m3fn)
    scf = sc.float() * gs
    safe = torch.where(scf > 0, scf, torch.ones_like(scf))
    y = torch.where(scf[..., None] > 0, xb / safe[..., None], torch.zeros_like(xb)).clamp(-6.0, 6.0)
    code = _e2m1_encode(y).reshape(*shp, 128)
    packed = code[..., 0::2] | (code[..., 1::2] << 4)
    return packed.contiguous(), sc.view(torch.uint8).contiguous()


def synth_cache(kv_dtype: str, num_pages: int, num_kv_heads: int, head_dim: int, device,
                seed: int, chunk_pages: int = 4096):
    """Fill a uint8 [num_pages, page_bytes] cache with N(0,1) K/V in the given format.

    Returns (cache, k_global_scale, v_global_scale); the global scales are 1
    for bf16/fp8 and the NVFP4 per-tensor scales amax/(448*6) otherwise.
    """
    pb = page_bytes_for(kv_dtype, num_kv_heads, head_dim)
    cache = torch.empty(num_pages, pb, dtype=torch.uint8, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    Hkv, D = num_kv_heads, head_dim
    if kv_dtype == "nvfp4":
        # N(0,1) has a known spread; a fixed global scale from the expected amax
        # keeps generation chunked. We still compute it from a first pass of amax.
        amax_k, amax_v = 0.0, 0.0
        for p0 in range(0, num_pages, chunk_pages):
            n = min(chunk_pages, num_pages - p0)
            kv = torch.randn(n, Hkv, 2, PAGE_ROWS, D, generator=g, device=device)
            amax_k = max(amax_k, float(kv[:, :, 0].abs().max()))
            amax_v = max(amax_v, float(kv[:, :, 1].abs().max()))
        gk, gv = amax_k / (448.0 * 6.0), amax_v / (448.0 * 6.0)
        g.manual_seed(seed)
        for p0 in range(0, num_pages, chunk_pages):
            n = min(chunk_pages, num_pages - p0)
            kv = torch.randn(n, Hkv, 2, PAGE_ROWS, D, generator=g, device=device)
            ck, sk = _nvfp4_quantise(kv[:, :, 0], gk)
            cv, sv = _nvfp4_quantise(kv[:, :, 1], gv)
            # slot 2g = K of head g, slot 2g+1 = V; a slot is [16 x 64 codes][16 x 8 scales]
            slot_k = torch.cat([ck.reshape(n, Hkv, -1), sk.reshape(n, Hkv, -1)], -1)
            slot_v = torch.cat([cv.reshape(n, Hkv, -1), sv.reshape(n, Hkv, -1)], -1)
            cache[p0:p0 + n] = torch.stack([slot_k, slot_v], 2).reshape(n, pb)
        return cache, gk, gv
    for p0 in range(0, num_pages, chunk_pages):
        n = min(chunk_pages, num_pages - p0)
        kv = torch.randn(n, Hkv, PAGE_ROWS, 2 * D, generator=g, device=device)
        if kv_dtype == "bf16":
            cache[p0:p0 + n] = kv.to(torch.bfloat16).view(torch.uint8).reshape(n, pb)
        elif kv_dtype == "fp8_e4m3":
            cache[p0:p0 + n] = kv.to(torch.float8_e4m3fn).view(torch.uint8).reshape(n, pb)
        else:
            raise ValueError(kv_dtype)
    return cache, 1.0, 1.0


def _randn_bf16(shape, gen, device):
    return torch.randn(*shape, generator=gen, device=device).to(torch.bfloat16)


# --------------------------------------------------------------------------------------------
# builders
# --------------------------------------------------------------------------------------------

def _decode_positions(seq_lens: torch.Tensor, dql: int) -> torch.Tensor:
    # right-aligned query rows: row b*dql + i sits at seq_len - dql + i
    return (seq_lens.to(torch.int64)[:, None] - dql + torch.arange(dql)[None, :]).reshape(-1)


def _prefill_positions(q_lens: list[int], seq_lens: list[int]) -> tuple[torch.Tensor, torch.Tensor]:
    pos, req = [], []
    for r, (ql, sl) in enumerate(zip(q_lens, seq_lens)):
        pos.append(torch.arange(sl - ql, sl))
        req.append(torch.full((ql,), r))
    if not pos:
        return torch.empty(0, dtype=torch.int64), torch.empty(0, dtype=torch.int64)
    return torch.cat(pos), torch.cat(req)


def make_batch(name: str, *, kv_dtype: str, num_heads: int, num_kv_heads: int, head_dim: int,
               topk: int, dec_seq_lens: list[int] | None = None, decode_query_len: int = 1,
               pre_q_lens: list[int] | None = None, pre_ctx_lens: list[int] | None = None,
               future_prob: float = 0.0, seed: int = 0, device="cpu", exact_pool: bool = False,
               k_scale: float | None = None, v_scale: float | None = None,
               dec_topk: torch.Tensor | None = None) -> Batch:
    gen = torch.Generator()
    gen.manual_seed(seed)
    dec_seq_lens = dec_seq_lens or []
    pre_q_lens = pre_q_lens or []
    pre_ctx_lens = pre_ctx_lens or [0] * len(pre_q_lens)
    pre_seq_lens = [c + q for c, q in zip(pre_ctx_lens, pre_q_lens)]
    (dec_pt, pre_pt), pool_blocks = allocate_blocks(
        [[max(s, 0) for s in dec_seq_lens], pre_seq_lens], gen, exact_pool=exact_pool)
    num_pages = pool_blocks * PAGES_PER_BLOCK
    cache, gk, gv = synth_cache(kv_dtype, num_pages, num_kv_heads, head_dim, device, seed + 7)
    qgen = torch.Generator(device=device)
    qgen.manual_seed(seed + 11)
    if kv_dtype == "nvfp4":
        ks, vs = gk, gv
    elif kv_dtype == "fp8_e4m3":
        ks = k_scale if k_scale is not None else 0.5 + 1.5 * float(torch.rand(1, generator=gen))
        vs = v_scale if v_scale is not None else 0.5 + 1.5 * float(torch.rand(1, generator=gen))
    else:
        ks = 1.0 if k_scale is None else k_scale
        vs = 1.0 if v_scale is None else v_scale
    b = Batch(name=name, kv_dtype=kv_dtype, num_heads=num_heads, num_kv_heads=num_kv_heads,
              head_dim=head_dim, topk=topk, cache=cache, block_page_stride=PAGES_PER_BLOCK,
              softmax_scale=1.0 / math.sqrt(head_dim), k_scale=float(ks), v_scale=float(vs))
    if dec_seq_lens:
        sl = torch.tensor(dec_seq_lens, dtype=torch.int32)
        pos = _decode_positions(sl, decode_query_len)
        tk = dec_topk if dec_topk is not None else draw_topk(pos, topk, gen)
        b.dec = DecodePart(q=_randn_bf16((pos.numel(), num_heads, head_dim), qgen, device),
                           topk=tk.to(device), page_table=dec_pt.to(device), seq_lens=sl.to(device),
                           decode_query_len=decode_query_len)
    if pre_q_lens:
        pos, req = _prefill_positions(pre_q_lens, pre_seq_lens)
        nb = torch.tensor([math.ceil(s / BLOCK_TOKENS) for s in pre_seq_lens])[req]
        tk = draw_topk(pos, topk, gen, future_prob=future_prob, blocks_in_request=nb)
        cu = torch.zeros(len(pre_q_lens) + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(pre_q_lens), 0)
        b.pre = PrefillPart(q=_randn_bf16((pos.numel(), num_heads, head_dim), qgen, device),
                            topk=tk.to(device), page_table=pre_pt.to(device), cu_seqlens_q=cu.to(device),
                            seq_lens=torch.tensor(pre_seq_lens, dtype=torch.int32).to(device))
    return b


def tiny(device="cpu", seed: int = 1000, kv_dtype: str = "bf16") -> Batch:
    """1 request of 1024 tokens: prefill of all of them plus one decode token.

    The decode row reuses prefill token 1023's top-k row, so its table, context
    length and output must equal that prefill row's.
    """
    b = make_batch("tiny", kv_dtype=kv_dtype, num_heads=8, num_kv_heads=1, head_dim=128, topk=4,
                   pre_q_lens=[1024], seed=seed, device=device, exact_pool=True)
    # decode part: same request, same pages, same top-k row as token 1023
    b.dec = DecodePart(q=b.pre.q[1023:1024].clone(), topk=b.pre.topk[:, 1023:1024].clone(),
                       page_table=b.pre.page_table.clone(), seq_lens=b.pre.seq_lens.clone(),
                       decode_query_len=1)
    return b


def decode(device="cuda", seed: int = 1001, batch: int = 64, kv_dtype: str = "bf16") -> Batch:
    """The decode workload; kv_dtype "fp8_e4m3" / "nvfp4" gives the same shape on those caches."""
    gen = torch.Generator()
    gen.manual_seed(seed + 3)
    sl = torch.randint(16384, 32768 + 1, (batch,), generator=gen).tolist()
    return make_batch(f"decode_b{batch}_16k-32k_top16_{kv_dtype}", kv_dtype=kv_dtype, num_heads=64, num_kv_heads=8,
                      head_dim=128, topk=16, dec_seq_lens=sl, seed=seed, device=device)


def prefill(device="cuda", seed: int = 1002, kv_dtype: str = "bf16") -> Batch:
    """The varlen prefill workload; kv_dtype "fp8_e4m3" / "nvfp4" gives the same prompts on those caches."""
    return make_batch(f"prefill_varlen_2k4k8k8k_top16_{kv_dtype}", kv_dtype=kv_dtype, num_heads=64,
                      num_kv_heads=8, head_dim=128, topk=16, pre_q_lens=[2048, 4096, 8192, 8192],
                      future_prob=0.3, seed=seed, device=device)


def prefill_g16(device="cuda", seed: int = 1005) -> Batch:
    """The prefill workload's prompts with GQA 16 (64 query heads on 4 kv heads)."""
    return make_batch("prefill_varlen_2k4k8k8k_top16_gqa16_bf16", kv_dtype="bf16", num_heads=64,
                      num_kv_heads=4, head_dim=128, topk=16, pre_q_lens=[2048, 4096, 8192, 8192],
                      future_prob=0.3, seed=seed, device=device)


def mtp_fp8(device="cuda", seed: int = 1003) -> Batch:
    gen = torch.Generator()
    gen.manual_seed(seed + 3)
    sl = torch.randint(65536, 131072 + 1, (128,), generator=gen).tolist()
    return make_batch("mtp_b128_64k-128k_dql2_top32_fp8", kv_dtype="fp8_e4m3", num_heads=64,
                      num_kv_heads=8, head_dim=128, topk=32, dec_seq_lens=sl, decode_query_len=2,
                      seed=seed, device=device)


def mixed_nvfp4(device="cuda", seed: int = 1004) -> Batch:
    gen = torch.Generator()
    gen.manual_seed(seed + 3)
    sl = torch.randint(8192, 65536 + 1, (32,), generator=gen).tolist()
    return make_batch("mixed_32dec_2x4096pre_top16_nvfp4", kv_dtype="nvfp4", num_heads=64,
                      num_kv_heads=8, head_dim=128, topk=16, dec_seq_lens=sl,
                      pre_q_lens=[4096, 4096], pre_ctx_lens=[16384, 32768], seed=seed, device=device)


def small(*, kv_dtype: str = "bf16", num_heads: int = 16, num_kv_heads: int = 2, topk: int = 6,
          dec_seq_lens=None, decode_query_len: int = 1, pre_q_lens=None, pre_ctx_lens=None,
          future_prob: float = 0.3, seed: int = 7, device="cpu") -> Batch:
    """Parameterised small case that the oracle finishes in seconds."""
    return make_batch(f"small_{kv_dtype}", kv_dtype=kv_dtype, num_heads=num_heads,
                      num_kv_heads=num_kv_heads, head_dim=128, topk=topk, dec_seq_lens=dec_seq_lens,
                      decode_query_len=decode_query_len, pre_q_lens=pre_q_lens,
                      pre_ctx_lens=pre_ctx_lens, future_prob=future_prob, seed=seed, device=device)


CONFIGS = {"tiny": tiny, "decode": decode, "prefill": prefill, "mtp_fp8": mtp_fp8,
           "mixed_nvfp4": mixed_nvfp4, "prefill_g16": prefill_g16}
