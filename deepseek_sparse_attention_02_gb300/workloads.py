"""Seeded synthetic inputs for the DSA decode path.

This module only draws random numbers, quantises them into the cache formats
and lays out pages and block tables.  It holds none of the method's arithmetic
(no score, selection or attention) and is the one module that both the CUDA
path's tests/benchmark and the fp64 oracle consume.

Formats (bytes, little endian):

* FP8 indexer-key page (``FP8_PAGE_BYTES`` = 8448): ``page_tokens`` (64) keys
  of 128 e4m3 codes, then 64 f32 per-token scales.  Key of slot i at byte
  ``128*i``, its scale at byte ``8192 + 4*i``.
* MXFP4 indexer-key page (``FP4_PAGE_BYTES`` = 4352): 64 keys of 64 bytes
  (128 e2m1 values, element 2i in the low nibble of byte i), then 64 x 4
  UE8M0 bytes (byte g scales elements 32g..32g+31).
* Latent (MLA) page: ``[64, 576]`` bf16, 512 latent + 64 rope elements.

Token t of request b lives in page ``block_table[b, t // 64]``, slot ``t % 64``.
Query rows are flattened: row ``r = b*next_n + j``.

The recipes follow the workload statements: q and keys ~ N(0, 1), a seeded 5 %
of tokens shifted by +3.0 in every element before quantisation, FP8 per-token
(keys) / per-head (q) scale amax/448, head weights ~ N(0,1)/sqrt(64*128),
64-token pages in a shuffled block table, latents and MLA queries ~ N(0, 1) in
bf16.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PAGE_TOKENS = 64
INDEX_HEADS = 64
INDEX_DIM = 128
MLA_HEADS = 128
MLA_DQK = 576
MLA_DV = 512
FP8_KEY_BYTES = PAGE_TOKENS * INDEX_DIM                  # 8192
FP8_PAGE_BYTES = FP8_KEY_BYTES + 4 * PAGE_TOKENS         # 8448
FP4_KEY_BYTES = PAGE_TOKENS * INDEX_DIM // 2             # 4096
FP4_PAGE_BYTES = FP4_KEY_BYTES + PAGE_TOKENS * INDEX_DIM // 32  # 4352
E4M3_MAX = 448.0


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def quantize_e4m3(x: torch.Tensor):
    """Per-row (last dim) FP8 e4m3 quantisation with scale amax/448 (1 for an
    all-zero row).  Returns (codes uint8, scale float32) with x ~ codes*scale."""
    x = x.float()
    amax = x.abs().amax(dim=-1, keepdim=True)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    y = (x / scale).clamp_(-E4M3_MAX, E4M3_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, scale.squeeze(-1).float()


_E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def quantize_mxfp4(x: torch.Tensor):
    """OCP-MX style e2m1 quantisation with one UE8M0 scale per 32 elements of the
    last dim: shared exponent floor(log2(amax)) - 2, magnitudes rounded to the
    nearest e2m1 grid point (ties to the even code), clamped to 6.  Returns
    (packed uint8 [..., n/2], scale bytes uint8 [..., n/32])."""
    x = x.float()
    *lead, n = x.shape
    assert n % 32 == 0
    g = x.reshape(*lead, n // 32, 32)
    amax = g.abs().amax(dim=-1, keepdim=True)
    e = torch.where(amax > 0, torch.floor(torch.log2(amax)) - 2, torch.full_like(amax, -127.0))
    e = e.clamp(-127, 127)
    y = (g / torch.exp2(e)).abs().clamp(max=6.0)
    grid = torch.tensor(_E2M1_GRID, device=x.device)
    # nearest grid point; on an exact tie take the even code (RNE on the code)
    d = (y.unsqueeze(-1) - grid).abs()
    best = d.min(dim=-1, keepdim=True).values
    cand = (d == best)
    idx = torch.arange(8, device=x.device)
    even_tie = cand & ((idx % 2) == 0)
    pick = torch.where(even_tie.any(-1, keepdim=True), even_tie, cand)
    code = _first_true(pick)
    sign = (g < 0) & (code > 0)
    nib = (code | (sign.to(torch.int64) << 3)).to(torch.uint8).reshape(*lead, n)
    packed = (nib[..., 0::2] | (nib[..., 1::2] << 4)).to(torch.uint8)
    sf = (e.squeeze(-1) + 127).to(torch.uint8)
    return packed, sf


def _first_true(mask: torch.Tensor) -> torch.Tensor:
    idx = torch.arange(mask.shape[-1], device=mask.device)
    big = torch.full_like(idx, mask.shape[-1])
    return torch.where(mask, idx, big).amin(-1)


def bf16_bits(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.bfloat16).view(torch.int16)


def row_lengths(ctx_len: torch.Tensor, next_n: int) -> torch.Tensor:
    """L_r of the flattened rows (row j of a request sees ctx - (next_n-1-j))."""
    j = torch.arange(next_n, device=ctx_len.device)
    return (ctx_len.long()[:, None] - (next_n - 1 - j)[None, :]).clamp(min=0).reshape(-1)


@dataclass
class PagedLayout:
    """Pages of all requests and the block table that maps them (shuffled)."""
    ctx_len: torch.Tensor          # [B] int32
    block_table: torch.Tensor      # [B, max_pages] int32, -1 past the context
    num_pages: int
    pages_of: list = field(default_factory=list)  # per request: page ids (int64 tensor)


def make_layout(ctx_lens, seed: int, device="cpu", shuffle=True, spare_pages=0) -> PagedLayout:
    ctx = torch.as_tensor(list(ctx_lens), dtype=torch.int32)
    npg = [(int(c) + PAGE_TOKENS - 1) // PAGE_TOKENS for c in ctx.tolist()]
    total = sum(npg) + spare_pages
    g = _gen(seed * 7919 + 17, "cpu")
    perm = torch.randperm(total, generator=g) if shuffle else torch.arange(total)
    maxp = max(1, max(npg) if npg else 1)
    bt = torch.full((len(npg), maxp), -1, dtype=torch.int32)
    pages_of, o = [], 0
    for b, n in enumerate(npg):
        ids = perm[o:o + n]
        bt[b, :n] = ids.to(torch.int32)
        pages_of.append(ids.long())
        o += n
    return PagedLayout(ctx.to(device), bt.to(device), total, [p.to(device) for p in pages_of])


def _token_page_slot(layout: PagedLayout, device):
    """(page, slot) of every cached token, request-major."""
    pg, sl = [], []
    for b, c in enumerate(layout.ctx_len.tolist()):
        t = torch.arange(c, device=device)
        pg.append(layout.pages_of[b].to(device)[t // PAGE_TOKENS])
        sl.append(t % PAGE_TOKENS)
    return torch.cat(pg), torch.cat(sl)


@dataclass
class IndexerCase:
    q: torch.Tensor            # [R, 64, 128] uint8 e4m3
    q_scale: torch.Tensor      # [R, 64] f32
    w: torch.Tensor            # [R, 64] f32
    cache: torch.Tensor        # [P, 8448] uint8 (FP8 pages) or [P, 4352] (MXFP4 pages)
    layout: PagedLayout
    next_n: int
    fmt: str = "fp8"

    @property
    def rows(self) -> int:
        return self.q.shape[0]


def _queries(R, seed, device):
    g = _gen(seed * 104729 + 1, device)
    q = torch.randn(R, INDEX_HEADS, INDEX_DIM, generator=g, device=device)
    qc, qs = quantize_e4m3(q)
    w = torch.randn(R, INDEX_HEADS, generator=g, device=device) / math.sqrt(INDEX_HEADS * INDEX_DIM)
    return qc, qs, w.float()


def _keys_by_page(layout: PagedLayout, seed, device, heavy_frac, heavy_shift, chunk_pages=4096):
    """Yields (page ids, float keys [n, 64, 128], valid mask [n, 64]) page-chunk by
    page-chunk; tokens past a request's context are zero keys."""
    g = _gen(seed * 15485863 + 3, device)
    P = layout.num_pages
    valid = torch.zeros(P, PAGE_TOKENS, dtype=torch.bool, device=device)
    for b, c in enumerate(layout.ctx_len.tolist()):
        ids = layout.pages_of[b].to(device)
        full = c // PAGE_TOKENS
        valid[ids[:full]] = True
        if c % PAGE_TOKENS:
            valid[ids[full], : c % PAGE_TOKENS] = True
    for p0 in range(0, P, chunk_pages):
        p1 = min(P, p0 + chunk_pages)
        k = torch.randn(p1 - p0, PAGE_TOKENS, INDEX_DIM, generator=g, device=device)
        heavy = torch.rand(p1 - p0, PAGE_TOKENS, generator=g, device=device) < heavy_frac
        k = k + heavy.unsqueeze(-1).float() * heavy_shift
        v = valid[p0:p1]
        k = k * v.unsqueeze(-1).float()
        yield p0, p1, k


def make_indexer_case(ctx_lens, next_n=1, seed=0, device="cpu", shuffle=True,
                      heavy_frac=0.05, heavy_shift=3.0, fmt="fp8", layout=None) -> IndexerCase:
    """Paged indexer inputs for the dense (fmt='fp8') or candidate (fmt='mxfp4')
    path.  `layout` reuses the pages and block table of another case (as the
    layers of one model share them); by default the seed draws a new one."""
    if layout is None:
        layout = make_layout(ctx_lens, seed, device="cpu", shuffle=shuffle)
    else:
        layout = PagedLayout(**{f: getattr(layout, f) for f in layout.__dataclass_fields__})
        layout.ctx_len = layout.ctx_len.cpu()
        layout.block_table = layout.block_table.cpu()
        layout.pages_of = [p.cpu() for p in layout.pages_of]
    R = len(ctx_lens) * next_n
    qc, qs, w = _queries(R, seed, device)
    P = layout.num_pages
    if fmt == "fp8":
        cache = torch.zeros(P, FP8_PAGE_BYTES, dtype=torch.uint8, device=device)
        for p0, p1, k in _keys_by_page(layout, seed, device, heavy_frac, heavy_shift):
            kc, ks = quantize_e4m3(k)
            cache[p0:p1, :FP8_KEY_BYTES] = kc.reshape(p1 - p0, -1)
            cache[p0:p1, FP8_KEY_BYTES:] = ks.contiguous().view(torch.uint8).reshape(p1 - p0, -1)
    elif fmt == "mxfp4":
        cache = torch.zeros(P, FP4_PAGE_BYTES, dtype=torch.uint8, device=device)
        for p0, p1, k in _keys_by_page(layout, seed, device, heavy_frac, heavy_shift):
            pk, sf = quantize_mxfp4(k)
            cache[p0:p1, :FP4_KEY_BYTES] = pk.reshape(p1 - p0, -1)
            cache[p0:p1, FP4_KEY_BYTES:] = sf.reshape(p1 - p0, -1)
    else:
        raise ValueError(fmt)
    layout.ctx_len = layout.ctx_len.to(device)
    layout.block_table = layout.block_table.to(device)
    layout.pages_of = [p.to(device) for p in layout.pages_of]
    return IndexerCase(qc, qs, w, cache, layout, next_n, fmt)


def make_candidates(ctx_lens, next_n, bs, nb, seed=0, device="cpu", include_newest=True):
    """[R, nb] distinct candidate block ids per row, drawn uniformly from the
    blocks of the row's request; the block holding the newest token is always
    one of them.  Unsorted (as a source layer would publish them)."""
    g = _gen(seed * 32452843 + 5, "cpu")
    rows = []
    for c in ctx_lens:
        nblk = (int(c) + bs - 1) // bs
        for j in range(next_n):
            L = int(c) - (next_n - 1 - j)
            newest = (L - 1) // bs
            take = min(nb, nblk)
            if include_newest:
                others = torch.randperm(nblk - 1, generator=g)[: take - 1]
                others = others + (others >= newest).long()
                ids = torch.cat([others, torch.tensor([newest])])
            else:
                ids = torch.randperm(nblk, generator=g)[:take]
            ids = ids[torch.randperm(len(ids), generator=g)]
            if take < nb:  # pad with ids past the context (they sort last)
                ids = torch.cat([ids, torch.arange(nblk, nblk + nb - take)])
            rows.append(ids.to(torch.int32))
    return torch.stack(rows).to(device)


@dataclass
class MLACase:
    q: torch.Tensor       # [R, 128, 576] bf16
    kv: torch.Tensor      # [P, 64, 576] bf16
    scale: float


def make_index_queries(R, seed=0, device="cpu"):
    """Indexer queries of another layer over the same cache: (e4m3 codes
    [R, 64, 128], per-head scales [R, 64], head weights [R, 64])."""
    return _queries(R, seed, device)


def make_mla_queries(R, seed=0, device="cpu"):
    """Attention queries [R, 128, 576] bf16 of another layer."""
    g = _gen(seed * 49979687 + 13, device)
    return torch.randn(R, MLA_HEADS, MLA_DQK, generator=g, device=device).to(torch.bfloat16)


def make_mla_case(R, num_pages, seed=0, device="cpu", chunk_pages=2048) -> MLACase:
    g = _gen(seed * 49979687 + 11, device)
    q = torch.randn(R, MLA_HEADS, MLA_DQK, generator=g, device=device).to(torch.bfloat16)
    kv = torch.empty(num_pages, PAGE_TOKENS, MLA_DQK, dtype=torch.bfloat16, device=device)
    for p0 in range(0, num_pages, chunk_pages):
        p1 = min(num_pages, p0 + chunk_pages)
        kv[p0:p1] = torch.randn(p1 - p0, PAGE_TOKENS, MLA_DQK, generator=g, device=device).to(torch.bfloat16)
    return MLACase(q, kv, 1.0 / math.sqrt(MLA_DQK))


def random_indices(row_lens, k, seed=0, device="cpu"):
    """[R, k] distinct random token positions per row (all of them, then -1,
    when the row is shorter than k) -- a stand-in selection for attention-only
    checks."""
    g = _gen(seed * 86028121 + 13, "cpu")
    out = torch.full((len(row_lens), k), -1, dtype=torch.int32)
    for r, L in enumerate(row_lens):
        L = int(L)
        if L <= k:
            out[r, :L] = torch.randperm(L, generator=g).to(torch.int32)
        else:
            out[r] = torch.randperm(L, generator=g)[:k].to(torch.int32)
    return out.to(device)


# ------------------------------------------------------------ the workloads --

def config_ctx(cfg: int, scale: float = 1.0, seed: int = 0):
    """Context lengths, next_n and request count of each workload.  ``scale`` < 1
    shrinks it (same structure) for oracle-sized checks."""
    g = _gen(seed * 7 + cfg, "cpu")
    if cfg == 0:   # tiny indexer decode: 1 request, 8192 tokens, contiguous cache
        return dict(ctx=[max(1, int(8192 * scale))], next_n=1, shuffle=False)
    if cfg == 1:   # batched varlen decode: 64 requests, L ~ U[16K, 64K]
        n = max(1, int(round(64 * min(1.0, scale * 4))))
        lo, hi = int(16384 * scale), int(65536 * scale)
        ctx = torch.randint(max(1, lo), max(2, hi) + 1, (n,), generator=g).tolist()
        return dict(ctx=ctx, next_n=1, shuffle=True)
    if cfg == 2:   # long-context MTP decode: 32 x 131072, next_n = 2
        n = max(1, int(round(32 * min(1.0, scale * 4))))
        return dict(ctx=[max(2, int(131072 * scale))] * n, next_n=2, shuffle=True)
    if cfg == 3:   # two-level candidate-block indexer: 64 x 196608, 512 blocks
        n = max(1, int(round(64 * min(1.0, scale * 4))))
        return dict(ctx=[max(64, int(196608 * scale))] * n, next_n=1, shuffle=True,
                    candidate_block_size=64, candidate_topk_blocks=max(2, int(512 * min(1.0, scale * 4))),
                    layers=4)
    if cfg == 4:   # chunked prefill: 4096 queries at the end of a 65536-token cache
        L = max(2, int(65536 * scale))
        nq = max(1, int(4096 * scale))
        return dict(ctx=[L], next_n=nq, shuffle=True)
    raise ValueError(cfg)
