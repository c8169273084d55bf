"""Pins of the fp64 oracle against facts fixed outside itself: the worked
examples the pages print, library decoders (torch float8 / bf16 casts, numpy
stable sort, torch scaled-dot-product attention), exact rational brute force,
closed forms and invariants.  CPU only."""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


# ----------------------------------------------------------------- helpers --

def e4m3_codes(values) -> np.ndarray:
    """Codes of values that are exactly representable in e4m3 (via torch)."""
    t = torch.tensor(np.asarray(values, np.float32)).to(torch.float8_e4m3fn)
    back = t.to(torch.float32).numpy()
    assert np.array_equal(back, np.asarray(values, np.float32)), "not exact in e4m3"
    return t.view(torch.uint8).numpy()


def fp8_cache(key_codes, key_scales, page_tokens, seed=0, shuffle=True):
    """Pages [P, page_tokens*D + 4*page_tokens] for one request's keys plus its
    block table row.  Returns (cache, k_stride, scale_bytes, s_stride, bt)."""
    key_codes = np.asarray(key_codes, np.uint8)
    T, D = key_codes.shape
    P = (T + page_tokens - 1) // page_tokens
    rng = np.random.default_rng(seed)
    perm = rng.permutation(P) if shuffle else np.arange(P)
    page_bytes = page_tokens * D + 4 * page_tokens
    cache = np.zeros((P, page_bytes), np.uint8)
    for t in range(T):
        p, s = perm[t // page_tokens], t % page_tokens
        cache[p, s * D:(s + 1) * D] = key_codes[t]
        cache[p, page_tokens * D + 4 * s: page_tokens * D + 4 * s + 4] = (
            np.asarray([key_scales[t]], np.float32).view(np.uint8))
    flat = cache.reshape(-1)
    return flat, page_bytes, flat[page_tokens * D:], page_bytes, perm.astype(np.int32)[None, :]


def run_indexer(q_codes, q_scale, w, key_codes, key_scales, page_tokens=4, ctx=None,
                next_n=1, seed=0):
    q_codes = np.asarray(q_codes, np.uint8)
    R, H, D = q_codes.shape
    T = len(key_codes)
    cache, ks, sc, ss, bt = fp8_cache(key_codes, key_scales, page_tokens, seed)
    nreq = R // next_n  # every request reads the same cached keys
    ctx = np.full(nreq, T if ctx is None else ctx, np.int32)
    bt = np.repeat(bt, nreq, axis=0)
    return oracle.indexer_logits(q_codes, np.asarray(q_scale, np.float32).reshape(R, H),
                                 np.asarray(w, np.float32).reshape(R, H), cache, ks, sc, ss,
                                 page_tokens, bt, ctx, next_n)


def read_golden(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "worked_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, *kv = line.split()
            rows.append((kind, dict(x.split("=") for x in kv)))
    return rows


# --------------------------------------------------------------- decoders --

def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.tensor(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode_e4m3(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))
    assert np.flatnonzero(np.isnan(got)).tolist() == [0x7F, 0xFF]


def test_ue8m0_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.tensor(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = oracle.decode_ue8m0(codes)
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])


def test_e2m1_table_and_nibble_order():
    # OCP MX e2m1 magnitudes by code 0..7; bit 3 is the sign.
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    packed = np.array([(2 * i + 1) << 4 | (2 * i) for i in range(8)], np.uint8)
    got = oracle.decode_e2m1(packed, 16)
    expect = [(-1.0 if c & 8 else 1.0) * grid[c & 7] for c in range(16)]
    assert got.tolist() == expect
    # element 2i is the low nibble: byte 0x21 -> [0.5, 1.0]
    assert oracle.decode_e2m1(np.array([0x21], np.uint8), 2).tolist() == [0.5, 1.0]


def test_bf16_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = torch.tensor(bits.astype(np.int32)).to(torch.int16).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.decode_bf16(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ---------------------------------------------------------------- indexer --

def test_worked_dot_and_relu(golden_dir):
    for kind, kv in read_golden(golden_dir):
        if kind == "dot":
            q = [float(x) for x in kv["q"].split(",")]
            k = [float(x) for x in kv["k"].split(",")]
            logits, _ = run_indexer(e4m3_codes(q).reshape(1, 1, 2), [1.0], [1.0],
                                    e4m3_codes([k]), [1.0], page_tokens=4)
            assert logits[0, 0] == float(kv["value"])
        elif kind == "relu":
            x, out = float(kv["in"]), float(kv["out"])
            # one head, D = 2: q = (x, 0), k = (1, 0) gives q.k = x
            logits, _ = run_indexer(e4m3_codes([x, 0.0]).reshape(1, 1, 2), [1.0], [1.0],
                                    e4m3_codes([[1.0, 0.0]]), [1.0], page_tokens=4)
            assert logits[0, 0] == out


def _frac_e4m3(code):
    v = float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64))
    return Fraction(v)


def brute_indexer(q_codes, q_scale, w, key_codes, key_scales, ctx, next_n):
    """Exact rational evaluation of Eq. (1) for every row and token."""
    R, H, D = q_codes.shape
    out = {}
    for r in range(R):
        L = ctx - (next_n - 1 - r % next_n)
        for t in range(L):
            tot = Fraction(0)
            for h in range(H):
                dot = sum(Fraction(float(q_scale[r, h])) * _frac_e4m3(q_codes[r, h, d]) *
                          Fraction(float(key_scales[t])) * _frac_e4m3(key_codes[t, d])
                          for d in range(D))
                tot += Fraction(float(w[r, h])) * max(dot, Fraction(0))
            out[(r, t)] = tot
    return out


def test_indexer_matches_rational_brute_force():
    rng = np.random.default_rng(1)
    R, H, D, T, next_n = 4, 3, 5, 11, 2
    q = e4m3_codes(rng.choice([-2, -1.5, -1, -0.5, 0.25, 0.5, 1, 1.5, 3], size=(R, H, D)).astype(np.float32))
    qs = rng.uniform(0.1, 2, size=(R, H)).astype(np.float32)
    w = rng.normal(size=(R, H)).astype(np.float32)
    k = e4m3_codes(rng.choice([-3, -1, -0.75, 0.5, 1, 2, 4], size=(T, D)).astype(np.float32))
    ks = rng.uniform(0.1, 2, size=T).astype(np.float32)
    logits, mag = run_indexer(q.reshape(R, H, D), qs, w, k, ks, page_tokens=4, ctx=T,
                              next_n=next_n)
    ref = brute_indexer(q.reshape(R, H, D), qs, w, k, ks, T, next_n)
    for (r, t), v in ref.items():
        assert abs(logits[r, t] - float(v)) <= 1e-13 * max(1.0, abs(float(v)))
    # rows see ctx - (next_n - 1 - j) tokens: the first row of each pair stops one short
    assert np.isnan(logits[0, T - 1]) and not np.isnan(logits[1, T - 1])
    assert np.all(mag[~np.isnan(mag)] >= np.abs(logits[~np.isnan(logits)]) - 1e-12)


def test_indexer_all_negative_dot_gives_zero():
    rng = np.random.default_rng(2)
    H, D, T = 4, 8, 9
    q = e4m3_codes(rng.choice([0.5, 1, 2], size=(1, H, D)).astype(np.float32))
    k = e4m3_codes(-rng.choice([0.5, 1, 2], size=(T, D)).astype(np.float32))
    w = rng.normal(size=(1, H)).astype(np.float32)
    logits, _ = run_indexer(q.reshape(1, H, D), np.ones((1, H)), w, k, np.ones(T))
    assert np.all(logits[0, :T] == 0.0)


def test_indexer_one_hot_keys_closed_form():
    rng = np.random.default_rng(3)
    D, T = 16, 13
    qv = rng.choice([-2.0, -0.5, 0.5, 1.0, 1.5, 3.0], size=D).astype(np.float32)
    q = e4m3_codes(qv).reshape(1, 1, D)
    dims = rng.integers(0, D, size=T)
    cv = rng.choice([0.25, 0.5, 1.0, 2.0, 6.0], size=T).astype(np.float32)
    keys = np.zeros((T, D), np.float32)
    keys[np.arange(T), dims] = cv
    ks = rng.uniform(0.5, 2, T).astype(np.float32)
    wv, sq = np.float32(0.75), np.float32(1.25)
    logits, _ = run_indexer(q, [sq], [wv], e4m3_codes(keys), ks)
    for t in range(T):
        closed = float(wv) * float(sq) * float(ks[t]) * max(0.0, float(qv[dims[t]]) * float(cv[t]))
        assert logits[0, t] == pytest.approx(closed, rel=1e-15, abs=0)


def test_indexer_key_permutation_permutes_logits():
    rng = np.random.default_rng(4)
    H, D, T = 5, 8, 37
    q = e4m3_codes(rng.choice([-1, -0.5, 0.5, 1], size=(1, H, D)).astype(np.float32))
    k = e4m3_codes(rng.choice([-2, -1, 0.5, 1, 2], size=(T, D)).astype(np.float32))
    ks = rng.uniform(0.5, 2, T).astype(np.float32)
    w = rng.normal(size=(1, H)).astype(np.float32)
    perm = rng.permutation(T)
    a, _ = run_indexer(q.reshape(1, H, D), np.ones((1, H)), w, k, ks, seed=0)
    b, _ = run_indexer(q.reshape(1, H, D), np.ones((1, H)), w, k[perm], ks[perm], seed=5)
    assert np.array_equal(b[0, :T], a[0, perm])


# ------------------------------------------------------------------ top-k --

def test_worked_topk(golden_dir):
    for kind, kv in read_golden(golden_dir):
        if kind == "topk":
            s = np.array([float(x) for x in kv["scores"].split(",")])
            got = oracle.topk(s, len(s), int(kv["k"]))[0].tolist()
            assert got == [int(x) for x in kv["selected"].split(",")]


def test_topk_short_row_returns_all_then_pad():
    s = np.array([[0.1, -2.0, 7.0, 0.0, 0.0, 0.0]])
    got = oracle.topk(s, 4, 8)[0]
    assert sorted(got[:4].tolist()) == [0, 1, 2, 3] and got[4:].tolist() == [-1] * 4


def test_topk_matches_stable_argsort_with_ties():
    rng = np.random.default_rng(5)
    s = rng.integers(-20, 20, size=(6, 300)).astype(np.float64)  # many exact ties
    L = np.array([300, 1, 0, 57, 299, 128], np.int32)
    got = oracle.topk(s, L, 64)
    for i in range(6):
        order = np.argsort(-s[i, :L[i]], kind="stable")[:64]
        expect = np.full(64, -1)
        expect[:len(order)] = order
        assert got[i].tolist() == expect.tolist()


def test_topk_permutation_equivariance_and_split():
    rng = np.random.default_rng(6)
    s = rng.normal(size=1000)
    k = 100
    base = oracle.topk(s, 1000, k)[0]
    perm = rng.permutation(1000)
    moved = oracle.topk(s[perm], 1000, k)[0]
    assert sorted(perm[moved].tolist()) == sorted(base.tolist())
    sel = np.zeros(1000, bool)
    sel[base] = True
    assert s[sel].min() >= s[~sel].max()


def test_topk_column_to_token_map():
    s = np.array([[5.0, 1.0, 4.0, 3.0, 9.0, 0.0]])
    blocks = np.array([[7, 2, 30]], np.int32)  # bs = 2: columns 0..5 -> 14,15,4,5,60,61
    got = oracle.topk(s, 6, 3, col_blocks=blocks, bs=2)[0].tolist()
    assert got == [60, 14, 4]


# -------------------------------------------------------------- candidate --

def test_candidate_expand_brute_force():
    rng = np.random.default_rng(7)
    bs, nb = 4, 6
    ctx = np.array([23, 8, 40], np.int32)
    cand = np.stack([rng.permutation(12)[:nb] for _ in range(3)]).astype(np.int32)
    si, end = oracle.candidate_expand(cand, bs, ctx, 1)
    for r in range(3):
        assert si[r].tolist() == sorted(cand[r].tolist())
        toks = [b * bs + o for b in si[r] for o in range(bs)]
        valid = [0 <= t < ctx[r] for t in toks]
        assert end[r] == sum(valid)
        # the valid columns form a prefix once the blocks are sorted
        assert all(valid[:end[r]]) and not any(valid[end[r]:])


def test_candidate_expand_sparse_blocks_brute_force():
    """Candidate blocks of cbs tokens scored as sparse blocks of sbs tokens
    (cbs a multiple of sbs): the sparse columns must cover exactly the
    candidate blocks' tokens, in ascending token order, the valid ones first;
    the sparse block count is nb * cbs / sbs."""
    rng = np.random.default_rng(8)
    for cbs, sbs in ((8, 4), (12, 4), (16, 2), (6, 6)):
        nb = 5
        ctx = np.array([37, 9, 80, 1], np.int32)
        cand = np.stack([rng.permutation(10)[:nb] for _ in range(4)]).astype(np.int32)
        si, end = oracle.candidate_expand(cand, cbs, ctx, 1, sparse_bs=sbs)
        assert si.shape == (4, nb * cbs // sbs)
        for r in range(4):
            want = sorted(b * cbs + o for b in cand[r].tolist() for o in range(cbs))
            got = [int(si[r, c // sbs]) * sbs + c % sbs for c in range(si.shape[1] * sbs)]
            assert got == want
            assert end[r] == sum(1 for t in want if t < ctx[r])
    with pytest.raises(ValueError):
        oracle.candidate_expand(cand, 8, ctx, 1, sparse_bs=3)


def _mxfp4_keys(rng, T, D):
    nib = rng.integers(0, 16, size=(T, D)).astype(np.uint8)
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    sf = rng.integers(125, 130, size=(T, D // 32)).astype(np.uint8)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    val = np.where(nib & 8, -1.0, 1.0) * grid[nib & 7] * np.exp2(np.repeat(sf.astype(np.float64) - 127, 32, axis=1))
    return packed, sf, val


def _fp4_cache(packed, sf, perm, page_tokens):
    T, Dh = packed.shape
    G = sf.shape[1]
    P = len(perm)
    kbytes = np.zeros((P, page_tokens, Dh), np.uint8)
    sbytes = np.zeros((P, page_tokens, G), np.uint8)
    for t in range(T):
        kbytes[perm[t // page_tokens], t % page_tokens] = packed[t]
        sbytes[perm[t // page_tokens], t % page_tokens] = sf[t]
    return kbytes.reshape(-1), page_tokens * Dh, sbytes.reshape(-1), page_tokens * G


def test_candidate_all_blocks_equals_dense_indexer():
    """Scoring every block of the context through the MXFP4 path equals Eq. (1)
    on the same key values held exactly as e4m3 codes with unit scale."""
    rng = np.random.default_rng(8)
    H, D, T, pt = 4, 64, 40, 8
    packed, sf, val = _mxfp4_keys(rng, T, D)
    q = e4m3_codes(rng.choice([-1, -0.5, 0.5, 1, 2], size=(1, H, D)).astype(np.float32)).reshape(1, H, D)
    qs = rng.uniform(0.5, 2, (1, H)).astype(np.float32)
    w = rng.normal(size=(1, H)).astype(np.float32)
    dense, _ = run_indexer(q, qs, w, e4m3_codes(val.astype(np.float32)), np.ones(T, np.float32),
                           page_tokens=pt, seed=0)
    perm = np.random.default_rng(0).permutation(T // pt)
    kb, ks, sb, ss = _fp4_cache(packed, sf, perm, pt)
    nblk = T // pt
    cand = np.random.default_rng(9).permutation(nblk).astype(np.int32)[None, :]
    ctx = np.array([T], np.int32)
    si, end = oracle.candidate_expand(cand, pt, ctx, 1)
    got, _ = oracle.candidate_logits(q, qs, w, kb, ks, sb, ss, pt, perm.astype(np.int32)[None, :],
                                     1, si, pt, end)
    assert end[0] == T
    np.testing.assert_allclose(got[0, :T], dense[0, :T], rtol=1e-14, atol=1e-300)


def test_candidate_subset_brute_force():
    rng = np.random.default_rng(10)
    H, D, T, pt = 2, 32, 48, 8
    packed, sf, val = _mxfp4_keys(rng, T, D)
    q = e4m3_codes(rng.choice([-1, 0.5, 1, 3], size=(1, H, D)).astype(np.float32)).reshape(1, H, D)
    qs = np.array([[0.5, 2.0]], np.float32)
    w = np.array([[1.5, -0.25]], np.float32)
    perm = np.arange(T // pt)[::-1].copy()
    kb, ks, sb, ss = _fp4_cache(packed, sf, perm, pt)
    cand = np.array([[5, 1, 3]], np.int32)
    ctx = np.array([T - 3], np.int32)  # block 5 is partial: 8 - 3 = 5 valid tokens
    si, end = oracle.candidate_expand(cand, pt, ctx, 1)
    assert end[0] == 8 + 8 + 5
    got, _ = oracle.candidate_logits(q, qs, w, kb, ks, sb, ss, pt, perm.astype(np.int32)[None, :],
                                     1, si, pt, end)
    qd = oracle.decode_e4m3(q).reshape(H, D) * qs.reshape(H, 1)
    for c in range(end[0]):
        tok = si[0, c // pt] * pt + c % pt
        ref = sum(Fraction(float(w[0, h])) * max(Fraction(0), sum(Fraction(qd[h, d]) * Fraction(val[tok, d]) for d in range(D)))
                  for h in range(H))
        assert got[0, c] == pytest.approx(float(ref), rel=1e-14, abs=1e-300)
    assert np.all(np.isnan(got[0, end[0]:]))


# ------------------------------------------------------------- sparse MLA --

def _bf16(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)


def mla_inputs(rng_seed, R=2, Hq=3, Dqk=12, Dv=8, T=20, pt=4):
    g = torch.Generator().manual_seed(rng_seed)
    q = torch.randn(R, Hq, Dqk, generator=g).to(torch.bfloat16)
    P = (T + pt - 1) // pt
    kv = torch.randn(P, pt, Dqk, generator=g).to(torch.bfloat16)
    perm = torch.randperm(P, generator=g).to(torch.int32)[None, :]
    return q, kv, perm


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def _tokens(kv, perm, pt, toks):
    """Latents of logical tokens (through the block table), float64."""
    return torch.stack([kv[int(perm[0, t // pt]), t % pt].double() for t in toks])


def test_mla_single_token_returns_its_value():
    q, kv, perm = mla_inputs(0)
    idx = np.full((2, 5), -1, np.int32)
    idx[0, 3] = 7
    idx[1, 0] = 19
    out, lse = oracle.sparse_mla(_bits(q), _bits(kv), 4 * 12, 4, perm.numpy(), 2, idx, 0.3, dv=8)
    for r, t in ((0, 7), (1, 19)):
        c = _tokens(kv, perm, 4, [t])[0]
        for g in range(3):
            assert np.array_equal(out[r, g], c[:8].numpy())
            z = 0.3 * float(q[r, g].double() @ c)
            assert lse[r, g] == pytest.approx(z, rel=1e-12, abs=1e-12)


def test_mla_equals_masked_dense_attention():
    """Sparse attention over the selection equals dense attention over every
    token with the others masked out (torch SDPA, fp64)."""
    q, kv, perm = mla_inputs(1, R=2, T=20)
    rng = np.random.default_rng(11)
    idx = np.stack([rng.permutation(20)[:9] for _ in range(2)]).astype(np.int32)
    idx[1, 4] = -1
    bt = np.repeat(perm.numpy(), 2, axis=0)  # two requests over the same pages
    out, lse = oracle.sparse_mla(_bits(q), _bits(kv), 4 * 12, 4, bt, 1, idx, 0.25, dv=8)
    for r in range(2):
        c = _tokens(kv, perm, 4, range(20))                     # [20, 12] (request r uses the same table)
        mask = torch.zeros(20, dtype=torch.bool)
        mask[[t for t in idx[r] if t >= 0]] = True
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[r].double()[None], c[None], c[None, :, :8], attn_mask=mask[None, None, :].expand(1, 3, 20),
            scale=0.25)[0]
        np.testing.assert_allclose(out[r], ref.numpy(), rtol=1e-12, atol=1e-13)
        s = 0.25 * (q[r].double() @ c.T)
        s[:, ~mask] = -math.inf
        np.testing.assert_allclose(lse[r], torch.logsumexp(s, -1).numpy(), rtol=1e-12)


def test_mla_all_tokens_equals_dense_attention():
    q, kv, perm = mla_inputs(2, R=1, T=16)
    idx = np.arange(16, dtype=np.int32)[None, ::-1].copy()
    out, _ = oracle.sparse_mla(_bits(q), _bits(kv), 4 * 12, 4, perm.numpy(), 1, idx, 0.5, dv=8)
    c = _tokens(kv, perm, 4, range(16))
    ref = torch.nn.functional.scaled_dot_product_attention(q[0].double()[None], c[None], c[None, :, :8], scale=0.5)[0]
    np.testing.assert_allclose(out[0], ref.numpy(), rtol=1e-12, atol=1e-13)


def test_mla_index_order_invariance_and_prefix_guard():
    q, kv, perm = mla_inputs(3, R=1, T=20)
    rng = np.random.default_rng(12)
    sel = rng.permutation(np.arange(6, 20))[:6].astype(np.int32)
    a, _ = oracle.sparse_mla(_bits(q), _bits(kv), 48, 4, perm.numpy(), 1, sel[None, :], 0.3, dv=8)
    b, _ = oracle.sparse_mla(_bits(q), _bits(kv), 48, 4, perm.numpy(), 1, sel[None, ::-1].copy(), 0.3, dv=8)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)
    # a selection of later tokens must not equal the first-k-tokens answer
    pre, _ = oracle.sparse_mla(_bits(q), _bits(kv), 48, 4, perm.numpy(), 1,
                               np.arange(6, dtype=np.int32)[None, :], 0.3, dv=8)
    assert np.abs(a - pre).max() > 1e-3


def test_mla_no_valid_index():
    q, kv, perm = mla_inputs(4, R=1)
    out, lse = oracle.sparse_mla(_bits(q), _bits(kv), 48, 4, perm.numpy(), 1,
                                 np.full((1, 4), -1, np.int32), 0.3, dv=8)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ----------------------------------------------------- layer schedule (MLI) --
def read_schedules(golden_dir):
    out = []
    with open(os.path.join(golden_dir, "layer_schedule.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, *kv = line.split()
            d = dict(x.split("=") for x in kv)
            out.append(([int(x) for x in d["keep"].split(",")], int(d["mli"]),
                        [int(x) for x in d["src"].split(",")]))
    return out


def test_layer_sources_hand_worked(golden_dir):
    cases = read_schedules(golden_dir)
    assert len(cases) == 10
    for keep, mli, src in cases:
        assert oracle.layer_sources(keep, mli) == src, (keep, mli)


def test_layer_sources_cumulative_max_form():
    """The same rule written another way: the latest indexer layer at or
    before l (sequential), or before l (MLI, first layer its own), as a
    running maximum over the kept layer numbers."""
    rng = np.random.default_rng(11)
    for _ in range(200):
        n = int(rng.integers(1, 17))
        keep = rng.integers(0, 2, n)
        keep[0] = 1
        kept_at = np.where(keep == 1, np.arange(n), -1)
        upto = np.maximum.accumulate(kept_at)            # latest kept j <= l
        before = np.concatenate([[0], upto[:-1]])         # latest kept j < l
        assert oracle.layer_sources(keep, False) == upto.tolist()
        assert oracle.layer_sources(keep, True) == before.tolist()


def test_layer_sources_invariants():
    rng = np.random.default_rng(12)
    for _ in range(100):
        n = int(rng.integers(2, 12))
        keep = rng.integers(0, 2, n)
        keep[0] = 1
        for mli in (False, True):
            src = oracle.layer_sources(keep, mli)
            for layer, j in enumerate(src):
                assert keep[j] == 1                        # attends a real selection
                assert j <= layer                          # never a later layer
                if mli and layer > 0:
                    assert j < layer                       # never its own (MLI)
    with pytest.raises(ValueError):
        oracle.layer_sources([0, 1, 1], False)


# ---------------------------------------------------- prefill chunk plan --
def read_plans(golden_dir):
    out = []
    with open(os.path.join(golden_dir, "prefill_chunks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kind, *kv = line.split()
            d = dict(x.split("=") for x in kv)
            out.append(([int(x) for x in d["q"].split(",")], [int(x) for x in d["ctx"].split(",")],
                        int(d["budget"]), int(d["min"]),
                        [tuple(int(y) for y in x.split(":")) for x in d["pieces"].split(",")]))
    return out


def test_prefill_chunk_plan_hand_worked(golden_dir):
    plans = read_plans(golden_dir)
    assert len(plans) == 5
    for q, ctx, budget, mn, pieces in plans:
        assert oracle.prefill_chunk_plan(q, ctx, budget, mn) == pieces, (q, ctx, budget, mn)


def test_prefill_chunk_plan_invariants():
    rng = np.random.default_rng(31)
    for _ in range(300):
        nreq = int(rng.integers(1, 8))
        q = rng.integers(0, 40, nreq)
        ctx = rng.integers(1, 5000, nreq)
        mn = int(rng.choice([0, 64, 2048]))
        budget = int(rng.integers(16, 200000))
        pieces = oracle.prefill_chunk_plan(q, ctx, budget, mn)
        width = [(max(int(c), mn) + 3) // 4 * 4 for c in ctx]
        # every row exactly once, in order
        rows = [(b, j) for c, b, j0, j1 in pieces for j in range(j0, j1)]
        assert rows == [(b, j) for b in range(nreq) for j in range(int(q[b]))]
        chunks = sorted({p[0] for p in pieces})
        assert chunks == list(range(len(chunks)))
        for ch in chunks:
            ps = [p for p in pieces if p[0] == ch]
            n = sum(p[3] - p[2] for p in ps)
            w = max(width[p[1]] for p in ps)
            # within budget unless it is a single row
            assert n * w * 4 <= budget or n == 1
            # maximal: the next row would not have fit
            nxt = [p for p in pieces if p[0] == ch + 1]
            if nxt:
                w2 = max(w, width[nxt[0][1]])
                assert (n + 1) * w2 * 4 > budget
