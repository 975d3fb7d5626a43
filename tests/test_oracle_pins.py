"""Pins for the fp64 oracle: closed forms, invariants, an independent library
route and brute force, each chosen so that a plausible slip in the oracle (a
dropped term, a wrong sign or index, a transposed operand, a log2/ln mix-up,
a top-left instead of bottom-right causal diagonal, h % Hkv instead of h // r)
fails at least one of them. No GPU is needed.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.attention import _rows_attention  # noqa: F401  (import check only)
from exact_attention_qk_gb300 import inputs

RNG = np.random.default_rng(1234)


def rnd(*shape):
    return RNG.standard_normal(shape)


# ---- closed forms with q = 0: every visible score is 0 -----------------------
# => O_i = mean of the visible v_j, LSE_i = ln(#visible_i). This pins the mask,
#    the seqused handling, the LSE base and the bottom-right alignment at once.

def _zero_q_expect(v_rows, lo, hi):
    """mean of v over keys lo..hi inclusive and ln(count)."""
    n = hi - lo + 1
    return v_rows[lo:hi + 1].mean(axis=0), math.log(n)


@pytest.mark.parametrize("sq,sk", [(7, 7), (5, 9), (1, 6), (12, 12)])
def test_zero_query_causal_bottom_right(sq, sk):
    q = np.zeros((1, sq, 2, 4))
    k = rnd(1, sk, 2, 4)
    v = rnd(1, sk, 2, 3)
    o, lse = oracle.attention_forward(q, k, v, causal=True)
    off = sk - sq
    for h in range(2):
        for i in range(sq):
            eo, el = _zero_q_expect(v[0, :, h], 0, i + off)   # keys 0..i+off
            np.testing.assert_allclose(o[0, i, h], eo, rtol=0, atol=1e-12)
            assert abs(lse[0, h, i] - el) < 1e-12


@pytest.mark.parametrize("wl,wr", [(3, 0), (0, 0), (2, 1), (-1, 2), (4, -1)])
def test_zero_query_window(wl, wr):
    sq = sk = 10
    q = np.zeros((1, sq, 1, 4))
    k = rnd(1, sk, 1, 4)
    v = rnd(1, sk, 1, 2)
    o, lse = oracle.attention_forward(q, k, v, window_left=wl, window_right=wr)
    for i in range(sq):
        lo = 0 if wl < 0 else max(0, i - wl)
        hi = sk - 1 if wr < 0 else min(sk - 1, i + wr)
        eo, el = _zero_q_expect(v[0, :, 0], lo, hi)
        np.testing.assert_allclose(o[0, i, 0], eo, atol=1e-12)
        assert abs(lse[0, 0, i] - el) < 1e-12


def test_zero_query_seqused():
    B, sk_cap = 3, 11
    used = np.array([11, 4, 1], np.int32)
    q = np.zeros((B, 2, 2, 4))
    k = rnd(B, sk_cap, 1, 4)
    v = rnd(B, sk_cap, 1, 5)
    v[1, 4:] = np.nan        # slots past seqused must never be read
    k[1, 4:] = np.nan
    v[2, 1:] = np.nan
    o, lse = oracle.attention_forward(q, k, v, seqused_k=used)
    for b in range(B):
        for i in range(2):
            for h in range(2):
                eo, el = _zero_q_expect(v[b, :, 0], 0, used[b] - 1)
                np.testing.assert_allclose(o[b, i, h], eo, atol=1e-12)
                assert abs(lse[b, h, i] - el) < 1e-12


def test_zero_query_varlen_causal_window():
    lens = [5, 1, 9]
    cu = np.array([0, 5, 6, 15], np.int32)
    q = np.zeros((15, 2, 4))
    k = rnd(15, 2, 4)
    v = rnd(15, 2, 3)
    o, lse = oracle.attention_forward(q, k, v, causal=True, window_left=2,
                                      cu_seqlens_q=cu, cu_seqlens_k=cu)
    for b, n in enumerate(lens):
        s = cu[b]
        for i in range(n):
            eo, el = _zero_q_expect(v[s:s + n, 1], max(0, i - 2), i)
            np.testing.assert_allclose(o[s + i, 1], eo, atol=1e-12)
            assert abs(lse[1, s + i] - math.log(min(i, 2) + 1)) < 1e-12
            assert abs(lse[1, s + i] - el) < 1e-12


# ---- invariants the pages fix -------------------------------------------------

def test_rows_sum_to_one_via_one_hot_v():
    sq, sk = 6, 8
    q = rnd(1, sq, 1, 5)
    k = rnd(1, sk, 1, 5)
    v = np.eye(sk)[None, :, None, :]          # v_j = e_j  =>  O_i = P_i
    o, _ = oracle.attention_forward(q, k, v, causal=True)
    p = o[0, :, 0]
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-13)
    assert (p >= 0).all()
    off = sk - sq
    for i in range(sq):
        assert np.all(p[i, i + off + 1:] == 0.0)   # future keys get no weight


def test_constant_v_returns_constant():
    q = rnd(2, 9, 4, 8)
    k = rnd(2, 9, 2, 8)
    v = np.full((2, 9, 2, 6), 0.375)
    o, _ = oracle.attention_forward(q, k, v, causal=True, window_left=3)
    np.testing.assert_allclose(o, 0.375, atol=1e-14)


def test_first_causal_row_is_v0():
    q = rnd(1, 5, 1, 4)
    k = rnd(1, 5, 1, 4)
    v = rnd(1, 5, 1, 3)
    scale = 0.7
    o, lse = oracle.attention_forward(q, k, v, scale=scale, causal=True)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-14)
    assert abs(lse[0, 0, 0] - scale * float(q[0, 0, 0] @ k[0, 0, 0])) < 1e-12


@pytest.mark.parametrize("sq,sk,causal", [(6, 6, False), (4, 9, True), (6, 6, True)])
def test_zero_width_window_is_diagonal(sq, sk, causal):
    q = rnd(1, sq, 1, 4)
    k = rnd(1, sk, 1, 4)
    v = rnd(1, sk, 1, 3)
    o, lse = oracle.attention_forward(q, k, v, scale=0.5, causal=causal, window_left=0, window_right=0)
    off = sk - sq
    for i in range(sq):
        np.testing.assert_allclose(o[0, i, 0], v[0, i + off, 0], atol=1e-14)
        assert abs(lse[0, 0, i] - 0.5 * float(q[0, i, 0] @ k[0, i + off, 0])) < 1e-12


def test_gqa_equals_explicit_kv_repetition():
    r = 4
    q = rnd(2, 7, 8, 6)
    k = rnd(2, 7, 2, 6)
    v = rnd(2, 7, 2, 5)
    o1, l1 = oracle.attention_forward(q, k, v, causal=True)
    o2, l2 = oracle.attention_forward(q, np.repeat(k, r, axis=2), np.repeat(v, r, axis=2), causal=True)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_gqa_head_map_is_quotient():
    # kv group g has constant value g+1; head h must read group h // r (not h % Hkv)
    hq, hkv = 6, 3
    q = rnd(1, 4, hq, 4)
    k = rnd(1, 4, hkv, 4)
    v = np.zeros((1, 4, hkv, 2))
    for g in range(hkv):
        v[:, :, g] = g + 1
    o, _ = oracle.attention_forward(q, k, v)
    for h in range(hq):
        np.testing.assert_allclose(o[0, :, h], h // (hq // hkv) + 1, atol=1e-14)


def test_score_shift_moves_lse_only():
    # append a coordinate: q' = [q, c/scale], k' = [k, 1]  =>  s' = s + c
    c, scale = 2.5, 0.3
    q = rnd(1, 6, 2, 4)
    k = rnd(1, 6, 2, 4)
    v = rnd(1, 6, 2, 3)
    q2 = np.concatenate([q, np.full((1, 6, 2, 1), c / scale)], axis=-1)
    k2 = np.concatenate([k, np.ones((1, 6, 2, 1))], axis=-1)
    o1, l1 = oracle.attention_forward(q, k, v, scale=scale, causal=True)
    o2, l2 = oracle.attention_forward(q2, k2, v, scale=scale, causal=True)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l2 - l1, c, atol=1e-12)


def test_key_permutation_invariance_dense():
    q = rnd(1, 5, 2, 4)
    k = rnd(1, 8, 2, 4)
    v = rnd(1, 8, 2, 3)
    perm = RNG.permutation(8)
    o1, l1 = oracle.attention_forward(q, k, v)
    o2, l2 = oracle.attention_forward(q, k[:, perm], v[:, perm])
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


@pytest.mark.parametrize("S,L", [(1, 16), (2, 8), (3, 5), (5, 3), (6, 4)])
def test_split_then_combine_equals_unsplit(S, L):
    # (6, 4) has splits past every sequence's end (empty: O=0, LSE=-inf)
    used = np.array([13, 2, 9], np.int32)
    q = rnd(3, 3, 4, 4)
    k = rnd(3, 13, 2, 4)
    v = rnd(3, 13, 2, 3)
    kw = dict(causal=True, window_left=5, seqused_k=used)
    o, lse = oracle.attention_forward(q, k, v, **kw)
    op, lp = oracle.split_forward(q, k, v, S, L, **kw)
    if S * L < 13:
        pytest.skip("splits do not cover the keys")
    oc, lc = oracle.combine(op, np.swapaxes(lp, -1, -2))
    np.testing.assert_allclose(oc, o, atol=1e-13)
    np.testing.assert_allclose(lc, np.swapaxes(lse, -1, -2), atol=1e-13)


def test_combine_special_cases():
    o1 = rnd(4, 3)
    o2 = rnd(4, 3)
    ninf = np.full(4, -np.inf)
    # one split
    o, l = oracle.combine(o1[None], np.zeros((1, 4)) + 0.25)
    np.testing.assert_allclose(o, o1, atol=1e-15)
    np.testing.assert_allclose(l, 0.25)
    # equal weights: average, LSE + ln 2
    o, l = oracle.combine(np.stack([o1, o2]), np.zeros((2, 4)))
    np.testing.assert_allclose(o, (o1 + o2) / 2, atol=1e-15)
    np.testing.assert_allclose(l, math.log(2), atol=1e-15)
    # an empty split drops out, even with garbage O
    o, l = oracle.combine(np.stack([o1, np.full((4, 3), np.nan)]), np.stack([np.ones(4), ninf]))
    np.testing.assert_allclose(o, o1, atol=1e-15)
    np.testing.assert_allclose(l, 1.0)
    # all empty
    o, l = oracle.combine(np.stack([o1, o2]), np.stack([ninf, ninf]))
    assert (o == 0).all() and np.isneginf(l).all()


def test_empty_rows_and_sequences():
    q = rnd(2, 3, 1, 4)
    k = rnd(2, 5, 1, 4)
    v = rnd(2, 5, 1, 2)
    o, lse = oracle.attention_forward(q, k, v, seqused_k=np.array([0, 5], np.int32))
    assert (o[0] == 0).all() and np.isneginf(lse[0]).all()
    assert np.isfinite(lse[1]).all()
    # window that hides everything for the first rows: Sq > Sk with causal
    o, lse = oracle.attention_forward(rnd(1, 6, 1, 4), rnd(1, 2, 1, 4), rnd(1, 2, 1, 2), causal=True)
    assert np.isneginf(lse[0, 0, :4]).all() and (o[0, :4] == 0).all()   # off = -4
    assert np.isfinite(lse[0, 0, 4:]).all()
    # varlen with a zero-length query sequence
    cu_q = np.array([0, 0, 3], np.int32)
    cu_k = np.array([0, 4, 9], np.int32)
    o, lse = oracle.attention_forward(rnd(3, 1, 4), rnd(9, 1, 4), rnd(9, 1, 2),
                                      cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
    assert o.shape == (3, 1, 2) and np.isfinite(lse).all()


# ---- an independent library route: torch SDPA in float64 ---------------------

def _sdpa_ref(q, k, v, scale, causal, wl, wr):
    """torch SDPA + logsumexp with a mask built by torch.tril/triu offsets."""
    B, sq, hq, d = q.shape
    sk, hkv = k.shape[1], k.shape[2]
    r = hq // hkv
    qt = torch.from_numpy(q).permute(0, 2, 1, 3)
    kt = torch.from_numpy(k).permute(0, 2, 1, 3).repeat_interleave(r, dim=1)
    vt = torch.from_numpy(v).permute(0, 2, 1, 3).repeat_interleave(r, dim=1)
    off = sk - sq
    ones = torch.ones(sq, sk, dtype=torch.bool)
    mask = ones.clone()
    if causal:
        wr = 0
    if wr >= 0:
        mask &= torch.tril(ones, diagonal=off + wr)
    if wl >= 0:
        mask &= torch.triu(ones, diagonal=off - wl)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    s = (qt @ kt.transpose(-1, -2)) * scale
    lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy(), mask.numpy()


@pytest.mark.parametrize("case", [
    dict(B=2, sq=33, sk=33, hq=4, hkv=2, d=16, dv=16, causal=False, wl=-1, wr=-1),
    dict(B=1, sq=40, sk=40, hq=8, hkv=1, d=32, dv=16, causal=True, wl=-1, wr=-1),
    dict(B=2, sq=17, sk=50, hq=2, hkv=2, d=8, dv=24, causal=True, wl=-1, wr=-1),
    dict(B=1, sq=64, sk=64, hq=4, hkv=4, d=24, dv=8, causal=True, wl=7, wr=-1),
    dict(B=1, sq=30, sk=45, hq=6, hkv=3, d=8, dv=8, causal=False, wl=5, wr=3),
])
def test_matches_torch_sdpa_fp64(case):
    c = case
    q = rnd(c["B"], c["sq"], c["hq"], c["d"])
    k = rnd(c["B"], c["sk"], c["hkv"], c["d"])
    v = rnd(c["B"], c["sk"], c["hkv"], c["dv"])
    scale = 1.0 / math.sqrt(c["d"])
    o, lse = oracle.attention_forward(q, k, v, causal=c["causal"], window_left=c["wl"], window_right=c["wr"])
    so, sl, mask = _sdpa_ref(q, k, v, scale, c["causal"], c["wl"], c["wr"])
    ok = mask.any(axis=1)        # SDPA gives NaN on rows with no visible key
    np.testing.assert_allclose(o[:, ok], so[:, ok], atol=1e-12)
    np.testing.assert_allclose(np.swapaxes(lse, 1, 2)[:, ok], np.swapaxes(sl, 1, 2)[:, ok], atol=1e-12)


# ---- brute force on tiny inputs with Python floats ---------------------------

def test_brute_force_python_loops():
    sq, sk, hq, hkv, d, dv = 4, 6, 4, 2, 3, 2
    q = rnd(1, sq, hq, d)
    k = rnd(1, sk, hkv, d)
    v = rnd(1, sk, hkv, dv)
    scale, wl = 0.9, 2
    o, lse = oracle.attention_forward(q, k, v, scale=scale, causal=True, window_left=wl)
    off = sk - sq
    for h in range(hq):
        g = h // (hq // hkv)
        for i in range(sq):
            keys = [j for j in range(sk) if i + off - wl <= j <= i + off]
            sc = {j: scale * sum(q[0, i, h, t] * k[0, j, g, t] for t in range(d)) for j in keys}
            z = sum(math.exp(x) for x in sc.values())
            assert abs(lse[0, h, i] - math.log(z)) < 1e-12
            for t in range(dv):
                want = sum(math.exp(sc[j]) / z * v[0, j, g, t] for j in keys)
                assert abs(o[0, i, h, t] - want) < 1e-12


def test_hand_worked_example():
    """tests/golden/hand_example.txt: a 1x2 example solved by hand."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "hand_example.txt")
    vals = {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if "=" in line:
            key, val = line.split("=", 1)
            vals[key.strip()] = val.strip()
    q = np.array(eval(vals["q"]), float).reshape(1, 1, 1, -1)
    k = np.array(eval(vals["k"]), float).reshape(1, 2, 1, -1)
    v = np.array(eval(vals["v"]), float).reshape(1, 2, 1, -1)
    o, lse = oracle.attention_forward(q, k, v, scale=float(vals["scale"]))
    e = math.e
    want_o = np.array(eval(vals["O"], {"e": e}))
    want_lse = eval(vals["LSE"], {"e": e, "log": math.log})
    np.testing.assert_allclose(o[0, 0, 0], want_o, atol=1e-15)
    assert abs(lse[0, 0, 0] - want_lse) < 1e-15


def test_rows_helper_matches_full():
    w = inputs.batched("t", 7, 2, 37, 53, 4, 2, 16, 8, causal=True, window_left=9,
                       seqused_k=np.array([53, 20], np.int32))
    o, lse = oracle.attention_forward(w.q, w.k, w.v, causal=True, window_left=9, seqused_k=w.seqused_k)
    rows = [(0, 0, 0), (0, 3, 36), (1, 1, 5), (1, 2, 36)]
    ro, rl = oracle.attention_rows(w.q, w.k, w.v, rows, causal=True, window_left=9, seqused_k=w.seqused_k)
    for n, (b, h, i) in enumerate(rows):
        np.testing.assert_allclose(ro[n], o[b, i, h], atol=1e-14)
        assert rl[n] == lse[b, h, i] or abs(rl[n] - lse[b, h, i]) < 1e-13


def test_visible_count_closed_forms():
    n = 300
    assert oracle.visible_count(n, n, True, -1, -1) == n * (n + 1) // 2
    assert oracle.visible_count(n, n, False, -1, -1) == n * n
    wl = 17
    assert oracle.visible_count(n, n, True, wl, -1) == sum(min(i, wl) + 1 for i in range(n))
    assert oracle.visible_count(1, 1000, False, -1, -1) == 1000


# ---- widen(): bf16 bit patterns -> float64 ---------------------------------------
# Every GPU parity check hands the oracle raw bf16 bits (uint16), so the widening
# is pinned on its own: hand-decoded patterns (sign bit 15, biased exponent bits
# 14..7 with bias 127, seven mantissa bits), then all 65536 patterns against
# torch's bfloat16 -> float64 conversion (a library route).

@pytest.mark.parametrize("bits,want", [
    (0x3F80, 1.0),
    (0xC000, -2.0),
    (0x3F81, 1.0 + 2.0 ** -7),
    (0x4049, 3.140625),                         # 2 * (1 + 73/128)
    (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127),   # largest finite
    (0x0080, 2.0 ** -126),                      # smallest normal
    (0x0001, 2.0 ** -133),                      # smallest subnormal
    (0x7F80, math.inf),
    (0xFF80, -math.inf),
    (0x0000, 0.0),
])
def test_widen_bf16_hand_decoded(bits, want):
    got = oracle.widen(np.array([bits], np.uint16))
    assert got.dtype == np.float64
    assert got[0] == want


def test_widen_bf16_signed_zero_and_nan():
    got = oracle.widen(np.array([0x8000, 0x7FC0, 0xFFC1], np.uint16))
    assert got[0] == 0.0 and math.copysign(1.0, got[0]) == -1.0
    assert np.isnan(got[1]) and np.isnan(got[2])


def test_widen_bf16_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()
    assert (np.signbit(got[~nan]) == np.signbit(ref[~nan])).all()


def test_forward_on_bf16_bits_equals_forward_on_their_values():
    """The same tiny case given as bf16 bits and as the float values those bits
    stand for (decoded by torch) gives identical O and LSE."""
    w = inputs.batched("t", 11, 2, 9, 13, 4, 2, 16, 8, causal=True, window_left=5)
    vals = [torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
            for a in (w.q, w.k, w.v)]
    o_bits, l_bits = oracle.attention_forward(w.q, w.k, w.v, causal=True, window_left=5)
    o_vals, l_vals = oracle.attention_forward(*vals, causal=True, window_left=5)
    assert np.array_equal(o_bits, o_vals)
    assert np.array_equal(l_bits, l_vals)
