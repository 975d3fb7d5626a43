"""Pins of the fp64 backward oracle (CPU only): central finite differences of
a scalar loss through the oracle's own forward (independent of the gradient
formulas), torch autograd in float64 on a masked softmax, and closed forms."""
import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")


def _loss(q, k, v, w, **kw):
    o, _ = oracle.attention_forward(q, k, v, **kw)
    return float((o * w).sum())


@pytest.mark.parametrize("causal,wl,hq,hkv", [(False, -1, 2, 2), (True, -1, 4, 2), (True, 3, 2, 1)])
def test_finite_differences(causal, wl, hq, hkv):
    rng = np.random.default_rng(3)
    B, Sq, Sk, D = 1, 5, 7, 4
    q = rng.standard_normal((B, Sq, hq, D))
    k = rng.standard_normal((B, Sk, hkv, D))
    v = rng.standard_normal((B, Sk, hkv, D))
    w = rng.standard_normal((B, Sq, hq, D))     # dL/dO for L = sum(O * w)
    kw = dict(scale=0.7, causal=causal, window_left=wl)
    dq, dk, dv = oracle.attention_backward(q, k, v, w, **kw)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if a is x else a for a in (q, k, v)]
            args_m = [xm if a is x else a for a in (q, k, v)]
            num[idx] = (_loss(*args_p, w, **kw) - _loss(*args_m, w, **kw)) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=0, atol=1e-7)


def test_torch_autograd_float64():
    rng = np.random.default_rng(4)
    B, Sq, Sk, hq, hkv, D = 2, 6, 9, 4, 2, 8
    q = rng.standard_normal((B, Sq, hq, D))
    k = rng.standard_normal((B, Sk, hkv, D))
    v = rng.standard_normal((B, Sk, hkv, D))
    do = rng.standard_normal((B, Sq, hq, D))
    scale = 0.35
    dq, dk, dv = oracle.attention_backward(q, k, v, do, scale=scale, causal=True)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    kr = tk.repeat_interleave(hq // hkv, dim=2)
    vr = tv.repeat_interleave(hq // hkv, dim=2)
    s = torch.einsum("bihd,bjhd->bhij", tq, kr) * scale
    off = Sk - Sq
    i = torch.arange(Sq)[:, None]
    j = torch.arange(Sk)[None, :]
    s = s.masked_fill(j > i + off, float("-inf"))
    o = torch.einsum("bhij,bjhd->bihd", torch.softmax(s, dim=-1), vr)
    o.backward(torch.tensor(do))
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=0, atol=1e-12)


def test_closed_forms_with_zero_query():
    # q = 0: each row's P is uniform over its visible keys
    rng = np.random.default_rng(5)
    B, S, H, D = 1, 4, 1, 3
    q = np.zeros((B, S, H, D))
    k = rng.standard_normal((B, S, H, D))
    v = rng.standard_normal((B, S, H, D))
    do = rng.standard_normal((B, S, H, D))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=True)
    # row i sees keys 0..i with weight 1/(i+1): dV_j = sum_{i >= j} dO_i / (i + 1)
    exp_dv = np.stack([sum(do[0, i, 0] / (i + 1) for i in range(j, S)) for j in range(S)])
    np.testing.assert_allclose(dv[0, :, 0], exp_dv, rtol=0, atol=1e-12)
    # q = 0 makes every dK zero (dK_j = scale * sum_i dS_ij q_i)
    assert np.abs(dk).max() == 0.0


def test_rows_without_keys_have_zero_gradients():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((1, 6, 2, 4))
    k = rng.standard_normal((1, 3, 2, 4))
    v = rng.standard_normal((1, 3, 2, 4))
    do = rng.standard_normal((1, 6, 2, 4))
    # causal with Sq > Sk: the first Sq - Sk rows see no key
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=True)
    assert np.abs(dq[0, :3]).max() == 0.0
    assert np.isfinite(dk).all() and np.isfinite(dv).all()


def test_zero_output_gradient_gives_zero_gradients():
    rng = np.random.default_rng(7)
    q, k, v = (rng.standard_normal((1, 5, 2, 4)) for _ in range(3))
    grads = oracle.attention_backward(q, k, v, np.zeros((1, 5, 2, 4)), causal=True)
    assert all(np.abs(g).max() == 0.0 for g in grads)


def test_rows_seeing_one_key():
    # window [i, i] (causal, window_left 0): P is the identity, so O = V,
    # dV = dO, and dS = P (dP - D) = dO.v - dO.v = 0 gives dQ = dK = 0
    rng = np.random.default_rng(8)
    q, k, v, do = (rng.standard_normal((1, 6, 1, 4)) for _ in range(4))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=True, window_left=0)
    np.testing.assert_allclose(dv, do, rtol=0, atol=1e-15)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15


def test_constant_values_give_zero_query_and_key_gradients():
    # every v_j = c: O = c whatever P is, so the loss does not depend on q or k
    rng = np.random.default_rng(9)
    q, k, do = (rng.standard_normal((2, 5, 2, 4)) for _ in range(3))
    v = np.broadcast_to(rng.standard_normal(4), (2, 5, 2, 4)).copy()
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=True)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    # dV_j = sum_i P_ij dO_i still holds; its sum over keys is the sum of dO over rows
    np.testing.assert_allclose(dv.sum(axis=1), do.sum(axis=1), rtol=0, atol=1e-12)


def test_gqa_equals_explicit_repetition():
    rng = np.random.default_rng(10)
    q, do = (rng.standard_normal((1, 5, 4, 3)) for _ in range(2))
    k, v = (rng.standard_normal((1, 6, 2, 3)) for _ in range(2))
    dq, dk, dv = oracle.attention_backward(q, k, v, do, causal=True)
    rq, rk, rv = oracle.attention_backward(q, np.repeat(k, 2, axis=2), np.repeat(v, 2, axis=2), do, causal=True)
    np.testing.assert_allclose(dq, rq, rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk, rk.reshape(1, 6, 2, 2, 3).sum(axis=3), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, rv.reshape(1, 6, 2, 2, 3).sum(axis=3), rtol=0, atol=1e-14)


def test_hand_worked_golden_example():
    """tests/golden/hand_backward.txt: one query, two keys, solved by hand."""
    import math
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "hand_backward.txt")
    vals = {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if "=" in line:
            key, val = line.split("=", 1)
            vals[key.strip()] = val.strip()
    env = {"log": math.log}
    q = np.array(eval(vals["q"], env), float).reshape(1, 1, 1, -1)
    k = np.array(eval(vals["k"], env), float).reshape(1, 2, 1, -1)
    v = np.array(eval(vals["v"], env), float).reshape(1, 2, 1, -1)
    do = np.array(eval(vals["dO"], env), float).reshape(1, 1, 1, -1)
    dq, dk, dv = oracle.attention_backward(q, k, v, do, scale=float(vals["scale"]))
    np.testing.assert_allclose(dq[0, 0, 0], eval(vals["dQ"], env), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk[0, :, 0], eval(vals["dK"], env), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv[0, :, 0], eval(vals["dV"], env), rtol=0, atol=1e-14)


def test_seqused_k_finite_differences_and_unused_slots():
    """seqused_k: central finite differences of the forward oracle (with the
    same seqused_k) for every element, including cache slots past the used
    length, whose gradients must be exactly 0; NaN in those slots must not
    reach any gradient."""
    rng = np.random.default_rng(9)
    B, Sq, Sk, hq, hkv, D = 2, 4, 7, 2, 1, 3
    used = np.array([5, 2], np.int32)
    q = rng.standard_normal((B, Sq, hq, D))
    k = rng.standard_normal((B, Sk, hkv, D))
    v = rng.standard_normal((B, Sk, hkv, D))
    w = rng.standard_normal((B, Sq, hq, D))
    kw = dict(scale=0.6, causal=True, window_left=2, seqused_k=used)
    dq, dk, dv = oracle.attention_backward(q, k, v, w, **kw)
    eps = 1e-6
    for x, g in ((q, dq), (k, dk), (v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [xp if a is x else a for a in (q, k, v)]
            args_m = [xm if a is x else a for a in (q, k, v)]
            num[idx] = (_loss(*args_p, w, **kw) - _loss(*args_m, w, **kw)) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=0, atol=1e-7)
    for b in range(B):
        assert (dk[b, used[b]:] == 0).all() and (dv[b, used[b]:] == 0).all()
    kn, vn = k.copy(), v.copy()
    for b in range(B):
        kn[b, used[b]:] = np.nan
        vn[b, used[b]:] = np.nan
    gq, gk, gv = oracle.attention_backward(q, kn, vn, w, **kw)
    np.testing.assert_array_equal(gq, dq)
    np.testing.assert_array_equal(gk, dk)
    np.testing.assert_array_equal(gv, dv)
