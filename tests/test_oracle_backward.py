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
