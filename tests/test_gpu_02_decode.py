"""Split-KV decode and combine through the C ABI vs the fp64 oracle."""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_attention_qk_gb300 import inputs  # noqa: E402
import gpu_util as gu  # noqa: E402


def _decode_wl(B=6, cap=700, hq=8, hkv=2, d=128, dv=128, seed=11, sq=1, used=None, **kw):
    if used is None:
        used = inputs.uniform_lengths(seed + 100, B, 1, cap)
    return inputs.batched("dec", seed, B, sq, cap, hq, hkv, d, dv, seqused_k=np.asarray(used, np.int32), **kw)


@pytest.mark.parametrize("ns", [0, 1, 2, 3, 16])
def test_decode_seqused_nan_padding(ns):
    # cache slots past seqused_k hold NaN: any use of them would show in O
    w = _decode_wl(used=[700, 1, 64, 65, 300, 129])
    print(gu.check_workload(w, num_splits=ns))


@pytest.mark.parametrize("hq,hkv,d,dv", [(8, 8, 64, 64), (16, 2, 128, 128), (4, 1, 192, 128),
                                         (8, 4, 256, 256), (16, 1, 128, 128)])
def test_decode_head_shapes(hq, hkv, d, dv):
    w = _decode_wl(B=3, cap=333, hq=hq, hkv=hkv, d=d, dv=dv, seed=d + hq)
    print(gu.check_workload(w))


@pytest.mark.parametrize("sq,causal,wl", [(2, True, -1), (3, False, 17), (4, True, 40)])
def test_decode_multi_row_masks(sq, causal, wl):
    w = _decode_wl(B=2, cap=300, hq=4, hkv=1, sq=sq, causal=causal, window_left=wl,
                   used=[300, 150])
    print(gu.check_workload(w))


def test_decode_varlen():
    lens_q = [1, 1, 2, 1]
    lens_k = [900, 17, 333, 1]
    w = inputs.packed("decvar", 21, lens_q, lens_k, 8, 2, 128, 128, causal=True)
    print(gu.check_workload(w))
    print(gu.check_workload(w, num_splits=5))


def test_splitkv_partials_and_combine():
    from exact_attention_qk_gb300 import fa
    w = _decode_wl(B=4, cap=1000, used=[1000, 10, 513, 257], seed=5)
    q, k, v = gu.to_dev(w.q), gu.to_dev(w.k), gu.to_dev(w.v)
    su = gu.i32(w.seqused_k)
    ns = 4
    args = fa.make_args(q, k, v, seqused_k=su, softmax_scale=w.softmax_scale)
    L = fa.fa_split_len(args, ns)
    assert L == 64 * math.ceil(math.ceil(1000 / ns) / 64)
    op, lp = fa.fa_fwd_splitkv(q, k, v, ns, seqused_k=su, softmax_scale=w.softmax_scale)
    assert fa.fa_get_status() == fa.FA_OK
    o_s, l_s = oracle.split_forward(w.q, w.k, w.v, ns, L, scale=w.softmax_scale, seqused_k=w.seqused_k)
    opg = op.cpu().numpy().astype(np.float64)
    lpg = lp.cpu().numpy().astype(np.float64)
    fin = np.isfinite(l_s)
    assert (np.isneginf(lpg[~fin])).all()          # empty splits
    assert np.abs(lpg[fin] - l_s[fin]).max() <= gu.TOL_MAX_LSE
    # partial O rows of empty splits are 0; the others carry the rounding of P
    # to bf16 ahead of the P.V product (as every P.V here does), so they meet
    # the output tolerances
    d = np.abs(opg - o_s)
    assert d.max() <= gu.TOL_MAX_O and d.mean() <= gu.TOL_MEAN_O
    out, lse = fa.fa_combine(op, lp)
    o_ref, l_ref = oracle.attention_forward(w.q, w.k, w.v, scale=w.softmax_scale, seqused_k=w.seqused_k)
    print(gu.compare(out, lse, o_ref, l_ref, "combine"))


def test_combine_all_empty_and_single_split():
    from exact_attention_qk_gb300 import fa
    op = torch.randn(3, 2, 1, 4, 128, device="cuda")
    lp = torch.full((3, 2, 4, 1), float("-inf"), device="cuda")
    lp[1, 0] = 0.5
    op[0] = float("nan")       # an empty split's O is never read
    out, lse = fa.fa_combine(op, lp)
    torch.cuda.synchronize()
    o = out.float().cpu().numpy()
    assert np.isneginf(lse[1].cpu().numpy()).all() and (o[1] == 0).all()
    np.testing.assert_allclose(o[0], op[1, 0].cpu().numpy(), atol=1e-2)
    np.testing.assert_allclose(lse[0].cpu().numpy(), 0.5, atol=1e-6)
