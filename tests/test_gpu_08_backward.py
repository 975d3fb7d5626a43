"""Attention backward through the C ABI vs the fp64 oracle: dQ, dK, dV for
head dims 64, 128, (192, 128) and 256 (the last two with the dK/dV kernel in
two passes and the streamed tiles in rings of their own), causal and
sliding-window masks with Sq != Sk, GQA and
MQA, ragged tails, empty axes, determinism, and the full-size causal workload
checked on one KV head group.

Tolerance. The kernels round P and dS to bf16 (relative error at most 2^-9 per
element) before the GEMMs that accumulate them in fp32, take D = rowsum(dO * O)
from the bf16 O of the forward, and round dQ, dK and dV to bf16 (again at most
2^-9 relative). The sums run over many terms of both signs, so an element's
error is about 2^-9 of its magnitude: per tensor, max|err| <= 1.5e-2 max|ref|
and mean|err| <= 4e-3 mean|ref| leave a margin of about 3 over that."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_attention_qk_gb300 import inputs  # noqa: E402
import gpu_util as gu  # noqa: E402

TOL_MAX_REL = 1.5e-2
TOL_MEAN_REL = 4e-3
# An all-zero reference that comes from cancellation (a row seeing one key:
# P = 1 and dS = dP - D = dO.v - dO.O = 0 exactly) leaves fp32 rounding behind:
# dP and D are dot products of at most 128 N(0,1) bf16 pairs (|.| <~ 50) summed
# in different orders, so |dP - D| <~ 50 x 2^-20 ~ 5e-5, and dQ / dK take it
# times scale (<= 1/8) times one key or query row (|.| <~ 5): below 1e-4.
TOL_CANCELLED_ZERO = 1e-4


def run_bwd(w, do_bits, concurrent=True):
    from exact_attention_qk_gb300 import fa
    q, k, v, do = gu.to_dev(w.q), gu.to_dev(w.k), gu.to_dev(w.v), gu.to_dev(do_bits)
    kw = dict(gu.kw_of(w))
    if w.varlen:
        kw.update(cu_seqlens_q=gu.i32(w.cu_seqlens_q), cu_seqlens_k=gu.i32(w.cu_seqlens_k),
                  max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k)
    if w.seqused_k is not None:
        kw["seqused_k"] = gu.i32(w.seqused_k)
    o, lse = fa.fa_fwd(q, k, v, **kw)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, lse, do, concurrent=concurrent, **kw)
    assert fa.fa_get_status() == fa.FA_OK
    return dq, dk, dv


def oracle_bwd(w, do_bits):
    kw = dict(scale=w.softmax_scale, causal=w.causal, window_left=w.window_left, window_right=w.window_right)
    if not w.varlen:
        return oracle.attention_backward(w.q, w.k, w.v, do_bits, seqused_k=w.seqused_k, **kw)
    # packed varlen: each sequence is its own batched problem of batch 1
    dq = np.zeros(w.q.shape, np.float64)
    dk = np.zeros(w.k.shape, np.float64)
    dv = np.zeros(w.v.shape, np.float64)
    cq, ck = w.cu_seqlens_q, w.cu_seqlens_k
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        if q1 == q0 or k1 == k0:
            continue   # no query row or no key: every gradient of the sequence is 0
        used = None if w.seqused_k is None else w.seqused_k[b:b + 1]
        rq, rk, rv = oracle.attention_backward(w.q[None, q0:q1], w.k[None, k0:k1], w.v[None, k0:k1],
                                               do_bits[None, q0:q1], seqused_k=used, **kw)
        dq[q0:q1], dk[k0:k1], dv[k0:k1] = rq[0], rk[0], rv[0]
    return dq, dk, dv


def compare(got, ref, what):
    g = gu.to64(got)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    err = np.abs(g - ref)
    mx, mean = float(np.abs(ref).max()) if ref.size else 0.0, float(np.abs(ref).mean()) if ref.size else 0.0
    if mx == 0.0:
        assert err.size == 0 or err.max() <= TOL_CANCELLED_ZERO, f"{what}: expected ~0, max|got| {err.max():.3e}"
        return f"{what}: zeros (max|got| {err.max() if err.size else 0.0:.1e})"
    assert err.max() <= TOL_MAX_REL * mx, f"{what}: max|err| {err.max():.3e} > {TOL_MAX_REL} x {mx:.3e}"
    assert err.mean() <= TOL_MEAN_REL * mean, f"{what}: mean|err| {err.mean():.3e} > {TOL_MEAN_REL} x {mean:.3e}"
    return f"{what}: max {err.max() / mx:.2e} mean {err.mean() / mean:.2e} (relative)"


def check_bwd(w):
    do = inputs.grad_out(w)
    got = run_bwd(w, do)
    ref = oracle_bwd(w, do)
    return "; ".join(compare(g, r, n) for g, r, n in zip(got, ref, ("dQ", "dK", "dV")))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dims_gqa(d, causal):
    # 300 rows: two full 128-row tiles and a 44-row tail; GQA 4/2
    w = inputs.batched("bwd", 400 + d, 2, 300, 300, 4, 2, d, d, causal=causal)
    print(check_bwd(w))


@pytest.mark.parametrize("causal", [False, True])
def test_head_dims_192_128(causal):
    # Dqk = 192, Dv = 128: 300 rows (two tiles and a tail), GQA 4/2
    w = inputs.batched("bwd192", 480 + causal, 2, 300, 300, 4, 2, 192, 128, causal=causal)
    print(check_bwd(w))


def test_head_dims_192_128_many_jobs_and_windows():
    # several query tiles per key block and q heads per KV head, so each single-stage
    # ring turns over many times; Sq != Sk with a two-sided window
    w = inputs.batched("bwd192j", 482, 1, 700, 600, 8, 2, 192, 128, causal=True)
    print(check_bwd(w))
    w2 = inputs.batched("bwd192w", 483, 2, 390, 450, 4, 1, 192, 128, window_left=150, window_right=60)
    print(check_bwd(w2))


def test_head_dims_192_128_varlen_window():
    # the varlen shape of the forward's sliding-window workload, small: causal, window 200
    lens = [300, 1, 129, 513, 64]
    w = inputs.packed("bwd192vl", 484, lens, lens, 4, 4, 192, 128, causal=True, window_left=200)
    print(check_bwd(w))


def test_head_dims_192_128_seqused_k():
    used = np.array([700, 1, 129], np.int32)
    w = inputs.batched("bwd192su", 485, 3, 200, 768, 4, 2, 192, 128, causal=True, seqused_k=used)
    print(check_bwd(w))


@pytest.mark.parametrize("sq,sk", [(200, 520), (520, 200), (1, 300), (300, 1), (128, 129), (129, 128)])
def test_causal_unequal_lengths(sq, sk):
    # bottom-right causal: with sq > sk the first sq - sk rows see no key (dQ = 0)
    w = inputs.batched("bwdne", 410 + sq % 97 + sk % 89, 1, sq, sk, 4, 1, 128, 128, causal=True)
    print(check_bwd(w))


@pytest.mark.parametrize("wl,wr", [(100, 0), (50, 70), (0, 0), (300, -1), (-1, 40)])
def test_sliding_window(wl, wr):
    w = inputs.batched("bwdw", 420 + max(wl, 0) + max(wr, 0), 2, 390, 450, 4, 2, 128, 128, window_left=wl,
                       window_right=wr)
    print(check_bwd(w))


def test_mqa_and_head_dim_64_window():
    w = inputs.batched("bwdmqa", 430, 1, 333, 333, 8, 1, 64, 64, causal=True, window_left=77)
    print(check_bwd(w))


def test_explicit_scale_and_several_kv_blocks():
    w = inputs.batched("bwdsc", 431, 1, 700, 1100, 2, 2, 128, 128, scale=0.05)
    print(check_bwd(w))


def test_tiny_shapes():
    for sq, sk in ((1, 1), (5, 3), (3, 5), (17, 17)):
        w = inputs.batched("bwdtiny", 432 + sq, 1, sq, sk, 2, 1, 64, 64, causal=(sq == 17))
        print(check_bwd(w))


def test_empty_query_axis_zeroes_dk_dv():
    from exact_attention_qk_gb300 import fa
    w = inputs.batched("bwdeq", 433, 1, 1, 200, 2, 1, 128, 128)
    q = torch.zeros(1, 0, 2, 128, dtype=torch.bfloat16, device="cuda")
    k, v = gu.to_dev(w.k), gu.to_dev(w.v)
    o = torch.zeros(1, 0, 2, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 2, 0, dtype=torch.float32, device="cuda")
    dk = torch.full_like(k, float("nan"))
    dv = torch.full_like(v, float("nan"))
    _, dk, dv = fa.fa_bwd(q, k, v, o, lse, o.clone(), dk=dk, dv=dv)
    assert fa.fa_get_status() == fa.FA_OK
    assert torch.count_nonzero(dk).item() == 0 and torch.count_nonzero(dv).item() == 0


def test_empty_key_axis_zeroes_dq():
    from exact_attention_qk_gb300 import fa
    w = inputs.batched("bwdek", 436, 1, 200, 1, 2, 1, 128, 128)
    q, do = gu.to_dev(w.q), gu.to_dev(inputs.grad_out(w))
    k = torch.zeros(1, 0, 1, 128, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.full((1, 2, 200), float("-inf"), dtype=torch.float32, device="cuda")
    dq = torch.full_like(q, float("nan"))
    dq, _, _ = fa.fa_bwd(q, k, k.clone(), o, lse, do, dq=dq)
    assert fa.fa_get_status() == fa.FA_OK
    assert torch.count_nonzero(dq).item() == 0


def test_keys_no_query_sees_get_zero_gradients():
    # a 100-key window behind each row: keys past the last row's window never count
    w = inputs.batched("bwdunseen", 434, 1, 150, 600, 2, 1, 128, 128, window_left=100, window_right=0)
    do = inputs.grad_out(w)
    dq, dk, dv = run_bwd(w, do)
    rq, rk, rv = oracle_bwd(w, do)
    assert np.all(rk[0, :350] == 0) and np.all(rv[0, :350] == 0)
    assert torch.count_nonzero(dk[0, :350]).item() == 0 and torch.count_nonzero(dv[0, :350]).item() == 0
    print(compare(dq, rq, "dQ"), compare(dk, rk, "dK"), compare(dv, rv, "dV"))


def test_deterministic():
    w = inputs.batched("bwddet", 435, 2, 600, 600, 8, 2, 128, 128, causal=True)
    do = inputs.grad_out(w)
    a = run_bwd(w, do)
    b = run_bwd(w, do)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_one_stream_equals_two_streams():
    """fa_bwd (every kernel on the caller's stream) and fa_bwd_two_streams (dK/dV
    on the caller's second stream) run the same kernels: the same bits."""
    w = inputs.batched("bwd1s", 436, 2, 700, 650, 8, 2, 128, 128, causal=True, window_left=200)
    do = inputs.grad_out(w)
    a = run_bwd(w, do, concurrent=False)
    b = run_bwd(w, do, concurrent=True)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    print(check_bwd(w))


@pytest.mark.parametrize("d", [64, 128])
def test_varlen_self_attention(d):
    # packed sequences of mixed lengths (one row, tails, several tiles), causal, GQA 8/2
    lens = [300, 1, 129, 513, 64]
    w = inputs.packed("bwdvl", 440 + d, lens, lens, 8, 2, d, d, causal=True)
    print(check_bwd(w))


def test_varlen_unequal_lengths_window_and_empty_sequences():
    # bottom-right causal with a window, Sq != Sk per sequence, a sequence
    # without keys (its dQ is 0) and one without queries (its dK, dV are 0)
    lens_q = [200, 77, 0, 300, 40]
    lens_k = [520, 77, 90, 0, 1000]
    w = inputs.packed("bwdvl2", 442, lens_q, lens_k, 4, 4, 128, 128, causal=True, window_left=150)
    print(check_bwd(w))


def test_varlen_dense_mqa():
    lens_q = [130, 257, 1]
    lens_k = [400, 300, 640]
    w = inputs.packed("bwdvl3", 443, lens_q, lens_k, 8, 1, 64, 64)
    print(check_bwd(w))


@pytest.mark.slow
def test_full_size_causal_one_kv_group():
    """The causal workload (B=2, S=4096, Hq=32, Hkv=4, D=128): every element of
    dK and dV of KV head 3 of sequence 1, and dQ of the 8 q heads reading it."""
    w = inputs.workload("causal")
    do = inputs.grad_out(w)
    dq, dk, dv = run_bwd(w, do)
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all().item()
    b, g, r = 1, 3, w.num_heads_q // w.num_heads_kv
    hs = slice(g * r, (g + 1) * r)
    rq, rk, rv = oracle.attention_backward(w.q[b:b + 1, :, hs], w.k[b:b + 1, :, g:g + 1], w.v[b:b + 1, :, g:g + 1],
                                           do[b:b + 1, :, hs], scale=w.softmax_scale, causal=True)
    print(compare(dq[b:b + 1, :, hs], rq, "dQ"), compare(dk[b:b + 1, :, g:g + 1], rk, "dK"),
          compare(dv[b:b + 1, :, g:g + 1], rv, "dV"))


@pytest.mark.parametrize("causal", [False, True])
def test_head_dims_256(causal):
    # D = 256: the dK/dV kernel in two passes, one stage of K / Q and V / dO in
    # halves through one slot; 300 rows (two tiles and a tail), GQA 4/2
    w = inputs.batched("bwd256", 490 + causal, 2, 300, 300, 4, 2, 256, 256, causal=causal)
    print(check_bwd(w))


def test_head_dims_256_varlen_window_and_seqused_k():
    lens = [300, 1, 129, 400]
    w = inputs.packed("bwd256vl", 492, lens, lens, 4, 2, 256, 256, causal=True, window_left=200)
    print(check_bwd(w))
    w2 = inputs.batched("bwd256su", 493, 3, 200, 768, 4, 2, 256, 256, causal=True,
                        seqused_k=np.array([700, 1, 129], np.int32))
    print(check_bwd(w2))


@pytest.mark.slow
def test_full_size_varlen_window_192_128_short_sequences():
    """The varlen sliding-window workload's backward (16 sequences, Hq=Hkv=16,
    Dqk=192, Dv=128, causal, window 1024) run at full size: every element of
    dQ, dK and dV of its five shortest sequences (425..837 rows, all heads)."""
    w = inputs.workload("varlen_bwd")
    do = inputs.grad_out(w)
    dq, dk, dv = run_bwd(w, do)
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all().item()
    cq, ck = w.cu_seqlens_q, w.cu_seqlens_k
    lens = np.diff(cq)
    kw = dict(scale=w.softmax_scale, causal=True, window_left=w.window_left, window_right=w.window_right)
    for b in np.argsort(lens)[:5]:
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        rq, rk, rv = oracle.attention_backward(w.q[None, q0:q1], w.k[None, k0:k1], w.v[None, k0:k1],
                                               do[None, q0:q1], **kw)
        print(int(b), q1 - q0, compare(dq[q0:q1], rq[0], "dQ"), compare(dk[k0:k1], rk[0], "dK"),
              compare(dv[k0:k1], rv[0], "dV"))


@pytest.mark.parametrize("d", [64, 128])
def test_seqused_k_with_nan_cache_slots(d):
    """seqused_k: keys [0, seqused_k[b]) exist; the cache slots past them hold
    NaN, which must not reach any gradient, and their dK and dV are written 0."""
    used = np.array([700, 1, 129, 300], np.int32)   # a tail inside a block, one key, 128+1, ...
    w = inputs.batched("bwdsu", 450 + d, 4, 200, 768, 8, 2, d, d, causal=True, seqused_k=used)
    print(check_bwd(w))
    w2 = inputs.batched("bwdsu2", 460 + d, 3, 257, 512, 4, 4, d, d, window_left=100, window_right=30,
                        seqused_k=np.array([512, 95, 260], np.int32))
    print(check_bwd(w2))


def test_seqused_k_varlen():
    """seqused_k with packed varlen: each sequence's keys [0, seqused_k[b]) of
    its cu_seqlens_k rows exist; the rest of its rows get dK = dV = 0 and the
    next sequence's rows are not touched."""
    lens_q = [130, 64, 1, 300]
    lens_k = [400, 64, 260, 300]
    w = inputs.packed("bwdsuvl", 470, lens_q, lens_k, 8, 2, 128, 128, causal=True)
    used = np.array([257, 64, 3, 150], np.int32)
    w.seqused_k = used
    for b in range(len(used)):   # NaN in every slot past the used keys
        k0, k1 = int(w.cu_seqlens_k[b]), int(w.cu_seqlens_k[b + 1])
        w.k[k0 + used[b]:k1] = inputs.BF16_NAN_BITS
        w.v[k0 + used[b]:k1] = inputs.BF16_NAN_BITS
    print(check_bwd(w))
