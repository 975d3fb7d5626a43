"""tcgen05 prefill through the C ABI vs the fp64 oracle, on sizes the oracle
finishes in seconds that still span several 128-row / 128-key tiles and end in
a ragged tail; every head-dim variant, mask kind and layout."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_attention_qk_gb300 import inputs  # noqa: E402
import gpu_util as gu  # noqa: E402


def test_tiny_workload():
    print(gu.check_workload(inputs.workload("tiny")))


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (192, 128), (256, 256)])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dims(d, dv, causal):
    w = inputs.batched("hd", 30 + d, 2, 600, 600, 4, 2, d, dv, causal=causal)
    print(gu.check_workload(w))


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 1), (16, 2)])
def test_gqa_mqa(hq, hkv):
    w = inputs.batched("gqa", 40 + hq + hkv, 1, 384, 384, hq, hkv, 128, 128, causal=True)
    print(gu.check_workload(w))


@pytest.mark.parametrize("sq,sk,causal", [(200, 500, True), (500, 200, True), (130, 700, False), (1000, 129, False)])
def test_unequal_lengths_bottom_right(sq, sk, causal):
    w = inputs.batched("neq", 50 + sq, 1, sq, sk, 4, 2, 128, 128, causal=causal)
    print(gu.check_workload(w))


@pytest.mark.parametrize("wl,wr,causal", [(100, -1, True), (0, 0, False), (37, 200, False), (-1, 5, False),
                                         (300, 0, False)])
def test_windows(wl, wr, causal):
    w = inputs.batched("win", 60 + wl, 1, 700, 700, 4, 1, 128, 128, causal=causal, window_left=wl,
                       window_right=wr)
    print(gu.check_workload(w))


def test_window_256_head():
    w = inputs.batched("win256", 61, 1, 520, 520, 2, 1, 256, 256, causal=True, window_left=150)
    print(gu.check_workload(w))


def test_varlen_causal_window_192():
    lens = [300, 5, 777, 129, 1, 256]
    w = inputs.packed("var", 70, lens, lens, 4, 4, 192, 128, causal=True, window_left=100, window_right=0)
    print(gu.check_workload(w))


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (256, 256)])
def test_varlen_unequal_q_k(d, dv):
    lens_q = [100, 300, 17, 0, 257]
    lens_k = [400, 300, 17, 50, 600]
    w = inputs.packed("varqk", 71 + d, lens_q, lens_k, 4, 2, d, dv, causal=True)
    print(gu.check_workload(w))


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (192, 128), (256, 256)])
def test_prefill_seqused_k_nan_padding(d, dv):
    # cache slots past seqused_k hold NaN: prefill loads them with the tile but
    # must never let them into O (tail V rows cleared, S columns masked)
    w = inputs.batched("pfsu", 80 + d, 3, 300, 640, 4, 2, d, dv, causal=True,
                       seqused_k=np.array([640, 300, 431], np.int32))
    print(gu.check_workload(w))


def test_strided_output_with_canaries():
    from exact_attention_qk_gb300 import fa
    w = inputs.batched("can", 90, 2, 333, 333, 4, 2, 128, 128, causal=True)
    q, k, v = gu.to_dev(w.q), gu.to_dev(w.k), gu.to_dev(w.v)
    # out is a view with one guard row before and after each sequence and a guard head
    big = torch.full((2, 333 + 2, 5, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    out = big[:, 1:-1, :4]
    lse_big = torch.full((2 * 4 * 333 + 64,), 7.0, dtype=torch.float32, device="cuda")
    lse = lse_big[32:-32].view(2, 4, 333)
    fa.fa_fwd(q, k, v, out=out, lse=lse, **gu.kw_of(w))
    assert fa.fa_get_status() == fa.FA_OK
    torch.cuda.synchronize()
    assert (big[:, 0] == 7).all() and (big[:, -1] == 7).all() and (big[:, :, 4] == 7).all()
    assert (lse_big[:32] == 7).all() and (lse_big[-32:] == 7).all()
    o_ref, l_ref = oracle.attention_forward(w.q, w.k, w.v, **gu.oracle_kw(w))
    print(gu.compare(out, lse, o_ref, l_ref, "strided"))


def test_rows_without_keys():
    # Sq > Sk with causal bottom-right alignment: the first rows see nothing
    w = inputs.batched("nokey", 95, 1, 400, 150, 2, 1, 128, 128, causal=True)
    print(gu.check_workload(w))


def test_repeat_calls_are_bitwise_stable():
    w = inputs.batched("rep", 96, 1, 512, 512, 8, 2, 128, 128, causal=True)
    o1, l1 = gu.run_gpu(w)
    o2, l2 = gu.run_gpu(w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def _scale_rows(bits, factors, axis_len):
    """Multiply row j (axis 1 of a [B, S, H, D] tensor) by factors[j], back to bf16."""
    x = inputs.bf16_bits_to_f32(bits).astype(np.float64)
    x *= factors.reshape(1, axis_len, 1, 1)
    return inputs.f32_to_bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (192, 128), (256, 256)])
@pytest.mark.parametrize("causal", [False, True])
def test_running_max_grows_every_block(d, dv, causal):
    """Keys grow in magnitude toward the start of the sequence. Key blocks run
    from the last one down, so nearly every block raises some row's max by
    more than the lazy-rescale threshold: O and l are rescaled (and the block
    exponentiated again) block after block. Such sharp rows make O close to a
    single V row, so V is scaled down to keep |O| (and its bf16 rounding) small."""
    sk = 1000
    w = inputs.batched("grow", 130 + d, 1, 300, sk, 4, 2, d, dv, causal=causal)
    blocks = np.arange(sk) // 128
    w.k = _scale_rows(w.k, 1.0 + 1.3 * (blocks.max() - blocks), sk)
    w.v = _scale_rows(w.v, np.full(sk, 0.25), sk)
    print(gu.check_workload(w))


def test_running_max_grows_for_some_rows_only():
    """Only odd query rows see growing maxima (their q is large), so a warp
    mixes rows that rescale with rows that keep their base."""
    sq, sk = 260, 900
    w = inputs.batched("growmix", 139, 1, sq, sk, 4, 4, 128, 128, causal=True)
    blocks = np.arange(sk) // 128
    w.k = _scale_rows(w.k, 1.0 + 0.9 * (blocks.max() - blocks), sk)
    w.q = _scale_rows(w.q, np.where(np.arange(sq) % 2 == 1, 2.5, 0.3), sq)
    w.v = _scale_rows(w.v, np.full(sk, 0.25), sk)
    print(gu.check_workload(w))
