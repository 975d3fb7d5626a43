"""Edge cases through the C ABI vs the fp64 oracle: head ratios that force row
chunking, every decode head-dim variant with explicit splits, varlen with
seqused_k, sequences with no keys, odd head counts, split-KV on prefill
shapes, shifted diagonals and non-default scales."""
import dataclasses

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_attention_qk_gb300 import inputs  # noqa: E402
import gpu_util as gu  # noqa: E402


@pytest.mark.parametrize("ns", [0, 4])
def test_mqa_decode_32_heads_per_kv(ns):
    # Hq/Hkv = 32 packed rows: the prefill kernel, unsplit (ns=0) or in 4 key splits + combine
    w = inputs.batched("mqa", 101, 3, 1, 600, 32, 1, 128, 128,
                       seqused_k=np.array([600, 77, 300], np.int32))
    print(gu.check_workload(w, num_splits=ns))


@pytest.mark.parametrize("d,dv", [(64, 64), (192, 128), (256, 256)])
def test_decode_head_dims_explicit_splits(d, dv):
    w = inputs.batched("dechd", 102 + d, 4, 1, 900, 8, 2, d, dv,
                       seqused_k=np.array([900, 65, 1, 500], np.int32))
    print(gu.check_workload(w, num_splits=3))


def test_varlen_prefill_with_seqused():
    lens_q = [130, 257, 64]
    lens_k = [400, 300, 640]
    w = inputs.packed("vsu", 103, lens_q, lens_k, 4, 2, 128, 128, causal=True)
    # only a prefix of each sequence's keys is live; poison the rest
    w.seqused_k = np.array([390, 257, 100], np.int32)
    for b, used in enumerate(w.seqused_k):
        w.k[w.cu_seqlens_k[b] + used:w.cu_seqlens_k[b + 1]] = inputs.BF16_NAN_BITS
        w.v[w.cu_seqlens_k[b] + used:w.cu_seqlens_k[b + 1]] = inputs.BF16_NAN_BITS
    print(gu.check_workload(w))


def test_varlen_sequences_without_keys():
    lens_q = [50, 40, 200]
    lens_k = [0, 90, 200]
    w = inputs.packed("nokeys", 104, lens_q, lens_k, 2, 1, 128, 128, causal=False)
    o, l = gu.run_gpu(w)
    o_ref, l_ref = oracle.attention_forward(w.q, w.k, w.v, **gu.oracle_kw(w))
    print(gu.compare(o, l, o_ref, l_ref, "no keys"))
    assert np.isneginf(l[:, :50].cpu().numpy()).all() and (o[:50].float() == 0).all().item()


def test_batched_seqused_zero():
    w = inputs.batched("su0", 105, 3, 200, 300, 4, 4, 128, 128, seqused_k=np.array([0, 300, 129], np.int32))
    print(gu.check_workload(w))


def test_odd_heads_and_lengths():
    w = inputs.batched("odd", 106, 2, 257, 257, 12, 3, 128, 128, causal=True)
    print(gu.check_workload(w))


@pytest.mark.parametrize("ns", [2, 5])
def test_split_kv_on_prefill_shape(ns):
    # fa_fwd with an explicit split count on a prefill-shaped problem: the
    # prefill kernel over whole 128-key blocks per split, then the combine
    w = inputs.batched("pfsplit", 107, 1, 70, 700, 4, 2, 128, 128, causal=True, window_left=200)
    print(gu.check_workload(w, num_splits=ns))


@pytest.mark.parametrize("sq,sk", [(64, 300), (300, 64)])
def test_zero_width_window_shifted_diagonal(sq, sk):
    w = inputs.batched("diag", 108 + sq, 1, sq, sk, 2, 1, 64, 64, window_left=0, window_right=0)
    print(gu.check_workload(w))


@pytest.mark.parametrize("scale", [0.3, 0.02])
def test_explicit_scales(scale):
    w = inputs.batched("sc", 109, 1, 300, 300, 4, 2, 128, 128, scale=scale, causal=True)
    print(gu.check_workload(w))


def test_decode_repeat_is_bitwise_stable():
    w = inputs.batched("drep", 110, 8, 1, 3000, 32, 8, 128, 128,
                       seqused_k=inputs.uniform_lengths(7, 8, 1, 3000))
    o1, l1 = gu.run_gpu(w)
    o2, l2 = gu.run_gpu(w)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def _bf16_bits(x: float) -> np.uint16:
    return np.uint16(np.array([x], np.float32).view(np.uint32)[0] >> 16)


@pytest.mark.parametrize("d,dv,wl", [(128, 128, -1), (64, 64, -1), (192, 128, -1), (256, 256, -1),
                                     (128, 128, 100)])
def test_masked_keys_with_scores_far_above_the_visible_ones(d, dv, wl):
    """Keys a row must not see score about 150-290 (base 2, scaled) above every
    key it sees, inside the same key block. A block max taken over all of a
    masked block's columns would put every visible P of such a row below the
    float range; the kernel must notice and use the visible max."""
    w = inputs.batched("maskfar", 61, 1, 256, 256, 2, 1, d, dv, causal=True, window_left=wl)
    q, k = w.q.copy(), w.k.copy()
    q[..., 0] = _bf16_bits(8.0)
    if wl < 0:
        k[:, 64:128, :, 0] = _bf16_bits(200.0)    # rows 0-63 see none of these keys
    else:
        k[:, 0:100, :, 0] = _bf16_bits(200.0)     # rows 200+ see none of these keys
    w = dataclasses.replace(w, q=q, k=k)
    print(gu.check_workload(w))
