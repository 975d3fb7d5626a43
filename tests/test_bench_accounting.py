"""The work counts every reported rate divides by (bench.py), on the CPU:
visible (row, key) pairs against the oracle's own mask, the headline's FLOPs
against their closed form, the backward's five GEMMs against the forward's
two, and decode bytes against a hand sum over the workload's lengths."""
import numpy as np
import pytest

import bench
import oracle
from exact_attention_qk_gb300 import inputs


@pytest.mark.parametrize("sq,sk", [(1, 1), (5, 3), (3, 5), (37, 53), (128, 129), (300, 64)])
@pytest.mark.parametrize("causal,wl,wr", [(False, -1, -1), (True, -1, -1), (True, 7, -1), (False, 4, 9),
                                          (False, 0, 0), (False, -1, 3), (False, 20, -1)])
def test_visible_pairs_match_the_oracle_mask(sq, sk, causal, wl, wr):
    want = int(oracle.visible_mask(sq, sk, causal, wl, wr).sum())
    assert bench.visible_pairs(sq, sk, causal, wl, wr) == want


def test_headline_flops_closed_form():
    # causal, Sq = Sk = 4096: row i sees i + 1 keys; 2 (Dqk + Dv) = 4 D per pair
    w = inputs.workload("causal")
    assert bench.flops(w) == 4 * 128 * (4096 * 4097 // 2) * 2 * 32


def test_backward_flops_are_five_gemms():
    w = inputs.workload("causal_bwd")
    assert bench.backward_flops(w) == pytest.approx(2.5 * bench.flops(w), rel=1e-15)
    # (192, 128): 2 (3*192 + 2*128) per pair against 2 (192 + 128)
    v = inputs.batched("acc", 1, 1, 10, 10, 2, 2, 192, 128)
    pairs = 10 * 10 * 2
    assert bench.backward_flops(v) == 2 * (3 * 192 + 2 * 128) * pairs


def test_decode_bytes_hand_sum():
    w = inputs.batched("accd", 5, 4, 1, 2048, 32, 8, 128, 128, seqused_k=np.array([2048, 1, 700, 1025], np.int32))
    used = w.seqused_k.astype(np.int64)
    hq, hkv, d = w.num_heads_q, w.num_heads_kv, w.head_dim_qk
    want = w.batch * hq * d * 2 + int(used.sum()) * hkv * 2 * d * 2 + w.batch * hq * d * 2 + w.batch * hq * 4
    assert bench.decode_bytes(w) == want
    # an fp8 cache moves one byte per K/V element, plus the two descales per (sequence, KV head)
    f = inputs.fp8_batched("acc8", 5, 4, 1, 2048, 32, 8, 128, "e4m3", seqused_k=w.seqused_k)
    want8 = want - int(used.sum()) * hkv * 2 * d + 2 * 4 * hkv * 4
    assert bench.decode_bytes(f) == want8
