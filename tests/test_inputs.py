"""The seeded input generator: bf16 rounding and determinism (no GPU)."""
import numpy as np

from exact_attention_qk_gb300 import inputs


def test_bf16_round_nearest_even():
    f = np.array([0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F808001, 0xBF808000, 0x00000000],
                 np.uint32).view(np.float32)
    got = inputs.f32_to_bf16_bits(f)
    # halfway cases go to the even mantissa; others to the nearest
    assert list(got) == [0x3F80, 0x3F82, 0x3F80, 0x3F81, 0xBF80, 0x0000]
    assert inputs.bf16_bits_to_f32(np.array([0x3F80, 0xC000, 0x3F81], np.uint16)).tolist() == \
        [1.0, -2.0, 1.0 + 2.0 ** -7]


def test_blocks_are_reproducible_and_independent():
    a = inputs.normal_bf16(5, 1, 3, (4, 2, 8))
    b = inputs.normal_bf16(5, 1, 3, (4, 2, 8))
    c = inputs.normal_bf16(5, 1, 4, (4, 2, 8))
    assert (a == b).all() and not (a == c).all()
    w = inputs.batched("t", 9, 3, 2, 10, 2, 1, 8, 8, seqused_k=np.array([10, 3, 7], np.int32))
    assert (w.k[1, 3:] == inputs.BF16_NAN_BITS).all()
    assert (w.k[1, :3] == inputs.normal_bf16(9, 1, 1, (3, 1, 8))).all()


def test_named_workload_lengths():
    lens = inputs.varlen_lengths()
    assert lens.shape == (16,) and lens.min() >= 256 and lens.max() <= 8192
    used = inputs.decode_seqused()
    assert used.shape == (64,) and used.min() >= 1024 and used.max() <= 16384
    t = inputs.workload("tiny")
    assert t.q.shape == (1, 128, 2, 64) and abs(t.softmax_scale - 0.125) < 1e-15
