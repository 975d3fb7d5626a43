"""Pins of the oracle's KV-cache forms (CPU only): fp8 decoding against the
formats' own landmarks and torch's float8 conversions, descales, and the page
gather against hand-written cases and a scatter/gather round trip."""
import numpy as np
import pytest

import oracle
from exact_attention_qk_gb300 import inputs

torch = pytest.importorskip("torch")


@pytest.mark.parametrize("fmt,tdtype", [("e4m3", "float8_e4m3fn"), ("e5m2", "float8_e5m2")])
def test_fp8_decode_matches_torch_for_every_code(fmt, tdtype):
    if not hasattr(torch, tdtype):
        pytest.skip(f"torch has no {tdtype}")
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.fp8_to_float(codes, fmt)
    ref = torch.from_numpy(codes).view(getattr(torch, tdtype)).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert np.array_equal(mine[fin], ref[fin])


def test_fp8_landmarks_from_the_pages_and_the_format():
    e4 = oracle.fp8_to_float(np.arange(256, dtype=np.uint8), "e4m3")
    e5 = oracle.fp8_to_float(np.arange(256, dtype=np.uint8), "e5m2")
    # largest finite values (the FP8 max_offset passage: 448 and 57344)
    assert np.nanmax(e4[np.isfinite(e4)]) == 448.0
    assert np.nanmax(e5[np.isfinite(e5)]) == 57344.0
    # e4m3 has no infinities and one NaN per sign; e5m2 has +-inf at 0x7C / 0xFC
    assert not np.isinf(e4).any() and np.isnan(e4).sum() == 2 and np.isnan(e4[0x7F])
    assert e5[0x7C] == np.inf and e5[0xFC] == -np.inf and np.isnan(e5).sum() == 6
    # smallest subnormals 2^-9 and 2^-16, signed zero, one
    assert e4[0x01] == 2.0 ** -9 and e5[0x01] == 2.0 ** -16
    assert e4[0x00] == 0.0 and np.signbit(e4[0x80]) and e4[0x38] == 1.0 and e5[0x3C] == 1.0
    # a few hand-decoded codes: e4m3 0x4B = 0 1001 011 = 2^2 * 1.375; e5m2 0xC6 = 1 10001 10 = -2^2 * 1.5
    assert e4[0x4B] == 5.5 and e5[0xC6] == -6.0


def test_generated_codes_stay_in_their_window():
    for fmt in inputs.FP8_FORMATS:
        c = inputs.fp8_codes(1, 1, 0, (4096,), fmt)
        v = np.abs(oracle.fp8_to_float(c, fmt))
        assert np.isfinite(v).all() and v.min() >= 0.125 and v.max() < 2.0


def test_dequant_applies_the_descale_of_each_sequence_and_head():
    codes = np.array([0x38, 0x40, 0xB8], np.uint8)       # 1, 2, -1 in e4m3
    k = np.broadcast_to(codes[None, :, None, None], (2, 3, 2, 1)).copy()
    ds = np.array([[0.5, 2.0], [3.0, 0.25]], np.float32)
    out = oracle.dequant_kv(k, ds, "e4m3")
    assert out[0, :, 0, 0].tolist() == [0.5, 1.0, -0.5]
    assert out[0, :, 1, 0].tolist() == [2.0, 4.0, -2.0]
    assert out[1, :, 0, 0].tolist() == [3.0, 6.0, -3.0]
    assert out[1, :, 1, 0].tolist() == [0.25, 0.5, -0.25]


def test_gather_pages_hand_case():
    # 3 pages of 2 rows; sequence 0 uses pages 2 then 0, sequence 1 uses page 1 then 2
    pool = np.arange(3 * 2).reshape(3, 2, 1, 1) * 10
    table = np.array([[2, 0], [1, 2]], np.int32)
    out = oracle.gather_pages(pool, table, 2)
    assert out[:, :, 0, 0].tolist() == [[40, 50, 0, 10], [20, 30, 40, 50]]


def test_paged_workload_round_trip():
    w = inputs.batched("pg", 11, 3, 2, 256, 4, 2, 64, 64, seqused_k=np.array([256, 70, 129], np.int32))
    p = inputs.to_paged(w, 64)
    assert p.k.shape == (3 * 4 + 3, 64, 2, 64)
    assert sorted(p.page_table.reshape(-1).tolist()) == sorted(set(p.page_table.reshape(-1).tolist()))
    for src, pool in ((w.k, p.k), (w.v, p.v)):
        g = oracle.gather_pages(pool, p.page_table, 64)
        assert np.array_equal(g, src)
    # and the oracle's plain view gives the same attention as the original layout
    k0, v0 = oracle.plain_kv(w)
    k1, v1 = oracle.plain_kv(p)
    o0, l0 = oracle.attention_forward(w.q, k0, v0, seqused_k=w.seqused_k)
    o1, l1 = oracle.attention_forward(p.q, k1, v1, seqused_k=p.seqused_k)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
