"""KV-cache forms of the attention inputs, for the fp64 oracle.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg use this module; the product path never imports it, and it shares
no code with the CUDA library.

Two forms turn into the plain (batched) K and V that `attention_forward` takes:

  * an fp8 cache: one byte per element, in the E4M3 or E5M2 format, with a
    descale per (sequence b, KV head g); the element's value is
        code value x descale[b, g]
  * a paged cache: K and V are pools of pages (num_pages, page_size, Hkv, D);
    key j of sequence b is row j % page_size of page page_table[b, j // page_size]

Sources (page title, then the passage):
  * the FlashAttention sm_120 pull-request page, "fp8 KV-cache decode
    (e4m3/e5m2)": a bf16 query against a quantized K/V cache with per-(batch,
    kv_head) k_descale / v_descale, checked against an fp8-quantized reference,
    i.e. attention over the dequantized cache.
  * "[CuTe, SM100] Make FP8 max_offset dtype-aware ...": e4m3fn's largest
    finite value is 448 and e5m2's is 57344 (pinned in the tests).
  * "mslk/attention/flash_attn/interface.py", `_flash_attn_fwd`: page_table is
    int32 (batch, max_num_pages_per_seq); k and v are (num_pages, page_size,
    num_head_kv, head_dim); the key capacity is max_num_pages_per_seq x page_size.

The bit layouts are those of the 8-bit floating-point formats the pages name:
  E4M3 ("fn"): sign, 4 exponent bits (bias 7), 3 mantissa bits; no infinities;
               exponent and mantissa all ones is NaN.
  E5M2:        sign, 5 exponent bits (bias 15), 2 mantissa bits; IEEE-style
               infinities (exponent all ones, mantissa 0) and NaNs.
  Exponent field 0 encodes subnormals: 2^(1 - bias) x mantissa / 2^mbits.
Reading where the pages are silent: key j of sequence b lives on page
page_table[b, j // page_size] at row j % page_size (pages fill in key order).
"""
from __future__ import annotations

import numpy as np

_FIELDS = {
    # format: (exponent bits, mantissa bits, bias)
    "e4m3": (4, 3, 7),
    "e5m2": (5, 2, 15),
}


def fp8_to_float(codes, fmt: str) -> np.ndarray:
    """Value of each fp8 code (uint8) in float64, NaN and +-inf included."""
    if fmt not in _FIELDS:
        raise ValueError(fmt)
    ebits, mbits, bias = _FIELDS[fmt]
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> mbits) & ((1 << ebits) - 1)
    m = c & ((1 << mbits) - 1)
    frac = m.astype(np.float64) / float(1 << mbits)
    normal = np.ldexp(1.0 + frac, (e - bias).astype(np.int64))
    subnormal = np.ldexp(frac, 1 - bias)
    val = sign * np.where(e > 0, normal, subnormal)
    e_max = (1 << ebits) - 1
    if fmt == "e4m3":
        nan = (e == e_max) & (m == (1 << mbits) - 1)
        inf = np.zeros_like(nan)
    else:
        nan = (e == e_max) & (m != 0)
        inf = (e == e_max) & (m == 0)
    val = np.where(inf, sign * np.inf, val)
    return np.where(nan, np.nan, val)


def dequant_kv(codes, descale, fmt: str) -> np.ndarray:
    """codes (B, S, Hkv, D) uint8, descale (B, Hkv) -> float64 (B, S, Hkv, D)."""
    vals = fp8_to_float(codes, fmt)
    ds = np.asarray(descale, dtype=np.float64)
    return vals * ds[:, None, :, None]


def gather_pages(pool, page_table, page_size: int) -> np.ndarray:
    """Page pool (num_pages, page_size, Hkv, D) -> batched (B, max_pages*page_size, Hkv, D).

    Row j of sequence b is pool[page_table[b, j // page_size], j % page_size].
    Any element type (bf16 bits, fp8 codes, floats) is moved as is.
    """
    pool = np.asarray(pool)
    table = np.asarray(page_table, dtype=np.int64)
    B, per = table.shape
    assert pool.shape[1] == page_size
    j = np.arange(per * page_size)
    return pool[table[:, j // page_size], (j % page_size)[None, :]]


def plain_kv(w):
    """K and V of a workload as the batched arrays `attention_forward` takes:
    pages gathered, fp8 codes dequantized with their descales."""
    k, v = w.k, w.v
    if w.page_table is not None:
        k = gather_pages(k, w.page_table, w.page_size)
        v = gather_pages(v, w.page_table, w.page_size)
    if w.kv_format != "bf16":
        k = dequant_kv(k, w.k_descale, w.kv_format)
        v = dequant_kv(v, w.v_descale, w.kv_format)
    return k, v
