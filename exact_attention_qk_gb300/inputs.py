"""Seeded synthetic inputs for the attention forward workloads.

This module is the only code shared by the fp64 oracle side and the CUDA side.
It draws numbers and lays them out; it holds none of the attention arithmetic.

Every tensor is drawn with numpy's PCG64 generator from a SeedSequence keyed by
(seed, tensor id, sequence index), so one sequence's block can be regenerated
alone (the oracle checks sampled sequences of the full-size workloads without
drawing the whole KV cache) and the bits are identical on any machine.
Standard-normal float32 draws are rounded to bfloat16 with round-to-nearest-even.

Workloads (the shapes the FlashAttention pages benchmark: dense/causal GQA
prefill, a large head dim, varlen packing with a sliding window and the
(192,128) head shape, and split-KV decode over a KV cache):

  tiny     B=1  Hq=Hkv=2  Sq=Sk=128  D=64, dense
  causal   B=2  Hq=32 Hkv=4  Sq=Sk=4096  D=128, causal
  dense    the causal shape (and the same draws) without a mask
  large    B=1  Hq=16 Hkv=2  Sq=Sk=8192  D=256, dense and causal, scale 1/16
  varlen   16 sequences, lengths uniform in [256, 8192], Hq=Hkv=16,
           Dqk=192, Dv=128, causal, window_left=1024
  decode   Sq=1, B=64, Hq=32, Hkv=8, D=128, KV cache capacity 16384,
           seqused_k uniform in [1024, 16384]

KV-cache variants of the decode workload (the fp8 KV-cache decode and paged-KV
passages of the FlashAttention pages):

  decode_fp8    the decode shape with an e4m3 K/V cache (one byte per element)
                and per-(sequence, KV head) descales
  decode_paged  the decode shape with the cache split into 128-key pages held
                in a shuffled page pool, located through a page table
  causal_paged  the causal prefill workload with its K/V cache paged the same way
  chunk_gqa     chunked prefill: 8 sequences of 128 new rows against 8192 keys,
                Hq=32 Hkv=4 D=128, causal (the pack-GQA prefill case)
  chunk_single  one sequence's 256 new rows against 16384 keys, Hq=32 Hkv=8
                D=128, causal (a grid of 32 tiles: the key-split prefill case)
  decode_*_small  the first 16 sequences of a decode workload (profiling cases)

Backward workloads (dQ, dK, dV given dO; dO is N(0,1) bf16 from its own stream):

  causal_bwd    the causal prefill shape (B=2 Hq=32 Hkv=4 S=4096 D=128)
  dense_bwd     the same shape without a mask
  varlen_bwd    the varlen sliding-window workload (Dqk=192 Dv=128; the same
                q, k, v draws)
  large_causal_bwd  the large-head causal shape (B=1 Hq=16 Hkv=2 S=8192 D=256;
                the same q, k, v draws)
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# tensor ids inside a workload's SeedSequence (_DO: the output gradient of a backward)
_Q, _K, _V, _DO = 0, 1, 2, 3

# bfloat16 bit pattern of a quiet NaN; written into KV-cache slots past
# seqused_k so that any read of them that reaches the arithmetic shows up.
BF16_NAN_BITS = 0x7FC0

# fp8 element formats of a quantized KV cache, and a NaN code of each
# (e4m3: exponent and mantissa all ones; e5m2: exponent all ones, mantissa != 0)
FP8_FORMATS = ("e4m3", "e5m2")
FP8_NAN_CODE = {"e4m3": 0x7F, "e5m2": 0x7F}


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bits to float32 exactly."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, tensor_id: int, index: int, shape) -> np.ndarray:
    """N(0,1) draws for one sequence block, rounded to bf16 bits."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id, index])))
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def fp8_codes(seed: int, tensor_id: int, index: int, shape, fmt: str) -> np.ndarray:
    """Random fp8 element codes (uint8) for one sequence block.

    Each code is assembled from independent draws of its fields: a random sign,
    a biased exponent from a window that spans magnitudes 1/8 to 2 (the scale
    of the bf16 workloads' normal draws), and a uniform mantissa. No
    floating-point arithmetic is involved.
    """
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id, index, 8])))
    sign = rng.integers(0, 2, size=shape, dtype=np.uint8)
    if fmt == "e4m3":      # 1 sign, 4 exponent (bias 7), 3 mantissa bits
        e = rng.integers(4, 8, size=shape, dtype=np.uint8)
        m = rng.integers(0, 8, size=shape, dtype=np.uint8)
        return (sign << 7) | (e << 3) | m
    if fmt == "e5m2":      # 1 sign, 5 exponent (bias 15), 2 mantissa bits
        e = rng.integers(12, 16, size=shape, dtype=np.uint8)
        m = rng.integers(0, 4, size=shape, dtype=np.uint8)
        return (sign << 7) | (e << 2) | m
    raise ValueError(fmt)


def uniform_f32(seed: int, tensor_id: int, shape, lo: float, hi: float) -> np.ndarray:
    """float32 draws uniform in [lo, hi)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id, 9])))
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def uniform_lengths(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform in [lo, hi] inclusive (int32)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed])))
    return rng.integers(lo, hi + 1, size=n).astype(np.int32)


@dataclasses.dataclass
class Workload:
    """Host-side (numpy) inputs; bf16 tensors are uint16 bit arrays."""
    name: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    num_heads_q: int
    num_heads_kv: int
    head_dim_qk: int
    head_dim_v: int
    softmax_scale: float
    causal: bool = False
    window_left: int = -1
    window_right: int = -1
    batch: int = 1
    seqlen_q: int = 0          # batched layout only
    seqlen_k: int = 0          # batched layout: K/V capacity per sequence
    cu_seqlens_q: Optional[np.ndarray] = None   # int32 [B+1], varlen layout
    cu_seqlens_k: Optional[np.ndarray] = None
    seqused_k: Optional[np.ndarray] = None      # int32 [B]
    max_seqlen_q: int = 0
    max_seqlen_k: int = 0
    seed: int = 0
    # KV-cache forms (defaults: a bf16 cache in the batched or packed layout)
    kv_format: str = "bf16"                     # "bf16", "e4m3" or "e5m2"
    k_descale: Optional[np.ndarray] = None      # float32 [B, Hkv]: K element = code value x descale
    v_descale: Optional[np.ndarray] = None
    page_table: Optional[np.ndarray] = None     # int32 [B, max_pages]; k/v then hold the page pool
    page_size: int = 0

    @property
    def varlen(self) -> bool:
        return self.cu_seqlens_q is not None


def batched(name, seed, B, Sq, Sk, Hq, Hkv, Dqk, Dv, scale=None, causal=False,
            window_left=-1, window_right=-1, seqused_k=None, pad_bits=BF16_NAN_BITS):
    """Batched layout: q (B,Sq,Hq,Dqk), k (B,Sk,Hkv,Dqk), v (B,Sk,Hkv,Dv).

    Sequence b's block of each tensor comes from its own stream. With seqused_k,
    only the first seqused_k[b] cache rows are drawn; the rest are filled with
    `pad_bits` (a NaN by default), which a correct kernel never lets reach O.
    """
    q = np.empty((B, Sq, Hq, Dqk), np.uint16)
    k = np.empty((B, Sk, Hkv, Dqk), np.uint16)
    v = np.empty((B, Sk, Hkv, Dv), np.uint16)
    for b in range(B):
        q[b] = normal_bf16(seed, _Q, b, (Sq, Hq, Dqk))
        n = Sk if seqused_k is None else int(seqused_k[b])
        k[b, :n] = normal_bf16(seed, _K, b, (n, Hkv, Dqk))
        v[b, :n] = normal_bf16(seed, _V, b, (n, Hkv, Dv))
        if n < Sk:
            k[b, n:] = pad_bits
            v[b, n:] = pad_bits
    if scale is None:
        scale = 1.0 / float(np.sqrt(Dqk))
    return Workload(name=name, q=q, k=k, v=v, num_heads_q=Hq, num_heads_kv=Hkv,
                    head_dim_qk=Dqk, head_dim_v=Dv, softmax_scale=scale, causal=causal,
                    window_left=window_left, window_right=window_right, batch=B,
                    seqlen_q=Sq, seqlen_k=Sk,
                    seqused_k=None if seqused_k is None else np.asarray(seqused_k, np.int32),
                    max_seqlen_q=Sq, max_seqlen_k=Sk, seed=seed)


def grad_out(w: Workload) -> np.ndarray:
    """dO for the backward of a workload: N(0,1) bf16 bits with the output's
    shape, (B, Sq, Hq, Dv) or packed (T, Hq, Dv), one stream per sequence."""
    if w.varlen:
        cu = w.cu_seqlens_q
        do = np.empty((int(cu[-1]), w.num_heads_q, w.head_dim_v), np.uint16)
        for b in range(len(cu) - 1):
            do[cu[b]:cu[b + 1]] = normal_bf16(w.seed, _DO, b, (int(cu[b + 1] - cu[b]), w.num_heads_q, w.head_dim_v))
        return do
    do = np.empty((w.batch, w.seqlen_q, w.num_heads_q, w.head_dim_v), np.uint16)
    for b in range(w.batch):
        do[b] = normal_bf16(w.seed, _DO, b, (w.seqlen_q, w.num_heads_q, w.head_dim_v))
    return do


def fp8_batched(name, seed, B, Sq, Sk, Hq, Hkv, D, fmt, seqused_k=None, scale=None, causal=False):
    """Batched layout with an fp8 K/V cache: q bf16 (B,Sq,Hq,D); k, v uint8
    codes (B,Sk,Hkv,D); descales float32 (B,Hkv) in [0.25, 1). Cache rows at or
    past seqused_k hold NaN codes."""
    q = np.empty((B, Sq, Hq, D), np.uint16)
    k = np.empty((B, Sk, Hkv, D), np.uint8)
    v = np.empty((B, Sk, Hkv, D), np.uint8)
    for b in range(B):
        q[b] = normal_bf16(seed, _Q, b, (Sq, Hq, D))
        n = Sk if seqused_k is None else int(seqused_k[b])
        k[b, :n] = fp8_codes(seed, _K, b, (n, Hkv, D), fmt)
        v[b, :n] = fp8_codes(seed, _V, b, (n, Hkv, D), fmt)
        if n < Sk:
            k[b, n:] = FP8_NAN_CODE[fmt]
            v[b, n:] = FP8_NAN_CODE[fmt]
    if scale is None:
        scale = 1.0 / float(np.sqrt(D))
    return Workload(name=name, q=q, k=k, v=v, num_heads_q=Hq, num_heads_kv=Hkv,
                    head_dim_qk=D, head_dim_v=D, softmax_scale=scale, causal=causal, batch=B,
                    seqlen_q=Sq, seqlen_k=Sk,
                    seqused_k=None if seqused_k is None else np.asarray(seqused_k, np.int32),
                    max_seqlen_q=Sq, max_seqlen_k=Sk, seed=seed, kv_format=fmt,
                    k_descale=uniform_f32(seed, 3, (B, Hkv), 0.25, 1.0),
                    v_descale=uniform_f32(seed, 4, (B, Hkv), 0.25, 1.0))


def to_paged(w: Workload, page_size: int, extra_pages: int = 3) -> Workload:
    """The same batched cache, moved into a page pool.

    Sequence b's keys [j*page_size, (j+1)*page_size) go to page page_table[b, j];
    the pages of all sequences are a random permutation of the pool, which also
    holds `extra_pages` pages no sequence uses. Pool rows that no visible key
    maps to (past seqused_k, and the extra pages) hold NaN patterns.
    """
    assert w.page_table is None and not w.varlen and w.seqlen_k % page_size == 0
    B, Sk = w.batch, w.seqlen_k
    per = Sk // page_size
    n_pages = B * per + extra_pages
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([w.seed, 7, page_size])))
    perm = rng.permutation(n_pages).astype(np.int32)
    table = perm[:B * per].reshape(B, per)
    nan = FP8_NAN_CODE[w.kv_format] if w.kv_format in FP8_FORMATS else BF16_NAN_BITS
    pools = []
    for src in (w.k, w.v):
        pool = np.full((n_pages, page_size) + src.shape[2:], nan, src.dtype)
        pool[table.reshape(-1)] = src.reshape((B * per, page_size) + src.shape[2:])
        pools.append(pool)
    return dataclasses.replace(w, name=w.name + "_paged", k=pools[0], v=pools[1],
                               page_table=np.ascontiguousarray(table), page_size=page_size)


def packed(name, seed, lens_q, lens_k, Hq, Hkv, Dqk, Dv, scale=None, causal=False,
           window_left=-1, window_right=-1):
    """Varlen packed layout: q (Tq,Hq,Dqk), k (Tk,Hkv,Dqk), v (Tk,Hkv,Dv)."""
    lens_q = np.asarray(lens_q, np.int64)
    lens_k = np.asarray(lens_k, np.int64)
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    q = np.empty((int(cu_q[-1]), Hq, Dqk), np.uint16)
    k = np.empty((int(cu_k[-1]), Hkv, Dqk), np.uint16)
    v = np.empty((int(cu_k[-1]), Hkv, Dv), np.uint16)
    for b in range(len(lens_q)):
        q[cu_q[b]:cu_q[b + 1]] = normal_bf16(seed, _Q, b, (int(lens_q[b]), Hq, Dqk))
        k[cu_k[b]:cu_k[b + 1]] = normal_bf16(seed, _K, b, (int(lens_k[b]), Hkv, Dqk))
        v[cu_k[b]:cu_k[b + 1]] = normal_bf16(seed, _V, b, (int(lens_k[b]), Hkv, Dv))
    if scale is None:
        scale = 1.0 / float(np.sqrt(Dqk))
    return Workload(name=name, q=q, k=k, v=v, num_heads_q=Hq, num_heads_kv=Hkv,
                    head_dim_qk=Dqk, head_dim_v=Dv, softmax_scale=scale, causal=causal,
                    window_left=window_left, window_right=window_right, batch=len(lens_q),
                    cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                    max_seqlen_q=int(lens_q.max()) if len(lens_q) else 0,
                    max_seqlen_k=int(lens_k.max()) if len(lens_k) else 0, seed=seed)


# ---- the named workloads -----------------------------------------------------

VARLEN_LENGTH_SEED = 40
DECODE_SEQUSED_SEED = 50


def varlen_lengths() -> np.ndarray:
    return uniform_lengths(VARLEN_LENGTH_SEED, 16, 256, 8192)


def decode_seqused() -> np.ndarray:
    return uniform_lengths(DECODE_SEQUSED_SEED, 64, 1024, 16384)


def workload(name: str) -> Workload:
    if name == "tiny":
        return batched("tiny", 1, 1, 128, 128, 2, 2, 64, 64)
    if name in ("causal", "dense"):
        # the causal GQA prefill and its unmasked twin (the same q, k, v draws)
        return batched(name, 2, 2, 4096, 4096, 32, 4, 128, 128, causal=(name == "causal"))
    if name in ("large_dense", "large_causal", "large_causal_bwd"):
        return batched(name, 3, 1, 8192, 8192, 16, 2, 256, 256, scale=1.0 / 16,
                       causal=(name != "large_dense"))
    if name in ("varlen", "varlen_bwd"):
        lens = varlen_lengths()
        return packed(name, 4, lens, lens, 16, 16, 192, 128, causal=True,
                      window_left=1024, window_right=0)
    if name == "decode":
        return batched("decode", 5, 64, 1, 16384, 32, 8, 128, 128, seqused_k=decode_seqused())
    if name == "decode_fp8":
        return fp8_batched("decode_fp8", 5, 64, 1, 16384, 32, 8, 128, "e4m3", seqused_k=decode_seqused())
    if name == "decode_paged":
        return to_paged(workload("decode"), 128)
    if name == "chunk_gqa":
        # chunked prefill: 128 new query rows of each of 8 sequences against an
        # 8192-key cache (bottom-right causal), GQA 32/4
        return batched("chunk_gqa", 6, 8, 128, 8192, 32, 4, 128, 128, causal=True)
    if name == "chunk_single":
        # one request's 256-row prefill chunk against a 16384-key cache, GQA
        # 32/8: 32 tiles of 256 rows (one per q head; 256 rows are too many to
        # pack), a grid the library splits over the keys
        return batched("chunk_single", 7, 1, 256, 16384, 32, 8, 128, 128, causal=True)
    if name == "causal_paged":
        # the causal prefill workload with its K/V cache in shuffled 128-key pages
        return to_paged(workload("causal"), 128)
    if name == "decode_fp8_small":
        return fp8_batched("decode_fp8_small", 5, 16, 1, 16384, 32, 8, 128, "e4m3", seqused_k=decode_seqused()[:16])
    if name == "decode_paged_small":
        return to_paged(workload("decode_small"), 128)
    if name in ("causal_bwd", "dense_bwd"):
        # the backward of the causal prefill shape (same q, k, v draws), and its unmasked twin
        return batched(name, 2, 2, 4096, 4096, 32, 4, 128, 128, causal=(name == "causal_bwd"))
    if name == "decode_small":
        # the decode shape with 16 sequences (about 1 GB of cache): a profiling case
        return batched("decode_small", 5, 16, 1, 16384, 32, 8, 128, 128, seqused_k=decode_seqused()[:16])
    raise KeyError(name)


WORKLOADS = ("tiny", "causal", "dense", "large_dense", "large_causal", "varlen", "decode", "decode_small",
             "decode_fp8", "decode_paged", "causal_paged", "chunk_gqa",
             "decode_fp8_small", "decode_paged_small", "causal_bwd", "dense_bwd", "chunk_single",
             "varlen_bwd", "large_causal_bwd")
