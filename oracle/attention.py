"""fp64 CPU oracle for the exact attention forward.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg use this module; the product path never imports it. It shares no
code with the CUDA library: it is the plain definition written out, one
(sequence, head) at a time, with the full score matrix materialised in float64.

What it computes (all four FlashAttention pages agree on this definition):

  For sequence b, query head h, query row i, key j:
    s_ij   = scale * sum_d q[i,h,d] k[j,g(h),d]          g(h) = h // (Hq/Hkv)
    LSE_i  = log( sum_{j visible} exp(s_ij) )            natural log
    O_i    = sum_{j visible} exp(s_ij - LSE_i) v[j,g(h),:]
  A row with no visible key has O_i = 0 and LSE_i = -inf.

Sources (page title, then the passage):
  * "mslk/attention/flash_attn/interface.py", `_flash_attn_fwd`: the default
    scale 1/sqrt(head_dim_qk); the O/LSE shapes (B,Sq,Hq,Dv)/(B,Hq,Sq) and the
    packed (Tq,Hq,Dv)/(Hq,Tq) varlen shapes; causal => window_right = 0.
  * "mslk/attention/flash_attn/flash_bwd_sm100.py", the backward preprocess
    multiplies the stored LSE by log2(e) before using it with exp2, so the stored
    LSE is a natural log; its causal/window block bound
    `(m_block+1)*tile_m + seqlen_k - seqlen_q (+ window_right)` fixes the
    bottom-right alignment of the causal diagonal (offset Sk - Sq); its GQA head
    map is the integer quotient h // (Hq/Hkv).
  * "mslk/attention/fmha/triton_splitk.py", `merge_attentions` and the empty
    input branch of `FwOp.apply`: split partials merge by LSE weights, and an
    empty key set gives O = 0, LSE = -inf.
  * "mslk/attention/flash_attn/interface.py", `_flash_attn_fwd_combine`: the
    combine of (num_splits, ...) fp32 partials into O and LSE.

Readings where the pages are silent (each also listed in the design notes):
  * window: key j is visible from row i iff
        j < Sk_b and (wl < 0 or j >= i + off - wl) and (wr < 0 or j <= i + off + wr)
    with off = Sk_b - Sq_b; -1 means unbounded on that side.
  * seqused_k[b] overrides the per-sequence key count (keys at or past it are
    never visible).
  * split s of a split-KV run covers key positions [s*L, (s+1)*L) of every
    sequence; an empty split has O = 0, LSE = -inf.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import List, Optional, Sequence, Tuple

import numpy as np


def widen(x) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 exactly; float arrays -> float64."""
    a = np.asarray(x)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


@dataclass
class Seq:
    q_start: int   # first row of this sequence in q's row axis
    sq: int        # query rows
    k_start: int   # first row in k/v's row axis
    sk: int        # visible-key count before masking (seqused or length)


def sequences(q_shape, k_shape, cu_seqlens_q=None, cu_seqlens_k=None, seqused_k=None) -> List[Seq]:
    """Per-sequence row ranges. Batched layouts index rows inside batch b."""
    if cu_seqlens_q is not None:
        cq = np.asarray(cu_seqlens_q, np.int64)
        ck = np.asarray(cu_seqlens_k, np.int64)
        out = []
        for b in range(len(cq) - 1):
            sk = int(ck[b + 1] - ck[b])
            if seqused_k is not None:
                sk = int(seqused_k[b])
            out.append(Seq(int(cq[b]), int(cq[b + 1] - cq[b]), int(ck[b]), sk))
        return out
    B, Sq = q_shape[0], q_shape[1]
    Sk = k_shape[1]
    return [Seq(0, Sq, 0, Sk if seqused_k is None else int(seqused_k[b])) for b in range(B)]


def visible_mask(sq: int, sk: int, causal: bool, wl: int, wr: int,
                 rows: Optional[np.ndarray] = None, key_lo: int = 0, key_hi: Optional[int] = None) -> np.ndarray:
    """Boolean [len(rows), sk] mask; keys outside [key_lo, key_hi) are hidden."""
    if causal:
        wr = 0
    off = sk - sq
    i = (np.arange(sq) if rows is None else np.asarray(rows)).astype(np.int64)[:, None]
    j = np.arange(sk, dtype=np.int64)[None, :]
    m = np.ones((i.shape[0], sk), dtype=bool)
    if wl >= 0:
        m &= j >= i + off - wl
    if wr >= 0:
        m &= j <= i + off + wr
    m &= j >= key_lo
    if key_hi is not None:
        m &= j < key_hi
    return m


def _rows_attention(qr: np.ndarray, kk: np.ndarray, vv: np.ndarray, mask: np.ndarray,
                    scale: float) -> Tuple[np.ndarray, np.ndarray]:
    """Definition for a block of rows: qr [n,Dk], kk [sk,Dk], vv [sk,Dv], mask [n,sk]."""
    n = qr.shape[0]
    dv = vv.shape[1]
    o = np.zeros((n, dv))
    lse = np.full(n, -np.inf)
    if kk.shape[0] == 0 or n == 0:
        return o, lse
    s = scale * (qr @ kk.T)
    s = np.where(mask, s, -np.inf)
    has = mask.any(axis=1)
    if not has.any():
        return o, lse
    m = np.max(np.where(mask, s, -np.inf), axis=1)
    m = np.where(has, m, 0.0)
    e = np.where(mask, np.exp(s - m[:, None]), 0.0)
    tot = e.sum(axis=1)
    lse = np.where(has, m + np.log(np.where(has, tot, 1.0)), -np.inf)
    p = np.where(mask, np.exp(s - np.where(has, lse, 0.0)[:, None]), 0.0)
    o = p @ vv
    return o, lse


def attention_forward(q, k, v, scale: Optional[float] = None, causal: bool = False,
                      window_left: int = -1, window_right: int = -1,
                      cu_seqlens_q=None, cu_seqlens_k=None, seqused_k=None,
                      key_range: Optional[Tuple[int, int]] = None):
    """Full forward in float64.

    Batched: q (B,Sq,Hq,Dk), k (B,Sk,Hkv,Dk), v (B,Sk,Hkv,Dv) -> O (B,Sq,Hq,Dv), LSE (B,Hq,Sq).
    Varlen:  q (Tq,Hq,Dk),   k (Tk,Hkv,Dk),   v (Tk,Hkv,Dv)   -> O (Tq,Hq,Dv),   LSE (Hq,Tq).
    key_range=(lo, hi) restricts every sequence to key positions [lo, hi) (one split).
    """
    qf, kf, vf = widen(q), widen(k), widen(v)
    varlen = cu_seqlens_q is not None
    hq, dk = qf.shape[-2], qf.shape[-1]
    hkv, dv = kf.shape[-2], vf.shape[-1]
    if hq % hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    r = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    seqs = sequences(qf.shape, kf.shape, cu_seqlens_q, cu_seqlens_k, seqused_k)
    o = np.zeros(qf.shape[:-1] + (dv,))
    lse = np.full((hq, qf.shape[0]) if varlen else (qf.shape[0], hq, qf.shape[1]), -np.inf)
    lo, hi = (0, None) if key_range is None else key_range
    for b, sq in enumerate(seqs):
        if sq.sq == 0:
            continue
        for h in range(hq):
            g = h // r
            if varlen:
                qr = qf[sq.q_start:sq.q_start + sq.sq, h]
                kk = kf[sq.k_start:sq.k_start + sq.sk, g]
                vv = vf[sq.k_start:sq.k_start + sq.sk, g]
            else:
                qr = qf[b, :sq.sq, h]
                kk = kf[b, :sq.sk, g]
                vv = vf[b, :sq.sk, g]
            mask = visible_mask(sq.sq, sq.sk, causal, window_left, window_right, key_lo=lo, key_hi=hi)
            ob, lb = _rows_attention(qr, kk, vv, mask, scale)
            if varlen:
                o[sq.q_start:sq.q_start + sq.sq, h] = ob
                lse[h, sq.q_start:sq.q_start + sq.sq] = lb
            else:
                o[b, :sq.sq, h] = ob
                lse[b, h, :sq.sq] = lb
    return o, lse


def attention_rows(q, k, v, rows: Sequence[Tuple[int, int, int]], scale: Optional[float] = None,
                   causal: bool = False, window_left: int = -1, window_right: int = -1,
                   cu_seqlens_q=None, cu_seqlens_k=None, seqused_k=None,
                   key_range: Optional[Tuple[int, int]] = None):
    """O and LSE for selected (b, h, i) rows only (i local to sequence b).

    Only the rows' own sequences are widened, so this runs on full-size inputs.
    Returns O [n, Dv] and LSE [n] in float64.
    """
    q, k, v = np.asarray(q), np.asarray(k), np.asarray(v)
    varlen = cu_seqlens_q is not None
    hq, dk = q.shape[-2], q.shape[-1]
    hkv, dv = k.shape[-2], v.shape[-1]
    r = hq // hkv
    if scale is None:
        scale = 1.0 / math.sqrt(dk)
    seqs = sequences(q.shape, k.shape, cu_seqlens_q, cu_seqlens_k, seqused_k)
    lo, hi = (0, None) if key_range is None else key_range
    o = np.zeros((len(rows), dv))
    lse = np.full(len(rows), -np.inf)
    for n, (b, h, i) in enumerate(rows):
        sq = seqs[b]
        g = h // r
        if varlen:
            qr = widen(q[sq.q_start + i, h])[None, :]
            kk = widen(k[sq.k_start:sq.k_start + sq.sk, g])
            vv = widen(v[sq.k_start:sq.k_start + sq.sk, g])
        else:
            qr = widen(q[b, i, h])[None, :]
            kk = widen(k[b, :sq.sk, g])
            vv = widen(v[b, :sq.sk, g])
        mask = visible_mask(sq.sq, sq.sk, causal, window_left, window_right,
                            rows=np.array([i]), key_lo=lo, key_hi=hi)
        ob, lb = _rows_attention(qr, kk, vv, mask, scale)
        o[n], lse[n] = ob[0], lb[0]
    return o, lse


def split_forward(q, k, v, num_splits: int, split_len: int, **kw):
    """Per-split partials: split s covers key positions [s*L, (s+1)*L).

    Returns O_s with a leading split axis (S, *O.shape) and LSE_s (S, *LSE.shape).
    """
    os_, ls_ = [], []
    for s in range(num_splits):
        o, l = attention_forward(q, k, v, key_range=(s * split_len, (s + 1) * split_len), **kw)
        os_.append(o)
        ls_.append(l)
    return np.stack(os_), np.stack(ls_)


def combine(o_partial: np.ndarray, lse_partial: np.ndarray, o_axis_map=None):
    """Merge split partials by their LSE weights.

    o_partial (S, ..., Dv) and lse_partial (S, ...) must broadcast row-wise:
    lse_partial[s][idx] weighs o_partial[s][idx, :]. Callers pass the LSE
    already permuted to O's row order.
      M   = max_s LSE_s
      LSE = M + log sum_s exp(LSE_s - M)      (-inf when every split is empty)
      O   = sum_s exp(LSE_s - LSE) O_s        (0 when every split is empty)
    """
    lp = np.asarray(lse_partial, np.float64)
    op = np.asarray(o_partial, np.float64)
    m = lp.max(axis=0)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    w = np.where(np.isfinite(lp), np.exp(lp - m_safe[None]), 0.0)
    tot = w.sum(axis=0)
    lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, tot)))
    wn = np.where(np.isfinite(lp), np.exp(lp - np.where(empty, 0.0, lse)[None]), 0.0)
    o = (wn[..., None] * np.where(np.isfinite(lp)[..., None], op, 0.0)).sum(axis=0)
    o = np.where(empty[..., None], 0.0, o)
    return o, lse


def lse_to_row_order(lse: np.ndarray, varlen: bool) -> np.ndarray:
    """(B,Hq,Sq) -> (B,Sq,Hq) or (Hq,Tq) -> (Tq,Hq), matching O's row order."""
    return np.swapaxes(lse, -1, -2) if not varlen else lse.T


def visible_count(sq: int, sk: int, causal: bool, wl: int, wr: int) -> int:
    """Number of visible (i, j) pairs in one sequence (FLOP accounting)."""
    if sq == 0 or sk == 0:
        return 0
    if causal:
        wr = 0
    off = sk - sq
    i = np.arange(sq, dtype=np.int64)
    lo = np.zeros(sq, np.int64) if wl < 0 else np.maximum(0, i + off - wl)
    hi = np.full(sq, sk - 1, np.int64) if wr < 0 else np.minimum(sk - 1, i + off + wr)
    return int(np.maximum(0, hi - lo + 1).sum())
