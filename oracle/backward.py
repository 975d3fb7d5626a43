"""fp64 CPU oracle for the attention backward (dQ, dK, dV).

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg use this module; the product path never imports it, and it shares
no code with the CUDA library.

It is the gradient of the forward in `attention.py`, written out per (sequence,
q head) with the full matrices in float64 ("mslk/attention/flash_attn/
flash_bwd_sm100.py", the backward kernel; its preprocess computes
D = rowsum(dO * O); the main loop recomputes P from the stored LSE and forms
dV = P^T dO, dP = dO V^T, dS = P * (dP - D), dQ = dS K, dK = dS^T Q, with the
softmax scale applied to dQ and dK):

    s_ij  = scale * q_i . k_j        (visible (i, j) only)
    P     = softmax over visible j   (rows with no visible key: P = 0)
    dV_j  = sum_i P_ij dO_i
    dP_ij = dO_i . v_j
    D_i   = sum_j P_ij dP_ij  ( = dO_i . O_i )
    dS_ij = P_ij (dP_ij - D_i)
    dQ_i  = scale * sum_j dS_ij k_j
    dK_j  = scale * sum_i dS_ij q_i
GQA: dK and dV of KV head g sum over the q heads h with h // (Hq/Hkv) = g.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from .attention import visible_mask, widen


def attention_backward(q, k, v, do, scale: Optional[float] = None, causal: bool = False, window_left: int = -1,
                       window_right: int = -1, seqused_k=None):
    """Batched layout: q (B,Sq,Hq,D), k/v (B,Sk,Hkv,D/Dv), do (B,Sq,Hq,Dv).

    Returns float64 dq (B,Sq,Hq,D), dk (B,Sk,Hkv,D), dv (B,Sk,Hkv,Dv). Keys at
    or past seqused_k[b] get zero gradients.
    """
    qf, kf, vf, dof = widen(q), widen(k), widen(v), widen(do)
    B, Sq, Hq, D = qf.shape
    Sk, Hkv = kf.shape[1], kf.shape[2]
    r = Hq // Hkv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    dq = np.zeros_like(qf)
    dk = np.zeros_like(kf)
    dv = np.zeros_like(vf)
    for b in range(B):
        sk = Sk if seqused_k is None else int(seqused_k[b])
        mask = visible_mask(Sq, sk, causal, window_left, window_right)
        for h in range(Hq):
            g = h // r
            qq, kk, vv, dd = qf[b, :, h], kf[b, :sk, g], vf[b, :sk, g], dof[b, :, h]
            s = scale * (qq @ kk.T)
            s = np.where(mask, s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            has = np.isfinite(m)
            e = np.where(mask, np.exp(s - np.where(has, m, 0.0)), 0.0)
            den = e.sum(axis=1, keepdims=True)
            p = np.where(den > 0, e / np.where(den > 0, den, 1.0), 0.0)
            dv[b, :sk, g] += p.T @ dd
            dp = dd @ vv.T
            drow = (p * dp).sum(axis=1, keepdims=True)
            ds = p * (dp - drow)
            dq[b, :, h] = scale * (ds @ kk)
            dk[b, :sk, g] += scale * (ds.T @ qq)
    return dq, dk, dv
