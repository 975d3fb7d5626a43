"""Helpers for the GPU parity tests: upload seeded inputs, run the CUDA path
through the C ABI, compare with the fp64 oracle under the stated tolerances."""
import numpy as np
import torch

import oracle

# bf16 inputs, fp32 accumulation, bf16 output: max|dO| <= 1.5e-2,
# mean|dO| <= 1e-3, max|dLSE| <= 1e-3 (all elements of O, all rows of LSE).
TOL_MAX_O = 1.5e-2
TOL_MEAN_O = 1e-3
TOL_MAX_LSE = 1e-3


def to_dev(a: np.ndarray, dev="cuda:0") -> torch.Tensor:
    """uint16 bf16 bits -> torch bf16 on the device (bits preserved)."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


def i32(a, dev="cuda:0"):
    return None if a is None else torch.from_numpy(np.asarray(a, np.int32)).to(dev)


def to64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def kw_of(w):
    return dict(softmax_scale=w.softmax_scale, causal=w.causal, window_left=w.window_left,
                window_right=w.window_right)


def oracle_kw(w):
    return dict(scale=w.softmax_scale, causal=w.causal, window_left=w.window_left,
                window_right=w.window_right, cu_seqlens_q=w.cu_seqlens_q, cu_seqlens_k=w.cu_seqlens_k,
                seqused_k=w.seqused_k)


def kv_to_dev(w, dev="cuda:0"):
    """K and V of a workload on the device: bf16 bits, or fp8 codes as uint8."""
    if w.kv_format == "bf16":
        return to_dev(w.k, dev), to_dev(w.v, dev)
    return (torch.from_numpy(np.ascontiguousarray(w.k)).to(dev),
            torch.from_numpy(np.ascontiguousarray(w.v)).to(dev))


def kv_kw(w, dev="cuda:0"):
    """fa_fwd keywords of a workload's KV-cache form (fp8 descales, page table)."""
    kw = {}
    if w.kv_format != "bf16":
        kw.update(kv_format=w.kv_format, k_descale=torch.from_numpy(w.k_descale).to(dev),
                  v_descale=torch.from_numpy(w.v_descale).to(dev))
    if w.page_table is not None:
        kw["page_table"] = i32(w.page_table, dev)
    return kw


def oracle_kv(w):
    """K and V for the oracle: pages gathered, fp8 codes dequantized."""
    if w.kv_format == "bf16" and w.page_table is None:
        return w.k, w.v
    return oracle.plain_kv(w)


def run_gpu(w, num_splits=0, out=None):
    from exact_attention_qk_gb300 import fa
    q = to_dev(w.q)
    k, v = kv_to_dev(w)
    extra = kv_kw(w)
    if w.varlen:
        extra = dict(cu_seqlens_q=i32(w.cu_seqlens_q), cu_seqlens_k=i32(w.cu_seqlens_k),
                     max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k)
    if w.seqused_k is not None:
        extra["seqused_k"] = i32(w.seqused_k)
    o, l = fa.fa_fwd(q, k, v, out=out, num_splits=num_splits, **kw_of(w), **extra)
    st = fa.fa_get_status()
    assert st == fa.FA_OK, f"device status {st}"
    return o, l


def compare(o_gpu, l_gpu, o_ref, l_ref, label=""):
    o = to64(o_gpu)
    l = l_gpu.cpu().numpy().astype(np.float64)
    assert o.shape == o_ref.shape, (o.shape, o_ref.shape)
    assert np.isfinite(o).all(), f"{label}: non-finite O"
    d_o = np.abs(o - o_ref)
    fin = np.isfinite(l_ref)
    assert (np.isneginf(l[~fin])).all(), f"{label}: rows with no visible key must have LSE=-inf"
    d_l = np.abs(l[fin] - l_ref[fin]) if fin.any() else np.zeros(1)
    msg = (f"{label}: max|dO|={d_o.max():.3e} mean|dO|={d_o.mean():.3e} "
           f"max|dLSE|={d_l.max():.3e}")
    assert d_o.max() <= TOL_MAX_O and d_o.mean() <= TOL_MEAN_O and d_l.max() <= TOL_MAX_LSE, msg
    return msg


def check_workload(w, num_splits=0):
    o, l = run_gpu(w, num_splits=num_splits)
    k, v = oracle_kv(w)
    o_ref, l_ref = oracle.attention_forward(w.q, k, v, **oracle_kw(w))
    return compare(o, l, o_ref, l_ref, w.name)
