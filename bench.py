"""Benchmark of the exact attention forward (and its backward) on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload <name from inputs.WORKLOADS>] [--only] [--dry-run]

One step is one call of the named workload (inputs resident in HBM): for the
prefill workloads one persistent tcgen05 kernel (plus the varlen prepare
kernel, or the combine when the library splits a small grid over the keys),
for decode the split-KV kernel plus the combine kernel, for the backward
workloads (`*_bwd`) one backward call (fa_bwd_two_streams: the preprocess,
then the dK/dV kernel (a dV and a dK pass in one grid at head dims 192/128
and 256) on a second,
torch-owned stream concurrent with the dQ kernel; the forward's O and LSE are
made once, untimed). The headline line is the causal
GQA prefill (B=2, Hq=32, Hkv=4, Sq=Sk=4096, D=128) in TFLOP/s with the
standard attention FLOP count 2*(Dqk+Dv)*#visible(i,j). The other workloads
(the same shape without a mask, the tiny case, the large head dim, varlen,
decode and its cache forms, chunked prefill, the backward of the causal, dense,
varlen and large-head causal shapes) are measured in the
same run and listed compactly at the end of the line under "workloads" as
[value, roofline fraction, kernel ms] (decode in GB/s of algorithmic bytes:
Q + visible K/V rows + O + LSE; the backward in TFLOP/s of its five GEMMs,
2*(3*Dqk+2*Dv)*#visible(i,j)); their full records go to stderr as one JSON line.

Timing: W untimed steps, then K steps each bracketed by CUDA events on the
launching stream, with an L2 flush (a 512 MB write) before every timed step
and a barrier + synchronize around the timed region; max over ranks.
`--impl reference` times the fp64 CPU oracle on a bounded sample instead.
With N > 1 every rank runs an independent replica of the workload (the path
needs no exchange); value = all ranks' work / max time. Started with
`--gpus N` outside torchrun, the script re-launches itself under
torch.distributed.run with N processes. `--dry-run` skips the GPU work and
only exercises the launch and the rank helpers (gloo; a CPU check).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from exact_attention_qk_gb300 import inputs  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0


# ---------------------------------------------------------------- accounting --
def visible_pairs(sq: int, sk: int, causal: bool, wl: int, wr: int) -> int:
    """#(i, j) with key j visible from row i (bottom-right aligned diagonal)."""
    if sq <= 0 or sk <= 0:
        return 0
    if causal:
        wr = 0
    off = sk - sq
    i = np.arange(sq, dtype=np.int64)
    lo = np.zeros(sq, np.int64) if wl < 0 else np.maximum(0, i + off - wl)
    hi = np.full(sq, sk - 1, np.int64) if wr < 0 else np.minimum(sk - 1, i + off + wr)
    return int(np.maximum(0, hi - lo + 1).sum())


def seq_lengths(w):
    if w.varlen:
        lq = np.diff(w.cu_seqlens_q)
        lk = np.diff(w.cu_seqlens_k) if w.seqused_k is None else w.seqused_k
        return list(zip(lq.tolist(), lk.tolist()))
    lk = [w.seqlen_k] * w.batch if w.seqused_k is None else w.seqused_k.tolist()
    return [(w.seqlen_q, k) for k in lk]


def flops(w) -> float:
    pairs = sum(visible_pairs(sq, sk, w.causal, w.window_left, w.window_right) for sq, sk in seq_lengths(w))
    return 2.0 * (w.head_dim_qk + w.head_dim_v) * pairs * w.num_heads_q


def decode_bytes(w) -> float:
    """Q + visible K/V rows + O + LSE, plus the descales of an fp8 cache and
    the page-table entries of a paged one."""
    rows = sum(sq for sq, _ in seq_lengths(w))
    keys = sum(sk for _, sk in seq_lengths(w))
    es = 2 if w.kv_format == "bf16" else 1
    q = rows * w.num_heads_q * w.head_dim_qk * 2
    kv = keys * w.num_heads_kv * (w.head_dim_qk + w.head_dim_v) * es
    o = rows * w.num_heads_q * w.head_dim_v * 2
    lse = rows * w.num_heads_q * 4
    extra = 0
    if w.kv_format != "bf16":
        extra += 2 * w.batch * w.num_heads_kv * 4
    if w.page_table is not None:
        extra += sum(-(-sk // w.page_size) for _, sk in seq_lengths(w)) * 4
    return float(q + kv + o + lse + extra)


def is_decode(name):
    return name.startswith("decode")


def is_backward(name):
    return name.endswith("_bwd")


def backward_flops(w) -> float:
    """The five GEMMs of the backward per visible (row, key) pair: S = QK^T
    recomputed, dP = dO V^T, dV = P^T dO, dQ = dS K, dK = dS^T Q (2.5x the
    forward's two for equal head dims)."""
    pairs = sum(visible_pairs(sq, sk, w.causal, w.window_left, w.window_right) for sq, sk in seq_lengths(w))
    return 2.0 * (3 * w.head_dim_qk + 2 * w.head_dim_v) * pairs * w.num_heads_q


# ------------------------------------------------------------- ncu traffic ----
def kernel_source_hash(files=None) -> str:
    """sha256 over CUDA sources (a changed kernel invalidates old counters):
    the named files of the library's csrc folder, or all of them."""
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_attention_qk_gb300", "csrc")
    paths = sorted(glob.glob(os.path.join(csrc, "*"))) if files is None else [os.path.join(csrc, f) for f in files]
    for f in paths:
        h.update(os.path.basename(f).encode())
        h.update(open(f, "rb").read())
    return h.hexdigest()


def measured_traffic(workload: str):
    """DRAM bytes per launch of the workload's dominant kernel from the committed
    ncu summary, or None when that capture predates the kernel's current sources
    (each entry names the source files of its kernel and their hash)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
    except Exception:
        return None
    e = d.get("workloads", {}).get(workload)
    if not e or not e.get("sources") or e.get("source_sha256") != kernel_source_hash(e["sources"]):
        return None
    return e.get("dram_bytes_per_launch")


# ------------------------------------------------------------------- peaks ----
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            hbm = d.get("hbm_gbs") or d.get("hbm_GBs")
            bf = d.get("bf16_tflops")
            bfs = d.get("bf16_tflops_sustained") or bf
            if hbm and bf:
                return dict(hbm=float(hbm), bf16=float(bf), bf16_sustained=float(bfs), source="measured")
        except Exception:
            pass
    return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS, bf16_sustained=FALLBACK_BF16_TFLOPS_SUSTAINED,
                source="fallback")


# ------------------------------------------------------------------ clocks ----
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms while running.

    start() returns once the first sample has arrived (or after 3 s), so that
    sampling covers the warm-up and the timed steps that follow it."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None
        self._first = threading.Event()

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            self._first.wait(timeout=3.0)
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())
            self._first.set()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- GPU timing ------
class Runner:
    """Device-resident inputs and pre-marshalled C-ABI calls for one workload."""

    def __init__(self, name, dev):
        import torch
        from exact_attention_qk_gb300 import fa
        self.torch, self.fa = torch, fa
        self.name = name
        self.w = w = inputs.workload(name)
        self.dev = dev

        def up(a):
            if a.dtype == np.uint8:      # fp8 codes
                return torch.from_numpy(np.ascontiguousarray(a)).to(dev)
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

        self.q, self.k, self.v = up(w.q), up(w.k), up(w.v)
        self.extra = {}
        if w.kv_format != "bf16":
            self.extra.update(kv_format=w.kv_format, k_descale=torch.from_numpy(w.k_descale).to(dev),
                              v_descale=torch.from_numpy(w.v_descale).to(dev))
        if w.page_table is not None:
            self.extra["page_table"] = torch.from_numpy(w.page_table).to(dev)
        if w.varlen:
            self.extra.update(cu_seqlens_q=torch.from_numpy(w.cu_seqlens_q).to(dev),
                              cu_seqlens_k=torch.from_numpy(w.cu_seqlens_k).to(dev),
                              max_seqlen_q=w.max_seqlen_q, max_seqlen_k=w.max_seqlen_k)
        if w.seqused_k is not None:
            self.extra["seqused_k"] = torch.from_numpy(w.seqused_k).to(dev)
        self.kw = dict(softmax_scale=w.softmax_scale, causal=w.causal, window_left=w.window_left,
                       window_right=w.window_right)
        hq = w.num_heads_q
        self.out = torch.empty(w.q.shape[:-1] + (w.head_dim_v,), dtype=torch.bfloat16, device=dev)
        lshape = (hq, w.q.shape[0]) if w.varlen else (w.batch, hq, w.seqlen_q)
        self.lse = torch.empty(lshape, dtype=torch.float32, device=dev)
        self.args = fa.make_args(self.q, self.k, self.v, self.out, self.lse, **self.kw, **self.extra)
        self.ws_bytes = fa.fa_workspace_size(self.args)
        self.ws = torch.empty(max(self.ws_bytes, 256), dtype=torch.uint8, device=dev)
        self.decode = is_decode(name)
        if self.decode:
            self.ns = fa.fa_num_splits(self.args, 0)
            rows = w.q.shape[:-2] if not w.varlen else w.q.shape[:1]
            self.opart = torch.empty((self.ns,) + tuple(rows) + (hq, w.head_dim_v), dtype=torch.float32,
                                     device=dev)
            self.lpart = torch.empty((self.ns,) + tuple(lshape), dtype=torch.float32, device=dev)
        self.work = decode_bytes(w) if self.decode else flops(w)
        self.launches_per_step = 2 if (self.decode or w.varlen) else 1
        self.backward = is_backward(name)
        if self.backward:
            # the forward's O and LSE are inputs of the backward: made once, untimed
            self.step()
            self.do = up(inputs.grad_out(w))
            self.dq, self.dk, self.dv = (torch.empty_like(t) for t in (self.q, self.k, self.v))
            self.bws_bytes = fa.fa_bwd_workspace_size(self.args)
            self.bws = torch.empty(max(self.bws_bytes, 256), dtype=torch.uint8, device=dev)
            self.work = backward_flops(w)
            # preprocess, dQ, dK/dV (its dV and dK passes share one grid at the head
            # dims whose accumulators do not fit tensor memory together)
            self.launches_per_step = 3

    def stream_ptr(self):
        import ctypes
        return ctypes.c_void_p(self.torch.cuda.current_stream().cuda_stream)

    def step(self):
        import ctypes
        rc = self.fa.lib().fa_fwd(ctypes.byref(self.args), self.ws.data_ptr(), self.ws_bytes, self.stream_ptr())
        if rc != 0:
            raise RuntimeError(f"fa_fwd: {self.fa.fa_status_string(rc)}")

    def step_bwd(self):
        import ctypes
        side, fork, join = self.fa.side_stream_objects(self.dev)
        rc = self.fa.lib().fa_bwd_two_streams(ctypes.byref(self.args), self.do.data_ptr(), self.dq.data_ptr(),
                                              self.dk.data_ptr(), self.dv.data_ptr(), self.bws.data_ptr(),
                                              self.bws_bytes, self.stream_ptr(), ctypes.c_void_p(side.cuda_stream),
                                              ctypes.c_void_p(fork.cuda_event), ctypes.c_void_p(join.cuda_event))
        if rc != 0:
            raise RuntimeError(f"fa_bwd_two_streams: {self.fa.fa_status_string(rc)}")

    def step_split(self):
        """decode as its two kernels, returning the events around the split-KV kernel."""
        import ctypes
        t = self.torch
        e0, e1 = t.cuda.Event(enable_timing=True), t.cuda.Event(enable_timing=True)
        e0.record()
        rc = self.fa.lib().fa_fwd_splitkv(ctypes.byref(self.args), self.ns, self.opart.data_ptr(),
                                          self.lpart.data_ptr(), None, 0, self.stream_ptr())
        e1.record()
        if rc != 0:
            raise RuntimeError(f"fa_fwd_splitkv: {self.fa.fa_status_string(rc)}")
        w = self.w
        o_bs, o_rs, o_hs = (0, self.out.stride(0), self.out.stride(1)) if w.varlen else \
            (self.out.stride(0), self.out.stride(1), self.out.stride(2))
        rc = self.fa.lib().fa_combine(
            self.opart.data_ptr(), self.lpart.data_ptr(), self.ns, w.batch, 0 if w.varlen else w.seqlen_q,
            w.num_heads_q, w.head_dim_v, self.extra["cu_seqlens_q"].data_ptr() if w.varlen else None,
            w.q.shape[0] if w.varlen else 0, self.out.data_ptr(), o_bs, o_rs, o_hs, self.lse.data_ptr(),
            self.stream_ptr())
        if rc != 0:
            raise RuntimeError(f"fa_combine: {self.fa.fa_status_string(rc)}")
        return e0, e1


def l2_flush_buffer(torch, dev):
    return torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)


def time_steps(r: Runner, steps: int, warmup: int, flush):
    """Returns per-step ms and per-step ms of the dominant kernel."""
    torch = r.torch
    for _ in range(warmup):
        if r.decode:
            r.step_split()
        elif r.backward:
            r.step_bwd()
        else:
            r.step()
    torch.cuda.synchronize()
    st = r.fa.fa_get_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    step_ms, kern_ms = [], []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        if r.decode:
            e0, e1 = r.step_split()
        elif r.backward:
            r.step_bwd()
        else:
            r.step()
        b.record()
        torch.cuda.synchronize()
        step_ms.append(a.elapsed_time(b))
        kern_ms.append(e0.elapsed_time(e1) if r.decode else step_ms[-1])
    st = r.fa.fa_get_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after timing")
    return step_ms, kern_ms


def time_e2e(r: Runner, steps: int, warmup: int):
    """Public API end to end: pinned host inputs -> H2D, fa_fwd, O and LSE -> host
    (for a backward workload: q, k, v, O, LSE and dO -> H2D, fa_bwd, dQ, dK, dV -> host)."""
    torch, fa = r.torch, r.fa
    w = r.w
    if r.backward:
        return time_e2e_bwd(r, steps, warmup)
    def host(a):
        a = np.ascontiguousarray(a)
        return torch.from_numpy(a if a.dtype == np.uint8 else a.view(np.int16)).pin_memory()

    def bits(t):   # the device tensor as the host copy's element type
        return t if t.dtype == torch.uint8 else t.view(torch.int16)

    hq, hk, hv = host(w.q), host(w.k), host(w.v)
    ho = torch.empty(r.out.shape, dtype=torch.int16).pin_memory()
    hl = torch.empty(r.lse.shape, dtype=torch.float32).pin_memory()
    dq, dk, dv = bits(r.q), bits(r.k), bits(r.v)
    # the small per-call inputs (sequence offsets and lengths, a KV-cache form's descales and page table) travel too
    small = small_inputs(r)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv)) + \
        sum(h.numel() * h.element_size() for h, _ in small)
    d2h = ho.numel() * 2 + hl.numel() * 4

    def one():
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        for h, d in small:
            d.copy_(h, non_blocking=True)
        fa.fa_fwd(r.q, r.k, r.v, out=r.out, lse=r.lse, workspace=r.ws, **r.kw, **r.extra)
        ho.copy_(r.out.view(torch.int16), non_blocking=True)
        hl.copy_(r.lse, non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        one()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, h2d, d2h


def small_inputs(r: Runner):
    """(pinned host copy, device tensor) of each small per-call input the step
    reads: varlen offsets, seqused_k, fp8 descales, a page table."""
    import numpy as np
    w = r.w
    src = (("cu_seqlens_q", w.cu_seqlens_q), ("cu_seqlens_k", w.cu_seqlens_k), ("seqused_k", w.seqused_k),
           ("k_descale", w.k_descale), ("v_descale", w.v_descale), ("page_table", w.page_table))
    return [(r.torch.from_numpy(np.ascontiguousarray(x)).pin_memory(), r.extra[name])
            for name, x in src if name in r.extra]


def time_e2e_bwd(r: Runner, steps: int, warmup: int):
    torch, fa = r.torch, r.fa
    dev_in = [r.q, r.k, r.v, r.out, r.lse, r.do]
    host_in = [(t.view(torch.int16) if t.dtype == torch.bfloat16 else t).cpu().pin_memory() for t in dev_in]
    host_out = [torch.empty(t.shape, dtype=torch.int16).pin_memory() for t in (r.dq, r.dk, r.dv)]
    small = small_inputs(r)
    h2d = sum(h.numel() * h.element_size() for h in host_in) + sum(h.numel() * h.element_size() for h, _ in small)
    d2h = sum(h.numel() * 2 for h in host_out)

    def one():
        for h, d in zip(host_in, dev_in):
            (d.view(torch.int16) if d.dtype == torch.bfloat16 else d).copy_(h, non_blocking=True)
        for h, d in small:
            d.copy_(h, non_blocking=True)
        fa.fa_bwd(r.q, r.k, r.v, r.out, r.lse, r.do, dq=r.dq, dk=r.dk, dv=r.dv, workspace=r.bws, **r.kw,
                  **r.extra)
        for h, d in zip(host_out, (r.dq, r.dk, r.dv)):
            h.copy_(d.view(torch.int16), non_blocking=True)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        one()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps, h2d, d2h


# --------------------------------------------------------------- CPU oracle ---
def oracle_sample(w, budget_s: float, max_pairs=None):
    """Time the fp64 oracle on whole (sequence, head) pairs until ~budget_s.

    Returns (work units done, seconds, description)."""
    import dataclasses
    import oracle
    kshape = w.k.shape if w.page_table is None else (w.batch, w.page_table.shape[1] * w.page_size) + w.k.shape[2:]
    seqs = oracle.sequences(w.q.shape, kshape, w.cu_seqlens_q, w.cu_seqlens_k, w.seqused_k)
    r = w.num_heads_q // w.num_heads_kv
    plain = {}

    def plain_kv(b):
        # fp8 / paged caches: the oracle's plain K and V of sequence b (timed with it)
        if b not in plain:
            sub = dict(q=w.q[b:b + 1], batch=1)
            if w.page_table is not None:
                sub["page_table"] = w.page_table[b:b + 1]
            else:
                sub.update(k=w.k[b:b + 1], v=w.v[b:b + 1])
            if w.kv_format != "bf16":
                sub.update(k_descale=w.k_descale[b:b + 1], v_descale=w.v_descale[b:b + 1])
            plain.clear()
            plain[b] = oracle.plain_kv(dataclasses.replace(w, **sub))
        return plain[b]
    done_work, t_total, pairs = 0.0, 0.0, 0
    order = [(b, h) for b in range(len(seqs)) for h in range(w.num_heads_q)]
    for b, h in order:
        s = seqs[b]
        if s.sq == 0:
            continue
        if w.varlen:
            q = w.q[s.q_start:s.q_start + s.sq, h][:, None, None, :].transpose(1, 0, 2, 3)
            k = w.k[s.k_start:s.k_start + s.sk, h // r][None, :, None, :]
            v = w.v[s.k_start:s.k_start + s.sk, h // r][None, :, None, :]
        else:
            t0 = time.perf_counter()
            kk, vv = (w.k, w.v) if (w.kv_format == "bf16" and w.page_table is None) else plain_kv(b)
            bb = b if kk is w.k else 0
            t_total += time.perf_counter() - t0
            q = w.q[b:b + 1, :, h:h + 1]
            k = kk[bb:bb + 1, :s.sk, h // r:h // r + 1]
            v = vv[bb:bb + 1, :s.sk, h // r:h // r + 1]
        t0 = time.perf_counter()
        if is_backward(w.name):
            # dO of this (sequence, head) pair alone, in the batched layout of q here
            do = inputs.grad_out(dataclasses.replace(w, q=q, batch=1, num_heads_q=1, seqlen_q=q.shape[1],
                                                     cu_seqlens_q=None, cu_seqlens_k=None))
            t0 = time.perf_counter()
            oracle.attention_backward(q, k, v, do, scale=w.softmax_scale, causal=w.causal,
                                      window_left=w.window_left, window_right=w.window_right)
        else:
            oracle.attention_forward(q, k, v, scale=w.softmax_scale, causal=w.causal, window_left=w.window_left,
                                     window_right=w.window_right)
        t_total += time.perf_counter() - t0
        pairs += 1
        if is_backward(w.name):
            done_work += 2.0 * (3 * w.head_dim_qk + 2 * w.head_dim_v) * visible_pairs(
                s.sq, s.sk, w.causal, w.window_left, w.window_right)
        elif is_decode(w.name):
            es = 2 if w.kv_format == "bf16" else 1
            done_work += s.sq * w.head_dim_qk * 2 + s.sk * (w.head_dim_qk + w.head_dim_v) * es / r + \
                s.sq * (w.head_dim_v * 2 + 4)
        else:
            done_work += 2.0 * (w.head_dim_qk + w.head_dim_v) * visible_pairs(
                s.sq, s.sk, w.causal, w.window_left, w.window_right)
        if t_total >= budget_s or (max_pairs and pairs >= max_pairs):
            break
    desc = f"{pairs} (sequence, q-head) pairs of the {w.name} workload, full rows, fp64"
    return done_work, t_total, desc


def unit_of(name):
    return "GB/s" if is_decode(name) else "TFLOP/s"


def rate(work, ms, name):
    return work / (ms * 1e-3) / (1e9 if is_decode(name) else 1e12)


# ------------------------------------------------------- ranks (replicas) ----
def max_over_ranks(x: float, world: int, device=None) -> float:
    """Largest value of x over all ranks (the slowest replica sets the time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(work_per_rank: float, ms_per_step: float, world: int, name: str) -> float:
    """Whole-job throughput: every rank processes its own replica of the workload."""
    return rate(work_per_rank * world, ms_per_step, name)


# -------------------------------------------------------------------- main ----
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="causal", choices=list(inputs.WORKLOADS))
    ap.add_argument("--only", action="store_true", help="measure the headline workload only")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--dry-run", action="store_true",
                    help="no GPU work: launch the ranks (gloo) and report the rank count only")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if args.gpus > 1 and "WORLD_SIZE" not in os.environ and args.impl == "ours":
        sys.exit(relaunch(args.gpus))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "ours" and world != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}")

    if args.dry_run:
        dry_run(args, world, rank)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args)
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks = load_peaks()
    flush = l2_flush_buffer(torch, dev)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    names = [args.workload] + ([] if args.only else [n for n in SECONDARY if n != args.workload])
    results = {}
    clocks = None
    for n in names:
        r = Runner(n, dev)
        primary = n == args.workload
        sampler = ClockSampler(local_rank) if primary else None
        barrier()
        if sampler:
            sampler.start()
        step_ms, kern_ms = time_steps(r, args.steps, args.warmup, flush)
        barrier()
        if sampler:
            clocks = sampler.stop()
        total_ms = max_over_ranks(sum(step_ms), world, dev)
        ms_step = total_ms / args.steps
        kern_avg = max_over_ranks(sum(kern_ms) / len(kern_ms), world, dev)
        value = job_rate(r.work, ms_step, world, n)
        if r.decode:
            roof = {"bound": "hbm", "achieved": rate(r.work, kern_avg, n), "peak": peaks["hbm"], "unit": "GB/s"}
        else:
            roof = {"bound": "tensor", "achieved": rate(r.work, kern_avg, n), "peak": peaks["bf16"],
                    "unit": "TFLOP/s"}
        roof["frac"] = roof["achieved"] / roof["peak"]
        roof["peak_source"] = peaks["source"] + (" (HBM copy)" if r.decode else " (dense bf16 burst)")
        if r.backward:
            roof["scope"] = "the whole fa_bwd call (preprocess, dQ and dK/dV kernels)"
        roof["traffic"] = measured_traffic(n)
        res = {"value": value, "unit": unit_of(n), "ms_per_step": ms_step, "kernel_ms": kern_avg,
               "work_per_step": r.work, "roofline": roof, "launches_per_step": r.launches_per_step,
               "median_step_ms": statistics.median(step_ms)}
        if r.decode:
            res["num_splits"] = r.ns
        if primary:
            e2e_ms, h2d, d2h = time_e2e(r, max(3, args.steps // 4), 2)
            e2e_ms = max_over_ranks(e2e_ms, world, dev)
            res["e2e"] = {"value": job_rate(r.work, e2e_ms, world, n), "unit": unit_of(n),
                          "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
        results[n] = res
        del r
        torch.cuda.empty_cache()

    p = results[args.workload]
    w0 = inputs.workload(args.workload)
    cpu = None
    if rank == 0:
        work, secs, desc = oracle_sample(w0, args.cpu_budget)
        cpu = {"value": rate(work, secs * 1e3, args.workload), "unit": unit_of(args.workload),
               "cores": os.cpu_count(), "kind": "oracle", "sample": desc, "seconds": secs}
    if rank == 0:
        line = {
            "metric": metric_name(args.workload),
            "value": p["value"],
            "unit": p["unit"],
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": p["ms_per_step"],
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": dtype_of(w0),
            "data": DATA,
            "config": config_of(w0, world),
            "roofline": p["roofline"],
            "cpu_baseline": cpu,
            "e2e": p["e2e"],
            "gpu_launches": p["launches_per_step"] * args.steps,
            "clocks": clocks,
        }
        # every workload's full record on stderr; the compact list last on the line
        sys.stderr.write(json.dumps({"workload_records": results}) + "\n")
        line["workloads_fields"] = ["value (TFLOP/s; GB/s for decode*)", "roofline frac of measured peak",
                                    "kernel ms"]
        line["workloads"] = {n: [float(f"{res['value']:.5g}"), round(res["roofline"]["frac"], 4),
                                 float(f"{res['kernel_ms']:.4g}")] for n, res in results.items()}
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


SECONDARY = ("dense", "tiny", "large_dense", "large_causal", "varlen", "decode", "decode_fp8", "decode_paged",
             "causal_paged", "chunk_gqa", "chunk_single", "causal_bwd", "dense_bwd", "varlen_bwd",
             "large_causal_bwd")
DATA = "synthetic (seeded N(0,1) bf16, numpy PCG64)"


def dtype_of(w):
    return "bf16" if w.kv_format == "bf16" else f"bf16 q/o, {w.kv_format} K/V"


def config_of(w, world):
    """The `config` object of the line, the same for both arms."""
    return {"workload": w.name, "shape": workload_desc(w), "l2": "flushed between steps",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def relaunch(n):
    """Run this script under torch.distributed.run with n processes on this node."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
    return subprocess.call(cmd)


def dry_run(args, world, rank):
    """The launch path without the GPU: gloo ranks agree on a max over ranks and
    rank 0 prints the line's rank fields."""
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("gloo", init_method="env://")
    slowest = max_over_ranks(float(rank + 1), world)
    if rank == 0:
        print(json.dumps({"dry_run": True, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                          "max_over_ranks": slowest, "config": {"workload": args.workload}}))
    if world > 1:
        dist.destroy_process_group()


def metric_name(name):
    if is_decode(name):
        return "split-KV decode KV GB/s"
    w = inputs.workload(name)
    if w.varlen:
        shape = f"varlen {w.batch} seqs Hq={w.num_heads_q} Hkv={w.num_heads_kv} Dqk={w.head_dim_qk} Dv={w.head_dim_v}"
    else:
        d = f"D={w.head_dim_qk}" if w.head_dim_qk == w.head_dim_v else f"Dqk={w.head_dim_qk} Dv={w.head_dim_v}"
        s = f"S={w.seqlen_q}" if w.seqlen_q == w.seqlen_k else f"Sq={w.seqlen_q} Sk={w.seqlen_k}"
        shape = f"B={w.batch} Hq={w.num_heads_q} Hkv={w.num_heads_kv} {s} {d}"
    mode = "causal" if w.causal else "dense"
    if w.window_left >= 0:
        mode += f" window {w.window_left}"
    if is_backward(name):
        return f"attn bwd TFLOP/s (dQ, dK, dV; {mode} {shape})"
    gqa = "GQA " if w.num_heads_q != w.num_heads_kv else ""
    return f"attn fwd TFLOP/s (prefill, {mode} {gqa}{shape})"


def workload_desc(w):
    d = {"Hq": w.num_heads_q, "Hkv": w.num_heads_kv, "Dqk": w.head_dim_qk, "Dv": w.head_dim_v,
         "causal": w.causal, "window": [w.window_left, w.window_right], "scale": w.softmax_scale}
    if w.varlen:
        d.update(batch=w.batch, total_q=int(w.cu_seqlens_q[-1]), varlen=True)
    else:
        d.update(batch=w.batch, seqlen_q=w.seqlen_q, seqlen_k=w.seqlen_k)
    if w.seqused_k is not None:
        d["seqused_k"] = "uniform [1024, 16384], seeded"
    if w.kv_format != "bf16":
        d["kv_cache"] = f"{w.kv_format}, descale per (sequence, KV head)"
    if w.page_table is not None:
        d["paged"] = f"page_size {w.page_size}, {w.k.shape[0]} pages, shuffled"
    return d


def run_reference(args):
    """The fp64 CPU oracle on the host cores, one bounded sample per step."""
    w = inputs.workload(args.workload)
    per_step_budget = max(1.0, min(20.0, 120.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, per_step_budget, max_pairs=1)
    works, secs = 0.0, 0.0
    desc = ""
    for _ in range(args.steps):
        wk, s, desc = oracle_sample(w, per_step_budget, max_pairs=1)
        works += wk
        secs += s
    value = rate(works, secs * 1e3, args.workload)
    line = {
        "impl": "reference",
        "metric": metric_name(args.workload),
        "value": value,
        "unit": unit_of(args.workload),
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": secs * 1e3 / max(1, args.steps),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": DATA,
        "config": config_of(w, 1),
        "cpu_baseline": {"value": value, "unit": unit_of(args.workload), "cores": os.cpu_count(), "kind": "oracle",
                         "sample": desc + " per step"},
        "e2e": {"value": value, "unit": unit_of(args.workload), "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
