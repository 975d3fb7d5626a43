"""Every-element parity of the full-size workloads against the fp64 oracle.

    python tests/full_parity.py [--workloads causal dense ...] [--out FILE] [--workers N]

The GPU tests compare sampled rows at full size; this script compares ALL
elements of O and all rows of LSE. It runs in two phases:
  1. GPU (a child process): each workload once through the C ABI (fa_fwd, in
     the launch configuration the benchmark times); O and LSE are copied to
     the host and saved as .npy files in a scratch folder.
  2. CPU (this process, which never touches CUDA): the inputs are drawn again
     from their seeds, and a forked process pool runs the oracle one
     (sequence, q head) at a time, accumulating per workload max|dO| and
     sum|dO| over every element of O, and max|dLSE| over every row that has a
     visible key (rows without one must be -inf on both sides).
Tolerances: max|dO| <= 1.5e-2, mean|dO| <= 1e-3, max|dLSE| <= 1e-3, with the
mean taken over all elements of O. Prints one JSON object (and writes it to
--out); exits 1 when a workload fails.

Test infrastructure: it imports the oracle, so only a test run calls it.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import multiprocessing as mp
import os
import subprocess
import sys
import tempfile
import time

# one BLAS thread per oracle worker (the pool provides the parallelism)
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

TOL_MAX_O, TOL_MEAN_O, TOL_MAX_LSE = 1.5e-2, 1e-3, 1e-3
DEFAULT = ("tiny", "causal", "dense", "large_dense", "large_causal", "varlen", "decode",
           "decode_fp8", "decode_paged", "causal_paged", "chunk_gqa", "chunk_single")


# ------------------------------------------------------------------ GPU side ---
def gpu_phase(names, folder):
    import torch
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import gpu_util as gu
    from exact_attention_qk_gb300 import fa, inputs
    for name in names:
        w = inputs.workload(name)
        o, l = gu.run_gpu(w)
        torch.cuda.synchronize()
        np.save(os.path.join(folder, name + "_o.npy"), o.float().cpu().numpy())
        np.save(os.path.join(folder, name + "_l.npy"), l.cpu().numpy())
        del w, o, l
        torch.cuda.empty_cache()
        print(f"[gpu] {name} done", file=sys.stderr, flush=True)
    st = fa.fa_get_status()
    if st != fa.FA_OK:
        raise RuntimeError(f"device status {st}")


# ------------------------------------------------------------------ CPU side ---
_W = None          # the workload being checked (inherited by the forked workers)
_FOLDER = None


def _sequence_kv(w, b):
    """Plain K and V of sequence b for the oracle (pages gathered, fp8 decoded)."""
    import oracle
    if w.kv_format == "bf16" and w.page_table is None:
        return w.k[b:b + 1], w.v[b:b + 1]
    sub = dict(q=w.q[b:b + 1], batch=1)
    if w.page_table is not None:
        sub["page_table"] = w.page_table[b:b + 1]
    else:
        sub.update(k=w.k[b:b + 1], v=w.v[b:b + 1])
    if w.kv_format != "bf16":
        sub.update(k_descale=w.k_descale[b:b + 1], v_descale=w.v_descale[b:b + 1])
    if w.seqused_k is not None:
        sub["seqused_k"] = w.seqused_k[b:b + 1]
    return oracle.plain_kv(dataclasses.replace(w, **sub))


def _task(args):
    """Oracle of sequence b, q heads [h0, h1), against the saved GPU output."""
    b, h0, h1 = args
    import oracle
    w = _W
    og = np.load(os.path.join(_FOLDER, w.name + "_o.npy"), mmap_mode="r")
    lg = np.load(os.path.join(_FOLDER, w.name + "_l.npy"), mmap_mode="r")
    r = w.num_heads_q // w.num_heads_kv
    kw = dict(scale=w.softmax_scale, causal=w.causal, window_left=w.window_left, window_right=w.window_right)
    res = dict(max_do=0.0, sum_do=0.0, n_o=0, max_dl=0.0, n_l=0, bad_inf=0, nonfinite=0)
    if not w.varlen:
        kb, vb = _sequence_kv(w, b)
    for h in range(h0, h1):
        g = h // r
        if w.varlen:
            q0, q1 = int(w.cu_seqlens_q[b]), int(w.cu_seqlens_q[b + 1])
            k0, k1 = int(w.cu_seqlens_k[b]), int(w.cu_seqlens_k[b + 1])
            o_ref, l_ref = oracle.attention_forward(w.q[q0:q1, h][None, :, None, :], w.k[k0:k1, g][None, :, None, :],
                                                    w.v[k0:k1, g][None, :, None, :], **kw)
            o_gpu = np.asarray(og[q0:q1, h], np.float64)
            l_gpu = np.asarray(lg[h, q0:q1], np.float64)
        else:
            su = None if w.seqused_k is None else w.seqused_k[b:b + 1]
            o_ref, l_ref = oracle.attention_forward(w.q[b:b + 1, :, h:h + 1], kb[:, :, g:g + 1], vb[:, :, g:g + 1],
                                                    seqused_k=su, **kw)
            o_gpu = np.asarray(og[b, :, h], np.float64)
            l_gpu = np.asarray(lg[b, h], np.float64)
        o_ref = o_ref.reshape(o_gpu.shape)
        l_ref = l_ref.reshape(l_gpu.shape)
        d = np.abs(o_gpu - o_ref)
        res["nonfinite"] += int((~np.isfinite(o_gpu)).sum())
        if d.size:
            res["max_do"] = max(res["max_do"], float(np.nanmax(d)))
        res["sum_do"] += float(np.nansum(d))
        res["n_o"] += d.size
        fin = np.isfinite(l_ref)
        res["bad_inf"] += int((~np.isneginf(l_gpu[~fin])).sum())
        if fin.any():
            res["max_dl"] = max(res["max_dl"], float(np.abs(l_gpu[fin] - l_ref[fin]).max()))
        res["n_l"] += int(fin.sum())
    return res


def cpu_phase(name, folder, workers):
    global _W, _FOLDER
    from exact_attention_qk_gb300 import inputs
    _W = inputs.workload(name)
    _FOLDER = folder
    w = _W
    rows_per_seq = 2 if w.varlen else w.seqlen_q
    per_head = rows_per_seq > 1 and w.num_heads_q * w.batch > 1 and name != "tiny"
    tasks = ([(b, h, h + 1) for b in range(w.batch) for h in range(w.num_heads_q)] if per_head
             else [(b, 0, w.num_heads_q) for b in range(w.batch)])
    tot = dict(max_do=0.0, sum_do=0.0, n_o=0, max_dl=0.0, n_l=0, bad_inf=0, nonfinite=0)
    with mp.get_context("fork").Pool(min(workers, len(tasks))) as pool:
        for res in pool.imap_unordered(_task, tasks, chunksize=1):
            tot["max_do"] = max(tot["max_do"], res["max_do"])
            tot["max_dl"] = max(tot["max_dl"], res["max_dl"])
            for key in ("sum_do", "n_o", "n_l", "bad_inf", "nonfinite"):
                tot[key] += res[key]
    _W = None
    return tot


def mem_available_gb():
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) / 1024 / 1024
    except OSError:
        pass
    return 16.0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workloads", nargs="*", default=list(DEFAULT))
    ap.add_argument("--out", default="")
    ap.add_argument("--workers", type=int, default=0)
    ap.add_argument("--folder", default="")
    ap.add_argument("--phase", default="all", choices=["all", "gpu", "cpu"])
    args = ap.parse_args()
    folder = args.folder or tempfile.mkdtemp(prefix="fa_full_parity_")
    if args.phase == "gpu":
        gpu_phase(args.workloads, folder)
        return
    t0 = time.time()
    if args.phase == "all":
        # the GPU phase runs in a child, so that this process can fork oracle workers
        rc = subprocess.call([sys.executable, os.path.abspath(__file__), "--phase", "gpu", "--folder", folder,
                              "--workloads", *args.workloads])
        if rc != 0:
            sys.exit(rc)
    t_gpu = time.time() - t0
    # one oracle task holds up to ~3 GB (an 8192 x 8192 fp64 score matrix and its temporaries)
    workers = args.workers or max(1, min(os.cpu_count() or 1, int(mem_available_gb() * 0.5 / 3.0)))
    report = {"tolerances": {"max_do": TOL_MAX_O, "mean_do": TOL_MEAN_O, "max_dlse": TOL_MAX_LSE},
              "workers": workers, "gpu_phase_s": round(t_gpu, 1), "workloads": {}}
    t1 = time.time()
    ok_all = True
    for name in args.workloads:
        ts = time.time()
        t = cpu_phase(name, folder, workers)
        mean = t["sum_do"] / max(1, t["n_o"])
        ok = (t["max_do"] <= TOL_MAX_O and mean <= TOL_MEAN_O and t["max_dl"] <= TOL_MAX_LSE
              and t["bad_inf"] == 0 and t["nonfinite"] == 0 and not math.isnan(t["max_do"]))
        ok_all &= ok
        report["workloads"][name] = {"max_do": t["max_do"], "mean_do": mean, "max_dlse": t["max_dl"],
                                     "o_elements": t["n_o"], "lse_rows": t["n_l"],
                                     "lse_inf_mismatch": t["bad_inf"], "nonfinite_o": t["nonfinite"], "pass": ok,
                                     "oracle_s": round(time.time() - ts, 1)}
        print(f"[cpu] {name}: {report['workloads'][name]}", file=sys.stderr, flush=True)
    report["oracle_phase_s"] = round(time.time() - t1, 1)
    report["pass"] = ok_all
    text = json.dumps(report, indent=1)
    print(text)
    if args.out:
        with open(args.out, "w") as f:
            f.write(text + "\n")
    sys.exit(0 if ok_all else 1)


if __name__ == "__main__":
    main()
