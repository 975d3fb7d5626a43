"""Full-size workloads, in the launch configuration bench.py times, checked
against the fp64 oracle on sampled rows (plus tile-boundary and sequence-end
rows), and for finiteness / empty-row conventions everywhere."""
import numpy as np
import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_attention_qk_gb300 import inputs  # noqa: E402
import gpu_util as gu  # noqa: E402


def _rows(w, n_random=48, seed=0):
    rng = np.random.default_rng(seed)
    seqs = oracle.sequences(w.q.shape, w.k.shape, w.cu_seqlens_q, w.cu_seqlens_k, w.seqused_k)
    rows = set()
    for _ in range(n_random):
        b = int(rng.integers(len(seqs)))
        if seqs[b].sq == 0:
            continue
        rows.add((b, int(rng.integers(w.num_heads_q)), int(rng.integers(seqs[b].sq))))
    for b in (0, len(seqs) - 1):
        sq = seqs[b].sq
        for i in (0, 1, 127, 128, 255, 256, sq - 1):
            if 0 <= i < sq:
                rows.add((b, w.num_heads_q - 1, i))
                rows.add((b, 0, i))
    return sorted(rows)


def _gather(o, l, w, rows):
    seqs = oracle.sequences(w.q.shape, w.k.shape, w.cu_seqlens_q, w.cu_seqlens_k, w.seqused_k)
    og, lg = [], []
    for b, h, i in rows:
        if w.varlen:
            t = seqs[b].q_start + i
            og.append(o[t, h])
            lg.append(l[h, t])
        else:
            og.append(o[b, i, h])
            lg.append(l[b, h, i])
    return torch.stack(og), torch.stack(lg)


@pytest.mark.parametrize("name", ["causal", "large_dense", "large_causal", "varlen", "decode"])
def test_full_size_sampled_rows(name):
    w = inputs.workload(name)
    o, l = gu.run_gpu(w)
    assert torch.isfinite(o).all().item(), "non-finite O"
    assert torch.isfinite(l).all().item(), "every row of these workloads sees at least one key"
    rows = _rows(w)
    og, lg = _gather(o, l, w, rows)
    ro, rl = oracle.attention_rows(w.q, w.k, w.v, rows, **gu.oracle_kw(w))
    print(gu.compare(og, lg, ro, rl, f"{name} ({len(rows)} rows)"))
