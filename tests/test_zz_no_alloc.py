"""fa_fwd_decode_noalloc: the decode entry point for callers that cannot
allocate device memory where they call it (an engine whose device memory
belongs to another allocator, a latency-critical path that must not take the
driver's allocation locks). Its split partials live in a fixed array inside
the library instead of a caller workspace.

Checked through the C ABI on two calls in a row, against fa_fwd (the entry
point that takes caller-allocated workspace) within the parity tolerances,
and against the fp64 oracle. The second call is a smaller problem, so
partials left over from the first would show if any were read instead of
rewritten. Collected last on purpose: a run that stops at the first failure
has run every other test before this one."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_attention_qk_gb300 import inputs  # noqa: E402
import gpu_util as gu  # noqa: E402


def _problem(seed, B, cap, used, hq=32, hkv=8):
    w = inputs.batched("noalloc", seed, B, 1, cap, hq, hkv, 128, 128, seqused_k=np.asarray(used, np.int32))
    return w, gu.to_dev(w.q), gu.to_dev(w.k), gu.to_dev(w.v), gu.i32(w.seqused_k)


def _call_noalloc(fa, w, q, k, v, su):
    out = torch.empty(w.q.shape[:-1] + (128,), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.batch, w.num_heads_q, 1), dtype=torch.float32, device="cuda")
    args = fa.make_args(q, k, v, out, lse, seqused_k=su, softmax_scale=w.softmax_scale)
    rc = fa.lib().fa_fwd_decode_noalloc(ctypes.byref(args),
                                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == fa.FA_OK, fa.fa_status_string(rc)
    assert fa.fa_get_status() == fa.FA_OK
    return out, lse


def _oracle(w):
    """O and LSE of the oracle, one sequence at a time (only its used keys widened)."""
    o = np.zeros(w.q.shape[:-1] + (128,))
    lse = np.zeros((w.batch, w.num_heads_q, 1))
    for b in range(w.batch):
        n = int(w.seqused_k[b])
        ob, lb = oracle.attention_forward(w.q[b:b + 1], w.k[b:b + 1, :n], w.v[b:b + 1, :n],
                                          scale=w.softmax_scale)
        o[b], lse[b] = ob[0], lb[0]
    return o, lse


def test_noalloc_matches_workspace_entry_point_and_oracle_twice():
    from exact_attention_qk_gb300 import fa
    first = _problem(31, 16, 16384, inputs.uniform_lengths(131, 16, 1024, 16384))
    second = _problem(32, 5, 3000, [3000, 1, 700, 2049, 64])
    for w, q, k, v, su in (first, second):
        args = fa.make_args(q, k, v, seqused_k=su)
        assert fa.fa_num_splits(args) > 1      # the scratch path is the one exercised
        o1, l1 = _call_noalloc(fa, w, q, k, v, su)
        o2, l2 = fa.fa_fwd(q, k, v, seqused_k=su, softmax_scale=w.softmax_scale)
        assert fa.fa_get_status() == fa.FA_OK
        d_o = (o1.float() - o2.float()).abs()
        d_l = (l1 - l2).abs()
        assert d_o.max().item() <= gu.TOL_MAX_O and d_o.mean().item() <= gu.TOL_MEAN_O
        assert d_l.max().item() <= gu.TOL_MAX_LSE
        o_ref, l_ref = _oracle(w)
        gu.compare(o1, l1, o_ref, l_ref, "noalloc vs oracle")


def test_noalloc_rejects_problems_beyond_the_scratch():
    from exact_attention_qk_gb300 import fa
    # 128 sequences x 32 heads x 8 splits x 129 floats > 16 MiB: refused before any launch
    q = torch.zeros((128, 1, 32, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((128, 64, 8, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((128, 64, 8, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((128, 1, 32, 128), dtype=torch.bfloat16, device="cuda")
    used = torch.full((128,), 16, dtype=torch.int32, device="cuda")
    args = fa.make_args(q, k, v, out, seqused_k=used, num_splits=8)
    rc = fa.lib().fa_fwd_decode_noalloc(ctypes.byref(args), None)
    assert rc == fa.FA_ERR_WORKSPACE


def test_noalloc_rejects_prefill_shapes():
    from exact_attention_qk_gb300 import fa
    # 64 query rows x 4 heads per KV head is not decode-shaped: refused before any launch
    q = torch.zeros((1, 64, 8, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 256, 2, 128), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros((1, 256, 2, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((1, 64, 8, 128), dtype=torch.bfloat16, device="cuda")
    args = fa.make_args(q, k, v, out)
    rc = fa.lib().fa_fwd_decode_noalloc(ctypes.byref(args), None)
    assert rc == fa.FA_ERR_UNSUPPORTED
