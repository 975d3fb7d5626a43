"""KV-cache forms through the C ABI vs the fp64 oracle: fp8 (E4M3 / E5M2) caches
with per-(sequence, KV head) descales, paged caches of several page sizes,
both together, and the full-size decode workloads in those forms."""
import dataclasses

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from exact_attention_qk_gb300 import inputs  # noqa: E402
import gpu_util as gu  # noqa: E402

SEQUSED = np.array([900, 65, 1, 500], np.int32)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("ns", [0, 3])
def test_fp8_decode(fmt, d, ns):
    w = inputs.fp8_batched("fp8", 200 + d, 4, 1, 900, 8, 2, d, fmt, seqused_k=SEQUSED)
    print(gu.check_workload(w, num_splits=ns))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_several_query_rows(fmt):
    # 3 query rows x 4 heads per KV head = 12 packed rows: two row chunks per KV head
    w = inputs.fp8_batched("fp8rows", 210, 2, 3, 700, 8, 2, 128, fmt, seqused_k=np.array([700, 333], np.int32),
                           causal=True)
    print(gu.check_workload(w))


def test_fp8_prefill_shape_is_correct():
    # fp8 caches run on the decode kernel for any row count (correct, not the fast path)
    w = inputs.fp8_batched("fp8pf", 211, 1, 200, 300, 4, 2, 128, "e4m3", causal=True)
    print(gu.check_workload(w))


def test_fp8_descale_matters():
    # the same codes with every descale doubled must not give the same output
    w = inputs.fp8_batched("fp8ds", 212, 2, 1, 400, 8, 2, 128, "e4m3")
    o1, _ = gu.run_gpu(w)
    w2 = dataclasses.replace(w, k_descale=w.k_descale * 2, v_descale=w.v_descale * 2)
    o2, _ = gu.run_gpu(w2)
    assert not torch.equal(o1, o2)
    print(gu.check_workload(w2))


@pytest.mark.parametrize("page_size", [16, 64, 128, 256])
@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (192, 128), (256, 256)])
def test_paged_decode(page_size, d, dv):
    w = inputs.batched("pg", 220 + d, 4, 1, 1024, 8, 2, d, dv, seqused_k=np.array([1024, 65, 1, 513], np.int32))
    print(gu.check_workload(inputs.to_paged(w, page_size)))


@pytest.mark.parametrize("ns", [2, 5])
def test_paged_decode_explicit_splits(ns):
    w = inputs.batched("pgs", 230, 3, 1, 2048, 16, 4, 128, 128, seqused_k=np.array([2048, 777, 1500], np.int32))
    print(gu.check_workload(inputs.to_paged(w, 128), num_splits=ns))


def test_paged_page_size_8_and_32():
    for ps in (8, 32):
        w = inputs.batched("pg8", 231 + ps, 2, 1, 256, 4, 1, 128, 128, seqused_k=np.array([256, 37], np.int32))
        print(gu.check_workload(inputs.to_paged(w, ps)))


@pytest.mark.parametrize("page_size", [16, 64, 128, 192, 256])
@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (192, 128), (256, 256)])
@pytest.mark.parametrize("causal", [False, True])
def test_paged_prefill(page_size, d, dv, causal):
    # prefill shapes with a page table run on the tensor-memory prefill kernel;
    # 192-key pages are moved in 64-row pieces, smaller pages one page a piece
    w = inputs.batched("pgpf", 240 + d, 2, 300, 768, 4, 2, d, dv, causal=causal,
                       seqused_k=np.array([768, 517], np.int32))
    print(gu.check_workload(inputs.to_paged(w, page_size)))


def test_paged_prefill_window_and_gqa():
    w = inputs.batched("pgpfw", 245, 2, 400, 1024, 16, 2, 128, 128, causal=True, window_left=200,
                       seqused_k=np.array([1024, 700], np.int32))
    print(gu.check_workload(inputs.to_paged(w, 64)))


def test_paged_fp8():
    w = inputs.fp8_batched("pgfp8", 232, 3, 1, 1024, 8, 2, 128, "e4m3", seqused_k=np.array([1024, 200, 700], np.int32))
    print(gu.check_workload(inputs.to_paged(w, 128)))


def test_paged_table_entries_past_the_used_keys_are_never_used():
    """Page-table entries of pages that hold no used key may be anything: out of
    the pool (negative, past its end). With 270 used keys and 32-key pages, the
    64-key tile [256, 320) reads the entry of the unused page [288, 320)."""
    w = inputs.to_paged(inputs.batched("pgbad", 233, 3, 1, 1024, 8, 2, 128, 128,
                                       seqused_k=np.array([1024, 100, 270], np.int32)), 32)
    t = w.page_table.copy()
    for b, used in enumerate(w.seqused_k):
        first_unused = (int(used) + 31) // 32
        t[b, first_unused:] = np.where(np.arange(t.shape[1] - first_unused) % 2 == 0, -5, 10 ** 6)
    w2 = dataclasses.replace(w, page_table=t)
    o, l = gu.run_gpu(w2)
    k, v = gu.oracle_kv(w)   # the oracle reads the intact table
    ro, rl = oracle.attention_forward(w.q, k, v, **gu.oracle_kw(w))
    print(gu.compare(o, l, ro, rl, "bad tail entries"))


def test_paged_rejected_with_varlen():
    """A page table with cu_seqlens is an argument error ("page_table is not
    supported with cu_seqlens_k"), reported before any launch."""
    import ctypes
    from exact_attention_qk_gb300 import fa
    q = torch.zeros(2, 4, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(256, 1, 64, dtype=torch.bfloat16, device="cuda")
    a = fa.make_args(q, k, k, torch.empty_like(q), cu_seqlens_q=gu.i32([0, 1, 2]),
                     cu_seqlens_k=gu.i32([0, 128, 256]), max_seqlen_q=1, max_seqlen_k=128)
    table = gu.i32([[0, 1], [2, 3]])
    a.page_table, a.max_pages_per_seq, a.page_size, a.num_pages = table.data_ptr(), 2, 64, 4
    assert fa.lib().fa_fwd(ctypes.byref(a), None, 0, None) == fa.FA_ERR_INVALID_ARG


def _one_sequence(w, b):
    """Workload w restricted to sequence b (same pool / codes, one table row)."""
    kw = dict(q=w.q[b:b + 1], batch=1, seqused_k=None if w.seqused_k is None else w.seqused_k[b:b + 1])
    if w.page_table is not None:
        kw["page_table"] = w.page_table[b:b + 1]
    else:
        kw.update(k=w.k[b:b + 1], v=w.v[b:b + 1])
    if w.kv_format != "bf16":
        kw.update(k_descale=w.k_descale[b:b + 1], v_descale=w.v_descale[b:b + 1])
    return dataclasses.replace(w, **kw)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode_fp8", "decode_paged"])
def test_full_size_kvcache_decode_sampled_sequences(name):
    w = inputs.workload(name)
    o, l = gu.run_gpu(w)
    assert torch.isfinite(o).all().item() and torch.isfinite(l).all().item()
    for b in (0, 17, 40, w.batch - 1):
        s = _one_sequence(w, b)
        k, v = gu.oracle_kv(s)
        ro, rl = oracle.attention_forward(s.q, k, v, **gu.oracle_kw(s))
        print(gu.compare(o[b:b + 1], l[b:b + 1], ro, rl, f"{name} sequence {b}"))


@pytest.mark.parametrize("page_size", [32, 64, 192, 256])
def test_paged_fp8_page_sizes(page_size):
    # fp8 tiles are 128 keys: pages of 64 or 192 keys are moved in 64-row pieces
    w = inputs.fp8_batched("pgfp8ps", 250 + page_size, 2, 1, 768, 8, 2, 128, "e5m2",
                           seqused_k=np.array([768, 333], np.int32))
    print(gu.check_workload(inputs.to_paged(w, page_size)))
