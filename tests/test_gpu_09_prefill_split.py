"""Key splits on the prefill kernel through the C ABI vs the fp64 oracle.

Prefill grids that would fill at most half of the SMs are split by the
library (fa_num_splits > 1); explicit split counts on prefill shapes run the
same path. Each split writes fp32 partials of whole 128-key blocks, and the
combine merges them. The cases cover both automatic forms (unpacked and
pack-GQA) and explicit counts over every head dim, causal and window masks,
NaN-padded caches, varlen, paged caches, and splits that are empty for some
or all rows."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from exact_attention_qk_gb300 import inputs  # noqa: E402
import gpu_util as gu  # noqa: E402


def _auto_splits(w):
    from exact_attention_qk_gb300 import fa
    q, k = gu.to_dev(w.q), gu.to_dev(w.k)
    a = fa.make_args(q, k, k, torch.empty_like(q), **gu.kw_of(w))
    return fa.fa_num_splits(a, torch.cuda.get_device_properties(0).multi_processor_count)


@pytest.mark.parametrize("causal", [False, True])
def test_auto_split_unpacked(causal):
    # 8 query tiles against 8192 keys: split by the library
    w = inputs.batched("pfs_auto", 500, 1, 256, 8192, 8, 8, 128, 128, causal=causal)
    ns = _auto_splits(w)
    assert ns > 1, ns
    print(ns, gu.check_workload(w))


def test_auto_split_packed():
    # 100 query rows x r = 8 heads per KV head, 4 KV heads: 16 packed tiles
    w = inputs.batched("pfs_pack", 501, 1, 100, 4000, 32, 4, 128, 128, causal=True)
    ns = _auto_splits(w)
    assert ns > 1, ns
    print(ns, gu.check_workload(w))


def test_full_grid_is_not_split():
    w = inputs.workload("chunk_gqa")
    assert _auto_splits(w) == 1


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (192, 128), (256, 256)])
@pytest.mark.parametrize("ns", [2, 3, 7])
def test_explicit_splits_head_dims(d, dv, ns):
    w = inputs.batched("pfs_hd", 510 + d + ns, 2, 300, 900, 4, 2, d, dv, causal=True)
    print(gu.check_workload(w, num_splits=ns))


def test_window_and_nan_padded_cache():
    w = inputs.batched("pfs_win", 520, 2, 200, 1500, 8, 2, 128, 128, causal=True, window_left=300,
                       seqused_k=np.array([1500, 700], np.int32))
    print(gu.check_workload(w, num_splits=4))


def test_more_splits_than_key_blocks():
    # 3 key blocks, 8 splits: five splits are empty for every row
    w = inputs.batched("pfs_many", 521, 1, 200, 300, 4, 4, 64, 64, causal=True)
    print(gu.check_workload(w, num_splits=8))


def test_varlen_splits():
    lens_q = [130, 257, 64, 1]
    lens_k = [400, 1300, 640, 900]
    w = inputs.packed("pfs_vl", 522, lens_q, lens_k, 8, 2, 128, 128, causal=True)
    print(gu.check_workload(w, num_splits=3))


def test_paged_splits():
    w = inputs.batched("pfs_pg", 523, 2, 150, 1024, 16, 2, 128, 128, causal=True,
                       seqused_k=np.array([1024, 600], np.int32))
    print(gu.check_workload(inputs.to_paged(w, 64), num_splits=3))
