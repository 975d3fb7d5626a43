"""Pack-GQA prefill through the C ABI vs the fp64 oracle: short query sequences
(<= 128 rows) whose r q heads per KV head fold into the tile rows, for every
head dim, GQA ratio, mask kind, varlen and paged caches; and the shapes next to
the switch (129 rows, a ratio that does not divide 128) that stay unpacked."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from exact_attention_qk_gb300 import inputs  # noqa: E402
import gpu_util as gu  # noqa: E402


@pytest.mark.parametrize("d,dv", [(64, 64), (128, 128), (192, 128), (256, 256)])
@pytest.mark.parametrize("sq", [3, 50, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_head_dims(d, dv, sq, causal):
    w = inputs.batched("pack", 300 + d + sq, 2, sq, 700, 32, 4, d, dv, causal=causal)
    print(gu.check_workload(w))


@pytest.mark.parametrize("r", [2, 4, 16, 32])
def test_packed_ratios(r):
    w = inputs.batched("packr", 310 + r, 2, 100, 600, 2 * r, 2, 128, 128, causal=True)
    print(gu.check_workload(w))


def test_packed_window_and_nan_padded_cache():
    w = inputs.batched("packw", 320, 3, 77, 900, 16, 2, 128, 128, causal=True, window_left=150,
                       seqused_k=np.array([900, 300, 78], np.int32))
    print(gu.check_workload(w))


def test_packed_varlen_short_queries():
    lens_q = [50, 128, 7, 1, 33]
    lens_k = [500, 300, 1000, 60, 33]
    w = inputs.packed("packvl", 321, lens_q, lens_k, 16, 2, 128, 128, causal=True)
    print(gu.check_workload(w))


def test_packed_paged_cache():
    w = inputs.batched("packpg", 322, 2, 64, 1024, 32, 4, 128, 128, causal=True,
                       seqused_k=np.array([1024, 513], np.int32))
    print(gu.check_workload(inputs.to_paged(w, 64)))


@pytest.mark.parametrize("sq,hq,hkv", [(129, 32, 4), (100, 6, 2)])
def test_unpacked_neighbours(sq, hq, hkv):
    # 129 query rows, or a ratio (3) that does not divide 128: the unpacked path
    w = inputs.batched("nopack", 323 + sq, 2, sq, 500, hq, hkv, 128, 128, causal=True)
    print(gu.check_workload(w))
