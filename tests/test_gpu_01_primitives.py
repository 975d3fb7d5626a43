"""tcgen05 building blocks on single tiles (test-only library), against numpy:
S = Q K^T with both operands K-major and 128B-swizzled, and O = P V with P read
from tensor memory and V MN-major. A descriptor or layout mistake fails here
before it can hide inside the full kernel."""
import ctypes
import os

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

from exact_attention_qk_gb300 import inputs  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(os.path.dirname(HERE), "exact_attention_qk_gb300", "libfa_selftest.so")


@pytest.fixture(scope="module")
def st():
    from exact_attention_qk_gb300 import fa  # noqa: F401  (same runtime)
    lib = ctypes.CDLL(LIB)
    vp = ctypes.c_void_p
    lib.fa_selftest_qk.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp]
    lib.fa_selftest_pv.argtypes = [vp, vp, ctypes.c_int, vp, vp, vp]
    return lib


def _bf16(shape, seed):
    bits = inputs.normal_bf16(seed, 9, 0, shape)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    return t, inputs.bf16_bits_to_f32(bits).astype(np.float64)


@pytest.mark.parametrize("dk", [64, 128, 192, 256])
def test_qk_tile(st, dk):
    q, qf = _bf16((128, dk), 1)
    k, kf = _bf16((128, dk), 2)
    s = torch.zeros(128, 128, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = st.fa_selftest_qk(q.data_ptr(), k.data_ptr(), dk, s.data_ptr(), status.data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and status.item() == 0
    ref = qf @ kf.T
    np.testing.assert_allclose(s.cpu().numpy(), ref, rtol=0, atol=2e-3 * np.sqrt(dk))


@pytest.mark.parametrize("dv", [64, 128, 256])
def test_pv_tile_p_from_tmem(st, dv):
    p, pf = _bf16((128, 128), 3)
    v, vf = _bf16((128, dv), 4)
    o = torch.zeros(128, dv, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = st.fa_selftest_pv(p.data_ptr(), v.data_ptr(), dv, o.data_ptr(), status.data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and status.item() == 0
    ref = pf @ vf
    np.testing.assert_allclose(o.cpu().numpy(), ref, rtol=0, atol=2e-2)


def test_bounded_wait_gives_up_and_reports(st):
    """A wait on a barrier nothing arrives on ends after its limit (2 ms here),
    records the failure in the status word and makes the CTA's other waiters
    give up as well; the kernel exits normally (no trap, no hang)."""
    st.fa_selftest_wait_timeout.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_void_p]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    report = torch.zeros(2, dtype=torch.int32, device="cuda")
    rc = st.fa_selftest_wait_timeout(status.data_ptr(), report.data_ptr(), 2_000_000,
                                     torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0
    assert status.item() == 1                      # the timeout bit
    assert report.tolist() == [1, 1]
    # the context is still healthy afterwards
    x = torch.ones(4, device="cuda")
    assert (x + x).sum().item() == 8.0
