"""Single-tile probes of the sm_103a primitives (TMA + 128-byte swizzle,
tcgen05.mma with shared-memory and tensor-memory operands, TMEM ld/st),
checked against exact float64 products on the host."""

import ctypes
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

LIB = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "exact_attention_16_gb300", "_lib", "libfa_probes.so")


@pytest.fixture(scope="module")
def probes():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = ctypes.CDLL(LIB)
    for name in ("fa_probe_qk", "fa_probe_pv"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    return lib


def ints(seed, shape, lo=-2, hi=2):
    # small integers: every product and 128-term sum is exact in fp32
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi, shape, generator=g).float()


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("kind", ["ints", "normal"])
def test_probe_qk_matches_a_bt(probes, dt, kind):
    if kind == "ints":
        a, b = ints(1, (128, 128)), ints(2, (128, 128))
    else:
        g = torch.Generator().manual_seed(3)
        a, b = torch.randn(128, 128, generator=g), torch.randn(128, 128, generator=g)
    a, b = a.to(dt), b.to(dt)
    out = torch.full((128, 128), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ad, bd = a.cuda(), b.cuda()
    rc = probes.fa_probe_qk(ad.data_ptr(), bd.data_ptr(), out.data_ptr(), int(dt == torch.bfloat16),
                            err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(err.item()) == 0
    ref = a.double().numpy() @ b.double().numpy().T
    got = out.cpu().double().numpy()
    tol = 0.0 if kind == "ints" else 1e-4
    np.testing.assert_allclose(got, ref, rtol=0, atol=tol)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("kind", ["ints", "normal"])
def test_probe_pv_matches_p_v(probes, dt, kind):
    if kind == "ints":
        p, v = ints(4, (128, 128), 0, 3), ints(5, (128, 128))
    else:
        g = torch.Generator().manual_seed(6)
        p, v = torch.rand(128, 128, generator=g), torch.randn(128, 128, generator=g)
    p, v = p.to(dt), v.to(dt)
    out = torch.full((128, 128), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pd, vd = p.cuda(), v.cuda()
    rc = probes.fa_probe_pv(pd.data_ptr(), vd.data_ptr(), out.data_ptr(), int(dt == torch.bfloat16),
                            err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert rc == 0 and int(err.item()) == 0
    ref = p.double().numpy() @ v.double().numpy()
    got = out.cpu().double().numpy()
    tol = 0.0 if kind == "ints" else 1e-4
    np.testing.assert_allclose(got, ref, rtol=0, atol=tol)


def test_probe_ex2_rate_is_plausible(probes):
    # 152 SMs x 16 to 32 ex2 per clock x ~2 GHz: some 5e12 to 1e13 per second;
    # accept a wide band around it (the probe sets the softmax's roof in the
    # bench line)
    probes.fa_probe_ex2_rate.restype = ctypes.c_int
    probes.fa_probe_ex2_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                         ctypes.c_void_p]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rate = ctypes.c_double(0.0)
    assert probes.fa_probe_ex2_rate(4 * sms, 512, ctypes.byref(rate), None) == 0
    assert 1e12 < rate.value < 1e14, rate.value
