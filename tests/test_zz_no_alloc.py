"""fa_fwd_decode_noalloc: the decode call whose split workspace is the
library's fixed device array, for callers that cannot allocate device memory
when they call. Called through the C ABI on two calls in a row with
different inputs (so that a second call cannot pass on what the first left
in the shared array), and compared on each with the fp64 oracle and with
fa_fwd_decode (caller-provided workspace). The second call must leave both
PyTorch's allocator and the device's free memory unchanged. Kept in a file
that runs last so a failure here comes after every other test has run."""

import ctypes
import math

import pytest

torch = pytest.importorskip("torch")

from exact_attention_16_gb300 import api  # noqa: E402
from exact_attention_16_gb300.workloads import Workload, draw_inputs  # noqa: E402

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _noalloc_into(q, k, v, o, lse, causal, num_splits):
    B, Sq, Hq, D = q.shape
    _, Sk, Hkv, _ = k.shape
    return api.lib().fa_fwd_decode_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                           B, Sq, Sk, Hq, Hkv, D, ctypes.c_float(1.0 / math.sqrt(D)), int(causal),
                                           api.FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else api.FA_DTYPE_FP16,
                                           num_splits, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _noalloc(q, k, v, causal, num_splits):
    o = torch.full_like(q, float("nan"))
    lse = torch.full((q.shape[0], q.shape[2], q.shape[1]), float("nan"), dtype=torch.float32, device=q.device)
    return _noalloc_into(q, k, v, o, lse, causal, num_splits), o, lse


@pytest.mark.parametrize("splits", [0, 7])
def test_noalloc_matches_oracle_and_workspace_call_twice(splits):
    import oracle
    from parity import compare

    shapes = [Workload("na1", 4, 1, 3000, 32, 4, 128, "bf16", True, 1.0, 1.0, 41),
              Workload("na2", 2, 4, 1800, 16, 2, 128, "bf16", False, 2.0, 1.0, 42)]
    for n, w in enumerate(shapes):                     # two calls in a row, different inputs
        q_h, k_h, v_h = draw_inputs(w)
        q, k, v = q_h.cuda(), k_h.cuda(), v_h.cuda()
        need = api.fa_decode_workspace_size(w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.D, splits)
        assert 0 < need <= SCRATCH_BYTES
        o = torch.full_like(q, float("nan"))
        lse = torch.full((w.B, w.Hq, w.Sq), float("nan"), dtype=torch.float32, device=q.device)
        torch.cuda.synchronize()
        before = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
        rc = _noalloc_into(q, k, v, o, lse, w.causal, splits)
        torch.cuda.synchronize()
        after = (torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0])
        assert rc == api.FA_OK
        assert api.fa_status() == 0
        if n == 1:
            # the first call on a device may load the scratch module; later
            # calls allocate nothing at all
            assert after == before, (before, after)
        o_ref, l_ref = oracle.attention(q_h.float().numpy(), k_h.float().numpy(), v_h.float().numpy(), w.scale,
                                        w.causal)
        compare(o.float().cpu().numpy().transpose(0, 2, 1, 3), lse.cpu().numpy(), o_ref.transpose(0, 2, 1, 3), l_ref)
        o_ws, l_ws = api.fa_fwd_decode(q, k, v, causal=w.causal, num_splits=splits)
        assert api.fa_status() == 0
        err = (o.float() - o_ws.float()).abs()
        assert err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
        assert (lse - l_ws).abs().max().item() <= 1e-3


def test_noalloc_rejects_workspace_beyond_the_array():
    # 64 query heads x 16 positions x 8 batch rows over 5+ splits need > 16 MiB
    B, Sq, Sk, Hq, Hkv, D = 8, 16, 4096, 64, 8, 128
    need = api.fa_decode_workspace_size(B, Sq, Sk, Hq, Hkv, D, 8)
    assert need > SCRATCH_BYTES
    q = torch.zeros(B, Sq, Hq, D, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(B, Sk, Hkv, D, dtype=torch.bfloat16, device="cuda")
    rc, _, _ = _noalloc(q, k, k, True, 8)
    assert rc == api.FA_ERR_UNSUPPORTED
