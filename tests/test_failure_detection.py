"""Failure detection and memory discipline on the GPU, without faulting it.

- A stalled pipeline: the library's test control (mla_verify_attn_set_test_controls)
  makes one work unit withhold a cache load; its bounded waits run out (2 s), the kernels unwind,
  the device status reports MLA_ERR_DEVICE_TIMEOUT, and the next call on the
  same context is correct.
- Guard bands: out, lse and the workspace are surrounded by sentinel bytes
  that must be untouched after a call (a stand-in for a sanitizer, which is
  not available here), on split, unsplit and ragged calls.
"""
import numpy as np
import pytest

import oracle
from mla_verify_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL_OUT = 2e-3
TOL_LSE = 1e-3


def _dev(case):
    import torch

    def t(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a)).view(dt).cuda()

    return [t(case.q_nope.view(np.int16), torch.bfloat16), t(case.q_rope.view(np.int16), torch.bfloat16),
            t(case.kv.view(np.int16), torch.bfloat16), t(case.seq_lens, torch.int32),
            t(case.mask.view(np.int32), torch.int32)]


def _check(case, out, lse):
    ref_out, ref_lse = oracle.case_reference(case)
    o = out.cpu().numpy().astype(np.float64).reshape(ref_out.shape)
    l = lse.cpu().numpy().astype(np.float64).reshape(ref_lse.shape)
    assert np.abs(o - ref_out).max() <= TOL_OUT
    assert np.abs(l - ref_lse).max() <= TOL_LSE


def test_stalled_pipeline_reports_timeout_and_recovers():
    import torch
    import mla_verify_attention_gb300 as mva
    case = I.make_case(I.WORKLOADS["chain9_p256"])
    inputs = _dev(case)
    assert mva.last_device_error() == 0
    with mva.forced(stall=True):
        mva.verify_attn(*inputs, float(case.scale))    # enqueued: the stall is device-side
        torch.cuda.synchronize()
    assert mva.last_device_error() == -7               # MLA_ERR_DEVICE_TIMEOUT, then cleared
    out, lse = mva.verify_attn(*inputs, float(case.scale))
    torch.cuda.synchronize()
    assert mva.last_device_error() == 0
    _check(case, out, lse)


GUARD = 4096      # bytes on each side (keeps the 256-byte workspace alignment)


@pytest.mark.parametrize("name,nsplit", [("tree9_p4096", None), ("chain9_p256", 1),
                                         ("ragged8_tree9", None)])
def test_guard_bands_untouched(name, nsplit):
    import mla_verify_attention_gb300 as mva
    with mva.forced(nsplit=nsplit):
        _guard_bands(name, nsplit)


def _guard_bands(name, nsplit):
    import torch
    import mla_verify_attention_gb300 as mva
    case = I.make_case(I.WORKLOADS[name])
    B, q, H, Smax = case.B, case.q, case.H, case.Smax
    n_out, n_lse = B * q * H * 512 * 4, B * q * H * 4
    need = mva.workspace_size(B, q, H, Smax)
    if nsplit is None:
        assert need > 0, "case must use the workspace"
    bufs = {}
    for key, n in (("out", n_out), ("lse", n_lse), ("ws", need)):
        b = torch.full((n + 2 * GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
        bufs[key] = b
    out = bufs["out"][GUARD:GUARD + n_out].view(torch.float32).view(B, q, H, 512)
    lse = bufs["lse"][GUARD:GUARD + n_lse].view(torch.float32).view(B, q, H)
    ws = bufs["ws"][GUARD:GUARD + need] if need else None
    mva.verify_attn(*_dev(case), float(case.scale), out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()
    assert mva.last_device_error() == 0
    for key, n in (("out", n_out), ("lse", n_lse), ("ws", need)):
        b = bufs[key].cpu().numpy()
        assert (b[:GUARD] == 0xA5).all() and (b[GUARD + n:] == 0xA5).all(), key
    _check(case, out, lse)
