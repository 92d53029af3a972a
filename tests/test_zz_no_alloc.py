"""The scratch-free entry point, mla_verify_attn_noalloc.

Some callers cannot allocate device memory for the key-split scratch: code
whose device memory is fully pre-planned by its own arena, latency-critical
loops where cudaMalloc/cudaFree would synchronise the device, or plain C callers
with no allocator.  For them the library keeps one fixed scratch array on each
device.  These tests call that entry point through the C ABI, twice in a row on
a workload whose key range is split (so the array really holds partials), and
compare each result with the workspace-taking entry point, bit for bit (same
plan, same kernels, same arithmetic order); then check that a
call needing more scratch than the array holds is rejected with nothing run.

This file sorts last so that a run stopping at its first failure has already
run every other test; it sets up everything it needs itself.
"""
import ctypes

import numpy as np
import pytest

from mla_verify_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

NOALLOC_SCRATCH_BYTES = 32 << 20


def _lib():
    import mla_verify_attention_gb300 as mva
    lib = mva.load_library()
    P, Ii, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.mla_verify_attn_noalloc.argtypes = [P, P, P, P, P, Ii, Ii, Ii, Ii, F, P, P, P]
    lib.mla_verify_attn_noalloc.restype = Ii
    return lib


def _dev(case):
    import torch
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).view(dt).cuda()
    return (t(case.q_nope.view(np.int16), torch.bfloat16), t(case.q_rope.view(np.int16), torch.bfloat16),
            t(case.kv.view(np.int16), torch.bfloat16), t(case.seq_lens, torch.int32),
            t(case.mask.view(np.int32), torch.int32))


def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    import mla_verify_attention_gb300 as mva
    lib = _lib()
    case = I.make_case(I.WORKLOADS["tree9_p4096"])
    B, q, H, Smax = case.B, case.q, case.H, case.Smax
    assert mva.plan(B, q, H, Smax)[1] > 1, "workload must split the key range"
    need = mva.workspace_size(B, q, H, Smax)
    assert 0 < need <= NOALLOC_SCRATCH_BYTES
    qn, qr, kv, sl, m = _dev(case)
    ref_out, ref_lse = mva.verify_attn(qn, qr, kv, sl, m, float(case.scale))
    torch.cuda.synchronize()
    assert mva.last_device_error() == 0
    stream = int(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = torch.full((B, q, H, 512), float("nan"), device="cuda")
        lse = torch.full((B, q, H), float("nan"), device="cuda")
        st = lib.mla_verify_attn_noalloc(qn.data_ptr(), qr.data_ptr(), kv.data_ptr(), sl.data_ptr(),
                                         m.data_ptr(), B, q, H, Smax, float(case.scale),
                                         out.data_ptr(), lse.data_ptr(), stream)
        assert st == 0, mva.strerror(st)
        torch.cuda.synchronize()
        assert mva.last_device_error() == 0
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()
        # Same plan, same kernels, same arithmetic order: equal bit for bit.
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_noalloc_rejects_more_scratch_than_it_has():
    import torch
    import mla_verify_attention_gb300 as mva
    lib = _lib()
    B, q, H, Smax = 8, 9, 64, 32832     # ragged-batch shape: ~76 MB of partials
    assert mva.workspace_size(B, q, H, Smax) > NOALLOC_SCRATCH_BYTES
    small = torch.zeros(1024, dtype=torch.float32, device="cuda")
    out = torch.full((16,), 7.0, device="cuda")
    p = small.data_ptr()
    st = lib.mla_verify_attn_noalloc(p, p, p, p, p, B, q, H, Smax, 0.1, out.data_ptr(), p,
                                     int(torch.cuda.current_stream().cuda_stream))
    assert st == -4, mva.strerror(st)                # MLA_ERR_WORKSPACE, nothing enqueued
    torch.cuda.synchronize()
    assert (out == 7.0).all()
