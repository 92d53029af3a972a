"""The verify call captured in a CUDA graph and replayed on new inputs.

The launch never reads device data on the host: grid, split plan and tensor
maps depend only on (B, q_len, H, Smax), the pointers and the device.  A
captured call therefore stays valid when the contents of its inputs change in
place between replays, seq_lens included (within Smax).  The first call on a
device does one-time setup (kernel attributes, occupancy query) and is made
before capture.  The captured call here takes the split path, so the graph
holds the split kernel and the slice merge (a programmatic dependent launch).
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
    assert np.isfinite(o).all() and np.isfinite(l).all()
    assert np.abs(o - ref_out).max() <= TOL_OUT
    assert np.abs(l - ref_lse).max() <= TOL_LSE


def test_graph_replay_matches_eager_and_follows_new_inputs():
    import torch
    import mla_verify_attention_gb300 as mva
    w = I.WORKLOADS["tree9_p4096"]
    case_a = I.make_case(w)
    # Same shapes, other values, and a shorter stream: its drafts are cache
    # rows 3000..3008 and everything from row 3009 on is NaN.
    case_b = I.make_case(w, seed=w.seed + 1000)
    case_b.seq_lens = np.array([3009], dtype=np.int32)
    case_b.kv[:, 3009:, :] = 0x7FC0
    B, q, H, Smax, scale = case_a.B, case_a.q, case_a.H, case_a.Smax, float(case_a.scale)
    assert case_b.Smax == Smax and float(case_b.scale) == scale
    assert mva.plan(B, q, H, Smax)[1] > 1, "the captured call must take the split path"

    inputs = _dev(case_a)
    out = torch.empty((B, q, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, q, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(mva.workspace_size(B, q, H, Smax), dtype=torch.uint8, device="cuda")

    mva.verify_attn(*inputs, scale, out=out, lse=lse, workspace=ws)   # setup, outside capture
    torch.cuda.synchronize()
    eager_out, eager_lse = out.clone(), lse.clone()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mva.verify_attn(*inputs, scale, out=out, lse=lse, workspace=ws)

    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert mva.last_device_error() == 0
    assert torch.equal(out, eager_out) and torch.equal(lse, eager_lse)
    _check(case_a, out, lse)

    for dst, src in zip(inputs, _dev(case_b)):
        dst.copy_(src)
    graph.replay()
    torch.cuda.synchronize()
    assert mva.last_device_error() == 0
    _check(case_b, out, lse)
    ref_out, ref_lse = mva.verify_attn(*inputs, scale)
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_graph_replay_with_device_plan_follows_new_stream_lengths():
    # Several streams: the slice count is chosen on the device from seq_lens
    # (a planner launch inside the captured sequence), so replays with other
    # lengths re-plan and stay exact.
    import torch
    import mla_verify_attention_gb300 as mva
    prefixes_a = [3000, 400, 1500, 6000]
    prefixes_b = [200, 5900, 100, 900]
    w = I.Workload("custom", 4, 9, 0, "random", 5, None, H=64, index=0)
    case_a = I.make_case(w, seed=71, prefixes=prefixes_a)
    case_b = I.make_case(w, seed=72, prefixes=prefixes_b, smax_align=case_a.Smax)
    assert case_b.Smax == case_a.Smax
    B, q, H, Smax, scale = case_a.B, case_a.q, case_a.H, case_a.Smax, float(case_a.scale)
    assert mva.plan(B, q, H, Smax)[1] > 1

    inputs = _dev(case_a)
    out = torch.empty((B, q, H, 512), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, q, H), dtype=torch.float32, device="cuda")
    ws = torch.empty(mva.workspace_size(B, q, H, Smax), dtype=torch.uint8, device="cuda")
    mva.verify_attn(*inputs, scale, out=out, lse=lse, workspace=ws)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mva.verify_attn(*inputs, scale, out=out, lse=lse, workspace=ws)
    for case in (case_a, case_b, case_a):
        for dst, src in zip(inputs, _dev(case)):
            dst.copy_(src)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert mva.last_device_error() == 0
        _check(case, out, lse)
