"""Back-to-back calls on one stream see their own inputs.

Every kernel of a call is launched as a programmatic dependent of the grid
before it (a launch that may start while that grid finishes) and waits for
that grid before reading anything; the copy of a paged cache and the split
plan sit between them on some paths.  Here a torch kernel rewrites the inputs
between two calls on the same stream, and each call's output must match the
oracle on its own inputs: any read of an input before the grid that wrote it
had finished would show up as a mismatch.  The cases cover the one-stream
path (merge of slices), the device-planned several-stream path and the
copied paged cache.
"""
import numpy as np
import pytest

import oracle
from mla_verify_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL_OUT = 2e-3
TOL_LSE = 1e-3


def _case(B, prefixes, seed):
    w = I.Workload("order", B, 9, 0, "random", 5, None, H=64, index=0)
    return I.make_case(w, seed=seed, prefixes=prefixes)


def _check(case, out, lse):
    ref_out, ref_lse = oracle.case_reference(case)
    o = out.cpu().numpy().astype(np.float64).reshape(ref_out.shape)
    l = lse.cpu().numpy().astype(np.float64).reshape(ref_lse.shape)
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(l), empty)
    assert np.abs(o - ref_out).max() <= TOL_OUT
    assert np.abs(l[~empty] - ref_lse[~empty]).max() <= TOL_LSE


@pytest.mark.parametrize("B,prefixes,page", [
    (1, [3000], 0),                  # one stream: split kernel, then the merge
    (3, [2500, 400, 1800], 0),       # device plan, split kernel, merge
    (3, [2500, 400, 1800], 16),      # cache copy, device plan, split kernel, merge
    (1, [3000], 16),                 # cache copy, split kernel, merge
])
def test_inputs_rewritten_between_calls(B, prefixes, page):
    import torch
    import mla_verify_attention_gb300 as mva

    a = _case(B, prefixes, seed=510 + B + page)
    b = _case(B, prefixes, seed=610 + B + page)

    def t(x, dt):
        return torch.from_numpy(np.ascontiguousarray(x)).view(dt).cuda()

    def host(case):
        if page:
            pool, table = I.to_paged(case, page, seed=3)
            cache = [pool.view(np.int16), table]
        else:
            cache = [case.kv.view(np.int16)]
        return [case.q_nope.view(np.int16), case.q_rope.view(np.int16), *cache,
                case.seq_lens, case.mask.view(np.int32)]

    ha, hb = host(a), host(b)
    dts = [torch.bfloat16, torch.bfloat16] + ([torch.bfloat16, torch.int32] if page else [torch.bfloat16]) \
        + [torch.int32, torch.int32]
    dev = [t(x, dt) for x, dt in zip(ha, dts)]
    src_b = [t(x, dt) for x, dt in zip(hb, dts)]

    def call():
        if page:
            qn, qr, pool, table, sl, m = dev
            return mva.verify_attn_paged(qn, qr, pool, table, page, sl, m, float(a.scale))
        qn, qr, kv, sl, m = dev
        return mva.verify_attn(qn, qr, kv, sl, m, float(a.scale))

    torch.cuda.synchronize()
    out_a, lse_a = call()
    for d, s in zip(dev, src_b):      # torch copy kernels on the same stream
        d.copy_(s)
    out_b, lse_b = call()
    torch.cuda.synchronize()
    assert mva.last_device_error() == 0
    _check(a, out_a, lse_a)
    _check(b, out_b, lse_b)
