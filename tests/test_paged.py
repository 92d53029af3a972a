"""The paged-cache entry point (mla_verify_attn_paged) through the C ABI.

Each case lays a seeded cache out as a page pool (random page order, NaN in
unused pages and past each stream's length) and compares the paged call with
the oracle on the logical cache, at the same tolerances as the contiguous
path; two cases also check that paged and contiguous calls agree bit for bit.
Pages of a multiple of 64 keys are read in place through the block table;
other sizes are first copied into a contiguous cache in the workspace.
"""
import numpy as np
import pytest

import oracle
from mla_verify_attention_gb300 import inputs as I

pytestmark = pytest.mark.gpu

TOL_OUT = 2e-3
TOL_LSE = 1e-3


def _t(a, dt):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).view(dt).cuda()


def run_paged(case, page_size, seed=11, extra_pages=3):
    import torch
    import mla_verify_attention_gb300 as mva
    pool, table = I.to_paged(case, page_size, seed, extra_pages)
    out, lse = mva.verify_attn_paged(
        _t(case.q_nope.view(np.int16), torch.bfloat16), _t(case.q_rope.view(np.int16), torch.bfloat16),
        _t(pool.view(np.int16), torch.bfloat16), _t(table, torch.int32), page_size,
        _t(case.seq_lens, torch.int32), _t(case.mask.view(np.int32), torch.int32), float(case.scale))
    torch.cuda.synchronize()
    st = mva.last_device_error()
    assert st == 0, mva.strerror(st)
    return out, lse


def check(case, out, lse):
    ref_out, ref_lse = oracle.case_reference(case)
    o = out.cpu().numpy().astype(np.float64).reshape(ref_out.shape)
    l = lse.cpu().numpy().astype(np.float64).reshape(ref_lse.shape)
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(l), empty)
    assert np.isfinite(o).all()
    assert np.abs(o - ref_out).max() <= TOL_OUT
    assert np.abs(l[~empty] - ref_lse[~empty]).max() <= TOL_LSE


@pytest.mark.parametrize("B,q,H,prefixes,page_size", [
    (1, 9, 64, [4096], 64),            # split path, one tile per page
    (1, 9, 64, [700], 256),            # tiles inside larger pages, partial last page
    (3, 5, 8, [10, 900, 2000], 128),   # ragged streams
    (2, 33, 64, [300, 1500], 64),      # two mask words
    # page sizes that are not whole key tiles: rows copied into the workspace first
    (1, 9, 64, [4096], 1),             # one row per page (scattered rows), split path
    (3, 5, 8, [10, 900, 2000], 16),    # ragged streams, 16-row pages
    (1, 33, 64, [700], 96),            # pages straddling key tiles
])
def test_paged_matches_oracle(B, q, H, prefixes, page_size):
    w = I.Workload("paged", B, q, 0, "random", 5, None, H=H)
    case = I.make_case(w, seed=123 + B + q + page_size, prefixes=prefixes)
    out, lse = run_paged(case, page_size)
    check(case, out, lse)


@pytest.mark.parametrize("B,prefixes,page_size", [
    (1, [991], 16),                 # Smax = 1000 keys: 63 pages of 16 = 1008 keys
    (3, [100, 991, 500], 7),        # 143 pages of 7 = 1001 keys, ragged
    (1, [4096], 48),                # 86 pages of 48 = 4128 keys, split path
])
def test_paged_smax_not_multiple_of_tile(B, prefixes, page_size):
    # The copied cache then has a row count that is not a whole number of
    # 64-key tiles: the last key box of a stream runs past it.
    w = I.Workload("paged", B, 9, 0, "random", 5, None, H=64)
    case = I.make_case(w, seed=77 + page_size, prefixes=prefixes, smax_align=1)
    max_blocks = -(-case.Smax // page_size)
    assert (max_blocks * page_size) % 64 != 0
    out, lse = run_paged(case, page_size)
    check(case, out, lse)


@pytest.mark.parametrize("page_size", [64, 16])
def test_paged_dominant_key_correction(page_size):
    # One term plus the dominant key's correction, whose value row is read
    # through the block table (64-key pages) or from the copy (16-row pages).
    # Without the correction these inputs are off by 3.8e-3.
    w = I.Workload("custom", 1, 9, 0, "random", 5, None, H=64, index=0)
    case = I.make_case(w, seed=2, prefixes=[6000])
    I.scale_key_rope(case, 0, 5100, 8.0)
    out, lse = run_paged(case, page_size)
    check(case, out, lse)
    ref_out, _ = oracle.case_reference(case)
    d = np.abs(out.cpu().numpy().astype(np.float64).reshape(ref_out.shape) - ref_out).max()
    assert d <= 1.2e-3, d


def test_paged_equals_contiguous_bitwise():
    import torch
    import mla_verify_attention_gb300 as mva
    case = I.make_case(I.WORKLOADS["tree9_p4096"])
    out_p, lse_p = run_paged(case, 64)
    ref = mva.verify_attn(_t(case.q_nope.view(np.int16), torch.bfloat16),
                          _t(case.q_rope.view(np.int16), torch.bfloat16),
                          _t(case.kv.view(np.int16), torch.bfloat16), _t(case.seq_lens, torch.int32),
                          _t(case.mask.view(np.int32), torch.int32), float(case.scale))
    torch.cuda.synchronize()
    # Smax is a whole number of 64-key pages, so both calls use the same split
    # plan and the same arithmetic order.
    assert case.Smax % 64 == 0
    assert torch.equal(out_p, ref[0]) and torch.equal(lse_p, ref[1])


def test_paged_bad_block_entry_is_reported():
    import torch
    import mla_verify_attention_gb300 as mva
    case = I.make_case(I.WORKLOADS["chain9_p256"])
    pool, table = I.to_paged(case, 64, seed=3)
    table = table.copy()
    table[0, 1] = pool.shape[0] // 64          # one past the last page
    out, lse = mva.verify_attn_paged(
        _t(case.q_nope.view(np.int16), torch.bfloat16), _t(case.q_rope.view(np.int16), torch.bfloat16),
        _t(pool.view(np.int16), torch.bfloat16), _t(table, torch.int32), 64,
        _t(case.seq_lens, torch.int32), _t(case.mask.view(np.int32), torch.int32), float(case.scale))
    torch.cuda.synchronize()
    assert mva.last_device_error() == -10          # MLA_ERR_PAGE, then cleared
    assert mva.last_device_error() == 0


def test_copied_pages_equal_contiguous_bitwise():
    """Page size 1: the split kernel reads a contiguous copy of the cache, so the
    result is the contiguous call's, bit for bit."""
    import torch
    import mla_verify_attention_gb300 as mva
    case = I.make_case(I.WORKLOADS["tree9_p4096"])
    out_p, lse_p = run_paged(case, 1)
    ref = mva.verify_attn(_t(case.q_nope.view(np.int16), torch.bfloat16),
                          _t(case.q_rope.view(np.int16), torch.bfloat16),
                          _t(case.kv.view(np.int16), torch.bfloat16), _t(case.seq_lens, torch.int32),
                          _t(case.mask.view(np.int32), torch.int32), float(case.scale))
    torch.cuda.synchronize()
    assert torch.equal(out_p, ref[0]) and torch.equal(lse_p, ref[1])


def test_paged_workspace_sizes():
    import torch
    import mla_verify_attention_gb300 as mva
    B, q, H, mb = 2, 9, 64, 70
    for ps in (64, 128):   # read in place: the contiguous call's workspace
        assert mva.paged_workspace_size(B, q, H, mb, ps) == mva.workspace_size(B, q, H, mb * ps)
    for ps in (1, 16, 96):  # plus the contiguous copy, after the partials at 256 bytes
        part = mva.workspace_size(B, q, H, mb * ps)
        assert mva.paged_workspace_size(B, q, H, mb, ps) == -(-part // 256) * 256 + B * mb * ps * 1152
    # one byte short is refused before anything is enqueued
    case = I.make_case(I.WORKLOADS["chain9_p256"])
    pool, table = I.to_paged(case, 1, seed=3)
    need = mva.paged_workspace_size(case.B, case.q, case.H, table.shape[1], 1)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = (_t(case.q_nope.view(np.int16), torch.bfloat16), _t(case.q_rope.view(np.int16), torch.bfloat16),
            _t(pool.view(np.int16), torch.bfloat16), _t(table, torch.int32), 1,
            _t(case.seq_lens, torch.int32), _t(case.mask.view(np.int32), torch.int32), float(case.scale))
    with pytest.raises(mva.MLAError) as e:
        mva.verify_attn_paged(*args, workspace=ws[:need - 1])
    assert e.value.status == -4
    out, lse = mva.verify_attn_paged(*args, workspace=ws)
    torch.cuda.synchronize()
    assert mva.last_device_error() == 0
    check(case, out, lse)
