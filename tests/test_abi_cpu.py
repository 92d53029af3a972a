"""The C ABI without a GPU: the library builds, loads and exports every
function the header declares; host-side argument checks return their codes
before touching the device; the split planner's arithmetic."""
import ctypes
import os
import re

import pytest

import mla_verify_attention_gb300 as mva
from mla_verify_attention_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", src, re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    return mva.load_library()


def test_every_declared_symbol_is_exported(lib):
    names = header_functions()
    assert set(_lib.EXPORTED) <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_strerror(lib):
    for code, name in _lib.STATUS_NAMES.items():
        assert mva.strerror(code).startswith(name)
    assert "unknown" in mva.strerror(12345)


def call(lib, **kw):
    a = dict(qn=16, qr=16, kv=16, sl=16, m=16, B=1, q=9, H=64, Smax=320, scale=0.07,
             out=16, lse=16, ws=0, wsb=0)
    a.update(kw)
    return lib.mla_verify_attn(a["qn"], a["qr"], a["kv"], a["sl"], a["m"], a["B"], a["q"], a["H"],
                               a["Smax"], a["scale"], a["out"], a["lse"], a["ws"], a["wsb"], None)


def test_host_argument_checks(lib):
    assert call(lib, q=0) == -2 and call(lib, q=65) == -2 and call(lib, H=0) == -2
    assert call(lib, Smax=0) == -2 and call(lib, B=-1) == -2 and call(lib, Smax=1 << 24) == -2
    assert call(lib, scale=float("nan")) == -9 and call(lib, scale=float("inf")) == -9
    assert call(lib, B=0, qn=0, kv=0) == 0                      # nothing to do
    for k in ("qn", "qr", "kv", "sl", "m", "out", "lse"):
        assert call(lib, **{k: 0}) == -1, k
    assert call(lib, kv=24) == -3 and call(lib, out=8) == -3 and call(lib, lse=2) == -3
    assert call(lib, ws=272) == -3


def test_no_device_is_reported(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert call(lib) == -5
    assert lib.mla_verify_attn_workspace_size(1, 9, 64, 320) == 0


def test_plan_arithmetic(lib):
    # 152 SMs -> 76 two-CTA clusters.  One 64k stream of 9 drafts x 64 heads:
    # 576 rows = 5 row tiles; 15 slices of 69 tiles fill 75 clusters.
    assert mva.plan(1, 9, 64, 65600, 76) == (5, 15, 69)
    # 33 drafts over 16k: 17 row tiles, 4 slices.
    assert mva.plan(1, 33, 64, 16448, 76) == (17, 4, 65)
    # short prefix: slices are at least 2 tiles long
    assert mva.plan(1, 9, 64, 320, 76) == (5, 3, 2)
    # 4k prefix: 15 slices would be wanted; 5-tile slices give 13
    assert mva.plan(1, 9, 64, 4160, 76) == (5, 13, 5)
    # ragged batch: smaller slices for balance
    nrt, ns, ct = mva.plan(8, 9, 64, 32832, 76)
    assert nrt == 5 and ns * ct >= 513 and (ns - 1) * ct < 513 and ct >= 2
    # streams that alone fill a wave (16 x 5 row tiles > 76 clusters) are still
    # cut into about four waves' worth of slices: 304 / 80 -> 4
    assert mva.plan(16, 9, 64, 24320, 76)[1] == 4
    # H other than 64 and one query row
    assert mva.plan(1, 1, 1, 64, 76)[0] == 1
    assert mva.plan(2, 3, 16, 1000, 76)[0] == 1


def test_forced_slice_count(lib, monkeypatch):
    with mva.forced(nsplit=3):
        assert mva.plan(1, 9, 64, 320, 76) == (5, 3, 2)
    with mva.forced(nsplit=100):
        assert mva.plan(1, 9, 64, 320, 76) == (5, 5, 1)
    assert mva.plan(1, 9, 64, 320, 76) == (5, 3, 2)          # own plan again
    # the environment is never consulted
    monkeypatch.setenv("MLA_VERIFY_NSPLIT", "100")
    assert mva.plan(1, 9, 64, 4160, 76) == (5, 13, 5)
    assert lib.mla_verify_attn_set_test_controls(-1, 0) == -9   # MLA_ERR_ARG
    assert mva.plan(1, 9, 64, 4160, 76) == (5, 13, 5)


def test_two_term_limit_setter(lib):
    assert lib.mla_verify_attn_set_two_term_max_keys(-1) == -9   # MLA_ERR_ARG
    with pytest.raises(mva.MLAError):
        mva.set_two_term_max_keys(-5)
    for v in (0, 2**31 - 1, mva.TWO_TERM_MAX_KEYS_DEFAULT):
        mva.set_two_term_max_keys(v)


def paged(lib, **kw):
    a = dict(qn=16, qr=16, pool=16, rows=640, bt=16, mb=5, ps=128, sl=16, m=16, B=1, q=9, H=64,
             scale=0.07, out=16, lse=16, ws=0, wsb=0)
    a.update(kw)
    return lib.mla_verify_attn_paged(a["qn"], a["qr"], a["pool"], a["rows"], a["bt"], a["mb"],
                                     a["ps"], a["sl"], a["m"], a["B"], a["q"], a["H"], a["scale"],
                                     a["out"], a["lse"], a["ws"], a["wsb"], None)


def test_paged_host_argument_checks(lib):
    # page sizes >= 1; the pool is whole pages, < 2^31 rows
    for ps in (0, -64):
        assert paged(lib, ps=ps) == -2, ps
    assert paged(lib, rows=650) == -2 and paged(lib, rows=0) == -2 and paged(lib, mb=0) == -2
    assert paged(lib, ps=100, rows=750) == -2                  # 750 rows: not whole pages
    assert paged(lib, rows=1 << 31) == -2
    assert paged(lib, mb=1 << 18, ps=64) == -2                  # Smax = 2^24
    assert paged(lib, bt=0) == -1 and paged(lib, pool=0) == -1
    assert paged(lib, bt=2) == -3
    assert paged(lib, B=0, bt=0, pool=0) == 0                   # nothing to do
    assert paged(lib, q=0) == -2 and paged(lib, scale=float("nan")) == -9


def test_paged_workspace_size_rejects_bad_arguments(lib):
    # Arguments mla_verify_attn_paged rejects size no workspace (and without a
    # GPU every size is 0: the plan depends on the device).
    for mb, ps in ((0, 64), (5, 0), (1 << 18, 64), (1 << 24, 1)):
        assert mva.paged_workspace_size(1, 9, 64, mb, ps) == 0, (mb, ps)


def test_paged_layout_helper():
    from mla_verify_attention_gb300 import inputs as I
    case = I.make_case(I.Workload("t", 2, 3, 100, "chain", H=2), smax_align=64)
    pool, table = I.to_paged(case, 64, seed=5)
    assert table.shape == (2, 2) and pool.shape == ((2 * 2 + 3) * 64, 576)
    assert len(set(table.ravel().tolist())) == table.size        # distinct pages
    for b in range(2):
        for t in (0, 63, 64, int(case.seq_lens[b]) - 1):
            row = int(table[b, t // 64]) * 64 + t % 64
            assert (pool[row] == case.kv[b, t]).all()
