"""The seeded input generator: reproducible, correctly rounded, and shaped
like the pages' workloads."""
import numpy as np
import pytest

from mla_verify_attention_gb300 import inputs as I


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    x = np.concatenate([I.normal_f32(1, "r", 100000) * 37.0,
                        np.array([0.0, -0.0, 1e-40, 3.0e38, -1.5, np.inf, -np.inf], np.float32)])
    ours = I.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)


def test_streams_are_reproducible_and_distinct():
    a = I.normal_bf16(5, "kv", (3, 7))
    np.testing.assert_array_equal(a, I.normal_bf16(5, "kv", (3, 7)))
    assert not np.array_equal(a, I.normal_bf16(5, "q_nope", (3, 7)))
    assert not np.array_equal(a, I.normal_bf16(6, "kv", (3, 7)))
    # chunked generation is identical to one-shot generation
    np.testing.assert_array_equal(I.normal_bf16(5, "kv", (1000,), chunk=64),
                                  I.normal_bf16(5, "kv", (1000,)))


def test_normal_statistics():
    x = I.normal_f32(3, "stats", 400000).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert abs((x ** 4).mean() - 3.0) < 0.05      # Gaussian kurtosis
    u = I.uniform(3, "u", 200000)
    assert u.min() >= 0.0 and u.max() < 1.0 and abs(u.mean() - 0.5) < 0.01


@pytest.mark.parametrize("q,dmax,kids", [(9, 5, None), (33, 8, 4), (64, 3, 4)])
def test_random_tree_limits(q, dmax, kids):
    for seed in range(20):
        par = I.random_tree_parents(q, seed, "t", dmax, kids)
        depth = [0] * q
        count = [0] * q
        for i in range(1, q):
            assert 0 <= par[i] < i
            depth[i] = depth[par[i]] + 1
            count[par[i]] += 1
        assert max(depth) <= dmax
        if kids is not None:
            assert max(count) <= kids
        m = I.ancestor_mask(par)
        for i in range(q):
            seen = {j for j in range(q) if (m[i, j >> 5] >> (j & 31)) & 1}
            path, j = set(), i
            while j >= 0:
                path.add(j)
                j = par[j]
            assert seen == path


def test_log_uniform_prefixes_in_range():
    v = I.log_uniform_ints(7, "seqlens", 5000, 1024, 32768)
    assert v.min() >= 1024 and v.max() <= 32768
    # log-uniform: the median sits near the geometric mean
    assert abs(np.log(np.median(v)) - 0.5 * (np.log(1024) + np.log(32768))) < 0.1


def test_workload_shapes():
    w = I.WORKLOADS["chain9_p256"]
    c = I.make_case(w)
    assert c.q_nope.shape == (1, 9, 64, 512) and c.q_rope.shape == (1, 9, 64, 64)
    assert c.kv.shape == (1, 320, 576) and list(c.seq_lens) == [265]
    assert np.isnan(I.bf16_bits_to_f32(c.kv[0, 265:])).all()
    assert not np.isnan(I.bf16_bits_to_f32(c.kv[0, :265])).any()
    np.testing.assert_array_equal(c.mask[0, :, 0], [(1 << (i + 1)) - 1 for i in range(9)])
    r = I.make_case(I.Workload("t", 8, 9, (1024, 32768), "random", 5, index=5,
                               Dl=8, Dr=4, H=2))
    assert r.kv.shape[1] % 64 == 0 and r.kv.shape[1] >= r.seq_lens.max()
    assert r.seq_lens.min() >= 1024 + 9
    assert float(c.scale) == float(np.float32(1 / np.sqrt(192)))


def test_scale_key_rope_changes_only_that_rope_part():
    w = I.Workload("t", 1, 9, 0, "random", 5, None, H=4, index=0)
    case = I.make_case(w, seed=3, prefixes=[200])
    before = case.kv.copy()
    I.scale_key_rope(case, 0, 150, 8.0)
    changed = np.argwhere(case.kv != before)
    assert set(changed[:, 1]) == {150} and changed[:, 2].min() >= 512
    old = I.bf16_bits_to_f32(before[0, 150, 512:])
    new = I.bf16_bits_to_f32(case.kv[0, 150, 512:])
    np.testing.assert_array_equal(new, old * np.float32(8.0))   # a power of two: exact in bf16
