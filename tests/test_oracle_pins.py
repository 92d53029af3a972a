"""Pins of the fp64 oracle to facts fixed by the pages and by mathematics.

None of these re-derive the oracle's own loop: each checks a closed form, an
invariant, or an independent library routine (torch's scaled-dot-product
attention and scipy's logsumexp) on inputs where the answer is known.  The
definition being pinned: score = q_nope . kv_c + q_pe . k_pe, scaled; tree-
masked softmax over visible keys; output = weighted sum of the 512-wide latent
(page "The Flash Attention Kernel That Had to Be Built: Designing sm_120 MLA
Verify for Blackwell Consumer GPUs", section "What Input Knowledge Is Required
to Understand This Message"); split partial states merged with the online-
softmax combine (page "The Decisive Microbench: When Theory Meets Silicon",
section "The KV-Split Solution").
"""
import math

import numpy as np
import pytest

import oracle
from mla_verify_attention_gb300 import inputs as I


def bf(x):
    return I.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def f(bits):
    return I.bf16_bits_to_f32(bits).astype(np.float64)


def small_case(seed, B=2, q=3, H=2, Dl=8, Dr=4, prefixes=(5, 0), pad=3, tree="random"):
    prefixes = np.asarray(prefixes[:B])
    seq = (prefixes + q).astype(np.int32)
    smax = int(seq.max()) + pad
    qn = I.normal_bf16(seed, "qn", (B, q, H, Dl))
    qr = I.normal_bf16(seed, "qr", (B, q, H, Dr))
    kv = I.normal_bf16(seed, "kv", (B, smax, Dl + Dr))
    for b in range(B):
        kv[b, seq[b]:] = 0x7FC0  # NaN padding
    masks = []
    for b in range(B):
        par = (I.chain_parents(q) if tree == "chain"
               else I.random_tree_parents(q, seed, "t%d" % b, 2, None))
        masks.append(I.ancestor_mask(par))
    return qn, qr, kv, seq, np.stack(masks)


def test_single_visible_key_closed_form():
    # One query, prefix of one key, the draft does not see itself: only key 0
    # is visible, so out = latent of key 0 and lse = its scaled score.
    Dl, Dr = 16, 8
    qn = np.zeros((1, 1, 1, Dl), np.float32); qn[0, 0, 0, 3] = 1.0
    qr = np.zeros((1, 1, 1, Dr), np.float32); qr[0, 0, 0, 5] = 2.0
    kv = np.random.default_rng(0).standard_normal((1, 4, Dl + Dr)).astype(np.float32)
    kv[0, 0, 3] = 2.0          # latent part contributes 1 * 2
    kv[0, 0, Dl + 5] = 3.0     # rope part contributes 2 * 3
    kv_b = bf(kv); kv_b[0, 2:] = 0x7FC0
    mask = np.zeros((1, 1, 1), np.uint32)
    scale = np.float32(0.125)
    out, lse = oracle.verify_attn(bf(qn), bf(qr), kv_b, np.array([2], np.int32), mask, scale)
    np.testing.assert_array_equal(out[0, 0, 0], f(kv_b[0, 0, :Dl]))
    assert lse[0, 0, 0] == pytest.approx(8.0 * 0.125, abs=1e-15)


def test_two_keys_exact_weights():
    # Integer inputs (exact in bf16).  Both keys score 1 on the latent part;
    # key 1 scores -2 more on the RoPE part, so with scale 1/2 the scaled
    # scores are +1/2 and -1/2 and the weights are e/(1+e) and 1/(1+e).
    Dl, Dr = 8, 4
    qn = np.zeros((1, 1, 1, Dl), np.float32); qn[0, 0, 0, 0] = 1.0
    qr = np.zeros((1, 1, 1, Dr), np.float32); qr[0, 0, 0, 1] = -1.0
    kv = np.zeros((1, 2, Dl + Dr), np.float32)
    kv[0, :, 0] = 1.0
    kv[0, 0, 1:Dl] = np.arange(1, Dl)            # latent of key 0
    kv[0, 1, 1:Dl] = -np.arange(1, Dl) * 2.0     # latent of key 1
    kv[0, 1, Dl + 1] = 2.0
    mask = np.ones((1, 1, 1), np.uint32)         # the draft (key 1) sees itself
    out, lse = oracle.verify_attn(bf(qn), bf(qr), bf(kv), np.array([2], np.int32), mask,
                                  np.float32(0.5))
    w0 = math.e / (1.0 + math.e)
    kv64 = kv.astype(np.float64)
    exp_out = w0 * kv64[0, 0, :Dl] + (1.0 - w0) * kv64[0, 1, :Dl]
    np.testing.assert_allclose(out[0, 0, 0], exp_out, rtol=0, atol=1e-14)
    assert lse[0, 0, 0] == pytest.approx(0.5 + math.log1p(math.exp(-1.0)), abs=1e-15)


def test_scale_zero_gives_mean_of_visible_latents():
    qn, qr, kv, seq, mask = small_case(11, B=2, q=5, H=3, prefixes=(7, 2))
    out, lse = oracle.verify_attn(qn, qr, kv, seq, mask, np.float32(0.0))
    Dl = qn.shape[3]
    for b in range(2):
        P = seq[b] - 5
        for i in range(5):
            vis = list(range(P)) + [P + j for j in range(5) if (mask[b, i, 0] >> j) & 1]
            mean = f(kv[b, vis, :Dl]).mean(0)
            for h in range(3):
                np.testing.assert_allclose(out[b, i, h], mean, atol=1e-13, rtol=0)
                assert lse[b, i, h] == pytest.approx(math.log(len(vis)), abs=1e-14)


def test_identical_latents_return_that_latent():
    qn, qr, kv, seq, mask = small_case(12, prefixes=(6, 3))
    Dl = qn.shape[3]
    v = bf(np.linspace(-2, 2, Dl))
    for b in range(2):
        kv[b, :seq[b], :Dl] = v
    out, _ = oracle.verify_attn(qn, qr, kv, seq, mask, np.float32(0.7))
    np.testing.assert_allclose(out.reshape(-1, Dl), np.broadcast_to(f(v), (out.size // Dl, Dl)),
                               atol=1e-13, rtol=0)


def test_empty_row_is_zero_and_minus_inf():
    qn, qr, kv, seq, mask = small_case(13, B=1, q=2, prefixes=(0,))
    mask[0, 0, 0] = 0               # draft 0 sees nothing, no prefix
    mask[0, 1, 0] = 0b10
    out, lse = oracle.verify_attn(qn, qr, kv, seq, mask, np.float32(0.3))
    assert np.all(out[0, 0] == 0.0) and np.all(np.isneginf(lse[0, 0]))
    assert np.all(np.isfinite(lse[0, 1]))


def test_masked_drafts_and_padding_have_no_influence():
    qn, qr, kv, seq, mask = small_case(14, B=2, q=4, H=2, prefixes=(5, 1), pad=4)
    scale = np.float32(0.4)
    out0, lse0 = oracle.verify_attn(qn, qr, kv, seq, mask, scale)
    for b in range(2):
        P = seq[b] - 4
        for i in range(4):
            hidden = [j for j in range(4) if not (mask[b, i, 0] >> j) & 1]
            for j in hidden:
                kv2 = kv.copy()
                kv2[b, P + j] = bf(np.full(kv.shape[2], 1e4))      # huge, finite
                kv2[b, seq[b]:] = bf(np.full(kv.shape[2], -3e4))   # padding changes too
                o2, l2 = oracle.verify_attn(qn, qr, kv2, seq, mask, scale)
                np.testing.assert_array_equal(o2[b, i], out0[b, i])
                np.testing.assert_array_equal(l2[b, i], lse0[b, i])


def test_prefix_permutation_invariance():
    qn, qr, kv, seq, mask = small_case(15, B=1, q=3, prefixes=(9,))
    scale = np.float32(0.35)
    out0, lse0 = oracle.verify_attn(qn, qr, kv, seq, mask, scale)
    perm = np.random.default_rng(1).permutation(9)
    kv2 = kv.copy(); kv2[0, :9] = kv[0, perm]
    out1, lse1 = oracle.verify_attn(qn, qr, kv2, seq, mask, scale)
    np.testing.assert_allclose(out1, out0, atol=1e-13, rtol=0)
    np.testing.assert_allclose(lse1, lse0, atol=1e-13, rtol=0)


@pytest.mark.parametrize("seed", [21, 22, 23])
def test_split_merge_equals_unsplit(seed):
    qn, qr, kv, seq, mask = small_case(seed, B=2, q=4, H=2, prefixes=(17, 3))
    scale = np.float32(0.3)
    out0, lse0 = oracle.verify_attn(qn, qr, kv, seq, mask, scale)
    rng = np.random.default_rng(seed)
    ns = 4
    cuts = np.stack([np.sort(np.concatenate([[0], rng.integers(0, s + 1, ns - 1), [s]]))
                     for s in seq])                            # ragged, empty slices allowed
    accs, ms, ls = [], [], []
    for k in range(ns):
        a, m, l = oracle.partial(qn, qr, kv, seq, mask, scale, cuts[:, k], cuts[:, k + 1])
        accs.append(a); ms.append(m); ls.append(l)
    out, lse = oracle.combine(np.stack(accs), np.stack(ms), np.stack(ls))
    np.testing.assert_allclose(out, out0.reshape(out.shape), atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, lse0.reshape(-1), atol=1e-12, rtol=0)


def test_weights_sum_to_one_and_vanish_on_hidden_keys():
    qn, qr, kv, seq, mask = small_case(16, B=1, q=5, H=2, prefixes=(8,), pad=5)
    for i in range(5):
        w = oracle.row_weights(qn, qr, kv, seq, mask, np.float32(0.9), 0, i, 1)
        assert abs(w.sum() - 1.0) < 1e-12
        P = seq[0] - 5
        for j in range(5):
            if not (mask[0, i, 0] >> j) & 1:
                assert w[P + j] == 0.0
        assert np.all(w[seq[0]:] == 0.0)


def _dense_visibility(seq, mask, q, smax):
    B = len(seq)
    vis = np.zeros((B, q, smax), bool)
    for b in range(B):
        P = seq[b] - q
        vis[b, :, :P] = True
        for i in range(q):
            for j in range(q):
                vis[b, i, P + j] = bool((mask[b, i, j >> 5] >> (j & 31)) & 1)
    return vis


@pytest.mark.parametrize("tree", ["chain", "random"])
def test_matches_torch_sdpa_and_scipy_logsumexp(tree):
    torch = pytest.importorskip("torch")
    from scipy.special import logsumexp
    qn, qr, kv, seq, mask = small_case(17, B=2, q=6, H=3, Dl=16, Dr=8, prefixes=(11, 4),
                                       tree=tree)
    scale = np.float32(0.21)
    out, lse = oracle.verify_attn(qn, qr, kv, seq, mask, scale)
    B, q, H, Dl = qn.shape
    vis = _dense_visibility(seq, mask, q, kv.shape[1])
    Q = np.concatenate([f(qn), f(qr)], axis=-1)        # [B,q,H,576-like]
    for b in range(B):
        S = seq[b]
        K = f(kv[b, :S])                                # only real rows
        V = K[:, :Dl]
        qb = torch.from_numpy(Q[b].transpose(1, 0, 2).copy())          # [H, q, D]
        kb = torch.from_numpy(np.broadcast_to(K, (H,) + K.shape).copy())
        vb = torch.from_numpy(np.broadcast_to(V, (H,) + V.shape).copy())
        am = torch.from_numpy(np.broadcast_to(vis[b, :, :S], (H, q, S)).copy())
        ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, attn_mask=am,
                                                               scale=float(scale))
        np.testing.assert_allclose(out[b].transpose(1, 0, 2), ref.numpy(), atol=1e-12, rtol=0)
        sc = float(scale) * np.einsum("qhd,sd->hqs", Q[b], K)
        sc = np.where(vis[b, None, :, :S], sc, -np.inf)
        np.testing.assert_allclose(lse[b].T, logsumexp(sc, axis=-1), atol=1e-12, rtol=0)


def test_chain_mask_is_causal_over_prefix_and_drafts():
    # A chain of drafts is ordinary causal attention over prefix + drafts.
    qn, qr, kv, seq, mask = small_case(18, B=1, q=7, H=2, prefixes=(6,), tree="chain")
    P = seq[0] - 7
    causal = np.zeros((1, 7, kv.shape[1]), bool)
    for i in range(7):
        causal[0, i, :P + i + 1] = True
    np.testing.assert_array_equal(_dense_visibility(seq, mask, 7, kv.shape[1]), causal)
    dense = np.tril(np.ones((7, 7), bool))[None]
    np.testing.assert_array_equal(I.pack_mask(dense), mask)


def test_rejects_bad_seq_lens():
    qn, qr, kv, seq, mask = small_case(19, B=1, q=3, prefixes=(4,))
    with pytest.raises(ValueError):
        oracle.verify_attn(qn, qr, kv, np.array([2], np.int32), mask, np.float32(1))
    with pytest.raises(ValueError):
        oracle.verify_attn(qn, qr, kv, np.array([kv.shape[1] + 1], np.int32), mask, np.float32(1))


def test_mask_word_boundary_q33():
    # Draft 32 lives in the second mask word; a tree whose node 32 is visible
    # only through that word must change the result when the bit is cleared.
    q = 33
    qn = I.normal_bf16(30, "qn", (1, q, 1, 8))
    qr = I.normal_bf16(30, "qr", (1, q, 1, 4))
    kv = I.normal_bf16(30, "kv", (1, 4 + q, 12))
    seq = np.array([4 + q], np.int32)
    mask = I.ancestor_mask(I.chain_parents(q))[None]
    out0, _ = oracle.verify_attn(qn, qr, kv, seq, mask, np.float32(0.5))
    m2 = mask.copy(); m2[0, 32, 1] = 0           # draft 32 no longer sees itself
    out1, _ = oracle.verify_attn(qn, qr, kv, seq, m2, np.float32(0.5))
    assert not np.array_equal(out0[0, 32], out1[0, 32])
    np.testing.assert_array_equal(out0[0, :32], out1[0, :32])


def test_golden_fixture_regression():
    # Inputs and expected values written by tests/golden/make_golden.py, which
    # calls only the oracle; guards against unintended changes to it.
    import json, os
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_small.json")
    g = json.load(open(path))
    arr = {k: np.array(v, dtype=g["dtypes"][k]).reshape(g["shapes"][k]) for k, v in g["inputs"].items()}
    out, lse = oracle.verify_attn(arr["q_nope"], arr["q_rope"], arr["kv"], arr["seq_lens"],
                                  arr["mask"], np.float32(g["scale"]))
    np.testing.assert_allclose(out.reshape(-1), np.array(g["out"]), atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse.reshape(-1), np.array(g["lse"]), atol=1e-12, rtol=0)
