"""Seeded synthetic inputs for absorbed-MLA verify attention.

This module only makes numbers: bf16 query/cache tensors drawn from N(0, 1),
random draft trees, their bit-packed ancestor masks and ragged sequence
lengths.  It holds none of the attention arithmetic, so the CPU oracle and the
CUDA path can both be fed from it without sharing any of the method.

Random numbers come from a counter-based generator: value ``i`` of a tensor is
``splitmix64(key + (i + 1) * 0x9E3779B97F4A7C15)``, where ``key`` hashes the
base seed with the tensor's tag (FNV-1a 64 of the tag bytes).  splitmix64 is
the finaliser published by Steele, Lea and Flood ("Fast splittable
pseudorandom number generators", OOPSLA 2014).  Each 64-bit draw gives two
32-bit uniforms and, through the Box-Muller transform, two normals; normals are
rounded to bf16 with round-to-nearest-even.

Workload shapes follow the verify-attention benchmark of the pages: H = 64
heads, a 512-wide latent plus a 64-wide RoPE part (576-wide cache rows), q_len
9 or 33 draft tokens, prefixes from 256 to 65536 (page "The Moment of Truth:
Benchmarking a Custom sm_120 Flash Attention Kernel", section "The Message: Raw
Performance Data", the ``verify_attn (MLA absorb, H=64 Dl=512 Dr=64)`` table).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
BASE_SEED = 0x4D4C41
DL, DR = 512, 64
H_DEFAULT = 64

_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser on a uint64 array (wrapping arithmetic)."""
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def _fnv1a64(data: bytes) -> int:
    h = 0xCBF29CE484222325
    for b in data:
        h ^= b
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def stream_key(seed: int, tag: str) -> np.uint64:
    """64-bit key of one named random stream under a base seed."""
    k = np.uint64((_fnv1a64(tag.encode()) ^ ((seed * 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF))
                  & 0xFFFFFFFFFFFFFFFF)
    return _mix(np.array([k], dtype=np.uint64))[0]


def raw64(seed: int, tag: str, start: int, n: int) -> np.ndarray:
    """Draws ``start .. start+n-1`` of the stream as uint64."""
    key = stream_key(seed, tag)
    ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix(key + ctr * GOLDEN)


def uniform(seed: int, tag: str, n: int, start: int = 0) -> np.ndarray:
    """n uniforms in [0, 1) (53-bit resolution), float64."""
    z = raw64(seed, tag, start, n)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal_f32(seed: int, tag: str, n: int, start: int = 0) -> np.ndarray:
    """n standard normals (Box-Muller, two per 64-bit draw), float32.

    ``start`` must be even so that chunks line up with the pairs.
    """
    assert start % 2 == 0
    npair = (n + 1) // 2
    z = raw64(seed, tag, start // 2, npair)
    hi = (z >> np.uint64(32)).astype(np.float64)
    lo = (z & np.uint64(0xFFFFFFFF)).astype(np.float64)
    u1 = (hi + 0.5) * (1.0 / 4294967296.0)          # (0, 1)
    u2 = lo * (1.0 / 4294967296.0)                  # [0, 1)
    r = np.sqrt(-2.0 * np.log(u1))
    t = 2.0 * math.pi * u2
    out = np.empty(2 * npair, dtype=np.float64)
    out[0::2] = r * np.cos(t)
    out[1::2] = r * np.sin(t)
    return out[:n].astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    r = np.where(nan, (u >> 16) | 0x40, r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(seed: int, tag: str, shape, chunk: int = 1 << 22) -> np.ndarray:
    """N(0, 1) rounded to bf16, as uint16 bits of the given shape."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    chunk -= chunk % 2
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = f32_to_bf16_bits(normal_f32(seed, tag, e - s, start=s))
    return out.reshape(shape)


# ----------------------------------------------------------------------------
# Draft trees and masks
# ----------------------------------------------------------------------------

def chain_parents(q: int) -> list[int]:
    """A linear chain of drafts: draft i follows draft i-1."""
    return [-1] + list(range(q - 1))


def random_tree_parents(q: int, seed: int, tag: str, max_depth: int,
                        max_children: int | None = None) -> list[int]:
    """Random draft tree in topological order.

    Node 0 is the root at depth 0.  Node i > 0 takes its parent uniformly
    among the earlier nodes whose depth is below ``max_depth`` and that have
    fewer than ``max_children`` children, so every node has depth <=
    ``max_depth`` and branching <= ``max_children``.
    """
    u = uniform(seed, tag, max(q, 1))
    parent, depth, kids = [-1], [0], [0]
    for i in range(1, q):
        cand = [j for j in range(i)
                if depth[j] < max_depth and (max_children is None or kids[j] < max_children)]
        if not cand:
            raise ValueError("tree limits leave no parent for node %d" % i)
        p = cand[min(len(cand) - 1, int(u[i] * len(cand)))]
        parent.append(p)
        depth.append(depth[p] + 1)
        kids.append(0)
        kids[p] += 1
    return parent


def ancestor_mask(parents: list[int]) -> np.ndarray:
    """Bit-packed ancestors-or-self mask, shape [q, ceil(q/32)] uint32.

    Word w, bit k of row i (LSB first) is set iff draft 32*w+k is draft i or
    one of its ancestors.
    """
    q = len(parents)
    words = (q + 31) // 32
    m = np.zeros((q, words), dtype=np.uint32)
    for i in range(q):
        j = i
        while j >= 0:
            m[i, j >> 5] |= np.uint32(1 << (j & 31))
            j = parents[j]
    return m


def pack_mask(dense: np.ndarray) -> np.ndarray:
    """Pack a boolean [..., q, q] visibility matrix into [..., q, ceil(q/32)] uint32."""
    dense = np.asarray(dense, dtype=bool)
    q = dense.shape[-1]
    words = (q + 31) // 32
    out = np.zeros(dense.shape[:-1] + (words,), dtype=np.uint32)
    for j in range(q):
        out[..., j >> 5] |= (dense[..., j].astype(np.uint32) << np.uint32(j & 31))
    return out


def log_uniform_ints(seed: int, tag: str, n: int, lo: int, hi: int) -> np.ndarray:
    u = uniform(seed, tag, n)
    v = np.floor(np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).astype(np.int64)
    return np.clip(v, lo, hi)


# ----------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class Workload:
    """One verify-attention workload (sizes and draft-tree recipe)."""
    name: str
    B: int
    q: int
    prefix: int | tuple[int, int]          # fixed prefix, or (lo, hi) log-uniform per stream
    tree: str                              # "chain" or "random"
    max_depth: int = 5
    max_children: int | None = None
    H: int = H_DEFAULT
    Dl: int = DL
    Dr: int = DR
    index: int = 0

    @property
    def seed(self) -> int:
        return BASE_SEED + self.index


# The five shapes: a short chain, a mid-length tree, a wide 33-node tree over
# 16k, the long-context 64k case and ragged batched streams.
WORKLOADS = {
    "chain9_p256": Workload("chain9_p256", 1, 9, 256, "chain", index=1),
    "tree9_p4096": Workload("tree9_p4096", 1, 9, 4096, "random", 5, None, index=2),
    "tree33_p16384": Workload("tree33_p16384", 1, 33, 16384, "random", 8, 4, index=3),
    "tree9_p65536": Workload("tree9_p65536", 1, 9, 65536, "random", 5, None, index=4),
    "ragged8_tree9": Workload("ragged8_tree9", 8, 9, (1024, 32768), "random", 5, None, index=5),
}


@dataclass
class Case:
    """Concrete inputs of one call (host arrays, bf16 as uint16 bits)."""
    q_nope: np.ndarray        # [B, q, H, Dl] uint16
    q_rope: np.ndarray        # [B, q, H, Dr] uint16
    kv: np.ndarray            # [B, Smax, Dl+Dr] uint16
    seq_lens: np.ndarray      # [B] int32, prefix + q
    mask: np.ndarray          # [B, q, ceil(q/32)] uint32
    scale: np.float32
    parents: list = field(default_factory=list)

    @property
    def B(self):
        return self.q_nope.shape[0]

    @property
    def q(self):
        return self.q_nope.shape[1]

    @property
    def H(self):
        return self.q_nope.shape[2]

    @property
    def Smax(self):
        return self.kv.shape[1]


def round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


def default_scale() -> np.float32:
    """1/sqrt(192): the fp32 value handed to both the oracle and the kernels."""
    return np.float32(1.0 / math.sqrt(192.0))


def to_paged(case: "Case", page_size: int, seed: int, extra_pages: int = 3):
    """Lay a case's cache out as a page pool for the paged entry point.

    Each stream's keys 0 .. max_blocks*page_size-1 are cut into blocks of
    page_size rows and placed at pages given by a seeded random permutation of
    the pool (which has ``extra_pages`` pages no stream uses).  Rows of the
    logical cache past Smax, and unused pages, are NaN.  Returns
    (kv_pool [pool_rows, 576] uint16, block_table [B, max_blocks] int32).
    """
    B, Smax, D = case.kv.shape
    max_blocks = -(-Smax // page_size)
    pages = B * max_blocks + extra_pages
    order = np.argsort(uniform(seed, "pages", pages), kind="stable").astype(np.int32)
    table = order[: B * max_blocks].reshape(B, max_blocks)
    pool = np.full((pages * page_size, D), 0x7FC0, dtype=np.uint16)
    for b in range(B):
        for k in range(max_blocks):
            lo, hi = k * page_size, min((k + 1) * page_size, Smax)
            if lo < hi:
                dst = int(table[b, k]) * page_size
                pool[dst:dst + hi - lo] = case.kv[b, lo:hi]
    return pool, np.ascontiguousarray(table)


def scale_key_rope(case: "Case", b: int, key: int, factor: float) -> None:
    """Scale the rope part (the last Dr values) of one cache row in place.

    The key's score grows in every row whose q_pe agrees with its k_pe, so it
    dominates those rows' softmax while its value row (the latent part) keeps
    the distribution of the others: inputs on which a rounded weight of the
    dominant key shows in the output.
    """
    row = bf16_bits_to_f32(case.kv[b, key]).copy()
    row[-case.kv.shape[2] + 512:] *= np.float32(factor)
    case.kv[b, key] = f32_to_bf16_bits(row)


def make_case(w: Workload, seed: int | None = None, pad: str = "nan",
              smax_align: int = 64, prefixes=None) -> Case:
    """Materialise a workload.

    ``pad`` fills cache rows at or beyond each stream's length: ``"nan"`` (for
    tests: those rows must have no influence) or ``"normal"`` (for timing).
    """
    seed = w.seed if seed is None else seed
    B, q, H = w.B, w.q, w.H
    if prefixes is None:
        if isinstance(w.prefix, tuple):
            prefixes = log_uniform_ints(seed, "seqlens", B, *w.prefix)
        else:
            prefixes = np.full(B, w.prefix, dtype=np.int64)
    prefixes = np.asarray(prefixes, dtype=np.int64)
    seq = (prefixes + q).astype(np.int32)
    smax = round_up(int(seq.max()), smax_align)
    D = w.Dl + w.Dr
    q_nope = normal_bf16(seed, "q_nope", (B, q, H, w.Dl))
    q_rope = normal_bf16(seed, "q_rope", (B, q, H, w.Dr))
    kv = normal_bf16(seed, "kv", (B, smax, D))
    if pad == "nan":
        for b in range(B):
            kv[b, seq[b]:, :] = 0x7FC0
    elif pad != "normal":
        raise ValueError(pad)
    masks, parents = [], []
    for b in range(B):
        if w.tree == "chain":
            par = chain_parents(q)
        else:
            par = random_tree_parents(q, seed, "tree%d" % b, w.max_depth, w.max_children)
        parents.append(par)
        masks.append(ancestor_mask(par))
    return Case(q_nope, q_rope, kv, seq, np.stack(masks), default_scale(), parents)
