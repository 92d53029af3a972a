"""Writes oracle_small.json: a small seeded verify-attention case and the
oracle's out/lse for it.  Calls only the oracle (and the seeded generator for
the inputs).  Run: python tests/golden/make_golden.py"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from mla_verify_attention_gb300 import inputs as I  # noqa: E402


def main():
    seed, B, q, H, Dl, Dr = 99, 2, 3, 2, 8, 4
    prefixes = np.array([4, 1])
    seq = (prefixes + q).astype(np.int32)
    smax = int(seq.max()) + 2
    qn = I.normal_bf16(seed, "qn", (B, q, H, Dl))
    qr = I.normal_bf16(seed, "qr", (B, q, H, Dr))
    kv = I.normal_bf16(seed, "kv", (B, smax, Dl + Dr))
    mask = np.stack([I.ancestor_mask(I.random_tree_parents(q, seed, "t%d" % b, 2)) for b in range(B)])
    scale = float(np.float32(0.25))
    out, lse = oracle.verify_attn(qn, qr, kv, seq, mask, np.float32(scale))
    arrs = {"q_nope": qn, "q_rope": qr, "kv": kv, "seq_lens": seq, "mask": mask}
    g = {
        "what": "oracle out/lse on a small seeded case (regression fixture)",
        "scale": scale,
        "inputs": {k: v.reshape(-1).tolist() for k, v in arrs.items()},
        "shapes": {k: list(v.shape) for k, v in arrs.items()},
        "dtypes": {k: str(v.dtype) for k, v in arrs.items()},
        "out": out.reshape(-1).tolist(),
        "lse": lse.reshape(-1).tolist(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.json")
    with open(path, "w") as fh:
        json.dump(g, fh)
    print("wrote", path)


if __name__ == "__main__":
    main()
