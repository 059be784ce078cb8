"""Writes tests/golden/oracle_small_case.json from the CPU oracle alone.

Inputs are drawn with numpy's PCG64 generator (platform independent) and
stored as 16-bit patterns; the expected output is the oracle's fp64 result.
The file is a regression fixture for the oracle (any change of its
arithmetic shows up), not an independent pin.  Run from the repository root:
    python tests/golden/make_golden.py
"""
import json
import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402


def main():
    rng = np.random.default_rng(2111)
    B, Hq, Hkv, D, NB, BS = 3, 4, 2, 8, 8, 16
    lens = np.array([5, 17, 40], np.int32)
    perm = rng.permutation(NB).astype(np.int32)
    tables = np.stack([perm[0:3], perm[3:6], np.r_[perm[6:8], perm[0]]]).astype(np.int32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float16).view(np.uint16)
    k = rng.standard_normal((NB, BS, Hkv, D)).astype(np.float16).view(np.uint16)
    v = rng.standard_normal((NB, BS, Hkv, D)).astype(np.float16).view(np.uint16)
    scale = 1.0 / math.sqrt(D)
    out = oracle.decode_attention(oracle.F16, q, k, v, tables, lens, scale)
    slots = oracle.slot_mapping(tables, lens, BS, NB)
    doc = {
        "_what": "oracle regression fixture written by tests/golden/make_golden.py (oracle only)",
        "dtype": "f16", "block_size": BS, "num_blocks": NB, "num_q_heads": Hq,
        "num_kv_heads": Hkv, "head_dim": D, "scale": scale,
        "context_lens": lens.tolist(), "block_tables": tables.tolist(),
        "q_bits": q.ravel().tolist(), "k_bits": k.ravel().tolist(), "v_bits": v.ravel().tolist(),
        "expected_out": [float(x).hex() for x in out.ravel()],
        "expected_slots": slots.tolist(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small_case.json")
    with open(path, "w") as f:
        json.dump(doc, f)
    print("wrote", path)


if __name__ == "__main__":
    main()
