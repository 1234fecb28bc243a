"""Writes the stored expected values under tests/golden/ from the CPU oracle alone.

Run from the repository root:  python tests/golden/make_golden.py
Each fixture holds, for one seeded workload of ``wq4_inputs``, sampled fp64 outputs of the oracle
with the row sums of |Y| (compared to 1e-12 relative: BLAS summation order may differ between
hosts), plus the SHA-256 of the prepacked blob the oracle builds for the same weight (integer
work, compared bit for bit).
"""
import hashlib
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
import wq4_inputs as I  # noqa: E402

CASES = {
    "tiny_m16_n256_k512_fp16_u4b8": dict(M=16, N=256, K=512, dtype="fp16", qtype="u4b8", seed=1001),
    "small_m5_n384_k256_bf16_u4zp": dict(M=5, N=384, K=256, dtype="bf16", qtype="u4_zp", seed=77),
    "small_m7_n256_k512_fp16_u4fzp": dict(M=7, N=256, K=512, dtype="fp16", qtype="u4_fzp", seed=91),
    "small_m6_n128_k384_bf16_u4zp_g64": dict(M=6, N=128, K=384, dtype="bf16", qtype="u4_zp", seed=64, group_size=64),
}
SAMPLES = [(0, 0), (1, 5), (3, 127), (4, 255), (2, 200), (15, 31), (9, 130), (4, 383)]


def golden(spec):
    p = I.make_problem(**spec)
    Y = O.mm_problem(p)
    blob = O.prepack(p.Wq, p.S_bits, p.N, p.K, p.dtype, p.qtype, p.Z, group_size=p.group_size)
    return {
        "spec": spec,
        "y_row_abs_sums": [float(v).hex() for v in np.abs(Y).sum(axis=1)],
        "y_samples": [[m, n, float(Y[m, n]).hex()] for m, n in SAMPLES if m < p.M and n < p.N],
        "blob_sha256": hashlib.sha256(blob.tobytes()).hexdigest(),
        "blob_bytes": int(blob.size),
    }


if __name__ == "__main__":
    here = os.path.dirname(os.path.abspath(__file__))
    for name, spec in CASES.items():
        with open(os.path.join(here, name + ".json"), "w") as f:
            json.dump(golden(spec), f, indent=1)
            f.write("\n")
        print("wrote", name)
