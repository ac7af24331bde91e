"""Writes the stored oracle outputs under tests/golden/.

The method's pages print no worked numerical example, so the stored values
here are the oracle's own outputs on the small seeded workloads, kept to
catch any later drift of the oracle (and any difference between the x86
build host and the Arm GPU host).  This script calls only ``oracle/`` and the
input generator.  Run from the repository root:

    python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth_inputs as si  # noqa: E402


def tiny_case():
    c = si.CONFIGS["tiny"]
    d = si.make_projection(c)
    _, out = oracle.Oracle().rmsnorm_linear(d["x"], d["gamma"], d["W"], c["eps"], c["norm_mode"], 0)
    return out


def small_w8a8_case():
    c = si.scaled(si.CONFIGS["w8a8"], T=8, K=256, N=64)
    d = si.make_w8a8(c)
    r = oracle.Oracle().rmsnorm_linear_w8a8(d["x"], d["gamma"], d["Wq"], d["w_scale"], c["eps"],
                                            c["norm_mode"])
    return r


def digest(a: np.ndarray) -> str:
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def main():
    out = tiny_case()
    with open(os.path.join(HERE, "tiny_rmsnorm_linear_bf16.txt"), "w") as f:
        f.write("# oracle output of the tiny workload (x[16,256], W[128,256]), bf16 bits, row-major\n")
        for row in out:
            f.write(" ".join("%04x" % int(v) for v in row) + "\n")
    r = small_w8a8_case()
    meta = {"q_sha256": digest(r["q"]), "acc_sha256": digest(r["acc"]),
            "out_sha256": digest(r["out"]), "x_scale": [float(v) for v in r["x_scale"]]}
    with open(os.path.join(HERE, "w8a8_T8_K256_N64.json"), "w") as f:
        json.dump(meta, f, indent=1)


if __name__ == "__main__":
    main()
