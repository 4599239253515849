"""Writes tests/golden/oracle_small_bf16.json: the oracle's outputs on a small
seeded bf16 workload, so that later changes to the oracle's arithmetic show up as
a diff. Calls only `oracle/` and the seeded input generator `synth/`.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

WL = synth.Workload("golden-small-bf16", B=1, T=24, d=16, n=8, dk=8, W=4, dtype="bf16",
                    seed=4242)


def compute():
    p = synth.make_params(WL)
    tok = synth.make_tokens(WL)
    out = oracle.prefill_sequence(tok["x"][0], p, tok["alpha"][0], tok["beta"][0], WL.W)
    return {
        "what": "oracle outputs of one small bf16 SDM sequence (regression fixture)",
        "cite": "written by tests/golden/make_golden.py from oracle/ only; workload "
                "golden-small-bf16 (B=1, T=24, d=16, n=8, dk=8, W=4, seed 4242)",
        "S": out["S"].tolist(), "R": out["R"].tolist(),
        "k": [[float.hex(float(a)) for a in row] for row in out["k"]],
        "y": [[float.hex(float(a)) for a in row] for row in out["y"]],
        "M_bits": np.asarray(out["M"]).astype(np.uint16).tolist(),
    }


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small_bf16.json")
    with open(path, "w") as f:
        json.dump(compute(), f)
    print("wrote", path)
