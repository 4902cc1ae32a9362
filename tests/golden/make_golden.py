"""Writes tests/golden/oracle_tiny.json: a regression record of the oracle on the tiny
workload (T=256, H=512, I=256, E=8, top-2, the seeded inputs of synth).  It calls only
oracle/ and synth/.  Rerun it (python tests/golden/make_golden.py) only when the oracle's
arithmetic changes on purpose, and say in the commit which reading of the method the
change follows."""
import hashlib
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402


def record() -> dict:
    synth.build_host()
    oracle.build()
    wl = synth.WORKLOADS["tiny"]
    h = synth.host_inputs(wl)
    ref = oracle.forward(h["x"], h["Wr"], None, h["W1"], h["W2"], wl.k)
    sha = lambda a: hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()  # noqa: E731
    return {
        "workload": "tiny: T=256 H=512 I=256 E=8 top-2, seed 0",
        "logits_sha256": sha(ref["logits"].view(np.uint32)),
        "ids_sha256": sha(ref["ids"].astype(np.int32)),
        "w_sha256": sha(ref["w"].view(np.uint32)),
        "counts": [int(c) for c in ref["counts"]],
        "y_sha256": sha(ref["y"].astype(np.uint16)),
        "ids_first_tokens": ref["ids"][:4].astype(int).tolist(),
        "y_first_row_bits": [int(b) for b in ref["y"][0, :8]],
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as f:
        json.dump(record(), f, indent=1)
        f.write("\n")
