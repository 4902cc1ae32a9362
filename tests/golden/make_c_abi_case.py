"""Writes the inputs and the oracle's expectations of the tiny workload (T=256, H=512, I=256,
E=8, top-2, the seeded inputs of synth) as raw little-endian binary files for the plain-C GPU
caller tests/c_abi_gpu.c.  It calls only oracle/ and synth/.

    python tests/golden/make_c_abi_case.py DIR

Files: x, Wr, W1, W2 (bf16 bit patterns, uint16), ids (int32 [T,k]), y (bf16 bits [T,H], the
oracle's output), ylo, yhi (float64 [T,H], the interval of y before rounding that the oracle's
flagged intermediates allow; see oracle.forward(bounds=True)), and shape.txt (T H I E k)."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402


def write_case(out_dir: str) -> dict:
    synth.build_host()
    oracle.build()
    wl = synth.WORKLOADS["tiny"]
    h = synth.host_inputs(wl)
    ref = oracle.forward(h["x"], h["Wr"], None, h["W1"], h["W2"], wl.k, bounds=True)
    os.makedirs(out_dir, exist_ok=True)
    arrays = {"x": h["x"], "Wr": h["Wr"], "W1": h["W1"], "W2": h["W2"],
              "ids": ref["ids"].astype(np.int32), "y": ref["y"].astype(np.uint16),
              "ylo": ref["ylo"].astype(np.float64), "yhi": ref["yhi"].astype(np.float64)}
    for name, a in arrays.items():
        np.ascontiguousarray(a).astype(a.dtype.newbyteorder("<")).tofile(os.path.join(out_dir, name + ".bin"))
    with open(os.path.join(out_dir, "shape.txt"), "w") as f:
        f.write(f"{wl.T} {wl.H} {wl.I} {wl.E} {wl.k}\n")
    return {"T": wl.T, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k}


if __name__ == "__main__":
    print(write_case(sys.argv[1] if len(sys.argv) > 1 else os.path.join(HERE, "c_abi_case")))
