"""Write tests/golden/tiny_oracle.json: the tiny workload's inputs and the
CPU oracle's outputs for them.

The sampler's pages print no worked example, so this file is not a pin taken
from the pages: it is a regression anchor that records what the (pinned)
oracle computes, so that any later change to the oracle's arithmetic shows up
as a diff.  It calls only oracle/ and the seeded workload generators.
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from logits_sampling_gb300 import workloads as W  # noqa: E402


def main():
    w = W.make_tiny()
    r = oracle.sample(w.logits, oracle.DTYPE_F32, w.n, w.temperature, w.top_k, w.top_p, w.seed, step=0,
                      want_lp=True)
    out = {
        "source": "CPU oracle on the tiny workload (4 x 1000 fp32 ~ N(0, 2), seed 0; T=1, top_k=50, "
                  "top_p=0.9, Philox seed of row r = r, step 0)",
        "logits_hex": [[float(v).hex() for v in row] for row in w.logits],
        "temperature": w.temperature.tolist(), "top_k": w.top_k.tolist(), "top_p": w.top_p.tolist(),
        "seed": [int(s) for s in w.seed], "step": 0,
        "ids": r["ids"].tolist(), "flags": r["flags"].tolist(),
        "kept": [np.nonzero(k)[0].tolist() for k in r["kept"]],
        "log_probs_kept_hex": [[float(v).hex() for v in r["lp"][i][r["kept"][i]]] for i in range(w.n)],
    }
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as f:
        json.dump(out, f, indent=0)


if __name__ == "__main__":
    main()
