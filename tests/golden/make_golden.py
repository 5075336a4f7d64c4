"""Writes tiny_oracle.json: the fp64 oracle's output for the tiny workload
(B=2, H=16, q_len=1, seq_lens {37, 64}, page_size 32, seed 1001).

Calls only ``oracle/`` (inputs from ``mla_inputs``).  The pages print no worked
numeric example, so this file is a regression record of the oracle, not an
external pin; the external pins are the closed forms in test_oracle_pins.py.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import mla_inputs  # noqa: E402
import oracle  # noqa: E402


def main():
    w = mla_inputs.tiny()
    out, lse = oracle.run(w, n_threads=1)
    doc = {
        "workload": w.name, "seed": w.seed,
        "source": "oracle/oracle.c via tests/golden/make_golden.py",
        "lse": lse.tolist(),
        # dims 0, 1, 255, 511 of every (token, head)
        "out_dims": [0, 1, 255, 511],
        "out": out[..., [0, 1, 255, 511]].tolist(),
    }
    with open(os.path.join(HERE, "tiny_oracle.json"), "w") as f:
        json.dump(doc, f, indent=1)


if __name__ == "__main__":
    main()
