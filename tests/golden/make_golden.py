"""Write tests/golden/oracle_tiny.txt: fp64 oracle outputs for a tiny seeded case.

Calls only the oracle and the seeded input generators.  The stored values pin
the oracle against silent drift; its correctness pins are in tests/test_oracle.py.
Run:  python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402
import torch  # noqa: E402

import fa_inputs  # noqa: E402
import oracle  # noqa: E402

CASES = [
    # name, B, Hq, Hkv, Sq, Sk, D, causal, dtype, scale, seed
    ("gqa_causal_bottom_right", 1, 4, 2, 5, 9, 8, True, torch.bfloat16, 0.35, 7),
    ("mha_noncausal_fp16", 2, 2, 2, 3, 6, 8, False, torch.float16, 0.5, 11),
]


def main():
    lines = ["# fp64 oracle outputs, written by tests/golden/make_golden.py"]
    for name, B, Hq, Hkv, Sq, Sk, D, causal, dt, scale, seed in CASES:
        q, k, v = fa_inputs.prefill_inputs(B, Hq, Hkv, Sq, Sk, D, dt, seed)
        o = oracle.attention(q, k, v, scale, causal)
        dts = "bf16" if dt == torch.bfloat16 else "fp16"
        lines.append(f"case {name} {B} {Hq} {Hkv} {Sq} {Sk} {D} {int(causal)} {dts} "
                     f"{scale!r} {seed}")
        lines.append(" ".join(f"{x:.17g}" for x in o.ravel()))
    with open(os.path.join(HERE, "oracle_tiny.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
