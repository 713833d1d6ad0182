"""Write tests/golden/tiny_layer_oracle.txt from the CPU oracle.

Calls only `oracle/` and the seeded input generators. The stored values are
the oracle's outputs for the tiny layer (33 tokens, hidden 64, 8 experts,
top-2, intermediate 128, SwiGLU, packed w13, softmax over the selected
logits, seed 0), written as hex so that a later change to the oracle's
arithmetic or to the input generators shows up as a diff.

    python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import moe_inputs as I  # noqa: E402

OUT = os.path.join(HERE, "tiny_layer_oracle.txt")


def compute() -> dict:
    case = I.TINY
    d = I.layer_inputs(case)
    r = oracle.forward(d["x"], d["logits"], d["w13"], d["w2"], case.k, case.gating,
                       act=case.act, layout=case.layout)
    keys = ["topk_indx", "topk_vals", "col_sum", "offs", "col_sorted", "row_sorted",
            "gate_scal", "out"]
    return {key: np.asarray(r[key]) for key in keys}


def _fmt(a: np.ndarray) -> str:
    if a.dtype == np.uint16:
        return " ".join(f"{int(v):04x}" for v in a.ravel())
    return " ".join(str(int(v)) for v in a.ravel())


def main() -> None:
    vals = compute()
    with open(OUT, "w") as f:
        f.write("# Oracle outputs for the tiny layer (n=33, H=64, E=8, k=2, I=128, seed 0).\n")
        f.write("# Written by tests/golden/make_golden.py (calls only oracle/). bf16 as hex bits.\n")
        for key, a in vals.items():
            f.write(f"{key} {a.dtype.name} {' '.join(map(str, a.shape))}\n{_fmt(a)}\n")


def load() -> dict:
    out = {}
    with open(OUT) as f:
        lines = [ln.rstrip("\n") for ln in f if not ln.startswith("#")]
    for head, body in zip(lines[0::2], lines[1::2]):
        key, dtype, *shape = head.split()
        shape = tuple(int(s) for s in shape)
        if dtype == "uint16":
            a = np.array([int(v, 16) for v in body.split()], dtype=np.uint16)
        else:
            a = np.array([int(v) for v in body.split()], dtype=dtype)
        out[key] = a.reshape(shape)
    return out


if __name__ == "__main__":
    main()
    print(OUT)
