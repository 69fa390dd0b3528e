"""Write tiny_oracle_regression.txt and tiny_ffn_oracle_regression.txt from
the float64 oracle (oracle/ only).

Inputs: the tiny workload (hidden 256, 4x64 MHA, batch 1, position 128,
float32 storage) and the tiny FFN workload (hidden 256, intermediate 688,
batch 1, float32 storage), each drawn on the CPU with seed 0 by the shared
input module.
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from attention_block_gb300 import synth  # noqa: E402


def compute():
    w = synth.WORKLOADS[synth.TINY]
    t = synth.make_layer(w, seed=0, device="cpu")
    f = {k: synth.to_f64(v) for k, v in t.items() if k != "positions"}
    pos = t["positions"].numpy()
    r = oracle.decode(w.oracle_cfg(), f["hidden"], f["ln_weight"], f["w_qkv"], f["w_o"],
                      f["k_cache"], f["v_cache"], pos)
    return r


def compute_ffn():
    w = synth.FFN_WORKLOADS[synth.TINY_FFN]
    t = synth.make_ffn(w, seed=0, device="cpu")
    f = {k: synth.to_f64(v) for k, v in t.items()}
    return oracle.ffn(f["hidden"], f["ln_weight"], f["w_gate"], f["w_up"], f["w_down"],
                      w.rms_eps)


if __name__ == "__main__":
    r = compute()
    path = os.path.join(HERE, "tiny_oracle_regression.txt")
    with open(path, "w") as fh:
        fh.write("# oracle output for the tiny workload, seed 0 (see README.md)\n")
        for key in ("out", "o"):
            fh.write(key + " " + " ".join(repr(float(v)) for v in r[key][0]) + "\n")
    print("wrote", path)
    rf = compute_ffn()
    path = os.path.join(HERE, "tiny_ffn_oracle_regression.txt")
    with open(path, "w") as fh:
        fh.write("# FFN oracle output for the tiny FFN workload, seed 0 (see README.md)\n")
        fh.write("out " + " ".join(repr(float(v)) for v in rf["out"][0]) + "\n")
    print("wrote", path)
