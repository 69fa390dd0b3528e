"""Write tiny_oracle_regression.txt, tiny_ffn_oracle_regression.txt and
tiny_mla_oracle_regression.txt from the float64 oracle (oracle/ only).

Inputs: the tiny workload (hidden 256, 4x64 MHA, batch 1, position 128,
float32 storage), the tiny FFN workload (hidden 256, intermediate 688,
batch 1, float32 storage) and the tiny MLA workload (hidden 512, 8 heads of
128 + 64 query/key and 128 value dims, latent 512, batch 1, position 128,
bf16 storage), each drawn on the CPU with seed 0 by the shared input module.
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


def compute_mla():
    w = synth.MLA_WORKLOADS[synth.MLA_TINY]
    t = synth.make_mla_layer(w, seed=0, device="cpu")
    f = {k: synth.to_f64(v) for k, v in t.items() if k != "positions"}
    lc = f["latent_cache"][0].copy()
    return oracle.mla_row(w.oracle_cfg(), f["hidden"][0], f["ln_weight"], f["w_q"], f["w_dkv"],
                          f["kv_norm_weight"], f["w_ukv"], f["w_o"], lc, int(t["positions"][0]))


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
    rm = compute_mla()
    path = os.path.join(HERE, "tiny_mla_oracle_regression.txt")
    with open(path, "w") as fh:
        fh.write("# MLA oracle output for the tiny MLA workload, seed 0 (see README.md)\n")
        for key in ("out", "o"):
            fh.write(key + " " + " ".join(repr(float(v)) for v in rm[key]) + "\n")
    print("wrote", path)
