"""Writes tiny_layer_seed0.txt: the oracle's decode of the tiny layer
(hidden 256, 16 experts, sigmoid top-2 + 1 shared expert, intermediate 64,
batch 1, seed 0; NVFP4 weights N(0, 0.02) quantised per 16-element block,
router bf16 N(0, 0.02), x bf16 N(0, 1)). Calls only the oracle and the input
generator. Run from the repository root: python tests/golden/make_tiny_golden.py
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))

import synth  # noqa: E402
from oracle import moe, nvfp4  # noqa: E402

CFG = moe.Config(hidden=256, num_experts=16, top_k=2, inter=64, n_shared=1)


def tiny_inputs(seed=0, B=1):
    x = moe.bf16_bits_to_f64(synth.x_bf16(seed, 0, B, CFG.hidden))
    router = moe.bf16_bits_to_f64(synth.router_bf16(seed, 0, CFG.num_experts, CFG.hidden))

    def get(e):
        mats = synth.expert_f32(seed, 0, e, CFG.hidden, CFG.inter)
        return tuple(moe.NVFP4Matrix(*nvfp4.quantize(m)) for m in mats)
    return x, router, get


def main():
    x, router, get = tiny_inputs()
    out, r = moe.moe_layer(x, router, get, CFG)
    bits = moe.f64_to_bf16_bits(out[0])
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_layer_seed0.txt")
    with open(path, "w") as f:
        f.write("# Oracle decode of the tiny MoE layer, batch 1, seed 0 (see make_tiny_golden.py).\n")
        f.write("# A regression record of the oracle, not a value printed on the pages.\n")
        f.write("idx " + " ".join(str(int(i)) for i in r.idx[0]) + "\n")
        f.write("w " + " ".join(repr(float(v)) for v in r.w[0]) + "\n")
        f.write("out_bf16_hex " + " ".join("%04x" % int(b) for b in bits) + "\n")


if __name__ == "__main__":
    main()
