"""Writes flint_stack_bias.txt: the selection bias of the 47-layer Flint stack
workload. A constant beta is added to the routing keys of experts 0..25 (10 % of
256) so that they take 50 % (+-1 %) of the top-6 picks; beta is found by
bisection on 4096 calibration tokens (bf16 N(0, 1), generator seed 1000,
layer index 999, which no stack layer uses) routed by the layer-0 router of the
stack (seed 1000, layer 0) with the oracle's routing. Calls only the oracle and
the input generator. Run from the repository root:
python tests/golden/make_stack_bias.py
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))

import synth  # noqa: E402
from oracle import moe  # noqa: E402

CFG = moe.Config(hidden=2048, num_experts=256, top_k=6, inter=512, n_shared=1)
SEED, CAL_LAYER, N_CAL, N_BIASED, TARGET = 1000, 999, 4096, 26, 0.5
PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "flint_stack_bias.txt")


def calibration_inputs():
    x = moe.bf16_bits_to_f64(synth.x_bf16(SEED, CAL_LAYER, N_CAL, CFG.hidden))
    router = moe.bf16_bits_to_f64(synth.router_bf16(SEED, 0, CFG.num_experts, CFG.hidden))
    return x, router


def bias_vector(beta: float) -> np.ndarray:
    b = np.zeros(CFG.num_experts, np.float32)
    b[:N_BIASED] = np.float32(beta)
    return b


def biased_fraction(x, router, beta: float) -> float:
    r = moe.route(x, router, CFG, bias_vector(beta))
    return float(np.mean(r.idx < N_BIASED))


def read_beta(path: str = PATH) -> float:
    with open(path) as f:
        for line in f:
            if line.startswith("beta_f32_hex "):
                return float(np.frombuffer(bytes.fromhex(line.split()[1])[::-1], np.float32)[0])
    raise ValueError("no beta in " + path)


def main():
    x, router = calibration_inputs()
    lo, hi = 0.0, 1.0
    beta, frac = 0.5, biased_fraction(x, router, 0.5)
    for _ in range(30):
        if abs(frac - TARGET) <= 0.002:
            break
        if frac < TARGET:
            lo = beta
        else:
            hi = beta
        beta = float(np.float32((lo + hi) / 2))
        frac = biased_fraction(x, router, beta)
    with open(PATH, "w") as f:
        f.write("# Selection bias of the 47-layer Flint stack workload (see make_stack_bias.py): added to\n")
        f.write("# the routing keys of experts 0..25 so that they take about half of the top-6 picks.\n")
        f.write("# A workload parameter calibrated with the oracle, not a value printed on the pages.\n")
        f.write("biased_experts %d\n" % N_BIASED)
        f.write("beta %r\n" % beta)
        f.write("beta_f32_hex %s\n" % np.float32(beta).tobytes()[::-1].hex())
        f.write("calibration_fraction %.6f\n" % frac)


if __name__ == "__main__":
    main()
