"""Derive the end-to-end tolerance of the matched 16-bit decision (bf16 weights and
activations, M = 63, 18 layers x 10 steps, prefix 788) from the oracle alone and
write it to bf16_envelope_expert_bf16_m63.txt, one line per checked decision.

The bf16 decision rounds every GEMM input, the attention operands and the
attention probabilities to bf16 (thousands of values per layer-step); a value
within fp32 rounding distance of a bf16 tie can round either way in any fp32
implementation, and each flip propagates through the remaining layers and steps.
The envelope is the largest action difference between the oracle and the same
oracle whose bf16 roundings are fed the fp32-rounded value (a perturbation of at
most 2^-24 relative), relative to RMS(actions).

Decision d uses noise draw d and the prefix whose 768 image-token rows come from
refresh version d // 5 (version 0 = the initial prefix), as in the persistence run.
Run: python tests/golden/make_bf16_envelope.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import fm_synth  # noqa: E402
from oracle import codecs as C  # noqa: E402
from oracle import model as O  # noqa: E402

NAME = "expert_bf16_m63"
DECISIONS = (0, 4, 5, 6, 50, 99)
IMAGE_ROWS, REFRESH_EVERY = 768, 5


def prefix_at(cfg, kp, vp, decision):
    k, v = kp.copy(), vp.copy()
    version = decision // REFRESH_EVERY
    if version > 0:
        k[:, :IMAGE_ROWS], v[:, :IMAGE_ROWS] = fm_synth.prefix_kv_rows(cfg, version, IMAGE_ROWS)
    return k, v


def main():
    cfg = fm_synth.config(NAME)
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    model = O.Model(cfg, layers, fm_synth.final_weights(cfg))
    kp, vp = fm_synth.prefix_kv(cfg)
    plain = C.bf16
    rows = []
    for d in DECISIONS:
        k, v = prefix_at(cfg, kp, vp, d)
        nz = fm_synth.noise(cfg, d)
        ref = O.decode(model, nz, k, v, None)
        C.bf16 = lambda x: plain(C.fp32(x))
        try:
            alt = O.decode(model, nz, k, v, None)
        finally:
            C.bf16 = plain
        env = float(np.max(np.abs(alt - ref)) / np.sqrt(np.mean(ref ** 2)))
        rows.append((d, env))
        print(d, env, flush=True)
    path = os.path.join(HERE, f"bf16_envelope_{NAME}.txt")
    with open(path, "w") as f:
        f.write("# decision  max|oracle(fp32-rounded bf16 inputs) - oracle| / RMS(oracle actions)\n")
        for d, env in rows:
            f.write(f"{d} {env:.6e}\n")
    print(path)


if __name__ == "__main__":
    main()
