"""Derive the end-to-end tolerance of the 18-layer x 10-step FP8 decision from the
oracle alone, and write it to fp8_envelope_expert_fp8_m50.txt.

The FP8 decision requantises 4 activations per layer-step (720 times per
decision); a value landing within rounding distance of an E4M3 tie can round
either way, and one flipped code moves every later activation. The envelope is
the largest action difference between the oracle and the same oracle whose
pre-quantisation values are first rounded to fp32 (a perturbation of at most
2^-24 relative, i.e. what any fp32 implementation of the same arithmetic may
differ by), relative to RMS(actions). Uses the calibrated scales and noise draw 0.
Run: python tests/golden/make_fp8_envelope.py [workload ...]
(default: expert_fp8_m50 and expert_fp8attn_m50, the same expert with FP8 attention,
and expert_fp8_m50_warm: the one-step warm start of that expert at warm_t = 0.5 from
the oracle's decision on noise draw 0, 3 actions executed, fresh noise draw 1).
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import fm_synth  # noqa: E402
from oracle import codecs as C  # noqa: E402
from oracle import model as O  # noqa: E402


WARM = {"expert_fp8_m50_warm": ("expert_fp8_m50", 0.5, 3)}   # base workload, warm_t, executed


def main(name="expert_fp8_m50"):
    base, warm_t, executed = WARM.get(name, (name, 0.0, 0))
    cfg = fm_synth.config(base, warm_t=warm_t)
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    model = O.Model(cfg, layers, fm_synth.final_weights(cfg))
    kp, vp = fm_synth.prefix_kv(cfg)
    sc = np.loadtxt(os.path.join(HERE, f"act_scales_{base}.txt"), dtype=np.float32, ndmin=2)
    nz = fm_synth.noise(cfg, 0)
    if warm_t > 0:
        prev = O.decode(model, nz, kp, vp, sc)
        nz1 = fm_synth.noise(cfg, 1)
        run = lambda: O.decode_warm(model, nz1, prev, executed, kp, vp, sc)
    else:
        run = lambda: O.decode(model, nz, kp, vp, sc)
    ref = run()
    plain = O.quant_codes

    def quant_fp32_input(h, s, fmt):   # the same quantiser, fed an fp32-rounded value
        if fmt == "fp8":
            return C.e4m3(C.fp32(C.fp32(h) * O.recip32(s)))
        return plain(h, s, fmt)

    O.quant_codes = quant_fp32_input
    try:
        alt = run()
    finally:
        O.quant_codes = plain
    env = float(np.max(np.abs(alt - ref)) / np.sqrt(np.mean(ref ** 2)))
    path = os.path.join(HERE, f"fp8_envelope_{name}.txt")
    with open(path, "w") as f:
        what = (f"warm start (warm_t {warm_t}, {executed} executed, noise draw 1) from the decision on noise draw 0"
                if warm_t > 0 else "noise draw 0")
        f.write(f"# max|oracle(fp32-rounded pre-quant) - oracle| / RMS(oracle actions), {what}\n")
        f.write(f"{env:.6e}\n")
    print(path, env)


if __name__ == "__main__":
    for name in sys.argv[1:] or ("expert_fp8_m50", "expert_fp8attn_m50", "expert_fp8_m50_warm"):
        main(name)
