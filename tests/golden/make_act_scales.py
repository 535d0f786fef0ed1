"""Write the calibrated static activation-scale tables used by the GPU parity tests
([L][4]; [L][7] for the FP8-attention workload, columns 4-6 = Q, K, V).

Calls only the CPU oracle (oracle.model.calibrate): one calibration decision
with noise draw 1000 and the workload's prefix, starting from the data-independent
table in fm_synth, per layer and quant point amax over all steps / 448.
Run: python tests/golden/make_act_scales.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import fm_synth  # noqa: E402
from oracle import model as O  # noqa: E402


def main(names=("layer_fp8_m10", "expert_fp8_m50", "expert_fp8attn_m50", "wam_nvfp4_m256")):
    for name in names:
        cfg = fm_synth.config(name)
        layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
        conds = fm_synth.step_conds(cfg) if cfg.cond == "given" else None
        model = O.Model(cfg, layers, fm_synth.final_weights(cfg), conds)
        kp, vp = fm_synth.prefix_kv(cfg)
        if cfg.cond == "given":
            # single-layer workload: calibrate on the layer input itself
            amax = np.zeros((cfg.L, 4))
            x = fm_synth.layer_input(cfg)
            q = O.pre_attn_quant(model, 0, 0, x, fm_synth.default_act_scales(cfg), amax)
            O.layer_forward(model, 0, 0, x, q, kp, vp, fm_synth.default_act_scales(cfg), amax)
            sc = (amax.astype(np.float32) / np.float32(448)).astype(np.float32)
            how = "oracle calibration on the single-layer input"
        else:
            sc = O.calibrate(model, fm_synth.noise(cfg, 1000), kp, vp, fm_synth.default_act_scales(cfg))
            how = "oracle calibration decision, noise draw 1000"
        path = os.path.join(HERE, f"act_scales_{name}.txt")
        with open(path, "w") as f:
            f.write(f"# static activation scales [L][{sc.shape[1]}] for {name}: {how}\n")
            for row in sc:
                f.write(" ".join(f"{float(v):.9e}" for v in row) + "\n")
        print(path)


if __name__ == "__main__":
    main(sys.argv[1:] or ("layer_fp8_m10", "expert_fp8_m50", "expert_fp8attn_m50", "wam_nvfp4_m256"))
