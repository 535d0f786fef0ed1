"""Full-size world-action-model decisions pinned on sampled layer-steps.

The 28-layer x 10-step decoder (d = 2048, 16 x 128 heads over 2 KV heads, F = 8192,
M = 256 rows, prefix 1024) with NVFP4 weights, with FP8 activations (W4A8) and with
four-bit activations (W4A4), runs traced as one whole decision at its full size; the
traced actions equal the graph decision's bitwise (so the checked kernels are the
decision's), and layer-steps at the start, the middle and the end of the decision
(the last with the final step's Euler update) are checked stage by stage against the
oracle applied to their own recorded inputs. Only the sampled records leave the
device, and the oracle is prepared for the sampled layers alone; the whole decision
at this size is too slow for the CPU oracle end to end (about a minute per decision).
"""
import dataclasses

import numpy as np
import pytest
import torch

import fm_synth
import flow_matching_action_denoise_gb300 as fmad
from oracle import model as O

from _gpu import dev, read_trace_records, require_gpu
from _stagewise import check_close, check_increment, check_layer_stages, check_step_end

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["wam_nvfp4_m256", "wam_w4a4_m256"])
def test_full_decision_sampled_layer_steps(name):
    device = require_gpu()
    cfg = fm_synth.config(name)
    L, S = cfg.L, cfg.S
    samples = [(0, 0), (S // 2, L // 2), (S - 1, L - 1)]
    final = fm_synth.final_weights(cfg)
    kp, vp = fm_synth.prefix_kv(cfg)
    scales = fm_synth.default_act_scales(cfg)
    layers = [fm_synth.layer_weights(cfg, l) for l in range(L)]
    weights = fmad.DeviceWeights(cfg, layers, final, device=device)
    kept = {l: layers[l] for _, l in samples}
    del layers
    pol = fmad.Policy(cfg, act_scales=scales, weights=weights)
    pol.set_prefix_kv(dev(kp, device, torch.bfloat16), dev(vp, device, torch.bfloat16))
    assert fmad.kernel_count(pol.handle) == (8, 1 + L * S * 8)
    # 16 row tiles x 2 KV heads of 1280 keys: 7-CTA clusters take three waves of 152
    # SMs, the wide slice's 5-CTA clusters two
    assert fmad.attn_plan(pol.handle) == (256, 5)
    nbytes = fmad.trace_size(pol.handle)
    trace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    nz = fm_synth.noise(cfg, 0)
    act = torch.empty((cfg.M, cfg.A), dtype=torch.float32, device=device)
    fmad.decode_trace(pol.handle, dev(nz, device), act, trace, nbytes)
    assert fmad.device_status(pol.handle) == 0
    assert torch.equal(act.cpu(), pol.decode(dev(nz, device)).cpu())
    recs = read_trace_records(trace, cfg, pol, samples + [(S - 2, L - 1)])
    del trace
    pol.close()
    del weights
    torch.cuda.empty_cache()

    check_close(recs[(0, 0)]["x_in"], np.asarray(nz, np.float64) @ np.asarray(final["w_in"], np.float64).T +
                np.asarray(final["b_in"], np.float64), f"{name} step head x")
    one = dataclasses.replace(cfg, L=1)
    for k, l in samples:
        model = O.Model(one, [kept[l]], final)   # layer l's weights and modulation alone
        r = recs[(k, l)]
        where = f"{name} step {k} layer {l}"
        inc, x_res = check_layer_stages(cfg, model.w[0], model.mods[k][0][0], r, scales[l],
                                        np.asarray(kp[l], np.float64), np.asarray(vp[l], np.float64), None, where)
        if l < L - 1:
            check_increment(r["x_out"], r["x_mid"], inc, where + " down GEMM + MLP residual")
        else:
            a_prev = recs[(k - 1, L - 1)]["actions"].astype(np.float64)
            check_step_end(model, k, r, x_res, a_prev, -1.0 / S, k < S - 1, where)
    np.testing.assert_array_equal(recs[(S - 1, L - 1)]["actions"], act.cpu().numpy())
