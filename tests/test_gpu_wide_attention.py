"""The wide attention slice on its other input path: with FP8 weights the QKV GEMM
writes no transposed copy of the chunk's values, so the slice holding the chunk
gathers them from the QKV output itself. The world-action-model shape (16 row tiles x
2 KV heads, 1280 keys) takes the wide slice (asserted through the policy's plan); a
one-layer, one-step decision is then checked stage by stage against the oracle, and
graph == the traced run bitwise. (The attention is bf16 whatever the weights; BF16
weights at this width are not used: their K = 2048 gate|up GEMM rounds 2.5e-3 of the
GeGLU's bf16 codes across a tie, beyond the stage checker's 1e-3, derived for K = 1024.)"""
import dataclasses

import numpy as np
import pytest
import torch

import fm_synth
import flow_matching_action_denoise_gb300 as fmad
from oracle import model as O

from _gpu import dev, parse_trace, require_gpu
from _stagewise import check_decision_stages

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt", ["fp8"])
def test_wide_slice_gathers_chunk_values(fmt):
    device = require_gpu()
    cfg = dataclasses.replace(fm_synth.config("wam_nvfp4_m256"), L=1, S=1, weight_fmt=fmt, act_fmt=fmt)
    layers = [fm_synth.layer_weights(cfg, 0)]
    final = fm_synth.final_weights(cfg)
    kp, vp = fm_synth.prefix_kv(cfg)
    scales = fm_synth.default_act_scales(cfg) if fmt == "fp8" else None
    pol = fmad.Policy(cfg, layers, final, act_scales=scales, device=device)
    pol.set_prefix_kv(dev(kp, device, torch.bfloat16), dev(vp, device, torch.bfloat16))
    assert fmad.attn_plan(pol.handle) == (256, 5)
    nbytes = fmad.trace_size(pol.handle)
    trace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    nz = fm_synth.noise(cfg, 0)
    act = torch.empty((cfg.M, cfg.A), dtype=torch.float32, device=device)
    fmad.decode_trace(pol.handle, dev(nz, device), act, trace, nbytes)
    assert fmad.device_status(pol.handle) == 0
    assert torch.equal(act.cpu(), pol.decode(dev(nz, device)).cpu())
    recs = parse_trace(trace.cpu().numpy(), cfg, pol)
    pol.close()
    last = check_decision_stages(cfg, O.Model(cfg, layers, final), recs, nz, kp, vp, scales)
    np.testing.assert_array_equal(last, act.cpu().numpy())
