"""One-step warm start on the GPU (the 18-layer FP8 expert, M = 50).

- warm_t = 1: the warm decision equals, bitwise, the full decision of a one-step
  policy on the same noise (the previous chunk and the executed count drop out);
- without a previous chunk (episode start, after fm_episode_reset) the warm call
  runs the full S-step decision, bitwise equal to decode_actions;
- warm_t = 0.5, 3 actions executed: within twice the oracle's own FP8 envelope of
  the oracle's warm decision from the GPU's previous chunk (teacher forced);
- teacher forced stage by stage (fm_decode_warm_trace), for 0, 3 and M executed
  actions: the mixed input a_tau (shift, pad with the last action, mix with the
  noise) equals the oracle's within fp32 rounding, and every kernel of the single
  Euler step matches the oracle's stage applied to its recorded input;
- the warm decision takes a fraction of the full decision's time.
"""
import dataclasses
import os

import numpy as np
import pytest
import torch

import fm_synth
import flow_matching_action_denoise_gb300 as fmad
from oracle import model as O

from _gpu import GOLDEN, dev, load_scales, parse_trace, require_gpu
from _stagewise import check_decision_stages

pytestmark = pytest.mark.gpu


class Ex:
    def __init__(self, device):
        self.device = device
        self.cfg = fm_synth.config("expert_fp8_m50")
        self.layers = [fm_synth.layer_weights(self.cfg, l) for l in range(self.cfg.L)]
        self.final = fm_synth.final_weights(self.cfg)
        self.kp, self.vp = fm_synth.prefix_kv(self.cfg)
        self.scales = load_scales("expert_fp8_m50")
        self.weights = fmad.DeviceWeights(self.cfg, self.layers, self.final, device=device)

    def policy(self, **over):
        cfg = dataclasses.replace(self.cfg, **over)
        p = fmad.Policy(cfg, act_scales=self.scales, weights=self.weights, device=self.device)
        p.set_prefix_kv(dev(self.kp, self.device, torch.bfloat16), dev(self.vp, self.device, torch.bfloat16))
        return p

    def noise(self, i):
        return dev(fm_synth.noise(self.cfg, i), self.device)


@pytest.fixture(scope="module")
def ex():
    return Ex(require_gpu())


def test_warm_t_one_equals_one_step_decision(ex):
    warm = ex.policy(warm_t=1.0)
    warm.decode(ex.noise(0))
    got = warm.decode_warm(ex.noise(1), 5)
    one = ex.policy(S=1)
    want = one.decode(ex.noise(1))
    torch.cuda.synchronize()
    assert fmad.device_status(warm.handle) == 0 and fmad.device_status(one.handle) == 0
    assert torch.equal(got, want)
    warm.close()
    one.close()


def test_episode_start_runs_the_full_decision(ex):
    p = ex.policy(warm_t=0.5)
    first = p.decode_warm(ex.noise(2), 0)          # no previous chunk yet
    p.decode(ex.noise(3))
    p.episode_reset()
    again = p.decode_warm(ex.noise(2), 7)
    ref = ex.policy()
    want = ref.decode(ex.noise(2))
    torch.cuda.synchronize()
    assert torch.equal(first, want) and torch.equal(again, want)
    p.close()
    ref.close()


def test_warm_decision_within_oracle_envelope(ex):
    p = ex.policy(warm_t=0.5)
    prev = p.decode(ex.noise(0)).cpu().numpy().astype(np.float64)
    got = p.decode_warm(ex.noise(1), 3).cpu().numpy().astype(np.float64)
    assert fmad.device_status(p.handle) == 0
    p.close()
    cfg = dataclasses.replace(ex.cfg, warm_t=0.5)
    model = O.Model(cfg, ex.layers, ex.final)
    ref = O.decode_warm(model, fm_synth.noise(cfg, 1), prev, 3, ex.kp, ex.vp, ex.scales)
    env = float(np.loadtxt(os.path.join(GOLDEN, "fp8_envelope_expert_fp8_m50_warm.txt")))
    err = np.max(np.abs(got - ref)) / np.sqrt(np.mean(ref ** 2))
    assert err <= 2 * env, (err, env)
    # and it moved: not the noise, not the shifted chunk
    assert np.max(np.abs(got - prev[np.minimum(np.arange(cfg.M) + 3, cfg.M - 1)])) > 1e-3


def test_warm_decision_is_one_step_of_time(ex):
    p = ex.policy(warm_t=0.5)
    nz = ex.noise(4)
    for _ in range(3):
        p.decode(nz)
        p.decode_warm(nz, 2)
    e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    e[0].record()
    p.decode(nz)
    e[1].record()
    e[2].record()
    p.decode_warm(nz, 2)
    e[3].record()
    torch.cuda.synchronize()
    full, warm = e[0].elapsed_time(e[1]), e[2].elapsed_time(e[3])
    assert warm < 0.25 * full, (warm, full)
    p.close()


@pytest.mark.parametrize("executed", [0, 3, 50])
def test_warm_start_teacher_forced(ex, executed):
    cfg = dataclasses.replace(ex.cfg, warm_t=0.5)
    p = ex.policy(warm_t=0.5)
    prev = p.decode(ex.noise(0)).cpu().numpy().astype(np.float64)
    nz = fm_synth.noise(cfg, 1)
    nbytes = fmad.warm_trace_size(p.handle)
    trace = torch.empty(nbytes, dtype=torch.uint8, device=ex.device)
    actions = torch.empty((cfg.M, cfg.A), dtype=torch.float32, device=ex.device)
    fmad.decode_warm_trace(p.handle, dev(nz, ex.device), executed, actions, trace, nbytes)
    assert fmad.device_status(p.handle) == 0
    raw = trace.cpu().numpy()
    got = actions.cpu().numpy()
    ab = cfg.M * cfg.A * 4
    recs = parse_trace(raw[ab:], dataclasses.replace(cfg, S=1), p)
    p.close()
    a_tau = raw[:ab].view(np.float32).reshape(cfg.M, cfg.A).astype(np.float64)
    tau = O.warm_time(cfg)
    want = O.warm_start_input(prev, executed, tau, nz)
    shifted = prev[np.minimum(np.arange(cfg.M) + executed, cfg.M - 1)]
    # one fp32 product and one fp32 fused multiply-add
    allow = 2.0 ** -23 * (tau * np.abs(nz) + (1.0 - tau) * np.abs(shifted))
    assert np.all(np.abs(a_tau - want) <= allow)
    if executed == cfg.M:   # every row is the last action, mixed with its own noise row
        assert np.allclose(a_tau - tau * nz, (1.0 - tau) * prev[-1], rtol=0, atol=1e-6)
    model = O.Model(cfg, ex.layers, ex.final)
    last = check_decision_stages(cfg, model, recs, a_tau, ex.kp, ex.vp, ex.scales, mod_rows=[cfg.S], dt=-tau)
    np.testing.assert_array_equal(got, last.astype(np.float32))
