"""Whole-path parity on the GPU: one decoder layer (M = 10) and whole FP8 decisions
(18 layers x 10 Euler steps, M = 50, prefix 788) against the CPU oracle, plus the
bitwise invariants of the execution contract: graph == eager launch, PDL on == off,
repeat runs identical, refreshed prefix == freshly set prefix, snapshot -> restore
-> decode == uninterrupted run, and capsule binding to the plan and address.

Tolerances: max |gpu - oracle| <= 2e-2 * RMS(oracle) for one FP8 layer (the
workload definition's bound). The whole FP8 decision requantises 720 times and
is ill-conditioned at the rounding level (the oracle moves by ~16% of RMS when
only its pre-quantisation values are rounded to fp32), so it is pinned stage by
stage instead, and end to end within twice that derived envelope.
"""
import os

import numpy as np
import pytest
import torch

import fm_synth
import flow_matching_action_denoise_gb300 as fmad
from oracle import codecs as C
from oracle import model as O

from _gpu import GOLDEN, code_step_distance, dev, load_scales, parse_trace, require_gpu
from _stagewise import check_decision_stages

pytestmark = pytest.mark.gpu
TOL_FP8 = 2e-2


@pytest.fixture(scope="module")
def device():
    return require_gpu()


# ---------------------------------------------------------------- single layer (M = 10)

PLACEMENTS = {"separate": 0, "fused": fmad.FLAG_FUSED_CONSUMERS, "o_fused": fmad.FLAG_O_CONSUMER_IN_GEMM}


@pytest.mark.parametrize("placement", list(PLACEMENTS))
def test_single_layer_vs_oracle(device, placement):
    cfg = fm_synth.config("layer_fp8_m10")
    layers = [fm_synth.layer_weights(cfg, 0)]
    final = fm_synth.final_weights(cfg)
    conds = fm_synth.step_conds(cfg)
    kp, vp = fm_synth.prefix_kv(cfg)
    x = fm_synth.layer_input(cfg)
    scales = load_scales("layer_fp8_m10")
    model = O.Model(cfg, layers, final, conds)
    x_ref, q_ref, _ = O.single_layer(model, x, kp, vp, scales)

    flags = fmad.FLAG_USE_GRAPH | fmad.FLAG_USE_PDL | PLACEMENTS[placement]
    pol = fmad.Policy(cfg, layers, final, act_scales=scales, conds=conds, flags=flags)
    pol.set_prefix_kv(dev(kp, device, torch.bfloat16), dev(vp, device, torch.bfloat16))
    xin = dev(x, device)
    xout = torch.empty_like(xin)
    q = torch.empty((cfg.M, cfg.d), dtype=torch.uint8, device=device)
    fmad.fm_test_layer(pol.handle, xin, 0, 0, xout, q)
    torch.cuda.synchronize()
    assert fmad.device_status(pol.handle) == 0
    dx_ref = x_ref - x
    dx = xout.cpu().numpy().astype(np.float64) - x
    assert np.max(np.abs(dx - dx_ref)) <= TOL_FP8 * np.sqrt(np.mean(dx_ref ** 2))
    dist = code_step_distance(q.cpu().numpy(), C.e4m3_encode_code(q_ref))
    assert np.max(dist) <= 1 and np.mean(dist > 0) <= 1e-2
    per_layer, per_decision = fmad.kernel_count(pol.handle)
    assert (per_layer, per_decision) == {"o_fused": (6, 1 + 6), "fused": (5, 1 + 5 + 1),
                                         "separate": (7, 1 + 7)}[placement]
    pol.close()


# ---------------------------------------------------------------- full FP8 decisions (M = 50)

class Expert:
    """Raw weights on the device once; policies built from them share nothing else."""

    def __init__(self, device):
        self.cfg = cfg = fm_synth.config("expert_fp8_m50")
        self.layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
        self.final = fm_synth.final_weights(cfg)
        self.kp, self.vp = fm_synth.prefix_kv(cfg)
        self.scales = load_scales("expert_fp8_m50")
        self.weights = fmad.DeviceWeights(cfg, self.layers, self.final, device=device)
        self.k = dev(self.kp, device, torch.bfloat16)
        self.v = dev(self.vp, device, torch.bfloat16)
        self.device = device
        self._oracle = None

    def policy(self, flags=fmad.FLAG_USE_GRAPH | fmad.FLAG_USE_PDL, ksplit=(0, 0, 0, 0)):
        p = fmad.Policy(self.cfg, act_scales=self.scales, flags=flags, ksplit=ksplit, weights=self.weights)
        p.set_prefix_kv(self.k, self.v)
        return p

    def oracle(self):
        if self._oracle is None:
            self._oracle = O.Model(self.cfg, self.layers, self.final)
        return self._oracle

    def noise(self, i):
        return dev(fm_synth.noise(self.cfg, i), self.device)


@pytest.fixture(scope="module")
def expert(device):
    return Expert(device)


def test_decision_fp8_end_to_end_within_oracle_envelope(expert):
    """End to end: the FP8 decision requantises 720 times, so the oracle itself moves
    by `env` (tests/golden/make_fp8_envelope.py) when only its pre-quantisation values
    are rounded to fp32. The GPU must stay within twice that envelope; the
    stage-by-stage test below pins every kernel tightly."""
    nz = fm_synth.noise(expert.cfg, 0)
    ref = O.decode(expert.oracle(), nz, expert.kp, expert.vp, expert.scales)
    env = float(np.loadtxt(os.path.join(GOLDEN, "fp8_envelope_expert_fp8_m50.txt")))
    base = fmad.FLAG_USE_GRAPH | fmad.FLAG_USE_PDL
    # every consumer as its own kernel (default, 7 kernels per layer), the O GEMM's
    # consumer in its epilogue (6), and the consumers inside the GEMMs (5 kernels per layer
    # plus one step-boundary kernel per step)
    for flags, counts in [(base, (7, 1 + 18 * 10 * 7)), (base | fmad.FLAG_O_CONSUMER_IN_GEMM, (6, 1 + 18 * 10 * 6)),
                          (base | fmad.FLAG_FUSED_CONSUMERS, (5, 1 + 18 * 10 * 5 + 10))]:
        pol = expert.policy(flags)
        act = pol.decode(dev(nz, expert.device))
        torch.cuda.synchronize()
        assert fmad.device_status(pol.handle) == 0
        got = act.cpu().numpy().astype(np.float64)
        err = np.max(np.abs(got - ref)) / np.sqrt(np.mean(ref ** 2))
        assert err <= 2 * env, (flags, err, env)
        assert fmad.kernel_count(pol.handle) == counts
        # 838 keys in 7 slices of 128 (the small grid splits O's head dims; no wide slice)
        assert fmad.attn_plan(pol.handle) == (128, 7)
        pol.close()


@pytest.mark.parametrize("placement", list(PLACEMENTS))
def test_decision_fp8_every_stage_vs_oracle(expert, placement):
    """Teacher-forced parity of every kernel of all 180 layer-steps: each recorded
    output equals the oracle's stage applied to the GPU's own recorded input -
    fp32 outputs within 1e-5 * RMS, quantised codes within one E4M3 step with at
    most 0.1% near-tie differences."""
    cfg, model = expert.cfg, expert.oracle()
    pol = expert.policy(fmad.FLAG_USE_GRAPH | fmad.FLAG_USE_PDL | PLACEMENTS[placement])
    nbytes = fmad.trace_size(pol.handle)
    trace = torch.empty(nbytes, dtype=torch.uint8, device=expert.device)
    nz = fm_synth.noise(cfg, 0)
    act = torch.empty((cfg.M, cfg.A), dtype=torch.float32, device=expert.device)
    fmad.decode_trace(pol.handle, dev(nz, expert.device), act, trace, nbytes)
    assert fmad.device_status(pol.handle) == 0
    # the traced (eager) run is bitwise the graph run
    assert torch.equal(act.cpu(), pol.decode(dev(nz, expert.device)).cpu())
    recs = parse_trace(trace.cpu().numpy(), cfg, pol)
    last = check_decision_stages(cfg, model, recs, nz, expert.kp, expert.vp, expert.scales)
    np.testing.assert_array_equal(last, act.cpu().numpy())
    pol.close()


def test_launch_modes_bitwise_identical(expert):
    nz = expert.noise(3)
    outs = []
    for flags in [fmad.FLAG_USE_GRAPH | fmad.FLAG_USE_PDL, fmad.FLAG_USE_GRAPH, fmad.FLAG_USE_PDL, 0]:
        pol = expert.policy(flags)
        outs.append(pol.decode(nz).cpu())
        outs.append(pol.decode(nz).cpu())   # repeat run on the same policy
        assert fmad.device_status(pol.handle) == 0
        pol.close()
    for o in outs[1:]:
        assert torch.equal(o, outs[0])


def test_ksplit_choices_agree(expert):
    nz = expert.noise(4)
    base = expert.policy()
    ref = base.decode(nz).cpu().numpy()
    base.close()
    pol = expert.policy(ksplit=(4, 2, 8, 8))
    got = pol.decode(nz).cpu().numpy()
    pol.close()
    # a different split changes only the fp32 summation order; through 720 requantisations
    # that is bounded by the same rounding envelope as the oracle comparison
    env = float(np.loadtxt(os.path.join(GOLDEN, "fp8_envelope_expert_fp8_m50.txt")))
    assert np.max(np.abs(got - ref)) <= 2 * env * np.sqrt(np.mean(ref ** 2))


def test_refresh_prefix_equals_fresh_set(expert):
    cfg = expert.cfg
    rows = 768
    kr, vr = fm_synth.prefix_kv_rows(cfg, 1, rows)
    nz = expert.noise(5)
    a = expert.policy()
    a.refresh_prefix(0, rows, dev(kr, expert.device, torch.bfloat16), dev(vr, expert.device, torch.bfloat16))
    out_a = a.decode(nz).cpu()
    b = expert.policy()
    k2, v2 = expert.kp.copy(), expert.vp.copy()
    k2[:, :rows], v2[:, :rows] = kr, vr
    b.set_prefix_kv(dev(k2, expert.device, torch.bfloat16), dev(v2, expert.device, torch.bfloat16))
    out_b = b.decode(nz).cpu()
    assert torch.equal(out_a, out_b)
    # and the refresh changed the result (the prefix reaches the attention)
    c = expert.policy()
    assert not torch.equal(c.decode(nz).cpu(), out_a)
    for p in (a, b, c):
        p.close()


def test_snapshot_restore_roundtrip(expert):
    cfg = expert.cfg
    pol = expert.policy()
    n = fmad.state_size(pol.handle)
    assert n >= 2 * cfg.L * cfg.P * cfg.Hkv * cfg.Dh * 2
    cap_host = torch.empty(n, dtype=torch.uint8).pin_memory()
    cap_dev = torch.empty(n, dtype=torch.uint8, device=expert.device)
    fmad.snapshot_state(pol.handle, cap_host, n, False)
    fmad.snapshot_state(pol.handle, cap_dev, n, True)
    nz = expert.noise(6)
    first = pol.decode(nz).cpu()
    # another session overwrites the state
    kr, vr = fm_synth.prefix_kv_rows(cfg, 2, cfg.P)
    pol.set_prefix_kv(dev(kr, expert.device, torch.bfloat16), dev(vr, expert.device, torch.bfloat16))
    other = pol.decode(expert.noise(7)).cpu()
    assert not torch.equal(other, first)
    for cap, on_dev in [(cap_host, False), (cap_dev, True)]:
        assert fmad.restore_state(pol.handle, cap, n, on_dev) == 0
        assert torch.equal(pol.decode(nz).cpu(), first)
    # the capsule's noise buffer is restored too: decode from it (noise = NULL)
    assert fmad.restore_state(pol.handle, cap_host, n, False) == 0
    out = torch.empty_like(nz)
    fmad.decode_actions(pol.handle, None, out)
    # the capsule was taken before any decision: its noise buffer is zero
    zero_start = pol.decode(torch.zeros_like(nz)).cpu()
    assert torch.equal(out.cpu(), zero_start)
    # bound to the plan and the address: another policy rejects it
    other_pol = expert.policy()
    st = fmad.restore_state(other_pol.handle, cap_host, n, False)
    assert st == 6
    bad = cap_host.clone()
    bad[0] ^= 0xFF
    assert fmad.restore_state(pol.handle, bad, n, False) == 6
    pol.close()
    other_pol.close()


def test_decode_host_buffers_match_device(expert):
    pol = expert.policy()
    nz = fm_synth.noise(expert.cfg, 8)
    dev_out = pol.decode(dev(nz, expert.device)).cpu()
    h_in = torch.from_numpy(nz).pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    fmad.decode_actions_host(pol.handle, h_in, h_out)
    assert torch.equal(h_out, dev_out)
    pol.close()
