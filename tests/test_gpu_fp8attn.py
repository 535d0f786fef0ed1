"""FP8 attention mode on the GPU (E4M3 Q, K, V with static per-layer scales, the
prefix cache's E4M3 copy, probabilities coded E4M3(P * 448)) against the CPU
oracle, on the 18-layer x 10-step FP8 expert (M = 50, prefix 788).

- the prefix copy is bit-exact after set_prefix_kv, refresh_prefix, a scale
  change and a capsule restore (codes = E4M3(fp32(x * fp32(1/s))));
- every kernel of a whole decision is pinned teacher-forced (QKV codes within one
  E4M3 step of the exact product's, attention within the coarse-probability
  allowance), and the decision end to end within twice the oracle's envelope;
- graph + PDL equals eager launches bitwise.
"""
import os

import numpy as np
import pytest
import torch

import fm_synth
import flow_matching_action_denoise_gb300 as fmad
from oracle import model as O

from _gpu import GOLDEN, dev, load_scales, parse_trace, require_gpu
from _stagewise import check_decision_stages, prefix_codes

pytestmark = pytest.mark.gpu
NAME = "expert_fp8attn_m50"


@pytest.fixture(scope="module")
def device():
    return require_gpu()


@pytest.fixture(scope="module")
def ex(device):
    cfg = fm_synth.config(NAME)
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    final = fm_synth.final_weights(cfg)
    kp, vp = fm_synth.prefix_kv(cfg)
    scales = load_scales(NAME)
    assert scales.shape == (cfg.L, 7)
    return dict(cfg=cfg, layers=layers, final=final, kp=kp, vp=vp, scales=scales, device=device,
                weights=fmad.DeviceWeights(cfg, layers, final, device=device), model=[None])


def policy(ex, flags=fmad.FLAG_USE_GRAPH | fmad.FLAG_USE_PDL, scales=None):
    p = fmad.Policy(ex["cfg"], act_scales=ex["scales"] if scales is None else scales, flags=flags,
                    weights=ex["weights"])
    p.set_prefix_kv(dev(ex["kp"], ex["device"], torch.bfloat16), dev(ex["vp"], ex["device"], torch.bfloat16))
    return p


def oracle(ex):
    if ex["model"][0] is None:
        ex["model"][0] = O.Model(ex["cfg"], ex["layers"], ex["final"])
    return ex["model"][0]


def read_prefix8(pol, cfg):
    p16 = (cfg.P + 15) // 16 * 16
    k8 = pol.buffer("prefix_k8", torch.uint8).cpu().numpy().reshape(cfg.L, cfg.P, cfg.Hkv, cfg.Dh)
    v8t = pol.buffer("prefix_v8", torch.uint8).cpu().numpy().reshape(cfg.L, cfg.Hkv, cfg.Dh, p16)
    from oracle import codecs as C
    kv = C.e4m3_decode_code(k8)
    vv = C.e4m3_decode_code(v8t[..., :cfg.P]).transpose(0, 3, 1, 2)   # -> [L][P][Hkv][Dh]
    assert not np.any(v8t[..., cfg.P:])   # the padding stays zero
    return kv, vv


def expect_prefix8(kp, vp, scales):
    pc = prefix_codes(kp, vp, scales)
    return np.stack([a for a, _ in pc]), np.stack([b for _, b in pc])


def test_prefix_copy_bit_exact(ex):
    cfg = ex["cfg"]
    pol = policy(ex)
    torch.cuda.synchronize()
    k8, v8 = read_prefix8(pol, cfg)
    ek, ev = expect_prefix8(ex["kp"], ex["vp"], ex["scales"])
    np.testing.assert_array_equal(k8, ek)
    np.testing.assert_array_equal(v8, ev)
    # refresh rows [0, 768): only those rows change
    kr, vr = fm_synth.prefix_kv_rows(cfg, 3, 768)
    pol.refresh_prefix(0, 768, dev(kr, ex["device"], torch.bfloat16), dev(vr, ex["device"], torch.bfloat16))
    torch.cuda.synchronize()
    k2, v2 = ex["kp"].copy(), ex["vp"].copy()
    k2[:, :768], v2[:, :768] = kr, vr
    k8, v8 = read_prefix8(pol, cfg)
    ek, ev = expect_prefix8(k2, v2, ex["scales"])
    np.testing.assert_array_equal(k8, ek)
    np.testing.assert_array_equal(v8, ev)
    # new scales re-derive the copy
    sc2 = ex["scales"].copy()
    sc2[:, 5:7] *= 1.5
    fmad.fm_set_act_scales(pol.handle, sc2)
    k8, v8 = read_prefix8(pol, cfg)
    ek, ev = expect_prefix8(k2, v2, sc2)
    np.testing.assert_array_equal(k8, ek)
    np.testing.assert_array_equal(v8, ev)
    pol.close()


def test_fp8_attention_decision_every_stage_vs_oracle(ex):
    cfg = ex["cfg"]
    pol = policy(ex)
    assert fmad.kernel_count(pol.handle) == (7, 1 + 18 * 10 * 7)
    nbytes = fmad.trace_size(pol.handle)
    trace = torch.empty(nbytes, dtype=torch.uint8, device=ex["device"])
    nz = fm_synth.noise(cfg, 0)
    act = torch.empty((cfg.M, cfg.A), dtype=torch.float32, device=ex["device"])
    fmad.decode_trace(pol.handle, dev(nz, ex["device"]), act, trace, nbytes)
    assert fmad.device_status(pol.handle) == 0
    assert torch.equal(act.cpu(), pol.decode(dev(nz, ex["device"])).cpu())
    recs = parse_trace(trace.cpu().numpy(), cfg, pol)
    last = check_decision_stages(cfg, oracle(ex), recs, nz, ex["kp"], ex["vp"], ex["scales"])
    np.testing.assert_array_equal(last, act.cpu().numpy())
    pol.close()


def test_fp8_attention_decision_within_envelope(ex):
    cfg = ex["cfg"]
    nz = fm_synth.noise(cfg, 0)
    pol = policy(ex)
    got = pol.decode(dev(nz, ex["device"])).cpu().numpy().astype(np.float64)
    assert fmad.device_status(pol.handle) == 0
    pol.close()
    ref = O.decode(oracle(ex), nz, ex["kp"], ex["vp"], ex["scales"])
    env = float(np.loadtxt(os.path.join(GOLDEN, f"fp8_envelope_{NAME}.txt")))
    err = np.max(np.abs(got - ref)) / np.sqrt(np.mean(ref ** 2))
    assert err <= 2 * env, (err, env)


def test_fp8_attention_launch_modes_and_restore(ex):
    cfg = ex["cfg"]
    nz = dev(fm_synth.noise(cfg, 4), ex["device"])
    a = policy(ex)
    b = policy(ex, flags=0)
    ya, yb = a.decode(nz).cpu(), b.decode(nz).cpu()
    assert torch.equal(ya, yb)
    # capsule: snapshot, disturb the prefix and the scales, restore -> the same decision
    n = fmad.state_size(a.handle)
    cap = torch.empty(n, dtype=torch.uint8, device=ex["device"])
    fmad.snapshot_state(a.handle, cap, n, True)
    kr, vr = fm_synth.prefix_kv_rows(cfg, 9, 768)
    a.refresh_prefix(0, 768, dev(kr, ex["device"], torch.bfloat16), dev(vr, ex["device"], torch.bfloat16))
    assert not torch.equal(a.decode(nz).cpu(), ya)
    assert fmad.restore_state(a.handle, cap, n, True) == 0
    assert torch.equal(a.decode(nz).cpu(), ya)
    a.close()
    b.close()
