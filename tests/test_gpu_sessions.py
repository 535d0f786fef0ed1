"""Sessions and capsule fork on the GPU (the 18-layer FP8 expert, M = 50).

- a session shares the base's weights: its workspace is a small fraction of the
  base's, and its decisions equal the base's bitwise on the same prefix and noise;
- a fork starts from a capsule: base and fork continue identically from the
  capsule's action buffer; afterwards each evolves alone (a refresh of the base's
  prefix does not reach the fork); restore_state stays bound to the capsule's own
  workspace;
- two sessions decide concurrently on two streams with the results of sequential
  runs;
- a base with live sessions is not destroyed.
"""
import numpy as np
import pytest
import torch

import fm_synth
import flow_matching_action_denoise_gb300 as fmad

from _gpu import dev, load_scales, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def base():
    device = require_gpu()
    cfg = fm_synth.config("expert_fp8_m50")
    p = fmad.Policy(cfg, [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)], fm_synth.final_weights(cfg),
                    act_scales=load_scales("expert_fp8_m50"), device=device)
    kp, vp = fm_synth.prefix_kv(cfg)
    p.kv = (dev(kp, device, torch.bfloat16), dev(vp, device, torch.bfloat16))
    p.set_prefix_kv(*p.kv)
    yield p
    p.close()


def noise(p, i):
    return dev(fm_synth.noise(p.cfg, i), p.device)


def test_session_shares_weights_and_decides_identically(base):
    s = base.session()
    assert s.ws_bytes < 0.05 * base.ws_bytes
    s.set_prefix_kv(*base.kv)
    for i in range(3):
        a, b = base.decode(noise(base, i)), s.decode(noise(base, i))
        torch.cuda.synchronize()
        assert torch.equal(a, b)
    assert fmad.device_status(s.handle) == 0
    s.close()


def test_fork_continues_from_the_capsule_then_diverges(base):
    base.decode(noise(base, 5))
    n = fmad.state_size(base.handle)
    cap = torch.empty(n, dtype=torch.uint8, device=base.device)
    fmad.snapshot_state(base.handle, cap, n, True)
    f = base.fork(cap)
    # both continue from the capsule's action buffer (noise = None)
    a = base.decode(None, torch.empty((base.cfg.M, base.cfg.A), device=base.device))
    b = f.decode(None, torch.empty((base.cfg.M, base.cfg.A), device=base.device))
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    # a capsule of the base does not restore into the fork's workspace (STATE_MISMATCH)
    assert fmad.restore_state(f.handle, cap, n, True) == 6
    # the base's prefix refresh stays in the base
    kr, vr = fm_synth.prefix_kv_rows(base.cfg, 4, 768)
    base.refresh_prefix(0, 768, dev(kr, base.device, torch.bfloat16), dev(vr, base.device, torch.bfloat16))
    ya, yb = base.decode(noise(base, 6)), f.decode(noise(base, 6))
    torch.cuda.synchronize()
    assert not torch.equal(ya, yb)
    base.set_prefix_kv(*base.kv)
    assert torch.equal(base.decode(noise(base, 6)), yb)
    f.close()


def test_sessions_decide_concurrently_on_two_streams(base):
    s1, s2 = base.session(), base.session()
    for s in (s1, s2):
        s.set_prefix_kv(*base.kv)
    torch.cuda.synchronize()
    want1, want2 = s1.decode(noise(base, 7)).clone(), s2.decode(noise(base, 8)).clone()
    torch.cuda.synchronize()
    st1, st2 = torch.cuda.Stream(), torch.cuda.Stream()
    n7, n8 = noise(base, 7), noise(base, 8)
    torch.cuda.synchronize()
    outs = []
    for _ in range(3):
        with torch.cuda.stream(st1):
            o1 = s1.decode(n7, stream=st1)
        with torch.cuda.stream(st2):
            o2 = s2.decode(n8, stream=st2)
        outs.append((o1, o2))
    torch.cuda.synchronize()
    for o1, o2 in outs:
        assert torch.equal(o1, want1) and torch.equal(o2, want2)
    s1.close()
    s2.close()


def test_base_with_live_sessions_is_not_destroyed(base):
    s = base.session()
    with pytest.raises(fmad.FmError) as e:
        fmad.policy_destroy(base.handle)
    assert e.value.status == 1
    s.close()
    # the base still works
    assert torch.isfinite(base.decode(noise(base, 0))).all()
