"""Device decision noise (Philox4x32-10 + Box-Muller) against the oracle's
generator, and decisions driven by it.

- the Philox words are bit-exact (integer work) for full and ragged chunks and
  for seeds / counters that use all 64 bits;
- the Gaussian values equal the oracle's float64 values rounded to float32, up to
  one float32 step where the two libraries' last-bit rounding differs (at most
  0.1% of elements);
- a seeded decision equals decode_actions on the same noise bitwise; the
  decision's timestamps are ordered and plausible.
"""
import numpy as np
import pytest
import torch

import fm_synth
import flow_matching_action_denoise_gb300 as fmad
from oracle import philox as X

from _gpu import load_scales, require_gpu

pytestmark = pytest.mark.gpu

STREAMS = [(0, 0), (7, 3), (0x0123456789ABCDEF, 0xFEDCBA9876543210), (2 ** 64 - 1, 2 ** 32 + 5)]


@pytest.fixture(scope="module")
def device():
    return require_gpu()


@pytest.mark.parametrize("n", [1600, 1603, 4])
@pytest.mark.parametrize("seed,counter", STREAMS)
def test_philox_words_bit_exact(device, n, seed, counter):
    nb = (n + 3) // 4
    out = torch.empty(n, dtype=torch.float32, device=device)
    raw = torch.zeros(nb * 4, dtype=torch.int32, device=device)
    fmad.philox_noise(out, seed, counter, raw)
    torch.cuda.synchronize()
    got = raw.cpu().numpy().view(np.uint32).reshape(nb, 4)
    np.testing.assert_array_equal(got, X.raw_blocks(seed, counter, nb))


@pytest.mark.parametrize("seed,counter", STREAMS)
def test_noise_values_match_oracle(device, seed, counter):
    M, A = 50, 32
    out = torch.empty(M * A + 3, dtype=torch.float32, device=device)   # ragged tail
    fmad.philox_noise(out, seed, counter)
    torch.cuda.synchronize()
    got = out.cpu().numpy().astype(np.float64)
    want64 = X.decision_noise(seed, counter, 1, M * A + 3).ravel()
    want = want64.astype(np.float32).astype(np.float64)
    ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
    diff = np.abs(got - want)
    assert np.all(diff <= ulp), float(np.max(diff / ulp))
    assert np.mean(diff > 0) <= 1e-3


def test_seeded_decision_equals_decode_on_same_noise(device):
    cfg = fm_synth.config("expert_fp8_m50")
    pol = fmad.Policy(cfg, [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)], fm_synth.final_weights(cfg),
                      act_scales=load_scales("expert_fp8_m50"), device=device)
    kp, vp = fm_synth.prefix_kv(cfg)
    pol.set_prefix_kv(torch.from_numpy(kp).to(device, torch.bfloat16), torch.from_numpy(vp).to(device, torch.bfloat16))
    noise = torch.empty((cfg.M, cfg.A), dtype=torch.float32, device=device)
    fmad.philox_noise(noise, 42, 9)
    want = pol.decode(noise.clone())
    got = pol.decode_seeded(42, 9)
    torch.cuda.synchronize()
    assert fmad.device_status(pol.handle) == 0
    assert torch.equal(got, want)
    other = pol.decode_seeded(42, 10)
    assert not torch.equal(other, got)
    # timestamps of the last decision
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    pol.decode_seeded(42, 11)
    e1.record()
    t = pol.last_timing()
    ms = e0.elapsed_time(e1)
    assert t["host_submit_ns"] > 0 and t["device_end_ns"] > t["device_start_ns"] > 0
    assert 0.2 * ms < t["t_infer_ns"] * 1e-6 <= ms * 1.05 + 0.05, (t, ms)
    pol.close()
