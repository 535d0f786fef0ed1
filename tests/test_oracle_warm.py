"""Pins for the oracle's one-step warm start (CPU only).

- shift and pad: brute force on a tiny chunk for executed = 0, 2, M-1, M + 3;
- tau = 1 reduces to the ordinary one-step decision of the same noise (the chunk
  and the executed count drop out);
- tau = 0 returns the shifted, padded previous chunk exactly (a zero step);
- with W_out = 0 the velocity is the constant b_out, so the result is the closed
  form a_tau - tau * b_out (pins the step size dt = -tau);
- the config's warm_t row of the modulation table is the modulation at that time.
"""
import dataclasses

import numpy as np
import pytest

import fm_synth
from oracle import model as O


def tiny(**kw):
    base = dict(name="tiny", L=2, S=3, M=5, d=32, H=2, Hkv=1, Dh=16, F=64, P=4, A=4,
                weight_fmt="fp8", act_fmt="fp8", seed=11)
    base.update(kw)
    return fm_synth.Config(**base)


def setup(cfg, zero_out=False):
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    final = fm_synth.final_weights(cfg)
    if zero_out:
        final = dict(final)
        final["w_out"] = np.zeros_like(final["w_out"])
    model = O.Model(cfg, layers, final)
    kp, vp = fm_synth.prefix_kv(cfg)
    sc = np.full((cfg.L, 4), 0.05, np.float32)
    return model, kp, vp, sc


@pytest.mark.parametrize("e", [0, 2, 4, 8])
def test_shift_and_pad_brute_force(e):
    rng = np.random.default_rng(1)
    prev = rng.standard_normal((5, 3))
    got = O.warm_start_input(prev, e, 0.0, np.zeros((5, 3)))
    for i in range(5):
        src = i + e if i + e < 5 else 4
        np.testing.assert_array_equal(got[i], prev[src])


def test_tau_one_is_a_one_step_decision():
    cfg = tiny(warm_t=1.0)
    model, kp, vp, sc = setup(cfg)
    nz, prev = fm_synth.noise(cfg, 0), fm_synth.noise(cfg, 1)
    got = O.decode_warm(model, nz, prev, 2, kp, vp, sc)
    one = dataclasses.replace(cfg, S=1, warm_t=0.0)
    model1, _, _, _ = setup(one)
    np.testing.assert_array_equal(got, O.decode(model1, nz, kp, vp, sc))


def test_tau_zero_returns_the_shifted_chunk():
    cfg = tiny()
    model, kp, vp, sc = setup(cfg)
    prev = fm_synth.noise(cfg, 3)
    got = O.decode_warm(model, fm_synth.noise(cfg, 4), prev, 3, kp, vp, sc, tau=0.0)
    np.testing.assert_array_equal(got, prev[np.minimum(np.arange(cfg.M) + 3, cfg.M - 1)])


def test_constant_velocity_closed_form():
    cfg = tiny(warm_t=0.375)
    model, kp, vp, sc = setup(cfg, zero_out=True)
    nz, prev = fm_synth.noise(cfg, 5), fm_synth.noise(cfg, 6)
    got = O.decode_warm(model, nz, prev, 1, kp, vp, sc)
    a_tau = O.warm_start_input(prev, 1, 0.375, nz)
    np.testing.assert_allclose(got, a_tau - 0.375 * model.final["b_out"], rtol=0, atol=1e-15)


def test_warm_row_is_the_modulation_at_warm_t():
    cfg = tiny(warm_t=0.3)
    model, _, _, _ = setup(cfg)
    assert len(model.mods) == cfg.S + 1
    t = float(np.float32(0.3))
    want = model.mods_at(t)
    for l in range(cfg.L):
        for i in range(6):
            np.testing.assert_array_equal(model.mods[cfg.S][0][l][i], want[0][l][i])
    # and it differs from every scheduled step's
    assert all(not np.array_equal(model.mods[k][0][0][0], want[0][0][0]) for k in range(cfg.S))
