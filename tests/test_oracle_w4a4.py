"""Pins for the oracle's four-bit activations (W4A4 NVFP4; CPU only).

- every element lands on the E2M1 grid and every block scale on the E4M3 grid;
- a block built from grid values (its largest element 6 * bs * ts) round-trips
  exactly;
- the error bound |h - e bs ts| <= bs ts + amax_b / 16 (half the widest E2M1 gap at
  the block's scale, plus the block scale's E4M3 rounding) holds on random data;
- power-of-two scalings of h and ts commute with the quantiser; zero blocks stay
  zero; a too-small tensor scale saturates at bs = 448, |e| = 6;
- the W4A4 product equals a library matmul of the dequantised operands;
- calibration maps each site's largest pre-quantisation value to bs = 448, e = 6.
"""
import numpy as np
import pytest

import fm_synth
from oracle import codecs as C
from oracle import model as O

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def test_codes_on_their_grids():
    rng = np.random.default_rng(3)
    h = rng.standard_normal((5, 64)) * np.exp(rng.standard_normal((5, 1)))
    ts = float(np.float32(np.max(np.abs(h)) / 2688.0))
    vals, bs = O.quant_nvfp4_act(h, ts)
    assert np.array_equal(C.e4m3(bs), bs) and np.all(bs >= 0)
    e = vals.reshape(5, 4, 16) / np.where(bs > 0, bs, 1.0)[..., None]
    assert np.all(np.isin(np.abs(e), E2M1_GRID))


def test_grid_block_round_trips_exactly():
    ts, bs = 2.0 ** -4, 1.5                       # both exact; bs on the E4M3 grid
    e = np.array([6.0, -4.0, 3.0, 0.5, -0.5, 0.0, 1.0, -1.5, 2.0, -6.0, 4.0, 1.5, -2.0, 3.0, 0.0, -1.0])
    h = (e * bs * ts)[None, :]
    vals, got_bs = O.quant_nvfp4_act(h, ts)
    assert got_bs[0, 0] == bs
    np.testing.assert_array_equal(vals[0] * ts, h[0])


def test_error_bound():
    rng = np.random.default_rng(4)
    h = rng.standard_normal((8, 128)) * rng.uniform(0.1, 10.0, (8, 1))
    ts = float(np.float32(np.max(np.abs(h)) / 2688.0))
    vals, bs = O.quant_nvfp4_act(h, ts)
    err = np.abs(h - vals * ts).reshape(8, 8, 16)
    amax_b = np.max(np.abs(h.reshape(8, 8, 16)), axis=-1)
    bound = bs * ts + amax_b / 16.0
    assert np.all(err <= bound[..., None] * (1 + 1e-12))


def test_power_of_two_scaling_zero_blocks_and_saturation():
    rng = np.random.default_rng(5)
    h = rng.standard_normal((3, 32))
    h[1, 16:] = 0.0
    ts = float(np.float32(np.max(np.abs(h)) / 2688.0))
    v1, b1 = O.quant_nvfp4_act(h, ts)
    v2, b2 = O.quant_nvfp4_act(h * 8.0, ts * 8.0)
    np.testing.assert_array_equal(v1, v2)
    np.testing.assert_array_equal(b1, b2)
    assert b1[1, 1] == 0.0 and np.all(v1[1, 16:] == 0.0)
    vs, bss = O.quant_nvfp4_act(h, ts / 64.0)    # far too small: block scales saturate
    assert np.max(bss) == 448.0
    assert np.max(np.abs(vs / np.repeat(np.where(bss > 0, bss, 1.0), 16, axis=1))) == 6.0


def test_w4a4_gemm_is_the_product_of_dequantised_operands():
    rng = np.random.default_rng(6)
    a = rng.standard_normal((4, 64))
    w = rng.standard_normal((32, 64)) * 0.02
    pw = O.prep_weight(w, None, "nvfp4")
    ts_a = float(np.float32(np.max(np.abs(a)) / 2688.0))
    vals, _ = O.quant_nvfp4_act(a, ts_a)
    got = O.gemm(vals, ts_a, pw)
    want = (vals * ts_a) @ (pw.codes * pw.scale).T
    np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-12)


def test_calibration_maps_each_site_amax_to_the_top_codes():
    cfg = fm_synth.Config(name="tiny_w4a4", L=1, S=1, M=3, d=32, H=2, Hkv=1, Dh=16, F=64, P=4, A=4,
                          weight_fmt="nvfp4", act_fmt="nvfp4", seed=9)
    layers = [fm_synth.layer_weights(cfg, 0)]
    model = O.Model(cfg, layers, fm_synth.final_weights(cfg))
    kp, vp = fm_synth.prefix_kv(cfg)
    nz = fm_synth.noise(cfg, 0)
    prov = np.ones((1, 4), np.float32)
    sc = O.calibrate(model, nz, kp, vp, prov)
    # the pre-attention input of layer 0 at step 0: its largest element codes as 6 * 448
    x = np.asarray(nz, np.float64) @ model.final["w_in"].T + model.final["b_in"]
    sc1, sh1 = model.mods[0][0][0][0], model.mods[0][0][0][1]
    h = O.ada_norm(x, sc1, sh1, cfg.eps)
    vals, bs = O.quant_nvfp4_act(h, float(sc[0, O.SITE_ATTN_IN]))
    assert np.max(bs) == 448.0
    assert np.max(np.abs(vals)) == 6.0 * 448.0
    out = O.decode(model, nz, kp, vp, sc)
    assert np.all(np.isfinite(out))
