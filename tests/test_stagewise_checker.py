"""The stage-by-stage checker the GPU parity tests use (tests/_stagewise.py),
exercised on CPU for FP8, BF16, FP8-attention and four-bit (W4A4: NVFP4 weights and
activations) decisions: records produced by the oracle
itself in the trace's layout pass, and records from an implementation with a
plausible mistake (gate and up
swapped, a dropped residual gate, the Euler sign, the next layer's modulation in
the pre-MLP norm, K and V swapped in the QKV output, a wrong dequantisation
scale) each fail it."""
import numpy as np
import pytest

import fm_synth
from oracle import codecs as C
from oracle import model as O

from _stagewise import check_decision_stages, prefix_codes


def tiny(fmt="fp8"):
    attn8 = fmt == "fp8attn"
    fmt = "fp8" if attn8 else fmt
    wfmt, afmt = ("nvfp4", "nvfp4") if fmt == "w4a4" else (fmt, fmt)
    cfg = fm_synth.Config(name="tiny_stages", L=2, S=2, M=3, d=32, H=2, Hkv=1, Dh=16, F=64, P=4, A=4,
                          weight_fmt=wfmt, act_fmt=afmt, seed=21, attn_fmt="fp8" if attn8 else "bf16")
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    model = O.Model(cfg, layers, fm_synth.final_weights(cfg))
    kp, vp = fm_synth.prefix_kv(cfg)
    nz = fm_synth.noise(cfg, 0)
    cols = 7 if attn8 else 4
    sc = (O.calibrate(model, nz, kp, vp, np.full((cfg.L, cols), 0.05, np.float32))
          if afmt in ("fp8", "nvfp4") else None)
    return cfg, model, kp, vp, nz, sc


def records(cfg, model, kp, vp, nz, sc, mistake=None):
    """What a decision's trace holds, computed by the oracle's stages (optionally
    with one planted mistake)."""
    M, H, Dh, F, L, S, d = cfg.M, cfg.H, cfg.Dh, cfg.F, cfg.L, cfg.S, cfg.d
    fmt = cfg.act_fmt
    attn8 = cfg.attn_fmt == "fp8"
    prefix8 = prefix_codes(kp, vp, sc) if attn8 else None
    s_act = lambda l, i: float(sc[l][i]) if fmt in ("fp8", "nvfp4") else 1.0
    fin = model.final
    nq, nk = H * Dh, cfg.Hkv * Dh
    dq = lambda l, i, w: np.float64(np.float32(s_act(l, i)) * np.float32(w.scale)) * (
        2.0 if mistake == "dequant" and i == 1 else 1.0)
    kp64, vp64 = np.asarray(kp, np.float64), np.asarray(vp, np.float64)
    a = np.asarray(nz, np.float64)
    x = a @ fin["w_in"].T + fin["b_in"]
    recs = [[{} for _ in range(L)] for _ in range(S)]
    for k in range(S):
        for l in range(L):
            r = recs[k][l]
            W = model.w[l]
            sc1, sh1, g1, sc2, sh2, g2 = model.mods[k][0][l]
            if mistake == "next_layer_mod":
                sc2, sh2 = model.mods[k][0][(l + 1) % L][3], model.mods[k][0][(l + 1) % L][4]
            r["x_in"] = x
            r["q"] = O.quant_codes(O.ada_norm(x, sc1, sh1, cfg.eps), s_act(l, 0),
                                   "fp8" if mistake == "act_e4m3" else fmt)
            exact = (r["q"] @ W["qkv"].codes.T) * dq(l, 0, W["qkv"])
            if attn8:   # E4M3 Q | K | V codes with their static scales; attention on codes
                s3 = [s_act(l, O.SITE_Q), s_act(l, O.SITE_K), s_act(l, O.SITE_V)]
                qkv = np.concatenate([O.quant_codes(exact[:, a:b], sx, "fp8") for (a, b), sx in
                                      zip(((0, nq), (nq, nq + nk), (nq + nk, exact.shape[1])), s3)], axis=1)
            else:
                qkv = C.bf16(exact)
            if mistake == "kv_swapped":
                qkv = np.concatenate([qkv[:, :nq], qkv[:, nq + nk:], qkv[:, nq:nq + nk]], axis=1)
            r["y_qkv"] = qkv
            if attn8:
                s_v = s3[2] * (2.0 if mistake == "dequant_v" else 1.0)
                att = O.attention_fp8(qkv[:, :nq], qkv[:, nq:nq + nk], qkv[:, nq + nk:], prefix8[l][0],
                                      prefix8[l][1], H, cfg.Hkv, Dh, s3[0], s3[1], s_v)
            else:
                att = O.attention(qkv[:, :nq], qkv[:, nq:nq + nk], qkv[:, nq + nk:], kp64[l], vp64[l], H, cfg.Hkv,
                                  Dh)
            r["attn_out"] = O.quant_codes(att, s_act(l, 1), fmt)
            yo = r["attn_out"] @ W["o"].codes.T
            r["y_o"] = np.zeros((0, M, d))
            x_mid = x + (1.0 if mistake == "dropped_gate" else g1) * yo * dq(l, 1, W["o"])
            r["x_mid"] = x_mid
            r["q2"] = O.quant_codes(O.ada_norm(x_mid, sc2, sh2, cfg.eps), s_act(l, 2), fmt)
            gu = (r["q2"] @ W["gu"].codes.T) * dq(l, 2, W["gu"])
            g, u = (gu[:, F:], gu[:, :F]) if mistake == "gate_up_swapped" else (gu[:, :F], gu[:, F:])
            r["geglu_out"] = O.quant_codes(O.gelu_tanh(g) * u, s_act(l, 3), fmt)
            r["y_d"] = np.zeros((0, M, d))
            x = x_mid + g2 * (r["geglu_out"] @ W["d"].codes.T) * dq(l, 3, W["d"])
            if l == L - 1:
                scf, shf = model.mods[k][1]
                v = (O.ada_norm(x, scf, shf, cfg.eps) * fin["gamma_f"]) @ fin["w_out"].T + fin["b_out"]
                a = a + ((1.0 if mistake == "euler_sign" else -1.0) / S) * v
                r["actions"] = a.astype(np.float32)
                a = r["actions"].astype(np.float64)
                if k < S - 1:
                    x = a @ fin["w_in"].T + fin["b_in"]
            r["x_out"] = x
    return recs


@pytest.fixture(scope="module", params=["fp8", "bf16", "fp8attn", "w4a4"])
def case(request):
    return tiny(request.param)


def test_oracle_records_pass(case):
    cfg, model, kp, vp, nz, sc = case
    last = check_decision_stages(cfg, model, records(cfg, model, kp, vp, nz, sc), nz, kp, vp, sc)
    # the records hold the action state in fp32 between steps, as the GPU does; with E4M3
    # probabilities that rounding alone can flip a code of the next step
    np.testing.assert_allclose(last, O.decode(model, nz, kp, vp, sc), rtol=0,
                               atol=1e-3 if cfg.attn_fmt == "fp8" else 1e-5)


@pytest.mark.parametrize("mistake", ["gate_up_swapped", "dropped_gate", "euler_sign", "next_layer_mod",
                                     "kv_swapped", "dequant"])
def test_planted_mistake_fails(case, mistake):
    cfg, model, kp, vp, nz, sc = case
    with pytest.raises(AssertionError):
        check_decision_stages(cfg, model, records(cfg, model, kp, vp, nz, sc, mistake), nz, kp, vp, sc)


def test_w4a4_planted_e4m3_activations_fail():
    """Four-bit activations quantised as E4M3 codes instead (the wrong operand format)."""
    cfg, model, kp, vp, nz, sc = tiny("w4a4")
    with pytest.raises(AssertionError):
        check_decision_stages(cfg, model, records(cfg, model, kp, vp, nz, sc, "act_e4m3"), nz, kp, vp, sc)


def test_fp8_attention_planted_scale_fails():
    cfg, model, kp, vp, nz, sc = tiny("fp8attn")
    with pytest.raises(AssertionError):
        check_decision_stages(cfg, model, records(cfg, model, kp, vp, nz, sc, "dequant_v"), nz, kp, vp, sc)
