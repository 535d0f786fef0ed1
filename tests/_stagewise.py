"""Teacher-forced, stage-by-stage check of a recorded decision (fm_decode_trace)
against the oracle: every kernel's recorded output must equal the oracle's stage
applied to the GPU's own recorded input. Shared by the FP8 and bf16 decision tests.

Tolerances:
- fp32 outputs (GEMM partial sums, residual stream, Euler update): 1e-5 * RMS;
- quantised operands (E4M3 codes or bf16 values): one grid step at the larger
  magnitude plus abs_tol * RMS, with at most max_frac of the values differing
  (a value within rounding distance of a tie may round either way);
- the QKV epilogue's bf16 outputs: within one bf16 rounding of the exact product.
"""
import numpy as np

from oracle import codecs as C
from oracle import model as O


def e4m3_ulp(v):
    """Spacing of the E4M3 grid at |v| (code units): 2^(e-3) for normal values, 2^-9 below 2^-6."""
    a = np.abs(np.asarray(v, np.float64))
    _, E = np.frexp(a)
    return np.ldexp(1.0, np.maximum(E - 1, -6) - 3)


def bf16_ulp(v):
    """Spacing of the bf16 grid at |v|: 8 significant bits, 2^(e-7) for |v| in [2^e, 2^(e+1))."""
    a = np.abs(np.asarray(v, np.float64))
    _, E = np.frexp(a)
    return np.ldexp(1.0, np.maximum(E - 1, -126) - 7)


def nvfp4_step(got, ref):
    """One grid step of four-bit activation values e * bs (E2M1 e, E4M3 block scale bs
    per 16 consecutive elements of the last axis) at the larger of the two magnitudes:
    every block's largest code is 6 (the block scale is amax / 6, rounded), so bs is the
    block's largest magnitude / 6; the E2M1 step is 0.5, 1 or 2 for |e| below 2, 4, 6.
    The larger of the two block scales covers a block whose scale rounded differently."""
    g, r = np.abs(got), np.abs(ref)
    shp = g.shape
    gb, rb = g.reshape(-1, 16), r.reshape(-1, 16)
    bs = np.maximum(gb.max(axis=1), rb.max(axis=1))[:, None] / 6.0
    v = np.maximum(gb, rb)
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.where(bs > 0, v / np.where(bs > 0, bs, 1.0), 0.0)
    step = np.where(e < 2, 0.5, np.where(e < 4, 1.0, 2.0)) * bs
    return step.reshape(shp)


def check_codes(got_values, ref_values, what, fmt="fp8", max_frac=1e-3, abs_tol=1e-3, extra=0.0):
    """Quantised operands agree when they differ by at most one grid step at the larger
    magnitude plus abs_tol * RMS (plus a per-element `extra`): a near-tie input rounds
    either way, and near zero (subnormal steps) a tiny upstream difference can span
    several steps."""
    got, ref = np.asarray(got_values, np.float64), np.asarray(ref_values, np.float64)
    diff = np.abs(got - ref)
    if fmt == "nvfp4":
        step = nvfp4_step(got, ref)
    else:
        step = (e4m3_ulp if fmt == "fp8" else bf16_ulp)(np.maximum(np.abs(got), np.abs(ref)))
    allow = step + abs_tol * np.sqrt(np.mean(ref ** 2)) + extra
    bad = diff > allow * (1 + 1e-12)
    if np.any(bad):
        i = np.unravel_index(np.argmax(diff - allow), diff.shape)
        raise AssertionError(f"{what}: {np.sum(bad)} codes beyond tolerance, worst at {i}: "
                             f"got {got[i]} ref {ref[i]} (allow {allow[i]:.3g})")
    frac = np.mean(diff > 0)
    assert frac <= max_frac, f"{what}: {frac:.2e} of codes differ"


def check_close(got, ref, what, tol=1e-5):
    err = np.max(np.abs(np.asarray(got, np.float64) - ref)) / (np.sqrt(np.mean(ref ** 2)) + 1e-30)
    assert err <= tol, f"{what}: {err:.2e} > {tol:.0e}"


def check_increment(new, old, inc_ref, what, tol=1e-5):
    """A residual update x_new = fp32(x_old + inc): the increment within tol * RMS(inc),
    plus the fp32 rounding of the stored sum (2^-22 of |x_new| covers it with room)."""
    new, old = np.asarray(new, np.float64), np.asarray(old, np.float64)
    err = np.abs((new - old) - inc_ref)
    allow = tol * np.sqrt(np.mean(inc_ref ** 2)) + 2.0 ** -22 * np.abs(new)
    if np.any(err > allow):
        i = np.unravel_index(np.argmax(err - allow), err.shape)
        raise AssertionError(f"{what}: increment off by {err[i]:.3g} at {i} (allow {allow[i]:.3g})")


def prefix_codes(kp, vp, scales):
    """The E4M3 prefix copy the FP8-attention path keeps: per layer
    E4M3(fp32(x * fp32(1 / s))) with the layer's K and V scales."""
    out = []
    for l in range(kp.shape[0]):
        rk = np.float64(np.float32(1.0) / np.float32(scales[l][O.SITE_K]))
        rv = np.float64(np.float32(1.0) / np.float32(scales[l][O.SITE_V]))
        out.append((C.e4m3(C.fp32(np.asarray(kp[l], np.float64) * rk)),
                    C.e4m3(C.fp32(np.asarray(vp[l], np.float64) * rv))))
    return out


_E4M3_POS = np.unique(np.abs(C.e4m3_decode_code(np.arange(0, 127))))


def fp8_attention_allowance(qc, kc, vc, kpre_c, vpre_c, H, Hkv, Dh, s_q, s_k, s_v, rel=1e-5):
    """Largest change of O when probability codes whose exact value P * 448 lies within
    `rel` of an E4M3 rounding boundary round the other way (fp32 softmax on the GPU vs
    the exact one here): per element, sum over such keys of one code step * |v| *
    fp32(s_v / 448). Returns [M][H*Dh]."""
    ds = np.float64(np.float32(s_q) * np.float32(s_k))
    dv = np.float64(np.float32(s_v) / np.float32(448.0))
    out = np.zeros((qc.shape[0], H * Dh))
    for h in range(H):
        g = (h * Hkv) // H
        keys = np.concatenate([kpre_c[:, g, :], kc[:, g * Dh:(g + 1) * Dh]], axis=0)
        vals = np.concatenate([vpre_c[:, g, :], vc[:, g * Dh:(g + 1) * Dh]], axis=0)
        x = O.softmax((qc[:, h * Dh:(h + 1) * Dh] @ keys.T) * ds / np.sqrt(Dh)) * 448.0
        hi = np.clip(np.searchsorted(_E4M3_POS, x), 1, _E4M3_POS.size - 1)
        g0, g1 = _E4M3_POS[hi - 1], _E4M3_POS[hi]
        near = np.abs(x - (g0 + g1) / 2) <= rel * np.maximum(x, 1e-30)
        out[:, h * Dh:(h + 1) * Dh] = (near * (g1 - g0)) @ np.abs(vals) * dv
    return out


def check_layer_stages(cfg, W, mods, r, sl, kp_l, vp_l, prefix8_l, where, attn_max_frac=1e-3,
                       attn_abs_tol=2.0 ** -7):
    """Teacher-forced checks of one layer-step's record r: every stage recomputed by the
    oracle from the record's own inputs. W: the layer's prepared weights; mods: its
    (sc1, sh1, g1, sc2, sh2, g2) at this step; sl: its activation scales ([4], or [7]
    with FP8 attention; ignored for bf16); kp_l, vp_l: its prefix rows; prefix8_l: their
    E4M3 codes (FP8 attention only). Returns (inc, x_res): the MLP branch's increment
    and x_mid + inc, which the caller checks against the layer-step's output."""
    fmt = cfg.act_fmt
    attn8 = getattr(cfg, "attn_fmt", "bf16") == "fp8"
    H, Dh, F = cfg.H, cfg.Dh, cfg.F

    def s_act(i):
        return float(sl[i]) if fmt in ("fp8", "nvfp4") else 1.0

    def dq(i, w):   # dequantisation factor fp32(s_a * s_w) the epilogues apply
        return np.float64(np.float32(s_act(i)) * np.float32(w.scale))

    sc1, sh1, g1, sc2, sh2, g2 = mods
    check_codes(r["q"], O.quant_codes(O.ada_norm(r["x_in"], sc1, sh1, cfg.eps), s_act(0), fmt),
                where + " pre-attention quantise", fmt)
    qkv = r["y_qkv"]
    exact = (r["q"] @ W["qkv"].codes.T) * dq(0, W["qkv"])
    nq, nk = H * Dh, cfg.Hkv * Dh
    if attn8:
        # E4M3 Q | K | V codes with their static scales, from the exact product
        s3 = [s_act(O.SITE_Q), s_act(O.SITE_K), s_act(O.SITE_V)]
        for (a, b), sx, nm in zip(((0, nq), (nq, nq + nk), (nq + nk, exact.shape[1])), s3, "QKV"):
            check_codes(qkv[:, a:b], O.quant_codes(exact[:, a:b], sx, "fp8"), where + f" QKV GEMM ({nm} codes)")
        # the attention stage's input is exactly the recorded codes and the prefix copy
        args = (qkv[:, :nq], qkv[:, nq:nq + nk], qkv[:, nq + nk:], prefix8_l[0], prefix8_l[1], H, cfg.Hkv, Dh, *s3)
        Oref = O.attention_fp8(*args)
        # probability codes at a rounding boundary may round either way
        extra = fp8_attention_allowance(*args) / s_act(1)
    else:
        extra = 0.0
        # QKV: the GEMM epilogue emits bf16(sum * dequant); within one bf16 rounding
        # of the exact dequantised product
        assert np.all(np.abs(qkv - exact) <= 2.0 ** -8 * np.abs(exact) +
                      1e-5 * np.sqrt(np.mean(exact ** 2))), where + " QKV GEMM"
        # the attention stage's input is exactly the recorded bf16 Q | K | V
        Oref = O.attention(qkv[:, :nq], qkv[:, nq:nq + nk], qkv[:, nq + nk:], kp_l, vp_l, H, cfg.Hkv, Dh)
    # attention rounds its probabilities (bf16, or E4M3 with 3 mantissa bits): a
    # near-tie probability rounding either way moves a row of O by a fraction of
    # P * |V|, so its allowance is abs_tol * RMS
    check_codes(r["attn_out"], O.quant_codes(Oref, s_act(1), fmt), where + " attention", fmt,
                max_frac=attn_max_frac, abs_tol=attn_abs_tol, extra=extra)
    # the O GEMM: its partial planes when recorded, then the gated residual (the
    # increment is compared, so the tolerance is relative to the branch itself)
    yo_ref = r["attn_out"] @ W["o"].codes.T
    if r["y_o"].shape[0]:
        check_close(r["y_o"].sum(0), yo_ref, where + " O GEMM")
    check_increment(r["x_mid"], r["x_in"], g1 * yo_ref * dq(1, W["o"]), where + " O GEMM + attention residual")
    check_codes(r["q2"], O.quant_codes(O.ada_norm(r["x_mid"], sc2, sh2, cfg.eps), s_act(2), fmt),
                where + " pre-MLP quantise", fmt)
    # gate|up GEMM with GeGLU + quantise in its epilogue
    gu = (r["q2"] @ W["gu"].codes.T) * dq(2, W["gu"])
    check_codes(r["geglu_out"], O.quant_codes(O.gelu_tanh(gu[:, :F]) * gu[:, F:], s_act(3), fmt),
                where + " gate|up GEMM + GeGLU", fmt)
    yd_ref = r["geglu_out"] @ W["d"].codes.T
    if r["y_d"].shape[0]:
        check_close(r["y_d"].sum(0), yd_ref, where + " down GEMM")
    inc = g2 * yd_ref * dq(3, W["d"])
    return inc, r["x_mid"] + inc


def check_step_end(model, k, r, x_res, a_prev, dt, next_head, where):
    """The last layer of step k: the final AdaRMSNorm, W_out and the Euler update from
    a_prev, then the next step's head (next_head) or the residual itself."""
    fin = model.final
    scf, shf = model.mods[k][1]
    v = (O.ada_norm(x_res, scf, shf, model.cfg.eps) * fin["gamma_f"]) @ fin["w_out"].T + fin["b_out"]
    check_close(r["actions"], a_prev + dt * v, where + " Euler update")
    if next_head:
        check_close(r["x_out"], r["actions"].astype(np.float64) @ fin["w_in"].T + fin["b_in"], where + " next step head")
    else:
        check_close(r["x_out"], x_res, where + " MLP residual")


def check_decision_stages(cfg, model, recs, noise, kp, vp, scales, attn_max_frac=1e-3, attn_abs_tol=2.0 ** -7,
                          mod_rows=None, dt=None):
    """recs[k][l] as parse_trace returns them; scales [L][4] ([L][7] with FP8
    attention; ignored for bf16). mod_rows: the modulation row of each recorded step
    (default 0 .. S-1); dt: the Euler step (default -1/S). The one-step warm start
    is mod_rows=[S], dt=-warm_t from its mixed input a_tau as `noise`."""
    attn8 = getattr(cfg, "attn_fmt", "bf16") == "fp8"
    prefix8 = prefix_codes(kp, vp, scales) if attn8 else None
    L, S = cfg.L, cfg.S
    fin = model.final
    kp, vp = np.asarray(kp, np.float64), np.asarray(vp, np.float64)
    rows = list(range(S)) if mod_rows is None else list(mod_rows)
    dt = -1.0 / S if dt is None else dt
    a_prev = np.asarray(noise, np.float64)
    check_close(recs[0][0]["x_in"], a_prev @ fin["w_in"].T + fin["b_in"], "step head x")
    for i, k in enumerate(rows):
        for l in range(L):
            r = recs[i][l]
            where = f"step {k} layer {l}"
            inc, x_res = check_layer_stages(cfg, model.w[l], model.mods[k][0][l], r,
                                            scales[l] if scales is not None else None, kp[l], vp[l],
                                            prefix8[l] if attn8 else None, where, attn_max_frac, attn_abs_tol)
            if l < L - 1:
                check_increment(r["x_out"], r["x_mid"], inc, where + " down GEMM + MLP residual")
                continue
            check_step_end(model, k, r, x_res, a_prev, dt, i < len(rows) - 1, where)
            a_prev = r["actions"].astype(np.float64)
    return recs[len(rows) - 1][L - 1]["actions"]
