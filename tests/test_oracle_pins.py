"""Pins for the oracle's model arithmetic (CPU only).

Each check ties the oracle to something other than itself: a closed form
(RMSNorm of constant / one-hot rows, the gamma-fold identity, the K-split
identity, Euler with a constant velocity), an invariant (softmax rows, gate = 0
leaves the residual unchanged), special cases (Q = 0, one key, a dominant key,
GQA grouping), an error bound (E4M3 relative error), or a brute-force scalar
restatement on tiny shapes.
"""
import math

import numpy as np
import pytest

import fm_synth
from oracle import codecs as C
from oracle import model as O


def tiny_cfg(**kw):
    base = dict(name="tiny", L=2, S=2, M=3, d=32, H=2, Hkv=1, Dh=16, F=64, P=4, A=4,
                weight_fmt="fp8", act_fmt="fp8", seed=7)
    base.update(kw)
    return fm_synth.Config(**base)


def tiny_model(cfg):
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    conds = fm_synth.step_conds(cfg) if cfg.cond == "given" else None
    return O.Model(cfg, layers, fm_synth.final_weights(cfg), conds), layers


# ---------------------------------------------------------------- RMSNorm / AdaRMSNorm

def test_rms_norm_constant_row():
    for c in [0.5, -3.0, 1e-2]:
        x = np.full((1, 64), c)
        np.testing.assert_allclose(O.rms_norm(x, 1e-6), c / math.sqrt(c * c + 1e-6), rtol=1e-14)


def test_rms_norm_one_hot():
    d, a, eps = 128, 2.5, 1e-6
    x = np.zeros((1, d))
    x[0, 17] = a
    y = O.rms_norm(x, eps)
    assert y[0, 17] == pytest.approx(a / math.sqrt(a * a / d + eps), rel=1e-14)
    assert np.count_nonzero(y) == 1


def test_ada_norm_uses_one_plus_scale():
    x = np.full((1, 8), 2.0)
    xh = 2.0 / math.sqrt(4.0 + 1e-6)
    y = O.ada_norm(x, np.full(8, 0.5), np.full(8, -0.25), 1e-6)
    np.testing.assert_allclose(y, xh * 1.5 - 0.25, rtol=1e-14)
    y0 = O.ada_norm(x, np.zeros(8), np.zeros(8), 1e-6)
    np.testing.assert_allclose(y0, O.rms_norm(x, 1e-6), rtol=0)


# ---------------------------------------------------------------- fold / quant / GEMM

def test_gamma_fold_identity():
    """(x_hat * gamma) W^T == x_hat (W diag(gamma))^T  (blog post, fold equation)."""
    rng = np.random.default_rng(3)
    xh = rng.standard_normal((5, 64))
    w = rng.standard_normal((48, 64)).astype(np.float32) * 0.02
    g = (1 + 0.1 * rng.standard_normal(64)).astype(np.float32)
    lhs = (xh * g) @ w.astype(np.float64).T
    rhs = xh @ O.fold_gamma(w, g).T
    # W' is stored in fp32: each element carries at most 2^-24 relative rounding
    bound = (np.abs(xh) @ np.abs(w.astype(np.float64) * g).T) * 2.0 ** -24 * 1.0001
    assert np.all(np.abs(rhs - lhs) <= bound)
    # exact on small integers (every product and sum representable)
    xi = rng.integers(-3, 4, (4, 16)).astype(np.float64)
    wi = rng.integers(-3, 4, (8, 16)).astype(np.float32)
    gi = rng.integers(-2, 3, 16).astype(np.float32)
    np.testing.assert_array_equal(xi @ O.fold_gamma(wi, gi).T, (xi * gi) @ wi.astype(np.float64).T)


def test_fp8_weight_prep_scale_and_bound():
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((64, 128)) * 0.02).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(128)).astype(np.float32)
    pw = O.prep_weight(w, g, "fp8")
    wf = O.fold_gamma(w, g)
    assert pw.scale == pytest.approx(np.max(np.abs(wf)) / 448.0, rel=1e-7)
    assert np.max(np.abs(pw.codes)) == 448.0
    deq = pw.codes * pw.scale
    # E4M3 RNE: relative error <= 2^-4 for normal codes, absolute <= 2^-10 * s in the subnormal range
    err = np.abs(deq - wf)
    bound = np.maximum(np.abs(wf) * 2.0 ** -4, 2.0 ** -10 * pw.scale) * (1 + 1e-6)
    assert np.all(err <= bound)
    assert np.all(np.isin(pw.codes, C.e4m3_decode_code(np.arange(256))))


def test_zero_weight_scale_is_one():
    pw = O.prep_weight(np.zeros((16, 32), np.float32), None, "fp8")
    assert pw.scale == 1.0 and not np.any(pw.codes)


def test_nvfp4_prep():
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((32, 64)) * 0.02).astype(np.float32)
    pw = O.prep_weight(w, None, "nvfp4")
    e2m1_grid = C.e2m1_decode_code(np.arange(16))
    bs = pw.block_scales
    assert bs.shape == (32, 4)
    elems = pw.codes.reshape(32, 4, 16) / np.where(bs > 0, bs, 1)[..., None]
    assert np.all(np.isin(elems, e2m1_grid))
    assert np.all(np.isin(bs, C.e4m3_decode_code(np.arange(128))))
    np.testing.assert_array_equal(C.bf16(pw.codes), pw.codes)   # e*bs exact in bf16
    deq = pw.codes * pw.scale
    amax_b = np.max(np.abs(w.reshape(32, 4, 16)), axis=-1, keepdims=True)
    # element error <= half an E2M1 step at the top binade (1.0 of 6) of the block scale,
    # plus the block-scale rounding (2^-4 relative)
    err = np.abs(deq.reshape(32, 4, 16) - w.reshape(32, 4, 16))
    assert np.all(err <= amax_b * (1.0 / 6.0 + 2.0 ** -4) * 1.01)
    assert pw.scale == pytest.approx(np.max(np.abs(w)) / 2688.0, rel=1e-7)


def test_ksplit_identity_integer_exact():
    """C = sum_j A_j W_j (blog post, "Small-M GEMM"), bit-exact on small integers."""
    case = fm_synth.gemm_case(10, 1024, 256, integer=True)
    pw = O.PreparedWeight(case["w"].astype(np.float64), 1.0, "fp8")
    full = case["a"].astype(np.float64) @ pw.codes.T
    for s in [1, 2, 4, 8, 16]:
        parts = O.gemm_ksplit(case["a"], pw, s)
        assert parts.shape == (s, 10, 256)
        np.testing.assert_array_equal(parts.sum(axis=0), full)
        # every partial and every running fp32 sum is exact: |sum| <= 9 * K < 2^24
        acc = np.zeros_like(full, dtype=np.float32)
        for j in range(s):
            acc = acc + parts[j].astype(np.float32)
        np.testing.assert_array_equal(acc.astype(np.float64), full)


def test_gemm_dequant_error_bound():
    rng = np.random.default_rng(6)
    a = rng.standard_normal((8, 256))
    w = (rng.standard_normal((64, 256)) * 0.02).astype(np.float32)
    s_a = float(np.float32(np.max(np.abs(a)) / 448))
    qa = O.quant_codes(a, s_a, "fp8")
    pw = O.prep_weight(w, None, "fp8")
    y = O.gemm(qa, s_a, pw)
    exact = a @ w.astype(np.float64).T
    bound = (np.abs(a) @ np.abs(w.astype(np.float64)).T) * (2 * 2.0 ** -4 + 2.0 ** -8) \
        + 256 * 2.0 ** -9 * s_a * np.max(np.abs(w)) * 2
    assert np.all(np.abs(y - exact) <= bound)


# ---------------------------------------------------------------- softmax / attention

def test_softmax_rows_sum_to_one():
    s = np.random.default_rng(7).standard_normal((20, 300)) * 5
    np.testing.assert_allclose(O.softmax(s).sum(-1), 1.0, atol=1e-12)


def _attn_inputs(M=3, P=5, H=2, Hkv=1, Dh=16, seed=8):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((M, H * Dh)), rng.standard_normal((M, Hkv * Dh)),
            rng.standard_normal((M, Hkv * Dh)), rng.standard_normal((P, Hkv, Dh)),
            rng.standard_normal((P, Hkv, Dh)))


def test_attention_zero_query_is_mean_of_values():
    q, kc, vc, kp, vp = _attn_inputs()
    q[:] = 0
    o = O.attention(q, kc, vc, kp, vp, 2, 1, 16, round_p=False)
    vals = np.concatenate([vp[:, 0, :], vc], axis=0)
    for h in range(2):
        np.testing.assert_allclose(o[:, h * 16:(h + 1) * 16], np.tile(vals.mean(0), (3, 1)), rtol=1e-12)


def test_attention_single_key():
    q, kc, vc, kp, vp = _attn_inputs(M=1, P=0)
    o = O.attention(q, kc, vc, kp, vp, 2, 1, 16)
    np.testing.assert_allclose(o, np.tile(vc, (1, 2)), rtol=0)


def test_attention_dominant_key():
    q, kc, vc, kp, vp = _attn_inputs(M=2, P=6)
    kp[3, 0, :] = q[0, :16] / np.linalg.norm(q[0, :16]) * 400.0   # score gap >> 50 for head 0, row 0
    o = O.attention(q, kc, vc, kp, vp, 2, 1, 16, round_p=False)
    np.testing.assert_allclose(o[0, :16], vp[3, 0], rtol=1e-9, atol=1e-9)


def test_attention_gqa_grouping():
    """Heads h use KV group floor(h*Hkv/H): with H=4, Hkv=2, heads 0,1 -> group 0."""
    M, P, Dh = 2, 3, 8
    rng = np.random.default_rng(9)
    q = rng.standard_normal((M, 4 * Dh))
    kc, kp = rng.standard_normal((M, 2 * Dh)), rng.standard_normal((P, 2, Dh))
    vc = np.concatenate([np.full((M, Dh), 1.0), np.full((M, Dh), 5.0)], axis=1)
    vp = np.stack([np.full((P, Dh), 1.0), np.full((P, Dh), 5.0)], axis=1)
    o = O.attention(q, kc, vc, kp, vp, 4, 2, Dh)
    np.testing.assert_allclose(o[:, :2 * Dh], 1.0, rtol=1e-2)
    np.testing.assert_allclose(o[:, 2 * Dh:], 5.0, rtol=1e-2)


# ---------------------------------------------------------------- GELU / embedding

def test_gelu_tanh_close_to_erf_form():
    g = np.linspace(-8, 8, 4001)
    erf_form = 0.5 * g * (1 + np.vectorize(math.erf)(g / math.sqrt(2)))
    assert np.max(np.abs(O.gelu_tanh(g) - erf_form)) < 1e-3
    assert O.gelu_tanh(np.array([0.0]))[0] == 0.0
    assert O.gelu_tanh(np.array([20.0]))[0] == pytest.approx(20.0)
    assert abs(O.gelu_tanh(np.array([-20.0]))[0]) < 1e-12


def test_time_embedding_closed_form():
    e0 = O.time_embedding(0.0, 64)
    np.testing.assert_array_equal(e0[:32], 0.0)
    np.testing.assert_array_equal(e0[32:], 1.0)
    e = O.time_embedding(1e-3, 64)           # quarter period of the shortest period 4e-3
    assert e[0] == pytest.approx(1.0, abs=1e-12)
    assert e[32] == pytest.approx(0.0, abs=1e-12)
    # the longest period is 4.0: at t = 1 its phase is pi/2
    e1 = O.time_embedding(1.0, 64)
    assert e1[31] == pytest.approx(1.0, abs=1e-12)


# ---------------------------------------------------------------- layer / loop invariants

def _zero_gates(layers, d):
    for lw in layers:
        lw["w_mod"][2 * d:3 * d] = 0
        lw["w_mod"][5 * d:6 * d] = 0


def test_zero_gates_leave_residual_unchanged():
    cfg = tiny_cfg(cond="given")
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    _zero_gates(layers, cfg.d)
    model = O.Model(cfg, layers, fm_synth.final_weights(cfg), fm_synth.step_conds(cfg))
    kp, vp = fm_synth.prefix_kv(cfg)
    x = fm_synth.layer_input(cfg)
    scales = fm_synth.default_act_scales(cfg)
    x_out, _, _ = O.single_layer(model, x, kp, vp, scales)
    np.testing.assert_array_equal(x_out, x.astype(np.float64))


def test_euler_zero_network_gives_noise_minus_bias():
    """All layer weights 0 and W_out = 0: v = b_out at every step, so a_0 = noise - b_out."""
    cfg = tiny_cfg()
    layers = [{k: np.zeros_like(v) for k, v in fm_synth.layer_weights(cfg, l).items()}
              for l in range(cfg.L)]
    fin = fm_synth.final_weights(cfg)
    fin["w_out"][:] = 0
    model = O.Model(cfg, layers, fin)
    kp, vp = fm_synth.prefix_kv(cfg)
    nz = fm_synth.noise(cfg)
    a = O.decode(model, nz, kp, vp, fm_synth.default_act_scales(cfg))
    np.testing.assert_allclose(a, nz - fin["b_out"].astype(np.float64), rtol=0, atol=1e-15)


def test_euler_velocity_independent_of_state():
    """W_in = 0: the velocity depends on t only, so a_0 = noise - (1/S) sum_k v(t_k)."""
    cfg = tiny_cfg(S=3)
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    fin = fm_synth.final_weights(cfg)
    fin["w_in"][:] = 0
    model = O.Model(cfg, layers, fin)
    kp, vp = fm_synth.prefix_kv(cfg)
    sc = fm_synth.default_act_scales(cfg)
    nz = fm_synth.noise(cfg)
    zero = np.zeros_like(nz, dtype=np.float64)
    vs = [(O.euler_step(model, k, zero, kp, vp, sc) - zero) / (-1.0 / cfg.S) for k in range(cfg.S)]
    expect = nz - sum(vs) / cfg.S
    np.testing.assert_allclose(O.decode(model, nz, kp, vp, sc), expect, rtol=1e-12, atol=1e-12)
    # and the velocities really differ between steps (the embedding reaches the network)
    assert not np.allclose(vs[0], vs[1])


def test_calibration_hits_448():
    cfg = tiny_cfg()
    model, _ = tiny_model(cfg)
    kp, vp = fm_synth.prefix_kv(cfg)
    sc = O.calibrate(model, fm_synth.noise(cfg, 1000), kp, vp, fm_synth.default_act_scales(cfg))
    amax = np.zeros((cfg.L, 4))
    O.decode(model, fm_synth.noise(cfg, 1000), kp, vp, sc, amax)
    # with the calibrated scales the largest pre-quant value maps to ~448
    assert np.all(sc > 0)
    ratio = amax / sc.astype(np.float64)
    assert np.all(ratio > 300) and np.all(ratio < 800)


# ---------------------------------------------------------------- brute-force scalar restatement

def _scalar_step(cfg, layers, fin, k, a, kp, vp, sc):
    """One Euler step written with scalar loops, independent of the vectorised oracle."""
    d, H, Hkv, Dh, F, M, A = cfg.d, cfg.H, cfg.Hkv, cfg.Dh, cfg.F, cfg.M, cfg.A
    t = 1.0 - k / cfg.S
    half = d // 2
    cond = [0.0] * d
    for i in range(half):
        p = 4e-3 * (4.0 / 4e-3) ** (i / (half - 1))
        cond[i] = math.sin(2 * math.pi * t / p)
        cond[half + i] = math.cos(2 * math.pi * t / p)

    def linear_mod(w, b, n_out):
        return [float(np.float32(sum(cond[i] * float(w[o][i]) for i in range(d)) + float(b[o])))
                for o in range(n_out)]

    def norm_row(row, scale, shift):
        ms = sum(v * v for v in row) / len(row)
        r = 1.0 / math.sqrt(ms + cfg.eps)
        return [row[i] * r * (1 + scale[i]) + shift[i] for i in range(len(row))]

    def q8(v, s):
        return float(C.e4m3(np.array([v * float(np.float32(1) / np.float32(s))]))[0])

    def prep(w, gamma):
        n, kk = len(w), len(w[0])
        wf = [[float(np.float32(float(w[i][j]) * (float(gamma[j]) if gamma is not None else 1.0)))
               for j in range(kk)] for i in range(n)]
        amax = max(abs(v) for r in wf for v in r)
        s = float(np.float32(amax) / np.float32(448))
        r = float(np.float32(1) / np.float32(s))
        codes = [[float(C.e4m3(np.array([float(np.float32(v * r))]))[0]) for v in row] for row in wf]
        return codes, s

    def mm(xq, sa, wc):
        codes, sw = wc
        comb = float(np.float32(sa) * np.float32(sw))
        return [[sum(xq[m][j] * codes[n][j] for j in range(len(xq[m]))) * comb
                 for n in range(len(codes))] for m in range(len(xq))]

    bf = lambda v: float(C.bf16(np.array([v]))[0])
    x = [[sum(float(a[m][j]) * float(fin["w_in"][n][j]) for j in range(A)) + float(fin["b_in"][n])
          for n in range(d)] for m in range(M)]
    for l, lw in enumerate(layers):
        mod = linear_mod(lw["w_mod"], lw["b_mod"], 6 * d)
        sc1, sh1, g1, sc2, sh2, g2 = [mod[i * d:(i + 1) * d] for i in range(6)]
        wq, wo = prep(lw["w_qkv"], lw["gamma1"]), prep(lw["w_o"], None)
        wgu, wd = prep(lw["w_gu"], lw["gamma2"]), prep(lw["w_d"], None)
        q = [[q8(v, sc[l][0]) for v in norm_row(x[m], sc1, sh1)] for m in range(M)]
        qkv = mm(q, sc[l][0], wq)
        Q = [[bf(v) for v in r[:H * Dh]] for r in qkv]
        Kc = [[bf(v) for v in r[H * Dh:(H + Hkv) * Dh]] for r in qkv]
        Vc = [[bf(v) for v in r[(H + Hkv) * Dh:]] for r in qkv]
        att = [[0.0] * (H * Dh) for _ in range(M)]
        for h in range(H):
            g = h * Hkv // H
            keys = [list(kp[l][p][g]) for p in range(cfg.P)] + [Kc[m][g * Dh:(g + 1) * Dh] for m in range(M)]
            vals = [list(vp[l][p][g]) for p in range(cfg.P)] + [Vc[m][g * Dh:(g + 1) * Dh] for m in range(M)]
            for m in range(M):
                sco = [sum(Q[m][h * Dh + e] * float(kk[e]) for e in range(Dh)) / math.sqrt(Dh) for kk in keys]
                mx = max(sco)
                ex = [math.exp(s - mx) for s in sco]
                tot = sum(ex)
                pr = [bf(e / tot) for e in ex]
                for e in range(Dh):
                    att[m][h * Dh + e] = sum(pr[j] * float(vals[j][e]) for j in range(len(keys)))
        o = mm([[q8(v, sc[l][1]) for v in r] for r in att], sc[l][1], wo)
        x = [[x[m][n] + g1[n] * o[m][n] for n in range(d)] for m in range(M)]
        q2 = [[q8(v, sc[l][2]) for v in norm_row(x[m], sc2, sh2)] for m in range(M)]
        gu = mm(q2, sc[l][2], wgu)
        mid = []
        for m in range(M):
            row = []
            for f in range(F):
                gg, uu = gu[m][f], gu[m][F + f]
                row.append(0.5 * gg * (1 + math.tanh(math.sqrt(2 / math.pi) * (gg + 0.044715 * gg ** 3))) * uu)
            mid.append(row)
        dn = mm([[q8(v, sc[l][3]) for v in r] for r in mid], sc[l][3], wd)
        x = [[x[m][n] + g2[n] * dn[m][n] for n in range(d)] for m in range(M)]
    condf = cond
    modf = [float(np.float32(sum(condf[i] * float(fin["w_mod_f"][o][i]) for i in range(d)) + float(fin["b_mod_f"][o])))
            for o in range(2 * d)]
    out = []
    for m in range(M):
        hf = norm_row(x[m], modf[:d], modf[d:])
        hf = [hf[i] * float(fin["gamma_f"][i]) for i in range(d)]
        v = [sum(hf[i] * float(fin["w_out"][j][i]) for i in range(d)) + float(fin["b_out"][j]) for j in range(A)]
        out.append([float(a[m][j]) - v[j] / cfg.S for j in range(A)])
    return np.array(out)


def test_brute_force_scalar_step_matches_oracle():
    cfg = tiny_cfg(L=2, S=2, M=2, d=32, H=4, Hkv=2, Dh=8, F=32, P=3, A=3)
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    fin = fm_synth.final_weights(cfg)
    model = O.Model(cfg, layers, fin)
    kp, vp = fm_synth.prefix_kv(cfg)
    sc = fm_synth.default_act_scales(cfg) * np.float32(0.5)
    a0 = fm_synth.noise(cfg)
    ref = O.euler_step(model, 1, a0.astype(np.float64), kp, vp, sc)
    brute = _scalar_step(cfg, layers, fin, 1, a0, kp, vp, sc)
    np.testing.assert_allclose(brute, ref, rtol=1e-9, atol=1e-11)


# ---------------------------------------------------------------- FP8 attention mode

def _e4m3_grid_values(rng, shape):
    grid = C.e4m3_decode_code(np.arange(0, 0x70))   # finite positive codes up to 240 and their signs
    vals = rng.choice(grid, size=shape)
    return vals * rng.choice([-1.0, 1.0], size=shape)


def test_attention_fp8_brute_force_tiny():
    """Scalar loops over a tiny case (2 query heads sharing 1 KV head, Dh = 4, 3 prefix
    keys + 2 chunk keys): scores scaled by fp32(s_q s_k)/sqrt(Dh), exact softmax,
    probabilities coded E4M3(P * 448), output scaled by fp32(s_v / 448)."""
    rng = np.random.default_rng(11)
    H, Hkv, Dh, M, P = 2, 1, 4, 2, 3
    qc = _e4m3_grid_values(rng, (M, H * Dh)) / 64
    kc = _e4m3_grid_values(rng, (M, Hkv * Dh)) / 64
    vc = _e4m3_grid_values(rng, (M, Hkv * Dh)) / 64
    kp = _e4m3_grid_values(rng, (P, Hkv, Dh)) / 64
    vp = _e4m3_grid_values(rng, (P, Hkv, Dh)) / 64
    s_q, s_k, s_v = 0.03, 0.05, 0.07
    got = O.attention_fp8(qc, kc, vc, kp, vp, H, Hkv, Dh, s_q, s_k, s_v)
    ds = float(np.float32(s_q) * np.float32(s_k))
    dv = float(np.float32(s_v) / np.float32(448.0))
    for m in range(M):
        for h in range(H):
            keys = [list(kp[j, 0]) for j in range(P)] + [list(kc[j, 0:Dh]) for j in range(M)]
            vals = [list(vp[j, 0]) for j in range(P)] + [list(vc[j, 0:Dh]) for j in range(M)]
            sc = []
            for kk in keys:
                acc = 0.0
                for e in range(Dh):
                    acc += qc[m, h * Dh + e] * kk[e]
                sc.append(acc * ds / math.sqrt(Dh))
            mx = max(sc)
            ex = [math.exp(x - mx) for x in sc]
            tot = sum(ex)
            pcode = [float(C.e4m3(np.array([x / tot * 448.0]))[0]) for x in ex]
            for e in range(Dh):
                ref = sum(pcode[j] * vals[j][e] for j in range(len(vals))) * dv
                assert got[m, h * Dh + e] == pytest.approx(ref, rel=1e-12, abs=1e-15)


def test_attention_fp8_single_key_returns_scaled_value():
    """One key: P = 1 is coded exactly (E4M3(448) = 448), so O = v * 448 * (s_v / 448) =
    v * s_v exactly when s_v / 448 is a power of two (s_v = 1.75: 1.75 / 448 = 2^-8)."""
    rng = np.random.default_rng(12)
    Dh = 8
    qc = _e4m3_grid_values(rng, (1, Dh))
    kc = _e4m3_grid_values(rng, (1, Dh))
    vc = _e4m3_grid_values(rng, (1, Dh))
    empty = np.zeros((0, 1, Dh))
    out = O.attention_fp8(qc, kc, vc, empty, empty, 1, 1, Dh, 0.5, 0.25, 1.75)
    np.testing.assert_array_equal(out, vc * 1.75)


def test_attention_fp8_uniform_scores():
    """Equal keys: P = 1/7 for 7 keys, coded E4M3(448 / 7) = 64 exactly, so
    O = 64 * sum(v) * (1.75 / 448) = sum(v) / 4."""
    rng = np.random.default_rng(13)
    Dh = 8
    k = _e4m3_grid_values(rng, (Dh,))
    kp = np.tile(k, (6, 1))[:, None, :]
    kc = k[None, :]
    vp = _e4m3_grid_values(rng, (6, 1, Dh))
    vc = _e4m3_grid_values(rng, (1, Dh))
    qc = _e4m3_grid_values(rng, (1, Dh))
    out = O.attention_fp8(qc, kc, vc, kp, vp, 1, 1, Dh, 0.125, 0.5, 1.75)
    np.testing.assert_array_equal(out[0], (vp[:, 0, :].sum(axis=0) + vc[0]) / 4)
