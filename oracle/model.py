"""FP64 CPU oracle of the flow-matching action-decoder hot path.

TEST INFRASTRUCTURE ONLY: the tests, the package's smoke check and the
benchmark's CPU-baseline leg may use this module; the GPU library never does.
It shares no code with the CUDA path; the only thing both sides use is the
seeded input generator in ``fm_synth``, which holds no arithmetic of the method.

What it computes follows the FlashRT-PAI pages (the blog post "Embodied
inference acceleration: first ask how old the observation is", its sections
"CUDA Graph vs graph simplification" (RMSNorm and the gamma fold), "Static
quantisation changes the work between two GEMMs" (static activation scales,
gated residual + AdaRMSNorm + FP8 convert, next layer's condition parameters),
"Small-M GEMM" (the K-split identity) and "Few-step denoise"; and the news
article's section "It optimises the relay" (prefix reuse, refresh of the
image-dependent part)). The layer form (attention over a prefix KV cache, GeGLU
MLP, 10 Euler steps) is the workload definition's. Rounding is emulated at
exactly the points where the GPU path rounds (E4M3 codes, bf16 operands, fp32
scales); everything else is float64.

Readings where the pages are silent (each also listed in the design notes):
  eps = 1e-6; gamma multiplies the modulated normalised input, so it folds
  exactly into W; gate is a raw linear output; modulation = cond . W_mod^T +
  b_mod, stored fp32; sinusoidal t-embedding with periods 4e-3 .. 4; keys =
  prefix + the chunk's own K/V, no mask, scale 1/sqrt(Dh), GQA group
  g = floor(h * Hkv / H); no positional rotation; tanh GELU; E4M3 RNE with
  saturation, multiply by the fp32 reciprocal of the static scale, dequant by
  fp32(s_a * s_w); weight scale amax/448 (1 if the matrix is all zero); noise at
  t = 1, t_k = 1 - k/S, Euler step dt = -1/S; adaptive final norm (no gate)
  with gamma_f, then W_out; attention probabilities rounded to bf16 before P.V.
  FP8 attention mode: Q, K, V (chunk and prefix) quantised with static per-layer
  scales (fp32 reciprocal multiply, E4M3 RNE with saturation), scores dequantised
  by fp32(s_q * s_k), probabilities P in [0, 1] stored as E4M3(P * 448) (static
  scale 1/448), output dequantised by fp32(s_v / 448).
"""
from __future__ import annotations

import math

import numpy as np

from . import codecs as C

F32 = np.float32

# quant points per layer (index into the [L][4] activation-scale table; the FP8
# attention mode adds Q, K and V as columns 4-6 of an [L][7] table)
SITE_ATTN_IN, SITE_ATTN_OUT, SITE_MLP_IN, SITE_GEGLU = 0, 1, 2, 3
SITE_Q, SITE_K, SITE_V = 4, 5, 6
P_CODE_SCALE = 448.0   # E4M3 probabilities: code = E4M3(P * 448), value = code / 448


# ---------------------------------------------------------------- primitives

def rms_norm(x: np.ndarray, eps: float) -> np.ndarray:
    """x_hat = x / sqrt(mean(x^2) + eps), row-wise (blog post, RMSNorm equation)."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)


def ada_norm(x, scale, shift, eps):
    """AdaRMSNorm: x_hat * (1 + scale) + shift, scale/shift generated from the condition."""
    return rms_norm(x, eps) * (1.0 + np.asarray(scale, np.float64)) + np.asarray(shift, np.float64)


def recip32(s) -> np.float64:
    """fp32 reciprocal of a static scale, as the GPU multiplies by it."""
    return np.float64(F32(1.0) / F32(s))


def quant_nvfp4_act(h: np.ndarray, ts: float):
    """NVFP4 activation operand for a four-bit (W4A4) GEMM (news article "FlashRT-PAI",
    sections "It optimises the relay" and the four-bit pi0.5 results): the tensor scale
    ts is static (calibrated like the FP8 scales, amax / (448 * 6)); the block scales
    are the activation's own, one per 16 consecutive K elements of a row:
    bs = E4M3_RNE_sat(fp32(amax_b / fp32(6 ts))), e = E2M1_RNE_sat(fp32(h / fp32(bs ts))),
    0 where bs ts = 0. Returns (e * bs as values [M][K], bs [M][K/16])."""
    h = np.asarray(h, np.float64)
    m, k = h.shape
    blocks = h.reshape(m, k // 16, 16)
    amax_b = np.max(np.abs(blocks), axis=-1)
    six_ts = np.float64(F32(6.0) * F32(ts))
    bs = C.e4m3(C.fp32(amax_b / six_ts))
    denom = C.fp32(bs * np.float64(F32(ts)))
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.where(denom[..., None] > 0,
                     C.e2m1(C.fp32(blocks / np.where(denom > 0, denom, 1.0)[..., None])), 0.0)
    return (e * bs[..., None]).reshape(m, k), bs


def quant_codes(h: np.ndarray, s: float, fmt: str) -> np.ndarray:
    """Static-scale activation quantisation; returns the operand codes as values.

    fp8: code = E4M3_RNE_sat(h * fp32(1/s)); the GEMM later multiplies by s.
    bf16: code = bf16_RNE(h) (no scale).
    nvfp4: e * bs of quant_nvfp4_act with tensor scale s; the GEMM multiplies by s.
    """
    if fmt == "fp8":
        return C.e4m3(np.asarray(h, np.float64) * recip32(s))
    if fmt == "bf16":
        return C.bf16(h)
    if fmt == "nvfp4":
        return quant_nvfp4_act(h, s)[0]
    raise ValueError(fmt)


def gelu_tanh(g: np.ndarray) -> np.ndarray:
    g = np.asarray(g, np.float64)
    return 0.5 * g * (1.0 + np.tanh(math.sqrt(2.0 / math.pi) * (g + 0.044715 * g ** 3)))


def softmax(s: np.ndarray) -> np.ndarray:
    s = np.asarray(s, np.float64)
    e = np.exp(s - np.max(s, axis=-1, keepdims=True))
    return e / np.sum(e, axis=-1, keepdims=True)


def time_embedding(t: float, d: int, min_period=4e-3, max_period=4.0) -> np.ndarray:
    """Sinusoidal embedding of the flow time t: [sin(2 pi t / p_i), cos(2 pi t / p_i)],
    p_i geometric from min_period to max_period over i = 0 .. d/2 - 1."""
    half = d // 2
    frac = np.arange(half, dtype=np.float64) / (half - 1)
    period = min_period * (max_period / min_period) ** frac
    arg = 2.0 * math.pi * t / period
    return np.concatenate([np.sin(arg), np.cos(arg)])


# ---------------------------------------------------------------- weight prep

class PreparedWeight:
    """A GEMM weight as the GPU stores it: operand codes (as values) and a scale.

    y = (a_codes @ codes.T) * fp32(s_a * scale).
    """

    def __init__(self, codes: np.ndarray, scale: float, fmt: str, block_scales=None):
        self.codes = codes            # float64 [N][K]
        self.scale = float(scale)
        self.fmt = fmt
        self.block_scales = block_scales


def fold_gamma(w: np.ndarray, gamma) -> np.ndarray:
    """W' = W diag(gamma) in the [out][in] layout: W'[n][k] = W[n][k] * gamma[k],
    rounded to fp32 (the stored precision of the folded weight)."""
    w = np.asarray(w, np.float64)
    if gamma is None:
        return C.fp32(w)
    return C.fp32(w * np.asarray(gamma, np.float64)[None, :])


def prep_weight(w: np.ndarray, gamma, fmt: str) -> PreparedWeight:
    wf = fold_gamma(w, gamma)
    if fmt == "fp8":
        amax = float(np.max(np.abs(wf))) if wf.size else 0.0
        s = float(F32(amax) / F32(448.0)) if amax > 0 else 1.0
        codes = C.e4m3(C.fp32(wf * recip32(s)))
        return PreparedWeight(codes, s, fmt)
    if fmt == "bf16":
        return PreparedWeight(C.bf16(wf), 1.0, fmt)
    if fmt == "nvfp4":
        return _prep_nvfp4(wf)
    raise ValueError(fmt)


def _prep_nvfp4(wf: np.ndarray) -> PreparedWeight:
    """NVFP4: E2M1 elements, one E4M3 scale per 16 consecutive K elements, one fp32
    tensor scale. ts = amax/(448*6); bs = E4M3(amax_b / (6 ts)); e = E2M1(w / (bs ts)).
    The GEMM operand is e*bs (exact in bf16); ts multiplies in the epilogue."""
    n, k = wf.shape
    amax = float(np.max(np.abs(wf)))
    ts = float(F32(amax) / F32(2688.0)) if amax > 0 else 1.0
    blocks = wf.reshape(n, k // 16, 16)
    amax_b = np.max(np.abs(blocks), axis=-1)
    six_ts = np.float64(F32(6.0) * F32(ts))
    bs = C.e4m3(C.fp32(amax_b / six_ts))
    denom = C.fp32(bs * ts)
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.where(denom[..., None] > 0,
                     C.e2m1(C.fp32(blocks / np.where(denom > 0, denom, 1.0)[..., None])), 0.0)
    codes = (e * bs[..., None]).reshape(n, k)
    return PreparedWeight(codes, ts, "nvfp4", block_scales=bs)


def gemm(a_codes: np.ndarray, s_a: float, w: PreparedWeight) -> np.ndarray:
    """Dequantised product: (A_codes W_codes^T) * fp32(s_a * s_w), accumulated exactly."""
    acc = np.asarray(a_codes, np.float64) @ w.codes.T
    return acc * np.float64(F32(s_a) * F32(w.scale))


def gemm_ksplit(a_codes, w: PreparedWeight, s: int) -> np.ndarray:
    """The K-split identity C = sum_j A_j W_j (blog post, "Small-M GEMM"):
    s equal contiguous K slices, partials returned as [s][M][N] (unscaled)."""
    k = a_codes.shape[1]
    ks = k // s
    return np.stack([np.asarray(a_codes[:, j * ks:(j + 1) * ks], np.float64)
                     @ w.codes[:, j * ks:(j + 1) * ks].T for j in range(s)])


# ---------------------------------------------------------------- model pieces

def attention(q, kc, vc, kpre, vpre, H, Hkv, Dh, round_p=True):
    """Chunk queries over [prefix; chunk] keys, no mask, softmax(QK^T/sqrt(Dh)) V.

    q [M][H*Dh], kc/vc [M][Hkv*Dh], kpre/vpre [P][Hkv][Dh]. Returns O [M][H*Dh].
    """
    M = q.shape[0]
    out = np.empty((M, H * Dh), np.float64)
    for h in range(H):
        g = (h * Hkv) // H
        keys = np.concatenate([kpre[:, g, :], kc[:, g * Dh:(g + 1) * Dh]], axis=0)
        vals = np.concatenate([vpre[:, g, :], vc[:, g * Dh:(g + 1) * Dh]], axis=0)
        s = (q[:, h * Dh:(h + 1) * Dh] @ keys.T) / math.sqrt(Dh)
        p = softmax(s)
        if round_p:
            p = C.bf16(p)
        out[:, h * Dh:(h + 1) * Dh] = p @ vals
    return out


def attention_fp8(qc, kc, vc, kpre_c, vpre_c, H, Hkv, Dh, s_q, s_k, s_v):
    """FP8 attention over [prefix; chunk] keys. All operands are E4M3 code values
    (without their static scales): qc [M][H*Dh], kc/vc [M][Hkv*Dh], kpre_c/vpre_c
    [P][Hkv][Dh]. Scores s = (qc . k^T) * fp32(s_q * s_k) / sqrt(Dh); P = softmax(s);
    P codes = E4M3(P * 448); O = (P codes . v) * fp32(s_v / 448). Returns O [M][H*Dh]."""
    M = qc.shape[0]
    ds = np.float64(F32(s_q) * F32(s_k))
    dv = np.float64(F32(s_v) / F32(P_CODE_SCALE))
    out = np.empty((M, H * Dh), np.float64)
    for h in range(H):
        g = (h * Hkv) // H
        keys = np.concatenate([kpre_c[:, g, :], kc[:, g * Dh:(g + 1) * Dh]], axis=0)
        vals = np.concatenate([vpre_c[:, g, :], vc[:, g * Dh:(g + 1) * Dh]], axis=0)
        sc = (qc[:, h * Dh:(h + 1) * Dh] @ keys.T) * ds / math.sqrt(Dh)
        pc = C.e4m3(softmax(sc) * P_CODE_SCALE)
        out[:, h * Dh:(h + 1) * Dh] = (pc @ vals) * dv
    return out


class Model:
    """Prepared weights and the per-step modulation table of one policy."""

    def __init__(self, cfg, layers: list, final: dict, conds=None):
        """layers: list of per-layer raw dicts (fm_synth.layer_weights); final: final_weights.
        conds: [S][d] cond vectors for cond == "given" workloads."""
        self.cfg = cfg
        wf = cfg.weight_fmt
        self.w = []
        self.mod_w = []
        for lw in layers:
            self.w.append({
                "qkv": prep_weight(lw["w_qkv"], lw["gamma1"], wf),
                "o": prep_weight(lw["w_o"], None, wf),
                "gu": prep_weight(lw["w_gu"], lw["gamma2"], wf),
                "d": prep_weight(lw["w_d"], None, wf),
            })
            self.mod_w.append((np.asarray(lw["w_mod"], np.float64), np.asarray(lw["b_mod"], np.float64)))
        self.final = {k: np.asarray(v, np.float64) for k, v in final.items()} if final else None
        self.conds = None if conds is None else np.asarray(conds, np.float64)
        self.mods = [self._mods_for_cond(self.cond(k)) for k in range(cfg.S)]
        # the one-step warm start's modulation (flow time warm_t) is row S
        if getattr(cfg, "warm_t", 0.0) > 0:
            self.mods.append(self.mods_at(warm_time(cfg)))

    def cond(self, k: int) -> np.ndarray:
        cfg = self.cfg
        if cfg.cond == "given":
            return self.conds[k]
        return time_embedding(1.0 - k / cfg.S, cfg.d)

    def mods_at(self, t: float):
        """Modulation at an arbitrary flow time t (time-conditioned models only)."""
        return self._mods_for_cond(time_embedding(t, self.cfg.d))

    def _mods_for_cond(self, c: np.ndarray):
        """Modulation for a cond vector: per layer [scale1, shift1, gate1, scale2, shift2,
        gate2] (each [d], fp32-rounded) and the final [scale_f, shift_f]."""
        d = self.cfg.d
        per_layer = []
        for wm, bm in self.mod_w:
            m = C.fp32(c @ wm.T + bm)
            per_layer.append([m[i * d:(i + 1) * d] for i in range(6)])
        fin = None
        if self.final is not None:
            m = C.fp32(c @ self.final["w_mod_f"].T + self.final["b_mod_f"])
            fin = [m[:d], m[d:]]
        return per_layer, fin


def layer_forward(model: Model, l: int, k: int, x: np.ndarray, q: np.ndarray,
                  kpre, vpre, act_scales, amax=None):
    """One decoder layer. q holds the already-quantised pre-attention input codes.

    Returns x after the layer. amax (optional [L][4] array) records max |pre-quant value|.
    """
    cfg = model.cfg
    H, Hkv, Dh, F, af = cfg.H, cfg.Hkv, cfg.Dh, cfg.F, cfg.act_fmt
    sc1, sh1, g1, sc2, sh2, g2 = model.mods[k][0][l]
    w = model.w[l]
    s = act_scales[l] if af in ("fp8", "nvfp4") else None   # bf16 operands carry no scale
    sa = lambda i: float(s[i]) if af in ("fp8", "nvfp4") else 1.0

    qkv = gemm(q, sa(SITE_ATTN_IN), w["qkv"])
    nq, nk = H * Dh, Hkv * Dh
    if getattr(cfg, "attn_fmt", "bf16") == "fp8":
        if amax is not None:
            amax[l, SITE_Q] = max(amax[l, SITE_Q], np.max(np.abs(qkv[:, :nq])))
            amax[l, SITE_K] = max(amax[l, SITE_K], np.max(np.abs(qkv[:, nq:nq + nk])), np.max(np.abs(kpre[l])))
            amax[l, SITE_V] = max(amax[l, SITE_V], np.max(np.abs(qkv[:, nq + nk:])), np.max(np.abs(vpre[l])))
        s_q, s_k, s_v = sa(SITE_Q), sa(SITE_K), sa(SITE_V)
        O = attention_fp8(quant_codes(qkv[:, :nq], s_q, "fp8"), quant_codes(qkv[:, nq:nq + nk], s_k, "fp8"),
                          quant_codes(qkv[:, nq + nk:], s_v, "fp8"), quant_codes(kpre[l], s_k, "fp8"),
                          quant_codes(vpre[l], s_v, "fp8"), H, Hkv, Dh, s_q, s_k, s_v)
    else:
        Q = C.bf16(qkv[:, :nq])
        Kc = C.bf16(qkv[:, nq:nq + nk])
        Vc = C.bf16(qkv[:, nq + nk:])
        O = attention(Q, Kc, Vc, kpre[l], vpre[l], H, Hkv, Dh)
    if amax is not None:
        amax[l, SITE_ATTN_OUT] = max(amax[l, SITE_ATTN_OUT], np.max(np.abs(O)))
    o = gemm(quant_codes(O, sa(SITE_ATTN_OUT), af), sa(SITE_ATTN_OUT), w["o"])
    x = x + g1 * o

    h2 = ada_norm(x, sc2, sh2, cfg.eps)
    if amax is not None:
        amax[l, SITE_MLP_IN] = max(amax[l, SITE_MLP_IN], np.max(np.abs(h2)))
    gu = gemm(quant_codes(h2, sa(SITE_MLP_IN), af), sa(SITE_MLP_IN), w["gu"])
    m = gelu_tanh(gu[:, :F]) * gu[:, F:]
    if amax is not None:
        amax[l, SITE_GEGLU] = max(amax[l, SITE_GEGLU], np.max(np.abs(m)))
    dd = gemm(quant_codes(m, sa(SITE_GEGLU), af), sa(SITE_GEGLU), w["d"])
    return x + g2 * dd


def pre_attn_quant(model: Model, l: int, k: int, x, act_scales, amax=None):
    cfg = model.cfg
    sc1, sh1 = model.mods[k][0][l][0], model.mods[k][0][l][1]
    h = ada_norm(x, sc1, sh1, cfg.eps)
    if amax is not None:
        amax[l, SITE_ATTN_IN] = max(amax[l, SITE_ATTN_IN], np.max(np.abs(h)))
    s = float(act_scales[l][SITE_ATTN_IN]) if cfg.act_fmt in ("fp8", "nvfp4") else 1.0
    return quant_codes(h, s, cfg.act_fmt)


def euler_step(model: Model, k: int, a: np.ndarray, kpre, vpre, act_scales, amax=None, dt=None):
    """One flow-matching Euler step: a <- a + dt * v(a, t_k) with step k's modulation,
    dt = -1/S unless given."""
    cfg, fin = model.cfg, model.final
    x = np.asarray(a, np.float64) @ fin["w_in"].T + fin["b_in"]
    for l in range(cfg.L):
        q = pre_attn_quant(model, l, k, x, act_scales, amax)
        x = layer_forward(model, l, k, x, q, kpre, vpre, act_scales, amax)
    scf, shf = model.mods[k][1]
    hf = ada_norm(x, scf, shf, cfg.eps) * fin["gamma_f"]
    v = hf @ fin["w_out"].T + fin["b_out"]
    return a + ((-1.0 / cfg.S) if dt is None else dt) * v


def decode(model: Model, noise, kpre, vpre, act_scales, amax=None) -> np.ndarray:
    """A whole decision: S Euler steps from noise (t = 1) to the action chunk (t = 0)."""
    a = np.asarray(noise, np.float64)
    kpre = np.asarray(kpre, np.float64)
    vpre = np.asarray(vpre, np.float64)
    for k in range(model.cfg.S):
        a = euler_step(model, k, a, kpre, vpre, act_scales, amax)
    return a


def warm_time(cfg) -> float:
    """The warm start's flow time as the library holds it (an fp32 config field)."""
    return float(np.float32(cfg.warm_t))


def warm_start_input(prev, executed: int, tau: float, noise) -> np.ndarray:
    """One-step warm start (blog post, section "Few-step denoise brings the error back
    into consecutive decisions"): the previous chunk moved forward by the number of
    actions already executed, its tail padded with its last action, then mixed with
    fresh noise at flow time tau: a_tau = tau * noise + (1 - tau) * shifted."""
    prev = np.asarray(prev, np.float64)
    M = prev.shape[0]
    shifted = prev[np.minimum(np.arange(M) + executed, M - 1)]
    return tau * np.asarray(noise, np.float64) + (1.0 - tau) * shifted


def decode_warm(model: Model, noise, prev, executed: int, kpre, vpre, act_scales, tau=None,
                amax=None) -> np.ndarray:
    """The warm-start decision: one Euler step from a_tau (warm_start_input) at flow
    time tau to t = 0, i.e. dt = -tau, with the modulation at t = tau. tau defaults
    to the config's warm_t (fp32)."""
    kpre = np.asarray(kpre, np.float64)
    vpre = np.asarray(vpre, np.float64)
    given = tau is not None
    if not given:
        tau = warm_time(model.cfg)
    model.mods.append(model.mods_at(tau) if given else model.mods[model.cfg.S])
    try:
        a = warm_start_input(prev, executed, tau, noise)
        return euler_step(model, len(model.mods) - 1, a, kpre, vpre, act_scales, amax, dt=-tau)
    finally:
        model.mods.pop()


def calibrate(model: Model, noise, kpre, vpre, provisional_scales) -> np.ndarray:
    """Static activation scales from one calibration decision: for every layer and
    quant point, amax of the pre-quantisation value over all S steps (run with the
    provisional table), divided by 448 and rounded to fp32; a point whose amax is 0
    keeps its provisional scale."""
    cfg = model.cfg
    amax = np.zeros(np.shape(provisional_scales), np.float64)
    decode(model, noise, kpre, vpre, provisional_scales, amax)
    out = np.asarray(provisional_scales, np.float32).copy()
    nz = amax > 0
    # E4M3: amax / 448; NVFP4 activations: the tensor scale amax / (448 * 6)
    div = F32(2688.0) if cfg.act_fmt == "nvfp4" else F32(448.0)
    out[nz] = (amax[nz].astype(np.float32) / div).astype(np.float32)
    return out


def single_layer(model: Model, x_in, kpre, vpre, act_scales, layer=0, step=0):
    """One layer on a given residual input, plus the quantised input it hands to the
    next layer (layer (l+1) mod L's pre-attention params stand in for the next layer).

    Returns (x_out, q_next_codes, q_in_codes)."""
    cfg = model.cfg
    kpre = np.asarray(kpre, np.float64)
    vpre = np.asarray(vpre, np.float64)
    x = np.asarray(x_in, np.float64)
    q = pre_attn_quant(model, layer, step, x, act_scales)
    x_out = layer_forward(model, layer, step, x, q, kpre, vpre, act_scales)
    q_next = pre_attn_quant(model, (layer + 1) % cfg.L, step, x_out, act_scales)
    return x_out, q_next, q


def gemm_consumer(a_codes, s_a, w: PreparedWeight, bias, x, gate, scale, shift, s_q, eps,
                  act_fmt="fp8"):
    """Standalone skinny GEMM + fused consumer: y = A W^T (dequantised) + bias,
    x_out = x + gate * y, q = Q(AdaRMSNorm(x_out; scale, shift)).

    Returns (y, x_out, q_codes)."""
    y = gemm(a_codes, s_a, w) + np.asarray(bias, np.float64)
    x_out = np.asarray(x, np.float64) + np.asarray(gate, np.float64) * y
    h = ada_norm(x_out, scale, shift, eps)
    return y, x_out, quant_codes(h, s_q, act_fmt)
