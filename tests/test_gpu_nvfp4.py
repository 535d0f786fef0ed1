"""NVFP4 weights on the GPU against the CPU oracle: packing (bit-exact), the
NVFP4-weight GEMM (bit-exact on integer data, 1e-5 * RMS on random data) and a
world-action-model-shaped decision (d = 2048, 16 x 128 heads over 2 KV heads,
GeGLU 2048 -> 2 x 8192, M = 256 rows, prefix 1024) at 2 layers x 2 Euler steps,
pinned stage by stage and end to end within twice the oracle's own envelope.
"""
import numpy as np
import pytest
import torch

import fm_synth
import flow_matching_action_denoise_gb300 as fmad
from oracle import codecs as C
from oracle import model as O

from _gpu import aligned_empty, dev, parse_trace, require_gpu
from _stagewise import check_decision_stages

pytestmark = pytest.mark.gpu
BLOCK = 4608   # bytes of one packed (128 rows x 64 K) block: 4096 code bytes + 512 scale bytes


@pytest.fixture(scope="module")
def device():
    return require_gpu()


def gpu_pack(device, w, gamma):
    N, K = w.shape
    nbytes = fmad.fm_packed_weight_bytes(N, K, fmad.FMT_NVFP4)
    assert nbytes == N * K * 9 // 16
    buf, ptr = aligned_empty(nbytes, device)
    ts = torch.empty(1, dtype=torch.float32, device=device)
    fmad.fm_pack_weight(dev(w, device), dev(gamma, device) if gamma is not None else None, N, K, fmad.FMT_NVFP4,
                        ptr, ts)
    torch.cuda.synchronize()
    off = ptr - buf.data_ptr()
    return buf, ptr, buf[off:off + nbytes].cpu().numpy(), float(ts.item())


def unpack(packed, N, K):
    """Packed bytes -> (element values e [N][K], block-scale values bs [N][K/16])."""
    blocks = packed.reshape(N // 128, K // 64, BLOCK)
    codes = blocks[:, :, :4096].reshape(N // 128, K // 64, 128, 32)
    scales = blocks[:, :, 4096:].reshape(N // 128, K // 64, 128, 4)
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(N // 128, K // 64, 128, 64)
    e = C.e2m1_decode_code(nib).transpose(0, 2, 1, 3).reshape(N, K)
    bs = C.e4m3_decode_code(scales).transpose(0, 2, 1, 3).reshape(N, K // 16)
    return e, bs


@pytest.mark.parametrize("N,K,with_gamma", [(1024, 2048, True), (256, 1024, False)])
def test_pack_nvfp4_bit_exact(device, N, K, with_gamma):
    rng = np.random.default_rng(N * 7 + K)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    w[3] = 0.0                                   # an all-zero row: block scales 0, elements 0
    w[5, :16] = 1e-9                             # a block whose scale rounds into the E4M3 subnormals / zero
    w[7, 16:32] = 0.5                            # a block far above the rest (saturating neighbourhood)
    g = (1 + 0.1 * rng.standard_normal(K)).astype(np.float32) if with_gamma else None
    _, _, packed, ts = gpu_pack(device, w, g)
    ref = O.prep_weight(w, g, "nvfp4")
    assert np.float32(ts) == np.float32(ref.scale)
    e, bs = unpack(packed, N, K)
    np.testing.assert_array_equal(bs, ref.block_scales)
    np.testing.assert_array_equal(e * np.repeat(bs, 16, axis=1), ref.codes)


def run_nvfp4_gemm(device, a_values, w_ptr, M, K, N, s):
    a = dev(a_values.astype(np.float16), device)
    out = torch.full((s, M, N), float("nan"), dtype=torch.float32, device=device)
    fmad.fm_test_skinny_gemm(a, M, K, w_ptr, N, fmad.FMT_NVFP4, s, 1, out)
    torch.cuda.synchronize()
    assert fmad.standalone_status() == 0, "a GEMM pipeline wait expired"
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("M,K,N", [(1, 1024, 256), (10, 1024, 384), (63, 2048, 256), (256, 1024, 512)])
def test_nvfp4_gemm_integer_bit_exact(device, M, K, N):
    """Integer A in [-3, 3] and W in [-6, 6]: every block scale is an integer >= 74 and
    every decoded weight e * bs an integer <= 2688, so each fp32 partial sum is exact
    and every K-split must reproduce the oracle's exact planes."""
    case = fm_synth.gemm_case(M, K, N, integer=True)
    a = case["a"].astype(np.float64)
    w = (case["w"] * 2).astype(np.float32)
    buf, ptr, _, _ = gpu_pack(device, w, None)
    pw = O.prep_weight(w, None, "nvfp4")
    for s in [1, 2, 4, 8]:
        if (K // 64) % s:
            continue
        parts = run_nvfp4_gemm(device, a, ptr, M, K, N, s)
        np.testing.assert_array_equal(parts, O.gemm_ksplit(a, pw, s), err_msg=f"s={s}")
    del buf


@pytest.mark.parametrize("M,K,N,s", [(256, 2048, 2560, 4), (256, 8192, 2048, 8), (50, 2048, 1024, 2),
                                     (17, 1024, 384, 1)])
def test_nvfp4_gemm_random_vs_oracle(device, M, K, N, s):
    case = fm_synth.gemm_case(M, K, N, seed=13)
    s_a = float(np.float32(np.max(np.abs(case["a"])) / np.float32(448)))
    a_codes = O.quant_codes(case["a"], s_a, "fp8")
    buf, ptr, _, _ = gpu_pack(device, case["w"], None)
    pw = O.prep_weight(case["w"], None, "nvfp4")
    parts = run_nvfp4_gemm(device, a_codes, ptr, M, K, N, s)
    ref = O.gemm_ksplit(a_codes, pw, s)
    rms = np.sqrt(np.mean(ref.sum(axis=0) ** 2))
    assert np.max(np.abs(parts - ref)) <= 1e-5 * rms
    del buf


# ---------------------------------------------------------------- decision (2 layers x 2 steps)

@pytest.fixture(scope="module")
def wam(device):
    cfg = fm_synth.config("wam_nvfp4_m256", L=2, S=2)
    layers = [fm_synth.layer_weights(cfg, l) for l in range(cfg.L)]
    final = fm_synth.final_weights(cfg)
    kp, vp = fm_synth.prefix_kv(cfg)
    model = O.Model(cfg, layers, final)
    scales = O.calibrate(model, fm_synth.noise(cfg, 1000), kp, vp, fm_synth.default_act_scales(cfg))
    weights = fmad.DeviceWeights(cfg, layers, final, device=device)
    return dict(cfg=cfg, model=model, kp=kp, vp=vp, scales=scales, weights=weights, device=device)


def wam_policy(wam, flags=fmad.FLAG_USE_GRAPH | fmad.FLAG_USE_PDL):
    p = fmad.Policy(wam["cfg"], act_scales=wam["scales"], flags=flags, weights=wam["weights"])
    p.set_prefix_kv(dev(wam["kp"], wam["device"], torch.bfloat16), dev(wam["vp"], wam["device"], torch.bfloat16))
    return p


def test_wam_decision_every_stage_vs_oracle(wam):
    cfg = wam["cfg"]
    pol = wam_policy(wam)
    per_layer, per_decision = fmad.kernel_count(pol.handle)
    assert (per_layer, per_decision) == (8, 1 + cfg.L * cfg.S * 8)
    nbytes = fmad.trace_size(pol.handle)
    trace = torch.empty(nbytes, dtype=torch.uint8, device=wam["device"])
    nz = fm_synth.noise(cfg, 0)
    act = torch.empty((cfg.M, cfg.A), dtype=torch.float32, device=wam["device"])
    fmad.decode_trace(pol.handle, dev(nz, wam["device"]), act, trace, nbytes)
    assert fmad.device_status(pol.handle) == 0
    assert torch.equal(act.cpu(), pol.decode(dev(nz, wam["device"])).cpu())
    recs = parse_trace(trace.cpu().numpy(), cfg, pol)
    last = check_decision_stages(cfg, wam["model"], recs, nz, wam["kp"], wam["vp"], wam["scales"])
    np.testing.assert_array_equal(last, act.cpu().numpy())
    pol.close()


def test_wam_decision_end_to_end_within_envelope(wam):
    """End to end the decision is chaotic at the rounding level (it requantises four
    activations per layer-step). The GPU differs from the oracle in two places of the
    same arithmetic: fp32 (not exact) pre-quantisation values and fp32 (not exact)
    GEMM accumulation. Each source alone, applied to the oracle, moves its actions by
    env_i; the GPU must stay within twice their sum."""
    cfg, model, kp, vp, sc = wam["cfg"], wam["model"], wam["kp"], wam["vp"], wam["scales"]
    nz = fm_synth.noise(cfg, 0)
    pol = wam_policy(wam)
    got = pol.decode(dev(nz, wam["device"])).cpu().numpy().astype(np.float64)
    pol.close()
    ref = O.decode(model, nz, kp, vp, sc)
    rms = np.sqrt(np.mean(ref ** 2))
    plain_quant, plain_gemm = O.quant_codes, O.gemm

    def quant_fp32_input(h, s, fmt):   # the same quantiser fed fp32-rounded values
        if fmt == "fp8":
            return C.e4m3(C.fp32(C.fp32(h) * O.recip32(s)))
        return plain_quant(h, s, fmt)

    def gemm_fp32_sum(a, s_a, w):      # the same product with its sum rounded to fp32
        acc = C.fp32(np.asarray(a, np.float64) @ w.codes.T)
        return acc * np.float64(np.float32(s_a) * np.float32(w.scale))

    env = []
    for name, fn in (("quant_codes", quant_fp32_input), ("gemm", gemm_fp32_sum)):
        plain = getattr(O, name)
        setattr(O, name, fn)
        try:
            alt = O.decode(model, nz, kp, vp, sc)
        finally:
            setattr(O, name, plain)
        env.append(np.max(np.abs(alt - ref)) / rms)
    assert O.quant_codes is plain_quant and O.gemm is plain_gemm
    err = np.max(np.abs(got - ref)) / rms
    assert err <= 2 * sum(env), (err, env)


def test_wam_launch_modes_bitwise(wam):
    nz = dev(fm_synth.noise(wam["cfg"], 3), wam["device"])
    outs = []
    for flags in [fmad.FLAG_USE_GRAPH | fmad.FLAG_USE_PDL, 0]:
        pol = wam_policy(wam, flags)
        outs.append(pol.decode(nz).cpu())
        pol.close()
    assert torch.equal(outs[0], outs[1])
