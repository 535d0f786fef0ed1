"""GPU building blocks against the CPU oracle, element by element, through the C ABI.

Bars: integer and byte work (E4M3 codes, packed weights, integer split-K
partials) bit-exact; the fp32 GEMM product within 1e-5 * RMS; consumer outputs
within fp32 rounding, quantised codes equal except rare 1-step near-tie flips.
"""
import numpy as np
import pytest
import torch

import fm_synth
import flow_matching_action_denoise_gb300 as fmad
from oracle import codecs as C
from oracle import model as O

from _gpu import (aligned_empty, code_step_distance, dev, e4m3_values_of_bytes, require_gpu, tile_codes,
                  untile_codes)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def device():
    return require_gpu()


# ---------------------------------------------------------------- quantiser

def test_quant_e4m3_midpoint_sweep_bit_exact(device):
    grid = np.unique(np.abs(C.e4m3_decode_code(np.arange(127))))
    mids = (grid[:-1] + grid[1:]) / 2
    eps = (grid[1:] - grid[:-1]) * 1e-3
    x = np.concatenate([mids, -mids, mids - eps, mids + eps, grid, [449.0, 500.0, 1e9, -1e9, 0.0]])
    x = x.astype(np.float32)
    for scale in [1.0, 0.125, 0.0137, 3.7]:
        xd = dev(x, device)
        codes = torch.empty(x.size, dtype=torch.uint8, device=device)
        fmad.fm_test_quant_e4m3(xd, scale, codes)
        torch.cuda.synchronize()
        r = np.float32(1.0) / np.float32(scale)
        expect = C.e4m3_encode_code(C.e4m3(C.fp32(x.astype(np.float64) * np.float64(r))))
        got = codes.cpu().numpy()
        # -0.0 and +0.0 are both valid encodings of a zero result
        zero = C.e4m3(C.fp32(x.astype(np.float64) * np.float64(r))) == 0
        np.testing.assert_array_equal(got[~zero], expect[~zero])
        assert np.all(e4m3_values_of_bytes(got[zero]) == 0)


# ---------------------------------------------------------------- weight packing

@pytest.mark.parametrize("N,K,with_gamma", [(1280, 1024, True), (1024, 4096, False)])
def test_pack_fp8_bit_exact(device, N, K, with_gamma):
    rng = np.random.default_rng(N + K)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(K)).astype(np.float32) if with_gamma else None
    nbytes = fmad.fm_packed_weight_bytes(N, K, fmad.FMT_FP8)
    buf, ptr = aligned_empty(nbytes, device)
    scale = torch.empty(1, dtype=torch.float32, device=device)
    fmad.fm_pack_weight(dev(w, device), dev(g, device) if g is not None else None, N, K, fmad.FMT_FP8, ptr, scale)
    torch.cuda.synchronize()
    off = ptr - buf.data_ptr()
    packed = buf[off:off + nbytes].cpu().numpy()
    codes = untile_codes(packed, N, K, 128)
    ref = O.prep_weight(w, g, "fp8")
    assert np.float32(scale.item()) == np.float32(ref.scale)
    np.testing.assert_array_equal(e4m3_values_of_bytes(codes), ref.codes)


def test_pack_bf16_bit_exact(device):
    N, K = 1024, 1024
    rng = np.random.default_rng(5)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    g = (1 + 0.1 * rng.standard_normal(K)).astype(np.float32)
    nbytes = fmad.fm_packed_weight_bytes(N, K, fmad.FMT_BF16)
    buf, ptr = aligned_empty(nbytes, device)
    scale = torch.empty(1, dtype=torch.float32, device=device)
    fmad.fm_pack_weight(dev(w, device), dev(g, device), N, K, fmad.FMT_BF16, ptr, scale)
    torch.cuda.synchronize()
    off = ptr - buf.data_ptr()
    packed = buf[off:off + nbytes].cpu().numpy().view(np.uint16)
    vals = C.bf16_decode_bits(untile_codes(packed, N, K, 64))
    np.testing.assert_array_equal(vals, O.prep_weight(w, g, "bf16").codes)
    assert scale.item() == 1.0


# ---------------------------------------------------------------- skinny GEMM

def run_gemm(device, a_bytes_or_bf16, M, K, packed_host, N, fmt, s, cs, tile=128):
    """a: host uint8 [M][K] codes (fp8) or uint16 bf16 bits; packed_host: tiled bytes/bits;
    tile: weight rows per CTA (128, or 64: half of a packed tile)."""
    a = dev(a_bytes_or_bf16, device)
    raw = np.ascontiguousarray(packed_host).view(np.uint8).reshape(-1)
    buf, ptr = aligned_empty(raw.size, device)
    off = ptr - buf.data_ptr()
    buf[off:off + raw.size].copy_(torch.from_numpy(raw).to(device))
    nparts = s // cs
    out = torch.full((nparts, M, N), float("nan"), dtype=torch.float32, device=device)
    if tile == 128:
        fmad.fm_test_skinny_gemm(a, M, K, ptr, N, fmt, s, cs, out)
    else:
        fmad.fm_test_skinny_gemm_tile(a, M, K, ptr, N, fmt, s, cs, tile, out)
    torch.cuda.synchronize()
    assert fmad.standalone_status() == 0, "a GEMM pipeline wait expired"
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("tile", [128, 64])
@pytest.mark.parametrize("M,K,N", [(1, 1024, 1024), (10, 1024, 1280), (50, 4096, 1024), (63, 2048, 4096),
                                   (100, 1024, 1024), (256, 1024, 1024)])
def test_skinny_gemm_integer_split_invariance_bit_exact(device, M, K, N, tile):
    """Integer A, W in [-3, 3] (exact E4M3 codes, scale 1): every partial and every fp32
    sum is exact, so each K-split and cluster size must give the exact product, with
    128-row tiles and with 64-row tiles (each CTA half of a packed tile), for MMA N
    (the activation rows rounded up to 16) from 16 to 256."""
    case = fm_synth.gemm_case(M, K, N, integer=True)
    a, w = case["a"].astype(np.float64), case["w"].astype(np.float64)
    a_codes = C.e4m3_encode_code(a)
    packed = tile_codes(C.e4m3_encode_code(w), 128)
    exact = a @ w.T
    nkb = K // 128
    for s in [1, 2, 4, 8, 16]:
        if nkb % s:
            continue
        for cs in [1, 2, 4, 8]:
            if s % cs:
                continue
            parts = run_gemm(device, a_codes, M, K, packed, N, fmad.FMT_FP8, s, cs, tile)
            ref = O.gemm_ksplit(a, O.PreparedWeight(w, 1.0, "fp8"), s)
            ref = ref.reshape(s // cs, cs, M, N).sum(axis=1)
            np.testing.assert_array_equal(parts, ref, err_msg=f"s={s} cs={cs}")
            np.testing.assert_array_equal(parts.sum(axis=0), exact)


@pytest.mark.parametrize("M,K,N,s,cs", [(10, 1024, 1280, 8, 8), (50, 4096, 1024, 16, 8), (63, 1024, 8192, 2, 2),
                                        (50, 1024, 16384, 4, 4), (1, 2048, 4096, 1, 1)])
def test_skinny_gemm_fp8_random_vs_oracle(device, M, K, N, s, cs):
    case = fm_synth.gemm_case(M, K, N)
    s_a = float(np.float32(np.max(np.abs(case["a"])) / np.float32(448)))
    a_codes = O.quant_codes(case["a"], s_a, "fp8")
    pw = O.prep_weight(case["w"], None, "fp8")
    packed = tile_codes(C.e4m3_encode_code(pw.codes), 128)
    parts = run_gemm(device, C.e4m3_encode_code(a_codes), M, K, packed, N, fmad.FMT_FP8, s, cs)
    got = parts.sum(axis=0)
    ref = a_codes @ pw.codes.T
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.max(np.abs(got - ref)) <= 1e-5 * rms


@pytest.mark.parametrize("tile", [128, 64])
@pytest.mark.parametrize("M,K,N,s,cs", [(63, 1024, 1280, 4, 4), (10, 4096, 1024, 8, 8), (16, 1024, 2048, 1, 1)])
def test_skinny_gemm_bf16_vs_oracle(device, M, K, N, s, cs, tile):
    case = fm_synth.gemm_case(M, K, N, seed=11)
    a = C.bf16(case["a"])
    pw = O.prep_weight(case["w"], None, "bf16")
    a_bits = torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).view(torch.uint16).numpy()
    w_bits = torch.from_numpy(pw.codes.astype(np.float32)).to(torch.bfloat16).view(torch.uint16).numpy()
    parts = run_gemm(device, a_bits, M, K, tile_codes(w_bits, 64), N, fmad.FMT_BF16, s, cs, tile)
    ref = a @ pw.codes.T
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.max(np.abs(parts.sum(axis=0) - ref)) <= 1e-5 * rms


# ---------------------------------------------------------------- fused consumer

@pytest.mark.parametrize("M,N,nparts", [(10, 1024, 1), (50, 1024, 2), (63, 4096, 4), (1, 16384, 1)])
def test_consumer_vs_oracle(device, M, N, nparts):
    K = 1024
    case = fm_synth.gemm_case(M, K, N)
    s_a = float(np.float32(np.max(np.abs(case["a"])) / np.float32(448)))
    a_codes = O.quant_codes(case["a"], s_a, "fp8")
    pw = O.prep_weight(case["w"], None, "fp8")
    partials = O.gemm_ksplit(a_codes, pw, nparts)          # exact; fp32-representable here
    y_ref, x_ref, _ = O.gemm_consumer(a_codes, s_a, pw, case["bias"], case["x"], case["gate"],
                                      case["scale"], case["shift"], 1.0, 1e-6)
    h = O.ada_norm(x_ref, case["scale"], case["shift"], 1e-6)
    s_q = float(np.float32(np.max(np.abs(h)) / np.float32(448)))
    _, x_ref, q_ref = O.gemm_consumer(a_codes, s_a, pw, case["bias"], case["x"], case["gate"],
                                      case["scale"], case["shift"], s_q, 1e-6)
    f32 = lambda v: dev(np.asarray(v, np.float32), device)
    x = f32(case["x"])
    q = torch.empty((M, N), dtype=torch.uint8, device=device)
    fmad.fm_test_consumer(f32(partials), nparts, M, N, f32([s_a]), f32([pw.scale]), f32(case["bias"]), x,
                          f32(case["gate"]), f32(case["scale"]), f32(case["shift"]), 1e-6, f32([s_q]), q,
                          fmad.FMT_FP8)
    torch.cuda.synchronize()
    xg = x.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(xg - x_ref)) <= 1e-5 * np.sqrt(np.mean(x_ref ** 2))
    qg = q.cpu().numpy()
    qr = C.e4m3_encode_code(q_ref)
    dist = code_step_distance(qg, qr)
    assert np.max(dist) <= 1
    assert np.mean(dist > 0) <= 1e-3


# ---------------------------------------------------------------- GEMM + fused consumer in one call

def gemm_consumer_case(device, M, K, N, fmt, seed=2):
    """Inputs for fm_gemm_consumer on the device and the oracle's expected outputs."""
    case = fm_synth.gemm_case(M, K, N, seed=seed)
    act = "fp8" if fmt == fmad.FMT_FP8 else "bf16"
    if act == "fp8":
        s_a = float(np.float32(np.max(np.abs(case["a"])) / np.float32(448)))
        a_codes = O.quant_codes(case["a"], s_a, "fp8")
        a_dev = dev(C.e4m3_encode_code(a_codes), device)
    else:
        s_a = 1.0
        a_codes = C.bf16(case["a"])
        a_dev = dev(a_codes.astype(np.float32), device, torch.bfloat16)
    pw = O.prep_weight(case["w"], None, act)
    y, x_ref, _ = O.gemm_consumer(a_codes, s_a, pw, case["bias"], case["x"], case["gate"], case["scale"],
                                  case["shift"], 1.0, 1e-6, act)
    h = O.ada_norm(x_ref, case["scale"], case["shift"], 1e-6)
    s_q = float(np.float32(np.max(np.abs(h)) / np.float32(448))) if act == "fp8" else 1.0
    q_ref = O.quant_codes(h, s_q, act)
    nbytes = fmad.fm_packed_weight_bytes(N, K, fmt)
    wbuf, wptr = aligned_empty(nbytes, device)
    w_scale = torch.empty(1, dtype=torch.float32, device=device)
    fmad.fm_pack_weight(dev(case["w"], device), None, N, K, fmt, wptr, w_scale)
    f32 = lambda v: dev(np.asarray(v, np.float32), device)
    inputs = dict(a=a_dev, w=(wbuf, wptr), s_a=f32([s_a]), s_w=w_scale, bias=f32(case["bias"]),
                  x0=f32(case["x"]), gate=f32(case["gate"]), scale=f32(case["scale"]), shift=f32(case["shift"]),
                  s_q=f32([s_q]))
    return inputs, x_ref, q_ref


def run_gemm_consumer(device, inp, M, K, N, fmt, s, entry="scratch"):
    x = inp["x0"].clone()
    q = torch.empty((M, N), dtype=torch.uint8 if fmt == fmad.FMT_FP8 else torch.bfloat16, device=device)
    args = (inp["a"], M, K, inp["w"][1], N, fmt, s, inp["s_a"], inp["s_w"], inp["bias"], x, inp["gate"],
            inp["scale"], inp["shift"], 1e-6, inp["s_q"], q)
    if entry == "scratch":
        nbytes = fmad.gemm_consumer_scratch_bytes(M, N, K, fmt, s)
        scratch = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device=device)
        fmad.fm_gemm_consumer(*args, scratch, nbytes)
    else:
        fmad.fm_gemm_consumer_noalloc(*args)
    torch.cuda.synchronize()
    assert fmad.standalone_status() == 0, "a GEMM pipeline wait expired"
    return x.cpu().numpy().astype(np.float64), q


def check_gemm_consumer_outputs(x, q, x_ref, q_ref, fmt):
    assert np.max(np.abs(x - x_ref)) <= 1e-5 * np.sqrt(np.mean(x_ref ** 2))
    if fmt == fmad.FMT_FP8:
        dist = code_step_distance(q.cpu().numpy(), C.e4m3_encode_code(q_ref))
        assert np.max(dist) <= 1 and np.mean(dist > 0) <= 1e-3
    else:
        # a near-tie input may round to the neighbouring bf16 value: one step is at most
        # 2^-7 of the value
        qv = q.float().cpu().numpy().astype(np.float64)
        assert np.all(np.abs(qv - q_ref) <= 2.0 ** -7 * np.abs(q_ref) + 1e-6 * np.sqrt(np.mean(q_ref ** 2)))


@pytest.mark.parametrize("M,K,N,s,fmt", [(1, 1024, 1024, 1, fmad.FMT_FP8), (10, 2048, 4096, 4, fmad.FMT_FP8),
                                         (50, 4096, 1024, 16, fmad.FMT_FP8), (63, 1024, 16384, 2, fmad.FMT_FP8),
                                         (63, 1024, 4096, 2, fmad.FMT_BF16)])
def test_gemm_consumer_vs_oracle(device, M, K, N, s, fmt):
    inp, x_ref, q_ref = gemm_consumer_case(device, M, K, N, fmt)
    x, q = run_gemm_consumer(device, inp, M, K, N, fmt, s)
    check_gemm_consumer_outputs(x, q, x_ref, q_ref, fmt)
