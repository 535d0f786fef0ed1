"""Helpers shared by the GPU tests: device buffers, tile layouts, tolerances."""
import os

import numpy as np
import pytest
import torch

import flow_matching_action_denoise_gb300 as fmad
from oracle import codecs as C

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    fmad.load()   # raises if the compiled library is missing: no fallback
    return torch.device("cuda:0")


def dev(a, device, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.to(device)


def aligned_empty(nbytes, device, align=1024):
    """A uint8 device buffer whose returned pointer is `align`-aligned (buffer, ptr)."""
    buf = torch.empty(nbytes + align, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % align
    return buf, buf.data_ptr() + off


def _chunk_perm(rows):
    """Chunk index (0..7, 16 bytes each) where row r of a 128-byte-row tile stores its
    chunk c under the 128-byte swizzle: c ^ (r mod 8)."""
    r = np.arange(rows)[:, None]
    c = np.arange(8)[None, :]
    return r, c, c ^ (r % 8)


def tile_codes(codes, elems_per_row_block):
    """[N][K] -> the packed tile order [N/128][K/e][128][e] (e = 128 fp8 or 64 bf16), each
    128-byte row stored with the 128-byte swizzle (the layout the MMA reads)."""
    n, k = codes.shape
    e = elems_per_row_block
    t = codes.reshape(n // 128, 128, k // e, e).transpose(0, 2, 1, 3).reshape(n // 128, k // e, 128, 8, e // 8)
    r, c, sw = _chunk_perm(128)
    out = np.empty_like(t)
    out[:, :, r, sw, :] = t[:, :, r, c, :]
    return out.reshape(n // 128, k // e, 128, e).copy()


def untile_codes(packed, n, k, e):
    t = np.asarray(packed).reshape(n // 128, k // e, 128, 8, e // 8)
    r, c, sw = _chunk_perm(128)
    plain = t[:, :, r, sw, :]   # chunk c of row r lives at position c ^ (r mod 8)
    return plain.reshape(n // 128, k // e, 128, e).transpose(0, 2, 1, 3).reshape(n, k)


def e4m3_values_of_bytes(b):
    return C.e4m3_decode_code(np.asarray(b, np.uint8))


def bf16_values_of_bits(bits):
    return C.bf16_decode_bits(np.asarray(bits).view(np.uint16))


def code_step_distance(a_codes, b_codes):
    """Distance in representable E4M3 steps between codes (sign-magnitude order)."""
    def ordinal(c):
        c = np.asarray(c, np.int64)
        mag = c & 0x7F
        return np.where(c & 0x80, -mag, mag)
    return np.abs(ordinal(a_codes) - ordinal(b_codes))


def load_scales(name):
    path = os.path.join(GOLDEN, f"act_scales_{name}.txt")
    return np.loadtxt(path, dtype=np.float32, ndmin=2)


def _trace_fields(cfg, pol):
    """The fields of one trace record (one layer-step) in order: (name, kind, shape,
    bytes); kind f = fp32, b = the QKV output, c = activation codes."""
    M, d = cfg.M, cfg.d
    fp8 = cfg.act_fmt == "fp8"
    f16_codes = cfg.weight_fmt == "nvfp4"   # E4M3 codes stored as their f16 values
    qkv8 = getattr(cfg, "attn_fmt", "bf16") == "fp8"   # Q | K | V as E4M3 codes
    ab = 1 if fp8 and not f16_codes else 2

    def parts(name, n):
        _, nbytes = fmad.named_buffer(pol.handle, name)
        return nbytes // (M * n * 4)

    layout = [("x_in", "f", (M, d)), ("q", "c", (M, d)),
              ("y_qkv", "b", (M, cfg.n_qkv)),
              ("attn_out", "c", (M, cfg.H * cfg.Dh)), ("y_o", "f", (parts("y_o", d), M, d)),
              ("x_mid", "f", (M, d)), ("q2", "c", (M, d)),
              ("geglu_out", "c", (M, cfg.F)),
              ("y_d", "f", (parts("y_d", d), M, d)), ("x_out", "f", (M, d)), ("actions", "f", (M, cfg.A))]
    out = []
    for name, kind, shape in layout:
        n = int(np.prod(shape))
        out.append((name, kind, shape, n * (4 if kind == "f" else (1 if qkv8 else 2) if kind == "b" else ab)))
    return out


def _decode_record(raw, cfg, fields):
    fp8 = cfg.act_fmt == "fp8"
    f16_codes = cfg.weight_fmt == "nvfp4"
    qkv8 = getattr(cfg, "attn_fmt", "bf16") == "fp8"
    r, off = {}, 0
    for name, kind, shape, nb in fields:
        chunk = raw[off:off + nb]
        off += nb
        if kind == "b" and qkv8:
            r[name] = C.e4m3_decode_code(chunk).reshape(shape)
        elif kind == "b":
            r[name] = C.bf16_decode_bits(chunk.view(np.uint16)).reshape(shape)
        elif kind == "f":
            r[name] = chunk.view(np.float32).reshape(shape).astype(np.float64)
        elif f16_codes:
            r[name] = chunk.view(np.float16).astype(np.float64).reshape(shape)
        elif fp8:
            r[name] = C.e4m3_decode_code(chunk).reshape(shape)
        else:
            r[name] = C.bf16_decode_bits(chunk.view(np.uint16)).reshape(shape)
    assert off == raw.size
    return r


def parse_trace(raw, cfg, pol):
    """Split an fm_decode_trace buffer into records[k][l] of numpy arrays; codes are
    returned as decoded values (E4M3 codes without their scale, or bf16 values)."""
    fields = _trace_fields(cfg, pol)
    rec = sum(f[3] for f in fields)
    assert raw.size == rec * cfg.S * cfg.L, (raw.size, rec * cfg.S * cfg.L)
    return [[_decode_record(raw[(k * cfg.L + l) * rec:(k * cfg.L + l + 1) * rec], cfg, fields)
             for l in range(cfg.L)] for k in range(cfg.S)]


def read_trace_records(trace, cfg, pol, wanted):
    """{(k, l): record} for the layer-steps in `wanted`, copying only those records out
    of the device trace buffer (a uint8 tensor): the records are laid out layer-step by
    layer-step, step-major, each of the same size."""
    fields = _trace_fields(cfg, pol)
    rec = sum(f[3] for f in fields)
    assert trace.numel() >= rec * cfg.S * cfg.L
    out = {}
    for k, l in wanted:
        i = k * cfg.L + l
        out[(k, l)] = _decode_record(trace[i * rec:(i + 1) * rec].cpu().numpy(), cfg, fields)
    return out
