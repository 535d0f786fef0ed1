"""Python binding of libfmad.so, the GB300 flow-matching action decoder.

Argument marshalling only: every step of the decoder runs in the library's CUDA
kernels. PyTorch supplies device memory and streams. The functions keep the C
names (include/fmad.h); they take torch tensors (or raw integer pointers) and
raise FmError on a non-zero status. Loading fails loudly when the compiled
library is missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "FmError", "lib", "load", "FmConfig", "make_config", "workspace_size", "policy_create",
    "policy_destroy", "set_prefix_kv", "refresh_prefix", "decode_actions", "decode_actions_host",
    "state_size", "snapshot_state", "restore_state", "fm_set_act_scales", "device_status", "standalone_status",
    "kernel_count", "philox_noise", "decode_actions_seeded", "last_timing", "decode_warm", "episode_reset", "Session",
    "session_workspace_size", "session_create", "session_fork", "FmTiming", "fm_test_quant_e4m3", "fm_packed_weight_bytes", "fm_pack_weight",
    "fm_test_skinny_gemm", "fm_test_consumer", "fm_test_layer", "named_buffer", "Policy", "DeviceWeights",
    "FMT_BF16", "FMT_FP8", "FMT_NVFP4", "FLAG_USE_GRAPH", "FLAG_USE_PDL", "FLAG_FUSED_CONSUMERS",
    "FLAG_O_CONSUMER_IN_GEMM", "COND_TIME", "COND_GIVEN",
    "ABI_VERSION", "STATUS",
]

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfmad.so")

ABI_VERSION = 3
FMT_BF16, FMT_FP8, FMT_NVFP4 = 0, 1, 2
FLAG_USE_GRAPH, FLAG_USE_PDL, FLAG_FUSED_CONSUMERS, FLAG_O_CONSUMER_IN_GEMM = 1, 2, 4, 8
COND_TIME, COND_GIVEN = 0, 1
STATUS = {0: "FM_OK", 1: "FM_ERR_INVALID_ARG", 2: "FM_ERR_SHAPE", 3: "FM_ERR_ALIGN",
          4: "FM_ERR_WORKSPACE", 5: "FM_ERR_CUDA", 6: "FM_ERR_STATE_MISMATCH",
          7: "FM_ERR_DEVICE", 8: "FM_ERR_UNSUPPORTED"}
EXPORTS = [
    "fm_status_string", "fm_last_error", "fm_workspace_size", "policy_create", "policy_destroy",
    "fm_set_act_scales", "set_prefix_kv", "refresh_prefix", "decode_actions", "decode_actions_host",
    "fm_state_size", "snapshot_state", "restore_state", "fm_device_status", "fm_test_kernel_count",
    "fm_test_quant_e4m3", "fm_packed_weight_bytes", "fm_pack_weight", "fm_test_skinny_gemm",
    "fm_test_consumer", "fm_test_layer", "fm_named_buffer", "fm_trace_size", "fm_decode_trace",
    "fm_gemm_consumer_scratch_bytes", "fm_gemm_consumer", "fm_gemm_consumer_noalloc",
    "fm_philox_noise", "fm_decode_actions_seeded", "fm_last_timing", "fm_decode_warm", "fm_episode_reset",
    "fm_session_workspace_size", "fm_session_create", "fm_session_fork", "fm_abi_sizes", "fm_standalone_status",
    "fm_warm_trace_size", "fm_decode_warm_trace", "fm_test_launch_kernel", "fm_decode_timeline",
    "fm_test_skinny_gemm_tile", "fm_test_pdl_chain", "fm_test_grid_barrier", "fm_test_attn_plan",
]


class FmError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}" + (f" ({detail})" if detail else ""))


class FmConfig(ctypes.Structure):
    _fields_ = [("abi_version", ctypes.c_int),
                ("L", ctypes.c_int), ("S", ctypes.c_int), ("M", ctypes.c_int), ("d", ctypes.c_int),
                ("H", ctypes.c_int), ("Hkv", ctypes.c_int), ("Dh", ctypes.c_int), ("F", ctypes.c_int),
                ("P", ctypes.c_int), ("A", ctypes.c_int),
                ("weight_fmt", ctypes.c_int), ("act_fmt", ctypes.c_int), ("attn_fmt", ctypes.c_int),
                ("cond_mode", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("ksplit", ctypes.c_int * 4), ("flags", ctypes.c_uint),
                ("warm_t", ctypes.c_float)]


class FmTiming(ctypes.Structure):
    _fields_ = [("host_submit_ns", ctypes.c_uint64), ("device_start_ns", ctypes.c_uint64),
                ("device_end_ns", ctypes.c_uint64)]


class FmLayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("w_qkv", "w_o", "w_gu", "w_d", "gamma1", "gamma2", "w_mod", "b_mod")]


class FmWeights(ctypes.Structure):
    _fields_ = [("layers", ctypes.POINTER(FmLayerWeights))] + [
        (n, ctypes.c_void_p) for n in
        ("w_in", "b_in", "w_out", "b_out", "gamma_f", "w_mod_f", "b_mod_f", "conds")]


_lib = None


def load() -> ctypes.CDLL:
    """Load the in-tree libfmad.so (build it with __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sig = {
        "fm_status_string": (ctypes.c_char_p, [i]),
        "fm_last_error": (ctypes.c_char_p, [vp]),
        "fm_workspace_size": (i, [ctypes.POINTER(FmConfig), ctypes.POINTER(sz)]),
        "policy_create": (i, [ctypes.POINTER(FmConfig), ctypes.POINTER(FmWeights), vp, vp, sz, vp,
                              ctypes.POINTER(vp)]),
        "policy_destroy": (i, [vp]),
        "fm_set_act_scales": (i, [vp, vp, vp]),
        "set_prefix_kv": (i, [vp, vp, vp, vp]),
        "refresh_prefix": (i, [vp, i, i, vp, vp, vp]),
        "decode_actions": (i, [vp, vp, vp, vp]),
        "decode_actions_host": (i, [vp, vp, vp, vp]),
        "fm_state_size": (i, [vp, ctypes.POINTER(sz)]),
        "snapshot_state": (i, [vp, vp, sz, i, vp]),
        "restore_state": (i, [vp, vp, sz, i, vp]),
        "fm_device_status": (i, [vp, vp, ctypes.POINTER(i)]),
        "fm_standalone_status": (i, [vp, ctypes.POINTER(i)]),
        "fm_test_kernel_count": (i, [vp, ctypes.POINTER(i), ctypes.POINTER(i)]),
        "fm_test_quant_e4m3": (i, [vp, ctypes.c_int64, ctypes.c_float, vp, vp]),
        "fm_packed_weight_bytes": (i, [i, i, i, ctypes.POINTER(sz)]),
        "fm_pack_weight": (i, [vp, vp, i, i, i, vp, vp, vp]),
        "fm_test_skinny_gemm": (i, [vp, i, i, vp, i, i, i, i, vp, vp]),
        "fm_test_skinny_gemm_tile": (i, [vp, i, i, vp, i, i, i, i, i, vp, vp]),
        "fm_test_consumer": (i, [vp, i, i, i, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, i, vp]),
        "fm_test_layer": (i, [vp, vp, i, i, vp, vp, vp]),
        "fm_named_buffer": (i, [vp, ctypes.c_char_p, ctypes.POINTER(vp), ctypes.POINTER(sz)]),
        "fm_trace_size": (i, [vp, ctypes.POINTER(sz)]),
        "fm_gemm_consumer_scratch_bytes": (i, [i, i, i, i, i, ctypes.POINTER(sz)]),
        "fm_gemm_consumer": (i, [vp, i, i, vp, i, i, i, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp, vp, sz,
                                 vp]),
        "fm_gemm_consumer_noalloc": (i, [vp, i, i, vp, i, i, i, vp, vp, vp, vp, vp, vp, vp, ctypes.c_float, vp, vp,
                                         vp]),
        "fm_decode_trace": (i, [vp, vp, vp, vp, sz, vp]),
        "fm_warm_trace_size": (i, [vp, ctypes.POINTER(sz)]),
        "fm_test_launch_kernel": (i, [vp, i, i, i, vp]),
        "fm_decode_timeline": (i, [vp, vp, vp, vp, sz, vp]),
        "fm_decode_warm_trace": (i, [vp, vp, i, vp, vp, sz, vp]),
        "fm_philox_noise": (i, [vp, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint64, vp, vp]),
        "fm_decode_actions_seeded": (i, [vp, ctypes.c_uint64, ctypes.c_uint64, vp, vp]),
        "fm_last_timing": (i, [vp, ctypes.POINTER(FmTiming), vp]),
        "fm_decode_warm": (i, [vp, vp, i, vp, vp]),
        "fm_episode_reset": (i, [vp]),
        "fm_session_workspace_size": (i, [vp, ctypes.POINTER(sz)]),
        "fm_abi_sizes": (i, [ctypes.POINTER(sz)] * 4),
        "fm_session_create": (i, [vp, vp, sz, vp, ctypes.POINTER(vp)]),
        "fm_session_fork": (i, [vp, vp, sz, i, vp, sz, vp, ctypes.POINTER(vp)]),
        "fm_test_pdl_chain": (i, [i, i, i, i, i, i, i, vp, sz, ctypes.POINTER(ctypes.c_float)]),
        "fm_test_grid_barrier": (i, [i, i, i, i, ctypes.c_ulonglong, vp, vp, vp]),
        "fm_test_attn_plan": (i, [vp, ctypes.POINTER(i), ctypes.POINTER(i)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def lib() -> ctypes.CDLL:
    return load()


# ---------------------------------------------------------------- marshalling helpers

def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str, policy=None):
    if status != 0:
        detail = load().fm_last_error(policy).decode(errors="replace")
        raise FmError(status, where, detail)


def make_config(cfg, flags: int = FLAG_USE_GRAPH | FLAG_USE_PDL, ksplit=(0, 0, 0, 0)) -> FmConfig:
    """fm_config from an fm_synth.Config-like object."""
    fmts = {"bf16": FMT_BF16, "fp8": FMT_FP8, "nvfp4": FMT_NVFP4}
    c = FmConfig()
    c.abi_version = ABI_VERSION
    for k in ("L", "S", "M", "d", "H", "Hkv", "Dh", "F", "P", "A"):
        setattr(c, k, int(getattr(cfg, k)))
    c.weight_fmt = fmts[cfg.weight_fmt]
    c.act_fmt = fmts[cfg.act_fmt]
    c.attn_fmt = fmts[getattr(cfg, "attn_fmt", "bf16")]
    c.cond_mode = COND_GIVEN if cfg.cond == "given" else COND_TIME
    c.rms_eps = float(cfg.eps)
    for i, s in enumerate(ksplit):
        c.ksplit[i] = int(s)
    c.flags = int(flags)
    c.warm_t = float(getattr(cfg, "warm_t", 0.0))
    return c


def workspace_size(cfg: FmConfig) -> int:
    n = ctypes.c_size_t()
    _check(load().fm_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "fm_workspace_size")
    return n.value


def policy_create(cfg: FmConfig, weights: FmWeights, act_scales, workspace, ws_bytes: int, stream=None) -> int:
    """act_scales: host float32 numpy array [L][4] (or None for BF16 activations)."""
    import numpy as np
    out = ctypes.c_void_p()
    sc = None
    if act_scales is not None:
        act_scales = np.ascontiguousarray(act_scales, dtype=np.float32)
        sc = act_scales.ctypes.data
    _check(load().policy_create(ctypes.byref(cfg), ctypes.byref(weights), sc, _ptr(workspace), ws_bytes,
                                _stream(stream), ctypes.byref(out)), "policy_create")
    return out.value


def policy_destroy(p: int):
    _check(load().policy_destroy(p), "policy_destroy")


def fm_set_act_scales(p: int, act_scales, stream=None):
    import numpy as np
    a = np.ascontiguousarray(act_scales, dtype=np.float32)
    _check(load().fm_set_act_scales(p, a.ctypes.data, _stream(stream)), "fm_set_act_scales", p)


def set_prefix_kv(p: int, k, v, stream=None):
    _check(load().set_prefix_kv(p, _ptr(k), _ptr(v), _stream(stream)), "set_prefix_kv", p)


def refresh_prefix(p: int, tok_begin: int, tok_end: int, k, v, stream=None):
    _check(load().refresh_prefix(p, tok_begin, tok_end, _ptr(k), _ptr(v), _stream(stream)), "refresh_prefix", p)


def decode_actions(p: int, noise, actions, stream=None):
    _check(load().decode_actions(p, _ptr(noise), _ptr(actions), _stream(stream)), "decode_actions", p)


def decode_actions_host(p: int, noise_host, actions_host, stream=None):
    """noise_host / actions_host: pinned (or pageable) CPU float32 tensors."""
    _check(load().decode_actions_host(p, _ptr(noise_host), _ptr(actions_host), _stream(stream)),
           "decode_actions_host", p)


def session_workspace_size(base: int) -> int:
    n = ctypes.c_size_t()
    _check(load().fm_session_workspace_size(base, ctypes.byref(n)), "fm_session_workspace_size", base)
    return n.value


def session_create(base: int, workspace: int, ws_bytes: int, stream=None) -> int:
    out = ctypes.c_void_p()
    _check(load().fm_session_create(base, workspace, ws_bytes, _stream(stream), ctypes.byref(out)),
           "fm_session_create")
    return out.value


def session_fork(base: int, capsule, nbytes: int, capsule_on_device: bool, workspace: int, ws_bytes: int,
                 stream=None) -> int:
    out = ctypes.c_void_p()
    _check(load().fm_session_fork(base, _ptr(capsule), nbytes, int(capsule_on_device), workspace, ws_bytes,
                                  _stream(stream), ctypes.byref(out)), "fm_session_fork")
    return out.value


def philox_noise(out, seed: int, counter: int, raw_words=None, stream=None):
    """Fill the device float32 tensor `out` with the decision noise of stream
    (seed, counter); raw_words: None or a device int32/uint32 tensor of
    ceil(n/4)*4 words receiving the Philox output words."""
    _check(load().fm_philox_noise(_ptr(out), out.numel(), seed & (2 ** 64 - 1), counter & (2 ** 64 - 1),
                                  _ptr(raw_words), _stream(stream)), "fm_philox_noise")


def decode_actions_seeded(p: int, seed: int, counter: int, actions, stream=None):
    _check(load().fm_decode_actions_seeded(p, seed & (2 ** 64 - 1), counter & (2 ** 64 - 1), _ptr(actions),
                                           _stream(stream)), "fm_decode_actions_seeded", p)


def decode_warm(p: int, noise, executed: int, actions, stream=None):
    _check(load().fm_decode_warm(p, _ptr(noise), int(executed), _ptr(actions), _stream(stream)), "fm_decode_warm", p)


def episode_reset(p: int):
    _check(load().fm_episode_reset(p), "fm_episode_reset", p)


def last_timing(p: int, stream=None) -> dict:
    """Timestamps of the last decision: host submit (steady clock, ns) and the GPU
    globaltimer at its first kernel's start and last kernel's end; t_infer_ns is
    their difference."""
    t = FmTiming()
    _check(load().fm_last_timing(p, ctypes.byref(t), _stream(stream)), "fm_last_timing", p)
    return {"host_submit_ns": t.host_submit_ns, "device_start_ns": t.device_start_ns,
            "device_end_ns": t.device_end_ns, "t_infer_ns": t.device_end_ns - t.device_start_ns}


def state_size(p: int) -> int:
    n = ctypes.c_size_t()
    _check(load().fm_state_size(p, ctypes.byref(n)), "fm_state_size", p)
    return n.value


def snapshot_state(p: int, dst, nbytes: int, dst_on_device: bool, stream=None):
    _check(load().snapshot_state(p, _ptr(dst), nbytes, int(dst_on_device), _stream(stream)), "snapshot_state", p)


def restore_state(p: int, src, nbytes: int, src_on_device: bool, stream=None) -> int:
    """Returns the status (FM_ERR_STATE_MISMATCH = 6 is an expected outcome, not raised)."""
    st = load().restore_state(p, _ptr(src), nbytes, int(src_on_device), _stream(stream))
    if st not in (0, 6):
        _check(st, "restore_state", p)
    return st


def device_status(p: int, stream=None) -> int:
    w = ctypes.c_int()
    st = load().fm_device_status(p, _stream(stream), ctypes.byref(w))
    if st not in (0, 7):
        _check(st, "fm_device_status", p)
    return w.value


def standalone_status(stream=None) -> int:
    """Read and clear the error word of the policy-free building blocks (fm_test_skinny_gemm,
    fm_gemm_consumer, fm_gemm_consumer_noalloc) after synchronising the stream; 0 = no
    kernel of theirs abandoned a bounded wait."""
    w = ctypes.c_int()
    st = load().fm_standalone_status(_stream(stream), ctypes.byref(w))
    if st not in (0, 7):
        _check(st, "fm_standalone_status")
    return w.value


def named_buffer(p: int, name: str):
    """(device pointer, bytes) of a policy's named persistent buffer."""
    ptr, n = ctypes.c_void_p(), ctypes.c_size_t()
    _check(load().fm_named_buffer(p, name.encode(), ctypes.byref(ptr), ctypes.byref(n)), "fm_named_buffer")
    return ptr.value, n.value


def trace_size(p: int) -> int:
    n = ctypes.c_size_t()
    _check(load().fm_trace_size(p, ctypes.byref(n)), "fm_trace_size", p)
    return n.value


def decode_trace(p: int, noise, actions, trace, nbytes: int, stream=None):
    _check(load().fm_decode_trace(p, _ptr(noise), _ptr(actions), _ptr(trace), nbytes, _stream(stream)),
           "fm_decode_trace", p)


def warm_trace_size(p: int) -> int:
    n = ctypes.c_size_t()
    _check(load().fm_warm_trace_size(p, ctypes.byref(n)), "fm_warm_trace_size", p)
    return n.value


def decode_warm_trace(p: int, noise, executed: int, actions, trace, nbytes: int, stream=None):
    _check(load().fm_decode_warm_trace(p, _ptr(noise), int(executed), _ptr(actions), _ptr(trace), nbytes,
                                       _stream(stream)), "fm_decode_warm_trace", p)


def pdl_chain(ctas: int, threads: int, kernels: int, reps: int, pdl: bool, scratch, cluster: int = 1,
              writes: int = 0) -> float:
    """Microseconds per kernel of a CUDA graph of `kernels` dependent nearly empty kernels
    (programmatic dependent launch when pdl, else plain stream order), in clusters of
    `cluster` CTAs, each thread storing `writes` words after its wait. Synchronous;
    scratch: a device tensor of >= 4 * (1 + ctas * threads * writes) bytes."""
    us = ctypes.c_float()
    nbytes = scratch.numel() * scratch.element_size()
    _check(load().fm_test_pdl_chain(int(ctas), int(threads), int(kernels), int(reps), int(bool(pdl)), int(cluster),
                                    int(writes), _ptr(scratch), nbytes, ctypes.byref(us)), "fm_test_pdl_chain")
    return us.value


def grid_barrier(ctas: int, threads: int, rounds: int, mode: int, budget_ns: int, scratch, out, stream=None) -> int:
    """One cooperative launch running `rounds` grid-wide barriers (mode 0 release/acquire,
    1 fences around relaxed atomics, 2 a CTA that never arrives). Synchronous. out:
    device int64 [ctas][2] (ns over the completed rounds, rounds completed). Returns the
    status: 0, or 7 (FM_ERR_DEVICE) when a bounded wait ran out; raises on others."""
    st = load().fm_test_grid_barrier(int(ctas), int(threads), int(rounds), int(mode), int(budget_ns), _ptr(scratch),
                                     _ptr(out), _stream(stream))
    if st not in (0, 7):
        _check(st, "fm_test_grid_barrier")
    return st


def launch_kernel(p: int, layer: int, step: int, index: int, stream=None):
    """Launch one kernel of a layer-step exactly as the decision does (with programmatic
    dependent launch when the policy's flags hold FLAG_USE_PDL)."""
    _check(load().fm_test_launch_kernel(p, layer, step, index, _stream(stream)), "fm_test_launch_kernel", p)


def decode_timeline(p: int, noise, actions, buf, nbytes: int, stream=None):
    """One decision whose kernels record per-CTA timestamps into buf (see the header)."""
    _check(load().fm_decode_timeline(p, _ptr(noise), _ptr(actions), _ptr(buf), nbytes, _stream(stream)),
           "fm_decode_timeline", p)


def parse_timeline(raw) -> list:
    """Records of a timeline buffer (numpy uint8) as dicts: kind, grid, block, sm, t[15]."""
    count, cap = (int(v) for v in raw[:8].view(np.uint32))
    recs = raw[64:64 + 128 * min(count, cap)].view(np.uint64).reshape(-1, 16)
    out = []
    for r in recs:
        w = int(r[0])
        out.append({"kind": w & 0xff, "grid": ((w >> 8) & 0xfff, (w >> 20) & 0xfff),
                    "block": ((w >> 32) & 0xfff, (w >> 44) & 0xfff), "sm": (w >> 56) & 0xff,
                    "t": [int(x) for x in r[1:]]})
    return out


def kernel_count(p: int):
    a, b = ctypes.c_int(), ctypes.c_int()
    _check(load().fm_test_kernel_count(p, ctypes.byref(a), ctypes.byref(b)), "fm_test_kernel_count", p)
    return a.value, b.value


def attn_plan(p: int):
    """(keys per slice, slices) of the policy's attention."""
    a, b = ctypes.c_int(), ctypes.c_int()
    _check(load().fm_test_attn_plan(p, ctypes.byref(a), ctypes.byref(b)), "fm_test_attn_plan", p)
    return a.value, b.value


def fm_test_quant_e4m3(x, scale: float, codes, stream=None):
    _check(load().fm_test_quant_e4m3(_ptr(x), x.numel(), float(scale), _ptr(codes), _stream(stream)),
           "fm_test_quant_e4m3")


def fm_packed_weight_bytes(N: int, K: int, fmt: int) -> int:
    n = ctypes.c_size_t()
    _check(load().fm_packed_weight_bytes(N, K, fmt, ctypes.byref(n)), "fm_packed_weight_bytes")
    return n.value


def fm_pack_weight(w, gamma, N: int, K: int, fmt: int, packed, scale_out, stream=None):
    _check(load().fm_pack_weight(_ptr(w), _ptr(gamma), N, K, fmt, _ptr(packed), _ptr(scale_out),
                                 _stream(stream)), "fm_pack_weight")


def fm_test_skinny_gemm(a, M: int, K: int, w_packed, N: int, fmt: int, s: int, cluster_reduce: int,
                        partials, stream=None):
    _check(load().fm_test_skinny_gemm(_ptr(a), M, K, _ptr(w_packed), N, fmt, s, cluster_reduce,
                                      _ptr(partials), _stream(stream)), "fm_test_skinny_gemm")


def fm_test_skinny_gemm_tile(a, M: int, K: int, w_packed, N: int, fmt: int, s: int, cluster_reduce: int,
                             tile_rows: int, partials, stream=None):
    _check(load().fm_test_skinny_gemm_tile(_ptr(a), M, K, _ptr(w_packed), N, fmt, s, cluster_reduce, tile_rows,
                                           _ptr(partials), _stream(stream)), "fm_test_skinny_gemm_tile")


def fm_test_consumer(partials, nparts: int, M: int, N: int, s_a, s_w, bias, x, gate, scale, shift,
                     eps: float, s_q, q, act_fmt: int, stream=None):
    _check(load().fm_test_consumer(_ptr(partials), nparts, M, N, _ptr(s_a), _ptr(s_w), _ptr(bias), _ptr(x),
                                   _ptr(gate), _ptr(scale), _ptr(shift), float(eps), _ptr(s_q), _ptr(q),
                                   act_fmt, _stream(stream)), "fm_test_consumer")


def gemm_consumer_scratch_bytes(M: int, N: int, K: int, fmt: int, s: int) -> int:
    n = ctypes.c_size_t()
    _check(load().fm_gemm_consumer_scratch_bytes(M, N, K, fmt, s, ctypes.byref(n)), "fm_gemm_consumer_scratch_bytes")
    return n.value


def fm_gemm_consumer(a, M: int, K: int, w_packed, N: int, fmt: int, s: int, s_a, s_w, bias, x, gate, scale,
                     shift, eps: float, s_q, q, scratch, scratch_bytes: int, stream=None):
    _check(load().fm_gemm_consumer(_ptr(a), M, K, _ptr(w_packed), N, fmt, s, _ptr(s_a), _ptr(s_w), _ptr(bias),
                                   _ptr(x), _ptr(gate), _ptr(scale), _ptr(shift), float(eps), _ptr(s_q), _ptr(q),
                                   _ptr(scratch), scratch_bytes, _stream(stream)), "fm_gemm_consumer")


def fm_gemm_consumer_noalloc(a, M: int, K: int, w_packed, N: int, fmt: int, s: int, s_a, s_w, bias, x, gate,
                             scale, shift, eps: float, s_q, q, stream=None):
    """fm_gemm_consumer without a scratch argument, for callers that cannot allocate
    device memory: the library's built-in 8 MiB device array holds the partials."""
    _check(load().fm_gemm_consumer_noalloc(_ptr(a), M, K, _ptr(w_packed), N, fmt, s, _ptr(s_a), _ptr(s_w),
                                           _ptr(bias), _ptr(x), _ptr(gate), _ptr(scale), _ptr(shift), float(eps),
                                           _ptr(s_q), _ptr(q), _stream(stream)), "fm_gemm_consumer_noalloc")


def fm_test_layer(p: int, x_in, layer: int, step: int, x_out, q_out, stream=None):
    _check(load().fm_test_layer(p, _ptr(x_in), layer, step, _ptr(x_out), _ptr(q_out), _stream(stream)),
           "fm_test_layer", p)


# ---------------------------------------------------------------- convenience owner

class DeviceWeights:
    """Device copies of a policy's raw parameters and the fm_weights struct pointing at them.

    layers: list of per-layer dicts of numpy arrays ([out][in] fp32 GEMM weights,
    gamma1/2, w_mod (bf16 values), b_mod); final: dict with w_in, b_in, w_out, b_out,
    gamma_f, w_mod_f, b_mod_f; conds: [S][d] for cond == "given" workloads.
    """

    def __init__(self, cfg, layers, final, conds=None, device="cuda"):
        import torch
        self.device = torch.device(device)
        to = lambda a, dt=torch.float32: torch.from_numpy(np.ascontiguousarray(a)).to(self.device, dt)
        bf = lambda a: to(a, torch.bfloat16)
        self.tensors = []
        self._lw = (FmLayerWeights * cfg.L)()
        for l, d in enumerate(layers):
            t = {k: to(d[k]) for k in ("w_qkv", "w_o", "w_gu", "w_d", "gamma1", "gamma2", "b_mod")}
            t["w_mod"] = bf(d["w_mod"])
            self.tensors.append(t)
            for k in ("w_qkv", "w_o", "w_gu", "w_d", "gamma1", "gamma2", "w_mod", "b_mod"):
                setattr(self._lw[l], k, t[k].data_ptr())
        fin = {k: bf(final[k]) for k in ("w_in", "w_out", "w_mod_f")}
        fin.update({k: to(final[k]) for k in ("b_in", "b_out", "gamma_f", "b_mod_f")})
        if conds is not None:
            fin["conds"] = to(conds)
        self.tensors.append(fin)
        w = FmWeights()
        w.layers = self._lw
        for k in ("w_in", "b_in", "w_out", "b_out", "gamma_f", "w_mod_f", "b_mod_f"):
            setattr(w, k, fin[k].data_ptr())
        w.conds = fin["conds"].data_ptr() if conds is not None else None
        self.struct = w


class Policy:
    """Owns a policy's workspace and handle (and, optionally, its raw device weights).

    weights: a DeviceWeights, or (layers, final) numpy dicts as DeviceWeights takes
    them; the raw copies made here are released after create.
    """

    def __init__(self, cfg, layers=None, final=None, act_scales=None, conds=None,
                 flags: int = FLAG_USE_GRAPH | FLAG_USE_PDL, ksplit=(0, 0, 0, 0), device="cuda",
                 weights: "DeviceWeights | None" = None):
        import torch
        self.torch = torch
        self.cfg = cfg
        self.fmcfg = make_config(cfg, flags, ksplit)
        self.device = torch.device(device)
        own = weights is None
        if own:
            weights = DeviceWeights(cfg, layers, final, conds, device)
        self.ws_bytes = workspace_size(self.fmcfg)
        self.workspace = torch.empty(self.ws_bytes + 1024, dtype=torch.uint8, device=self.device)
        off = (-self.workspace.data_ptr()) % 1024
        self.ws_ptr = self.workspace.data_ptr() + off
        self.handle = policy_create(self.fmcfg, weights.struct, act_scales, self.ws_ptr, self.ws_bytes)
        if own:
            del weights
            torch.cuda.empty_cache()

    def set_prefix_kv(self, k, v, stream=None):
        set_prefix_kv(self.handle, k, v, stream)

    def refresh_prefix(self, b, e, k, v, stream=None):
        refresh_prefix(self.handle, b, e, k, v, stream)

    def buffer(self, name: str, dtype=None, shape=None):
        """Zero-copy torch view of a named persistent buffer (a session's shared
        buffers live in its base policy's workspace)."""
        ptr, n = named_buffer(self.handle, name)
        space = self.workspace
        base = getattr(self, "base", None)
        if base is not None and not (space.data_ptr() <= ptr < space.data_ptr() + space.numel()):
            space = base.workspace
        off = ptr - space.data_ptr()
        view = space[off:off + n]
        if dtype is not None:
            view = view.view(dtype)
        if shape is not None:
            count = 1
            for s_ in shape:
                count *= s_
            view = view[:count].view(*shape)
        return view

    def decode(self, noise, actions=None, stream=None):
        if actions is None:
            actions = self.torch.empty_like(noise)
        decode_actions(self.handle, noise, actions, stream)
        return actions

    def decode_seeded(self, seed: int, counter: int, actions=None, stream=None):
        """One decision from device-generated noise (seed, counter)."""
        if actions is None:
            actions = self.torch.empty((self.cfg.M, self.cfg.A), dtype=self.torch.float32, device=self.device)
        decode_actions_seeded(self.handle, seed, counter, actions, stream)
        return actions

    def last_timing(self, stream=None) -> dict:
        return last_timing(self.handle, stream)

    def decode_warm(self, noise, executed: int, actions=None, stream=None):
        """One-step warm start from the previous chunk (the full decision at an
        episode's start)."""
        if actions is None:
            actions = self.torch.empty_like(noise)
        decode_warm(self.handle, noise, executed, actions, stream)
        return actions

    def episode_reset(self):
        episode_reset(self.handle)

    def session(self, stream=None) -> "Session":
        """A new session sharing this policy's weights, with its own state."""
        return Session(self, stream=stream)

    def fork(self, capsule, capsule_on_device: bool = True, stream=None) -> "Session":
        """A new session started from a capsule of this policy (or of a session of it)."""
        return Session(self, capsule, capsule_on_device, stream)

    def close(self):
        if getattr(self, "handle", None):
            policy_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Session(Policy):
    """A session of a base Policy: shares the base's plan and read-only buffers,
    owns its state (prefix cache, scales, action buffer, activations) in its own
    workspace. Holds a reference to the base, which must outlive it."""

    def __init__(self, base: Policy, capsule=None, capsule_on_device: bool = True, stream=None):
        torch = base.torch
        self.torch = torch
        self.cfg = base.cfg
        self.fmcfg = base.fmcfg
        self.device = base.device
        self.base = base
        self.ws_bytes = session_workspace_size(base.handle)
        self.workspace = torch.empty(self.ws_bytes + 1024, dtype=torch.uint8, device=self.device)
        self.ws_ptr = self.workspace.data_ptr() + (-self.workspace.data_ptr()) % 1024
        if capsule is None:
            self.handle = session_create(base.handle, self.ws_ptr, self.ws_bytes, stream)
        else:
            self.handle = session_fork(base.handle, capsule, capsule.numel() * capsule.element_size(),
                                       capsule_on_device, self.ws_ptr, self.ws_bytes, stream)
