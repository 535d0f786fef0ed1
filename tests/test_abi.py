"""The C-ABI library loads and exports every entry point include/fmad.h declares,
and host-side validation returns the documented status codes (no GPU needed:
nothing here launches a kernel)."""
import ctypes
import os
import re

import pytest

import fm_synth
import flow_matching_action_denoise_gb300 as fmad

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    text = open(os.path.join(ROOT, "include", "fmad.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\([^;{]*\)\s*;", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fmad.LIB_PATH):
        from flow_matching_action_denoise_gb300 import build
        build.build()
    return fmad.load()


def test_header_declares_the_boundary():
    names = header_functions()
    for required in ["policy_create", "set_prefix_kv", "refresh_prefix", "decode_actions",
                     "snapshot_state", "restore_state", "policy_destroy"]:
        assert required in names
    assert sorted(names) == sorted(fmad.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in fmad.STATUS.items():
        assert lib.fm_status_string(code).decode() == name


def test_workspace_size_and_validation(lib):
    cfg = fmad.make_config(fm_synth.config("expert_fp8_m50"))
    n = fmad.workspace_size(cfg)
    # packed FP8 weights alone are 18 x 14.94 MB
    assert n > 18 * 14_942_208
    bad = fmad.make_config(fm_synth.config("expert_fp8_m50"))
    bad.M = 300
    with pytest.raises(fmad.FmError) as e:
        fmad.workspace_size(bad)
    assert e.value.status == 2
    bad = fmad.make_config(fm_synth.config("expert_fp8_m50"))
    bad.abi_version = 99
    with pytest.raises(fmad.FmError) as e:
        fmad.workspace_size(bad)
    assert e.value.status == 1
    bad = fmad.make_config(fm_synth.config("expert_fp8_m50"), ksplit=(3, 0, 0, 0))
    with pytest.raises(fmad.FmError) as e:
        fmad.workspace_size(bad)
    assert e.value.status == 2


def test_policy_create_rejects_bad_arguments_without_touching_the_gpu(lib):
    cfg = fmad.make_config(fm_synth.config("expert_fp8_m50"))
    out = ctypes.c_void_p()
    w = fmad.FmWeights()
    # NULL weights
    st = lib.policy_create(ctypes.byref(cfg), ctypes.byref(w), None, 1024, 1 << 30, None, ctypes.byref(out))
    assert st == 1 and out.value is None
    assert b"NULL" in lib.fm_last_error(None)


def test_policy_free_exports_validate(lib):
    n = ctypes.c_size_t()
    assert lib.fm_packed_weight_bytes(1280, 1024, fmad.FMT_FP8, ctypes.byref(n)) == 0
    assert n.value == 1280 * 1024
    assert lib.fm_packed_weight_bytes(1280, 1000, fmad.FMT_FP8, ctypes.byref(n)) == 2
    assert lib.fm_packed_weight_bytes(1280, 1024, fmad.FMT_BF16, ctypes.byref(n)) == 0
    assert n.value == 1280 * 1024 * 2
    # GEMM: split must divide the K-block count; pointers are checked before any launch
    assert lib.fm_test_skinny_gemm(None, 10, 1024, None, 1024, fmad.FMT_FP8, 8, 8, None, None) == 1
    assert lib.fm_test_skinny_gemm(1024, 10, 1024, 1024, 1024, fmad.FMT_FP8, 3, 1, 1024, None) == 2
    assert lib.fm_test_skinny_gemm(1024, 300, 1024, 1024, 1024, fmad.FMT_FP8, 1, 1, 1024, None) == 2
    assert lib.fm_test_skinny_gemm(1032, 10, 1024, 1024, 1024, fmad.FMT_FP8, 1, 1, 1024, None) == 3
    assert lib.fm_test_quant_e4m3(1024, 16, ctypes.c_float(0.0), 1024, None) == 1


def test_warm_start_config_validation(lib):
    base = fmad.make_config(fm_synth.config("expert_fp8_m50"))
    warm = fmad.make_config(fm_synth.config("expert_fp8_m50", warm_t=0.5))
    # the warm start adds one modulation row: [L][6][d] + [2][d] fp32 and its [d] double cond
    extra = fmad.workspace_size(warm) - fmad.workspace_size(base)
    row = 18 * 6 * 1024 * 4 + 2 * 1024 * 4 + 1024 * 8
    assert row <= extra < row + 3 * 1024
    for t in (-0.1, 1.5, float("nan")):
        bad = fmad.make_config(fm_synth.config("expert_fp8_m50", warm_t=t))
        with pytest.raises(fmad.FmError) as e:
            fmad.workspace_size(bad)
        assert e.value.status == 1
    given = fmad.make_config(fm_synth.config("layer_fp8_m10", warm_t=0.5))   # cond given per step
    with pytest.raises(fmad.FmError) as e:
        fmad.workspace_size(given)
    assert e.value.status == 1


def test_noise_and_warm_entry_points_validate_without_a_gpu(lib):
    assert lib.fm_philox_noise(None, 16, 1, 2, None, None) == 1
    assert lib.fm_decode_warm(None, None, 0, None, None) == 1
    assert lib.fm_episode_reset(None) == 1
    assert lib.fm_last_timing(None, None, None) == 1
    assert lib.fm_decode_actions_seeded(None, 1, 2, None, None) == 1


def test_session_entry_points_validate_without_a_gpu(lib):
    n = ctypes.c_size_t()
    assert lib.fm_session_workspace_size(None, ctypes.byref(n)) == 1
    out = ctypes.c_void_p(1)
    assert lib.fm_session_create(None, 1024, 1 << 20, None, ctypes.byref(out)) == 1 and out.value is None
    assert lib.fm_session_fork(None, None, 0, 1, 1024, 1 << 20, None, ctypes.byref(out)) == 1
    assert lib.policy_destroy(None) == 1


def test_binding_struct_mirrors_match_the_library(lib):
    sizes = [ctypes.c_size_t() for _ in range(4)]
    assert lib.fm_abi_sizes(*[ctypes.byref(s) for s in sizes]) == 0
    cfg, w, lw, t = (s.value for s in sizes)
    assert cfg == ctypes.sizeof(fmad.FmConfig)
    assert w == ctypes.sizeof(fmad.FmWeights)
    assert lw == ctypes.sizeof(fmad.FmLayerWeights)
    assert t == ctypes.sizeof(fmad.FmTiming)


def test_attention_plan_limits_are_validated(lib):
    # keys = P + M must fit 8 key slices of at most 192 keys
    ok = fmad.make_config(fm_synth.config("expert_fp8_m50", P=1536 - 50))
    assert fmad.workspace_size(ok) > 0
    bad = fmad.make_config(fm_synth.config("expert_fp8_m50", P=1536 - 49))
    with pytest.raises(fmad.FmError) as e:
        fmad.workspace_size(bad)
    assert e.value.status == 2 and "attention plan" in str(e.value)


def test_handoff_diagnostics_validate_without_a_gpu(lib):
    # host addresses stand in for device buffers: every call below is rejected before
    # any CUDA call, and the alignment case needs a pointer that is not 16-byte aligned
    buf = ctypes.create_string_buffer(4096 + 16)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    out = ctypes.c_ulonglong()
    us = ctypes.c_float()
    gb = lib.fm_test_grid_barrier
    assert gb(4, 128, 10, 0, 10**6, None, ctypes.byref(out), None) == 1          # NULL scratch
    assert gb(4, 128, 10, 0, 10**6, base, None, None) == 1                       # NULL result
    assert gb(0, 128, 10, 0, 10**6, base, ctypes.byref(out), None) == 2          # no CTAs
    assert gb(4, 100, 10, 0, 10**6, base, ctypes.byref(out), None) == 2          # threads not a warp multiple
    assert gb(4, 128, 10, 3, 10**6, base, ctypes.byref(out), None) == 2          # unknown mode
    assert gb(4, 128, 10, 0, 10, base, ctypes.byref(out), None) == 2             # wait budget under 1 us
    assert gb(4, 128, 10, 0, 10**6, base + 4, ctypes.byref(out), None) == 3      # scratch misaligned
    pc = lib.fm_test_pdl_chain
    assert pc(8, 128, 4, 2, 1, 1, 0, None, 4096, ctypes.byref(us)) == 1          # NULL scratch
    assert pc(8, 128, 4, 2, 1, 1, 0, base, 4096, None) == 1                      # NULL result
    assert pc(8, 128, 4, 2, 1, 3, 0, base, 4096, ctypes.byref(us)) == 2          # cluster not a power of two
    assert pc(6, 128, 4, 2, 1, 4, 0, base, 4096, ctypes.byref(us)) == 2          # CTAs not whole clusters
    assert pc(8, 128, 0, 2, 1, 1, 0, base, 4096, ctypes.byref(us)) == 2          # no kernels
    assert pc(8, 128, 4, 2, 1, 1, 65, base, 4096, ctypes.byref(us)) == 2         # too many writes per thread
    # 8 CTAs x 128 threads x 1 write needs 4 * (1 + 1024) bytes
    assert pc(8, 128, 4, 2, 1, 1, 1, base, 4 * 1025 - 1, ctypes.byref(us)) == 4


def test_policy_diagnostics_reject_a_null_policy(lib):
    a, b = ctypes.c_int(-1), ctypes.c_int(-1)
    assert lib.fm_test_attn_plan(None, ctypes.byref(a), ctypes.byref(b)) == 1
    assert (a.value, b.value) == (-1, -1)   # outputs untouched on error
    assert lib.fm_test_launch_kernel(None, 0, 0, 0, None) == 1
    assert lib.fm_standalone_status(None, None) == 1


@pytest.mark.parametrize("field,value,status", [
    ("act_fmt", fmad.FMT_BF16, 1),      # FP8 weights with bf16 activations: no such pair
    ("attn_fmt", fmad.FMT_NVFP4, 1),    # attention runs in bf16 or E4M3 only
    ("cond_mode", 7, 1),
    ("Dh", 64, 2),                      # the kernels are built for 128-dim heads
    ("Hkv", 3, 2),                      # 8 query heads do not share 3 KV heads evenly
    ("d", 1000, 2),                     # not a multiple of 128
    ("F", 4100, 2),
    ("A", 33, 2),
    ("M", 0, 2),
    ("rms_eps", 0.0, 1),
])
def test_config_preconditions(lib, field, value, status):
    cfg = fmad.make_config(fm_synth.config("expert_fp8_m50"))
    setattr(cfg, field, value)
    with pytest.raises(fmad.FmError) as e:
        fmad.workspace_size(cfg)
    assert e.value.status == status


def test_unsupported_mode_combinations_and_splits(lib):
    # E4M3 attention is built for FP8 weights and activations only
    cfg = fmad.make_config(fm_synth.config("expert_bf16_m63"))
    cfg.attn_fmt = fmad.FMT_FP8
    with pytest.raises(fmad.FmError) as e:
        fmad.workspace_size(cfg)
    assert e.value.status == 8
    # the QKV and gate|up GEMMs reduce every K slice inside one cluster (at most 8)
    with pytest.raises(fmad.FmError) as e:
        fmad.workspace_size(fmad.make_config(fm_synth.config("expert_fp8_m50"), ksplit=(16, 0, 0, 0)))
    assert e.value.status == 2 and "1, 2, 4 or 8" in str(e.value)
    # a split must divide the K blocks: the down GEMM's K = 4096 holds 32 FP8 blocks
    with pytest.raises(fmad.FmError) as e:
        fmad.workspace_size(fmad.make_config(fm_synth.config("expert_fp8_m50"), ksplit=(0, 0, 0, 5)))
    assert e.value.status == 2
    # with NVFP4 weights the gate|up GEMM applies GeGLU itself and keeps its whole K
    with pytest.raises(fmad.FmError) as e:
        fmad.workspace_size(fmad.make_config(fm_synth.config("wam_nvfp4_m256"), ksplit=(0, 0, 2, 0)))
    assert e.value.status == 2 and "GeGLU" in str(e.value)
    # the accepted splits still size a workspace
    assert fmad.workspace_size(fmad.make_config(fm_synth.config("expert_fp8_m50"), ksplit=(4, 4, 2, 8))) > 0
