"""Seeded synthetic inputs for the flow-matching action-decoder workloads.

This module is shared by the CPU oracle, the tests and the benchmark. It holds
the workload shapes and the seeded random draws only: no step of the method's
arithmetic (no folding, quantisation, normalisation or matrix product) lives
here. Values that the workloads store in bf16 are rounded with torch's dtype
cast, a plain format conversion.

Every tensor is drawn from its own counter-style stream,
``numpy.random.default_rng([seed, tag, layer])`` (PCG64 seeded through
SeedSequence), so any layer can be regenerated on its own. Draws are float32.

Distributions (FlashRT-PAI pages, "CUDA Graph vs graph simplification" for the
RMSNorm/fold form; the workload definitions fix the rest):
  * layer weights W ~ N(0, 0.02^2), stored [out][in] (the GEMM's N x K);
  * gamma = 1 + 0.1 * N(0, 1)  (fixed per-channel norm scale, folded into W);
  * modulation weights W_mod ~ N(0, 0.02^2) rounded to bf16, b_mod = 0;
  * in/out projections W_in, W_out ~ N(0, 0.02^2) rounded to bf16,
    biases b_in, b_out ~ N(0, 0.02^2) in fp32;
  * prefix K/V cache ~ N(0, 1) rounded to bf16, layout [L][P][Hkv][Dh];
  * noise ~ N(0, 1), [M][A] fp32; single-layer x and cond ~ N(0, 1).
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np

__all__ = [
    "Config", "CONFIGS", "config", "rng", "layer_weights", "final_weights",
    "prefix_kv", "prefix_kv_rows", "noise", "layer_input", "gemm_case",
    "default_act_scales",
]


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    L: int            # decoder layers
    S: int            # Euler steps per decision
    M: int            # action-chunk rows
    d: int            # model width
    H: int            # query heads
    Hkv: int          # key/value heads
    Dh: int           # head dim
    F: int            # GeGLU hidden width
    P: int            # prefix tokens in the KV cache
    A: int            # action dim
    weight_fmt: str   # "fp8" | "bf16" | "nvfp4"
    act_fmt: str      # "fp8" | "bf16"
    seed: int
    cond: str = "time"   # "time": sinusoidal t-embedding; "given": cond vector drawn per step
    eps: float = 1e-6
    attn_fmt: str = "bf16"   # "bf16" | "fp8": attention operands (Q, K, V, P)
    warm_t: float = 0.0      # flow time of the one-step warm start (0: none)

    @property
    def n_qkv(self) -> int:
        return (self.H + 2 * self.Hkv) * self.Dh

    @property
    def gemm_shapes(self):
        """(N, K) of the four per-layer GEMMs: QKV, O, gate|up, down."""
        return [(self.n_qkv, self.d), (self.d, self.H * self.Dh),
                (2 * self.F, self.d), (self.d, self.F)]


CONFIGS = {
    # one action-decoder layer, one denoise step, given cond vector
    "layer_fp8_m10": Config("layer_fp8_m10", L=1, S=1, M=10, d=1024, H=8, Hkv=1, Dh=128,
                            F=4096, P=64, A=32, weight_fmt="fp8", act_fmt="fp8",
                            seed=0, cond="given"),
    # full action expert, FP8: 18 layers x 10 steps, M=50, prefix 3x256+20
    "expert_fp8_m50": Config("expert_fp8_m50", L=18, S=10, M=50, d=1024, H=8, Hkv=1, Dh=128,
                             F=4096, P=788, A=32, weight_fmt="fp8", act_fmt="fp8", seed=1),
    # matched 16-bit variant, M=63
    # the same expert with FP8 attention (E4M3 Q, K, V and probabilities)
    "expert_fp8attn_m50": Config("expert_fp8attn_m50", L=18, S=10, M=50, d=1024, H=8, Hkv=1, Dh=128,
                                 F=4096, P=788, A=32, weight_fmt="fp8", act_fmt="fp8", seed=1,
                                 attn_fmt="fp8"),
    "expert_bf16_m63": Config("expert_bf16_m63", L=18, S=10, M=63, d=1024, H=8, Hkv=1, Dh=128,
                              F=4096, P=788, A=32, weight_fmt="bf16", act_fmt="bf16", seed=3),
    # world-action-model-sized decoder, NVFP4 weights, FP8 activations
    "wam_nvfp4_m256": Config("wam_nvfp4_m256", L=28, S=10, M=256, d=2048, H=16, Hkv=2, Dh=128,
                             F=8192, P=1024, A=32, weight_fmt="nvfp4", act_fmt="fp8", seed=4),
    # the same decoder with four-bit activations too (W4A4: NVFP4 weights and activations)
    "wam_w4a4_m256": Config("wam_w4a4_m256", L=28, S=10, M=256, d=2048, H=16, Hkv=2, Dh=128,
                            F=8192, P=1024, A=32, weight_fmt="nvfp4", act_fmt="nvfp4", seed=4),
}


def config(name: str, **overrides) -> Config:
    return dataclasses.replace(CONFIGS[name], **overrides)


def _tag(name: str) -> int:
    return zlib.crc32(name.encode())


def rng(seed: int, tag: str, index: int = 0) -> np.random.Generator:
    return np.random.default_rng([int(seed), _tag(tag), int(index)])


def _normal(seed, tag, index, shape, std=1.0, mean=0.0) -> np.ndarray:
    x = rng(seed, tag, index).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return x


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (torch cast, round-to-nearest-even); returns float32."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).to(torch.float32).numpy()


def layer_weights(cfg: Config, layer: int) -> dict:
    """Per-layer tensors, [out][in] layout, float32 (W_mod holds bf16 values)."""
    s, d = cfg.seed, cfg.d
    out = {}
    for name, (n, k) in zip(("w_qkv", "w_o", "w_gu", "w_d"), cfg.gemm_shapes):
        out[name] = _normal(s, name, layer, (n, k), std=0.02)
    out["gamma1"] = _normal(s, "gamma1", layer, (d,), std=0.1, mean=1.0)
    out["gamma2"] = _normal(s, "gamma2", layer, (d,), std=0.1, mean=1.0)
    out["w_mod"] = to_bf16_values(_normal(s, "w_mod", layer, (6 * d, d), std=0.02))
    out["b_mod"] = np.zeros((6 * d,), np.float32)
    return out


def final_weights(cfg: Config) -> dict:
    s, d, a = cfg.seed, cfg.d, cfg.A
    return {
        "w_in": to_bf16_values(_normal(s, "w_in", 0, (d, a), std=0.02)),
        "b_in": _normal(s, "b_in", 0, (d,), std=0.02),
        "w_out": to_bf16_values(_normal(s, "w_out", 0, (a, d), std=0.02)),
        "b_out": _normal(s, "b_out", 0, (a,), std=0.02),
        "gamma_f": _normal(s, "gamma_f", 0, (d,), std=0.1, mean=1.0),
        "w_mod_f": to_bf16_values(_normal(s, "w_mod_f", 0, (2 * d, d), std=0.02)),
        "b_mod_f": np.zeros((2 * d,), np.float32),
    }


def prefix_kv(cfg: Config, version: int = 0):
    """Prefix K and V caches, [L][P][Hkv][Dh], bf16 values as float32."""
    shape = (cfg.L, cfg.P, cfg.Hkv, cfg.Dh)
    k = to_bf16_values(_normal(cfg.seed, "prefix_k", version, shape))
    v = to_bf16_values(_normal(cfg.seed, "prefix_v", version, shape))
    return k, v


def prefix_kv_rows(cfg: Config, version: int, rows: int):
    """Fresh rows [0, rows) of every layer's K and V (an observation refresh)."""
    shape = (cfg.L, rows, cfg.Hkv, cfg.Dh)
    k = to_bf16_values(_normal(cfg.seed, "refresh_k", version, shape))
    v = to_bf16_values(_normal(cfg.seed, "refresh_v", version, shape))
    return k, v


def noise(cfg: Config, decision: int = 0) -> np.ndarray:
    return _normal(cfg.seed, "noise", decision, (cfg.M, cfg.A))


def step_conds(cfg: Config) -> np.ndarray:
    """Per-step cond vectors for cond == "given" workloads, [S][d] ~ N(0, 1)."""
    return _normal(cfg.seed, "cond", 0, (cfg.S, cfg.d))


def layer_input(cfg: Config) -> np.ndarray:
    """Residual-stream input x [M][d] ~ N(0, 1) for single-layer workloads."""
    return _normal(cfg.seed, "x", 0, (cfg.M, cfg.d))


def default_act_scales(cfg: Config) -> np.ndarray:
    """A data-independent static activation-scale table [L][4] (fp32; [L][7] with FP8 attention).

    Quant points per layer: 0 = pre-attention norm output, 1 = attention output,
    2 = pre-MLP norm output, 3 = GeGLU output. Used where no calibrated table is
    supplied; the values are plain constants sized for the distributions above.
    """
    base = [24.0, 1.0, 24.0, 16.0]
    if cfg.attn_fmt == "fp8":   # FP8 attention adds Q, K, V (columns 4-6 of an [L][7] table)
        base += [8.0, 8.0, 8.0]
    # E4M3 codes: amax / 448; four-bit activations: the tensor scale amax / (448 * 6)
    div = np.float32(2688.0) if cfg.act_fmt == "nvfp4" else np.float32(448.0)
    return np.tile(np.array(base, np.float32) / div, (cfg.L, 1)).astype(np.float32)


def gemm_case(M: int, K: int, N: int, seed: int = 2, integer: bool = False) -> dict:
    """Standalone skinny-GEMM + consumer case.

    A [M][K] ~ N(0,1), W [N][K] ~ N(0, 0.02^2); consumer tensors: bias [N] ~ N(0, 0.02^2),
    x [M][N] ~ N(0,1), gate/scale/shift [N] ~ N(0, 0.1^2).
    integer=True draws A, W uniformly from the integers -3..3 (exact in E4M3 with
    scale 1), for the bit-exact split-K invariance check.
    """
    idx = M * 1_000_003 + K * 101 + N
    if integer:
        a = rng(seed, "int_a", idx).integers(-3, 4, size=(M, K)).astype(np.float32)
        w = rng(seed, "int_w", idx).integers(-3, 4, size=(N, K)).astype(np.float32)
    else:
        a = _normal(seed, "gemm_a", idx, (M, K))
        w = _normal(seed, "gemm_w", idx, (N, K), std=0.02)
    return {
        "a": a, "w": w,
        "bias": _normal(seed, "gemm_bias", idx, (N,), std=0.02),
        "x": _normal(seed, "gemm_x", idx, (M, N)),
        "gate": _normal(seed, "gemm_gate", idx, (N,), std=0.1),
        "scale": _normal(seed, "gemm_scale", idx, (N,), std=0.1),
        "shift": _normal(seed, "gemm_shift", idx, (N,), std=0.1),
    }
