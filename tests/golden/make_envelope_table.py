"""Tabulate the oracle's own rounding envelope of a whole decision against its depth
(layers L x Euler steps S), and write envelope_table_<workload>.txt.

A decision re-rounds its activations at every quant point of every layer-step (E4M3
codes in FP8 mode, bf16 values in BF16 mode). A value within fp32 rounding distance
of a rounding boundary may round either way in any fp32 implementation of the same
arithmetic, and each flip moves every later activation, so the spread grows with
the number of layer-steps. The envelope at (L, S) is the largest action difference,
relative to RMS(actions), between the oracle and three perturbed copies of it whose
rounding inputs are moved by at most 2^-23 relative:
  * fp32: the value is first rounded to fp32;
  * jitter 1, jitter 2: the value is multiplied by (1 + 2^-23 u), u uniform in
    [-1, 1) from a seeded generator (seeds 1 and 2).
The policies are the workload's first L layers (their weights, prefix rows and
calibrated activation scales) run for S steps on noise draw 0.
Run: python tests/golden/make_envelope_table.py [workload ...]
(default: expert_fp8_m50 and expert_bf16_m63)
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import fm_synth  # noqa: E402
from oracle import codecs as C  # noqa: E402
from oracle import model as O  # noqa: E402

DEPTHS_L = (1, 2, 6, 18)
DEPTHS_S = (1, 2, 10)


def perturbations(fmt):
    """(name, install, uninstall) triples patching the oracle's rounding inputs."""
    plain_q, plain_b = O.quant_codes, C.bf16

    def fp8_with(move):
        def q(h, s, f):
            if f == "fp8":
                return C.e4m3(C.fp32(move(np.asarray(h, np.float64)) * O.recip32(s)))
            return plain_q(h, s, f)
        return q

    def jitter(seed):
        rng = np.random.default_rng(seed)
        return lambda x: x * (1.0 + 2.0 ** -23 * rng.uniform(-1.0, 1.0, np.shape(x)))

    moves = [("fp32", lambda: C.fp32)] + [(f"jitter{s}", (lambda s=s: jitter(s))) for s in (1, 2)]
    out = []
    for name, make in moves:
        if fmt == "fp8":
            def install(make=make):
                O.quant_codes = fp8_with(make())

            def uninstall():
                O.quant_codes = plain_q
        else:
            def install(make=make):
                mv = make()
                C.bf16 = lambda x: plain_b(mv(np.asarray(x, np.float64)))

            def uninstall():
                C.bf16 = plain_b
        out.append((name, install, uninstall))
    return out


def envelope(name, L, S, layers_all, final, kp_all, vp_all, sc_all):
    cfg = fm_synth.config(name, L=L, S=S)
    model = O.Model(cfg, layers_all[:L], final)
    kp, vp = kp_all[:L], vp_all[:L]
    sc = None if sc_all is None else sc_all[:L]
    nz = fm_synth.noise(cfg, 0)
    ref = O.decode(model, nz, kp, vp, sc)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    envs = []
    for _, install, uninstall in perturbations(cfg.act_fmt):
        install()
        try:
            alt = O.decode(model, nz, kp, vp, sc)
        finally:
            uninstall()
        envs.append(float(np.max(np.abs(alt - ref)) / rms))
    return envs


def main(name):
    base = fm_synth.config(name)
    layers_all = [fm_synth.layer_weights(base, l) for l in range(base.L)]
    final = fm_synth.final_weights(base)
    kp_all, vp_all = fm_synth.prefix_kv(base)
    sc_all = None
    if base.act_fmt == "fp8":
        sc_all = np.loadtxt(os.path.join(HERE, f"act_scales_{name}.txt"), dtype=np.float32, ndmin=2)
    rows = []
    for L in DEPTHS_L:
        for S in DEPTHS_S:
            envs = envelope(name, L, S, layers_all, final, kp_all, vp_all, sc_all)
            rows.append((L, S, max(envs), envs))
            print(name, L, S, max(envs), flush=True)
    path = os.path.join(HERE, f"envelope_table_{name}.txt")
    with open(path, "w") as f:
        f.write("# L S envelope(max) fp32 jitter1 jitter2 : max|perturbed oracle - oracle| / RMS(oracle actions),\n")
        f.write(f"# first L layers of {name}, S Euler steps, noise draw 0\n")
        for L, S, env, envs in rows:
            f.write(f"{L} {S} {env:.6e} " + " ".join(f"{e:.6e}" for e in envs) + "\n")
    print(path)


if __name__ == "__main__":
    for n in sys.argv[1:] or ("expert_fp8_m50", "expert_bf16_m63"):
        main(n)
