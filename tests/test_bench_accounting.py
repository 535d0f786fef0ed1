"""The benchmark's algorithmic byte and FLOP counts (the roofline numerators), checked
against totals worked out by hand from each workload's shapes, and the rule that the
dominant kernel's DRAM traffic is reported only while its source is the profiled one."""
import hashlib

import bench
import fm_synth


def test_expert_fp8_decision_bytes():
    # per layer (1 byte per FP8 weight): QKV 1280x1024 + O 1024x1024 + gate|up 8192x1024
    # + down 1024x4096 = 14,942,208; 18 layers x 10 steps = 180 layer-steps
    b = bench.algorithmic_bytes(fm_synth.config("expert_fp8_m50"))
    assert b["weights"] == 180 * 14_942_208 == 2_689_597_440
    # K and V of 788 prefix rows x 1 KV head x 128 dims x 2 bytes, every layer-step
    assert b["kv"] == 180 * 2 * 788 * 128 * 2 == 72_622_080
    # six fp32 modulation rows of 1024 per layer and step, two final rows per step
    assert b["mod"] == 10 * 18 * 6 * 1024 * 4 + 10 * 2 * 1024 * 4 == 4_505_600
    # W_in and W_out (bf16, 1024 x 32) once per step
    assert b["io"] == 10 * 2 * 1024 * 32 * 2 == 1_310_720
    assert b["total"] == 2_768_035_840


def test_expert_bf16_decision_bytes():
    b = bench.algorithmic_bytes(fm_synth.config("expert_bf16_m63"))
    assert b["weights"] == 2 * 2_689_597_440   # two bytes per weight
    assert b["total"] == 5_457_633_280


def test_world_action_model_decision_bytes_and_flops():
    cfg = fm_synth.config("wam_nvfp4_m256")
    # per layer: QKV 2560x2048 + O 2048x2048 + gate|up 16384x2048 + down 2048x8192 =
    # 59,768,832 weights at 4.5 bits (E2M1 code + an E4M3 scale per 16) = 33,619,968 B
    b = bench.algorithmic_bytes(cfg)
    assert b["weights"] == 280 * 33_619_968 == 9_413_591_040
    assert b["kv"] == 280 * 2 * 1024 * 2 * 128 * 2 == 293_601_280
    assert b["mod"] == 10 * 28 * 6 * 2048 * 4 + 10 * 2 * 2048 * 4 == 13_926_400
    assert b["total"] == 9_723_740_160
    f = bench.algorithmic_flops(cfg)
    assert f["gemm"] == 280 * 2 * 256 * 59_768_832 == 8_568_459_755_520
    # Q K^T and P V: 256 rows x 16 heads x (1024 + 256) keys x 128 dims, 2 FLOPs each
    assert f["attn"] == 280 * 2 * 2 * 256 * 16 * 1280 * 128 == 751_619_276_800


def test_expert_fp8_decision_flops():
    f = bench.algorithmic_flops(fm_synth.config("expert_fp8_m50"))
    assert f["gemm"] == 180 * 2 * 50 * 14_942_208 == 268_959_744_000
    assert f["attn"] == 180 * 2 * 2 * 50 * 8 * 838 * 128 == 30_892_032_000


def test_single_layer_bytes():
    # one FP8 layer (14,942,208), K and V of 64 prefix rows, its six modulation rows
    assert bench.layer_bytes(fm_synth.config("layer_fp8_m10")) == 14_942_208 + 2 * 64 * 128 * 2 + 6 * 1024 * 4
    assert bench.layer_bytes(fm_synth.config("layer_fp8_m10")) == 14_999_552


def test_traffic_only_while_the_source_is_the_profiled_one(tmp_path, monkeypatch):
    src = tmp_path / "flow_matching_action_denoise_gb300" / "csrc" / "gemm.cu"
    src.parent.mkdir(parents=True)
    src.write_bytes(b"// kernel source\n")
    (tmp_path / "profiles").mkdir()
    sha = hashlib.sha256(src.read_bytes()).hexdigest()[:16]
    (tmp_path / "profiles" / "p.md").write_text(f"Kernel source sha256 prefix: {sha}\ntraffic_bytes_per_launch: 123\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("p.md") == 123
    src.write_bytes(b"// kernel source, changed\n")
    assert bench.profiled_traffic("p.md") is None
    assert bench.profiled_traffic("missing.md") is None
