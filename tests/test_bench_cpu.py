"""The benchmark's reference arm on the CPU: `bench.py --impl reference` times the
float64 oracle (the reference arm of this build) and prints one JSON line with the
driver contract's keys. Run on the tiny workload with a short sample so that the CPU
suite stays quick; the GPU arm is exercised on a GB300."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         capture_output=True, text=True, timeout=600, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.strip()]
    assert len(lines) == 1, out
    return json.loads(lines[0])


def test_reference_arm_prints_the_contract_line():
    d = _run("--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "0")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 2 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny" and d["config"]["batch"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_names_a_micro_batch():
    d = _run("--impl", "reference", "--workload", "tiny", "--batch", "2", "--steps", "1",
             "--warmup", "0")
    assert d["config"]["workload"] == "tiny-b2" and d["config"]["batch"] == 2


def test_long_workload_sample_extrapolates_from_component_rates():
    """Past 4096 tokens one sample times the oracle's projection of one attention
    shard over the whole sequence, the attention of 256 sampled rows and their MLP;
    the full-layer time is the sum of the layer's three FLOP classes at those rates."""
    sys.path.insert(0, ROOT)
    import bench
    import tsp_inputs
    cfg = tsp_inputs.LayerConfig("long-narrow", 2, 8192, 256, 4, 688, 7)
    bits = tsp_inputs.layer_inputs(cfg)
    t, tokens_per_s, rates = bench.oracle_sample(cfg, bits)
    assert t > 0 and tokens_per_s > 0
    S, H, F = cfg.S, cfg.hidden, cfg.ffn
    t_full = (8.0 * S * H * H / (rates["projection_gflops"] * 1e9)
              + 2.0 * H * S * (S + 1) / (rates["attention_gflops"] * 1e9)
              + 6.0 * S * H * F / (rates["mlp_gflops"] * 1e9))
    assert abs(t_full - rates["extrapolated_layer_s"]) <= 0.05 * t_full + 0.1
    assert abs(S / t_full - tokens_per_s) <= 0.05 * tokens_per_s
    assert "EXTRAPOLATED" in bench.oracle_sample_desc(cfg)
