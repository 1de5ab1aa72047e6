"""The JSON line of bench.py's reference arm (the CPU oracle, no GPU needed)
carries every key of the benchmark contract."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_decode", "--steps", "2", "--warmup", "1", "--ref-seconds", "0.6"],
                       capture_output=True, text=True, cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"].startswith("tiny_decode")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_roofline_arithmetic_mixed_tick():
    """The algorithmic work the bench divides by: the mixed tick's chunks are
    2048 rows after prefixes 0 and 3072 (visible query-key pairs 2,098,176 +
    8,389,632, times 4 * d flop per pair per q head), and every roofline is the
    work of one launch over its average duration."""
    sys.path.insert(0, ROOT)
    import bench
    from paged_kv_attention_mapping_gb300 import workloads as W
    w = W.make_workload("mixed_tick")
    work = bench.tick_work(w)
    pairs = (2048 * 2049 // 2) + (2048 * 3072 + 2048 * 2049 // 2)
    assert pairs == 2_098_176 + 8_389_632
    assert work["prefill_flops"] == 4 * 128 * 32 * pairs == 171_832_246_272
    # decode rows: K and V of every row's context, 8 KV heads x 128 dims x 2 bytes
    dec = [r for r in w.requests if r.q_len == 1]
    assert work["decode_kv_bytes"] == sum(2 * r.kv_len * 8 * 128 * 2 for r in dec)
    assert work["append_bytes"] == 2 * w.total_q * 8 * 128 * (2 + 2)
    peaks = dict(hbm_gbs=1000.0, bf16_tflops=1000.0, source="test")
    ktimes = {"prefill_tc": (2, 2 * 0.1718322462720), "decode": (1, 1.0)}   # ms totals
    r = bench.kernel_roofline("prefill_tc", ktimes, work, peaks, "none")
    assert abs(r["achieved"] - 1000.0) < 1e-6 and abs(r["frac"] - 1.0) < 1e-9 and r["unit"] == "TFLOP/s"
    r = bench.kernel_roofline("decode", ktimes, work, peaks, "none")
    assert abs(r["achieved"] - work["decode_bytes"] / 1e-3 / 1e9) < 1e-6
    t = bench.tick_roofline(work, peaks, 1.0)
    assert abs(t["t_serial_us"] - t["t_mem_us"] - t["t_flop_us"]) < 1e-9
    assert abs(t["t_flop_us"] - 171.832246272) < 1e-6
