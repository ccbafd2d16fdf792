"""bench.py's reference arm runs on the CPU (it times the oracle), so its
JSON line is checked here without a GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1", "--cpu-sample", "2"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] == "llama3_8b_b64"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_algorithmic_bytes_follow_the_keep_sets_and_the_layout():
    """The bench's algorithmic bytes: each kept token's K and V rows of every
    kv head once (plus its two fp32 scales per kv head in FP8 / INT8 pools),
    counted from the pinned keep-sets, and the workloads' published totals
    (about 1.14 GB for the batch-64 Llama-3-8B layer, 1.107 GB for 4 x 128K
    FP8 tokens with scales)."""
    import random

    import bench
    import oracle
    import workloads

    modes = {"full": oracle.MASK_FULL, "sliding": oracle.MASK_SLIDING, "sink_window": oracle.MASK_SINK_WINDOW}
    rng = random.Random(3)
    for name, make in workloads.ALL.items():
        wl = make()
        elem = {"fp32": 4, "bf16": 2, "fp8": 1, "int8": 1}[wl.kv_dtype]
        scales = 2 * wl.n_kv_heads * 4 if wl.kv_dtype in ("fp8", "int8") else 0
        assert bench._kv_bytes_per_token(wl) == 2 * wl.n_kv_heads * wl.head_dim * elem + scales, name
        for L in [0, 1, wl.num_sinks + wl.window, wl.num_sinks + wl.window + 1] + [rng.randint(1, 140000)
                                                                                   for _ in range(20)]:
            if L > 20000 and wl.mask == "full":
                continue  # the full keep-set is every position: checked on the short lengths
            want = len(oracle.keep_set(L, modes[wl.mask], wl.num_sinks, wl.window))
            assert bench._kept(L, wl) == want, (name, L)
    llama = workloads.llama3_8b_batch64()
    total = sum(llama.lens) * bench._kv_bytes_per_token(llama)
    assert total == sum(llama.lens) * 8 * 128 * 2 * 2 and 1.0e9 < total < 1.3e9
    fp8 = workloads.long_context_fp8()
    assert sum(fp8.lens) * bench._kv_bytes_per_token(fp8) == 4 * 131072 * (8 * 128 * 2 + 2 * 8 * 4)
