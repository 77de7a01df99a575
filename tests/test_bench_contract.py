"""The bench's reference arm (the CPU oracle, no GPU needed) prints the contract's JSON line,
and a non-zero rank of a multi-process launch prints nothing and exits 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=300, env=env)


def test_reference_arm_prints_the_contract_line():
    res = run(["--impl", "reference", "--workload", "single_seq_300", "--steps", "2", "--warmup", "3"])
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] == (os.cpu_count() or 1)
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == "single_seq_300"


def test_reference_arm_other_ranks_do_no_work():
    res = run(["--impl", "reference", "--workload", "single_seq_300", "--steps", "1", "--warmup", "3",
               "--gpus", "2"], {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert res.returncode == 0, res.stderr
    assert res.stdout.strip() == ""


def test_gpus_flag_disagreeing_with_the_launch_is_refused():
    res = run(["--impl", "reference", "--workload", "single_seq_300", "--steps", "1",
               "--gpus", "3"], {"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"})
    assert res.returncode == 2 and "--gpus 3" in res.stderr


def test_gpus_flag_alone_starts_one_rank_per_gpu():
    """`bench.py --gpus 2` started as a single process relaunches itself as two ranks under
    torch.distributed.run; rank 0 alone prints the line, which reports n_gpus 2."""
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "single_seq_300", "--steps", "1", "--warmup", "3",
                          "--gpus", "2"], cwd=ROOT, capture_output=True, text=True, timeout=300,
                         env=env)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["n_gpus"] == 2


def test_traffic_figures_name_existing_kernels_and_sources():
    """The committed DRAM figures name each kernel's source file and its hash; the bench
    returns a byte count only while the source is unchanged, else None."""
    sys.path.insert(0, ROOT)
    import hashlib
    import bench
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        figures = json.load(f)
    for kernel, entry in figures.items():
        if kernel.startswith("_"):
            continue
        src = os.path.join(ROOT, entry["source"])
        assert os.path.exists(src), src
        current = hashlib.sha256(open(src, "rb").read()).hexdigest() == entry["source_sha256"]
        for workload, fig in entry["workloads"].items():
            got = bench.ncu_traffic(kernel, workload)
            assert got == (fig["dram_bytes_per_launch"] if current else None)
            assert fig["dram_bytes_per_launch"] == fig["read"] + fig["write"]
    assert bench.ncu_traffic("no_such_kernel", "decode_b256") is None


def test_decode_roofline_uses_the_timed_region_only_for_overlapped_layer_steps():
    """A step made only of fused decode launches over several layers reports the timed
    region's time per launch (the layers overlap), with one launch timed alone beside it;
    every other step reports the launch timed alone."""
    sys.path.insert(0, ROOT)
    import types
    import bench
    from paged_kv_cache_299_gb300 import workloads as wl

    w = wl.decode_batch256_lognormal(layers=16)
    per_launch = w.decode_kv_bytes() / w.layers

    def fake(**kw):
        d = dict(w=w, fused_append=True, ws_merge_kernel=False, unified=False)
        d.update(kw)
        return types.SimpleNamespace(**d)

    r = bench.decode_roofline(fake(), "decode_b256", 0.125, 6694.2, "measured", step_ms=1.6)
    assert r["launch_ms"] == round(0.1, 5)
    assert r["achieved"] == round(per_launch / 0.1e-3 / 1e9, 1)
    assert r["isolated"]["launch_ms"] == 0.125
    assert r["isolated"]["achieved"] == round(per_launch / 0.125e-3 / 1e9, 1)
    assert r["frac"] == round(r["achieved"] / 6694.2, 4)
    # a store launched separately, or a merge kernel in the step: the launch timed alone
    for st in (fake(fused_append=False), fake(ws_merge_kernel=True)):
        r = bench.decode_roofline(st, "decode_b256", 0.125, 6694.2, "measured", step_ms=1.6)
        assert r["launch_ms"] == 0.125 and "isolated" not in r
    w1 = wl.decode_batch64_uniform()  # one layer
    r = bench.decode_roofline(fake(w=w1), "decode_b64", 0.04, 6694.2, "measured", step_ms=0.039)
    assert r["launch_ms"] == 0.04 and "isolated" not in r


def test_clock_summary_keeps_the_samples_of_the_marked_region():
    """nvidia-smi rows (timestamp first) outside the marked region are left out of the
    clock summary; a region without samples falls back to every sample, and says so."""
    sys.path.insert(0, ROOT)
    import datetime
    import bench
    rows = [
        "2026/12/03 10:00:00.000, 0, 1200, 2070, 300.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/03 10:00:00.500, 0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Active",
        "2026/12/03 10:00:00.520, 0, 2070, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/12/03 10:00:01.000, 0, 1000, 2070, 200.0, 0x0, Active, Not Active, Not Active, Not Active",
    ]
    text = "\n".join(rows)
    t = lambda x: datetime.datetime.strptime("2026/12/03 " + x, "%Y/%m/%d %H:%M:%S.%f")
    got = bench.ClockSampler.summarise(text, t("10:00:00.400"), t("10:00:00.600"))
    assert got["samples"] == 2 and got["sm_mhz"] == 2070 and got["sm_max_mhz"] == 2070
    assert got["reasons"] == ["sw_power_cap"] and got["samples_from"] == "the marked region"
    everything = bench.ClockSampler.summarise(text, t("10:00:02.000"), t("10:00:03.000"))
    assert everything["samples"] == 4 and "hw_slowdown" in everything["reasons"]
    assert everything["samples_from"].startswith("the whole sampling")
    assert bench.ClockSampler.summarise("")["samples"] == 0


def test_concurrent_split_balances_the_two_kernels():
    """The decode's SM share beside a chunk prefill: both modelled kernels end together,
    more prefill work leaves fewer SMs to the decode, and the share stays within 1 .. SMs-1."""
    import bench
    d = bench.concurrent_decode_sms(1056923648, 45134905344, 152)  # the mixed step
    assert 80 <= d <= 96
    assert bench.concurrent_decode_sms(1056923648, 4 * 45134905344, 152) < d
    assert bench.concurrent_decode_sms(4 * 1056923648, 45134905344, 152) > d
    assert bench.concurrent_decode_sms(1.0, 1e15, 152) == 1
    # a decode-only load takes the SMs it can use: past DECODE_GBS_MAX more SMs add nothing
    cap = int(bench.DECODE_GBS_MAX / bench.DECODE_GBS_PER_SM)
    assert cap <= bench.concurrent_decode_sms(1e15, 1.0, 152) <= cap + 1
