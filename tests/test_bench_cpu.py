"""The benchmark's JSON contract and helpers, on the CPU: the reference arm
(the oracle on a bounded window) prints one line with the required keys, and
the clock sampler parses nvidia-smi rows and reports throttle reasons."""
import json
import os
import subprocess
import sys

import bench
from synth import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr
    lines = [x for x in out.stdout.splitlines() if x.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e", "impl"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 2 and d["higher_is_better"] is True
    assert d["value"] > 0 and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"] == bench.workload_config(W.LLAMA_7B_STAGE3, 1)
    assert "llama-7b-stage3" in d["config"]["workload"]
    assert d["config"]["bytes_per_step"] == bench.algorithmic_bytes(16, 6_738_415_616, 2)


def test_reference_arm_of_each_workload_kind():
    """The reference arm runs the oracle's step of every workload kind (fused,
    bucketed with the clip, stage-3 group) and reports that workload's
    config."""
    for name in ("gpt2-small", "llama-1.4b"):
        out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
                              "reference", "--workload", name, "--steps", "1", "--warmup", "0"],
                             capture_output=True, text=True, timeout=600, cwd=ROOT)
        assert out.returncode == 0, out.stderr
        d = json.loads(out.stdout.strip().splitlines()[-1])
        assert d["config"] == bench.workload_config(W.ALL[name], 1)
        assert d["value"] > 0 and name in d["cpu_baseline"]["sample"]


def test_reference_arm_under_torchrun_prints_once():
    """Launched as the driver launches N > 1 (torchrun, 2 ranks, gloo on the
    CPU): rank 0 alone runs the oracle and prints the line; rank 1 exits 0."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                          "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                          "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                          "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [x for x in out.stdout.splitlines() if x.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0


def test_clock_sampler_parses_rows_and_reasons():
    cs = bench.ClockSampler(0)
    cs.out = "\n".join([
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2070, 2070, 1300.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 345, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 2040, 2070, 1350.0, 0x0, Not Active, Not Active, Active, Not Active",
    ])
    s = cs.summary()
    assert s["sm_max_mhz"] == 2070.0 and s["samples"] == 4
    assert s["sm_mhz"] == 2070.0                    # idle samples (< half the top) are ignored
    assert s["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]
    cs.out = ""
    assert cs.summary()["reasons"] == ["nvidia-smi unavailable"]


def test_algorithmic_bytes_formula():
    # N sources of the gradient dtype + 12 B state read + 12 B written + 2 B bf16 out
    assert bench.algorithmic_bytes(8, 124_439_808, 2) == 124_439_808 * 42
    assert bench.algorithmic_bytes(64, 10, 2) == 10 * 154
    assert bench.algorithmic_bytes(8, 10, 4) == 10 * 58


def test_overlap_fraction():
    import bench
    assert bench._hidden(10.0, 30.0, 30.0) == 1.0     # gathers entirely behind the consumer
    assert bench._hidden(10.0, 30.0, 40.0) == 0.0     # one after the other
    assert bench._hidden(8.0, 4.0, 10.0) == 0.5


def test_host_placement_helpers_fail_soft_without_a_gpu():
    """The end-to-end leg's placement helpers: the GPU's NUMA node is None
    when there is no device to ask, the default memory policy can always be
    restored, and the local rank count follows LOCAL_WORLD_SIZE."""
    import os
    assert bench.gpu_numa_node(0) is None or isinstance(bench.gpu_numa_node(0), int)
    assert bench._set_mempolicy(None) in (True, False)
    old = os.environ.get("LOCAL_WORLD_SIZE")
    try:
        os.environ["LOCAL_WORLD_SIZE"] = "4"
        assert bench.local_ranks() == 4
        os.environ["LOCAL_WORLD_SIZE"] = "0"
        assert bench.local_ranks() == 1
    finally:
        if old is None:
            os.environ.pop("LOCAL_WORLD_SIZE", None)
        else:
            os.environ["LOCAL_WORLD_SIZE"] = old


def test_traffic_records_match_the_current_kernel_sources():
    """Every DRAM traffic record in profiles/traffic.json was taken on the
    kernel sources the repository holds now (the bench reports a record only
    while the source hash matches), and carries the command that made it."""
    import json
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    seen = 0
    for workload, kernels in rec.items():
        for key, entry in kernels.items():
            kernel = key.replace("_block", "").replace("_step", "")
            assert entry["source_hash"] == bench.kernel_source_hash(kernel), (workload, key)
            assert entry["bytes_per_launch"] > 0
            if not key.endswith("_step"):
                assert entry["command"].startswith("ncu ") and "--clock-control none" in \
                    entry["command"], (workload, key)
            seen += 1
    assert seen >= 8
