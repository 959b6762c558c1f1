"""Host-side logic of bench.py (no GPU): the cost model behind the roofline,
workload names, and the reference arm's JSON line."""

import json
import os
import subprocess
import sys

import numpy as np

import dmoe_synth as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_op_costs_follow_the_operand_sizes():
    cfg = syn.CONFIGS["moe_xs"]
    P, nnz, live = 11776, 1472, 64
    c = bench.op_costs(cfg, P, nnz, live)
    blk = nnz * 128 * 128 * 2
    W = live * cfg.d * cfg.F * 2
    assert c["sdd_fwd"] == (P * cfg.d * 2 + W + 2 * blk, 2.0 * P * cfg.d * cfg.F)
    assert c["dsd_fwd"] == (blk + W + P * cfg.d * 2, 2.0 * P * cfg.d * cfg.F)
    assert c["dstd_dw1"][0] == c["dstd_dw2"][0] == blk + P * cfg.d * 2 + W
    # the products' flops count padded rows: P, not the A = T k assignments
    assert c["sdd_bwd"][1] == 2.0 * P * cfg.d * cfg.F
    # the gate: x and W_g in, logits and the routing out; 2 T d E flops
    A = cfg.T * cfg.k
    assert c["gate_route_topk"] == (cfg.T * cfg.d * 2 + cfg.E * cfg.d * 2 + cfg.T * cfg.E * 4 + A * 8,
                                    2.0 * cfg.T * cfg.d * cfg.E)
    # a 64-row block format: four times the blocks of a quarter of the size
    c64 = bench.op_costs(cfg, P, 4 * nnz, live, block=64)
    assert c64["sdd_fwd"][0] == c["sdd_fwd"][0]


def test_swiglu_costs_count_both_halves():
    cfg = syn.CONFIGS["mixtral"]
    P, nnz, live = 16896, 14784, 8
    c = bench.op_costs(cfg, P, nnz, live)
    blk = nnz * 128 * 128 * 2
    W = live * cfg.d * cfg.F * 2
    assert c["sdd_fwd"] == (P * cfg.d * 2 + 2 * W + 3 * blk, 2.0 * 2.0 * P * cfg.d * cfg.F)
    assert c["dsd_t_dx"][1] == 2.0 * 2.0 * P * cfg.d * cfg.F
    assert "dstd_dw3" in c
    # useful flops: 3 GEMMs forward for SwiGLU, times 3 for fwd + bwd, on A rows
    assert bench.useful_flops(cfg) == 3.0 * 3 * 2.0 * cfg.A * cfg.d * cfg.F


def test_workload_names():
    cfg = syn.CONFIGS["fine"]
    base = bench.workload_name(cfg)
    assert base.startswith("fine: T=4096 d=3584 E=64 F=2560 top-8 swiglu")
    assert bench.workload_name(cfg, depth=2).endswith("depth=2")
    assert bench.workload_name(cfg, block=64).endswith("block=64")
    assert bench.workload_name(cfg, gate=True).endswith("linear-gate")
    assert bench.workload_name(cfg, block=128) == base


def test_gate_weights_are_seeded():
    cfg = syn.CONFIGS["tiny"]
    a, b = bench.gate_weights(cfg), bench.gate_weights(cfg)
    assert a.shape == (cfg.E, cfg.d) and np.array_equal(a, b)


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    r = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in r, key
    assert r["impl"] == "reference" and r["value"] > 0 and r["higher_is_better"] is True
    assert r["cpu_baseline"]["kind"] == "oracle" and r["cpu_baseline"]["value"] == r["value"]
    # the threads the oracle kept busy (CPU time over wall time, counted in
    # clock ticks over a short step, so it is not bounded by `cores`), and the
    # host's own CPU figures beside the affinity count
    assert r["cpu_baseline"]["threads_effective"] > 0
    host = r["cpu_baseline"]["host"]
    assert host["affinity"] == r["cpu_baseline"]["cores"] >= 1 and host["cpu_count"] >= 1
    assert host["cgroup_quota_cores"] is None or host["cgroup_quota_cores"] > 0
    assert r["e2e"]["h2d_bytes_per_step"] == 0 and r["e2e"]["d2h_bytes_per_step"] == 0
    assert r["config"]["workload"].startswith("tiny:")


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun only rank 0 times the oracle and prints; another rank
    exits 0 at once without output."""
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=120, cwd=ROOT,
                         env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip() == ""


def test_cpu_samples_are_bounded_by_work():
    """The CPU legs size their token samples by fp64 work: the largest
    workload gets its floor of 64 tokens, the MoE-XS reference arm keeps
    T/16."""
    mx, xs = syn.CONFIGS["mixtral"], syn.CONFIGS["moe_xs"]
    assert bench.sample_tokens(mx, 50.0, cap=mx.T // 16) == 64
    assert bench.sample_tokens(xs, 50.0, cap=xs.T // 16) == xs.T // 16
    assert bench.per_token_flops(mx) * 64 < 200e9


def test_default_workload_is_the_largest():
    """With no --config the bench runs the Mixtral-shaped layer, the
    largest of the workloads by useful flops."""
    name = bench.parser().parse_args([]).config
    assert name == "mixtral"
    assert bench.useful_flops(syn.CONFIGS[name]) == max(bench.useful_flops(c) for c in syn.CONFIGS.values())


def test_warmup_below_three_is_rejected():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                          "--steps", "1", "--warmup", "2"], capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert out.returncode != 0 and "warmup" in out.stderr


def test_traffic_counters_follow_the_kernel_sources(tmp_path, monkeypatch):
    """ncu counters keyed by a source hash count only while the kernel's
    sources are those the capture ran on: an edit to one of them turns the
    roofline's traffic into null for the kernels built from it, and only
    for those."""
    src = os.path.join(ROOT, "dropless_moe_block_gb300", "csrc")
    csrc = tmp_path / "dropless_moe_block_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in os.listdir(src):
        if f.endswith((".cu", ".cuh")):
            (csrc / f).write_bytes(open(os.path.join(src, f), "rb").read())
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h_prod = bench.kernel_source_hash("dsd_t_dx")
    h_comb = bench.kernel_source_hash("unpermute_combine")
    assert h_prod != h_comb
    (tmp_path / "profiles" / "traffic.txt").write_text(
        "# op workload bytes hash\n"
        f"dsd_t_dx moe_xs 100 {h_prod}\n"
        "dsd_fwd moe_xs 200 000000000000\n"
        f"unpermute_combine moe_xs 300 {h_comb}\n")
    assert bench.load_traffic() == {("dsd_t_dx", "moe_xs"): 100.0, ("unpermute_combine", "moe_xs"): 300.0}
    # the products' tensor-map code changes: their counters no longer apply
    (csrc / "tmap.cuh").write_text((csrc / "tmap.cuh").read_text() + "\n// edited\n")
    assert bench.load_traffic() == {("unpermute_combine", "moe_xs"): 300.0}
    # the helpers every kernel includes change: nothing applies
    (csrc / "common.cuh").write_text((csrc / "common.cuh").read_text() + "\n// edited\n")
    assert bench.load_traffic() == {}
