"""Host-side logic of bench.py on CPU: aggregation over ranks (world size 2
over gloo), clock-record parsing, and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [12.5, 20.0][rank]
    m = bench.reduce_max(ms, dist, "cpu")
    value, rows = bench.aggregate(world, 1000, 10, 4, m)
    q.put((rank, m, value, rows))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, value, rows in got:
        assert m == 20.0                                   # slowest rank's time
        assert value == pytest.approx(2 * 1000 * 4 / 0.020 / 1e9)
        assert rows == pytest.approx(2 * 10 * 4 / 0.020)


def test_aggregate_single_rank():
    v, r = bench.aggregate(1, 9438336, 4096, 1000, 3.0)
    assert v == pytest.approx(9438336 * 1000 / 3e-3 / 1e9)
    assert r == pytest.approx(4096 * 1000 / 3e-3)
    assert bench.reduce_max(3.5, None, "cpu") == 3.5


def test_clock_summary_flags_slowdown():
    s = bench.ClockSampler(None)
    s.samples = [(1.0, ["2070", "2070", "500", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]),
                 (2.0, ["1900", "2070", "900", "0x4", "Not Active", "Not Active", "Not Active", "Active"]),
                 (3.0, ["2000", "2070", "800", "0x0", "Active", "Not Active", "Not Active", "Not Active"]),
                 (9.0, ["300", "2070", "90", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"])]
    c = s.summary(0.5, 3.5)
    assert c["samples"] == 3 and c["sm_mhz"] == 2000 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]
    c2 = s.summary(100.0, 101.0)   # nothing in the window: falls back to the whole run
    assert c2["samples"] == 4


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "5", "--warmup", "3"], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"]["workload"] == "bf16_res_65536x8192_w"
    import bench as B
    from row_reduction_norm_gb300 import workloads as W
    # the same config object as the GPU arm prints
    assert line["config"] == B.bench_config(W.WORKLOADS[B.HEADLINE], 1)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "5", "--warmup", "3"], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_floor():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "5", "--warmup", "2"], capture_output=True, text=True, timeout=120)
    assert r.returncode != 0


def test_device_code_tokens_ignore_comments_only():
    """A profile stays valid across comment edits, not across code edits."""
    a = "int f(int x) {  // doubles x\n  return 2 * x; /* twice */ }\n"
    b = "/* header */\nint f(int x) {\n    return 2 * x;\n}\n"
    c = "int f(int x) { return 3 * x; }"
    s = 'const char *s = "a // not a comment"; char q = \'/\';'
    assert bench.code_tokens(a) == bench.code_tokens(b)
    assert bench.code_tokens(a) != bench.code_tokens(c)
    assert "// not a comment" in bench.code_tokens(s)


def test_row_slice_profiles_scale_to_the_full_workload():
    import bench
    plan = {"kernel": "reg", "regime": "cta", "threads_per_row": 256, "chunks_per_thread": 4, "vec_elems": 8,
            "block": 256, "grid": 65536}
    v, why = bench.profiled_traffic("bf16_res_65536x8192_w", plan, with_source=True, rows=65536)
    if v is None:   # the summary predates the device code or the plan
        assert "predates" in why or "another launch plan" in why
    else:
        assert "scaled by 65536/8192" in why and v > 0
    # a slice counts only when the caller says how many rows to scale to
    v, why = bench.profiled_traffic("bf16_res_65536x8192_w", plan, with_source=True)
    assert v is None


def test_e2e_steps_are_bounded():
    import bench
    from row_reduction_norm_gb300 import workloads as W
    assert bench.e2e_steps_for(W.WORKLOADS["bf16_res_65536x8192_w"], 0) < 200
    assert bench.e2e_steps_for(W.WORKLOADS["bf16_4096x576"], 0) == 4096
    assert bench.e2e_steps_for(W.WORKLOADS["bf16_4096x576"], 7) == 7


def test_e2e_chunks_are_about_64_mib_of_rows():
    import bench
    from row_reduction_norm_gb300 import workloads as W
    head = W.WORKLOADS["bf16_res_65536x8192_w"]
    assert bench.e2e_chunk_rows(head) == 4096                # 4096 x 16 KiB = 64 MiB
    small = W.WORKLOADS["bf16_4096x576"]
    assert bench.e2e_chunk_rows(small) == small.rows         # the whole batch fits one chunk
    for wl in W.WORKLOADS.values():
        c = bench.e2e_chunk_rows(wl)
        assert 1 <= c <= wl.rows and c * wl.hidden * wl.elem_bytes <= max(64 << 20, wl.hidden * wl.elem_bytes)


def test_plan_summary_names_the_cluster_size():
    import bench
    from row_reduction_norm_gb300 import _native as N
    import row_reduction_norm_gb300 as R
    p = R.rmsnorm_plan_ex(100, 65536, N.RMSNORM_BF16, True, True, 152, 4)
    d = bench.plan_summary(p)
    assert d["kernel"] == "cluster" and d["cluster_ctas"] == 8 and "rows_per_block" not in d
    q = R.rmsnorm_plan(100, 8192, N.RMSNORM_BF16, True, 152, 4)
    assert "cluster_ctas" not in bench.plan_summary(q)


def test_traffic_source_says_why():
    import bench
    v, why = bench.profiled_traffic("no_such_workload", None, with_source=True)
    assert v is None and "no ncu summary" in why
    v, why = bench.profiled_traffic("bf16_4096x576", {"kernel": "none"}, with_source=True)
    assert v is None and "another launch plan" in why
    assert bench.profiled_traffic("no_such_workload") is None
