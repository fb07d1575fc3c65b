"""The bench's multi-rank host logic on CPU with world size 2 (gloo): the step
time is the maximum over ranks and the throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms_local = [3.0, 5.0][rank]           # rank 1 is the slower one
        value, ms = bench.aggregate_throughput(4096, ms_local, world)
        q.put((rank, value, ms, bench.max_over_ranks(float(rank), world)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, ms, mx in res:
        assert ms == 5.0 and mx == 1.0
        assert value == pytest.approx(2 * 4096 / 5e-3)


def test_single_rank_is_local_time():
    import bench
    value, ms = bench.aggregate_throughput(100, 2.0, 1)
    assert ms == 2.0 and value == pytest.approx(100 / 2e-3)


def test_kernel_labels_map_to_layer_stages():
    import bench
    labels = ["router_logits", "router_select", "permute_rank", "permute_scan", "permute_scatter",
              "quantize_act_rows", "grouped_gemm_fc1_n256_w8a8", "quantize_act_rows",
              "grouped_gemm_fc2_n256_short_w8a8", "finalize"]
    seen = {}
    stages = []
    for lab in labels:
        st = bench._stage_of(lab, seen)
        seen[st] = seen.get(st, 0.0) + 1.0
        stages.append(st)
    assert stages == ["route", "route", "permute", "permute", "permute", "quant_x", "fc1", "quant_h", "fc2",
                      "finalize"]


def test_layer_bytes_count_each_tensor_once():
    import bench
    import moe_inputs as mi
    cfg = mi.MoEConfig("b", T=2, H=64, I=128, E=4, k=2, renorm=False, n_shared=1, I_shared=64)
    rows, active = 4, 3
    wk = bench._work(cfg, rows, active)
    H, I, Ish, T = 64, 128, 64, 2
    w1 = active * 2 * I * H * 2 + 2 * Ish * H * 2
    w2 = active * H * I * 2 + H * Ish * 2
    fc1 = w1 + (rows + T) * H * 2 + rows * I * 2 + T * Ish * 2          # A rows in, h out
    fc2 = w2 + rows * I * 2 + T * Ish * 2 + rows * H * 2 + T * H * 2     # h in, y out
    assert wk["fc1_bytes"] == fc1 and wk["fc2_bytes"] == fc2
    # + fp32 gate weights, x for the router, x_perm written, y and y_shared read back, out
    assert wk["layer_bytes"] == fc1 + fc2 + 4 * H * 4 + T * H * 2 + rows * H * 2 + rows * H * 2 + T * H * 2 + T * H * 2


def test_clock_sampler_keeps_region_samples_and_reasons(tmp_path):
    import bench
    cs = bench.ClockSampler(0)
    path = tmp_path / "clocks.csv"
    # index, sm, max sm, power, active mask, hw_slowdown, hw_thermal, sw_thermal, sw_power_cap
    lines = ["0, 1200, 2070, 300.0, 0x0, Not Active, Not Active, Not Active, Not Active",   # before the region
             "0, 2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",   # last one before
             "0, 2055, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active",      # inside the region
             "0, 1980, 2070, 1390.0, 0x20, Not Active, Not Active, Active, Not Active",     # inside the region
             "garbled line"]
    path.write_text("\n".join(lines) + "\n")

    class _Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    cs.path, cs.proc, cs.n_before = str(path), _Done(), 2
    cs.f = open(tmp_path / "unused", "w")
    rec = cs.stop()
    assert rec["samples_in_region"] == 2  # parsed samples after the region opened
    assert rec["samples"] == 3            # the last sample before it plus the two inside
    assert rec["sm_mhz"] == 2055.0 and rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == ["sw_power_cap", "sw_thermal_slowdown"]


def _bench_cli(args, env_extra):
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(root, "bench.py")] + args, cwd=root, env=env,
                          capture_output=True, text=True, timeout=300)


def test_bench_refuses_inconsistent_rank_options_before_touching_a_gpu():
    # a launcher's world size must match --gpus
    r = _bench_cli(["--gpus", "1"], {"WORLD_SIZE": "2", "RANK": "0"})
    assert r.returncode != 0 and "--gpus 1 but the launcher started 2 ranks" in r.stderr
    # the one-GPU rank modes hold every rank in one process: not under a multi-rank launcher
    for mode in ("--a2a-ranks", "--ep-ranks"):
        r = _bench_cli(["--gpus", "2", mode, "4"], {"WORLD_SIZE": "2", "RANK": "0"})
        assert r.returncode != 0 and "hold every rank in one process" in r.stderr, (mode, r.stderr[-500:])


def test_bench_help_lists_the_partitions_and_reductions():
    r = _bench_cli(["--help"], {})
    assert r.returncode == 0
    for word in ("--partition", "a2a", "--reduce", "peer", "--a2a-ranks", "--ep-ranks"):
        assert word in r.stdout
