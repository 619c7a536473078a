"""bench.py on the host: the multi-rank path with gloo (world size 2), the
reference arm under torchrun, the traffic model and the clock summary."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, _ = bench.setup_dist()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 + 5 * rank, w, "cpu")
    out.put((rank, m))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 15.0), (1, 15.0)]


def test_reference_arm_under_torchrun_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3",
           "--workload", "adam_small", "--ref-budget", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == bench.UNIT and rec["metric"] == bench.METRIC
    assert rec["value"] > 0 and rec["higher_is_better"] is True
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] == 1
    assert rec["e2e"] == {"value": rec["value"], "unit": bench.UNIT, "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}


def test_algorithmic_bytes_model():
    wl = bench.WORKLOADS["adam_4096"]()
    # fp32 Adam: read p, g, 2 codes; write p, 2 codes = 16 B/elem; absmax 2 x (r+w) x 4 B / 256
    assert wl.algorithmic_bytes() == 16 * 4096 * 4096 + 16 * (4096 * 4096 // 256)
    wl = bench.WORKLOADS["momentum_64m"]()
    assert wl.algorithmic_bytes() == 8 * (1 << 26) + 8 * ((1 << 26) // 256)
    wl = bench.WORKLOADS["ademamix_64m"]()
    assert wl.algorithmic_bytes() == 18 * (1 << 26) + 24 * ((1 << 26) // 256)
    wl = bench.WORKLOADS["momentum_embedding"]()
    n = 50257 * 1024
    assert wl.algorithmic_bytes(0.1) == int(2 * n + 0.1 * (6 * n + 8 * (n // 256)))


def test_clock_summary():
    rows = [dict(t=1.0, sm=1900.0, sm_max=2070.0, power="900", hw="Not Active",
                 hw_thermal="Not Active", sw_thermal="Not Active", sw_power="Active"),
            dict(t=1.1, sm=1800.0, sm_max=2070.0, power="950", hw="Not Active",
                 hw_thermal="Not Active", sw_thermal="Not Active", sw_power="Not Active"),
            dict(t=9.0, sm=300.0, sm_max=2070.0, power="100", hw="Active",
                 hw_thermal="Not Active", sw_thermal="Not Active", sw_power="Not Active")]
    s = bench.summarize_clocks(rows, 1.0, 1.1)
    assert s["sm_mhz"] == 1850.0 and s["sm_max_mhz"] == 2070.0
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 2


def test_traffic_is_null_for_other_kernel_sources(tmp_path, monkeypatch):
    assert bench.ncu_traffic("no-such-workload") is None


@pytest.mark.parametrize("name,unorm", [("adam_4096", 0.0), ("gpt2xl", 0.0), ("gpt2xl", 1.0),
                                        ("momentum_embedding", 0.0)])
def test_e2e_groups_cover_every_element_once(name, unorm):
    # the end-to-end pipeline's launches: every element of every tensor in
    # exactly one piece, pieces block-aligned, whole tensors under max_unorm
    import torch
    import bit_block_wise_gb300 as bnb8
    wl = bench.WORKLOADS[name]()
    wl.hp = dict(wl.hp, max_unorm=unorm)
    if name == "gpt2xl":   # a shortened list of the same shapes keeps host memory small
        wl.sizes, wl.bits = wl.sizes[:40], wl.bits[:40]
    params = []
    for n, b in zip(wl.sizes, wl.bits):
        p = torch.empty(n, dtype=torch.float32)
        s1, s2, a1, a2 = bnb8.zero_state(p, wl.optim, b, wl.blocksize)
        params.append(bnb8.ParamState(p, torch.empty_like(p), s1, s2, a1, a2, b))
    groups = bench.e2e_groups(bnb8, params, wl, 4)
    assert 1 <= len(groups) <= 5
    covered = {i: [] for i in range(len(params))}
    for grp in groups:
        for i, (lo, hi), pc in grp:
            assert pc.p.numel() == hi - lo
            assert lo % wl.blocksize == 0
            assert pc.p.data_ptr() == params[i].p.data_ptr() + 4 * lo
            covered[i].append((lo, hi))
    for i, ranges in covered.items():
        ranges.sort()
        assert ranges[0][0] == 0 and ranges[-1][1] == wl.sizes[i]
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
        if unorm > 0:
            assert len(ranges) == 1


@pytest.mark.parametrize("name", ["quantize_4096", "dequantize_4096"])
def test_codec_workloads_bytes_and_reference_arm(name, capsys):
    # the stand-alone conversion: x (4 B) + codes (1 B) + absmax (4 B per block)
    wl = bench.WORKLOADS[name]()
    n = 4096 * 4096
    assert wl.algorithmic_bytes() == n * 4 + n + (n // 256) * 4
    bench.main(["--impl", "reference", "--workload", name, "--steps", "1", "--warmup", "3",
                "--ref-budget", "2"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
