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
    # a carried ||p|| spares the pre-pass its read of p (2 B/elem in bf16) only
    # where the direction does not need p: decoupled decay, not Adam's coupled one
    plain, carried = bench.WORKLOADS["gpt2xl_adamw"](), bench.WORKLOADS["gpt2xl_adamw_carried"]()
    assert plain.algorithmic_bytes() - carried.algorithmic_bytes() == 2 * plain.elements
    assert bench.WORKLOADS["gpt2xl"]().algorithmic_bytes() == \
        bench.WORKLOADS["gpt2xl_carried"]().algorithmic_bytes()


def test_read_bytes_and_the_pages_baseline():
    # what a step reads (p, g, codes, absmax), against the L2 for --l2 none
    wl = bench.WORKLOADS["adam_4096"]()
    n = 4096 * 4096
    assert wl.read_bytes() == 2 * 4 * n + 2 * n + 2 * 4 * (n // 256)
    assert wl.read_bytes() >= 1.2 * bench.L2_BYTES
    assert bench.WORKLOADS["adam_small"]().read_bytes() < 1.2 * bench.L2_BYTES
    # vs_baseline only where the pages give a figure for the workload: the
    # PR #1692 step, 1.2875 ms for 4096 x 4096 elements
    pages = bench.WORKLOADS["adam_4096_bf16_pages"]()
    gelem = n / 1.2875e-3 / 1e9
    assert bench.vs_pages(pages, 10 * gelem) == 10.0
    assert bench.vs_pages(wl, 100.0) is None
    assert bench.WORKLOADS["ademamix_4096_bf16_pages"]().pages == pages.pages


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


def _cpu_params(wl, seed):
    import torch
    import bit_block_wise_gb300 as bnb8
    import workloads
    params, grads = [], []
    for i, n in enumerate(wl.sizes):
        nb = -(-n // wl.blocksize)
        p = torch.from_numpy(workloads.normal(n, 0.02, seed + i))
        s1 = torch.from_numpy(workloads.random_codes(n, seed + 10 + i))
        s2 = torch.from_numpy(workloads.random_codes(n, seed + 20 + i))
        a1 = torch.from_numpy(workloads.random_absmax(nb, 1e-3, seed + 30 + i))
        a2 = torch.from_numpy(workloads.random_absmax(nb, 1e-6, seed + 40 + i))
        params.append(bnb8.ParamState(p, None, s1, s2, a1, a2, 8))
        grads.append(torch.from_numpy(workloads.normal(n, 1e-3, seed + 50 + i)))
    return params, grads


def _oracle_full_step(wl, params, grads, step):
    # a stand-in for the GPU step that is right by construction: the oracle
    # on the whole tensors
    import torch
    import oracle
    q1, q2 = oracle.create_qmap(True), oracle.create_qmap(False)
    for ps, g in zip(params, grads):
        t = oracle.TensorState(ps.p.numpy().copy(), ps.s1.numpy().copy(), ps.s2.numpy().copy(),
                               ps.absmax1.numpy().copy(), ps.absmax2.numpy().copy(), 8)
        oracle.step(oracle.HParams(optim=wl.optim, step=step, **wl.hp), t, g.numpy(), "f32",
                    wl.blocksize, q1, q2)
        for dst, src in ((ps.p, t.p), (ps.s1, t.s1), (ps.s2, t.s2), (ps.absmax1, t.absmax1),
                         (ps.absmax2, t.absmax2)):
            dst.copy_(torch.from_numpy(src))


@pytest.mark.parametrize("plant", [None, "code", "absmax", "p"])
def test_sampled_parity_counts_what_differs(plant):
    wl = bench.Workload("t", "t", "adam", "f32", [256 * 40 + 77], [8], 256,
                        dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=1e-2),
                        ("normal", 1e-3))
    params, grads = _cpu_params(wl, 500)
    ps = params[0]
    n = ps.p.numel()

    def gpu_step():
        _oracle_full_step(wl, params, grads, 3)
        if plant == "code":        # block 0 is always sampled; the last block too
            ps.s1[5] = (int(ps.s1[5]) + 3) % 256
        elif plant == "absmax":
            ps.absmax2[-1] = ps.absmax2[-1] * 2
        elif plant == "p":
            ps.p[n - 1] = ps.p[n - 1] + 1.0

    rep = bench.sampled_parity(wl, params, gpu_step, 3, grads)
    assert rep["blocks"] >= 2 and rep["codes"] > 0 and rep["p_compared"] > 0
    assert rep["code_mismatches"] == (1 if plant == "code" else 0)
    assert rep["code_mismatch_max_index_delta"] == (3 if plant == "code" else 0)
    assert rep["absmax_mismatches"] == (1 if plant == "absmax" else 0)
    assert rep["p_mismatches"] == (1 if plant == "p" else 0)
