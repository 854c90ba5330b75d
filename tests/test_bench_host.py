"""bench.py's host side without a GPU: the reference arm's JSON line, its
launch under torchrun with two gloo ranks (rank 0 alone prints), and the
max-over-ranks reduction the timed region uses, with world_size 2 on gloo."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
REF_CMD = ["bench.py", "--impl", "reference", "--workload", "toy", "--steps", "2", "--warmup", "3",
           "--ref-tokens", "16"]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env():
    env = dict(os.environ)
    env["CUDA_VISIBLE_DEVICES"] = ""  # CPU only, also on a machine with a GPU
    env["OMP_NUM_THREADS"] = "2"
    return env


def _json_lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def _check_reference_line(d):
    assert d["impl"] == "reference"
    for key, typ in [("metric", str), ("value", float), ("unit", str), ("n_gpus", int), ("steps", int),
                     ("warmup", int), ("ms_per_step", float), ("higher_is_better", bool), ("scaling", str),
                     ("dtype", str), ("data", str), ("config", dict), ("cpu_baseline", dict), ("e2e", dict)]:
        assert isinstance(d[key], typ), key
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["steps"] == 2 and d["warmup"] == 3
    assert d["vs_baseline"] is None and d["higher_is_better"] is True
    assert d["config"]["workload"] == "toy" and d["config"]["sample_tokens_per_step"] == 16
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable] + REF_CMD, cwd=ROOT, env=_env(), capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    _check_reference_line(lines[0])


def test_reference_arm_under_torchrun_two_gloo_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port())] + REF_CMD + ["--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1, r.stdout
    _check_reference_line(lines[0])
    assert lines[0]["n_gpus"] == 2


def _rank_main(rank, world, port, out):
    # gloo on the CPU, also on a machine with a GPU (set before any CUDA query)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(1.5 + rank, w)
    dist.destroy_process_group()


@pytest.mark.skipif(not torch.distributed.is_available(), reason="torch.distributed unavailable")
def test_max_over_ranks_two_gloo_ranks():
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_memory_kernel_bytes_follow_the_row_types():
    """The algorithmic bytes bench.py divides by the event-timed duration:
    finalize reads fp32 expert and shared rows for bf16 weights and bf16 rows
    for fp8 weights; the h conversion reads fp32 h, or bf16 h for fp8 weights
    stored K-contiguous."""
    sys.path.insert(0, ROOT)
    import bench
    import workloads

    q = workloads.CONFIGS["qwen3_prefill"]
    T, D, k, R = q.T, q.D, q.k, q.R
    assert bench.memory_kernel_bytes(q, "finalize", 2) == R * D * 4 + 4 * R + 4 * T * k + T * D * 2
    assert bench.memory_kernel_bytes(q, "w13_gate_up", 2) is None
    ling = workloads.CONFIGS["ling_prefill"]
    T, D, k, R, I, Is = ling.T, ling.D, ling.k, ling.R, ling.I, ling.I_shared
    for nk in (False, True):
        assert bench.memory_kernel_bytes(ling, "finalize", 2, nk) == \
            R * D * 2 + 4 * R + 4 * T * k + T * D * 2 + T * D * 2
        assert bench.memory_kernel_bytes(ling, "x_to_e4m3x2", 2, nk) == T * D * 2 + T * D * 2 + 4 * T
    hb = {False: 4, True: 2}
    for nk in (False, True):
        assert bench.memory_kernel_bytes(ling, "h_to_e4m3x2", 2, nk) == R * I * hb[nk] + R * I * 2 + 4 * R
        assert bench.memory_kernel_bytes(ling, "shared_h_to_e4m3x2", 2, nk) == \
            T * Is * hb[nk] + T * Is * 2 + 4 * T


@pytest.mark.parametrize("name", sorted(__import__("workloads").CONFIGS))
@pytest.mark.parametrize("layout", ["kn", "nk"])
def test_bench_kernel_names_match_launch_count(name, layout):
    """bench.py names each kernel moe_layer launches (per-kernel timings):
    one name per launch the library reports, for every workload."""
    sys.path.insert(0, ROOT)
    import bench
    import mixture_experts_layer_gating_gb300 as moe
    import workloads
    from tests._lib import ensure_library

    ensure_library()
    shape = workloads.CONFIGS[name]
    nk = layout == "nk" and shape.w_dtype == "fp8_e4m3"
    cfg = moe.config_from_shape(shape, "nk" if nk else "kn")
    assert len(bench.kernel_names(shape, nk)) == moe.moe_layer_launch_count(cfg)
    old = moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, 1)
    try:
        in_gemm = (shape.I_shared == shape.I and shape.I_shared > 0 and shape.act_dtype == "bf16" and
                   (nk or shape.w_dtype != "fp8_e4m3"))
        assert len(bench.kernel_names(shape, nk, shared_in_gemm=in_gemm)) == \
            moe.moe_layer_launch_count(cfg)
    finally:
        moe.moe_set_option(moe.MOE_OPT_SHARED_IN_GEMM, old)
    old = moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, 0)
    try:
        assert len(bench.kernel_names(shape, nk, fused_routing=False)) == \
            moe.moe_layer_launch_count(cfg)
    finally:
        moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, old)
    old = moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, 3)
    try:
        assert len(bench.kernel_names(shape, nk, hist_sort=False)) == \
            moe.moe_layer_launch_count(cfg)
    finally:
        moe.moe_set_option(moe.MOE_OPT_FUSED_ROUTING, old)


def test_bench_percentiles():
    sys.path.insert(0, ROOT)
    import bench

    v = [5.0, 1.0, 3.0, 2.0, 4.0]
    assert bench.pct(v, 50) == 3.0 and bench.pct(v, 0) == 1.0 and bench.pct(v, 100) == 5.0
    assert bench.pct(v, 10) == pytest.approx(1.4) and bench.pct(v, 90) == pytest.approx(4.6)
