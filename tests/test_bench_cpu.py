"""Host-side logic of bench.py, on the CPU: the reference arm's JSON line, rank
handling under torchrun, and the max-over-ranks reduction of the timed
intervals with world_size 2 over gloo."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _run_bench(args, env_extra=None):
    env = dict(os.environ)
    env.update(env_extra or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                          env=env, timeout=600)


def test_reference_arm_prints_one_json_line():
    r = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"])
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["host_cores"] == os.cpu_count() and d["cpu_baseline"]["affinity_cores"] >= 1
    # ms_per_step is the timed sample's wall time; the whole batch's step is extrapolated beside it
    assert 0 < d["ms_per_step"] and d["ms_per_step_extrapolated"] > 0
    assert d["value"] == pytest.approx(256 / (d["ms_per_step_extrapolated"] / 1e3), rel=1e-9)
    assert d["n_gpus"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"].startswith("tiny")
    assert d["steps"] == 2 and d["warmup"] == 3


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3", "--gpus", "2"],
                   {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_gpus_n_launches_n_ranks_itself():
    """Without a launcher, --gpus 2 starts two ranks (torch's launcher, rendezvous on 127.0.0.1);
    the ranks' timings are reduced with a max over gloo and rank 0 alone prints."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--selftest-launch"],
                       capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert lines == [{"selftest": "launch", "world": 2, "max_ms": [11.0, 50.0]}]


def test_gpus_disagreeing_with_world_size_is_an_error():
    r = _run_bench(["--gpus", "2", "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"],
                   {"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert r.returncode != 0 and "WORLD_SIZE" in r.stderr


def test_warmup_below_three_is_rejected():
    r = _run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "2"])
    assert r.returncode != 0


def test_whole_job_throughput():
    import bench
    # 2 ranks x 8192 tokens x 10 steps over a slowest-rank interval of 40 ms
    assert bench.whole_job_tokens_per_s(2, 8192, 10, 40.0) == pytest.approx(2 * 8192 * 10 / 0.040)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [10.0 + rank * 5.0, 30.0 - rank * 7.0]       # rank 0: (10, 30); rank 1: (15, 23)
    got = bench.reduce_max_over_ranks(mine, "cpu")
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo_world_size_2():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        assert out[r] == [15.0, 30.0]


def test_stage_report_bytes_and_roofline_bound():
    """GEMM stages carry algorithmic bytes beside FLOPs; at the measured peaks the
    Mixtral-like up projection is tensor-bound and the 2,304-expert one HBM-bound
    (about 3 GB of expert weights against a few hundred GFLOP)."""
    import bench
    from dropless_moe_expert_router_gb300 import workloads as W
    peaks = {"hbm_gbs": 6806.2, "bf16_tflops": 1906.5}

    def bound(name, stage):
        wl = W.get(name)
        R = wl.T * wl.K
        ms = {stage: 1.0}
        out, flops, nbytes = bench.stage_report(wl, R, ms, active=wl.E)
        assert "GB/s" in out[stage] and "TFLOP/s" in out[stage]
        peak_f = peaks["bf16_tflops"] * (2 if wl.precision == "mxfp8" else 1)
        return "hbm" if nbytes[stage] / (peaks["hbm_gbs"] * 1e9) > flops[stage] / (peak_f * 1e12) else "tensor"

    assert bound("mixtral", "gemm_up") == "tensor"
    assert bound("dsv3", "gemm_down") == "tensor"
    assert bound("large_e", "gemm_up") == "hbm"
    assert bound("large_e", "gemm_down") == "hbm"
    # up projection bytes, large-E shape: x_perm + W1|W3 + h, bf16
    wl = W.get("large_e")
    R = wl.T * wl.K
    _, _, nbytes = bench.stage_report(wl, R, {"gemm_up": 1.0}, active=wl.E)
    assert nbytes["gemm_up"] == R * wl.H * 2 + wl.E * wl.H * 2 * wl.F * 2 + R * wl.F * 2


def test_stage_report_nvfp4_and_sigmoid_bytes():
    """NVFP4 operands count half a byte plus a 1/16 scale share per element; the NVFP4 permute
    reads x twice (the routed tokens' amax, then the scatter) and writes codes and scales; the
    up projection writes bf16 h (quantised by its own stage); the sigmoid router also reads the
    expert bias."""
    import bench
    from dropless_moe_expert_router_gb300 import workloads as W
    wl = W.get("dsv3_nvfp4")
    T, H, E, K, F = wl.T, wl.H, wl.E, wl.K, wl.F
    R = T * K
    ms = {"permute": 1.0, "gemm_up": 1.0, "quant_h": 1.0, "gemm_down": 1.0}
    out, flops, nb = bench.stage_report(wl, R, ms, active=E)
    q = 0.5 + 1 / 16
    assert nb["permute"] == 2 * T * H * 2 + R * H * q + T * K * (4 + 4) + R * 4
    assert nb["gemm_up"] == R * H * q + E * H * 2 * F * q + R * F * 2
    assert nb["quant_h"] == R * F * 2 + R * F * q
    assert nb["gemm_down"] == R * F * q + E * F * H * q + R * H * 2
    assert flops["gemm_up"] == 4.0 * R * H * F and "TFLOP/s" in out["gemm_up"]
    ws = W.get("dsv3_sigmoid")
    _, _, nb_s = bench.stage_report(ws, ws.T * ws.K, {"route": 1.0}, active=ws.E)
    _, _, nb_m = bench.stage_report(W.get("dsv3"), ws.T * ws.K, {"route": 1.0}, active=ws.E)
    assert nb_s["route"] - nb_m["route"] == ws.E * 4
