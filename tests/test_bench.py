"""bench.py's JSON line: the oracle arm on the host, and the CUDA arm on a small workload."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                         text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_reference_arm_runs_the_oracle_on_the_host():
    line = _run(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0",
                 "--ref-seconds", "1"], timeout=300)
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"]
    st = line["cpu_baseline"]["stage_seconds"]
    assert set(st) == {"reshard", "attention", "merge"} and all(v >= 0 for v in st.values())
    assert line["e2e"] == {"value": line["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"]["workload"].startswith("tiny-")
    assert {"bytes_per_step", "parallelism", "l2"} <= set(line["config"])


def test_reference_arm_loads_only_the_oracle():
    """The oracle arm's inputs are built without the product library (no import, no workspace)."""
    code = ("import sys, torch; sys.path.insert(0, %r); import bench; "
            "wl = bench.Workload('tiny', torch.device('cpu'), oracle_only=True); "
            "assert wl.ws is None; "
            "assert 'decode_context_paged_gb300' not in sys.modules, 'product imported'; print('ok')") % ROOT
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and "ok" in out.stdout, out.stderr[-2000:]


@pytest.mark.gpu
def test_cuda_arm_line(cuda_device):
    line = _run(["--config", "tiny", "--steps", "4", "--warmup", "3", "--no-cpu-baseline"], timeout=600)
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["steps"] == 4 and line["warmup"] == 3
    assert line["n_gpus"] == 1 and line["scaling"] == "weak" and line["vs_baseline"] is None
    roof = line["roofline"]
    assert roof["bound"] in ("hbm", "tensor") and roof["unit"] in ("GB/s", "TFLOP/s")
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    assert "traffic" in roof
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert line["gpu_launches"] > 0
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(line["clocks"])
    assert line["stages"]["pass"]["ms_per_step"] > 0


def _rank_main(rank, world, port, q):
    import os
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="")  # gloo CPU ranks on any machine
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist, r, ws, _ = bench.dist_setup()
    bench.barrier(dist)
    m = bench.max_over_ranks(dist, 1.5 + r)
    q.put((r, ws, m))
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_on_two_gloo_ranks():
    import multiprocessing as mp
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    ps = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 2.5), (1, 2, 2.5)]


def test_reference_arm_under_torchrun_prints_once():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                          "--master-addr", "127.0.0.1", "--master-port", str(port),
                          os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny", "--gpus", "2",
                          "--steps", "1", "--warmup", "0", "--ref-seconds", "1"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300,
                         env={**os.environ, "CUDA_VISIBLE_DEVICES": ""})
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2


@pytest.mark.gpu
def test_layer_pipeline_equals_the_stages_in_order(cuda_device):
    """The bench's layer pipeline (the reshard layer by layer on its own stream, each layer's
    attention after its layer) computes bit for bit what the stages in order compute."""
    import torch
    sys.path.insert(0, ROOT)
    import bench
    import dcp_inputs as di
    import decode_context_paged_gb300 as dcp
    wl = bench.Workload("layers4", cuda_device)
    assert wl.layer_pipe and wl.L == 4 and wl.n_cp == 2
    outs = []
    for pipelined in (True, False, True):
        for p in wl.rc.dst_pools:
            p.view(torch.uint8).fill_(di.SENTINEL_BYTE)
        wl.o.fill_(7.0)
        wl.lse.fill_(7.0)
        wl.step(dcp, events=None if pipelined else {})
        torch.cuda.synchronize()
        assert int(wl.err.item()) == 0
        outs.append((wl.o.clone(), wl.lse.clone()))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])
    assert bool(torch.isfinite(outs[0][0]).all())
