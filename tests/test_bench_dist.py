"""The bench's multi-process plumbing on CPU (gloo, world size 2): the layer has no
cross-GPU exchange, so N processes run N replicas; what must hold is the barrier, the
max-over-ranks timing and one JSON line from rank 0 (and, for the reference arm, that only
rank 0 does any work)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local, d = bench.dist_setup(None)
    assert (w, r, local) == (world, rank, rank) and d is not None
    bench.barrier(d, torch.device("cpu"))
    got = bench.max_over_ranks(d, float(10 * (rank + 1)), torch.device("cpu"))
    q.put((rank, got))
    d.destroy_process_group()


def test_barrier_and_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert res == [(0, 20.0), (1, 20.0)]


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"), "--impl", "reference",
           "--gpus", "2", "--workload", "tiny", "--steps", "5", "--warmup", "1"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_traffic_is_reported_only_for_the_captured_configuration(tmp_path):
    # The committed ncu byte counts belong to one configuration and one version of the kernel
    # sources; any other configuration, or an edited source, reports null rather than a
    # stale count.
    sys.path.insert(0, ROOT)
    import bench
    srcs = ["video_diffusion_dit_gb300/csrc/apply.cu", "video_diffusion_dit_gb300/csrc/ptx.cuh",
            "video_diffusion_dit_gb300/csrc/lin_attn_internal.cuh"]
    cfg = {"workload": "720p_193f", "mode": "high", "out_dtype": "f32", "layout": "hnd", "fused": False}
    cap = {"captures": [
        {"config": cfg, "kernels": {"apply_tc_kernel": {"sources": srcs, "sources_sha256": bench.sources_sha256(srcs),
                                                         "bytes_per_launch_full": 123}}},
        {"config": {**cfg, "layout": "nhd"},
         "kernels": {"apply_tc_kernel": {"sources": srcs, "sources_sha256": bench.sources_sha256(srcs),
                                         "bytes_per_launch_full": 456}}},
    ]}
    cur = tmp_path / "current.json"
    cur.write_text(json.dumps(cap))
    assert bench.kernel_traffic("apply_tc_kernel", cfg, str(cur)) == 123
    assert bench.kernel_traffic("apply_tc_kernel", {**cfg, "layout": "nhd"}, str(cur)) == 456
    for key, other in (("workload", "480p_81f"), ("mode", "lossless"), ("out_dtype", "bf16"), ("fused", True)):
        assert bench.kernel_traffic("apply_tc_kernel", {**cfg, key: other}, str(cur)) is None
    assert bench.kernel_traffic("apply_fused_kernel", cfg, str(cur)) is None
    for c in cap["captures"]:
        c["kernels"]["apply_tc_kernel"]["sources_sha256"] = "0" * 64
    old = tmp_path / "stale.json"
    old.write_text(json.dumps(cap))
    assert bench.kernel_traffic("apply_tc_kernel", cfg, str(old)) is None
    # The committed captures parse, and each names sources that exist.
    with open(os.path.join(ROOT, "profiles", "ncu_dram_traffic.json")) as f:
        committed = json.load(f)
    for c in committed["captures"]:
        for ent in c["kernels"].values():
            assert bench.sources_sha256(ent["sources"]) is not None
