"""bench.py host logic without a GPU: the workload arithmetic, and the N > 1
replica path over a world-size-2 gloo process group (barrier, max over ranks,
rank 0 alone prints the reference arm's JSON line)."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

import bench
from gated_delta_rule_chunk_gb300.inputs import make_inputs


def test_headline_roofline_arithmetic():
    x = make_inputs(2)
    assert bench.algorithmic_bytes(x) == 105906176          # 25.9 KB/token
    assert abs(bench.algorithmic_flops(x) - 21.65e9) < 0.01e9
    assert bench.n_chunks(x["lengths"]) == 64


def test_stage_boundary_bytes():
    # Headline shape: the scan reads q and k (2 x 16 MiB bf16), w and u in bf16 (2 x 32 MiB:
    # 64 chunks x 32 value heads x 64 x 128 x 2 B each), G (64 x 32 x 64 x 4 B = 0.5 MiB)
    # and the initial state (2 MiB), and writes out (32 MiB bf16) and the final state
    # (2 MiB); the intra stage reads q, k, v (32 MiB), g and beta (0.5 MiB each) and writes
    # w, u and G. 132.5 MiB (138.9 MB) for the scan.
    x = make_inputs(2)
    sb = bench.method_stage_bytes(x)
    MiB = 1 << 20
    assert sb["inter"] == 32 * MiB + 64 * MiB + MiB // 2 + 4 * MiB + 32 * MiB
    assert sb["intra"] == 32 * MiB + 32 * MiB + MiB + 64 * MiB + MiB // 2
    # the whole call's compulsory bytes are what the two stages exchange with the caller
    assert bench.algorithmic_bytes(x) == 32 * MiB + 32 * MiB + 32 * MiB + MiB + 4 * MiB


def test_traffic_entries_are_documented_captures():
    """Each kernel's recorded DRAM traffic names its source file and the profile summary of
    the capture, and that summary names the source revision (SHA-1) the bytes were taken
    on; the bytes are at least the stage's compulsory bytes (a capture cannot move less)."""
    import re
    x = make_inputs(bench.NCU_WORKLOAD)
    sb = bench.method_stage_bytes(x)
    for stage, e in bench.NCU_TRAFFIC.items():
        assert os.path.exists(os.path.join(bench.ROOT, e["source"])), stage
        prof = os.path.join(bench.ROOT, e["profile"])
        assert os.path.exists(prof), stage
        assert re.fullmatch(r"[0-9a-f]{40}", e["sha1"]), stage
        with open(prof) as f:
            assert e["sha1"] in f.read(), stage
        assert e["bytes"] >= sb[stage], stage


def test_backward_roofline_arithmetic():
    # T = 4096, H = 16, Hv = 32, d = 128, bf16 q/k/v, fp32 upstream and output gradients
    x = make_inputs(2)
    # in: q, k (2 x 16 MiB bf16), v (32 MiB), g and beta (1 MiB), the initial state and
    # d_final (2 MiB each), dO (64 MiB fp32); out: dq, dk (64 MiB), dv (64 MiB), dg and
    # dbeta (1 MiB), d_initial_state (2 MiB). The in and out parts equal the end-to-end
    # copies bench.py counts from its tensors (host to device also carries cu_seqlens, 8 B).
    assert bench.bwd_bytes(x) == 139460608 + 137363456
    # per (chunk, value head): S and dS (64 KiB each), v_new and dv_new (32 KiB each),
    # dO (32 KiB) in, three 64 x 128 fp32 results out: 320 KiB, over 64 chunks x 32 heads
    assert bench.bwd_state_bytes(x) == 2048 * 327680
    f = bench.bwd_stage_flops(x)
    # ten 64 x 64 x 128 products, two 64 x 64 x 64 ones and the triangular inverse per
    # (chunk, value head): 2048 x (10485760 + 1048576 + 87381.33)
    assert abs(f["chunk_grads"] - 23801277098.67) < 1.0
    # the reverse scan: three 64 x 128 x 128 products and one 64 x 64 x 128 per step
    assert f["reverse_scan"] == 2048 * (6 * 64 * 128 * 128 + 2 * 64 * 64 * 128)
    assert f["state_products"] == 2048 * 6291456


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=2)
    m = bench.max_over_ranks(float(rank + 1), 2)
    bench.barrier(2)
    dist.destroy_process_group()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--workload", "0", "--steps", "1", "--warmup", "0",
                    "--gpus", "2"])
    q.put((rank, m, buf.getvalue()))


def test_two_rank_replicas_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict()
    for _ in range(2):
        rank, m, out = q.get(timeout=300)
        res[rank] = (m, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == 2.0 and res[1][0] == 2.0
    assert res[1][1].strip() == ""
    line = json.loads(res[0][1].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
