"""Host-side logic of bench.py on CPU: the replica timing reduction over two
gloo ranks, the rank-0-only reference arm, and the byte accounting."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.reduce_max(10.0 + rank * 5.0, world)
        ref = bench.run_reference(type("A", (), {"steps": 1, "warmup": 0})(), rank, world) \
            if rank == 1 else "skipped"
        q.put((rank, got, ref))
    finally:
        dist.destroy_process_group()


def test_replica_max_time_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][1] == 15.0 and res[1][1] == 15.0   # both ranks see the max
    assert res[1][2] is None                          # rank 1 runs no reference work


def test_single_process_reduce_is_identity():
    assert bench.reduce_max(3.5, 1) == 3.5


def test_step_bytes_counts_weights_scales_and_activations():
    # q: 6144 x 5120 nvfp4 = 0.5625 B per weight, plus M*K*2 activation bytes
    assert bench.weight_bytes(6144, 5120) == 6144 * 5120 * 9 // 16
    assert bench.weight_bytes(6144, 5120, "q4_0") == 6144 * 5120 * 9 // 16
    total = sum(n * k * 9 // 16 + 8 * k * 2 for _, n, k in bench.STEP)
    assert bench.step_bytes(8) == total
    assert abs(bench.step_bytes(8) / 1e6 - 192.2) < 0.1
    # the packed step holds exactly the seven linears' weights; the shared
    # inputs of q/k/v and gate/up are read once instead of three and two times
    w7 = sum(n * k * 9 // 16 for _, n, k in bench.LAYER)
    w4 = sum(n * k * 9 // 16 for _, n, k in bench.STEP)
    assert w7 == w4
    assert bench.step_bytes(8, spec=bench.LAYER) - total == 8 * 5120 * 2 * 3


def test_depth_controller_summary_over_sixteen_widths():
    """The bench's controller summary from per-M step times (M = 1..16):
    widths interpolated, depths 0..15 rated, the choice the best rate."""
    lay = {"1": 57.2, "2": 57.5, "4": 57.5, "8": 57.6, "16": 73.4}
    per_m = {"nvfp4": {m: {"layer_us": us} for m, us in lay.items()}}
    d = bench.depth_controller_summary(per_m)
    assert sorted(d["verify_us"]) == list(range(1, 17))
    assert d["verify_us"][12] == pytest.approx(57.6 + (73.4 - 57.6) * 4 / 8, abs=0.01)
    rates = d["committed_tokens_per_ms"]
    assert sorted(rates) == list(range(16))
    assert d["chosen_depth"] == max(rates, key=lambda k: (rates[k], -k))
