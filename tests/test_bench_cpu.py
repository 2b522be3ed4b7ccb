"""bench.py's host-side logic without a GPU: the reference arm's JSON line and the rank aggregation."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    sys.path.insert(0, ROOT)
    import bench

    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == bench.host_cores()
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["steps"] == 2 and line["warmup"] == 3
    assert line["metric"] == bench.METRIC  # the GPU arm prints the same metric string


def test_packed_views_are_aligned_and_hold_the_arrays():
    """The per-step inputs and outputs live in one buffer each (one host copy per direction): every view starts
    on a 256-byte boundary (the kernels want 16) and holds its array's values and type."""
    import numpy as np

    sys.path.insert(0, ROOT)
    import bench

    arrays = [np.arange(7, dtype=np.float32), np.arange(6, dtype=np.int32).reshape(2, 3),
              np.full((3, 5), 2.5, np.float32)]
    buf, views = bench.packed(arrays, "cpu")
    for a, v in zip(arrays, views):
        assert (v.data_ptr() - buf.data_ptr()) % 256 == 0
        assert tuple(v.shape) == a.shape and np.array_equal(v.numpy(), a)
    assert buf.numel() == 3 * 256


@pytest.mark.parametrize("n,parts", [(1, 4), (7, 3), (18944, 16), (5, 8), (64, 1)])
def test_row_chunks_cover_the_rows_once(n, parts):
    sys.path.insert(0, ROOT)
    import bench

    ch = bench.row_chunks(n, parts)
    assert len(ch) <= parts and ch[0][0] == 0 and ch[-1][1] == n
    assert all(lo < hi for lo, hi in ch) and all(a[1] == b[0] for a, b in zip(ch, ch[1:]))


def test_oracle_on_row_chunks_equals_the_whole(oracle_lib):
    """The multithreaded host leg splits every call's rows over threads: the oracle's rows are independent, so
    the chunks' results side by side are the whole call's, bit for bit."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    sys.path.insert(0, ROOT)
    import bench
    import synth

    g = synth.make_gateup(3, 70, 512)
    whole = oracle_lib.fused_gateup_q4k_gemv(g["w_gate"], g["w_up"], g["x"], g["gamma"], 1e-5)
    with ThreadPoolExecutor(4) as pool:
        parts = list(pool.map(lambda r: oracle_lib.fused_gateup_q4k_gemv(g["w_gate"][r[0]:r[1]], g["w_up"][r[0]:r[1]],
                                                                         g["x"], g["gamma"], 1e-5),
                              bench.row_chunks(70, 4)))
    for s in range(2):
        for k in range(2):
            assert np.array_equal(np.concatenate([p[s][k] for p in parts]), whole[s][k])


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--warmup", "2"],
                       capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode != 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    secs = [0.5, 0.8][rank]  # the slower rank sets the job's time
    value, t = bench.aggregate(secs, bytes_per_step=1e9, steps=10, world=world)
    bench.barrier(world)
    q.put((rank, value, t))
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, t in res:
        assert t == pytest.approx(0.8)
        assert value == pytest.approx(2 * 1e9 * 10 / 0.8 / 1e9)
