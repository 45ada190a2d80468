"""The benchmark's multi-process (replica) logic on CPU with gloo, world size 2:
rank setup from the torchrun environment, barrier, and max-over-ranks of the
step time that rank 0 reports."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    d = bench.Dist(backend="gloo")
    d.barrier()
    ms = 1.0 + rank * 2.5          # rank 1 is the slow one
    m = d.max(ms)
    d.barrier()
    q.put((rank, d.world, m))
    d.close()


def test_two_ranks_agree_on_max_step_time():
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
    assert res == [(0, 2, 3.5), (1, 2, 3.5)]


def test_single_process_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    import bench
    d = bench.Dist()
    assert d.world == 1 and d.rank == 0 and d.pg is None
    assert d.max(4.0) == 4.0


def test_oracle_sample_counts_bytes_and_threads():
    """The CPU baseline's sampler: bytes are whole (request, kv head) units of
    K+V, and the one-core run reports one thread."""
    import bench
    from split_kv_decode_attention_gb300 import workloads as W
    shp = W.small_shape("cpu_base", batch=2, num_q_heads=4, num_kv_heads=2, lo=50, hi=90, seed=5)
    inp = W.make_host_inputs(shp)
    nbytes, secs, threads, note = bench.oracle_sample(inp, 30.0, max_passes=1, threads=1)
    assert threads == 1 and secs > 0
    # one full pass: every (request, kv head) unit once, K and V rows of 128 bf16
    assert nbytes == int(inp.seq_lens.sum()) * shp.num_kv_heads * shp.head_dim * 2 * 2
    assert note.startswith(f"{shp.batch * shp.num_kv_heads} (request, kv head) units")


def test_reference_arm_prints_the_contract_line():
    """bench.py --impl reference runs the fp64 oracle on the host cores (no
    GPU) and prints one JSON line with the contract's keys."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "0", "--workload", "c1_b1_h32kv8_L4096"],
                         capture_output=True, text=True, timeout=300, cwd=root)
    assert res.returncode == 0, res.stderr[-2000:]
    d = json.loads(res.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert (d["n_gpus"], d["steps"], d["warmup"], d["gpu_launches"]) == (1, 2, 0, 0)
    assert d["higher_is_better"] is True and d["config"]["workload"] == "c1_b1_h32kv8_L4096"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_default_run_times_every_gate_workload_with_c3_as_headline():
    """The default bench covers the five gate workloads; the headline is the
    largest single-GPU one (c3), and the reference arm follows it."""
    import bench
    from split_kv_decode_attention_gb300 import workloads as W
    args = bench.parse_args([])
    assert args.workload == bench.DEFAULT_WORKLOAD
    assert bench.HEADLINE_WORKLOAD in bench.GATE_WORKLOADS
    assert bench.GATE_WORKLOADS == W.WORKLOAD_ORDER   # the five workload recipes
    lens = {n: W.draw_seq_lens(W.WORKLOADS[n], __import__("numpy").random.default_rng(
        W.WORKLOADS[n].seed)) for n in bench.GATE_WORKLOADS}
    kv = {n: int(lens[n].sum()) * W.WORKLOADS[n].num_kv_heads for n in lens}
    assert max(kv, key=kv.get) == bench.HEADLINE_WORKLOAD
