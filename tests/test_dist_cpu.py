"""The multi-GPU host logic of the bench on CPU: two gloo ranks (world size 2).

The forward shards by whole documents (attention is block-diagonal), so ranks exchange nothing on the
data path: each rank runs its own copy of the workload's documents (weak scaling) and the only
collective is the max-over-ranks of the timed region."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import bench
    import synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.WORKLOADS["video_audio_bf16"]
        docs = bench.rank_documents(w["docs"], rank, world)
        lay = synth.build_layout(docs)
        seed = bench.rank_seed(w["seed"], rank)
        ms = bench.reduce_max_ms(10.0 + rank * 5.0, dist)  # rank 1 is the slow one
        q.put((rank, lay["n_tokens"], [int(v) for v in lay["cu_seqlens"]], seed, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling_and_max_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    # every rank holds the full per-rank workload: 17,408 tokens in 2 documents
    assert [r[1] for r in res] == [17408, 17408]
    assert res[0][2] == res[1][2] == [0, 8704, 17408]
    assert res[0][3] != res[1][3]  # independent requests: different seeded inputs per rank
    assert [r[4] for r in res] == [15.0, 15.0]  # the job time is the slowest rank's


def test_single_process_helpers():
    import bench
    assert bench.reduce_max_ms(3.5, None) == 3.5
    fl = bench.step_flops({"hidden": 3072, "ffn_hidden": 8192, "n_blocks": 8}, [0, 8704, 17408])
    assert abs(fl["total"] / 1e12 - 46.437) < 1e-3  # 31.54 TFLOP of GEMMs + 14.90 of attention
