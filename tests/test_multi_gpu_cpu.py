"""The multi-GPU host logic on CPU with two gloo ranks: whole-document partitioning and the Ulysses
head-scatter exchange for one long document.  The attention and forward each rank runs here are the
oracle's (the kernels' stand-in on a machine without GPUs); the exchanges and the partition are the
library's own host code, and each result must equal the one-process oracle run bit for bit, since
both only move data."""
import os
import socket

import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _spawn(target, world, *args):
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, world, port, q) + args) for r in range(world)]
    for p in procs:
        p.start()
    # drain the queue before joining: a child cannot exit while its large result is still in the pipe
    try:
        res = [q.get(timeout=300) for _ in range(world)]
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return sorted(res, key=lambda t: t[0])


def test_even_shards_and_partition():
    from video_audio_gen_gb300 import multi_gpu as mg
    assert mg.even_shards(1001, 2) == [(0, 501), (501, 1001)]
    assert mg.even_shards(5, 3) == [(0, 2), (2, 4), (4, 5)]
    assert mg.even_shards(2, 4) == [(0, 1), (1, 2), (2, 2), (2, 2)]
    m = synth.C2_MODEL
    # the loop's two ragged requests on two GPUs: one each
    loop = synth.WORKLOADS["denoise_loop"]
    lens = [synth.doc_tokens(d) for d in loop["docs"]]
    assert mg.partition_documents(lens, 2, m) == [[0], [1]]
    # 13 short documents on 3 GPUs: every document exactly once, work balanced
    lens = [synth.doc_tokens(d) for d in synth.WORKLOADS["many_docs"]["docs"]]
    parts = mg.partition_documents(lens, 3, m)
    assert sorted(j for p in parts for j in p) == list(range(len(lens)))
    loads = [sum(mg.document_cost(lens[j], m) for j in p) for p in parts]
    assert max(loads) <= 1.25 * (sum(loads) / 3) + max(mg.document_cost(n, m) for n in lens) * 0.01
    # more ranks than documents: the spare ranks get nothing
    assert mg.partition_documents([10, 20], 3, m) == [[1], [0], []]


def _ulysses_worker(rank, world, port, q, n, H, Dh):
    import torch.distributed as dist

    import oracle
    from video_audio_gen_gb300 import multi_gpu as mg
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        d = H * Dh
        qf = synth.normal(500, "uq", (n, d), 1.0).astype(np.float64)
        kf = synth.normal(500, "uk", (n, d), 1.0).astype(np.float64)
        vf = synth.normal(500, "uv", (n, d), 1.0).astype(np.float64)
        a, b = mg.even_shards(n, world)[rank]
        t = lambda x: torch.from_numpy(np.ascontiguousarray(x[a:b]))

        def attend(qh, kh, vh, h):
            return torch.from_numpy(oracle.attention(qh.numpy(), kh.numpy(), vh.numpy(),
                                                     np.array([0, n], dtype=np.int32), h, Dh))

        o = mg.ulysses_attention(t(qf), t(kf), t(vf), n, H, Dh, attend)
        q.put((rank, a, b, o.numpy()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("n,H", [(1001, 5), (640, 4)])
def test_ulysses_attention_two_ranks_equals_one_process(n, H):
    """One document split by tokens over two ranks (uneven tokens and heads in the first case): the
    head-scatter all-to-all, per-head attention over the whole document and the gather back give the
    one-process attention bit for bit."""
    import oracle
    Dh = 16
    res = _spawn(_ulysses_worker, 2, n, H, Dh)
    d = H * Dh
    qf = synth.normal(500, "uq", (n, d), 1.0).astype(np.float64)
    kf = synth.normal(500, "uk", (n, d), 1.0).astype(np.float64)
    vf = synth.normal(500, "uv", (n, d), 1.0).astype(np.float64)
    ref = oracle.attention(qf, kf, vf, np.array([0, n], dtype=np.int32), H, Dh)
    got = np.concatenate([r[3] for r in res])
    assert [(r[1], r[2]) for r in res] == [(0, (n + 1) // 2), ((n + 1) // 2, n)]
    assert np.array_equal(got, ref)


def _partition_worker(rank, world, port, q):
    import torch.distributed as dist

    import oracle
    from video_audio_gen_gb300 import multi_gpu as mg
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = synth.WORKLOADS["many_docs"]
        m = dict(w["model"], n_blocks=1)
        full = synth.build_layout(w["docs"])
        x = synth.make_tokens(w, full)
        W = synth.make_weights(dict(w, model=m))
        lens = [synth.doc_tokens(dd) for dd in w["docs"]]
        mine = mg.partition_documents(lens, world, m)[rank]
        lay = synth.build_layout([w["docs"][j] for j in mine])
        cu = full["cu_seqlens"]
        rows = np.concatenate([np.arange(cu[j], cu[j + 1]) for j in mine])
        out, _ = oracle.forward(m, W, x[rows], lay, 0.61)
        got = [None] * world
        dist.all_gather_object(got, (rows, out))
        q.put((rank, got if rank == 0 else None))
    finally:
        dist.destroy_process_group()


def test_document_partition_two_ranks_equals_one_process():
    """13 documents split over two ranks by the partition: each rank runs the forward on its own
    documents only, and the gathered rows equal the one-process forward over all of them, bit for
    bit (documents share no data-path step)."""
    import oracle
    res = _spawn(_partition_worker, 2)
    w = synth.WORKLOADS["many_docs"]
    m = dict(w["model"], n_blocks=1)
    full = synth.build_layout(w["docs"])
    x = synth.make_tokens(w, full)
    W = synth.make_weights(dict(w, model=m))
    ref, _ = oracle.forward(m, W, x, full, 0.61)
    got = np.full_like(ref, np.nan)
    seen = np.zeros(full["n_tokens"], dtype=int)
    for rows, out in res[0][1]:
        got[rows] = out
        seen[rows] += 1
    assert (seen == 1).all()
    assert np.array_equal(got, ref)
