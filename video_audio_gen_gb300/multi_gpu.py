"""Host logic for running the forward on several GPUs, one process per GPU.

Two ways to split the work:

* Whole documents.  Attention is block-diagonal over cu_seqlens, so documents (requests) are
  independent: each rank runs the forward on its own subset of whole documents with the weights
  replicated, and no data-path collective is needed.  `partition_documents` assigns documents to
  ranks, balancing the algorithmic work (linear maps grow with a document's length, attention with
  its square).

* One long document, split by tokens (sequence parallelism in the Ulysses style; [H3] "Not yet
  built -- honestly recorded" lists this multi-GPU USP path as unbuilt upstream).  Every per-token
  step (norms, linear maps, RoPE with the tokens' own positions) runs on each rank's token shard;
  attention needs every key of the document, so around it the shards are exchanged with one
  all-to-all: `scatter_heads` turns [own tokens, all heads] into [all tokens, own heads], attention
  runs per head over the whole document, and `gather_tokens` turns the result back into [own tokens,
  all heads].  Both exchanges move data only, so the result equals the one-GPU attention.

Every function takes sizes and a torch.distributed group; nothing here computes the method.
"""
from __future__ import annotations


def even_shards(n: int, world: int) -> list[tuple[int, int]]:
    """[start, stop) of `world` contiguous shards of n items whose sizes differ by at most one (the
    first n % world shards hold the extra item)."""
    assert n >= 0 and world >= 1
    base, extra = divmod(n, world)
    out, a = [], 0
    for r in range(world):
        b = a + base + (1 if r < extra else 0)
        out.append((a, b))
        a = b
    return out


def document_cost(length: int, model: dict) -> float:
    """Algorithmic FLOPs of one document through the block stack: the linear maps,
    2 S (4 d^2 + 3 d F) per block, and the attention, 4 S^2 d per block."""
    d, F, L = model["hidden"], model["ffn_hidden"], model["n_blocks"]
    S = float(length)
    return L * (2.0 * S * (4.0 * d * d + 3.0 * d * F) + 4.0 * S * S * d)


def partition_documents(lengths, world: int, model: dict) -> list[list[int]]:
    """Assign whole documents to ranks: longest-processing-time first (each document, most expensive
    first, goes to the rank with the least work so far; ties to the lower rank).  Returns, per rank,
    its document indices in packed order.  A rank may receive no document when there are fewer
    documents than ranks."""
    assert world >= 1
    order = sorted(range(len(lengths)), key=lambda j: (-document_cost(lengths[j], model), j))
    load = [0.0] * world
    parts: list[list[int]] = [[] for _ in range(world)]
    for j in order:
        r = min(range(world), key=lambda i: (load[i], i))
        parts[r].append(j)
        load[r] += document_cost(lengths[j], model)
    return [sorted(p) for p in parts]


def _split_sizes(world, rank, n_tokens, n_heads, head_dim):
    ts = even_shards(n_tokens, world)
    hs = even_shards(n_heads, world)
    n_own = ts[rank][1] - ts[rank][0]
    h_own = hs[rank][1] - hs[rank][0]
    return ts, hs, n_own, h_own


def scatter_heads(x_own, n_tokens: int, n_heads: int, head_dim: int, group=None):
    """[own tokens, n_heads * head_dim] -> [n_tokens, own heads * head_dim] across the group.

    Rank r holds the contiguous token shard even_shards(n_tokens, world)[r] and, after the exchange,
    the contiguous head range even_shards(n_heads, world)[r] of every token (rank order is token
    order, so the received blocks stack into the document's rows)."""
    import torch
    import torch.distributed as dist
    world, rank = dist.get_world_size(group), dist.get_rank(group)
    ts, hs, n_own, h_own = _split_sizes(world, rank, n_tokens, n_heads, head_dim)
    assert tuple(x_own.shape) == (n_own, n_heads * head_dim)
    send = torch.cat([x_own[:, a * head_dim:b * head_dim].reshape(-1) for a, b in hs])
    in_split = [n_own * (b - a) * head_dim for a, b in hs]
    out_split = [(b - a) * h_own * head_dim for a, b in ts]
    recv = torch.empty(sum(out_split), dtype=x_own.dtype, device=x_own.device)
    dist.all_to_all_single(recv, send, out_split, in_split, group=group)
    return recv.view(n_tokens, h_own * head_dim)


def gather_tokens(o_heads, n_tokens: int, n_heads: int, head_dim: int, group=None):
    """The inverse exchange: [n_tokens, own heads * head_dim] -> [own tokens, n_heads * head_dim]."""
    import torch
    import torch.distributed as dist
    world, rank = dist.get_world_size(group), dist.get_rank(group)
    ts, hs, n_own, h_own = _split_sizes(world, rank, n_tokens, n_heads, head_dim)
    assert tuple(o_heads.shape) == (n_tokens, h_own * head_dim)
    send = torch.cat([o_heads[a:b].reshape(-1) for a, b in ts])
    in_split = [(b - a) * h_own * head_dim for a, b in ts]
    out_split = [n_own * (b - a) * head_dim for a, b in hs]
    recv = torch.empty(sum(out_split), dtype=o_heads.dtype, device=o_heads.device)
    dist.all_to_all_single(recv, send, out_split, in_split, group=group)
    blocks, off = [], 0
    for (a, b), size in zip(hs, out_split):
        blocks.append(recv[off:off + size].view(n_own, (b - a) * head_dim))
        off += size
    return torch.cat(blocks, dim=1)


def ulysses_attention(q_own, k_own, v_own, n_tokens: int, n_heads: int, head_dim: int, attend, group=None):
    """Attention of one document split by tokens across the group.  q_own, k_own, v_own: this
    rank's token shard [own tokens, n_heads * head_dim], RoPE already applied with the tokens'
    global positions.  attend(q, k, v, h) computes the attention of h heads over the whole document
    ([n_tokens, h * head_dim] each way): on a GPU the library's attention call.  Returns this rank's
    token shard of the output, [own tokens, n_heads * head_dim]."""
    import torch.distributed as dist
    world, rank = dist.get_world_size(group), dist.get_rank(group)
    hs = even_shards(n_heads, world)
    h_own = hs[rank][1] - hs[rank][0]
    q = scatter_heads(q_own, n_tokens, n_heads, head_dim, group)
    k = scatter_heads(k_own, n_tokens, n_heads, head_dim, group)
    v = scatter_heads(v_own, n_tokens, n_heads, head_dim, group)
    o = attend(q, k, v, h_own)
    return gather_tokens(o, n_tokens, n_heads, head_dim, group)
