"""Head-sharded multi-GPU execution of the quantized attention path.

Every (batch, head) attention problem is independent, so a multi-GPU run puts
whole heads on ranks.  The pages name the layout for distributed execution:
QKV tiles land in rank-destined Ulysses buffers and the attention output goes
back to the caller's local token-major layout ("H3 Performance Roadmap",
section "Phase 3: NVFP4 Fused Projection Prototype", the paragraph on the
direct-layout target).  That is one exchange step on each side of the
attention:

  * ``ulysses_heads``: the all-to-all that turns a sequence-sharded tensor
    (this rank's tokens of every head) into a head-sharded one (this rank's
    heads, every token).  Remote tiles arrive in a receive buffer and are
    copied into local memory before any kernel reads them.
  * the attention of the rank's heads, in the library's kernels
    (``sage_attention`` on device buffers);
  * ``ulysses_tokens``: the inverse all-to-all, back to this rank's tokens of
    every head.

Heads and tokens are split by ``sage_shard_range`` of the C library
(contiguous ranges in rank order, the first ``units % world`` ranks one more).
The int8 KV-cache prompt attention shards whole kv-head groups instead (a kv
head and its Hq/Hkv query heads stay on one rank), with no exchange at all:
``int8kv_group_heads`` gives a rank's kv heads and query heads.

The collectives are torch.distributed ``all_to_all_single`` calls (NCCL
between GPUs, gloo in the CPU tests); the payload travels as raw bytes, so
every dtype crosses bit for bit.  Nothing here computes attention.
"""

from __future__ import annotations

from . import sage_attention, sage_shard_range


def _dist():
    import torch.distributed as dist

    return dist


def _world_rank(group):
    dist = _dist()
    if not dist.is_available() or not dist.is_initialized():
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


def _as_bytes(t):
    """A contiguous tensor's storage as a flat uint8 tensor (no copy)."""
    import torch

    return t.contiguous().view(-1).view(torch.uint8)


def _exchange(send_chunks, recv_shapes, dtype, device, group):
    """all_to_all of one chunk per destination rank (in rank order) into
    buffers of the given shapes (one per source rank); returns the received
    tensors.  With a single rank the chunk is returned as it is."""
    import torch

    world, _ = _world_rank(group)
    if world == 1:
        return [send_chunks[0].reshape(recv_shapes[0])]
    dist = _dist()
    send = torch.cat([_as_bytes(c) for c in send_chunks])
    in_split = [c.numel() * c.element_size() for c in send_chunks]
    esize = torch.empty((), dtype=dtype).element_size()
    out_split = [int(torch.Size(s).numel()) * esize for s in recv_shapes]
    recv = torch.empty(sum(out_split), dtype=torch.uint8, device=device)
    dist.all_to_all_single(recv, send, out_split, in_split, group=group)
    out, off = [], 0
    for s, n in zip(recv_shapes, out_split):
        out.append(recv[off:off + n].view(dtype).view(s))
        off += n
    return out


def head_range(units: int, group=None) -> tuple[int, int]:
    """This rank's [begin, end) of `units` heads."""
    world, rank = _world_rank(group)
    return sage_shard_range(units, world, rank)


def ulysses_heads(x_tok, n_total: int, group=None):
    """Sequence-sharded -> head-sharded.

    x_tok: [BH, n_local, D], this rank's token range (``sage_shard_range(n_total,
    world, rank)``) of all BH heads.  Returns [h1 - h0, n_total, D]: this rank's
    heads (``sage_shard_range(BH, world, rank)``) over every token."""
    import torch

    world, rank = _world_rank(group)
    BH, n_local, D = x_tok.shape
    t0, t1 = sage_shard_range(n_total, world, rank)
    if t1 - t0 != n_local:
        raise ValueError(f"rank {rank} holds {n_local} tokens, its shard of {n_total} is {t1 - t0}")
    heads = [sage_shard_range(BH, world, r) for r in range(world)]
    toks = [sage_shard_range(n_total, world, r) for r in range(world)]
    h0, h1 = heads[rank]
    send = [x_tok[b:e] for b, e in heads]                       # to rank s: its heads, my tokens
    recv_shapes = [(h1 - h0, e - b, D) for b, e in toks]         # from rank r: my heads, its tokens
    parts = _exchange(send, recv_shapes, x_tok.dtype, x_tok.device, group)
    return torch.cat(parts, dim=1)                               # tokens in order: a local copy


def ulysses_tokens(y_heads, BH: int, group=None):
    """Head-sharded -> sequence-sharded, the inverse of ``ulysses_heads``.

    y_heads: [h1 - h0, n_total, D] (this rank's heads).  Returns [BH, n_local, D]:
    this rank's token range of every head."""
    import torch

    world, rank = _world_rank(group)
    hh, n_total, D = y_heads.shape
    heads = [sage_shard_range(BH, world, r) for r in range(world)]
    toks = [sage_shard_range(n_total, world, r) for r in range(world)]
    if heads[rank][1] - heads[rank][0] != hh:
        raise ValueError(f"rank {rank} holds {hh} heads, its shard of {BH} is {heads[rank][1] - heads[rank][0]}")
    t0, t1 = toks[rank]
    send = [y_heads[:, b:e] for b, e in toks]                    # to rank s: my heads, its tokens
    recv_shapes = [(e - b, t1 - t0, D) for b, e in heads]        # from rank r: its heads, my tokens
    parts = _exchange(send, recv_shapes, y_heads.dtype, y_heads.device, group)
    return torch.cat(parts, dim=0)


def sage_attention_ulysses(q_tok, k_tok, v_tok, Nq: int, Nk: int, q_block: int = 64, k_block: int = 64,
                           sm_scale: float = 0.0, causal: bool = False, group=None, attend=None):
    """Dense quantized attention on sequence-sharded inputs, heads sharded over ranks.

    q_tok: [BH, nq_local, 128], k_tok, v_tok: [BH, nk_local, 128] bf16, this rank's
    token ranges of Nq queries and Nk keys.  Returns [BH, nq_local, 128] bf16: the
    attention output of this rank's queries for every head, equal bit for bit to a
    single-process run over all heads.  ``attend(q, k, v)`` maps head-sharded
    [hh, N, 128] tensors to the output [hh, Nq, 128]; by default the library's
    one-call dense path on the rank's GPU."""
    if attend is None:
        def attend(q, k, v):
            out = sage_attention(q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), q_block, k_block,
                                 sm_scale=sm_scale, causal=causal)
            return out.squeeze(0)
    BH = q_tok.shape[0]
    q = ulysses_heads(q_tok, Nq, group)
    k = ulysses_heads(k_tok, Nk, group)
    v = ulysses_heads(v_tok, Nk, group)
    return ulysses_tokens(attend(q, k, v), BH, group)


def int8kv_group_heads(Hq: int, Hkv: int, group=None) -> tuple[tuple[int, int], tuple[int, int]]:
    """This rank's kv heads [g0, g1) of the int8 cache and the query heads
    [g0 * G, g1 * G) that read them (G = Hq / Hkv): whole groups per rank, so the
    rank's cache shard serves its queries with no exchange."""
    if Hkv < 1 or Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    g0, g1 = head_range(Hkv, group)
    G = Hq // Hkv
    return (g0, g1), (g0 * G, g1 * G)
