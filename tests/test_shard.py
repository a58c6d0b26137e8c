"""Head-sharded multi-rank execution on CPU (gloo): the partition of the C
library, the Ulysses exchange around the attention (sequence-sharded ->
head-sharded -> attention -> sequence-sharded) and the int8-KV group split.

Each rank computes the attention of its own heads with the oracle (these
tests run without a GPU); the reassembled result must equal a single-process
oracle run over all heads bit for bit, so the partition, the exchanges and the
reassembly lose, duplicate or reorder nothing."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import quantized_attention_sage_gb300 as qas
import synth


@pytest.fixture(scope="module", autouse=True)
def built():
    qas.build()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("units", [0, 1, 5, 24, 37810, 3 * 2**31])
@pytest.mark.parametrize("world", [1, 2, 3, 7, 8])
def test_shard_range_is_a_balanced_contiguous_partition(units, world):
    ranges = [qas.sage_shard_range(units, world, r) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == units
    for (b0, e0), (b1, e1) in zip(ranges, ranges[1:]):
        assert e0 == b1                                   # contiguous, in rank order, disjoint
    sizes = [e - b for b, e in ranges]
    assert min(sizes) >= 0 and max(sizes) - min(sizes) <= 1
    assert max(sizes) == -(-units // world)               # no rank holds more than ceil(units / world)
    assert sizes == sorted(sizes, reverse=True)           # the larger shares come first


def test_shard_range_rejects_bad_arguments():
    for args in ((-1, 2, 0), (10, 0, 0), (10, 2, 2), (10, 2, -1)):
        with pytest.raises(qas.SageError):
            qas.sage_shard_range(*args)


# ---------------------------------------------------------------------------
# dense path: Ulysses exchange + per-rank heads
# ---------------------------------------------------------------------------

BQ = BK = 64


def _workload(nq, nk, H):
    w = synth.DenseWorkload("shard", 11, 1, H, nq, nk, BQ, sub=H)
    return w, synth.dense_inputs(w)


def _bf16_tensor(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def _oracle_attend(q, k, v):
    """attention of head-sharded [hh, N, 128] bf16 tensors by the oracle, bf16 out"""
    outs = []
    for h in range(q.shape[0]):
        bits = [t[h].contiguous().view(torch.int16).numpy().view(np.uint16) for t in (q, k, v)]
        outs.append(oracle.sage_head(*bits, BQ, BK, nthreads=1)["out_bf16"])
    return _bf16_tensor(np.stack(outs))


def _dense_rank(rank, world, port, nq, nk, H, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    from quantized_attention_sage_gb300 import shard

    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, x = _workload(nq, nk, H)
    q, k, v = (_bf16_tensor(x[n][0]) for n in ("q", "k", "v"))      # [H, N, 128]
    tq0, tq1 = qas.sage_shard_range(nq, world, rank)
    tk0, tk1 = qas.sage_shard_range(nk, world, rank)
    seen = {}

    def attend(qh, kh, vh):
        seen["heads"] = (qh.clone(), kh.clone(), vh.clone())
        return _oracle_attend(qh, kh, vh)

    out_tok = shard.sage_attention_ulysses(q[:, tq0:tq1].contiguous(), k[:, tk0:tk1].contiguous(),
                                           v[:, tk0:tk1].contiguous(), nq, nk, BQ, BK, attend=attend)
    h0, h1 = shard.head_range(H)
    results[rank] = dict(out=out_tok.view(torch.int16).numpy().copy(), heads=(h0, h1), tok=(tq0, tq1),
                         exchanged=all(torch.equal(a.view(torch.int16), b[h0:h1].view(torch.int16))
                                       for a, b in zip(seen["heads"], (q, k, v))))
    dist.destroy_process_group()


def _spawn(fn, world, *args):
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=fn, args=(r, world, port) + args + (results,)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0
    return dict(results)


@pytest.mark.parametrize("world,nq,nk,H", [(2, 150, 150, 5), (3, 97, 230, 4)])
def test_ulysses_head_sharded_attention_equals_one_process(world, nq, nk, H):
    res = _spawn(_dense_rank, world, nq, nk, H)
    w, x = _workload(nq, nk, H)
    want = np.stack([oracle.sage_head(x["q"][0, h], x["k"][0, h], x["v"][0, h], BQ, BK, nthreads=1)["out_bf16"]
                     for h in range(H)]).view(np.int16)                                   # [H, Nq, 128]
    covered = []
    for r in range(world):
        t0, t1 = res[r]["tok"]
        assert res[r]["exchanged"], f"rank {r}: the head-sharded inputs are not the rank's heads"
        assert np.array_equal(res[r]["out"], want[:, t0:t1]), f"rank {r}"
        covered.append(res[r]["heads"])
    # every head was computed by exactly one rank
    assert sorted(covered)[0][0] == 0 and sorted(covered)[-1][1] == H
    assert sum(e - b for b, e in covered) == H


# ---------------------------------------------------------------------------
# int8 KV cache: whole kv-head groups per rank
# ---------------------------------------------------------------------------

def _kv_workload(Hkv):
    return synth.Int8KVWorkload("shard_kv", 6, 40, 200, 4 * Hkv, Hkv, 0.01, 8.0, sub=Hkv)


def _kv_rank(rank, world, port, Hkv, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist

    from kv_helpers import oracle_cache
    from quantized_attention_sage_gb300 import shard

    dist.init_process_group("gloo", rank=rank, world_size=world)
    w = _kv_workload(Hkv)
    x = oracle_cache(synth.int8kv_inputs(w))
    (g0, g1), (h0, h1) = shard.int8kv_group_heads(w.Hq, w.Hkv)
    local = torch.zeros((w.Nq, 0, 128), dtype=torch.float64)
    if g1 > g0:  # a rank with no kv head has nothing to compute
        # the rank holds only its kv heads' cache and its query heads
        q = np.ascontiguousarray(x["q"][:, h0:h1])
        rows, heads = np.meshgrid(np.arange(w.Nq), np.arange(h1 - h0), indexing="ij")
        out, _ = oracle.int8kv_rows(q, x["k"][g0:g1], x["k_scale"][g0:g1], x["v"][g0:g1], x["v_scale"][g0:g1],
                                    w.q_pos0, rows.ravel(), heads.ravel(), nthreads=1)
        local = torch.from_numpy(out.reshape(w.Nq, h1 - h0, 128))
    # gather the query heads of all ranks (uneven shares: pad to the largest)
    G = w.Hq // w.Hkv
    most = -(-w.Hkv // world) * G
    pad = torch.zeros((w.Nq, most, 128), dtype=torch.float64)
    pad[:, :h1 - h0] = local
    got = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(got, pad)
    parts = []
    for r in range(world):
        b, e = qas.sage_shard_range(w.Hkv, world, r)
        parts.append(got[r][:, :(e - b) * G])
    results[rank] = dict(out=torch.cat(parts, dim=1).numpy(), groups=(g0, g1), heads=(h0, h1))
    dist.destroy_process_group()


@pytest.mark.parametrize("world,Hkv", [(2, 3), (3, 2)])
def test_int8kv_group_sharded_attention_equals_one_process(world, Hkv):
    # uneven shares (3 groups over 2 ranks) and a rank with none (2 over 3)
    res = _spawn(_kv_rank, world, Hkv)
    from kv_helpers import oracle_cache

    w = _kv_workload(Hkv)
    x = oracle_cache(synth.int8kv_inputs(w))
    rows, heads = np.meshgrid(np.arange(w.Nq), np.arange(w.Hq), indexing="ij")
    want, _ = oracle.int8kv_rows(x["q"], x["k"], x["k_scale"], x["v"], x["v_scale"], w.q_pos0, rows.ravel(),
                                 heads.ravel(), nthreads=1)
    want = want.reshape(w.Nq, w.Hq, 128)
    G = w.Hq // w.Hkv
    for r in range(world):
        g0, g1 = res[r]["groups"]
        assert res[r]["heads"] == (g0 * G, g1 * G)
        assert np.array_equal(res[r]["out"], want)
