"""Parity of int8kv_prompt_attn (CUDA) with the fp64 oracle of the int8
KV-cache prompt attention: bf16 output within max-abs 2e-3 and rel-L2 1e-3
of the oracle rounded to bf16.  Each side reads its own copy of the cache (the
oracle's quantiser on the host, the library's cache writer on the device),
checked bit for bit first."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_output_close, assert_output_close_rows, bf16_to_f64
from kv_helpers import both_caches

pytestmark = pytest.mark.gpu


def run(qas, w, x):
    """Both caches, then the attention on the device one; returns (oracle inputs, output)."""
    host, (q, kc, ks, vc, vs) = both_caches(qas, x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = qas.int8kv_prompt_attn(q, kc, ks, vc, vs, w.q_pos0, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return host, out


def oracle_bf16(w, x, rows, heads):
    ref, _ = oracle.int8kv_rows(x["q"], x["k"], x["k_scale"], x["v"], x["v_scale"], w.q_pos0, rows, heads)
    return oracle.bf16_value(oracle.f32_to_bf16(ref.astype(np.float32))), ref


SMALL = [
    synth.int8kv_workload("tiny_kv_q96_k300"),
    synth.Int8KVWorkload("kv_g1", 9, 70, 200, 2, 2, sub=1),
    synth.Int8KVWorkload("kv_g8", 9, 40, 333, 16, 2, sub=2),
    synth.Int8KVWorkload("kv_g3_ragged", 9, 50, 129, 6, 2, sub=3),
    synth.Int8KVWorkload("kv_from_zero", 9, 200, 200, 4, 1, sub=4),
    synth.Int8KVWorkload("kv_one_query", 9, 1, 1000, 8, 8, sub=5),
    # wide query-head groups: 5 (125 rows per tile), 32 (4 queries per tile) and
    # the largest, 128 (one query per tile)
    synth.Int8KVWorkload("kv_g5", 9, 37, 261, 10, 2, sub=8),
    synth.Int8KVWorkload("kv_g32", 9, 9, 300, 64, 2, sub=9),
    synth.Int8KVWorkload("kv_g128", 9, 3, 140, 128, 1, sub=10),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_int8kv_matches_oracle_all_rows(cuda_lib, w):
    x, out = run(cuda_lib, w, synth.int8kv_inputs(w))
    rows, heads = np.meshgrid(np.arange(w.Nq), np.arange(w.Hq), indexing="ij")
    ref_b, _ = oracle_bf16(w, x, rows.ravel(), heads.ravel())
    got = bf16_to_f64(out).reshape(-1, 128)
    assert_output_close(got, ref_b, w.name)


# Mid-size cases whose query tiles fill the GPU without split-KV, so one CTA
# walks 16-40 key tiles and every shared-memory ring wraps many times.
LONG = [
    synth.Int8KVWorkload("kv_long_g4", 9, 1024, 4096, 32, 8, sub=6),
    synth.Int8KVWorkload("kv_long_g8_outliers", 9, 640, 5000, 64, 8, 0.01, sub=7),
]


@pytest.mark.parametrize("w", LONG, ids=lambda w: w.name)
def test_int8kv_long_key_range_sampled(cuda_lib, w):
    x, out = run(cuda_lib, w, synth.int8kv_inputs(w))
    rng = np.random.default_rng(5)
    rows = np.concatenate([rng.integers(0, w.Nq, 60), [0, w.Nq - 1]])
    heads = np.concatenate([rng.integers(0, w.Hq, 60), [0, w.Hq - 1]])
    ref_b, _ = oracle_bf16(w, x, rows, heads)
    got = bf16_to_f64(out[torch.as_tensor(rows).cuda(), torch.as_tensor(heads).cuda()])
    assert_output_close(got, ref_b, w.name)


@pytest.mark.parametrize("name", ["prompt32k_q1024", "prompt64k_q512_outliers"])
def test_int8kv_full_size_sampled(cuda_lib, name):
    w = synth.int8kv_workload(name)
    x, out = run(cuda_lib, w, synth.int8kv_inputs(w))
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(11)
    rows = np.concatenate([rng.integers(0, w.Nq, 40), [0, w.Nq - 1, 31, 32]])
    heads = np.concatenate([rng.integers(0, w.Hq, 40), [0, w.Hq - 1, 5, 6]])
    ref_b, ref = oracle_bf16(w, x, rows, heads)
    got = bf16_to_f64(out[torch.as_tensor(rows).cuda(), torch.as_tensor(heads).cuda()])
    max_abs, rel = assert_output_close(got, ref_b, name)
    scale = np.abs(ref).max()
    print(f"{name}: max-abs {max_abs:.2e} rel-L2 {rel:.2e} (output scale {scale:.2f}); "
          f"vs unrounded fp64 max-abs {np.abs(got - ref).max():.2e}")


@pytest.mark.parametrize("name", ["prompt32k_q1024", "prompt64k_q512_outliers"])
def test_int8kv_full_size_whole_kv_group(cuda_lib, name):
    """Every row of one whole kv-head group (its 4 query heads x all queries)
    of the full-size chunk against the fp64 oracle at the full bar."""
    w = synth.int8kv_workload(name)
    x, out = run(cuda_lib, w, synth.int8kv_inputs(w))
    G = w.Hq // w.Hkv
    g = w.Hkv - 1
    rows, heads = np.meshgrid(np.arange(w.Nq), np.arange(g * G, (g + 1) * G), indexing="ij")
    rows, heads = rows.ravel(), heads.ravel()
    ref_b, ref = oracle_bf16(w, x, rows, heads)
    got = bf16_to_f64(out[torch.as_tensor(rows).cuda(), torch.as_tensor(heads).cuda()])
    max_abs, rel = assert_output_close(got, ref_b, f"{name} kv group {g}")
    print(f"{name} kv group {g}: {rows.size} rows, max-abs {max_abs:.2e} rel-L2 {rel:.2e}; "
          f"vs unrounded fp64 rel-L2 {np.linalg.norm(got - ref) / np.linalg.norm(ref):.2e}")


def test_int8kv_late_dominant_keys(cuda_lib):
    """Keys far above everything before them, in key tiles after the first of a
    split piece: in every kv head the keys at four positions are 20 x one query
    vector of that head group, so that query's row (and about half of the
    others) sees a logit tens to hundreds of units of log2 above the maximum
    of the earlier tiles.  Every row against the fp64 oracle, at the bar for
    rows that one or two keys dominate (their outputs are of order one, where a
    bf16 step is 2^-7 to 2^-5: rel-L2 <= 1e-3 and every element within
    max(2e-3, one bf16 step of the oracle's value)); the aligned rows of the
    oracle return that key's dequantised V."""
    w = synth.Int8KVWorkload("kv_late_spikes", 9, 256, 2048, 32, 8, sub=14)
    x = synth.int8kv_inputs(w)
    G = w.Hq // w.Hkv
    qv = oracle.bf16_value(x["q"])  # [Nq, Hq, 128]
    aligned = []
    for g in range(w.Hkv):
        for i, pos in enumerate((300, 777, 1500, 1900)):
            row, head = 40 * i + 7, g * G + i % G
            assert pos <= w.q_pos0 + row  # visible to the aligned query
            x["k_raw"][g, pos] = (20.0 * qv[row, head]).astype(np.float32)
            aligned.append((row, head, g, pos))
    host, out = run(cuda_lib, w, x)
    rows, heads = np.meshgrid(np.arange(w.Nq), np.arange(w.Hq), indexing="ij")
    ref_b, ref = oracle_bf16(w, host, rows.ravel(), heads.ravel())
    got = bf16_to_f64(out).reshape(-1, 128)
    assert_output_close_rows(got, ref_b, w.name)
    for row, head, g, pos in aligned:
        v_deq = host["v"][g, pos].astype(np.float64) * float(host["v_scale"][g, pos])
        k = row * w.Hq + head
        assert np.abs(ref[k] - v_deq).max() < 1e-6 * max(1.0, np.abs(v_deq).max())


def test_int8kv_quarter_million_token_cache_sampled(cuda_lib):
    """64 queries at the end of a 262,144-token cache (2,048 key tiles, the largest
    split-KV factor): sampled rows against the fp64 oracle."""
    w = synth.Int8KVWorkload("kv_256k", 9, 64, 262144, 8, 2, sub=11)
    x, out = run(cuda_lib, w, synth.int8kv_inputs(w))
    rows = np.array([0, 5, 31, 32, 63, 63, 17])
    heads = np.array([0, 7, 3, 4, 0, 7, 5])
    ref_b, _ = oracle_bf16(w, x, rows, heads)
    got = bf16_to_f64(out[torch.as_tensor(rows).cuda(), torch.as_tensor(heads).cuda()])
    assert_output_close(got, ref_b, w.name)


def test_int8kv_strided_queries_and_output(cuda_lib):
    """q read through a [Nq, Hq, 192] buffer's first 128 channels and the output
    written into a [Nq, Hq + 3, 128] buffer give the same bits as contiguous ones."""
    w = synth.Int8KVWorkload("kv_strided", 9, 45, 400, 8, 2, sub=12)
    _, (q, kc, ks, vc, vs) = both_caches(cuda_lib, synth.int8kv_inputs(w))
    ref = cuda_lib.int8kv_prompt_attn(q, kc, ks, vc, vs, w.q_pos0)
    wide = torch.zeros((w.Nq, w.Hq, 192), dtype=torch.bfloat16, device="cuda")
    wide[:, :, :128] = q
    qv = wide[:, :, :128]
    big = torch.full((w.Nq, w.Hq + 3, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    ov = big[:, 1:w.Hq + 1, :]
    assert not qv.is_contiguous() and not ov.is_contiguous()
    cuda_lib.int8kv_prompt_attn(qv, kc, ks, vc, vs, w.q_pos0, out=ov)
    torch.cuda.synchronize()
    assert torch.equal(ov.view(torch.int16), ref.view(torch.int16))
    assert torch.isnan(big[:, 0].float()).all() and torch.isnan(big[:, w.Hq + 1:].float()).all()


def test_int8kv_chunk_inside_a_longer_cache(cuda_lib):
    """Queries that end before the cache does (q_pos0 + Nq < Nk, e.g. a chunk of a
    prompt whose later tokens are already cached): every row against the fp64
    oracle; the positions no query sees are never read (other codes and NaN scales
    there change no bit); and the result equals the call on the cache cut to the
    visible keys (same images, split and scaling)."""
    w = synth.Int8KVWorkload("kv_mid", 9, 70, 3000, 8, 2, sub=13)
    host, (q, kc, ks, vc, vs) = both_caches(cuda_lib, synth.int8kv_inputs(w))
    p0 = 900
    nvis = p0 + w.Nq  # keys 0..969 are visible to some query, 970..2999 to none
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = cuda_lib.int8kv_prompt_attn(q, kc, ks, vc, vs, p0, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    rows, heads = np.meshgrid(np.arange(w.Nq), np.arange(w.Hq), indexing="ij")
    ref, _ = oracle.int8kv_rows(host["q"], host["k"], host["k_scale"], host["v"], host["v_scale"], p0,
                                rows.ravel(), heads.ravel())
    ref_b = oracle.bf16_value(oracle.f32_to_bf16(ref.astype(np.float32)))
    assert_output_close(bf16_to_f64(out).reshape(-1, 128), ref_b, w.name)

    kc2, vc2, ks2, vs2 = kc.clone(), vc.clone(), ks.clone(), vs.clone()
    g = torch.Generator(device="cuda").manual_seed(3)
    kc2[:, nvis:] = torch.randint(-127, 128, kc2[:, nvis:].shape, generator=g, device="cuda", dtype=torch.int8)
    vc2[:, nvis:] = torch.randint(-127, 128, vc2[:, nvis:].shape, generator=g, device="cuda", dtype=torch.int8)
    ks2.view(torch.int16)[:, nvis:] = 0x7E00  # fp16 NaN
    vs2.view(torch.int16)[:, nvis:] = 0x7E00
    out2 = cuda_lib.int8kv_prompt_attn(q, kc2, ks2, vc2, vs2, p0)
    out3 = cuda_lib.int8kv_prompt_attn(q, kc[:, :nvis], ks[:, :nvis], vc[:, :nvis], vs[:, :nvis], p0)
    torch.cuda.synchronize()
    assert torch.equal(out2.view(torch.int16), out.view(torch.int16))
    assert torch.equal(out3.view(torch.int16), out.view(torch.int16))
