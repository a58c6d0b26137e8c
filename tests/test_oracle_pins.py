"""Pins of the CPU oracle against things other than itself.

Each test ties one oracle function to a library routine, a closed form, brute
force on a tiny input, or an invariant of the quantized program, so that a
dropped term, a wrong index or sign, or a transposed operand in the oracle
fails here.  No expected value comes from the CUDA library.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from kv_helpers import oracle_cache

D = 128
RNG = np.random.default_rng(20261202)


def bf16(x):
    """numbers -> bf16 bits through the library (torch) conversion"""
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16f(h):
    return oracle.bf16_value(h)


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def test_e4m3_decode_matches_library():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_value(codes)
    lib = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(lib)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # S.1111.111 only
    assert np.array_equal(ours[~nan], lib[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9


def _e4m3_probe_values():
    finite = oracle.e4m3_value(np.arange(0, 0x7F, dtype=np.uint8))  # 0 .. 448
    mids = (finite[:-1] + finite[1:]) / 2
    pts = np.concatenate([finite, mids, [464.0, 465.0, 480.0, 1e4, 3e38, 1e-30, 2.0 ** -10]])
    pts32 = pts.astype(np.float32)
    up = np.nextafter(pts32, np.float32(np.inf))
    dn = np.nextafter(pts32, np.float32(0))
    rnd = RNG.uniform(0, 500, 20000).astype(np.float32)
    tiny = (RNG.uniform(0, 2.0 ** -5, 20000)).astype(np.float32)
    allv = np.concatenate([pts32, up, dn, rnd, tiny])
    return np.concatenate([allv, -allv])


def test_e4m3_encode_matches_library_rne_and_saturates():
    x = _e4m3_probe_values()
    codes = oracle.f32_to_e4m3(x)
    ours = oracle.e4m3_value(codes)
    lib_codes = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).double().numpy()
    big = np.abs(x) > 464.0
    # code bits, so the sign of a zero result counts too
    assert np.array_equal(codes[~big], lib_codes[~big])
    assert np.array_equal(ours[~big], lib[~big])
    tiny_neg = (x < 0) & (x > -(2.0 ** -10))
    assert tiny_neg.any() and np.all(codes[tiny_neg] == 0x80)
    assert np.all(np.abs(ours[big]) == 448.0)
    assert np.array_equal(np.sign(ours[big]), np.sign(x[big]))


def test_e4m3_encode_is_nearest_by_brute_force():
    finite = oracle.e4m3_value(np.arange(0, 0x7F, dtype=np.uint8))
    x = _e4m3_probe_values()
    x = x[np.abs(x) <= 448.0]
    got = np.abs(oracle.e4m3_value(oracle.f32_to_e4m3(x)))
    a = np.abs(x.astype(np.float64))
    dist = np.abs(a[:, None] - finite[None, :])
    best = dist.min(axis=1)
    assert np.all(np.abs(a - got) == best)
    # ties go to the code with an even last mantissa bit
    tie = np.sum(dist == best[:, None], axis=1) == 2
    codes = oracle.f32_to_e4m3(x[tie]) & 0x7F
    assert tie.sum() > 100 and np.all(codes % 2 == 0)


def test_bf16_encode_matches_library():
    bits = np.arange(0, 1 << 32, 4093, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 3e38)]
    ours = oracle.f32_to_bf16(x)
    lib = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, lib)


def test_f16_decode_matches_library():
    h = np.arange(1 << 16, dtype=np.uint16)
    ours = oracle.f16_value(h)
    lib = h.view(np.float16).astype(np.float64)
    fin = np.isfinite(lib)
    assert np.array_equal(ours[fin], lib[fin])
    assert np.array_equal(np.isnan(ours), np.isnan(lib))


# ---------------------------------------------------------------------------
# K smoothing mean
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("nk", [1, 5, 255, 256, 257, 700])
def test_k_mean_close_to_exact_mean(nk):
    k = bf16(RNG.normal(0, 1, (nk, D)) + RNG.normal(0, 2, D)[None, :])
    mu = oracle.k_mean(k).astype(np.float64)
    kv = bf16f(k)
    exact = np.array([math.fsum(kv[:, c]) / nk for c in range(D)])
    bound = (nk + 2) * 2.0 ** -24 * np.abs(kv).max(axis=0) + 2.0 ** -24 * np.abs(exact)
    assert np.all(np.abs(mu - exact) <= bound)
    if nk == 1:
        assert np.array_equal(mu, kv[0])


def test_k_mean_constant_column_exact():
    k = bf16(np.full((300, D), 1.5))
    assert np.all(oracle.k_mean(k) == 1.5)


# ---------------------------------------------------------------------------
# Q/K INT8 per-block quantisation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,blk", [(1, 64), (63, 64), (129, 64), (300, 128)])
def test_int8_quant_properties(n, blk):
    q = bf16(RNG.normal(0, 1, (n, D)) * 3)
    codes, scales = oracle.quant_q(q, blk)
    x = bf16f(q)
    assert scales.shape == ((n + blk - 1) // blk,)
    assert np.abs(codes.astype(int)).max() <= 127
    for b in range(scales.size):
        blkx = x[b * blk:(b + 1) * blk]
        blkc = codes[b * blk:(b + 1) * blk].astype(np.float64)
        amax = np.abs(blkx).max()
        # the block's largest magnitude lands on +-127
        i = np.unravel_index(np.argmax(np.abs(blkx)), blkx.shape)
        assert abs(blkc[i]) == 127 and np.sign(blkc[i]) == np.sign(blkx[i])
        assert abs(scales[b] - amax / 127) <= 2.0 ** -23 * amax / 127
        # reconstruction within half a step
        err = np.abs(blkx - blkc * np.float64(scales[b]))
        assert np.all(err <= (0.5 + 1e-4) * scales[b])


def test_int8_quant_power_of_two_and_block_locality():
    q = bf16(RNG.normal(0, 1, (200, D)))
    c0, s0 = oracle.quant_q(q, 64)
    for k in (-3, -1, 2, 3):
        c1, s1 = oracle.quant_q(bf16(bf16f(q) * 2.0 ** k), 64)
        assert np.array_equal(c0, c1)
        assert np.array_equal(s1.astype(np.float64), s0.astype(np.float64) * 2.0 ** k)
    # changing block 1 only changes block 1
    x = bf16f(q).copy()
    x[64:128] *= 5.0
    c2, s2 = oracle.quant_q(bf16(x), 64)
    keep = np.r_[0:64, 128:200]
    assert np.array_equal(c2[keep], c0[keep])
    assert s2[0] == s0[0] and np.array_equal(s2[2:], s0[2:]) and s2[1] != s0[1]


def test_zero_block_gives_zero_scale_and_codes():
    q = np.zeros((70, D), dtype=np.uint16)
    c, s = oracle.quant_q(q, 64)
    assert not c.any() and not s.any()


def test_k_quant_uses_smoothed_values():
    k = bf16(RNG.normal(0, 1, (130, D)) + 40.0)
    mu = oracle.k_mean(k)
    c, s = oracle.quant_k(k, 64, mu)
    # after removing the ~40 mean the step is set by the spread (~4), not by ~44
    assert s.max() < 6.0 / 127
    recon = c.astype(np.float64) * np.repeat(s, 64)[:130, None] + mu[None, :]
    assert np.abs(recon - bf16f(k)).max() <= 0.51 * s.max() + 1e-5


# ---------------------------------------------------------------------------
# V FP8 per-channel quantisation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("nk", [1, 100, 128, 257])
def test_fp8_v_quant_properties(nk):
    v = bf16(RNG.normal(0, 1, (nk, D)) * np.exp(RNG.normal(0, 1, D))[None, :])
    codes, sv = oracle.quant_v(v)
    x = bf16f(v)
    assert codes.shape == (D, oracle.nk_pad(nk))
    assert not codes[:, nk:].any()
    val = oracle.e4m3_value(codes[:, :nk]).T  # [nk, D]
    amax = np.abs(x).max(axis=0)
    assert np.all(np.abs(sv - amax / 448) <= 2.0 ** -23 * amax / 448)
    i = np.argmax(np.abs(x), axis=0)
    assert np.all(np.abs(val[i, np.arange(D)]) == 448.0)
    scaled = x / sv[None, :].astype(np.float64)
    normal = np.abs(scaled) >= 2.0 ** -6
    rel = np.abs(val - scaled) / np.maximum(np.abs(scaled), 1e-30)
    assert np.all(rel[normal] <= 2.0 ** -4 * (1 + 1e-5))
    assert np.all(np.abs(val - scaled)[~normal] <= 2.0 ** -10 * (1 + 1e-5))


def test_fp8_v_quant_power_of_two():
    v = bf16(RNG.normal(0, 1, (150, D)))
    c0, s0 = oracle.quant_v(v)
    c1, s1 = oracle.quant_v(bf16(bf16f(v) * 8.0))
    assert np.array_equal(c0, c1) and np.array_equal(s1, s0 * 8)


# ---------------------------------------------------------------------------
# the attention program
# ---------------------------------------------------------------------------

def softmax_attn_f64(q, k, v, sm):
    s = (q @ k.T) * sm
    s -= s.max(axis=1, keepdims=True)
    p = np.exp(s)
    return (p / p.sum(axis=1, keepdims=True)) @ v


@pytest.mark.parametrize("nq,nk", [(1, 1), (5, 127), (3, 128), (7, 129), (4, 300)])
@pytest.mark.parametrize("tile", [1, 7, 128, 1000])
def test_tile_loop_equals_bruteforce_softmax_when_unquantised(nq, nk, tile):
    q = RNG.normal(0, 1, (nq, D))
    k = RNG.normal(0, 1, (nk, D)) * 1.5
    v = RNG.normal(0, 1, (nk, D))
    sm = 1 / math.sqrt(D)
    ours = oracle.attn_rows_f64(q, k, v, sm, tile)
    ref = softmax_attn_f64(q, k, v, sm)
    assert np.abs(ours - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def quantized_head(q, k, v, blk=64):
    return oracle.sage_head(q, k, v, blk, blk, nthreads=1)


def f64_attention(q, k, v):
    return softmax_attn_f64(bf16f(q), bf16f(k), bf16f(v), 1 / math.sqrt(D))


def rel_l2(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def test_single_key_returns_dequantised_v_row():
    q = bf16(RNG.normal(0, 1, (9, D)))
    k = bf16(RNG.normal(0, 1, (1, D)))
    v = bf16(RNG.normal(0, 1, (1, D)))
    r = quantized_head(q, k, v)
    assert not r["kc"].any() and r["sk"][0] == 0.0
    vdeq = oracle.e4m3_value(r["vct"][:, 0]) * r["sv"].astype(np.float64)
    for row in r["out"]:
        assert np.all(np.abs(row - vdeq) <= 2.0 ** -22 * np.abs(vdeq))


@pytest.mark.parametrize("nk", [1, 64, 127, 129, 257])
def test_zero_query_averages_dequantised_v(nk):
    q = np.zeros((3, D), dtype=np.uint16)
    k = bf16(RNG.normal(0, 1, (nk, D)))
    v = bf16(RNG.normal(0, 1, (nk, D)))
    r = quantized_head(q, k, v)
    vdeq = oracle.e4m3_value(r["vct"][:, :nk]).T * r["sv"][None, :].astype(np.float64)
    mean = vdeq.mean(axis=0)
    for row in r["out"]:
        assert np.all(np.abs(row - mean) <= 1e-6 * np.abs(vdeq).max())


def test_bit_exact_invariants_of_the_quantized_program():
    q = bf16(RNG.normal(0, 1, (70, D)))
    k = bf16(RNG.normal(0, 1, (200, D)) + RNG.normal(0, 2, D)[None, :])
    v = bf16(RNG.normal(0, 1, (200, D)))
    base = quantized_head(q, k, v)["out"].astype(np.float64)
    for e in (-3, -1, 2, 3):
        out_v = quantized_head(q, k, bf16(bf16f(v) * 2.0 ** e))["out"].astype(np.float64)
        assert np.array_equal(out_v, base * 2.0 ** e)
        out_qk = quantized_head(bf16(bf16f(q) * 2.0 ** e), bf16(bf16f(k) * 2.0 ** -e), v)["out"]
        assert np.array_equal(out_qk.astype(np.float64), base)


def test_close_to_fp64_attention_on_the_tiny_workload():
    w = synth.dense_workload("tiny_b1h2n256")
    x = synth.dense_inputs(w)
    for h in range(w.H):
        out = quantized_head(x["q"][0, h], x["k"][0, h], x["v"][0, h], w.block)["out"]
        assert rel_l2(out, f64_attention(x["q"][0, h], x["k"][0, h], x["v"][0, h])) <= 5e-2


def test_per_block_and_per_channel_scales_are_applied_where_they_belong():
    nq, nk = 192, 256
    q = RNG.normal(0, 1, (nq, D)) * np.repeat(2.0 ** np.array([0, 2, -1]), 64)[:, None]
    k = RNG.normal(0, 1, (nk, D)) * np.repeat(2.0 ** np.array([1, -2, 0, 3]), 64)[:, None] / 2
    v = RNG.normal(0, 1, (nk, D)) * (2.0 ** (np.arange(D) % 5))[None, :]
    q, k, v = bf16(q), bf16(k), bf16(v)
    out = quantized_head(q, k, v)["out"]
    assert rel_l2(out, f64_attention(q, k, v)) <= 5e-2


def test_k_smoothing_removes_a_large_channel_offset():
    q = bf16(RNG.normal(0, 1, (64, D)))
    # quarter-integers in [-3.75, 3.75]: K and K + 48 are both exact in bf16
    kr = np.clip(np.round(RNG.normal(0, 1, (256, D)) * 4) / 4, -3.75, 3.75)
    v = bf16(RNG.normal(0, 1, (256, D)))
    k0 = bf16(kr)
    k1 = bf16(kr + 48.0 * RNG.choice([-1.0, 1.0], D)[None, :])
    assert np.array_equal(bf16f(k1) - bf16f(k0), np.round(bf16f(k1) - bf16f(k0)))
    o0 = quantized_head(q, k0, v)["out"]
    o1 = quantized_head(q, k1, v)["out"]
    # softmax ignores a per-channel shift of K; with smoothing so does the program
    # (an unsmoothed step of ~52/127 would put it far off the fp64 result)
    assert rel_l2(o1, f64_attention(q, k1, v)) <= 5e-2
    assert rel_l2(o1, o0) <= 1e-2


# ---------------------------------------------------------------------------
# int8 KV-cache prompt attention (fp64 exact program)
# ---------------------------------------------------------------------------

def _dequant(codes, scales):
    return codes.astype(np.float64) * np.asarray(scales, dtype=np.float64)[..., None]


def test_int8kv_zero_query_is_the_causal_mean_per_group():
    Nq, Nk, Hq, Hkv = 6, 20, 4, 2
    p0 = Nk - Nq
    q = np.zeros((Nq, Hq, D), dtype=np.uint16)
    kc = RNG.integers(-127, 128, (Hkv, Nk, D)).astype(np.int8)
    vc = RNG.integers(-127, 128, (Hkv, Nk, D)).astype(np.int8)
    ks = RNG.uniform(0.01, 0.05, (Hkv, Nk)).astype(np.float16)
    vs = RNG.uniform(0.01, 0.05, (Hkv, Nk)).astype(np.float16)
    rows, heads = np.meshgrid(np.arange(Nq), np.arange(Hq), indexing="ij")
    out, _ = oracle.int8kv_rows(q, kc, ks, vc, vs, p0, rows.ravel(), heads.ravel(), nthreads=1)
    vdeq = _dequant(vc, vs)
    for n, (i, h) in enumerate(zip(rows.ravel(), heads.ravel())):
        g = h // (Hq // Hkv)
        expect = vdeq[g, :p0 + i + 1].mean(axis=0)
        assert np.abs(out[n] - expect).max() <= 1e-12


def test_int8kv_dominant_key_is_selected():
    Nq, Nk, Hq, Hkv = 4, 50, 2, 1
    p0 = Nk - Nq
    kc = np.zeros((Hkv, Nk, D), dtype=np.int8)
    target = 17
    kc[0, target, 3] = 127
    ks = np.full((Hkv, Nk), 0.02, dtype=np.float16)
    vc = RNG.integers(-127, 128, (Hkv, Nk, D)).astype(np.int8)
    vs = RNG.uniform(0.01, 0.05, (Hkv, Nk)).astype(np.float16)
    qv = np.zeros((Nq, Hq, D), dtype=np.float32)
    qv[:, :, 3] = 200.0
    out, _ = oracle.int8kv_rows(bf16(qv), kc, ks, vc, vs, p0, [0, 3], [0, 1], nthreads=1)
    expect = _dequant(vc, vs)[0, target]
    assert np.abs(out - expect[None, :]).max() <= 1e-9 * np.abs(expect).max()


def test_int8kv_scale_exchange_and_group_sharing():
    w = synth.int8kv_workload("tiny_kv_q96_k300")
    x = oracle_cache(synth.int8kv_inputs(w))
    rows = np.array([0, 5, 95, 95, 40])
    heads = np.array([0, 3, 7, 4, 1])
    base, _ = oracle.int8kv_rows(x["q"], x["k"], x["k_scale"], x["v"], x["v_scale"], w.q_pos0,
                                 rows, heads, nthreads=1)
    # q * 4 with key scales / 4: identical logits
    q4 = bf16(bf16f(x["q"]) * 4.0)
    ks4 = (x["k_scale"].astype(np.float32) / 4).astype(np.float16)
    alt, _ = oracle.int8kv_rows(q4, x["k"], ks4, x["v"], x["v_scale"], w.q_pos0, rows, heads,
                                nthreads=1)
    assert np.abs(alt - base).max() <= 1e-12
    # two query heads of one group with the same q row give the same output
    q2 = x["q"].copy()
    q2[:, 1] = q2[:, 0]
    o2, _ = oracle.int8kv_rows(q2, x["k"], x["k_scale"], x["v"], x["v_scale"], w.q_pos0,
                               [10, 10], [0, 1], nthreads=1)
    assert np.array_equal(o2[0], o2[1])


def _int8kv_softmax_f64(q_bits, kc, ks, vc, vs, q_pos0, sm_scale):
    """Test-side restatement of the int8-KV prompt attention ("Strata PR #2092",
    description and the table "... error against FP64"): for query i of head h,
    kv head g = h // (Hq // Hkv), visible keys j <= q_pos0 + i,
    logits sm_scale * ks_j * (q_i . kc_j) in the natural base, softmax weights
    times the dequantised values vs_j * vc_j.  Vectorised numpy in fp64."""
    q = bf16f(q_bits)                                      # [Nq, Hq, 128]
    Nq, Hq, _ = q.shape
    Hkv, Nk, _ = kc.shape
    G = Hq // Hkv
    kd = kc.astype(np.float64)
    vdeq = vc.astype(np.float64) * vs.astype(np.float64)[..., None]
    out = np.empty((Nq, Hq, D))
    for h in range(Hq):
        g = h // G
        logits = sm_scale * ks[g].astype(np.float64)[None, :] * (q[:, h] @ kd[g].T)   # [Nq, Nk]
        visible = np.arange(Nk)[None, :] <= (q_pos0 + np.arange(Nq))[:, None]
        logits = np.where(visible, logits, -np.inf)
        e = np.exp(logits - logits.max(axis=1, keepdims=True))
        out[:, h] = (e @ vdeq[g]) / e.sum(axis=1, keepdims=True)
    return out


@pytest.mark.parametrize("Hq,Hkv,Nq,Nk", [(3, 3, 7, 301), (8, 2, 5, 190)])
def test_int8kv_equals_a_numpy_fp64_softmax_at_ordinary_logits(Hq, Hkv, Nq, Nk):
    # logits of order 1-10 (not the one-hot or uniform limits), a ragged cache
    # length and a causal window that moves with the query: a wrong logit scale,
    # exp2 in place of exp, an off-by-one window or a wrong group map all fail
    rng = np.random.default_rng(Hq * 1000 + Nk)
    q_pos0 = Nk - Nq - 3
    q = bf16(rng.normal(0, 2.0, (Nq, Hq, D)))
    kc = rng.integers(-127, 128, (Hkv, Nk, D)).astype(np.int8)
    vc = rng.integers(-127, 128, (Hkv, Nk, D)).astype(np.int8)
    ks = rng.uniform(0.002, 0.03, (Hkv, Nk)).astype(np.float16)
    vs = rng.uniform(0.005, 0.05, (Hkv, Nk)).astype(np.float16)
    sm = 1.0 / math.sqrt(128.0)
    want = _int8kv_softmax_f64(q, kc, ks, vc, vs, q_pos0, sm)
    logits = sm * ks[0].astype(np.float64) * (bf16f(q)[:, 0] @ kc[0].astype(np.float64).T)
    assert 1.0 < np.abs(logits).max() < 30.0          # ordinary logits, not a limit case
    rows, heads = np.meshgrid(np.arange(Nq), np.arange(Hq), indexing="ij")
    got, _ = oracle.int8kv_rows(q, kc, ks, vc, vs, q_pos0, rows.ravel(), heads.ravel(), nthreads=1)
    want = want.reshape(-1, D)
    assert np.abs(got - want).max() <= 1e-12 * max(1.0, np.abs(want).max())


def _row_logits_f32(qc_row, sq, kc, sk, bk, C):
    """s_j = fl(S_j * fl(fl(sq * sk_blk(j)) * C)) rebuilt from codes and scales."""
    S = kc.astype(np.int64) @ qc_row.astype(np.int64)
    t = (np.float32(sq) * sk[np.arange(kc.shape[0]) // bk]).astype(np.float32) * np.float32(C)
    return (S.astype(np.float32) * t.astype(np.float32)).astype(np.float32)


def test_dense_denominator_sums_fp32_p_before_the_fp8_conversion():
    # Reading A8 ("Sage2 SM89 Temporal Pair Experiment", "Candidate": the order
    # accumulate_d -> RS_32_to_8): the row sum l adds the fp32 p, not the FP8
    # P/448.  Logits spread over ~25 binades put 448 p into every E4M3 binade,
    # the subnormals and below, where the two sums differ by percents; the lse
    # of the row exposes l directly.
    rng = np.random.default_rng(88)
    nq, nk, bk = 6, 333, 64
    qc = rng.integers(-127, 128, (nq, D)).astype(np.int8)
    kc = rng.integers(-127, 128, (nk, D)).astype(np.int8)
    sq = rng.uniform(0.5, 1.0, (nq + 63) // 64).astype(np.float32)
    sk = rng.uniform(0.5, 1.0, (nk + bk - 1) // bk).astype(np.float32) * np.float32(8.0 / 60000.0 / 0.0884)
    sk = sk.astype(np.float32)
    vct = np.zeros((D, oracle.nk_pad(nk)), dtype=np.uint8)
    vct[:, :nk] = oracle.f32_to_e4m3(rng.uniform(-400, 400, (D, nk)).astype(np.float32))
    sv = np.full(D, 1.0, dtype=np.float32)
    _, _, _, lse = oracle.sage_attn_rows(qc, sq, 64, kc, sk, bk, vct, sv, nq, nk, with_lse=True)
    C = np.float32(oracle.SM_SCALE_D128) * np.float32(1.4426950408889634)
    spread = []
    for i in range(nq):
        s = _row_logits_f32(qc[i], sq[i // 64], kc, sk, bk, C).astype(np.float64)
        M = s.max()
        want = math.log(2.0) * (M + math.log2(np.exp2(s - M).sum()))
        assert abs(lse[i] - want) <= 2e-6 * max(1.0, abs(want)), (i, lse[i], want)
        # the FP8 sum would be far off: the pin separates the two readings
        p = np.exp2(s - M).astype(np.float32)
        p8 = oracle.e4m3_value(oracle.f32_to_e4m3((np.float32(448.0) * p).astype(np.float32))) / 448.0
        spread.append(abs(math.log(p8.sum()) - math.log(p.astype(np.float64).sum())))
        assert (s.max() - s.min()) > 20.0
    assert max(spread) > 1e-3


# ---------------------------------------------------------------------------
# fp16 encoder and the per-token int8 KV cache quantiser
# ("Strata PR #2092": int8 K/V cache with per-token fp16 scales)
# ---------------------------------------------------------------------------

def test_f16_encode_matches_library_rne():
    rng = np.random.default_rng(21)
    mant = rng.integers(0, 1 << 23, 400_000).astype(np.uint32)
    expo = rng.integers(127 - 30, 127 + 17, 400_000).astype(np.uint32)
    sign = rng.integers(0, 2, 400_000).astype(np.uint32) << 31
    x = (sign | (expo << 23) | mant).view(np.float32)
    # exact halfway points between fp16 neighbours (ties), across the subnormal range too
    h = np.arange(0, 0x7BFF, 7, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    ties = ((lo + hi) / 2).astype(np.float32)
    edges = np.array([0.0, -0.0, 65504.0, 65519.996, 65520.0, 1e9, 2.0**-24, 2.0**-25, 2.0**-25 * 1.0001,
                      2.0**-14, 2.0**-14 * (1 - 2.0**-11), np.inf, -np.inf], dtype=np.float32)
    allx = np.concatenate([x, ties, -ties, edges])
    with np.errstate(over="ignore"):
        want = allx.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.f32_to_f16(allx), want)


def test_int8_code_rounds_half_to_even_and_saturates():
    k = np.arange(-140, 141, dtype=np.float64)
    half = (k + 0.5).astype(np.float32)
    x = np.concatenate([half, np.nextafter(half, np.float32(np.inf)), np.nextafter(half, np.float32(-np.inf)),
                        np.array([0.0, -0.0, 1e9, -1e9, 126.5, 127.5, -127.5, 2.0**-30], dtype=np.float32),
                        np.random.default_rng(4).uniform(-200, 200, 10000).astype(np.float32)])
    want = np.clip(np.rint(x.astype(np.float64)), -127, 127).astype(np.int8)  # numpy rint: ties to even
    assert np.array_equal(oracle.f32_to_i8(x), want)
    assert oracle.f32_to_i8(np.float32([2.5, 3.5, -2.5]))[:3].tolist() == [2, 4, -2]


def _cache_rows(seed, n, gain=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((n, 128)) * gain).astype(np.float32)


def test_cache_quantise_properties():
    x = _cache_rows(5, 3000, gain=np.float32(3.0))
    x[7] *= 1e-4                      # small row (normal fp16 scale)
    x[8] *= 1e-9                      # scale below the fp16 subnormal range -> 0
    codes, sc = oracle.cache_quantise(x)
    s = oracle.f16_value(sc)
    amax = np.abs(x.astype(np.float64)).max(axis=1)
    # the scale is fp16(fl32(amax / 127))
    assert np.array_equal(sc, oracle.f32_to_f16((x.__abs__().max(axis=1) / np.float32(127.0)).astype(np.float32)))
    assert np.all(np.abs(codes.astype(np.int32)) <= 127)
    live = s > 0
    # the largest element of a row encodes to +-127 (fp16 rounding moves the
    # scale by at most 2^-11 relative, far less than half a code)
    arg = np.abs(x).argmax(axis=1)
    assert np.all(np.abs(codes[np.arange(len(x)), arg][live].astype(np.int32)) == 127)
    # reconstruction within half a code (plus the scale's own rounding at the top)
    err = np.abs(x.astype(np.float64) - codes.astype(np.float64) * s[:, None])
    bound = 0.5 * s[:, None] * (1 + 2.0**-20) + 127 * s[:, None] * 2.0**-11
    assert np.all(err[live] <= bound[live])
    # a scale that rounds to 0 gives zero codes
    assert sc[8] == 0 and not codes[8].any()


def _cache_quantise_numpy(x32):
    """Independent numpy restatement of the per-token cache recipe: fp32
    division amax / 127, rounded to fp16; codes rint(fl(x / scale)) (ties to
    even) clamped to +-127; zero codes where the fp16 scale is 0."""
    amax = np.max(np.abs(x32), axis=-1)
    scale16 = (amax / np.float32(127.0)).astype(np.float32).astype(np.float16)
    s32 = scale16.astype(np.float32)
    safe = np.where(s32 > 0, s32, np.float32(1.0))
    quot = (x32 / safe[..., None]).astype(np.float32)
    codes = np.clip(np.where(s32[..., None] > 0, np.rint(quot), 0.0), -127, 127).astype(np.int8)
    return codes, scale16.view(np.uint16)


def test_cache_quantise_agrees_with_a_numpy_restatement_including_exact_ties():
    x = _cache_rows(7, 2000, gain=np.float32(0.7))
    _, s16 = _cache_quantise_numpy(x)
    s = s16.view(np.float16).astype(np.float32)
    rng = np.random.default_rng(70)
    # put quotients exactly on half-integers (k + 1/2) * scale, and one fp32 step
    # to either side of them, below the row's amax so the scale stays the same
    amax = np.abs(x).max(axis=1)
    for r in range(0, 2000, 2):
        for c in rng.choice(np.arange(128), 12, replace=False):
            k = int(rng.integers(-126, 126))
            v = np.float32((k + 0.5) * float(s[r]))
            if abs(v) >= amax[r] or abs(x[r, c]) == amax[r]:
                continue
            x[r, c] = [v, np.nextafter(v, np.float32(np.inf)), np.nextafter(v, np.float32(-np.inf))][c % 3]
    codes, sc = oracle.cache_quantise(x)
    c2, s2 = _cache_quantise_numpy(x)
    assert np.array_equal(sc, s2)
    assert np.array_equal(codes, c2)
    # ties really were hit, and some went to the even neighbour below
    quot = x / s[:, None]
    ties = np.abs(quot - np.floor(quot) - 0.5) == 0
    assert ties.sum() > 1000
    assert np.any(np.abs(codes[ties].astype(np.float32)) < np.abs(quot[ties]))


def test_cache_quantise_zero_row_and_power_of_two():
    x = _cache_rows(6, 64)
    x[3] = 0.0
    codes, sc = oracle.cache_quantise(x)
    assert sc[3] == 0 and not codes[3].any()
    for k in (-3, 2, 5):
        c2, s2 = oracle.cache_quantise(x * np.float32(2.0**k))
        assert np.array_equal(c2, codes)
        np.testing.assert_array_equal(oracle.f16_value(s2), oracle.f16_value(sc) * 2.0**k)


# ---------------------------------------------------------------------------
# causal window and log-sum-exp of the dense program
# ---------------------------------------------------------------------------

def _bruteforce_causal(q, k, v, sm_scale, off):
    """fp64 causal softmax(q k^T * sm_scale) v with query i seeing keys j <= i + off; and lse."""
    s = (q @ k.T) * sm_scale
    n_q, n_k = s.shape
    mask = np.arange(n_k)[None, :] > (np.arange(n_q)[:, None] + off)
    s = np.where(mask, -np.inf, s)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return (e @ v) / e.sum(axis=1, keepdims=True), (m[:, 0] + np.log(e.sum(axis=1)))


@pytest.mark.parametrize("nq,nk,tile", [(200, 200, 128), (200, 200, 32), (70, 300, 64), (1, 129, 128)])
def test_causal_tile_loop_and_lse_equal_bruteforce_when_unquantised(nq, nk, tile):
    rng = np.random.default_rng(nq * 7 + nk)
    q, k, v = (rng.standard_normal((n, 128)) for n in (nq, nk, nk))
    sm = 1.0 / math.sqrt(128.0)
    out, lse = oracle.attn_rows_f64(q, k, v, sm_scale=sm, tile=tile, causal=True, with_lse=True)
    want, want_lse = _bruteforce_causal(q, k, v, sm, nk - nq)
    np.testing.assert_allclose(out, want, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(lse, want_lse, rtol=1e-12, atol=1e-12)
    # non-causal lse as well
    _, lse_nc = oracle.attn_rows_f64(q, k, v, sm_scale=sm, tile=tile, causal=False, with_lse=True)
    _, want_nc = _bruteforce_causal(q, k, v, sm, nk)
    np.testing.assert_allclose(lse_nc, want_nc, rtol=1e-12, atol=1e-12)


def _quantised_head(seed, nq, nk, blk=64):
    w = synth.DenseWorkload("pin", 9, 1, 1, nq, nk, blk, sub=seed)
    x = synth.dense_inputs(w)
    q, k, v = x["q"][0, 0], x["k"][0, 0], x["v"][0, 0]
    mu = oracle.k_mean(k)
    qc, sq = oracle.quant_q(q, blk)
    kc, sk = oracle.quant_k(k, blk, mu)
    vct, sv = oracle.quant_v(v)
    return qc, sq, kc, sk, vct, sv


@pytest.mark.parametrize("nq,nk", [(150, 150), (40, 230)])
def test_causal_row_equals_the_program_on_its_visible_prefix(nq, nk):
    # the masked program on the full key set and the unmasked program on the
    # row's visible keys only are the same computation: bit-identical
    qc, sq, kc, sk, vct, sv = _quantised_head(11, nq, nk)
    rows = np.array([r for r in (0, 1, 63, 64, 65, nq - 1) if r < nq])
    out, outb, _, lse = oracle.sage_attn_rows(qc, sq, 64, kc, sk, 64, vct, sv, nq, nk, rows=rows, causal=True,
                                              with_lse=True)
    for r_i, i in enumerate(rows):
        nvis = i + (nk - nq) + 1
        o2, b2, _, l2 = oracle.sage_attn_rows(qc, sq, 64, kc[:nvis], sk, 64, np.ascontiguousarray(vct[:, :nvis]),
                                              sv, nq, nvis, rows=np.array([i]), with_lse=True)
        assert np.array_equal(out[r_i], o2[0]) and np.array_equal(outb[r_i], b2[0])
        assert lse[r_i] == l2[0]


def test_causal_first_row_is_the_dequantised_first_v_row_and_its_lse():
    nq = nk = 90
    qc, sq, kc, sk, vct, sv = _quantised_head(12, nq, nk)
    out, outb, _, lse = oracle.sage_attn_rows(qc, sq, 64, kc, sk, 64, vct, sv, nq, nk, rows=np.array([0]),
                                              causal=True, with_lse=True)
    # a single visible key: p = 1, P = 448, out = V_0 * sv
    v0 = oracle.e4m3_value(vct[:, 0]) * sv.astype(np.float64)
    np.testing.assert_allclose(out[0], v0, rtol=2.0**-22, atol=0)
    # lse = ln 2 * s_00 with s_00 = fl(S_00 * fl(fl(sq*sk) * C))
    C = np.float32(oracle.SM_SCALE_D128 * np.float32(1.4426950408889634))
    t = np.float32(np.float32(sq[0] * sk[0]) * C)
    s00 = np.float32(np.float32(int(qc[0].astype(np.int64) @ kc[0].astype(np.int64))) * t)
    assert lse[0] == pytest.approx(math.log(2.0) * float(s00), rel=1e-15)


def _golden(name):
    vals = {}
    for line in open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", name)):
        line = line.split("|")[0].strip()
        if line and not line.startswith("#"):
            key, val = (s.strip() for s in line.split("="))
            vals[key] = int(val)
    return vals


def test_workloads_match_the_sizes_the_pages_print():
    """The synthetic stand-ins have the sizes the pages measure on (golden fixture
    with citations): the 37,810-token dense self-attention and the int8-KV prompt
    chunks 32K x 1024 and 64K x 512."""
    g = _golden("page_workloads.txt")
    w = synth.dense_workload("videodit_b1h24n37810")
    assert w.Nq == w.Nk == g["dense.tokens"]
    a = synth.int8kv_workload("prompt32k_q1024")
    assert (a.Nk, a.Nq) == (g["int8kv.context_32k"], g["int8kv.queries_32k"])
    b = synth.int8kv_workload("prompt64k_q512_outliers")
    assert (b.Nk, b.Nq) == (g["int8kv.context_64k"], g["int8kv.queries_64k"])
