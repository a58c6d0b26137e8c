"""Parity of the int8 KV-cache writer (int8kv_cache_write) with the oracle's
per-token quantiser: codes and fp16 scales bit-exact; rows outside the written
positions untouched; the workload's own cache reproduced from its fp32 rows;
a non-finite scale reported in the status word."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_output_close, bf16_to_f64
from kv_helpers import oracle_cache

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A


def _empty_cache(Hkv, Ncache):
    kc = torch.full((Hkv, Ncache, 128), SENTINEL, dtype=torch.int8, device="cuda")
    vc = torch.full((Hkv, Ncache, 128), SENTINEL, dtype=torch.int8, device="cuda")
    ks = torch.full((Hkv, Ncache), -1.0, dtype=torch.float16, device="cuda")
    vs = torch.full((Hkv, Ncache), -1.0, dtype=torch.float16, device="cuda")
    return kc, vc, ks, vs


def _write(qas, k, v, Ncache, pos0):
    Hkv = k.shape[1]
    kc, vc, ks, vs = _empty_cache(Hkv, Ncache)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qas.int8kv_cache_write(k, v, kc, ks, vc, vs, pos0, status=status)
    torch.cuda.synchronize()
    return kc, vc, ks, vs, int(status.item())


def _check_rows(x_f32, cache, scale, pos0):
    """x_f32 [N, Hkv, 128] source rows as fp32; cache [Hkv, Ncache, 128]."""
    N = x_f32.shape[0]
    want_c, want_s = oracle.cache_quantise(np.ascontiguousarray(x_f32.transpose(1, 0, 2)))
    got_c = cache[:, pos0:pos0 + N].cpu().numpy()
    got_s = scale[:, pos0:pos0 + N].cpu().numpy().view(np.uint16)
    assert np.array_equal(got_c, want_c)
    assert np.array_equal(got_s, want_s)
    # nothing else was written
    c = cache.cpu().numpy()
    assert (c[:, :pos0] == SENTINEL).all() and (c[:, pos0 + N:] == SENTINEL).all()
    s = scale.cpu().numpy()
    assert (s[:, :pos0] == -1).all() and (s[:, pos0 + N:] == -1).all()


@pytest.mark.parametrize("N,Hkv,pos0,Ncache", [(300, 3, 17, 400), (1, 1, 0, 1), (129, 8, 127, 256),
                                              (1, 7, 4, 6), (2, 5, 0, 2), (3, 2, 1, 4)])
def test_cache_write_bf16_matches_oracle(cuda_lib, N, Hkv, pos0, Ncache):
    rng = np.random.default_rng(N * 31 + Hkv)
    x = (rng.standard_normal((2, N, Hkv, 128)) * rng.uniform(0.01, 40, (2, N, Hkv, 1))).astype(np.float32)
    bits = synth.f32_to_bf16_bits(x)
    x16 = synth.bf16_bits_to_f32(bits)            # the bf16 values as fp32 (exact)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    kc, vc, ks, vs, st = _write(cuda_lib, t[0], t[1], Ncache, pos0)
    assert st == 0
    _check_rows(x16[0], kc, ks, pos0)
    _check_rows(x16[1], vc, vs, pos0)


def test_cache_write_f32_strided_and_special_rows(cuda_lib):
    N, Hkv, Ncache, pos0 = 70, 2, 96, 20
    rng = np.random.default_rng(3)
    full = (rng.standard_normal((N, Hkv, 256)) * 3).astype(np.float32)
    full[5, 0, :128] = 0.0                        # zero row: scale 0, codes 0
    full[6, 1, :128] *= 1e-9                       # scale below fp16's range: 0, codes 0
    full[7, 0, :128] *= 1e5                        # large row, scale ~ 3e3
    full[8, 1, :128] = np.float32(2.0**-12)        # fp16-subnormal scale
    src = torch.from_numpy(full).cuda()[:, :, :128]  # token stride 2*256, head stride 256
    v = torch.from_numpy(full[:, :, ::-1].copy()).cuda()[:, :, :128]
    assert src.stride() == v.stride()
    kc, vc, ks, vs, st = _write(cuda_lib, src, v, Ncache, pos0)
    assert st == 0
    _check_rows(full[:, :, :128], kc, ks, pos0)
    _check_rows(full[:, :, ::-1][:, :, :128], vc, vs, pos0)


def test_cache_write_reports_a_non_finite_scale(cuda_lib):
    x = np.ones((4, 1, 128), dtype=np.float32)
    x[2] *= np.float32(1e7)                        # amax / 127 beyond fp16's largest finite value
    t = torch.from_numpy(x).cuda()
    *_, st = _write(cuda_lib, t, t, 8, 0)
    assert st == 7


def test_cache_write_reproduces_the_workload_cache_and_feeds_the_attention(cuda_lib):
    w = synth.int8kv_workload("tiny_kv_q96_k300")
    x = oracle_cache(synth.int8kv_inputs(w))
    raw = synth.int8kv_raw(w)
    # new rows arrive token-major [N, Hkv, 128]; write the whole cache in two appends
    k = torch.from_numpy(np.ascontiguousarray(raw["k"].transpose(1, 0, 2))).cuda()
    v = torch.from_numpy(np.ascontiguousarray(raw["v"].transpose(1, 0, 2))).cuda()
    kc, vc, ks, vs = _empty_cache(w.Hkv, w.Nk)
    cut = 173
    for a, b in ((0, cut), (cut, w.Nk)):
        cuda_lib.int8kv_cache_write(k[a:b], v[a:b], kc, ks, vc, vs, a)
    torch.cuda.synchronize()
    assert np.array_equal(kc.cpu().numpy(), x["k"]) and np.array_equal(vc.cpu().numpy(), x["v"])
    assert np.array_equal(ks.cpu().numpy().view(np.uint16), x["k_scale"].view(np.uint16))
    assert np.array_equal(vs.cpu().numpy().view(np.uint16), x["v_scale"].view(np.uint16))
    q = torch.from_numpy(x["q"].view(np.int16)).view(torch.bfloat16).cuda()
    out = cuda_lib.int8kv_prompt_attn(q, kc, ks, vc, vs, w.q_pos0)
    torch.cuda.synchronize()
    rows, heads = np.meshgrid(np.arange(w.Nq), np.arange(w.Hq), indexing="ij")
    ref, _ = oracle.int8kv_rows(x["q"], x["k"], x["k_scale"], x["v"], x["v_scale"], w.q_pos0, rows.ravel(),
                                heads.ravel())
    ref_b = oracle.bf16_value(oracle.f32_to_bf16(ref.astype(np.float32)))
    assert_output_close(bf16_to_f64(out).reshape(-1, 128), ref_b, w.name)


def test_cache_write_codes_at_rounding_boundaries(cuda_lib):
    """Rows whose quotients x / scale fall exactly on half-integers (ties to even)
    and one fp32 step either side of them, for scales 1, 1/2, 3/8 and an
    fp16-subnormal scale: the codes must equal the oracle's IEEE-division codes."""
    rows = []
    for amax, s in ((127.0, 1.0), (63.5, 0.5), (47.625, 0.375)):
        k = np.arange(-126, 127, dtype=np.float64)
        half = (k + 0.5) * s
        for x in (half, np.nextafter(half.astype(np.float32), np.float32(np.inf)).astype(np.float64),
                  np.nextafter(half.astype(np.float32), np.float32(-np.inf)).astype(np.float64)):
            for start in range(0, x.size, 127):
                r = np.zeros(128)
                seg = x[start:start + 127]
                r[:seg.size] = seg
                r[127] = amax  # fixes the scale to fp16(amax / 127) = s
                rows.append(r)
    # fp16-subnormal scale: amax / 127 below 2^-14
    tiny = np.zeros(128)
    tiny[:5] = [1e-6, -7.5e-7, 3.1e-7, 6e-8, -1e-6]
    rows.append(tiny)
    x = np.asarray(rows, dtype=np.float32)[:, None, :]          # [N, 1, 128] fp32
    t = torch.from_numpy(x).cuda()
    kc, vc, ks, vs, st = _write(cuda_lib, t, t, x.shape[0], 0)
    assert st == 0
    _check_rows(x, kc, ks, 0)
    _check_rows(x, vc, vs, 0)


def test_cache_write_bf16_rows_without_16_byte_alignment(cuda_lib):
    """bf16 rows whose token stride is 4 elements short of a 16-byte multiple take
    the one-warp-per-row kernel; its codes and scales equal the oracle's too."""
    N, Hkv, Ncache, pos0 = 93, 3, 120, 9
    rng = np.random.default_rng(17)
    x = (rng.standard_normal((2, N, Hkv * 128 + 4)) * rng.uniform(0.05, 20, (2, N, 1))).astype(np.float32)
    bits = synth.f32_to_bf16_bits(x)
    x16 = synth.bf16_bits_to_f32(bits)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    k = t[0].as_strided((N, Hkv, 128), (Hkv * 128 + 4, 128, 1))
    v = t[1].as_strided((N, Hkv, 128), (Hkv * 128 + 4, 128, 1))
    assert (k.stride(0) * 2) % 16 == 8
    kc, vc, ks, vs, st = _write(cuda_lib, k, v, Ncache, pos0)
    assert st == 0
    _check_rows(x16[0][:, :Hkv * 128].reshape(N, Hkv, 128), kc, ks, pos0)
    _check_rows(x16[1][:, :Hkv * 128].reshape(N, Hkv, 128), vc, vs, pos0)
