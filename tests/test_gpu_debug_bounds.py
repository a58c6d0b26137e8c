"""Every kernel of the library run through the bounds-checking debug build
(the stand-in for a memory sanitizer, which this GPU pool does not offer):
small and ragged shapes of each entry point must record no out-of-bounds
site and give outputs bit for bit equal to the normal build's."""

import numpy as np
import pytest
import torch

import quantized_attention_sage_gb300 as qas
import synth
from gpu_helpers import bf16_dev
from kv_helpers import device_cache

pytestmark = pytest.mark.gpu


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16).cuda()


def _f32(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).cuda()


def _dense_cases():
    cases = []
    for i, (B, H, nq, nk, bq, bk, causal) in enumerate([
            (1, 2, 1, 1, 64, 64, False), (1, 2, 65, 129, 64, 128, False), (2, 3, 191, 257, 128, 64, True),
            (1, 1, 300, 1000, 128, 128, False), (1, 2, 384, 384, 64, 64, True)]):
        q, k, v = _bf16((B, H, nq, 128), 10 * i + 1), _bf16((B, H, nk, 128), 10 * i + 2), _bf16((B, H, nk, 128), 10 * i + 3)
        cases.append((f"dense{i}", q, k, v, bq, bk, causal))
    return cases


def _run_all(cases, kv):
    """Every entry point on every case; returns a flat dict of output tensors (cloned)."""
    res = {}
    for name, q, k, v, bq, bk, causal in cases:
        out, lse = qas.sage_attention(q, k, v, bq, bk, causal=causal, return_lse=True)
        res[name + "/one_call"], res[name + "/lse"] = out.clone(), lse.clone()
        qk = qas.sage_quantize_qk(q, k, bq, bk)
        vq = qas.sage_quantize_v(v)
        for key, t in list(qk.items()) + list(vq.items()):
            res[f"{name}/{key}"] = t.clone()
        res[name + "/three_calls"] = qas.sage_attn_fwd(qk, vq, bq, bk, causal=causal).clone()
        for images in (False, True):
            prep = qas.sage_quantize_qkv(q, k, v, bq, bk, images=images)
            for key, t in prep.items():
                res[f"{name}/qkv{int(images)}/{key}"] = t.clone()
            if images:
                res[name + "/f16"] = qas.sage_attn_fwd_f16(prep, bq, bk, causal=causal).clone()
    # token-major views of one case
    B, H, N = 1, 3, 200
    qt, kt, vt = (_bf16((B, N, H, 128), 90 + j).permute(0, 2, 1, 3) for j in range(3))
    res["token_major"] = qas.sage_attention(qt, kt, vt, 64, 64).clone()
    # int8 KV cache: writer (bf16 and fp32 rows) and the prompt attention
    for name, Nq, Nk, Hq, Hkv, f32 in kv:
        mk = _f32 if f32 else _bf16
        k, v = mk((Nk, Hkv, 128), 200 + Nk), mk((Nk, Hkv, 128), 300 + Nk)
        kc = torch.empty((Hkv, Nk, 128), dtype=torch.int8, device="cuda")
        vc = torch.empty_like(kc)
        ks = torch.empty((Hkv, Nk), dtype=torch.float16, device="cuda")
        vs = torch.empty_like(ks)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        qas.int8kv_cache_write(k, v, kc, ks, vc, vs, 0, status=status)
        qry = _bf16((Nq, Hq, 128), 400 + Nq)
        st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
        o = qas.int8kv_prompt_attn(qry, kc, ks, vc, vs, Nk - Nq, status=st2)
        torch.cuda.synchronize()
        assert status.item() == 0 and st2.item() == 0, name
        for key, t in (("kc", kc), ("ks", ks), ("vc", vc), ("vs", vs), ("out", o)):
            res[f"{name}/{key}"] = t.clone()
    x = _f32((4096,), 77, 100.0)
    for key, t in qas.sage_conversion_check(x).items():
        res["conv/" + key] = t.clone()
    torch.cuda.synchronize()
    return res


KV = [("kv_tiny", 96, 300, 8, 2, False), ("kv_gqa3", 33, 1000, 6, 2, True), ("kv_one", 1, 129, 4, 4, False),
      ("kv_split", 256, 4096, 32, 8, False)]


def test_every_kernel_in_bounds_and_equal_to_the_normal_build(cuda_lib):
    cases = _dense_cases()
    qas.use_debug_bounds(False)
    normal = _run_all(cases, KV)
    assert qas.debug_bounds_site() == 0
    try:
        qas.use_debug_bounds(True)
        assert qas.lib().sage_debug_bounds_enabled() == 1
        assert qas.debug_bounds_site() == 0  # nothing left over
        debug = _run_all(cases, KV)
        site = qas.debug_bounds_site()
        assert site == 0, f"out-of-bounds access recorded at file {site // 100000}, line {site % 100000}"
    finally:
        qas.use_debug_bounds(False)
    assert qas.lib().sage_debug_bounds_enabled() == 0
    assert normal.keys() == debug.keys()
    as_int = {torch.float32: torch.int32, torch.bfloat16: torch.int16, torch.float16: torch.int16}
    for key in normal:
        a, b = normal[key], debug[key]
        assert a.dtype == b.dtype and a.shape == b.shape, key
        if a.dtype in as_int:
            a, b = a.contiguous().view(as_int[a.dtype]), b.contiguous().view(as_int[b.dtype])
        assert torch.equal(a, b), key


def test_full_size_workloads_in_bounds_and_equal_to_the_normal_build(cuda_lib):
    """The benchmark's own launches through the bounds-checking build: the
    37,810-token, 24-head dense path in one call (fused preparation, then the
    attention over the images, last-wave single-tile CTAs included) and both
    int8-KV prompt chunks (split-KV): no out-of-bounds site, same bits."""
    w = synth.dense_workload("videodit_b1h24n37810")
    x = synth.dense_inputs(w)
    q, k, v = bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"])
    del x
    caches = [(wk, device_cache(qas, synth.int8kv_inputs(wk)))
              for wk in (synth.int8kv_workload("prompt32k_q1024"), synth.int8kv_workload("prompt64k_q512_outliers"))]

    def run_all():
        res = {"dense": qas.sage_attention(q, k, v, w.block, w.block).clone()}
        for wk, (qq, kc, ks, vc, vs) in caches:
            st = torch.zeros(1, dtype=torch.int32, device="cuda")
            res[wk.name] = qas.int8kv_prompt_attn(qq, kc, ks, vc, vs, wk.q_pos0, status=st).clone()
            torch.cuda.synchronize()
            assert st.item() == 0, wk.name
        return res

    qas.use_debug_bounds(False)
    normal = run_all()
    try:
        qas.use_debug_bounds(True)
        assert qas.debug_bounds_site() == 0
        debug = run_all()
        site = qas.debug_bounds_site()
        assert site == 0, f"out-of-bounds access recorded at file {site // 100000}, line {site % 100000}"
    finally:
        qas.use_debug_bounds(False)
    for key in normal:
        assert torch.equal(normal[key].view(torch.int16), debug[key].view(torch.int16)), key
    assert np.isfinite(normal["dense"].float().cpu().numpy()).all()
