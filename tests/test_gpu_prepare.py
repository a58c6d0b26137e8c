"""The fused preparation (sage_quantize_qkv: one reduction pass over K and V,
one finalisation, one encoding pass over Q, K and V) against the separate
quantizers, and the attention over its fp16 images (sage_attn_fwd_f16)
against the attention over int8 codes: every code, scale and mean must be the
same bits, every fp16 image the exact value of its code, every output the
same bits.  The separate quantizers are checked against the oracle elsewhere;
one case here goes to the oracle directly as well."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_output_close, bf16_dev, bf16_to_f64, bits_to_f64

pytestmark = pytest.mark.gpu

CASES = [("tiny_b1h2n256", None), ("sweep_b1h4n1", None), ("sweep_b1h4n65", None), ("sweep_b1h4n257", None),
         ("mixed", (3, 2, 300, 1031, 64, 128)), ("mixed2", (1, 5, 700, 129, 128, 64))]


def _inputs(name, spec):
    if spec is None:
        w = synth.dense_workload(name)
        return w, w.block, w.block
    B, H, nq, nk, bq, bk = spec
    return synth.DenseWorkload(name, 13, B, H, nq, nk, bq, sub=H), bq, bk


def _separate(qas, q, k, v, bq, bk):
    qk = qas.sage_quantize_qk(q, k, bq, bk)
    vq = qas.sage_quantize_v(v)
    return qk, vq


@pytest.mark.parametrize("name,spec", CASES, ids=[c[0] for c in CASES])
def test_fused_preparation_equals_the_separate_quantizers(cuda_lib, name, spec):
    w, bq, bk = _inputs(name, spec)
    x = synth.dense_inputs(w)
    q, k, v = bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"])
    qk, vq = _separate(cuda_lib, q, k, v, bq, bk)
    for images in (False, True):
        p = cuda_lib.sage_quantize_qkv(q, k, v, bq, bk, images=images)
        torch.cuda.synchronize()
        for key in ("q_scales", "k_scales", "k_mean"):
            assert torch.equal(p[key], qk[key]), f"{name} {key}"
        for key in ("v_codes", "v_scales"):
            assert torch.equal(p[key], vq[key]), f"{name} {key}"
        for key in ("q_codes", "k_codes"):
            if images:
                # the exact fp16 value of every code (|code| <= 127)
                assert torch.equal(p[key].float(), qk[key].float()), f"{name} {key} image"
            else:
                assert torch.equal(p[key], qk[key]), f"{name} {key}"


def test_fused_preparation_on_token_major_strided_views(cuda_lib):
    w = synth.DenseWorkload("strided_prep", 13, 2, 3, 333, 333, 64, sub=7)
    x = synth.dense_inputs(w)
    # [B, N, H, 128] storage viewed as [B, H, N, 128]
    q, k, v = (bf16_dev(np.ascontiguousarray(x[t].transpose(0, 2, 1, 3))).permute(0, 2, 1, 3) for t in "qkv")
    qk, vq = _separate(cuda_lib, q.contiguous(), k.contiguous(), v.contiguous(), 64, 64)
    p = cuda_lib.sage_quantize_qkv(q, k, v, 64, 64, images=True)
    torch.cuda.synchronize()
    assert torch.equal(p["q_codes"].float(), qk["q_codes"].float())
    assert torch.equal(p["k_codes"].float(), qk["k_codes"].float())
    assert torch.equal(p["v_codes"], vq["v_codes"]) and torch.equal(p["k_mean"], qk["k_mean"])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("name,spec", CASES[2:], ids=[c[0] for c in CASES[2:]])
def test_attention_over_images_equals_attention_over_codes(cuda_lib, name, spec, causal):
    w, bq, bk = _inputs(name, spec)
    if causal and w.Nq > w.Nk:
        pytest.skip("causal needs Nq <= Nk")
    x = synth.dense_inputs(w)
    q, k, v = bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"])
    qk, vq = _separate(cuda_lib, q, k, v, bq, bk)
    ref, ref_lse = cuda_lib.sage_attn_fwd(qk, vq, bq, bk, causal=causal, return_lse=True)
    p = cuda_lib.sage_quantize_qkv(q, k, v, bq, bk, images=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = cuda_lib.sage_attn_fwd_f16(p, bq, bk, causal=causal, return_lse=True, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(lse, ref_lse)


def test_fused_path_full_size_videodit_matches_the_oracle_on_a_head(cuda_lib):
    """The 37,810-token, 24-head workload through the fused preparation and the
    attention over images (the benchmark's launch configuration); head 5's
    codes, scales and mean against the oracle in full, 64 sampled rows of its
    output at the full bar."""
    w = synth.dense_workload("videodit_b1h24n37810")
    x = synth.dense_inputs(w)
    q, k, v = bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"])
    p = cuda_lib.sage_quantize_qkv(q, k, v, w.block, w.block, images=True)
    out = cuda_lib.sage_attn_fwd_f16(p, w.block, w.block)
    torch.cuda.synchronize()
    h = 5
    rows = np.unique(np.random.default_rng(3).integers(0, w.Nq, 64))
    ref = oracle.sage_head(x["q"][0, h], x["k"][0, h], x["v"][0, h], w.block, w.block, rows=rows)
    assert np.array_equal(p["k_mean"][0, h].cpu().numpy(), ref["mu"])
    assert np.array_equal(p["q_scales"][0, h].cpu().numpy(), ref["sq"])
    assert np.array_equal(p["k_scales"][0, h].cpu().numpy(), ref["sk"])
    assert np.array_equal(p["q_codes"][0, h].float().cpu().numpy(), ref["qc"].astype(np.float32))
    assert np.array_equal(p["k_codes"][0, h].float().cpu().numpy(), ref["kc"].astype(np.float32))
    assert np.array_equal(p["v_codes"][0, h].cpu().numpy(), ref["vct"])
    assert np.array_equal(p["v_scales"][0, h].cpu().numpy(), ref["sv"])
    got = bf16_to_f64(out[0, h][torch.as_tensor(rows).cuda()])
    assert_output_close(got, bits_to_f64(ref["out_bf16"]), "videodit fused head 5")
