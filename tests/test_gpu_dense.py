"""Parity of the dense CUDA path (sage_quantize_qk, sage_quantize_v,
sage_attn_fwd) against the CPU oracle, element by element.

Codes, scales and the K mean are compared bit-exactly; the bf16 output within
max-abs 2e-3 and rel-L2 1e-3 of the oracle's result rounded to bf16."""

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import assert_output_close, assert_output_close_rows, bf16_dev, bf16_to_f64, bits_to_f64, errors

pytestmark = pytest.mark.gpu

SMALL = [w.name for w in synth.dense_workloads() if w.config in (1, 2)]


def run_dense(qas, q, k, v, bq, bk):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qk = qas.sage_quantize_qk(q, k, bq, bk)
    vq = qas.sage_quantize_v(v)
    out = qas.sage_attn_fwd(qk, vq, bq, bk, status=status)
    torch.cuda.synchronize()
    assert status.item() == 0
    return qk, vq, out


def three_calls(qas, q, k, v, bq, bk, causal=False, return_lse=False):
    """The dense path as its three entry points called in a row on one stream."""
    qk = qas.sage_quantize_qk(q, k, bq, bk)
    vq = qas.sage_quantize_v(v)
    return qas.sage_attn_fwd(qk, vq, bq, bk, causal=causal, return_lse=return_lse)


def check_head(qk, vq, out, b, h, qbits, kbits, vbits, bq, bk, rows=None, tag=""):
    ref = oracle.sage_head(qbits, kbits, vbits, bq, bk, rows=rows)
    assert np.array_equal(qk["k_mean"][b, h].cpu().numpy(), ref["mu"]), f"{tag} k_mean"
    assert np.array_equal(qk["q_scales"][b, h].cpu().numpy(), ref["sq"]), f"{tag} q_scales"
    assert np.array_equal(qk["k_scales"][b, h].cpu().numpy(), ref["sk"]), f"{tag} k_scales"
    assert np.array_equal(qk["q_codes"][b, h].cpu().numpy(), ref["qc"]), f"{tag} q_codes"
    assert np.array_equal(qk["k_codes"][b, h].cpu().numpy(), ref["kc"]), f"{tag} k_codes"
    assert np.array_equal(vq["v_scales"][b, h].cpu().numpy(), ref["sv"]), f"{tag} v_scales"
    assert np.array_equal(vq["v_codes"][b, h].cpu().numpy(), ref["vct"]), f"{tag} v_codes"
    got = bf16_to_f64(out[b, h]) if rows is None else bf16_to_f64(out[b, h][torch.as_tensor(rows).cuda()])
    return assert_output_close(got, bits_to_f64(ref["out_bf16"]), f"{tag} out"), ref


@pytest.mark.parametrize("name", SMALL)
def test_dense_matches_oracle(cuda_lib, name):
    w = synth.dense_workload(name)
    x = synth.dense_inputs(w)
    qk, vq, out = run_dense(cuda_lib, bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"]), w.block, w.block)
    for h in range(w.H):
        check_head(qk, vq, out, 0, h, x["q"][0, h], x["k"][0, h], x["v"][0, h], w.block, w.block, tag=f"{name} h{h}")


@pytest.mark.parametrize("nq,nk,bq,bk", [(100, 300, 128, 64), (300, 100, 64, 128), (1, 513, 64, 64), (257, 1, 128, 128)])
def test_dense_unequal_lengths_and_blocks(cuda_lib, nq, nk, bq, bk):
    w = synth.DenseWorkload(f"mixed_{nq}_{nk}", 7, 2, 3, nq, nk, 64, sub=(nq * 7 + nk) % 97)
    x = synth.dense_inputs(w)
    qk, vq, out = run_dense(cuda_lib, bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"]), bq, bk)
    for b in range(w.B):
        for h in range(w.H):
            check_head(qk, vq, out, b, h, x["q"][b, h], x["k"][b, h], x["v"][b, h], bq, bk, tag=f"b{b}h{h}")


def test_dense_accepts_token_major_strided_views(cuda_lib):
    """[B, N, H, d] storage read through [B, H, N, d] views gives the same bits."""
    w = synth.dense_workload("sweep_b1h4n191")
    x = synth.dense_inputs(w)
    base = [bf16_dev(x[t]) for t in ("q", "k", "v")]
    views = [t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3) for t in base]
    assert not views[0].is_contiguous()
    _, _, o1 = run_dense(cuda_lib, *base, 64, 64)
    out_nhd = torch.empty((1, w.Nq, w.H, 128), dtype=torch.bfloat16, device="cuda").permute(0, 2, 1, 3)
    qk = cuda_lib.sage_quantize_qk(views[0], views[1], 64, 64)
    vq = cuda_lib.sage_quantize_v(views[2])
    o2 = cuda_lib.sage_attn_fwd(qk, vq, 64, 64, out=out_nhd)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_dense_zero_query_and_single_key_closed_forms(cuda_lib):
    """Q = 0 gives the mean of the dequantised V rows; Nk = 1 gives the V row."""
    w = synth.DenseWorkload("closed", 8, 1, 2, 130, 200, 64)
    x = synth.dense_inputs(w)
    q = torch.zeros((1, 2, 130, 128), dtype=torch.bfloat16, device="cuda")
    qk, vq, out = run_dense(cuda_lib, q, bf16_dev(x["k"]), bf16_dev(x["v"]), 64, 64)
    for h in range(2):
        vdeq = oracle.e4m3_value(vq["v_codes"][0, h, :, :200].cpu().numpy()).T * vq["v_scales"][0, h].cpu().numpy()
        got = bf16_to_f64(out[0, h])
        assert np.abs(got - vdeq.mean(axis=0)[None, :]).max() <= 2.0 ** -8 * np.abs(vdeq.mean(axis=0)).max() + 1e-6
    k1 = bf16_dev(x["k"][:, :, :1])
    v1 = bf16_dev(x["v"][:, :, :1])
    qk, vq, out = run_dense(cuda_lib, bf16_dev(x["q"]), k1, v1, 64, 64)
    for h in range(2):
        vrow = oracle.e4m3_value(vq["v_codes"][0, h, :, 0].cpu().numpy()) * vq["v_scales"][0, h].cpu().numpy()
        got = bf16_to_f64(out[0, h])
        assert np.all(np.abs(got - vrow[None, :]) <= 2.0 ** -8 * np.abs(vrow)[None, :] + 1e-30)


def test_dense_full_size_videodit_sampled(cuda_lib):
    """The 37,810-token, 24-head workload on the GPU; two heads checked against the
    oracle (codes and scales in full, 48 sampled output rows each)."""
    w = synth.dense_workload("videodit_b1h24n37810")
    x = synth.dense_inputs(w)
    q, k, v = bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"])
    qk, vq, out = run_dense(cuda_lib, q, k, v, w.block, w.block)
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(7)
    for h in (0, 17):
        rows = np.unique(np.concatenate([rng.integers(0, w.Nq, 44), [0, 127, 128, w.Nq - 1]]))
        (max_abs, rel), ref = check_head(qk, vq, out, 0, h, x["q"][0, h], x["k"][0, h], x["v"][0, h],
                                         w.block, w.block, rows=rows, tag=f"videodit h{h}")
        # distance of the quantized program from unquantised fp64 attention (reported)
        qf = bits_to_f64(x["q"][0, h][rows])
        kf = bits_to_f64(x["k"][0, h])
        vf = bits_to_f64(x["v"][0, h])
        s = qf @ kf.T / np.sqrt(128.0)
        s -= s.max(axis=1, keepdims=True)
        pr = np.exp(s)
        f64 = (pr / pr.sum(axis=1, keepdims=True)) @ vf
        got = bf16_to_f64(out[0, h][torch.as_tensor(rows).cuda()])
        _, rel64 = errors(got, f64)
        print(f"videodit h{h}: vs oracle max-abs {max_abs:.2e} rel-L2 {rel:.2e}; vs fp64 attention rel-L2 {rel64:.3e}")
        assert rel64 < 0.1


def test_dense_full_size_videodit_whole_head(cuda_lib):
    """The 37,810-token, 24-head workload in the launch configuration the
    benchmark times; one whole head (all 37,810 rows and 128 channels, plus
    its codes, scales and K mean) against the oracle at the full bar."""
    w = synth.dense_workload("videodit_b1h24n37810")
    x = synth.dense_inputs(w)
    q, k, v = bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"])
    qk, vq, out = run_dense(cuda_lib, q, k, v, w.block, w.block)
    h = 11
    (max_abs, rel), _ = check_head(qk, vq, out, 0, h, x["q"][0, h], x["k"][0, h], x["v"][0, h],
                                   w.block, w.block, tag=f"videodit whole head {h}")
    print(f"videodit whole head {h}: {w.Nq} rows, vs oracle max-abs {max_abs:.2e} rel-L2 {rel:.2e}")


@pytest.mark.parametrize("name", ["tiny_b1h2n256", "sweep_b1h4n1", "sweep_b1h4n129", "sweep_b1h4n257"])
def test_dense_int32_scores_are_exact(cuda_lib, name):
    """The scores the tensor cores produce (kind::f16 over fp16 images of the
    INT8 codes) equal the exact integer dot products of the oracle's codes."""
    w = synth.dense_workload(name)
    x = synth.dense_inputs(w)
    qk = cuda_lib.sage_quantize_qk(bf16_dev(x["q"]), bf16_dev(x["k"]), w.block, w.block)
    vq = cuda_lib.sage_quantize_v(bf16_dev(x["v"]))
    out, scores = cuda_lib.sage_attn_fwd_scores_dump(qk, vq, w.block, w.block)
    out_ref = cuda_lib.sage_attn_fwd(qk, vq, w.block, w.block)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16))
    for h in range(w.H):
        ref = oracle.sage_head(x["q"][0, h], x["k"][0, h], x["v"][0, h], w.block, w.block, rows=[0])
        exact = ref["qc"].astype(np.int64) @ ref["kc"].astype(np.int64).T
        got = scores[0, h, :w.Nq, :w.Nk].cpu().numpy().astype(np.int64)
        assert np.array_equal(got, exact), f"{name} h{h}"
        assert np.abs(exact).max() <= 128 * 127 * 127


def check_lse(lse_gpu: torch.Tensor, lse_ref: np.ndarray, what: str):
    """Row log-sum-exp: both sides take the same running max m; the sums differ
    only by fp32 summation order and the GPU's ex2, so 1e-5 absolute + relative."""
    got = lse_gpu.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), what
    err = np.abs(got - lse_ref)
    bound = 1e-5 * (1.0 + np.abs(lse_ref))
    assert np.all(err <= bound), f"{what}: lse error {err.max():.3e}"


@pytest.mark.parametrize("nq,nk,bq,bk", [(257, 257, 64, 64), (100, 300, 128, 64), (1, 513, 64, 64),
                                         (600, 600, 128, 128), (383, 700, 64, 128), (129, 129, 128, 64)])
def test_dense_causal_with_lse_matches_oracle(cuda_lib, nq, nk, bq, bk):
    """Causal (query i sees keys j <= i + Nk - Nq) with the row log-sum-exp, against
    the oracle's causal program: codes bit-exact, outputs and lse within the bar."""
    w = synth.DenseWorkload(f"causal_{nq}_{nk}", 9, 1, 3, nq, nk, 64, sub=(nq * 5 + nk) % 89)
    x = synth.dense_inputs(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qk = cuda_lib.sage_quantize_qk(bf16_dev(x["q"]), bf16_dev(x["k"]), bq, bk)
    vq = cuda_lib.sage_quantize_v(bf16_dev(x["v"]))
    out, lse = cuda_lib.sage_attn_fwd(qk, vq, bq, bk, status=status, causal=True, return_lse=True)
    torch.cuda.synchronize()
    assert status.item() == 0
    for h in range(w.H):
        ref = oracle.sage_head(x["q"][0, h], x["k"][0, h], x["v"][0, h], bq, bk, causal=True)
        assert np.array_equal(qk["q_codes"][0, h].cpu().numpy(), ref["qc"])
        assert np.array_equal(qk["k_codes"][0, h].cpu().numpy(), ref["kc"])
        assert_output_close_rows(bf16_to_f64(out[0, h]), bits_to_f64(ref["out_bf16"]), f"causal {nq}x{nk} h{h} out")
        check_lse(lse[0, h], ref["lse"], f"causal {nq}x{nk} h{h}")


@pytest.mark.parametrize("name", ["sweep_b1h4n65", "sweep_b1h4n257", "tiny_b1h2n256"])
def test_dense_lse_non_causal(cuda_lib, name):
    """return_lse without the mask: the same output bits as the plain call, and the
    oracle's log-sum-exp."""
    w = synth.dense_workload(name)
    x = synth.dense_inputs(w)
    qk = cuda_lib.sage_quantize_qk(bf16_dev(x["q"]), bf16_dev(x["k"]), w.block, w.block)
    vq = cuda_lib.sage_quantize_v(bf16_dev(x["v"]))
    out, lse = cuda_lib.sage_attn_fwd(qk, vq, w.block, w.block, return_lse=True)
    plain = cuda_lib.sage_attn_fwd(qk, vq, w.block, w.block)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), plain.view(torch.int16))
    for h in range(w.H):
        ref = oracle.sage_head(x["q"][0, h], x["k"][0, h], x["v"][0, h], w.block, w.block)
        check_lse(lse[0, h], ref["lse"], f"{name} h{h}")


def test_dense_causal_square_first_row_is_first_v_row(cuda_lib):
    """Nq = Nk causal: row 0 sees key 0 alone, so its output is the dequantised
    V row 0 (within one bf16 rounding) and its lse is that key's scaled logit."""
    w = synth.DenseWorkload("causal_row0", 10, 1, 2, 300, 300, 64)
    x = synth.dense_inputs(w)
    qk = cuda_lib.sage_quantize_qk(bf16_dev(x["q"]), bf16_dev(x["k"]), 64, 64)
    vq = cuda_lib.sage_quantize_v(bf16_dev(x["v"]))
    out, lse = cuda_lib.sage_attn_fwd(qk, vq, 64, 64, causal=True, return_lse=True)
    torch.cuda.synchronize()
    for h in range(2):
        vrow = oracle.e4m3_value(vq["v_codes"][0, h, :, 0].cpu().numpy()) * vq["v_scales"][0, h].cpu().numpy()
        got = bf16_to_f64(out[0, h, 0])
        assert np.all(np.abs(got - vrow) <= 2.0 ** -8 * np.abs(vrow) + 1e-30)
        s00 = float(np.dot(qk["q_codes"][0, h, 0].cpu().numpy().astype(np.int64),
                           qk["k_codes"][0, h, 0].cpu().numpy().astype(np.int64)))
        logit = s00 * float(qk["q_scales"][0, h, 0]) * float(qk["k_scales"][0, h, 0]) / np.sqrt(128.0)
        assert abs(float(lse[0, h, 0]) - logit) <= 1e-5 * (1.0 + abs(logit))


def test_dense_causal_full_size_videodit_sampled(cuda_lib):
    """The 37,810-token, 24-head workload with the causal mask; sampled rows of two
    heads (outputs and lse) against the oracle's causal program."""
    w = synth.dense_workload("videodit_b1h24n37810")
    x = synth.dense_inputs(w)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qk = cuda_lib.sage_quantize_qk(bf16_dev(x["q"]), bf16_dev(x["k"]), w.block, w.block)
    vq = cuda_lib.sage_quantize_v(bf16_dev(x["v"]))
    out, lse = cuda_lib.sage_attn_fwd(qk, vq, w.block, w.block, status=status, causal=True, return_lse=True)
    torch.cuda.synchronize()
    assert status.item() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(11)
    for h in (3, 22):
        rows = np.unique(np.concatenate([rng.integers(0, w.Nq, 40), [0, 1, 255, 256, w.Nq - 1]]))
        ref = oracle.sage_head(x["q"][0, h], x["k"][0, h], x["v"][0, h], w.block, w.block, rows=rows, causal=True)
        got = bf16_to_f64(out[0, h][torch.as_tensor(rows).cuda()])
        assert_output_close_rows(got, bits_to_f64(ref["out_bf16"]), f"videodit causal h{h}")
        check_lse(lse[0, h][torch.as_tensor(rows).cuda()], ref["lse"], f"videodit causal h{h}")


@pytest.mark.parametrize("B,H,nq,nk,chunk,causal", [(2, 3, 300, 300, 4, False), (1, 5, 257, 513, 2, True),
                                                    (1, 2, 129, 129, 8, False), (1, 7, 200, 333, 1, False)])
def test_host_pipeline_equals_the_device_path(cuda_lib, B, H, nq, nk, chunk, causal):
    """sage_attention_host (copies of one head group overlapped with the kernels of
    the previous one) gives the same bits as the three device entry points; two
    calls in a row share the workspace."""
    w = synth.DenseWorkload(f"host_{B}_{H}_{nq}_{nk}", 13, B, H, nq, nk, 64, sub=(nq + nk) % 71)
    x = synth.dense_inputs(w)

    def host(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()

    hq, hk, hv = host(x["q"]), host(x["k"]), host(x["v"])
    ref = three_calls(cuda_lib, hq.cuda(), hk.cuda(), hv.cuda(), 64, 64, causal=causal)
    side = torch.cuda.Stream()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(cuda_lib.lib().sage_attention_host_workspace(B, H, nq, nk, chunk), dtype=torch.uint8,
                     device="cuda")
    with torch.cuda.stream(side):
        for rep in range(2):
            out = torch.full((B, H, nq, 128), float("nan"), dtype=torch.bfloat16).pin_memory()
            cuda_lib.sage_attention_host(hq, hk, hv, out, 64, 64, causal=causal, head_chunk=chunk, workspace=ws,
                                         status=status)
            side.synchronize()
            assert torch.equal(out.view(torch.int16), ref.cpu().view(torch.int16)), f"call {rep}"
    assert status.item() == 0


def test_dense_many_heads_and_batches(cuda_lib):
    """B = 3, H = 101 (303 (b, h) problems in the grid's second dimension), ragged
    length: a spread of heads against the oracle."""
    w = synth.DenseWorkload("many_heads", 14, 3, 101, 70, 70, 64, sub=3)
    x = synth.dense_inputs(w)
    qk, vq, out = run_dense(cuda_lib, bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"]), 64, 64)
    for b, h in ((0, 0), (0, 100), (1, 37), (2, 0), (2, 100)):
        check_head(qk, vq, out, b, h, x["q"][b, h], x["k"][b, h], x["v"][b, h], 64, 64, tag=f"b{b}h{h}")


def test_dense_causal_single_query_sees_every_key(cuda_lib):
    """Nq = 1 causal over Nk keys: the one query is the last row, so it sees all keys
    and equals the non-causal result bit for bit."""
    w = synth.DenseWorkload("causal_one_query", 15, 1, 2, 1, 700, 64, sub=1)
    x = synth.dense_inputs(w)
    qk = cuda_lib.sage_quantize_qk(bf16_dev(x["q"]), bf16_dev(x["k"]), 64, 64)
    vq = cuda_lib.sage_quantize_v(bf16_dev(x["v"]))
    o1 = cuda_lib.sage_attn_fwd(qk, vq, 64, 64, causal=True)
    o2 = cuda_lib.sage_attn_fwd(qk, vq, 64, 64)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_dense_long_sequence_sampled(cuda_lib):
    """One head of 200,003 tokens (1,563 key tiles per CTA, 782 CTAs): sampled rows
    against the oracle, codes and scales in full."""
    w = synth.DenseWorkload("long_seq", 16, 1, 1, 200003, 200003, 128, sub=1)
    x = synth.dense_inputs(w)
    qk, vq, out = run_dense(cuda_lib, bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"]), 128, 128)
    rows = np.array([0, 1, 4095, 100000, 131071, 200002])
    check_head(qk, vq, out, 0, 0, x["q"][0, 0], x["k"][0, 0], x["v"][0, 0], 128, 128, rows=rows, tag="long")


@pytest.mark.parametrize("B,H,nq,nk,causal,token_major", [(1, 24, 300, 300, False, False),
                                                          (1, 2, 129, 200, True, False),
                                                          (3, 2, 257, 257, False, False),
                                                          (2, 5, 190, 321, False, True)])
def test_one_call_equals_the_three_entry_points(cuda_lib, B, H, nq, nk, causal, token_major):
    """sage_attention (the three steps in one call, intermediates in its workspace)
    gives the bits of the three entry points in a row, output and lse, also on
    token-major strided views; two calls share the workspace."""
    w = synth.DenseWorkload(f"one_{B}_{H}_{nq}_{nk}", 17, B, H, nq, nk, 64, sub=(nq + 3 * nk) % 89)
    x = synth.dense_inputs(w)
    if token_major:  # [B, N, H, 128] storage viewed as [B, H, N, 128]
        q, k, v = (bf16_dev(np.ascontiguousarray(x[t].transpose(0, 2, 1, 3))).permute(0, 2, 1, 3)
                   for t in ("q", "k", "v"))
    else:
        q, k, v = bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"])
    ref, ref_lse = three_calls(cuda_lib, q, k, v, 64, 128, causal=causal, return_lse=True)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(cuda_lib.lib().sage_attention_workspace(B, H, nq, nk), dtype=torch.uint8, device="cuda")
    for rep in range(2):
        out, lse = cuda_lib.sage_attention(q, k, v, 64, 128, causal=causal, return_lse=True, status=status,
                                           workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"call {rep}"
        assert torch.equal(lse, ref_lse), f"call {rep} lse"
    assert status.item() == 0


def test_dense_last_wave_single_tile_ctas(cuda_lib):
    """One head of 41,372 tokens: 162 pairs of query tiles, so on 152 SMs the last
    10 pairs run as 20 single-tile CTAs, the very last one past Nq (it returns at
    once).  Rows on both sides of the switch and of every converted tile's border
    against the oracle."""
    n = 162 * 256 - 100
    w = synth.DenseWorkload("tail_wave", 18, 1, 1, n, n, 128, sub=2)
    x = synth.dense_inputs(w)
    qk, vq, out = run_dense(cuda_lib, bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"]), 128, 128)
    rows = np.array([0, 38911, 38912, 39039, 39040, 39167, 41215, 41216, 41343, n - 1])
    check_head(qk, vq, out, 0, 0, x["q"][0, 0], x["k"][0, 0], x["v"][0, 0], 128, 128, rows=rows, tag="tail")
