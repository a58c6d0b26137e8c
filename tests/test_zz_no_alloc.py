"""sage_quantize_qk_noalloc: the allocation-free variant of sage_quantize_qk.

Some callers cannot allocate device memory (an engine that reserves all of
HBM at start-up, a plug-in whose host framework owns every allocation, a
latency-bound loop where cudaMalloc could synchronise the device).  This
entry point keeps its scratch in a fixed array inside the library; the
caller passes only inputs and outputs.  Its results must equal those of
sage_quantize_qk bit for bit (the codes, scales and K mean are exact), also
on a second call that reuses the shared scratch with a different problem.
"""

import ctypes as C

import numpy as np
import pytest
import torch

import synth
from gpu_helpers import bf16_dev
from quantized_attention_sage_gb300 import Strides

pytestmark = pytest.mark.gpu

SAGE_ERR_TOO_LARGE = 6


def noalloc_fn(qas):
    f = qas.lib().sage_quantize_qk_noalloc
    vp, i32 = C.c_void_p, C.c_int
    f.restype = i32
    f.argtypes = [vp, Strides, vp, Strides, i32, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
    return f


def strides(t):
    return Strides(t.stride(0), t.stride(1), t.stride(2))


def call_noalloc(qas, q, k, bq, bk):
    B, H, Nq, D = q.shape
    Nk = k.shape[2]
    out = dict(q_codes=torch.empty((B, H, Nq, D), dtype=torch.int8, device="cuda"),
               q_scales=torch.empty((B, H, -(-Nq // bq)), dtype=torch.float32, device="cuda"),
               k_codes=torch.empty((B, H, Nk, D), dtype=torch.int8, device="cuda"),
               k_scales=torch.empty((B, H, -(-Nk // bk)), dtype=torch.float32, device="cuda"),
               k_mean=torch.empty((B, H, D), dtype=torch.float32, device="cuda"))
    code = noalloc_fn(qas)(q.data_ptr(), strides(q), k.data_ptr(), strides(k), B, H, Nq, Nk, D, bq, bk,
                           out["q_codes"].data_ptr(), out["q_scales"].data_ptr(), out["k_codes"].data_ptr(),
                           out["k_scales"].data_ptr(), out["k_mean"].data_ptr(),
                           torch.cuda.current_stream().cuda_stream)
    assert code == 0, qas.lib().sage_status_string(code)
    return out


def test_noalloc_matches_the_workspace_entry_point_on_two_calls(cuda_lib):
    cases = [(synth.dense_workload("tiny_b1h2n256"), 64, 64),
             (synth.DenseWorkload("noalloc_second", 10, 2, 3, 700, 1031, 128), 128, 64)]
    for w, bq, bk in cases:  # two calls in a row, different shapes, same scratch
        x = synth.dense_inputs(w)
        q, k = bf16_dev(x["q"]), bf16_dev(x["k"])
        got = call_noalloc(cuda_lib, q, k, bq, bk)
        ref = cuda_lib.sage_quantize_qk(q, k, bq, bk)
        torch.cuda.synchronize()
        for key in ("q_codes", "q_scales", "k_codes", "k_scales", "k_mean"):
            assert torch.equal(got[key], ref[key]), f"{w.name}: {key}"


def test_noalloc_accepts_a_problem_exactly_at_its_scratch_limit(cuda_lib):
    # B*H*ceil(Nk/256) == 16384 fills the 8 MiB array exactly: accepted, and
    # equal to the workspace entry point (a one-off in the size check, or in
    # the partial rows the kernels touch, would show here)
    B, H, Nq, Nk = 1, 64, 64, 256 * 256
    gen = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn((B, H, Nq, 128), generator=gen, device="cuda").to(torch.bfloat16)
    k = (torch.randn((B, H, Nk, 128), generator=gen, device="cuda") + 3.0).to(torch.bfloat16)
    got = call_noalloc(cuda_lib, q, k, 64, 128)
    ref = cuda_lib.sage_quantize_qk(q, k, 64, 128)
    torch.cuda.synchronize()
    for key in ("q_codes", "q_scales", "k_codes", "k_scales", "k_mean"):
        assert torch.equal(got[key], ref[key]), key
    del q, k, got, ref
    torch.cuda.empty_cache()


def test_noalloc_rejects_problems_beyond_its_scratch(cuda_lib):
    f = noalloc_fn(cuda_lib)
    fake = 1 << 20  # aligned, never dereferenced: the size check rejects first
    H, Nk = 65, 256 * 253  # 65 * 253 partial rows > 16384
    assert H * (Nk // 256) > 16384
    st = Strides(H * Nk * 128, Nk * 128, 128)
    code = f(fake, st, fake, st, 1, H, Nk, Nk, 128, 64, 64, fake, fake, fake, fake, fake, None)
    assert code == SAGE_ERR_TOO_LARGE
    assert b"scratch" in cuda_lib.lib().sage_status_string(code)
    # one more chunk of keys than fits, with a single head
    code = f(fake, st, fake, st, 1, 1, 8, 256 * 16384 + 1, 128, 64, 64, fake, fake, fake, fake, fake, None)
    assert code == SAGE_ERR_TOO_LARGE
