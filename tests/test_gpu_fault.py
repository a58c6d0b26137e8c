"""Failure detection of the dense attention kernel, without a GPU fault.

The fault-test entry point launches the real attention kernel with its load
warp stopped early, so the consumer warps' bounded waits run out: in mode 1 no
copy is ever issued; in mode 2 the query tiles and the first key tile are
loaded and their Q.K^T issued before the waits give up, so the kernel must wait
for those copies and MMAs before it frees its memory.  Either way it must
report SAGE_ERR_TIMEOUT in its status word, return on its own (tensor memory
freed), and leave the CUDA context usable: the next normal call still matches
the oracle."""

import time

import pytest
import torch

import synth
from gpu_helpers import bf16_dev
from test_gpu_dense import check_head, run_dense

pytestmark = pytest.mark.gpu

SAGE_ERR_TIMEOUT = 5


@pytest.mark.parametrize("mode", [1, 2])
def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib, mode):
    w = synth.dense_workload("tiny_b1h2n256")
    x = synth.dense_inputs(w)
    q, k, v = bf16_dev(x["q"]), bf16_dev(x["k"]), bf16_dev(x["v"])
    qk = cuda_lib.sage_quantize_qk(q, k, w.block, w.block)
    vq = cuda_lib.sage_quantize_v(v)
    torch.cuda.synchronize()

    limit_ns = 20_000_000  # 20 ms
    t0 = time.perf_counter()
    status = cuda_lib.sage_attn_fwd_fault_test(qk, vq, limit_ns, w.block, w.block, mode=mode)
    elapsed = time.perf_counter() - t0
    assert status == SAGE_ERR_TIMEOUT
    # the wait gave up near its limit, not at the 2 s default
    assert elapsed < 1.0, elapsed
    # a second injected failure behaves the same (the first left no state behind)
    assert cuda_lib.sage_attn_fwd_fault_test(qk, vq, limit_ns, w.block, w.block, mode=mode) == SAGE_ERR_TIMEOUT

    # the context is still usable: a normal call afterwards is exact
    qk2, vq2, out = run_dense(cuda_lib, q, k, v, w.block, w.block)
    for h in range(w.H):
        check_head(qk2, vq2, out, 0, h, x["q"][0, h], x["k"][0, h], x["v"][0, h], w.block, w.block,
                   tag=f"after-timeout mode {mode} h{h}")


def test_fault_test_rejects_bad_arguments(cuda_lib):
    L = cuda_lib.lib()
    # NULL status word or a zero limit: refused on the host, nothing launched
    rc = L.sage_attn_fwd_fault_test(None, None, None, None, None, None, 1, 1, 128, 128, 128, 64, 64, 0.0,
                                    None, cuda_lib.Strides(0, 0, 0), None, 0, None, 1000, 1, None)
    assert rc == 1
    # an unknown mode: refused on the host as well
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.sage_attn_fwd_fault_test(None, None, None, None, None, None, 1, 1, 128, 128, 128, 64, 64, 0.0,
                                    None, cuda_lib.Strides(0, 0, 0), None, 0, status.data_ptr(), 1000, 3, None)
    assert rc == 1


# The int8-KV kernel: its softmax warps also meet at named barriers, which
# cannot time out; after a bounded wait gives up, every warp must still pass
# the same number of them.  Mode 2 loads Q and two K tiles, so the Q copy into
# tensor memory, two Q.K^T MMAs and the first scores are done before the waits
# for V give up; split-KV (several CTAs per query tile) is on in the larger case.
@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("wname", ["tiny_kv_q96_k300", "kv_split_fault"])
def test_int8kv_bounded_wait_reports_timeout_and_context_survives(cuda_lib, mode, wname):
    from test_gpu_int8kv import oracle_bf16, run
    from gpu_helpers import assert_output_close, bf16_to_f64
    import numpy as np

    w = (synth.int8kv_workload(wname) if wname.startswith("tiny")
         else synth.Int8KVWorkload(wname, 9, 256, 4096, 32, 8, sub=11))
    x = synth.int8kv_inputs(w)
    from kv_helpers import device_cache
    q, kc, ks, vc, vs = device_cache(cuda_lib, x)

    limit_ns = 20_000_000  # 20 ms
    t0 = time.perf_counter()
    status = cuda_lib.int8kv_prompt_attn_fault_test(q, kc, ks, vc, vs, w.q_pos0, limit_ns, mode)
    elapsed = time.perf_counter() - t0
    assert status == SAGE_ERR_TIMEOUT
    assert elapsed < 2.0, elapsed
    assert cuda_lib.int8kv_prompt_attn_fault_test(q, kc, ks, vc, vs, w.q_pos0, limit_ns, mode) == SAGE_ERR_TIMEOUT

    # the context is still usable: a normal call afterwards matches the oracle
    host, out = run(cuda_lib, w, x)
    rng = np.random.default_rng(3)
    rows = rng.integers(0, w.Nq, 64)
    heads = rng.integers(0, w.Hq, 64)
    ref_b, _ = oracle_bf16(w, host, rows, heads)
    got = bf16_to_f64(out[torch.from_numpy(rows), torch.from_numpy(heads)])
    assert_output_close(got, ref_b, f"int8kv after timeout, mode {mode}")


def test_int8kv_fault_test_rejects_bad_arguments(cuda_lib):
    L = cuda_lib.lib()
    rc = L.int8kv_prompt_attn_fault_test(None, 0, 0, None, None, None, None, 0, 0, 1, 0, 1, 1, 1, 128, 0.0, None, 0,
                                         0, None, 0, None, 1000, 1, None)
    assert rc == 1  # NULL status word
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = L.int8kv_prompt_attn_fault_test(None, 0, 0, None, None, None, None, 0, 0, 1, 0, 1, 1, 1, 128, 0.0, None, 0,
                                         0, None, 0, status.data_ptr(), 0, 1, None)
    assert rc == 1  # zero limit
    rc = L.int8kv_prompt_attn_fault_test(None, 0, 0, None, None, None, None, 0, 0, 1, 0, 1, 1, 1, 128, 0.0, None, 0,
                                         0, None, 0, status.data_ptr(), 1000, 3, None)
    assert rc == 1  # unknown mode
