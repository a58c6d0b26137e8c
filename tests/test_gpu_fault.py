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
