"""Shared helpers of the GPU parity tests (marshalling and the comparison bar)."""

import numpy as np
import torch

# Output bar: GPU bf16 against the oracle's result rounded to bf16, errors in fp64.
MAX_ABS = 2e-3
REL_L2 = 1e-3


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def errors(got: np.ndarray, ref: np.ndarray):
    d = got - ref
    max_abs = float(np.abs(d).max()) if d.size else 0.0
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-300))
    return max_abs, rel


def assert_output_close(got: np.ndarray, ref: np.ndarray, what: str):
    max_abs, rel = errors(got, ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max-abs {max_abs:.3e}, rel-L2 {rel:.3e}"
    return max_abs, rel
