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


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def assert_output_close_rows(got: np.ndarray, ref: np.ndarray, what: str):
    """The bar for outputs whose rows may average only a few keys (causal rows near
    the start): rel-L2 <= 1e-3 as always, and every element within max-abs 2e-3 or
    one bf16 step of the oracle's value, whichever is larger.  A row that sees one
    or two keys has outputs of order one, where a single bf16 rounding that falls
    the other way (fp32 sums in another order) is already 2^-8 or 2^-7."""
    max_abs, rel = errors(got, ref)
    bound = np.maximum(MAX_ABS, bf16_ulp(ref))
    worst = float(np.max(np.abs(got - ref) / bound)) if got.size else 0.0
    assert rel <= REL_L2 and worst <= 1.0, f"{what}: rel-L2 {rel:.3e}, max-abs {max_abs:.3e}, worst/bound {worst:.2f}"
    return max_abs, rel
