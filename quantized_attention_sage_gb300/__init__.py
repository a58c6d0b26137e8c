"""GB300 (sm_103a) quantized attention: Python binding of ``libsage_gb300.so``.

This module only marshals arguments: it turns torch tensors into device
pointers, element strides and the current CUDA stream, allocates outputs and
workspaces with torch, and calls the C ABI declared in
``include/sage_gb300.h``.  Every step of the computation runs in the library's
CUDA kernels; there is no CPU or PyTorch fallback.  If the library has not
been built (``build()``), every call raises.

Entry points (same names as the C ABI):
  sage_quantize_qk, sage_quantize_v, sage_attn_fwd, int8kv_prompt_attn
plus ``sage_attention`` (the three dense steps in one call) and ``sage_attention_host`` (the
same on host buffers, with the copies and quantizers of one group of heads overlapped with the
attention of another).
"""

from __future__ import annotations

import ctypes as C
import math
import os

from .build import DEBUG_LIB, LIB, build as _build_lib

__all__ = [
    "SageError", "build", "lib", "sage_quantize_qk", "sage_quantize_v", "sage_attn_fwd",
    "sage_attn_fwd_scores_dump", "sage_attn_fwd_fault_test", "int8kv_prompt_attn", "int8kv_prompt_attn_fault_test", "int8kv_cache_write",
    "sage_attention", "sage_attention_host", "sage_shard_range", "sage_quantize_qkv", "sage_attn_fwd_f16",
    "Strides", "STATUS", "use_debug_bounds", "debug_bounds_site",
]

STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration", 3: "CUDA error",
          4: "workspace too small", 5: "bounded device wait timed out", 6: "problem too large",
          7: "non-finite input or scale"}
D = 128


class SageError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, 'unknown')} (status {code})")
        self.code = code


class Strides(C.Structure):
    _fields_ = [("b", C.c_int64), ("h", C.c_int64), ("n", C.c_int64)]


_lib = None


def build(force: bool = False) -> str:
    """Compile the CUDA library for sm_103a (in-tree) and load it."""
    global _lib
    path = _build_lib(force=force)
    _lib = None
    lib()
    return path


def use_debug_bounds(enable: bool = True) -> str:
    """Route every entry point to the bounds-checking debug library (built on
    first use) or back to the normal one; returns the library path."""
    global LIB, _lib
    LIB = _build_lib(debug_bounds=True) if enable else _build_lib()
    _lib = None
    lib()
    return LIB


def debug_bounds_site() -> int:
    """First out-of-bounds access site recorded by the debug library since the
    last call (0: none; always 0 for the normal library); clears the record."""
    site = C.c_int32(0)
    code = lib().sage_debug_bounds(C.byref(site))
    if code != 0:
        raise SageError(code, "sage_debug_bounds")
    return int(site.value)


def lib():
    """The loaded C library with argument types set; raises if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise RuntimeError(f"{LIB} is missing: the CUDA library must be built (call build())")
    L = C.CDLL(LIB)
    vp, i32, i64, sz, f32 = C.c_void_p, C.c_int, C.c_int64, C.c_size_t, C.c_float
    L.sage_status_string.restype = C.c_char_p
    L.sage_status_string.argtypes = [i32]
    L.sage_abi_version.restype = i32
    L.sage_quantize_qk_workspace.restype = sz
    L.sage_quantize_qk_workspace.argtypes = [i32, i32, i32]
    L.sage_quantize_qk.restype = i32
    L.sage_quantize_qk.argtypes = [vp, Strides, vp, Strides, i32, i32, i32, i32, i32, i32, i32,
                                   vp, vp, vp, vp, vp, vp, sz, vp]
    L.sage_quantize_v_workspace.restype = sz
    L.sage_quantize_v_workspace.argtypes = [i32, i32, i32]
    L.sage_quantize_v.restype = i32
    L.sage_quantize_v.argtypes = [vp, Strides, i32, i32, i32, i32, vp, vp, vp, sz, vp]
    L.sage_attn_fwd_workspace.restype = sz
    L.sage_attn_fwd_workspace.argtypes = [i32, i32, i32, i32]
    L.sage_attn_fwd.restype = i32
    L.sage_attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32,
                                vp, Strides, vp, sz, vp, vp]
    L.sage_attn_fwd_scores_dump.restype = i32
    L.sage_attn_fwd_scores_dump.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32,
                                            vp, Strides, vp, sz, vp, vp, vp]
    L.sage_attention_host_workspace.restype = sz
    L.sage_attention_host_workspace.argtypes = [i32, i32, i32, i32, i32]
    L.sage_attention_host.restype = i32
    L.sage_attention_host.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32, i32, vp, sz, vp,
                                      vp, vp]
    L.sage_attention_workspace.restype = sz
    L.sage_attention_workspace.argtypes = [i32, i32, i32, i32]
    L.sage_attention.restype = i32
    L.sage_attention.argtypes = [vp, Strides, vp, Strides, vp, Strides, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                 vp, Strides, vp, vp, sz, vp, vp]
    L.sage_attn_fwd_ex.restype = i32
    L.sage_attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32,
                                   vp, Strides, vp, vp, sz, vp, vp]
    L.sage_attn_fwd_fault_test.restype = i32
    L.sage_attn_fwd_fault_test.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32,
                                           vp, Strides, vp, sz, vp, C.c_uint64, i32, vp]
    L.sage_conversion_check.restype = i32
    L.sage_conversion_check.argtypes = [vp, i64, vp, vp, vp, vp, vp]
    L.sage_probe_rates.restype = i32
    L.sage_probe_rates.argtypes = [i32, i32, vp, vp, vp, vp]
    L.sage_quantize_qkv_workspace.restype = sz
    L.sage_quantize_qkv_workspace.argtypes = [i32, i32, i32]
    L.sage_quantize_qkv.restype = i32
    L.sage_quantize_qkv.argtypes = [vp, Strides, vp, Strides, vp, Strides, i32, i32, i32, i32, i32, i32, i32, i32,
                                    vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.sage_attn_fwd_f16.restype = i32
    L.sage_attn_fwd_f16.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, f32, i32, vp, Strides,
                                    vp, vp, vp]
    L.sage_debug_bounds.restype = i32
    L.sage_debug_bounds.argtypes = [C.POINTER(C.c_int32)]
    L.sage_debug_bounds_enabled.restype = i32
    L.sage_shard_range.restype = i32
    L.sage_shard_range.argtypes = [i64, i32, i32, C.POINTER(i64), C.POINTER(i64)]
    L.int8kv_cache_write.restype = i32
    L.int8kv_cache_write.argtypes = [vp, vp, i32, i64, i64, i32, i32, i32, i32, vp, vp, i64, i32, vp, vp, i64,
                                     vp, vp]
    L.int8kv_prompt_attn_workspace.restype = sz
    L.int8kv_prompt_attn_workspace.argtypes = [i32, i32, i32, i32]
    L.int8kv_prompt_attn_fault_test.restype = i32
    L.int8kv_prompt_attn_fault_test.argtypes = [vp, i64, i64, vp, vp, vp, vp, i64, i64, i32, i32, i32, i32, i32,
                                                i32, f32, vp, i64, i64, vp, sz, vp, C.c_uint64, i32, vp]
    L.int8kv_prompt_attn.restype = i32
    L.int8kv_prompt_attn.argtypes = [vp, i64, i64, vp, vp, vp, vp, i64, i64, i32, i32, i32, i32, i32,
                                     i32, f32, vp, i64, i64, vp, sz, vp, vp]
    _lib = L
    return _lib


def _torch():
    import torch
    return torch


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _strides4(t) -> Strides:
    if t.dim() != 4 or t.shape[3] != D or t.stride(3) != 1:
        raise ValueError("expected a [B, H, N, 128] tensor with unit channel stride")
    return Strides(t.stride(0), t.stride(1), t.stride(2))


def _require(t, dtype, name: str, dims: int = None):
    """Device tensors only: there is no CPU path."""
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dimensions, got {t.dim()}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")


def _require_codes(torch, qk: dict, vq: dict):
    """The attention calls take the quantisers' outputs as they come."""
    _require(qk["q_codes"], torch.int8, "q_codes", 4)
    _require(qk["k_codes"], torch.int8, "k_codes", 4)
    _require(qk["q_scales"], torch.float32, "q_scales")
    _require(qk["k_scales"], torch.float32, "k_scales")
    _require(vq["v_codes"], torch.uint8, "v_codes", 4)
    _require(vq["v_scales"], torch.float32, "v_scales")


def _check(code: int, where: str):
    if code != 0:
        raise SageError(code, where)


def _workspace(nbytes: int, device, ws=None):
    torch = _torch()
    if ws is not None:
        if ws.numel() * ws.element_size() < nbytes:
            raise ValueError(f"workspace needs {nbytes} bytes")
        return ws
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------
# dense path
# ---------------------------------------------------------------------------

def sage_quantize_qk(q, k, q_block: int = 64, k_block: int = 64, out=None, workspace=None, stream=None):
    """INT8 per-block codes of Q and of the mean-smoothed K.

    q: [B,H,Nq,128] bf16, k: [B,H,Nk,128] bf16 (any 16-byte aligned strides).
    Returns dict(q_codes, q_scales, k_codes, k_scales, k_mean)."""
    torch = _torch()
    _require(q, torch.bfloat16, "q", 4)
    _require(k, torch.bfloat16, "k", 4)
    if q.shape[:2] != k.shape[:2] or q.shape[3] != D or k.shape[3] != D or q.device != k.device:
        raise ValueError("q and k must be [B, H, N, 128] on one device with the same B and H")
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    dev = q.device
    if out is None:
        out = dict(
            q_codes=torch.empty((B, H, Nq, D), dtype=torch.int8, device=dev),
            q_scales=torch.empty((B, H, -(-Nq // q_block)), dtype=torch.float32, device=dev),
            k_codes=torch.empty((B, H, Nk, D), dtype=torch.int8, device=dev),
            k_scales=torch.empty((B, H, -(-Nk // k_block)), dtype=torch.float32, device=dev),
            k_mean=torch.empty((B, H, D), dtype=torch.float32, device=dev))
    L = lib()
    nbytes = L.sage_quantize_qk_workspace(B, H, Nk)
    ws = _workspace(nbytes, dev, workspace)
    _check(L.sage_quantize_qk(_ptr(q), _strides4(q), _ptr(k), _strides4(k), B, H, Nq, Nk, D, q_block,
                              k_block, _ptr(out["q_codes"]), _ptr(out["q_scales"]), _ptr(out["k_codes"]),
                              _ptr(out["k_scales"]), _ptr(out["k_mean"]), _ptr(ws), nbytes,
                              _stream(stream)), "sage_quantize_qk")
    return out


def nk_pad(nk: int) -> int:
    return (nk + 127) // 128 * 128


def sage_quantize_v(v, out=None, workspace=None, stream=None):
    """FP8 E4M3 per-channel codes of V, transposed to [B,H,128,Nk_pad], and scales [B,H,128]."""
    torch = _torch()
    _require(v, torch.bfloat16, "v", 4)
    if v.shape[3] != D:
        raise ValueError("v must be [B, H, Nk, 128]")
    B, H, Nk, _ = v.shape
    dev = v.device
    if out is None:
        out = dict(v_codes=torch.empty((B, H, D, nk_pad(Nk)), dtype=torch.uint8, device=dev),
                   v_scales=torch.empty((B, H, D), dtype=torch.float32, device=dev))
    L = lib()
    nbytes = L.sage_quantize_v_workspace(B, H, Nk)
    ws = _workspace(nbytes, dev, workspace)
    _check(L.sage_quantize_v(_ptr(v), _strides4(v), B, H, Nk, D, _ptr(out["v_codes"]), _ptr(out["v_scales"]),
                             _ptr(ws), nbytes, _stream(stream)), "sage_quantize_v")
    return out


def sage_attn_fwd(qk: dict, vq: dict, q_block: int = 64, k_block: int = 64, sm_scale: float = 0.0,
                  out=None, workspace=None, status=None, stream=None, causal: bool = False,
                  return_lse: bool = False):
    """Quantized attention forward over the two quantisers' outputs; bf16 [B,H,Nq,128].

    ``causal``: query i sees keys j <= i + (Nk - Nq).  ``return_lse``: also return the
    rows' natural log-sum-exp, fp32 [B,H,Nq]."""
    torch = _torch()
    _require_codes(torch, qk, vq)
    qc, kc = qk["q_codes"], qk["k_codes"]
    B, H, Nq, _ = qc.shape
    Nk = kc.shape[2]
    dev = qc.device
    if out is None:
        out = torch.empty((B, H, Nq, D), dtype=torch.bfloat16, device=dev)
    L = lib()
    nbytes = L.sage_attn_fwd_workspace(B, H, Nq, Nk)
    ws = _workspace(nbytes, dev, workspace)
    if not causal and not return_lse:
        _check(L.sage_attn_fwd(_ptr(qc), _ptr(qk["q_scales"]), _ptr(kc), _ptr(qk["k_scales"]),
                               _ptr(vq["v_codes"]), _ptr(vq["v_scales"]), B, H, Nq, Nk, D, q_block, k_block,
                               float(sm_scale), _ptr(out), _strides4(out), _ptr(ws), nbytes, _ptr(status),
                               _stream(stream)), "sage_attn_fwd")
        return out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev) if return_lse else None
    _check(L.sage_attn_fwd_ex(_ptr(qc), _ptr(qk["q_scales"]), _ptr(kc), _ptr(qk["k_scales"]),
                              _ptr(vq["v_codes"]), _ptr(vq["v_scales"]), B, H, Nq, Nk, D, q_block, k_block,
                              float(sm_scale), int(bool(causal)), _ptr(out), _strides4(out), _ptr(lse), _ptr(ws),
                              nbytes, _ptr(status), _stream(stream)), "sage_attn_fwd_ex")
    return (out, lse) if return_lse else out


SAGE_QK_INT8, SAGE_QK_F16 = 0, 1


def sage_quantize_qkv(q, k, v, q_block: int = 64, k_block: int = 64, images: bool = True, out=None,
                      workspace=None, stream=None):
    """The whole preparation (K smoothing, Q/K INT8 codes, V FP8 codes) in three launches.

    q: [B,H,Nq,128], k, v: [B,H,Nk,128] bf16 CUDA tensors.  Returns dict(q_codes, q_scales,
    k_codes, k_scales, k_mean, v_codes, v_scales); with ``images`` the Q/K codes are their exact
    fp16 images (what sage_attn_fwd_f16 reads), otherwise int8 as sage_quantize_qk writes them."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, torch.bfloat16, name, 4)
    if (q.shape[:2] != k.shape[:2] or k.shape != v.shape or q.shape[3] != D or k.shape[3] != D
            or not (q.device == k.device == v.device)):
        raise ValueError("q [B,H,Nq,128], k and v [B,H,Nk,128] on one device")
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    dev = q.device
    cd = torch.float16 if images else torch.int8
    if out is None:
        out = dict(q_codes=torch.empty((B, H, Nq, D), dtype=cd, device=dev),
                   q_scales=torch.empty((B, H, -(-Nq // q_block)), dtype=torch.float32, device=dev),
                   k_codes=torch.empty((B, H, Nk, D), dtype=cd, device=dev),
                   k_scales=torch.empty((B, H, -(-Nk // k_block)), dtype=torch.float32, device=dev),
                   k_mean=torch.empty((B, H, D), dtype=torch.float32, device=dev),
                   v_codes=torch.empty((B, H, D, nk_pad(Nk)), dtype=torch.uint8, device=dev),
                   v_scales=torch.empty((B, H, D), dtype=torch.float32, device=dev))
    L = lib()
    nbytes = L.sage_quantize_qkv_workspace(B, H, Nk)
    ws = _workspace(nbytes, dev, workspace)
    _check(L.sage_quantize_qkv(_ptr(q), _strides4(q), _ptr(k), _strides4(k), _ptr(v), _strides4(v), B, H, Nq, Nk, D,
                               q_block, k_block, SAGE_QK_F16 if images else SAGE_QK_INT8, _ptr(out["q_codes"]),
                               _ptr(out["q_scales"]), _ptr(out["k_codes"]), _ptr(out["k_scales"]),
                               _ptr(out["k_mean"]), _ptr(out["v_codes"]), _ptr(out["v_scales"]), _ptr(ws), nbytes,
                               _stream(stream)), "sage_quantize_qkv")
    return out


def sage_attn_fwd_f16(prep: dict, q_block: int = 64, k_block: int = 64, sm_scale: float = 0.0, out=None,
                      status=None, stream=None, causal: bool = False, return_lse: bool = False):
    """The attention over sage_quantize_qkv(..., images=True)'s outputs (fp16 images of the
    Q/K codes); bf16 [B,H,Nq,128], or (out, lse) with ``return_lse``.  No workspace."""
    torch = _torch()
    _require(prep["q_codes"], torch.float16, "q images", 4)
    _require(prep["k_codes"], torch.float16, "k images", 4)
    _require(prep["v_codes"], torch.uint8, "v_codes", 4)
    qi, ki = prep["q_codes"], prep["k_codes"]
    B, H, Nq, _ = qi.shape
    Nk = ki.shape[2]
    dev = qi.device
    if out is None:
        out = torch.empty((B, H, Nq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev) if return_lse else None
    _check(lib().sage_attn_fwd_f16(_ptr(qi), _ptr(prep["q_scales"]), _ptr(ki), _ptr(prep["k_scales"]),
                                   _ptr(prep["v_codes"]), _ptr(prep["v_scales"]), B, H, Nq, Nk, D, q_block, k_block,
                                   float(sm_scale), int(bool(causal)), _ptr(out), _strides4(out), _ptr(lse),
                                   _ptr(status), _stream(stream)), "sage_attn_fwd_f16")
    return (out, lse) if return_lse else out


def sage_attn_fwd_scores_dump(qk: dict, vq: dict, q_block: int = 64, k_block: int = 64, sm_scale: float = 0.0,
                              stream=None):
    """sage_attn_fwd plus the exact int32 scores Q.K^T the tensor cores produced.

    Returns (out bf16 [B,H,Nq,128], scores int32 [B,H,Nq_pad,Nk_pad]).  For checking small problems."""
    torch = _torch()
    _require_codes(torch, qk, vq)
    qc, kc = qk["q_codes"], qk["k_codes"]
    B, H, Nq, _ = qc.shape
    Nk = kc.shape[2]
    dev = qc.device
    out = torch.empty((B, H, Nq, D), dtype=torch.bfloat16, device=dev)
    nq_pad = (Nq + 255) // 256 * 256
    scores = torch.zeros((B, H, nq_pad, nk_pad(Nk)), dtype=torch.int32, device=dev)
    L = lib()
    nbytes = L.sage_attn_fwd_workspace(B, H, Nq, Nk)
    ws = _workspace(nbytes, dev)
    _check(L.sage_attn_fwd_scores_dump(_ptr(qc), _ptr(qk["q_scales"]), _ptr(kc), _ptr(qk["k_scales"]),
                                       _ptr(vq["v_codes"]), _ptr(vq["v_scales"]), B, H, Nq, Nk, D, q_block,
                                       k_block, float(sm_scale), _ptr(out), _strides4(out), _ptr(ws), nbytes,
                                       None, _ptr(scores), _stream(stream)), "sage_attn_fwd_scores_dump")
    return out, scores


def sage_attn_fwd_fault_test(qk: dict, vq: dict, wait_limit_ns: int, q_block: int = 64, k_block: int = 64,
                             stream=None, mode: int = 1) -> int:
    """Launch sage_attn_fwd with its load warp stopped early, so the bounded waits run out.

    mode 1: no copy is issued; mode 2: the query tiles and the first key tile are
    loaded (and their Q.K^T issued) before the waits give up.  Returns the device
    status word after synchronising (SAGE_ERR_TIMEOUT when the failure detection
    works).  Test hook: the output is not written."""
    torch = _torch()
    _require_codes(torch, qk, vq)
    qc, kc = qk["q_codes"], qk["k_codes"]
    B, H, Nq, _ = qc.shape
    Nk = kc.shape[2]
    dev = qc.device
    out = torch.zeros((B, H, Nq, D), dtype=torch.bfloat16, device=dev)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    L = lib()
    nbytes = L.sage_attn_fwd_workspace(B, H, Nq, Nk)
    ws = _workspace(nbytes, dev)
    _check(L.sage_attn_fwd_fault_test(_ptr(qc), _ptr(qk["q_scales"]), _ptr(kc), _ptr(qk["k_scales"]),
                                      _ptr(vq["v_codes"]), _ptr(vq["v_scales"]), B, H, Nq, Nk, D, q_block,
                                      k_block, 0.0, _ptr(out), _strides4(out), _ptr(ws), nbytes, _ptr(status),
                                      int(wait_limit_ns), int(mode), _stream(stream)), "sage_attn_fwd_fault_test")
    torch.cuda.synchronize(dev)
    return int(status.item())


_copy_streams = {}


def _side_stream(cache: dict, dev):
    s = cache.get(dev.index)
    if s is None:
        s = cache[dev.index] = _torch().cuda.Stream(device=dev)
    return s


def sage_attention(q, k, v, q_block: int = 64, k_block: int = 64, sm_scale: float = 0.0, out=None,
                   stream=None, causal: bool = False, return_lse: bool = False, workspace=None, status=None):
    """The dense path in one call (C ``sage_attention``): quantize Q/K, quantize V, attention.

    q: [B,H,Nq,128], k, v: [B,H,Nk,128] bf16 CUDA tensors (16-byte aligned strides).
    Returns out bf16 [B,H,Nq,128], or (out, lse) with ``return_lse``."""
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, torch.bfloat16, name, 4)
    if (q.shape[:2] != k.shape[:2] or k.shape != v.shape or q.shape[3] != D or k.shape[3] != D
            or not (q.device == k.device == v.device)):
        raise ValueError("q [B,H,Nq,128], k and v [B,H,Nk,128] on one device")
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    dev = q.device
    if out is None:
        out = torch.empty((B, H, Nq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev) if return_lse else None
    L = lib()
    nbytes = L.sage_attention_workspace(B, H, Nq, Nk)
    ws = _workspace(nbytes, dev, workspace)
    _check(L.sage_attention(_ptr(q), _strides4(q), _ptr(k), _strides4(k), _ptr(v), _strides4(v), B, H, Nq, Nk, D,
                            q_block, k_block, float(sm_scale), int(bool(causal)), _ptr(out), _strides4(out),
                            _ptr(lse), _ptr(ws), nbytes, _ptr(status), _stream(stream)),
           "sage_attention")
    return (out, lse) if return_lse else out


def sage_attention_host(q, k, v, out, q_block: int = 64, k_block: int = 64, sm_scale: float = 0.0,
                        causal: bool = False, head_chunk: int = 4, workspace=None, status=None, stream=None,
                        copy_stream=None):
    """The dense path on host tensors q, out [B,H,Nq,128] and k, v [B,H,Nk,128] (bf16, contiguous;
    page-locked for the copies to overlap the kernels).  Groups of up to ``head_chunk`` heads are
    copied in and out and quantized on ``copy_stream`` while the attention of another group runs on
    ``stream``; ``out`` is complete once ``stream`` reaches the end of the call.  Both streams must
    differ (non-default streams overlap)."""
    torch = _torch()
    for t in (q, k, v, out):
        if t.device.type != "cpu" or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q, k, v, out must be contiguous bf16 [B, H, N, 128] host tensors")
    B, H, Nq, _ = q.shape
    Nk = k.shape[2]
    dev = torch.device("cuda", torch.cuda.current_device())
    if copy_stream is None:
        copy_stream = _side_stream(_copy_streams, dev)
    L = lib()
    nbytes = L.sage_attention_host_workspace(B, H, Nq, Nk, head_chunk)
    ws = _workspace(nbytes, dev, workspace)
    _check(L.sage_attention_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, Nq, Nk, D, q_block, k_block,
                                 float(sm_scale), int(bool(causal)), int(head_chunk), _ptr(ws), nbytes,
                                 _ptr(status), _stream(stream), _stream(copy_stream)), "sage_attention_host")
    return out


# ---------------------------------------------------------------------------
# int8 KV-cache prompt attention
# ---------------------------------------------------------------------------

def int8kv_prompt_attn(q, k_cache, k_scale, v_cache, v_scale, q_pos0: int, sm_scale: float = 0.0,
                       out=None, workspace=None, status=None, stream=None, _fault=None):
    """Causal prompt attention of q [Nq,Hq,128] bf16 over an int8 cache.

    k_cache, v_cache: int8 [Hkv, Nk, 128] (token rows contiguous);
    k_scale, v_scale: fp16 [Hkv, Nk].  Returns bf16 [Nq, Hq, 128]."""
    torch = _torch()
    Nq, Hq, _ = q.shape
    Hkv, Nk, _ = k_cache.shape
    if k_cache.stride() != v_cache.stride() or k_cache.stride(1) != D or k_cache.stride(2) != 1:
        raise ValueError("k_cache and v_cache must share a [Hkv, Nk, 128] layout with contiguous token rows")
    if k_scale.stride() != v_scale.stride() or k_scale.stride(1) != 1:
        raise ValueError("k_scale and v_scale must share a [Hkv, Nk] layout")
    if q.stride(2) != 1:
        raise ValueError("q channel stride must be 1")
    dev = q.device
    if out is None:
        out = torch.empty((Nq, Hq, D), dtype=torch.bfloat16, device=dev)
    L = lib()
    nbytes = L.int8kv_prompt_attn_workspace(Nq, Hq, Hkv, Nk)
    ws = _workspace(nbytes, dev, workspace)
    args = (_ptr(q), q.stride(0), q.stride(1), _ptr(k_cache), _ptr(k_scale), _ptr(v_cache), _ptr(v_scale),
            k_cache.stride(0), k_scale.stride(0), Nq, int(q_pos0), Nk, Hq, Hkv, D, float(sm_scale), _ptr(out),
            out.stride(0), out.stride(1), _ptr(ws), nbytes, _ptr(status))
    if _fault is not None:  # (wait_limit_ns, mode): int8kv_prompt_attn_fault_test
        _check(L.int8kv_prompt_attn_fault_test(*args, int(_fault[0]), int(_fault[1]), _stream(stream)),
               "int8kv_prompt_attn_fault_test")
        return out
    _check(L.int8kv_prompt_attn(*args, _stream(stream)), "int8kv_prompt_attn")
    return out


def int8kv_prompt_attn_fault_test(q, k_cache, k_scale, v_cache, v_scale, q_pos0: int, wait_limit_ns: int,
                                  mode: int, stream=None) -> int:
    """int8kv_prompt_attn with its load warp stopped early (mode 1: no copy; mode 2: Q and two K
    tiles), so the bounded waits run out after wait_limit_ns; returns the device status word
    (SAGE_ERR_TIMEOUT expected).  Test hook only."""
    torch = _torch()
    status = torch.zeros(1, dtype=torch.int32, device=q.device)
    int8kv_prompt_attn(q, k_cache, k_scale, v_cache, v_scale, q_pos0, status=status, stream=stream,
                       _fault=(wait_limit_ns, mode))
    torch.cuda.synchronize(q.device)
    return int(status.item())


def int8kv_cache_write(k, v, k_cache, k_scale, v_cache, v_scale, pos0: int, status=None, stream=None):
    """Quantize new rows k, v [N, Hkv, 128] (bf16 or fp32) into the int8 cache at positions pos0..pos0+N-1.

    k_cache, v_cache: int8 [Hkv, Ncache, 128] (token rows contiguous); k_scale, v_scale: fp16 [Hkv, Ncache]."""
    torch = _torch()
    N, Hkv, _ = k.shape
    if k.dtype != v.dtype or k.stride() != v.stride() or k.stride(2) != 1:
        raise ValueError("k and v must share dtype and a [N, Hkv, 128] layout with unit channel stride")
    if k.dtype == torch.bfloat16:
        dt = 0
    elif k.dtype == torch.float32:
        dt = 1
    else:
        raise ValueError("k and v must be bf16 or fp32")
    if k_cache.stride() != v_cache.stride() or k_cache.stride(1) != D or k_cache.stride(2) != 1:
        raise ValueError("k_cache and v_cache must share a [Hkv, Ncache, 128] layout with contiguous token rows")
    if k_scale.stride() != v_scale.stride() or k_scale.stride(1) != 1:
        raise ValueError("k_scale and v_scale must share a [Hkv, Ncache] layout")
    L = lib()
    _check(L.int8kv_cache_write(_ptr(k), _ptr(v), dt, k.stride(0), k.stride(1), N, Hkv, D, int(pos0),
                                _ptr(k_cache), _ptr(v_cache), k_cache.stride(0), k_cache.shape[1], _ptr(k_scale),
                                _ptr(v_scale), k_scale.stride(0), _ptr(status), _stream(stream)),
           "int8kv_cache_write")


def default_sm_scale() -> float:
    return 1.0 / math.sqrt(D)


def sage_shard_range(units: int, world: int, rank: int) -> tuple[int, int]:
    """[begin, end) of the `units` independent problems (heads, kv-head groups or
    tokens) that rank `rank` of `world` processes: contiguous, in rank order, the
    first units % world ranks one more (the C ABI's sage_shard_range)."""
    b, e = C.c_int64(0), C.c_int64(0)
    _check(lib().sage_shard_range(int(units), int(world), int(rank), C.byref(b), C.byref(e)), "sage_shard_range")
    return b.value, e.value


def sage_conversion_check(x, stream=None) -> dict:
    """The kernels' four conversions of every fp32 element of the CUDA tensor x
    (even length): dict(e4m3 uint8, i8 int8, bf16 int16 bits, f16 int16 bits)."""
    torch = _torch()
    _require(x, torch.float32, "x", 1)
    n = x.numel()
    dev = x.device
    out = dict(e4m3=torch.empty(n, dtype=torch.uint8, device=dev), i8=torch.empty(n, dtype=torch.int8, device=dev),
               bf16=torch.empty(n, dtype=torch.int16, device=dev), f16=torch.empty(n, dtype=torch.int16, device=dev))
    _check(lib().sage_conversion_check(_ptr(x), n, _ptr(out["e4m3"]), _ptr(out["i8"]), _ptr(out["bf16"]),
                                       _ptr(out["f16"]), _stream(stream)), "sage_conversion_check")
    return out


def sage_probe_rates(kind: int, iters: int, device=None) -> dict:
    """Per-SM rate of one kind of work (0: tcgen05 kind::f16 M128N128K16 MMAs,
    1: kind::f8f6f4 M128N128K32, 2: MUFU ex2), one CTA per SM, synchronised.

    Returns dict(per_clock = MACs (or ex2) per SM per clock (median over SMs),
    ms = the launch's duration, mhz = the SM clock implied by cycles / duration)."""
    torch = _torch()
    dev = torch.device("cuda") if device is None else torch.device(device)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    cycles = torch.zeros(sms, dtype=torch.int64, device=dev)
    sink = torch.zeros(1, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    L = lib()
    a.record(stream)
    _check(L.sage_probe_rates(int(kind), int(iters), _ptr(cycles), _ptr(sink), _ptr(status),
                              _stream(stream)), "sage_probe_rates")
    b.record(stream)
    torch.cuda.synchronize(dev)
    if status.item() != 0:
        raise SageError(int(status.item()), "sage_probe_rates")
    cyc = cycles.double().cpu()
    work = iters * (128 ** 3 if kind in (0, 1) else 64 * 8 * 384)
    ms = a.elapsed_time(b)
    med = float(cyc.median())
    return {"per_clock": work / med, "ms": ms, "mhz": float(cyc.max()) / (ms * 1e3)}
