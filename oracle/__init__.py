"""Python front of the plain C oracle (``sage_oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` use it.  The CUDA library and its binding
never import it.

The C file is compiled with gcc (``-O2 -ffp-contract=off``, no fast-math) into
``oracle/_build/liborc.so`` the first time it is needed, or by ``build()``.
All functions work on one (batch, head) at a time; helpers at the bottom loop
over heads of a whole workload.
"""

from __future__ import annotations

import ctypes as C
import math
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "sage_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "liborc.so")
D = 128
SM_SCALE_D128 = float(np.float32(1.0 / math.sqrt(128.0)))

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle library (gcc, OpenMP) if it is missing or stale."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(LIB)) or os.path.getmtime(LIB) < os.path.getmtime(SRC)
    if force or stale:
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-o", tmp, SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    return LIB


def _p(a: np.ndarray, ct):
    return a.ctypes.data_as(C.POINTER(ct))


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(LIB)
        i32, i64, f32, f64 = C.c_int, C.c_int64, C.c_float, C.c_double
        P = C.POINTER
        L.orc_k_mean.argtypes = [P(C.c_uint16), i32, P(f32)]
        L.orc_quant_q.argtypes = [P(C.c_uint16), i32, i32, P(C.c_int8), P(f32)]
        L.orc_quant_k.argtypes = [P(C.c_uint16), i32, i32, P(f32), P(C.c_int8), P(f32)]
        L.orc_quant_v.argtypes = [P(C.c_uint16), i32, i32, P(C.c_uint8), P(f32)]
        L.orc_sage_attn_rows.argtypes = [P(C.c_int8), P(f32), i32, P(C.c_int8), P(f32), i32,
                                         P(C.c_uint8), i32, P(f32), i32, i32, f32, i32,
                                         P(i32), i32, P(f32), P(C.c_uint16), i32, i32, P(f64)]
        L.orc_sage_attn_rows.restype = i32
        L.orc_attn_rows_f64.argtypes = [P(f64), P(f64), P(f64), i32, i32, f64, i32, P(i32), i32, P(f64),
                                        i32, P(f64)]
        L.orc_int8kv_rows.argtypes = [P(C.c_uint16), P(C.c_int8), P(C.c_uint16), P(C.c_int8),
                                      P(C.c_uint16), i32, i32, i32, i32, i32, f64,
                                      P(i32), P(i32), i32, P(f64), i32]
        L.orc_int8kv_rows.restype = i32
        L.orc_f32_to_bf16_array.argtypes = [P(f32), i64, P(C.c_uint16)]
        L.orc_f32_to_e4m3_array.argtypes = [P(f32), i64, P(C.c_uint8)]
        L.orc_e4m3_value_array.argtypes = [P(C.c_uint8), i64, P(f64)]
        L.orc_f16_value_array.argtypes = [P(C.c_uint16), i64, P(f64)]
        L.orc_f32_to_f16_array.argtypes = [P(f32), i64, P(C.c_uint16)]
        L.orc_cache_quantise_rows.argtypes = [P(f32), i64, P(C.c_int8), P(C.c_uint16)]
        L.orc_f32_to_i8_array.argtypes = [P(f32), i64, P(C.c_int8)]
        _lib = L
    return _lib


# ---------------------------------------------------------------------------
# conversions
# ---------------------------------------------------------------------------

def f32_to_bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_bf16_array(_p(x, C.c_float), x.size, _p(out, C.c_uint16))
    return out


def f32_to_e4m3(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_f32_to_e4m3_array(_p(x, C.c_float), x.size, _p(out, C.c_uint8))
    return out


def e4m3_value(c) -> np.ndarray:
    c = np.ascontiguousarray(c, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().orc_e4m3_value_array(_p(c, C.c_uint8), c.size, _p(out, C.c_double))
    return out


def f16_value(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    lib().orc_f16_value_array(_p(h, C.c_uint16), h.size, _p(out, C.c_double))
    return out


def f32_to_f16(x) -> np.ndarray:
    """fp32 -> fp16 bits, round to nearest even (overflow to infinity)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().orc_f32_to_f16_array(_p(x, C.c_float), x.size, _p(out, C.c_uint16))
    return out


def f32_to_i8(x) -> np.ndarray:
    """fp32 -> int8 code: round half to even, saturated to [-127, 127]."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.int8)
    lib().orc_f32_to_i8_array(_p(x, C.c_float), x.size, _p(out, C.c_int8))
    return out


def cache_quantise(x) -> tuple[np.ndarray, np.ndarray]:
    """Per-token int8 KV cache rows: x fp32 [..., 128] -> (int8 codes, fp16 scale bits [...])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape[-1] == 128
    n = x.size // 128
    codes = np.empty(x.shape, dtype=np.int8)
    scales = np.empty(x.shape[:-1], dtype=np.uint16)
    lib().orc_cache_quantise_rows(_p(x, C.c_float), n, _p(codes, C.c_int8), _p(scales, C.c_uint16))
    return codes, scales


def bf16_value(h) -> np.ndarray:
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# dense path, one head
# ---------------------------------------------------------------------------

def k_mean(k: np.ndarray) -> np.ndarray:
    k = np.ascontiguousarray(k, dtype=np.uint16)
    mu = np.empty(D, dtype=np.float32)
    lib().orc_k_mean(_p(k, C.c_uint16), k.shape[0], _p(mu, C.c_float))
    return mu


def quant_q(q: np.ndarray, bq: int):
    q = np.ascontiguousarray(q, dtype=np.uint16)
    n = q.shape[0]
    codes = np.empty((n, D), dtype=np.int8)
    scales = np.empty((n + bq - 1) // bq, dtype=np.float32)
    lib().orc_quant_q(_p(q, C.c_uint16), n, bq, _p(codes, C.c_int8), _p(scales, C.c_float))
    return codes, scales


def quant_k(k: np.ndarray, bk: int, mu: np.ndarray):
    k = np.ascontiguousarray(k, dtype=np.uint16)
    mu = np.ascontiguousarray(mu, dtype=np.float32)
    n = k.shape[0]
    codes = np.empty((n, D), dtype=np.int8)
    scales = np.empty((n + bk - 1) // bk, dtype=np.float32)
    lib().orc_quant_k(_p(k, C.c_uint16), n, bk, _p(mu, C.c_float), _p(codes, C.c_int8),
                      _p(scales, C.c_float))
    return codes, scales


def nk_pad(nk: int) -> int:
    return (nk + 127) // 128 * 128


def quant_v(v: np.ndarray):
    v = np.ascontiguousarray(v, dtype=np.uint16)
    n = v.shape[0]
    npad = nk_pad(n)
    codes = np.empty((D, npad), dtype=np.uint8)
    scales = np.empty(D, dtype=np.float32)
    lib().orc_quant_v(_p(v, C.c_uint16), n, npad, _p(codes, C.c_uint8), _p(scales, C.c_float))
    return codes, scales


def sage_attn_rows(qc, sq, bq, kc, sk, bk, vct, sv, Nq, Nk, rows=None, sm_scale=SM_SCALE_D128,
                   tile=128, nthreads=0, causal=False, with_lse=False):
    """The quantized program for the given query rows of one head.

    Returns (out_f32 [n,128] before rounding, out_bf16 bits [n,128], threads used), plus the
    rows' log-sum-exp (fp64 [n]) when ``with_lse``."""
    rows = np.arange(Nq, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    qc = np.ascontiguousarray(qc, dtype=np.int8)
    kc = np.ascontiguousarray(kc, dtype=np.int8)
    vct = np.ascontiguousarray(vct, dtype=np.uint8)
    sq = np.ascontiguousarray(sq, dtype=np.float32)
    sk = np.ascontiguousarray(sk, dtype=np.float32)
    sv = np.ascontiguousarray(sv, dtype=np.float32)
    n = rows.size
    out = np.empty((n, D), dtype=np.float32)
    outb = np.empty((n, D), dtype=np.uint16)
    lse = np.empty(n, dtype=np.float64)
    used = lib().orc_sage_attn_rows(_p(qc, C.c_int8), _p(sq, C.c_float), bq, _p(kc, C.c_int8),
                                    _p(sk, C.c_float), bk, _p(vct, C.c_uint8), vct.shape[1],
                                    _p(sv, C.c_float), Nq, Nk, float(sm_scale), tile,
                                    _p(rows, C.c_int), n, _p(out, C.c_float), _p(outb, C.c_uint16),
                                    int(nthreads), int(bool(causal)),
                                    _p(lse, C.c_double) if with_lse else None)
    return (out, outb, used, lse) if with_lse else (out, outb, used)


def attn_rows_f64(q, k, v, sm_scale=1.0 / math.sqrt(128.0), tile=128, rows=None, causal=False,
                  with_lse=False):
    """Quantisation-off twin of the same tile loop (fp64, identity quantisers)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    k = np.ascontiguousarray(k, dtype=np.float64)
    v = np.ascontiguousarray(v, dtype=np.float64)
    Nq, Nk = q.shape[0], k.shape[0]
    rows = np.arange(Nq, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    out = np.empty((rows.size, D), dtype=np.float64)
    lse = np.empty(rows.size, dtype=np.float64)
    lib().orc_attn_rows_f64(_p(q, C.c_double), _p(k, C.c_double), _p(v, C.c_double), Nq, Nk,
                            float(sm_scale), tile, _p(rows, C.c_int), rows.size, _p(out, C.c_double),
                            int(bool(causal)), _p(lse, C.c_double))
    return (out, lse) if with_lse else out


def sage_head(q, k, v, bq, bk, rows=None, sm_scale=SM_SCALE_D128, nthreads=0, causal=False):
    """Whole dense path for one head: bf16 bits [N,128] in, everything out (incl. the rows' lse)."""
    mu = k_mean(k)
    qc, sq = quant_q(q, bq)
    kc, sk = quant_k(k, bk, mu)
    vct, sv = quant_v(v)
    out, outb, used, lse = sage_attn_rows(qc, sq, bq, kc, sk, bk, vct, sv, q.shape[0], k.shape[0],
                                          rows=rows, sm_scale=sm_scale, nthreads=nthreads, causal=causal,
                                          with_lse=True)
    return dict(mu=mu, qc=qc, sq=sq, kc=kc, sk=sk, vct=vct, sv=sv, out=out, out_bf16=outb, lse=lse,
                threads=used)


# ---------------------------------------------------------------------------
# int8 KV-cache prompt attention
# ---------------------------------------------------------------------------

def int8kv_rows(q, kc, ks, vc, vs, q_pos0, rows, heads, Hkv=None, sm_scale=1.0 / math.sqrt(128.0),
                nthreads=0):
    """fp64 exact program for the (row, head) pairs given.

    q bf16 bits [Nq, Hq, 128]; kc, vc int8 [Hkv, Nk, 128]; ks, vs fp16 [Hkv, Nk]."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kc = np.ascontiguousarray(kc, dtype=np.int8)
    vc = np.ascontiguousarray(vc, dtype=np.int8)
    ks = np.ascontiguousarray(np.asarray(ks, dtype=np.float16).view(np.uint16))
    vs = np.ascontiguousarray(np.asarray(vs, dtype=np.float16).view(np.uint16))
    Nq, Hq = q.shape[0], q.shape[1]
    Hkv = kc.shape[0] if Hkv is None else Hkv
    Nk = kc.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    heads = np.ascontiguousarray(heads, dtype=np.int32)
    out = np.empty((rows.size, D), dtype=np.float64)
    used = lib().orc_int8kv_rows(_p(q, C.c_uint16), _p(kc, C.c_int8), _p(ks, C.c_uint16),
                                 _p(vc, C.c_int8), _p(vs, C.c_uint16), Nq, q_pos0, Nk, Hq, Hkv,
                                 float(sm_scale), _p(rows, C.c_int), _p(heads, C.c_int), rows.size,
                                 _p(out, C.c_double), int(nthreads))
    return out, used
