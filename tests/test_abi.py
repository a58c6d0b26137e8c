"""The C-ABI library: it builds for sm_103a, loads, exports every function the
header declares, and rejects bad arguments on the host before any launch.
No compute call is made here (these tests run without a GPU)."""

import ctypes as C
import os
import re

import pytest

import quantized_attention_sage_gb300 as qas
from quantized_attention_sage_gb300 import Strides

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sage_gb300.h")


@pytest.fixture(scope="module")
def L():
    qas.build()
    return qas.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z][a-z0-9_]*)\s*\(", text)
    skip = {"sizeof", "if", "return"}
    return sorted({n for n in names if n not in skip and (n.startswith("sage_") or n.startswith("int8kv_"))})


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("sage_quantize_qk", "sage_quantize_v", "sage_attn_fwd", "int8kv_prompt_attn"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n


def test_abi_version_and_status_strings(L):
    assert L.sage_abi_version() == 2
    assert L.sage_status_string(0) == b"ok"
    assert L.sage_status_string(4) == b"workspace too small"
    assert L.sage_status_string(99) == b"unknown status"


def test_workspace_queries(L):
    assert L.sage_quantize_qk_workspace(1, 24, 37810) >= 24 * 148 * 128 * 4
    assert L.sage_quantize_v_workspace(1, 24, 37810) >= 24 * 149 * 128 * 4
    assert L.sage_attn_fwd_workspace(1, 24, 37810, 37810) >= 2 * 24 * 37810 * 128 * 2
    assert L.int8kv_prompt_attn_workspace(1024, 32, 8, 32768) > 2 * 8 * 32768 * 128 * 2
    assert L.sage_quantize_qk_workspace(0, 1, 1) == 0
    assert L.int8kv_prompt_attn_workspace(4, 6, 4, 10) == 0  # Hq % Hkv != 0


FAKE = 1 << 20  # 16-byte aligned, never dereferenced: validation fails first


def s4(b, h, n):
    return Strides(b, h, n)


def test_quantize_qk_rejects_bad_arguments(L):
    st = s4(2 * 256 * 128, 256 * 128, 128)
    ok_args = dict(q=FAKE, qs=st, k=FAKE, ks=st, B=1, H=2, Nq=256, Nk=256, d=128, qb=64, kb=64)

    def call(**kw):
        a = dict(ok_args)
        a.update(kw)
        return L.sage_quantize_qk(a["q"], a["qs"], a["k"], a["ks"], a["B"], a["H"], a["Nq"], a["Nk"], a["d"],
                                  a["qb"], a["kb"], FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                  a.get("wsb", 0), None)
    assert call(d=64) == 2
    assert call(qb=32) == 2
    assert call(kb=256) == 2
    assert call(Nq=0) == 1
    assert call(B=0) == 1
    assert call(q=None) == 1
    assert call(k=FAKE + 8) == 1                       # misaligned
    assert call(qs=s4(2 * 256 * 128, 256 * 128, 100)) == 1  # stride not a multiple of 8
    assert call(wsb=0) == 4                            # workspace too small


def test_quantize_v_and_attn_reject_bad_arguments(L):
    st = s4(2 * 256 * 128, 256 * 128, 128)
    assert L.sage_quantize_v(FAKE, st, 1, 2, 256, 100, FAKE, FAKE, FAKE, 1 << 30, None) == 2
    assert L.sage_quantize_v(None, st, 1, 2, 256, 128, FAKE, FAKE, FAKE, 1 << 30, None) == 1
    assert L.sage_quantize_v(FAKE, st, 1, 2, 256, 128, FAKE, FAKE, FAKE, 0, None) == 4
    assert L.sage_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 256, 128, 64, 48, 0.0, FAKE, st,
                           FAKE, 1 << 30, None, None) == 2
    assert L.sage_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 256, 128, 64, 64, 0.0, None, st,
                           FAKE, 1 << 30, None, None) == 1
    assert L.sage_attn_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 256, 128, 64, 64, 0.0, FAKE, st,
                           FAKE, 16, None, None) == 4


def test_int8kv_rejects_bad_arguments(L):
    def call(Nq=8, q_pos0=8, Nk=16, Hq=4, Hkv=2, d=128, kvhs=16 * 128, q=FAKE, wsb=1 << 30):
        return L.int8kv_prompt_attn(q, Hq * 128, 128, FAKE, FAKE, FAKE, FAKE, kvhs, Nk, Nq, q_pos0, Nk, Hq,
                                    Hkv, d, 0.0, FAKE, Hq * 128, 128, FAKE, wsb, None, None)
    assert call(d=96) == 2
    assert call(Hq=6, Hkv=4) == 1        # not a whole number of query heads per kv head
    assert call(q_pos0=9) == 1           # q_pos0 + Nq > Nk
    assert call(q_pos0=-1) == 1
    assert call(kvhs=100) == 1           # kv head stride below Nk * 128
    assert call(q=FAKE + 4) == 1
    assert call(wsb=0) == 4


def test_cache_write_rejects_bad_arguments(L):
    def call(dt=0, N=8, Hkv=2, d=128, pos0=0, Ncache=16, src=FAKE, tok=256, head=128, chs=16 * 128, cache=FAKE,
             sc=FAKE, schs=16):
        return L.int8kv_cache_write(src, src, dt, tok, head, N, Hkv, d, pos0, cache, cache, chs, Ncache, sc, sc,
                                    schs, None, None)
    assert call(d=64) == 2
    assert call(dt=5) == 2
    assert call(pos0=9) == 1              # pos0 + N > Ncache
    assert call(pos0=-1) == 1
    assert call(N=0) == 1
    assert call(chs=100) == 1             # cache head stride below Ncache * 128
    assert call(schs=8) == 1              # scale head stride below Ncache
    assert call(src=FAKE + 2) == 1        # bf16 rows need 8-byte alignment
    assert call(dt=1, src=FAKE + 8) == 1  # fp32 rows need 16-byte alignment
    assert call(tok=258) == 1             # strides in multiples of 4 elements
    assert call(cache=FAKE + 8) == 1
    assert call(sc=FAKE + 1) == 1
    assert L.sage_status_string(7) != L.sage_status_string(99)


def test_host_pipeline_rejects_bad_arguments(L):
    ws = L.sage_attention_host_workspace(1, 4, 256, 256, 2)
    assert ws > 2 * 3 * 2 * 256 * 128 * 2
    assert L.sage_attention_host_workspace(1, 4, 256, 256, 0) == 0

    def call(d=128, qb=64, causal=0, chunk=2, Nq=256, Nk=256, q=FAKE, wsb=ws, cs=FAKE, xs=FAKE + 64):
        return L.sage_attention_host(q, FAKE, FAKE, FAKE, 1, 4, Nq, Nk, d, qb, 64, 0.0, causal, chunk, FAKE, wsb,
                                     None, cs, xs)
    assert call(d=64) == 2
    assert call(qb=32) == 2
    assert call(causal=2) == 1
    assert call(causal=1, Nq=300) == 2     # causal needs Nq <= Nk
    assert call(chunk=0) == 1
    assert call(q=None) == 1
    assert call(xs=FAKE) == 1               # the two streams must differ
    assert call(xs=None) == 1
    assert call(wsb=ws - 1) == 4


def test_attn_fwd_ex_rejects_bad_arguments(L):
    st = s4(2 * 256 * 128, 256 * 128, 128)

    def call(causal=0, Nq=256, Nk=256, lse=None):
        return L.sage_attn_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, Nq, Nk, 128, 64, 64, 0.0, causal, FAKE,
                                  st, lse, FAKE, 1 << 30, None, None)
    assert call(causal=2) == 1                 # causal is 0 or 1
    assert call(causal=1, Nq=300) == 2         # the causal window needs Nq <= Nk
    assert call(lse=FAKE + 2) == 1             # lse must be 4-byte aligned
    assert L.sage_attn_fwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 256, 256, 96, 64, 64, 0.0, 0, FAKE, st,
                              None, FAKE, 1 << 30, None, None) == 2   # d != 128


def test_binding_rejects_wrong_dtypes_and_host_tensors():
    """The Python binding checks dtypes, ranks and the device before it calls the
    library, so a CPU tensor is an error, never a silent host computation."""
    torch = pytest.importorskip("torch")
    q = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        qas.sage_quantize_qk(q, q)
    with pytest.raises(ValueError, match="bfloat16"):
        qas.sage_quantize_qk(q.float(), q)
    with pytest.raises(ValueError, match="CUDA"):
        qas.sage_quantize_v(q)
    with pytest.raises(ValueError, match="dimensions"):
        qas.sage_quantize_v(q[0])
    qk = dict(q_codes=torch.zeros((1, 1, 64, 128), dtype=torch.int8),
              k_codes=torch.zeros((1, 1, 64, 128), dtype=torch.int8),
              q_scales=torch.zeros((1, 1, 1)), k_scales=torch.zeros((1, 1, 1)))
    vq = dict(v_codes=torch.zeros((1, 1, 128, 128), dtype=torch.uint8), v_scales=torch.zeros((1, 1, 128)))
    with pytest.raises(ValueError, match="CUDA"):
        qas.sage_attn_fwd(qk, vq)
    with pytest.raises(ValueError, match="int8"):
        qas.sage_attn_fwd(dict(qk, q_codes=qk["q_codes"].to(torch.uint8)), vq)


def test_one_call_dense_path_rejects_bad_arguments(L):
    ws = L.sage_attention_workspace(1, 24, 256, 256)
    assert ws > 24 * 256 * 128 * 3
    assert L.sage_attention_workspace(1, 24, 0, 256) == 0
    st = s4(24 * 256 * 128, 256 * 128, 128)

    def call(d=128, qb=64, causal=0, Nq=256, Nk=256, q=FAKE, qs=st, lse=None, wsb=ws):
        return L.sage_attention(q, qs, FAKE, st, FAKE, st, 1, 24, Nq, Nk, d, qb, 64, 0.0, causal, FAKE, st, lse,
                                FAKE, wsb, None, None)
    assert call(d=96) == 2
    assert call(qb=32) == 2
    assert call(causal=2) == 1
    assert call(causal=1, Nq=300) == 2      # causal needs Nq <= Nk
    assert call(q=None) == 1
    assert call(q=FAKE + 8) == 1            # 16-byte aligned rows only
    assert call(qs=s4(24 * 256 * 128, 256 * 128, 132)) == 1
    assert call(lse=FAKE + 2) == 1
    assert call(wsb=ws - 1) == 4


def test_noalloc_size_check_accepts_exactly_the_limit_and_rejects_one_more(L):
    """The allocation-free entry point's size check, on the host only: a problem
    with B*H*ceil(Nk/256) == 16384 K-mean partial rows fills its fixed 8 MiB
    scratch exactly and passes the check; one more row is SAGE_ERR_TOO_LARGE.
    Without a GPU the accepted call then stops at the CUDA device query
    (SAGE_ERR_CUDA) before anything could be launched on the fake pointers, so
    this test runs only where no CUDA device is visible."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("host-only check: a visible GPU would run the accepted call")
    f = L.sage_quantize_qk_noalloc
    f.restype = C.c_int
    f.argtypes = [C.c_void_p, Strides, C.c_void_p, Strides] + [C.c_int] * 7 + [C.c_void_p] * 6
    H, Nk = 64, 256 * 256
    st = Strides(H * Nk * 128, Nk * 128, 128)
    at_limit = f(FAKE, st, FAKE, st, 1, H, 64, Nk, 128, 64, 64, FAKE, FAKE, FAKE, FAKE, FAKE, None)
    assert at_limit != 6 and at_limit == 3
    over = f(FAKE, st, FAKE, st, 1, H, 64, Nk + 1, 128, 64, 64, FAKE, FAKE, FAKE, FAKE, FAKE, None)
    assert over == 6
