"""The kernels' number-format conversions on the GPU against the oracle's
encoders, bit for bit: a dense stride through all finite fp32 bit patterns
plus every rounding midpoint (and one fp32 step to either side) of E4M3, int8,
bf16 and fp16.  The conversions are the ones the kernels use:
cvt.rn.satfinite.e4m3x2.f32 (V codes, FP8 P), round-to-nearest-even int8 with
saturation to +-127 (Q/K and cache codes), bf16 rn (outputs), fp16 rn (cache
scales); the library's sage_conversion_check applies them to given inputs."""

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def _finite(bits_u32):
    bits_u32 = bits_u32[(bits_u32 & 0x7F800000) != 0x7F800000]
    return bits_u32.view(np.float32)


def _around(mid):
    """each midpoint, and the fp32 neighbours on either side, both signs"""
    mid = np.asarray(mid, dtype=np.float32)
    pts = np.concatenate([mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(-np.inf))])
    return np.concatenate([pts, -pts])


def _inputs():
    sweep = _finite(np.arange(0, 2**32, 97, dtype=np.uint64).astype(np.uint32))
    # E4M3: midpoints between neighbouring codes and past the largest (448)
    e4 = np.unique(oracle.e4m3_value(np.arange(0, 0x7F, dtype=np.uint8)))
    e4_mid = np.concatenate([(e4[1:] + e4[:-1]) / 2, [464.0, 480.0, 1e6]])
    # int8: half-integers up to beyond the clamp
    i8_mid = np.arange(-130, 131) + 0.5
    # bf16: the midpoint below every finite positive bf16 (bits << 16 | 0x8000)
    b = np.arange(0, 0x7F80, dtype=np.uint32)
    bf_mid = ((b << 16) | 0x8000).view(np.float32)
    # fp16: midpoints between neighbours, subnormals included, and the overflow edge
    h = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    f16_mid = np.concatenate([(h[1:] + h[:-1]) / 2, [65520.0, 65504.0 + 8.0]])
    x = np.concatenate([sweep, _around(e4_mid), _around(i8_mid), _around(bf_mid), _around(f16_mid),
                        np.float32([0.0, -0.0, 448.0, -448.0, 127.0, -127.0, 65504.0])])
    if x.size % 2:
        x = np.append(x, np.float32(1.0))
    return np.ascontiguousarray(x, dtype=np.float32)


def test_device_conversions_equal_the_oracle_encoders_bit_for_bit(cuda_lib):
    x = _inputs()
    assert x.size > 40_000_000
    got = cuda_lib.sage_conversion_check(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    checks = (("e4m3", oracle.f32_to_e4m3, np.uint8), ("i8", oracle.f32_to_i8, np.int8),
              ("bf16", oracle.f32_to_bf16, np.uint16), ("f16", oracle.f32_to_f16, np.uint16))
    for key, enc, dt in checks:
        g = got[key].cpu().numpy().view(dt)
        want = enc(x)
        bad = np.flatnonzero(g != want)
        assert bad.size == 0, (f"{key}: {bad.size} mismatches, e.g. x={x[bad[:4]]!r} "
                               f"gpu={g[bad[:4]]!r} oracle={want[bad[:4]]!r}")
