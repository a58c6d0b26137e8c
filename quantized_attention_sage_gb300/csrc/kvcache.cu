// Int8 KV-cache writer: new K/V rows (bf16 or fp32, token-major) quantized per
// (kv head, token) into the int8 cache with fp16 scales, at cache positions
// pos0 .. pos0 + N - 1.
//
// Page: "Strata PR #2092" (an int8 K/V cache with per-token fp16 scales,
// written upstream of the prompt attention).  Per row of 128 channels:
//   amax  = max |x_c|
//   scale = fp16_rn(fl(amax / 127))      (IEEE fp32 division, then fp16)
//   code  = clamp(rint_even(fl(x_c / float(scale))), -127, 127); 0 where the
//           fp16 scale is 0.
//
// GB300 design: HBM-bound streaming.  Rows whose source is 16-byte aligned
// take a wide kernel (8 lanes per row, four rows per warp, rows walked head by
// head so every address advances by a constant, source slices staged through
// shared memory with cp.async several steps ahead); others one warp per row,
// four channels per lane (8- or 16-byte loads, 4-byte code stores: a row is
// one 128-byte line of the cache).  The row maximum by warp shuffles, one
// division-free code per channel (a multiply by the correctly rounded
// reciprocal of the scale, with the exact quotient taken only next to a
// rounding boundary), no 64-bit division in the row loop; one wave of equal
// CTAs, as many as fit on the SMs at once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace sg {

SG_BOUNDS_FILE(kvcache, 3)

namespace kvc {

template <bool kF32>
__device__ __forceinline__ void load_row(const void *src, int64_t off, float (&x)[4]) {
  if (kF32) {
    const float4 v = *reinterpret_cast<const float4 *>(static_cast<const float *>(src) + off);
    x[0] = v.x;
    x[1] = v.y;
    x[2] = v.z;
    x[3] = v.w;
  } else {
    const uint2 w = *reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(src) + off);
    x[0] = __uint_as_float(w.x << 16);
    x[1] = __uint_as_float(w.x & 0xFFFF0000u);
    x[2] = __uint_as_float(w.y << 16);
    x[3] = __uint_as_float(w.y & 0xFFFF0000u);
  }
}

// fl(a / 127) without a division, by Markstein's correction step: with
// y = fl(1/127), q0 = fl(a * y) is within an ulp of a / 127, the remainder
// a - 127 * q0 is exact in one fma, and fl(q0 + remainder * y) is the
// correctly rounded quotient.  Equal to IEEE division for every finite a >= 0
// (all 2^31 such fp32 values compared on the GPU); a non-finite a gives a * y,
// which is a / 127 (infinity or NaN) as well.
__device__ __forceinline__ float div127(float a) {
  const float y = 0x1.020408p-7f;  // fl(1/127)
  const float q0 = __fmul_rn(a, y);
  if (!(a <= 3.40282347e38f)) return q0;
  return __fmaf_rn(__fmaf_rn(-127.f, q0, a), y, q0);
}

// The correctly rounded fp32 reciprocal of a positive finite fp16 value s:
// the MUFU approximation refined by one Newton-Raphson step,
// r1 = r0 + r0 (1 - s r0).  Equal to the correctly rounded 1/s for every
// positive finite fp16 s (all 31,743 compared on the GPU).
__device__ __forceinline__ float rcp_of_f16(float s) {
  float r0;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r0) : "f"(s));
  return __fmaf_rn(r0, __fmaf_rn(-s, r0, 1.f), r0);
}

// One row of 128 channels held four per lane: fp16 scale and int8 codes.
// q = x * fl(1/s) is within 3 * 2^-24 * |x/s| of fl(x/s); |x/s| stays below
// 2 * 127 even for an fp16-subnormal scale, so q and fl(x/s) round to the same
// integer unless q lies within 1e-4 of a half-integer, where the quotient is
// divided out with IEEE division.
__device__ __forceinline__ void encode_row(const float (&x)[4], int lane, int8_t *dst_codes, __half *dst_scale,
                                           int32_t *status) {
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const __half s16 = __float2half_rn(div127(amax));
  const float sc = __half2float(s16);
  uint32_t packed = 0;
  if (sc > 0.f) {
    const float inv = sc <= 65504.f ? rcp_of_f16(sc) : 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float q = __fmul_rn(x[k], inv);
      float rq = rintf(q);
      if (0.5f - fabsf(q - rq) < 1e-4f) rq = rintf(__fdiv_rn(x[k], sc));
      int c = int(rq);
      c = c > 127 ? 127 : (c < -127 ? -127 : c);
      packed |= (uint32_t(c) & 0xFFu) << (8 * k);
    }
  }
  *reinterpret_cast<uint32_t *>(dst_codes + 4 * lane) = packed;
  if (lane == 0) {
    *dst_scale = s16;
    if (!(fabsf(sc) <= 65504.f) && status) atomicCAS(status, 0, SAGE_ERR_NONFINITE);
  }
}

// Each warp takes a contiguous range of (token, head) pairs, head fastest, so
// that consecutive rows of the source are read in address order, and encodes
// the K and the V row of each pair (two loads in flight).
template <bool kF32>
__global__ void __launch_bounds__(256) cache_write_kernel(CacheWriteArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t P = int64_t(a.N) * a.Hkv;  // (token, head) pairs, head fastest
  const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t chunk = (P + nwarps - 1) / nwarps;
  int64_t p = warp0 * chunk;
  const int64_t pend = min(P, p + chunk);
  if (p >= pend) return;
  int t = int(p / a.Hkv), h = int(p - int64_t(t) * a.Hkv);
  for (; p < pend; ++p) {
    if (!SG_BOUNDS(t < a.N && h < a.Hkv && int64_t(a.pos0) + t < a.ncache)) return;
    const int64_t off = int64_t(t) * a.src_tok + int64_t(h) * a.src_head + 4 * lane;
    float xk[4], xv[4];
    load_row<kF32>(a.k_src, off, xk);
    load_row<kF32>(a.v_src, off, xv);
    const int64_t pos = int64_t(a.pos0) + t;
    const int64_t co = int64_t(h) * a.cache_head + pos * kD, so = int64_t(h) * a.scale_head + pos;
    encode_row(xk, lane, a.k_cache + co, static_cast<__half *>(a.k_scale) + so, a.status);
    encode_row(xv, lane, a.v_cache + co, static_cast<__half *>(a.v_scale) + so, a.status);
    if (++h == a.Hkv) {
      h = 0;
      ++t;
    }
  }
}

// Wide variant for 16-byte aligned rows: 8 lanes per row, 16 channels per
// lane (16-byte slices), four rows per warp step: the K and V rows of two
// consecutive tokens of one kv head.  Rows are taken head by head, tokens in
// order, so a warp's steps advance every address by a constant (two source
// token rows, 256 bytes of codes, two scales) and its codes land contiguously.
// Source slices stream through shared memory with cp.async, kDepth steps
// ahead (the bytes in flight cost no registers; each thread reads back only
// its own slots).  The scale and every code equal encode_row's: the same
// rounding decisions, reached with fewer instructions.
template <bool kF32>
__global__ void __launch_bounds__(256) cache_write_wide_kernel(CacheWriteArgs a) {
  const int lane = threadIdx.x & 31, grp = lane >> 3, l8 = lane & 7;
  const int64_t F = int64_t(a.N) * a.Hkv;  // rows pairs, head-major: f = h * N + t
  const int64_t F2 = (F + 1) >> 1;          // warp steps
  const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t chunk = (F2 + nwarps - 1) / nwarps;
  int64_t q = warp0 * chunk;
  const int64_t qend = min(F2, q + chunk);
  if (q >= qend) return;
  const bool isv = grp & 1;
  const char *src = static_cast<const char *>(isv ? a.v_src : a.k_src);
  int8_t *cache = isv ? a.v_cache : a.k_cache;
  __half *scale = static_cast<__half *>(isv ? a.v_scale : a.k_scale);
  constexpr int kVec = kF32 ? 4 : 2;  // 16-byte pieces of a 16-channel slice
  constexpr int64_t kEsz = kF32 ? 4 : 2;
  // A cursor over this lane's rows: f = 2 q + (grp >> 1) as (t, h), with the
  // byte offset of its source slice.
  struct Cursor {
    int64_t f;
    int t, h;
    int64_t src;
  };
  auto at = [&](int64_t f) {
    Cursor c;
    c.f = f;
    c.h = int(f / a.N);
    c.t = int(f - int64_t(c.h) * a.N);
    c.src = (int64_t(c.t) * a.src_tok + int64_t(c.h) * a.src_head + 16 * l8) * kEsz;
    return c;
  };
  auto step = [&](Cursor &c) {  // f += 2
    c.f += 2;
    c.t += 2;
    c.src += 2 * a.src_tok * kEsz;
    if (c.t >= a.N) {  // next head (rare)
      c = at(c.f);
    }
  };
  constexpr int kDepth = kF32 ? 2 : 4;
  __shared__ uint4 stage[kDepth][256][kVec];
  Cursor ci = at(2 * q + (grp >> 1));  // issue cursor, kDepth - 1 steps ahead
  Cursor cc = ci;                      // the step being encoded
  auto issue = [&](int64_t qq) {
    uint4 *slot = stage[qq % kDepth][threadIdx.x];
    if (qq < qend && ci.f < F && SG_BOUNDS(ci.t < a.N && ci.h < a.Hkv)) {
      const char *g4 = src + ci.src;
#pragma unroll
      for (int u = 0; u < kVec; ++u)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(slot + u)), "l"(g4 + 16 * u)
                     : "memory");
    } else {
#pragma unroll
      for (int u = 0; u < kVec; ++u) slot[u] = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (qq < qend) step(ci);
  };
#pragma unroll
  for (int i = 0; i < kDepth - 1; ++i) issue(q + i);
  for (; q < qend; ++q) {
    issue(q + kDepth - 1);
    asm volatile("cp.async.wait_group %0;" ::"n"(kDepth - 1) : "memory");
    uint4 cur[kVec];
#pragma unroll
    for (int u = 0; u < kVec; ++u) cur[u] = stage[q % kDepth][threadIdx.x][u];
    float x[16];
    if (kF32) {
#pragma unroll
      for (int u = 0; u < kVec; ++u) {
        x[4 * u] = __uint_as_float(cur[u].x);
        x[4 * u + 1] = __uint_as_float(cur[u].y);
        x[4 * u + 2] = __uint_as_float(cur[u].z);
        x[4 * u + 3] = __uint_as_float(cur[u].w);
      }
    } else {
#pragma unroll
      for (int u = 0; u < kVec; ++u) {
        const uint32_t ww[4] = {cur[u].x, cur[u].y, cur[u].z, cur[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          x[8 * u + 2 * k] = __uint_as_float(ww[k] << 16);
          x[8 * u + 2 * k + 1] = __uint_as_float(ww[k] & 0xFFFF0000u);
        }
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 16; k += 2) amax = fmax3(amax, fabsf(x[k]), fabsf(x[k + 1]));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const __half s16 = __float2half_rn(div127(amax));
    const float sc = __half2float(s16);
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
    // With a normal fp16 scale (>= 2^-14), |x / s| <= 127 (1 + 2^-11), so the
    // codes need no clamp; only fp16-subnormal scales can exceed 127.  (The
    // vote is taken by the whole warp, before any lane branches.)
    const bool clamp = __any_sync(0xffffffffu, sc > 0.f && sc < 6.103515625e-05f);
    if (!clamp) {
      // Round to nearest even by adding M = 1.5 * 2^23: the sum's ulp is 1,
      // so fl(q + M) = M + rint(q) for |q| < 2^22, the code is the low byte of
      // the sum's bits (two's complement), and q - (fl(q + M) - M) is exact.
      // A q within 1e-4 of a half-integer is redone from the IEEE quotient.
      const float inv = sc > 0.f && sc <= 65504.f ? rcp_of_f16(sc) : 0.f;
      const float2 M2 = make_float2(12582912.f, 12582912.f);
      uint32_t rb[16];
      float dmax = 0.f;
#pragma unroll
      for (int k = 0; k < 16; k += 2) {
        const float2 q2 = fmul2(make_float2(x[k], x[k + 1]), make_float2(inv, inv));
        const float2 r2 = fadd2(q2, M2);
        const float2 d2 = fsub2(q2, fsub2(r2, M2));
        dmax = fmax3(dmax, fabsf(d2.x), fabsf(d2.y));
        rb[k] = __float_as_uint(r2.x);
        rb[k + 1] = __float_as_uint(r2.y);
      }
      if (dmax > 0.5f - 1e-4f) {
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float qk = __fmul_rn(x[k], inv);
          if (fabsf(__fsub_rn(qk, float(__float2int_rn(qk)))) > 0.5f - 1e-4f)
            rb[k] = uint32_t(__float2int_rn(__fdiv_rn(x[k], sc)));
        }
      }
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4)
        packed[k4] = __byte_perm(__byte_perm(rb[4 * k4], rb[4 * k4 + 1], 0x0040u),
                                 __byte_perm(rb[4 * k4 + 2], rb[4 * k4 + 3], 0x0040u), 0x5410u);
      // scale 0, NaN or infinite (flagged below): every code 0, as the IEEE path gives
      if (!(sc > 0.f && sc <= 65504.f)) packed[0] = packed[1] = packed[2] = packed[3] = 0u;
    } else if (sc > 0.f) {
      const float inv = rcp_of_f16(sc);  // fp16-subnormal scales reach this path
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        int c[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float qk = __fmul_rn(x[4 * k4 + u], inv);
          int cv = __float2int_rn(qk);  // round half to even, as rint
          if (fabsf(__fsub_rn(qk, float(cv))) > 0.5f - 1e-4f) cv = __float2int_rn(__fdiv_rn(x[4 * k4 + u], sc));
          c[u] = max(-127, min(127, cv));
        }
        // bytes 0 of c0..c3 -> one word
        packed[k4] = __byte_perm(__byte_perm(c[0], c[1], 0x0040u), __byte_perm(c[2], c[3], 0x0040u), 0x5410u);
      }
    }
    if (cc.f < F && SG_BOUNDS(cc.t < a.N && cc.h < a.Hkv && int64_t(a.pos0) + cc.t < a.ncache)) {
      const int64_t pos = int64_t(a.pos0) + cc.t;
      *reinterpret_cast<uint4 *>(cache + int64_t(cc.h) * a.cache_head + pos * kD + 16 * l8) =
          make_uint4(packed[0], packed[1], packed[2], packed[3]);
      if (l8 == 0) {
        scale[int64_t(cc.h) * a.scale_head + pos] = s16;
        if (!(fabsf(sc) <= 65504.f) && a.status) atomicCAS(a.status, 0, SAGE_ERR_NONFINITE);
      }
    }
    step(cc);
  }
}

}  // namespace kvc

cudaError_t launch_cache_write(const CacheWriteArgs &a, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t nrows = 2 * int64_t(a.Hkv) * a.N;
  // 16-byte aligned rows (fp32 rows always are) take the wide kernel
  const int64_t esz = a.f32 ? 4 : 2;
  const bool wide = ((reinterpret_cast<uintptr_t>(a.k_src) | reinterpret_cast<uintptr_t>(a.v_src)) & 15u) == 0 &&
                    (a.src_tok * esz) % 16 == 0 && (a.src_head * esz) % 16 == 0;
  const void *fn = wide ? (a.f32 ? reinterpret_cast<const void *>(kvc::cache_write_wide_kernel<true>)
                                 : reinterpret_cast<const void *>(kvc::cache_write_wide_kernel<false>))
                        : (a.f32 ? reinterpret_cast<const void *>(kvc::cache_write_kernel<true>)
                                 : reinterpret_cast<const void *>(kvc::cache_write_kernel<false>));
  // One wave of equal CTAs (as many as fit on the SMs at once): each warp
  // walks one contiguous range of rows, so no partial last wave is left.
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, 256, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
  const int64_t want = (nrows + 7) / 8, cap = int64_t(sms) * per_sm;
  const int blocks = int(want < cap ? want : cap);
  if (wide) {
    if (a.f32) kvc::cache_write_wide_kernel<true><<<blocks, 256, 0, st>>>(a);
    else kvc::cache_write_wide_kernel<false><<<blocks, 256, 0, st>>>(a);
  } else {
    if (a.f32) kvc::cache_write_kernel<true><<<blocks, 256, 0, st>>>(a);
    else kvc::cache_write_kernel<false><<<blocks, 256, 0, st>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace sg
