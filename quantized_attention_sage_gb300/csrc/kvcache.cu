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
// take a wide kernel (8 lanes per row, four rows per warp); others one warp
// per row, four channels per lane (8- or 16-byte loads, 4-byte code stores: a
// row is one 128-byte line of the cache), the row maximum by warp shuffles, one division-free code per
// channel (a multiply by the correctly rounded reciprocal of the scale, with
// the exact quotient taken only next to a rounding boundary), no 64-bit
// division in the row loop; one resident grid of 8 blocks of 256 threads per
// SM.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

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
  const __half s16 = __float2half_rn(__fdiv_rn(amax, 127.f));
  const float sc = __half2float(s16);
  uint32_t packed = 0;
  if (sc > 0.f) {
    const float inv = __frcp_rn(sc);
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
// lane (16-byte loads and code stores), four rows per warp (the K and V rows
// of two consecutive (token, head) pairs), the row maximum over 16 values and
// three shuffles: about half the instructions per row of the narrow kernel.
// The codes follow the same steps as encode_row.
template <bool kF32>
__global__ void __launch_bounds__(256) cache_write_wide_kernel(CacheWriteArgs a) {
  const int lane = threadIdx.x & 31, grp = lane >> 3, l8 = lane & 7;
  const int64_t P = int64_t(a.N) * a.Hkv;
  const int64_t P2 = (P + 1) >> 1;  // pair couples
  const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  const int64_t chunk = (P2 + nwarps - 1) / nwarps;
  int64_t q = warp0 * chunk;
  const int64_t qend = min(P2, q + chunk);
  if (q >= qend) return;
  // this lane's pair: 2q + (grp >> 1); K for even groups, V for odd
  int64_t p = 2 * q + (grp >> 1);
  int t = int(p / a.Hkv), h = int(p - int64_t(t) * a.Hkv);
  const bool isv = grp & 1;
  const void *src = isv ? a.v_src : a.k_src;
  int8_t *cache = isv ? a.v_cache : a.k_cache;
  __half *scale = static_cast<__half *>(isv ? a.v_scale : a.k_scale);
  // raw source bytes of a row slice: 2 x 16 bytes (bf16) or 4 x 16 bytes (fp32)
  constexpr int kVec = kF32 ? 4 : 2;
  auto load = [&](int64_t pp, int tt, int hh, uint4 (&r)[kVec]) {
    if (pp < P && SG_BOUNDS(tt < a.N && hh < a.Hkv)) {
      const int64_t off = int64_t(tt) * a.src_tok + int64_t(hh) * a.src_head + 16 * l8;
      const uint4 *s4 = kF32 ? reinterpret_cast<const uint4 *>(static_cast<const float *>(src) + off)
                             : reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(src) + off);
#pragma unroll
      for (int u = 0; u < kVec; ++u) r[u] = s4[u];
    } else {
#pragma unroll
      for (int u = 0; u < kVec; ++u) r[u] = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  uint4 nxt[kVec];
  load(p, t, h, nxt);
  for (; q < qend; ++q) {
    // this couple's bytes; the next couple's loads are issued before the math
    uint4 cur[kVec];
#pragma unroll
    for (int u = 0; u < kVec; ++u) cur[u] = nxt[u];
    const bool live = p < P;
    const int tc = t, hcur = h;
    p += 2;
    h += 2;
    while (h >= a.Hkv) {
      h -= a.Hkv;
      ++t;
    }
    if (q + 1 < qend) load(p, t, h, nxt);
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
    for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const __half s16 = __float2half_rn(__fdiv_rn(amax, 127.f));
    const float sc = __half2float(s16);
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
    // With a normal fp16 scale (>= 2^-14), |x / s| <= 127 (1 + 2^-11), so the
    // codes need no clamp; only fp16-subnormal scales can exceed 127.  (The
    // vote is taken by the whole warp, before any lane branches.)
    const bool clamp = __any_sync(0xffffffffu, sc > 0.f && sc < 6.103515625e-05f);
    if (sc > 0.f) {
      const float inv = __frcp_rn(sc);
      auto encode4 = [&](int k4, auto clamp_c) {
        int c[4];
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
          const float2 q2 = fmul2(make_float2(x[4 * k4 + u], x[4 * k4 + u + 1]), make_float2(inv, inv));
          const float qv[2] = {q2.x, q2.y};
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            int cv = __float2int_rn(qv[v]);  // round half to even, as rint
            if (fabsf(__fsub_rn(qv[v], float(cv))) > 0.5f - 1e-4f)
              cv = __float2int_rn(__fdiv_rn(x[4 * k4 + u + v], sc));
            if (decltype(clamp_c)::value) cv = max(-127, min(127, cv));
            c[u + v] = cv;
          }
        }
        // bytes 0 of c0..c3 -> one word
        return __byte_perm(__byte_perm(c[0], c[1], 0x0040u), __byte_perm(c[2], c[3], 0x0040u), 0x5410u);
      };
      if (clamp) {
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) packed[k4] = encode4(k4, std::true_type{});
      } else {
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) packed[k4] = encode4(k4, std::false_type{});
      }
    }
    if (live && SG_BOUNDS(tc < a.N && hcur < a.Hkv && int64_t(a.pos0) + tc < a.ncache)) {
      const int64_t pos = int64_t(a.pos0) + tc;
      *reinterpret_cast<uint4 *>(cache + int64_t(hcur) * a.cache_head + pos * kD + 16 * l8) =
          make_uint4(packed[0], packed[1], packed[2], packed[3]);
      if (l8 == 0) {
        scale[int64_t(hcur) * a.scale_head + pos] = s16;
        if (!(fabsf(sc) <= 65504.f) && a.status) atomicCAS(a.status, 0, SAGE_ERR_NONFINITE);
      }
    }
  }
}

}  // namespace kvc

cudaError_t launch_cache_write(const CacheWriteArgs &a, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t nrows = 2 * int64_t(a.Hkv) * a.N;
  const int64_t want = (nrows + 7) / 8, cap = int64_t(sms) * 8;
  const int blocks = int(want < cap ? want : cap);
  // 16-byte aligned rows (fp32 rows always are) take the wide kernel
  const int64_t esz = a.f32 ? 4 : 2;
  const bool wide = ((reinterpret_cast<uintptr_t>(a.k_src) | reinterpret_cast<uintptr_t>(a.v_src)) & 15u) == 0 &&
                    (a.src_tok * esz) % 16 == 0 && (a.src_head * esz) % 16 == 0;
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
