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
// GB300 design: HBM-bound streaming.  One warp per row, four channels per
// lane (8- or 16-byte loads, 4-byte code stores: a row is one 128-byte line
// of the cache), the row maximum by warp shuffles, a grid-stride loop over
// rows ordered so that consecutive warps write consecutive cache rows.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace sg {
namespace kvc {

template <bool kF32>
__global__ void __launch_bounds__(256) cache_write_kernel(CacheWriteArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t rows_per = int64_t(a.Hkv) * a.N;  // rows of one tensor
  const int64_t nrows = 2 * rows_per;
  const int64_t step = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; row < nrows; row += step) {
    const int which = row >= rows_per ? 1 : 0;  // 0: K, 1: V
    const int64_t rr = row - which * rows_per;
    const int h = int(rr / a.N), t = int(rr - int64_t(h) * a.N);
    const int64_t src_off = int64_t(t) * a.src_tok + int64_t(h) * a.src_head + 4 * lane;
    float x[4];
    if (kF32) {
      const float4 v = *reinterpret_cast<const float4 *>(static_cast<const float *>(which ? a.v_src : a.k_src) +
                                                         src_off);
      x[0] = v.x;
      x[1] = v.y;
      x[2] = v.z;
      x[3] = v.w;
    } else {
      const uint2 w = *reinterpret_cast<const uint2 *>(
          static_cast<const __nv_bfloat16 *>(which ? a.v_src : a.k_src) + src_off);
      x[0] = __uint_as_float(w.x << 16);
      x[1] = __uint_as_float(w.x & 0xFFFF0000u);
      x[2] = __uint_as_float(w.y << 16);
      x[3] = __uint_as_float(w.y & 0xFFFF0000u);
    }
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const __half s16 = __float2half_rn(__fdiv_rn(amax, 127.f));
    const float s = __half2float(s16);
    uint32_t packed = 0;
    if (s > 0.f) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        int c = __float2int_rn(__fdiv_rn(x[u], s));
        c = c > 127 ? 127 : (c < -127 ? -127 : c);
        packed |= (uint32_t(c) & 0xFFu) << (8 * u);
      }
    }
    const int64_t pos = int64_t(a.pos0) + t;
    int8_t *cache = which ? a.v_cache : a.k_cache;
    *reinterpret_cast<uint32_t *>(cache + int64_t(h) * a.cache_head + pos * kD + 4 * lane) = packed;
    if (lane == 0) {
      __half *sc = static_cast<__half *>(which ? a.v_scale : a.k_scale);
      sc[int64_t(h) * a.scale_head + pos] = s16;
      if (!(fabsf(s) <= 65504.f) && a.status) atomicCAS(a.status, 0, SAGE_ERR_NONFINITE);
    }
  }
}

}  // namespace kvc

cudaError_t launch_cache_write(const CacheWriteArgs &a, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t nrows = 2 * int64_t(a.Hkv) * a.N;
  const int64_t want = (nrows + 7) / 8, cap = int64_t(sms) * 16;
  const int blocks = int(want < cap ? want : cap);
  if (a.f32) kvc::cache_write_kernel<true><<<blocks, 256, 0, st>>>(a);
  else kvc::cache_write_kernel<false><<<blocks, 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace sg
