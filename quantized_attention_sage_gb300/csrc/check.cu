// Check hook: the number-format conversions of the kernels, applied to
// arbitrary fp32 inputs, so that tests can compare them bit for bit with
// independent encoders over dense sweeps of fp32 bit patterns and every
// rounding midpoint.  Each line below is the conversion a kernel uses:
//   E4M3   cvt.rn.satfinite.e4m3x2.f32     (V codes, P in the dense softmax)
//   int8   __float2int_rn, clamped to +-127 (Q/K codes, int8 cache codes)
//   bf16   __floats2bfloat162_rn           (attention outputs)
//   fp16   __float2half_rn                 (int8 cache scales)
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace sg {

SG_BOUNDS_FILE(check, 6)

__global__ void __launch_bounds__(256) conversion_check_kernel(const float *__restrict__ x, int64_t npairs,
                                                               uint8_t *__restrict__ e4m3, int8_t *__restrict__ i8,
                                                               uint16_t *__restrict__ bf16,
                                                               uint16_t *__restrict__ f16) {
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < npairs; i += int64_t(gridDim.x) * blockDim.x) {
    const float2 v = reinterpret_cast<const float2 *>(x)[i];
    const uint32_t e = cvt_e4m3x2(v.x, v.y);
    reinterpret_cast<uint16_t *>(e4m3)[i] = uint16_t(e);
    const int a = max(-127, min(127, __float2int_rn(v.x)));
    const int b = max(-127, min(127, __float2int_rn(v.y)));
    reinterpret_cast<uint16_t *>(i8)[i] = uint16_t((uint32_t(a) & 0xFFu) | ((uint32_t(b) & 0xFFu) << 8));
    const __nv_bfloat162 h2 = __floats2bfloat162_rn(v.x, v.y);
    reinterpret_cast<uint32_t *>(bf16)[i] = *reinterpret_cast<const uint32_t *>(&h2);
    const __half lo = __float2half_rn(v.x), hi = __float2half_rn(v.y);
    reinterpret_cast<uint32_t *>(f16)[i] =
        uint32_t(__half_as_ushort(lo)) | (uint32_t(__half_as_ushort(hi)) << 16);
  }
}

cudaError_t launch_conversion_check(const float *x, int64_t n, uint8_t *e4m3, int8_t *i8, uint16_t *bf16,
                                    uint16_t *f16, cudaStream_t st) {
  const int64_t npairs = n / 2;
  const int64_t want = (npairs + 255) / 256, cap = int64_t(current_sm_count()) * 16;
  int blocks = int(want < cap ? want : cap);
  if (blocks < 1) blocks = 1;
  conversion_check_kernel<<<blocks, 256, 0, st>>>(x, npairs, e4m3, i8, bf16, f16);
  return cudaGetLastError();
}

}  // namespace sg
