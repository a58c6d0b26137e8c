// Rate probes for the roofline: how many MACs per clock one SM's tensor core
// completes for the two MMA shapes the dense attention issues, and how many
// ex2 per clock its MUFU units complete.  One CTA per SM; each CTA counts its
// own SM clock cycles (clock64) around a fixed amount of work and writes them
// to cycles[blockIdx.x].  The operands are pseudo-random finite values in
// shared memory (zeros would understate the power draw).
//   kind 0: tcgen05.mma kind::f16, M128 N128 K16, A and B from shared memory,
//           8 K-steps per iteration (a 128 x 128 x 128 block), fp32 in TMEM;
//   kind 1: tcgen05.mma kind::f8f6f4 (E4M3), M128 N128 K32, 4 K-steps per
//           iteration (the same block);
//   kind 2: ex2.approx.ftz.f32 on all 384 threads, 8 independent chains per
//           thread, 64 per chain per iteration.
#include "internal.h"
#include "ptx.cuh"

namespace sg {

namespace {

constexpr int kProbeThreads = 384;
constexpr uint32_t kProbeSmem = 64 * 1024 + 1024;

__global__ void __launch_bounds__(kProbeThreads, 1) rate_probe_kernel(int kind, int iters, unsigned long long *cycles,
                                                                      float *sink, int32_t *status) {
  extern __shared__ uint8_t raw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar;
  __shared__ uint32_t tbase;
  __shared__ int abort_flag;
  // pseudo-random operands: fp16 pairs in [-64, 64] (exponent field 16..21)
  // whose bytes, read as E4M3, are finite as well (bit 7 of every byte clear
  // of the all-ones pattern by masking with 0x7E)
  for (int i = threadIdx.x; i < 64 * 1024 / 16; i += blockDim.x) {
    uint32_t h = uint32_t(i) * 2654435761u + 12345u + blockIdx.x;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      h ^= h >> 13;
      h *= 0x5bd1e995u;
      h ^= h >> 15;
      const uint32_t lo = (h & 0x83FFu) | ((0x10u + (h >> 10) % 6u) << 10);
      const uint32_t hi = ((h >> 16) & 0x83FFu) | ((0x10u + (h >> 26) % 6u) << 10);
      w[q] = (lo | (hi << 16)) & 0x7E7E7E7Eu;
    }
    reinterpret_cast<uint4 *>(sm)[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  fence_proxy_async_smem();
  if (threadIdx.x < 32) {
    tmem_alloc(&tbase, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tm = tbase;
  if (kind == 2) {
    float x[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = -0.001f * float(threadIdx.x + c);
    __syncthreads();
    const unsigned long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int r = 0; r < 64; ++r) {
#pragma unroll
        for (int c = 0; c < 8; ++c) x[c] = ex2(x[c]) - 1.0f;
      }
    }
    __syncthreads();
    const unsigned long long t1 = clock64();
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) s += x[c];
    if (s == 12345.f) sink[0] = s;  // keeps the chains alive
  } else if (threadIdx.x == 0) {
    const uint32_t a = smem_u32(sm), b = smem_u32(sm + 32768);
    const unsigned long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
      const uint32_t d = tm + uint32_t(it & 1) * 128;
      if (kind == 0) {
        constexpr uint32_t id = make_idesc(kFmtF32, kFmtF16, kFmtF16, 128, 128);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          umma_f16(d, sdesc_sw128(a + (k >> 2) * 16384 + (k & 3) * 32), sdesc_sw128(b + (k >> 2) * 16384 + (k & 3) * 32),
                   id, k > 0);
      } else {
        constexpr uint32_t id = make_idesc(kFmtF32, kFmtE4M3, kFmtE4M3, 128, 128);
#pragma unroll
        for (int k = 0; k < 4; ++k) umma_f8f6f4(d, sdesc_sw128(a + k * 32), sdesc_sw128(b + k * 32), id, k > 0);
      }
    }
    tc_commit(&bar);
    // the chain completes by itself; the wait is bounded all the same
    if (!mbar_drain(&bar, 0)) atomicCAS(status, 0, SAGE_ERR_TIMEOUT);
    const unsigned long long t1 = clock64();
    cycles[blockIdx.x] = t1 - t0;
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x < 32) {
    tc_fence_after();
    tmem_dealloc(tm, 512);
  }
}

}  // namespace

cudaError_t launch_rate_probe(int kind, int iters, unsigned long long *cycles, float *sink, int32_t *status,
                              cudaStream_t st) {
  static CtxOnce attr_done;
  cudaError_t e = set_smem_attr_once(reinterpret_cast<const void *>(rate_probe_kernel), kProbeSmem, &attr_done);
  if (e != cudaSuccess) return e;
  rate_probe_kernel<<<current_sm_count(), kProbeThreads, kProbeSmem, st>>>(kind, iters, cycles, sink, status);
  return cudaGetLastError();
}

}  // namespace sg
