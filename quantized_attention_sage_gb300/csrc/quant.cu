// Quantisers of the dense path: K smoothing mean, INT8 per-block Q/K codes,
// FP8 E4M3 per-channel V codes written transposed.
//
// Pages: "H3 Performance Roadmap", section "Measured GB10 Baseline", table
// "SageAttention 2.2.0 internals" (Q/K INT8 quantization, V FP8 quantization,
// K smoothing) and section "Phase 4: Dense Sage-Compatible Attention".
//
// All three are HBM-bound streams: 16-byte (or 4-byte bf16x2) coalesced loads,
// one pass per tensor, fp32 arithmetic with explicitly rounded operations so
// the codes are bit-identical to the fp32 program they implement.
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace sg {

SG_BOUNDS_FILE(quant, 1)

// -------------------------------------------------------------------------
// K1: channel sums of K over chunks of 256 tokens, ascending token order.
// (Also serves V: with kMax it takes channel maxima of |V| instead.)
// grid (chunks, B*H), 64 threads: thread c2 owns channels 2*c2, 2*c2+1.
// -------------------------------------------------------------------------
template <bool kMax>
__global__ void __launch_bounds__(64) chunk_reduce_kernel(const __nv_bfloat16 *__restrict__ x, int64_t sb,
                                                          int64_t sh, int64_t sn, int H, int N, int nchunks,
                                                          float *__restrict__ partial) {
  const int chunk = blockIdx.x, bh = blockIdx.y;
  const int b = bh / H, h = bh - b * H;
  const int c2 = threadIdx.x;
  const __nv_bfloat16 *base = x + b * sb + h * sh + 2 * c2;
  const int t0 = chunk * kMeanChunk;
  const int t1 = min(t0 + kMeanChunk, N);
  if (!SG_BOUNDS(chunk < nchunks && t0 < N && 2 * c2 + 1 < kD)) return;
  float a0 = 0.f, a1 = 0.f;
  int t = t0;
  // 32 rows of loads in flight per round (the additions stay in ascending
  // token order): with few heads each chunk's CTA is alone on its SM and the
  // chunk time is the number of memory round trips
  for (; t + 32 <= t1; t += 32) {
    __nv_bfloat162 v[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) v[u] = *reinterpret_cast<const __nv_bfloat162 *>(base + int64_t(t + u) * sn);
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const float2 f = __bfloat1622float2(v[u]);
      if (kMax) {
        a0 = fmaxf(a0, fabsf(f.x));
        a1 = fmaxf(a1, fabsf(f.y));
      } else {
        a0 = __fadd_rn(a0, f.x);
        a1 = __fadd_rn(a1, f.y);
      }
    }
  }
  for (; t < t1; ++t) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(base + int64_t(t) * sn));
    if (kMax) {
      a0 = fmaxf(a0, fabsf(f.x));
      a1 = fmaxf(a1, fabsf(f.y));
    } else {
      a0 = __fadd_rn(a0, f.x);
      a1 = __fadd_rn(a1, f.y);
    }
  }
  const int64_t off = (int64_t(bh) * nchunks + chunk) * kD + 2 * c2;
  if (SG_BOUNDS(off + 2 <= int64_t(gridDim.y) * nchunks * kD))
    *reinterpret_cast<float2 *>(partial + off) = make_float2(a0, a1);
}

// K1b: mean = (chunk sums added in ascending order) / Nk.  grid B*H, 128 threads.
__global__ void __launch_bounds__(128) k_mean_finalize_kernel(const float *__restrict__ partial, int nchunks,
                                                              int Nk, float *__restrict__ mean) {
  const int bh = blockIdx.x, c = threadIdx.x;
  const float *p = partial + int64_t(bh) * nchunks * kD + c;
  float tot = 0.f;
  int i = 0;
  // 16 partials loaded per round, added in ascending chunk order
  for (; i + 16 <= nchunks; i += 16) {
    float v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) v[u] = p[int64_t(i + u) * kD];
#pragma unroll
    for (int u = 0; u < 16; ++u) tot = __fadd_rn(tot, v[u]);
  }
  for (; i < nchunks; ++i) tot = __fadd_rn(tot, p[int64_t(i) * kD]);
  if (SG_BOUNDS(c < kD && bh < int(gridDim.x))) mean[bh * kD + c] = __fdiv_rn(tot, float(Nk));
}

// -------------------------------------------------------------------------
// K2: INT8 per-block codes of Q and of K - mean.  grid (nbq + nbk, B*H),
// 256 threads, one block of BLK tokens per CTA, 16-byte loads and 8-byte
// stores, block-wide amax in shared memory.
// -------------------------------------------------------------------------
struct QKQuantArgs {
  const __nv_bfloat16 *q, *k;
  sage_strides qs, ks;
  const float *mean;
  int H, Nq, Nk, nbq, nbk;
  int8_t *q_codes, *k_codes;
  float *q_scales, *k_scales;
};

template <int BLK>
__global__ void __launch_bounds__(256, 4) quant_qk_kernel(const QKQuantArgs a) {
  constexpr int CH = BLK * 16 / 256;  // 16-byte chunks per thread
  __shared__ float red[8];
  const bool isk = int(blockIdx.x) >= a.nbq;
  const int blk = isk ? blockIdx.x - a.nbq : blockIdx.x;
  const int bh = blockIdx.y;
  const int b = bh / a.H, h = bh - b * a.H;
  const int N = isk ? a.Nk : a.Nq;
  const sage_strides s = isk ? a.ks : a.qs;
  const __nv_bfloat16 *src = (isk ? a.k : a.q) + b * s.b + h * s.h;
  const int t0 = blk * BLK;
  const int nt = min(BLK, N - t0);
  // every thread owns one 8-channel column group: col = (tid & 15) * 8
  const int col = (threadIdx.x & 15) * 8;
  float mu[8];
  if (isk) {
    const float4 m0 = *reinterpret_cast<const float4 *>(a.mean + bh * kD + col);
    const float4 m1 = *reinterpret_cast<const float4 *>(a.mean + bh * kD + col + 4);
    mu[0] = m0.x, mu[1] = m0.y, mu[2] = m0.z, mu[3] = m0.w, mu[4] = m1.x, mu[5] = m1.y, mu[6] = m1.z, mu[7] = m1.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) mu[j] = 0.f;
  }
  // raw bf16 chunks stay packed in registers; both passes convert on the fly
  uint4 raw[CH];
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int row = (threadIdx.x >> 4) + 16 * i;
    raw[i] = (row < nt && SG_BOUNDS(t0 + row < N && col + 8 <= kD))
                 ? *reinterpret_cast<const uint4 *>(src + int64_t(t0 + row) * s.n + col)
                 : make_uint4(0u, 0u, 0u, 0u);
  }
  auto value = [&](const uint4 &w, int j) -> float {
    const uint32_t word = j < 2 ? w.x : j < 4 ? w.y : j < 6 ? w.z : w.w;
    const float f = __uint_as_float((j & 1) ? (word & 0xFFFF0000u) : (word << 16));
    return isk ? __fsub_rn(f, mu[j]) : f;
  };
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int row = (threadIdx.x >> 4) + 16 * i;
    if (row < nt) {
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(value(raw[i], j)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);

  const float inv = amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f;
  if (threadIdx.x == 0) {
    float *scales = isk ? a.k_scales : a.q_scales;
    if (SG_BOUNDS(blk < (isk ? a.nbk : a.nbq) && t0 < N))
      scales[bh * (isk ? a.nbk : a.nbq) + blk] = __fdiv_rn(amax, 127.f);
  }
  int8_t *dst = (isk ? a.k_codes : a.q_codes) + (int64_t(bh) * N + t0) * kD;
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int row = (threadIdx.x >> 4) + 16 * i;
    if (row < nt) {
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        int c = __float2int_rn(__fmul_rn(value(raw[i], j), inv));
        c = max(-127, min(127, c));
        w[j >> 2] |= (uint32_t(c) & 0xFFu) << (8 * (j & 3));
      }
      if (SG_BOUNDS(t0 + row < N && col + 8 <= kD))
        *reinterpret_cast<uint2 *>(dst + int64_t(row) * kD + col) = make_uint2(w[0], w[1]);
    }
  }
}

// -------------------------------------------------------------------------
// K3b: V scales from the chunk maxima.  grid B*H, 128 threads.
// -------------------------------------------------------------------------
__global__ void __launch_bounds__(128) v_finalize_kernel(const float *__restrict__ partial, int nchunks,
                                                         float *__restrict__ v_scales, float *__restrict__ inv) {
  const int bh = blockIdx.x, c = threadIdx.x;
  const float *p = partial + int64_t(bh) * nchunks * kD + c;
  float amax = 0.f;
  int i = 0;
  for (; i + 16 <= nchunks; i += 16) {
    float v[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) v[u] = p[int64_t(i + u) * kD];
#pragma unroll
    for (int u = 0; u < 16; ++u) amax = fmaxf(amax, v[u]);
  }
  for (; i < nchunks; ++i) amax = fmaxf(amax, p[int64_t(i) * kD]);
  if (SG_BOUNDS(c < kD && bh < int(gridDim.x))) {
    v_scales[bh * kD + c] = __fdiv_rn(amax, 448.f);
    inv[bh * kD + c] = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
  }
}

// -------------------------------------------------------------------------
// K3c: E4M3 codes of one 128-token tile, transposed through shared memory to
// [128 channels][128 tokens].  grid (Nk_pad/128, B*H), 256 threads.
// Shared layout: 32-bit word (channel ch, token quad) at
// ch*32 + (quad ^ 2*(ch/8)), which keeps the 16 channel groups of a warp's
// stores in distinct banks.
// -------------------------------------------------------------------------
__global__ void __launch_bounds__(256) v_encode_kernel(const __nv_bfloat16 *__restrict__ v, sage_strides vs,
                                                       int H, int Nk, int Nk_pad, const float *__restrict__ inv,
                                                       uint8_t *__restrict__ codes) {
  __shared__ uint32_t tile[kD * 32];
  const int kt = blockIdx.x, bh = blockIdx.y;
  const int b = bh / H, h = bh - b * H;
  const __nv_bfloat16 *src = v + b * vs.b + h * vs.h;
  const float *iv = inv + bh * kD;
#pragma unroll
  for (int rep = 0; rep < 2; ++rep) {
    const int p = threadIdx.x + 256 * rep;
    const int cg = p & 15, quad = p >> 4;
    float sc[8];
    {
      const float4 i0 = *reinterpret_cast<const float4 *>(iv + cg * 8);
      const float4 i1 = *reinterpret_cast<const float4 *>(iv + cg * 8 + 4);
      sc[0] = i0.x, sc[1] = i0.y, sc[2] = i0.z, sc[3] = i0.w;
      sc[4] = i1.x, sc[5] = i1.y, sc[6] = i1.z, sc[7] = i1.w;
    }
    uint32_t word[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int tok = kt * kTile + quad * 4 + r;
      if (tok < Nk && SG_BOUNDS(cg * 8 + 8 <= kD)) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(src + int64_t(tok) * vs.n + cg * 8);
        const __nv_bfloat162 *v2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(v2[j]);
          const uint32_t pr = cvt_e4m3x2(__fmul_rn(f.x, sc[2 * j]), __fmul_rn(f.y, sc[2 * j + 1]));
          word[2 * j] |= (pr & 0xFFu) << (8 * r);
          word[2 * j + 1] |= ((pr >> 8) & 0xFFu) << (8 * r);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int ch = cg * 8 + j;
      tile[ch * 32 + (quad ^ (2 * cg))] = word[j];
    }
  }
  __syncthreads();
  uint8_t *dst = codes + int64_t(bh) * kD * Nk_pad + int64_t(kt) * kTile;
#pragma unroll
  for (int rep = 0; rep < 4; ++rep) {
    const int p = threadIdx.x + 256 * rep;
    const int ch = p >> 3, k16 = p & 7;
    const int sw = 2 * (ch >> 3);
    uint4 o;
    o.x = tile[ch * 32 + ((4 * k16 + 0) ^ sw)];
    o.y = tile[ch * 32 + ((4 * k16 + 1) ^ sw)];
    o.z = tile[ch * 32 + ((4 * k16 + 2) ^ sw)];
    o.w = tile[ch * 32 + ((4 * k16 + 3) ^ sw)];
    if (SG_BOUNDS(ch < kD && kt * kTile + k16 * 16 + 16 <= Nk_pad))
      *reinterpret_cast<uint4 *>(dst + int64_t(ch) * Nk_pad + k16 * 16) = o;
  }
}

// -------------------------------------------------------------------------
// host launchers
// -------------------------------------------------------------------------
cudaError_t launch_quantize_qk(const void *q, sage_strides qs, const void *k, sage_strides ks, int B, int H,
                               int Nq, int Nk, int q_block, int k_block, int8_t *q_codes, float *q_scales,
                               int8_t *k_codes, float *k_scales, float *k_mean, float *partial,
                               cudaStream_t st) {
  const int nchunks = ceil_div(Nk, kMeanChunk);
  const auto *kk = static_cast<const __nv_bfloat16 *>(k);
  chunk_reduce_kernel<false><<<dim3(nchunks, B * H), 64, 0, st>>>(kk, ks.b, ks.h, ks.n, H, Nk, nchunks, partial);
  k_mean_finalize_kernel<<<B * H, 128, 0, st>>>(partial, nchunks, Nk, k_mean);
  QKQuantArgs a;
  a.q = static_cast<const __nv_bfloat16 *>(q);
  a.k = kk;
  a.qs = qs;
  a.ks = ks;
  a.mean = k_mean;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.nbq = ceil_div(Nq, q_block);
  a.nbk = ceil_div(Nk, k_block);
  a.q_codes = q_codes;
  a.k_codes = k_codes;
  a.q_scales = q_scales;
  a.k_scales = k_scales;
  // Q and K blocks of the same size share one launch; otherwise two.
  if (q_block == k_block) {
    dim3 grid(a.nbq + a.nbk, B * H);
    if (q_block == 64) quant_qk_kernel<64><<<grid, 256, 0, st>>>(a);
    else quant_qk_kernel<128><<<grid, 256, 0, st>>>(a);
  } else {
    QKQuantArgs aq = a, ak = a;
    aq.nbk = 0;  // grid covers Q blocks only
    ak.nbq = 0;
    ak.nbk = a.nbk;
    // Q-only launch: blocks [0, nbq); K-only launch: blocks [nbq', ...) with nbq' = 0
    if (q_block == 64) quant_qk_kernel<64><<<dim3(a.nbq, B * H), 256, 0, st>>>(aq);
    else quant_qk_kernel<128><<<dim3(a.nbq, B * H), 256, 0, st>>>(aq);
    if (k_block == 64) quant_qk_kernel<64><<<dim3(a.nbk, B * H), 256, 0, st>>>(ak);
    else quant_qk_kernel<128><<<dim3(a.nbk, B * H), 256, 0, st>>>(ak);
  }
  return cudaGetLastError();
}

cudaError_t launch_quantize_v(const void *v, sage_strides vs, int B, int H, int Nk, uint8_t *v_codes,
                              float *v_scales, float *partial, float *inv, cudaStream_t st) {
  const int nchunks = ceil_div(Nk, kMeanChunk);
  const auto *vv = static_cast<const __nv_bfloat16 *>(v);
  chunk_reduce_kernel<true><<<dim3(nchunks, B * H), 64, 0, st>>>(vv, vs.b, vs.h, vs.n, H, Nk, nchunks, partial);
  v_finalize_kernel<<<B * H, 128, 0, st>>>(partial, nchunks, v_scales, inv);
  const int npad = nk_pad(Nk);
  v_encode_kernel<<<dim3(npad / kTile, B * H), 256, 0, st>>>(vv, vs, H, Nk, npad, inv, v_codes);
  return cudaGetLastError();
}

// -------------------------------------------------------------------------
// Allocation-free variant of sage_quantize_qk.  Its K-mean chunk partials
// live in this fixed device array instead of a caller workspace; every GPU
// that loads the library holds it until the process exits.
// -------------------------------------------------------------------------
static __device__ __align__(256) float g_qk_scratch[kNoAllocScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;

// Device address of g_qk_scratch on the current device, looked up with
// cudaGetSymbolAddress (that device current) once per device context: the
// first call on a device, and again when the device's context is no longer
// the one the address was taken in (after cudaDeviceReset the module is
// loaded anew, possibly elsewhere).  In host code the array's name is only a
// host-side stand-in, never a device address.
static cudaError_t noalloc_scratch(float **out) {
  static std::mutex mu;
  static float *ptrs[kMaxDevices] = {};
  static unsigned long long ctxs[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();
  if (ptrs[dev] == nullptr || ctx == 0 || ctx != ctxs[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_qk_scratch);
    if (e != cudaSuccess) return e;
    ptrs[dev] = static_cast<float *>(p);
    ctxs[dev] = current_context_id();  // the lookup made the context current
  }
  *out = ptrs[dev];
  return cudaSuccess;
}

cudaError_t launch_quantize_qk_noalloc(const void *q, sage_strides qs, const void *k, sage_strides ks, int B,
                                       int H, int Nq, int Nk, int q_block, int k_block, int8_t *q_codes,
                                       float *q_scales, int8_t *k_codes, float *k_scales, float *k_mean,
                                       cudaStream_t st) {
  float *scratch = nullptr;
  cudaError_t e = noalloc_scratch(&scratch);
  if (e != cudaSuccess) return e;
  return launch_quantize_qk(q, qs, k, ks, B, H, Nq, Nk, q_block, k_block, q_codes, q_scales, k_codes, k_scales,
                            k_mean, scratch, st);
}

}  // namespace sg
