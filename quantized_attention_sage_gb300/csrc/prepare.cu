// The dense path's preparation in three launches for all heads: K smoothing,
// INT8 per-block codes of Q and of the smoothed K, FP8 E4M3 per-channel
// codes of V (transposed).
//
// Pages: "H3 Performance Roadmap", section "Measured GB10 Baseline", table
// "SageAttention 2.2.0 internals" (K smoothing, Q/K INT8 quantization, V FP8
// quantization as separate steps) and section "Phase 4: Dense
// Sage-Compatible Attention", item 4 (fuse the Q/K/V preparation where it
// pays).
//
// The separate quantizers (quant.cu) take six launches and leave INT8 codes
// that the attention first turns into fp16 images (two more passes).  Here:
//   1. prep_reduce_kernel: one pass over K and V together, fp32 channel sums
//      of K and channel maxima of |V| per chunk of 256 tokens;
//   2. prep_finalize_kernel: the K mean and the V scales of every head;
//   3. prep_encode_kernel: Q blocks, K blocks and V tiles in one grid; the
//      Q/K codes go out either as int8 or directly as their exact fp16
//      images (what the attention's tensor cores read), so no image pass and
//      no int8 round trip through HBM is left.
// The arithmetic is that of quant.cu step for step (same reduction order,
// same rounding of every operation), so codes, scales and means are the same
// bits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace sg {

SG_BOUNDS_FILE(prepare, 2)

namespace prep {

// 1. channel sums of K (z = 0) or maxima of |V| (z = 1) over chunks of 256
// tokens, ascending token order.  grid (chunks, B*H, 2), 64 threads: thread
// c2 owns channels 2*c2 and 2*c2 + 1.
__global__ void __launch_bounds__(64) prep_reduce_kernel(const __nv_bfloat16 *__restrict__ k, sage_strides ks,
                                                         const __nv_bfloat16 *__restrict__ v, sage_strides vs,
                                                         int H, int N, int nchunks, float *__restrict__ part_k,
                                                         float *__restrict__ part_v) {
  const bool isv = blockIdx.z == 1;
  const int chunk = blockIdx.x, bh = blockIdx.y;
  const int b = bh / H, h = bh - b * H;
  const int c2 = threadIdx.x;
  const sage_strides s = isv ? vs : ks;
  const __nv_bfloat16 *base = (isv ? v : k) + b * s.b + h * s.h + 2 * c2;
  const int t0 = chunk * kMeanChunk;
  const int t1 = min(t0 + kMeanChunk, N);
  if (!SG_BOUNDS(chunk < nchunks && t0 < N && 2 * c2 + 1 < kD)) return;
  float a0 = 0.f, a1 = 0.f;
  auto take = [&](const __nv_bfloat162 w) {
    const float2 f = __bfloat1622float2(w);
    if (isv) {
      a0 = fmaxf(a0, fabsf(f.x));
      a1 = fmaxf(a1, fabsf(f.y));
    } else {
      a0 = __fadd_rn(a0, f.x);
      a1 = __fadd_rn(a1, f.y);
    }
  };
  int t = t0;
  // 32 rows of loads in flight per round; the additions stay in ascending order
  for (; t + 32 <= t1; t += 32) {
    __nv_bfloat162 w[32];
#pragma unroll
    for (int u = 0; u < 32; ++u) w[u] = *reinterpret_cast<const __nv_bfloat162 *>(base + int64_t(t + u) * s.n);
#pragma unroll
    for (int u = 0; u < 32; ++u) take(w[u]);
  }
  for (; t < t1; ++t) take(*reinterpret_cast<const __nv_bfloat162 *>(base + int64_t(t) * s.n));
  float *part = isv ? part_v : part_k;
  const int64_t off = (int64_t(bh) * nchunks + chunk) * kD + 2 * c2;
  if (SG_BOUNDS(off + 2 <= int64_t(gridDim.y) * nchunks * kD))
    *reinterpret_cast<float2 *>(part + off) = make_float2(a0, a1);
}

// 2. per head: K mean = (chunk sums added in ascending order) / N (y = 0);
// V scale = amax / 448 and its inverse 448 / amax (y = 1).  grid (B*H, 2),
// 128 threads (one channel each).
__global__ void __launch_bounds__(128) prep_finalize_kernel(const float *__restrict__ part_k,
                                                            const float *__restrict__ part_v, int nchunks, int N,
                                                            float *__restrict__ k_mean, float *__restrict__ v_scales,
                                                            float *__restrict__ v_inv) {
  const int bh = blockIdx.x, c = threadIdx.x;
  const bool isv = blockIdx.y == 1;
  const float *p = (isv ? part_v : part_k) + int64_t(bh) * nchunks * kD + c;
  float acc = 0.f;
  int i = 0;
  for (; i + 16 <= nchunks; i += 16) {
    float w[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) w[u] = p[int64_t(i + u) * kD];
#pragma unroll
    for (int u = 0; u < 16; ++u) acc = isv ? fmaxf(acc, w[u]) : __fadd_rn(acc, w[u]);
  }
  for (; i < nchunks; ++i) acc = isv ? fmaxf(acc, p[int64_t(i) * kD]) : __fadd_rn(acc, p[int64_t(i) * kD]);
  if (!SG_BOUNDS(c < kD && bh < int(gridDim.x))) return;
  if (isv) {
    v_scales[bh * kD + c] = __fdiv_rn(acc, 448.f);
    v_inv[bh * kD + c] = acc > 0.f ? __fdiv_rn(448.f, acc) : 0.f;
  } else {
    k_mean[bh * kD + c] = __fdiv_rn(acc, float(N));
  }
}

struct EncodeArgs {
  const __nv_bfloat16 *q, *k, *v;
  sage_strides qs, ks, vs;
  const float *k_mean, *v_inv;
  int H, Nq, Nk, Nk_pad, nbq, nbk, nvt;
  void *q_out, *k_out;  // int8 codes or fp16 images [B, H, N, 128]
  float *q_scales, *k_scales;
  uint8_t *v_codes;  // [B, H, 128, Nk_pad]
};

// One block of BLK tokens of Q (mean 0) or of K - mean: amax over the block,
// scale = fl(amax / 127), codes rint(fl(x * fl(127 / amax))) clamped to +-127,
// stored as int8 or as their exact fp16 images.  256 threads; thread t owns
// the 8-channel group (t & 15) of rows t/16, t/16 + 16, ...
template <int BLK, bool kImages>
__device__ __forceinline__ void encode_qk_block(const __nv_bfloat16 *__restrict__ src, int64_t sn, int N, int blk,
                                                const float *__restrict__ mean, float *__restrict__ scale_out,
                                                void *__restrict__ dst_base, float *red) {
  constexpr int CH = BLK * 16 / 256;  // 16-byte chunks per thread
  const int t0 = blk * BLK;
  const int nt = min(BLK, N - t0);
  const int col = (threadIdx.x & 15) * 8;
  float mu[8];
  if (mean != nullptr) {
    const float4 m0 = *reinterpret_cast<const float4 *>(mean + col);
    const float4 m1 = *reinterpret_cast<const float4 *>(mean + col + 4);
    mu[0] = m0.x, mu[1] = m0.y, mu[2] = m0.z, mu[3] = m0.w, mu[4] = m1.x, mu[5] = m1.y, mu[6] = m1.z, mu[7] = m1.w;
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) mu[j] = 0.f;
  }
  uint4 raw[CH];
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int row = (threadIdx.x >> 4) + 16 * i;
    raw[i] = (row < nt && SG_BOUNDS(t0 + row < N && col + 8 <= kD))
                 ? *reinterpret_cast<const uint4 *>(src + int64_t(t0 + row) * sn + col)
                 : make_uint4(0, 0, 0, 0);
  }
  const bool smooth = mean != nullptr;
  auto value = [&](const uint4 &w, int j) -> float {
    const uint32_t word = j < 2 ? w.x : j < 4 ? w.y : j < 6 ? w.z : w.w;
    const float f = __uint_as_float((j & 1) ? (word & 0xFFFF0000u) : (word << 16));
    return smooth ? __fsub_rn(f, mu[j]) : f;
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
  if (threadIdx.x == 0 && SG_BOUNDS(t0 < N)) scale_out[blk] = __fdiv_rn(amax, 127.f);
#pragma unroll
  for (int i = 0; i < CH; ++i) {
    const int row = (threadIdx.x >> 4) + 16 * i;
    if (row >= nt || !SG_BOUNDS(t0 + row < N && col + 8 <= kD)) continue;
    const int64_t off = int64_t(t0 + row) * kD + col;
    if (kImages) {
      // rint (ties to even, as the int8 path's conversion) and the clamp in
      // fp32; integers below 2^11 are exact in fp16
      uint32_t h[4];
#pragma unroll
      for (int j = 0; j < 8; j += 2) {
        const float r0 = fminf(fmaxf(rintf(__fmul_rn(value(raw[i], j), inv)), -127.f), 127.f);
        const float r1 = fminf(fmaxf(rintf(__fmul_rn(value(raw[i], j + 1), inv)), -127.f), 127.f);
        const __half2 p = __floats2half2_rn(r0, r1);
        h[j >> 1] = *reinterpret_cast<const uint32_t *>(&p);
      }
      *reinterpret_cast<uint4 *>(static_cast<__half *>(dst_base) + off) = make_uint4(h[0], h[1], h[2], h[3]);
    } else {
      uint32_t w[2] = {0u, 0u};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        int c = __float2int_rn(__fmul_rn(value(raw[i], j), inv));
        c = max(-127, min(127, c));
        w[j >> 2] |= (uint32_t(c) & 0xFFu) << (8 * (j & 3));
      }
      *reinterpret_cast<uint2 *>(static_cast<int8_t *>(dst_base) + off) = make_uint2(w[0], w[1]);
    }
  }
}

// One 128-token tile of V: E4M3 codes of fl(v * inv_c), transposed through
// shared memory to [128 channels][128 tokens] (the layout of quant.cu's V
// encoder: 32-bit word (channel ch, token quad) at ch*32 + (quad ^ 2*(ch/8))).
__device__ __forceinline__ void encode_v_tile(const __nv_bfloat16 *__restrict__ src, int64_t sn, int Nk, int Nk_pad,
                                              int kt, const float *__restrict__ iv, uint8_t *__restrict__ codes,
                                              uint32_t *tile) {
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
      if (tok < Nk) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(src + int64_t(tok) * sn + cg * 8);
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
    for (int j = 0; j < 8; ++j) tile[(cg * 8 + j) * 32 + (quad ^ (2 * cg))] = word[j];
  }
  __syncthreads();
  uint8_t *dst = codes + int64_t(kt) * kTile;
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

// 3. grid (nbq + nbk + nvt, B*H), 256 threads: blockIdx.x picks a Q block, a
// K block or a V tile of head blockIdx.y.  The V tiles come first (their CTAs
// read the V just reduced, most of which the reduction's last waves left in
// L2), then K, then Q.
template <int QB, int KB, bool kImages>
__global__ void __launch_bounds__(256, 4) prep_encode_kernel(const EncodeArgs a) {
  __shared__ uint32_t tile[kD * 32];
  __shared__ float red[8];
  const int bh = blockIdx.y;
  const int b = bh / a.H, h = bh - b * a.H;
  int u = blockIdx.x;
  if (u < a.nvt) {
    encode_v_tile(a.v + b * a.vs.b + h * a.vs.h, a.vs.n, a.Nk, a.Nk_pad, u, a.v_inv + bh * kD,
                  a.v_codes + int64_t(bh) * kD * a.Nk_pad, tile);
    return;
  }
  u -= a.nvt;
  const size_t esize = kImages ? 2 : 1;
  if (u < a.nbk) {
    void *dst = static_cast<uint8_t *>(a.k_out) + int64_t(bh) * a.Nk * kD * esize;
    encode_qk_block<KB, kImages>(a.k + b * a.ks.b + h * a.ks.h, a.ks.n, a.Nk, u, a.k_mean + bh * kD,
                                 a.k_scales + bh * a.nbk, dst, red);
    return;
  }
  u -= a.nbk;
  void *dst = static_cast<uint8_t *>(a.q_out) + int64_t(bh) * a.Nq * kD * esize;
  encode_qk_block<QB, kImages>(a.q + b * a.qs.b + h * a.qs.h, a.qs.n, a.Nq, u, nullptr, a.q_scales + bh * a.nbq, dst,
                               red);
}

template <bool kImages>
void launch_encode(const EncodeArgs &a, int qb, int kb, dim3 grid, cudaStream_t st) {
  if (qb == 64 && kb == 64) prep_encode_kernel<64, 64, kImages><<<grid, 256, 0, st>>>(a);
  else if (qb == 64) prep_encode_kernel<64, 128, kImages><<<grid, 256, 0, st>>>(a);
  else if (kb == 64) prep_encode_kernel<128, 64, kImages><<<grid, 256, 0, st>>>(a);
  else prep_encode_kernel<128, 128, kImages><<<grid, 256, 0, st>>>(a);
}

}  // namespace prep

size_t prepare_workspace_bytes(int B, int H, int Nk) {
  const size_t BH = size_t(B) * H, nch = size_t(ceil_div(Nk, kMeanChunk));
  return (2 * BH * nch * kD + BH * kD) * sizeof(float) + 16;
}

cudaError_t launch_prepare(const PrepArgs &a, cudaStream_t st) {
  using namespace prep;
  const int BH = a.B * a.H;
  const int nch = ceil_div(a.Nk, kMeanChunk);
  float *part_k = a.workspace;
  float *part_v = part_k + size_t(BH) * nch * kD;
  float *v_inv = part_v + size_t(BH) * nch * kD;
  const auto *k = static_cast<const __nv_bfloat16 *>(a.k);
  const auto *v = static_cast<const __nv_bfloat16 *>(a.v);
  prep_reduce_kernel<<<dim3(nch, BH, 2), 64, 0, st>>>(k, a.ks, v, a.vs, a.H, a.Nk, nch, part_k, part_v);
  prep_finalize_kernel<<<dim3(BH, 2), 128, 0, st>>>(part_k, part_v, nch, a.Nk, a.k_mean, a.v_scales, v_inv);
  EncodeArgs e;
  e.q = static_cast<const __nv_bfloat16 *>(a.q);
  e.k = k;
  e.v = v;
  e.qs = a.qs;
  e.ks = a.ks;
  e.vs = a.vs;
  e.k_mean = a.k_mean;
  e.v_inv = v_inv;
  e.H = a.H;
  e.Nq = a.Nq;
  e.Nk = a.Nk;
  e.Nk_pad = nk_pad(a.Nk);
  e.nbq = ceil_div(a.Nq, a.q_block);
  e.nbk = ceil_div(a.Nk, a.k_block);
  e.nvt = e.Nk_pad / kTile;
  e.q_out = a.q_out;
  e.k_out = a.k_out;
  e.q_scales = a.q_scales;
  e.k_scales = a.k_scales;
  e.v_codes = a.v_codes;
  const dim3 grid(e.nvt + e.nbk + e.nbq, BH);
  if (a.images) launch_encode<true>(e, a.q_block, a.k_block, grid, st);
  else launch_encode<false>(e, a.q_block, a.k_block, grid, st);
  return cudaGetLastError();
}

}  // namespace sg
