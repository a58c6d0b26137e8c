// Dense quantized attention forward (SageAttention-2 style) for sm_103a.
//
// Pages: "Sage2 SM89 Temporal Pair Experiment", section "Candidate" (per KV
// tile: QK -> online-softmax update of m, d, O -> denominator from the fp32
// scores -> scores to FP8 -> PV; V scale in the epilogue), and "H3
// Performance Roadmap", section "Phase 4: Dense Sage-Compatible Attention".
//
// GB300 design (not the pages' SM89 warp-register schedule):
//  * Q.K^T runs on tcgen05.mma kind::f16 over exact fp16 images of the INT8
//    codes (sm_103a has no kind::i8).  Every product is an integer below 2^14
//    and every 128-term sum is below 2^21, so the fp32 accumulator holds the
//    exact int32 dot product.
//  * P.V runs on tcgen05.mma kind::f8f6f4 (E4M3 x E4M3, fp32 accumulate in
//    TMEM).
//  * Q, K (fp16 images) and V^T (E4M3) tiles arrive by TMA into 128-byte
//    swizzled shared memory; S (double-buffered) and O live in TMEM.
//  * Warp roles: warp 0 issues TMA, warp 1 issues MMAs and owns TMEM, warps
//    4-7 own one query row per thread (TMEM lane = row): softmax, the O
//    rescale in TMEM when the row maximum grows, and the epilogue.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace sg {
namespace dense {

constexpr int BM = 128, BN = 128, NS = 3;
constexpr int kThreads = 256;
constexpr uint32_t kQBytes = BM * kD * 2;    // 32 KB fp16
constexpr uint32_t kKBytes = BN * kD * 2;    // 32 KB fp16
constexpr uint32_t kVBytes = kD * BN;        // 16 KB e4m3
constexpr uint32_t kPBytes = BM * BN;        // 16 KB e4m3
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffV = kOffK + NS * kKBytes;
constexpr uint32_t kOffP = kOffV + NS * kVBytes;
constexpr uint32_t kOffBar = kOffP + 2 * kPBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // barriers + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;

constexpr uint32_t kIdescQK = make_idesc(kFmtF32, kFmtF16, kFmtF16, BM, BN);
constexpr uint32_t kIdescPV = make_idesc(kFmtF32, kFmtE4M3, kFmtE4M3, BM, kD);

struct Params {
  const float *q_scales, *k_scales, *v_scales;
  int H, Nq, Nk, q_block, k_block, nbq, nbk;
  float C;  // fl(sm_scale * log2 e)
  __nv_bfloat16 *out;
  sage_strides os;
  int32_t *status;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[NS], k_empty[NS], v_full[NS], v_empty[NS];
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

__device__ __forceinline__ void report(int32_t *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__global__ void __launch_bounds__(kThreads, 1)
    sage_attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars *bars = reinterpret_cast<Bars *>(smem + kOffBar);
  volatile int *abort = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x, bh = blockIdx.y;
  const int q0 = qt * BM;
  const int T = ceil_div(p.Nk, BN);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b], 4);
    }
    mbar_init(&bars->pv_done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      uint8_t *sQ = smem + kOffQ;
      mbar_arrive_expect_tx(&bars->q_full, kQBytes);
      tma_load_3d(sQ, &tmQ, &bars->q_full, 0, q0, bh);
      tma_load_3d(sQ + kQBytes / 2, &tmQ, &bars->q_full, 64, q0, bh);
      auto load_k = [&](int j) -> bool {
        const int s = j % NS;
        if (j >= NS && !mbar_wait(&bars->k_empty[s], ((j / NS) + 1) & 1, abort)) return false;
        uint8_t *dst = smem + kOffK + s * kKBytes;
        mbar_arrive_expect_tx(&bars->k_full[s], kKBytes);
        tma_load_3d(dst, &tmK, &bars->k_full[s], 0, j * BN, bh);
        tma_load_3d(dst + kKBytes / 2, &tmK, &bars->k_full[s], 64, j * BN, bh);
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = j % NS;
        if (j >= NS && !mbar_wait(&bars->v_empty[s], ((j / NS) + 1) & 1, abort)) return false;
        mbar_arrive_expect_tx(&bars->v_full[s], kVBytes);
        tma_load_3d(smem + kOffV + s * kVBytes, &tmV, &bars->v_full[s], j * BN, 0, bh);
        return true;
      };
      bool ok = load_k(0);
      for (int j = 0; ok && j < T; ++j) {
        if (j + 1 < T) ok = load_k(j + 1);
        if (ok) ok = load_v(j);
      }
      if (!ok) report(p.status, SAGE_ERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sQ = smem_u32(smem + kOffQ);
      auto issue_qk = [&](int j) -> bool {
        const int s = j % NS;
        if (!mbar_wait(&bars->k_full[s], (j / NS) & 1, abort)) return false;
        tc_fence_after();
        const uint32_t sK = smem_u32(smem + kOffK + s * kKBytes);
        const uint32_t dS = tmem + ((j & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {
          const uint32_t off = (k >> 2) * (kQBytes / 2) + (k & 3) * 32;
          umma_f16(dS, sdesc_sw128(sQ + off), sdesc_sw128(sK + off), kIdescQK, k > 0);
        }
        tc_commit(&bars->s_full[j & 1]);
        tc_commit(&bars->k_empty[s]);
        return true;
      };
      bool ok = mbar_wait(&bars->q_full, 0, abort) && issue_qk(0);
      for (int j = 0; ok && j < T; ++j) {
        if (j + 1 < T) ok = issue_qk(j + 1);
        if (!ok) break;
        const int s = j % NS;
        ok = mbar_wait(&bars->p_full[j & 1], (j >> 1) & 1, abort) && mbar_wait(&bars->v_full[s], (j / NS) & 1, abort);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sP = smem_u32(smem + kOffP + (j & 1) * kPBytes);
        const uint32_t sV = smem_u32(smem + kOffV + s * kVBytes);
#pragma unroll
        for (int k = 0; k < BN / 32; ++k)
          umma_f8f6f4(tmem + kColO, sdesc_sw128(sP + k * 32), sdesc_sw128(sV + k * 32), kIdescPV, (j > 0) || (k > 0));
        tc_commit(&bars->v_empty[s]);
        tc_commit(&bars->pv_done);
      }
      if (!ok) report(p.status, SAGE_ERR_TIMEOUT);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / correction / epilogue
    const int r = (warp - 4) * 32 + lane;  // query row in the tile == TMEM lane
    const int row = q0 + r;
    const bool valid = row < p.Nq;
    const uint32_t lane_base = tmem + (uint32_t((warp & 3) * 32) << 16);
    const float sq = valid ? p.q_scales[bh * p.nbq + row / p.q_block] : 0.f;
    const float *sk = p.k_scales + bh * p.nbk;
    float m = -INFINITY, l = 0.f;
    uint8_t *sPbase = smem + kOffP + r * 128;
    const uint32_t sw = r & 7;
    bool ok = true;
    for (int j = 0; j < T; ++j) {
      ok = mbar_wait(&bars->s_full[j & 1], (j >> 1) & 1, abort);
      if (!ok) break;
      tc_fence_after();
      uint32_t S[128];
      {
        const uint32_t a = lane_base + ((j & 1) ? kColS1 : kColS0);
        tmem_ld32(a + 0, *reinterpret_cast<uint32_t(*)[32]>(&S[0]));
        tmem_ld32(a + 32, *reinterpret_cast<uint32_t(*)[32]>(&S[32]));
        tmem_ld32(a + 64, *reinterpret_cast<uint32_t(*)[32]>(&S[64]));
        tmem_ld32(a + 96, *reinterpret_cast<uint32_t(*)[32]>(&S[96]));
        tmem_ld_wait();
      }
      // dequantisation multipliers: t = fl(fl(sq * sk) * C) per key block
      float t_lo, t_hi;
      if (p.k_block == 128) {
        t_lo = t_hi = __fmul_rn(__fmul_rn(sq, sk[j]), p.C);
      } else {
        t_lo = __fmul_rn(__fmul_rn(sq, sk[2 * j]), p.C);
        t_hi = (2 * j + 1 < p.nbk) ? __fmul_rn(__fmul_rn(sq, sk[2 * j + 1]), p.C) : 0.f;
      }
      const int nvalid = min(BN, p.Nk - j * BN);
      float s[128];
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < 128; ++i) {
        float v = __fmul_rn(__uint_as_float(S[i]), i < 64 ? t_lo : t_hi);
        if (i >= nvalid) v = -INFINITY;
        s[i] = v;
        mt = fmaxf(mt, v);
      }
      const float mnew = fmaxf(m, mt);
      const float alpha = (m == -INFINITY) ? 0.f : ex2(__fsub_rn(m, mnew));
      float rowsum = 0.f;
      uint32_t pk[32];
#pragma unroll
      for (int i = 0; i < 128; i += 4) {
        const float p0 = ex2(__fsub_rn(s[i], mnew));
        const float p1 = ex2(__fsub_rn(s[i + 1], mnew));
        const float p2 = ex2(__fsub_rn(s[i + 2], mnew));
        const float p3 = ex2(__fsub_rn(s[i + 3], mnew));
        rowsum = __fadd_rn(rowsum, p0);
        rowsum = __fadd_rn(rowsum, p1);
        rowsum = __fadd_rn(rowsum, p2);
        rowsum = __fadd_rn(rowsum, p3);
        const uint32_t lo = cvt_e4m3x2(__fmul_rn(448.f, p0), __fmul_rn(448.f, p1));
        const uint32_t hi = cvt_e4m3x2(__fmul_rn(448.f, p2), __fmul_rn(448.f, p3));
        pk[i >> 2] = lo | (hi << 16);
      }
      l = __fadd_rn(__fmul_rn(alpha, l), rowsum);
      // PV of the previous tile must be complete: it frees this P buffer's
      // previous user and leaves O stable for the rescale below.
      if (j >= 1) {
        ok = mbar_wait(&bars->pv_done, (j - 1) & 1, abort);
        if (!ok) break;
        tc_fence_after();
      }
      uint8_t *dstP = sPbase + (j & 1) * kPBytes;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4 *>(dstP + ((c ^ sw) << 4)) =
            make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + kColO + 32 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__fmul_rn(alpha, __uint_as_float(o[i])));
          tmem_st32(lane_base + kColO + 32 * c, o);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[j & 1]);
      m = mnew;
    }
    if (ok) ok = mbar_wait(&bars->pv_done, (T - 1) & 1, abort);
    if (!ok) {
      report(p.status, SAGE_ERR_TIMEOUT);
    } else {
      tc_fence_after();
      const float *sv = p.v_scales + bh * kD;
      const int b = bh / p.H, h = bh - b * p.H;
      __nv_bfloat16 *dst = p.out + b * p.os.b + h * p.os.h + int64_t(row) * p.os.n;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(lane_base + kColO + 32 * c, o);
        tmem_ld_wait();
        uint32_t packed[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float y0 = __fmul_rn(__fdiv_rn(__uint_as_float(o[i]), l), __fdiv_rn(sv[32 * c + i], 448.f));
          const float y1 =
              __fmul_rn(__fdiv_rn(__uint_as_float(o[i + 1]), l), __fdiv_rn(sv[32 * c + i + 1], 448.f));
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(y0, y1);
          packed[i >> 1] = *reinterpret_cast<const uint32_t *>(&b2);
        }
        if (valid) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4 *>(dst + 32 * c + 8 * u) =
                make_uint4(packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// int8 codes -> exact fp16 images (|code| <= 127 is exact in fp16).
// Each byte b is placed as the fp16 bit pattern 0x6400 | (b ^ 0x80), which is
// 1024 + (code + 128); subtracting 1152 leaves the code.
__global__ void __launch_bounds__(256) codes_to_f16_kernel(const int8_t *__restrict__ in, __half *__restrict__ out,
                                                           int64_t n16) {
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n16; i += int64_t(gridDim.x) * blockDim.x) {
    const uint4 w = reinterpret_cast<const uint4 *>(in)[i];
    const uint32_t ws[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
    uint32_t h[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t a = __byte_perm(ws[k], 0x64646464u, 0x4140);
      uint32_t b = __byte_perm(ws[k], 0x64646464u, 0x4342);
      __half2 ha = __hsub2(*reinterpret_cast<__half2 *>(&a), bias);
      __half2 hb = __hsub2(*reinterpret_cast<__half2 *>(&b), bias);
      h[2 * k] = *reinterpret_cast<uint32_t *>(&ha);
      h[2 * k + 1] = *reinterpret_cast<uint32_t *>(&hb);
    }
    uint4 *o = reinterpret_cast<uint4 *>(out) + 2 * i;
    o[0] = make_uint4(h[0], h[1], h[2], h[3]);
    o[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
}

}  // namespace dense

size_t dense_workspace_bytes(int B, int H, int Nq, int Nk) {
  return (size_t(B) * H * Nq + size_t(B) * H * Nk) * kD * sizeof(__half) + 256;
}

static int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

cudaError_t launch_codes_to_f16(const int8_t *codes, void *img, int64_t n, cudaStream_t st) {
  const int64_t n16 = n / 16;
  const int64_t want = (n16 + 255) / 256, cap = int64_t(sm_count()) * 8;
  int blocks = int(want < cap ? want : cap);
  if (blocks < 1) blocks = 1;
  dense::codes_to_f16_kernel<<<blocks, 256, 0, st>>>(codes, static_cast<__half *>(img), n16);
  return cudaGetLastError();
}

cudaError_t launch_attn_dense(const DenseArgs &a, cudaStream_t st) {
  using namespace dense;
  const int BH = a.B * a.H;
  const int64_t nq = int64_t(BH) * a.Nq * kD, nk = int64_t(BH) * a.Nk * kD;
  cudaError_t e = launch_codes_to_f16(a.q_codes, a.q_img, nq, st);
  if (e != cudaSuccess) return e;
  e = launch_codes_to_f16(a.k_codes, a.k_img, nk, st);
  if (e != cudaSuccess) return e;

  CUtensorMap tq, tk, tv;
  const int npad = nk_pad(a.Nk);
  if (!encode_tmap_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.q_img, kD, a.Nq, BH, kD * 2, uint64_t(a.Nq) * kD * 2, 64,
                      BM, 1) ||
      !encode_tmap_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.k_img, kD, a.Nk, BH, kD * 2, uint64_t(a.Nk) * kD * 2, 64,
                      BN, 1) ||
      !encode_tmap_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.v_codes, npad, kD, BH, npad, uint64_t(npad) * kD, BN, kD,
                      1))
    return cudaErrorInvalidValue;

  Params p;
  p.q_scales = a.q_scales;
  p.k_scales = a.k_scales;
  p.v_scales = a.v_scales;
  p.H = a.H;
  p.Nq = a.Nq;
  p.Nk = a.Nk;
  p.q_block = a.q_block;
  p.k_block = a.k_block;
  p.nbq = ceil_div(a.Nq, a.q_block);
  p.nbk = ceil_div(a.Nk, a.k_block);
  p.C = a.sm_scale * 1.44269504f;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.os = a.os;
  p.status = a.status;

  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(sage_attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid(ceil_div(a.Nq, BM), BH);
  sage_attn_fwd_kernel<<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace sg
