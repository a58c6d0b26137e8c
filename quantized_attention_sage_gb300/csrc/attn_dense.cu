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
//  * One CTA owns two 128-row query tiles of one (b, h); every K/V tile read
//    serves both.  (When the last wave of CTAs would leave more than half of
//    the SMs idle, its pairs run as single-tile CTAs instead.)  Warp 0 issues
//    TMA; warps 1 and 3 issue Q.K^T of tile 0 and tile 1, warp 2 issues both
//    P.V (one issuing warp per sub-partition); warps 4-7 and 8-11 are two
//    softmax warpgroups, one per query tile, one query row per thread (TMEM
//    lane = row).  TMEM: S0, S1, O0, O1, 128 columns each.  The role
//    warpgroup hands registers to the softmax warpgroups (setmaxnreg).
//  * S_t is free as soon as the softmax has loaded it into registers, so
//    QK_t(j+1) is issued right then (barrier s_free): the next scores are
//    computed while the softmax of the current tile runs.  P_t (E4M3) goes
//    to a 128-byte-swizzled shared tile per query tile, read by PV_t(j).
//  * The two softmax warps of a sub-partition take turns for the arithmetic
//    (one computes while the other loads S, stores P or rescales O).
//  * Softmax per element: row max on the raw int32-valued S (the dequant
//    multiplier is positive, so max(fl(S*t)) = fl(max(S)*t)); for a key tile
//    with no masked key it comes with the two 64-column S loads
//    (tcgen05.ld.red with .max returns the values and each half's maximum,
//    one per 64-key scale block).  Then one FFMA for S*t - m' + log2(448), ex2
//    on MUFU (448*p directly), fp32 row sums of 448*p, E4M3 conversion of
//    448*p; the ex2 of one group of keys are issued between the sums and
//    conversions of the previous group.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace sg {

SG_BOUNDS_FILE(dense, 4)

namespace dense {

constexpr int BM = 128, BN = 128, NSK = 2, NSV = 2;
constexpr int kThreads = 384;
constexpr uint32_t kQBytes = BM * kD * 2;    // 32 KB fp16 per query tile
constexpr uint32_t kKBytes = BN * kD * 2;    // 32 KB fp16
constexpr uint32_t kVBytes = kD * BN;        // 16 KB e4m3
constexpr uint32_t kPBytes = BM * BN;        // 16 KB e4m3 per query tile
constexpr uint32_t kOffQ = 0;                // two query tiles
constexpr uint32_t kOffK = kOffQ + 2 * kQBytes;
constexpr uint32_t kOffV = kOffK + NSK * kKBytes;
constexpr uint32_t kOffP = kOffV + NSV * kVBytes;  // two P tiles
constexpr uint32_t kOffBar = kOffP + 2 * kPBytes;
constexpr uint32_t kSmemBytes = kOffBar + 256 + 1024;  // barriers + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory");
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_s(int t) { return t ? 128u : 0u; }
__host__ __device__ constexpr uint32_t col_o(int t) { return t ? 384u : 256u; }

constexpr uint32_t kIdescQK = make_idesc(kFmtF32, kFmtF16, kFmtF16, BM, BN);
constexpr uint32_t kIdescPV = make_idesc(kFmtF32, kFmtE4M3, kFmtE4M3, BM, kD);
constexpr float kLog2_448 = 8.807354922057604f;  // log2(448)

struct Params {
  const float *q_scales, *k_scales, *v_scales;
  int H, Nq, Nk, q_block, k_block, nbq, nbk;
  float C;  // fl(sm_scale * log2 e)
  __nv_bfloat16 *out;
  sage_strides os;
  int32_t *status;
  int32_t *s_dump;  // diagnostic: exact scores [B*H][Nq_pad][Nk_pad], or null
  int nq_pad, nk_pad;
  int causal;        // query i sees keys j <= i + (Nk - Nq)
  float *lse;        // per-row log-sum-exp [B*H][Nq] (natural base), or null
  uint64_t wait_ns;  // limit of every bounded wait
  int fault;         // test hook: 1 = the producer issues no loads; 2 = only Q and the first K tile
  int pairs;         // query-tile pairs per head
  int n_pairs;       // 1-D grid: the first n_pairs CTAs take pairs, the rest single tiles; -1: 2-D grid
#ifdef SAGE_DEBUG_BOUNDS
  int BH;  // B * H, for the bounds checks of the debug build
#endif
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV];
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  // turn[t][k]: the softmax warp of tile t in TMEM lane quadrant k may run its
  // arithmetic (the two tiles' warps of one sub-partition alternate)
  uint64_t turn[2][4];
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
  int bh, q0, ntile;
  if (p.n_pairs >= 0) {
    // last-wave balancing: pairs of query tiles in (head, pair) order, then the
    // tiles of the remaining pairs one per CTA, so that the last wave spreads
    // over twice as many SMs
    const int u = blockIdx.x;
    if (u < p.n_pairs) {
      bh = u / p.pairs;
      q0 = (u - bh * p.pairs) * 2 * BM;
      ntile = (q0 + BM < p.Nq) ? 2 : 1;
    } else {
      const int v = u - p.n_pairs, g = p.n_pairs + (v >> 1);
      bh = g / p.pairs;
      q0 = (g - bh * p.pairs) * 2 * BM + (v & 1) * BM;
      ntile = 1;
    }
  } else {
    bh = blockIdx.y;
    // causal: the CTAs with the most key tiles (the last query rows) start first
    const int qpair = p.causal ? int(gridDim.x) - 1 - int(blockIdx.x) : int(blockIdx.x);
    q0 = qpair * 2 * BM;
    ntile = (q0 + BM < p.Nq) ? 2 : 1;  // second query tile present?
  }
  if (q0 >= p.Nq) return;  // the second tile of a ragged last pair: nothing to do
  if (!SG_BOUNDS(bh < p.BH && q0 >= 0)) return;
  const int coff = p.Nk - p.Nq;                 // causal offset: row i sees keys <= i + coff
  const int T = p.causal ? (min(q0 + ntile * BM, p.Nq) - 1 + coff) / BN + 1 : ceil_div(p.Nk, BN);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < NSK; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], ntile);  // one commit per query tile's Q.K^T
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->s_free[t], 4);
      mbar_init(&bars->p_full[t], 4);
      mbar_init(&bars->pv_done[t], 1);
      for (int k = 0; k < 4; ++k) mbar_init(&bars->turn[t][k], 1);
    }
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

  // Registers: the role warpgroup (warps 0-3) needs few, the softmax arithmetic
  // schedules better with more.  128 x 48 + 256 x 208 = 59,392 <= 384 x 168,
  // the registers the CTA was launched with.
  if (warp < 4) {
  setmaxnreg_dec<48>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop (uniform values); one elected lane issues.
    const bool leader = elect_one();
    // Test hooks: fault == 1 issues nothing; fault == 2 loads Q and the first
    // K tile and stops.  Either way the consumers' bounded waits run out and
    // the kernel reports SAGE_ERR_TIMEOUT.
    int nk = 0, nv = 0;  // K and V tiles issued
    bool q_issued = false;
    if (p.fault != 1) {
      if (leader) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        mbar_arrive_expect_tx(&bars->q_full, ntile * kQBytes);
        for (int t = 0; t < ntile; ++t) {
          uint8_t *sQ = smem + kOffQ + t * kQBytes;
          tma_load_3d(sQ, &tmQ, &bars->q_full, 0, q0 + t * BM, bh);
          tma_load_3d(sQ + kQBytes / 2, &tmQ, &bars->q_full, 64, q0 + t * BM, bh);
        }
      }
      q_issued = true;
      __syncwarp();
      auto load_k = [&](int j) -> bool {
        const int s = j % NSK;
        if (j >= NSK && !mbar_wait(&bars->k_empty[s], ((j / NSK) + 1) & 1, abort, p.wait_ns)) return false;
        if (leader) {
          uint8_t *dst = smem + kOffK + s * kKBytes;
          mbar_arrive_expect_tx(&bars->k_full[s], kKBytes);
          tma_load_3d(dst, &tmK, &bars->k_full[s], 0, j * BN, bh);
          tma_load_3d(dst + kKBytes / 2, &tmK, &bars->k_full[s], 64, j * BN, bh);
        }
        __syncwarp();
        ++nk;
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = j % NSV;
        if (j >= NSV && !mbar_wait(&bars->v_empty[s], ((j / NSV) + 1) & 1, abort, p.wait_ns)) return false;
        if (leader) {
          mbar_arrive_expect_tx(&bars->v_full[s], kVBytes);
          tma_load_3d(smem + kOffV + s * kVBytes, &tmV, &bars->v_full[s], j * BN, 0, bh);
        }
        __syncwarp();
        ++nv;
        return true;
      };
      bool ok = load_k(0);
      if (p.fault != 2) {
        for (int j = 0; ok && j < T; ++j) {
          if (j + 1 < T) ok = load_k(j + 1);
          if (ok) ok = load_v(j);
        }
      }
      if (!ok && leader) report(p.status, SAGE_ERR_TIMEOUT);
    }
    // Every copy issued here lands in this CTA's shared memory: wait for the
    // last phase of each barrier it armed before the CTA may exit, also when
    // the consumers gave up and no longer wait for them.
    bool drained = !q_issued || mbar_drain(&bars->q_full, 0, p.wait_ns);
    for (int s = 0; s < NSK; ++s)
      if (nk > s) drained &= mbar_drain(&bars->k_full[s], ((nk - 1 - s) / NSK) & 1, p.wait_ns);
    for (int s = 0; s < NSV; ++s)
      if (nv > s) drained &= mbar_drain(&bars->v_full[s], ((nv - 1 - s) / NSV) & 1, p.wait_ns);
    if (!drained && leader) report(p.status, SAGE_ERR_TIMEOUT);
  } else if (warp <= 3) {
    // ------------------------------------------------------------ MMA issuers
    // tcgen05.mma issue blocks for about one MMA's execution time and takes
    // issue slots from the softmax warps of the issuing warp's sub-partition,
    // which gate everyone through the barriers.  So the issue is spread over
    // three sub-partitions, each issuer in a fixed order with blocking waits:
    // warp 1 issues Q.K^T of tile 0, warp 3 Q.K^T of tile 1, warp 2 both P.V.
    // A commit tracks the MMAs of its own thread only; the issuers touch
    // disjoint TMEM columns (S_0, S_1, O_t), and a K stage is released when
    // both Q.K^T warps' commits have arrived (k_empty counts the tiles).
    // Each whole warp runs the loop (uniform values); one elected lane issues.
    const bool leader = elect_one();
    // Shared-memory descriptors are built once; a K-step only adds a constant:
    // +32 bytes (2 in the address field) inside a 128-byte swizzle row, +16 KB
    // (1024) to the second 64-column block of an fp16 tile.
    constexpr uint64_t kQStep = kQBytes >> 4, kKStep = kKBytes >> 4, kVStep = kVBytes >> 4, kPStep = kPBytes >> 4;
    bool ok = true;
    if (warp == 1 || warp == 3) {
      const int t = warp == 1 ? 0 : 1;
      if (t < ntile) {
        const uint64_t dq = sdesc_sw128(smem_u32(smem + kOffQ)) + uint64_t(t) * kQStep;
        const uint64_t dK0 = sdesc_sw128(smem_u32(smem + kOffK));
        ok = mbar_wait(&bars->q_full, 0, abort, p.wait_ns);
        int last = -1;  // last key tile whose Q.K^T was committed to s_full[t]
        for (int j = 0; ok && j < T; ++j) {
          const int s = j % NSK;
          ok = mbar_wait(&bars->k_full[s], (j / NSK) & 1, abort, p.wait_ns);
          // S_t(j) overwrites S_t(j-1): the softmax must have loaded it
          if (ok && j >= 1) ok = mbar_wait(&bars->s_free[t], (j - 1) & 1, abort, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dk = dK0 + uint64_t(s) * kKStep;
          if (leader) {
#pragma unroll
            for (int k = 0; k < kD / 16; ++k) {
              const uint64_t off = uint64_t((k >> 2) * (kQBytes / 2 / 16) + (k & 3) * 2);
              umma_f16(tmem + col_s(t), dq + off, dk + off, kIdescQK, k > 0);
            }
            tc_commit(&bars->s_full[t]);
            tc_commit(&bars->k_empty[s]);
          }
          __syncwarp();
          last = j;
        }
        // the MMAs issued here read shared memory and write TMEM: wait for the
        // last commit (it covers all of them) before the CTA may free either
        if (last >= 0 && !mbar_drain(&bars->s_full[t], last & 1, p.wait_ns)) ok = false;
      }
    } else {
      const uint64_t dV0 = sdesc_sw128(smem_u32(smem + kOffV));
      const uint64_t dP0 = sdesc_sw128(smem_u32(smem + kOffP));
      int last_j = -1, last_t = 0;  // last P.V committed to pv_done[last_t]
      for (int j = 0; ok && j < T; ++j) {
        const int s = j % NSV;
        ok = mbar_wait(&bars->v_full[s], (j / NSV) & 1, abort, p.wait_ns);
        for (int t = 0; ok && t < ntile; ++t) {
          ok = mbar_wait(&bars->p_full[t], j & 1, abort, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dp = dP0 + uint64_t(t) * kPStep, dv = dV0 + uint64_t(s) * kVStep;
          if (leader) {
#pragma unroll
            for (int k = 0; k < BN / 32; ++k)
              umma_f8f6f4(tmem + col_o(t), dp + uint64_t(2 * k), dv + uint64_t(2 * k), kIdescPV, (j > 0) || (k > 0));
            tc_commit(&bars->pv_done[t]);
          }
          __syncwarp();
          last_j = j;
          last_t = t;
        }
        if (ok && leader) tc_commit(&bars->v_empty[s]);
        __syncwarp();
      }
      if (last_j >= 0 && !mbar_drain(&bars->pv_done[last_t], last_j & 1, p.wait_ns)) ok = false;
    }
    if (!ok && leader) report(p.status, SAGE_ERR_TIMEOUT);
  }
  } else {
    setmaxnreg_inc<208>();
    // ------------------------------------------------------------ softmax / rescale / epilogue
    const int t = (warp - 4) >> 2;  // query tile of this warpgroup
    if (t < ntile) {
      const int r = (warp & 3) * 32 + lane;  // row in the tile == TMEM lane
      const int row = q0 + t * BM + r;
      const bool valid = row < p.Nq;
      const uint32_t lane_base = tmem + (uint32_t((warp & 3) * 32) << 16);
      const uint32_t colS = lane_base + col_s(t), colO = lane_base + col_o(t);
      uint8_t *sP = smem + kOffP + t * kPBytes + r * 128;
      const uint32_t sw = r & 7;
      const float sq = (valid && SG_BOUNDS(row / p.q_block < p.nbq)) ? p.q_scales[bh * p.nbq + row / p.q_block] : 0.f;
      const float *skp = p.k_scales + bh * p.nbk;
      float m = -INFINITY, l = 0.f;  // l sums 448 * p
      bool ok = true;
      // dequantisation multipliers t = fl(fl(sq * sk) * C) of a tile's key blocks
      auto tile_t = [&](int j, float &lo, float &hi) {
        if (p.k_block == 128) {
          lo = hi = SG_BOUNDS(j < p.nbk) ? __fmul_rn(__fmul_rn(sq, skp[j]), p.C) : 0.f;
        } else {
          lo = SG_BOUNDS(2 * j < p.nbk) ? __fmul_rn(__fmul_rn(sq, skp[2 * j]), p.C) : 0.f;
          hi = (2 * j + 1 < p.nbk) ? __fmul_rn(__fmul_rn(sq, skp[2 * j + 1]), p.C) : 0.f;
        }
      };
      float t_lo, t_hi;
      tile_t(0, t_lo, t_hi);
      for (int j = 0; j < T; ++j) {
        ok = mbar_wait(&bars->s_full[t], j & 1, abort, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
        uint32_t S[128];
        // the two loads also return the maximum of each 64-key half (used
        // when no key of the tile is masked)
        float mh[2];
        tmem_ld64_max(colS + 0, *reinterpret_cast<uint32_t(*)[64]>(&S[0]), mh[0]);
        tmem_ld64_max(colS + 64, *reinterpret_cast<uint32_t(*)[64]>(&S[64]), mh[1]);
        // keys of this tile that exist and, when causal, that the row may see
        const int nvalid = p.causal ? min(min(BN, p.Nk - j * BN), row + coff - j * BN + 1) : min(BN, p.Nk - j * BN);
        float nt_lo = 0.f, nt_hi = 0.f;  // next tile's multipliers, loaded while S is in flight
        if (j + 1 < T) tile_t(j + 1, nt_lo, nt_hi);
        tmem_ld_wait(S);
        asm volatile("" : "+f"(mh[0]), "+f"(mh[1]));
        if (p.s_dump != nullptr && SG_BOUNDS(q0 + t * BM + r < p.nq_pad && j * BN + BN <= p.nk_pad)) {
          // diagnostic copy of the exact integer scores
          int32_t *d = p.s_dump + (int64_t(bh) * p.nq_pad + (q0 + t * BM + r)) * p.nk_pad + j * BN;
#pragma unroll
          for (int i = 0; i < 128; i += 4)
            *reinterpret_cast<int4 *>(d + i) =
                make_int4(__float2int_rn(__uint_as_float(S[i])), __float2int_rn(__uint_as_float(S[i + 1])),
                          __float2int_rn(__uint_as_float(S[i + 2])), __float2int_rn(__uint_as_float(S[i + 3])));
        }
        // S_t(j) is in registers: the MMA warp may compute S_t(j+1) now
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->s_free[t]);
        float *Sf = reinterpret_cast<float *>(S);
        float mnew, alpha, rowsum;
        uint32_t pk[32];
        // The tile's softmax; kMasked (keys past Nk in this tile) is a
        // compile-time flag so that full tiles carry no per-element predicates.
        const int quad = warp & 3;
        bool turn_ok = true;
        auto softmax_tile = [&](auto masked_c) {
          constexpr bool kMasked = decltype(masked_c)::value;
          if (kMasked) {
#pragma unroll
            for (int i = 0; i < 128; ++i)
              if (i >= nvalid) Sf[i] = -INFINITY;
          }
          // row maximum of the raw scores: from the loads for a full tile,
          // four independent chains over the masked scores otherwise
          float mlo, mhi;
          if (!kMasked) {
            mlo = mh[0];
            mhi = mh[1];
          } else {
            float c0 = fmax3(Sf[0], Sf[1], Sf[2]), c1 = fmax3(Sf[32], Sf[33], Sf[34]);
            float c2 = fmax3(Sf[64], Sf[65], Sf[66]), c3 = fmax3(Sf[96], Sf[97], Sf[98]);
#pragma unroll
            for (int i = 3; i < 31; i += 2) {
              c0 = fmax3(c0, Sf[i], Sf[i + 1]);
              c1 = fmax3(c1, Sf[32 + i], Sf[33 + i]);
              c2 = fmax3(c2, Sf[64 + i], Sf[65 + i]);
              c3 = fmax3(c3, Sf[96 + i], Sf[97 + i]);
            }
            mlo = fmax3(fmax3(c0, c1, Sf[31]), Sf[63], Sf[63]);
            mhi = fmax3(fmax3(c2, c3, Sf[95]), Sf[127], Sf[127]);
          }
          float mt;
          if (kMasked) {
            mt = fmaxf(mlo == -INFINITY ? -INFINITY : __fmul_rn(mlo, t_lo),
                       mhi == -INFINITY ? -INFINITY : __fmul_rn(mhi, t_hi));
          } else {
            mt = fmaxf(__fmul_rn(mlo, t_lo), __fmul_rn(mhi, t_hi));
          }
          mnew = fmaxf(m, mt);
          alpha = (m == -INFINITY) ? 0.f : ex2(__fsub_rn(m, mnew));
          // only the exponential phase takes turns with the other tile's warp
          if (ntile == 2 && (t == 1 || j >= 1)) {
            turn_ok = mbar_wait(&bars->turn[t][quad], (t == 1 ? j : j - 1) & 1, abort, p.wait_ns);
            if (!turn_ok) return;
          }
          // x = S * t - (m' - log2 448): 2^x = 448 * p
          const float nb = __fsub_rn(kLog2_448, mnew);
          float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
          // Groups of four keys, software-pipelined by hand: the four ex2 of
          // group g+1 are issued between the sums and E4M3 conversions of
          // group g (the _ord helpers keep this order), so the MUFU pipe and
          // the FMA/ALU pipes work side by side.
          auto group_x = [&](int i, float2 &x01, float2 &x23) {
            const float tt = i < 64 ? t_lo : t_hi;
            x01 = ffma2_ord(make_float2(Sf[i], Sf[i + 1]), make_float2(tt, tt), make_float2(nb, nb));
            x23 = ffma2_ord(make_float2(Sf[i + 2], Sf[i + 3]), make_float2(tt, tt), make_float2(nb, nb));
            if (kMasked) {  // keys past Nk: p = 0 (also when t = 0, where -inf * 0 would be NaN)
              if (i >= nvalid) x01.x = -INFINITY;
              if (i + 1 >= nvalid) x01.y = -INFINITY;
              if (i + 2 >= nvalid) x23.x = -INFINITY;
              if (i + 3 >= nvalid) x23.y = -INFINITY;
            }
          };
          float2 x01, x23;
          group_x(0, x01, x23);
          float2 q01 = make_float2(ex2_ord(x01.x), ex2_ord(x01.y));
          float2 q23 = make_float2(ex2_ord(x23.x), ex2_ord(x23.y));
#pragma unroll
          for (int i = 4; i <= 128; i += 4) {
            const bool more = i < 128;
            float2 n01, n23;
            if (more) group_x(i, n01, n23);
            float2 r01, r23;
            if (more) r01.x = ex2_ord(n01.x);
            acc0 = fadd2_ord(acc0, q01);
            if (more) r01.y = ex2_ord(n01.y);
            const uint32_t lo = cvt_e4m3x2_ord(q01.x, q01.y);
            if (more) r23.x = ex2_ord(n23.x);
            acc1 = fadd2_ord(acc1, q23);
            if (more) r23.y = ex2_ord(n23.y);
            const uint32_t hi = cvt_e4m3x2_ord(q23.x, q23.y);
            pk[(i - 4) >> 2] = __byte_perm(lo, hi, 0x5410);
            if (more) {
              q01 = r01;
              q23 = r23;
            }
          }
          rowsum = __fadd_rn(__fadd_rn(acc0.x, acc0.y), __fadd_rn(acc1.x, acc1.y));
        };
        // The warps of the two tiles that share a sub-partition take turns
        // for the arithmetic, so that one computes while the other loads S
        // or waits for its P.V, instead of both competing for issue slots
        // and then idling together.  Tile 0 goes first in every round.
        if (__any_sync(0xffffffffu, nvalid < BN)) softmax_tile(std::true_type{});
        else softmax_tile(std::false_type{});
        if (!turn_ok) {
          ok = false;
          break;
        }
        if (ntile == 2) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->turn[t ^ 1][quad]);
        }
        l = __fadd_rn(__fmul_rn(alpha, l), rowsum);
        // PV_t(j-1) must be complete: it read P_t and accumulated into O_t
        if (j >= 1) {
          ok = mbar_wait(&bars->pv_done[t], (j - 1) & 1, abort, p.wait_ns);
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4 *>(sP + ((c ^ sw) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
          // rescale O_t in TMEM: one load round trip, one store round trip
          uint32_t o[128];
          tmem_ld32(colO + 0, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
          tmem_ld32(colO + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
          tmem_ld32(colO + 64, *reinterpret_cast<uint32_t(*)[32]>(&o[64]));
          tmem_ld32(colO + 96, *reinterpret_cast<uint32_t(*)[32]>(&o[96]));
          tmem_ld_wait(o);
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int i = 0; i < 128; i += 2) {
            const float2 v = fmul2(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2);
            o[i] = __float_as_uint(v.x);
            o[i + 1] = __float_as_uint(v.y);
          }
          tmem_st32(colO + 0, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
          tmem_st32(colO + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
          tmem_st32(colO + 64, *reinterpret_cast<uint32_t(*)[32]>(&o[64]));
          tmem_st32(colO + 96, *reinterpret_cast<uint32_t(*)[32]>(&o[96]));
          tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->p_full[t]);
        m = mnew;
        t_lo = nt_lo;
        t_hi = nt_hi;
      }
      if (ok) ok = mbar_wait(&bars->pv_done[t], (T - 1) & 1, abort, p.wait_ns);
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
          tmem_ld32(colO + 32 * c, o);
          tmem_ld_wait(o);
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float y0 = __fmul_rn(__fdiv_rn(__uint_as_float(o[i]), l), sv[32 * c + i]);
            const float y1 = __fmul_rn(__fdiv_rn(__uint_as_float(o[i + 1]), l), sv[32 * c + i + 1]);
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(y0, y1);
            packed[i >> 1] = *reinterpret_cast<const uint32_t *>(&b2);
          }
          if (valid && SG_BOUNDS(row < p.Nq && bh < p.BH)) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              *reinterpret_cast<uint4 *>(dst + 32 * c + 8 * u) =
                  make_uint4(packed[4 * u], packed[4 * u + 1], packed[4 * u + 2], packed[4 * u + 3]);
          }
        }
        // log-sum-exp in the natural base: l sums 448 * 2^(s - m)
        if (p.lse != nullptr && valid && SG_BOUNDS(row < p.Nq && bh < p.BH))
          p.lse[int64_t(bh) * p.Nq + row] = (m + (log2f(l) - kLog2_448)) * 0.6931471805599453f;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
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

cudaError_t launch_codes_to_f16(const int8_t *codes, void *img, int64_t n, cudaStream_t st) {
  const int64_t n16 = n / 16;
  const int64_t want = (n16 + 255) / 256, cap = int64_t(current_sm_count()) * 8;
  int blocks = int(want < cap ? want : cap);
  if (blocks < 1) blocks = 1;
  dense::codes_to_f16_kernel<<<blocks, 256, 0, st>>>(codes, static_cast<__half *>(img), n16);
  return cudaGetLastError();
}

cudaError_t launch_attn_dense(const DenseArgs &a, cudaStream_t st) {
  using namespace dense;
  const int BH = a.B * a.H;
  const int64_t nq = int64_t(BH) * a.Nq * kD, nk = int64_t(BH) * a.Nk * kD;
  cudaError_t e = cudaSuccess;
  if (!a.images_ready) {
    e = launch_codes_to_f16(a.q_codes, a.q_img, nq, st);
    if (e != cudaSuccess) return e;
    e = launch_codes_to_f16(a.k_codes, a.k_img, nk, st);
    if (e != cudaSuccess) return e;
  }

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
#ifdef SAGE_DEBUG_BOUNDS
  p.BH = BH;
#endif
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
  p.s_dump = a.s_dump;
  p.nq_pad = ceil_div(a.Nq, 2 * BM) * 2 * BM;
  p.nk_pad = npad;
  p.causal = a.causal;
  p.lse = a.lse;
  p.wait_ns = a.wait_ns;
  p.fault = a.fault;

  static CtxOnce attr_done;
  e = set_smem_attr_once(reinterpret_cast<const void *>(sage_attn_fwd_kernel), kSmemBytes, &attr_done);
  if (e != cudaSuccess) return e;
  dim3 grid(ceil_div(a.Nq, 2 * BM), BH);
  p.pairs = ceil_div(a.Nq, 2 * BM);
  p.n_pairs = -1;
  {
    // Equal CTAs fill whole waves of one CTA per SM; when the last wave is at
    // most half full, its pairs are split into single-tile CTAs (a single tile
    // takes ~0.8 of a pair's time, measured), which shortens the tail.
    // Causal CTAs are unequal and keep the longest-first 2-D order.
    const long long total = (long long)BH * p.pairs;
    const int sms = current_sm_count();
    const int rem = sms > 0 ? int(total % sms) : 0;
    if (!a.causal && total > sms && rem > 0 && 2 * rem <= sms) {
      p.n_pairs = int(total - rem);
      grid = dim3(unsigned(p.n_pairs + 2 * rem), 1);
    }
  }
  sage_attn_fwd_kernel<<<grid, kThreads, kSmemBytes, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace sg
