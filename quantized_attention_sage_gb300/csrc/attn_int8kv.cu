// Causal prompt attention over an int8 KV cache with per-token fp16 scales,
// grouped-query heads, for sm_103a.
//
// Pages: "Strata PR #2092" (v2 int8 prompt attention: a chunk of new queries
// attends to the int8 KV cache; K/V staged per chunk together with their
// scales; error reported against FP64) and "Strata PR #2146" (the same kernel,
// one stage).
//
// GB300 design:
//  * One 128-row tile holds QT = floor(128 / G) queries x the G query heads of
//    one kv head (G = Hq / Hkv), so each K/V tile read serves all G heads.
//  * S = Q.K^T on tcgen05 kind::f16 (bf16 queries x exact bf16 images of the
//    int8 K codes), fp32 in TMEM.  Q is copied into TMEM once per CTA and read
//    from there (A operand): the MMAs that read both operands from shared
//    memory take all of its bandwidth while they run, and the TMA copies of
//    the next K/V tiles and the scale loads share it.
//  * softmax per row in fp32: s = S * fl(ks * sm_scale * log2 e), causal mask
//    by absolute position, p = 2^(s - m) with the exponent taken from the raw
//    score in one FMA (S * kt - (m + E)) once the row has a reference m.
//  * P.V: the weight w = p * vs (scaled by a power of two so that w < 2^15) is
//    split into fp16 hi + lo parts and multiplied with exact fp16 images of the
//    V codes by one K = 256 kind::f16 MMA chain ([hi | lo] . [V ; V]), so the
//    fp16 rounding of w does not reach the output.  hi and lo are written
//    with tcgen05.st over the consumed S buffer and read by the MMA from TMEM.
//  * Four softmax warpgroups, one per 32-key quarter of every key tile, one
//    query row per thread: four warps per SM sub-partition.  They share one
//    O accumulator and one reference maximum per row: each quarter's maximum
//    is exchanged through shared memory under a named barrier of the four
//    warps that hold the same rows, and each rescales its own 32 columns of O.
//    The reference is the exact maximum of the first tile; later tiles take
//    their weights against the kept reference before the exchange and are
//    redone only when their maximum passes it by more than 15 (the weights
//    are fp16 hi + lo, whose range holds 2^15).
//  * S is double-buffered in TMEM and QK(j+2) is issued right behind PV(j),
//    so the next scores are ready when the softmax finishes a tile; the MMA
//    and TMA warps run converged with one elected lane issuing.
//  * The key range of each query tile is split into `nsplit` contiguous pieces
//    (split-KV) so the grid fills the SMs; a combine kernel merges the (m, l,
//    O) partials of one row in split order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace sg {

SG_BOUNDS_FILE(int8kv, 5)

namespace kv {

constexpr int BM = 128, BN = 128, NSK = 3, NSV = 3;
constexpr int kQuarter = BN / 4;  // keys of a tile per softmax warpgroup
// warp 0 TMA, warp 1 MMA, warps 2-17 softmax (quarter (w - 2) / 4, TMEM lane
// quadrant w % 4: four consecutive warps cover the four quadrants)
constexpr int kSoftmaxWarp0 = 2;
constexpr int kThreads = (kSoftmaxWarp0 + 16) * 32;
constexpr uint32_t kQBytes = BM * kD * 2;
constexpr uint32_t kKTile = BN * kD * 2;                // bf16 K image
constexpr uint32_t kVBytes = kD * BN * 2;               // fp16 V^T image
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kQBytes;
constexpr uint32_t kOffV = kOffK + 2 * kKTile;
// K ring: stages 0 and 1 at kOffK, stage 2 in the Q tile, which is free once
// Q has been copied into TMEM
__host__ __device__ constexpr uint32_t k_stage(int s) { return s == 2 ? kOffQ : kOffK + uint32_t(s) * kKTile; }
// the tile's kt and vs (128 fp32 each) ride with its V tile
constexpr uint32_t kOffKt = kOffV + NSV * kVBytes;
constexpr uint32_t kOffVs = kOffKt + NSV * BN * 4;
constexpr uint32_t kOffBar = kOffVs + NSV * BN * 4;
// per row and quarter: the quarter maxima of a tile (two tiles in flight) and
// the final partial row sums
constexpr uint32_t kOffXm = kOffBar + 256;
constexpr uint32_t kOffXl = kOffXm + 2 * BM * 4 * 4;
constexpr uint32_t kSmemBytes = kOffXl + BM * 4 * 4 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory");
constexpr uint32_t kTmemCols = 512;
// TMEM: S double buffer at columns 0 and 128, O at 256, Q (bf16 pairs) at
// 384-447.  Quarter g's P (fp16 hi of its 32 keys in 16 columns, then lo in
// 16) overwrites that quarter's own 32 columns of the consumed S buffer.
__host__ __device__ constexpr uint32_t col_s(int b) { return b ? 128u : 0u; }
constexpr uint32_t kColO = 256, kColQ = 384;

constexpr uint32_t kIdescQK = make_idesc(kFmtF32, kFmtBF16, kFmtBF16, BM, BN);
constexpr uint32_t kIdescPV = make_idesc(kFmtF32, kFmtF16, kFmtF16, BM, kD);

struct Params {
  int Nq, q_pos0, Nk, Hkv, G, QT, nsplit, Npad;
  const float *kt, *vs;        // [Hkv][Npad] fl(ks*C), vs
  const uint32_t *vmax_bits;   // max vs over the cache (fp32 bits)
  float *part_o;               // [units][128][128]
  float2 *part_ml;             // [units][128] (m, l)
  int32_t *status;
  uint64_t wait_ns;  // limit of every bounded wait
  int fault;         // test hook: 1 = the producer issues no copy; 2 = only Q and the first two K tiles
};

struct Bars {
  uint64_t q_full, q_tmem;  // Q in shared memory; Q copied into TMEM
  uint64_t k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV];
  // s_full, p_full and pv_done per S buffer (tile j uses j & 1): a softmax
  // warp may finish tile j+1 before another finishes tile j (never two
  // tiles: the quarters meet at a named barrier every tile), so one barrier
  // per kind could be completed by the wrong tile's arrivals.
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

// Two weights w (fp32, below 2^15) as fp16 pairs hi + lo: hi = fp16_rn(w),
// lo = fp16_rn(w - hi).  w - hi is exact in fp32 (hi keeps the leading 11
// bits of w, or w's fp16-subnormal grid), taken in one mixed-precision FMA
// per weight (fp32 = fp16 * fp16 + fp32: hi * -1 + w), so hi + lo is w to
// within 2^-22 relative (2^-25 absolute below fp16's normal range).  Pairs
// in the bf16x2/f16x2 order: the first weight in the low half.
__device__ __forceinline__ void split_f16(float2 w, uint32_t &hi, uint32_t &lo) {
  asm("{\n\t.reg .b16 a, b, m;\n\t.reg .f32 ra, rb;\n\t"
      "mov.b16 m, 0xBC00;\n\t"
      "cvt.rn.f16x2.f32 %0, %3, %2;\n\t"
      "mov.b32 {a, b}, %0;\n\t"
      "fma.rn.f32.f16 ra, a, m, %2;\n\t"
      "fma.rn.f32.f16 rb, b, m, %3;\n\t"
      "cvt.rn.f16x2.f32 %1, rb, ra;\n\t}"
      : "=r"(hi), "=r"(lo)
      : "f"(w.x), "f"(w.y));
}
__device__ __forceinline__ void report(int32_t *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ int kv_tiles_for(const Params &p, int qtile) {
  const int last_q = min((qtile + 1) * p.QT, p.Nq) - 1;
  const int last_key = min(p.q_pos0 + last_q, p.Nk - 1);
  return last_key / BN + 1;
}

// Roles: warp 0 TMA, warp 1 MMA; warps 2-17 the softmax, warp w taking key
// quarter (w - 2) / 4 of every tile for the 32 query rows of TMEM lane
// quadrant w % 4, one row per thread (TMEM lane = row).  The four quarters of
// a row agree on the row maximum every tile (named barrier 1 + quadrant) and
// keep partial row sums that are added in quarter order at the end; the
// oracle of this path is the exact softmax, so splitting the keys only
// changes the fp32 summation order.
__global__ void __launch_bounds__(kThreads, 1)
    int8kv_attn_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars *bars = reinterpret_cast<Bars *>(smem + kOffBar);
  float4 *xm = reinterpret_cast<float4 *>(smem + kOffXm);  // [tile & 1][row]: the four quarter maxima
  float4 *xl = reinterpret_cast<float4 *>(smem + kOffXl);  // [row]: the four partial row sums
  volatile int *abort = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, qtile = blockIdx.y, g = blockIdx.z;
  const int unit = (g * gridDim.y + qtile) * p.nsplit + split;
  const int i0 = qtile * p.QT;
  const int tiles = kv_tiles_for(p, qtile);
  const int tb = int((int64_t(tiles) * split) / p.nsplit);
  const int te = int((int64_t(tiles) * (split + 1)) / p.nsplit);
  const int T = te - tb;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_tmem, 4);  // the four warps of quarter 0
    for (int s = 0; s < NSK; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
    }
    for (int s = 0; s < NSV; ++s) {
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b], 16);  // one arrive per softmax warp
      mbar_init(&bars->pv_done[b], 1);
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

  if (T <= 0) {
    // empty key range: record an empty partial for the combine
    if (warp >= kSoftmaxWarp0 && warp < kSoftmaxWarp0 + 4 &&
        SG_BOUNDS(unit < int(gridDim.x * gridDim.y * gridDim.z))) {
      const int r = (warp & 3) * 32 + lane;
      p.part_ml[int64_t(unit) * BM + r] = make_float2(-INFINITY, 0.f);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (converged warp)
    const bool leader = elect_one();
    // Test hooks: fault == 1 issues nothing; fault == 2 loads Q and the first
    // two K tiles and stops.  Either way the consumers' bounded waits run out
    // and the kernel reports SAGE_ERR_TIMEOUT.
    const bool q_issued = p.fault != 1;
    if (leader && q_issued) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(&bars->q_full, uint32_t(p.QT * p.G) * 256u);
      tma_load_3d(smem + kOffQ, &tmQ, &bars->q_full, 0, g * p.G, i0);
      tma_load_3d(smem + kOffQ + kQBytes / 2, &tmQ, &bars->q_full, 64, g * p.G, i0);
    }
    __syncwarp();
    int nk = 0, nv = 0;  // K and V tiles issued
    auto load_k = [&](int j) -> bool {
      const int s = j % NSK;
      if (j >= NSK && !mbar_wait(&bars->k_empty[s], ((j / NSK) + 1) & 1, abort, p.wait_ns)) return false;
      if (j == 2 && !mbar_wait(&bars->q_tmem, 0, abort, p.wait_ns)) return false;  // stage 2 is the Q tile
      if (leader) {
        const int key0 = (tb + j) * BN;
        uint8_t *dst = smem + k_stage(s);
        mbar_arrive_expect_tx(&bars->k_full[s], kKTile);
        tma_load_3d(dst, &tmK, &bars->k_full[s], 0, key0, g);
        tma_load_3d(dst + kKTile / 2, &tmK, &bars->k_full[s], 64, key0, g);
      }
      __syncwarp();
      ++nk;
      return true;
    };
    auto load_v = [&](int j) -> bool {
      const int s = j % NSV;
      if (j >= NSV && !mbar_wait(&bars->v_empty[s], ((j / NSV) + 1) & 1, abort, p.wait_ns)) return false;
      if (leader) {
        const int key0 = (tb + j) * BN;
        uint8_t *dst = smem + kOffV + s * kVBytes;
        mbar_arrive_expect_tx(&bars->v_full[s], kVBytes + 2 * BN * 4);
        tma_load_3d(dst, &tmV, &bars->v_full[s], key0, 0, g);
        tma_load_3d(dst + kVBytes / 2, &tmV, &bars->v_full[s], key0 + 64, 0, g);
        const int64_t row = int64_t(g) * p.Npad + key0;
        bulk_load(smem + kOffKt + s * BN * 4, p.kt + row, BN * 4, &bars->v_full[s]);
        bulk_load(smem + kOffVs + s * BN * 4, p.vs + row, BN * 4, &bars->v_full[s]);
      }
      __syncwarp();
      ++nv;
      return true;
    };
    // order of first use: K0, K1, V0, K2, V1, K3, ...; K(j+2) waits for the
    // Q.K^T of tile j-1, one tile earlier than a two-stage ring would
    bool ok = p.fault == 1 || (load_k(0) && (T < 2 || load_k(1)));
    for (int j = 0; ok && p.fault == 0 && j < T; ++j) {
      ok = load_v(j);
      if (ok && j + 2 < T) ok = load_k(j + 2);
    }
    // Every copy issued here lands in this CTA's shared memory: wait for the
    // last phase of each barrier it armed before the CTA may exit, also when
    // the consumers gave up and no longer wait for them.
    bool drained = !q_issued || mbar_drain(&bars->q_full, 0, p.wait_ns);
    for (int s = 0; s < NSK; ++s)
      if (nk > s) drained &= mbar_drain(&bars->k_full[s], ((nk - 1 - s) / NSK) & 1, p.wait_ns);
    for (int s = 0; s < NSV; ++s)
      if (nv > s) drained &= mbar_drain(&bars->v_full[s], ((nv - 1 - s) / NSV) & 1, p.wait_ns);
    if ((!ok || !drained) && leader) report(p.status, SAGE_ERR_TIMEOUT);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (converged warp)
    // Order: QK(0), QK(1), then per tile j: PV (A = the four quarters' P from
    // TMEM), QK(j+2) into the same TMEM buffer (MMAs of one thread execute in
    // order, so QK(j+2) overwrites P_j only after P.V has read it).
    const bool leader = elect_one();
    // the barrier and phase parity of the last commit (it covers every MMA
    // issued before it)
    uint64_t *last_bar = nullptr;
    uint32_t last_par = 0;
    auto issue_qk = [&](int j) -> bool {
      const int s = j % NSK;
      if (!mbar_wait(&bars->k_full[s], (j / NSK) & 1, abort, p.wait_ns)) return false;
      tc_fence_after();
      const uint32_t sK = smem_u32(smem + k_stage(s));
      if (leader) {
#pragma unroll
        for (int k = 0; k < kD / 16; ++k) {
          const uint32_t off = (k >> 2) * (kKTile / 2) + (k & 3) * 32;
          umma_f16_ts(tmem + col_s(j & 1), tmem + kColQ + 8 * k, sdesc_sw128(sK + off), kIdescQK, k > 0);
        }
        tc_commit(&bars->s_full[j & 1]);
        tc_commit(&bars->k_empty[s]);
      }
      __syncwarp();
      last_bar = &bars->s_full[j & 1];
      last_par = (j >> 1) & 1;
      return true;
    };
    bool ok = mbar_wait(&bars->q_tmem, 0, abort, p.wait_ns);
    tc_fence_after();
    ok = ok && issue_qk(0) && (T < 2 || issue_qk(1));
    for (int j = 0; ok && j < T; ++j) {
      const int s = j % NSV, b = j & 1;
      ok = mbar_wait(&bars->v_full[s], (j / NSV) & 1, abort, p.wait_ns) &&
           mbar_wait(&bars->p_full[b], (j >> 1) & 1, abort, p.wait_ns);
      if (!ok) break;
      tc_fence_after();
      const uint32_t sV = smem_u32(smem + kOffV + s * kVBytes);
      if (leader) {
        // O += sum over quarters g of [P_hi,g | P_lo,g] . [V_g ; V_g]: per
        // quarter two K-steps of 16 keys over hi and two over lo, against
        // keys 32g..32g+31 of the V^T tile (64-key blocks 16 KB apart,
        // 16 keys = 32 bytes of a 128-byte swizzled row)
#pragma unroll
        for (int g = 0; g < 4; ++g) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t off = (g >> 1) * (kVBytes / 2) + ((g & 1) * 2 + (k & 1)) * 32;
            umma_f16_ts(tmem + kColO, tmem + col_s(b) + kQuarter * g + 8 * k, sdesc_sw128(sV + off), kIdescPV,
                        (j > 0) || (g > 0) || (k > 0));
          }
        }
        tc_commit(&bars->pv_done[b]);
        tc_commit(&bars->v_empty[s]);
      }
      __syncwarp();
      last_bar = &bars->pv_done[b];
      last_par = (j >> 1) & 1;
      if (j + 2 < T) ok = issue_qk(j + 2);
    }
    // the MMAs read shared memory and write TMEM: wait for the last commit
    // before the CTA may free either
    if (last_bar != nullptr && !mbar_drain(last_bar, last_par, p.wait_ns)) ok = false;
    if (!ok && leader) report(p.status, SAGE_ERR_TIMEOUT);
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------------------------------ softmax of one key quarter
    const int g = (warp - kSoftmaxWarp0) >> 2;  // key quarter
    const int quad = warp & 3;                  // TMEM lane quadrant
    const int r = quad * 32 + lane;
    const int il = r / p.G;
    const int qi = i0 + il;
    const bool valid = (il < p.QT) && (qi < p.Nq);
    const int pos = p.q_pos0 + qi;  // keys 0..pos are visible
    const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16);
    const uint32_t colO = lane_base + kColO + kQuarter * g;  // this quarter's 32 columns of O
    // w = p * vs * 2^-E with 2^E > max vs: w < p = 2^(s - m), which stays
    // inside fp16 while s - m <= 15.  The factor 2^-E is taken into the
    // exponent (p' = 2^(s - m - E)), so the row sum is l * 2^-E as well and
    // O / l is unchanged.
    const float vmax = __uint_as_float(*p.vmax_bits);
    const int E = vmax > 0.f ? int((__float_as_uint(vmax) >> 23) & 0xFF) - 127 + 1 : 0;
    const float Ef = float(E);
    float m = -INFINITY, l = 0.f;  // m: the row's reference maximum (same in all quarters); l: this quarter's sum
    bool ok = true;
    // Named barriers cannot time out, so every warp of a quadrant passes
    // exactly T + 1 of them (one per tile and one at the end), also after a
    // bounded wait gave up: a warp that left the loop early makes up the
    // ones it skipped, without work, so that the others are never stranded.
    // All of them are the reducing form (bar.red), which must not be mixed
    // with bar.sync on the same barrier.
    int nbar = 0;
    if (g == 0) {
      // Q into TMEM: row r's 128 bf16 (two 128-byte swizzled rows of the TMA
      // boxes; 16-byte chunk c of row r sits at chunk c ^ (r & 7)) become 64
      // columns of bf16 pairs, the A-operand layout of Q.K^T
      ok = mbar_wait(&bars->q_full, 0, abort, p.wait_ns);
      if (ok) {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint8_t *row = smem + kOffQ + half * (kQBytes / 2) + r * 128;
          uint32_t qw[32];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4 *>(row + ((c ^ (r & 7)) << 4));
            qw[4 * c] = v.x;
            qw[4 * c + 1] = v.y;
            qw[4 * c + 2] = v.z;
            qw[4 * c + 3] = v.w;
          }
          tmem_st32(lane_base + kColQ + 32 * half, qw);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->q_tmem);
      }
    }
    for (int j = 0; ok && j < T; ++j) {
      const int b = j & 1;
      ok = mbar_wait(&bars->s_full[b], (j >> 1) & 1, abort, p.wait_ns);
      if (!ok) break;
      tc_fence_after();
      const uint32_t sa = lane_base + col_s(b) + kQuarter * g;
      uint32_t S[kQuarter];
      tmem_ld32(sa, S);
      const int key0 = (tb + j) * BN + kQuarter * g;
      const int nvis = min(kQuarter, pos - key0 + 1);  // visible keys of this quarter (<= 0: none)
      // kt and vs of this tile arrived with V(j); its slot is reused only
      // after the P.V of tile j, which waits for this warp's p_full
      const int sv = j % NSV;
      ok = mbar_wait(&bars->v_full[sv], (j / NSV) & 1, abort, p.wait_ns);
      if (!ok) break;
      const float4 *kt4 = reinterpret_cast<const float4 *>(smem + kOffKt + sv * BN * 4) + kQuarter / 4 * g;
      const float4 *vs4 = reinterpret_cast<const float4 *>(smem + kOffVs + sv * BN * 4) + kQuarter / 4 * g;
      tmem_ld_wait(S);
      float *Sf = reinterpret_cast<float *>(S);
      float mnew, alpha, rowsum;
      // The quarter tile's softmax; kMasked (some row of the warp sees only
      // part of the quarter) is a compile-time flag so that the tiles below
      // the diagonal carry no per-element predicates.
      auto softmax_quarter = [&](auto masked_c) {
        constexpr bool kMasked = decltype(masked_c)::value;
        // p' = 2^x, the row sum, and w = p' * vs split into fp16 hi + lo,
        // written over this quarter's S columns: hi at +0..15, lo at +16..31,
        // in blocks of 8 keys (4 columns each: fewer registers live at once);
        // returns the quarter's row sum.  x = s - nb (nb = reference + E):
        // from the base-2 logits already in Sf (kRaw false), or from the raw
        // scores in one FMA, x = S * kt - nb (kRaw true), which also gives
        // the quarter's largest x in xq (masked keys are -inf)
        auto weights = [&](float nb, auto raw_c, float &xq) -> float {
          constexpr bool kRaw = decltype(raw_c)::value;
          const float2 nb2 = make_float2(nb, nb), nbn2 = make_float2(-nb, -nb);
          float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
          float q0 = -INFINITY, q1 = -INFINITY;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int i = 0; i < 8; i += 4) {
              const int e = 8 * c + i;
              const float4 v4 = lds_f4_in_order(vs4 + (e >> 2));
              float2 x01, x23;
              if (kRaw) {
                const float4 k4 = lds_f4_in_order(kt4 + (e >> 2));
                x01 = ffma2(make_float2(Sf[e], Sf[e + 1]), make_float2(k4.x, k4.y), nbn2);
                x23 = ffma2(make_float2(Sf[e + 2], Sf[e + 3]), make_float2(k4.z, k4.w), nbn2);
                if (kMasked) {  // keys past the query's position
                  if (e >= nvis) x01.x = -INFINITY;
                  if (e + 1 >= nvis) x01.y = -INFINITY;
                  if (e + 2 >= nvis) x23.x = -INFINITY;
                  if (e + 3 >= nvis) x23.y = -INFINITY;
                }
                q0 = fmax3(q0, x01.x, x01.y);
                q1 = fmax3(q1, x23.x, x23.y);
              } else {
                x01 = fsub2(make_float2(Sf[e], Sf[e + 1]), nb2);
                x23 = fsub2(make_float2(Sf[e + 2], Sf[e + 3]), nb2);
              }
              const float2 p01 = make_float2(ex2(x01.x), ex2(x01.y));
              const float2 p23 = make_float2(ex2(x23.x), ex2(x23.y));
              acc0 = fadd2(acc0, p01);
              acc1 = fadd2(acc1, p23);
              const float2 w01 = fmul2(p01, make_float2(v4.x, v4.y));
              const float2 w23 = fmul2(p23, make_float2(v4.z, v4.w));
              split_f16(w01, hi[i >> 1], lo[i >> 1]);
              split_f16(w23, hi[(i >> 1) + 1], lo[(i >> 1) + 1]);
            }
            tmem_st4(sa + 4 * c, hi);
            tmem_st4(sa + 16 + 4 * c, lo);
          }
          xq = fmaxf(q0, q1);
          return __fadd_rn(__fadd_rn(acc0.x, acc0.y), __fadd_rn(acc1.x, acc1.y));
        };
        // The reference maximum m of the weights.  While some row of the warp
        // has none, the tile's exact maximum is exchanged first (the four
        // warps holding these rows meet at named barrier 1 + quad; xm is
        // double-buffered by tile, and no warp can be two tiles ahead of
        // another since each tile has exactly one such barrier) and becomes
        // it.  After that the reference is kept: the tile's weights are taken
        // against it at once, from the raw scores, and the exchange follows
        // them, so the exponentials do not wait for it.  The weights are fp16
        // hi + lo, not FP8, so a reference below the tile's maximum only
        // scales them (O / l does not change), and up to 2^15 they stay inside
        // fp16 (w < 2^(s - m), since vs * 2^-E < 1).  A tile whose maximum
        // passes the reference by more than 15 (x > 15 - E) is redone against
        // the new running maximum, and O and l are rescaled.  All four warps
        // of a quadrant hold the same rows, the same m and the same exchanged
        // maxima, so they take the same branch.
        float xq;
        if (__any_sync(0xffffffffu, m == -INFINITY)) {
          // s = S * kt (base-2 logits), masked, and the quarter's maximum
#pragma unroll
          for (int i = 0; i < kQuarter; i += 4) {
            const float4 k4 = kt4[i >> 2];
            const float2 a = fmul2(make_float2(Sf[i], Sf[i + 1]), make_float2(k4.x, k4.y));
            const float2 c = fmul2(make_float2(Sf[i + 2], Sf[i + 3]), make_float2(k4.z, k4.w));
            Sf[i] = a.x;
            Sf[i + 1] = a.y;
            Sf[i + 2] = c.x;
            Sf[i + 3] = c.y;
          }
          if (kMasked) {
#pragma unroll
            for (int i = 0; i < kQuarter; ++i)
              if (i >= nvis) Sf[i] = -INFINITY;
          }
          float c0 = fmax3(Sf[0], Sf[1], Sf[2]), c1 = fmax3(Sf[16], Sf[17], Sf[18]);
#pragma unroll
          for (int i = 3; i < 15; i += 2) {
            c0 = fmax3(c0, Sf[i], Sf[i + 1]);
            c1 = fmax3(c1, Sf[16 + i], Sf[17 + i]);
          }
          reinterpret_cast<float *>(&xm[b * BM + r])[g] = fmax3(fmax3(c0, c1, Sf[15]), Sf[31], Sf[31]);
          named_bar_or(1 + quad, 128, false);
          ++nbar;
          const float4 mx = xm[b * BM + r];
          mnew = fmaxf(m, fmaxf(fmaxf(mx.x, mx.y), fmaxf(mx.z, mx.w)));
          // x = s - (m' + E); masked entries stay -inf (p' = 0)
          rowsum = weights(mnew == -INFINITY ? 0.f : __fadd_rn(mnew, Ef), std::false_type{}, xq);
        } else {
          const float nb = __fadd_rn(m, Ef);
          rowsum = weights(nb, std::true_type{}, xq);
          mnew = m;
          // the exchange: the barrier itself reports whether any quarter of
          // any row of the quadrant passed the reference by more than 15; the
          // quarter maxima (as logits, xq + nb) are read back only then
          reinterpret_cast<float *>(&xm[b * BM + r])[g] = __fadd_rn(xq, nb);
          ++nbar;
          if (named_bar_or(1 + quad, 128, xq > 15.f - Ef)) {
            const float4 mx = xm[b * BM + r];
            mnew = fmaxf(m, fmaxf(fmaxf(mx.x, mx.y), fmaxf(mx.z, mx.w)));
            tmem_st_wait();  // the first weights are written before they are replaced
            rowsum = weights(__fadd_rn(mnew, Ef), std::true_type{}, xq);
          }
        }
        alpha = (m == -INFINITY) ? (mnew == -INFINITY ? 1.f : 0.f) : (mnew == m ? 1.f : ex2(__fsub_rn(m, mnew)));
      };
      if (__any_sync(0xffffffffu, nvis < kQuarter)) softmax_quarter(std::true_type{});
      else softmax_quarter(std::false_type{});
      l = __fadd_rn(__fmul_rn(alpha, l), rowsum);
      // O is stable once the P.V of tile j-1 is complete; this quarter's
      // warps rescale their 32 columns of it when the reference moved
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
        ok = mbar_wait(&bars->pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, abort, p.wait_ns);
        if (!ok) break;
        tc_fence_after();
        uint32_t o[32];
        tmem_ld32(colO, o);
        tmem_ld_wait(o);
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 v = fmul2(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])), a2);
          o[i] = __float_as_uint(v.x);
          o[i + 1] = __float_as_uint(v.y);
        }
        tmem_st32(colO, o);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[b]);
      m = mnew;
    }
    if (ok) ok = mbar_wait(&bars->pv_done[(T - 1) & 1], ((T - 1) >> 1) & 1, abort, p.wait_ns);
    // L = l_0 + l_1 + l_2 + l_3 in quarter order; every quarter writes its 32
    // channels of the partial O, quarter 0 also (m, L)
    if (ok) reinterpret_cast<float *>(&xl[r])[g] = l;
    for (; nbar <= T; ++nbar) named_bar_or(1 + quad, 128, false);
    if (!ok) {
      report(p.status, SAGE_ERR_TIMEOUT);
    } else {
      tc_fence_after();
      uint32_t o[32];
      tmem_ld32(colO, o);
      tmem_ld_wait(o);
      const bool unit_ok = SG_BOUNDS(unit < int(gridDim.x * gridDim.y * gridDim.z) && r < BM);
      if (valid && unit_ok) {
        float *dst = p.part_o + (int64_t(unit) * BM + r) * kD + kQuarter * g;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<float4 *>(dst + 4 * u) =
              make_float4(__uint_as_float(o[4 * u]), __uint_as_float(o[4 * u + 1]), __uint_as_float(o[4 * u + 2]),
                          __uint_as_float(o[4 * u + 3]));
      }
      if (g == 0 && unit_ok) {
        const float4 ls = xl[r];
        p.part_ml[int64_t(unit) * BM + r] =
            make_float2(m, __fadd_rn(__fadd_rn(__fadd_rn(ls.x, ls.y), ls.z), ls.w));
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

// Prepare the cache for the tensor cores: bf16 images of the K codes
// [Hkv][Npad][128], fp16 images of the V codes transposed [Hkv][128][Npad],
// kt = fl(ks * C) and vs as fp32 [Hkv][Npad], and the maximum of vs, for the
// first Nk keys (the visible ones; images and scales are zero from Nk to the
// end of the last tile).  grid (ceil(Nk / 128), Hkv), 256 threads.
__global__ void __launch_bounds__(256) int8kv_prep_kernel(const int8_t *__restrict__ kc, const int8_t *__restrict__ vc,
                                                          const __half *__restrict__ ks, const __half *__restrict__ vs,
                                                          int64_t kv_hs, int64_t sc_hs, int Nk, int Npad, float C,
                                                          __nv_bfloat16 *__restrict__ kimg, __half *__restrict__ vtimg,
                                                          float *__restrict__ kt, float *__restrict__ vsf,
                                                          uint32_t *__restrict__ vmax_bits) {
  __shared__ uint32_t vw[BN][kD / 4];  // the V tile's codes, key-major, 4 codes per word
  // the tile's fp16 images, channel-major; the 16-byte chunk of keys 8q..8q+7
  // of channel ch sits at chunk q ^ ((ch >> 2) & 15) of its row, so that the
  // transposing writes (one channel quad per lane) and the row reads below
  // spread over the banks
  __shared__ uint4 vt[kD][BN / 8];
  const int tile = blockIdx.x, g = blockIdx.y;
  const int key0 = tile * BN;
  const int8_t *ksrc = kc + g * kv_hs;
  const int8_t *vsrc = vc + g * kv_hs;
  // K: 128 keys x 128 codes -> bf16, 16 codes per thread-step
#pragma unroll
  for (int rep = 0; rep < 4; ++rep) {
    const int e = threadIdx.x + 256 * rep;  // 1024 chunks of 16 codes
    const int key = e >> 3, c16 = (e & 7) * 16;
    const int gk = key0 + key;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (gk < Nk) w = *reinterpret_cast<const uint4 *>(ksrc + int64_t(gk) * kD + c16);
    const int8_t *b = reinterpret_cast<const int8_t *>(&w);
    uint32_t o[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const __nv_bfloat162 t = __floats2bfloat162_rn(float(b[2 * u]), float(b[2 * u + 1]));
      o[u] = *reinterpret_cast<const uint32_t *>(&t);
    }
    if (SG_BOUNDS(gk < Npad && g < int(gridDim.y) && c16 + 16 <= kD)) {
      uint4 *dst = reinterpret_cast<uint4 *>(kimg + (int64_t(g) * Npad + gk) * kD + c16);
      dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
      dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
  }
  // V: the int8 tile lands key-major in shared memory (16-byte loads and
  // stores); each thread then reads one 4-code word of 8 consecutive keys
  // (a warp reads 32 consecutive words of a key row: no bank conflicts),
  // transposes the 4 x 8 bytes with byte permutes and puts 8 keys of each of
  // its 4 channels as fp16 into the channel-major shared tile, which then
  // leaves in whole 256-byte rows.  An int8 code b becomes the fp16 bit
  // pattern 0x6400 | (b ^ 0x80) = 1024 + b + 128, and subtracting 1152 leaves b.
#pragma unroll
  for (int rep = 0; rep < 4; ++rep) {
    const int e = threadIdx.x + 256 * rep;  // 1024 chunks of 16 codes
    const int key = e >> 3, w4 = (e & 7) * 4;
    const int gk = key0 + key;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (gk < Nk) w = *reinterpret_cast<const uint4 *>(vsrc + int64_t(gk) * kD + 4 * w4);
    *reinterpret_cast<uint4 *>(&vw[key][w4]) = w;
  }
  __syncthreads();
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
#pragma unroll
  for (int rep = 0; rep < 2; ++rep) {
    const int e = threadIdx.x + 256 * rep;  // 512 tasks: word (4 channels) x group of 8 keys
    const int wd = e & 31, kg = e >> 5;
    uint32_t x[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = vw[kg * 8 + k][wd] ^ 0x80808080u;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[4];
#pragma unroll
      for (int k = 0; k < 8; k += 2) {
        // bytes c of keys k and k+1, each under a 0x64 high byte
        const uint32_t t = __byte_perm(x[k], x[k + 1], uint32_t(c) | (uint32_t(4 + c) << 4));
        const uint32_t hb = __byte_perm(t, 0x64646464u, 0x5140u);
        const __half2 hv = __hsub2(*reinterpret_cast<const __half2 *>(&hb), bias);
        o[k >> 1] = *reinterpret_cast<const uint32_t *>(&hv);
      }
      const int ch = 4 * wd + c;
      vt[ch][kg ^ (wd & 15)] = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  __syncthreads();
  // rows out: 16 threads write the 256 bytes of one channel's 128 keys
#pragma unroll
  for (int rep = 0; rep < 8; ++rep) {
    const int ch = rep * 16 + (threadIdx.x >> 4), q = threadIdx.x & 15;
    if (SG_BOUNDS(ch < kD && key0 + q * 8 + 8 <= Npad && g < int(gridDim.y)))
      *reinterpret_cast<uint4 *>(vtimg + (int64_t(g) * kD + ch) * Npad + key0 + q * 8) = vt[ch][q ^ ((ch >> 2) & 15)];
  }
  if (threadIdx.x < BN) {
    const int gk = key0 + threadIdx.x;
    float ktv = 0.f, vsv = 0.f;
    if (gk < Nk) {
      ktv = __fmul_rn(__half2float(ks[g * sc_hs + gk]), C);
      vsv = __half2float(vs[g * sc_hs + gk]);
    }
    if (SG_BOUNDS(gk < Npad && g < int(gridDim.y))) {
      kt[int64_t(g) * Npad + gk] = ktv;
      vsf[int64_t(g) * Npad + gk] = vsv;
    }
    float mx = fabsf(vsv);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0) atomicMax(vmax_bits, __float_as_uint(mx));
  }
}

__global__ void zero_word_kernel(uint32_t *w) { *w = 0u; }

// Merge the split partials of each (query, head) row in split order and write
// bf16 output.  One warp per row, 4 channels per lane.
__global__ void __launch_bounds__(256) int8kv_combine_kernel(const float *__restrict__ part_o,
                                                             const float2 *__restrict__ part_ml,
                                                             int Nq, int Hq,
                                                             int G, int QT, int nqt, int nsplit,
                                                             __nv_bfloat16 *__restrict__ out, int64_t o_tok,
                                                             int64_t o_head) {
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= Nq * Hq) return;
  const int qi = gw / Hq, h = gw - qi * Hq;
  const int g = h / G, hl = h - g * G;
  const int qtile = qi / QT, r = (qi - qtile * QT) * G + hl;
  const int64_t unit0 = (int64_t(g) * nqt + qtile) * nsplit;
  if (!SG_BOUNDS(qtile < nqt && r < BM && g * G + hl < Hq)) return;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, part_ml[(unit0 + s) * BM + r].x);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < nsplit; ++s) {
    const float2 ml = part_ml[(unit0 + s) * BM + r];
    if (ml.x == -INFINITY) continue;
    const float wgt = ex2(__fsub_rn(ml.x, M));
    L = __fadd_rn(L, __fmul_rn(wgt, ml.y));
    const float4 o = *reinterpret_cast<const float4 *>(part_o + ((unit0 + s) * BM + r) * kD + 4 * lane);
    acc.x = __fadd_rn(acc.x, __fmul_rn(wgt, o.x));
    acc.y = __fadd_rn(acc.y, __fmul_rn(wgt, o.y));
    acc.z = __fadd_rn(acc.z, __fmul_rn(wgt, o.z));
    acc.w = __fadd_rn(acc.w, __fmul_rn(wgt, o.w));
  }
  // O and l both carry the factor 2^-E of the weights
  const float inv = __fdiv_rn(1.f, L);
  const __nv_bfloat162 a = __floats2bfloat162_rn(__fmul_rn(acc.x, inv), __fmul_rn(acc.y, inv));
  const __nv_bfloat162 b = __floats2bfloat162_rn(__fmul_rn(acc.z, inv), __fmul_rn(acc.w, inv));
  uint2 packed;
  packed.x = *reinterpret_cast<const uint32_t *>(&a);
  packed.y = *reinterpret_cast<const uint32_t *>(&b);
  *reinterpret_cast<uint2 *>(out + int64_t(qi) * o_tok + int64_t(h) * o_head + 4 * lane) = packed;
}

struct Layout {
  int G, QT, nqt, nsplit, Npad;
  size_t off_kimg, off_vt, off_kt, off_vs, off_vmax, off_po, off_pml, total;
};

// split-KV: the split count that minimises waves x (key tiles per unit + 2)
static int choose_nsplit(int64_t base_units, int tiles, int sms) {
  double best = 1e300;
  int nsplit = 1;
  for (int s = 1; s <= 16 && s <= tiles; ++s) {
    const int64_t units = base_units * s;
    const int64_t waves = (units + sms - 1) / sms;
    const double cost = double(waves) * (double(tiles) / s + 2.0);
    if (cost < best - 1e-9) {
      best = cost;
      nsplit = s;
    }
  }
  return nsplit;
}

// Workspace layout for a cache of Nk tokens (the split partials sized for the
// split count of the whole cache, an upper bound for any launch on it).
static Layout layout(int Nq, int Hq, int Hkv, int Nk, int sms) {
  Layout L;
  L.G = Hq / Hkv;
  L.QT = BM / L.G;
  L.nqt = ceil_div(Nq, L.QT);
  L.Npad = nk_pad(Nk);
  L.nsplit = choose_nsplit(int64_t(Hkv) * L.nqt, ceil_div(Nk, BN), sms);
  const int64_t units = int64_t(Hkv) * L.nqt * L.nsplit;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += (bytes + 255) & ~size_t(255);
    return o;
  };
  L.off_kimg = take(size_t(Hkv) * L.Npad * kD * 2);
  L.off_vt = take(size_t(Hkv) * L.Npad * kD * 2);
  L.off_kt = take(size_t(Hkv) * L.Npad * 4);
  L.off_vs = take(size_t(Hkv) * L.Npad * 4);
  L.off_vmax = take(4);
  L.off_po = take(size_t(units) * BM * kD * 4);
  L.off_pml = take(size_t(units) * BM * 8);
  L.total = off + 256;
  return L;
}

}  // namespace kv

size_t int8kv_workspace_bytes(int Nq, int Hq, int Hkv, int Nk) {
  return kv::layout(Nq, Hq, Hkv, Nk, current_sm_count()).total;
}

cudaError_t launch_int8kv(const Int8KVArgs &a, cudaStream_t st) {
  using namespace kv;
  const int sms = current_sm_count();
  const Layout L = layout(a.Nq, a.Hq, a.Hkv, a.Nk, sms);
  // Keys at positions q_pos0 + Nq and beyond are visible to no query: the
  // images, the split and the key loop cover only the first nvis keys, and
  // the rest of the cache is never read.
  const int nvis = a.q_pos0 + a.Nq;
  const int tiles_vis = ceil_div(nvis, BN);
  const int nsplit = std::min(choose_nsplit(int64_t(a.Hkv) * L.nqt, tiles_vis, sms), L.nsplit);
  uint8_t *ws = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(a.workspace) + 255) & ~uintptr_t(255));
  auto *kimg = reinterpret_cast<__nv_bfloat16 *>(ws + L.off_kimg);
  auto *vtimg = reinterpret_cast<__half *>(ws + L.off_vt);
  auto *kt = reinterpret_cast<float *>(ws + L.off_kt);
  auto *vsf = reinterpret_cast<float *>(ws + L.off_vs);
  auto *vmax = reinterpret_cast<uint32_t *>(ws + L.off_vmax);
  auto *po = reinterpret_cast<float *>(ws + L.off_po);
  auto *pml = reinterpret_cast<float2 *>(ws + L.off_pml);
  const float C = a.sm_scale * 1.44269504f;

  zero_word_kernel<<<1, 1, 0, st>>>(vmax);
  int8kv_prep_kernel<<<dim3(tiles_vis, a.Hkv), 256, 0, st>>>(
      a.k_cache, a.v_cache, static_cast<const __half *>(a.k_scale), static_cast<const __half *>(a.v_scale),
      a.kv_head_stride, a.scale_head_stride, nvis, L.Npad, C, kimg, vtimg, kt, vsf, vmax);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  CUtensorMap tq, tk, tv;
  if (!encode_tmap_3d(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.q, kD, a.Hq, a.Nq, uint64_t(a.q_head) * 2,
                      uint64_t(a.q_tok) * 2, 64, L.G, L.QT) ||
      !encode_tmap_3d(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kimg, kD, L.Npad, a.Hkv, kD * 2,
                      uint64_t(L.Npad) * kD * 2, 64, BN, 1) ||
      !encode_tmap_3d(&tv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, vtimg, L.Npad, kD, a.Hkv, uint64_t(L.Npad) * 2,
                      uint64_t(L.Npad) * kD * 2, 64, kD, 1))
    return cudaErrorInvalidValue;

  Params p;
  p.Nq = a.Nq;
  p.q_pos0 = a.q_pos0;
  p.Nk = a.Nk;
  p.Hkv = a.Hkv;
  p.G = L.G;
  p.QT = L.QT;
  p.nsplit = nsplit;
  p.Npad = L.Npad;
  p.kt = kt;
  p.vs = vsf;
  p.vmax_bits = vmax;
  p.part_o = po;
  p.part_ml = pml;
  p.status = a.status;
  p.wait_ns = a.wait_ns;
  p.fault = a.fault;
  static CtxOnce attr_done;
  e = set_smem_attr_once(reinterpret_cast<const void *>(int8kv_attn_kernel), kSmemBytes, &attr_done);
  if (e != cudaSuccess) return e;
  int8kv_attn_kernel<<<dim3(nsplit, L.nqt, a.Hkv), kThreads, kSmemBytes, st>>>(tq, tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int rows = a.Nq * a.Hq;
  int8kv_combine_kernel<<<ceil_div(rows, 8), 256, 0, st>>>(po, pml, a.Nq, a.Hq, L.G, L.QT, L.nqt, nsplit,
                                                          static_cast<__nv_bfloat16 *>(a.out), a.o_tok, a.o_head);
  return cudaGetLastError();
}

}  // namespace sg
