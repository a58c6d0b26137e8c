// Internal launchers shared by the C-ABI layer (api.cu) and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdint>

#include "../../include/sage_gb300.h"

namespace sg {

constexpr int kD = 128;          // head dimension
constexpr int kMeanChunk = 256;  // tokens per K-mean partial sum
constexpr int kTile = 128;       // keys per softmax tile

__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Bounds checks of the debug build (compiled with -DSAGE_DEBUG_BOUNDS, the
// stand-in for a memory sanitizer): SG_BOUNDS(cond) guards a global memory
// access whose index was computed in the kernel.  When cond is false the
// access is skipped and the first such site (file id * 100000 + source line)
// is recorded in a device word of the kernel's file; sage_debug_bounds reads
// and clears the words of all files.  Nothing traps.  In the normal build
// SG_BOUNDS(cond) is `true` and costs nothing.  Each kernel file names its id
// with SG_BOUNDS_FILE(name, id) at namespace sg scope.
#ifdef SAGE_DEBUG_BOUNDS
__device__ __forceinline__ bool bounds_check(bool ok, int32_t *word, int32_t site) {
  if (!ok) atomicCAS(word, 0, site);
  return ok;
}
#define SG_BOUNDS_FILE(name, id)                                             \
  namespace {                                                                \
  __device__ int32_t g_bounds_site;                                          \
  constexpr int32_t kBoundsFile = (id);                                      \
  }                                                                          \
  int32_t bounds_take_##name() {                                             \
    int32_t v = 0;                                                           \
    const int32_t z = 0;                                                     \
    if (cudaMemcpyFromSymbol(&v, g_bounds_site, sizeof(v)) != cudaSuccess) v = -1; \
    cudaMemcpyToSymbol(g_bounds_site, &z, sizeof(z));                        \
    return v;                                                                \
  }
#define SG_BOUNDS(cond) (::sg::bounds_check((cond), &g_bounds_site, kBoundsFile * 100000 + __LINE__))
#else
#define SG_BOUNDS_FILE(name, id) \
  int32_t bounds_take_##name() { return 0; }
#define SG_BOUNDS(cond) true
#endif
// the per-file readers (sage_debug_bounds calls them in file-id order)
int32_t bounds_take_quant();
int32_t bounds_take_prepare();
int32_t bounds_take_kvcache();
int32_t bounds_take_dense();
int32_t bounds_take_int8kv();
int32_t bounds_take_check();

// SM count of the current device (queried per call: a process may drive GPUs
// of different sizes).
int current_sm_count();
// Unique id (+1) of the calling thread's current CUDA context, 0 if none or
// unknown.  A new context (after cudaDeviceReset, say) gets a new id.
unsigned long long current_context_id();
// Per-device record of the context in which a one-time set-up was done.
struct CtxOnce {
  static constexpr int kDevices = 64;
  std::atomic<unsigned long long> ctx[kDevices] = {};
};
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per (kernel, device
// context): the attribute belongs to the context, so a process-wide "done"
// flag would leave a second device, or the device after a reset, without it.
cudaError_t set_smem_attr_once(const void *kernel, int bytes, CtxOnce *once);
__host__ __device__ inline int nk_pad(int nk) { return ceil_div(nk, kTile) * kTile; }

// Host-side argument checks shared by the entry points.
// A non-null pointer on a 16-byte boundary (TMA and vector accesses).
inline bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Element strides of bf16 rows that keep every row on a 16-byte boundary.
inline bool strides_ok(const sage_strides &s) {
  return s.b >= 0 && s.h >= 0 && s.n >= 0 && (s.b % 8) == 0 && (s.h % 8) == 0 && (s.n % 8) == 0;
}
// Problem sizes the grids and 32-bit index arithmetic support.
inline bool sizes_ok(int B, int H, int N) {
  return B >= 1 && H >= 1 && N >= 1 && int64_t(B) * H <= 65535 && N <= (1 << 28);
}
// sm_scale <= 0 selects 1/sqrt(d).
inline float default_scale(float sm_scale) { return sm_scale > 0.f ? sm_scale : float(1.0 / std::sqrt(double(kD))); }

// quantisers (quant.cu)
cudaError_t launch_quantize_qk(const void *q, sage_strides qs, const void *k, sage_strides ks, int B, int H,
                               int Nq, int Nk, int q_block, int k_block, int8_t *q_codes, float *q_scales,
                               int8_t *k_codes, float *k_scales, float *k_mean, float *partial,
                               cudaStream_t st);
// allocation-free variant: scratch in a static device array of this size
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
cudaError_t launch_quantize_qk_noalloc(const void *q, sage_strides qs, const void *k, sage_strides ks, int B,
                                       int H, int Nq, int Nk, int q_block, int k_block, int8_t *q_codes,
                                       float *q_scales, int8_t *k_codes, float *k_scales, float *k_mean,
                                       cudaStream_t st);
cudaError_t launch_quantize_v(const void *v, sage_strides vs, int B, int H, int Nk, uint8_t *v_codes,
                              float *v_scales, float *partial, float *inv, cudaStream_t st);

// the whole preparation in three launches (prepare.cu)
struct PrepArgs {
  const void *q, *k, *v;  // bf16 [B, H, N, 128] with element strides
  sage_strides qs, ks, vs;
  int B, H, Nq, Nk, q_block, k_block;
  bool images;            // Q/K out as exact fp16 images (else int8 codes)
  void *q_out, *k_out;    // [B, H, N, 128] int8 or fp16, contiguous
  float *q_scales, *k_scales, *k_mean;
  uint8_t *v_codes;       // [B, H, 128, Nk_pad]
  float *v_scales;
  float *workspace;       // prepare_workspace_bytes(B, H, Nk)
};
size_t prepare_workspace_bytes(int B, int H, int Nk);
cudaError_t launch_prepare(const PrepArgs &a, cudaStream_t st);

// dense attention (attn_dense.cu)
struct DenseArgs {
  const int8_t *q_codes;
  const float *q_scales;
  const int8_t *k_codes;
  const float *k_scales;
  const uint8_t *v_codes;
  const float *v_scales;
  int B, H, Nq, Nk, q_block, k_block;
  float sm_scale;
  void *out;
  sage_strides os;
  void *q_img, *k_img;  // workspace: fp16 images of the codes
  int32_t *status;
  int32_t *s_dump = nullptr;  // diagnostic score dump or null
  uint64_t wait_ns = 2000000000ull;  // limit of every bounded wait inside the kernel
  int fault = 0;                     // test hook (see sage_attn_fwd_fault_test)
  int causal = 0;                    // query i sees keys j <= i + (Nk - Nq)
  float *lse = nullptr;              // per-row log-sum-exp [B*H][Nq], or null
  bool images_ready = false;         // q_img / k_img already hold the images (no conversion launches)
};
size_t dense_workspace_bytes(int B, int H, int Nq, int Nk);
cudaError_t launch_attn_dense(const DenseArgs &a, cudaStream_t st);
// exact fp16 images of n int8 codes (16-byte aligned, n a multiple of 16)
cudaError_t launch_codes_to_f16(const int8_t *codes, void *img, int64_t n, cudaStream_t st);

// int8 KV-cache prompt attention (attn_int8kv.cu)
struct Int8KVArgs {
  const void *q;
  int64_t q_tok, q_head;
  const int8_t *k_cache, *v_cache;
  const void *k_scale, *v_scale;
  int64_t kv_head_stride, scale_head_stride;
  int Nq, q_pos0, Nk, Hq, Hkv;
  float sm_scale;
  void *out;
  int64_t o_tok, o_head;
  void *workspace;
  int32_t *status;
  uint64_t wait_ns = 2000000000ull;  // limit of every bounded wait in the kernel
  int fault = 0;                     // test hook of int8kv_prompt_attn_fault_test
};
size_t int8kv_workspace_bytes(int Nq, int Hq, int Hkv, int Nk);
cudaError_t launch_int8kv(const Int8KVArgs &a, cudaStream_t st);

// int8 KV-cache writer (kvcache.cu)
struct CacheWriteArgs {
  const void *k_src, *v_src;  // [N tokens][Hkv heads][128], bf16 or fp32
  int64_t src_tok, src_head;  // element strides
  bool f32;
  int N, Hkv, pos0, ncache;
  int8_t *k_cache, *v_cache;  // [Hkv][Ncache][128]
  int64_t cache_head;         // element stride between heads
  void *k_scale, *v_scale;    // fp16 [Hkv][Ncache]
  int64_t scale_head;
  int32_t *status;
};
cudaError_t launch_cache_write(const CacheWriteArgs &a, cudaStream_t st);

// check hook: the kernels' number-format conversions (check.cu)
cudaError_t launch_conversion_check(const float *x, int64_t n, uint8_t *e4m3, int8_t *i8, uint16_t *bf16,
                                    uint16_t *f16, cudaStream_t st);

// rate probes for the roofline (probe.cu)
cudaError_t launch_rate_probe(int kind, int iters, unsigned long long *cycles, float *sink, int32_t *status,
                              cudaStream_t st);

// tensor-map encoding through the driver entry point (api.cu)
bool encode_tmap_3d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                    uint32_t box2);

}  // namespace sg
