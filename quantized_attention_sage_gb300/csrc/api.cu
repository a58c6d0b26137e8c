// C ABI of the library: argument validation, workspace sizing, tensor-map
// encoding and the launches.  Declarations and their contracts are in
// include/sage_gb300.h.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "internal.h"

namespace sg {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D tiled tensor map, 128-byte swizzle, zero fill outside the tensor.
bool encode_tmap_3d(CUtensorMap *map, CUtensorMapDataType dtype, const void *base, uint64_t d0, uint64_t d1,
                    uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                    uint32_t box2) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {box0, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  CUresult r = fn(map, dtype, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Driver entry points for the current context's unique id (cuCtxGetId,
// CUDA 12.0+).  Ids are never reused within a process, so a cache keyed on the
// id notices when a device's context was destroyed and created again (after
// cudaDeviceReset, for instance), where a device ordinal would not.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext *);
  using GetId = CUresult (*)(CUcontext, unsigned long long *);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(p);
  });
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id + 1;  // 0 stands for "unknown"
}

int current_sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 148;
}

cudaError_t set_smem_attr_once(const void *kernel, int bytes, CtxOnce *once) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool slot = dev >= 0 && dev < CtxOnce::kDevices;
  const unsigned long long ctx = current_context_id();
  if (slot && ctx != 0 && once->ctx[dev].load(std::memory_order_acquire) == ctx) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  // the call above made the device's context current if it was not yet
  if (e == cudaSuccess && slot) once->ctx[dev].store(current_context_id(), std::memory_order_release);
  return e;
}

}  // namespace sg

using namespace sg;

namespace {

constexpr int kAbiVersion = 2;

sage_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SAGE_OK : SAGE_ERR_CUDA; }

}  // namespace

extern "C" {

const char *sage_status_string(sage_status s) {
  switch (s) {
    case SAGE_OK: return "ok";
    case SAGE_ERR_INVALID_ARG: return "invalid argument";
    case SAGE_ERR_UNSUPPORTED: return "unsupported configuration";
    case SAGE_ERR_CUDA: return "CUDA error";
    case SAGE_ERR_WORKSPACE: return "workspace too small";
    case SAGE_ERR_TIMEOUT: return "bounded device wait timed out";
    case SAGE_ERR_TOO_LARGE: return "problem exceeds the fixed scratch of the allocation-free entry point";
    case SAGE_ERR_NONFINITE: return "non-finite input or scale";
    default: return "unknown status";
  }
}

int sage_abi_version(void) { return kAbiVersion; }

sage_status sage_debug_bounds(int32_t *site) {
  if (site == nullptr) return SAGE_ERR_INVALID_ARG;
  *site = 0;
#ifdef SAGE_DEBUG_BOUNDS
  if (cudaDeviceSynchronize() != cudaSuccess) return SAGE_ERR_CUDA;
  int32_t (*const readers[])() = {bounds_take_quant, bounds_take_prepare, bounds_take_kvcache,
                                  bounds_take_dense,  bounds_take_int8kv,  bounds_take_check};
  for (auto rd : readers) {
    const int32_t v = rd();  // reads and clears that file's record
    if (v < 0) return SAGE_ERR_CUDA;
    if (*site == 0) *site = v;
  }
#endif
  return SAGE_OK;
}

int sage_debug_bounds_enabled(void) {
#ifdef SAGE_DEBUG_BOUNDS
  return 1;
#else
  return 0;
#endif
}

size_t sage_quantize_qk_workspace(int B, int H, int Nk) {
  if (B < 1 || H < 1 || Nk < 1) return 0;
  return size_t(B) * H * ceil_div(Nk, kMeanChunk) * kD * sizeof(float) + 16;
}

sage_status sage_quantize_qk(const void *q_bf16, sage_strides qs, const void *k_bf16, sage_strides ks, int B,
                             int H, int Nq, int Nk, int d, int q_block, int k_block, int8_t *q_codes,
                             float *q_scales, int8_t *k_codes, float *k_scales, float *k_mean, void *workspace,
                             size_t workspace_bytes, void *stream) {
  if (d != kD) return SAGE_ERR_UNSUPPORTED;
  if ((q_block != 64 && q_block != 128) || (k_block != 64 && k_block != 128)) return SAGE_ERR_UNSUPPORTED;
  if (!sizes_ok(B, H, Nq) || !sizes_ok(B, H, Nk)) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(q_bf16) || !aligned16(k_bf16) || !aligned16(q_codes) || !aligned16(k_codes) ||
      !aligned16(k_mean) || q_scales == nullptr || k_scales == nullptr || !aligned16(workspace))
    return SAGE_ERR_INVALID_ARG;
  if (!strides_ok(qs) || !strides_ok(ks)) return SAGE_ERR_INVALID_ARG;
  if (workspace_bytes < sage_quantize_qk_workspace(B, H, Nk)) return SAGE_ERR_WORKSPACE;
  return from_cuda(launch_quantize_qk(q_bf16, qs, k_bf16, ks, B, H, Nq, Nk, q_block, k_block, q_codes, q_scales,
                                      k_codes, k_scales, k_mean, static_cast<float *>(workspace),
                                      static_cast<cudaStream_t>(stream)));
}

sage_status sage_quantize_qk_noalloc(const void *q_bf16, sage_strides qs, const void *k_bf16, sage_strides ks,
                                     int B, int H, int Nq, int Nk, int d, int q_block, int k_block,
                                     int8_t *q_codes, float *q_scales, int8_t *k_codes, float *k_scales,
                                     float *k_mean, void *stream) {
  if (d != kD) return SAGE_ERR_UNSUPPORTED;
  if ((q_block != 64 && q_block != 128) || (k_block != 64 && k_block != 128)) return SAGE_ERR_UNSUPPORTED;
  if (!sizes_ok(B, H, Nq) || !sizes_ok(B, H, Nk)) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(q_bf16) || !aligned16(k_bf16) || !aligned16(q_codes) || !aligned16(k_codes) ||
      !aligned16(k_mean) || q_scales == nullptr || k_scales == nullptr)
    return SAGE_ERR_INVALID_ARG;
  if (!strides_ok(qs) || !strides_ok(ks)) return SAGE_ERR_INVALID_ARG;
  if (sage_quantize_qk_workspace(B, H, Nk) - 16 > kNoAllocScratchBytes) return SAGE_ERR_TOO_LARGE;
  return from_cuda(launch_quantize_qk_noalloc(q_bf16, qs, k_bf16, ks, B, H, Nq, Nk, q_block, k_block, q_codes,
                                              q_scales, k_codes, k_scales, k_mean,
                                              static_cast<cudaStream_t>(stream)));
}

size_t sage_quantize_qkv_workspace(int B, int H, int Nk) {
  if (B < 1 || H < 1 || Nk < 1) return 0;
  return prepare_workspace_bytes(B, H, Nk);
}

sage_status sage_quantize_qkv(const void *q_bf16, sage_strides qs, const void *k_bf16, sage_strides ks,
                              const void *v_bf16, sage_strides vs, int B, int H, int Nq, int Nk, int d, int q_block,
                              int k_block, int qk_format, void *q_out, float *q_scales, void *k_out, float *k_scales,
                              float *k_mean, uint8_t *v_codes, float *v_scales, void *workspace,
                              size_t workspace_bytes, void *stream) {
  if (d != kD) return SAGE_ERR_UNSUPPORTED;
  if ((q_block != 64 && q_block != 128) || (k_block != 64 && k_block != 128)) return SAGE_ERR_UNSUPPORTED;
  if (qk_format != SAGE_QK_INT8 && qk_format != SAGE_QK_F16) return SAGE_ERR_INVALID_ARG;
  if (!sizes_ok(B, H, Nq) || !sizes_ok(B, H, Nk)) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(q_bf16) || !aligned16(k_bf16) || !aligned16(v_bf16) || !aligned16(q_out) || !aligned16(k_out) ||
      !aligned16(k_mean) || !aligned16(v_codes) || !aligned16(v_scales) || q_scales == nullptr ||
      k_scales == nullptr || !aligned16(workspace))
    return SAGE_ERR_INVALID_ARG;
  if (!strides_ok(qs) || !strides_ok(ks) || !strides_ok(vs)) return SAGE_ERR_INVALID_ARG;
  if (workspace_bytes < sage_quantize_qkv_workspace(B, H, Nk)) return SAGE_ERR_WORKSPACE;
  PrepArgs a;
  a.q = q_bf16;
  a.k = k_bf16;
  a.v = v_bf16;
  a.qs = qs;
  a.ks = ks;
  a.vs = vs;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.q_block = q_block;
  a.k_block = k_block;
  a.images = qk_format == SAGE_QK_F16;
  a.q_out = q_out;
  a.k_out = k_out;
  a.q_scales = q_scales;
  a.k_scales = k_scales;
  a.k_mean = k_mean;
  a.v_codes = v_codes;
  a.v_scales = v_scales;
  a.workspace = static_cast<float *>(workspace);
  return from_cuda(launch_prepare(a, static_cast<cudaStream_t>(stream)));
}

size_t sage_quantize_v_workspace(int B, int H, int Nk) {
  if (B < 1 || H < 1 || Nk < 1) return 0;
  return (size_t(B) * H * ceil_div(Nk, kMeanChunk) * kD + size_t(B) * H * kD) * sizeof(float) + 16;
}

sage_status sage_quantize_v(const void *v_bf16, sage_strides vs, int B, int H, int Nk, int d, uint8_t *v_codes,
                            float *v_scales, void *workspace, size_t workspace_bytes, void *stream) {
  if (d != kD) return SAGE_ERR_UNSUPPORTED;
  if (!sizes_ok(B, H, Nk)) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(v_bf16) || !aligned16(v_codes) || !aligned16(v_scales) || !aligned16(workspace))
    return SAGE_ERR_INVALID_ARG;
  if (!strides_ok(vs)) return SAGE_ERR_INVALID_ARG;
  if (workspace_bytes < sage_quantize_v_workspace(B, H, Nk)) return SAGE_ERR_WORKSPACE;
  float *partial = static_cast<float *>(workspace);
  float *inv = partial + size_t(B) * H * ceil_div(Nk, kMeanChunk) * kD;
  return from_cuda(
      launch_quantize_v(v_bf16, vs, B, H, Nk, v_codes, v_scales, partial, inv, static_cast<cudaStream_t>(stream)));
}

size_t sage_attn_fwd_workspace(int B, int H, int Nq, int Nk) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return 0;
  return dense_workspace_bytes(B, H, Nq, Nk);
}

static sage_status attn_fwd_impl(const int8_t *q_codes, const float *q_scales, const int8_t *k_codes,
                                 const float *k_scales, const uint8_t *v_codes, const float *v_scales, int B, int H,
                                 int Nq, int Nk, int d, int q_block, int k_block, float sm_scale, void *out_bf16,
                                 sage_strides os, void *workspace, size_t workspace_bytes, int32_t *status_dev,
                                 int32_t *s_dump, void *stream, int fault = 0,
                                 uint64_t wait_ns = 2000000000ull, int causal = 0, float *lse = nullptr) {
  if (d != kD) return SAGE_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return SAGE_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return SAGE_ERR_UNSUPPORTED;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SAGE_ERR_INVALID_ARG;
  if ((q_block != 64 && q_block != 128) || (k_block != 64 && k_block != 128)) return SAGE_ERR_UNSUPPORTED;
  if (!sizes_ok(B, H, Nq) || !sizes_ok(B, H, Nk)) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(q_codes) || !aligned16(k_codes) || !aligned16(v_codes) || q_scales == nullptr ||
      k_scales == nullptr || v_scales == nullptr || !aligned16(out_bf16) || !aligned16(workspace))
    return SAGE_ERR_INVALID_ARG;
  if (!strides_ok(os)) return SAGE_ERR_INVALID_ARG;
  if (workspace_bytes < sage_attn_fwd_workspace(B, H, Nq, Nk)) return SAGE_ERR_WORKSPACE;
  DenseArgs a;
  a.q_codes = q_codes;
  a.q_scales = q_scales;
  a.k_codes = k_codes;
  a.k_scales = k_scales;
  a.v_codes = v_codes;
  a.v_scales = v_scales;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.q_block = q_block;
  a.k_block = k_block;
  a.sm_scale = default_scale(sm_scale);
  a.out = out_bf16;
  a.os = os;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  a.q_img = ws;
  a.k_img = ws + size_t(B) * H * Nq * kD * 2;
  a.status = status_dev;
  a.s_dump = s_dump;
  a.fault = fault;
  a.wait_ns = wait_ns;
  a.causal = causal;
  a.lse = lse;
  return from_cuda(launch_attn_dense(a, static_cast<cudaStream_t>(stream)));
}

sage_status sage_attn_fwd_f16(const void *q_f16, const float *q_scales, const void *k_f16, const float *k_scales,
                              const uint8_t *v_codes, const float *v_scales, int B, int H, int Nq, int Nk, int d,
                              int q_block, int k_block, float sm_scale, int causal, void *out_bf16, sage_strides os,
                              float *lse, int32_t *status_dev, void *stream) {
  if (d != kD) return SAGE_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return SAGE_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return SAGE_ERR_UNSUPPORTED;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SAGE_ERR_INVALID_ARG;
  if ((q_block != 64 && q_block != 128) || (k_block != 64 && k_block != 128)) return SAGE_ERR_UNSUPPORTED;
  if (!sizes_ok(B, H, Nq) || !sizes_ok(B, H, Nk)) return SAGE_ERR_INVALID_ARG;
  if (!aligned16(q_f16) || !aligned16(k_f16) || !aligned16(v_codes) || q_scales == nullptr || k_scales == nullptr ||
      v_scales == nullptr || !aligned16(out_bf16))
    return SAGE_ERR_INVALID_ARG;
  if (!strides_ok(os)) return SAGE_ERR_INVALID_ARG;
  DenseArgs a;
  a.q_codes = nullptr;
  a.q_scales = q_scales;
  a.k_codes = nullptr;
  a.k_scales = k_scales;
  a.v_codes = v_codes;
  a.v_scales = v_scales;
  a.B = B;
  a.H = H;
  a.Nq = Nq;
  a.Nk = Nk;
  a.q_block = q_block;
  a.k_block = k_block;
  a.sm_scale = default_scale(sm_scale);
  a.out = out_bf16;
  a.os = os;
  a.q_img = const_cast<void *>(q_f16);
  a.k_img = const_cast<void *>(k_f16);
  a.status = status_dev;
  a.causal = causal;
  a.lse = lse;
  a.images_ready = true;
  return from_cuda(launch_attn_dense(a, static_cast<cudaStream_t>(stream)));
}

sage_status sage_attn_fwd_ex(const int8_t *q_codes, const float *q_scales, const int8_t *k_codes,
                             const float *k_scales, const uint8_t *v_codes, const float *v_scales, int B, int H,
                             int Nq, int Nk, int d, int q_block, int k_block, float sm_scale, int causal,
                             void *out_bf16, sage_strides os, float *lse, void *workspace, size_t workspace_bytes,
                             int32_t *status_dev, void *stream) {
  return attn_fwd_impl(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, B, H, Nq, Nk, d, q_block, k_block,
                       sm_scale, out_bf16, os, workspace, workspace_bytes, status_dev, nullptr, stream, 0,
                       2000000000ull, causal, lse);
}

sage_status sage_attn_fwd(const int8_t *q_codes, const float *q_scales, const int8_t *k_codes,
                          const float *k_scales, const uint8_t *v_codes, const float *v_scales, int B, int H,
                          int Nq, int Nk, int d, int q_block, int k_block, float sm_scale, void *out_bf16,
                          sage_strides os, void *workspace, size_t workspace_bytes, int32_t *status_dev,
                          void *stream) {
  return attn_fwd_impl(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, B, H, Nq, Nk, d, q_block, k_block,
                       sm_scale, out_bf16, os, workspace, workspace_bytes, status_dev, nullptr, stream);
}

sage_status sage_attn_fwd_scores_dump(const int8_t *q_codes, const float *q_scales, const int8_t *k_codes,
                                      const float *k_scales, const uint8_t *v_codes, const float *v_scales, int B,
                                      int H, int Nq, int Nk, int d, int q_block, int k_block, float sm_scale,
                                      void *out_bf16, sage_strides os, void *workspace, size_t workspace_bytes,
                                      int32_t *status_dev, int32_t *s_dump, void *stream) {
  if (s_dump == nullptr || (reinterpret_cast<uintptr_t>(s_dump) & 15u)) return SAGE_ERR_INVALID_ARG;
  return attn_fwd_impl(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, B, H, Nq, Nk, d, q_block, k_block,
                       sm_scale, out_bf16, os, workspace, workspace_bytes, status_dev, s_dump, stream);
}



sage_status sage_attn_fwd_fault_test(const int8_t *q_codes, const float *q_scales, const int8_t *k_codes,
                                     const float *k_scales, const uint8_t *v_codes, const float *v_scales, int B,
                                     int H, int Nq, int Nk, int d, int q_block, int k_block, float sm_scale,
                                     void *out_bf16, sage_strides os, void *workspace, size_t workspace_bytes,
                                     int32_t *status_dev, uint64_t wait_limit_ns, int mode, void *stream) {
  if (status_dev == nullptr || wait_limit_ns == 0 || (mode != 1 && mode != 2)) return SAGE_ERR_INVALID_ARG;
  return attn_fwd_impl(q_codes, q_scales, k_codes, k_scales, v_codes, v_scales, B, H, Nq, Nk, d, q_block, k_block,
                       sm_scale, out_bf16, os, workspace, workspace_bytes, status_dev, nullptr, stream, mode,
                       wait_limit_ns);
}

size_t int8kv_prompt_attn_workspace(int Nq, int Hq, int Hkv, int Nk) {
  if (Nq < 1 || Hq < 1 || Hkv < 1 || Nk < 1 || Hq % Hkv != 0) return 0;
  return int8kv_workspace_bytes(Nq, Hq, Hkv, Nk);
}

}  // extern "C"

namespace {
sage_status int8kv_impl(const void *q_bf16, int64_t q_tok_stride, int64_t q_head_stride, const int8_t *k_cache,
                        const void *k_scale_f16, const int8_t *v_cache, const void *v_scale_f16,
                        int64_t kv_head_stride, int64_t scale_head_stride, int Nq, int q_pos0, int Nk, int Hq,
                        int Hkv, int d, float sm_scale, void *out_bf16, int64_t o_tok_stride,
                        int64_t o_head_stride, void *workspace, size_t workspace_bytes, int32_t *status_dev,
                        void *stream, uint64_t wait_ns, int fault) {
  if (d != kD) return SAGE_ERR_UNSUPPORTED;
  if (Nq < 1 || Nk < 1 || Hq < 1 || Hkv < 1 || q_pos0 < 0 || int64_t(q_pos0) + Nq > Nk) return SAGE_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return SAGE_ERR_INVALID_ARG;
  if (Hq / Hkv > 128 || Hkv > 65535 || Nk > (1 << 28)) return SAGE_ERR_UNSUPPORTED;
  if (!aligned16(q_bf16) || !aligned16(k_cache) || !aligned16(v_cache) || k_scale_f16 == nullptr ||
      v_scale_f16 == nullptr || !aligned16(out_bf16) || workspace == nullptr)
    return SAGE_ERR_INVALID_ARG;
  if (q_tok_stride < 0 || q_head_stride < 0 || (q_tok_stride % 8) || (q_head_stride % 8)) return SAGE_ERR_INVALID_ARG;
  if (o_tok_stride < 0 || o_head_stride < 0 || (o_tok_stride % 4) || (o_head_stride % 4)) return SAGE_ERR_INVALID_ARG;
  if (kv_head_stride < int64_t(Nk) * kD || (kv_head_stride % 16) || scale_head_stride < Nk)
    return SAGE_ERR_INVALID_ARG;
  if (workspace_bytes < int8kv_prompt_attn_workspace(Nq, Hq, Hkv, Nk)) return SAGE_ERR_WORKSPACE;
  Int8KVArgs a;
  a.q = q_bf16;
  a.q_tok = q_tok_stride;
  a.q_head = q_head_stride;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.k_scale = k_scale_f16;
  a.v_scale = v_scale_f16;
  a.kv_head_stride = kv_head_stride;
  a.scale_head_stride = scale_head_stride;
  a.Nq = Nq;
  a.q_pos0 = q_pos0;
  a.Nk = Nk;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.sm_scale = default_scale(sm_scale);
  a.out = out_bf16;
  a.o_tok = o_tok_stride;
  a.o_head = o_head_stride;
  a.workspace = workspace;
  a.status = status_dev;
  a.wait_ns = wait_ns;
  a.fault = fault;
  return from_cuda(launch_int8kv(a, static_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" {

sage_status int8kv_prompt_attn(const void *q_bf16, int64_t q_tok_stride, int64_t q_head_stride,
                               const int8_t *k_cache, const void *k_scale_f16, const int8_t *v_cache,
                               const void *v_scale_f16, int64_t kv_head_stride, int64_t scale_head_stride, int Nq,
                               int q_pos0, int Nk, int Hq, int Hkv, int d, float sm_scale, void *out_bf16,
                               int64_t o_tok_stride, int64_t o_head_stride, void *workspace,
                               size_t workspace_bytes, int32_t *status_dev, void *stream) {
  return int8kv_impl(q_bf16, q_tok_stride, q_head_stride, k_cache, k_scale_f16, v_cache, v_scale_f16, kv_head_stride,
                     scale_head_stride, Nq, q_pos0, Nk, Hq, Hkv, d, sm_scale, out_bf16, o_tok_stride, o_head_stride,
                     workspace, workspace_bytes, status_dev, stream, 2000000000ull, 0);
}

sage_status int8kv_prompt_attn_fault_test(const void *q_bf16, int64_t q_tok_stride, int64_t q_head_stride,
                                          const int8_t *k_cache, const void *k_scale_f16, const int8_t *v_cache,
                                          const void *v_scale_f16, int64_t kv_head_stride,
                                          int64_t scale_head_stride, int Nq, int q_pos0, int Nk, int Hq, int Hkv,
                                          int d, float sm_scale, void *out_bf16, int64_t o_tok_stride,
                                          int64_t o_head_stride, void *workspace, size_t workspace_bytes,
                                          int32_t *status_dev, uint64_t wait_limit_ns, int mode, void *stream) {
  if (status_dev == nullptr || wait_limit_ns == 0 || (mode != 1 && mode != 2)) return SAGE_ERR_INVALID_ARG;
  return int8kv_impl(q_bf16, q_tok_stride, q_head_stride, k_cache, k_scale_f16, v_cache, v_scale_f16, kv_head_stride,
                     scale_head_stride, Nq, q_pos0, Nk, Hq, Hkv, d, sm_scale, out_bf16, o_tok_stride, o_head_stride,
                     workspace, workspace_bytes, status_dev, stream, wait_limit_ns, mode);
}

sage_status sage_conversion_check(const float *x, int64_t n, uint8_t *e4m3, int8_t *i8, uint16_t *bf16,
                                  uint16_t *f16, void *stream) {
  if (n < 2 || (n % 2) || !aligned16(x) || !aligned16(e4m3) || !aligned16(i8) || !aligned16(bf16) ||
      !aligned16(f16))
    return SAGE_ERR_INVALID_ARG;
  return from_cuda(launch_conversion_check(x, n, e4m3, i8, bf16, f16, static_cast<cudaStream_t>(stream)));
}

sage_status sage_probe_rates(int kind, int iters, unsigned long long *cycles, float *sink, int32_t *status_dev,
                             void *stream) {
  if (kind < 0 || kind > 2 || iters < 1 || iters > (1 << 20) || cycles == nullptr || sink == nullptr ||
      status_dev == nullptr)
    return SAGE_ERR_INVALID_ARG;
  return from_cuda(launch_rate_probe(kind, iters, cycles, sink, status_dev, static_cast<cudaStream_t>(stream)));
}

sage_status sage_shard_range(int64_t units, int world, int rank, int64_t *begin, int64_t *end) {
  if (units < 0 || world < 1 || rank < 0 || rank >= world || begin == nullptr || end == nullptr)
    return SAGE_ERR_INVALID_ARG;
  const int64_t base = units / world, extra = units % world;
  // ranks below `extra` take base + 1 units, the rest base
  const int64_t b = int64_t(rank) * base + (rank < extra ? rank : extra);
  *begin = b;
  *end = b + base + (rank < extra ? 1 : 0);
  return SAGE_OK;
}

sage_status int8kv_cache_write(const void *k_src, const void *v_src, int src_dtype, int64_t src_tok_stride,
                               int64_t src_head_stride, int N, int Hkv, int d, int pos0, int8_t *k_cache,
                               int8_t *v_cache, int64_t cache_head_stride, int Ncache, void *k_scale_f16,
                               void *v_scale_f16, int64_t scale_head_stride, int32_t *status_dev, void *stream) {
  if (d != kD) return SAGE_ERR_UNSUPPORTED;
  if (src_dtype != SAGE_DTYPE_BF16 && src_dtype != SAGE_DTYPE_F32) return SAGE_ERR_UNSUPPORTED;
  if (N < 1 || Hkv < 1 || pos0 < 0 || Ncache < 1 || int64_t(pos0) + N > Ncache) return SAGE_ERR_INVALID_ARG;
  const uintptr_t src_align = src_dtype == SAGE_DTYPE_F32 ? 15u : 7u;
  if (k_src == nullptr || v_src == nullptr || (reinterpret_cast<uintptr_t>(k_src) & src_align) ||
      (reinterpret_cast<uintptr_t>(v_src) & src_align))
    return SAGE_ERR_INVALID_ARG;
  if (src_tok_stride < 0 || src_head_stride < 0 || (src_tok_stride % 4) || (src_head_stride % 4))
    return SAGE_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || cache_head_stride < int64_t(Ncache) * kD ||
      (cache_head_stride % 16))
    return SAGE_ERR_INVALID_ARG;
  if (k_scale_f16 == nullptr || v_scale_f16 == nullptr || (reinterpret_cast<uintptr_t>(k_scale_f16) & 1u) ||
      (reinterpret_cast<uintptr_t>(v_scale_f16) & 1u) || scale_head_stride < Ncache)
    return SAGE_ERR_INVALID_ARG;
  CacheWriteArgs a;
  a.k_src = k_src;
  a.v_src = v_src;
  a.src_tok = src_tok_stride;
  a.src_head = src_head_stride;
  a.f32 = src_dtype == SAGE_DTYPE_F32;
  a.N = N;
  a.Hkv = Hkv;
  a.pos0 = pos0;
  a.ncache = Ncache;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.cache_head = cache_head_stride;
  a.k_scale = k_scale_f16;
  a.v_scale = v_scale_f16;
  a.scale_head = scale_head_stride;
  a.status = status_dev;
  return from_cuda(launch_cache_write(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
