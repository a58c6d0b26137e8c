// The dense path as one call: sage_attention on device buffers (the fused
// preparation, sage_quantize_qkv with fp16 images of the Q/K codes, then the
// attention kernel, intermediates in the caller's workspace) and
// sage_attention_host on host-resident Q, K, V and output, with the
// host<->device copies and the preparation overlapped with the attention
// kernels (the rest of this comment).
//
// The (batch, head) problems are independent, so the heads are cut into
// chunks (growing 1, 2, 4, ... up to the chunk size and shrinking again at
// the end, so that the first copy in and the last copy out are short).  Two
// streams share the work:
//   staging stream (the caller's copy stream): host->device copies, the
//            preparation (three launches: reduction, finalisation, encoding
//            into fp16 images of the Q/K codes and E4M3 V codes),
//            device->host copies;
//   compute stream: the attention kernel of one chunk after another.
// While the compute stream attends chunk c, the staging stream copies chunk
// c+2 in, then (once chunk c is done) copies its output out and quantizes
// chunk c+2, so that neither the copies nor the short quantizer launches
// sit between two attention launches.  Inputs, outputs and the quantized
// intermediates (codes, scales, images) are double-buffered in the caller's
// workspace (slot c % 2), and so are the events that order the streams.
//
// Per chunk c (slot s = c % 2), in stream order:
//   staging: H2D q, k, v -> in[s]; prepare in[s] -> images[s], codes[s];
//            record q_ready[s]
//   compute: wait q_ready[s]; attention kernel on images[s], codes[s] -> out[s];
//            record done[s]
//   staging: wait done[s]; D2H out[s]; prepare chunk c+2 into images[s], codes[s]
// H2D of chunk c+2 is queued before the wait for done[c]: in[s] was last read
// by the preparation of chunk c, earlier on the same stream.  The preparation
// of chunk c+2 follows done[c] (images[s] have been read) and D2H of chunk c
// (out[s] is drained before attention(c+2), which waits for q_ready[s] as
// recorded for chunk c+2).
// The staging stream first waits for the work already queued on the compute
// stream; at the end the compute stream waits for the last D2H, so the caller
// synchronises one stream.  The cross-stream order uses six events (q_ready
// and done as two-slot rings, start, last), created once per thread and device
// context and reused by every call: recording an event again is safe because
// every wait on its previous record has been enqueued by then, and a call
// then creates and destroys no driver objects.
#include <cuda_runtime.h>

#include <vector>

#include "internal.h"

namespace {

constexpr size_t kAlign = 256;

// The six events of sage_attention_host for the calling thread and the current
// device context (created on first use; a context created again after a reset
// gets new ones).
struct HostEvents {
  unsigned long long ctx = 0;
  cudaEvent_t ev[6] = {};
};
cudaError_t host_events(cudaEvent_t (&out)[6]) {
  thread_local HostEvents cache[sg::CtxOnce::kDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= sg::CtxOnce::kDevices) return cudaErrorInvalidDevice;
  HostEvents &h = cache[dev];
  const unsigned long long ctx = sg::current_context_id();
  if (ctx == 0) return cudaErrorDeviceUninitialized;  // no current context
  if (h.ctx != ctx) {  // first use here, or the context was destroyed with its events
    for (cudaEvent_t &x : h.ev) {
      e = cudaEventCreateWithFlags(&x, cudaEventDisableTiming);
      if (e != cudaSuccess) {
        h.ctx = 0;
        return e;
      }
    }
    h.ctx = ctx;
  }
  for (int i = 0; i < 6; ++i) out[i] = h.ev[i];
  return cudaSuccess;
}

size_t up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

struct HostLayout {
  int hc;                               // heads per chunk
  size_t q_bytes, k_bytes, o_bytes;     // bf16 chunk buffers
  size_t off_in[2][3], off_out[2];      // inputs (q, k, v) and output per slot
  size_t off_qs[2], off_ks[2], off_mu[2], off_vc[2], off_vs[2], off_wp[2];
  size_t off_qi[2], off_ki[2];          // fp16 images of the Q and K codes the attention reads
  size_t wp, total;
};

HostLayout host_layout(int B, int H, int Nq, int Nk, int head_chunk) {
  HostLayout L{};
  const int BH = B * H;
  L.hc = head_chunk < BH ? head_chunk : BH;
  const size_t hc = size_t(L.hc);
  L.q_bytes = hc * Nq * sg::kD * 2;
  L.k_bytes = hc * Nk * sg::kD * 2;
  L.o_bytes = L.q_bytes;
  L.wp = sage_quantize_qkv_workspace(1, L.hc, Nk);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += up(bytes);
    return o;
  };
  for (int s = 0; s < 2; ++s) {
    L.off_in[s][0] = take(L.q_bytes);
    L.off_in[s][1] = take(L.k_bytes);
    L.off_in[s][2] = take(L.k_bytes);
    L.off_out[s] = take(L.o_bytes);
    L.off_qs[s] = take(hc * sg::ceil_div(Nq, 64) * sizeof(float));  // blocks of 64 or 128 tokens
    L.off_ks[s] = take(hc * sg::ceil_div(Nk, 64) * sizeof(float));
    L.off_mu[s] = take(hc * sg::kD * sizeof(float));
    L.off_vc[s] = take(hc * sg::kD * size_t(sg::nk_pad(Nk)));
    L.off_vs[s] = take(hc * sg::kD * sizeof(float));
    L.off_wp[s] = take(L.wp);
    L.off_qi[s] = take(hc * Nq * sg::kD * 2);
    L.off_ki[s] = take(hc * Nk * sg::kD * 2);
  }
  L.total = off + kAlign;  // room to align the base
  return L;
}

// First head of each chunk, then B*H: sizes 1, 2, 4, ... up to hc, hc while
// heads remain, then halving again towards 1, so that the copies nothing can
// hide (the first chunk in, the last chunk out) are small.
std::vector<int> chunk_starts(int BH, int hc) {
  std::vector<int> up_sz, down_sz, mid, first;
  int left = BH;
  for (int n = 1; n < hc && left > 0; n *= 2) {
    const int a = n < left ? n : left;
    up_sz.push_back(a);
    left -= a;
    if (left > 0) {
      const int b = n < left ? n : left;
      down_sz.push_back(b);
      left -= b;
    }
  }
  while (left > 0) {
    const int a = hc < left ? hc : left;
    mid.push_back(a);
    left -= a;
  }
  int h = 0;
  for (int n : up_sz) first.push_back(h), h += n;
  for (int n : mid) first.push_back(h), h += n;
  for (auto it = down_sz.rbegin(); it != down_sz.rend(); ++it) first.push_back(h), h += *it;
  first.push_back(h);
  return first;
}

// sage_attention: the preparation and the attention on device buffers in one
// call.  The intermediates of all heads live in the caller's workspace.
struct DeviceLayout {
  size_t off_qi, off_ki, off_qs, off_ks, off_mu, off_vc, off_vs, off_wp;
  size_t wp, total;
};

DeviceLayout device_layout(int B, int H, int Nq, int Nk) {
  DeviceLayout L{};
  const size_t BH = size_t(B) * H;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += up(bytes);
    return o;
  };
  L.off_qi = take(BH * Nq * sg::kD * 2);
  L.off_ki = take(BH * Nk * sg::kD * 2);
  L.off_qs = take(BH * sg::ceil_div(Nq, 64) * sizeof(float));  // blocks of 64 or 128 tokens
  L.off_ks = take(BH * sg::ceil_div(Nk, 64) * sizeof(float));
  L.off_mu = take(BH * sg::kD * sizeof(float));
  L.off_vc = take(BH * sg::kD * size_t(sg::nk_pad(Nk)));
  L.off_vs = take(BH * sg::kD * sizeof(float));
  L.wp = sage_quantize_qkv_workspace(B, H, Nk);
  L.off_wp = take(L.wp);
  L.total = off + kAlign;  // room to align the base
  return L;
}

}  // namespace

extern "C" {

size_t sage_attention_workspace(int B, int H, int Nq, int Nk) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return 0;
  return device_layout(B, H, Nq, Nk).total;
}

sage_status sage_attention(const void *q_bf16, sage_strides qs, const void *k_bf16, sage_strides ks,
                           const void *v_bf16, sage_strides vs, int B, int H, int Nq, int Nk, int d, int q_block,
                           int k_block, float sm_scale, int causal, void *out_bf16, sage_strides os, float *lse,
                           void *workspace, size_t workspace_bytes, int32_t *status_dev, void *stream) {
  // every argument is checked here, before the first step is enqueued
  if (d != sg::kD) return SAGE_ERR_UNSUPPORTED;
  if ((q_block != 64 && q_block != 128) || (k_block != 64 && k_block != 128)) return SAGE_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return SAGE_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return SAGE_ERR_UNSUPPORTED;
  if (!sg::sizes_ok(B, H, Nq) || !sg::sizes_ok(B, H, Nk)) return SAGE_ERR_INVALID_ARG;
  if (!sg::aligned16(q_bf16) || !sg::aligned16(k_bf16) || !sg::aligned16(v_bf16) || !sg::aligned16(out_bf16) ||
      workspace == nullptr)
    return SAGE_ERR_INVALID_ARG;
  if (!sg::strides_ok(qs) || !sg::strides_ok(ks) || !sg::strides_ok(vs) || !sg::strides_ok(os))
    return SAGE_ERR_INVALID_ARG;
  if (lse != nullptr && (reinterpret_cast<uintptr_t>(lse) & 3u)) return SAGE_ERR_INVALID_ARG;
  const DeviceLayout L = device_layout(B, H, Nq, Nk);
  if (workspace_bytes < L.total) return SAGE_ERR_WORKSPACE;
  uint8_t *ws = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(workspace) + kAlign - 1) &
                                            ~uintptr_t(kAlign - 1));
  auto *qsc = reinterpret_cast<float *>(ws + L.off_qs);
  auto *ksc = reinterpret_cast<float *>(ws + L.off_ks);
  auto *vc = reinterpret_cast<uint8_t *>(ws + L.off_vc);
  auto *vsc = reinterpret_cast<float *>(ws + L.off_vs);
  sage_status r = sage_quantize_qkv(q_bf16, qs, k_bf16, ks, v_bf16, vs, B, H, Nq, Nk, sg::kD, q_block, k_block,
                                    SAGE_QK_F16, ws + L.off_qi, qsc, ws + L.off_ki, ksc,
                                    reinterpret_cast<float *>(ws + L.off_mu), vc, vsc, ws + L.off_wp, L.wp, stream);
  if (r == SAGE_OK)
    r = sage_attn_fwd_f16(ws + L.off_qi, qsc, ws + L.off_ki, ksc, vc, vsc, B, H, Nq, Nk, sg::kD, q_block, k_block,
                          sm_scale, causal, out_bf16, os, lse, status_dev, stream);
  return r;
}

size_t sage_attention_host_workspace(int B, int H, int Nq, int Nk, int head_chunk) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || head_chunk < 1) return 0;
  return host_layout(B, H, Nq, Nk, head_chunk).total;
}

sage_status sage_attention_host(const void *q_host, const void *k_host, const void *v_host, void *out_host, int B,
                                int H, int Nq, int Nk, int d, int q_block, int k_block, float sm_scale, int causal,
                                int head_chunk, void *workspace, size_t workspace_bytes, int32_t *status_dev,
                                void *compute_stream, void *copy_stream) {
  if (d != sg::kD) return SAGE_ERR_UNSUPPORTED;
  if ((q_block != 64 && q_block != 128) || (k_block != 64 && k_block != 128)) return SAGE_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return SAGE_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return SAGE_ERR_UNSUPPORTED;
  if (!sg::sizes_ok(B, H, Nq) || !sg::sizes_ok(B, H, Nk) || head_chunk < 1) return SAGE_ERR_INVALID_ARG;
  if (q_host == nullptr || k_host == nullptr || v_host == nullptr || out_host == nullptr || workspace == nullptr)
    return SAGE_ERR_INVALID_ARG;
  if (copy_stream == nullptr || copy_stream == compute_stream) return SAGE_ERR_INVALID_ARG;
  const HostLayout L = host_layout(B, H, Nq, Nk, head_chunk);
  if (workspace_bytes < L.total) return SAGE_ERR_WORKSPACE;
  uint8_t *ws = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(workspace) + kAlign - 1) &
                                            ~uintptr_t(kAlign - 1));
  cudaStream_t cs = static_cast<cudaStream_t>(compute_stream), xs = static_cast<cudaStream_t>(copy_stream);

  const std::vector<int> first = chunk_starts(B * H, L.hc);
  const int C = int(first.size()) - 1;
  sage_status st = SAGE_OK;
  auto fail = [&](sage_status s) {
    if (st == SAGE_OK) st = s;
  };
  auto ck = [&](cudaError_t e) {
    if (e != cudaSuccess) fail(SAGE_ERR_CUDA);
    return e == cudaSuccess;
  };
  cudaEvent_t evs[6];
  if (!ck(host_events(evs))) return st;
  cudaEvent_t *q_ready = evs, *done = evs + 2;  // slot c & 1 for head group c
  cudaEvent_t start = evs[4], last = evs[5];
  // the staging stream starts after everything already queued on the compute
  // stream (e.g. a previous call that used the same workspace)
  if (st == SAGE_OK && ck(cudaEventRecord(start, cs))) ck(cudaStreamWaitEvent(xs, start, 0));

  const size_t qrow = size_t(Nq) * sg::kD * 2, krow = size_t(Nk) * sg::kD * 2;  // bytes per head
  auto heads_of = [&](int c) { return first[c + 1] - first[c]; };
  auto q_strides = [&](int n) { return sage_strides{int64_t(n) * Nq * sg::kD, int64_t(Nq) * sg::kD, sg::kD}; };
  auto kv_strides = [&](int n) { return sage_strides{int64_t(n) * Nk * sg::kD, int64_t(Nk) * sg::kD, sg::kD}; };
  auto h2d = [&](int c) {
    const int s = c & 1, n = heads_of(c);
    const size_t h0 = size_t(first[c]);
    ck(cudaMemcpyAsync(ws + L.off_in[s][0], static_cast<const uint8_t *>(q_host) + h0 * qrow, n * qrow,
                       cudaMemcpyHostToDevice, xs));
    ck(cudaMemcpyAsync(ws + L.off_in[s][1], static_cast<const uint8_t *>(k_host) + h0 * krow, n * krow,
                       cudaMemcpyHostToDevice, xs));
    ck(cudaMemcpyAsync(ws + L.off_in[s][2], static_cast<const uint8_t *>(v_host) + h0 * krow, n * krow,
                       cudaMemcpyHostToDevice, xs));
  };
  // the preparation of chunk c on the staging stream (fp16 images of the Q/K
  // codes, so that only the attention kernel runs on the compute stream),
  // then q_ready[c]
  auto quantize = [&](int c) {
    const int s = c & 1, n = heads_of(c);
    const sage_status r = sage_quantize_qkv(
        ws + L.off_in[s][0], q_strides(n), ws + L.off_in[s][1], kv_strides(n), ws + L.off_in[s][2], kv_strides(n), 1,
        n, Nq, Nk, sg::kD, q_block, k_block, SAGE_QK_F16, ws + L.off_qi[s], reinterpret_cast<float *>(ws + L.off_qs[s]),
        ws + L.off_ki[s], reinterpret_cast<float *>(ws + L.off_ks[s]), reinterpret_cast<float *>(ws + L.off_mu[s]),
        reinterpret_cast<uint8_t *>(ws + L.off_vc[s]), reinterpret_cast<float *>(ws + L.off_vs[s]), ws + L.off_wp[s],
        L.wp, xs);
    if (r != SAGE_OK) {
      fail(r);
      return;
    }
    if (st == SAGE_OK) ck(cudaEventRecord(q_ready[c & 1], xs));
  };
  for (int c = 0; c < 2 && c < C && st == SAGE_OK; ++c) {
    h2d(c);
    if (st == SAGE_OK) quantize(c);
  }
  for (int c = 0; c < C && st == SAGE_OK; ++c) {
    const int s = c & 1, n = heads_of(c);
    if (!ck(cudaStreamWaitEvent(cs, q_ready[c & 1], 0))) break;
    // the attention kernel alone (arguments checked above; images written by the staging stream)
    sg::DenseArgs a;
    a.q_codes = nullptr;  // the attention reads the images
    a.q_scales = reinterpret_cast<const float *>(ws + L.off_qs[s]);
    a.k_codes = nullptr;
    a.k_scales = reinterpret_cast<const float *>(ws + L.off_ks[s]);
    a.v_codes = reinterpret_cast<const uint8_t *>(ws + L.off_vc[s]);
    a.v_scales = reinterpret_cast<const float *>(ws + L.off_vs[s]);
    a.B = 1;
    a.H = n;
    a.Nq = Nq;
    a.Nk = Nk;
    a.q_block = q_block;
    a.k_block = k_block;
    a.sm_scale = sg::default_scale(sm_scale);
    a.out = ws + L.off_out[s];
    a.os = q_strides(n);
    a.q_img = ws + L.off_qi[s];
    a.k_img = ws + L.off_ki[s];
    a.status = status_dev;
    a.causal = causal;
    a.images_ready = true;
    if (!ck(sg::launch_attn_dense(a, cs))) break;
    if (!ck(cudaEventRecord(done[c & 1], cs))) break;
    if (c + 2 < C) h2d(c + 2);  // in[s] was last read by quantize(c), earlier on this stream
    if (st != SAGE_OK || !ck(cudaStreamWaitEvent(xs, done[c & 1], 0))) break;
    ck(cudaMemcpyAsync(static_cast<uint8_t *>(out_host) + size_t(first[c]) * qrow, ws + L.off_out[s], n * qrow,
                       cudaMemcpyDeviceToHost, xs));
    if (c + 2 < C && st == SAGE_OK) quantize(c + 2);
  }
  if (st == SAGE_OK && ck(cudaEventRecord(last, xs))) ck(cudaStreamWaitEvent(cs, last, 0));
  return st;
}

}  // extern "C"
