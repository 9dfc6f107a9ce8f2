// attn_host.cu - attention on host buffers, declared in include/attn_fwd.h.
//
// The caller's inputs and output live in host memory (page-locked for the
// copies to overlap anything). The problem is cut into chunks; each chunk's
// inputs go to the device on one internal stream, its kernel runs on one of two
// compute streams once they have landed, and its output comes back on a third
// stream once the kernel is done. So chunk i's kernel overlaps chunk i+1's
// upload and chunk i-1's download, and neighbouring kernels can fill each
// other's tail waves. Events order everything; nothing on the host waits. The
// device tensors are in the caller's workspace, each chunk's share packed
// densely there in the caller's layout.
//
// How a problem is cut into chunks is in host_plan.h. A chunk of a dense
// problem is an attn_fwd_ex call on its own dense sub-tensors; a chunk of a
// packed variable-length batch is attn_fwd_varlen over the full tensors with
// the offsets array advanced to its first sequence (the offsets stay absolute).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "attn_fwd.h"
#include "host_plan.h"

namespace {

using attn_plan::Chunk;
using attn_plan::kMaxChunks;
using attn_plan::round_up;
using attn_plan::SeqChunk;
using attn_plan::Span;

constexpr int kMaxDevices = 64;
constexpr int64_t kAlign = 256;

// Per device: the three internal streams and the events of one call. A call
// holds the device's mutex while it enqueues (no host waits inside), so calls
// from several threads are serialised only for that short time.
struct DeviceStreams {
  std::mutex mu;
  bool ready = false;
  int status = ATTN_OK;
  cudaStream_t in = nullptr, out = nullptr, comp[2] = {nullptr, nullptr};
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t landed[kMaxChunks] = {}, computed[kMaxChunks] = {}, comp_done[2] = {};
};
DeviceStreams g_dev[kMaxDevices];

int setup(DeviceStreams& d) {
  if (d.ready) return ATTN_OK;
  if (d.status != ATTN_OK) return d.status;
  bool ok = cudaStreamCreateWithFlags(&d.in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&d.out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&d.comp[0], cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&d.comp[1], cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&d.start, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&d.done, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < kMaxChunks; ++i)
    ok = cudaEventCreateWithFlags(&d.landed[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&d.computed[i], cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; ok && i < 2; ++i)
    ok = cudaEventCreateWithFlags(&d.comp_done[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    d.status = ATTN_ERR_LAUNCH;
    return d.status;
  }
  d.ready = true;
  return ATTN_OK;
}

// One span's copy (nothing for rows == 0): a plain copy when its runs are
// contiguous on both sides, else a 2-D copy.
bool copy_span(char* dst_base, const char* src_base, const Span& s, cudaMemcpyKind kind,
               cudaStream_t st) {
  if (s.rows == 0) return true;
  const attn_plan::CopyArgs a = attn_plan::copy_args(s, kind == cudaMemcpyHostToDevice);
  if (a.rows == 1 || (a.dpitch == a.width && a.spitch == a.width))
    return cudaMemcpyAsync(dst_base + a.dst, src_base + a.src, a.width * a.rows, kind, st) ==
           cudaSuccess;
  return cudaMemcpy2DAsync(dst_base + a.dst, a.dpitch, src_base + a.src, a.spitch, a.width,
                           a.rows, kind, st) == cudaSuccess;
}

}  // namespace

extern "C" {

int64_t attn_fwd_host_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk,
                                      int64_t d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Sk < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  const int64_t kLim = int64_t(1) << 31;
  if (B > kLim || Hq > kLim || Sq > kLim || Sk > kLim) return ATTN_ERR_TOO_LARGE;
  const int64_t big = int64_t(1) << 58;  // keeps the byte counts below 2^62
  if (B * Hq > big / 256 / Sq || B * Hkv > big / 256 / Sk) return ATTN_ERR_TOO_LARGE;
  return 2 * round_up(B * Hq * Sq * 256, kAlign) + 2 * round_up(B * Hkv * Sk * 256, kAlign);
}

int attn_fwd_host(const void* q, const void* k, const void* v, void* out, int layout, int64_t B,
                  int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t d, float scale,
                  int rounding_mode, int flags, void* workspace, int64_t workspace_bytes,
                  void* stream) {
  // ---- validation before anything is enqueued (each chunk's attn_fwd_ex call
  // checks its sub-problem again)
  if (!q || !k || !v || !out || !workspace) return ATTN_ERR_INVALID_ARG;
  const int64_t need = attn_fwd_host_workspace_bytes(B, Hq, Hkv, Sq, Sk, d);
  if (need < 0) return static_cast<int>(need);
  if (!(scale - scale == 0.f)) return ATTN_ERR_INVALID_ARG;  // NaN or Inf
  if (flags & ~ATTN_FLAG_CAUSAL) return ATTN_ERR_UNSUPPORTED;
  if (layout != ATTN_LAYOUT_BHSD && layout != ATTN_LAYOUT_BSHD) return ATTN_ERR_UNSUPPORTED;
  if (rounding_mode < ATTN_ROUND_RTNE || rounding_mode > ATTN_ROUND_RTZ) return ATTN_ERR_UNSUPPORTED;
  if (workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) return ATTN_ERR_MISALIGNED;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  DeviceStreams& ds = g_dev[dev];
  std::lock_guard<std::mutex> lock(ds.mu);
  const int st0 = setup(ds);
  if (st0 != ATTN_OK) return st0;

  const bool causal = (flags & ATTN_FLAG_CAUSAL) != 0;
  const std::vector<Chunk> chunks = attn_plan::plan(layout, B, Hq, Hkv, Sq, Sk, causal);
  if (chunks.empty() || chunks.size() > static_cast<size_t>(kMaxChunks)) return ATTN_ERR_LAUNCH;
  const int64_t q_region = round_up(B * Hq * Sq * 256, kAlign);
  const int64_t kv_region = round_up(B * Hkv * Sk * 256, kAlign);
  char* wq = static_cast<char*>(workspace);
  char* wo = wq + q_region;
  char* wk = wo + q_region;
  char* wv = wk + kv_region;
  const char* hq = static_cast<const char*>(q);
  const char* hk = static_cast<const char*>(k);
  const char* hv = static_cast<const char*>(v);
  char* ho = static_cast<char*>(out);
  const cudaStream_t caller = static_cast<cudaStream_t>(stream);

  // Everything starts after the work already on the caller's stream.
  bool ok = cudaEventRecord(ds.start, caller) == cudaSuccess;
  for (cudaStream_t s : {ds.in, ds.out, ds.comp[0], ds.comp[1]})
    ok = ok && cudaStreamWaitEvent(s, ds.start, 0) == cudaSuccess;
  int status = ok ? ATTN_OK : ATTN_ERR_LAUNCH;
  for (size_t i = 0; i < chunks.size() && status == ATTN_OK; ++i) {
    const Chunk& c = chunks[i];
    const cudaStream_t cs = ds.comp[i & 1];
    ok = copy_span(wq, hq, c.q, cudaMemcpyHostToDevice, ds.in) &&
         copy_span(wk, hk, c.kv, cudaMemcpyHostToDevice, ds.in) &&
         copy_span(wv, hv, c.kv, cudaMemcpyHostToDevice, ds.in);
    ok = ok && cudaEventRecord(ds.landed[i], ds.in) == cudaSuccess &&
         cudaStreamWaitEvent(cs, ds.landed[i], 0) == cudaSuccess;
    if (!ok) {
      status = ATTN_ERR_LAUNCH;
      break;
    }
    status = attn_fwd_ex(wq + c.q.dev, wk + c.kv.dev, wv + c.kv.dev, wo + c.q.dev, layout, c.B,
                         c.Hq, c.Hkv, c.Sq, c.Sk, d, scale, rounding_mode, flags, cs);
    if (status != ATTN_OK) break;
    ok = cudaEventRecord(ds.computed[i], cs) == cudaSuccess &&
         cudaStreamWaitEvent(ds.out, ds.computed[i], 0) == cudaSuccess &&
         copy_span(ho, wo, c.q, cudaMemcpyDeviceToHost, ds.out);
    if (!ok) status = ATTN_ERR_LAUNCH;
  }
  // The caller's stream waits for everything enqueued above, also after an error.
  ok = cudaEventRecord(ds.comp_done[0], ds.comp[0]) == cudaSuccess &&
       cudaEventRecord(ds.comp_done[1], ds.comp[1]) == cudaSuccess &&
       cudaEventRecord(ds.done, ds.out) == cudaSuccess &&
       cudaStreamWaitEvent(caller, ds.comp_done[0], 0) == cudaSuccess &&
       cudaStreamWaitEvent(caller, ds.comp_done[1], 0) == cudaSuccess &&
       cudaStreamWaitEvent(caller, ds.done, 0) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    if (status == ATTN_OK) status = ATTN_ERR_LAUNCH;
  }
  return status;
}

int64_t attn_fwd_varlen_host_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t total_q,
                                             int64_t total_k, int64_t d) {
  if (B < 1 || Hq < 1 || Hkv < 1 || total_q < 1 || total_k < 1 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  const int64_t kLim = (int64_t(1) << 31) - 1;
  if (B > kLim || total_q > kLim || total_k > kLim || Hq > kLim) return ATTN_ERR_TOO_LARGE;
  return 2 * round_up(total_q * Hq * 256, kAlign) + 2 * round_up(total_k * Hkv * 256, kAlign) +
         2 * round_up((B + 1) * 4, kAlign);
}

int attn_fwd_varlen_host(const void* q, const void* k, const void* v, void* out,
                         const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int64_t B,
                         int64_t Hq, int64_t Hkv, int64_t total_q, int64_t total_k, int64_t d,
                         float scale, int rounding_mode, int flags, void* workspace,
                         int64_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !out || !cu_seqlens_q || !cu_seqlens_k || !workspace)
    return ATTN_ERR_INVALID_ARG;
  const int64_t need = attn_fwd_varlen_host_workspace_bytes(B, Hq, Hkv, total_q, total_k, d);
  if (need < 0) return static_cast<int>(need);
  if (!(scale - scale == 0.f)) return ATTN_ERR_INVALID_ARG;  // NaN or Inf
  if (flags & ~ATTN_FLAG_CAUSAL) return ATTN_ERR_UNSUPPORTED;
  if (rounding_mode < ATTN_ROUND_RTNE || rounding_mode > ATTN_ROUND_RTZ) return ATTN_ERR_UNSUPPORTED;
  if (workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) return ATTN_ERR_MISALIGNED;
  // The offsets are on the host here, so they are checked before anything runs.
  if (cu_seqlens_q[0] != 0 || cu_seqlens_k[0] != 0 || cu_seqlens_q[B] != total_q ||
      cu_seqlens_k[B] != total_k)
    return ATTN_ERR_SEQLENS;
  for (int64_t b = 0; b < B; ++b)
    if (cu_seqlens_q[b + 1] < cu_seqlens_q[b] || cu_seqlens_k[b + 1] < cu_seqlens_k[b])
      return ATTN_ERR_SEQLENS;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  DeviceStreams& ds = g_dev[dev];
  std::lock_guard<std::mutex> lock(ds.mu);
  const int st0 = setup(ds);
  if (st0 != ATTN_OK) return st0;

  const std::vector<SeqChunk> chunks = attn_plan::plan_varlen(cu_seqlens_q, B, Hq);
  if (chunks.empty() || chunks.size() > static_cast<size_t>(kMaxChunks)) return ATTN_ERR_LAUNCH;
  const int64_t q_region = round_up(total_q * Hq * 256, kAlign);
  const int64_t kv_region = round_up(total_k * Hkv * 256, kAlign);
  const int64_t cu_region = round_up((B + 1) * 4, kAlign);
  char* wq = static_cast<char*>(workspace);
  char* wo = wq + q_region;
  char* wk = wo + q_region;
  char* wv = wk + kv_region;
  int32_t* wcq = reinterpret_cast<int32_t*>(wv + kv_region);
  int32_t* wck = reinterpret_cast<int32_t*>(wv + kv_region + cu_region);
  const char* hq = static_cast<const char*>(q);
  const char* hk = static_cast<const char*>(k);
  const char* hv = static_cast<const char*>(v);
  char* ho = static_cast<char*>(out);
  const int64_t qrow = Hq * 256, kvrow = Hkv * 256;  // bytes per token
  const cudaStream_t caller = static_cast<cudaStream_t>(stream);

  bool ok = cudaEventRecord(ds.start, caller) == cudaSuccess;
  for (cudaStream_t s : {ds.in, ds.out, ds.comp[0], ds.comp[1]})
    ok = ok && cudaStreamWaitEvent(s, ds.start, 0) == cudaSuccess;
  // The offsets go up first (they are small); every chunk's kernel reads them.
  ok = ok && cudaMemcpyAsync(wcq, cu_seqlens_q, (B + 1) * 4, cudaMemcpyHostToDevice, ds.in) ==
                 cudaSuccess &&
       cudaMemcpyAsync(wck, cu_seqlens_k, (B + 1) * 4, cudaMemcpyHostToDevice, ds.in) ==
           cudaSuccess;
  int status = ok ? ATTN_OK : ATTN_ERR_LAUNCH;
  for (size_t i = 0; i < chunks.size() && status == ATTN_OK; ++i) {
    const SeqChunk& c = chunks[i];
    const cudaStream_t cs = ds.comp[i & 1];
    const int64_t q0 = cu_seqlens_q[c.b0], q1 = cu_seqlens_q[c.b1];
    const int64_t k0 = cu_seqlens_k[c.b0], k1 = cu_seqlens_k[c.b1];
    ok = true;
    if (q1 > q0)
      ok = cudaMemcpyAsync(wq + q0 * qrow, hq + q0 * qrow, (q1 - q0) * qrow,
                           cudaMemcpyHostToDevice, ds.in) == cudaSuccess;
    if (ok && k1 > k0)
      ok = cudaMemcpyAsync(wk + k0 * kvrow, hk + k0 * kvrow, (k1 - k0) * kvrow,
                           cudaMemcpyHostToDevice, ds.in) == cudaSuccess &&
           cudaMemcpyAsync(wv + k0 * kvrow, hv + k0 * kvrow, (k1 - k0) * kvrow,
                           cudaMemcpyHostToDevice, ds.in) == cudaSuccess;
    ok = ok && cudaEventRecord(ds.landed[i], ds.in) == cudaSuccess &&
         cudaStreamWaitEvent(cs, ds.landed[i], 0) == cudaSuccess;
    if (!ok) {
      status = ATTN_ERR_LAUNCH;
      break;
    }
    if (c.max_sq == 0) continue;  // only sequences without queries
    status = attn_fwd_varlen(wq, wk, wv, wo, wcq + c.b0, wck + c.b0, c.b1 - c.b0, Hq, Hkv,
                             total_q, total_k, c.max_sq, d, scale, rounding_mode, flags, cs);
    if (status != ATTN_OK) break;
    ok = cudaEventRecord(ds.computed[i], cs) == cudaSuccess &&
         cudaStreamWaitEvent(ds.out, ds.computed[i], 0) == cudaSuccess &&
         cudaMemcpyAsync(ho + q0 * qrow, wo + q0 * qrow, (q1 - q0) * qrow, cudaMemcpyDeviceToHost,
                         ds.out) == cudaSuccess;
    if (!ok) status = ATTN_ERR_LAUNCH;
  }
  ok = cudaEventRecord(ds.comp_done[0], ds.comp[0]) == cudaSuccess &&
       cudaEventRecord(ds.comp_done[1], ds.comp[1]) == cudaSuccess &&
       cudaEventRecord(ds.done, ds.out) == cudaSuccess &&
       cudaStreamWaitEvent(caller, ds.comp_done[0], 0) == cudaSuccess &&
       cudaStreamWaitEvent(caller, ds.comp_done[1], 0) == cudaSuccess &&
       cudaStreamWaitEvent(caller, ds.done, 0) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    if (status == ATTN_OK) status = ATTN_ERR_LAUNCH;
  }
  return status;
}

}  // extern "C"
