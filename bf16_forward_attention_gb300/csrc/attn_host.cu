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
// Chunks (every chunk attends only within itself, so each is an attn_fwd_ex
// call on its own dense sub-tensors):
//   BHSD: (b, h) pairs are contiguous blocks, and (B, H, S, d) is the same memory
//         as (1, B*H, S, d); chunks are runs of whole key/value heads with their
//         query heads (a multiple of the group size).
//   BSHD: batch entries are contiguous blocks; chunks are runs of batch
//         entries. With fewer entries than chunks, each entry is cut into runs
//         of key/value heads with their query heads: strided in the caller's
//         tensors (one row of the run's heads per token), copied with 2-D copies
//         and packed densely on the device, so that the first chunk's upload is
//         one run's Q, K and V, and each chunk's CTAs share one run's K/V in L2.
//         With a single key/value head, the entry is cut into runs of query rows
//         instead (contiguous; the entry's K/V go up with its first chunk). A
//         row chunk [s0, s1) of a causal problem is the causal problem with
//         Sq' = s1 - s0 and Sk' = s1 + Sk - Sq: row i' sees keys up to
//         i' + s0 + Sk - Sq, the same keys as row s0 + i' of the whole problem.
//   packed variable-length batch (attn_fwd_varlen_host): runs of whole
//         sequences, contiguous in the packed tensors; a chunk's kernel is
//         attn_fwd_varlen over the full tensors with the offsets array advanced
//         to its first sequence (the offsets stay absolute).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "attn_fwd.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxChunks = 8;
constexpr int64_t kCtasPerChunk = 256;  // a chunk smaller than this is not split
constexpr int64_t kAlign = 256;

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
int64_t qpairs(int64_t Sq) { return (Sq + 255) / 256; }

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

// One tensor's share of a chunk: `rows` runs of `width` bytes, `pitch` bytes
// apart, from byte `host` of the caller's tensor, packed densely from byte `dev`
// of the device tensor. rows == 0: already on the device (K/V of a row chunk).
struct Span {
  int64_t host, dev, width, rows, pitch;
};

// A contiguous share: the same offset on host and device.
Span flat(int64_t off, int64_t bytes, bool copy = true) {
  return {off, off, bytes, copy ? 1 : 0, bytes};
}

// One chunk: its shares of Q (and of O, which has Q's shape), of K and V (alike),
// and the sub-problem they form.
struct Chunk {
  Span q, kv;
  int64_t B, Hq, Hkv, Sq, Sk;
};

bool copy_span(char* dst_base, const char* src_base, const Span& s, cudaMemcpyKind kind,
               cudaStream_t st) {
  if (s.rows == 0) return true;
  const bool up = kind == cudaMemcpyHostToDevice;
  char* dst = dst_base + (up ? s.dev : s.host);
  const char* src = src_base + (up ? s.host : s.dev);
  if (s.rows == 1 || s.pitch == s.width)
    return cudaMemcpyAsync(dst, src, s.width * s.rows, kind, st) == cudaSuccess;
  return cudaMemcpy2DAsync(dst, up ? s.width : s.pitch, src, up ? s.pitch : s.width, s.width,
                           s.rows, kind, st) == cudaSuccess;
}

// Splits the problem into at most kMaxChunks chunks of at least kCtasPerChunk
// CTAs (one CTA per 256 query rows of one head) where possible.
std::vector<Chunk> plan(int layout, int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk,
                        bool causal) {
  std::vector<Chunk> out;
  const int64_t row = 256;  // bytes per (token, head) row of d = 128 bf16
  const int64_t total_ctas = B * Hq * qpairs(Sq);
  int64_t want = total_ctas / kCtasPerChunk;
  want = want < 1 ? 1 : (want > kMaxChunks ? kMaxChunks : want);
  if (layout == ATTN_LAYOUT_BHSD) {
    // Runs of key/value heads over the flattened (b, h_kv) index.
    const int64_t units = B * Hkv, group = Hq / Hkv;
    const int64_t n = want < units ? want : units;
    for (int64_t c = 0; c < n; ++c) {
      const int64_t u0 = units * c / n, u1 = units * (c + 1) / n;
      out.push_back({flat(u0 * group * Sq * row, (u1 - u0) * group * Sq * row),
                     flat(u0 * Sk * row, (u1 - u0) * Sk * row), 1, (u1 - u0) * group, u1 - u0,
                     Sq, Sk});
    }
    return out;
  }
  const int64_t q_batch = Sq * Hq * row, kv_batch = Sk * Hkv * row;
  if (want <= B) {
    for (int64_t c = 0; c < want; ++c) {
      const int64_t b0 = B * c / want, b1 = B * (c + 1) / want;
      out.push_back({flat(b0 * q_batch, (b1 - b0) * q_batch), flat(b0 * kv_batch, (b1 - b0) * kv_batch),
                     b1 - b0, Hq, Hkv, Sq, Sk});
    }
    return out;
  }
  // Runs per entry: enough for `want` chunks, but at most kMaxChunks in all.
  int64_t per = (want + B - 1) / B;
  if (per > kMaxChunks / B) per = kMaxChunks / B;
  if (per < 1) per = 1;
  if (Hkv > 1) {
    // Runs of key/value heads of each entry, with their query heads; each run's
    // rows are packed densely on the device, one run after the other.
    const int64_t group = Hq / Hkv;
    const int64_t n = per < Hkv ? per : Hkv;
    int64_t dq = 0, dkv = 0;
    for (int64_t b = 0; b < B; ++b) {
      for (int64_t c = 0; c < n; ++c) {
        const int64_t u0 = Hkv * c / n, u1 = Hkv * (c + 1) / n;
        const int64_t qw = (u1 - u0) * group * row, kvw = (u1 - u0) * row;
        out.push_back({{b * q_batch + u0 * group * row, dq, qw, Sq, Hq * row},
                       {b * kv_batch + u0 * row, dkv, kvw, Sk, Hkv * row}, 1, (u1 - u0) * group,
                       u1 - u0, Sq, Sk});
        dq += qw * Sq;
        dkv += kvw * Sk;
      }
    }
    return out;
  }
  // A single key/value head: cut each entry's query rows. Boundaries are
  // multiples of 256 rows; under the causal mask the first chunk of an entry
  // also takes every row that sees no key (Sk' = s1 + Sk - Sq must be >= 1).
  for (int64_t b = 0; b < B; ++b) {
    int64_t s0 = 0;
    bool first = true;
    for (int64_t c = 1; c <= per; ++c) {
      int64_t s1 = c == per ? Sq : round_up(Sq * c / per, 256);
      if (s1 > Sq) s1 = Sq;
      if (s1 <= s0) continue;
      if (causal && s1 + Sk - Sq < 1) continue;  // merge into the next chunk
      out.push_back({flat(b * q_batch + s0 * Hq * row, (s1 - s0) * Hq * row),
                     flat(b * kv_batch, kv_batch, first), 1, Hq, Hkv, s1 - s0,
                     causal ? s1 + Sk - Sq : Sk});
      first = false;
      s0 = s1;
    }
  }
  return out;
}

// Runs of whole sequences of a packed batch, at most kMaxChunks, each of at
// least kCtasPerChunk CTAs where the batch allows.
struct SeqChunk {
  int64_t b0, b1, max_sq;
};

std::vector<SeqChunk> plan_varlen(const int32_t* cq, int64_t B, int64_t Hq) {
  int64_t total = 0;
  for (int64_t b = 0; b < B; ++b) total += Hq * qpairs(cq[b + 1] - cq[b]);
  int64_t want = total / kCtasPerChunk;
  want = want < 1 ? 1 : (want > kMaxChunks ? kMaxChunks : want);
  std::vector<SeqChunk> out;
  int64_t b0 = 0, acc = 0, max_sq = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t sq = cq[b + 1] - cq[b];
    acc += Hq * qpairs(sq);
    max_sq = sq > max_sq ? sq : max_sq;
    // The last chunk takes every remaining sequence (also ones without queries),
    // so there are at most `want` chunks.
    const int64_t goal = total * (static_cast<int64_t>(out.size()) + 1) / want;
    if ((acc >= goal && static_cast<int64_t>(out.size()) + 1 < want) || b == B - 1) {
      out.push_back({b0, b + 1, max_sq});
      b0 = b + 1;
      max_sq = 0;
    }
  }
  return out;
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
  const std::vector<Chunk> chunks = plan(layout, B, Hq, Hkv, Sq, Sk, causal);
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

  const std::vector<SeqChunk> chunks = plan_varlen(cu_seqlens_q, B, Hq);
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
