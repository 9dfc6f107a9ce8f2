// host_plan.h - how the host-buffer entry points (attn_fwd_host,
// attn_fwd_varlen_host) cut a problem into chunks. Plain C++ with no CUDA
// dependency, so that the plans can be built and checked on any host.
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
//   packed variable-length batch: runs of whole sequences, contiguous in the
//         packed tensors.
#pragma once

#include <cstdint>
#include <vector>

#include "attn_fwd.h"

namespace attn_plan {

constexpr int kMaxChunks = 8;
constexpr int64_t kCtasPerChunk = 256;  // a chunk smaller than this is not split

inline int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }
inline int64_t qpairs(int64_t Sq) { return (Sq + 255) / 256; }

// One tensor's share of a chunk: `rows` runs of `width` bytes, `pitch` bytes
// apart, from byte `host` of the caller's tensor, packed densely from byte `dev`
// of the device tensor. rows == 0: already on the device (K/V of a row chunk).
struct Span {
  int64_t host, dev, width, rows, pitch;
};

// A contiguous share: the same offset on host and device.
inline Span flat(int64_t off, int64_t bytes, bool copy = true) {
  return {off, off, bytes, copy ? 1 : 0, bytes};
}

// The arguments of the (2-D) copy of a span, upload (host to device) or
// download: byte offsets into the destination and source tensors, their pitches,
// and the width and number of the runs.
struct CopyArgs {
  int64_t dst, dpitch, src, spitch, width, rows;
};

inline CopyArgs copy_args(const Span& s, bool upload) {
  return upload ? CopyArgs{s.dev, s.width, s.host, s.pitch, s.width, s.rows}
                : CopyArgs{s.host, s.pitch, s.dev, s.width, s.width, s.rows};
}

// One chunk: its shares of Q (and of O, which has Q's shape), of K and V (alike),
// and the sub-problem they form.
struct Chunk {
  Span q, kv;
  int64_t B, Hq, Hkv, Sq, Sk;
};

// Splits the problem into at most kMaxChunks chunks of at least kCtasPerChunk
// CTAs (one CTA per 256 query rows of one head) where possible. The sizes are
// the validated ones of attn_fwd_host (all >= 1, Hq a multiple of Hkv, d = 128).
inline std::vector<Chunk> plan(int layout, int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq,
                               int64_t Sk, bool causal) {
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
// least kCtasPerChunk CTAs where the batch allows. `cq` holds the B + 1 query
// offsets, already checked (cq[0] = 0, non-decreasing).
struct SeqChunk {
  int64_t b0, b1, max_sq;
};

inline std::vector<SeqChunk> plan_varlen(const int32_t* cq, int64_t B, int64_t Hq) {
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

}  // namespace attn_plan
