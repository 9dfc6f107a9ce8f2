// attn_fwd.cu - host side of the C ABI declared in include/attn_fwd.h.
//
// Validates the call on the host, builds the four TMA tensor maps (Q, K, V, O;
// the layout only changes their strides and coordinate order, so both BSHD and
// BHSD are read in place), sizes the grid (one CTA per pair of 128-row query
// tiles of one (batch, head), consecutive CTAs on the same head so that K/V
// stay in L2) and launches the kernel on the caller's stream.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_fwd.h"
#include "attn_fwd_kernel.cuh"
#include "splitkv_combine.cuh"

namespace {

constexpr int kVersion = 100;  // 0.1.0
constexpr unsigned long long kTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr int kMaxDevices = 64;

std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qres;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &qres) == cudaSuccess &&
        qres == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

std::mutex g_dev_mutex;
int g_dev_state[kMaxDevices];  // 0 = not set up, 1 = ready, negative = status to return
int g_dev_sms[kMaxDevices];    // streaming multiprocessors of each device (once ready)
int g_dev_pairs[kMaxDevices];  // 2-CTA clusters of the pair variant that fit at once

// Whole-range problems with at most this many key tiles run on the persistent
// variant (one CTA per SM looping over the items) when they have more items
// than SMs: their items are short, and one CTA per item leaves each SM idle
// through every item's first loads and final store.
constexpr int64_t kPersistMaxKvTiles = 16;

// Whole-range problems with at least this many key tiles run the items of their
// last, partial wave on the pair variant (each item's keys split between the two
// CTAs of a cluster), when those items fit on the GPU at once as clusters: the
// wave then takes about half an item's time instead of a whole one.
constexpr int64_t kPairMinKvTiles = 8;

// Once per device: check the architecture and raise the shared-memory limit.
int device_ready(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_dev_state[dev] != 0) return g_dev_state[dev] > 0 ? ATTN_OK : g_dev_state[dev];
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  if (major != 10 || minor != 3) {
    g_dev_state[dev] = ATTN_ERR_ARCH;
    return ATTN_ERR_ARCH;
  }
  // Every variant of the fused kernel (whole key range / split; causal; packed
  // variable-length batch, without and with the causal mask).
  const void* variants[] = {
      reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, false, false>),
      reinterpret_cast<const void*>(attn::attn_fwd_kernel<true, false, false>),
      reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, true, false>),
      reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, false, true>),
      reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, true, true>),
      reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, false, false, true>),
      reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, false, false, false, true>),
      reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, false, false, true, false, 1>),
      reinterpret_cast<const void*>(attn::attn_fwd_kernel<false, false, false, true, false, 2>)};
  for (const void* fn : variants) {
    const bool persist = fn == variants[5] || fn == variants[7] || fn == variants[8];
    const bool pair = fn == variants[6];
    const bool row_limit = fn == variants[2] || fn == variants[3] || fn == variants[4];
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             persist ? attn::kSmemBytesPersist
                             : pair  ? attn::kSmemBytesPair
                                     : (row_limit ? attn::kSmemBytesRowLimit : attn::kSmemBytes)) !=
        cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
  }
  // The kernel's warpgroups re-split the registers a CTA is launched with
  // (setmaxnreg); the split only adds up if each thread starts with exactly
  // kLaunchRegs. A build with another count would make setmaxnreg.inc wait
  // forever, so it is refused here.
  for (const void* fn : variants) {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
    if (fa.numRegs != attn::kLaunchRegs) {
      g_dev_state[dev] = ATTN_ERR_LAUNCH;
      return ATTN_ERR_LAUNCH;
    }
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  g_dev_sms[dev] = sms;
  // How many 2-CTA clusters of the pair variant the device holds at once (SMs
  // are paired within their GPC, so this can be below half the SM count). If the
  // query fails the pair variant is not used.
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * static_cast<unsigned>(sms));
    cfg.blockDim = dim3(attn::kThreads);
    cfg.dynamicSmemBytes = attn::kSmemBytesPair;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, variants[6], &cfg) != cudaSuccess) {
      cudaGetLastError();
      clusters = 0;
    }
    g_dev_pairs[dev] = clusters;
  }
  g_dev_state[dev] = 1;
  return ATTN_OK;
}

// Under ATTN_FLAG_SPLIT_TAIL: how many items (those of the last, partial wave of a
// one-CTA-per-item launch) run on pairs; 0 if none. Problems that take the
// persistent variant keep it.
int64_t pair_tail_items(int dev, int64_t n_items, int64_t kv_tiles) {
  // The pair launch numbers its CTAs' work items 2 * item + half in an int.
  if (n_items > (int64_t(1) << 30) - 1) return 0;
  const int64_t sms = g_dev_sms[dev];
  if (kv_tiles <= kPersistMaxKvTiles && n_items > sms) return 0;
  const int64_t tail = n_items % sms;
  return (tail > 0 && tail <= g_dev_pairs[dev] && kv_tiles >= kPairMinKvTiles) ? tail : 0;
}

// 4-D map over a (B, H, S, 128) bf16 tensor in the given layout, box of
// 64 columns x box_rows rows, 128-byte swizzle, zero fill outside the tensor.
bool make_map(CUtensorMap* map, const void* ptr, int layout, int64_t B, int64_t H, int64_t S,
              uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t row = 128 * 2;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4];
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  if (layout == ATTN_LAYOUT_BHSD) {
    dims[0] = 128; dims[1] = S; dims[2] = H; dims[3] = B;
    strides[0] = row; strides[1] = S * row; strides[2] = H * S * row;
    box[0] = 64; box[1] = box_rows; box[2] = 1; box[3] = 1;
  } else {
    dims[0] = 128; dims[1] = H; dims[2] = S; dims[3] = B;
    strides[0] = row; strides[1] = H * row; strides[2] = S * H * row;
    box[0] = 64; box[1] = 1; box[2] = box_rows; box[3] = 1;
  }
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims,
                            strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

int64_t kv_tiles_of(int64_t Sk) { return (Sk + attn::kBN - 1) / attn::kBN; }

// Causal schedule: (batch, head) items per longest-first group, so that the K/V
// of one group (512 bytes per key and head) take at most 48 MiB of the 126 MiB L2.
int head_group_of(int64_t BH, int64_t keys_per_head) {
  const int64_t per = 512 * (keys_per_head > 0 ? keys_per_head : 1);
  int64_t g = (int64_t(48) << 20) / per;
  if (g < 1) g = 1;
  if (g > BH) g = BH;
  return static_cast<int>(g);
}
int64_t qpairs_of(int64_t Sq) { return (Sq + 2 * attn::kBM - 1) / (2 * attn::kBM); }

// Split workspace: unnormalised rows (128 fp32) then (reference max, row sum).
int64_t splitkv_bytes(int64_t B, int64_t H, int64_t Sq, int64_t n_splits) {
  const int64_t rows = n_splits * B * H * qpairs_of(Sq) * 2 * attn::kBM;
  return rows * (attn::kD + 2) * 4;
}

}  // namespace

extern "C" {

const char* attn_status_str(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument (null pointer, size < 1 or non-finite scale)";
    case ATTN_ERR_UNSUPPORTED: return "unsupported (head_dim must be 128; unknown layout or rounding mode)";
    case ATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case ATTN_ERR_ALIASING: return "output overlaps an input";
    case ATTN_ERR_NO_DEVICE: return "no usable CUDA device";
    case ATTN_ERR_ARCH: return "device is not compute capability 10.3 (sm_103)";
    case ATTN_ERR_LAUNCH: return "CUDA launch or tensor-map setup failed";
    case ATTN_ERR_TIMEOUT: return "a device-side wait timed out";
    case ATTN_ERR_TOO_LARGE: return "size beyond tensor-map or grid limits";
    case ATTN_ERR_SCRATCH: return "split workspace needed exceeds the library's fixed 32 MiB device scratch";
    case ATTN_ERR_SEQLENS: return "invalid cu_seqlens contents (found on the device; those sequences were not computed)";
    case ATTN_ERR_DEBUG_CHECK: return "a bounds or protocol check of the debug build failed (the access it guards was skipped)";
    default: return "unknown status";
  }
}

int attn_fwd_version(void) { return kVersion; }

}  // extern "C"

namespace {

int attn_fwd_impl(const void* q, const void* k, const void* v, void* out, int layout, int64_t B,
                  int64_t H, int64_t Sq, int64_t Sk, int64_t d, float scale, int rounding_mode,
                  void* stream, unsigned long long timeout_ns, int withhold_s0, int n_splits,
                  void* workspace, int64_t workspace_bytes, int64_t Hkv = 0, int causal = 0,
                  int dbg_poison = 0, int split_tail = 0) {
  if (Hkv == 0) Hkv = H;
  // ---- host-side validation (nothing is launched on failure)
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Sq < 1 || Sk < 1 || Hkv < 1 || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (causal && n_splits != 1) return ATTN_ERR_UNSUPPORTED;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  if (layout != ATTN_LAYOUT_BHSD && layout != ATTN_LAYOUT_BSHD) return ATTN_ERR_UNSUPPORTED;
  if (rounding_mode < ATTN_ROUND_RTNE || rounding_mode > ATTN_ROUND_RTZ) return ATTN_ERR_UNSUPPORTED;
  // TMA: coordinates are int32, strides < 2^40 bytes; grid.x < 2^31.
  const int64_t kLim31 = (int64_t(1) << 31) - 1;
  if (Sq > kLim31 || Sk > kLim31 || H > kLim31 || B > kLim31) return ATTN_ERR_TOO_LARGE;
  const int64_t kStrideLim = int64_t(1) << 40;
  if (H > kStrideLim / 256 / Sq || H > kStrideLim / 256 / Sk) return ATTN_ERR_TOO_LARGE;
  if (B > (int64_t(1) << 62) / 256 / H / (Sq > Sk ? Sq : Sk)) return ATTN_ERR_TOO_LARGE;
  const int64_t n_qpairs = qpairs_of(Sq);
  if (n_splits < 1 || n_splits > kv_tiles_of(Sk)) return ATTN_ERR_INVALID_ARG;
  if (B * H > kLim31 / n_qpairs / n_splits) return ATTN_ERR_TOO_LARGE;
  const uintptr_t ormask = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                           reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out);
  if (ormask & 15u) return ATTN_ERR_MISALIGNED;
  const uint64_t bytes_q = uint64_t(B) * H * Sq * 256, bytes_kv = uint64_t(B) * Hkv * Sk * 256;
  if (overlaps(out, bytes_q, q, bytes_q) || overlaps(out, bytes_q, k, bytes_kv) ||
      overlaps(out, bytes_q, v, bytes_kv))
    return ATTN_ERR_ALIASING;
  if (n_splits > 1) {
    const int64_t need = splitkv_bytes(B, H, Sq, n_splits);
    if (!workspace || workspace_bytes < need) return ATTN_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 15u) return ATTN_ERR_MISALIGNED;
    if (overlaps(workspace, need, q, bytes_q) || overlaps(workspace, need, k, bytes_kv) ||
        overlaps(workspace, need, v, bytes_kv) || overlaps(workspace, need, out, bytes_q))
      return ATTN_ERR_ALIASING;
  }

  // ---- device
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  const int st = device_ready(dev);
  if (st != ATTN_OK) return st;

  CUtensorMap tq, tk, tv, to;
  if (!make_map(&tq, q, layout, B, H, Sq, attn::kBM) || !make_map(&tk, k, layout, B, Hkv, Sk, attn::kBN) ||
      !make_map(&tv, v, layout, B, Hkv, Sk, attn::kBN) || !make_map(&to, out, layout, B, H, Sq, 32))
    return ATTN_ERR_LAUNCH;

  attn::Params p;
  p.Sq = static_cast<int>(Sq);
  p.Sk = static_cast<int>(Sk);
  p.H = static_cast<int>(H);
  p.n_qpairs = static_cast<int>(n_qpairs);
  p.kv_tiles = static_cast<int>(kv_tiles_of(Sk));
  p.kv_tail = static_cast<int>(Sk - int64_t(p.kv_tiles - 1) * attn::kBN);
  p.n_splits = n_splits;
  p.BH = static_cast<int>(B * H);
  p.sq_pad = static_cast<int>(n_qpairs * 2 * attn::kBM);
  p.part_o = static_cast<float*>(workspace);
  p.part_rl = n_splits > 1 ? p.part_o + static_cast<size_t>(n_splits) * B * H * p.sq_pad * attn::kD
                           : nullptr;
  p.layout = layout;
  p.mode = rounding_mode;
  p.c = scale * 1.4426950408889634f;
  p.timeout_ns = timeout_ns;
  p.withhold_s0 = withhold_s0;
  p.group = static_cast<int>(H / Hkv);
  p.causal = causal ? 1 : 0;
  p.cu_q = nullptr;
  p.cu_k = nullptr;
  p.max_sq = p.Sq;
  p.out = static_cast<uint16_t*>(out);
  p.head_group = head_group_of(B * H, Sk);
  p.dbg_poison = dbg_poison;
  p.n_items = static_cast<int>(B * H * n_qpairs * n_splits);
  p.item_base = 0;
  p.early_dependents = 0;

  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int64_t n_items1 = B * H * n_qpairs;
  const int64_t n_tail =
      (split_tail && !causal && n_splits == 1 && !dbg_poison) ? pair_tail_items(dev, n_items1, p.kv_tiles)
                                                              : 0;
  const unsigned grid = static_cast<unsigned>(B * H * n_qpairs * n_splits);
  if (causal) {
    attn::attn_fwd_kernel<false, true, false>
        <<<grid, attn::kThreads, attn::kSmemBytesRowLimit, cs>>>(tq, tk, tv, to, p);
  } else if (n_splits == 1 && p.kv_tiles <= kPersistMaxKvTiles && p.n_items > g_dev_sms[dev]) {
    // Items of at most 4 key tiles ending in a ragged one: a short persistent
    // variant (the partial in TMEM until the epilogue, S kept in registers between
    // the softmax passes, the ragged tile's P V cut at its last key chunk). One
    // tile and 2 to 4 tiles are separate instantiations: the general form cost the
    // one-tile case 4%.
    if (p.kv_tiles == 1 && p.kv_tail < attn::kBN)
      attn::attn_fwd_kernel<false, false, false, true, false, 1>
          <<<static_cast<unsigned>(g_dev_sms[dev]), attn::kThreads, attn::kSmemBytesPersist, cs>>>(
              tq, tk, tv, to, p);
    else if (p.kv_tiles <= attn::kShortMaxKvTiles && p.kv_tail < attn::kBN)
      attn::attn_fwd_kernel<false, false, false, true, false, 2>
          <<<static_cast<unsigned>(g_dev_sms[dev]), attn::kThreads, attn::kSmemBytesPersist, cs>>>(
              tq, tk, tv, to, p);
    else
      attn::attn_fwd_kernel<false, false, false, true>
          <<<static_cast<unsigned>(g_dev_sms[dev]), attn::kThreads, attn::kSmemBytesPersist, cs>>>(
              tq, tk, tv, to, p);
  } else if (n_tail > 0) {
    // The full waves as usual, then the tail items as 2-CTA clusters, each with
    // its key range split in two halves and merged on chip (pair variant).
    const int64_t n_full = n_items1 - n_tail;
    if (n_full > 0) {
      attn::Params pf = p;
      pf.early_dependents = 1;
      attn::attn_fwd_kernel<false, false, false>
          <<<static_cast<unsigned>(n_full), attn::kThreads, attn::kSmemBytes, cs>>>(tq, tk, tv, to, pf);
    }
    attn::Params pp = p;
    pp.n_splits = 2;
    pp.item_base = static_cast<int>(2 * n_full);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * n_tail));
    cfg.blockDim = dim3(attn::kThreads);
    cfg.dynamicSmemBytes = attn::kSmemBytesPair;
    cfg.stream = cs;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // A programmatic dependent of the full waves: its clusters take SMs as the
    // last full wave drains instead of after the whole launch.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = n_full > 0 ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, attn::attn_fwd_kernel<false, false, false, false, true>, tq, tk,
                           tv, to, pp) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
  } else if (n_splits == 1) {
    attn::attn_fwd_kernel<false, false, false>
        <<<grid, attn::kThreads, attn::kSmemBytes, cs>>>(tq, tk, tv, to, p);
  } else {
    attn::attn_fwd_kernel<true, false, false>
        <<<grid, attn::kThreads, attn::kSmemBytes, cs>>>(tq, tk, tv, to, p);
    attn::CombineParams cp;
    cp.part_o = p.part_o;
    cp.part_rl = p.part_rl;
    cp.out = static_cast<uint16_t*>(out);
    cp.n_splits = n_splits;
    cp.BH = p.BH;
    cp.H = p.H;
    cp.Sq = p.Sq;
    cp.sq_pad = p.sq_pad;
    cp.layout = layout;
    cp.mode = rounding_mode;
    // Programmatic dependent launch: the merge grid is set up while the split
    // kernel runs and waits on the device for its completion.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((Sq + attn::kCombineRows - 1) / attn::kCombineRows),
                       static_cast<unsigned>(B * H));
    cfg.blockDim = dim3(attn::kD);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = cs;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, attn::attn_splitkv_combine, cp) != cudaSuccess) {
      cudaGetLastError();
      return ATTN_ERR_LAUNCH;
    }
  }
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

}  // namespace

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* out, int layout, int64_t B,
             int64_t H, int64_t Sq, int64_t Sk, int64_t d, float scale, int rounding_mode,
             void* stream) {
  return attn_fwd_impl(q, k, v, out, layout, B, H, Sq, Sk, d, scale, rounding_mode, stream,
                       kTimeoutNs, 0, 1, nullptr, 0);
}

int attn_fwd_ex(const void* q, const void* k, const void* v, void* out, int layout, int64_t B,
                int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t d, float scale,
                int rounding_mode, int flags, void* stream) {
  if (flags & ~(ATTN_FLAG_CAUSAL | ATTN_FLAG_SPLIT_TAIL)) return ATTN_ERR_UNSUPPORTED;
  if (Hkv < 1) return ATTN_ERR_INVALID_ARG;
  return attn_fwd_impl(q, k, v, out, layout, B, Hq, Sq, Sk, d, scale, rounding_mode, stream,
                       kTimeoutNs, 0, 1, nullptr, 0, Hkv, (flags & ATTN_FLAG_CAUSAL) ? 1 : 0, 0,
                       (flags & ATTN_FLAG_SPLIT_TAIL) ? 1 : 0);
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* out,
                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int64_t B,
                    int64_t Hq, int64_t Hkv, int64_t total_q, int64_t total_k,
                    int64_t max_seqlen_q, int64_t d, float scale, int rounding_mode, int flags,
                    void* stream) {
  // ---- host-side validation (nothing is launched on failure); the offsets
  // themselves live on the device and are checked by the kernel.
  if (!q || !k || !v || !out || !cu_seqlens_q || !cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (total_q < 1 || total_k < 1 || max_seqlen_q < 1 || max_seqlen_q > total_q)
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (flags & ~ATTN_FLAG_CAUSAL) return ATTN_ERR_UNSUPPORTED;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  if (rounding_mode < ATTN_ROUND_RTNE || rounding_mode > ATTN_ROUND_RTZ) return ATTN_ERR_UNSUPPORTED;
  const int64_t kLim31 = (int64_t(1) << 31) - 1;
  if (total_q > kLim31 || total_k > kLim31 || Hq > kLim31 || B > kLim31) return ATTN_ERR_TOO_LARGE;
  const int64_t kStrideLim = int64_t(1) << 40;
  if (Hq > kStrideLim / 256 / total_q || Hkv > kStrideLim / 256 / total_k) return ATTN_ERR_TOO_LARGE;
  const int64_t n_qpairs = qpairs_of(max_seqlen_q);
  if (B * Hq > kLim31 / n_qpairs) return ATTN_ERR_TOO_LARGE;
  const uintptr_t ormask = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                           reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out);
  if (ormask & 15u) return ATTN_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) | reinterpret_cast<uintptr_t>(cu_seqlens_k)) & 3u)
    return ATTN_ERR_MISALIGNED;
  const uint64_t bytes_q = uint64_t(total_q) * Hq * 256, bytes_kv = uint64_t(total_k) * Hkv * 256;
  if (overlaps(out, bytes_q, q, bytes_q) || overlaps(out, bytes_q, k, bytes_kv) ||
      overlaps(out, bytes_q, v, bytes_kv) ||
      overlaps(out, bytes_q, cu_seqlens_q, uint64_t(B + 1) * 4) ||
      overlaps(out, bytes_q, cu_seqlens_k, uint64_t(B + 1) * 4))
    return ATTN_ERR_ALIASING;

  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  const int st = device_ready(dev);
  if (st != ATTN_OK) return st;

  // The packed tensors are BSHD with one batch entry and S = total tokens.
  CUtensorMap tq, tk, tv, to;
  const int lay = ATTN_LAYOUT_BSHD;
  if (!make_map(&tq, q, lay, 1, Hq, total_q, attn::kBM) ||
      !make_map(&tk, k, lay, 1, Hkv, total_k, attn::kBN) ||
      !make_map(&tv, v, lay, 1, Hkv, total_k, attn::kBN) ||
      !make_map(&to, out, lay, 1, Hq, total_q, 32))
    return ATTN_ERR_LAUNCH;

  attn::Params p;
  p.Sq = static_cast<int>(total_q);
  p.Sk = static_cast<int>(total_k);
  p.H = static_cast<int>(Hq);
  p.n_qpairs = static_cast<int>(n_qpairs);
  p.kv_tiles = static_cast<int>(kv_tiles_of(total_k));
  p.kv_tail = static_cast<int>(total_k - int64_t(p.kv_tiles - 1) * attn::kBN);
  p.n_splits = 1;
  p.BH = static_cast<int>(B * Hq);
  p.sq_pad = 0;
  p.part_o = nullptr;
  p.part_rl = nullptr;
  p.layout = lay;
  p.mode = rounding_mode;
  p.c = scale * 1.4426950408889634f;
  p.timeout_ns = kTimeoutNs;
  p.withhold_s0 = 0;
  p.group = static_cast<int>(Hq / Hkv);
  p.causal = (flags & ATTN_FLAG_CAUSAL) ? 1 : 0;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.max_sq = static_cast<int>(max_seqlen_q);
  p.out = static_cast<uint16_t*>(out);
  p.head_group = p.causal ? head_group_of(B * Hq, total_k / B) : 1;
  p.dbg_poison = 0;
  p.n_items = static_cast<int>(B * Hq * n_qpairs);
  p.item_base = 0;
  p.early_dependents = 0;

  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const unsigned grid = static_cast<unsigned>(B * Hq * n_qpairs);
  if (p.causal)
    attn::attn_fwd_kernel<false, true, true>
        <<<grid, attn::kThreads, attn::kSmemBytesRowLimit, cs>>>(tq, tk, tv, to, p);
  else
    attn::attn_fwd_kernel<false, false, true>
        <<<grid, attn::kThreads, attn::kSmemBytesRowLimit, cs>>>(tq, tk, tv, to, p);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_LAUNCH;
  return ATTN_OK;
}

int64_t attn_fwd_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d,
                                         int num_splits) {
  if (B < 1 || H < 1 || Sq < 1 || Sk < 1 || num_splits < 1) return ATTN_ERR_INVALID_ARG;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  if (num_splits > kv_tiles_of(Sk)) return ATTN_ERR_INVALID_ARG;
  // The launch's own limits, checked before anything is multiplied: every
  // factor below 2^31 and at most 2^31 - 1 CTAs (batch x head x query-tile pair
  // x split), so the byte count below stays under 2^31 * 256 * 520 < 2^48.
  const int64_t kLim31 = (int64_t(1) << 31) - 1;
  if (B > kLim31 || H > kLim31 || Sq > kLim31 || Sk > kLim31) return ATTN_ERR_TOO_LARGE;
  if (B * H > kLim31 / qpairs_of(Sq) / num_splits) return ATTN_ERR_TOO_LARGE;
  if (num_splits == 1) return 0;
  return splitkv_bytes(B, H, Sq, num_splits);
}

int attn_fwd_splitkv_num_splits(int64_t B, int64_t H, int64_t Sq, int64_t Sk) {
  if (B < 1 || H < 1 || Sq < 1 || Sk < 1) return ATTN_ERR_INVALID_ARG;
  int sms = 152, dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  else
    cudaGetLastError();
  const int64_t items = B * H * qpairs_of(Sq);
  const int64_t tiles = kv_tiles_of(Sk);
  if (items >= sms) return 1;
  // Enough CTAs to fill the GPU once, keeping at least 4 key tiles per split.
  int64_t s = (sms + items - 1) / items;
  const int64_t max_s = tiles / 4 > 0 ? tiles / 4 : 1;
  if (s > max_s) s = max_s;
  if (s > 64) s = 64;
  return static_cast<int>(s);
}

int attn_fwd_split_tail_items(int64_t B, int64_t Hq, int64_t Sq, int64_t Sk) {
  if (B < 1 || Hq < 1 || Sq < 1 || Sk < 1) return ATTN_ERR_INVALID_ARG;
  const int64_t kLim31 = (int64_t(1) << 31) - 1;
  if (B > kLim31 || Hq > kLim31 || Sq > kLim31 || Sk > kLim31) return ATTN_ERR_TOO_LARGE;
  if (B * Hq > kLim31 / qpairs_of(Sq)) return ATTN_ERR_TOO_LARGE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  const int st = device_ready(dev);
  if (st != ATTN_OK) return st;
  return static_cast<int>(pair_tail_items(dev, B * Hq * qpairs_of(Sq), kv_tiles_of(Sk)));
}

int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* out, int layout,
                     int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, float scale,
                     int rounding_mode, int num_splits, void* workspace, int64_t workspace_bytes,
                     void* stream) {
  return attn_fwd_impl(q, k, v, out, layout, B, H, Sq, Sk, d, scale, rounding_mode, stream,
                       kTimeoutNs, 0, num_splits, workspace, workspace_bytes);
}

int attn_fwd_timeout_selftest(const void* q, const void* k, const void* v, void* out, int layout,
                              int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, float scale,
                              int rounding_mode, void* stream, uint64_t timeout_ns, int flags) {
  if (timeout_ns == 0 || timeout_ns > kTimeoutNs) return ATTN_ERR_INVALID_ARG;
  if (flags & ~ATTN_FLAG_SPLIT_TAIL) return ATTN_ERR_UNSUPPORTED;
  return attn_fwd_impl(q, k, v, out, layout, B, H, Sq, Sk, d, scale, rounding_mode, stream,
                       timeout_ns, 1, 1, nullptr, 0, 0, 0, 0, (flags & ATTN_FLAG_SPLIT_TAIL) ? 1 : 0);
}

int attn_fwd_debug_build(void) { return ATTN_DEBUG ? 1 : 0; }

int attn_fwd_debug_selftest(const void* q, const void* k, const void* v, void* out, int layout,
                            int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, float scale,
                            int rounding_mode, void* stream) {
  if (!ATTN_DEBUG) return ATTN_ERR_UNSUPPORTED;
  return attn_fwd_impl(q, k, v, out, layout, B, H, Sq, Sk, d, scale, rounding_mode, stream,
                       kTimeoutNs, 0, 1, nullptr, 0, 0, 0, 1);
}

int attn_fwd_last_error(void) {
  unsigned int s = 0;
  if (cudaMemcpyFromSymbol(&s, attn::g_attn_status, sizeof(s)) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  if (s == 0) return ATTN_OK;
  const unsigned int zero = 0;
  cudaMemcpyToSymbol(attn::g_attn_status, &zero, sizeof(zero));
  if (s & 1u) return ATTN_ERR_TIMEOUT;
  return (s & 2u) ? ATTN_ERR_SEQLENS : ATTN_ERR_DEBUG_CHECK;
}

}  // extern "C"

// ---------------------------------------------------------------- no-allocation split-KV
//
// Some callers cannot allocate device memory when they need attention: a plugin
// inside a framework whose own pool owns every device allocation, a serving loop
// that must not call cudaMalloc / cudaFree after start-up (those calls can
// synchronise the device and stall every stream), or a host with no allocator
// beyond what this library brings. For them the split workspace lives in a fixed
// array in the library's device memory. Every GPU that loads the library holds
// these 32 MiB until the process exits.
static constexpr int64_t kNoAllocScratchBytes = int64_t(32) << 20;
static __device__ __align__(256) unsigned char g_attn_noalloc_scratch[kNoAllocScratchBytes];

namespace {
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices];  // device address of the scratch array, per device
}  // namespace

extern "C" int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* out,
                                        int layout, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                                        int64_t d, float scale, int rounding_mode, int num_splits,
                                        void* stream) {
  if (!q || !k || !v || !out) return ATTN_ERR_INVALID_ARG;
  const int64_t need = attn_fwd_splitkv_workspace_bytes(B, H, Sq, Sk, d, num_splits);
  // A negative size is one of the status codes above; pass on only those.
  if (need == ATTN_ERR_INVALID_ARG || need == ATTN_ERR_UNSUPPORTED || need == ATTN_ERR_TOO_LARGE)
    return static_cast<int>(need);
  if (need < 0) return ATTN_ERR_TOO_LARGE;
  if (need > kNoAllocScratchBytes) return ATTN_ERR_SCRATCH;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ATTN_ERR_NO_DEVICE;
  }
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NO_DEVICE;
  void* scratch = nullptr;
  {
    // Once per device, with that device current: the array's name is only a
    // host-side stand-in, so the kernel is given the device address instead.
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_attn_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return ATTN_ERR_LAUNCH;
      }
      g_scratch_addr[dev] = ptr;
    }
    scratch = g_scratch_addr[dev];
  }
  return attn_fwd_impl(q, k, v, out, layout, B, H, Sq, Sk, d, scale, rounding_mode, stream,
                       kTimeoutNs, 0, num_splits, scratch, kNoAllocScratchBytes);
}
