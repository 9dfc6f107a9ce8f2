/*
 * attn_fwd.h - C ABI of the GB300 (sm_103a) bf16 forward-attention library.
 *
 * The operation is the fused forward attention described on the pages about
 * MoonMath AI's bf16 attention kernel:
 *   - snilld.dk, "Open source attention-kernel i HIP slaar AITER v3 paa MI300X -
 *     hurtigere bf16-attention uden assembly":
 *       "Hvordan kernen arbejder": O = softmax(Q K^T / sqrt(d)) V in one fused
 *         pass, bf16 output;
 *       "Hvad er udgivet": BSHD and BHSD inputs read without a transpose,
 *         head_dim 128, arbitrary sequence lengths, cross-attention (Sq != Sk);
 *       "Numerik samlet eet sted": output rounded to bf16 per mode, finite
 *         values within 1 bf16 ULP, NaN/Inf bit-identical, deterministic.
 *   - tilnote.io note on the same kernel, performance section: the modes are
 *     RTNE, RTNA and RTZ; no causal mask, no GQA, no varlen batching.
 *
 * Every entry point is a plain C function. Pointers marked "device" must point
 * to memory of the current CUDA device; the library never copies them to the
 * host, never frees them and keeps no reference after the call returns.
 */
#ifndef ATTN_FWD_H
#define ATTN_FWD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Tensor layouts. Q, K, V and O all use the one layout given to the call.
 *   BHSD: element (b, h, s, c) at ((b*H + h)*S + s)*128 + c
 *   BSHD: element (b, h, s, c) at ((b*S + s)*H + h)*128 + c
 * with S = Sq for Q and O, S = Sk for K and V. Tensors are contiguous. */
typedef enum { ATTN_LAYOUT_BHSD = 0, ATTN_LAYOUT_BSHD = 1 } attn_layout_t;

/* bf16 rounding of the output (from the fp32 accumulator):
 *   RTNE nearest, ties to even; RTNA nearest, ties away from zero;
 *   RTZ toward zero. NaN outputs are written as 0x7FC0; signed zeros and
 *   bf16 subnormals are kept. */
typedef enum { ATTN_ROUND_RTNE = 0, ATTN_ROUND_RTNA = 1, ATTN_ROUND_RTZ = 2 } attn_round_t;

/* Status codes. Errors other than ATTN_ERR_LAUNCH, ATTN_ERR_TIMEOUT and
 * ATTN_ERR_SEQLENS are found on the host before anything is launched. */
enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = -1, /* null pointer, a size < 1, non-finite scale     */
  ATTN_ERR_UNSUPPORTED = -2, /* d != 128, unknown layout or rounding mode      */
  ATTN_ERR_MISALIGNED = -3,  /* a pointer not 16-byte aligned                  */
  ATTN_ERR_ALIASING = -4,    /* out overlaps q, k or v                         */
  ATTN_ERR_NO_DEVICE = -5,   /* no current CUDA device                         */
  ATTN_ERR_ARCH = -6,        /* current device is not compute capability 10.3  */
  ATTN_ERR_LAUNCH = -7,      /* the CUDA launch (or tensor-map setup) failed   */
  ATTN_ERR_TIMEOUT = -8,     /* a bounded device-side wait expired             */
  ATTN_ERR_TOO_LARGE = -9,   /* a size beyond the tensor-map / grid limits     */
  ATTN_ERR_SCRATCH = -10,    /* attn_fwd_splitkv_noalloc: workspace > 32 MiB   */
  ATTN_ERR_SEQLENS = -11,    /* attn_fwd_varlen: invalid offsets, found on the
                                device and reported by attn_fwd_last_error     */
  ATTN_ERR_DEBUG_CHECK = -12 /* debug build: a bounds or protocol check failed,
                                reported by attn_fwd_last_error                */
};

/*
 * attn_fwd - O = softmax(Q K^T * scale) V for every (b, h).
 *
 *   q    device, bf16, B*H*Sq*d elements in `layout`      (read only)
 *   k    device, bf16, B*H*Sk*d elements in `layout`      (read only)
 *   v    device, bf16, B*H*Sk*d elements in `layout`      (read only)
 *   out  device, bf16, B*H*Sq*d elements in `layout`      (written; must not
 *        overlap q, k or v)
 *   layout         ATTN_LAYOUT_BHSD or ATTN_LAYOUT_BSHD
 *   B, H, Sq, Sk   batch, heads, query length, key length; each >= 1, Sq and
 *                  Sk need not be multiples of anything and may differ
 *   d              head dimension; must be 128
 *   scale          logit scale, any finite float (1/sqrt(128) in the pages)
 *   rounding_mode  ATTN_ROUND_RTNE, ATTN_ROUND_RTNA or ATTN_ROUND_RTZ
 *   stream         cudaStream_t to run on (NULL = legacy default stream)
 *
 * Asynchronous: returns after the launch; `out` is valid once the stream has
 * reached the call. All pointers must be 16-byte aligned. The call allocates
 * no device memory. Results are bit-identical from run to run, and each
 * (batch, head, query row)'s result is independent of the rest of the call.
 * Thread-safe. Returns ATTN_OK or a negative status code.
 *
 * Schedule (invisible in the result): one CTA per (batch, head, pair of
 * 128-row query tiles); when Sk <= 2048 and there are more such items than
 * SMs, one CTA per SM loops over them instead, overlapping each item's loads
 * and stores with its neighbours'.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* out, int layout,
             int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, float scale,
             int rounding_mode, void* stream);

/* Flags of attn_fwd_ex. */
enum { ATTN_FLAG_CAUSAL = 1, ATTN_FLAG_SPLIT_TAIL = 2 };

/*
 * attn_fwd_ex - attn_fwd with two of the follow-on steps the pages list as
 * missing from their kernel (tilnote.io note, performance section; snilld.dk,
 * "Hvad er udgivet"): grouped-query attention and a causal mask.
 *
 *   Hq, Hkv  query heads and key/value heads; Hq must be a multiple of Hkv, and
 *            query head h reads key/value head h / (Hq / Hkv). q and out have Hq
 *            heads, k and v have Hkv heads, all in `layout`.
 *   flags    0, or either or both of ATTN_FLAG_CAUSAL and ATTN_FLAG_SPLIT_TAIL
 *            (any other bit: ATTN_ERR_UNSUPPORTED).
 *            ATTN_FLAG_CAUSAL: key j is visible to query i iff
 *            j <= i + (Sk - Sq) (aligned at the bottom right, so the last query
 *            sees every key); hidden logits are -Inf, and a query that sees no
 *            key (possible when Sq > Sk) comes out NaN. Key tiles that no row of
 *            a query tile can see are skipped. A hidden key takes no part at
 *            all: a NaN or infinity in V at a key a query does not see does not
 *            reach that query's output, while a query that sees it gets NaN or
 *            that infinity in the column.
 *            ATTN_FLAG_SPLIT_TAIL (without the mask; no effect with it): when
 *            the items of the launch's last, partial wave fit on the GPU at once
 *            as pairs of CTAs (2-CTA clusters) and the key range has at least 8
 *            tiles of 128 keys (more than 16 when there are more items than
 *            SMs), each of those items runs on a pair, each CTA taking half of
 *            its key tiles, merged on chip with the same arithmetic as
 *            attn_fwd_splitkv with 2 splits. The last wave then takes about
 *            half as long. The price: an item's bits then depend on how many
 *            items the call has (they stay within the numerics contract and the
 *            same from run to run). Without the flag every item's result is
 *            independent of the rest of the call: a sub-batch or a slice of the
 *            heads gives the same bits as the whole call.
 * Other arguments, ownership, errors and the numerics contract as attn_fwd.
 */
int attn_fwd_ex(const void* q, const void* k, const void* v, void* out, int layout, int64_t B,
                int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t d, float scale,
                int rounding_mode, int flags, void* stream);

/*
 * attn_fwd_split_tail_items - how many of the (batch, head, query-tile pair)
 * items of an attn_fwd_ex call of this size with ATTN_FLAG_SPLIT_TAIL (and no
 * mask) run on pairs of CTAs on the current device: 0 when the flag changes
 * nothing. When the result is above 0 and below the item count
 * B * Hq * ceil(Sq / 256), the call makes two kernel launches (the full waves,
 * then the pairs); otherwise one.
 *
 * Returns the count (>= 0), ATTN_ERR_INVALID_ARG if a size is below 1,
 * ATTN_ERR_TOO_LARGE beyond the launch limits of attn_fwd, or
 * ATTN_ERR_NO_DEVICE / ATTN_ERR_ARCH for the current device. Launches nothing.
 * Neither this query nor ATTN_FLAG_SPLIT_TAIL has a counterpart on the pages:
 * they concern how the work fills this GPU, not what is computed.
 */
int attn_fwd_split_tail_items(int64_t B, int64_t Hq, int64_t Sq, int64_t Sk);

/*
 * Split-KV: the same operation with each query tile's key range cut into
 * `num_splits` contiguous parts handled by different CTAs, for shapes with too
 * few (batch, head, query-tile) units to fill the GPU (short queries against long
 * keys). Each part writes an unnormalised fp32 partial result and its running max
 * and row sum to `workspace`; a second kernel merges the parts in a fixed order,
 * normalises and rounds to bf16 per mode into `out`. The numerics contract of
 * attn_fwd holds; results are bit-identical from run to run for a given
 * num_splits (but not bit-identical to other split counts: the fp32 sums run in
 * another order). This is the first of the follow-on steps after the fused
 * kernel; the pages' kernel processes each query tile's keys in one CTA.
 *
 *   num_splits       1 .. ceil(Sk / 128); 1 runs attn_fwd and needs no workspace
 *   workspace        device, 16-byte aligned, at least
 *                    attn_fwd_splitkv_workspace_bytes(...) bytes, owned by the
 *                    caller, not overlapping q, k, v or out; its contents on
 *                    entry do not matter and are overwritten
 *   workspace_bytes  its size in bytes
 * Other arguments as attn_fwd. Two kernels are launched on `stream`; calls that
 * share a workspace must not overlap in time. Returns ATTN_OK or a status code
 * (ATTN_ERR_INVALID_ARG for a bad split count or a missing / short workspace).
 */
int attn_fwd_splitkv(const void* q, const void* k, const void* v, void* out, int layout,
                     int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, float scale,
                     int rounding_mode, int num_splits, void* workspace, int64_t workspace_bytes,
                     void* stream);

/*
 * attn_fwd_varlen - attention over a packed batch of variable-length sequences,
 * the follow-on step the pages call varlen batching and list as missing
 * (snilld.dk, "Hvad er udgivet" and "Autoregressiv serving, de praktiske
 * hager": serving mixes sequence lengths in one batch).
 *
 *   q    device, bf16, total_q * Hq * d elements, token-major: (token, head, d)
 *   k, v device, bf16, total_k * Hkv * d elements, token-major
 *   out  device, bf16, like q (written; must not overlap q, k, v or the offsets)
 *   cu_seqlens_q, cu_seqlens_k
 *        device, int32, B + 1 entries each: sequence b owns query tokens
 *        cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key tokens cu_seqlens_k[b] ..
 *        cu_seqlens_k[b+1]-1, and attends only within itself (another
 *        sequence's keys take no part, NaN or infinite values in its V
 *        included). Offsets start at
 *        0, do not decrease and end at total_q / total_k; a sequence may have no
 *        queries (nothing to do) or no keys (its rows come out NaN).
 *   B             number of sequences, >= 1
 *   Hq, Hkv       query and key/value heads, as attn_fwd_ex
 *   total_q, total_k   packed token counts, each >= 1
 *   max_seqlen_q  an upper bound on every sequence's query count (1 .. total_q);
 *                 it sizes the grid (a loose bound only adds grid slots that
 *                 exit at once)
 *   flags         0 or ATTN_FLAG_CAUSAL; the causal alignment is per sequence
 *                 (key j visible to query i iff j <= i + Sk_b - Sq_b)
 * The offsets stay on the device: the kernel checks each sequence's offsets
 * against the totals and max_seqlen_q, skips a sequence whose offsets are
 * invalid (its rows of out are left unwritten) and raises a device status that
 * attn_fwd_last_error() returns as ATTN_ERR_SEQLENS. Other arguments,
 * ownership, errors and the numerics contract as attn_fwd.
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* out,
                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int64_t B,
                    int64_t Hq, int64_t Hkv, int64_t total_q, int64_t total_k,
                    int64_t max_seqlen_q, int64_t d, float scale, int rounding_mode, int flags,
                    void* stream);

/* Workspace bytes attn_fwd_splitkv needs (0 for num_splits == 1), or a negative
 * status code: ATTN_ERR_INVALID_ARG / ATTN_ERR_UNSUPPORTED for invalid sizes,
 * ATTN_ERR_TOO_LARGE when a size exceeds 2^31 - 1 or the launch would need more
 * than 2^31 - 1 CTAs (B * H * ceil(Sq / 256) * num_splits). The limits are
 * checked before any product is formed, so the result never overflows. Host
 * only. */
int64_t attn_fwd_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d,
                                         int num_splits);

/* A split count that fills the current device once (1 when the problem already
 * has at least one query-tile pair per SM), keeping at least 4 key tiles per
 * split and at most 64 splits. Negative status code for invalid sizes. */
int attn_fwd_splitkv_num_splits(int64_t B, int64_t H, int64_t Sq, int64_t Sk);

/*
 * attn_fwd_splitkv_noalloc - attn_fwd_splitkv for callers that cannot allocate.
 *
 * The pages have no counterpart of this entry point. It exists because some
 * callers cannot allocate device memory when they need attention: a plugin
 * inside a framework whose own pool owns every device allocation, a serving loop
 * that must not call cudaMalloc / cudaFree after start-up (those calls can
 * synchronise the device and stall every stream), or a host with no allocator
 * of its own. Here the split workspace is a fixed 32 MiB array in the library's
 * device memory, held by every GPU that loads the library until the process
 * exits; the call allocates nothing. The caller still passes q, k, v and out.
 *
 *   - Arguments and results as attn_fwd_splitkv, without the workspace.
 *   - A problem whose split workspace (attn_fwd_splitkv_workspace_bytes) exceeds
 *     32 MiB is rejected with ATTN_ERR_SCRATCH before anything is launched.
 *   - The first call on a device looks up the array's device address for that
 *     device (cudaGetSymbolAddress); make that first call before any stream
 *     capture. The address is kept for the life of the process: after a
 *     cudaDeviceReset of that device the library's device memory is gone, and
 *     this entry point must not be called on that device again.
 *   - Every call on a device shares the one array, and each call overwrites the
 *     part it uses before reading it (nothing has to start at zero). Calls that
 *     overlap in time on the GPU, from any stream or thread, race on it: order
 *     them on one stream or synchronise between them.
 */
int attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* out, int layout,
                             int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, float scale,
                             int rounding_mode, int num_splits, void* stream);

/* Static English text for a status code (never NULL). */
const char* attn_status_str(int status);

/*
 * attn_fwd_host - attn_fwd_ex on HOST buffers, with the copies overlapped.
 * The pages measure the kernel alone; a caller that holds its tensors in host
 * memory pays for the copies too, and this entry hides most of them behind
 * the kernel. It has no counterpart on the pages.
 *
 *   q, k, v, out   host memory, in `layout`, sizes as attn_fwd_ex (out written).
 *                  Page-locked memory (cudaHostAlloc / cudaHostRegister) lets
 *                  the copies run asynchronously and overlap the kernels;
 *                  pageable memory works but the copies then serialise.
 *   flags          0 or ATTN_FLAG_CAUSAL (ATTN_FLAG_SPLIT_TAIL or any other
 *                  bit: ATTN_ERR_UNSUPPORTED).
 *   workspace      device memory of attn_fwd_host_workspace_bytes() bytes,
 *                  256-byte aligned, owned by the caller; it receives copies of
 *                  q, k, v and out, each chunk's share packed densely in
 *                  `layout`. Calls in flight at the same time need separate
 *                  workspaces.
 *   stream         the call is ordered after the work already on `stream`, and
 *                  later work on `stream` is ordered after all of it: `out` is
 *                  valid once `stream` has reached this point.
 * The problem is cut into up to 8 chunks: runs of heads for BHSD; for BSHD,
 * runs of batch entries, or with fewer entries than chunks runs of key/value
 * heads of each entry (strided on the host, copied with 2-D copies), or with a
 * single key/value head runs of query rows. Each chunk's upload, kernel
 * (attn_fwd_ex on the chunk's dense sub-tensors) and download run on internal
 * streams ordered by events, so chunk i's kernel overlaps the copies of its
 * neighbours. Results are bit-identical to attn_fwd_ex.
 * Errors: as attn_fwd_ex, and ATTN_ERR_INVALID_ARG for a missing or short
 * workspace, ATTN_ERR_MISALIGNED for a workspace not 256-byte aligned.
 */
int64_t attn_fwd_host_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk,
                                      int64_t d);
int attn_fwd_host(const void* q, const void* k, const void* v, void* out, int layout, int64_t B,
                  int64_t Hq, int64_t Hkv, int64_t Sq, int64_t Sk, int64_t d, float scale,
                  int rounding_mode, int flags, void* workspace, int64_t workspace_bytes,
                  void* stream);

/*
 * attn_fwd_varlen_host - attn_fwd_varlen on HOST buffers, copies overlapped.
 *   q, k, v, out       host memory, packed (token, head, d) as attn_fwd_varlen
 *   cu_seqlens_q/_k    HOST int32 arrays of B + 1 offsets; being on the host they
 *                      are checked before anything runs (ATTN_ERR_SEQLENS: not
 *                      starting at 0, decreasing, or not ending at the totals)
 *   workspace          device memory of attn_fwd_varlen_host_workspace_bytes()
 *                      bytes, 256-byte aligned (copies of the four tensors and
 *                      of both offset arrays)
 * Chunks are runs of whole sequences (contiguous in every tensor); each chunk's
 * upload, attn_fwd_varlen launch and download run on internal streams ordered
 * by events, as attn_fwd_host. Stream, ownership and results as attn_fwd_host
 * (bit-identical to attn_fwd_varlen). No counterpart on the pages.
 */
int64_t attn_fwd_varlen_host_workspace_bytes(int64_t B, int64_t Hq, int64_t Hkv, int64_t total_q,
                                             int64_t total_k, int64_t d);
int attn_fwd_varlen_host(const void* q, const void* k, const void* v, void* out,
                         const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int64_t B,
                         int64_t Hq, int64_t Hkv, int64_t total_q, int64_t total_k, int64_t d,
                         float scale, int rounding_mode, int flags, void* workspace,
                         int64_t workspace_bytes, void* stream);

/*
 * Debug build. The library built with -DATTN_DEBUG=1 (libattn_fwd_debug.so)
 * checks, inside the kernel, every computed tile coordinate, global row index
 * and the producer's count of ring fills; a failed check skips the access it
 * guards and raises a status that attn_fwd_last_error() returns as
 * ATTN_ERR_DEBUG_CHECK (no trap, no assert). It has no counterpart on the pages.
 *   attn_fwd_debug_build()     1 in the debug build, 0 in the release build
 *   attn_fwd_debug_selftest()  debug build: an attn_fwd launch (same arguments)
 *                              whose first thread reports one failed check
 *                              without any bad access, to test the reporting;
 *                              release build: ATTN_ERR_UNSUPPORTED, no launch
 */
int attn_fwd_debug_build(void);
int attn_fwd_debug_selftest(const void* q, const void* k, const void* v, void* out, int layout,
                            int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, float scale,
                            int rounding_mode, void* stream);

/*
 * Device-side status of earlier launches on the current device: ATTN_OK;
 * ATTN_ERR_TIMEOUT if some launch gave up on a wait that did not finish within
 * its time limit (the kernel then stops its work, waits for its own copies in
 * flight, frees its tensor memory and returns; its output is undefined); else
 * ATTN_ERR_SEQLENS if an attn_fwd_varlen launch found invalid offsets; else
 * ATTN_ERR_DEBUG_CHECK if a debug-build check failed.
 * Reading clears the status. Synchronize the stream that ran the calls first.
 */
int attn_fwd_last_error(void);

/*
 * attn_fwd_timeout_selftest - exercises the failure path on a real GPU.
 *
 * Same arguments, checks and launch as attn_fwd, plus a wait limit in
 * nanoseconds (1 .. 2e9) and flags (0 or ATTN_FLAG_SPLIT_TAIL, which runs the
 * launch as attn_fwd_ex with that flag would; any other bit gives
 * ATTN_ERR_UNSUPPORTED), but the kernel withholds one of its own internal
 * signals (the tensor-core warp never announces query tile 0's first S tile),
 * so a device-side wait must run out. Every role of the kernel then stops,
 * waits for the copies and matrix products it started, frees its tensor memory
 * and returns; no output is written (`out` keeps its old contents) and after the
 * stream is synchronized attn_fwd_last_error() reports ATTN_ERR_TIMEOUT. The
 * CUDA context stays usable. Returns ATTN_OK if the launch went out.
 */
int attn_fwd_timeout_selftest(const void* q, const void* k, const void* v, void* out, int layout,
                              int64_t B, int64_t H, int64_t Sq, int64_t Sk, int64_t d, float scale,
                              int rounding_mode, void* stream, uint64_t timeout_ns, int flags);

/* Library version, as MAJOR*10000 + MINOR*100 + PATCH. */
int attn_fwd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_H */
