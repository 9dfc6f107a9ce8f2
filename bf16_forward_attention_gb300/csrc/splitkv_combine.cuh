// splitkv_combine.cuh - merge of key-range splits for bf16 forward attention.
//
// A split s of the keys leaves, for every query row, an unnormalised output
// O_s = sum_j 2^(t_j - r_s) v_j and a row sum l_s = sum_j 2^(t_j - r_s), both
// relative to its own reference r_s (t_j = scaled logits in log2 units). The
// exact softmax over all keys is
//   O = sum_s 2^(r_s - R) O_s / sum_s 2^(r_s - R) l_s   for any common R,
// here R = max_s r_s (r_s = -Inf for a split with no finite logit). The sums
// run over s in a fixed order, so the result is bit-identical from run to run. Then the output is rounded to bf16 per mode as
// in the fused kernel (snilld.dk, "Open source attention-kernel i HIP slaar AITER
// v3 paa MI300X", section "Numerik samlet eet sted").
#pragma once
#include <stdint.h>

#include "attn_fwd_kernel.cuh"

namespace attn {

struct CombineParams {
  const float* part_o;   // [split][bh][sq_pad][128]
  const float* part_rl;  // [split][bh][sq_pad][2]
  uint16_t* out;         // bf16 bits, caller's layout
  int n_splits, BH, H, Sq, sq_pad, layout, mode;
};

// Four query rows per block of 128 threads: 32 threads per row, each owning four
// consecutive output columns (16-byte loads of the partial rows); the merge
// itself is merge_splits4, shared with the split kernel's own merge.
constexpr int kCombineRows = 4;

// Launched as a programmatic dependent of the split kernel: it may start while
// the split kernel's last CTAs still run, and waits here for that grid's writes.
__global__ void __launch_bounds__(kD) attn_splitkv_combine(const CombineParams p) {
  ptx::grid_dependency_wait();
  const int q = blockIdx.x * kCombineRows + (threadIdx.x >> 5);
  if (q >= p.Sq) return;
  const int bh = blockIdx.y;
  const int c0 = (threadIdx.x & 31) * 4;
  const size_t split_pitch = static_cast<size_t>(p.BH) * p.sq_pad;
  const uint2 o = merge_splits4(p.part_o, p.part_rl, static_cast<size_t>(bh) * p.sq_pad + q,
                                split_pitch, p.n_splits, c0, p.mode);
  const int b = bh / p.H, h = bh % p.H;
  const size_t idx = p.layout == 0 ? ((static_cast<size_t>(b) * p.H + h) * p.Sq + q) * kD + c0
                                   : ((static_cast<size_t>(b) * p.Sq + q) * p.H + h) * kD + c0;
  *reinterpret_cast<uint2*>(p.out + idx) = o;
}

}  // namespace attn
