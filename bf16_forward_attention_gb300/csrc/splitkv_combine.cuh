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
// consecutive output columns (16-byte loads of the partial rows). The loops over
// the splits are unrolled so that their independent loads overlap; the sums still
// run in split order.
constexpr int kCombineRows = 4;

__global__ void __launch_bounds__(kD) attn_splitkv_combine(const CombineParams p) {
  const int q = blockIdx.x * kCombineRows + (threadIdx.x >> 5);
  if (q >= p.Sq) return;
  const int bh = blockIdx.y;
  const int c0 = (threadIdx.x & 31) * 4;
  const float2* rl = reinterpret_cast<const float2*>(p.part_rl);
  const size_t split_pitch = static_cast<size_t>(p.BH) * p.sq_pad;
  const size_t row0 = static_cast<size_t>(bh) * p.sq_pad + q;

  // R = max over splits of r_s. A split with no finite logit has r_s = -Inf and
  // weight 0 (its sums are 0, or NaN which then propagates as it must). If every
  // split is like that, R = 0 keeps the weights at 0 and 0/0 gives NaN.
  float R = -__int_as_float(0x7F800000);
#pragma unroll 8
  for (int s = 0; s < p.n_splits; ++s) R = fmaxf(R, rl[row0 + s * split_pitch].x);
  if (R == -__int_as_float(0x7F800000)) R = 0.f;
  float L = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
  for (int s = 0; s < p.n_splits; ++s) {
    const size_t r = row0 + s * split_pitch;
    const float2 ml = rl[r];
    const float w = ptx::ex2(ml.x - R);  // NaN only if R = +Inf: that row is NaN anyway
    const float4 x = *reinterpret_cast<const float4*>(p.part_o + r * kD + c0);
    L = fmaf(ml.y, w, L);
    o.x = fmaf(x.x, w, o.x);
    o.y = fmaf(x.y, w, o.y);
    o.z = fmaf(x.z, w, o.z);
    o.w = fmaf(x.w, w, o.w);
  }
  const float inv = __frcp_rn(L);
  const int b = bh / p.H, h = bh % p.H;
  const size_t idx = p.layout == 0 ? ((static_cast<size_t>(b) * p.H + h) * p.Sq + q) * kD + c0
                                   : ((static_cast<size_t>(b) * p.Sq + q) * p.H + h) * kD + c0;
  const uint32_t lo = round_bf16_bits(o.x * inv, p.mode) | (round_bf16_bits(o.y * inv, p.mode) << 16);
  const uint32_t hi = round_bf16_bits(o.z * inv, p.mode) | (round_bf16_bits(o.w * inv, p.mode) << 16);
  *reinterpret_cast<uint2*>(p.out + idx) = make_uint2(lo, hi);
}

}  // namespace attn
