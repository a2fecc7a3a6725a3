// modsrc.cuh -- the broadcast modulation sources of the LayerNorm producers:
// scale and shift of N consecutive columns (N = 8 or 2), and the AWQ
// smoothing multiplier, held as the raw source words and widened to fp32 one
// pair at a time where they are used (fewer live registers than fp32 copies).
//
// Sources (adaptive-layernorm-producers README, "Available Functions" and
// "Tensor Contract"):
//   MOD_BCAST   bf16 (dim,) scale / shift
//   MOD_AWQ     the same, plus a bf16 (dim,) inv_s that multiplies the
//               modulated activation before the FP8 quantiser
//   MOD_MODFP8  e4m3 (dim,) scale_fp8 / shift_fp8, each times its fp32 device
//               scalar: scale = decode(scale_fp8) * scale_deq (one fp32
//               product, exact when deq has <= 20 significant bits)
#pragma once

#include "device.cuh"
#include "kernels.h"

namespace nvfp4ap {

// The fp32 multipliers of a source's decoded values: (scale_deq, shift_deq)
// for MOD_MODFP8, unused (1) otherwise.
template <int MOD>
__device__ __forceinline__ float2 source_deq(const LnArgs& a) {
  if constexpr (MOD == MOD_MODFP8) return make_float2(__ldg(a.scale_deq), __ldg(a.shift_deq));
  return make_float2(1.0f, 1.0f);
}

// scale and shift of the N columns [col, col + N) of a broadcast source.
// Alignment: bf16 sources 2N bytes, e4m3 sources N bytes.
template <int MOD, int N>
struct BcastCols {
  static_assert(N == 8 || N == 2, "8 or 2 columns");
  static constexpr bool kE4m3 = (MOD == MOD_MODFP8);
  // raw words: bf16 pairs (N/2 words) or e4m3 bytes (N bytes)
  static constexpr int W = kE4m3 ? (N == 8 ? 2 : 1) : N / 2;
  uint32_t s[W], t[W];

  __device__ __forceinline__ void load(const LnArgs& a, int64_t col) {
    if constexpr (kE4m3 && N == 8) {
      const uint2 u = ld_reuse_v2(a.scale8 + col), v = ld_reuse_v2(a.shift8 + col);
      s[0] = u.x; s[1] = u.y; t[0] = v.x; t[1] = v.y;
    } else if constexpr (kE4m3) {
      s[0] = ld_reuse_b16(a.scale8 + col);
      t[0] = ld_reuse_b16(a.shift8 + col);
    } else if constexpr (N == 8) {
      const uint4 u = ld_reuse_v4(a.scale + col), v = ld_reuse_v4(a.shift + col);
      s[0] = u.x; s[1] = u.y; s[2] = u.z; s[3] = u.w;
      t[0] = v.x; t[1] = v.y; t[2] = v.z; t[3] = v.w;
    } else {
      s[0] = ld_reuse_b32(a.scale + col);
      t[0] = ld_reuse_b32(a.shift + col);
    }
  }
  // e4m3 bytes 2i, 2i + 1 of the raw words
  static __device__ __forceinline__ uint32_t half(const uint32_t (&w)[W], int i) {
    return (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu);
  }
  // zero scale and shift (both encodings decode all-zero words to 0)
  __device__ __forceinline__ void clear() {
#pragma unroll
    for (int i = 0; i < W; ++i) s[i] = t[i] = 0u;
  }
  // columns col + 2i, col + 2i + 1 as fp32; deq from source_deq<MOD>
  __device__ __forceinline__ float2 scale(int i, float2 deq) const {
    if constexpr (kE4m3) return mul2(e4m3x2_to_f2(half(s, i)), splat2(deq.x));
    return bf16x2_to_f2(s[i]);
  }
  __device__ __forceinline__ float2 shift(int i, float2 deq) const {
    if constexpr (kE4m3) return mul2(e4m3x2_to_f2(half(t, i)), splat2(deq.y));
    return bf16x2_to_f2(t[i]);
  }
};

// AWQ multipliers inv_s of the N columns [col, col + N) (bf16, 2N-byte aligned)
template <int N>
struct AwqCols {
  uint32_t w[N / 2];
  __device__ __forceinline__ void load(const LnArgs& a, int64_t col) {
    if constexpr (N == 8) {
      const uint4 u = ld_reuse_v4(a.inv_s + col);
      w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
    } else {
      w[0] = ld_reuse_b32(a.inv_s + col);
    }
  }
  __device__ __forceinline__ float2 mult(int i) const { return bf16x2_to_f2(w[i]); }
};

}  // namespace nvfp4ap
