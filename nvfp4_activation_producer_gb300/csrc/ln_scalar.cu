// ln_scalar.cu -- element-wise LayerNorm producers (FP8 e4m3fn and NVFP4) for
// inputs and outputs that are only element-aligned.
//
// Operations (adaptive-layernorm-producers README, "Available Functions",
// "Tensor Contract"; NVFP4 encoding facts from the h3-blackwell-runtime
// compare page):
//   y = (x - mean) * rstd * (1 + scale) + shift, rstd = 1/sqrt(var + eps),
//   scale/shift from any modulation source of kernels.h
//   FP8:   out = e4m3fn(y / act_scale) [AWQ: y * inv_s / act_scale]
//   NVFP4: v = bf16(y); per 16 elements s = e4m3fn(amax/6); e2m1 codes of
//          v/s, two per byte (low nibble first); s in the 128x4 tiled layout
//          with zero padding.
//
// The tensor contract asks only for contiguous tensors, so a caller may pass
// views whose data pointers are not 16-byte aligned (a slice at an odd row or
// element offset).  The vectorised kernels cannot read those; this one reads
// every element with its own load (2-byte bf16, 1-byte e4m3, 4-byte fp32) and
// writes outputs byte by byte, so it needs element alignment only.  It is the
// fallback for such pointers, not a fast path: one CTA of 256 threads per row,
// the statistics with the same shifted one-pass sums and fp32 operations as
// the vectorised kernels (within the same bounds of the reference).
#include "device.cuh"
#include "kernels.h"

namespace nvfp4ap {

// Set when a row's segment index is outside [0, nseg) (that row is produced
// with zero modulation); read and cleared by take_scalar_seg_fault().
__device__ unsigned int g_scalar_seg_fault = 0u;

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float ldf_bf16(const uint16_t* p) { return __uint_as_float((uint32_t)__ldg(p) << 16); }

// fp32 (1 + scale, shift) of column d of row r, and inv_s for AWQ
template <int MOD>
struct ScalarMod {
  const LnArgs& a;
  int64_t r;
  int seg;  // MOD_SEG: the row's segment, -1 when out of range
  float sdeq, hdeq;
  __device__ __forceinline__ ScalarMod(const LnArgs& args, int64_t row) : a(args), r(row), seg(0), sdeq(1.f), hdeq(1.f) {
    if constexpr (MOD == MOD_MODFP8) {
      sdeq = __ldg(a.scale_deq);
      hdeq = __ldg(a.shift_deq);
    }
    if constexpr (MOD == MOD_SEG) {
      const int32_t g = __ldg(a.seg_idx + r);
      seg = (g >= 0 && (int64_t)g < a.nseg) ? g : -1;
    }
  }
  __device__ __forceinline__ void at(int64_t d, float& gain, float& shift) const {
    const int64_t D = a.dim;
    float s = 0.f, h = 0.f;
    if constexpr (MOD == MOD_BCAST || MOD == MOD_AWQ) {
      s = ldf_bf16(a.scale + d);
      h = ldf_bf16(a.shift + d);
    } else if constexpr (MOD == MOD_PTOK) {
      s = ldf_bf16(a.scale + r * D + d);
      h = ldf_bf16(a.shift + r * D + d);
    } else if constexpr (MOD == MOD_TABLE) {
      const uint16_t* te = a.temb + r * a.chunks * D;
      s = ldf_bf16(te + a.scale_idx * D + d) + __ldg(a.table + a.scale_idx * D + d);
      h = ldf_bf16(te + a.shift_idx * D + d) + __ldg(a.table + a.shift_idx * D + d);
    } else if constexpr (MOD == MOD_MODFP8) {
      s = e4m3_to_f32(__ldg(a.scale8 + d)) * sdeq;
      h = e4m3_to_f32(__ldg(a.shift8 + d)) * hdeq;
    } else if constexpr (MOD == MOD_SEG) {
      if (seg >= 0) {
        s = ldf_bf16(a.seg_scale + (int64_t)seg * D + d);
        h = ldf_bf16(a.seg_shift + (int64_t)seg * D + d);
      }
    }
    gain = 1.0f + s;
    shift = h;
  }
};

__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t ct) {
  return ((r >> 7) * ct + (c >> 2)) * 512 + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (c & 3);
}

template <bool FP8, int MOD>
__global__ void __launch_bounds__(kThreads) ln_scalar_kernel(const LnArgs a, const float inv_d) {
  __shared__ float2 red[kThreads / 32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t D = a.dim, row = blockIdx.x;
  const int64_t nblk = D >> 4, padc = (nblk + 3) & ~(int64_t)3, ct = padc >> 2;
  pdl_enter();
  if (row >= a.rows) {
    if constexpr (!FP8)  // a padding row of the last 128-row scale tile
      for (int64_t c = t; c < padc; c += kThreads) st_b8(reinterpret_cast<uint8_t*>(a.sf) + sf_offset(row, c, ct), 0u);
    return;
  }
  const uint16_t* xr = a.x + row * D;
  const float K = ldf_bf16(xr);
  float s1 = 0.f, s2 = 0.f;
  for (int64_t d = t; d < D; d += kThreads) {
    const float v = ldf_bf16(xr + d) - K;
    s1 += v;
    s2 = fmaf(v, v, s2);
  }
  float2 s = make_float2(s1, s2);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s.x += __shfl_xor_sync(0xFFFFFFFFu, s.x, o);
    s.y += __shfl_xor_sync(0xFFFFFFFFu, s.y, o);
  }
  if (lane == 0) red[warp] = s;
  __syncthreads();
  s = red[0];
#pragma unroll
  for (int v = 1; v < kThreads / 32; ++v) {
    s.x += red[v].x;
    s.y += red[v].y;
  }
  const float m1 = s.x * inv_d;  // mean - K
  const float var = fmaxf(fmaf(s.y, inv_d, -m1 * m1), 0.f);
  const float rstd = rsqrtf(var + a.eps);
  const ScalarMod<MOD> mod(a, row);
  if constexpr (MOD == MOD_SEG)
    if (mod.seg < 0 && t == 0) atomicOr(&g_scalar_seg_fault, 1u);

  if constexpr (FP8) {
    const float inv_act = 1.0f / __ldg(a.act_scale);
    const float A = MOD == MOD_NONE ? rstd * inv_act : rstd;
    uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) + row * D;
    for (int64_t d = t; d < D; d += kThreads) {
      float y = fmaf(ldf_bf16(xr + d) - K, A, -m1 * A);
      if constexpr (MOD != MOD_NONE) {
        float g, h;
        mod.at(d, g, h);
        const float f = MOD == MOD_AWQ ? ldf_bf16(a.inv_s + d) * inv_act : inv_act;
        y = fmaf(y, g, h) * f;
      }
      st_b8(orow + d, f2_to_e4m3x2(make_float2(y, 0.f)) & 0xFFu);
    }
    return;
  }
  uint8_t* prow = reinterpret_cast<uint8_t*>(a.out) + row * (D >> 1);
  uint8_t* sf = reinterpret_cast<uint8_t*>(a.sf);
  for (int64_t b = t; b < padc; b += kThreads) {
    if (b >= nblk) {  // a padding column of the scale tile
      st_b8(sf + sf_offset(row, b, ct), 0u);
      continue;
    }
    float v[16];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t d = b * 16 + i;
      float y = fmaf(ldf_bf16(xr + d) - K, rstd, -m1 * rstd);
      if constexpr (MOD != MOD_NONE) {
        float g, h;
        mod.at(d, g, h);
        y = fmaf(y, g, h);
      }
      v[i] = bf16_lo(f2_to_bf16x2(make_float2(y, 0.f)));  // the staged bf16 value
      amax = fmaxf(amax, fabsf(v[i]));
    }
    // amax * (1/6) in fp32 rounds to the same e4m3 byte as the exact quotient
    // (amax has 8 significant bits); codes from v * (r_hi + r_lo), the
    // Newton-corrected reciprocal: exact at every e2m1 midpoint
    const uint32_t sbyte = f2_to_e4m3x2(make_float2(amax * (1.0f / 6.0f), 0.f)) & 0xFFu;
    const float scl = e4m3_to_f32(sbyte);
    const float rh = (scl == 0.f) ? 0.f : rcp_approx(scl);
    const float rl = rh * fmaf(-scl, rh, 1.0f);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float2 q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 vv = make_float2(v[8 * j + 2 * i], v[8 * j + 2 * i + 1]);
        q[i] = fma2(vv, splat2(rh), mul2(vv, splat2(rl)));
      }
      const uint32_t c = f8_to_e2m1x8(q[0], q[1], q[2], q[3]);
#pragma unroll
      for (int k = 0; k < 4; ++k) st_b8(prow + b * 8 + j * 4 + k, (c >> (8 * k)) & 0xFFu);
    }
    st_b8(sf + sf_offset(row, b, ct), sbyte);
  }
}

template <bool FP8, int MOD>
cudaError_t launch_k(const LnArgs& a, cudaStream_t st) {
  const int64_t work = FP8 ? a.rows : (a.rows + 127) / 128 * 128;
  const float inv_d = (float)(1.0 / (double)a.dim);
  return launch_maybe_pdl(ln_scalar_kernel<FP8, MOD>, dim3((unsigned)work), dim3(kThreads), 0, st, a, inv_d);
}

}  // namespace

cudaError_t launch_ln_scalar(const LnArgs& a, bool nvfp4, int mod, cudaStream_t st) {
  if (nvfp4) {
    switch (mod) {
      case MOD_NONE: return launch_k<false, MOD_NONE>(a, st);
      case MOD_BCAST: return launch_k<false, MOD_BCAST>(a, st);
      case MOD_MODFP8: return launch_k<false, MOD_MODFP8>(a, st);
      case MOD_SEG: return launch_k<false, MOD_SEG>(a, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (mod) {
    case MOD_NONE: return launch_k<true, MOD_NONE>(a, st);
    case MOD_BCAST: return launch_k<true, MOD_BCAST>(a, st);
    case MOD_PTOK: return launch_k<true, MOD_PTOK>(a, st);
    case MOD_TABLE: return launch_k<true, MOD_TABLE>(a, st);
    case MOD_MODFP8: return launch_k<true, MOD_MODFP8>(a, st);
    case MOD_AWQ: return launch_k<true, MOD_AWQ>(a, st);
    case MOD_SEG: return launch_k<true, MOD_SEG>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t take_scalar_seg_fault(unsigned int* fault) {
  unsigned int zero = 0u;
  cudaError_t e = cudaMemcpyFromSymbol(fault, g_scalar_seg_fault, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_scalar_seg_fault, &zero, sizeof(unsigned int));
}

}  // namespace nvfp4ap
