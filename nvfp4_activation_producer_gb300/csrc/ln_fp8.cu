// ln_fp8.cu -- adaptive-LayerNorm -> FP8 (e4m3fn) producers for sm_103a.
//
// Operations (adaptive-layernorm-producers README, "Available Functions" and
// "Tensor Contract"):
//   ada_layer_norm_quant_fp8_bf16            broadcast (dim,) scale/shift
//   ada_layer_norm_quant_fp8_ptok_bf16       per-token (rows, dim) scale/shift
//   ada_layer_norm_quant_fp8_ptok_table_bf16 scale/shift = temb[r,idx,:] + table[idx,:]
//   layer_norm_no_affine_quant_fp8_static_bf16   no modulation
//   ada_layer_norm_quant_fp8_modfp8_bf16     e4m3 (dim,) scale/shift times fp32 deq scalars
//   awq_ada_layer_norm_quant_fp8_bf16        broadcast, y multiplied by inv_s
// For each row: mean and biased variance over dim, rstd = 1/sqrt(var+eps),
// y = (x - mean) * rstd * (1 + scale) + shift, out = e4m3fn(y / act_scale)
// rounded to nearest-even and saturated to +-448.
//
// This file serves the bf16-pair path: rows whose dim is even but not a
// multiple of 8, or bf16 pointers that are 4-byte but not 16-byte aligned (a
// thread loads one bf16 pair per vector, VEC = 2), and per-token rows too
// long for the register row kernels.
//
// Design: a row is owned by `tpr` threads (one warp up to one CTA, picked by
// dim on the host).  Every thread issues all of its loads of the row (and of
// per-token modulation rows) before any arithmetic, so x is read from HBM
// exactly once and a whole row is in flight per thread group; the values stay
// in registers.  Statistics: fp32 sum -> mean, then the centred sum of
// squares from the registers (two sweeps over registers, one pass over
// memory), warp shuffles then one shared-memory step across the row's warps.
// Packed fp32x2 arithmetic does the normalise/modulate/scale, and
// cvt.rn.satfinite.e4m3x2 produces two codes per instruction; each 8-element
// vector leaves as one 8-byte streaming store.
#include "device.cuh"
#include "kernels.h"
#include "modsrc.cuh"

namespace nvfp4ap {
namespace {

template <int VEC>
struct Vec {
  static constexpr int W = VEC / 2;  // 32-bit words (bf16 pairs) per vector
};

template <int VEC>
__device__ __forceinline__ void load_once(uint32_t (&w)[VEC / 2], const uint16_t* p) {
  if constexpr (VEC == 8) {
    uint4 v = ld_once_v4(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    w[0] = ld_once_b32(p);
  }
}

template <int VEC>
__device__ __forceinline__ void load_reuse(uint32_t (&w)[VEC / 2], const uint16_t* p) {
  if constexpr (VEC == 8) {
    uint4 v = ld_reuse_v4(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  } else {
    w[0] = ld_reuse_b32(p);
  }
}

// Largest number of threads per row (and per CTA) an (NV, VEC) instance is
// launched with.  It bounds the registers per thread (65536 / bound), which
// must hold NV vectors of x plus, per token, NV vectors each of scale and
// shift.  The host never picks a shape above it.
__host__ __device__ constexpr int fp8_max_tpr(int nv, int vec) {
  return vec == 8 ? (nv <= 2 ? 1024 : 512) : (nv <= 4 ? 1024 : 512);
}

template <int MOD, int NV, int VEC>
__global__ void __launch_bounds__(fp8_max_tpr(NV, VEC)) ln_fp8_kernel(const LnArgs a) {
  constexpr int W = Vec<VEC>::W;
  constexpr bool kPerToken = (MOD == MOD_PTOK || MOD == MOD_TABLE);
  // Per-token modulation rows are fetched together with x (more bytes in
  // flight) unless that would not fit the register budget of wide rows.
  constexpr bool kPerTokenRegs = kPerToken && NV * W <= 16;
  __shared__ float red_sum[4][32];
  __shared__ float red_sq[4][32];

  const int tpr = blockDim.x;
  const int t = threadIdx.x;
  const int ry = threadIdx.y;
  const int lane = t & 31, warp = t >> 5, nwarps = (tpr + 31) >> 5;
  const int64_t D = a.dim;
  const int nvec = (int)(D / VEC);
  const int64_t row = (int64_t)blockIdx.x * blockDim.y + ry;
  const bool active = row < a.rows;

  // ---- issue every load of this thread's part of the row ----------------
  uint32_t xw[NV][W];
  uint32_t scw[kPerTokenRegs ? NV : 1][W];
  uint32_t shw[kPerTokenRegs ? NV : 1][W];
  const uint16_t* xr = a.x + row * D;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int j = t + k * tpr;
    const bool valid = active && j < nvec;
#pragma unroll
    for (int i = 0; i < W; ++i) xw[k][i] = 0u;
    if (valid) {
      load_once<VEC>(xw[k], xr + (int64_t)j * VEC);
      if constexpr (MOD == MOD_PTOK && kPerTokenRegs) {
        load_once<VEC>(scw[k], a.scale + row * D + (int64_t)j * VEC);
        load_once<VEC>(shw[k], a.shift + row * D + (int64_t)j * VEC);
      } else if constexpr (MOD == MOD_TABLE && kPerTokenRegs) {
        const uint16_t* te = a.temb + row * a.chunks * D + (int64_t)j * VEC;
        load_once<VEC>(scw[k], te + a.scale_idx * D);
        load_once<VEC>(shw[k], te + a.shift_idx * D);
      }
    }
  }

  // ---- statistics: mean, then the centred sum of squares ------------------
  // x is widened to fp32 once; d = x - mean (exact for values near the mean)
  // replaces it in place and is what the output step scales.
  float2 d[NV][W];
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int i = 0; i < W; ++i) {
      d[k][i] = bf16x2_to_f2(xw[k][i]);
      acc = add2(acc, d[k][i]);  // padding words are 0
    }
  const float mean = row_sum(acc.x + acc.y, red_sum[ry], warp, nwarps, lane) / (float)D;

  float2 sq = make_float2(0.f, 0.f);
  const float2 nmean = splat2(-mean);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const bool valid = t + k * tpr < nvec;
#pragma unroll
    for (int i = 0; i < W; ++i) {
      d[k][i] = add2(d[k][i], nmean);
      if (valid) sq = fma2(d[k][i], d[k][i], sq);
    }
  }
  const float var = row_sum(sq.x + sq.y, red_sq[ry], warp, nwarps, lane) / (float)D;
  if (!active) return;  // no barrier follows

  // y = d * rstd * (1 + scale) + shift and q = y / act_scale, as
  // q = (d * a + shift) * inv with a = rstd + rstd * scale (one rounding)
  const float rstd = 1.0f / sqrtf(var + a.eps);
  const float inv_act = 1.0f / __ldg(a.act_scale);
  const float2 rstd2 = splat2(rstd), inv2 = splat2(inv_act), rinv2 = splat2(rstd * inv_act);
  const float2 deq = source_deq<MOD>(a);

  // ---- normalise, modulate, quantise, store -------------------------------
  uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) + row * D;
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int j = t + k * tpr;
    if (j >= nvec) continue;
    const int64_t col = (int64_t)j * VEC;
    uint32_t sc[W], sh[W];
    BcastCols<mod_is_bcast(MOD) ? MOD : MOD_BCAST, VEC> bc;
    AwqCols<VEC> aw;
    if constexpr (mod_is_bcast(MOD)) {
      bc.load(a, col);
      if constexpr (MOD == MOD_AWQ) aw.load(a, col);
    } else if constexpr (kPerTokenRegs) {
#pragma unroll
      for (int i = 0; i < W; ++i) { sc[i] = scw[k][i]; sh[i] = shw[k][i]; }
    } else if constexpr (MOD == MOD_PTOK) {
      load_once<VEC>(sc, a.scale + row * D + col);
      load_once<VEC>(sh, a.shift + row * D + col);
    } else if constexpr (MOD == MOD_TABLE) {
      const uint16_t* te = a.temb + row * a.chunks * D + col;
      load_once<VEC>(sc, te + a.scale_idx * D);
      load_once<VEC>(sh, te + a.shift_idx * D);
    }
    uint32_t codes[W];
#pragma unroll
    for (int i = 0; i < W; ++i) {
      float2 q;
      if constexpr (MOD == MOD_NONE) {
        q = mul2(d[k][i], rinv2);
      } else if constexpr (mod_is_bcast(MOD)) {
        const float2 f = MOD == MOD_AWQ ? mul2(aw.mult(i), inv2) : inv2;
        q = mul2(fma2(d[k][i], fma2(bc.scale(i, deq), rstd2, rstd2), bc.shift(i, deq)), f);
      } else {
        float2 s = bf16x2_to_f2(sc[i]);
        float2 h = bf16x2_to_f2(sh[i]);
        if constexpr (MOD == MOD_TABLE) {
          s = add2(s, ld_reuse_f2(a.table + a.scale_idx * D + col + 2 * i));
          h = add2(h, ld_reuse_f2(a.table + a.shift_idx * D + col + 2 * i));
        }
        q = mul2(fma2(d[k][i], fma2(s, rstd2, rstd2), h), inv2);
      }
      codes[i] = f2_to_e4m3x2(q);
    }
    if constexpr (VEC == 8) {
      st_stream_v2(orow + col, codes[0] | (codes[1] << 16), codes[2] | (codes[3] << 16));
    } else {
      st_stream_b16(orow + col, (uint16_t)codes[0]);
    }
  }
}

template <int MOD, int VEC>
cudaError_t launch_mod(const LnArgs& a, RowShape s, cudaStream_t st) {
  dim3 block(s.tpr, s.rpc);
  dim3 grid((unsigned)((a.rows + s.rpc - 1) / s.rpc));
#define NVFP4AP_CASE(N)                                     \
  case N:                                                   \
    ln_fp8_kernel<MOD, N, VEC><<<grid, block, 0, st>>>(a);  \
    break;
  switch (s.per_thread) {
    NVFP4AP_CASE(2)
    NVFP4AP_CASE(4)
    NVFP4AP_CASE(8)
    NVFP4AP_CASE(16)
    NVFP4AP_CASE(32)
    default: return cudaErrorInvalidValue;
  }
#undef NVFP4AP_CASE
  return cudaGetLastError();
}

template <int VEC>
cudaError_t launch_vec(const LnArgs& a, int mod, RowShape s, cudaStream_t st) {
  switch (mod) {
    case MOD_NONE: return launch_mod<MOD_NONE, VEC>(a, s, st);
    case MOD_BCAST: return launch_mod<MOD_BCAST, VEC>(a, s, st);
    case MOD_PTOK: return launch_mod<MOD_PTOK, VEC>(a, s, st);
    case MOD_TABLE: return launch_mod<MOD_TABLE, VEC>(a, s, st);
    case MOD_MODFP8: return launch_mod<MOD_MODFP8, VEC>(a, s, st);
    case MOD_AWQ: return launch_mod<MOD_AWQ, VEC>(a, s, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int ln_fp8_max_tpr(int vec, int per_thread) {
  if (vec == 2) {
    switch (per_thread) {
      case 2: case 4: case 8: case 16: case 32: return fp8_max_tpr(per_thread, 2);
      default: return 0;
    }
  }
  return 0;
}

cudaError_t launch_ln_fp8(const LnArgs& a, int mod, int vec, RowShape s, cudaStream_t st) {
  if (vec == 2) return launch_vec<2>(a, mod, s, st);
  return cudaErrorInvalidValue;
}

}  // namespace nvfp4ap
