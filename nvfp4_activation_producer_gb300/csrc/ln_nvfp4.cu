// ln_nvfp4.cu -- adaptive-LayerNorm -> NVFP4 producers for sm_103a.
//
// Operations (adaptive-layernorm-producers README, "Available Functions",
// "Tensor Contract", "Validation"):
//   ada_layer_norm_quant_nvfp4_swizzled_bf16        broadcast (dim,) scale/shift
//   layer_norm_no_affine_quant_nvfp4_swizzled_bf16  no modulation
// For each row: y = LayerNorm(x) * (1 + scale) + shift in fp32, staged to
// bf16 (v = bf16(y), the "staged BF16-norm plus FP4 quantizer" contract);
// per 16-element block: s = e4m3fn(amax/6), codes = e2m1 nearest of v/s
// (ties to even, sign kept, +-6 saturation), packed two per byte low nibble
// first; the block scale goes to the 128-row x 4-column tiled ("swizzled")
// layout, whose padding bytes are written as zero.  Rounding to nearest-even,
// signed zero and low-nibble-first packing follow the h3-blackwell-runtime
// compare page (PLAN.md "NVFP4 activation quantization status" and
// benchmarks/gb10-cute-nvfp4-conversion-contract.json); the tiled scale
// layout is its "general 128-row by 4-scale-column tiled offset".
//
// Design: `tpr` threads own a row; thread t owns the 16-element blocks
// t, t+tpr, ... (32 contiguous bytes each, so a warp reads 1 KB contiguous
// per step).  All loads of the row are issued first; statistics as in the
// FP8 kernels.  Per block, the staged bf16 values stay packed (bf16x2) for
// the magnitude max (max.xorsign.abs.bf16x2), the block scale is one fp32
// multiply and one cvt, and the e2m1 codes come from the hardware
// cvt.rn.satfinite.e2m1x2 applied to a quotient that is exact where it
// matters (see quotient() below).  Each block leaves as one 8-byte store of
// codes plus one scale byte; rows beyond `rows` up to the 128-row tile and
// block columns up to the 4-column tile get zero scale bytes from the
// threads that own them.
#include "device.cuh"
#include "kernels.h"

namespace nvfp4ap {
namespace {

// Byte offset of the scale of (row r, block column c) in the swizzled buffer
// with `ct` 4-column tiles per 128-row tile: tiles of 128x4 scales are 512
// contiguous bytes, row-tile major; inside a tile the byte is
// (r % 32) * 16 + ((r % 128) / 32) * 4 + c % 4.
__device__ __forceinline__ int64_t sf_off(int64_t r, int c, int ct) {
  return ((r >> 7) * ct + (c >> 2)) * 512 + (int)((r & 31) << 4) + (int)(((r >> 5) & 3) << 2) + (c & 3);
}

// v / s for the e2m1 decision.  q0 = v * rcp(s) is within a few ulp of v/s;
// the remainder e = v - q0*s is exact in fp32 (s has at most 4 significant
// bits and q0*s is within a few ulp of v), and q0 + e*rcp(s) rounds to v/s
// whenever v/s is a representable midpoint of the e2m1 grid.  Elsewhere v/s
// (8 significant bits over 4) is at least ~2^-9 (relative) away from every
// midpoint, far more than the error of either step, so the round-to-nearest
// decision of the hardware conversion equals that of the exact quotient.
// r = 0 when s = 0: then q = +-0 with the sign of v.
__device__ __forceinline__ float2 quotient(float2 v, float2 r2, float2 ns2) {
  float2 q0 = mul2(v, r2);
  float2 e = fma2(q0, ns2, v);
  return fma2(e, r2, q0);
}

__host__ __device__ constexpr int nvfp4_max_tpr(int bpt) { return bpt <= 2 ? 1024 : 512; }

template <int MOD, int BPT>
__global__ void __launch_bounds__(nvfp4_max_tpr(BPT)) ln_nvfp4_kernel(const LnArgs a) {
  __shared__ float red_sum[4][32];
  __shared__ float red_sq[4][32];

  const int tpr = blockDim.x;
  const int t = threadIdx.x;
  const int ry = threadIdx.y;
  const int lane = t & 31, warp = t >> 5, nwarps = (tpr + 31) >> 5;
  const int64_t D = a.dim;
  const int nblk = (int)(D >> 4);
  const int padc = (nblk + 3) & ~3;
  const int ct = padc >> 2;
  const int64_t row = (int64_t)blockIdx.x * blockDim.y + ry;
  const bool active = row < a.rows;
  uint8_t* sf = reinterpret_cast<uint8_t*>(a.sf);

  // ---- loads -----------------------------------------------------------------
  uint32_t xw[BPT][8];
  const uint16_t* xr = a.x + row * D;
#pragma unroll
  for (int k = 0; k < BPT; ++k) {
    const int b = t + k * tpr;
#pragma unroll
    for (int i = 0; i < 8; ++i) xw[k][i] = 0u;
    if (active && b < nblk) {
      uint4 lo = ld_once_v4(xr + (int64_t)b * 16);
      uint4 hi = ld_once_v4(xr + (int64_t)b * 16 + 8);
      xw[k][0] = lo.x; xw[k][1] = lo.y; xw[k][2] = lo.z; xw[k][3] = lo.w;
      xw[k][4] = hi.x; xw[k][5] = hi.y; xw[k][6] = hi.z; xw[k][7] = hi.w;
    }
  }

  // ---- statistics (as in the FP8 kernels; d = x - mean kept) ----------------
  float2 d[BPT][8];
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < BPT; ++k)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      d[k][i] = bf16x2_to_f2(xw[k][i]);
      acc = add2(acc, d[k][i]);
    }
  const float mean = row_sum(acc.x + acc.y, red_sum[ry], warp, nwarps, lane) / (float)D;
  float2 sq = make_float2(0.f, 0.f);
  const float2 nmean = splat2(-mean);
#pragma unroll
  for (int k = 0; k < BPT; ++k) {
    const bool valid = t + k * tpr < nblk;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      d[k][i] = add2(d[k][i], nmean);
      if (valid) sq = fma2(d[k][i], d[k][i], sq);
    }
  }
  const float var = row_sum(sq.x + sq.y, red_sq[ry], warp, nwarps, lane) / (float)D;

  if (!active) {
    // rows past the end inside the last 128-row tile: zero scale bytes
    const int64_t rows_pad = (a.rows + 127) & ~(int64_t)127;
    if (row < rows_pad)
      for (int c = t; c < padc; c += tpr) st_b8(sf + sf_off(row, c, ct), 0u);
    return;
  }

  const float rstd = 1.0f / sqrtf(var + a.eps);
  const float2 rstd2 = splat2(rstd);
  uint8_t* prow = reinterpret_cast<uint8_t*>(a.out) + row * (D >> 1);

#pragma unroll
  for (int k = 0; k < BPT; ++k) {
    const int b = t + k * tpr;
    if (b >= nblk) continue;
    uint32_t sc[8], sh[8];
    if constexpr (MOD == MOD_BCAST) {
      uint4 s0 = ld_reuse_v4(a.scale + (int64_t)b * 16), s1 = ld_reuse_v4(a.scale + (int64_t)b * 16 + 8);
      uint4 h0 = ld_reuse_v4(a.shift + (int64_t)b * 16), h1 = ld_reuse_v4(a.shift + (int64_t)b * 16 + 8);
      sc[0] = s0.x; sc[1] = s0.y; sc[2] = s0.z; sc[3] = s0.w;
      sc[4] = s1.x; sc[5] = s1.y; sc[6] = s1.z; sc[7] = s1.w;
      sh[0] = h0.x; sh[1] = h0.y; sh[2] = h0.z; sh[3] = h0.w;
      sh[4] = h1.x; sh[5] = h1.y; sh[6] = h1.z; sh[7] = h1.w;
    }
    // y = d * (rstd + rstd * scale) + shift, staged to bf16
    uint32_t vb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float2 y;
      if constexpr (MOD == MOD_BCAST)
        y = fma2(d[k][i], fma2(bf16x2_to_f2(sc[i]), rstd2, rstd2), bf16x2_to_f2(sh[i]));
      else
        y = mul2(d[k][i], rstd2);
      vb[i] = f2_to_bf16x2(y);
    }
    // block scale: e4m3(amax / 6).  amax is a bf16 value; multiplying by the
    // fp32 constant 1/6 instead of dividing by 6 gives the same e4m3 byte:
    // when 3 divides amax's significand the product rounds back to the exact
    // quotient (its error is below half an fp32 ulp), otherwise amax/6 is at
    // least ~2^-11 (relative) away from every e4m3 rounding boundary.
    uint32_t m = bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(vb[0], vb[1]), bf16x2_absmax(vb[2], vb[3])),
                               bf16x2_absmax(bf16x2_absmax(vb[4], vb[5]), bf16x2_absmax(vb[6], vb[7])));
    const float amax = fmaxf(fabsf(bf16_lo(m)), fabsf(bf16_hi(m)));
    const uint32_t sbyte = f2_to_e4m3x2(make_float2(amax * (1.0f / 6.0f), 0.f)) & 0xFFu;
    const float s = e4m3_to_f32(sbyte);
    const float r = (s == 0.f) ? 0.f : rcp_approx(s);
    const float2 r2 = splat2(r), ns2 = splat2(-s);
    float2 q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = quotient(bf16x2_to_f2(vb[i]), r2, ns2);
    const uint32_t w0 = f8_to_e2m1x8(q[0], q[1], q[2], q[3]);
    const uint32_t w1 = f8_to_e2m1x8(q[4], q[5], q[6], q[7]);
    st_stream_v2(prow + (int64_t)b * 8, w0, w1);
    st_b8(sf + sf_off(row, b, ct), sbyte);
  }
  // block columns past dim/16 inside the last 4-column tile: zero scale bytes
  for (int c = nblk + t; c < padc; c += tpr) st_b8(sf + sf_off(row, c, ct), 0u);
}

template <int MOD>
cudaError_t launch_mod(const LnArgs& a, RowShape s, cudaStream_t st) {
  const int64_t rows_pad = (a.rows + 127) & ~(int64_t)127;
  dim3 block(s.tpr, s.rpc);
  dim3 grid((unsigned)((rows_pad + s.rpc - 1) / s.rpc));
  switch (s.per_thread) {
#define NVFP4AP_CASE(N)                                       \
  case N:                                                     \
    ln_nvfp4_kernel<MOD, N><<<grid, block, 0, st>>>(a);       \
    break;
    NVFP4AP_CASE(1)
    NVFP4AP_CASE(2)
    NVFP4AP_CASE(3)
    NVFP4AP_CASE(4)
    NVFP4AP_CASE(6)
#undef NVFP4AP_CASE
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

int ln_nvfp4_max_tpr(int per_thread) {
  switch (per_thread) {
    case 1: case 2: case 3: case 4: case 6: return nvfp4_max_tpr(per_thread);
    default: return 0;
  }
}

cudaError_t launch_ln_nvfp4(const LnArgs& a, int mod, RowShape s, cudaStream_t st) {
  switch (mod) {
    case MOD_NONE: return launch_mod<MOD_NONE>(a, s, st);
    case MOD_BCAST: return launch_mod<MOD_BCAST>(a, s, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nvfp4ap
