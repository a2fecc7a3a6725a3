// ln_rows.cuh -- the register-row LayerNorm producer kernel template
// (FP8, NVFP4 single-level, and the two passes of the two-level NVFP4 contract)
// and its launch helper, shared by the translation units that instantiate it.
//
// Operations (adaptive-layernorm-producers README, "Available Functions",
// "Tensor Contract", "Validation"; NVFP4 encoding facts from the
// h3-blackwell-runtime compare page):
//   y = (x - mean) * rstd * (1 + scale) + shift, rstd = 1/sqrt(var + eps),
//   scale/shift from one of the modulation sources of kernels.h (the AWQ
//   source also multiplies y by inv_s)
//   FP8:   out = e4m3fn(y / act_scale), nearest-even, saturating
//   NVFP4: v = bf16(y); per 16 elements s = e4m3fn(amax/6); e2m1 codes of
//          v/s, two per byte (low nibble first); s in the 128x4 tiled layout
//          with zero padding.
//   Two-level NVFP4 (h3-blackwell-runtime compare page: "Numerical
//   Constraint" and the P1 checkpoint's "numerical_contract"), two launches:
//     KIND_AMAX: v as above; the largest |v| of the whole tensor into one
//                device word (atomic max of the non-negative fp32 bits);
//     KIND_NV2L: ts = bf16(amax / 2688) from that word; per 16 elements
//                s = e4m3fn(min((amax_b / 6) / ts, 448)) with both
//                quotients correctly rounded in fp32; e2m1 codes of v / (s * ts).
//
// Design.  A row is owned by `tpr` threads (a warp or a few warps); thread t
// owns the 8-element chunks t, t+tpr, ... of the row (a warp reads 512
// contiguous bytes per step).  Every load of the row -- and of its per-token
// modulation rows -- is issued before any arithmetic and the row stays in
// registers as packed bf16, so x is read from HBM exactly once.  The shape is
// chosen so that each thread holds many elements (up to 96): the per-row work
// (two-value reduction, rsqrt) is then small next to the per-element work,
// which is what bounds these kernels on GB300 (a 3-byte-per-element stream
// leaves ~18 instructions per element at full HBM bandwidth).
//
// Statistics in one pass over the registers, shifted by the row's first
// element K (exact and identical for every thread): s1 = sum(x - K),
// s2 = sum((x - K)^2); mean = K + s1/D, var = s2/D - (s1/D)^2.  The shift keeps
// the cancellation small for rows whose mean is large against their spread,
// and a constant row gives s1 = s2 = 0, so mean = K and x - mean = 0 exactly.
#pragma once

#include "device.cuh"
#include "kernels.h"
#include "modsrc.cuh"

// the maximum pass returns early from the shared NVFP4 path; the code after
// that return is unreachable in its instances by design
#pragma nv_diag_suppress 128

namespace nvfp4ap {
namespace {

enum { KIND_FP8 = 0, KIND_NVFP4 = 1, KIND_AMAX = 2, KIND_NV2L = 3 };

// Set when a row's segment index is outside [0, nseg): that row is produced
// with zero modulation instead of reading outside the tables.  One word per
// translation unit; only the unit that instantiates MOD_SEG writes it.
__device__ unsigned int g_seg_fault = 0u;

// fp32 -> the nearest bf16 value, as fp32 (round to nearest even)
__device__ __forceinline__ float round_bf16(float v) { return bf16_lo(f2_to_bf16x2(make_float2(v, 0.f))); }

// Resident 128-thread CTAs per SM the FULL instances are compiled for (40
// registers per thread): measured best on GB300 for the NVFP4 producers at
// dim 2048-4096 (32 registers spill, and uncapped instances hold fewer warps).
constexpr int kFullMinBlocks = 12;

__device__ __forceinline__ int64_t sf_off(int64_t r, int c, int ct) {
  return ((r >> 7) * ct + (c >> 2)) * 512 + (int)((r & 31) << 4) + (int)(((r >> 5) & 3) << 2) + (c & 3);
}

__device__ __forceinline__ void unpack4(uint4 v, uint32_t (&w)[4]) {
  w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
}

// Largest threads-per-row of an instance: NV chunks of 8 elements per thread,
// dim <= 32768 -> 4096 chunks per row.
__host__ __device__ constexpr int rows_max_tpr(int nv) {
  return ((4096 + nv - 1) / nv + 31) / 32 * 32 > 512 ? 512 : ((4096 + nv - 1) / nv + 31) / 32 * 32;
}

// FULL (FULLMB > 0): the row is exactly NV * tpr chunks (no thread holds a
// chunk past the end), the CTA is one row of at most 128 threads, and
// registers are capped for FULLMB resident CTAs of 128 threads per SM.
// Measured on GB300 for the NVFP4 layer norm at 5070 rows: 15% faster than
// the uncapped kernel at dim 3072, 13% at 4096 -- the NVFP4 encode is a chain
// of dependent steps, and more resident warps hide its latency.
template <int KIND, int MOD, int NV, int FULLMB = 0>
__global__ void __launch_bounds__(FULLMB ? 128 : 512, FULLMB ? FULLMB : 1) ln_rows_kernel(const LnArgs a, const float inv_d) {
  constexpr bool kPerToken = (MOD == MOD_PTOK || MOD == MOD_TABLE);
  constexpr bool kScales = (KIND == KIND_NVFP4 || KIND == KIND_NV2L);  // writes codes and scales
  __shared__ float2 red[16][16];  // [row group][warp of the row]

  const int tpr = blockDim.x;
  const int t = threadIdx.x, ry = FULLMB ? 0 : threadIdx.y;  // FULL: one row per CTA
  const int lane = t & 31, warp = t >> 5, nwarps = tpr >> 5;
  const int64_t D = a.dim;
  const int nch = (int)(D >> 3);
  constexpr bool FULL = FULLMB > 0;
  const int64_t row = (int64_t)blockIdx.x * blockDim.y + ry;
  const bool active = row < a.rows;
  const int64_t rbase = active ? row * D : 0;
  pdl_enter();

  // ---- all loads of the row first -------------------------------------------
  uint32_t xw[NV][4];
  uint32_t sw[kPerToken ? NV : 1][4], hw[kPerToken ? NV : 1][4];
  const uint16_t* sc_src = nullptr;
  const uint16_t* sh_src = nullptr;
  if constexpr (MOD == MOD_PTOK) {
    sc_src = a.scale + rbase;
    sh_src = a.shift + rbase;
  } else if constexpr (MOD == MOD_TABLE) {
    const uint16_t* te = a.temb + (active ? row * a.chunks * D : 0);
    sc_src = te + a.scale_idx * D;
    sh_src = te + a.shift_idx * D;
  }
  // segmented source: the row's segment selects one row of the (nseg, dim)
  // tables, read chunk by chunk where it is used (the tables are shared by
  // many rows and stay in L1/L2, like the broadcast vectors)
  bool have_src = true;
  if constexpr (MOD == MOD_SEG) {
    const int g = active ? __ldg(a.seg_idx + row) : 0;
    have_src = g >= 0 && g < a.nseg;
    if (active && !have_src && t == 0) atomicOr(&g_seg_fault, 1u);
    sc_src = a.seg_scale + (have_src ? (int64_t)g * D : 0);
    sh_src = a.seg_shift + (have_src ? (int64_t)g * D : 0);
  }
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int j = t + k * tpr;
    if (active && (FULL || j < nch)) {
      unpack4(ld_once_v4(a.x + rbase + (int64_t)j * 8), xw[k]);
      if constexpr (kPerToken) {
        unpack4(ld_once_v4(sc_src + (int64_t)j * 8), sw[k]);
        unpack4(ld_once_v4(sh_src + (int64_t)j * 8), hw[k]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) xw[k][i] = 0u;
    }
  }
  const float K = active ? __uint_as_float((uint32_t)__ldg(a.x + rbase) << 16) : 0.f;

  // ---- statistics: one pass, shifted by K -------------------------------------
  // dk = x - K stays in registers (fp32) for the output step.
  float2 dk[NV][4];
  float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
  const float2 nk = splat2(-K);
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const bool valid = FULL || t + k * tpr < nch;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      dk[k][i] = add2(bf16x2_to_f2(xw[k][i]), nk);
      if (valid) {
        s1 = add2(s1, dk[k][i]);
        s2 = fma2(dk[k][i], dk[k][i], s2);
      }
    }
  }
  float2 s = make_float2(s1.x + s1.y, s2.x + s2.y);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s.x += __shfl_xor_sync(0xFFFFFFFFu, s.x, o);
    s.y += __shfl_xor_sync(0xFFFFFFFFu, s.y, o);
  }
  if (nwarps > 1) {
    if (lane == 0) red[ry][warp] = s;
    __syncthreads();
    s = red[ry][0];
    for (int w = 1; w < nwarps; ++w) {
      const float2 u = red[ry][w];
      s.x += u.x;
      s.y += u.y;
    }
  }
  if (!active) {
    if constexpr (kScales) {
      // rows past the end inside the last 128-row tile: zero scale bytes
      const int nblk = nch >> 1, padc = (nblk + 3) & ~3, ct = padc >> 2;
      const int64_t rows_pad = (a.rows + 127) & ~(int64_t)127;
      if (row < rows_pad)
        for (int c = t; c < padc; c += tpr) st_b8(reinterpret_cast<uint8_t*>(a.sf) + sf_off(row, c, ct), 0u);
    }
    return;
  }
  const float m1 = s.x * inv_d;  // mean - K
  const float var = fmaxf(fmaf(s.y, inv_d, -m1 * m1), 0.f);
  const float rstd = rsqrtf(var + a.eps);
  const float2 nm1 = splat2(-m1);  // x - mean = dk - m1

  if constexpr (KIND == KIND_FP8) {
    // ---- FP8: q = (x - mean) * rstd * (1 + scale) + shift) / act_scale ------
    const float inv_act = 1.0f / __ldg(a.act_scale);
    const float2 rstd2 = splat2(rstd), inv2 = splat2(inv_act), rinv2 = splat2(rstd * inv_act);
    const float2 deq = source_deq<MOD>(a);
    uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) + row * D;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int j = t + k * tpr;
      if (!FULL && j >= nch) continue;
      uint32_t sc[4], sh[4];
      BcastCols<MOD, 8> bc;
      AwqCols<8> aw;
      if constexpr (mod_is_bcast(MOD)) {
        bc.load(a, (int64_t)j * 8);
        if constexpr (MOD == MOD_AWQ) aw.load(a, (int64_t)j * 8);
      } else if constexpr (kPerToken) {
#pragma unroll
        for (int i = 0; i < 4; ++i) { sc[i] = sw[k][i]; sh[i] = hw[k][i]; }
      } else if constexpr (MOD == MOD_SEG) {
        if (have_src) {
          unpack4(ld_reuse_v4(sc_src + (int64_t)j * 8), sc);
          unpack4(ld_reuse_v4(sh_src + (int64_t)j * 8), sh);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) sc[i] = sh[i] = 0u;
        }
      }
      float2 tg[4], th[4];
      if constexpr (MOD == MOD_TABLE) {
        // the two fp32 table rows of this chunk, 32 bytes each
        const float* ts = a.table + a.scale_idx * D + (int64_t)j * 8;
        const float* tsh = a.table + a.shift_idx * D + (int64_t)j * 8;
        const float4 t0 = ld_reuse_f4(ts), t1 = ld_reuse_f4(ts + 4), u0 = ld_reuse_f4(tsh), u1 = ld_reuse_f4(tsh + 4);
        tg[0] = make_float2(t0.x, t0.y); tg[1] = make_float2(t0.z, t0.w);
        tg[2] = make_float2(t1.x, t1.y); tg[3] = make_float2(t1.z, t1.w);
        th[0] = make_float2(u0.x, u0.y); th[1] = make_float2(u0.z, u0.w);
        th[2] = make_float2(u1.x, u1.y); th[3] = make_float2(u1.z, u1.w);
      }
      uint32_t q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 d = add2(dk[k][i], nm1);
        float2 y;
        if constexpr (MOD == MOD_NONE) {
          y = mul2(d, rinv2);
        } else if constexpr (mod_is_bcast(MOD)) {
          // AWQ: y * inv_s / act_scale as y * (inv_s * (1 / act_scale))
          const float2 f = MOD == MOD_AWQ ? mul2(aw.mult(i), inv2) : inv2;
          y = mul2(fma2(d, fma2(bc.scale(i, deq), rstd2, rstd2), bc.shift(i, deq)), f);
        } else {
          float2 g = bf16x2_to_f2(sc[i]), h = bf16x2_to_f2(sh[i]);
          if constexpr (MOD == MOD_TABLE) {
            g = add2(g, tg[i]);
            h = add2(h, th[i]);
          }
          y = mul2(fma2(d, fma2(g, rstd2, rstd2), h), inv2);
        }
        q[i] = f2_to_e4m3x2(y);
      }
      st_stream_v2(orow + (int64_t)j * 8, q[0] | (q[1] << 16), q[2] | (q[3] << 16));
    }
  } else {
    // ---- NVFP4: chunk j is half of block j/2; lanes t and t^1 hold the halves
    const int nblk = nch >> 1, padc = (nblk + 3) & ~3, ct = padc >> 2;
    const float2 rstd2 = splat2(rstd);
    uint8_t* prow = reinterpret_cast<uint8_t*>(a.out) + row * (D >> 1);
    // this row's part of the 128x4 tiled scale offset; a block column c adds
    // (c / 4) * 512 + c % 4
    uint8_t* sfrow = reinterpret_cast<uint8_t*>(a.sf) + (row >> 7) * (int64_t)ct * 512 +
                     (int)((row & 31) << 4) + (int)(((row >> 5) & 3) << 2);
    // Phase by phase over the thread's chunks, so that the chunks' dependency
    // chains (stage -> block max -> partner shuffle -> scale -> quotient ->
    // conversion) interleave instead of running one after another.
    const float2 deq = source_deq<MOD>(a);
    uint32_t vb[NV][4];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int j = t + k * tpr;
      const bool valid = FULL || j < nch;
      BcastCols<MOD, 8> bc;
      uint32_t sc[4] = {0u, 0u, 0u, 0u}, sh[4] = {0u, 0u, 0u, 0u};
      if constexpr (mod_is_bcast(MOD)) {
        if (valid)
          bc.load(a, (int64_t)j * 8);
        else
          bc.clear();
      } else if constexpr (MOD == MOD_SEG) {
        if (valid && have_src) {
          unpack4(ld_reuse_v4(sc_src + (int64_t)j * 8), sc);
          unpack4(ld_reuse_v4(sh_src + (int64_t)j * 8), sh);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 d = add2(dk[k][i], nm1);
        float2 y;
        if constexpr (mod_is_bcast(MOD))
          y = fma2(d, fma2(bc.scale(i, deq), rstd2, rstd2), bc.shift(i, deq));
        else if constexpr (MOD == MOD_SEG)
          y = fma2(d, fma2(bf16x2_to_f2(sc[i]), rstd2, rstd2), bf16x2_to_f2(sh[i]));
        else
          y = mul2(d, rstd2);
        vb[k][i] = valid ? f2_to_bf16x2(y) : 0u;
      }
    }
    float amax[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const uint32_t m = bf16x2_absmax(bf16x2_absmax(vb[k][0], vb[k][1]), bf16x2_absmax(vb[k][2], vb[k][3]));
      amax[k] = fmaxf(fabsf(bf16_lo(m)), fabsf(bf16_hi(m)));
    }
    if constexpr (KIND == KIND_AMAX) {
      // first pass of the two-level contract: the tensor's largest |v|.  One
      // value per warp, and the atomic only when it beats the word's current
      // value (read through L2): same-address atomics serialise in L2, and
      // after the first rows almost none are needed.  No barrier here: rows
      // past the end of the tensor have already returned.
      float m = amax[0];
#pragma unroll
      for (int k = 1; k < NV; ++k) m = fmaxf(m, amax[k]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
      if (lane == 0 && m > __uint_as_float(__ldcg(a.amax_ws))) atomicMax(a.amax_ws, __float_as_uint(m));
      return;
    }
#pragma unroll
    for (int k = 0; k < NV; ++k) amax[k] = fmaxf(amax[k], __shfl_xor_sync(0xFFFFFFFFu, amax[k], 1));
    // two-level: the tensor scale from the first pass's maximum (read through
    // L2: it was written by atomics of the previous launch)
    float ts = 1.0f, rts = 1.0f;
    if constexpr (KIND == KIND_NV2L) {
      ts = round_bf16(__fdiv_rn(__uint_as_float(__ldcg(a.amax_ws)), 2688.0f));
      rts = __frcp_rn(ts);
      if (blockIdx.x == 0 && t == 0 && ry == 0) a.tensor_scale[0] = ts;
    }
    uint32_t sbyte[NV], codes[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      float scl;
      if constexpr (KIND == KIND_NV2L) {
        // (amax_b / 6) / ts, both quotients correctly rounded (two_level_quot),
        // clamped at 448 (fminf takes
        // 448 for the 0/0 of an all-zero tensor); the divisor of the codes is
        // s * ts, exact in fp32 (4 + 8 significant bits)
        sbyte[k] = f2_to_e4m3x2(make_float2(fminf(two_level_quot(amax[k], ts, rts), 448.0f), 0.f)) & 0xFFu;
        scl = e4m3_to_f32(sbyte[k]) * ts;
      } else {
        // e4m3(amax/6) via the fp32 constant 1/6 gives the byte of the exact
        // quotient: amax has 8 significant bits, so amax/6 is either exact or
        // far from every e4m3 rounding boundary (checked on the CPU for every
        // bf16 amax).
        sbyte[k] = f2_to_e4m3x2(make_float2(amax[k] * (1.0f / 6.0f), 0.f)) & 0xFFu;
        scl = e4m3_to_f32(sbyte[k]);
      }
      // v/s as v * (r_hi + r_lo): r_hi ~ 1/s, r_lo = r_hi * (1 - s * r_hi), so
      // r_hi + r_lo = 1/s to ~2^-44 relative; q = fma(v, r_hi, v * r_lo) is then
      // the exact quotient rounded once, which equals every representable
      // midpoint of the e2m1 grid exactly and is otherwise far closer to v/s
      // than v/s is to any midpoint.  s = 0 gives r = 0 and q = +-0.
      // Two-level: a divisor below 2^-64 (a tensor scale near the bottom of
      // the fp32 range) and the block's values are both scaled by 2^64 --
      // exact -- so that the reciprocal is not flushed.
      float pre = 1.0f;
      if constexpr (KIND == KIND_NV2L) {
        if (scl != 0.f && scl < 0x1p-64f) {
          scl *= 0x1p64f;
          pre = 0x1p64f;
        }
      }
      const float rh = (scl == 0.f) ? 0.f : rcp_approx(scl);
      const float rl = rh * fmaf(-scl, rh, 1.0f);
      const float2 rh2 = splat2(rh), rl2 = splat2(rl);
      float2 q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 v = KIND == KIND_NV2L ? mul2(bf16x2_to_f2(vb[k][i]), splat2(pre)) : bf16x2_to_f2(vb[k][i]);
        q[i] = fma2(v, rh2, mul2(v, rl2));
      }
      codes[k] = f8_to_e2m1x8(q[0], q[1], q[2], q[3]);
    }
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int j = t + k * tpr;
      if (FULL || j < nch) {
        st_stream_b32(prow + (int64_t)j * 4, codes[k]);
        if ((j & 1) == 0) {
          const int c = j >> 1;
          st_b8(sfrow + (c >> 2) * 512 + (c & 3), sbyte[k]);
        }
      }
    }
    for (int c = nblk + t; c < padc; c += tpr) st_b8(sfrow + (c >> 2) * 512 + (c & 3), 0u);
  }
}

template <int KIND, int MOD>
cudaError_t launch_nv(const LnArgs& a, RowShape s, cudaStream_t st) {
  constexpr bool kPerToken = (MOD == MOD_PTOK || MOD == MOD_TABLE);
  const int64_t work_rows = (KIND == KIND_NVFP4 || KIND == KIND_NV2L) ? (a.rows + 127) / 128 * 128 : a.rows;
  const dim3 block(s.tpr, s.rpc);
  const dim3 grid((unsigned)((work_rows + s.rpc - 1) / s.rpc));
  const float inv_d = (float)(1.0 / (double)a.dim);
#define NVFP4AP_CASE(N)                                                            \
  case N:                                                                          \
    return launch_maybe_pdl(ln_rows_kernel<KIND, MOD, N>, grid, block, 0, st, a, inv_d);
  if constexpr (kPerToken) {
    switch (s.per_thread) {
      NVFP4AP_CASE(1)
      NVFP4AP_CASE(2)
      NVFP4AP_CASE(3)
      NVFP4AP_CASE(4)
      NVFP4AP_CASE(6)
      default: return cudaErrorInvalidValue;
    }
  } else {
    switch (s.per_thread) {
      NVFP4AP_CASE(1)
      NVFP4AP_CASE(2)
      NVFP4AP_CASE(3)
      NVFP4AP_CASE(4)
      NVFP4AP_CASE(6)
      NVFP4AP_CASE(8)
      NVFP4AP_CASE(12)
      default: return cudaErrorInvalidValue;
    }
  }
#undef NVFP4AP_CASE
  return cudaGetLastError();
}

}  // namespace
}  // namespace nvfp4ap
