// ln_blk.cuh -- block-per-lane LayerNorm producer kernel template (FP8
// e4m3fn, NVFP4 single-level, and the two passes of the two-level NVFP4
// contract) and its launch helper, shared by the translation units that
// instantiate it (ln_blk.cu, ln_blk2l.cu).
//
// Operations (adaptive-layernorm-producers README, "Available Functions",
// "Tensor Contract"; NVFP4 encoding facts, the two-level contract and the
// segmented modulation from the h3-blackwell-runtime compare page):
//   y = (x - mean) * rstd * (1 + scale) + shift, rstd = 1/sqrt(var + eps),
//   scale/shift from a broadcast source of kernels.h (none, bf16, e4m3 times
//   deq scalars; AWQ also multiplies y by inv_s) or the row's segment of
//   (nseg, dim) bf16 tables
//   FP8:   out = e4m3fn(y / act_scale), nearest-even, saturating
//   NVFP4: v = bf16(y); per 16 elements s = e4m3fn(amax/6); e2m1 codes of
//          v/s, two per byte (low nibble first); s in the 128x4 tiled layout
//          with zero padding.
//   Two-level NVFP4, two launches:
//     BK_AMAX: the largest |v| of the whole tensor into one device word;
//     BK_NV2L: ts = bf16(amax / 2688) from that word; per 16 elements
//              s = e4m3fn(min((amax_b / 6) / ts, 448)) with both
//              quotients correctly rounded in fp32; e2m1 codes of v / (s * ts).
//
// Design.  A lane owns whole 16-element blocks of a row: blocks t, t + tpr,
// ... (tpr = threads per row, a warp or a few), each read with one 256-bit
// load, so a warp reads 1 KB of contiguous row per instruction and the NVFP4
// block maximum, scale and codes of a block are computed once, in one lane,
// with no shuffle.  A CTA is a persistent group of rows: every row group of
// the CTA walks rows blockIdx.x + gridDim.x * (g + ngrp * k) (rows interleaved
// over the CTAs, so every SM gets the same number of rows to one row), the
// next row's blocks loaded into a second register buffer while the current
// row is reduced and written.  The warps of a row combine their sums through
// shared memory behind a named barrier of the row's threads (parity-indexed
// slots: one barrier per row).  The maximum pass keeps a running maximum in
// each thread and issues one atomic per CTA when its rows are done.
//
// The modulation is converted once per CTA to fp32 -- G = 1 + scale and
// H = shift (FP8: both times 1/act_scale, AWQ also times inv_s) -- and kept
// in shared memory in block-chunk-major order (float4 chunk q of block b at
// q * nblk + b; a segmented source keeps one such table per segment plus an
// identity table for rows whose index is out of range), so the 32 lanes of a
// warp read 32 consecutive float4s without bank conflicts; per element the
// modulation then costs one packed FMA and a quarter of a shared-memory load.
//
// Statistics in one pass over the registers, shifted by the row's first
// element K: s1 = sum(x - K), s2 = sum((x - K)^2); mean = K + s1/D,
// var = s2/D - (s1/D)^2.  The normalised value is recomputed from the staged
// bf16 pair as (x - K) * rstd - (s1/D) * rstd (no fp32 copy of the row is
// kept, which leaves registers for the prefetch buffer); x - K is 0 for a
// constant row, so such a row normalises to exactly 0.
#pragma once

#include <cstdlib>
#include <mutex>

#include "device.cuh"
#include "kernels.h"
#include "modsrc.cuh"

namespace nvfp4ap {
namespace {

enum { BK_FP8 = 0, BK_NVFP4 = 1, BK_AMAX = 2, BK_NV2L = 3 };

constexpr int kBlkThreads = 512;  // threads per CTA (row groups x threads per row)
constexpr int kWarpRowThreads = 1024;  // warp-per-row kernels: 32 warps per CTA
// dynamic shared memory the modulation tables may take (the static slots and
// the 227 KB per-CTA limit leave room above it)
constexpr int kBlkMaxSmem = 200 * 1024;

// Set when a row's segment index is outside [0, nseg): that row is produced
// with zero modulation.  One word per translation unit.
__device__ unsigned int g_blk_seg_fault = 0u;

// one 16-element bf16 block: 32 contiguous bytes, read once
__device__ __forceinline__ void ld_block(const uint16_t* p, uint32_t (&w)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}

__device__ __forceinline__ void bar_rows(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ float blk_round_bf16(float v) { return bf16_lo(f2_to_bf16x2(make_float2(v, 0.f))); }

template <int BPT, bool FULL>
__device__ __forceinline__ void load_row(uint32_t (&w)[BPT][8], const uint16_t* xr, int t, int tpr, int nblk) {
#pragma unroll
  for (int k = 0; k < BPT; ++k) {
    const int b = t + k * tpr;
    if (FULL || b < nblk) {
      ld_block(xr + (int64_t)b * 16, w[k]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[k][i] = 0u;
    }
  }
}

// largest |v| of a block of 16 staged bf16 values (8 packed pairs)
__device__ __forceinline__ float block_amax(const uint32_t (&vb)[8]) {
  const uint32_t m = bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(vb[0], vb[1]), bf16x2_absmax(vb[2], vb[3])),
                                   bf16x2_absmax(bf16x2_absmax(vb[4], vb[5]), bf16x2_absmax(vb[6], vb[7])));
  return fmaxf(fabsf(bf16_lo(m)), fabsf(bf16_hi(m)));
}

// fp32 G/H of the 8 columns [8 c8, 8 c8 + 8) into the chunk-major table `tab`
// (FP8: times 1/act_scale, AWQ also times inv_s)
template <int KIND, int MOD>
__device__ __forceinline__ void put_cols(float4* tab, int nblk, int c8, const float2 (&sc)[4], const float2 (&sh)[4],
                                         const float2 (&f)[4]) {
  float2 gv[4], hv[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    gv[i] = add2(sc[i], splat2(1.0f));
    hv[i] = sh[i];
    if constexpr (KIND == BK_FP8) {
      gv[i] = mul2(gv[i], f[i]);
      hv[i] = mul2(hv[i], f[i]);
    }
  }
  const int b = c8 >> 1, q0 = (c8 & 1) * 2;
  tab[q0 * nblk + b] = make_float4(gv[0].x, gv[0].y, gv[1].x, gv[1].y);
  tab[(q0 + 1) * nblk + b] = make_float4(gv[2].x, gv[2].y, gv[3].x, gv[3].y);
  tab[(4 + q0) * nblk + b] = make_float4(hv[0].x, hv[0].y, hv[1].x, hv[1].y);
  tab[(5 + q0) * nblk + b] = make_float4(hv[2].x, hv[2].y, hv[3].x, hv[3].y);
}

// shared-memory tables a modulated instance needs (float4 count)
__host__ __device__ constexpr int64_t blk_tab_float4s(int mod, int64_t nblk, int64_t nseg) {
  return mod == MOD_NONE ? 0 : (mod == MOD_SEG ? (nseg + 1) * 8 * nblk : 8 * nblk);
}

// The CTA's modulation tables in shared memory (G = 1 + scale and H = shift as
// fp32, FP8: both times 1/act_scale, AWQ also times inv_s; chunk-major; a
// segmented source: one table per segment, then the identity table).  Ends
// with a barrier when there are tables.
template <int KIND, int MOD>
__device__ __forceinline__ void blk_tables(const LnArgs& a, float4* gh, int nblk, float inv_act) {
  const int64_t D = a.dim;
  if constexpr (MOD == MOD_SEG) {
    // one table per segment, then the identity table (G = 1, H = 0; FP8: 1/act_scale, 0)
    const int nseg = (int)a.nseg;
    const float2 f[4] = {splat2(inv_act), splat2(inv_act), splat2(inv_act), splat2(inv_act)};
    for (int i = threadIdx.x; i < (nseg + 1) * 2 * nblk; i += blockDim.x) {
      const int sg = i / (2 * nblk), c8 = i - sg * 2 * nblk;
      float2 sc[4], sh[4];
      if (sg < nseg) {
        const uint4 u = ld_reuse_v4(a.seg_scale + (int64_t)sg * D + (int64_t)c8 * 8);
        const uint4 v = ld_reuse_v4(a.seg_shift + (int64_t)sg * D + (int64_t)c8 * 8);
        sc[0] = bf16x2_to_f2(u.x); sc[1] = bf16x2_to_f2(u.y); sc[2] = bf16x2_to_f2(u.z); sc[3] = bf16x2_to_f2(u.w);
        sh[0] = bf16x2_to_f2(v.x); sh[1] = bf16x2_to_f2(v.y); sh[2] = bf16x2_to_f2(v.z); sh[3] = bf16x2_to_f2(v.w);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) sc[j] = sh[j] = make_float2(0.f, 0.f);
      }
      put_cols<KIND, MOD>(gh + (int64_t)sg * 8 * nblk, nblk, c8, sc, sh, f);
    }
    __syncthreads();
  } else if constexpr (MOD != MOD_NONE) {
    const float2 deq = source_deq<MOD>(a);
    for (int c8 = threadIdx.x; c8 < 2 * nblk; c8 += blockDim.x) {
      BcastCols<MOD, 8> bc;
      AwqCols<8> aw;
      bc.load(a, (int64_t)c8 * 8);
      if constexpr (MOD == MOD_AWQ) aw.load(a, (int64_t)c8 * 8);
      float2 sc[4], sh[4], f[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sc[i] = bc.scale(i, deq);
        sh[i] = bc.shift(i, deq);
        f[i] = MOD == MOD_AWQ ? mul2(aw.mult(i), splat2(inv_act)) : splat2(inv_act);
      }
      put_cols<KIND, MOD>(gh, nblk, c8, sc, sh, f);
    }
    __syncthreads();
  }

}

template <int KIND, int MOD, int BPT, bool FULL>
__global__ void __launch_bounds__(kBlkThreads, 1) ln_blk_kernel(const LnArgs a, const float inv_d, const int tpr) {
  extern __shared__ float4 gh[];    // modulation tables, chunk-major (see the file comment)
  __shared__ float2 red[2][16][8];  // [row parity][row group][warp of the row]
  __shared__ float redm[kBlkThreads / 32];
  constexpr bool kNv = (KIND != BK_FP8);
  const int ngrp = blockDim.x / tpr;
  const int g = threadIdx.x / tpr, t = threadIdx.x - g * tpr;
  const int lane = threadIdx.x & 31, wig = t >> 5, wpr = tpr >> 5;
  const int64_t D = a.dim;
  const int nblk = (int)(D >> 4);
  pdl_enter();

  float inv_act = 1.0f;
  if constexpr (KIND == BK_FP8) inv_act = 1.0f / __ldg(a.act_scale);
  blk_tables<KIND, MOD>(a, gh, nblk, inv_act);

  // two-level: the tensor scale from the maximum pass's word (read through L2)
  float ts = 1.0f, rts = 1.0f;
  if constexpr (KIND == BK_NV2L) {
    ts = blk_round_bf16(__fdiv_rn(__uint_as_float(__ldcg(a.amax_ws)), 2688.0f));
    rts = __frcp_rn(ts);
    if (blockIdx.x == 0 && threadIdx.x == 0) a.tensor_scale[0] = ts;
  }
  float run = 0.0f;  // maximum pass: this thread's largest |v|

  const int padc = (nblk + 3) & ~3, ct = padc >> 2;
  const int64_t gstride = (int64_t)gridDim.x * ngrp;
  int64_t row = (int64_t)blockIdx.x + (int64_t)gridDim.x * g;
  uint32_t cur[BPT][8], nxt[BPT][8];
  if (row < a.rows) load_row<BPT, FULL>(cur, a.x + row * D, t, tpr, nblk);
  int par = 0;
  for (; row < a.rows; row += gstride) {
    const int64_t nrow = row + gstride;
    if (nrow < a.rows) load_row<BPT, FULL>(nxt, a.x + nrow * D, t, tpr, nblk);
    const float K = __uint_as_float((uint32_t)__ldg(a.x + row * D) << 16);
    const float4* tab = gh;
    if constexpr (MOD == MOD_SEG) {
      const int sg = __ldg(a.seg_idx + row);
      const bool ok = sg >= 0 && sg < a.nseg;
      if (!ok && t == 0) atomicOr(&g_blk_seg_fault, 1u);
      tab = gh + (int64_t)(ok ? sg : a.nseg) * 8 * nblk;
    }

    // ---- statistics: one pass, shifted by K --------------------------------
    const float2 nk = splat2(-K);
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < BPT; ++k) {
      if (FULL || t + k * tpr < nblk) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 d = add2(bf16x2_to_f2(cur[k][i]), nk);
          s1 = add2(s1, d);
          s2 = fma2(d, d, s2);
        }
      }
    }
    float2 s = make_float2(s1.x + s1.y, s2.x + s2.y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s.x += __shfl_xor_sync(0xFFFFFFFFu, s.x, o);
      s.y += __shfl_xor_sync(0xFFFFFFFFu, s.y, o);
    }
    if (wpr > 1) {
      // row r + 2 writes a slot only after every warp of the row has passed
      // row r + 1's barrier, i.e. finished reading row r's slots
      if (lane == 0) red[par][g][wig] = s;
      bar_rows(1 + g, tpr);
      s = red[par][g][0];
      for (int w = 1; w < wpr; ++w) {
        const float2 u = red[par][g][w];
        s.x += u.x;
        s.y += u.y;
      }
    }
    par ^= 1;
    const float m1 = s.x * inv_d;  // mean - K
    const float var = fmaxf(fmaf(s.y, inv_d, -m1 * m1), 0.f);
    const float rstd = rsqrtf(var + a.eps);
    if constexpr (KIND == BK_AMAX) {
      // the row's statistics for a flat quantising pass (the same fp32 values)
      if (a.row_stats != nullptr && t == 0)
        reinterpret_cast<float4*>(a.row_stats)[row] = make_float4(K, m1, rstd, 0.f);
    }
    // y = (x - K) * A + B (then * G + H): A = rstd, B = -(mean - K) * rstd
    // (FP8 without modulation: both times 1/act_scale)
    const float A = (KIND == BK_FP8 && MOD == MOD_NONE) ? rstd * inv_act : rstd;
    const float2 A2 = splat2(A), B2 = splat2(-m1 * A);

    uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) + row * (kNv ? (D >> 1) : D);
    uint8_t* sfrow = kNv ? reinterpret_cast<uint8_t*>(a.sf) + (row >> 7) * (int64_t)ct * 512 + (int)((row & 31) << 4) +
                               (int)(((row >> 5) & 3) << 2)
                         : nullptr;
#pragma unroll
    for (int k = 0; k < BPT; ++k) {
      const int b = t + k * tpr;
      if (!FULL && b >= nblk) continue;
      float2 y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        y[i] = fma2(add2(bf16x2_to_f2(cur[k][i]), nk), A2, B2);
        if constexpr (MOD != MOD_NONE) {
          const float4 G4 = tab[(i >> 1) * nblk + b], H4 = tab[(4 + (i >> 1)) * nblk + b];
          y[i] = (i & 1) ? fma2(y[i], make_float2(G4.z, G4.w), make_float2(H4.z, H4.w))
                         : fma2(y[i], make_float2(G4.x, G4.y), make_float2(H4.x, H4.y));
        }
      }
      if constexpr (KIND == BK_FP8) {
        uint32_t q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = f2_to_e4m3x2(y[i]);
        st_stream_v4(orow + (int64_t)b * 16,
                     make_uint4(q[0] | (q[1] << 16), q[2] | (q[3] << 16), q[4] | (q[5] << 16), q[6] | (q[7] << 16)));
      } else {
        uint32_t vb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) vb[i] = f2_to_bf16x2(y[i]);
        const float amax = block_amax(vb);
        if constexpr (KIND == BK_AMAX) {
          run = fmaxf(run, amax);
        } else {
          uint32_t sbyte, c0, c1;
          if constexpr (KIND == BK_NV2L) {
            // (amax_b / 6) / ts, both quotients correctly rounded (two_level_quot),
            // clamped at 448 (fminf takes
            // 448 for the 0/0 of an all-zero tensor); the divisor of the codes
            // is s * ts, exact in fp32 (4 + 8 significant bits)
            sbyte = f2_to_e4m3x2(make_float2(fminf(two_level_quot(amax, ts, rts), 448.0f), 0.f)) & 0xFFu;
            block_codes_2l(vb, e4m3_to_f32(sbyte) * ts, c0, c1);
          } else {
            // amax * (1/6) in fp32 rounds to the same e4m3 byte as the exact
            // quotient: amax has 8 significant bits, so amax/6 is exact or
            // lies far from every e4m3 rounding boundary
            sbyte = f2_to_e4m3x2(make_float2(amax * (1.0f / 6.0f), 0.f)) & 0xFFu;
            block_codes(vb, e4m3_to_f32(sbyte), c0, c1);
          }
          st_stream_v2(orow + (int64_t)b * 8, c0, c1);
          st_b8(sfrow + (b >> 2) * 512 + (b & 3), sbyte);
        }
      }
    }
    if constexpr (KIND == BK_NVFP4 || KIND == BK_NV2L)
      for (int c = nblk + t; c < padc; c += tpr) st_b8(sfrow + (c >> 2) * 512 + (c & 3), 0u);
#pragma unroll
    for (int k = 0; k < BPT; ++k)
#pragma unroll
      for (int i = 0; i < 8; ++i) cur[k][i] = nxt[k][i];
  }
  if constexpr (KIND == BK_NVFP4 || KIND == BK_NV2L) {
    // rows past the end inside the last 128-row tile: zero scale bytes
    const int64_t rows_pad = (a.rows + 127) & ~(int64_t)127;
    for (int64_t pr = a.rows + blockIdx.x + (int64_t)gridDim.x * g; pr < rows_pad; pr += gstride) {
      uint8_t* sfrow = reinterpret_cast<uint8_t*>(a.sf) + (pr >> 7) * (int64_t)ct * 512 + (int)((pr & 31) << 4) +
                       (int)(((pr >> 5) & 3) << 2);
      for (int c = t; c < padc; c += tpr) st_b8(sfrow + (c >> 2) * 512 + (c & 3), 0u);
    }
  }
  if constexpr (KIND == BK_AMAX) {
    // the CTA's largest |v| (non-negative fp32: its bits order like the values)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) run = fmaxf(run, __shfl_xor_sync(0xFFFFFFFFu, run, o));
    if (lane == 0) redm[threadIdx.x >> 5] = run;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = redm[0];
      for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, redm[w]);
      if (m > 0.f) atomicMax(a.amax_ws, __float_as_uint(m));
    }
  }
}

// 16 bf16 values (32 contiguous bytes), allocated in L1: the row is read twice
__device__ __forceinline__ void ld_block_l1(const uint16_t* p, uint32_t (&w)[8]) {
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}

// Warp-per-row kernel for many rows per warp (KIND BK_FP8, or BK_AMAX: the
// maximum pass of the two-level contract): each warp takes rows w, w + W, ...
// and sweeps a row twice -- the shifted sums (three 256-bit loads per lane in
// flight, allocated in L1), then the blocks read again (L1 or L2) to write the
// FP8 codes, or to take the staged values' maximum and store the row's
// statistics for the flat quantising pass.  No row stays in registers and
// warps never wait on each other, so 32 warps per SM stream rows
// independently.  The maximum pass issues one atomic per CTA.
template <int KIND, int MOD>
__global__ void __launch_bounds__(kWarpRowThreads, 1) warp_rows_kernel(const LnArgs a, const float inv_d) {
  extern __shared__ float4 gh[];
  __shared__ float redm[kWarpRowThreads / 32];
  const int lane = threadIdx.x & 31;
  const int64_t D = a.dim;
  const int nblk = (int)(D >> 4);
  pdl_enter();
  float inv_act = 1.0f;
  if constexpr (KIND == BK_FP8) inv_act = 1.0f / __ldg(a.act_scale);
  blk_tables<KIND, MOD>(a, gh, nblk, inv_act);

  float run = 0.0f;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < a.rows; row += nw) {
    const uint16_t* xr = a.x + row * D;
    const float K = __uint_as_float((uint32_t)__ldg(xr) << 16);
    const float2 nk = splat2(-K);
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
    for (int b0 = lane; b0 < nblk; b0 += 96) {
      uint32_t w[3][8];
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        if (b0 + 32 * k < nblk) {
          ld_block_l1(xr + (int64_t)(b0 + 32 * k) * 16, w[k]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) w[k][i] = 0u;
        }
      }
#pragma unroll
      for (int k = 0; k < 3; ++k) {
        if (b0 + 32 * k < nblk) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float2 d = add2(bf16x2_to_f2(w[k][i]), nk);
            s1 = add2(s1, d);
            s2 = fma2(d, d, s2);
          }
        }
      }
    }
    float2 s = make_float2(s1.x + s1.y, s2.x + s2.y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      s.x += __shfl_xor_sync(0xFFFFFFFFu, s.x, o);
      s.y += __shfl_xor_sync(0xFFFFFFFFu, s.y, o);
    }
    const float m1 = s.x * inv_d;  // mean - K
    const float var = fmaxf(fmaf(s.y, inv_d, -m1 * m1), 0.f);
    const float rstd = rsqrtf(var + a.eps);
    if (KIND == BK_AMAX && lane == 0) reinterpret_cast<float4*>(a.row_stats)[row] = make_float4(K, m1, rstd, 0.f);
    const float4* tab = gh;
    if constexpr (MOD == MOD_SEG) {
      const int sg = __ldg(a.seg_idx + row);
      const bool ok = sg >= 0 && sg < a.nseg;
      if (!ok && lane == 0) atomicOr(&g_blk_seg_fault, 1u);
      tab = gh + (int64_t)(ok ? sg : a.nseg) * 8 * nblk;
    }
    // the maximum pass: the same fp32 operations as the quantising pass
    const float A = (KIND == BK_FP8 && MOD == MOD_NONE) ? rstd * inv_act : rstd;
    const float2 A2 = splat2(A), B2 = splat2(-m1 * A);
    for (int b = lane; b < nblk; b += 32) {
      uint32_t w[8];
      ld_block_l1(xr + (int64_t)b * 16, w);
      float2 y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        y[i] = fma2(add2(bf16x2_to_f2(w[i]), nk), A2, B2);
        if constexpr (MOD != MOD_NONE) {
          const float4 G4 = tab[(i >> 1) * nblk + b], H4 = tab[(4 + (i >> 1)) * nblk + b];
          y[i] = (i & 1) ? fma2(y[i], make_float2(G4.z, G4.w), make_float2(H4.z, H4.w))
                         : fma2(y[i], make_float2(G4.x, G4.y), make_float2(H4.x, H4.y));
        }
      }
      if constexpr (KIND == BK_FP8) {
        uint32_t q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = f2_to_e4m3x2(y[i]);
        st_stream_v4(reinterpret_cast<uint8_t*>(a.out) + row * D + (int64_t)b * 16,
                     make_uint4(q[0] | (q[1] << 16), q[2] | (q[3] << 16), q[4] | (q[5] << 16), q[6] | (q[7] << 16)));
      } else {
        uint32_t vb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) vb[i] = f2_to_bf16x2(y[i]);
        run = fmaxf(run, block_amax(vb));
      }
    }
  }
  if constexpr (KIND == BK_AMAX) {
    // the CTA's largest |v| (non-negative fp32: its bits order like the values)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) run = fmaxf(run, __shfl_xor_sync(0xFFFFFFFFu, run, o));
    if (lane == 0) redm[threadIdx.x >> 5] = run;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = redm[0];
      for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, redm[w]);
      if (m > 0.f) atomicMax(a.amax_ws, __float_as_uint(m));
    }
  }
}

// Dynamic-memory limit of a kernel raised once per device (keyed by the
// kernel itself: instances share their function-pointer type).
inline bool flat_smem_limit(const void* k) {
  struct Entry { const void* k; int dev; };
  static Entry done[64];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (done[i].k == k && done[i].dev == dev) return true;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kBlkMaxSmem) != cudaSuccess) return false;
  if (n < 64) done[n++] = Entry{k, dev};
  return true;
}

// rows from which the warp-per-row kernels give every warp of the grid
// several (one 1024-thread CTA per SM)
inline int64_t warp_rows_min(int sms) { return (int64_t)sms * (kWarpRowThreads / 32) * 4; }

// ctas_per_sm > 0 caps the resident CTAs per SM (tests: many rows per warp)
template <int KIND, int MOD>
cudaError_t launch_warp_rows(const LnArgs& a, int sms, int ctas_per_sm, cudaStream_t st) {
  auto k = warp_rows_kernel<KIND, MOD>;
  const int64_t smem64 = blk_tab_float4s(MOD, a.dim / 16, a.nseg) * (int64_t)sizeof(float4);
  if (smem64 > kBlkMaxSmem || !flat_smem_limit((const void*)k)) return cudaErrorInvalidValue;
  const int smem = (int)smem64;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kWarpRowThreads, smem) != cudaSuccess || occ < 1)
    return cudaErrorInvalidConfiguration;
  if (ctas_per_sm > 0 && ctas_per_sm < occ) occ = ctas_per_sm;
  int64_t grid = (int64_t)sms * occ;
  const int64_t need = (a.rows + kWarpRowThreads / 32 - 1) / (kWarpRowThreads / 32);
  if (grid > need) grid = need;
  const float inv_d = (float)(1.0 / (double)a.dim);
  return launch_maybe_pdl(k, dim3((unsigned)grid), dim3(kWarpRowThreads), (size_t)smem, st, a, inv_d);
}

// Resident CTAs per SM of an instance with `smem` bytes of dynamic shared
// memory (queried once per key).  The instance's dynamic-memory limit is set
// once, to the largest size the launcher ever passes.
inline int blk_occupancy(const void* k, int smem) {
  struct Entry { const void* k; int smem, dev, occ; };
  static Entry cache[256];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> lock(mu);
  bool seen = false;
  for (int i = 0; i < n; ++i) {
    if (cache[i].k == k && cache[i].smem == smem && cache[i].dev == dev) return cache[i].occ;
    seen = seen || (cache[i].k == k && cache[i].dev == dev);
  }
  if (!seen && cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kBlkMaxSmem) != cudaSuccess)
    return -1;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kBlkThreads, smem) != cudaSuccess) return -1;
  if (n < 256) cache[n++] = Entry{k, smem, dev, occ};
  return occ;
}

template <int KIND, int MOD, int BPT>
cudaError_t launch_blk(const LnArgs& a, BlkShape s, int sms, cudaStream_t st) {
  const int nblk = (int)(a.dim / 16);
  const bool full = s.tpr * BPT == nblk;
  auto k = full ? ln_blk_kernel<KIND, MOD, BPT, true> : ln_blk_kernel<KIND, MOD, BPT, false>;
  const int64_t smem64 = blk_tab_float4s(MOD, nblk, a.nseg) * (int64_t)sizeof(float4);
  if (smem64 > kBlkMaxSmem) return cudaErrorInvalidValue;
  const int smem = (int)smem64;
  int occ = blk_occupancy((const void*)k, smem);
  if (occ < 1) return cudaErrorInvalidConfiguration;
  if (s.ctas_per_sm > 0 && s.ctas_per_sm < occ) occ = s.ctas_per_sm;
  const int ngrp = kBlkThreads / s.tpr;
  const int64_t need = (a.rows + ngrp - 1) / ngrp;
  int64_t grid = (int64_t)sms * occ;
  if (grid > need) grid = need;
  if (grid < 1) grid = 1;
  const float inv_d = (float)(1.0 / (double)a.dim);
  return launch_maybe_pdl(k, dim3((unsigned)grid), dim3(ngrp * s.tpr), (size_t)smem, st, a, inv_d, s.tpr);
}

template <int KIND, int MOD>
cudaError_t launch_blk_bpt(const LnArgs& a, BlkShape s, int sms, cudaStream_t st) {
  if (s.tpr % 32 != 0 || s.tpr > 256 || (int64_t)s.tpr * s.bpt < a.dim / 16) return cudaErrorInvalidValue;
  switch (s.bpt) {
    case 2: return launch_blk<KIND, MOD, 2>(a, s, sms, st);
    case 3: return launch_blk<KIND, MOD, 3>(a, s, sms, st);
    case 4: return launch_blk<KIND, MOD, 4>(a, s, sms, st);
    case 6: return launch_blk<KIND, MOD, 6>(a, s, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

inline cudaError_t take_blk_word(unsigned int* fault) {
  unsigned int zero = 0u;
  cudaError_t e = cudaMemcpyFromSymbol(fault, g_blk_seg_fault, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_blk_seg_fault, &zero, sizeof(unsigned int));
}

}  // namespace
}  // namespace nvfp4ap
