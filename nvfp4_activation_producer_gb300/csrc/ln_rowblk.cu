// ln_rowblk.cu -- one-row-per-CTA, block-per-lane LayerNorm producers (NVFP4
// and FP8 e4m3fn) for sm_103a.
//
// Operations (adaptive-layernorm-producers README, "Available Functions",
// "Tensor Contract"; NVFP4 encoding facts from the h3-blackwell-runtime
// compare page):
//   y = (x - mean) * rstd * (1 + scale) + shift, rstd = 1/sqrt(var + eps),
//   scale/shift: none, bf16 broadcast vectors, or e4m3 vectors times fp32 deq
//   scalars (modfp8); AWQ (FP8) also multiplies y by inv_s
//   FP8:   out = e4m3fn(y / act_scale), nearest-even, saturating
//   NVFP4: v = bf16(y); per 16 elements s = e4m3fn(amax/6); e2m1 codes of
//          v/s, two per byte (low nibble first); s in the 128x4 tiled layout
//          with zero padding.
//
// Design.  A CTA is one row of `tpr` threads (a few warps); a lane owns whole
// 16-element blocks t, t + tpr, ... of the row, read with 256-bit loads and
// kept in registers as packed bf16, so the block's maximum, scale byte and 16
// codes are computed once, in one lane.  Statistics in one pass over the
// registers (shifted by the row's first element K), warp shuffles then one
// shared-memory step.  Registers are capped so that many CTAs stay resident
// per SM: short rows of work per CTA and many rows in flight hide the encode's
// dependent steps.  Broadcast modulation is read per block through L1 (the
// vectors are shared by every row).
#include "device.cuh"
#include "kernels.h"
#include "modsrc.cuh"

namespace nvfp4ap {
namespace {

// one 16-element bf16 block: 32 contiguous bytes, read once
__device__ __forceinline__ void rb_load(const uint16_t* p, uint32_t (&w)[8]) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}

template <bool FP8, int MOD, int BPT, int TPR, int MINB>
__global__ void __launch_bounds__(TPR, MINB) ln_rowblk_kernel(const LnArgs a, const float inv_d) {
  __shared__ float2 red[TPR / 32];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t D = a.dim;
  const int nblk = (int)(D >> 4), padc = (nblk + 3) & ~3, ct = padc >> 2;
  const int64_t row = blockIdx.x;
  pdl_enter();

  if (row >= a.rows) {
    if constexpr (FP8) return;
    // rows past the end inside the last 128-row tile: zero scale bytes
    uint8_t* sfrow = reinterpret_cast<uint8_t*>(a.sf) + (row >> 7) * (int64_t)ct * 512 + (int)((row & 31) << 4) +
                     (int)(((row >> 5) & 3) << 2);
    for (int c = t; c < padc; c += TPR) st_b8(sfrow + (c >> 2) * 512 + (c & 3), 0u);
    return;
  }
  const uint16_t* xr = a.x + row * D;
  uint32_t w[BPT][8];
#pragma unroll
  for (int k = 0; k < BPT; ++k) rb_load(xr + (int64_t)(t + k * TPR) * 16, w[k]);
  const float K = __uint_as_float((uint32_t)__ldg(xr) << 16);
  const float2 nk = splat2(-K);
  float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < BPT; ++k)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 d = add2(bf16x2_to_f2(w[k][i]), nk);
      s1 = add2(s1, d);
      s2 = fma2(d, d, s2);
    }
  float2 s = make_float2(s1.x + s1.y, s2.x + s2.y);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    s.x += __shfl_xor_sync(0xFFFFFFFFu, s.x, o);
    s.y += __shfl_xor_sync(0xFFFFFFFFu, s.y, o);
  }
  if (TPR > 32) {
    if (lane == 0) red[warp] = s;
    __syncthreads();
    s = red[0];
#pragma unroll
    for (int v = 1; v < TPR / 32; ++v) {
      s.x += red[v].x;
      s.y += red[v].y;
    }
  }
  const float m1 = s.x * inv_d;  // mean - K
  const float var = fmaxf(fmaf(s.y, inv_d, -m1 * m1), 0.f);
  const float rstd = rsqrtf(var + a.eps);
  // y = (x - K) * A + B (then * G + H): A = rstd, B = -(mean - K) * rstd (FP8
  // without modulation: both times 1/act_scale; with it: (..) * G + H, then
  // times 1/act_scale, and inv_s for AWQ)
  const float inv_act = FP8 ? 1.0f / __ldg(a.act_scale) : 1.0f;
  const float A = (FP8 && MOD == MOD_NONE) ? rstd * inv_act : rstd;
  const float2 A2 = splat2(A), B2 = splat2(-m1 * A), inv2 = splat2(inv_act);
  const float2 deq = source_deq<MOD>(a);
  if constexpr (FP8) {
    uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) + row * D;
#pragma unroll
    for (int k = 0; k < BPT; ++k) {
      const int b = t + k * TPR;
      uint32_t q[8];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        BcastCols<MOD, 8> bc;
        AwqCols<8> aw;
        if constexpr (MOD != MOD_NONE) bc.load(a, (int64_t)b * 16 + h * 8);
        if constexpr (MOD == MOD_AWQ) aw.load(a, (int64_t)b * 16 + h * 8);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float2 y = fma2(add2(bf16x2_to_f2(w[k][h * 4 + i]), nk), A2, B2);
          if constexpr (MOD != MOD_NONE) {
            const float2 f = MOD == MOD_AWQ ? mul2(aw.mult(i), inv2) : inv2;
            y = mul2(fma2(y, add2(bc.scale(i, deq), splat2(1.0f)), bc.shift(i, deq)), f);
          }
          q[h * 4 + i] = f2_to_e4m3x2(y);
        }
      }
      st_stream_v4(orow + (int64_t)b * 16,
                   make_uint4(q[0] | (q[1] << 16), q[2] | (q[3] << 16), q[4] | (q[5] << 16), q[6] | (q[7] << 16)));
    }
    return;
  }
  uint8_t* prow = reinterpret_cast<uint8_t*>(a.out) + row * (D >> 1);
  uint8_t* sfrow = reinterpret_cast<uint8_t*>(a.sf) + (row >> 7) * (int64_t)ct * 512 + (int)((row & 31) << 4) +
                   (int)(((row >> 5) & 3) << 2);
#pragma unroll
  for (int k = 0; k < BPT; ++k) {
    const int b = t + k * TPR;
    uint32_t vb[8];
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // the block's two 8-column halves
      BcastCols<MOD, 8> bc;
      if constexpr (MOD != MOD_NONE) bc.load(a, (int64_t)b * 16 + h * 8);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 y = fma2(add2(bf16x2_to_f2(w[k][h * 4 + i]), nk), A2, B2);
        if constexpr (MOD != MOD_NONE) y = fma2(y, add2(bc.scale(i, deq), splat2(1.0f)), bc.shift(i, deq));
        vb[h * 4 + i] = f2_to_bf16x2(y);
      }
    }
    const uint32_t m = bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(vb[0], vb[1]), bf16x2_absmax(vb[2], vb[3])),
                                     bf16x2_absmax(bf16x2_absmax(vb[4], vb[5]), bf16x2_absmax(vb[6], vb[7])));
    const float amax = fmaxf(fabsf(bf16_lo(m)), fabsf(bf16_hi(m)));
    // amax * (1/6) in fp32 rounds to the same e4m3 byte as the exact quotient
    // (amax has 8 significant bits); codes from v * (r_hi + r_lo), the
    // Newton-corrected reciprocal: exact at every e2m1 midpoint
    const uint32_t sbyte = f2_to_e4m3x2(make_float2(amax * (1.0f / 6.0f), 0.f)) & 0xFFu;
    const float scl = e4m3_to_f32(sbyte);
    const float rh = (scl == 0.f) ? 0.f : rcp_approx(scl);
    const float rl = rh * fmaf(-scl, rh, 1.0f);
    const float2 rh2 = splat2(rh), rl2 = splat2(rl);
    float2 q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float2 v = bf16x2_to_f2(vb[i]);
      q[i] = fma2(v, rh2, mul2(v, rl2));
    }
    st_stream_v2(prow + (int64_t)b * 8, f8_to_e2m1x8(q[0], q[1], q[2], q[3]), f8_to_e2m1x8(q[4], q[5], q[6], q[7]));
    st_b8(sfrow + (b >> 2) * 512 + (b & 3), sbyte);
  }
  for (int c = nblk + t; c < padc; c += TPR) st_b8(sfrow + (c >> 2) * 512 + (c & 3), 0u);
}

template <bool FP8, int MOD, int BPT, int TPR, int MINB>
cudaError_t launch_rb(const LnArgs& a, cudaStream_t st) {
  const int64_t work = FP8 ? a.rows : (a.rows + 127) / 128 * 128;
  const float inv_d = (float)(1.0 / (double)a.dim);
  return launch_maybe_pdl(ln_rowblk_kernel<FP8, MOD, BPT, TPR, MINB>, dim3((unsigned)work), dim3(TPR), 0, st, a,
                          inv_d);
}

// Resident CTAs per SM the registers are capped for (the fewest registers per
// thread each shape compiles to without spills): 56 / 64 / 80 for two, three,
// four blocks per lane; the broadcast source keeps its column words live and
// takes 64 / 80 / 96 (AWQ: also inv_s).  The modfp8 source (e4m3 vectors, half
// the column words) fits two blocks per lane in 56, one CTA more per SM (NVFP4
// 5070x3072: 11.09 -> 10.94 us; a cap changes no arithmetic, so it still
// reduces to the broadcast source bit for bit).
template <int MOD>
constexpr int rb_minb(int bpt, int tpr) {
  const int regs = (MOD == MOD_NONE)                  ? (bpt == 2 ? 56 : bpt == 3 ? 64 : 80)
                   : (MOD == MOD_MODFP8 && bpt == 2) ? 56
                                                     : (bpt == 2 ? 64 : bpt == 3 ? 80 : 96);
  const int b = 65536 / (regs * tpr);
  return b > 32 ? 32 : b;
}

#define NVFP4AP_RB(B, T)                                                      \
  if (s.bpt == B && s.tpr == T) return launch_rb<FP8, MOD, B, T, rb_minb<MOD>(B, T)>(a, st);

template <bool FP8, int MOD>
cudaError_t launch_rb_shape(const LnArgs& a, RbShape s, cudaStream_t st) {
  NVFP4AP_RB(2, 32) NVFP4AP_RB(2, 64) NVFP4AP_RB(2, 96) NVFP4AP_RB(2, 128)
  NVFP4AP_RB(3, 32) NVFP4AP_RB(3, 64) NVFP4AP_RB(3, 96) NVFP4AP_RB(3, 128)
  NVFP4AP_RB(4, 32) NVFP4AP_RB(4, 64) NVFP4AP_RB(4, 96) NVFP4AP_RB(4, 128)
  return cudaErrorInvalidValue;
}
#undef NVFP4AP_RB

}  // namespace

bool pick_rowblk(int64_t dim, int forced_bpt, RbShape* s, bool two_first) {
  if (dim % 16 != 0) return false;
  const int64_t nblk = dim / 16;
  // three blocks per lane first; two first for the forms measured faster so
  // (dim 3072, 5070 rows: NVFP4 broadcast 11.58 -> 10.94 us, which the modfp8
  // source follows at 10.94 -> 11.07 us; 4096 rows: FP8 layer norm 7.68 ->
  // 7.41 us; the NVFP4 layer norm 8.32 -> 8.45 us the other way)
  static const int kPref3[] = {3, 2, 4}, kPref2[] = {2, 3, 4};
  for (int bpt : two_first ? kPref2 : kPref3) {
    if (forced_bpt > 0 && bpt != forced_bpt) continue;
    if (nblk % bpt != 0) continue;
    const int64_t tpr = nblk / bpt;
    // two to four warps per row: a one-warp row measured slower than the
    // register row kernels on GB300 (dim 1536)
    if (tpr % 32 != 0 || tpr < 64 || tpr > 128) continue;
    s->bpt = bpt;
    s->tpr = (int)tpr;
    return true;
  }
  return false;
}

cudaError_t launch_ln_rowblk(const LnArgs& a, bool nvfp4, int mod, RbShape s, cudaStream_t st) {
  if (nvfp4) {
    switch (mod) {
      case MOD_NONE: return launch_rb_shape<false, MOD_NONE>(a, s, st);
      case MOD_BCAST: return launch_rb_shape<false, MOD_BCAST>(a, s, st);
      case MOD_MODFP8: return launch_rb_shape<false, MOD_MODFP8>(a, s, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (mod) {
    case MOD_NONE: return launch_rb_shape<true, MOD_NONE>(a, s, st);
    case MOD_BCAST: return launch_rb_shape<true, MOD_BCAST>(a, s, st);
    case MOD_MODFP8: return launch_rb_shape<true, MOD_MODFP8>(a, s, st);
    case MOD_AWQ: return launch_rb_shape<true, MOD_AWQ>(a, s, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nvfp4ap
