// ln_rows.cu -- adaptive-LayerNorm producers (FP8 e4m3fn and NVFP4) for
// sm_103a, register-resident rows: the instances of the row kernel template
// (ln_rows.cuh) for the single-level producers, and the persistent broadcast
// kernel.
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
#include <cstdlib>
#include <mutex>

#include "ln_rows.cuh"

namespace nvfp4ap {
namespace {

// ---------------------------------------------------------------------------
// Persistent broadcast-modulation kernel (FP8 and NVFP4).
//
// The broadcast scale/shift are the same for every row, so a CTA that walks
// many rows with a fixed thread -> column mapping converts them to fp32 once
// (g = 1 + scale and h = shift from any broadcast source; FP8 pre-multiplied
// by 1/act_scale, AWQ by inv_s) and keeps them in registers; per element the
// output then costs two packed fp32 ops whatever the source.
// The CTA processes rows blockIdx.x, blockIdx.x + gridDim.x, ...; while one
// row is reduced and written, the next row's loads are already in flight in a
// second register buffer.  Statistics and encodings as in ln_rows_kernel.
// ---------------------------------------------------------------------------

template <int NV, bool FULL = false>
__device__ __forceinline__ void load_x(uint32_t (&w)[NV][4], const uint16_t* xr, int t, int tpr, int nch) {
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int j = t + k * tpr;
    if (FULL || j < nch) {
      unpack4(ld_once_v4(xr + (int64_t)j * 8), w[k]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) w[k][i] = 0u;
    }
  }
}

// FULL: the row is exactly NV * tpr chunks (no chunk-validity checks); measured
// 4-6% faster on GB300 at 3072 columns.
template <int KIND, int MOD, int NV, bool FULL = false>
__global__ void __launch_bounds__(256, 2) ln_bcast_persist_kernel(const LnArgs a, const float inv_d) {
  __shared__ float2 red[2][8];  // [row parity][warp]
  const int tpr = blockDim.x;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nwarps = tpr >> 5;
  const int64_t D = a.dim;
  const int nch = (int)(D >> 3);
  pdl_enter();

  // per-thread fp32 modulation of its columns
  const float inv_act = KIND == KIND_FP8 ? 1.0f / __ldg(a.act_scale) : 1.0f;
  const float2 deq = source_deq<MOD>(a);
  float2 G[NV][4], H[NV][4];
#pragma unroll
  for (int k = 0; k < NV; ++k) {
    const int j = t + k * tpr;
    BcastCols<MOD, 8> bc;
    AwqCols<8> aw;
    bc.clear();
    if (FULL || j < nch) {
      bc.load(a, (int64_t)j * 8);
      if constexpr (MOD == MOD_AWQ) aw.load(a, (int64_t)j * 8);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 g = add2(bc.scale(i, deq), splat2(1.0f));
      const float2 h = bc.shift(i, deq);
      if constexpr (KIND == KIND_FP8) {
        // output multiplier 1/act_scale, times inv_s for AWQ
        const float2 f = (MOD == MOD_AWQ && (FULL || j < nch)) ? mul2(aw.mult(i), splat2(inv_act)) : splat2(inv_act);
        G[k][i] = mul2(g, f);
        H[k][i] = mul2(h, f);
      } else {
        G[k][i] = g;
        H[k][i] = h;
      }
    }
  }

  const int nblk = nch >> 1, padc = (nblk + 3) & ~3, ct = padc >> 2;
  uint32_t cur[NV][4], nxt[NV][4];
  int64_t row = blockIdx.x;
  if (row < a.rows) load_x<NV, FULL>(cur, a.x + row * D, t, tpr, nch);
  int par = 0;
  for (; row < a.rows; row += gridDim.x) {
    const int64_t nrow = row + gridDim.x;
    if (nrow < a.rows) load_x<NV, FULL>(nxt, a.x + nrow * D, t, tpr, nch);
    const float K = __uint_as_float((uint32_t)__ldg(a.x + row * D) << 16);

    // statistics (one pass, shifted by K)
    float2 dk[NV][4];
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const bool valid = FULL || t + k * tpr < nch;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        dk[k][i] = add2(bf16x2_to_f2(cur[k][i]), splat2(-K));
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
      // two buffers by row parity: row r+2 writes a buffer only after every
      // thread has passed row r+1's barrier, i.e. finished reading row r's
      if (lane == 0) red[par][warp] = s;
      __syncthreads();
      s = red[par][0];
      for (int w = 1; w < nwarps; ++w) {
        const float2 u = red[par][w];
        s.x += u.x;
        s.y += u.y;
      }
    }
    par ^= 1;
    const float m1 = s.x * inv_d;
    const float var = fmaxf(fmaf(s.y, inv_d, -m1 * m1), 0.f);
    const float2 rstd2 = splat2(rsqrtf(var + a.eps)), nm1 = splat2(-m1);

    if constexpr (KIND == KIND_FP8) {
      uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) + row * D;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int j = t + k * tpr;
        if (!FULL && j >= nch) continue;
        uint32_t q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          q[i] = f2_to_e4m3x2(fma2(add2(dk[k][i], nm1), mul2(G[k][i], rstd2), H[k][i]));
        st_stream_v2(orow + (int64_t)j * 8, q[0] | (q[1] << 16), q[2] | (q[3] << 16));
      }
    } else {
      uint8_t* prow = reinterpret_cast<uint8_t*>(a.out) + row * (D >> 1);
      uint8_t* sfrow = reinterpret_cast<uint8_t*>(a.sf) + (row >> 7) * (int64_t)ct * 512 +
                       (int)((row & 31) << 4) + (int)(((row >> 5) & 3) << 2);
      uint32_t vb[NV][4];
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const bool valid = FULL || t + k * tpr < nch;
#pragma unroll
        for (int i = 0; i < 4; ++i)
          vb[k][i] = valid ? f2_to_bf16x2(fma2(add2(dk[k][i], nm1), mul2(G[k][i], rstd2), H[k][i])) : 0u;
      }
      float amax[NV];
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const uint32_t m = bf16x2_absmax(bf16x2_absmax(vb[k][0], vb[k][1]), bf16x2_absmax(vb[k][2], vb[k][3]));
        amax[k] = fmaxf(fabsf(bf16_lo(m)), fabsf(bf16_hi(m)));
      }
#pragma unroll
      for (int k = 0; k < NV; ++k) amax[k] = fmaxf(amax[k], __shfl_xor_sync(0xFFFFFFFFu, amax[k], 1));
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int j = t + k * tpr;
        const uint32_t sbyte = f2_to_e4m3x2(make_float2(amax[k] * (1.0f / 6.0f), 0.f)) & 0xFFu;
        const float scl = e4m3_to_f32(sbyte);
        const float rh = (scl == 0.f) ? 0.f : rcp_approx(scl);
        const float rl = rh * fmaf(-scl, rh, 1.0f);
        const float2 rh2 = splat2(rh), rl2 = splat2(rl);
        float2 q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 v = bf16x2_to_f2(vb[k][i]);
          q[i] = fma2(v, rh2, mul2(v, rl2));
        }
        const uint32_t codes = f8_to_e2m1x8(q[0], q[1], q[2], q[3]);
        if (FULL || j < nch) {
          st_stream_b32(prow + (int64_t)j * 4, codes);
          if ((j & 1) == 0) st_b8(sfrow + ((j >> 1) >> 2) * 512 + ((j >> 1) & 3), sbyte);
        }
      }
      for (int c = nblk + t; c < padc; c += tpr) st_b8(sfrow + (c >> 2) * 512 + (c & 3), 0u);
    }
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
      for (int i = 0; i < 4; ++i) cur[k][i] = nxt[k][i];
  }
  if constexpr (KIND == KIND_NVFP4) {
    // rows past the end inside the last 128-row tile: zero scale bytes
    const int64_t rows_pad = (a.rows + 127) & ~(int64_t)127;
    for (int64_t pr = a.rows + blockIdx.x; pr < rows_pad; pr += gridDim.x) {
      uint8_t* sfrow = reinterpret_cast<uint8_t*>(a.sf) + (pr >> 7) * (int64_t)ct * 512 +
                       (int)((pr & 31) << 4) + (int)(((pr >> 5) & 3) << 2);
      for (int c = t; c < padc; c += tpr) st_b8(sfrow + (c >> 2) * 512 + (c & 3), 0u);
    }
  }
}

// Resident CTAs per SM of a persistent instance (queried once per key).
template <typename K>
int persist_occupancy(K k, int threads) {
  struct Entry { const void* k; int threads; int dev; int occ; };
  static Entry cache[64];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].k == (const void*)k && cache[i].threads == threads && cache[i].dev == dev) return cache[i].occ;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, threads, 0) != cudaSuccess) return -1;
  if (n < 64) cache[n++] = Entry{(const void*)k, threads, dev, occ};
  return occ;
}

template <int KIND, int MOD>
cudaError_t launch_persist(const LnArgs& a, RowShape s, int sms, int ctas_per_sm, cudaStream_t st) {
  const float inv_d = (float)(1.0 / (double)a.dim);
  const int64_t work_rows = KIND == KIND_NVFP4 ? (a.rows + 127) / 128 * 128 : a.rows;
  // rows that exactly fill the threads' chunks take the FULL instance
  const bool full = (int64_t)s.tpr * s.per_thread * 8 == a.dim;
#define NVFP4AP_CASE(N)                                                                        \
  case N: {                                                                                    \
    auto k = (full && N >= 2 && N <= 4) ? ln_bcast_persist_kernel<KIND, MOD, N, (N >= 2 && N <= 4)> \
                                        : ln_bcast_persist_kernel<KIND, MOD, N, false>;        \
    int occ = persist_occupancy(k, s.tpr);                                                     \
    if (occ < 1) return cudaErrorInvalidConfiguration;                                         \
    if (ctas_per_sm > 0 && ctas_per_sm < occ) occ = ctas_per_sm;                               \
    int64_t grid = (int64_t)sms * occ;                                                         \
    if (grid > work_rows) grid = work_rows;                                                    \
    return launch_maybe_pdl(k, dim3((unsigned)grid), dim3(s.tpr), 0, st, a, inv_d);            \
  }
  switch (s.per_thread) {
    NVFP4AP_CASE(1)
    NVFP4AP_CASE(2)
    NVFP4AP_CASE(3)
    NVFP4AP_CASE(4)
    NVFP4AP_CASE(6)
    default:
      return cudaErrorInvalidValue;
  }
#undef NVFP4AP_CASE
}


}  // namespace

int ln_rows_max_tpr(int mod, int per_thread) {
  const bool per_token = (mod == MOD_PTOK || mod == MOD_TABLE);
  switch (per_thread) {
    case 1: case 2: case 3: case 4: case 6: return rows_max_tpr(per_thread);
    case 8: case 12: return per_token ? 0 : rows_max_tpr(per_thread);
    default: return 0;
  }
}

cudaError_t launch_ln_bcast_persistent(const LnArgs& a, bool nvfp4, int mod, RowShape s, int sms,
                                       int ctas_per_sm, cudaStream_t st) {
  if (s.tpr > 256 || s.rpc != 1) return cudaErrorInvalidValue;
  if (nvfp4) {
    switch (mod) {
      case MOD_BCAST: return launch_persist<KIND_NVFP4, MOD_BCAST>(a, s, sms, ctas_per_sm, st);
      case MOD_MODFP8: return launch_persist<KIND_NVFP4, MOD_MODFP8>(a, s, sms, ctas_per_sm, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (mod) {
    case MOD_BCAST: return launch_persist<KIND_FP8, MOD_BCAST>(a, s, sms, ctas_per_sm, st);
    case MOD_MODFP8: return launch_persist<KIND_FP8, MOD_MODFP8>(a, s, sms, ctas_per_sm, st);
    case MOD_AWQ: return launch_persist<KIND_FP8, MOD_AWQ>(a, s, sms, ctas_per_sm, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_ln_rows_full(const LnArgs& a, bool nvfp4, int mod, RowShape s, cudaStream_t st) {
  if (!nvfp4 || s.tpr > 128 || (int64_t)s.tpr * s.per_thread * 8 != a.dim) return cudaErrorInvalidValue;
  // one row per CTA (the kernel takes threadIdx.y as 0)
  const int64_t rows_pad = (a.rows + 127) / 128 * 128;
  const dim3 block(s.tpr, 1), grid((unsigned)rows_pad);
  const float inv_d = (float)(1.0 / (double)a.dim);
#define NVFP4AP_CASE(M, N)                                                                                        \
  case N:                                                                                                         \
    return launch_maybe_pdl(ln_rows_kernel<KIND_NVFP4, M, N, kFullMinBlocks>, grid, block, 0, st, a, inv_d);
#define NVFP4AP_MOD(M)          \
  case M:                       \
    switch (s.per_thread) {     \
      NVFP4AP_CASE(M, 2)        \
      NVFP4AP_CASE(M, 3)        \
      NVFP4AP_CASE(M, 4)        \
      default: return cudaErrorInvalidValue; \
    }
  switch (mod) {
    NVFP4AP_MOD(MOD_NONE)
    NVFP4AP_MOD(MOD_BCAST)
    NVFP4AP_MOD(MOD_MODFP8)
    default: return cudaErrorInvalidValue;
  }
#undef NVFP4AP_MOD
#undef NVFP4AP_CASE
}

cudaError_t launch_ln_rows(const LnArgs& a, bool nvfp4, int mod, RowShape s, cudaStream_t st) {
  if (nvfp4) {
    switch (mod) {
      case MOD_NONE: return launch_nv<KIND_NVFP4, MOD_NONE>(a, s, st);
      case MOD_BCAST: return launch_nv<KIND_NVFP4, MOD_BCAST>(a, s, st);
      case MOD_MODFP8: return launch_nv<KIND_NVFP4, MOD_MODFP8>(a, s, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (mod) {
    case MOD_NONE: return launch_nv<KIND_FP8, MOD_NONE>(a, s, st);
    case MOD_BCAST: return launch_nv<KIND_FP8, MOD_BCAST>(a, s, st);
    case MOD_PTOK: return launch_nv<KIND_FP8, MOD_PTOK>(a, s, st);
    case MOD_TABLE: return launch_nv<KIND_FP8, MOD_TABLE>(a, s, st);
    case MOD_MODFP8: return launch_nv<KIND_FP8, MOD_MODFP8>(a, s, st);
    case MOD_AWQ: return launch_nv<KIND_FP8, MOD_AWQ>(a, s, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nvfp4ap
