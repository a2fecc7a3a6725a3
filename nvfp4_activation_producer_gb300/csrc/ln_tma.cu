// ln_tma.cu -- persistent TMA-pipelined adaptive-LayerNorm producers (FP8 and
// NVFP4) for sm_103a.
//
// Same operations and numerics as ln_rows.cu (adaptive-layernorm-producers
// README, "Available Functions", "Tensor Contract", "Validation"; NVFP4
// encoding facts from the h3-blackwell-runtime compare page), organised so
// that HBM always has several rows per SM in flight:
//
//  * persistent CTAs of `tpr` threads, as many per SM as fit; CTA b owns rows
//    b, b + G, b + 2G, ... (G = grid size) and processes one row at a time
//    with all of its threads (thread t owns the 8-element chunks t, t+tpr, ..);
//  * a ring of S shared-memory stages per CTA; thread 0 fills a stage with one
//    row's inputs (x, and the per-token or temb rows) by 1-D bulk copies
//    (cp.async.bulk, the TMA engine) completing that stage's mbarrier, so S
//    rows per CTA are in flight while the CTA computes;
//  * per row: wait for the stage, move the row into registers (x - K in fp32,
//    per-token rows packed), reduce (warp shuffles, one shared-memory step),
//    and right after the reduction barrier -- the stage is no longer read --
//    refill it with the row S*G further on; the output is computed from
//    registers and written with streaming stores;
//  * broadcast scale/shift and the fp32 table rows are the same for every row
//    of a CTA: they are converted once into fp32 registers;
//  * every mbarrier wait is bounded by the `wait_limit` argument (SM clock
//    cycles; the library passes about one second); a CTA whose wait runs out
//    (decided CTA-wide at the reduction barrier) waits, with the library's
//    normal bound, for every copy it has in flight -- the one whose wait ran
//    out included -- then sets the fault word and returns, so no copy is
//    left writing into the shared memory of a CTA that has exited.
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "device.cuh"
#include "kernels.h"
#include "tma.cuh"

namespace nvfp4ap {

// Set (bit 0) by a TMA producer whose bounded wait ran out; read and cleared
// by nvfp4ap_take_device_fault().
__device__ unsigned int g_tma_fault = 0u;

namespace {

enum { KIND_FP8 = 0, KIND_NVFP4 = 1 };

__device__ __forceinline__ void unpack4(uint4 v, uint32_t (&w)[4]) {
  w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
}

// FULL: the row is exactly NV * tpr chunks (no chunk-validity checks).
template <int KIND, int MOD, int NV, bool FULL = false>
__global__ void __launch_bounds__(256)
    ln_tma_kernel(const LnArgs a, const float inv_d, const int S, const long long wait_limit) {
  constexpr bool kPerToken = (MOD == MOD_PTOK || MOD == MOD_TABLE);
  constexpr bool kConst = (MOD == MOD_BCAST || MOD == MOD_TABLE);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float2 red[2][8];  // [row parity][warp]
  __shared__ int red_bad[2][8];

  const int tpr = blockDim.x;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nwarps = tpr >> 5;
  const int64_t D = a.dim;
  const int nch = (int)(D >> 3);
  const uint32_t xbytes = (uint32_t)(D * 2);
  const uint32_t stage_bytes = kPerToken ? 3 * xbytes : xbytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* stages = smem + ((S * 8 + 127) & ~127);

  if (t < S) mbar_init(&bars[t], 1);
  mbar_init_fence();
  __syncthreads();
  pdl_enter();

  // ---- per-CTA constants in registers ----------------------------------------
  const float inv_act = KIND == KIND_FP8 ? 1.0f / __ldg(a.act_scale) : 1.0f;
  float2 G[kConst ? NV : 1][4], H[kConst ? NV : 1][4];
  if constexpr (MOD == MOD_BCAST) {
    // g = 1 + scale, h = shift (FP8: both times 1/act_scale)
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int j = t + k * tpr;
      uint32_t sc[4] = {0u, 0u, 0u, 0u}, sh[4] = {0u, 0u, 0u, 0u};
      if (FULL || j < nch) {
        unpack4(ld_reuse_v4(a.scale + (int64_t)j * 8), sc);
        unpack4(ld_reuse_v4(a.shift + (int64_t)j * 8), sh);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        G[k][i] = mul2(add2(bf16x2_to_f2(sc[i]), splat2(1.0f)), splat2(inv_act));
        H[k][i] = mul2(bf16x2_to_f2(sh[i]), splat2(inv_act));
      }
    }
  } else if constexpr (MOD == MOD_TABLE) {
    // the two fp32 table rows, added to the temb chunks of every row
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int j = t + k * tpr;
      float4 t0 = make_float4(0.f, 0.f, 0.f, 0.f), t1 = t0, u0 = t0, u1 = t0;
      if (FULL || j < nch) {
        const float* ts = a.table + a.scale_idx * D + (int64_t)j * 8;
        const float* th = a.table + a.shift_idx * D + (int64_t)j * 8;
        t0 = ld_reuse_f4(ts); t1 = ld_reuse_f4(ts + 4); u0 = ld_reuse_f4(th); u1 = ld_reuse_f4(th + 4);
      }
      G[k][0] = make_float2(t0.x, t0.y); G[k][1] = make_float2(t0.z, t0.w);
      G[k][2] = make_float2(t1.x, t1.y); G[k][3] = make_float2(t1.z, t1.w);
      H[k][0] = make_float2(u0.x, u0.y); H[k][1] = make_float2(u0.z, u0.w);
      H[k][2] = make_float2(u1.x, u1.y); H[k][3] = make_float2(u1.z, u1.w);
    }
  }

  // ---- ring of S stages, filled by thread 0 ------------------------------------
  const int64_t Gr = gridDim.x;
  uint32_t pending = 0u;  // thread 0: stages with a copy in flight
  uint32_t phase = 0u;    // thread 0: parity of each stage's next completion
  auto issue = [&](int64_t row, int s) {
    uint8_t* dst = stages + (size_t)s * stage_bytes;
    mbar_expect_tx(&bars[s], stage_bytes);
    bulk_g2s(dst, a.x + row * D, xbytes, &bars[s]);
    if constexpr (MOD == MOD_PTOK) {
      bulk_g2s(dst + xbytes, a.scale + row * D, xbytes, &bars[s]);
      bulk_g2s(dst + 2 * xbytes, a.shift + row * D, xbytes, &bars[s]);
    } else if constexpr (MOD == MOD_TABLE) {
      const uint16_t* te = a.temb + row * a.chunks * D;
      bulk_g2s(dst + xbytes, te + a.scale_idx * D, xbytes, &bars[s]);
      bulk_g2s(dst + 2 * xbytes, te + a.shift_idx * D, xbytes, &bars[s]);
    }
    pending |= 1u << s;
  };
  if (t == 0)
    for (int s = 0; s < S; ++s) {
      const int64_t r = blockIdx.x + (int64_t)s * Gr;
      if (r < a.rows) issue(r, s);
    }

  const int nblk = nch >> 1, padc = (nblk + 3) & ~3, ct = padc >> 2;
  int s = 0, par = 0;
  uint32_t parity = 0u;
  for (int64_t row = blockIdx.x; row < a.rows; row += Gr) {
    const bool ok = mbar_wait_bounded(&bars[s], parity, wait_limit);
    const uint8_t* st = stages + (size_t)s * stage_bytes;
    const uint4* xs = reinterpret_cast<const uint4*>(st);
    const float K = __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(st)) << 16);

    // row into registers: dk = x - K (fp32), per-token rows packed
    float2 dk[NV][4];
    uint32_t sw[kPerToken ? NV : 1][4], hw[kPerToken ? NV : 1][4];
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int j = t + k * tpr;
      const bool valid = FULL || j < nch;
      uint32_t xw[4] = {0u, 0u, 0u, 0u};
      if (valid) unpack4(xs[j], xw);
      if constexpr (kPerToken) {
        if (valid) {
          unpack4(reinterpret_cast<const uint4*>(st + xbytes)[j], sw[k]);
          unpack4(reinterpret_cast<const uint4*>(st + 2 * xbytes)[j], hw[k]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) sw[k][i] = hw[k][i] = 0u;
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        dk[k][i] = add2(bf16x2_to_f2(xw[i]), splat2(-K));
        if (valid) {
          s1 = add2(s1, dk[k][i]);
          s2 = fma2(dk[k][i], dk[k][i], s2);
        }
      }
    }
    float2 sum = make_float2(s1.x + s1.y, s2.x + s2.y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sum.x += __shfl_xor_sync(0xFFFFFFFFu, sum.x, o);
      sum.y += __shfl_xor_sync(0xFFFFFFFFu, sum.y, o);
    }
    const bool warp_ok = __all_sync(0xFFFFFFFFu, ok);
    if (lane == 0) {
      red[par][warp] = sum;
      red_bad[par][warp] = warp_ok ? 0 : 1;
    }
    __syncthreads();
    int bad = 0;
    sum = red[par][0];
    bad = red_bad[par][0];
    for (int w = 1; w < nwarps; ++w) {
      const float2 u = red[par][w];
      sum.x += u.x;
      sum.y += u.y;
      bad |= red_bad[par][w];
    }
    if (bad) {
      // the CTA stops: wait (bounded) for its copies still in flight, then report
      if (t == 0) {
        for (int q = 0; q < S; ++q)
          if (pending & (1u << q)) (void)mbar_wait(&bars[q], (phase >> q) & 1u);
        atomicOr(&g_tma_fault, 1u);
      }
      return;
    }
    // stage s is no longer read: refill it with the row S*G further on
    if (t == 0) {
      pending &= ~(1u << s);
      phase ^= 1u << s;
      const int64_t nr = row + (int64_t)S * Gr;
      if (nr < a.rows) issue(nr, s);
    }
    par ^= 1;
    if (++s == S) { s = 0; parity ^= 1u; }

    const float m1 = sum.x * inv_d;  // mean - K
    const float var = fmaxf(fmaf(sum.y, inv_d, -m1 * m1), 0.f);
    const float rstd = rsqrtf(var + a.eps);
    const float2 nm1 = splat2(-m1), rstd2 = splat2(rstd);

    // y (FP8: already divided by act_scale) of pair i of chunk k
    auto y_of = [&](int k, int i) -> float2 {
      const float2 d = add2(dk[k][i], nm1);
      if constexpr (MOD == MOD_NONE) {
        return mul2(d, KIND == KIND_FP8 ? splat2(rstd * inv_act) : rstd2);
      } else if constexpr (MOD == MOD_BCAST) {
        return fma2(d, mul2(G[k][i], rstd2), H[k][i]);
      } else {
        float2 g = bf16x2_to_f2(sw[k][i]), h = bf16x2_to_f2(hw[k][i]);
        if constexpr (MOD == MOD_TABLE) {
          g = add2(g, G[k][i]);
          h = add2(h, H[k][i]);
        }
        const float2 y = fma2(d, fma2(g, rstd2, rstd2), h);
        return KIND == KIND_FP8 ? mul2(y, splat2(inv_act)) : y;
      }
    };

    if constexpr (KIND == KIND_FP8) {
      uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) + row * D;
#pragma unroll
      for (int k = 0; k < NV; ++k) {
        const int j = t + k * tpr;
        if (!FULL && j >= nch) continue;
        uint32_t q[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) q[i] = f2_to_e4m3x2(y_of(k, i));
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
        for (int i = 0; i < 4; ++i) vb[k][i] = valid ? f2_to_bf16x2(y_of(k, i)) : 0u;
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
        // e4m3(amax/6) via the fp32 constant 1/6 (the byte of the exact
        // quotient, as in ln_rows.cuh) and the head/tail reciprocal quotient
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
  }

  if constexpr (KIND == KIND_NVFP4) {
    // rows past the end inside the last 128-row tile: zero scale bytes
    const int64_t rows_pad = (a.rows + 127) & ~(int64_t)127;
    for (int64_t pr = a.rows + blockIdx.x; pr < rows_pad; pr += Gr) {
      uint8_t* sfrow = reinterpret_cast<uint8_t*>(a.sf) + (pr >> 7) * (int64_t)ct * 512 +
                       (int)((pr & 31) << 4) + (int)(((pr >> 5) & 3) << 2);
      for (int c = t; c < padc; c += tpr) st_b8(sfrow + (c >> 2) * 512 + (c & 3), 0u);
    }
  }
}

using TmaKernel = void (*)(const LnArgs, const float, const int, const long long);

template <int KIND, int MOD>
TmaKernel pick_nv(int nv, bool full) {
  switch (nv) {
    case 1: return ln_tma_kernel<KIND, MOD, 1>;
    case 2: return full ? ln_tma_kernel<KIND, MOD, 2, true> : ln_tma_kernel<KIND, MOD, 2>;
    case 3: return full ? ln_tma_kernel<KIND, MOD, 3, true> : ln_tma_kernel<KIND, MOD, 3>;
    case 4: return full ? ln_tma_kernel<KIND, MOD, 4, true> : ln_tma_kernel<KIND, MOD, 4>;
    default: return nullptr;
  }
}

TmaKernel pick(bool nvfp4, int mod, int nv, bool full = false) {
  if (nvfp4) {
    if (mod == MOD_NONE) return pick_nv<KIND_NVFP4, MOD_NONE>(nv, full);
    if (mod == MOD_BCAST) return pick_nv<KIND_NVFP4, MOD_BCAST>(nv, full);
    return nullptr;
  }
  switch (mod) {
    case MOD_NONE: return pick_nv<KIND_FP8, MOD_NONE>(nv, full);
    case MOD_BCAST: return pick_nv<KIND_FP8, MOD_BCAST>(nv, full);
    case MOD_PTOK: return pick_nv<KIND_FP8, MOD_PTOK>(nv, full);
    case MOD_TABLE: return pick_nv<KIND_FP8, MOD_TABLE>(nv, full);
    default: return nullptr;
  }
}

int64_t tma_smem(int mod, int64_t dim, int stages) {
  const int64_t x = dim * 2;
  const int64_t stage = (mod == MOD_PTOK || mod == MOD_TABLE) ? 3 * x : x;
  return ((int64_t)stages * 8 + 127) / 128 * 128 + (int64_t)stages * stage;
}

// Stages and resident CTAs per SM for (kernel, tpr, dim), cached per key and
// device (queried on the first call, which should come before any stream
// capture).
struct TmaPlan {
  int stages, occ;
};
TmaPlan tma_plan(TmaKernel k, int mod, int64_t dim, int tpr, int forced_stages) {
  struct Entry { TmaKernel k; int64_t dim; int tpr, forced, dev; TmaPlan p; };
  static Entry cache[128];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return {0, 0};
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].k == k && cache[i].dim == dim && cache[i].tpr == tpr && cache[i].forced == forced_stages &&
        cache[i].dev == dev)
      return cache[i].p;
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, k) != cudaSuccess) return {0, 0};
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return {0, 0};
  const int64_t max_dyn = (int64_t)optin - (int64_t)fa.sharedSizeBytes;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)max_dyn) != cudaSuccess)
    return {0, 0};
  // fewest stages that keep >= 96 KB per SM in flight (measured best on
  // GB300: more stages cost resident CTAs), else the most bytes in flight
  TmaPlan best{0, 0};
  int64_t best_bytes = -1;
  const int64_t stage = tma_smem(mod, dim, 1) - 128;
  for (int S = 1; S <= 6; ++S) {
    if (forced_stages > 0 && S != forced_stages) continue;
    const int64_t smem = tma_smem(mod, dim, S);
    if (smem > max_dyn) break;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, tpr, (size_t)smem) != cudaSuccess || occ < 1)
      continue;
    const int64_t bytes = (int64_t)occ * S * stage;
    if (bytes > best_bytes) {
      best_bytes = bytes;
      best = {S, occ};
    }
    if (bytes >= 96 * 1024) break;
  }
  if (n < 128) cache[n++] = Entry{k, dim, tpr, forced_stages, dev, best};
  if (const char* dbg = env_get("NVFP4AP_DEBUG"))
    if (dbg[0] == '1')
      std::fprintf(stderr, "nvfp4ap: tma plan dim=%lld tpr=%d: stages=%d ctas/SM=%d\n", (long long)dim, tpr,
                   best.stages, best.occ);
  return best;
}

}  // namespace

bool ln_tma_supported(bool nvfp4, int mod, RowShape s) {
  return s.tpr <= 256 && s.rpc == 1 && pick(nvfp4, mod, s.per_thread) != nullptr;
}

cudaError_t launch_ln_tma(const LnArgs& a, bool nvfp4, int mod, RowShape s, int sms, int forced_stages,
                          int ctas_per_sm, long long wait_limit, cudaStream_t st) {
  // rows that exactly fill the threads' chunks take the FULL instance
  const bool full = (int64_t)s.tpr * s.per_thread * 8 == a.dim;
  TmaKernel k = pick(nvfp4, mod, s.per_thread, full);
  if (!k || s.tpr > 256 || s.rpc != 1) return cudaErrorInvalidValue;
  const TmaPlan p = tma_plan(k, mod, a.dim, s.tpr, forced_stages);
  if (p.stages < 1 || p.occ < 1) return cudaErrorInvalidConfiguration;
  int occ = p.occ;
  if (ctas_per_sm > 0 && ctas_per_sm < occ) occ = ctas_per_sm;
  int64_t grid = (int64_t)sms * occ;
  if (grid > a.rows) grid = a.rows;
  const float inv_d = (float)(1.0 / (double)a.dim);
  return launch_maybe_pdl(k, dim3((unsigned)grid), dim3(s.tpr), (size_t)tma_smem(mod, a.dim, p.stages), st, a,
                          inv_d, p.stages, wait_limit);
}

cudaError_t take_tma_fault(unsigned int* fault) {
  unsigned int zero = 0u;
  cudaError_t e = cudaMemcpyFromSymbol(fault, g_tma_fault, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_tma_fault, &zero, sizeof(unsigned int));
}

}  // namespace nvfp4ap
