// ln_ring.cu -- TMA-staged adaptive-LayerNorm producers (FP8 and NVFP4) for
// sm_103a.
//
// Same operations and numerics as ln_fp8.cu / ln_nvfp4.cu (adaptive-
// layernorm-producers README, "Available Functions", "Tensor Contract",
// "Validation"; NVFP4 encoding facts from the h3-blackwell-runtime compare
// page), organised so that HBM never waits for arithmetic:
//
//  * persistent CTAs (a multiple of the SM count), W warps each; warp g of
//    the grid owns rows g, g + G, g + 2G, ... (G = warps in the grid);
//  * each warp owns a ring of S shared-memory stages; lane 0 fills a stage
//    with one row's inputs (x, and the per-token or temb rows) by 1-D bulk
//    copies (cp.async.bulk, the TMA engine) that complete an mbarrier, so up
//    to S rows per warp -- W*S per CTA -- are in flight while the warp
//    computes; broadcast scale/shift or the two fp32 table rows are copied
//    into shared memory once per CTA;
//  * a warp reduces its row with shuffles only (no CTA barrier in the loop),
//    reading the staged row from shared memory three times (sum, centred sum
//    of squares, output), and writes the codes straight to global memory;
//  * every mbarrier wait is bounded by the `wait_limit` argument (SM clock
//    cycles; the library passes about one second); on expiry lane 0 waits,
//    with the library's normal bound, for every copy the warp has in flight
//    (the one whose wait ran out included), then sets the library's fault
//    word and the warp stops, so no copy is left writing into the shared
//    memory of a warp -- or a CTA -- that has exited.
#include <mutex>

#include "device.cuh"
#include "nvfp4ap.h"
#include "kernels.h"
#include "tma.cuh"

namespace nvfp4ap {

// Set (bit 0) by any ring kernel whose mbarrier wait ran out; read and cleared
// by the host through nvfp4ap_take_device_fault().
__device__ unsigned int g_ring_fault = 0u;

namespace {

enum { KIND_FP8 = 0, KIND_NVFP4 = 1 };

__device__ __forceinline__ int64_t sf_off(int64_t r, int c, int ct) {
  return ((r >> 7) * ct + (c >> 2)) * 512 + (int)((r & 31) << 4) + (int)(((r >> 5) & 3) << 2) + (c & 3);
}

// Row statistics of a staged row: mean, then 1/sqrt(mean((x-mean)^2) + eps).
__device__ __forceinline__ void row_stats(const uint4* xs, int nch, int lane, float D, float eps, float& mean,
                                          float& rstd) {
  float2 acc = make_float2(0.f, 0.f);
  for (int c = lane; c < nch; c += 32) {
    const uint4 v = xs[c];
    acc = add2(acc, add2(add2(bf16x2_to_f2(v.x), bf16x2_to_f2(v.y)), add2(bf16x2_to_f2(v.z), bf16x2_to_f2(v.w))));
  }
  mean = warp_sum(acc.x + acc.y) / D;
  const float2 nm = splat2(-mean);
  float2 sq = make_float2(0.f, 0.f);
  for (int c = lane; c < nch; c += 32) {
    const uint4 v = xs[c];
    float2 d;
    d = add2(bf16x2_to_f2(v.x), nm); sq = fma2(d, d, sq);
    d = add2(bf16x2_to_f2(v.y), nm); sq = fma2(d, d, sq);
    d = add2(bf16x2_to_f2(v.z), nm); sq = fma2(d, d, sq);
    d = add2(bf16x2_to_f2(v.w), nm); sq = fma2(d, d, sq);
  }
  const float var = warp_sum(sq.x + sq.y) / D;
  rstd = 1.0f / sqrtf(var + eps);
}

// y of one bf16 pair: d * (rstd + rstd * scale) + shift (or d * rstd).
template <int MOD>
__device__ __forceinline__ float2 modulate(uint32_t xw, float2 nm, float2 rstd2, float2 s, float2 h) {
  const float2 d = add2(bf16x2_to_f2(xw), nm);
  if constexpr (MOD == MOD_NONE) return mul2(d, rstd2);
  else return fma2(d, fma2(s, rstd2, rstd2), h);
}

// Scale / shift of the 8 elements of chunk c as four fp32 pairs each.
template <int MOD>
__device__ __forceinline__ void mod_chunk(const uint8_t* stage, const uint8_t* cst, int c, uint32_t xbytes,
                                          float2 (&s)[4], float2 (&h)[4]) {
  if constexpr (MOD == MOD_NONE) {
    return;
  } else {
    uint4 sv, hv;
    if constexpr (MOD == MOD_BCAST) {
      sv = reinterpret_cast<const uint4*>(cst)[c];
      hv = reinterpret_cast<const uint4*>(cst + xbytes)[c];
    } else {
      sv = reinterpret_cast<const uint4*>(stage + xbytes)[c];
      hv = reinterpret_cast<const uint4*>(stage + 2 * xbytes)[c];
    }
    s[0] = bf16x2_to_f2(sv.x); s[1] = bf16x2_to_f2(sv.y); s[2] = bf16x2_to_f2(sv.z); s[3] = bf16x2_to_f2(sv.w);
    h[0] = bf16x2_to_f2(hv.x); h[1] = bf16x2_to_f2(hv.y); h[2] = bf16x2_to_f2(hv.z); h[3] = bf16x2_to_f2(hv.w);
    if constexpr (MOD == MOD_TABLE) {
      // fp32 table rows: [scale row (dim)][shift row (dim)]
      const float4* ts = reinterpret_cast<const float4*>(cst) + 2 * c;
      const float4* th = reinterpret_cast<const float4*>(cst + 2 * xbytes) + 2 * c;
      const float4 t0 = ts[0], t1 = ts[1], u0 = th[0], u1 = th[1];
      s[0] = add2(s[0], make_float2(t0.x, t0.y)); s[1] = add2(s[1], make_float2(t0.z, t0.w));
      s[2] = add2(s[2], make_float2(t1.x, t1.y)); s[3] = add2(s[3], make_float2(t1.z, t1.w));
      h[0] = add2(h[0], make_float2(u0.x, u0.y)); h[1] = add2(h[1], make_float2(u0.z, u0.w));
      h[2] = add2(h[2], make_float2(u1.x, u1.y)); h[3] = add2(h[3], make_float2(u1.z, u1.w));
    }
  }
}

template <int MOD>
__device__ __forceinline__ void fp8_row(const LnArgs& a, int64_t row, const uint8_t* stage, const uint8_t* cst,
                                        int lane, float inv_act) {
  const int64_t D = a.dim;
  const int nch = (int)(D >> 3);
  const uint32_t xbytes = (uint32_t)(D * 2);
  const uint4* xs = reinterpret_cast<const uint4*>(stage);
  float mean, rstd;
  row_stats(xs, nch, lane, (float)D, a.eps, mean, rstd);
  const float2 nm = splat2(-mean), inv2 = splat2(inv_act);
  const float2 rstd2 = splat2(MOD == MOD_NONE ? rstd * inv_act : rstd);
  uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) + row * D;
  for (int c = lane; c < nch; c += 32) {
    const uint4 v = xs[c];
    float2 s[4], h[4];
    mod_chunk<MOD>(stage, cst, c, xbytes, s, h);
    uint32_t q[4];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 y = modulate<MOD>(w[i], nm, rstd2, s[i], h[i]);
      if constexpr (MOD != MOD_NONE) y = mul2(y, inv2);
      q[i] = f2_to_e4m3x2(y);
    }
    st_stream_v2(orow + (int64_t)c * 8, q[0] | (q[1] << 16), q[2] | (q[3] << 16));
  }
}

template <int MOD>
__device__ __forceinline__ void nvfp4_row(const LnArgs& a, int64_t row, const uint8_t* stage, const uint8_t* cst,
                                          int lane) {
  const int64_t D = a.dim;
  const int nch = (int)(D >> 3);  // 8-element chunks; a 16-element block is chunks 2b, 2b+1
  const int nblk = nch >> 1, padc = (nblk + 3) & ~3, ct = padc >> 2;
  const uint32_t xbytes = (uint32_t)(D * 2);
  const uint4* xs = reinterpret_cast<const uint4*>(stage);
  float mean, rstd;
  row_stats(xs, nch, lane, (float)D, a.eps, mean, rstd);
  const float2 nm = splat2(-mean), rstd2 = splat2(rstd);
  uint8_t* prow = reinterpret_cast<uint8_t*>(a.out) + row * (D >> 1);
  uint8_t* sf = reinterpret_cast<uint8_t*>(a.sf);
  // all lanes run the same number of iterations: the block amax pairs lanes
  for (int base = 0; base < nch; base += 32) {
    const int c = base + lane;
    const bool valid = c < nch;
    uint32_t vb[4] = {0u, 0u, 0u, 0u};
    if (valid) {
      const uint4 v = xs[c];
      float2 s[4], h[4];
      mod_chunk<MOD>(stage, cst, c, xbytes, s, h);
      vb[0] = f2_to_bf16x2(modulate<MOD>(v.x, nm, rstd2, s[0], h[0]));
      vb[1] = f2_to_bf16x2(modulate<MOD>(v.y, nm, rstd2, s[1], h[1]));
      vb[2] = f2_to_bf16x2(modulate<MOD>(v.z, nm, rstd2, s[2], h[2]));
      vb[3] = f2_to_bf16x2(modulate<MOD>(v.w, nm, rstd2, s[3], h[3]));
    }
    const uint32_t m = bf16x2_absmax(bf16x2_absmax(vb[0], vb[1]), bf16x2_absmax(vb[2], vb[3]));
    float amax = fmaxf(fabsf(bf16_lo(m)), fabsf(bf16_hi(m)));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));  // the other half of the block
    // e4m3(amax/6) through the fp32 constant 1/6: same byte as the exact quotient
    // (see ln_nvfp4.cu); e2m1 codes through the exact-at-midpoints quotient
    const uint32_t sbyte = f2_to_e4m3x2(make_float2(amax * (1.0f / 6.0f), 0.f)) & 0xFFu;
    const float sc = e4m3_to_f32(sbyte);
    const float r = (sc == 0.f) ? 0.f : rcp_approx(sc);
    const float2 r2 = splat2(r), ns2 = splat2(-sc);
    float2 q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 vv = bf16x2_to_f2(vb[i]);
      const float2 q0 = mul2(vv, r2);
      q[i] = fma2(fma2(q0, ns2, vv), r2, q0);
    }
    const uint32_t codes = f8_to_e2m1x8(q[0], q[1], q[2], q[3]);
    if (valid) {
      st_stream_b32(prow + (int64_t)c * 4, codes);
      if ((c & 1) == 0) st_b8(sf + sf_off(row, c >> 1, ct), sbyte);
    }
  }
  for (int cc = nblk + lane; cc < padc; cc += 32) st_b8(sf + sf_off(row, cc, ct), 0u);
}

// `cta_state` (may be null): one word per CTA; each warp adds the number of
// rows it finished, and bit 31 marks a CTA one of whose waits ran out.
template <int KIND, int MOD>
__global__ void __launch_bounds__(512)
    ln_ring_kernel(const LnArgs a, const int S, unsigned int* cta_state, const long long wait_limit) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int W = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t D = a.dim;
  const uint32_t xbytes = (uint32_t)(D * 2);
  constexpr bool kPerToken = (MOD == MOD_PTOK || MOD == MOD_TABLE);
  const uint32_t stage_bytes = kPerToken ? 3 * xbytes : xbytes;
  const uint32_t const_bytes = MOD == MOD_BCAST ? 2 * xbytes : (MOD == MOD_TABLE ? 4 * xbytes : 0);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* cst = smem + ((W * S * 8 + 127) & ~127);
  uint8_t* stages = cst + const_bytes;

  if (threadIdx.x < W * S) mbar_init(&bars[threadIdx.x], 1);
  mbar_init_fence();
  if constexpr (MOD == MOD_BCAST) {
    uint4* dst = reinterpret_cast<uint4*>(cst);
    const int n = (int)(xbytes >> 4);
    for (int i = threadIdx.x; i < 2 * n; i += blockDim.x)
      dst[i] = ld_reuse_v4(i < n ? (const void*)(a.scale + (int64_t)i * 8) : (const void*)(a.shift + (int64_t)(i - n) * 8));
  } else if constexpr (MOD == MOD_TABLE) {
    float4* dst = reinterpret_cast<float4*>(cst);
    const int n = (int)(D >> 2);
    const float* ts = a.table + a.scale_idx * D;
    const float* th = a.table + a.shift_idx * D;
    for (int i = threadIdx.x; i < 2 * n; i += blockDim.x)
      dst[i] = ld_reuse_f4(i < n ? ts + (int64_t)i * 4 : th + (int64_t)(i - n) * 4);
  }
  __syncthreads();

  const int64_t G = (int64_t)gridDim.x * W;
  const int64_t gw = (int64_t)blockIdx.x * W + w;
  uint8_t* ring = stages + (size_t)w * S * stage_bytes;
  uint64_t* wb = bars + w * S;
  const float inv_act = KIND == KIND_FP8 ? 1.0f / __ldg(a.act_scale) : 0.f;

  uint32_t pending = 0u;  // lane 0: stages with a copy in flight
  uint32_t phase = 0u;    // lane 0: parity of each stage's next completion
  auto issue = [&](int64_t row, int s) {
    uint8_t* dst = ring + (size_t)s * stage_bytes;
    pending |= 1u << s;
    mbar_expect_tx(&wb[s], stage_bytes);
    bulk_g2s(dst, a.x + row * D, xbytes, &wb[s]);
    if constexpr (MOD == MOD_PTOK) {
      bulk_g2s(dst + xbytes, a.scale + row * D, xbytes, &wb[s]);
      bulk_g2s(dst + 2 * xbytes, a.shift + row * D, xbytes, &wb[s]);
    } else if constexpr (MOD == MOD_TABLE) {
      const uint16_t* te = a.temb + row * a.chunks * D;
      bulk_g2s(dst + xbytes, te + a.scale_idx * D, xbytes, &wb[s]);
      bulk_g2s(dst + 2 * xbytes, te + a.shift_idx * D, xbytes, &wb[s]);
    }
  };

  if (lane == 0)
    for (int s = 0; s < S; ++s) {
      const int64_t r = gw + (int64_t)s * G;
      if (r < a.rows) issue(r, s);
    }
  __syncwarp();

  int s = 0;
  uint32_t parity = 0u;
  unsigned int done = 0u;
  for (int64_t row = gw; row < a.rows; row += G) {
    const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&wb[s], parity, wait_limit));
    if (!ok) {
      if (lane == 0) {
        // drain: every issued copy of this warp, the expired one included
        for (int q = 0; q < S; ++q)
          if (pending & (1u << q)) (void)mbar_wait(&wb[q], (phase >> q) & 1u);
        atomicOr(&g_ring_fault, 1u);
        if (cta_state) atomicOr(&cta_state[blockIdx.x], 0x80000000u);
      }
      return;
    }
    ++done;
    const uint8_t* stage = ring + (size_t)s * stage_bytes;
    if constexpr (KIND == KIND_FP8) fp8_row<MOD>(a, row, stage, cst, lane, inv_act);
    else nvfp4_row<MOD>(a, row, stage, cst, lane);
    __syncwarp();
    if (lane == 0) {
      pending &= ~(1u << s);
      phase ^= 1u << s;
      const int64_t nr = row + (int64_t)S * G;
      if (nr < a.rows) issue(nr, s);
    }
    if (++s == S) { s = 0; parity ^= 1u; }
  }
  if (cta_state && lane == 0 && done) atomicAdd(&cta_state[blockIdx.x], done);

  if constexpr (KIND == KIND_NVFP4) {
    // rows past the end inside the last 128-row tile: zero scale bytes
    const int nblk = (int)(D >> 4), padc = (nblk + 3) & ~3, ct = padc >> 2;
    const int64_t rows_pad = (a.rows + 127) & ~(int64_t)127;
    uint8_t* sf = reinterpret_cast<uint8_t*>(a.sf);
    for (int64_t pr = a.rows + gw; pr < rows_pad; pr += G)
      for (int cc = lane; cc < padc; cc += 32) st_b8(sf + sf_off(pr, cc, ct), 0u);
  }
}

using RingKernel = void (*)(const LnArgs, const int, unsigned int*, const long long);

RingKernel pick(int kind, int mod) {
  if (kind == KIND_FP8) {
    switch (mod) {
      case MOD_NONE: return ln_ring_kernel<KIND_FP8, MOD_NONE>;
      case MOD_BCAST: return ln_ring_kernel<KIND_FP8, MOD_BCAST>;
      case MOD_PTOK: return ln_ring_kernel<KIND_FP8, MOD_PTOK>;
      case MOD_TABLE: return ln_ring_kernel<KIND_FP8, MOD_TABLE>;
    }
  } else {
    switch (mod) {
      case MOD_NONE: return ln_ring_kernel<KIND_NVFP4, MOD_NONE>;
      case MOD_BCAST: return ln_ring_kernel<KIND_NVFP4, MOD_BCAST>;
    }
  }
  return nullptr;
}

}  // namespace

int64_t ring_smem_bytes(int mod, int64_t dim, int warps, int stages) {
  const int64_t x = dim * 2;
  const bool per_token = (mod == MOD_PTOK || mod == MOD_TABLE);
  const int64_t stage = per_token ? 3 * x : x;
  const int64_t cst = mod == MOD_BCAST ? 2 * x : (mod == MOD_TABLE ? 4 * x : 0);
  return ((int64_t)warps * stages * 8 + 127) / 128 * 128 + cst + (int64_t)warps * stages * stage;
}

// Resident CTAs per SM of (kernel, threads, dynamic smem) on a device.  The
// attribute set-up and the occupancy query run once per key, outside any
// stream capture that later calls reuse.
int ring_occupancy(RingKernel k, int threads, int64_t smem) {
  struct Entry { RingKernel k; int threads; int64_t smem; int dev; int occ; };
  static Entry cache[128];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].k == k && cache[i].threads == threads && cache[i].smem == smem && cache[i].dev == dev)
      return cache[i].occ;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess) return -1;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, threads, (size_t)smem) != cudaSuccess) return -1;
  if (n < 128) cache[n++] = Entry{k, threads, smem, dev, occ};
  return occ;
}

cudaError_t launch_ln_ring(const LnArgs& a, bool nvfp4, int mod, RingShape rs, int sms, long long wait_limit,
                           cudaStream_t st) {
  RingKernel k = pick(nvfp4 ? KIND_NVFP4 : KIND_FP8, mod);
  if (!k) return cudaErrorInvalidValue;
  const int64_t smem = ring_smem_bytes(mod, a.dim, rs.warps, rs.stages);
  int occ = ring_occupancy(k, rs.warps * 32, smem);
  if (occ < 0) return cudaErrorInvalidValue;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  if (rs.ctas_per_sm > 0 && rs.ctas_per_sm < occ) occ = rs.ctas_per_sm;
  const int64_t work_rows = nvfp4 ? (a.rows + 127) / 128 * 128 : a.rows;
  int64_t grid = (work_rows + rs.warps - 1) / rs.warps;
  if (grid > (int64_t)sms * occ) grid = (int64_t)sms * occ;
  k<<<(unsigned)grid, rs.warps * 32, (size_t)smem, st>>>(a, rs.stages, nullptr, wait_limit);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Allocation-free FP8 broadcast producer (see nvfp4ap.h,
// ada_layer_norm_quant_fp8_bf16_noalloc): the ring kernel's per-CTA words
// live in this fixed array instead of any allocated buffer.
// ---------------------------------------------------------------------------

constexpr int kNoAllocMaxCtas = 1024;  // 4 KB, held by every device that loads the library
static __device__ __align__(256) unsigned int g_noalloc_cta_state[kNoAllocMaxCtas];

// Device address of g_noalloc_cta_state on the current device, looked up once
// per device (the host-side name is only a stand-in for the device symbol).
static unsigned int* noalloc_scratch(int dev) {
  static std::mutex mu;
  static unsigned int* addr[64] = {nullptr};
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_cta_state) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned int*>(p);
  }
  return addr[dev];
}

// CTAs of the last allocation-free launch per device (host-side record for
// noalloc_progress)
static int64_t g_noalloc_ctas[64] = {0};

int noalloc_fp8_bcast(const LnArgs& a, int sms, long long wait_limit, cudaStream_t st) {
  // ring shape as for the allocating path: 8 warps, up to 4 stages in ~110 KB
  RingShape rs{8, 4, 0};
  while (rs.stages > 1 && ring_smem_bytes(MOD_BCAST, a.dim, rs.warps, rs.stages) > 110 * 1024) --rs.stages;
  while (rs.warps > 1 && ring_smem_bytes(MOD_BCAST, a.dim, rs.warps, rs.stages) > 110 * 1024) --rs.warps;
  const int64_t smem = ring_smem_bytes(MOD_BCAST, a.dim, rs.warps, rs.stages);
  if (smem > 227 * 1024) return NVFP4AP_ERR_DIM;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4AP_ERR_LAUNCH;
  unsigned int* state = noalloc_scratch(dev);
  if (!state) return NVFP4AP_ERR_LAUNCH;
  RingKernel k = ln_ring_kernel<KIND_FP8, MOD_BCAST>;
  const int occ = ring_occupancy(k, rs.warps * 32, smem);
  if (occ < 1) return NVFP4AP_ERR_LAUNCH;
  int64_t grid = (a.rows + rs.warps - 1) / rs.warps;
  if (grid > (int64_t)sms * occ) grid = (int64_t)sms * occ;
  if (grid > kNoAllocMaxCtas) return NVFP4AP_ERR_SCRATCH;
  if (cudaMemsetAsync(state, 0, (size_t)grid * sizeof(unsigned int), st) != cudaSuccess) return NVFP4AP_ERR_LAUNCH;
  k<<<(unsigned)grid, rs.warps * 32, (size_t)smem, st>>>(a, rs.stages, state, wait_limit);
  if (cudaGetLastError() != cudaSuccess) return NVFP4AP_ERR_LAUNCH;
  g_noalloc_ctas[dev] = grid;
  return NVFP4AP_OK;
}

int noalloc_progress(unsigned int* words, int64_t n, int64_t* used) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NVFP4AP_ERR_LAUNCH;
  const int64_t m = g_noalloc_ctas[dev];
  if (used) *used = m;
  if (!words || n <= 0 || m == 0) return NVFP4AP_OK;
  unsigned int* state = noalloc_scratch(dev);
  if (!state) return NVFP4AP_ERR_LAUNCH;
  const int64_t k = n < m ? n : m;
  if (cudaMemcpy(words, state, (size_t)k * sizeof(unsigned int), cudaMemcpyDeviceToHost) != cudaSuccess) {
    (void)cudaGetLastError();
    return NVFP4AP_ERR_LAUNCH;
  }
  return NVFP4AP_OK;
}

cudaError_t take_ring_fault(unsigned int* fault) {
  unsigned int zero = 0u;
  cudaError_t e = cudaMemcpyFromSymbol(fault, g_ring_fault, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_ring_fault, &zero, sizeof(unsigned int));
}

}  // namespace nvfp4ap
