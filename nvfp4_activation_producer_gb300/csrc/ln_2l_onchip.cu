// ln_2l_onchip.cu -- the two-level NVFP4 LayerNorm producers in one
// cooperative launch, for tensors that fit in the GPU's shared memory.
//
// Two-level NVFP4 (h3-blackwell-runtime compare page: NVFP4_STREAMING_DESIGN.md
// "Numerical Constraint" -- no block can be encoded before the whole tensor's
// maximum is known; the P1 checkpoint's "numerical_contract" -- block scale
// (amax_b / 6) / ts clamped at 448):
//   v = bf16(y), y the (modulated) LayerNorm of the row;
//   amax = max |v| over the tensor; ts = bf16(amax / 2688);
//   per 16 elements s = e4m3fn(min((amax_b / 6) / ts, 448)) with both quotients
//   correctly rounded in fp32; codes e2m1 of v / (s * ts).
//
// Design.  When every CTA's share of the rows fits in its shared memory
// (5070 x 3072 bf16 is 31 MB: 34 rows of 6 KB per SM), the tensor is read from
// HBM once: one CTA per SM (a cooperative launch, so all are resident) stages
// its rows by 1-D bulk copies, one mbarrier per row.  Phase 1, a warp per row
// as its copy lands: the statistics (shifted by the row's first element, as
// the other kernels), then v = bf16(y) written over the row in shared memory
// and the largest |v|.  The CTA's maximum goes to the caller's workspace word
// by one atomic; a grid-wide barrier (a counter in the workspace, cleared by
// the launch before) makes the maximum final.  Phase 2 encodes the staged v,
// one 16-value block per thread over all the CTA's rows, so that the scale
// and code arithmetic -- which cannot start before the barrier -- is spread
// evenly over the CTA.  Modulation vectors are read per block through L1.
//
// Every wait is bounded: the row copies by the `wait_limit` argument, the
// grid barrier by the library's normal bound.  A CTA whose wait runs out waits
// (with the normal bound) for every copy it issued, sets the fault word and
// returns without writing outputs.
#include <mutex>

#include "ln_blk.cuh"
#include "tma.cuh"

namespace nvfp4ap {

// Set (bit 0) when a bounded wait of the on-chip kernel ran out; read and
// cleared by take_onchip_fault().
__device__ unsigned int g_onchip_fault = 0u;

namespace {

constexpr int kOnchipThreads = 1024;
constexpr int kOnchipBarBytes = 1024;  // up to 128 row mbarriers

// workspace words: [0] the tensor's maximum (fp32 bits), [1] the grid
// barrier's arrival count
__global__ void onchip_clear_kernel(unsigned int* w) {
  pdl_enter();
  w[0] = 0u;
  w[1] = 0u;
}

__device__ __forceinline__ void red_release_add(unsigned int* p, unsigned int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ unsigned int ld_relaxed_u32(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Stage one half (8 values) of a block in place: x -> v = bf16(y); returns
// the packed pair of the half's largest magnitudes.
template <int MOD>
__device__ __forceinline__ uint32_t stage_half(const LnArgs& a, uint4* p, int64_t col, int seg, float2 nk, float2 A2,
                                               float2 B2) {
  const uint4 u = *p;
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t s[4] = {0u, 0u, 0u, 0u}, t[4] = {0u, 0u, 0u, 0u};
  if constexpr (MOD == MOD_BCAST) {
    const uint4 sv = ld_reuse_v4(a.scale + col), hv = ld_reuse_v4(a.shift + col);
    s[0] = sv.x; s[1] = sv.y; s[2] = sv.z; s[3] = sv.w;
    t[0] = hv.x; t[1] = hv.y; t[2] = hv.z; t[3] = hv.w;
  } else if constexpr (MOD == MOD_SEG) {
    if (seg >= 0) {
      const uint4 sv = ld_reuse_v4(a.seg_scale + (int64_t)seg * a.dim + col);
      const uint4 hv = ld_reuse_v4(a.seg_shift + (int64_t)seg * a.dim + col);
      s[0] = sv.x; s[1] = sv.y; s[2] = sv.z; s[3] = sv.w;
      t[0] = hv.x; t[1] = hv.y; t[2] = hv.z; t[3] = hv.w;
    }
  }
  uint32_t v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 y = fma2(add2(bf16x2_to_f2(w[i]), nk), A2, B2);
    if constexpr (MOD != MOD_NONE) y = fma2(y, add2(bf16x2_to_f2(s[i]), splat2(1.0f)), bf16x2_to_f2(t[i]));
    v[i] = f2_to_bf16x2(y);
  }
  *p = make_uint4(v[0], v[1], v[2], v[3]);
  return bf16x2_absmax(bf16x2_absmax(v[0], v[1]), bf16x2_absmax(v[2], v[3]));
}

// Dynamic shared memory: the row mbarriers (1 KB), the blocks' largest |v|
// as bf16 (nr * nblk * 2 bytes, padded to 128), then the nr rows (2 * dim
// bytes each).
__host__ __device__ __forceinline__ int64_t onchip_amax_bytes(int64_t dim, int64_t nr) {
  return (nr * (dim >> 4) * 2 + 127) / 128 * 128;
}

template <int MOD>
__global__ void __launch_bounds__(kOnchipThreads, 1)
    nv2l_onchip_kernel(const LnArgs a, const float inv_d, const long long wait_limit) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ unsigned int cta_max;
  __shared__ float gmax;
  __shared__ int bad;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5, nwarps = blockDim.x >> 5;
  const int64_t D = a.dim, G = gridDim.x;
  const int nblk = (int)(D >> 4), padc = (nblk + 3) & ~3, ct = padc >> 2, nq = (int)(D >> 3);
  const uint32_t xbytes = (uint32_t)(D * 2);
  const int nr = a.rows > (int64_t)blockIdx.x ? (int)((a.rows - blockIdx.x + G - 1) / G) : 0;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint16_t* bmax = reinterpret_cast<uint16_t*>(smem + kOnchipBarBytes);
  uint8_t* rows = smem + kOnchipBarBytes + onchip_amax_bytes(D, nr);
  unsigned int* counter = a.amax_ws + 1;
  // In phase 1 a lane takes the two 16-byte halves of its block in the order
  // h0, h0 ^ 1: the eight lanes of a quarter-warp then cover all 32 banks.
  // (Phase 2 reads them in order: there the reordering's selects cost more
  // than the conflicts, 15.0 -> 14.8 us at 5070x3072.)
  const int h0 = (lane >> 2) & 1;

  if (t < nr) mbar_init(&bars[t], 1);
  if (t == 0) {
    cta_max = 0u;
    bad = 0;
  }
  mbar_init_fence();
  __syncthreads();
  pdl_enter();
  if (t == 0)
    for (int j = 0; j < nr; ++j) {
      mbar_expect_tx(&bars[j], xbytes);
      bulk_g2s(rows + (size_t)j * xbytes, a.x + (blockIdx.x + (int64_t)j * G) * D, xbytes, &bars[j]);
    }

  // ---- phase 1, a warp per row as its copy lands: the statistics, then
  // v = bf16(y) written over the row, each block's largest |v| ---------------
  uint32_t wmax2 = 0u;  // packed pair of running magnitudes
  for (int j = warp; j < nr; j += nwarps) {
    const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bars[j], 0u, wait_limit));
    if (!ok) {
      if (lane == 0) bad = 1;
      continue;
    }
    const int64_t row = blockIdx.x + (int64_t)j * G;
    uint4* xq = reinterpret_cast<uint4*>(rows + (size_t)j * xbytes);
    const float K = __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(xq)[0] << 16);
    const float2 nk = splat2(-K);
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
    for (int q = lane; q < nq; q += 32) {
      const uint4 u = xq[q];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 d = add2(bf16x2_to_f2(w[i]), nk);
        s1 = add2(s1, d);
        s2 = fma2(d, d, s2);
      }
    }
    const float m1 = warp_sum(s1.x + s1.y) * inv_d;  // mean - K
    const float var = fmaxf(fmaf(warp_sum(s2.x + s2.y), inv_d, -m1 * m1), 0.f);
    const float rstd = rsqrtf(var + a.eps);
    int seg = 0;
    if constexpr (MOD == MOD_SEG) {
      const int sg = __ldg(a.seg_idx + row);
      seg = (sg >= 0 && sg < a.nseg) ? sg : -1;
      if (seg < 0 && lane == 0) atomicOr(&g_blk_seg_fault, 1u);
    }
    const float2 A2 = splat2(rstd), B2 = splat2(-m1 * rstd);
    // the statistics' reads of the row are done (warp_sum consumed them)
    // before any lane writes v over it
    uint16_t* brow = bmax + j * nblk;
    for (int b = lane; b < nblk; b += 32) {
      const int64_t col = (int64_t)b * 16;
      const uint32_t m = bf16x2_absmax(stage_half<MOD>(a, xq + 2 * b + h0, col + h0 * 8, seg, nk, A2, B2),
                                       stage_half<MOD>(a, xq + 2 * b + (h0 ^ 1), col + (h0 ^ 1) * 8, seg, nk, A2, B2));
      wmax2 = bf16x2_absmax(wmax2, m);
      brow[b] = (uint16_t)(__float_as_uint(fmaxf(fabsf(bf16_lo(m)), fabsf(bf16_hi(m)))) >> 16);
    }
  }
  float wmax = fmaxf(fabsf(bf16_lo(wmax2)), fabsf(bf16_hi(wmax2)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xFFFFFFFFu, wmax, o));
  if (lane == 0 && wmax > 0.f) atomicMax(&cta_max, __float_as_uint(wmax));
  __syncthreads();

  // ---- the grid-wide barrier: the CTA's maximum into the workspace word, a
  // release increment of the count, then (acquire) every CTA has arrived ------
  if (t == 0) {
    if (cta_max > 0u) atomicMax(a.amax_ws, cta_max);
    red_release_add(counter, 1u);
    const long long t0 = clock64();
    while (ld_acquire_u32(counter) < (unsigned int)G) {
      if (clock64() - t0 > kWaitCycles) {
        bad = 1;
        break;
      }
    }
    gmax = __uint_as_float(ld_relaxed_u32(a.amax_ws));
  }
  __syncthreads();
  if (bad) {
    // wait, with the normal bound, for every copy this CTA issued, then report
    if (t == 0) {
      for (int j = 0; j < nr; ++j) (void)mbar_wait(&bars[j], 0u);
      atomicOr(&g_onchip_fault, 1u);
    }
    return;
  }

  // ---- phase 2: block scales and codes of the staged v ----------------------
  // One block per thread and step over the CTA's (row, block) pairs, in
  // row-major order: consecutive lanes take consecutive blocks of a row.
  const float ts = blk_round_bf16(__fdiv_rn(gmax, 2688.0f));
  const float rts = __frcp_rn(ts);
  if (blockIdx.x == 0 && t == 0) a.tensor_scale[0] = ts;
  // 32-bit offsets: this CTA's rows are blockIdx.x + j * G, j < 128, and its
  // share of the tensor fits in shared memory, so j * G * dim / 2 and every
  // swizzled scale offset stay far below 2^31
  uint8_t* const out0 = reinterpret_cast<uint8_t*>(a.out) + (int64_t)blockIdx.x * (D >> 1);
  uint8_t* const sf = reinterpret_cast<uint8_t*>(a.sf);
  const int ostride = (int)G * (int)(D >> 1), tile = ct * 512;
  const int step = blockDim.x, step_j = step / nblk, step_b = step - step_j * nblk;
  int j = t / nblk, b = t - j * nblk;
  for (; j < nr; j += step_j, b += step_b) {
    if (b >= nblk) {
      b -= nblk;
      if (++j >= nr) break;
    }
    const int r = (int)blockIdx.x + j * (int)G;
    const uint4* p = reinterpret_cast<const uint4*>(rows + (size_t)j * xbytes) + 2 * b;
    const uint4 u0 = p[0], u1 = p[1];
    const uint32_t vb[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    const float amax = __uint_as_float((uint32_t)bmax[j * nblk + b] << 16);
    // (amax_b / 6) / ts, both quotients correctly rounded, clamped at 448
    // (fminf takes 448 for the 0/0 of an all-zero tensor); the divisor of
    // the codes is s * ts, exact in fp32
    const uint32_t sbyte = f2_to_e4m3x2(make_float2(fminf(two_level_quot(amax, ts, rts), 448.0f), 0.f)) & 0xFFu;
    uint32_t c0, c1;
    block_codes_2l(vb, e4m3_to_f32(sbyte) * ts, c0, c1);
    st_stream_v2(out0 + (j * ostride + b * 8), c0, c1);
    st_b8(sf + ((r >> 7) * tile + ((r & 31) << 4) + ((r >> 3) & 12) + (b >> 2) * 512 + (b & 3)), sbyte);
  }
  // scale columns past the last block of this CTA's rows, and rows past the
  // end inside the last 128-row tile: zero scale bytes
  if (padc > nblk)
    for (int i = t; i < nr * (padc - nblk); i += blockDim.x) {
      const int jj = i / (padc - nblk), c = nblk + i - jj * (padc - nblk);
      const int64_t row = blockIdx.x + (int64_t)jj * G;
      st_b8(sf + (row >> 7) * (int64_t)ct * 512 + (int)((row & 31) << 4) + (int)(((row >> 5) & 3) << 2) +
                (c >> 2) * 512 + (c & 3),
            0u);
    }
  const int64_t rows_pad = (a.rows + 127) & ~(int64_t)127;
  for (int64_t pr = a.rows + blockIdx.x; pr < rows_pad; pr += G) {
    uint8_t* sfrow = sf + (pr >> 7) * (int64_t)ct * 512 + (int)((pr & 31) << 4) + (int)(((pr >> 5) & 3) << 2);
    for (int c = t; c < padc; c += blockDim.x) st_b8(sfrow + (c >> 2) * 512 + (c & 3), 0u);
  }
}

using OnchipKernel = void (*)(const LnArgs, const float, const long long);

OnchipKernel pick(int mod) {
  switch (mod) {
    case MOD_NONE: return nv2l_onchip_kernel<MOD_NONE>;
    case MOD_BCAST: return nv2l_onchip_kernel<MOD_BCAST>;
    case MOD_SEG: return nv2l_onchip_kernel<MOD_SEG>;
    default: return nullptr;
  }
}

int64_t onchip_smem(int64_t dim, int64_t nr) { return kOnchipBarBytes + onchip_amax_bytes(dim, nr) + nr * dim * 2; }

// one CTA per SM, at most one per row
int64_t onchip_grid(int64_t rows, int sms) { return rows < sms ? rows : sms; }

// Largest dynamic shared memory the kernel may take on the current device
// (the opt-in limit minus its static use), set once per kernel and device.
int64_t onchip_max_smem(OnchipKernel k) {
  struct Entry { OnchipKernel k; int dev; int64_t max; };
  static Entry cache[8];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].k == k && cache[i].dev == dev) return cache[i].max;
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, k) != cudaSuccess) return -1;
  int optin = 0;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return -1;
  const int64_t mx = (int64_t)optin - (int64_t)fa.sharedSizeBytes;
  if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mx) != cudaSuccess) return -1;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kOnchipThreads, (size_t)mx) != cudaSuccess || occ < 1)
    return -1;
  if (n < 8) cache[n++] = Entry{k, dev, mx};
  return mx;
}

}  // namespace

bool ln_2level_onchip_fits(int mod, int64_t rows, int64_t dim, int sms) {
  OnchipKernel k = pick(mod);
  if (!k || sms <= 0 || rows < 1 || dim < 16 || dim % 16 != 0) return false;
  const int64_t G = onchip_grid(rows, sms), nr = (rows + G - 1) / G;
  if (nr > kOnchipBarBytes / 8) return false;
  const int64_t mx = onchip_max_smem(k);
  return mx > 0 && onchip_smem(dim, nr) <= mx;
}

cudaError_t launch_ln_2level_onchip(const LnArgs& a, int mod, int sms, long long wait_limit, cudaStream_t st) {
  OnchipKernel k = pick(mod);
  if (!k || !ln_2level_onchip_fits(mod, a.rows, a.dim, sms)) return cudaErrorInvalidValue;
  const int64_t G = onchip_grid(a.rows, sms), nr = (a.rows + G - 1) / G;
  cudaError_t e = launch_maybe_pdl(onchip_clear_kernel, dim3(1), dim3(1), 0, st, a.amax_ws);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)G);
  cfg.blockDim = dim3(kOnchipThreads);
  cfg.dynamicSmemBytes = (size_t)onchip_smem(a.dim, nr);
  cfg.stream = st;
  // cooperative (every CTA resident: the grid barrier) and, as every launch of
  // the library, programmatic serialisation (the kernel waits for the previous
  // grid before it touches memory); without the latter if refused
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  const float inv_d = (float)(1.0 / (double)a.dim);
  e = cudaLaunchKernelEx(&cfg, k, a, inv_d, wait_limit);
  if (e != cudaSuccess && cfg.numAttrs == 2) {
    (void)cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k, a, inv_d, wait_limit);
  }
  return e;
}

cudaError_t take_onchip_fault(unsigned int* fault) {
  unsigned int zero = 0u;
  cudaError_t e = cudaMemcpyFromSymbol(fault, g_onchip_fault, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_onchip_fault, &zero, sizeof(unsigned int));
}

// this translation unit's copy of the segment fault word (ln_blk.cuh)
cudaError_t take_onchip_seg_fault(unsigned int* fault) { return take_blk_word(fault); }

}  // namespace nvfp4ap
