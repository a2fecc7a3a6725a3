// ln_ring.cu -- the kernel of the allocation-free FP8 broadcast producer
// (ada_layer_norm_quant_fp8_bf16_noalloc) for sm_103a.
//
// Operation (adaptive-layernorm-producers README, "Available Functions":
// ada_layer_norm_quant_fp8_bf16; "Tensor Contract"):
//   y = (x - mean) * rstd * (1 + scale) + shift, rstd = 1/sqrt(var + eps),
//   out = e4m3fn(y / act_scale), nearest-even, saturating.
//
// Design: a warp per row with its rows staged through shared memory by the
// TMA engine, so the kernel keeps no per-row state outside the CTA except one
// progress word per CTA -- the only device scratch it needs, which the
// allocation-free entry point takes from a fixed array inside the library.
//  * persistent CTAs (up to a few per SM), W warps each; warp g of the grid
//    owns rows g, g + G, g + 2G, ... (G = warps in the grid);
//  * each warp owns a ring of S shared-memory stages; lane 0 fills a stage
//    with one row of x by a 1-D bulk copy (cp.async.bulk) completing that
//    stage's mbarrier, so up to S rows per warp are in flight while it
//    computes; scale and shift are copied into shared memory once per CTA;
//  * a warp reduces its row with shuffles only (no CTA barrier in the loop):
//    the mean, then the centred sum of squares, from the staged row; then the
//    codes, written straight to global memory;
//  * every mbarrier wait is bounded by the `wait_limit` argument (SM clock
//    cycles; the library passes about one second); on expiry lane 0 waits,
//    with the library's normal bound, for every copy the warp has in flight
//    (the one whose wait ran out included), then sets the library's fault
//    word and its CTA's bit 31 and the warp stops, so no copy is left writing
//    into the shared memory of a warp -- or a CTA -- that has exited.
#include <mutex>

#include "device.cuh"
#include "kernels.h"
#include "nvfp4ap.h"
#include "tma.cuh"

namespace nvfp4ap {

// Set (bit 0) by the ring kernel when an mbarrier wait ran out; read and
// cleared by the host through nvfp4ap_take_device_fault().
__device__ unsigned int g_ring_fault = 0u;

namespace {

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

// The codes of one staged row: y = (x - mean) * (rstd + rstd * scale) + shift,
// then / act_scale; scale and shift from the CTA's copy in shared memory.
__device__ __forceinline__ void fp8_row(const LnArgs& a, int64_t row, const uint8_t* stage, const uint8_t* cst,
                                        int lane, float inv_act) {
  const int64_t D = a.dim;
  const int nch = (int)(D >> 3);
  const uint32_t xbytes = (uint32_t)(D * 2);
  const uint4* xs = reinterpret_cast<const uint4*>(stage);
  float mean, rstd;
  row_stats(xs, nch, lane, (float)D, a.eps, mean, rstd);
  const float2 nm = splat2(-mean), inv2 = splat2(inv_act), rstd2 = splat2(rstd);
  uint8_t* orow = reinterpret_cast<uint8_t*>(a.out) + row * D;
  for (int c = lane; c < nch; c += 32) {
    const uint4 v = xs[c];
    const uint4 sv = reinterpret_cast<const uint4*>(cst)[c];
    const uint4 hv = reinterpret_cast<const uint4*>(cst + xbytes)[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w}, sw[4] = {sv.x, sv.y, sv.z, sv.w}, hw[4] = {hv.x, hv.y, hv.z, hv.w};
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 d = add2(bf16x2_to_f2(w[i]), nm);
      const float2 y = fma2(d, fma2(bf16x2_to_f2(sw[i]), rstd2, rstd2), bf16x2_to_f2(hw[i]));
      q[i] = f2_to_e4m3x2(mul2(y, inv2));
    }
    st_stream_v2(orow + (int64_t)c * 8, q[0] | (q[1] << 16), q[2] | (q[3] << 16));
  }
}

// `cta_state`: one word per CTA; each warp adds the number of rows it
// finished, and bit 31 marks a CTA one of whose waits ran out.
__global__ void __launch_bounds__(512)
    ln_ring_kernel(const LnArgs a, const int S, unsigned int* cta_state, const long long wait_limit) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int W = blockDim.x >> 5, w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t D = a.dim;
  const uint32_t xbytes = (uint32_t)(D * 2);

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint8_t* cst = smem + ((W * S * 8 + 127) & ~127);
  uint8_t* stages = cst + 2 * xbytes;

  if (threadIdx.x < W * S) mbar_init(&bars[threadIdx.x], 1);
  mbar_init_fence();
  {
    uint4* dst = reinterpret_cast<uint4*>(cst);
    const int n = (int)(xbytes >> 4);
    for (int i = threadIdx.x; i < 2 * n; i += blockDim.x)
      dst[i] = ld_reuse_v4(i < n ? (const void*)(a.scale + (int64_t)i * 8)
                                 : (const void*)(a.shift + (int64_t)(i - n) * 8));
  }
  __syncthreads();

  const int64_t G = (int64_t)gridDim.x * W;
  const int64_t gw = (int64_t)blockIdx.x * W + w;
  uint8_t* ring = stages + (size_t)w * S * xbytes;
  uint64_t* wb = bars + w * S;
  const float inv_act = 1.0f / __ldg(a.act_scale);

  uint32_t pending = 0u;  // lane 0: stages with a copy in flight
  uint32_t phase = 0u;    // lane 0: parity of each stage's next completion
  auto issue = [&](int64_t row, int s) {
    pending |= 1u << s;
    mbar_expect_tx(&wb[s], xbytes);
    bulk_g2s(ring + (size_t)s * xbytes, a.x + row * D, xbytes, &wb[s]);
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
        atomicOr(&cta_state[blockIdx.x], 0x80000000u);
      }
      return;
    }
    ++done;
    fp8_row(a, row, ring + (size_t)s * xbytes, cst, lane, inv_act);
    __syncwarp();
    if (lane == 0) {
      pending &= ~(1u << s);
      phase ^= 1u << s;
      const int64_t nr = row + (int64_t)S * G;
      if (nr < a.rows) issue(nr, s);
    }
    if (++s == S) {
      s = 0;
      parity ^= 1u;
    }
  }
  if (lane == 0 && done) atomicAdd(&cta_state[blockIdx.x], done);
}

int64_t ring_smem_bytes(int64_t dim, int warps, int stages) {
  const int64_t x = dim * 2;
  return ((int64_t)warps * stages * 8 + 127) / 128 * 128 + 2 * x + (int64_t)warps * stages * x;
}

// Resident CTAs per SM of the kernel for (threads, dynamic smem) on a device.
// The attribute set-up and the occupancy query run once per key, outside any
// stream capture that later calls reuse.
int ring_occupancy(int threads, int64_t smem) {
  struct Entry { int threads; int64_t smem; int dev; int occ; };
  static Entry cache[64];
  static int n = 0;
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n; ++i)
    if (cache[i].threads == threads && cache[i].smem == smem && cache[i].dev == dev) return cache[i].occ;
  if (cudaFuncSetAttribute(ln_ring_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
    return -1;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, ln_ring_kernel, threads, (size_t)smem) != cudaSuccess)
    return -1;
  if (n < 64) cache[n++] = Entry{threads, smem, dev, occ};
  return occ;
}

}  // namespace

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
  // 8 warps, up to 4 stages in ~110 KB, so that two CTAs share an SM
  int warps = 8, stages = 4;
  while (stages > 1 && ring_smem_bytes(a.dim, warps, stages) > 110 * 1024) --stages;
  while (warps > 1 && ring_smem_bytes(a.dim, warps, stages) > 110 * 1024) --warps;
  const int64_t smem = ring_smem_bytes(a.dim, warps, stages);
  if (smem > 227 * 1024) return NVFP4AP_ERR_DIM;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4AP_ERR_LAUNCH;
  unsigned int* state = noalloc_scratch(dev);
  if (!state) return NVFP4AP_ERR_LAUNCH;
  const int occ = ring_occupancy(warps * 32, smem);
  if (occ < 1) return NVFP4AP_ERR_LAUNCH;
  int64_t grid = (a.rows + warps - 1) / warps;
  if (grid > (int64_t)sms * occ) grid = (int64_t)sms * occ;
  if (grid > kNoAllocMaxCtas) return NVFP4AP_ERR_SCRATCH;
  if (cudaMemsetAsync(state, 0, (size_t)grid * sizeof(unsigned int), st) != cudaSuccess) return NVFP4AP_ERR_LAUNCH;
  ln_ring_kernel<<<(unsigned)grid, warps * 32, (size_t)smem, st>>>(a, stages, state, wait_limit);
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
