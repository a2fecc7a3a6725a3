// swiglu.cu -- SwiGLU -> two-level NVFP4 producer for sm_103a.
//
// Operation (h3-blackwell-runtime compare page, NVFP4_SWIGLU_FUSION_DESIGN.md:
// the SwiGLU values are recomputed inside the tensor-scale and pack passes
// with both bf16 boundaries kept -- silu(gate) rounded to bf16, then that
// value times bf16 up rounded to bf16 -- followed by the two-level NVFP4
// contract of the same page):
//   v = bf16(bf16(silu(g)) * u),  silu(g) = g / (1 + exp(-g))
//   amax = max |v|;  ts = bf16(amax / 2688)
//   per 16 elements: s = e4m3(min((amax_b / 6) / ts, 448)); codes e2m1(v / (s * ts))
//
// silu's bf16 boundary is taken on the binary32 value of silu.  A bf16 gate
// has only 65,536 bit patterns, so bf16(binary32(silu(g))) is a table built
// in float64 when the library is compiled (build.py); the kernels look the
// gate's pattern up (128 KB, read through L1: activations cluster on a few
// thousand patterns) instead of evaluating an exponential and a division per
// element.  The product of two bf16 values is exact in fp32, so its bf16
// rounding needs no care.
//
// Layout: gate and up are (rows, dim) bf16 with a common row stride `ld`
// (elements): two tensors, or the two halves of one (rows, 2*dim) FC1 output.
// Threads take 8-element chunks in a grid-stride loop whose bounds are warp-
// uniform (full-mask shuffles); chunks 2b and 2b+1 -- the halves of NVFP4
// block b -- sit in lanes t and t^1.  Two launches after a clear of the
// caller's word: the maximum pass (a running maximum per thread, one gated
// atomic per warp at the end) and the quantising pass.
#include "device.cuh"
#include "kernels.h"

namespace nvfp4ap {
namespace {

// bf16(binary32(silu(g))) for every bf16 pattern g (generated, see build.py)
__device__ const uint16_t kSiluBf16[65536] = {
#include "silu_bf16_table.inc"
};

__device__ __forceinline__ float round_bf16(float v) { return bf16_lo(f2_to_bf16x2(make_float2(v, 0.f))); }

// silu of a packed pair of bf16 gates, as a packed pair of bf16 values
__device__ __forceinline__ uint32_t silu_bf16x2(uint32_t g) {
  const uint32_t lo = __ldg(&kSiluBf16[g & 0xFFFFu]);
  const uint32_t hi = __ldg(&kSiluBf16[g >> 16]);
  return lo | (hi << 16);
}

// the 8 staged values of one chunk as four packed bf16 pairs
__device__ __forceinline__ void swiglu8(const uint16_t* g8, const uint16_t* u8, uint32_t (&vb)[4]) {
  const uint4 g = ld_once_v4(g8), u = ld_once_v4(u8);
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
    vb[i] = f2_to_bf16x2(mul2(bf16x2_to_f2(silu_bf16x2(gw[i])), bf16x2_to_f2(uw[i])));  // exact product, one rounding
}

struct SwArgs {
  const uint16_t* gate;
  const uint16_t* up;
  int64_t ld, rows, dim;
  uint8_t* packed;
  uint8_t* sf;
  float* tensor_scale;
  unsigned int* amax_ws;
};

__global__ void sw_clear_kernel(unsigned int* w) {
  pdl_enter();
  *w = 0u;
}

template <bool QUANT>
__global__ void __launch_bounds__(256) swiglu_kernel(const SwArgs a) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int nch = (int)(a.dim >> 3);
  const int64_t total = a.rows * nch;  // even: dim % 16 == 0
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int nblk = nch >> 1, padc = (nblk + 3) & ~3, ct = padc >> 2;

  float ts = 1.0f, run = 0.0f;
  if constexpr (QUANT) {
    ts = round_bf16(__fdiv_rn(__uint_as_float(__ldcg(a.amax_ws)), 2688.0f));
    if (blockIdx.x == 0 && threadIdx.x == 0) a.tensor_scale[0] = ts;
  }
  for (int64_t c0 = (int64_t)blockIdx.x * blockDim.x + (threadIdx.x & ~31); c0 < total; c0 += stride) {
    const int64_t c = c0 + lane;
    const bool valid = c < total;
    const int64_t r = valid ? c / nch : 0;
    const int j = valid ? (int)(c - r * nch) : 0;
    uint32_t vb[4] = {0u, 0u, 0u, 0u};
    if (valid) swiglu8(a.gate + r * a.ld + (int64_t)j * 8, a.up + r * a.ld + (int64_t)j * 8, vb);
    const uint32_t m2 = bf16x2_absmax(bf16x2_absmax(vb[0], vb[1]), bf16x2_absmax(vb[2], vb[3]));
    float amax = fmaxf(fabsf(bf16_lo(m2)), fabsf(bf16_hi(m2)));
    if constexpr (!QUANT) {
      run = fmaxf(run, amax);
    } else {
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));  // the block's other half
      const uint32_t sbyte =
          f2_to_e4m3x2(make_float2(fminf(__fdiv_rn(__fdiv_rn(amax, 6.0f), ts), 448.0f), 0.f)) & 0xFFu;
      float scl = e4m3_to_f32(sbyte) * ts, pre = 1.0f;
      if (scl != 0.f && scl < 0x1p-64f) {  // keep the reciprocal out of the flushed range (exact rescale)
        scl *= 0x1p64f;
        pre = 0x1p64f;
      }
      const float rh = (scl == 0.f) ? 0.f : rcp_approx(scl);
      const float rl = rh * fmaf(-scl, rh, 1.0f);
      const float2 rh2 = splat2(rh), rl2 = splat2(rl);
      float2 q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 v = mul2(bf16x2_to_f2(vb[i]), splat2(pre));
        q[i] = fma2(v, rh2, mul2(v, rl2));
      }
      const uint32_t codes = f8_to_e2m1x8(q[0], q[1], q[2], q[3]);
      if (valid) {
        st_stream_b32(a.packed + r * (a.dim >> 1) + (int64_t)j * 4, codes);
        if ((j & 1) == 0) {
          const int b = j >> 1;
          st_b8(a.sf + ((r >> 7) * ct + (b >> 2)) * 512 + (int)((r & 31) << 4) + (int)(((r >> 5) & 3) << 2) + (b & 3),
                sbyte);
        }
      }
    }
  }
  if constexpr (!QUANT) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) run = fmaxf(run, __shfl_xor_sync(0xFFFFFFFFu, run, o));
    if (lane == 0 && run > __uint_as_float(__ldcg(a.amax_ws))) atomicMax(a.amax_ws, __float_as_uint(run));
  } else {
    // padding of the swizzled scale buffer: columns nblk..padc-1 of every row,
    // and all columns of the rows up to the next multiple of 128
    const int64_t rows_pad = (a.rows + 127) & ~(int64_t)127;
    const int64_t pad_cols = (int64_t)(padc - nblk) * a.rows;
    const int64_t pad_rows = (rows_pad - a.rows) * padc;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < pad_cols + pad_rows; i += stride) {
      int64_t r;
      int b;
      if (i < pad_cols) {
        r = i / (padc - nblk);
        b = nblk + (int)(i - r * (padc - nblk));
      } else {
        const int64_t k = i - pad_cols;
        r = a.rows + k / padc;
        b = (int)(k % padc);
      }
      st_b8(a.sf + ((r >> 7) * ct + (b >> 2)) * 512 + (int)((r & 31) << 4) + (int)(((r >> 5) & 3) << 2) + (b & 3),
            0u);
    }
  }
}

// the staged values themselves (the materialised form), 16 bytes per chunk
__global__ void __launch_bounds__(256) swiglu_values_kernel(const SwArgs a, uint16_t* out) {
  pdl_enter();
  const int nch = (int)(a.dim >> 3);
  const int64_t total = a.rows * nch;
  for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < total; c += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = c / nch;
    const int j = (int)(c - r * nch);
    uint32_t vb[4];
    swiglu8(a.gate + r * a.ld + (int64_t)j * 8, a.up + r * a.ld + (int64_t)j * 8, vb);
    st_stream_v4(out + r * a.dim + (int64_t)j * 8, make_uint4(vb[0], vb[1], vb[2], vb[3]));
  }
}

int sw_grid(int sms) {
  static int occ = 0;
  if (occ == 0) {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, swiglu_kernel<true>, 256, 0) != cudaSuccess || o < 1) o = 1;
    occ = o;
  }
  return sms * occ;
}

}  // namespace

cudaError_t launch_swiglu_2level(const void* gate, const void* up, int64_t ld, int64_t rows, int64_t dim,
                                 void* packed, void* sf, float* tensor_scale, unsigned int* ws, int sms,
                                 cudaStream_t st) {
  SwArgs a{static_cast<const uint16_t*>(gate), static_cast<const uint16_t*>(up), ld, rows, dim,
           static_cast<uint8_t*>(packed), static_cast<uint8_t*>(sf), tensor_scale, ws};
  const int64_t chunks = rows * (dim / 8);
  int64_t grid = sw_grid(sms);
  const int64_t need = (chunks + 255) / 256;
  if (grid > need) grid = need < 1 ? 1 : need;
  cudaError_t e = launch_maybe_pdl(sw_clear_kernel, dim3(1), dim3(1), 0, st, ws);
  if (e != cudaSuccess) return e;
  e = launch_maybe_pdl(swiglu_kernel<false>, dim3((unsigned)grid), dim3(256), 0, st, a);
  if (e != cudaSuccess) return e;
  return launch_maybe_pdl(swiglu_kernel<true>, dim3((unsigned)grid), dim3(256), 0, st, a);
}

cudaError_t launch_swiglu_values(const void* gate, const void* up, int64_t ld, int64_t rows, int64_t dim, void* out,
                                 int sms, cudaStream_t st) {
  SwArgs a{static_cast<const uint16_t*>(gate), static_cast<const uint16_t*>(up), ld, rows, dim, nullptr, nullptr,
           nullptr, nullptr};
  const int64_t chunks = rows * (dim / 8);
  int64_t grid = sw_grid(sms);
  const int64_t need = (chunks + 255) / 256;
  if (grid > need) grid = need < 1 ? 1 : need;
  return launch_maybe_pdl(swiglu_values_kernel, dim3((unsigned)grid), dim3(256), 0, st, a,
                          static_cast<uint16_t*>(out));
}

}  // namespace nvfp4ap
