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
// Work items are 16-element blocks (two-level passes) or 8-element chunks
// (materialised values) in one flat grid-stride loop; an item's row comes
// from a multiply-high division by the invariant items-per-row count
// (divide.cuh), so the loop carries no 64-bit division.  In the two-level
// passes a lane owns a whole NVFP4 block: its gate and up are two 32-byte
// reads (one 256-bit load each when both are 32-byte aligned), and its
// maximum, scale and 16 codes are computed once, with no shuffle.  Two launches after a clear of the caller's
// word: the maximum pass (a running maximum per thread, one atomic per CTA)
// and the quantising pass.
#include "device.cuh"
#include "divide.cuh"
#include "kernels.h"

namespace nvfp4ap {
namespace {

// bf16(binary32(silu(g))) for every bf16 pattern g (generated, see build.py)
__device__ const uint16_t kSiluBf16[65536] = {
#include "silu_bf16_table.inc"
};

constexpr int kSwThreads = 256;

__device__ __forceinline__ float round_bf16(float v) { return bf16_lo(f2_to_bf16x2(make_float2(v, 0.f))); }

// silu of a packed pair of bf16 gates, as a packed pair of bf16 values
__device__ __forceinline__ uint32_t silu_bf16x2(uint32_t g) {
  const uint32_t lo = __ldg(&kSiluBf16[g & 0xFFFFu]);
  const uint32_t hi = __ldg(&kSiluBf16[g >> 16]);
  return lo | (hi << 16);
}

// v = bf16(silu(g) * u) for one packed pair (the product is exact, one rounding)
__device__ __forceinline__ uint32_t swiglu_pair(uint32_t g, uint32_t u) {
  return f2_to_bf16x2(mul2(bf16x2_to_f2(silu_bf16x2(g)), bf16x2_to_f2(u)));
}

// 32 contiguous bytes (16 bf16 values), read once
template <bool V8>
__device__ __forceinline__ void ld_block16(const uint16_t* p, uint32_t (&w)[8]) {
  if constexpr (V8) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
  } else {
    const uint4 a = ld_once_v4(p), b = ld_once_v4(p + 8);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  }
}

struct SwArgs {
  const uint16_t* gate;
  const uint16_t* up;
  int64_t ld, rows, dim;
  uint8_t* packed;
  uint8_t* sf;
  float* tensor_scale;
  unsigned int* amax_ws;
  uint32_t items;  // rows * items per row
  InvDiv per_row;  // items per row (16-element blocks or 8-element chunks)
};

__global__ void sw_clear_kernel(unsigned int* w) {
  pdl_enter();
  *w = 0u;
}

template <bool QUANT, bool V8>
__global__ void __launch_bounds__(kSwThreads) swiglu_kernel(const SwArgs a) {
  __shared__ float redm[kSwThreads / 32];
  pdl_enter();
  const int nblk = (int)(a.dim >> 4), padc = (nblk + 3) & ~3, ct = padc >> 2;
  const uint32_t stride = gridDim.x * blockDim.x;

  float ts = 1.0f, rts = 1.0f, run = 0.0f;
  if constexpr (QUANT) {
    ts = round_bf16(__fdiv_rn(__uint_as_float(__ldcg(a.amax_ws)), 2688.0f));
    rts = __frcp_rn(ts);
    if (blockIdx.x == 0 && threadIdx.x == 0) a.tensor_scale[0] = ts;
  }
  for (uint32_t n = blockIdx.x * blockDim.x + threadIdx.x; n < a.items; n += stride) {
    const uint32_t r = inv_div(n, a.per_row), b = n - r * (uint32_t)nblk;
    const int64_t off = (int64_t)r * a.ld + (int64_t)b * 16;
    uint32_t gw[8], uw[8], vb[8];
    ld_block16<V8>(a.gate + off, gw);
    ld_block16<V8>(a.up + off, uw);
#pragma unroll
    for (int i = 0; i < 8; ++i) vb[i] = swiglu_pair(gw[i], uw[i]);
    const uint32_t m = bf16x2_absmax(bf16x2_absmax(bf16x2_absmax(vb[0], vb[1]), bf16x2_absmax(vb[2], vb[3])),
                                     bf16x2_absmax(bf16x2_absmax(vb[4], vb[5]), bf16x2_absmax(vb[6], vb[7])));
    const float amax = fmaxf(fabsf(bf16_lo(m)), fabsf(bf16_hi(m)));
    if constexpr (!QUANT) {
      run = fmaxf(run, amax);
    } else {
      // (amax_b / 6) / ts, each quotient correctly rounded (two_level_quot),
      // clamped at 448 (fminf takes 448 for the 0/0 of an all-zero tensor); the
      // divisor of the codes is s * ts, exact in fp32
      const uint32_t sbyte = f2_to_e4m3x2(make_float2(fminf(two_level_quot(amax, ts, rts), 448.0f), 0.f)) & 0xFFu;
      uint32_t c0, c1;
      block_codes_2l(vb, e4m3_to_f32(sbyte) * ts, c0, c1);
      st_stream_v2(a.packed + (int64_t)r * (a.dim >> 1) + (int64_t)b * 8, c0, c1);
      st_b8(a.sf + ((int64_t)(r >> 7) * ct + (b >> 2)) * 512 + (int)((r & 31) << 4) + (int)(((r >> 5) & 3) << 2) +
                (b & 3),
            sbyte);
    }
  }
  if constexpr (!QUANT) {
    // the CTA's largest |v| (non-negative fp32: its bits order like the values)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) run = fmaxf(run, __shfl_xor_sync(0xFFFFFFFFu, run, o));
    if ((threadIdx.x & 31) == 0) redm[threadIdx.x >> 5] = run;
    __syncthreads();
    if (threadIdx.x == 0) {
      float mx = redm[0];
      for (int w = 1; w < (int)(blockDim.x >> 5); ++w) mx = fmaxf(mx, redm[w]);
      if (mx > 0.f) atomicMax(a.amax_ws, __float_as_uint(mx));
    }
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

// the staged values themselves (the materialised form): 8-element chunks,
// 16 bytes of gate, up and output each
__global__ void __launch_bounds__(kSwThreads) swiglu_values_kernel(const SwArgs a, uint16_t* out) {
  pdl_enter();
  const uint32_t nch = (uint32_t)(a.dim >> 3);
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t n = blockIdx.x * blockDim.x + threadIdx.x; n < a.items; n += stride) {
    const uint32_t r = inv_div(n, a.per_row), j = n - r * nch;
    const int64_t off = (int64_t)r * a.ld + (int64_t)j * 8;
    const uint4 g = ld_once_v4(a.gate + off), u = ld_once_v4(a.up + off);
    st_stream_v4(out + (int64_t)r * a.dim + (int64_t)j * 8,
                 make_uint4(swiglu_pair(g.x, u.x), swiglu_pair(g.y, u.y), swiglu_pair(g.z, u.z),
                            swiglu_pair(g.w, u.w)));
  }
}

template <typename K>
int sw_grid(K k, int sms, int64_t items) {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kSwThreads, 0) != cudaSuccess || occ < 1) occ = 1;
  int64_t grid = (int64_t)sms * occ;
  const int64_t need = (items + kSwThreads - 1) / kSwThreads;
  if (grid > need) grid = need < 1 ? 1 : need;
  return (int)grid;
}

}  // namespace

bool swiglu_items_fit(int64_t rows, int64_t dim) { return rows * (dim / 8) < ((int64_t)1 << 32); }

cudaError_t launch_swiglu_2level(const void* gate, const void* up, int64_t ld, int64_t rows, int64_t dim,
                                 void* packed, void* sf, float* tensor_scale, unsigned int* ws, int sms,
                                 cudaStream_t st) {
  if (!swiglu_items_fit(rows, dim)) return cudaErrorInvalidValue;
  const uint32_t nblk = (uint32_t)(dim / 16);
  SwArgs a{static_cast<const uint16_t*>(gate), static_cast<const uint16_t*>(up), ld, rows, dim,
           static_cast<uint8_t*>(packed), static_cast<uint8_t*>(sf), tensor_scale, ws,
           (uint32_t)(rows * nblk), make_inv_div(nblk)};
  const bool v8 = (reinterpret_cast<uintptr_t>(gate) % 32 == 0) && (reinterpret_cast<uintptr_t>(up) % 32 == 0) &&
                  (ld % 16 == 0);
  cudaError_t e = launch_maybe_pdl(sw_clear_kernel, dim3(1), dim3(1), 0, st, ws);
  if (e != cudaSuccess) return e;
  auto k0 = v8 ? swiglu_kernel<false, true> : swiglu_kernel<false, false>;
  auto k1 = v8 ? swiglu_kernel<true, true> : swiglu_kernel<true, false>;
  e = launch_maybe_pdl(k0, dim3(sw_grid(k0, sms, a.items)), dim3(kSwThreads), 0, st, a);
  if (e != cudaSuccess) return e;
  return launch_maybe_pdl(k1, dim3(sw_grid(k1, sms, a.items)), dim3(kSwThreads), 0, st, a);
}

cudaError_t launch_swiglu_values(const void* gate, const void* up, int64_t ld, int64_t rows, int64_t dim, void* out,
                                 int sms, cudaStream_t st) {
  if (!swiglu_items_fit(rows, dim)) return cudaErrorInvalidValue;
  const uint32_t nch = (uint32_t)(dim / 8);
  SwArgs a{static_cast<const uint16_t*>(gate), static_cast<const uint16_t*>(up), ld, rows, dim, nullptr, nullptr,
           nullptr, nullptr, (uint32_t)(rows * nch), make_inv_div(nch)};
  return launch_maybe_pdl(swiglu_values_kernel, dim3(sw_grid(swiglu_values_kernel, sms, a.items)), dim3(kSwThreads),
                          0, st, a, static_cast<uint16_t*>(out));
}

}  // namespace nvfp4ap
