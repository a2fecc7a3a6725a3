// modulation6.cu -- six-way fp32 -> bf16 modulation producer for sm_103a.
//
// Operation (adaptive-layernorm-producers README, "Available Functions" and
// "Tensor Contract": adaln_modulation6_bf16): params (batch, seq, 6, dim)
// fp32 plus modulation (6, dim) fp32 give six bf16 (batch, seq, dim)
// tensors, out_i[b,s,:] = bf16(params[b,s,i,:] + modulation[i,:]) with one
// binary32 addition and round-to-nearest-even.
//
// Design: a pure stream (24 bytes read, 12 written per element of the six
// outputs' total).  The flattened params are cut into 8-element chunks (32
// bytes in, 16 bytes out); each thread issues the loads of U chunks before
// converting any, the modulation rows (6*dim*4 bytes, shared by every token)
// come through L1, outputs leave as 16-byte streaming stores.
#include "device.cuh"
#include "kernels.h"

namespace nvfp4ap {
namespace {

struct Outs {
  uint16_t* p[6];
};

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// grid.y = i (the output chunk), grid.x walks tokens x dim/8 chunks of it.
template <typename IDX>
__global__ void __launch_bounds__(kThreads) mod6_vec8_kernel(const float* __restrict__ params,
                                                             const float* __restrict__ modulation,
                                                             const __grid_constant__ Outs out, IDX nch,
                                                             IDX total, int64_t dim) {
  const int i = blockIdx.y;
  const IDX base = (IDX)blockIdx.x * (kThreads * kUnroll) + threadIdx.x;
  const float* pbase = params + (int64_t)i * dim;
  pdl_enter();
  uint4 p0[kUnroll], p1[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const IDX c = base + (IDX)u * kThreads;
    if (c < total) {
      const IDX tok = c / nch;
      const IDX d8 = c - tok * nch;
      const float* src = pbase + (int64_t)tok * 6 * dim + (int64_t)d8 * 8;
      p0[u] = ld_once_v4(src);
      p1[u] = ld_once_v4(src + 4);
    }
  }
  const float* mrow = modulation + (int64_t)i * dim;
  uint16_t* orow = out.p[i];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const IDX c = base + (IDX)u * kThreads;
    if (c >= total) continue;
    const IDX tok = c / nch;
    const IDX d8 = c - tok * nch;
    const float4 m0 = ld_reuse_f4(mrow + (int64_t)d8 * 8), m1 = ld_reuse_f4(mrow + (int64_t)d8 * 8 + 4);
    const float2 s0 = add2(make_float2(__uint_as_float(p0[u].x), __uint_as_float(p0[u].y)), make_float2(m0.x, m0.y));
    const float2 s1 = add2(make_float2(__uint_as_float(p0[u].z), __uint_as_float(p0[u].w)), make_float2(m0.z, m0.w));
    const float2 s2 = add2(make_float2(__uint_as_float(p1[u].x), __uint_as_float(p1[u].y)), make_float2(m1.x, m1.y));
    const float2 s3 = add2(make_float2(__uint_as_float(p1[u].z), __uint_as_float(p1[u].w)), make_float2(m1.z, m1.w));
    uint4 o;
    o.x = f2_to_bf16x2(s0);
    o.y = f2_to_bf16x2(s1);
    o.z = f2_to_bf16x2(s2);
    o.w = f2_to_bf16x2(s3);
    st_stream_v4(orow + (int64_t)tok * dim + (int64_t)d8 * 8, o);
  }
}

// Any dim and any (element-aligned) pointers: one element per thread step.
__global__ void __launch_bounds__(kThreads) mod6_scalar_kernel(const float* __restrict__ params,
                                                               const float* __restrict__ modulation,
                                                               const __grid_constant__ Outs out,
                                                               int64_t total, int64_t dim) {
  const int i = blockIdx.y;
  uint16_t* orow = out.p[i];
  for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * kThreads) {
    const int64_t tok = e / dim;
    const int64_t d = e - tok * dim;
    const float s = __fadd_rn(__ldg(params + (tok * 6 + i) * dim + d), __ldg(modulation + (int64_t)i * dim + d));
    orow[e] = f_to_bf16(s);
  }
}

}  // namespace

cudaError_t launch_modulation6(const Mod6Args& a, bool vec8, cudaStream_t st) {
  Outs o;
  for (int i = 0; i < 6; ++i) o.p[i] = a.out[i];
  if (vec8) {
    const int64_t nch = a.dim / 8;
    const int64_t total = a.tokens * nch;  // chunks of one output
    const int64_t per_cta = (int64_t)kThreads * kUnroll;
    const int64_t gx = (total + per_cta - 1) / per_cta;
    if (gx > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)gx, 6);
    if (total + per_cta < ((int64_t)1 << 31))
      return launch_maybe_pdl(mod6_vec8_kernel<uint32_t>, grid, dim3(kThreads), 0, st, a.params, a.modulation, o,
                              (uint32_t)nch, (uint32_t)total, a.dim);
    else
      return launch_maybe_pdl(mod6_vec8_kernel<uint64_t>, grid, dim3(kThreads), 0, st, a.params, a.modulation, o,
                              (uint64_t)nch, (uint64_t)total, a.dim);
  } else {
    const int64_t total = a.tokens * a.dim;  // elements of one output
    int64_t gx = (total + kThreads - 1) / kThreads;
    if (gx > 152 * 16) gx = 152 * 16;
    mod6_scalar_kernel<<<dim3((unsigned)gx, 6), kThreads, 0, st>>>(a.params, a.modulation, o, total, a.dim);
  }
  return cudaGetLastError();
}

}  // namespace nvfp4ap
