// ln_blk2l.cu -- the two passes of the two-level NVFP4 contract on the
// block-per-lane kernels: a clear of the caller's maximum word, the maximum
// pass (ln_blk.cuh: rows in register-held groups, one atomic per CTA), the
// quantising pass; no modulation, broadcast bf16 or segmented modulation.
//
// Two-level NVFP4 (h3-blackwell-runtime compare page: NVFP4_STREAMING_DESIGN.md
// "Numerical Constraint" -- no block can be encoded before the whole tensor's
// maximum is known -- so two launches).  All three launches use programmatic
// serialisation: each may start while the previous drains, and each waits
// (griddepcontrol.wait) before it touches the word.
//
// The maximum pass stores each row's K, mean - K and rstd in the caller's
// workspace: on register-held row groups (ln_blk.cuh), or, when the rows give
// every warp of the grid several, a warp per row with two sweeps of the row
// (below).  The quantising pass is then flat: the rows * nblk blocks are spread over a persistent grid in one
// grid-stride loop (row of block n by a multiply-high division), each lane
// reads its block, the row's statistics (L1: the lanes of a warp mostly share
// a row) and its segment, and encodes with the same fp32 operations as the
// maximum pass, so both passes see the same staged values.  Without row
// reductions, barriers or register-held rows it keeps 32 warps per SM.
#include "divide.cuh"
#include "ln_blk.cuh"

namespace nvfp4ap {
namespace {

constexpr int kFlatThreads = 1024;

// Clears the maximum word: waits for the previous kernel on the stream (which
// may still read the word) before writing it.
__global__ void blk_clear_word_kernel(unsigned int* w) {
  pdl_enter();
  *w = 0u;
}

// The modulation tables of the block-per-lane passes (G = 1 + scale, H = shift
// as fp32, chunk-major; segmented: one per segment plus the identity table),
// built by the CTA; ends with a barrier when there are tables.
template <int MOD>
__device__ __forceinline__ void flat_tables(const LnArgs& a, float4* gh, int nblk) {
  const int64_t D = a.dim;
  const float2 one4[4] = {splat2(1.0f), splat2(1.0f), splat2(1.0f), splat2(1.0f)};
  if constexpr (MOD == MOD_SEG) {
    const int nseg = (int)a.nseg;
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
      put_cols<BK_NV2L, MOD>(gh + (int64_t)sg * 8 * nblk, nblk, c8, sc, sh, one4);
    }
    __syncthreads();
  } else if constexpr (MOD == MOD_BCAST) {
    const float2 deq = source_deq<MOD>(a);
    for (int c8 = threadIdx.x; c8 < 2 * nblk; c8 += blockDim.x) {
      BcastCols<MOD, 8> bc;
      bc.load(a, (int64_t)c8 * 8);
      float2 sc[4], sh[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        sc[i] = bc.scale(i, deq);
        sh[i] = bc.shift(i, deq);
      }
      put_cols<BK_NV2L, MOD>(gh, nblk, c8, sc, sh, one4);
    }
    __syncthreads();
  }
}

template <int MOD>
__global__ void __launch_bounds__(kFlatThreads, 1) flat_nv2l_kernel(const LnArgs a, const uint32_t items,
                                                                     const InvDiv per_row) {
  extern __shared__ float4 gh[];  // modulation tables, chunk-major (ln_blk.cuh)
  const int64_t D = a.dim;
  const int nblk = (int)(D >> 4), padc = (nblk + 3) & ~3, ct = padc >> 2;
  pdl_enter();

  flat_tables<MOD>(a, gh, nblk);

  const float ts = blk_round_bf16(__fdiv_rn(__uint_as_float(__ldcg(a.amax_ws)), 2688.0f));
  if (blockIdx.x == 0 && threadIdx.x == 0) a.tensor_scale[0] = ts;
  const float4* stats = reinterpret_cast<const float4*>(a.row_stats);
  const uint32_t stride = gridDim.x * blockDim.x;
  for (uint32_t n = blockIdx.x * blockDim.x + threadIdx.x; n < items; n += stride) {
    const uint32_t r = inv_div(n, per_row), b = n - r * (uint32_t)nblk;
    const int64_t row = r;
    const float4 st = stats[r];  // K, mean - K, rstd
    const float4* tab = gh;
    if constexpr (MOD == MOD_SEG) {
      const int sg = __ldg(a.seg_idx + row);
      tab = gh + (int64_t)((sg >= 0 && sg < a.nseg) ? sg : a.nseg) * 8 * nblk;
    }
    uint32_t w[8];
    ld_block(a.x + row * D + (int64_t)b * 16, w);
    const float2 nk = splat2(-st.x), A2 = splat2(st.z), B2 = splat2(-st.y * st.z);
    uint32_t vb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float2 y = fma2(add2(bf16x2_to_f2(w[i]), nk), A2, B2);
      if constexpr (MOD != MOD_NONE) {
        const float4 G4 = tab[(i >> 1) * nblk + b], H4 = tab[(4 + (i >> 1)) * nblk + b];
        y = (i & 1) ? fma2(y, make_float2(G4.z, G4.w), make_float2(H4.z, H4.w))
                    : fma2(y, make_float2(G4.x, G4.y), make_float2(H4.x, H4.y));
      }
      vb[i] = f2_to_bf16x2(y);
    }
    const float amax = block_amax(vb);
    // (amax_b / 6) / ts with IEEE divisions, clamped at 448 (fminf takes 448
    // for the 0/0 of an all-zero tensor); the divisor of the codes is s * ts,
    // exact in fp32; a divisor below 2^-64 and the values are scaled by 2^64
    const uint32_t sbyte =
        f2_to_e4m3x2(make_float2(fminf(__fdiv_rn(__fdiv_rn(amax, 6.0f), ts), 448.0f), 0.f)) & 0xFFu;
    float scl = e4m3_to_f32(sbyte) * ts, pre = 1.0f;
    if (scl != 0.f && scl < 0x1p-64f) {
      scl *= 0x1p64f;
      pre = 0x1p64f;
    }
    uint32_t c0, c1;
    block_codes(vb, scl, pre, c0, c1);
    st_stream_v2(reinterpret_cast<uint8_t*>(a.out) + row * (D >> 1) + (int64_t)b * 8, c0, c1);
    st_b8(reinterpret_cast<uint8_t*>(a.sf) + ((row >> 7) * ct + (b >> 2)) * 512 + (int)((row & 31) << 4) +
              (int)(((row >> 5) & 3) << 2) + (b & 3),
          sbyte);
  }
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
    st_b8(reinterpret_cast<uint8_t*>(a.sf) + ((r >> 7) * ct + (b >> 2)) * 512 + (int)((r & 31) << 4) +
              (int)(((r >> 5) & 3) << 2) + (b & 3),
          0u);
  }
}

// 16 bf16 values (32 contiguous bytes), allocated in L1: the row is read twice
__device__ __forceinline__ void ld_block_l1(const uint16_t* p, uint32_t (&w)[8]) {
  asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "l"(p));
}

// Maximum pass for many rows per warp: each warp takes rows w, w + W, ... and
// sweeps a row twice -- the shifted sums (three 256-bit loads per lane in
// flight, allocated in L1), then the staged values' maximum from the blocks
// read again (L1 or L2) -- and stores the row's statistics for the flat
// quantising pass.  No row stays in registers and warps never wait on each
// other, so 32 warps per SM stream rows independently.  One atomic per CTA.
template <int MOD>
__global__ void __launch_bounds__(kFlatThreads, 1) warp_amax_kernel(const LnArgs a, const float inv_d) {
  extern __shared__ float4 gh[];
  __shared__ float redm[kFlatThreads / 32];
  const int lane = threadIdx.x & 31;
  const int64_t D = a.dim;
  const int nblk = (int)(D >> 4);
  pdl_enter();
  flat_tables<MOD>(a, gh, nblk);

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
    if (lane == 0) reinterpret_cast<float4*>(a.row_stats)[row] = make_float4(K, m1, rstd, 0.f);
    const float4* tab = gh;
    if constexpr (MOD == MOD_SEG) {
      const int sg = __ldg(a.seg_idx + row);
      const bool ok = sg >= 0 && sg < a.nseg;
      if (!ok && lane == 0) atomicOr(&g_blk_seg_fault, 1u);
      tab = gh + (int64_t)(ok ? sg : a.nseg) * 8 * nblk;
    }
    // the same fp32 operations as the quantising pass
    const float2 A2 = splat2(rstd), B2 = splat2(-m1 * rstd);
    for (int b = lane; b < nblk; b += 32) {
      uint32_t w[8], vb[8];
      ld_block_l1(xr + (int64_t)b * 16, w);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float2 y = fma2(add2(bf16x2_to_f2(w[i]), nk), A2, B2);
        if constexpr (MOD != MOD_NONE) {
          const float4 G4 = tab[(i >> 1) * nblk + b], H4 = tab[(4 + (i >> 1)) * nblk + b];
          y = (i & 1) ? fma2(y, make_float2(G4.z, G4.w), make_float2(H4.z, H4.w))
                      : fma2(y, make_float2(G4.x, G4.y), make_float2(H4.x, H4.y));
        }
        vb[i] = f2_to_bf16x2(y);
      }
      run = fmaxf(run, block_amax(vb));
    }
  }
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

// Dynamic-memory limit of a kernel raised once per device (keyed by the
// kernel itself: instances share their function-pointer type).
bool flat_smem_limit(const void* k) {
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

template <int MOD>
cudaError_t launch_warp_amax(const LnArgs& a, int sms, cudaStream_t st) {
  auto k = warp_amax_kernel<MOD>;
  const int64_t smem64 = blk_tab_float4s(MOD, a.dim / 16, a.nseg) * (int64_t)sizeof(float4);
  if (smem64 > kBlkMaxSmem || !flat_smem_limit((const void*)k)) return cudaErrorInvalidValue;
  const int smem = (int)smem64;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kFlatThreads, smem) != cudaSuccess || occ < 1)
    return cudaErrorInvalidConfiguration;
  int64_t grid = (int64_t)sms * occ;
  const int64_t need = (a.rows + kFlatThreads / 32 - 1) / (kFlatThreads / 32);
  if (grid > need) grid = need;
  const float inv_d = (float)(1.0 / (double)a.dim);
  return launch_maybe_pdl(k, dim3((unsigned)grid), dim3(kFlatThreads), (size_t)smem, st, a, inv_d);
}

template <int MOD>
cudaError_t launch_flat_nv2l(const LnArgs& a, int sms, cudaStream_t st) {
  auto k = flat_nv2l_kernel<MOD>;
  const int nblk = (int)(a.dim / 16);
  const int64_t smem64 = blk_tab_float4s(MOD, nblk, a.nseg) * (int64_t)sizeof(float4);
  if (smem64 > kBlkMaxSmem) return cudaErrorInvalidValue;
  const int smem = (int)smem64;
  if (!flat_smem_limit((const void*)k)) return cudaErrorInvalidConfiguration;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kFlatThreads, smem) != cudaSuccess || occ < 1)
    return cudaErrorInvalidConfiguration;
  const uint32_t items = (uint32_t)(a.rows * nblk);
  int64_t grid = (int64_t)sms * occ;
  const int64_t need = ((int64_t)items + kFlatThreads - 1) / kFlatThreads;
  if (grid > need) grid = need < 1 ? 1 : need;
  return launch_maybe_pdl(k, dim3((unsigned)grid), dim3(kFlatThreads), (size_t)smem, st, a, items,
                          make_inv_div((uint32_t)nblk));
}

template <int MOD>
cudaError_t run_blk_2level(const LnArgs& a, BlkShape s, int sms, cudaStream_t st) {
  cudaError_t e = launch_maybe_pdl(blk_clear_word_kernel, dim3(1), dim3(1), 0, st, a.amax_ws);
  if (e != cudaSuccess) return e;
  // maximum pass: warp per row when the rows give every warp of the grid
  // several (NVFP4AP_2L_AMAX=1 forces it, 2 the row-group kernel)
  const char* v = std::getenv("NVFP4AP_2L_AMAX");
  const int force = v ? std::atoi(v) : 0;
  const bool warp_rows = a.row_stats != nullptr &&
                         (force == 1 || (force == 0 && a.rows >= (int64_t)sms * (kFlatThreads / 32) * 4));
  e = warp_rows ? launch_warp_amax<MOD>(a, sms, st) : launch_blk_bpt<BK_AMAX, MOD>(a, s, sms, st);
  if (e != cudaSuccess) return e;
  // flat quantising pass when the statistics were kept and the block index
  // fits 32 bits; otherwise the row-group pass
  if (a.row_stats != nullptr && a.rows * (a.dim / 16) < ((int64_t)1 << 32)) return launch_flat_nv2l<MOD>(a, sms, st);
  return launch_blk_bpt<BK_NV2L, MOD>(a, s, sms, st);
}

}  // namespace

cudaError_t launch_ln_2level_blk(const LnArgs& a, int mod, BlkShape s, int sms, cudaStream_t st) {
  switch (mod) {
    case MOD_NONE: return run_blk_2level<MOD_NONE>(a, s, sms, st);
    case MOD_BCAST: return run_blk_2level<MOD_BCAST>(a, s, sms, st);
    case MOD_SEG: return run_blk_2level<MOD_SEG>(a, s, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t take_blk2l_seg_fault(unsigned int* fault) { return take_blk_word(fault); }

}  // namespace nvfp4ap
