// ln_warpreg.cu -- warp-per-row producers that hold the whole row in
// registers: FP8 (no modulation, broadcast bf16, segmented) and the two-level
// NVFP4 maximum pass (the same sources).
//
// A warp takes whole rows; lane l owns the 16-element blocks l, l + 32, ...
// (BPL of them, BPL = ceil(blocks / 32), at most 12: dims up to 6144), reads
// each with one 256-bit non-allocating load, and keeps them as packed bf16.
// The row is read from HBM once: statistics from the registers (shifted
// one-pass sums, warp shuffles), then the codes (FP8) or the row's largest
// |bf16(y)| (two-level maximum pass, which also stores the row's K, mean - K
// and rstd for the flat quantising pass) from the same registers.  The
// two-sweep warp kernel (ln_blk.cuh) reads the row a second time from L2
// instead; both use the same fp32 operations in the same order, so their
// outputs are identical.  Modulation tables in shared memory as for the
// block-per-lane kernels (blk_tables); 512-thread CTAs, one per SM (the rows
// take up to 96 registers of a lane).
#include "ln_blk.cuh"

namespace nvfp4ap {
namespace {

constexpr int kWarpRegThreads = 512;

template <int KIND, int MOD, int BPL>
__global__ void __launch_bounds__(kWarpRegThreads, 1) warp_regs_kernel(const LnArgs a, const float inv_d) {
  extern __shared__ float4 gh[];
  __shared__ float redm[kWarpRegThreads / 32];
  const int lane = threadIdx.x & 31;
  const int64_t D = a.dim;
  const int nblk = (int)(D >> 4);
  pdl_enter();
  float inv_act = 1.0f;
  if constexpr (KIND == BK_FP8) inv_act = 1.0f / __ldg(a.act_scale);
  blk_tables<KIND, MOD>(a, gh, nblk, inv_act);

  float run = 0.0f;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < a.rows; row += nw) {
    const uint16_t* xr = a.x + row * D;
    uint32_t w[BPL][8];
#pragma unroll
    for (int k = 0; k < BPL; ++k) {
      if (lane + 32 * k < nblk) {
        ld_block(xr + (int64_t)(lane + 32 * k) * 16, w[k]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[k][i] = 0u;
      }
    }
    const float K = __uint_as_float((uint32_t)__ldg(xr) << 16);
    const float2 nk = splat2(-K);
    float2 s1 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < BPL; ++k) {
      if (lane + 32 * k < nblk) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 d = add2(bf16x2_to_f2(w[k][i]), nk);
          s1 = add2(s1, d);
          s2 = fma2(d, d, s2);
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
    if (KIND == BK_AMAX && lane == 0) reinterpret_cast<float4*>(a.row_stats)[row] = make_float4(K, m1, rstd, 0.f);
    const float4* tab = gh;
    if constexpr (MOD == MOD_SEG) {
      const int sg = __ldg(a.seg_idx + row);
      const bool ok = sg >= 0 && sg < a.nseg;
      if (!ok && lane == 0) atomicOr(&g_blk_seg_fault, 1u);
      tab = gh + (int64_t)(ok ? sg : a.nseg) * 8 * nblk;
    }
    const float A = (KIND == BK_FP8 && MOD == MOD_NONE) ? rstd * inv_act : rstd;
    const float2 A2 = splat2(A), B2 = splat2(-m1 * A);
#pragma unroll
    for (int k = 0; k < BPL; ++k) {
      const int b = lane + 32 * k;
      if (b >= nblk) continue;
      float2 y[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        y[i] = fma2(add2(bf16x2_to_f2(w[k][i]), nk), A2, B2);
        if constexpr (MOD != MOD_NONE) {
          const float4 G4 = tab[(i >> 1) * nblk + b], H4 = tab[(4 + (i >> 1)) * nblk + b];
          y[i] = (i & 1) ? fma2(y[i], make_float2(G4.z, G4.w), make_float2(H4.z, H4.w))
                         : fma2(y[i], make_float2(G4.x, G4.y), make_float2(H4.x, H4.y));
        }
      }
      if constexpr (KIND == BK_FP8) {
        uint32_t q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = f2_to_e4m3x2(y[i]);
        st_stream_v4(reinterpret_cast<uint8_t*>(a.out) + row * D + (int64_t)b * 16,
                     make_uint4(q[0] | (q[1] << 16), q[2] | (q[3] << 16), q[4] | (q[5] << 16), q[6] | (q[7] << 16)));
      } else {
        uint32_t vb[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) vb[i] = f2_to_bf16x2(y[i]);
        run = fmaxf(run, block_amax(vb));
      }
    }
  }
  if constexpr (KIND == BK_AMAX) {
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
}

template <int KIND, int MOD, int BPL>
cudaError_t launch_bpl(const LnArgs& a, int sms, int ctas_per_sm, cudaStream_t st) {
  auto k = warp_regs_kernel<KIND, MOD, BPL>;
  const int64_t smem64 = blk_tab_float4s(MOD, a.dim / 16, a.nseg) * (int64_t)sizeof(float4);
  if (smem64 > kBlkMaxSmem || !flat_smem_limit((const void*)k)) return cudaErrorInvalidValue;
  const int smem = (int)smem64;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kWarpRegThreads, smem) != cudaSuccess || occ < 1)
    return cudaErrorInvalidConfiguration;
  if (ctas_per_sm > 0 && ctas_per_sm < occ) occ = ctas_per_sm;
  int64_t grid = (int64_t)sms * occ;
  const int64_t need = (a.rows + kWarpRegThreads / 32 - 1) / (kWarpRegThreads / 32);
  if (grid > need) grid = need;
  const float inv_d = (float)(1.0 / (double)a.dim);
  return launch_maybe_pdl(k, dim3((unsigned)grid), dim3(kWarpRegThreads), (size_t)smem, st, a, inv_d);
}

template <int KIND, int MOD>
cudaError_t launch_kind_mod(const LnArgs& a, int sms, int ctas_per_sm, cudaStream_t st) {
  const int bpl = warp_regs_bpl(a.dim);
  switch (bpl) {
    case 6: return launch_bpl<KIND, MOD, 6>(a, sms, ctas_per_sm, st);
    case 8: return launch_bpl<KIND, MOD, 8>(a, sms, ctas_per_sm, st);
    case 11: return launch_bpl<KIND, MOD, 11>(a, sms, ctas_per_sm, st);
    case 12: return launch_bpl<KIND, MOD, 12>(a, sms, ctas_per_sm, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int warp_regs_bpl(int64_t dim) {
  if (dim % 16 != 0) return 0;
  const int64_t need = (dim / 16 + 31) / 32;
  for (int bpl : {6, 8, 11, 12})
    if (need <= bpl) return bpl;
  return 0;
}

bool warp_path_rows(int64_t rows, int64_t dim, int sms, bool regs) {
  const int64_t min_rows = (int64_t)sms * 32 * 4;
  return regs ? rows * dim >= min_rows * 3072 : rows >= min_rows;
}

// this translation unit's copy of the segment fault word (ln_blk.cuh), read and cleared
cudaError_t take_warpreg_seg_fault(unsigned int* fault) { return take_blk_word(fault); }

cudaError_t launch_warp_regs(const LnArgs& a, bool amax, int mod, int sms, int ctas_per_sm, cudaStream_t st) {
  if (amax) {
    switch (mod) {
      case MOD_NONE: return launch_kind_mod<BK_AMAX, MOD_NONE>(a, sms, ctas_per_sm, st);
      case MOD_BCAST: return launch_kind_mod<BK_AMAX, MOD_BCAST>(a, sms, ctas_per_sm, st);
      case MOD_SEG: return launch_kind_mod<BK_AMAX, MOD_SEG>(a, sms, ctas_per_sm, st);
      default: return cudaErrorInvalidValue;
    }
  }
  if (mod != MOD_SEG) return cudaErrorInvalidValue;
  return launch_kind_mod<BK_FP8, MOD_SEG>(a, sms, ctas_per_sm, st);
}

}  // namespace nvfp4ap
