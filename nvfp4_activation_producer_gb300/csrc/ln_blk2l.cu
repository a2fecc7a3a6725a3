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

template <int MOD>
__global__ void __launch_bounds__(kFlatThreads, 1) flat_nv2l_kernel(const LnArgs a, const uint32_t items,
                                                                     const InvDiv per_row) {
  extern __shared__ float4 gh[];  // modulation tables, chunk-major (ln_blk.cuh)
  const int64_t D = a.dim;
  const int nblk = (int)(D >> 4), padc = (nblk + 3) & ~3, ct = padc >> 2;
  pdl_enter();

  blk_tables<BK_NV2L, MOD>(a, gh, nblk, 1.0f);

  const float ts = blk_round_bf16(__fdiv_rn(__uint_as_float(__ldcg(a.amax_ws)), 2688.0f));
  const float rts = __frcp_rn(ts);
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
    // (amax_b / 6) / ts, each quotient correctly rounded (two_level_quot),
    // clamped at 448 (fminf takes 448 for the 0/0 of an all-zero tensor); the
    // divisor of the codes is s * ts, exact in fp32
    const uint32_t sbyte = f2_to_e4m3x2(make_float2(fminf(two_level_quot(amax, ts, rts), 448.0f), 0.f)) & 0xFFu;
    uint32_t c0, c1;
    block_codes_2l(vb, e4m3_to_f32(sbyte) * ts, c0, c1);
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
  // maximum pass: warp per row for large tensors (warp_path_rows; s.warp = 1
  // forces it, -1 the row-group kernel), the row held in registers where a
  // lane's share fits, else two sweeps of each row
  const bool regs_ok = warp_regs_bpl(a.dim) > 0;
  const bool warp_rows = a.row_stats != nullptr &&
                         (s.warp > 0 || (s.warp == 0 && warp_path_rows(a.rows, a.dim, sms, regs_ok)));
  const bool regs = warp_rows && regs_ok;
  e = regs        ? launch_warp_regs(a, true, MOD, sms, s.ctas_per_sm, st)
      : warp_rows ? launch_warp_rows<BK_AMAX, MOD>(a, sms, s.ctas_per_sm, st)
                  : launch_blk_bpt<BK_AMAX, MOD>(a, s, sms, st);
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
