// ln_twolevel.cu -- instances of the register-row kernel template
// (ln_rows.cuh) for the segmented modulation source and for the two passes
// of the two-level NVFP4 contract, and their launchers.
//
// Segmented modulation (h3-blackwell-runtime compare page: "segment-specific
// shift and scale selection", the request-layout segment index of the exact
// elementwise fusion phase): row r takes row seg_idx[r] of the (nseg, dim)
// scale/shift tables.
//
// Two-level NVFP4 (same page: NVFP4_STREAMING_DESIGN.md "Numerical
// Constraint" -- no block can be encoded before the whole tensor's maximum
// is known -- so two launches): the maximum pass writes the tensor's largest
// |v| to a caller-owned device word, the quantising pass derives the tensor
// scale from it and writes codes, block scales and the tensor scale.  The
// word is cleared first by a one-thread kernel.  All three launches use
// programmatic serialisation: each may start while the previous drains, and
// each waits (griddepcontrol.wait) before it touches the word.
#include "ln_rows.cuh"

namespace nvfp4ap {
namespace {

template <int KIND, int MOD>
cudaError_t launch_full(const LnArgs& a, RowShape s, bool pdl, cudaStream_t st) {
  if (s.tpr > 128 || (int64_t)s.tpr * s.per_thread * 8 != a.dim) return cudaErrorInvalidValue;
  const int64_t work_rows = KIND == KIND_AMAX ? a.rows : (a.rows + 127) / 128 * 128;
  const dim3 block(s.tpr, 1), grid((unsigned)work_rows);  // one row per CTA
  const float inv_d = (float)(1.0 / (double)a.dim);
  auto go = [&](auto k) -> cudaError_t {
    if (pdl) return launch_maybe_pdl(k, grid, block, 0, st, a, inv_d);
    k<<<grid, block, 0, st>>>(a, inv_d);
    return cudaGetLastError();
  };
  switch (s.per_thread) {
    case 2: return go(ln_rows_kernel<KIND, MOD, 2, kFullMinBlocks>);
    case 3: return go(ln_rows_kernel<KIND, MOD, 3, kFullMinBlocks>);
    case 4: return go(ln_rows_kernel<KIND, MOD, 4, kFullMinBlocks>);
    default: return cudaErrorInvalidValue;
  }
}

// Clears the maximum word: waits for the previous kernel on the stream (which
// may still read the word) before writing it.
__global__ void clear_word_kernel(unsigned int* w) {
  pdl_enter();
  *w = 0u;
}

template <int MOD>
cudaError_t run_2level(const LnArgs& a, RowShape s, bool full, cudaStream_t st) {
  cudaError_t e = launch_maybe_pdl(clear_word_kernel, dim3(1), dim3(1), 0, st, a.amax_ws);
  if (e != cudaSuccess) return e;
  if constexpr (MOD == MOD_NONE) {  // the modulated forms spill at the capped register count
    if (full) {
      e = launch_full<KIND_AMAX, MOD>(a, s, true, st);
      return e != cudaSuccess ? e : launch_full<KIND_NV2L, MOD>(a, s, true, st);
    }
  }
  e = launch_nv<KIND_AMAX, MOD>(a, s, st);
  return e != cudaSuccess ? e : launch_nv<KIND_NV2L, MOD>(a, s, st);
}

}  // namespace

cudaError_t launch_ln_seg(const LnArgs& a, bool nvfp4, RowShape s, cudaStream_t st) {
  return nvfp4 ? launch_nv<KIND_NVFP4, MOD_SEG>(a, s, st) : launch_nv<KIND_FP8, MOD_SEG>(a, s, st);
}

cudaError_t launch_ln_2level(const LnArgs& a, int mod, RowShape s, bool full, cudaStream_t st) {
  switch (mod) {
    case MOD_NONE: return run_2level<MOD_NONE>(a, s, full, st);
    case MOD_BCAST: return run_2level<MOD_BCAST>(a, s, full, st);
    case MOD_SEG: return run_2level<MOD_SEG>(a, s, false, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t take_seg_fault(unsigned int* fault) {
  unsigned int zero = 0u;
  cudaError_t e = cudaMemcpyFromSymbol(fault, g_seg_fault, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_seg_fault, &zero, sizeof(unsigned int));
}

}  // namespace nvfp4ap
