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
// word is cleared on the stream first.  The maximum pass is launched without
// programmatic serialisation, so it starts only after the clear; the
// quantising pass may overlap its ramp with the maximum pass's tail and waits
// (griddepcontrol.wait) before reading the word.
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
    case 2: return go(ln_rows_kernel<KIND, MOD, 2, false, kFullMinBlocks>);
    case 3: return go(ln_rows_kernel<KIND, MOD, 3, false, kFullMinBlocks>);
    case 4: return go(ln_rows_kernel<KIND, MOD, 4, false, kFullMinBlocks>);
    default: return cudaErrorInvalidValue;
  }
}

// the maximum pass without programmatic serialisation (it must follow the clear)
template <int MOD>
cudaError_t launch_amax_plain(const LnArgs& a, RowShape s, cudaStream_t st) {
  const dim3 block(s.tpr, s.rpc), grid((unsigned)((a.rows + s.rpc - 1) / s.rpc));
  const float inv_d = (float)(1.0 / (double)a.dim);
  constexpr bool kPerToken = false;  // the two-level sources (none, broadcast, segmented) keep no rows in registers
#define NVFP4AP_CASE(N)                                              \
  case N:                                                            \
    ln_rows_kernel<KIND_AMAX, MOD, N><<<grid, block, 0, st>>>(a, inv_d); \
    return cudaGetLastError();
  if constexpr (kPerToken) {
    switch (s.per_thread) {
      NVFP4AP_CASE(1)
      NVFP4AP_CASE(2)
      NVFP4AP_CASE(3)
      NVFP4AP_CASE(4)
      NVFP4AP_CASE(6)
      default: return cudaErrorInvalidValue;
    }
  } else {
    switch (s.per_thread) {
      NVFP4AP_CASE(1)
      NVFP4AP_CASE(2)
      NVFP4AP_CASE(3)
      NVFP4AP_CASE(4)
      NVFP4AP_CASE(6)
      NVFP4AP_CASE(8)
      NVFP4AP_CASE(12)
      default: return cudaErrorInvalidValue;
    }
  }
#undef NVFP4AP_CASE
}

template <int MOD>
cudaError_t run_2level(const LnArgs& a, RowShape s, bool full, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(a.amax_ws, 0, sizeof(unsigned int), st);
  if (e != cudaSuccess) return e;
  if constexpr (MOD == MOD_NONE) {  // the modulated forms spill at the capped register count
    if (full) {
      e = launch_full<KIND_AMAX, MOD>(a, s, false, st);
      return e != cudaSuccess ? e : launch_full<KIND_NV2L, MOD>(a, s, true, st);
    }
  }
  e = launch_amax_plain<MOD>(a, s, st);
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
