// ln_blk2l.cu -- the two passes of the two-level NVFP4 contract on the
// block-per-lane kernel template (ln_blk.cuh): a clear of the caller's
// maximum word, the maximum pass (one atomic per CTA), the quantising pass;
// no modulation, broadcast bf16 or segmented modulation.
//
// Two-level NVFP4 (h3-blackwell-runtime compare page: NVFP4_STREAMING_DESIGN.md
// "Numerical Constraint" -- no block can be encoded before the whole tensor's
// maximum is known -- so two launches).  All three launches use programmatic
// serialisation: each may start while the previous drains, and each waits
// (griddepcontrol.wait) before it touches the word.
#include "ln_blk.cuh"

namespace nvfp4ap {
namespace {

// Clears the maximum word: waits for the previous kernel on the stream (which
// may still read the word) before writing it.
__global__ void blk_clear_word_kernel(unsigned int* w) {
  pdl_enter();
  *w = 0u;
}

template <int MOD>
cudaError_t run_blk_2level(const LnArgs& a, BlkShape s, int sms, cudaStream_t st) {
  cudaError_t e = launch_maybe_pdl(blk_clear_word_kernel, dim3(1), dim3(1), 0, st, a.amax_ws);
  if (e != cudaSuccess) return e;
  e = launch_blk_bpt<BK_AMAX, MOD>(a, s, sms, st);
  return e != cudaSuccess ? e : launch_blk_bpt<BK_NV2L, MOD>(a, s, sms, st);
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
