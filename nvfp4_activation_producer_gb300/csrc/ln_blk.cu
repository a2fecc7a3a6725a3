// ln_blk.cu -- instances of the block-per-lane kernel template (ln_blk.cuh)
// for the single-level producers: FP8 (no modulation, broadcast bf16, modfp8,
// AWQ, segmented) and NVFP4 (no modulation, broadcast bf16, modfp8,
// segmented), and the shape choice; the warp-per-row FP8 segmented kernel
// (two sweeps of each row) for many rows.
#include "ln_blk.cuh"

namespace nvfp4ap {

bool pick_blk(int64_t dim, int forced_bpt, BlkShape* s, bool fp8) {
  if (dim % 16 != 0) return false;
  const int64_t nblk = dim / 16;
  // 3 blocks (48 elements) per lane first; the fewest idle block slots wins.
  // FP8 takes 2 blocks per lane before 4 (measured on GB300 for the broadcast
  // sources: dim 4096, 4096 rows 37.5 -> 34.1 us for the three sources, dim
  // 2048 21.9 -> 20.9 us); the NVFP4 and two-level passes keep 4 before 2.
  static const int kPref[] = {3, 4, 2, 6};
  static const int kPrefFp8[] = {3, 2, 4, 6};
  const int* pref = fp8 ? kPrefFp8 : kPref;
  int best = -1;
  int64_t best_waste = 0;
  for (int j = 0; j < 4; ++j) {
    const int bpt = pref[j];
    if (forced_bpt > 0 && bpt != forced_bpt) continue;
    const int64_t tpr = ((nblk + bpt - 1) / bpt + 31) / 32 * 32;
    if (tpr > 256) continue;  // at most 8 warps per row, at least 2 rows per CTA
    const int64_t waste = tpr * bpt - nblk;
    if (best < 0 || waste < best_waste) {
      best = bpt;
      best_waste = waste;
      s->tpr = (int)tpr;
    }
  }
  if (best < 0) return false;
  s->bpt = best;
  s->ctas_per_sm = 0;
  s->warp = 0;
  return true;
}

bool blk_default_shape(int64_t dim, bool fp8, BlkShape* s) {
  if (!pick_blk(dim, 0, s, fp8)) return false;
  return (int64_t)s->tpr * s->bpt == dim / 16 && kBlkThreads / s->tpr >= 3;
}

bool ln_blk_supported(int kind, int mod, int64_t dim, int64_t nseg) {
  if (dim % 16 != 0 || dim > kBlkMaxDim) return false;
  if (mod == MOD_SEG && (nseg < 1 || blk_tab_float4s(MOD_SEG, dim / 16, nseg) * 16 > kBlkMaxSmem)) return false;
  switch (kind) {
    case BLK_FP8: return mod == MOD_NONE || mod == MOD_BCAST || mod == MOD_MODFP8 || mod == MOD_AWQ || mod == MOD_SEG;
    case BLK_NVFP4: return mod == MOD_NONE || mod == MOD_BCAST || mod == MOD_MODFP8 || mod == MOD_SEG;
    case BLK_2LEVEL: return mod == MOD_NONE || mod == MOD_BCAST || mod == MOD_SEG;
    default: return false;
  }
}

cudaError_t launch_ln_blk(const LnArgs& a, bool nvfp4, int mod, BlkShape s, int sms, cudaStream_t st) {
  if (nvfp4) {
    switch (mod) {
      case MOD_NONE: return launch_blk_bpt<BK_NVFP4, MOD_NONE>(a, s, sms, st);
      case MOD_BCAST: return launch_blk_bpt<BK_NVFP4, MOD_BCAST>(a, s, sms, st);
      case MOD_MODFP8: return launch_blk_bpt<BK_NVFP4, MOD_MODFP8>(a, s, sms, st);
      case MOD_SEG: return launch_blk_bpt<BK_NVFP4, MOD_SEG>(a, s, sms, st);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (mod) {
    case MOD_NONE: return launch_blk_bpt<BK_FP8, MOD_NONE>(a, s, sms, st);
    case MOD_BCAST: return launch_blk_bpt<BK_FP8, MOD_BCAST>(a, s, sms, st);
    case MOD_MODFP8: return launch_blk_bpt<BK_FP8, MOD_MODFP8>(a, s, sms, st);
    case MOD_AWQ: return launch_blk_bpt<BK_FP8, MOD_AWQ>(a, s, sms, st);
    case MOD_SEG: return launch_blk_bpt<BK_FP8, MOD_SEG>(a, s, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_ln_warp_rows_fp8(const LnArgs& a, int mod, int sms, int ctas_per_sm, cudaStream_t st) {
  if (mod != MOD_SEG) return cudaErrorInvalidValue;
  return launch_warp_rows<BK_FP8, MOD_SEG>(a, sms, ctas_per_sm, st);
}

cudaError_t take_blk_seg_fault(unsigned int* fault) { return take_blk_word(fault); }

}  // namespace nvfp4ap
