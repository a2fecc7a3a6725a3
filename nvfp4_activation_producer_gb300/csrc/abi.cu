// abi.cu -- the C ABI of libnvfp4ap.so (declared in include/nvfp4ap.h).
//
// Each entry point checks its arguments on the host (shapes, dim rules,
// indices, pointer alignment, eps), picks the kernel variant and launch shape
// from dim, launches on the caller's stream and returns a status.  Nothing
// here allocates, synchronises or touches device memory.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include <cuda_runtime.h>
#include <unistd.h>

#include "kernels.h"
#include "nvfp4ap.h"

#define NVFP4AP_EXPORT extern "C" __attribute__((visibility("default")))

namespace nvfp4ap {
namespace {

inline bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

// Rows from which the block-per-lane persistent kernel is the default: the FP8
// broadcast sources, and the single-level NVFP4 forms whose row does not fit
// the one-row-per-CTA kernel (see run_fp8 and run_nvfp4 for the measurements).
constexpr int64_t kBlkBcastRows = 4096;
constexpr int64_t kBlkNvfp4Rows = 2048;

int env_int(const char* name) {
  const char* v = env_get(name);
  return v ? std::atoi(v) : 0;
}

// true when the variable is set to 0 (a default-on choice switched off)
bool env_off(const char* name) {
  const char* v = env_get(name);
  return v && v[0] == '0';
}

// Launch shape for a row of `nvec` units (vectors or blocks): the candidate
// per-thread counts are tried in order of preference and the one that wastes
// the fewest thread slots (tpr * per_thread - nvec, tpr a multiple of 32 not
// above the instance's limit) wins; ties keep the earlier candidate.
// `forced` (> 0) restricts the choice to that per-thread count when it fits.
template <typename MaxTpr>
bool pick_shape(int64_t nvec, const int* cands, int ncand, MaxTpr max_tpr, int forced, RowShape* out) {
  int64_t best_waste = -1;
  for (int i = 0; i < ncand; ++i) {
    const int nv = cands[i];
    if (forced > 0 && nv != forced) continue;
    const int lim = max_tpr(nv);
    if (lim <= 0) continue;
    int64_t tpr = (nvec + nv - 1) / nv;
    tpr = (tpr + 31) / 32 * 32;
    if (tpr > lim) continue;
    const int64_t waste = tpr * nv - nvec;
    if (best_waste < 0 || waste < best_waste) {
      best_waste = waste;
      out->tpr = (int)tpr;
      out->per_thread = nv;
    }
  }
  if (best_waste < 0) return false;
  out->rpc = out->tpr >= 128 ? 1 : 128 / out->tpr;
  return true;
}

bool grid_ok(int64_t rows, int rpc) { return (rows + rpc - 1) / rpc <= 0x7FFFFFFF; }

// Multiprocessor count of the current device (cached per device ordinal).
int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < 64) cache[dev] = n;
  return n;
}

// Shape of the TMA ring kernel for a row of `dim`: 8 warps per CTA and as
// many stages (up to 4) as fit a budget of ~110 KB of shared memory per CTA,
// so that two CTAs share an SM; fewer warps with one stage when a stage is
// large.  Returns false when not even one warp with one stage fits (227 KB).
bool pick_ring(int mod, int64_t dim, RingShape* rs) {
  const int64_t budget = (env_int("NVFP4AP_RING_SMEM_KB") > 0 ? env_int("NVFP4AP_RING_SMEM_KB") : 110) * 1024;
  int warps = env_int("NVFP4AP_RING_WARPS") > 0 ? env_int("NVFP4AP_RING_WARPS") : 8;
  if (warps > 16) warps = 16;
  int stages = env_int("NVFP4AP_RING_STAGES");
  rs->ctas_per_sm = env_int("NVFP4AP_RING_CTAS");
  if (stages <= 0) {
    stages = 4;
    while (stages > 1 && ring_smem_bytes(mod, dim, warps, stages) > budget) --stages;
    while (warps > 1 && ring_smem_bytes(mod, dim, warps, stages) > budget) --warps;
  }
  if (stages > 8) stages = 8;
  if (ring_smem_bytes(mod, dim, warps, stages) > 227 * 1024) return false;
  rs->warps = warps;
  rs->stages = stages;
  return true;
}

// Shape of the register row kernel: 8-element chunks per thread from a
// preference list (3 first: 24 elements per thread measured fastest on
// GB300 at dim 1536-3072), the first that wastes the fewest thread slots;
// up to 96 elements per thread for one input row, 48 for the per-token forms
// (three input rows in registers).  Rows per CTA fill 128 threads
// (NVFP4AP_ROWS_PER_CTA overrides).
bool pick_rows(int mod, int64_t dim, RowShape* s) {
  static const int kWide[] = {3, 4, 6, 2, 8, 12, 1};
  static const int kToken[] = {3, 4, 2, 6, 1};
  const bool per_token = (mod == MOD_PTOK || mod == MOD_TABLE);
  const int* c = per_token ? kToken : kWide;
  const int n = per_token ? 5 : 7;
  auto lim = [mod](int nv) { return ln_rows_max_tpr(mod, nv); };
  if (!pick_shape(dim / 8, c, n, lim, env_int("NVFP4AP_PER_THREAD"), s) && !pick_shape(dim / 8, c, n, lim, 0, s))
    return false;
  const int want = env_int("NVFP4AP_ROWS_PER_CTA");
  if (want > 0 && want <= 16 && want * s->tpr <= 512) s->rpc = want;  // the kernels are bounded to 512 threads
  return true;
}

// The persistent broadcast kernel takes one row per CTA of at most 256
// threads and up to 6 chunks per thread (NVFP4AP_PERSIST=0 turns it off).
bool persist_ok(const RowShape& s) {
  if (env_int("NVFP4AP_PERSIST") < 0) return false;
  const bool nv_ok = s.per_thread == 1 || s.per_thread == 2 || s.per_thread == 3 || s.per_thread == 4 ||
                     s.per_thread == 6;
  return nv_ok && s.tpr <= 256 && s.rpc == 1;
}

int finish(cudaError_t e) {
  if (e == cudaSuccess) return NVFP4AP_OK;
  if (env_int("NVFP4AP_DEBUG") > 0) std::fprintf(stderr, "nvfp4ap: launch failed: %s\n", cudaGetErrorString(e));
  (void)cudaGetLastError();
  return NVFP4AP_ERR_LAUNCH;
}

// The element-wise kernel (ln_scalar.cu) for pointers that are only
// element-aligned: bf16 tensors at 2 bytes, fp32 tables and scalars at 4,
// e4m3 and output bytes at 1 (the tensor contract asks for contiguity only).
// NVFP4AP_ERR_ALIGN when even that does not hold.
int run_scalar(const LnArgs& a, bool nvfp4, int mod, cudaStream_t st) {
  const void* bf[] = {a.x, a.scale, a.shift, a.temb, a.inv_s, a.seg_scale, a.seg_shift};
  for (const void* p : bf)
    if (p && !aligned(p, 2)) return NVFP4AP_ERR_ALIGN;
  const void* f32[] = {a.table, a.act_scale, a.scale_deq, a.shift_deq, a.seg_idx};
  for (const void* p : f32)
    if (p && !aligned(p, 4)) return NVFP4AP_ERR_ALIGN;
  const int64_t work = nvfp4 ? (a.rows + 127) / 128 * 128 : a.rows;
  if (!grid_ok(work, 1)) return NVFP4AP_ERR_SHAPE;
  return finish(launch_ln_scalar(a, nvfp4, mod, st));
}

int check_common(int64_t rows, int64_t dim, float eps) {
  if (rows < 0 || dim <= 0) return NVFP4AP_ERR_SHAPE;
  if (dim > NVFP4AP_MAX_DIM) return NVFP4AP_ERR_DIM;
  if (!std::isfinite(eps) || eps < 0.f) return NVFP4AP_ERR_VALUE;
  return NVFP4AP_OK;
}

// The modfp8 source: non-null e4m3 vectors and fp32 scalars; the scalars
// 4-byte aligned.
int check_modfp8(const LnArgs& a) {
  if (!a.scale8 || !a.shift8 || !a.scale_deq || !a.shift_deq) return NVFP4AP_ERR_NULL;
  if (!aligned(a.scale_deq, 4) || !aligned(a.shift_deq, 4)) return NVFP4AP_ERR_ALIGN;
  return NVFP4AP_OK;
}

// FP8 family: validation shared by every modulation source, then variant +
// shape + launch.
int run_fp8(LnArgs& a, int mod, cudaStream_t st) {
  int rc = check_common(a.rows, a.dim, a.eps);
  if (rc) return rc;
  if (a.dim % 2 != 0) return NVFP4AP_ERR_DIM;
  if (mod == MOD_TABLE && (a.chunks < 1 || a.shift_idx < 0 || a.shift_idx >= a.chunks ||
                           a.scale_idx < 0 || a.scale_idx >= a.chunks))
    return NVFP4AP_ERR_INDEX;
  if (a.rows == 0) return NVFP4AP_OK;
  if (!a.x || !a.out || !a.act_scale) return NVFP4AP_ERR_NULL;
  if ((mod == MOD_BCAST || mod == MOD_PTOK || mod == MOD_AWQ) && (!a.scale || !a.shift)) return NVFP4AP_ERR_NULL;
  if (mod == MOD_AWQ && !a.inv_s) return NVFP4AP_ERR_NULL;
  if (mod == MOD_TABLE && (!a.temb || !a.table)) return NVFP4AP_ERR_NULL;
  if (mod == MOD_MODFP8 && (rc = check_modfp8(a)) != NVFP4AP_OK) return rc;
  if (!aligned(a.act_scale, 4)) return NVFP4AP_ERR_ALIGN;

  // 16-byte vector path or bf16-pair path
  const void* bf_in[4] = {a.x, nullptr, nullptr, nullptr};
  if (mod == MOD_BCAST || mod == MOD_PTOK || mod == MOD_AWQ) { bf_in[1] = a.scale; bf_in[2] = a.shift; }
  if (mod == MOD_AWQ) bf_in[3] = a.inv_s;
  if (mod == MOD_TABLE) bf_in[1] = a.temb;
  bool vec8 = (a.dim % 8 == 0) && aligned(a.out, 8) && (mod != MOD_TABLE || aligned(a.table, 16));
  bool pair_ok = aligned(a.out, 2) && (mod != MOD_TABLE || aligned(a.table, 8));
  if (mod == MOD_MODFP8) {
    // e4m3 vectors: 8 bytes per 8-column chunk, 2 bytes per pair
    vec8 = vec8 && aligned(a.scale8, 8) && aligned(a.shift8, 8);
    pair_ok = pair_ok && aligned(a.scale8, 2) && aligned(a.shift8, 2);
  }
  for (const void* p : bf_in) {
    if (!p) continue;
    vec8 = vec8 && aligned(p, 16);
    pair_ok = pair_ok && aligned(p, 4);
  }
  if (!vec8 && !pair_ok) return run_scalar(a, false, mod, st);
  const int vec = vec8 ? 8 : 2;

  // NVFP4AP_KERNEL: 0 auto (below), 1 warp-per-row TMA ring, 2 first register
  // kernel, 3 register row kernels for every form, 4 TMA pipeline for every
  // form, 5 block-per-lane persistent kernel, 8 one-row-per-CTA block-per-lane
  // kernel.  The ring and TMA kernels have no modfp8 / AWQ source: those run
  // on the register kernels.
  int kernel = env_int("NVFP4AP_KERNEL");
  // default: the one-row-per-CTA block-per-lane kernel for the layer norm
  // form where the row fits it exactly (measured on GB300: 4096x3072 7.9 ->
  // 7.55 us), the TMA pipeline for the table form; for the three broadcast
  // sources (bf16, modfp8, AWQ: one rule, so that they reduce to each other
  // bit for bit) the block-per-lane persistent kernel from kBlkBcastRows rows
  // where its shape has no idle lane and three or more rows per CTA, else the
  // persistent broadcast kernel.  Measured on GB300 (graphs of 32 calls),
  // sum over the three sources: 3072 x 4096 rows 28.2 -> 27.1 us, x 32768
  // 177.7 -> 143.4 us; 1536 x 32768 100.1 -> 76.0 us; 6144 x 32768 351 ->
  // 290 us; below 4096 rows the persistent kernel is as fast or faster
  // (3072 x 2520: 20.3 against 21.1 us).
  if (kernel == 0) {
    BlkShape bs{};
    if (mod_is_bcast(mod) && a.rows >= kBlkBcastRows && vec8 && ln_blk_supported(BLK_FP8, mod, a.dim, 0) &&
        aligned(a.x, 32) && aligned(a.out, 16) && blk_default_shape(a.dim, true, &bs))
      kernel = 5;
    else
      kernel = (mod == MOD_NONE) ? 8 : (mod == MOD_TABLE) ? 4 : 3;
  }
  if (kernel == 1 && (mod == MOD_MODFP8 || mod == MOD_AWQ)) kernel = 3;
  if (kernel == 8) {
    // one-row-per-CTA block-per-lane kernel where the row fits it exactly
    // (the default for the layer norm form, see above), else the other defaults
    RbShape rb{};
    if (vec8 && (mod == MOD_NONE || mod_is_bcast(mod)) && aligned(a.x, 32) && aligned(a.out, 16) &&
        pick_rowblk(a.dim, env_int("NVFP4AP_RB_BPT"), &rb))
      return finish(launch_ln_rowblk(a, false, mod, rb, st));
    kernel = (mod == MOD_TABLE) ? 4 : 3;
  }
  if (kernel == 5) {
    // block-per-lane persistent kernel where it applies, else the default
    if (vec8 && ln_blk_supported(BLK_FP8, mod, a.dim, 0) && aligned(a.x, 32) && aligned(a.out, 16)) {
      BlkShape bs{};
      const int sms = sm_count();
      if (sms > 0 && pick_blk(a.dim, env_int("NVFP4AP_BLK_BPT"), &bs, true)) {
        bs.ctas_per_sm = env_int("NVFP4AP_BLK_CTAS");
        bs.max_ctas = env_int("NVFP4AP_BLK_GRID");
        return finish(launch_ln_blk(a, false, mod, bs, sms, st));
      }
    }
    kernel = (mod == MOD_TABLE) ? 4 : 3;
  }
  if (kernel == 6) {
    // warp-per-row kernel (two sweeps of each row) where it applies, else the default
    if (vec8 && (mod == MOD_NONE || mod == MOD_BCAST) && ln_blk_supported(BLK_FP8, mod, a.dim, 0) &&
        aligned(a.x, 32) && aligned(a.out, 16)) {
      const int sms = sm_count();
      if (sms > 0 && !env_off("NVFP4AP_WARPREG") && warp_regs_bpl(a.dim) > 0)
        return finish(launch_warp_regs(a, false, mod, sms, st));
      if (sms > 0) return finish(launch_ln_warp_rows_fp8(a, mod, sms, st));
    }
    kernel = (mod == MOD_TABLE) ? 4 : 3;
  }
  RingShape rs{};
  if (vec8 && kernel == 1 && pick_ring(mod, a.dim, &rs)) {
    const int sms = sm_count();
    if (sms > 0) return finish(launch_ln_ring(a, false, mod, rs, sms, wait_limit_cycles(), st));
  }
  RowShape rows_shape{};
  if (vec8 && (kernel == 3 || kernel == 4) && pick_rows(mod, a.dim, &rows_shape)) {
    if (!grid_ok(a.rows, rows_shape.rpc)) return NVFP4AP_ERR_SHAPE;
    const int sms = sm_count();
    if (kernel == 4 && sms > 0 && ln_tma_supported(false, mod, rows_shape))
      return finish(launch_ln_tma(a, false, mod, rows_shape, sms, env_int("NVFP4AP_TMA_STAGES"),
                                  env_int("NVFP4AP_TMA_CTAS"), wait_limit_cycles(), st));
    if (mod_is_bcast(mod) && persist_ok(rows_shape) && sms > 0)
      return finish(
          launch_ln_bcast_persistent(a, false, mod, rows_shape, sms, env_int("NVFP4AP_PERSIST_CTAS"), st));
    return finish(launch_ln_rows(a, false, mod, rows_shape, st));
  }

  static const int kVec8[] = {3, 4, 2, 6, 8, 1};
  static const int kVec2[] = {8, 4, 16, 2, 32};
  RowShape s{};
  const bool ok = vec8 ? pick_shape(a.dim / 8, kVec8, 6, [](int nv) { return ln_fp8_max_tpr(8, nv); },
                                    env_int("NVFP4AP_FP8_PER_THREAD"), &s)
                       : pick_shape(a.dim / 2, kVec2, 5, [](int nv) { return ln_fp8_max_tpr(2, nv); },
                                    env_int("NVFP4AP_FP8_PER_THREAD"), &s);
  if (!ok) {
    // a forced per-thread count that does not fit: fall back to the default choice
    if (!(vec8 ? pick_shape(a.dim / 8, kVec8, 6, [](int nv) { return ln_fp8_max_tpr(8, nv); }, 0, &s)
               : pick_shape(a.dim / 2, kVec2, 5, [](int nv) { return ln_fp8_max_tpr(2, nv); }, 0, &s)))
      return NVFP4AP_ERR_DIM;
  }
  if (!grid_ok(a.rows, s.rpc)) return NVFP4AP_ERR_SHAPE;
  return finish(launch_ln_fp8(a, mod, vec, s, st));
}

// Segmented modulation: index and tables present and aligned.
int check_seg(const LnArgs& a) {
  if (!a.seg_idx || !a.seg_scale || !a.seg_shift) return NVFP4AP_ERR_NULL;
  if (a.nseg < 1) return NVFP4AP_ERR_INDEX;
  if (!aligned(a.seg_idx, 4)) return NVFP4AP_ERR_ALIGN;
  return NVFP4AP_OK;
}

// Segmented modulation producers (FP8 and single-level NVFP4) on the register
// row kernels: dim % 8 (FP8) or % 16 (NVFP4), 16-byte aligned x and outputs.
int run_seg(LnArgs& a, bool nvfp4, cudaStream_t st) {
  int rc = check_common(a.rows, a.dim, a.eps);
  if (rc) return rc;
  if (a.dim % (nvfp4 ? 16 : 2) != 0) return NVFP4AP_ERR_DIM;
  if (a.rows == 0) return NVFP4AP_OK;
  if (!a.x || !a.out || (nvfp4 ? !a.sf : !a.act_scale)) return NVFP4AP_ERR_NULL;
  if ((rc = check_seg(a)) != NVFP4AP_OK) return rc;
  if (!nvfp4 && !aligned(a.act_scale, 4)) return NVFP4AP_ERR_ALIGN;
  // vector kernels: dim % 8, 16-byte aligned x and tables, 8-byte aligned
  // output; anything else takes the element-wise kernel
  if (a.dim % 8 != 0 || !aligned(a.x, 16) || !aligned(a.out, 8) || !aligned(a.seg_scale, 16) ||
      !aligned(a.seg_shift, 16))
    return run_scalar(a, nvfp4, MOD_SEG, st);
  if (env_int("NVFP4AP_KERNEL") == 5 && ln_blk_supported(nvfp4 ? BLK_NVFP4 : BLK_FP8, MOD_SEG, a.dim, a.nseg) &&
      aligned(a.x, 32) && aligned(a.out, 16)) {
    BlkShape bs{};
    const int sms = sm_count();
    if (sms > 0 && pick_blk(a.dim, env_int("NVFP4AP_BLK_BPT"), &bs, !nvfp4)) {
      bs.max_ctas = env_int("NVFP4AP_BLK_GRID");
      return finish(launch_ln_blk(a, nvfp4, MOD_SEG, bs, sms, st));
    }
  }
  // FP8, many rows: the warp-per-row kernel (NVFP4AP_SEG_WARP=1 forces it,
  // -1 turns it off)
  if (!nvfp4 && env_int("NVFP4AP_KERNEL") != 5 && env_int("NVFP4AP_SEG_WARP") >= 0 &&
      ln_blk_supported(BLK_FP8, MOD_SEG, a.dim, a.nseg) && aligned(a.x, 32) && aligned(a.out, 16)) {
    const int sms = sm_count();
    // the row held in registers where a lane's share fits (NVFP4AP_WARPREG=0:
    // the two-sweep kernel; measured on GB300 at 37810x5376: 119.7 -> 101.1 us)
    const bool regs = !env_off("NVFP4AP_WARPREG") && warp_regs_bpl(a.dim) > 0;
    if (sms > 0 && (env_int("NVFP4AP_SEG_WARP") > 0 || warp_path_rows(a.rows, a.dim, sms, regs))) {
      if (regs) return finish(launch_warp_regs(a, false, MOD_SEG, sms, st));
      return finish(launch_ln_warp_rows_fp8(a, MOD_SEG, sms, st));
    }
  }
  RowShape s{};
  if (!pick_rows(MOD_SEG, a.dim, &s)) return NVFP4AP_ERR_DIM;
  const int64_t work = nvfp4 ? (a.rows + 127) / 128 * 128 : a.rows;
  if (!grid_ok(work, s.rpc)) return NVFP4AP_ERR_SHAPE;
  return finish(launch_ln_seg(a, nvfp4, s, st));
}

// Two-level NVFP4 producers: as the NVFP4 producers, plus a 4-byte aligned
// tensor-scale output and workspace word.
int run_2level(LnArgs& a, int mod, cudaStream_t st) {
  int rc = check_common(a.rows, a.dim, a.eps);
  if (rc) return rc;
  if (a.dim % 16 != 0) return NVFP4AP_ERR_DIM;
  if (a.rows == 0) return NVFP4AP_OK;
  if (!a.x || !a.out || !a.sf || !a.tensor_scale || !a.amax_ws) return NVFP4AP_ERR_NULL;
  if (mod == MOD_BCAST && (!a.scale || !a.shift)) return NVFP4AP_ERR_NULL;
  if (mod == MOD_SEG && (rc = check_seg(a)) != NVFP4AP_OK) return rc;
  if (mod == MOD_SEG && (!aligned(a.seg_scale, 16) || !aligned(a.seg_shift, 16))) return NVFP4AP_ERR_ALIGN;
  if (!aligned(a.x, 16) || !aligned(a.out, 8) || !aligned(a.tensor_scale, 4) || !aligned(a.amax_ws, 16))
    return NVFP4AP_ERR_ALIGN;
  // the workspace's statistics slots follow the word (16 bytes in)
  a.row_stats = reinterpret_cast<float*>(reinterpret_cast<char*>(a.amax_ws) + 16);
  if (mod == MOD_BCAST && (!aligned(a.scale, 16) || !aligned(a.shift, 16))) return NVFP4AP_ERR_ALIGN;
  // default (and NVFP4AP_KERNEL=5): the block-per-lane kernels -- persistent,
  // one atomic per CTA in the maximum pass -- where they apply (measured on
  // GB300: 37810x5376 segmented 341 -> 284 us, 5070x3072 20.9 -> 18.5 us);
  // any other NVFP4AP_KERNEL value, or a shape they do not take: the register
  // row kernels
  const int kernel = env_int("NVFP4AP_KERNEL");
  if ((kernel == 0 || kernel == 5) && ln_blk_supported(BLK_2LEVEL, mod, a.dim, a.nseg) && aligned(a.x, 32)) {
    BlkShape bs{};
    const int sms = sm_count();
    if (sms > 0 && pick_blk(a.dim, env_int("NVFP4AP_BLK_BPT"), &bs)) {
      bs.max_ctas = env_int("NVFP4AP_BLK_GRID");
      return finish(launch_ln_2level_blk(a, mod, bs, sms, st));
    }
  }
  RowShape s{};
  if (!pick_rows(mod, a.dim, &s)) return NVFP4AP_ERR_DIM;
  if (!grid_ok((a.rows + 127) / 128 * 128, s.rpc)) return NVFP4AP_ERR_SHAPE;
  // the register-capped instances for rows that exactly fill the CTA's
  // chunks (NVFP4AP_FULL=0 turns them off); unmodulated rows only -- the
  // broadcast instances spill at 40 registers
  const bool full = !env_off("NVFP4AP_FULL") && mod == MOD_NONE && s.tpr <= 128 && s.per_thread >= 2 &&
                    s.per_thread <= 4 && (int64_t)s.tpr * s.per_thread * 8 == a.dim;
  return finish(launch_ln_2level(a, mod, s, full, st));
}

int run_nvfp4(LnArgs& a, int mod, cudaStream_t st) {
  int rc = check_common(a.rows, a.dim, a.eps);
  if (rc) return rc;
  if (a.dim % 16 != 0) return NVFP4AP_ERR_DIM;
  if (a.rows == 0) return NVFP4AP_OK;
  if (!a.x || !a.out || !a.sf) return NVFP4AP_ERR_NULL;
  if (mod == MOD_BCAST && (!a.scale || !a.shift)) return NVFP4AP_ERR_NULL;
  if (mod == MOD_MODFP8 && (rc = check_modfp8(a)) != NVFP4AP_OK) return rc;
  // vector kernels: 16-byte aligned x and bf16 vectors, 8-byte aligned packed
  // output and e4m3 vectors; anything else takes the element-wise kernel
  if (!aligned(a.x, 16) || !aligned(a.out, 8) ||
      (mod == MOD_BCAST && (!aligned(a.scale, 16) || !aligned(a.shift, 16))) ||
      (mod == MOD_MODFP8 && (!aligned(a.scale8, 8) || !aligned(a.shift8, 8))))
    return run_scalar(a, true, mod, st);

  int kernel = env_int("NVFP4AP_KERNEL");  // as for FP8, 8: one-row-per-CTA block-per-lane kernels
  // default: the one-row-per-CTA block-per-lane kernel where the row fits it
  // exactly (measured faster than the register row and persistent kernels on
  // GB300 at dims 2048-8192, 2,520-32,768 rows: 5070x3072 layer norm 10.0 ->
  // 8.5 us, broadcast 12.2 -> 10.6 us); where it does not, the block-per-lane
  // persistent kernel from kBlkNvfp4Rows rows when its shape has no idle lane
  // and three or more rows per CTA (dims 1024, 1536, 5120; measured at
  // 2,520-32,768 rows: faster at every size, 1536 x 32768 layer norm 33.4 ->
  // 22.2 us, broadcast 36.8 -> 28.3 us, 5120 x 4096 broadcast 20.1 -> 16.0
  // us), else the register row kernels
  const bool blk_ok = ln_blk_supported(BLK_NVFP4, mod, a.dim, 0) && aligned(a.x, 32);
  if (kernel == 0 || kernel == 8) {
    RbShape rb{};
    if ((mod == MOD_NONE || mod == MOD_BCAST || mod == MOD_MODFP8) && aligned(a.x, 32) &&
        pick_rowblk(a.dim, env_int("NVFP4AP_RB_BPT"), &rb))
      return finish(launch_ln_rowblk(a, true, mod, rb, st));
    BlkShape bs{};
    kernel = (kernel == 0 && a.rows >= kBlkNvfp4Rows && blk_ok && blk_default_shape(a.dim, false, &bs)) ? 5 : 3;
  }
  if (kernel == 5) {
    if (blk_ok) {
      BlkShape bs{};
      const int sms = sm_count();
      if (sms > 0 && pick_blk(a.dim, env_int("NVFP4AP_BLK_BPT"), &bs)) {
        bs.ctas_per_sm = env_int("NVFP4AP_BLK_CTAS");
        bs.max_ctas = env_int("NVFP4AP_BLK_GRID");
        return finish(launch_ln_blk(a, true, mod, bs, sms, st));
      }
    }
    kernel = 3;
  }
  // the modfp8 source runs on the register kernels only
  if (mod == MOD_MODFP8 && kernel != 3 && kernel != 4) kernel = 3;
  RingShape rs{};
  if (kernel == 1 && pick_ring(mod, a.dim, &rs)) {
    const int sms = sm_count();
    if (sms > 0) return finish(launch_ln_ring(a, true, mod, rs, sms, wait_limit_cycles(), st));
  }
  RowShape rows_shape{};
  if ((kernel == 3 || kernel == 4) && pick_rows(mod, a.dim, &rows_shape)) {
    const int64_t rows_pad = (a.rows + 127) / 128 * 128;
    if (!grid_ok(rows_pad, rows_shape.rpc)) return NVFP4AP_ERR_SHAPE;
    const int sms = sm_count();
    if (kernel == 4 && sms > 0 && ln_tma_supported(true, mod, rows_shape))
      return finish(launch_ln_tma(a, true, mod, rows_shape, sms, env_int("NVFP4AP_TMA_STAGES"),
                                  env_int("NVFP4AP_TMA_CTAS"), wait_limit_cycles(), st));
    // four rows of a scale tile per CTA (whole 16-byte scale chunks): opt-in
    // with NVFP4AP_TILE4=1 -- measured slower on GB300 than one row per CTA
    const bool tile4 = env_int("NVFP4AP_TILE4") > 0 && rows_shape.tpr <= 128 && rows_shape.per_thread <= 4 &&
                       aligned(a.sf, 16) && (mod == MOD_NONE || mod == MOD_BCAST);
    if (mod_is_bcast(mod) && persist_ok(rows_shape) && sms > 0 && !tile4)
      return finish(
          launch_ln_bcast_persistent(a, true, mod, rows_shape, sms, env_int("NVFP4AP_PERSIST_CTAS"), st));
    if (tile4) return finish(launch_ln_rows_tile4(a, mod, rows_shape, st));
    // rows that exactly fill the CTA's chunks: the register-capped instance
    // (NVFP4AP_FULL=0 turns it off)
    if (!env_off("NVFP4AP_FULL") && rows_shape.tpr <= 128 && rows_shape.per_thread >= 2 && rows_shape.per_thread <= 4 &&
        (int64_t)rows_shape.tpr * rows_shape.per_thread * 8 == a.dim)
      return finish(launch_ln_rows_full(a, true, mod, rows_shape, st));
    return finish(launch_ln_rows(a, true, mod, rows_shape, st));
  }

  static const int kCands[] = {2, 3, 1, 4, 6};
  RowShape s{};
  if (!pick_shape(a.dim / 16, kCands, 5, [](int b) { return ln_nvfp4_max_tpr(b); },
                  env_int("NVFP4AP_NVFP4_PER_THREAD"), &s) &&
      !pick_shape(a.dim / 16, kCands, 5, [](int b) { return ln_nvfp4_max_tpr(b); }, 0, &s))
    return NVFP4AP_ERR_DIM;
  const int64_t rows_pad = (a.rows + 127) / 128 * 128;
  if (!grid_ok(rows_pad, s.rpc)) return NVFP4AP_ERR_SHAPE;
  return finish(launch_ln_nvfp4(a, mod, s, st));
}

LnArgs ln_args(const void* x, float eps, void* out, int64_t rows, int64_t dim) {
  LnArgs a{};
  a.x = static_cast<const uint16_t*>(x);
  a.eps = eps;
  a.out = out;
  a.rows = rows;
  a.dim = dim;
  return a;
}

}  // namespace

// Bound of the TMA kernels' mbarrier waits (SM clock cycles); 0 = the
// default, about one second at 2 GHz.
namespace {
constexpr long long kDefaultWaitCycles = 2000000000LL;
std::atomic<long long> g_wait_limit{0};
}  // namespace

long long wait_limit_cycles() {
  const long long v = g_wait_limit.load(std::memory_order_relaxed);
  return v > 0 ? v : kDefaultWaitCycles;
}

bool pdl_enabled() {
  const char* v = env_get("NVFP4AP_PDL");
  return !(v && v[0] == '0');
}

// The NVFP4AP_* settings of this thread's current call: one pass over the
// environment per producer call (env_refresh, first thing in every producer
// entry point) keeps the entries that start with NVFP4AP_; env_get then reads
// those.  Each getenv is a scan of the whole environment (eight of them took
// 1.9 us on an x86 host with 114 variables), the pass about a tenth of that,
// and a setting changed between calls is still seen by the next call.
namespace {
struct EnvSnap {
  int n;
  const char* kv[64];
};
thread_local EnvSnap g_env = {0, {}};
}  // namespace

void env_refresh() {
  int n = 0;
  for (char** e = environ; e != nullptr && *e != nullptr; ++e) {
    const char* kv = *e;
    if (kv[0] == 'N' && std::strncmp(kv, "NVFP4AP_", 8) == 0 && n < 64) g_env.kv[n++] = kv;
  }
  g_env.n = n;
}

const char* env_get(const char* name) {
  const size_t len = std::strlen(name);
  for (int i = 0; i < g_env.n; ++i) {
    const char* kv = g_env.kv[i];
    if (std::strncmp(kv, name, len) == 0 && kv[len] == '=') return kv + len + 1;
  }
  return nullptr;
}

}  // namespace nvfp4ap

using namespace nvfp4ap;

NVFP4AP_EXPORT const char* nvfp4ap_status_string(int status) {
  switch (status) {
    case NVFP4AP_OK: return "ok";
    case NVFP4AP_ERR_NULL: return "a required pointer is NULL";
    case NVFP4AP_ERR_SHAPE: return "invalid shape (negative rows/batch/seq, dim <= 0, or grid too large)";
    case NVFP4AP_ERR_DIM: return "dim violates the op's rule (FP8: even; NVFP4: multiple of 16; <= NVFP4AP_MAX_DIM)";
    case NVFP4AP_ERR_INDEX: return "chunks < 1 or shift_idx/scale_idx out of range";
    case NVFP4AP_ERR_ALIGN: return "a pointer misses its alignment rule";
    case NVFP4AP_ERR_LAUNCH: return "CUDA launch failed";
    case NVFP4AP_ERR_VALUE: return "eps is negative or not finite";
    case NVFP4AP_ERR_TIMEOUT:
      return "a kernel's bounded wait ran out: its output is incomplete (read by nvfp4ap_take_device_fault)";
    case NVFP4AP_ERR_FAULT:
      return "a segment index was outside [0, nseg): that row was produced with zero modulation";
    case NVFP4AP_ERR_SCRATCH: return "the call needs more per-CTA words than the library's static scratch array holds";
    default: return "unknown status";
  }
}

NVFP4AP_EXPORT int nvfp4ap_version(void) { return 100; }

NVFP4AP_EXPORT int nvfp4ap_take_device_fault(void) {
  // wait words (ring and TMA kernels), then the segment-index words
  unsigned int f = 0u, g = 0u, h = 0u, i = 0u, j = 0u, k = 0u, l = 0u;
  if (take_ring_fault(&f) != cudaSuccess || take_tma_fault(&g) != cudaSuccess || take_seg_fault(&h) != cudaSuccess ||
      take_blk_seg_fault(&i) != cudaSuccess || take_blk2l_seg_fault(&j) != cudaSuccess ||
      take_warpreg_seg_fault(&k) != cudaSuccess || take_scalar_seg_fault(&l) != cudaSuccess) {
    (void)cudaGetLastError();
    return NVFP4AP_ERR_LAUNCH;
  }
  if (f | g) return NVFP4AP_ERR_TIMEOUT;
  return (h | i | j | k | l) ? NVFP4AP_ERR_FAULT : NVFP4AP_OK;
}

NVFP4AP_EXPORT int nvfp4ap_set_wait_limit(int64_t cycles) {
  g_wait_limit.store(cycles > 0 ? (long long)cycles : 0LL, std::memory_order_relaxed);
  return NVFP4AP_OK;
}

NVFP4AP_EXPORT int64_t nvfp4ap_wait_limit(void) { return (int64_t)wait_limit_cycles(); }

NVFP4AP_EXPORT int nvfp4ap_noalloc_progress(uint32_t* words, int64_t n, int64_t* used) {
  return noalloc_progress(words, n, used);
}

NVFP4AP_EXPORT int ada_layer_norm_quant_fp8_bf16(const void* x, const void* scale, const void* shift,
                                                 const float* act_scale, float eps, void* out, int64_t rows,
                                                 int64_t dim, nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, out, rows, dim);
  a.scale = static_cast<const uint16_t*>(scale);
  a.shift = static_cast<const uint16_t*>(shift);
  a.act_scale = act_scale;
  return run_fp8(a, MOD_BCAST, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int ada_layer_norm_quant_fp8_bf16_noalloc(const void* x, const void* scale, const void* shift,
                                                         const float* act_scale, float eps, void* out,
                                                         int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  env_refresh();
  int rc = check_common(rows, dim, eps);
  if (rc) return rc;
  if (dim % 8 != 0) return NVFP4AP_ERR_DIM;
  if (rows == 0) return NVFP4AP_OK;
  if (!x || !scale || !shift || !act_scale || !out) return NVFP4AP_ERR_NULL;
  if (!aligned(x, 16) || !aligned(scale, 16) || !aligned(shift, 16) || !aligned(out, 8) || !aligned(act_scale, 4))
    return NVFP4AP_ERR_ALIGN;
  const int sms = sm_count();
  if (sms <= 0) return NVFP4AP_ERR_LAUNCH;
  LnArgs a = ln_args(x, eps, out, rows, dim);
  a.scale = static_cast<const uint16_t*>(scale);
  a.shift = static_cast<const uint16_t*>(shift);
  a.act_scale = act_scale;
  rc = noalloc_fp8_bcast(a, sms, wait_limit_cycles(), reinterpret_cast<cudaStream_t>(stream));
  if (rc == NVFP4AP_ERR_LAUNCH) (void)cudaGetLastError();
  return rc;
}

NVFP4AP_EXPORT int ada_layer_norm_quant_fp8_ptok_bf16(const void* x, const void* scale, const void* shift,
                                                      const float* act_scale, float eps, void* out,
                                                      int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, out, rows, dim);
  a.scale = static_cast<const uint16_t*>(scale);
  a.shift = static_cast<const uint16_t*>(shift);
  a.act_scale = act_scale;
  return run_fp8(a, MOD_PTOK, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int ada_layer_norm_quant_fp8_ptok_table_bf16(const void* x, const void* temb, const float* table,
                                                            int64_t chunks, int64_t shift_idx, int64_t scale_idx,
                                                            const float* act_scale, float eps, void* out,
                                                            int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, out, rows, dim);
  a.temb = static_cast<const uint16_t*>(temb);
  a.table = table;
  a.chunks = chunks;
  a.shift_idx = shift_idx;
  a.scale_idx = scale_idx;
  a.act_scale = act_scale;
  return run_fp8(a, MOD_TABLE, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int ada_layer_norm_quant_fp8_modfp8_bf16(const void* x, const void* scale_fp8, const void* shift_fp8,
                                                        const float* scale_deq, const float* shift_deq,
                                                        const float* act_scale, float eps, void* out, int64_t rows,
                                                        int64_t dim, nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, out, rows, dim);
  a.scale8 = static_cast<const uint8_t*>(scale_fp8);
  a.shift8 = static_cast<const uint8_t*>(shift_fp8);
  a.scale_deq = scale_deq;
  a.shift_deq = shift_deq;
  a.act_scale = act_scale;
  return run_fp8(a, MOD_MODFP8, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int awq_ada_layer_norm_quant_fp8_bf16(const void* x, const void* scale, const void* shift,
                                                     const void* inv_s, const float* act_scale, float eps, void* out,
                                                     int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, out, rows, dim);
  a.scale = static_cast<const uint16_t*>(scale);
  a.shift = static_cast<const uint16_t*>(shift);
  a.inv_s = static_cast<const uint16_t*>(inv_s);
  a.act_scale = act_scale;
  return run_fp8(a, MOD_AWQ, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int layer_norm_no_affine_quant_fp8_static_bf16(const void* x, const float* act_scale, float eps,
                                                              void* out, int64_t rows, int64_t dim,
                                                              nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, out, rows, dim);
  a.act_scale = act_scale;
  return run_fp8(a, MOD_NONE, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int ada_layer_norm_quant_nvfp4_swizzled_bf16(const void* x, const void* scale, const void* shift,
                                                            float eps, void* packed, void* sf_swizzled,
                                                            int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, packed, rows, dim);
  a.scale = static_cast<const uint16_t*>(scale);
  a.shift = static_cast<const uint16_t*>(shift);
  a.sf = sf_swizzled;
  return run_nvfp4(a, MOD_BCAST, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(const void* x, const void* scale_fp8,
                                                                   const void* shift_fp8, const float* scale_deq,
                                                                   const float* shift_deq, float eps, void* packed,
                                                                   void* sf_swizzled, int64_t rows, int64_t dim,
                                                                   nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, packed, rows, dim);
  a.scale8 = static_cast<const uint8_t*>(scale_fp8);
  a.shift8 = static_cast<const uint8_t*>(shift_fp8);
  a.scale_deq = scale_deq;
  a.shift_deq = shift_deq;
  a.sf = sf_swizzled;
  return run_nvfp4(a, MOD_MODFP8, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int layer_norm_no_affine_quant_nvfp4_swizzled_bf16(const void* x, float eps, void* packed,
                                                                  void* sf_swizzled, int64_t rows, int64_t dim,
                                                                  nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, packed, rows, dim);
  a.sf = sf_swizzled;
  return run_nvfp4(a, MOD_NONE, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int ada_layer_norm_quant_fp8_seg_bf16(const void* x, const int32_t* seg_idx, const void* seg_scale,
                                                     const void* seg_shift, int64_t nseg, const float* act_scale,
                                                     float eps, void* out, int64_t rows, int64_t dim,
                                                     nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, out, rows, dim);
  a.seg_idx = seg_idx;
  a.seg_scale = static_cast<const uint16_t*>(seg_scale);
  a.seg_shift = static_cast<const uint16_t*>(seg_shift);
  a.nseg = nseg;
  a.act_scale = act_scale;
  return run_seg(a, false, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int ada_layer_norm_quant_nvfp4_swizzled_seg_bf16(const void* x, const int32_t* seg_idx,
                                                                const void* seg_scale, const void* seg_shift,
                                                                int64_t nseg, float eps, void* packed,
                                                                void* sf_swizzled, int64_t rows, int64_t dim,
                                                                nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, packed, rows, dim);
  a.seg_idx = seg_idx;
  a.seg_scale = static_cast<const uint16_t*>(seg_scale);
  a.seg_shift = static_cast<const uint16_t*>(seg_shift);
  a.nseg = nseg;
  a.sf = sf_swizzled;
  return run_seg(a, true, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int layer_norm_no_affine_quant_nvfp4_2level_bf16(const void* x, float eps, void* packed,
                                                                void* sf_swizzled, float* tensor_scale,
                                                                void* workspace, int64_t rows, int64_t dim,
                                                                nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, packed, rows, dim);
  a.sf = sf_swizzled;
  a.tensor_scale = tensor_scale;
  a.amax_ws = static_cast<unsigned int*>(workspace);
  return run_2level(a, MOD_NONE, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int ada_layer_norm_quant_nvfp4_2level_bf16(const void* x, const void* scale, const void* shift,
                                                          float eps, void* packed, void* sf_swizzled,
                                                          float* tensor_scale, void* workspace, int64_t rows,
                                                          int64_t dim, nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, packed, rows, dim);
  a.scale = static_cast<const uint16_t*>(scale);
  a.shift = static_cast<const uint16_t*>(shift);
  a.sf = sf_swizzled;
  a.tensor_scale = tensor_scale;
  a.amax_ws = static_cast<unsigned int*>(workspace);
  return run_2level(a, MOD_BCAST, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int ada_layer_norm_quant_nvfp4_2level_seg_bf16(const void* x, const int32_t* seg_idx,
                                                              const void* seg_scale, const void* seg_shift,
                                                              int64_t nseg, float eps, void* packed,
                                                              void* sf_swizzled, float* tensor_scale,
                                                              void* workspace, int64_t rows, int64_t dim,
                                                              nvfp4ap_stream_t stream) {
  env_refresh();
  LnArgs a = ln_args(x, eps, packed, rows, dim);
  a.seg_idx = seg_idx;
  a.seg_scale = static_cast<const uint16_t*>(seg_scale);
  a.seg_shift = static_cast<const uint16_t*>(seg_shift);
  a.nseg = nseg;
  a.sf = sf_swizzled;
  a.tensor_scale = tensor_scale;
  a.amax_ws = static_cast<unsigned int*>(workspace);
  return run_2level(a, MOD_SEG, reinterpret_cast<cudaStream_t>(stream));
}

NVFP4AP_EXPORT int swiglu_quant_nvfp4_2level_bf16(const void* gate, const void* up, int64_t ld, void* packed,
                                                  void* sf_swizzled, float* tensor_scale, void* workspace,
                                                  int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  env_refresh();
  if (rows < 0 || dim <= 0) return NVFP4AP_ERR_SHAPE;
  if (dim > NVFP4AP_MAX_DIM || dim % 16 != 0) return NVFP4AP_ERR_DIM;
  if (ld < dim || ld % 8 != 0 || !swiglu_items_fit(rows, dim)) return NVFP4AP_ERR_SHAPE;
  if (rows == 0) return NVFP4AP_OK;
  if (!gate || !up || !packed || !sf_swizzled || !tensor_scale || !workspace) return NVFP4AP_ERR_NULL;
  if (!aligned(gate, 16) || !aligned(up, 16) || !aligned(packed, 8) || !aligned(tensor_scale, 4) ||
      !aligned(workspace, 4))
    return NVFP4AP_ERR_ALIGN;
  const int sms = sm_count();
  if (sms <= 0) return NVFP4AP_ERR_LAUNCH;
  return finish(launch_swiglu_2level(gate, up, ld, rows, dim, packed, sf_swizzled, tensor_scale,
                                     static_cast<unsigned int*>(workspace), sms,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

NVFP4AP_EXPORT int swiglu_bf16(const void* gate, const void* up, int64_t ld, void* out, int64_t rows, int64_t dim,
                               nvfp4ap_stream_t stream) {
  env_refresh();
  if (rows < 0 || dim <= 0) return NVFP4AP_ERR_SHAPE;
  if (dim > NVFP4AP_MAX_DIM || dim % 8 != 0) return NVFP4AP_ERR_DIM;
  if (ld < dim || ld % 8 != 0 || !swiglu_items_fit(rows, dim)) return NVFP4AP_ERR_SHAPE;
  if (rows == 0) return NVFP4AP_OK;
  if (!gate || !up || !out) return NVFP4AP_ERR_NULL;
  if (!aligned(gate, 16) || !aligned(up, 16) || !aligned(out, 16)) return NVFP4AP_ERR_ALIGN;
  const int sms = sm_count();
  if (sms <= 0) return NVFP4AP_ERR_LAUNCH;
  return finish(launch_swiglu_values(gate, up, ld, rows, dim, out, sms, reinterpret_cast<cudaStream_t>(stream)));
}

NVFP4AP_EXPORT int64_t nvfp4ap_2level_workspace_bytes(int64_t rows) {
  if (rows < 0 || rows > (INT64_MAX - 16) / 16) return -1;
  return NVFP4AP_2LEVEL_WORKSPACE_BYTES(rows);
}

NVFP4AP_EXPORT int64_t swizzled_sf_size(int64_t rows, int64_t dim) {
  if (rows < 0 || dim <= 0 || dim % 16 != 0) return -1;
  const int64_t rows_pad = (rows + 127) / 128 * 128;
  const int64_t cols_pad = (dim / 16 + 3) / 4 * 4;
  return rows_pad * cols_pad;
}

NVFP4AP_EXPORT int adaln_modulation6_bf16(const float* params, const float* modulation, void* const out[6],
                                          int64_t batch, int64_t seq, int64_t dim, nvfp4ap_stream_t stream) {
  env_refresh();
  if (batch < 0 || seq < 0 || dim <= 0) return NVFP4AP_ERR_SHAPE;
  if (seq != 0 && batch > INT64_MAX / seq) return NVFP4AP_ERR_SHAPE;
  const int64_t tokens = batch * seq;
  if (tokens == 0) return NVFP4AP_OK;
  if (!params || !modulation || !out) return NVFP4AP_ERR_NULL;
  Mod6Args a{};
  a.params = params;
  a.modulation = modulation;
  a.tokens = tokens;
  a.dim = dim;
  bool vec8 = (dim % 8 == 0) && aligned(params, 16) && aligned(modulation, 16);
  bool natural = aligned(params, 4) && aligned(modulation, 4);
  for (int i = 0; i < 6; ++i) {
    if (!out[i]) return NVFP4AP_ERR_NULL;
    a.out[i] = static_cast<uint16_t*>(out[i]);
    vec8 = vec8 && aligned(out[i], 16);
    natural = natural && aligned(out[i], 2);
  }
  if (!natural) return NVFP4AP_ERR_ALIGN;
  return finish(launch_modulation6(a, vec8, reinterpret_cast<cudaStream_t>(stream)));
}
