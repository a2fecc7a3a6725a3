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

// Kernel families a call may be forced onto (NVFP4AP_KERNEL=F[:C]), for tests
// that cover each family's instances; every family meets the same output
// contract.  C caps the resident CTAs per SM of the persistent kernels, so a
// small problem still walks many rows through each CTA.
enum Family { FAM_AUTO = 0, FAM_ROWS = 3, FAM_TMA = 4, FAM_BLK = 5, FAM_WARP = 6, FAM_ROWBLK = 8 };
struct Force {
  int family, ctas;
};
Force forced() {
  Force f{FAM_AUTO, 0};
  const char* v = env_get("NVFP4AP_KERNEL");
  if (!v) return f;
  char* end = nullptr;
  const long fam = std::strtol(v, &end, 10);
  if (fam == FAM_ROWS || fam == FAM_TMA || fam == FAM_BLK || fam == FAM_WARP || fam == FAM_ROWBLK) f.family = (int)fam;
  if (end && *end == ':') {
    const long c = std::strtol(end + 1, nullptr, 10);
    if (c > 0 && c < 64) f.ctas = (int)c;
  }
  return f;
}

bool debug_on() {
  const char* v = env_get("NVFP4AP_DEBUG");
  return v && v[0] == '1';
}

// Launch shape for a row of `nvec` units (vectors or blocks): the candidate
// per-thread counts are tried in order of preference and the one that wastes
// the fewest thread slots (tpr * per_thread - nvec, tpr a multiple of 32 not
// above the instance's limit) wins; ties keep the earlier candidate.
template <typename MaxTpr>
bool pick_shape(int64_t nvec, const int* cands, int ncand, MaxTpr max_tpr, RowShape* out) {
  int64_t best_waste = -1;
  for (int i = 0; i < ncand; ++i) {
    const int nv = cands[i];
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

// Shape of the register row kernel: 8-element chunks per thread from a
// preference list (3 first: 24 elements per thread measured fastest on
// GB300 at dim 1536-3072), the first that wastes the fewest thread slots;
// up to 96 elements per thread for one input row, 48 for the per-token forms
// (three input rows in registers).  Rows per CTA fill 128 threads.
bool pick_rows(int mod, int64_t dim, RowShape* s) {
  static const int kWide[] = {3, 4, 6, 2, 8, 12, 1};
  static const int kToken[] = {3, 4, 2, 6, 1};
  const bool per_token = (mod == MOD_PTOK || mod == MOD_TABLE);
  const int* c = per_token ? kToken : kWide;
  const int n = per_token ? 5 : 7;
  return pick_shape(dim / 8, c, n, [mod](int nv) { return ln_rows_max_tpr(mod, nv); }, s);
}

// The persistent broadcast kernel takes one row per CTA of at most 256
// threads and 1, 2, 3, 4 or 6 chunks per thread.
bool persist_ok(const RowShape& s) {
  const bool nv_ok = s.per_thread == 1 || s.per_thread == 2 || s.per_thread == 3 || s.per_thread == 4 ||
                     s.per_thread == 6;
  return nv_ok && s.tpr <= 256 && s.rpc == 1;
}

int finish(cudaError_t e) {
  if (e == cudaSuccess) return NVFP4AP_OK;
  if (debug_on()) std::fprintf(stderr, "nvfp4ap: launch failed: %s\n", cudaGetErrorString(e));
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

// The register row kernels: the persistent broadcast kernel for the broadcast
// sources where its shape applies, the register-capped FULL instance for NVFP4
// rows that exactly fill the CTA's chunks, else the flat row kernel.
int run_rows(const LnArgs& a, bool nvfp4, int mod, const RowShape& rs, int ctas, cudaStream_t st) {
  const int64_t work = nvfp4 ? (a.rows + 127) / 128 * 128 : a.rows;
  if (!grid_ok(work, rs.rpc)) return NVFP4AP_ERR_SHAPE;
  const int sms = sm_count();
  if (mod_is_bcast(mod) && persist_ok(rs) && sms > 0)
    return finish(launch_ln_bcast_persistent(a, nvfp4, mod, rs, sms, ctas, st));
  if (nvfp4 && rs.tpr <= 128 && rs.per_thread >= 2 && rs.per_thread <= 4 &&
      (int64_t)rs.tpr * rs.per_thread * 8 == a.dim)
    return finish(launch_ln_rows_full(a, true, mod, rs, st));
  return finish(launch_ln_rows(a, nvfp4, mod, rs, st));
}

// FP8 family: validation shared by every modulation source, then the kernel
// and its shape.
//
// Default kernels (measured on GB300, graphs of 32 calls over rotating
// buffers): the layer norm form on the one-row-per-CTA block-per-lane kernel
// where the row fits it exactly (4096x3072 7.9 -> 7.55 us); the table form on
// the TMA pipeline (16.1 against 17.4 us for the register row kernel at
// 4096x3072); the three broadcast sources (bf16, modfp8, AWQ: one rule, so
// that they reduce to each other bit for bit) on the block-per-lane
// persistent kernel from kBlkBcastRows rows where its shape has no idle lane
// and three or more rows per CTA (3072 x 4096 rows 28.2 -> 27.1 us for the
// three sources, x 32768 177.7 -> 143.4 us; 1536 x 32768 100.1 -> 76.0 us;
// 6144 x 32768 351 -> 290 us), else the persistent broadcast kernel (as fast
// or faster below 4096 rows: 3072 x 2520 20.3 against 21.1 us); the
// per-token form on the register row kernels.
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

  // 16-byte vector kernels, bf16-pair kernel, or the element-wise kernel
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

  const Force f = forced();
  if (vec8) {
    const int sms = sm_count();
    int fam = f.family;
    if (fam == FAM_AUTO) {
      BlkShape bs{};
      if (mod_is_bcast(mod) && a.rows >= kBlkBcastRows && ln_blk_supported(BLK_FP8, mod, a.dim, 0) &&
          aligned(a.x, 32) && aligned(a.out, 16) && blk_default_shape(a.dim, true, &bs))
        fam = FAM_BLK;
      else
        fam = (mod == MOD_NONE) ? FAM_ROWBLK : (mod == MOD_TABLE) ? FAM_TMA : FAM_ROWS;
    }
    if (fam == FAM_ROWBLK) {
      RbShape rb{};
      if ((mod == MOD_NONE || mod_is_bcast(mod)) && aligned(a.x, 32) && aligned(a.out, 16) &&
          pick_rowblk(a.dim, 0, &rb, mod == MOD_NONE))
        return finish(launch_ln_rowblk(a, false, mod, rb, st));
    }
    if (fam == FAM_BLK && sms > 0 && ln_blk_supported(BLK_FP8, mod, a.dim, 0) && aligned(a.x, 32) &&
        aligned(a.out, 16)) {
      BlkShape bs{};
      if (pick_blk(a.dim, 0, &bs, true)) {
        bs.ctas_per_sm = f.ctas;
        return finish(launch_ln_blk(a, false, mod, bs, sms, st));
      }
    }
    RowShape rs{};
    if (pick_rows(mod, a.dim, &rs)) {
      if ((fam == FAM_TMA || mod == MOD_TABLE) && fam != FAM_ROWS && sms > 0 && ln_tma_supported(false, mod, rs))
        return finish(launch_ln_tma(a, false, mod, rs, sms, 0, f.ctas, wait_limit_cycles(), st));
      return run_rows(a, false, mod, rs, f.ctas, st);
    }
    // rows too long for the register row kernels (per-token dims above 24576):
    // the bf16-pair kernel below
  }
  static const int kVec2[] = {8, 4, 16, 2, 32};
  RowShape s{};
  if (!pick_shape(a.dim / 2, kVec2, 5, [](int nv) { return ln_fp8_max_tpr(2, nv); }, &s)) return NVFP4AP_ERR_DIM;
  if (!grid_ok(a.rows, s.rpc)) return NVFP4AP_ERR_SHAPE;
  return finish(launch_ln_fp8(a, mod, 2, s, st));
}

// Segmented modulation: index present and aligned, at least one segment.
int check_seg(const LnArgs& a) {
  if (!a.seg_idx || !a.seg_scale || !a.seg_shift) return NVFP4AP_ERR_NULL;
  if (a.nseg < 1) return NVFP4AP_ERR_INDEX;
  if (!aligned(a.seg_idx, 4)) return NVFP4AP_ERR_ALIGN;
  return NVFP4AP_OK;
}

// Segmented modulation producers (FP8 and single-level NVFP4).  Default: for
// FP8 on many rows the warp-per-row kernels (the row held in registers where a
// lane's share fits, measured on GB300 at 37810x5376: 119.7 -> 101.1 us),
// else the register row kernels.
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
  const Force f = forced();
  const int sms = sm_count();
  if (f.family == FAM_BLK && sms > 0 && ln_blk_supported(nvfp4 ? BLK_NVFP4 : BLK_FP8, MOD_SEG, a.dim, a.nseg) &&
      aligned(a.x, 32) && aligned(a.out, 16)) {
    BlkShape bs{};
    if (pick_blk(a.dim, 0, &bs, !nvfp4)) {
      bs.ctas_per_sm = f.ctas;
      return finish(launch_ln_blk(a, nvfp4, MOD_SEG, bs, sms, st));
    }
  }
  if (!nvfp4 && (f.family == FAM_AUTO || f.family == FAM_WARP) && sms > 0 &&
      ln_blk_supported(BLK_FP8, MOD_SEG, a.dim, a.nseg) && aligned(a.x, 32) && aligned(a.out, 16)) {
    const bool regs = warp_regs_bpl(a.dim) > 0;
    if (f.family == FAM_WARP || warp_path_rows(a.rows, a.dim, sms, regs)) {
      if (regs) return finish(launch_warp_regs(a, false, MOD_SEG, sms, f.ctas, st));
      return finish(launch_ln_warp_rows_fp8(a, MOD_SEG, sms, f.ctas, st));
    }
  }
  RowShape s{};
  if (!pick_rows(MOD_SEG, a.dim, &s)) return run_scalar(a, nvfp4, MOD_SEG, st);
  const int64_t work = nvfp4 ? (a.rows + 127) / 128 * 128 : a.rows;
  if (!grid_ok(work, s.rpc)) return NVFP4AP_ERR_SHAPE;
  return finish(launch_ln_seg(a, nvfp4, s, st));
}

// Two-level NVFP4 producers: as the NVFP4 producers, plus a 4-byte aligned
// tensor-scale output and workspace.  Default: the block-per-lane kernels --
// persistent, one atomic per CTA in the maximum pass, the flat quantising pass
// (measured on GB300: 37810x5376 segmented 341 -> 284 us, 5070x3072 20.9 ->
// 18.5 us), with the warp-per-row maximum pass for large tensors; the register
// row kernels where those do not apply (or forced: NVFP4AP_KERNEL=3).
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
  const Force f = forced();
  // default: one cooperative launch that reads the tensor once, where its rows
  // fit in the SMs' shared memory
  if (f.family == FAM_AUTO) {
    const int sms = sm_count();
    if (ln_2level_onchip_fits(mod, a.rows, a.dim, sms)) {
      // a cooperative launch the device refuses (fewer SMs available to this
      // context than it has, say) leaves nothing running: take the two passes
      if (launch_ln_2level_onchip(a, mod, sms, wait_limit_cycles(), st) == cudaSuccess) return NVFP4AP_OK;
      (void)cudaGetLastError();
    }
  }
  if (f.family != FAM_ROWS && ln_blk_supported(BLK_2LEVEL, mod, a.dim, a.nseg) && aligned(a.x, 32)) {
    BlkShape bs{};
    const int sms = sm_count();
    if (sms > 0 && pick_blk(a.dim, 0, &bs)) {
      bs.ctas_per_sm = f.ctas;
      bs.warp = f.family == FAM_WARP ? 1 : f.family == FAM_BLK ? -1 : 0;
      return finish(launch_ln_2level_blk(a, mod, bs, sms, st));
    }
  }
  RowShape s{};
  if (!pick_rows(mod, a.dim, &s)) return NVFP4AP_ERR_DIM;
  if (!grid_ok((a.rows + 127) / 128 * 128, s.rpc)) return NVFP4AP_ERR_SHAPE;
  // the register-capped instances for rows that exactly fill the CTA's
  // chunks; unmodulated rows only -- the broadcast instances spill at 40
  // registers
  const bool full = mod == MOD_NONE && s.tpr <= 128 && s.per_thread >= 2 && s.per_thread <= 4 &&
                    (int64_t)s.tpr * s.per_thread * 8 == a.dim;
  return finish(launch_ln_2level(a, mod, s, full, st));
}

// Single-level NVFP4 producers.  Default (measured on GB300 at dims
// 2048-8192, 2,520-32,768 rows): the one-row-per-CTA block-per-lane kernel
// where the row fits it exactly (5070x3072 layer norm 10.0 -> 8.5 us,
// broadcast 12.2 -> 10.6 us against the register row and persistent
// kernels); where it does not, the block-per-lane persistent kernel from
// kBlkNvfp4Rows rows when its shape has no idle lane and three or more rows
// per CTA (dims 1024, 1536, 5120: 1536 x 32768 layer norm 33.4 -> 22.2 us,
// broadcast 36.8 -> 28.3 us; 5120 x 4096 broadcast 20.1 -> 16.0 us), else the
// register row kernels.
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

  const Force f = forced();
  const int sms = sm_count();
  const bool blk_ok = ln_blk_supported(BLK_NVFP4, mod, a.dim, 0) && aligned(a.x, 32);
  int fam = f.family;
  if (fam == FAM_AUTO || fam == FAM_ROWBLK) {
    RbShape rb{};
    // the broadcast and modfp8 sources take the same shape, so that they
    // reduce to each other bit for bit
    if (aligned(a.x, 32) && pick_rowblk(a.dim, 0, &rb, mod == MOD_BCAST || mod == MOD_MODFP8))
      return finish(launch_ln_rowblk(a, true, mod, rb, st));
    BlkShape bs{};
    fam = (fam == FAM_AUTO && a.rows >= kBlkNvfp4Rows && blk_ok && blk_default_shape(a.dim, false, &bs)) ? FAM_BLK
                                                                                                         : FAM_ROWS;
  }
  if (fam == FAM_BLK && blk_ok && sms > 0) {
    BlkShape bs{};
    if (pick_blk(a.dim, 0, &bs)) {
      bs.ctas_per_sm = f.ctas;
      return finish(launch_ln_blk(a, true, mod, bs, sms, st));
    }
  }
  RowShape rs{};
  if (!pick_rows(mod, a.dim, &rs)) return run_scalar(a, true, mod, st);
  if (fam == FAM_TMA && mod != MOD_MODFP8 && sms > 0 && ln_tma_supported(true, mod, rs)) {
    if (!grid_ok((a.rows + 127) / 128 * 128, rs.rpc)) return NVFP4AP_ERR_SHAPE;
    return finish(launch_ln_tma(a, true, mod, rs, sms, 0, f.ctas, wait_limit_cycles(), st));
  }
  return run_rows(a, true, mod, rs, f.ctas, st);
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
  unsigned int f = 0u, g = 0u, o = 0u, h = 0u, i = 0u, j = 0u, k = 0u, l = 0u, m = 0u;
  if (take_ring_fault(&f) != cudaSuccess || take_tma_fault(&g) != cudaSuccess || take_onchip_fault(&o) != cudaSuccess ||
      take_seg_fault(&h) != cudaSuccess || take_blk_seg_fault(&i) != cudaSuccess ||
      take_blk2l_seg_fault(&j) != cudaSuccess || take_warpreg_seg_fault(&k) != cudaSuccess ||
      take_scalar_seg_fault(&l) != cudaSuccess || take_onchip_seg_fault(&m) != cudaSuccess) {
    (void)cudaGetLastError();
    return NVFP4AP_ERR_LAUNCH;
  }
  if (f | g | o) return NVFP4AP_ERR_TIMEOUT;
  return (h | i | j | k | l | m) ? NVFP4AP_ERR_FAULT : NVFP4AP_OK;
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

NVFP4AP_EXPORT int nvfp4ap_2level_single_read(int64_t rows, int64_t dim, int modulation, int* single_read) {
  if (!single_read) return NVFP4AP_ERR_NULL;
  *single_read = 0;
  if (rows < 0 || dim <= 0) return NVFP4AP_ERR_SHAPE;
  if (dim > NVFP4AP_MAX_DIM || dim % 16 != 0) return NVFP4AP_ERR_DIM;
  const int mod = modulation == 0 ? MOD_NONE : modulation == 1 ? MOD_BCAST : modulation == 2 ? MOD_SEG : -1;
  if (mod < 0) return NVFP4AP_ERR_VALUE;
  if (rows == 0 || forced().family != FAM_AUTO) return NVFP4AP_OK;
  const int sms = sm_count();
  if (sms <= 0) return NVFP4AP_ERR_LAUNCH;
  *single_read = ln_2level_onchip_fits(mod, rows, dim, sms) ? 1 : 0;
  return NVFP4AP_OK;
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
