// kernels.h -- internal interface between the C ABI (abi.cu) and the kernel
// translation units.  Not installed; the public interface is nvfp4ap.h.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace nvfp4ap {

// Bound of every mbarrier wait of the TMA kernels in SM clock cycles (about
// one second unless nvfp4ap_set_wait_limit changed it).
long long wait_limit_cycles();

// Launch `k` on `st` with programmatic stream serialisation (PDL) unless
// NVFP4AP_PDL=0: the kernel may then be dispatched while the previous kernel
// on the stream drains (the kernel itself waits for it, see pdl_enter()).
bool pdl_enabled();
// NVFP4AP_* settings of the current producer call (abi.cu): env_refresh takes
// one pass over the environment, env_get reads that snapshot (nullptr if unset)
void env_refresh();
const char* env_get(const char* name);
template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k, static_cast<KArgs>(args)...);
}

// modulation source of a LayerNorm producer
//   MOD_BCAST   bf16 (dim,) scale/shift
//   MOD_PTOK    bf16 (rows, dim) scale/shift
//   MOD_TABLE   temb[r, idx, :] (bf16) + table[idx, :] (fp32)
//   MOD_MODFP8  e4m3 (dim,) scale/shift times fp32 device scalars scale_deq/shift_deq
//   MOD_AWQ     bf16 (dim,) scale/shift, output multiplied by bf16 (dim,) inv_s
//   MOD_SEG     row r takes row seg_idx[r] of bf16 (nseg, dim) scale/shift tables
enum ModKind { MOD_NONE = 0, MOD_BCAST = 1, MOD_PTOK = 2, MOD_TABLE = 3, MOD_MODFP8 = 4, MOD_AWQ = 5, MOD_SEG = 6 };

// sources whose scale/shift are the same (dim,) vector for every row
constexpr bool mod_is_bcast(int mod) { return mod == MOD_BCAST || mod == MOD_MODFP8 || mod == MOD_AWQ; }

// Arguments of one LayerNorm producer launch (device pointers, element counts).
struct LnArgs {
  const uint16_t* x;      // (rows, dim) bf16
  const uint16_t* scale;  // BCAST: (dim,)  PTOK: (rows, dim)  bf16
  const uint16_t* shift;
  const uint16_t* temb;   // TABLE: (rows, chunks, dim) bf16
  const float* table;     // TABLE: (chunks, dim) fp32
  int64_t chunks, shift_idx, scale_idx;
  const float* act_scale; // FP8: device scalar
  const uint8_t* scale8;  // MODFP8: (dim,) e4m3
  const uint8_t* shift8;
  const float* scale_deq; // MODFP8: device scalars
  const float* shift_deq;
  const uint16_t* inv_s;  // AWQ: (dim,) bf16
  const int32_t* seg_idx;     // SEG: (rows,) segment of each row
  const uint16_t* seg_scale;  // SEG: (nseg, dim) bf16
  const uint16_t* seg_shift;
  int64_t nseg;
  unsigned int* amax_ws;      // two-level: one device word (the tensor's largest |v| as fp32 bits)
  float* tensor_scale;        // two-level: device fp32 output
  float* row_stats;           // two-level: (rows,) float4 K, mean - K, rstd, 0 per row (written by the
                              // block-per-lane maximum pass; nullptr: not kept)
  float eps;
  void* out;              // FP8: (rows, dim) e4m3; NVFP4: packed (rows, dim/2)
  void* sf;               // NVFP4: swizzled scales
  int64_t rows, dim;
};

// Launch shape of a row kernel: `tpr` threads per row, `per_thread` vectors
// (FP8) or 16-element blocks (NVFP4) per thread, `rpc` rows per CTA.
struct RowShape {
  int tpr, per_thread, rpc;
};

// FP8 producers on the bf16-pair kernel (every modulation source except the
// segmented one): `vec` must be 2 (one bf16 pair per vector).
cudaError_t launch_ln_fp8(const LnArgs& a, int mod, int vec, RowShape s, cudaStream_t st);
// Largest threads-per-row (and threads-per-CTA) the (vec, per_thread)
// instance accepts; 0 if there is no such instance.
int ln_fp8_max_tpr(int vec, int per_thread);

// Register-resident row kernels for FP8 (dim % 8 == 0, 16-byte aligned) and
// NVFP4: `per_thread` 8-element chunks per thread.
cudaError_t launch_ln_rows(const LnArgs& a, bool nvfp4, int mod, RowShape s, cudaStream_t st);
int ln_rows_max_tpr(int mod, int per_thread);
// NVFP4 row kernel for rows that exactly fill tpr * per_thread chunks: one
// row per CTA of tpr <= 128 threads, registers capped at 40 per thread;
// per_thread 2..4; mod MOD_NONE, MOD_BCAST or MOD_MODFP8.
cudaError_t launch_ln_rows_full(const LnArgs& a, bool nvfp4, int mod, RowShape s, cudaStream_t st);
// Persistent broadcast-modulation variant (one row per CTA at a time, the
// next row prefetched, fp32 modulation in registers): tpr <= 256, rpc == 1,
// per_thread in {1, 2, 3, 4, 6}; at most `ctas_per_sm` CTAs per SM (0 = as
// many as fit).
cudaError_t launch_ln_bcast_persistent(const LnArgs& a, bool nvfp4, int mod, RowShape s, int sms,
                                       int ctas_per_sm, cudaStream_t st);

// Block-per-lane persistent row kernels (ln_blk.cuh; ln_blk.cu, ln_blk2l.cu):
// a lane owns whole 16-element blocks (`bpt` of them), `tpr` threads per row
// (a multiple of 32, <= 256), 512-thread CTAs of 512 / tpr rows, at most
// `ctas_per_sm` CTAs per SM (0 = as many as fit).  Modulation as fp32 tables in
// shared memory.  `warp` (two-level only): 1 forces the warp-per-row maximum
// pass, -1 the row-group one, 0 chooses by size.
// dim % 16 == 0, dim <= kBlkMaxDim; x 32-byte aligned; FP8 out 16-byte
// aligned; broadcast bf16 sources and segment tables 16-byte aligned.
struct BlkShape {
  int tpr, bpt, ctas_per_sm, warp;
};
constexpr int64_t kBlkMaxDim = 8192;
enum { BLK_FP8 = 0, BLK_NVFP4 = 1, BLK_2LEVEL = 2 };
// `kind` BLK_*; nseg: segments of a MOD_SEG source (their tables must fit)
bool ln_blk_supported(int kind, int mod, int64_t dim, int64_t nseg);
// shape for `dim` (forced_bpt > 0: only that many blocks per lane); `fp8`:
// the FP8 preference (3, 2, 4, 6 blocks per lane) instead of 3, 4, 2, 6
bool pick_blk(int64_t dim, int forced_bpt, BlkShape* s, bool fp8 = false);
// the block-per-lane kernel as a default: a shape with no idle lane and at
// least three rows per CTA
bool blk_default_shape(int64_t dim, bool fp8, BlkShape* s);
cudaError_t launch_ln_blk(const LnArgs& a, bool nvfp4, int mod, BlkShape s, int sms, cudaStream_t st);
// two-level NVFP4 on the block-per-lane kernels: clears a.amax_ws, maximum
// pass, quantising pass; mod MOD_NONE, MOD_BCAST or MOD_SEG
cudaError_t launch_ln_2level_blk(const LnArgs& a, int mod, BlkShape s, int sms, cudaStream_t st);
// Warp-per-row FP8 segmented producer (ln_blk.cuh): each warp sweeps its rows
// twice (sums, then codes from the blocks read again through L1/L2); mod
// MOD_SEG (tables as for the block-per-lane kernels); ctas_per_sm as above.
cudaError_t launch_ln_warp_rows_fp8(const LnArgs& a, int mod, int sms, int ctas_per_sm, cudaStream_t st);
// Register-resident warp-per-row producers (ln_warpreg.cu): the same
// operations as the warp-per-row kernels with the row read once.  Lanes hold
// warp_regs_bpl(dim) blocks (0 when dim is not a multiple of 16 or above
// 6144); amax: the two-level maximum pass (mod MOD_NONE, MOD_BCAST or
// MOD_SEG), else the FP8 segmented producer (MOD_SEG); ctas_per_sm as above.
int warp_regs_bpl(int64_t dim);
// whether the warp-per-row path takes `rows` x `dim` on `sms` SMs: the two-sweep
// kernel from 4 rows per warp of its grid (sms * 128 rows); the
// register-resident one (regs) from the same number of elements, rows * dim >=
// sms * 128 * 3072 (measured on GB300: at 12000x5376 the two-level maximum pass
// 70.4 -> 60.9 us against the row-group kernel, at 12000x3072 a tie)
bool warp_path_rows(int64_t rows, int64_t dim, int sms, bool regs);
cudaError_t launch_warp_regs(const LnArgs& a, bool amax, int mod, int sms, int ctas_per_sm, cudaStream_t st);
// read and clear the segment-index fault words of the two translation units
cudaError_t take_blk_seg_fault(unsigned int* fault);
cudaError_t take_blk2l_seg_fault(unsigned int* fault);
cudaError_t take_warpreg_seg_fault(unsigned int* fault);

// One-row-per-CTA block-per-lane kernels (ln_rowblk.cu), NVFP4 and FP8: `tpr`
// threads per row (64..128, a multiple of 32), `bpt` 16-element blocks per
// thread (2..4), rows exactly tpr * bpt blocks; mod MOD_NONE, MOD_BCAST,
// MOD_MODFP8 (and MOD_AWQ for FP8); x 32-byte aligned, FP8 out 16-byte
// aligned.  pick_rowblk: the shape for `dim` (forced_bpt > 0: only that one;
// two_first: two blocks per lane preferred over three).
struct RbShape {
  int tpr, bpt;
};
bool pick_rowblk(int64_t dim, int forced_bpt, RbShape* s, bool two_first);
cudaError_t launch_ln_rowblk(const LnArgs& a, bool nvfp4, int mod, RbShape s, cudaStream_t st);

// Element-wise LayerNorm producers (ln_scalar.cu) for pointers that are only
// element-aligned: one CTA of 256 threads per row, FP8 (any modulation
// source) or NVFP4 (MOD_NONE, MOD_BCAST, MOD_MODFP8, MOD_SEG).
cudaError_t launch_ln_scalar(const LnArgs& a, bool nvfp4, int mod, cudaStream_t st);
cudaError_t take_scalar_seg_fault(unsigned int* fault);

// FP8 broadcast producer on the ring kernel with its per-CTA words in the
// library's static scratch array; returns an NVFP4AP_* status (arguments
// already validated, dim % 8 == 0, 16-byte aligned inputs).
int noalloc_fp8_bcast(const LnArgs& a, int sms, long long wait_limit, cudaStream_t st);
// Copies the first min(n, used) per-CTA words of the last allocation-free
// launch on the current device into `words` (a synchronising read); *used =
// that launch's CTA count (0 if none yet).
int noalloc_progress(unsigned int* words, int64_t n, int64_t* used);
// Reads and clears the fault word the ring kernels set when a bounded wait
// runs out (synchronising copy).
cudaError_t take_ring_fault(unsigned int* fault);

// Persistent TMA-pipelined row kernels (ln_tma.cu): one row per CTA at a
// time (rpc == 1, tpr <= 256, per_thread 1..4), rows staged through a ring of
// shared-memory stages by bulk copies.  forced_stages / ctas_per_sm: 0 = auto.
bool ln_tma_supported(bool nvfp4, int mod, RowShape s);
cudaError_t launch_ln_tma(const LnArgs& a, bool nvfp4, int mod, RowShape s, int sms, int forced_stages,
                          int ctas_per_sm, long long wait_limit, cudaStream_t st);
cudaError_t take_tma_fault(unsigned int* fault);

// Segmented modulation (MOD_SEG) on the register row kernels: FP8 (dim % 8
// == 0, 16-byte aligned inputs) or single-level NVFP4.
cudaError_t launch_ln_seg(const LnArgs& a, bool nvfp4, RowShape s, cudaStream_t st);
// Two-level NVFP4: clears a.amax_ws (a kernel), runs the maximum pass, then the
// quantising pass (writes packed, sf and *a.tensor_scale); mod MOD_NONE,
// MOD_BCAST or MOD_SEG.  `full`: rows exactly fill tpr * per_thread chunks
// (tpr <= 128) -- the register-capped instances.
cudaError_t launch_ln_2level(const LnArgs& a, int mod, RowShape s, bool full, cudaStream_t st);
// Reads and clears the word set when a segment index was out of range.
cudaError_t take_seg_fault(unsigned int* fault);

// Two-level NVFP4 in one cooperative launch (ln_2l_onchip.cu) for tensors
// whose rows fit in the SMs' shared memory (one CTA per SM, ceil(rows / sms)
// rows each): the tensor is read from HBM once.  mod MOD_NONE, MOD_BCAST or
// MOD_SEG; dim % 16 == 0; x 16-byte aligned; a.amax_ws holds the maximum word
// and, in the next word, the grid barrier's count (both cleared by a kernel
// launched first).  Copy waits bounded by wait_limit, the grid barrier by the
// normal bound; on expiry the fault word is set (take_onchip_fault).
bool ln_2level_onchip_fits(int mod, int64_t rows, int64_t dim, int sms);
cudaError_t launch_ln_2level_onchip(const LnArgs& a, int mod, int sms, long long wait_limit, cudaStream_t st);
cudaError_t take_onchip_fault(unsigned int* fault);
cudaError_t take_onchip_seg_fault(unsigned int* fault);

// SwiGLU work items (8-element chunks) of a (rows, dim) call fit the kernels'
// 32-bit item index: rows * (dim / 8) < 2^32.
bool swiglu_items_fit(int64_t rows, int64_t dim);
// SwiGLU -> two-level NVFP4 (swiglu.cu): clears ws, maximum pass, quantising
// pass.  gate/up (rows, dim) bf16 with row stride ld (elements), 16-byte
// aligned, ld % 8 == 0, dim % 16 == 0, swiglu_items_fit(rows, dim).
cudaError_t launch_swiglu_2level(const void* gate, const void* up, int64_t ld, int64_t rows, int64_t dim,
                                 void* packed, void* sf, float* tensor_scale, unsigned int* ws, int sms,
                                 cudaStream_t st);
// The SwiGLU values themselves, (rows, dim) bf16 contiguous (dim % 8 == 0).
cudaError_t launch_swiglu_values(const void* gate, const void* up, int64_t ld, int64_t rows, int64_t dim, void* out,
                                 int sms, cudaStream_t st);

// Six-way modulation (K7).
struct Mod6Args {
  const float* params;      // (tokens, 6, dim) fp32
  const float* modulation;  // (6, dim) fp32
  uint16_t* out[6];         // (tokens, dim) bf16 each
  int64_t tokens, dim;
};
cudaError_t launch_modulation6(const Mod6Args& a, bool vec8, cudaStream_t st);

}  // namespace nvfp4ap
