/*
 * nvfp4ap.h -- C ABI of libnvfp4ap.so: GB300 (sm_103a) adaptive-LayerNorm
 * activation producers (LayerNorm -> adaptive modulation -> FP8 e4m3fn or
 * NVFP4) and the six-way fp32 -> bf16 modulation producer.
 *
 * Source of the operations: the "adaptive-layernorm-producers" README,
 * sections "Available Functions" (the function list), "Tensor Contract"
 * (shapes, dtypes, contiguity, dim rules) and "Minimal Usage" (static
 * buffers for CUDA Graph capture, the table form, the NVFP4 pair).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers to contiguous row-major memory
 *    owned by the caller.  The producers never allocate, never free, never
 *    synchronise and never read device memory on the host, so every producer
 *    call can be captured in a CUDA graph with static buffers.  The only
 *    entry points that read device memory on the host (and so synchronise)
 *    are the diagnostics nvfp4ap_take_device_fault and
 *    nvfp4ap_noalloc_progress.
 *  - bf16 tensors are IEEE bfloat16 bit patterns (2 bytes), e4m3 tensors are
 *    OCP float8_e4m3fn bytes, fp32 tensors are IEEE binary32.
 *  - `stream` is the CUDA stream the kernel is launched on (NULL = legacy
 *    default stream).  The call returns after the launch is queued.
 *  - The return value is an NVFP4AP_* status.  Every argument is checked on
 *    the host before anything is launched; on a non-zero status nothing has
 *    been launched and no memory has been touched, except NVFP4AP_ERR_LAUNCH,
 *    which reports the CUDA error of the launch itself.
 *  - rows == 0 (or batch*seq == 0) is a valid no-op; pointers may then be NULL.
 *  - Alignment (the tensor contract asks for contiguity only): the
 *    LayerNorm producers, single-level, accept any element-aligned pointers
 *    -- bf16 tensors at 2 bytes, fp32 tables, scalars and segment indices at
 *    4, e4m3 vectors and the outputs at 1.  They run vectorised kernels when
 *    x, scale, shift, temb, inv_s and the segment tables are 16-byte aligned,
 *    the table 16 (FP8) or 8 bytes, the outputs 8 bytes and the e4m3 vectors
 *    8 bytes (FP8 also has a bf16-pair path at 4/2 bytes), and otherwise an
 *    element-wise kernel (one load per element, byte stores) with the same
 *    results within the same bounds.  A pointer that is not even
 *    element-aligned gives NVFP4AP_ERR_ALIGN.  The two-level, SwiGLU,
 *    six-way and allocation-free entry points keep the alignment rules
 *    stated beside them (NVFP4AP_ERR_ALIGN otherwise).
 *  - dim must be at most NVFP4AP_MAX_DIM for the LayerNorm ops (a whole row
 *    is held in registers); the six-way op has no such limit.
 *  - Environment: each producer call reads three variables (one pass over
 *    the environment per call); none is needed.  NVFP4AP_KERNEL=F[:C] forces
 *    a kernel family for tests -- F = 3 register row kernels, 4 TMA
 *    pipeline, 5 block-per-lane persistent kernels, 6 warp-per-row kernels
 *    (FP8 segmented form and the two-level maximum pass), 8 one-row-per-CTA
 *    block-per-lane kernels; a family that does not take a form or shape
 *    falls back to the register row kernels (the table form: the TMA
 *    pipeline) -- and C caps the persistent kernels at C CTAs per SM; every
 *    family meets the same output contract.
 *    NVFP4AP_PDL=0 launches without programmatic dependent launch;
 *    NVFP4AP_DEBUG=1 prints launch errors and the staged kernels' plans.
 */
#ifndef NVFP4AP_H
#define NVFP4AP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* nvfp4ap_stream_t; /* same type as cudaStream_t */

enum nvfp4ap_status {
  NVFP4AP_OK = 0,
  NVFP4AP_ERR_NULL = 1,    /* a required pointer is NULL (with rows > 0)      */
  NVFP4AP_ERR_SHAPE = 2,   /* negative rows/batch/seq, or dim <= 0           */
  NVFP4AP_ERR_DIM = 3,     /* dim odd (FP8), not a multiple of 16 (NVFP4), or
                              above NVFP4AP_MAX_DIM                          */
  NVFP4AP_ERR_INDEX = 4,   /* chunks < 1 or shift_idx/scale_idx out of range */
  NVFP4AP_ERR_ALIGN = 5,   /* a pointer misses its alignment rule            */
  NVFP4AP_ERR_LAUNCH = 6,  /* the CUDA launch failed (cudaGetLastError)      */
  NVFP4AP_ERR_TIMEOUT = 7, /* a kernel's bounded wait ran out; that kernel's
                              output is incomplete (reported by
                              nvfp4ap_take_device_fault)                      */
  NVFP4AP_ERR_VALUE = 8,   /* eps negative or not finite                      */
  NVFP4AP_ERR_SCRATCH = 9, /* the call needs more than the static scratch of
                              ada_layer_norm_quant_fp8_bf16_noalloc holds     */
  NVFP4AP_ERR_FAULT = 10   /* a segmented producer met a segment index
                              outside [0, nseg) (reported by
                              nvfp4ap_take_device_fault)                      */
};

#define NVFP4AP_MAX_DIM 32768

/* Bytes of the caller-owned device workspace of the two-level LayerNorm
 * NVFP4 producers for `rows` rows: the maximum word, a grid-barrier count word
 * (used when the whole tensor is encoded in one launch), padding to 16 bytes,
 * then one 16-byte slot per row where the maximum pass keeps the row's
 * statistics for the quantising pass (16-byte aligned).  The SwiGLU producer uses the
 * word only (4 bytes, 4-byte aligned). */
#define NVFP4AP_2LEVEL_WORKSPACE_BYTES(rows) (16 + 16 * (int64_t)(rows))
/* The same as a function (for callers that cannot use the macro); -1 for
 * rows < 0 or a size past INT64_MAX. */
int64_t nvfp4ap_2level_workspace_bytes(int64_t rows);

/* Whether the two-level LayerNorm producers, for a (rows, dim) tensor on the
 * current device, read it from HBM once (*single_read = 1: one cooperative
 * launch, its rows staged in shared memory) or twice (0: the maximum pass,
 * then the quantising pass), with the default kernel choice.  modulation: 0
 * none, 1 broadcast, 2 segmented.  Status: NVFP4AP_ERR_NULL (single_read),
 * _SHAPE, _DIM, _VALUE (modulation), _LAUNCH (no CUDA device); *single_read
 * is 0 whenever the status is not NVFP4AP_OK, for rows = 0, and when
 * NVFP4AP_KERNEL forces a kernel family.  A device that refuses the
 * cooperative launch at run time still gets the two passes.  Host-only:
 * launches nothing. */
int nvfp4ap_2level_single_read(int64_t rows, int64_t dim, int modulation, int* single_read);

/* Human-readable name of a status code (static string, never NULL). */
const char* nvfp4ap_status_string(int status);

/* Version of this ABI (major*10000 + minor*100 + patch). */
int nvfp4ap_version(void);

/* Some LayerNorm producer kernels (the table form's default kernel and the
 * allocation-free producer) stage rows through shared memory with
 * asynchronous bulk copies and wait on them with a bounded wait (about one
 * second by default).  If a wait runs out, the kernel waits (with that same
 * default bound) for every copy it still has in flight, stops early, leaves
 * its output incomplete and sets a device word instead of hanging.  The
 * segmented producers set a second word when a row's segment index is out
 * of range.  This call reads and clears both words on the current device:
 * NVFP4AP_ERR_TIMEOUT if a wait ran out since the last call (it takes
 * precedence), else NVFP4AP_ERR_FAULT if a segment index was out of range,
 * else NVFP4AP_OK; NVFP4AP_ERR_LAUNCH if the device could not be read.
 * Unlike the producers it synchronises with the device (a blocking copy). */
int nvfp4ap_take_device_fault(void);

/* The bound of those waits, for testing the failure path: `cycles` SM clock
 * cycles after a first non-blocking test of the copy; cycles <= 0 restores the
 * default (2e9 cycles, about one second).  A very small bound makes the first
 * wait of each CTA give up before its copy lands, so a test can check the
 * report above; the copies in flight are still waited for with the default
 * bound before the kernel returns.  Process-wide, read when a producer is
 * launched (a captured graph keeps the bound it was captured with).  Returns
 * NVFP4AP_OK.  nvfp4ap_wait_limit returns the bound in effect. */
int nvfp4ap_set_wait_limit(int64_t cycles);
int64_t nvfp4ap_wait_limit(void);

/* ------------------------------------------------------------------------
 * FP8 producers.  For each row r of x (rows, dim) bf16:
 *   mean, var = biased mean and variance of the row; rstd = 1/sqrt(var+eps)
 *   y[d] = (x[r,d] - mean) * rstd * (1 + scale[.]) + shift[.]
 *   out[r,d] = e4m3fn(y[d] / act_scale)   round-to-nearest-even, saturating
 *                                          to +-448 (e4m3fn has no inf)
 * act_scale: device pointer to ONE fp32 (the dequantisation scale, so the
 * output value is about out * act_scale).  eps: host float, >= 0.
 * out: (rows, dim) e4m3fn bytes.  dim must be even.
 * ---------------------------------------------------------------------- */

/* README "Available Functions": ada_layer_norm_quant_fp8_bf16.
 * scale, shift: (dim,) bf16, broadcast over rows. */
int ada_layer_norm_quant_fp8_bf16(const void* x, const void* scale, const void* shift,
                                  const float* act_scale, float eps, void* out,
                                  int64_t rows, int64_t dim, nvfp4ap_stream_t stream);

/* No counterpart in the paper: an addition of this library.
 *
 * ada_layer_norm_quant_fp8_bf16_noalloc computes the same operation as
 * ada_layer_norm_quant_fp8_bf16, with the same arguments and within the same
 * bounds against the library's reference (its kernel takes the row statistics
 * in two passes, so a byte can differ by one code step from the default
 * kernel's), for callers that cannot allocate device memory at all -- for
 * example code that runs under a device-memory budget fixed at start-up, or
 * inside a framework region whose caching allocator must not grow.  It runs
 * the TMA ring kernel, which keeps one progress word per CTA (rows finished;
 * bit 31 set if one of the CTA's bounded waits ran out) in device scratch;
 * here that scratch is a fixed array inside the library, 1024 words (4 KB),
 * 256-byte aligned, which every GPU that loads the library holds until the
 * process exits.  The words of the last call can be read back with
 * nvfp4ap_noalloc_progress (diagnostics).  The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine):
 * it clears the words it will use with cudaMemsetAsync on `stream`, then
 * launches.
 *  - dim % 8 == 0; x, scale, shift 16-byte aligned, out 8-byte aligned,
 *    act_scale 4-byte aligned (else NVFP4AP_ERR_DIM / NVFP4AP_ERR_ALIGN).
 *  - A call whose launch would need more than 1024 CTAs is rejected with
 *    NVFP4AP_ERR_SCRATCH before anything is launched (the persistent grid is
 *    at most a few CTAs per SM, so 1024 covers current GPUs).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) and sets up the kernel's shared-memory attribute;
 *    make that first call before any stream capture.
 *  - Every call shares the one array, which keeps the last call's contents:
 *    calls that overlap on the GPU (different streams, or different host
 *    threads) race on it.  Serialise them on one stream.
 *  - A bounded wait that runs out is reported by nvfp4ap_take_device_fault(). */
int ada_layer_norm_quant_fp8_bf16_noalloc(const void* x, const void* scale, const void* shift,
                                          const float* act_scale, float eps, void* out,
                                          int64_t rows, int64_t dim, nvfp4ap_stream_t stream);

/* No counterpart in the paper: diagnostics of the allocation-free producer.
 * *used (if not NULL) receives the CTA count of the last
 * ada_layer_norm_quant_fp8_bf16_noalloc launch on the current device (0 before
 * the first); the first min(n, *used) progress words of that launch are
 * copied into the host array `words` (if not NULL and n > 0): each holds the
 * rows its CTA finished in bits 0-30 and bit 31 if one of its waits ran out,
 * so after a complete call the words sum to rows.  A blocking read of device
 * memory (synchronises with the device); a later call overwrites the words.
 * Returns NVFP4AP_OK, or NVFP4AP_ERR_LAUNCH if the device could not be read. */
int nvfp4ap_noalloc_progress(uint32_t* words, int64_t n, int64_t* used);

/* README "Available Functions": ada_layer_norm_quant_fp8_ptok_bf16.
 * scale, shift: (rows, dim) bf16, one row of modulation per token. */
int ada_layer_norm_quant_fp8_ptok_bf16(const void* x, const void* scale, const void* shift,
                                       const float* act_scale, float eps, void* out,
                                       int64_t rows, int64_t dim, nvfp4ap_stream_t stream);

/* README "Available Functions" / "Minimal Usage" (fused host modulation table
 * add and chunk selection): ada_layer_norm_quant_fp8_ptok_table_bf16.
 * temb: (rows, chunks, dim) bf16; table: (chunks, dim) fp32;
 *   scale[r,d] = temb[r, scale_idx, d] + table[scale_idx, d]
 *   shift[r,d] = temb[r, shift_idx, d] + table[shift_idx, d]
 * (the sums are taken in fp32 and are not rounded to bf16).
 * 0 <= shift_idx, scale_idx < chunks, else NVFP4AP_ERR_INDEX. */
int ada_layer_norm_quant_fp8_ptok_table_bf16(const void* x, const void* temb, const float* table,
                                             int64_t chunks, int64_t shift_idx, int64_t scale_idx,
                                             const float* act_scale, float eps, void* out,
                                             int64_t rows, int64_t dim, nvfp4ap_stream_t stream);

/* README "Available Functions": ada_layer_norm_quant_fp8_modfp8_bf16;
 * "Tensor Contract": scale_fp8, shift_fp8 e4m3fn (dim,); scale_deq,
 * shift_deq fp32 scalars.
 * scale_fp8, shift_fp8: device (dim,) e4m3fn bytes, broadcast over rows.
 * scale_deq, shift_deq: device pointers to ONE fp32 each.  The modulation is
 *   scale[d] = decode(scale_fp8[d]) * (*scale_deq)
 *   shift[d] = decode(shift_fp8[d]) * (*shift_deq)
 * taken as one fp32 product each (exact whenever the scalar has at most 20
 * significant bits); the rest as ada_layer_norm_quant_fp8_bf16.  e4m3 NaN
 * bytes (0x7F, 0xFF) are out of contract.  A NULL pointer gives
 * NVFP4AP_ERR_NULL, a misaligned scalar NVFP4AP_ERR_ALIGN. */
int ada_layer_norm_quant_fp8_modfp8_bf16(const void* x, const void* scale_fp8, const void* shift_fp8,
                                         const float* scale_deq, const float* shift_deq,
                                         const float* act_scale, float eps, void* out, int64_t rows,
                                         int64_t dim, nvfp4ap_stream_t stream);

/* README "Available Functions": awq_ada_layer_norm_quant_fp8_bf16;
 * "Tensor Contract": inv_s bf16 (dim,).
 * scale, shift, inv_s: device (dim,) bf16, broadcast over rows.  The pages
 * do not say where inv_s applies; this library multiplies the modulated
 * activation by it before the quantiser (the AWQ smoothing of a GEMM input):
 *   out[r,d] = e4m3fn(y[d] * inv_s[d] / act_scale)
 * computed as y * (inv_s * (1 / act_scale)) in fp32. */
int awq_ada_layer_norm_quant_fp8_bf16(const void* x, const void* scale, const void* shift,
                                      const void* inv_s, const float* act_scale, float eps, void* out,
                                      int64_t rows, int64_t dim, nvfp4ap_stream_t stream);

/* Segmented modulation (h3-blackwell-runtime compare page: segment-specific
 * shift and scale selection with a per-row segment index).
 * seg_idx: device (rows,) int32, 4-byte aligned; row r takes row seg_idx[r] of
 * seg_scale, seg_shift: device (nseg, dim) bf16.
 *   y[d] = (x[r,d] - mean) * rstd * (1 + seg_scale[g,d]) + seg_shift[g,d]
 * dim even (FP8) or a multiple of 16 (NVFP4), else NVFP4AP_ERR_DIM.
 * nseg < 1 gives NVFP4AP_ERR_INDEX.  An index outside [0, nseg) cannot be
 * checked on the host: that row is produced with zero modulation and the
 * device fault word is set (nvfp4ap_take_device_fault). */
int ada_layer_norm_quant_fp8_seg_bf16(const void* x, const int32_t* seg_idx, const void* seg_scale,
                                      const void* seg_shift, int64_t nseg, const float* act_scale, float eps,
                                      void* out, int64_t rows, int64_t dim, nvfp4ap_stream_t stream);

/* README "Available Functions": layer_norm_no_affine_quant_fp8_static_bf16.
 * No modulation: y = (x - mean) * rstd. */
int layer_norm_no_affine_quant_fp8_static_bf16(const void* x, const float* act_scale, float eps,
                                               void* out, int64_t rows, int64_t dim,
                                               nvfp4ap_stream_t stream);

/* ------------------------------------------------------------------------
 * NVFP4 producers ("Tensor Contract": packed (rows, dim/2) uint8 and the
 * 128x4 swizzled uint8 scale layout; "Validation": the staged BF16-norm plus
 * FP4 quantizer contract).  For each row, y as above (no act_scale), then
 *   v = bf16(y)                                  (round-to-nearest-even)
 *   per 16-element block b: amax = max |v|, s = e4m3fn(amax / 6) (RNE,
 *     saturating); code_k = e2m1 nearest of v_k / decode(s), ties to the
 *     even code, saturating at 6, sign kept (a zero scale gives +-0 codes)
 *   packed[r, 8b + j] = code_{16b+2j} | code_{16b+2j+1} << 4
 *   sf_swizzled[off(r, b)] = s, with C4 = ceil(dim/16 / 4) and
 *     off(r,b) = ((r/128)*C4 + b/4)*512 + (r%32)*16 + ((r%128)/32)*4 + b%4
 *   and every padding byte of the swizzled buffer (rows up to a multiple of
 *   128, block columns up to a multiple of 4) is written as 0.
 * dim % 16 == 0.  packed: rows*dim/2 bytes; sf_swizzled:
 * swizzled_sf_size(rows, dim) bytes (any alignment, see the conventions).
 * ---------------------------------------------------------------------- */

/* README "Available Functions": ada_layer_norm_quant_nvfp4_swizzled_bf16.
 * scale, shift: (dim,) bf16 broadcast. */
int ada_layer_norm_quant_nvfp4_swizzled_bf16(const void* x, const void* scale, const void* shift,
                                             float eps, void* packed, void* sf_swizzled,
                                             int64_t rows, int64_t dim, nvfp4ap_stream_t stream);

/* README "Available Functions": ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16.
 * scale_fp8, shift_fp8: device (dim,) e4m3fn bytes;
 * scale_deq, shift_deq: device pointers to ONE fp32 each; the modulation is
 * decode(code) * deq as for ada_layer_norm_quant_fp8_modfp8_bf16, the output
 * as ada_layer_norm_quant_nvfp4_swizzled_bf16. */
int ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(const void* x, const void* scale_fp8, const void* shift_fp8,
                                                    const float* scale_deq, const float* shift_deq, float eps,
                                                    void* packed, void* sf_swizzled, int64_t rows, int64_t dim,
                                                    nvfp4ap_stream_t stream);

/* README "Available Functions": layer_norm_no_affine_quant_nvfp4_swizzled_bf16. */
int layer_norm_no_affine_quant_nvfp4_swizzled_bf16(const void* x, float eps, void* packed,
                                                   void* sf_swizzled, int64_t rows, int64_t dim,
                                                   nvfp4ap_stream_t stream);

/* Single-level NVFP4 with the segmented modulation of
 * ada_layer_norm_quant_fp8_seg_bf16 (same index and table rules). */
int ada_layer_norm_quant_nvfp4_swizzled_seg_bf16(const void* x, const int32_t* seg_idx, const void* seg_scale,
                                                 const void* seg_shift, int64_t nseg, float eps, void* packed,
                                                 void* sf_swizzled, int64_t rows, int64_t dim,
                                                 nvfp4ap_stream_t stream);

/* ------------------------------------------------------------------------
 * Two-level NVFP4 producers (h3-blackwell-runtime compare page:
 * NVFP4_STREAMING_DESIGN.md "Numerical Constraint" -- one exact global bf16
 * absolute maximum, one fp32 tensor scale derived from it, e4m3 block scales,
 * e2m1 codes using both; the P1 checkpoint's numerical contract -- block
 * scale (amax / 6) / global scale, clamped at 448).  For the staged values
 * v = bf16(y) of the whole (rows, dim) tensor:
 *   amax = max |v|;  ts = bf16(fp32(amax / 2688))   (2688 = 6 * 448)
 *   per 16-element block b: s = e4m3fn(fminf(fp32(fp32(amax_b / 6) / ts), 448))
 *   code_k = e2m1 nearest of v_k / (decode(s) * ts), ties to even, saturating;
 *            a zero divisor gives +-0 codes
 * The library divides exactly where the page's runtime multiplies by an
 * approximate reciprocal.  Outputs: packed and sf_swizzled as for the
 * single-level producers, and *tensor_scale = ts (device fp32, 4-byte
 * aligned) -- the dequantised value is e2m1 * decode(s) * ts.
 * workspace: caller-owned device memory of NVFP4AP_2LEVEL_WORKSPACE_BYTES(rows)
 * bytes, 16-byte aligned (NVFP4AP_ERR_ALIGN), cleared and used by the call
 * (two calls on concurrent streams need two workspaces); a smaller buffer is
 * written past its end.  Kernels on `stream`: a clear of the workspace words,
 * then -- when every SM's share of the rows fits in its shared memory -- one
 * cooperative launch that reads the tensor once (statistics and maximum, a
 * grid-wide barrier, then the codes), else (or when the device refuses that
 * launch) the maximum pass and the quantising pass (graph-capturable either
 * way). */
int layer_norm_no_affine_quant_nvfp4_2level_bf16(const void* x, float eps, void* packed, void* sf_swizzled,
                                                 float* tensor_scale, void* workspace, int64_t rows, int64_t dim,
                                                 nvfp4ap_stream_t stream);
/* broadcast scale, shift: (dim,) bf16, 16-byte aligned */
int ada_layer_norm_quant_nvfp4_2level_bf16(const void* x, const void* scale, const void* shift, float eps,
                                           void* packed, void* sf_swizzled, float* tensor_scale, void* workspace,
                                           int64_t rows, int64_t dim, nvfp4ap_stream_t stream);
/* segmented modulation as in ada_layer_norm_quant_fp8_seg_bf16 */
int ada_layer_norm_quant_nvfp4_2level_seg_bf16(const void* x, const int32_t* seg_idx, const void* seg_scale,
                                               const void* seg_shift, int64_t nseg, float eps, void* packed,
                                               void* sf_swizzled, float* tensor_scale, void* workspace,
                                               int64_t rows, int64_t dim, nvfp4ap_stream_t stream);

/* SwiGLU -> two-level NVFP4 (h3-blackwell-runtime compare page,
 * NVFP4_SWIGLU_FUSION_DESIGN.md: both bf16 boundaries kept):
 *   v = bf16(bf16(silu(gate)) * up),  silu(g) = g / (1 + exp(-g)),
 * the silu boundary taken on the binary32 value of silu (the library takes
 * bf16(binary32(silu(g))) from a table computed in float64 for all 65,536 bf16
 * gate patterns), then the two-level contract above on v (no LayerNorm).  gate, up: device
 * (rows, dim) bf16 with the common row stride ld (elements): two tensors, or
 * the halves of one (rows, 2*dim) tensor (up = gate + dim, ld = 2*dim).  dim %
 * 16 == 0, ld >= dim, ld % 8 == 0 and rows * (dim / 8) < 2^32 (NVFP4AP_ERR_DIM /
 * _SHAPE), gate and up 16-byte aligned (32-byte aligned with ld % 16 == 0 takes
 * 256-bit loads).  Outputs as for the two-level producers; workspace: the
 * maximum word only, 4 bytes, 4-byte aligned. */
int swiglu_quant_nvfp4_2level_bf16(const void* gate, const void* up, int64_t ld, void* packed, void* sf_swizzled,
                                   float* tensor_scale, void* workspace, int64_t rows, int64_t dim,
                                   nvfp4ap_stream_t stream);

/* The SwiGLU values of swiglu_quant_nvfp4_2level_bf16 themselves:
 * out (rows, dim) bf16 contiguous, v = bf16(bf16(silu(gate)) * up) -- the
 * materialised form.  dim % 8 == 0, gate/up/out 16-byte aligned, ld and rows as
 * above. */
int swiglu_bf16(const void* gate, const void* up, int64_t ld, void* out, int64_t rows, int64_t dim,
                nvfp4ap_stream_t stream);

/* README "Available Functions" / "Tensor Contract": swizzled_sf_size.
 * Bytes of the swizzled scale buffer: ceil(rows/128)*128 * ceil(dim/16/4)*4.
 * Returns -1 when rows < 0, dim <= 0 or dim % 16 != 0.  Host only. */
int64_t swizzled_sf_size(int64_t rows, int64_t dim);

/* ------------------------------------------------------------------------
 * README "Available Functions" / "Tensor Contract": adaln_modulation6_bf16.
 * params: (batch, seq, 6, dim) fp32; modulation: (6, dim) fp32;
 * out[i]: six device pointers, each (batch, seq, dim) bf16:
 *   out[i][b,s,d] = bf16( params[b,s,i,d] + modulation[i,d] )
 * with one binary32 addition and round-to-nearest-even to bf16.
 * `out` itself is a HOST array of six device pointers (read during the call).
 * ---------------------------------------------------------------------- */
int adaln_modulation6_bf16(const float* params, const float* modulation, void* const out[6],
                           int64_t batch, int64_t seq, int64_t dim, nvfp4ap_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4AP_H */
