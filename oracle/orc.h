/*
 * orc.h -- C interface of the CPU oracle for the adaptive-LayerNorm activation
 * producers.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, scalar, slow CPU restatement of
 * what the producers compute, used to check the CUDA library.  Only the tests,
 * the smoke check and the benchmark's CPU-baseline leg may load it.  It shares
 * no code, header, table or constant with the CUDA library, and the CUDA
 * library never calls it.
 *
 * Sources (web pages; section names as printed there):
 *   [README]  "adaptive-layernorm-producers" README: "Available Functions",
 *             "Tensor Contract", "Minimal Usage", "Validation".
 *   [H3]      "daniel/h3-blackwell-runtime" compare page: PLAN.md "NVFP4
 *             activation quantization status"; "Phase 3: NVFP4 Fused
 *             Projection Prototype"; benchmarks/gb10-cute-nvfp4-conversion-
 *             contract.json; the attn_out_proj/FC1 ring records (qdata_bytes,
 *             sfa_bytes).
 *
 * All arrays are host memory, row-major and contiguous.  bf16 values travel
 * as their uint16 bit patterns, e4m3 values as bytes.  Every op computes its
 * rows independently; `nthreads` > 1 splits the rows over POSIX threads.
 */
#ifndef ORC_H
#define ORC_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats ---------------------------------------------------- */
double   orc_bf16_to_f64(uint16_t bits);
uint16_t orc_bf16_from_f32(float v);               /* nearest, ties to even */
double   orc_e4m3_decode(uint8_t code);            /* NaN for 0x7F / 0xFF   */
uint8_t  orc_e4m3_encode(double v);                /* nearest, ties to even, |v|>448 -> 448 */
double   orc_e2m1_decode(uint8_t code4);           /* low 4 bits used       */
uint8_t  orc_e2m1_encode(double v, double s_dec);  /* nearest of v/s_dec    */

/* ---- swizzled scale layout --------------------------------------------- */
int64_t orc_swizzled_sf_size(int64_t rows, int64_t dim);          /* -1 if invalid */
int64_t orc_sf_offset(int64_t r, int64_t c, int64_t dim);
void    orc_swizzle_scales(const uint8_t* sf_logical, int64_t rows, int64_t dim,
                           uint8_t* sf_swizzled);

/* ---- row statistics ------------------------------------------------------ */
void orc_row_stats(const uint16_t* x, int64_t dim, float eps, double* mean, double* rstd);

/* ---- producers ---------------------------------------------------------- */
/* modulation sources */
enum { ORC_MOD_NONE = 0, ORC_MOD_BCAST = 1, ORC_MOD_PTOK = 2, ORC_MOD_TABLE = 3,
       ORC_MOD_MODFP8 = 4, ORC_MOD_AWQ = 5, ORC_MOD_SEG = 6 };

typedef struct {
  int kind;
  const uint16_t* scale;   /* BCAST, AWQ: (dim,)   PTOK: (rows, dim)       */
  const uint16_t* shift;
  const uint16_t* temb;    /* TABLE: (rows, chunks, dim) bf16             */
  const float*    table;   /* TABLE: (chunks, dim) fp32                    */
  int64_t chunks, shift_idx, scale_idx;
  const uint8_t*  scale_fp8;  /* MODFP8: (dim,) e4m3 codes                */
  const uint8_t*  shift_fp8;
  float scale_deq, shift_deq; /* MODFP8: fp32 multipliers of the decoded codes */
  const uint16_t* inv_s;      /* AWQ: (dim,) bf16 smoothing multipliers    */
  const int32_t*  seg_idx;    /* SEG: (rows,) segment of each row          */
  const uint16_t* seg_scale;  /* SEG: (nseg, dim) bf16                      */
  const uint16_t* seg_shift;
  int64_t nseg;
} orc_mod_t;

/* y = LN(x) * (1 + scale) + shift, as double, for all rows (rows, dim);
 * AWQ: y = (LN(x) * (1 + scale) + shift) * inv_s. */
int orc_modulated_rows(const uint16_t* x, const orc_mod_t* mod, float eps, double* y,
                       int64_t rows, int64_t dim, int nthreads);

/* FP8: out[r,d] = e4m3( fp32( y[r,d] / act_scale ) ). */
int orc_ln_quant_fp8(const uint16_t* x, const orc_mod_t* mod, float act_scale, float eps,
                     uint8_t* out, int64_t rows, int64_t dim, int nthreads);

/* NVFP4 with a logical (rows, dim/16) scale matrix. */
int orc_ln_quant_nvfp4(const uint16_t* x, const orc_mod_t* mod, float eps,
                       uint8_t* packed, uint8_t* sf_logical,
                       int64_t rows, int64_t dim, int nthreads);

/* NVFP4 with the swizzled scale buffer of orc_swizzled_sf_size(rows, dim) bytes. */
int orc_ln_quant_nvfp4_swizzled(const uint16_t* x, const orc_mod_t* mod, float eps,
                                uint8_t* packed, uint8_t* sf_swizzled,
                                int64_t rows, int64_t dim, int nthreads);

/* The bf16-staged modulated values v = bf16(fp32(y)) of the NVFP4 producers. */
int orc_ln_staged_bf16(const uint16_t* x, const orc_mod_t* mod, float eps, uint16_t* v,
                       int64_t rows, int64_t dim, int nthreads);

/* Two-level NVFP4 of bf16 values v (rows, dim): global amax -> fp32 tensor
 * scale (bf16-valued), e4m3 block scales relative to it, e2m1 codes.  Writes
 * packed (rows, dim/2), the swizzled scale buffer and *tensor_scale. */
int orc_nvfp4_2level(const uint16_t* v, int64_t rows, int64_t dim, uint8_t* packed,
                     uint8_t* sf_swizzled, float* tensor_scale, int nthreads);

/* LayerNorm producer with the two-level NVFP4 output. */
int orc_ln_quant_nvfp4_2level(const uint16_t* x, const orc_mod_t* mod, float eps, uint8_t* packed,
                              uint8_t* sf_swizzled, float* tensor_scale, int64_t rows, int64_t dim,
                              int nthreads);

/* SwiGLU values v = bf16(bf16(silu(gate)) * up) for (rows, dim) with row
 * stride ld (elements) for both inputs; v is (rows, dim) contiguous. */
int orc_swiglu_values(const uint16_t* gate, const uint16_t* up, int64_t ld, uint16_t* v,
                      int64_t rows, int64_t dim, int nthreads);

/* SwiGLU producer with the two-level NVFP4 output. */
int orc_swiglu_quant_nvfp4_2level(const uint16_t* gate, const uint16_t* up, int64_t ld, uint8_t* packed,
                                  uint8_t* sf_swizzled, float* tensor_scale, int64_t rows, int64_t dim,
                                  int nthreads);

/* six-way: out is (6, batch*seq, dim) bf16 bits; params (batch*seq, 6, dim). */
int orc_adaln_modulation6(const float* params, const float* modulation, uint16_t* out,
                          int64_t tokens, int64_t dim, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
