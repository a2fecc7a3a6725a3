/*
 * orc.c -- CPU oracle for the adaptive-LayerNorm activation producers.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the CUDA library.  Plain scalar C,
 * built with -O2 -ffp-contract=off and no fast-math so that every double and
 * float operation below is one IEEE-754 operation with round-to-nearest-even.
 *
 * What it computes (sources in orc.h):
 *   - "Available Functions" / "Tensor Contract" of the adaptive-layernorm-
 *     producers README: LayerNorm without affine over `dim`, adaptive
 *     modulation x_hat*(1+scale)+shift with a broadcast, per-token or
 *     temb+table source, then static e4m3fn quantisation or NVFP4 (e2m1 codes
 *     two per byte plus one e4m3 scale per 16 elements in the 128x4 swizzled
 *     layout), and the six-way fp32 -> bf16 modulation.
 *   - The README's "Validation" section: the NVFP4 producer follows a
 *     "staged BF16-norm plus FP4 quantizer" contract, i.e. the modulated value
 *     is materialised as bf16 before the FP4 quantiser sees it.
 *   - The h3-blackwell-runtime compare page: e2m1 rounding is
 *     round-to-nearest ties-to-even with signed zero kept (PLAN.md, "NVFP4
 *     activation quantization status"), packed low nibble first
 *     (gb10-cute-nvfp4-conversion-contract.json), and the block scales use
 *     the general 128-row by 4-scale-column tiled layout ("Phase 3: NVFP4
 *     Fused Projection Prototype").
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes of the repository):
 *   R1 statistics: biased variance, eps inside the square root (torch
 *      layer_norm semantics); computed here in double, two passes.
 *   R2 no intermediate rounding of (1+scale), of temb+table or of the FP8
 *      path's y; NVFP4 rounds y to bf16 (the staged contract).
 *   R3 FP8 quantisation divides by act_scale (act_scale is a dequant scale:
 *      value ~= code * act_scale); out-of-range values saturate to +-448.
 *   R4 NVFP4 block scale: s = e4m3(amax/6) with amax the largest |v| of the
 *      16-element block, single level (the producers take no global scale).
 *   R5 e2m1 code: nearest grid value to v/s_dec, ties to the even code,
 *      saturating at 6; a zero scale gives a signed zero code.
 *   R6 padding of the swizzled scale buffer is zero.
 *   R7 every value handed to a rounding step (y/act_scale for FP8, y for the
 *      bf16 stage, amax/6 for the block scale) is first rounded to binary32,
 *      the precision in which the GPU takes the same decision.
 *   R8 six-way: out_i = bf16(params[..., i, :] + modulation[i, :]) with the
 *      addition in binary32.
 *   R15 modfp8 producers: scale = decode(scale_fp8) * scale_deq and
 *      shift = decode(shift_fp8) * shift_deq, unrounded (double); the rest as
 *      for the broadcast producers.
 *   R16 AWQ producer: the bf16 smoothing vector inv_s multiplies the modulated
 *      activation, y * inv_s, before the FP8 quantiser (which then divides by
 *      act_scale as in R3).
 *   R17-R19 two-level NVFP4: see orc_nvfp4_2level.
 *   R20 segmented modulation: row r uses row seg_idx[r] of (nseg, dim) bf16
 *      scale/shift tables, with the broadcast producers' arithmetic.
 *   R21 SwiGLU: see orc_swiglu_values.
 */
#include "orc.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ======================================================================= */
/* bf16                                                                     */
/* ======================================================================= */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits_from_f32(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 is the upper half of a binary32 pattern. */
double orc_bf16_to_f64(uint16_t bits) { return (double)f32_from_bits((uint32_t)bits << 16); }

/* Nearest bf16 to a finite binary32 value, ties to the even pattern.
 * The two candidates are the truncation toward zero (`lo`) and the next bf16
 * away from zero (`hi`); both and `v` are exact in double, so are the two
 * distances (each is a difference of nearby binary32 values).  Past the
 * largest finite bf16 the next candidate is the infinity pattern, which
 * round-to-nearest treats as the value 2^128 (IEEE 754: a result at or
 * beyond the midpoint between the largest finite value and 2^128 overflows
 * to infinity). */
uint16_t orc_bf16_from_f32(float v) {
  uint32_t u = bits_from_f32(v);
  uint32_t lo = u & 0xFFFF0000u;
  if (lo == u) return (uint16_t)(lo >> 16);
  uint32_t hi = lo + 0x10000u;
  double dv = (double)v;
  double vhi = ((hi & 0x7FFFFFFFu) == 0x7F800000u) ? copysign(ldexp(1.0, 128), dv) : (double)f32_from_bits(hi);
  double dlo = fabs(dv - (double)f32_from_bits(lo));
  double dhi = fabs(vhi - dv);
  if (dlo < dhi) return (uint16_t)(lo >> 16);
  if (dhi < dlo) return (uint16_t)(hi >> 16);
  return ((lo >> 16) & 1u) ? (uint16_t)(hi >> 16) : (uint16_t)(lo >> 16);
}

/* ======================================================================= */
/* e4m3fn (OCP FP8: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits,   */
/* no infinities, S.1111.111 is NaN, largest finite 448)                    */
/* ======================================================================= */

double orc_e4m3_decode(uint8_t code) {
  int s = code >> 7, e = (code >> 3) & 0xF, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  double mag = (e == 0) ? ldexp((double)m, -9)          /* m/8 * 2^-6      */
                        : ldexp((double)(8 + m), e - 10); /* (1+m/8) * 2^(e-7) */
  return s ? -mag : mag;
}

/* Nearest finite e4m3fn value to v, ties to the even code, saturating.
 * Codes 0x00..0x7E are the non-negative finite values in increasing order and
 * the code's low bit is the mantissa's low bit, so "even code" is "even
 * mantissa".  A binary search finds the largest code not above |v|; the
 * answer is it or its successor.  Both distances are exact: consecutive
 * values differ by at most a factor of two (Sterbenz). */
uint8_t orc_e4m3_encode(double v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs(v);
  int c;
  if (a >= orc_e4m3_decode(0x7E)) {
    c = 0x7E;
  } else {
    int lo = 0, hi = 0x7E;
    while (lo < hi) {
      int mid = (lo + hi + 1) / 2;
      if (orc_e4m3_decode((uint8_t)mid) <= a) lo = mid; else hi = mid - 1;
    }
    c = lo;
    double d0 = a - orc_e4m3_decode((uint8_t)c);
    double d1 = orc_e4m3_decode((uint8_t)(c + 1)) - a;
    if (d1 < d0 || (d1 == d0 && (c & 1))) c += 1;
  }
  return (uint8_t)(sign | c);
}

/* ======================================================================= */
/* e2m1 (OCP FP4: 1 sign, 2 exponent bits with bias 1, 1 mantissa bit)     */
/* ======================================================================= */

double orc_e2m1_decode(uint8_t code4) {
  int s = (code4 >> 3) & 1, e = (code4 >> 1) & 3, m = code4 & 1;
  double mag = (e == 0) ? 0.5 * m                       /* subnormal: m/2  */
                        : ldexp((double)(2 + m), e - 2); /* (1+m/2)*2^(e-1) */
  return s ? -mag : mag;
}

/* Code of the e2m1 value nearest to v/s_dec, ties to the even code, with
 * saturation at 6 (the largest magnitude is simply the nearest one for any
 * quotient above 5).  Instead of dividing, the comparison is done on
 * |v| against g_k*s_dec: each g_k*s_dec has at most 7 significant bits, so it
 * and the distances near a tie are exact in double.  The sign of v is kept,
 * so a negative value that rounds to zero gives -0 (code 0x8).  A zero scale
 * (the whole block underflowed) gives signed zero codes. */
uint8_t orc_e2m1_encode(double v, double s_dec) {
  uint8_t sign = signbit(v) ? 0x8 : 0x0;
  if (s_dec == 0.0) return sign;
  double a = fabs(v);
  int best = 0;
  double best_d = a; /* distance to g_0 = 0 */
  for (int k = 1; k < 8; ++k) {
    double d = fabs(a - orc_e2m1_decode((uint8_t)k) * s_dec);
    if (d < best_d || (d == best_d && (k & 1) == 0)) { best = k; best_d = d; }
  }
  return (uint8_t)(sign | best);
}

/* ======================================================================= */
/* 128x4 swizzled block-scale layout                                         */
/* ======================================================================= */

static int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

/* Bytes of the swizzled scale buffer: the logical (rows, dim/16) scale
 * matrix padded to whole 128-row x 4-column tiles (README "Tensor Contract":
 * allocate with swizzled_sf_size(rows, dim); dim divisible by 16). */
int64_t orc_swizzled_sf_size(int64_t rows, int64_t dim) {
  if (rows < 0 || dim <= 0 || dim % 16 != 0) return -1;
  return round_up(rows, 128) * round_up(dim / 16, 4);
}

/* Byte offset of the scale of row r, block column c.  Tiles of 128 rows x 4
 * columns are 512 contiguous bytes, ordered row-tile major.  Inside a tile the
 * 128 rows are four 32-row groups; the 16-byte chunk index is r%32 and a
 * chunk holds, for that r%32, the 4 groups x 4 columns (group-major). */
int64_t orc_sf_offset(int64_t r, int64_t c, int64_t dim) {
  int64_t col_tiles = round_up(dim / 16, 4) / 4;
  int64_t tile = (r / 128) * col_tiles + (c / 4);
  return tile * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
}

void orc_swizzle_scales(const uint8_t* sf_logical, int64_t rows, int64_t dim, uint8_t* out) {
  int64_t nblk = dim / 16;
  int64_t size = orc_swizzled_sf_size(rows, dim);
  memset(out, 0, (size_t)size);
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < nblk; ++c) out[orc_sf_offset(r, c, dim)] = sf_logical[r * nblk + c];
}

/* ======================================================================= */
/* LayerNorm statistics and modulation                                       */
/* ======================================================================= */

/* Mean and 1/sqrt(var + eps) of one row, double, two passes (reading R1). */
void orc_row_stats(const uint16_t* x, int64_t dim, float eps, double* mean, double* rstd) {
  double s = 0.0;
  for (int64_t d = 0; d < dim; ++d) s += orc_bf16_to_f64(x[d]);
  double mu = s / (double)dim;
  double q = 0.0;
  for (int64_t d = 0; d < dim; ++d) {
    double t = orc_bf16_to_f64(x[d]) - mu;
    q += t * t;
  }
  double var = q / (double)dim;
  *mean = mu;
  *rstd = 1.0 / sqrt(var + (double)eps);
}

/* Scale and shift of element (r, d) for each modulation source (README
 * "Available Functions"/"Tensor Contract"; table form: "Fused host modulation
 * table add and chunk selection" in "Minimal Usage"). */
static void mod_at(const orc_mod_t* m, int64_t r, int64_t d, int64_t dim,
                   double* scale, double* shift) {
  switch (m->kind) {
    case ORC_MOD_BCAST:
      *scale = orc_bf16_to_f64(m->scale[d]);
      *shift = orc_bf16_to_f64(m->shift[d]);
      return;
    case ORC_MOD_PTOK:
      *scale = orc_bf16_to_f64(m->scale[r * dim + d]);
      *shift = orc_bf16_to_f64(m->shift[r * dim + d]);
      return;
    case ORC_MOD_TABLE: {
      const uint16_t* te = m->temb + r * m->chunks * dim;
      *scale = orc_bf16_to_f64(te[m->scale_idx * dim + d]) + (double)m->table[m->scale_idx * dim + d];
      *shift = orc_bf16_to_f64(te[m->shift_idx * dim + d]) + (double)m->table[m->shift_idx * dim + d];
      return;
    }
    case ORC_MOD_MODFP8:
      /* e4m3 (dim,) vectors, each dequantised by its own fp32 scalar
       * (README "Available Functions": the *_modfp8_* producers; "Tensor
       * Contract": scale_fp8/shift_fp8 e4m3 (dim,), scale_deq/shift_deq fp32
       * scalars).  Reading R15: value = decode(code) * deq, exact in double. */
      *scale = orc_e4m3_decode(m->scale_fp8[d]) * (double)m->scale_deq;
      *shift = orc_e4m3_decode(m->shift_fp8[d]) * (double)m->shift_deq;
      return;
    case ORC_MOD_AWQ:
      /* bf16 broadcast scale/shift as in BCAST; inv_s is applied by
       * modulated_row (README "Available Functions": awq_ada_layer_norm_...). */
      *scale = orc_bf16_to_f64(m->scale[d]);
      *shift = orc_bf16_to_f64(m->shift[d]);
      return;
    case ORC_MOD_SEG: {
      /* segmented modulation (h3-blackwell-runtime compare page: "segment-
       * specific shift and scale selection", the request-layout segment index
       * of Phase 1): row r takes row seg_idx[r] of the (nseg, dim) tables. */
      const int64_t g = m->seg_idx[r];
      *scale = orc_bf16_to_f64(m->seg_scale[g * dim + d]);
      *shift = orc_bf16_to_f64(m->seg_shift[g * dim + d]);
      return;
    }
    default:
      *scale = 0.0;
      *shift = 0.0;
      return;
  }
}

/* y[d] = (x[d] - mean) * rstd * (1 + scale) + shift, double.
 * AWQ (reading R16): the smoothing multiplier is applied to the modulated
 * activation, y[d] *= inv_s[d], before it is quantised -- the quantised
 * tensor is the input of the smoothed GEMM, whose weights carry s. */
static void modulated_row(const uint16_t* xr, const orc_mod_t* m, int64_t r, float eps,
                          double* y, int64_t dim) {
  double mu, rstd;
  orc_row_stats(xr, dim, eps, &mu, &rstd);
  for (int64_t d = 0; d < dim; ++d) {
    double sc, sh;
    mod_at(m, r, d, dim, &sc, &sh);
    double xhat = (orc_bf16_to_f64(xr[d]) - mu) * rstd;
    y[d] = xhat * (1.0 + sc) + sh;
    if (m->kind == ORC_MOD_AWQ) y[d] *= orc_bf16_to_f64(m->inv_s[d]);
  }
}

/* ======================================================================= */
/* row-parallel driver                                                       */
/* ======================================================================= */

typedef void (*row_fn)(void* ctx, int64_t r, double* scratch);
typedef struct {
  row_fn fn; void* ctx; int64_t r0, r1, dim;
} span_t;

static void* run_span(void* p) {
  span_t* s = (span_t*)p;
  double* scratch = (double*)malloc(sizeof(double) * (size_t)(s->dim > 0 ? s->dim : 1));
  for (int64_t r = s->r0; r < s->r1; ++r) s->fn(s->ctx, r, scratch);
  free(scratch);
  return NULL;
}

static void for_rows(row_fn fn, void* ctx, int64_t rows, int64_t dim, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((int64_t)nthreads > rows) nthreads = (int)(rows > 0 ? rows : 1);
  span_t spans[256];
  pthread_t tids[256];
  int64_t per = (rows + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    spans[t].fn = fn; spans[t].ctx = ctx; spans[t].dim = dim;
    spans[t].r0 = (int64_t)t * per < rows ? (int64_t)t * per : rows;
    spans[t].r1 = spans[t].r0 + per < rows ? spans[t].r0 + per : rows;
  }
  if (nthreads == 1) { run_span(&spans[0]); return; }
  for (int t = 0; t < nthreads; ++t) pthread_create(&tids[t], NULL, run_span, &spans[t]);
  for (int t = 0; t < nthreads; ++t) pthread_join(tids[t], NULL);
}

/* ======================================================================= */
/* producers                                                                 */
/* ======================================================================= */

typedef struct {
  const uint16_t* x; const orc_mod_t* mod; float eps; int64_t dim;
  double* y; float act_scale; uint8_t* out; uint8_t* packed; uint8_t* sf;
} op_ctx;

static void row_modulated(void* p, int64_t r, double* scratch) {
  op_ctx* c = (op_ctx*)p;
  (void)scratch;
  modulated_row(c->x + r * c->dim, c->mod, r, c->eps, c->y + r * c->dim, c->dim);
}

int orc_modulated_rows(const uint16_t* x, const orc_mod_t* mod, float eps, double* y,
                       int64_t rows, int64_t dim, int nthreads) {
  if (rows < 0 || dim <= 0) return -1;
  op_ctx c = {x, mod, eps, dim, y, 0.f, NULL, NULL, NULL};
  for_rows(row_modulated, &c, rows, dim, nthreads);
  return 0;
}

/* FP8 row: code = e4m3(fp32(y / act_scale)) (readings R3, R7). */
static void row_fp8(void* p, int64_t r, double* y) {
  op_ctx* c = (op_ctx*)p;
  modulated_row(c->x + r * c->dim, c->mod, r, c->eps, y, c->dim);
  uint8_t* o = c->out + r * c->dim;
  for (int64_t d = 0; d < c->dim; ++d) {
    float t = (float)(y[d] / (double)c->act_scale);
    o[d] = orc_e4m3_encode((double)t);
  }
}

int orc_ln_quant_fp8(const uint16_t* x, const orc_mod_t* mod, float act_scale, float eps,
                     uint8_t* out, int64_t rows, int64_t dim, int nthreads) {
  if (rows < 0 || dim <= 0) return -1;
  op_ctx c = {x, mod, eps, dim, NULL, act_scale, out, NULL, NULL};
  for_rows(row_fp8, &c, rows, dim, nthreads);
  return 0;
}

/* NVFP4 row (readings R2, R4, R5, R7):
 *   v = bf16(fp32(y));  per 16-element block: amax = max|v|,
 *   s = e4m3(fp32(amax/6)); code = e2m1 nearest of v/decode(s);
 *   element 2k goes to the low nibble of byte k, 2k+1 to the high nibble. */
static void row_nvfp4(void* p, int64_t r, double* y) {
  op_ctx* c = (op_ctx*)p;
  int64_t dim = c->dim, nblk = dim / 16;
  modulated_row(c->x + r * dim, c->mod, r, c->eps, y, dim);
  uint8_t* pk = c->packed + r * (dim / 2);
  uint8_t* sf = c->sf + r * nblk;
  for (int64_t b = 0; b < nblk; ++b) {
    double v[16];
    double amax = 0.0;
    for (int k = 0; k < 16; ++k) {
      v[k] = orc_bf16_to_f64(orc_bf16_from_f32((float)y[b * 16 + k]));
      if (fabs(v[k]) > amax) amax = fabs(v[k]);
    }
    uint8_t s = orc_e4m3_encode((double)(float)(amax / 6.0));
    double s_dec = orc_e4m3_decode(s);
    sf[b] = s;
    for (int k = 0; k < 16; k += 2) {
      uint8_t lo = orc_e2m1_encode(v[k], s_dec);
      uint8_t hi = orc_e2m1_encode(v[k + 1], s_dec);
      pk[b * 8 + k / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

int orc_ln_quant_nvfp4(const uint16_t* x, const orc_mod_t* mod, float eps,
                       uint8_t* packed, uint8_t* sf_logical,
                       int64_t rows, int64_t dim, int nthreads) {
  if (rows < 0 || dim <= 0 || dim % 16 != 0) return -1;
  op_ctx c = {x, mod, eps, dim, NULL, 0.f, NULL, packed, sf_logical};
  for_rows(row_nvfp4, &c, rows, dim, nthreads);
  return 0;
}

int orc_ln_quant_nvfp4_swizzled(const uint16_t* x, const orc_mod_t* mod, float eps,
                                uint8_t* packed, uint8_t* sf_swizzled,
                                int64_t rows, int64_t dim, int nthreads) {
  if (rows < 0 || dim <= 0 || dim % 16 != 0) return -1;
  uint8_t* logical = (uint8_t*)malloc((size_t)(rows * (dim / 16) + 1));
  if (!logical) return -2;
  int rc = orc_ln_quant_nvfp4(x, mod, eps, packed, logical, rows, dim, nthreads);
  if (rc == 0) orc_swizzle_scales(logical, rows, dim, sf_swizzled);
  free(logical);
  return rc;
}

/* ---- staged values and the two-level NVFP4 contract ---------------------- */

typedef struct {
  const uint16_t* x; const orc_mod_t* mod; float eps; int64_t dim; uint16_t* v;
} stage_ctx;

static void row_stage(void* p, int64_t r, double* y) {
  stage_ctx* c = (stage_ctx*)p;
  modulated_row(c->x + r * c->dim, c->mod, r, c->eps, y, c->dim);
  for (int64_t d = 0; d < c->dim; ++d) c->v[r * c->dim + d] = orc_bf16_from_f32((float)y[d]);
}

int orc_ln_staged_bf16(const uint16_t* x, const orc_mod_t* mod, float eps, uint16_t* v,
                       int64_t rows, int64_t dim, int nthreads) {
  if (rows < 0 || dim <= 0) return -1;
  stage_ctx c = {x, mod, eps, dim, v};
  for_rows(row_stage, &c, rows, dim, nthreads);
  return 0;
}

/* Two-level NVFP4 (h3-blackwell-runtime compare page: NVFP4_STREAMING_DESIGN.md
 * "Numerical Constraint" -- one exact global bf16 absolute maximum, one fp32
 * tensor scale derived from it, e4m3 block scales per 16 values, e2m1 codes
 * using both scales; the P1 producer-consumer checkpoint's
 * "numerical_contract" -- block scale (amax / 6.0f) / global_scale clamped by
 * fminf(., 448.0f)).  Readings:
 *   R17 tensor scale ts = bf16(fp32(amax_g / 2688)), 2688 = 6 (largest e2m1)
 *       x 448 (largest e4m3); every tensor scale the page prints is a bf16
 *       value.  All-zero input: ts = 0.
 *   R18 block scale s = e4m3(fminf(fp32(fp32(amax_b / 6) / ts), 448)), both
 *       divisions fp32 as printed; fminf returns 448 for the 0/0 of an
 *       all-zero tensor, which reproduces the page's scale byte 126 there.
 *   R19 code = e2m1 nearest of v / (decode(s) * ts), exact quotient (the
 *       product is exact); a zero denominator gives signed zeros.  The page's
 *       approximate reciprocal is replaced by the exact quotient, as in R5. */
typedef struct {
  const uint16_t* v; int64_t dim; uint8_t* packed; uint8_t* sf; float ts;
} tl_ctx;

static void row_2level(void* p, int64_t r, double* scratch) {
  tl_ctx* c = (tl_ctx*)p;
  (void)scratch;
  const int64_t dim = c->dim, nblk = dim / 16;
  const uint16_t* vr = c->v + r * dim;
  uint8_t* pk = c->packed + r * (dim / 2);
  uint8_t* sf = c->sf + r * nblk;
  for (int64_t b = 0; b < nblk; ++b) {
    double amax = 0.0;
    for (int k = 0; k < 16; ++k) {
      const double a = fabs(orc_bf16_to_f64(vr[b * 16 + k]));
      if (a > amax) amax = a;
    }
    float q = (float)amax / 6.0f;
    q = q / c->ts;
    q = fminf(q, 448.0f);
    const uint8_t s = orc_e4m3_encode((double)q);
    sf[b] = s;
    const double den = orc_e4m3_decode(s) * (double)c->ts;
    for (int k = 0; k < 16; k += 2) {
      const uint8_t lo = orc_e2m1_encode(orc_bf16_to_f64(vr[b * 16 + k]), den);
      const uint8_t hi = orc_e2m1_encode(orc_bf16_to_f64(vr[b * 16 + k + 1]), den);
      pk[b * 8 + k / 2] = (uint8_t)(lo | (hi << 4));
    }
  }
}

int orc_nvfp4_2level(const uint16_t* v, int64_t rows, int64_t dim, uint8_t* packed,
                     uint8_t* sf_swizzled, float* tensor_scale, int nthreads) {
  if (rows < 0 || dim <= 0 || dim % 16 != 0) return -1;
  double amax = 0.0;
  for (int64_t i = 0; i < rows * dim; ++i) {
    const double a = fabs(orc_bf16_to_f64(v[i]));
    if (a > amax) amax = a;
  }
  const float ts = (float)orc_bf16_to_f64(orc_bf16_from_f32((float)amax / 2688.0f));
  uint8_t* logical = (uint8_t*)malloc((size_t)(rows * (dim / 16) + 1));
  if (!logical) return -2;
  tl_ctx c = {v, dim, packed, logical, ts};
  for_rows(row_2level, &c, rows, dim, nthreads);
  orc_swizzle_scales(logical, rows, dim, sf_swizzled);
  free(logical);
  *tensor_scale = ts;
  return 0;
}

int orc_ln_quant_nvfp4_2level(const uint16_t* x, const orc_mod_t* mod, float eps, uint8_t* packed,
                              uint8_t* sf_swizzled, float* tensor_scale, int64_t rows, int64_t dim,
                              int nthreads) {
  if (rows < 0 || dim <= 0 || dim % 16 != 0) return -1;
  uint16_t* v = (uint16_t*)malloc((size_t)(rows * dim + 1) * sizeof(uint16_t));
  if (!v) return -2;
  int rc = orc_ln_staged_bf16(x, mod, eps, v, rows, dim, nthreads);
  if (rc == 0) rc = orc_nvfp4_2level(v, rows, dim, packed, sf_swizzled, tensor_scale, nthreads);
  free(v);
  return rc;
}

/* ---- SwiGLU producer (h3-blackwell-runtime compare page:
 * NVFP4_SWIGLU_FUSION_DESIGN.md -- the two bf16 boundaries: silu(gate)
 * rounded to bf16, then that bf16 value times bf16 up rounded to bf16; then the
 * tensor scale, e4m3 block scales and e2m1 codes of the two-level contract).
 * Reading R21: silu(g) = g / (1 + exp(-g)) in double, rounded to binary32 and
 * then to bf16 (R7: the value is first rounded to the precision in which the
 * GPU takes the decision); the product of two bf16 values is exact in double
 * and in binary32, then rounded to bf16. ------------------------------------ */
typedef struct {
  const uint16_t* gate; const uint16_t* up; int64_t ld, dim; uint16_t* v;
} sw_ctx;

static void row_swiglu(void* p, int64_t r, double* scratch) {
  sw_ctx* c = (sw_ctx*)p;
  (void)scratch;
  for (int64_t d = 0; d < c->dim; ++d) {
    const double g = orc_bf16_to_f64(c->gate[r * c->ld + d]);
    const double u = orc_bf16_to_f64(c->up[r * c->ld + d]);
    const double silu = g / (1.0 + exp(-g));
    const double s = orc_bf16_to_f64(orc_bf16_from_f32((float)silu));
    c->v[r * c->dim + d] = orc_bf16_from_f32((float)(s * u));
  }
}

int orc_swiglu_values(const uint16_t* gate, const uint16_t* up, int64_t ld, uint16_t* v,
                      int64_t rows, int64_t dim, int nthreads) {
  if (rows < 0 || dim <= 0 || ld < dim) return -1;
  sw_ctx c = {gate, up, ld, dim, v};
  for_rows(row_swiglu, &c, rows, dim, nthreads);
  return 0;
}

int orc_swiglu_quant_nvfp4_2level(const uint16_t* gate, const uint16_t* up, int64_t ld, uint8_t* packed,
                                  uint8_t* sf_swizzled, float* tensor_scale, int64_t rows, int64_t dim,
                                  int nthreads) {
  if (rows < 0 || dim <= 0 || dim % 16 != 0 || ld < dim) return -1;
  uint16_t* v = (uint16_t*)malloc((size_t)(rows * dim + 1) * sizeof(uint16_t));
  if (!v) return -2;
  int rc = orc_swiglu_values(gate, up, ld, v, rows, dim, nthreads);
  if (rc == 0) rc = orc_nvfp4_2level(v, rows, dim, packed, sf_swizzled, tensor_scale, nthreads);
  free(v);
  return rc;
}

/* ======================================================================= */
/* six-way modulation (README "Tensor Contract": fp32 (batch, seq, 6, dim)   */
/* params plus fp32 (6, dim) modulation -> six bf16 (batch, seq, dim))       */
/* ======================================================================= */

typedef struct {
  const float* params; const float* mod; uint16_t* out; int64_t tokens, dim;
} m6_ctx;

static void row_m6(void* p, int64_t t, double* scratch) {
  m6_ctx* c = (m6_ctx*)p;
  (void)scratch;
  for (int i = 0; i < 6; ++i) {
    const float* pr = c->params + (t * 6 + i) * c->dim;
    const float* mr = c->mod + i * c->dim;
    uint16_t* o = c->out + ((int64_t)i * c->tokens + t) * c->dim;
    for (int64_t d = 0; d < c->dim; ++d) {
      float s = pr[d] + mr[d]; /* one binary32 addition (reading R8) */
      o[d] = orc_bf16_from_f32(s);
    }
  }
}

int orc_adaln_modulation6(const float* params, const float* modulation, uint16_t* out,
                          int64_t tokens, int64_t dim, int nthreads) {
  if (tokens < 0 || dim <= 0) return -1;
  m6_ctx c = {params, modulation, out, tokens, dim};
  for_rows(row_m6, &c, tokens, 0, nthreads);
  return 0;
}
