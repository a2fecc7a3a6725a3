/* abi_stub.c -- a stand-in for libnvfp4ap.so's producer entry points, built by
 * tests/test_pycall_marshal.py on the CPU: each function records its name and
 * arguments (pointers and integers as 64-bit words, floats as their bit
 * pattern, the six outputs of adaln_modulation6_bf16 in order) and returns a
 * status that identifies it.  The test calls it through the binding's ctypes
 * declarations and through the C marshalling module and compares the records.
 */
#include <stdint.h>
#include <string.h>

#include "nvfp4ap.h"

static char g_name[96];
static uint64_t g_args[24];
static int g_n;

static void start(const char* name) {
  strncpy(g_name, name, sizeof(g_name) - 1);
  g_n = 0;
}
static void pp(const void* p) { g_args[g_n++] = (uint64_t)(uintptr_t)p; }
static void pi(int64_t v) { g_args[g_n++] = (uint64_t)v; }
static void pf(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  g_args[g_n++] = u;
}

/* the last call: its name into `name` (96 bytes), its words into `out` (24); returns their count */
__attribute__((visibility("default"))) int stub_last(char* name, uint64_t* out) {
  memcpy(name, g_name, sizeof(g_name));
  memcpy(out, g_args, sizeof(g_args));
  return g_n;
}

int ada_layer_norm_quant_fp8_bf16(const void* x, const void* scale, const void* shift, const float* act_scale,
                                  float eps, void* out, int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(scale); pp(shift); pp(act_scale); pf(eps); pp(out); pi(rows); pi(dim); pp(stream);
  return 101;
}
int ada_layer_norm_quant_fp8_bf16_noalloc(const void* x, const void* scale, const void* shift, const float* act_scale,
                                          float eps, void* out, int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(scale); pp(shift); pp(act_scale); pf(eps); pp(out); pi(rows); pi(dim); pp(stream);
  return 102;
}
int ada_layer_norm_quant_fp8_ptok_bf16(const void* x, const void* scale, const void* shift, const float* act_scale,
                                       float eps, void* out, int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(scale); pp(shift); pp(act_scale); pf(eps); pp(out); pi(rows); pi(dim); pp(stream);
  return 103;
}
int ada_layer_norm_quant_fp8_ptok_table_bf16(const void* x, const void* temb, const float* table, int64_t chunks,
                                             int64_t shift_idx, int64_t scale_idx, const float* act_scale, float eps,
                                             void* out, int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(temb); pp(table); pi(chunks); pi(shift_idx); pi(scale_idx); pp(act_scale); pf(eps);
  pp(out); pi(rows); pi(dim); pp(stream);
  return 104;
}
int ada_layer_norm_quant_fp8_modfp8_bf16(const void* x, const void* scale_fp8, const void* shift_fp8,
                                         const float* scale_deq, const float* shift_deq, const float* act_scale,
                                         float eps, void* out, int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(scale_fp8); pp(shift_fp8); pp(scale_deq); pp(shift_deq); pp(act_scale); pf(eps);
  pp(out); pi(rows); pi(dim); pp(stream);
  return 105;
}
int awq_ada_layer_norm_quant_fp8_bf16(const void* x, const void* scale, const void* shift, const void* inv_s,
                                      const float* act_scale, float eps, void* out, int64_t rows, int64_t dim,
                                      nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(scale); pp(shift); pp(inv_s); pp(act_scale); pf(eps); pp(out); pi(rows); pi(dim);
  pp(stream);
  return 106;
}
int ada_layer_norm_quant_fp8_seg_bf16(const void* x, const int32_t* seg_idx, const void* seg_scale,
                                      const void* seg_shift, int64_t nseg, const float* act_scale, float eps,
                                      void* out, int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(seg_idx); pp(seg_scale); pp(seg_shift); pi(nseg); pp(act_scale); pf(eps); pp(out);
  pi(rows); pi(dim); pp(stream);
  return 107;
}
int layer_norm_no_affine_quant_fp8_static_bf16(const void* x, const float* act_scale, float eps, void* out,
                                               int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(act_scale); pf(eps); pp(out); pi(rows); pi(dim); pp(stream);
  return 108;
}
int ada_layer_norm_quant_nvfp4_swizzled_bf16(const void* x, const void* scale, const void* shift, float eps,
                                             void* packed, void* sf_swizzled, int64_t rows, int64_t dim,
                                             nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(scale); pp(shift); pf(eps); pp(packed); pp(sf_swizzled); pi(rows); pi(dim); pp(stream);
  return 109;
}
int ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(const void* x, const void* scale_fp8, const void* shift_fp8,
                                                    const float* scale_deq, const float* shift_deq, float eps,
                                                    void* packed, void* sf_swizzled, int64_t rows, int64_t dim,
                                                    nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(scale_fp8); pp(shift_fp8); pp(scale_deq); pp(shift_deq); pf(eps); pp(packed);
  pp(sf_swizzled); pi(rows); pi(dim); pp(stream);
  return 110;
}
int layer_norm_no_affine_quant_nvfp4_swizzled_bf16(const void* x, float eps, void* packed, void* sf_swizzled,
                                                   int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pf(eps); pp(packed); pp(sf_swizzled); pi(rows); pi(dim); pp(stream);
  return 111;
}
int ada_layer_norm_quant_nvfp4_swizzled_seg_bf16(const void* x, const int32_t* seg_idx, const void* seg_scale,
                                                 const void* seg_shift, int64_t nseg, float eps, void* packed,
                                                 void* sf_swizzled, int64_t rows, int64_t dim,
                                                 nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(seg_idx); pp(seg_scale); pp(seg_shift); pi(nseg); pf(eps); pp(packed);
  pp(sf_swizzled); pi(rows); pi(dim); pp(stream);
  return 112;
}
int layer_norm_no_affine_quant_nvfp4_2level_bf16(const void* x, float eps, void* packed, void* sf_swizzled,
                                                 float* tensor_scale, void* workspace, int64_t rows, int64_t dim,
                                                 nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pf(eps); pp(packed); pp(sf_swizzled); pp(tensor_scale); pp(workspace); pi(rows); pi(dim);
  pp(stream);
  return 113;
}
int ada_layer_norm_quant_nvfp4_2level_bf16(const void* x, const void* scale, const void* shift, float eps,
                                           void* packed, void* sf_swizzled, float* tensor_scale, void* workspace,
                                           int64_t rows, int64_t dim, nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(scale); pp(shift); pf(eps); pp(packed); pp(sf_swizzled); pp(tensor_scale);
  pp(workspace); pi(rows); pi(dim); pp(stream);
  return 114;
}
int ada_layer_norm_quant_nvfp4_2level_seg_bf16(const void* x, const int32_t* seg_idx, const void* seg_scale,
                                               const void* seg_shift, int64_t nseg, float eps, void* packed,
                                               void* sf_swizzled, float* tensor_scale, void* workspace, int64_t rows,
                                               int64_t dim, nvfp4ap_stream_t stream) {
  start(__func__); pp(x); pp(seg_idx); pp(seg_scale); pp(seg_shift); pi(nseg); pf(eps); pp(packed);
  pp(sf_swizzled); pp(tensor_scale); pp(workspace); pi(rows); pi(dim); pp(stream);
  return 115;
}
int swiglu_quant_nvfp4_2level_bf16(const void* gate, const void* up, int64_t ld, void* packed, void* sf_swizzled,
                                   float* tensor_scale, void* workspace, int64_t rows, int64_t dim,
                                   nvfp4ap_stream_t stream) {
  start(__func__); pp(gate); pp(up); pi(ld); pp(packed); pp(sf_swizzled); pp(tensor_scale); pp(workspace);
  pi(rows); pi(dim); pp(stream);
  return 116;
}
int swiglu_bf16(const void* gate, const void* up, int64_t ld, void* out, int64_t rows, int64_t dim,
                nvfp4ap_stream_t stream) {
  start(__func__); pp(gate); pp(up); pi(ld); pp(out); pi(rows); pi(dim); pp(stream);
  return 117;
}
int adaln_modulation6_bf16(const float* params, const float* modulation, void* const out[6], int64_t batch,
                           int64_t seq, int64_t dim, nvfp4ap_stream_t stream) {
  start(__func__); pp(params); pp(modulation);
  for (int j = 0; j < 6; ++j) pp(out[j]);
  pi(batch); pi(seq); pi(dim); pp(stream);
  return 118;
}

/* the other entry points, so that the binding's declarations resolve */
int64_t nvfp4ap_2level_workspace_bytes(int64_t rows) { return 16 + 16 * rows; }
const char* nvfp4ap_status_string(int status) { return status ? "stub status" : "ok"; }
int nvfp4ap_version(void) { return 0; }
int nvfp4ap_take_device_fault(void) { return 0; }
int nvfp4ap_set_wait_limit(int64_t cycles) { (void)cycles; return 0; }
int64_t nvfp4ap_wait_limit(void) { return 0; }
int nvfp4ap_noalloc_progress(uint32_t* words, int64_t n, int64_t* used) {
  (void)words; (void)n;
  if (used) *used = 0;
  return 0;
}
int nvfp4ap_2level_single_read(int64_t rows, int64_t dim, int modulation, int* single_read) {
  (void)rows; (void)dim; (void)modulation;
  if (single_read) *single_read = 0;
  return 0;
}
int64_t swizzled_sf_size(int64_t rows, int64_t dim) { return (rows + 127) / 128 * 128 * ((dim / 16 + 3) / 4 * 4); }
