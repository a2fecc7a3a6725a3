/* pycall.c -- CPython argument marshalling for the producer entry points of
 * libnvfp4ap.so (include/nvfp4ap.h).
 *
 * Each function converts its Python arguments (ints for device pointers,
 * stream handles and sizes, None for a null pointer, a float for eps) into the
 * C types of the entry point of the same name and calls it; it returns the
 * entry point's status as an int.  No other work is done here: the library
 * validates every argument.  This replaces a ctypes call (about 3.4 us of host
 * time per call on a Grace core) by a direct C call (a fraction of a
 * microsecond).
 *
 * The entry points are resolved with dlopen/dlsym on the library path the
 * Python binding loads (bind(path)), so both refer to one loaded copy of the
 * library and its state (device fault words, launch-shape caches).  The
 * function-pointer types are taken from the header's prototypes, so every
 * call is type-checked against the C ABI.
 */
#define PY_SSIZE_T_CLEAN
#include <Python.h>
#include <dlfcn.h>
#include <stdint.h>
#include <string.h>

#include "nvfp4ap.h"

typedef union {
  void* p;
  int64_t i;
  float f;
} Arg;

/* sig: one letter per argument: p pointer (int or None), i int64, f float,
 * - skipped (converted by the caller) */
static int conv(PyObject* const* args, Py_ssize_t n, const char* sig, Arg* a, const char* name) {
  const Py_ssize_t want = (Py_ssize_t)strlen(sig);
  if (n != want) {
    PyErr_Format(PyExc_TypeError, "%s: %zd arguments given, %zd expected", name, n, want);
    return -1;
  }
  for (Py_ssize_t k = 0; k < n; ++k) {
    PyObject* o = args[k];
    switch (sig[k]) {
      case 'p':
        a[k].p = (o == Py_None) ? NULL : PyLong_AsVoidPtr(o);
        break;
      case 'i':
        a[k].i = (int64_t)PyLong_AsLongLong(o);
        break;
      case 'f':
        a[k].f = (float)PyFloat_AsDouble(o);
        break;
      default:
        break;
    }
    if (PyErr_Occurred()) return -1;
  }
  return 0;
}

#define ENTRY_POINTS(X)                               \
  X(ada_layer_norm_quant_fp8_bf16)                    \
  X(ada_layer_norm_quant_fp8_bf16_noalloc)            \
  X(ada_layer_norm_quant_fp8_ptok_bf16)               \
  X(ada_layer_norm_quant_fp8_ptok_table_bf16)         \
  X(ada_layer_norm_quant_fp8_modfp8_bf16)             \
  X(awq_ada_layer_norm_quant_fp8_bf16)                \
  X(ada_layer_norm_quant_fp8_seg_bf16)                \
  X(layer_norm_no_affine_quant_fp8_static_bf16)       \
  X(ada_layer_norm_quant_nvfp4_swizzled_bf16)         \
  X(ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16)  \
  X(layer_norm_no_affine_quant_nvfp4_swizzled_bf16)   \
  X(ada_layer_norm_quant_nvfp4_swizzled_seg_bf16)     \
  X(layer_norm_no_affine_quant_nvfp4_2level_bf16)     \
  X(ada_layer_norm_quant_nvfp4_2level_bf16)           \
  X(ada_layer_norm_quant_nvfp4_2level_seg_bf16)       \
  X(swiglu_quant_nvfp4_2level_bf16)                   \
  X(swiglu_bf16)                                      \
  X(adaln_modulation6_bf16)

#define DECLARE_PTR(name) static __typeof__(&name) p_##name = NULL;
ENTRY_POINTS(DECLARE_PTR)

#define BEGIN(name, sig)                                                                  \
  static PyObject* py_##name(PyObject* self, PyObject* const* args, Py_ssize_t n) {      \
    Arg a[16];                                                                            \
    int rc;                                                                               \
    (void)self;                                                                           \
    if (p_##name == NULL) {                                                               \
      PyErr_SetString(PyExc_RuntimeError, #name ": call bind(library path) first");       \
      return NULL;                                                                        \
    }                                                                                     \
    if (conv(args, n, sig, a, #name)) return NULL;
#define END          \
  return PyLong_FromLong(rc); \
  }
#define P(k) (a[k].p)
#define FP(k) ((float*)a[k].p)
#define IP(k) ((const int32_t*)a[k].p)
#define I(k) (a[k].i)
#define F(k) (a[k].f)
#define S(k) ((nvfp4ap_stream_t)a[k].p)

BEGIN(ada_layer_norm_quant_fp8_bf16, "ppppfpiip")
rc = p_ada_layer_norm_quant_fp8_bf16(P(0), P(1), P(2), FP(3), F(4), P(5), I(6), I(7), S(8));
END

BEGIN(ada_layer_norm_quant_fp8_bf16_noalloc, "ppppfpiip")
rc = p_ada_layer_norm_quant_fp8_bf16_noalloc(P(0), P(1), P(2), FP(3), F(4), P(5), I(6), I(7), S(8));
END

BEGIN(ada_layer_norm_quant_fp8_ptok_bf16, "ppppfpiip")
rc = p_ada_layer_norm_quant_fp8_ptok_bf16(P(0), P(1), P(2), FP(3), F(4), P(5), I(6), I(7), S(8));
END

BEGIN(ada_layer_norm_quant_fp8_ptok_table_bf16, "pppiiipfpiip")
rc = p_ada_layer_norm_quant_fp8_ptok_table_bf16(P(0), P(1), FP(2), I(3), I(4), I(5), FP(6), F(7), P(8), I(9), I(10),
                                                S(11));
END

BEGIN(ada_layer_norm_quant_fp8_modfp8_bf16, "ppppppfpiip")
rc = p_ada_layer_norm_quant_fp8_modfp8_bf16(P(0), P(1), P(2), FP(3), FP(4), FP(5), F(6), P(7), I(8), I(9), S(10));
END

BEGIN(awq_ada_layer_norm_quant_fp8_bf16, "pppppfpiip")
rc = p_awq_ada_layer_norm_quant_fp8_bf16(P(0), P(1), P(2), P(3), FP(4), F(5), P(6), I(7), I(8), S(9));
END

BEGIN(ada_layer_norm_quant_fp8_seg_bf16, "ppppipfpiip")
rc = p_ada_layer_norm_quant_fp8_seg_bf16(P(0), IP(1), P(2), P(3), I(4), FP(5), F(6), P(7), I(8), I(9), S(10));
END

BEGIN(layer_norm_no_affine_quant_fp8_static_bf16, "ppfpiip")
rc = p_layer_norm_no_affine_quant_fp8_static_bf16(P(0), FP(1), F(2), P(3), I(4), I(5), S(6));
END

BEGIN(ada_layer_norm_quant_nvfp4_swizzled_bf16, "pppfppiip")
rc = p_ada_layer_norm_quant_nvfp4_swizzled_bf16(P(0), P(1), P(2), F(3), P(4), P(5), I(6), I(7), S(8));
END

BEGIN(ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16, "pppppfppiip")
rc = p_ada_layer_norm_quant_nvfp4_swizzled_modfp8_bf16(P(0), P(1), P(2), FP(3), FP(4), F(5), P(6), P(7), I(8), I(9),
                                                       S(10));
END

BEGIN(layer_norm_no_affine_quant_nvfp4_swizzled_bf16, "pfppiip")
rc = p_layer_norm_no_affine_quant_nvfp4_swizzled_bf16(P(0), F(1), P(2), P(3), I(4), I(5), S(6));
END

BEGIN(ada_layer_norm_quant_nvfp4_swizzled_seg_bf16, "ppppifppiip")
rc = p_ada_layer_norm_quant_nvfp4_swizzled_seg_bf16(P(0), IP(1), P(2), P(3), I(4), F(5), P(6), P(7), I(8), I(9),
                                                    S(10));
END

BEGIN(layer_norm_no_affine_quant_nvfp4_2level_bf16, "pfppppiip")
rc = p_layer_norm_no_affine_quant_nvfp4_2level_bf16(P(0), F(1), P(2), P(3), FP(4), P(5), I(6), I(7), S(8));
END

BEGIN(ada_layer_norm_quant_nvfp4_2level_bf16, "pppfppppiip")
rc = p_ada_layer_norm_quant_nvfp4_2level_bf16(P(0), P(1), P(2), F(3), P(4), P(5), FP(6), P(7), I(8), I(9), S(10));
END

BEGIN(ada_layer_norm_quant_nvfp4_2level_seg_bf16, "ppppifppppiip")
rc = p_ada_layer_norm_quant_nvfp4_2level_seg_bf16(P(0), IP(1), P(2), P(3), I(4), F(5), P(6), P(7), FP(8), P(9), I(10),
                                                  I(11), S(12));
END

BEGIN(swiglu_quant_nvfp4_2level_bf16, "ppippppiip")
rc = p_swiglu_quant_nvfp4_2level_bf16(P(0), P(1), I(2), P(3), P(4), FP(5), P(6), I(7), I(8), S(9));
END

BEGIN(swiglu_bf16, "ppipiip")
rc = p_swiglu_bf16(P(0), P(1), I(2), P(3), I(4), I(5), S(6));
END

/* adaln_modulation6_bf16(params, modulation, outs, batch, seq, dim, stream):
 * outs is a sequence of six pointers */
BEGIN(adaln_modulation6_bf16, "pp-iiip")
{
  void* outs[6];
  PyObject* seq = PySequence_Fast(args[2], "adaln_modulation6_bf16: outs must be a sequence of six pointers");
  if (seq == NULL) return NULL;
  if (PySequence_Fast_GET_SIZE(seq) != 6) {
    Py_DECREF(seq);
    PyErr_SetString(PyExc_ValueError, "adaln_modulation6_bf16: outs must hold six pointers");
    return NULL;
  }
  for (int j = 0; j < 6; ++j) {
    PyObject* o = PySequence_Fast_GET_ITEM(seq, j);
    outs[j] = (o == Py_None) ? NULL : PyLong_AsVoidPtr(o);
  }
  Py_DECREF(seq);
  if (PyErr_Occurred()) return NULL;
  rc = p_adaln_modulation6_bf16((const float*)P(0), (const float*)P(1), outs, I(3), I(4), I(5), S(6));
}
END

/* bind(path): resolve every entry point in the library at `path` */
static PyObject* py_bind(PyObject* self, PyObject* arg) {
  (void)self;
  const char* path = PyUnicode_AsUTF8(arg);
  if (path == NULL) return NULL;
  void* h = dlopen(path, RTLD_NOW | RTLD_LOCAL);
  if (h == NULL) {
    PyErr_Format(PyExc_OSError, "bind: %s", dlerror());
    return NULL;
  }
#define RESOLVE(name)                                                     \
  p_##name = (__typeof__(&name))dlsym(h, #name);                          \
  if (p_##name == NULL) {                                                 \
    PyErr_Format(PyExc_OSError, "bind: %s lacks %s", path, #name);        \
    return NULL;                                                          \
  }
  ENTRY_POINTS(RESOLVE)
  Py_RETURN_NONE;
}

#define METHOD(name) {#name, (PyCFunction)(void (*)(void))py_##name, METH_FASTCALL, NULL},
static PyMethodDef kMethods[] = {
    {"bind", py_bind, METH_O, "bind(path): resolve the entry points of the library at path"},
    ENTRY_POINTS(METHOD){NULL, NULL, 0, NULL}};

static struct PyModuleDef kModule = {PyModuleDef_HEAD_INIT,
                                     "_pycall",
                                     "argument marshalling for libnvfp4ap.so's producer entry points",
                                     -1,
                                     kMethods,
                                     NULL,
                                     NULL,
                                     NULL,
                                     NULL};

PyMODINIT_FUNC PyInit__pycall(void) { return PyModule_Create(&kModule); }
