// divide.cuh -- unsigned 32-bit division by an invariant divisor, for the
// flat grid-stride kernels that map a work-item index to (row, item in row).
//
// Granlund and Montgomery, "Division by invariant integers using
// multiplication" (1994), the unsigned N = 32 case: for 1 <= d < 2^32 with
// l = ceil(log2 d) and m = floor(2^32 (2^l - d) / d) + 1 (fits 32 bits),
// t = mulhi(m, n) gives n / d = (t + ((n - t) >> min(l, 1))) >> max(l - 1, 0)
// for every n < 2^32.
#pragma once

#include <cstdint>

namespace nvfp4ap {

struct InvDiv {
  uint32_t m;
  int sh1, sh2;
};

inline InvDiv make_inv_div(uint32_t d) {
  int l = 0;
  while (l < 32 && ((uint64_t)1 << l) < d) ++l;
  InvDiv v;
  v.m = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << l) - d)) / d + 1);
  v.sh1 = l < 1 ? l : 1;
  v.sh2 = l - 1 > 0 ? l - 1 : 0;
  return v;
}

__device__ __forceinline__ uint32_t inv_div(uint32_t n, const InvDiv& v) {
  const uint32_t t = __umulhi(v.m, n);
  return (t + ((n - t) >> v.sh1)) >> v.sh2;
}

}  // namespace nvfp4ap
