// Division by a divisor fixed for a whole launch, as one 32 x 32 -> 64-bit multiply and
// a shift, with the multiplier computed once on the host.
//
// A GPU integer division by a value known only at run time is a short routine around the
// MUFU reciprocal. The attention kernels keep the MUFU unit saturated with exponentials,
// so such a division waits in its queue (measured on the forward's producer: several
// hundred cycles per division), and the work decode at every item boundary has several.
//
// Method: the round-up multiplier of Granlund and Montgomery ("Division by invariant
// integers using multiplication", PLDI 1994). For 1 <= d < 2^31 let l = ceil(log2 d),
// s = 31 + l and m = ceil(2^s / d), so 2^31 <= m < 2^32 (d > 2^(l-1) for l >= 1). For
// 0 <= n < 2^31, floor(n * m / 2^s) = floor(n / d): with m = 2^s / d + e, 0 <= e < 1, the
// quotient is n / d + n * e / 2^s, and n * e / 2^s < 2^31 / 2^(31 + l) = 2^-l <= 1 / d,
// too small to reach the next multiple of 1 / d above n / d.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define ATTN_HD __host__ __device__ __forceinline__
#else
#define ATTN_HD inline
#endif

namespace attn {

struct FastDiv {
  uint32_t d;  // the divisor
  uint32_t m;  // the multiplier ceil(2^s / d)
  uint32_t s;  // the shift 31 + ceil(log2 d)

  // d must lie in [1, 2^31); a divisor of 0 is treated as 1 (callers never divide by 0)
  static FastDiv make(uint32_t div) {
    FastDiv f;
    f.d = div == 0 ? 1u : div;
    uint32_t l = 0;
    while (l < 31 && (1u << l) < f.d) ++l;
    f.s = 31 + l;
    const uint64_t p = 1ull << f.s;
    f.m = (uint32_t)((p + f.d - 1) / f.d);
    return f;
  }
  // floor(n / d) for 0 <= n < 2^31
  ATTN_HD uint32_t div(uint32_t n) const { return (uint32_t)(((uint64_t)n * m) >> s); }
  // n mod d for 0 <= n < 2^31
  ATTN_HD uint32_t mod(uint32_t n) const { return n - div(n) * d; }
};

}  // namespace attn

#undef ATTN_HD
