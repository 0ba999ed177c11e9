// Instantiates every kernel of one bit width; compiled once per width with
// -DTFX_BITS=1..8 so the widths build in parallel.
#include "exl3_kernels.cuh"
#include "exl3_tc.cuh"

#ifndef TFX_BITS
#error "compile with -DTFX_BITS=<1..8>"
#endif

#define TFX_CAT2(a, b) a##b
#define TFX_CAT(a, b) TFX_CAT2(a, b)

// Launch-shape constants of the decode-rows kernel: prefetch depth and the
// minimum resident 8-warp CTAs per SM (4 -> 64 registers, 3 -> 80, 2 -> 128)
// for 1..8, 9..16, 17..32 and 33..64 rows.
#ifndef TFX_ROWS_PF1
#define TFX_ROWS_PF1 4
#endif
#ifndef TFX_ROWS_MINB1
#define TFX_ROWS_MINB1 ((TFX_BITS >= 5 && TFX_BITS <= 7) ? 3 : 4)
#endif
#ifndef TFX_ROWS_PF2
#define TFX_ROWS_PF2 (TFX_BITS == 4 ? 4 : 2)
#endif
#ifndef TFX_ROWS_MINB2
#define TFX_ROWS_MINB2 3
#endif
#ifndef TFX_ROWS_PF4
#define TFX_ROWS_PF4 2
#endif
#ifndef TFX_ROWS_MINB4
#define TFX_ROWS_MINB4 ((TFX_BITS >= 5 && TFX_BITS <= 7) ? 2 : 3)
#endif
#ifndef TFX_ROWS_PF8
#define TFX_ROWS_PF8 2
#endif
#ifndef TFX_ROWS_MINB8
#define TFX_ROWS_MINB8 2
#endif

namespace tfx {

KernelSet TFX_CAT(kernels_b, TFX_BITS)() {
  KernelSet k;
  k.linear_rows[0] =
      reinterpret_cast<const void*>(&linear_rows_kernel<TFX_BITS, 1, TFX_ROWS_PF1, TFX_ROWS_MINB1>);
  k.linear_rows[1] =
      reinterpret_cast<const void*>(&linear_rows_kernel<TFX_BITS, 2, TFX_ROWS_PF2, TFX_ROWS_MINB2>);
  k.linear_rows[2] =
      reinterpret_cast<const void*>(&linear_rows_kernel<TFX_BITS, 4, TFX_ROWS_PF4, TFX_ROWS_MINB4>);
  k.linear_rows[3] =
      reinterpret_cast<const void*>(&linear_rows_kernel<TFX_BITS, 8, TFX_ROWS_PF8, TFX_ROWS_MINB8>);
  k.linear_warp[0] = reinterpret_cast<const void*>(&linear_warp_kernel<TFX_BITS, 1, 2>);
  k.linear_warp[1] = reinterpret_cast<const void*>(&linear_warp_kernel<TFX_BITS, 2, 2>);
  k.linear_warp[2] = reinterpret_cast<const void*>(&linear_warp_kernel<TFX_BITS, 4, 1>);
  k.linear_warp[3] = reinterpret_cast<const void*>(&linear_warp_kernel<TFX_BITS, 8, 1>);
  k.linear_tc = reinterpret_cast<const void*>(&linear_tc_kernel<TFX_BITS>);
  k.decode = reinterpret_cast<const void*>(&decode_kernel<TFX_BITS>);
  k.decode_rate = reinterpret_cast<const void*>(&decode_rate_kernel<TFX_BITS>);
  return k;
}

}  // namespace tfx
