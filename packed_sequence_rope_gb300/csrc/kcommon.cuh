// Device helpers shared by the kernels: RoPE from the two-level tables,
// 128-byte-swizzled tile addressing and the launch-side TMA descriptor setup.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "aa_internal.h"
#include "ptx.cuh"

namespace aa {

// (cos, sin)(pos * theta_p) from the two-level tables: pos = 32*h + l and the
// angle-addition identity, evaluated with explicitly rounded fp32 operations
// so every kernel produces identical bits for the same (pos, p).
__device__ __forceinline__ float2 rope_cs(const float2* __restrict__ hi_tab, const float2* __restrict__ lo_tab,
                                          int pos, int p, int half) {
  const float2 a = __ldg(hi_tab + (size_t)(pos >> 5) * half + p);
  const float2 b = __ldg(lo_tab + (size_t)p * kRopeSplit + (pos & (kRopeSplit - 1)));
  const float c = __fmaf_rn(a.x, b.x, -__fmul_rn(a.y, b.y));
  const float s = __fmaf_rn(a.y, b.x, __fmul_rn(a.x, b.y));
  return make_float2(c, s);
}

// Rotate the pair (x, y) by (c, s): Eq. 6's 2x2 block [[c, -s], [s, c]].
__device__ __forceinline__ void rope_pair(float& x, float& y, float c, float s) {
  const float nx = __fmaf_rn(c, x, -__fmul_rn(s, y));
  const float ny = __fmaf_rn(s, x, __fmul_rn(c, y));
  x = nx;
  y = ny;
}

// Byte offset of the 16-byte chunk `c8` (8 bf16) of row `r` inside a
// [128 rows][64 bf16] tile block stored with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c8) {
  return (uint32_t)(r * 128 + ((c8 ^ (r & 7)) << 4));
}

// Rotate row `r` of a [128][HD] bf16 tile held as HD/64 swizzled blocks of
// 16 KB, in place. `inverse` applies R^T. layout: 0 adjacent, 1 half, 2 none.
template <int HD>
__device__ __forceinline__ void rope_row_smem(uint8_t* tile, int r, int pos, int layout, bool inverse,
                                              const float2* hi_tab, const float2* lo_tab) {
  constexpr int half = HD / 2;
  if (layout == 2) return;
  if (layout == 0) {
#pragma unroll
    for (int b = 0; b < HD / 64; ++b) {
#pragma unroll 2
      for (int c8 = 0; c8 < 8; ++c8) {
        uint4* ptr = reinterpret_cast<uint4*>(tile + b * 16384 + sw128_chunk(r, c8));
        uint4 w = *ptr;
        uint32_t* u = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int p = b * 32 + c8 * 4 + e;
          float2 cs = rope_cs(hi_tab, lo_tab, pos, p, half);
          if (inverse) cs.y = -cs.y;
          float2 xy = ptx::unpack_bf16x2(u[e]);
          rope_pair(xy.x, xy.y, cs.x, cs.y);
          u[e] = ptx::pack_bf16x2(xy.x, xy.y);
        }
        *ptr = w;
      }
    }
  } else {
    // pairs (p, p + HD/2): chunk c8 of the first half meets the chunk HD/16
    // chunks later (the next block for HD = 128, chunk c8 + 4 for HD = 64)
    constexpr int n_chunks = HD / 16;
#pragma unroll 2
    for (int c = 0; c < n_chunks; ++c) {
      const int c2 = c + n_chunks;
      uint4* pa = reinterpret_cast<uint4*>(tile + (c / 8) * 16384 + sw128_chunk(r, c % 8));
      uint4* pb = reinterpret_cast<uint4*>(tile + (c2 / 8) * 16384 + sw128_chunk(r, c2 % 8));
      uint4 wa = *pa, wb = *pb;
      __nv_bfloat16* xa = reinterpret_cast<__nv_bfloat16*>(&wa);
      __nv_bfloat16* xb = reinterpret_cast<__nv_bfloat16*>(&wb);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int p = c * 8 + e;
        float2 cs = rope_cs(hi_tab, lo_tab, pos, p, half);
        if (inverse) cs.y = -cs.y;
        float x = __bfloat162float(xa[e]), y = __bfloat162float(xb[e]);
        rope_pair(x, y, cs.x, cs.y);
        xa[e] = __float2bfloat16_rn(x);
        xb[e] = __float2bfloat16_rn(y);
      }
      *pa = wa;
      *pb = wb;
    }
  }
}

// Read element `c` of row `r` of a swizzled [128][HD] bf16 tile.
__device__ __forceinline__ float tile_elem(const uint8_t* tile, int r, int c) {
  const __nv_bfloat16* p = reinterpret_cast<const __nv_bfloat16*>(
      tile + (c >> 6) * 16384 + sw128_chunk(r, (c & 63) >> 3) + (c & 7) * 2);
  return __bfloat162float(*p);
}

// Host: tensor map over x [T, H, D] bf16 with a {64, 1, 128} box and the
// 128-byte swizzle (one 16 KB tile block per load).
aa_status make_tile_map(CUtensorMap* m, const void* base, int T, int H, int D);

}  // namespace aa
