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

// ---------------------------------------------------------------- tile RoPE
// Canonical rotation of a 128-row tile. Work unit = (quad qd of 4 consecutive
// pairs, 16-row group g). The group's first row, and any row whose position
// does not follow its predecessor's (a document start), take (cos, sin) from
// the two-level tables; the other rows advance each pair's angle by one
// theta_p with a complex product by (cos theta_p, sin theta_p) in fp32. A
// table value is off by at most 3 fp32 units in the last place (u = 2^-24) per
// component, each step adds at most 4.3u, and a unit takes at most 15 steps,
// so with the rotation's own roundings the result is within 72u (4.3e-6) of
// the pair's magnitude of the exact rotation: far below the bf16 rounding of
// the result (2^-9 relative). Any kernel that rotates a tile runs this
// same unit decomposition and arithmetic, so all rotations of a tile agree bit
// for bit.
//
// Usage: RopeUnits<HD, NT> st; st.begin(...) loads the positions and the
// group-start (cos, sin) values (issue it before waiting for the tile's data
// to hide their latency); st.run(tile, ...) then rotates in place.
// Tile accessors provide load4(r, qd, x[4], y[4]) / store4(r, qd, x, y) for
// the 4 pairs of quad qd in tile row r. NT threads (a multiple of 32) with ids
// t share the NU = HD/8 * 8 units.
template <int HD, int NT>
struct RopeUnits {
  static constexpr int NQ = HD / 8;      // quads per row
  static constexpr int NU = NQ * 8;      // units per tile
  static constexpr int UPT = (NU + NT - 1) / NT;
  static constexpr int RPL = 16 / NQ;    // positions each lane holds for its group
  int pos[UPT][RPL];                     // positions of this lane's slice of its group's rows
  float c0[UPT][4], s0[UPT][4];          // (cos, sin) at the group's first row

  __device__ __forceinline__ void begin(int row0, int T, const int32_t* __restrict__ pos_id, bool inverse,
                                        const float2* __restrict__ hi_tab, const float2* __restrict__ lo_tab, int t) {
    const int lane = t & 31;
#pragma unroll
    for (int k = 0; k < UPT; ++k) {
      const int u = t + k * NT;
      const int qd = u % NQ, g = u / NQ;
#pragma unroll
      for (int m = 0; m < RPL; ++m) {
        const int row = row0 + g * 16 + (lane % NQ) + m * NQ;
        pos[k][m] = (u < NU && row < T) ? __ldg(pos_id + row) : -1;
      }
      const int p0 = (u < NU && row0 + g * 16 < T) ? __ldg(pos_id + row0 + g * 16) : 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 cs = rope_cs(hi_tab, lo_tab, p0, qd * 4 + e, HD / 2);
        c0[k][e] = cs.x;
        s0[k][e] = inverse ? -cs.y : cs.y;
      }
    }
  }

  // Rotates each unit in two batches of 8 rows, each in three phases so the
  // row loads are in flight together: load, rotate in registers, store.
  template <class Tile>
  __device__ __forceinline__ void run(Tile& tile, bool inverse, const float2* __restrict__ hi_tab,
                                      const float2* __restrict__ lo_tab, const float2* __restrict__ step_tab,
                                      int t) const {
    const int lane = t & 31;
    const int gl = lane & ~(NQ - 1);  // first lane of this lane's group
#pragma unroll
    for (int k = 0; k < UPT; ++k) {
      const int u = t + k * NT;
      const int qd = u % NQ, g = u / NQ;
      const bool unit_ok = u < NU;
      float sc[4], ss[4], c[4], s[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 st = __ldg(step_tab + qd * 4 + e);
        sc[e] = st.x;
        ss[e] = inverse ? -st.y : st.y;
        c[e] = c0[k][e];
        s[e] = s0[k][e];
      }
      int prev = -2;
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // two batches of 8 rows
        int pr[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int rr = half * 8 + r;
          pr[r] = __shfl_sync(0xffffffffu, pos[k][rr / NQ], gl + (rr % NQ));
        }
        typename Tile::Raw raw[8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (unit_ok && pr[r] >= 0) raw[r] = tile.load_raw(g * 16 + half * 8 + r, qd);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          if (!unit_ok || pr[r] < 0) continue;
          if (half * 8 + r > 0) {
            if (pr[r] == prev + 1) {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float nc = __fmaf_rn(c[e], sc[e], -__fmul_rn(s[e], ss[e]));
                const float ns = __fmaf_rn(s[e], sc[e], __fmul_rn(c[e], ss[e]));
                c[e] = nc;
                s[e] = ns;
              }
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 cs = rope_cs(hi_tab, lo_tab, pr[r], qd * 4 + e, HD / 2);
                c[e] = cs.x;
                s[e] = inverse ? -cs.y : cs.y;
              }
            }
          }
          prev = pr[r];
          float x[4], y[4];
          Tile::unpack(raw[r], x, y);
#pragma unroll
          for (int e = 0; e < 4; ++e) rope_pair(x[e], y[e], c[e], s[e]);
          raw[r] = Tile::pack(x, y);
        }
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (unit_ok && pr[r] >= 0) tile.store_raw(g * 16 + half * 8 + r, qd, raw[r]);
      }
    }
  }
};

// Packing of one quad (4 pairs) for the two pair layouts: layout 0 keeps
// (2p, 2p+1) interleaved in 16 bytes; layout 1 holds the 4 first-half and the
// 4 second-half elements as two 8-byte words.
struct QuadRaw {
  uint4 w;
};
__device__ __forceinline__ void quad_unpack(int layout, const QuadRaw& q, float* x, float* y) {
  const uint32_t u[4] = {q.w.x, q.w.y, q.w.z, q.w.w};
  if (layout == 0) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 v = ptx::unpack_bf16x2(u[e]);
      x[e] = v.x;
      y[e] = v.y;
    }
  } else {
    const float2 a0 = ptx::unpack_bf16x2(u[0]), a1 = ptx::unpack_bf16x2(u[1]);
    const float2 b0 = ptx::unpack_bf16x2(u[2]), b1 = ptx::unpack_bf16x2(u[3]);
    x[0] = a0.x; x[1] = a0.y; x[2] = a1.x; x[3] = a1.y;
    y[0] = b0.x; y[1] = b0.y; y[2] = b1.x; y[3] = b1.y;
  }
}
__device__ __forceinline__ QuadRaw quad_pack(int layout, const float* x, const float* y) {
  QuadRaw q;
  if (layout == 0)
    q.w = make_uint4(ptx::pack_bf16x2(x[0], y[0]), ptx::pack_bf16x2(x[1], y[1]), ptx::pack_bf16x2(x[2], y[2]),
                     ptx::pack_bf16x2(x[3], y[3]));
  else
    q.w = make_uint4(ptx::pack_bf16x2(x[0], x[1]), ptx::pack_bf16x2(x[2], x[3]), ptx::pack_bf16x2(y[0], y[1]),
                     ptx::pack_bf16x2(y[2], y[3]));
  return q;
}

// Host: tensor map over x [T, H, D] bf16 with a {64, 1, 128} box and the
// 128-byte swizzle (one 16 KB tile block per load).
aa_status make_tile_map(CUtensorMap* m, const void* base, int T, int H, int D);

// Host: tensor map over x [T, H, D] fp32 with a {box_c, 1, box_t} box, no
// swizzle (a [box_t rows][box_c channels] fp32 block).
aa_status make_f32_map(CUtensorMap* m, const void* base, int T, int H, int D, int box_c, int box_t);

}  // namespace aa
