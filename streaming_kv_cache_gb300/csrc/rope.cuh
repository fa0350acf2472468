// Device helpers shared by the attention kernels for the rotary embedding
// applied on the fly: rotate-half rotation of bf16 pairs into fp16, logical
// positions of physical key rows, and the angle step R(p+1) = R(p) R(1).
//
// FlashDrive blog walkthrough, section 3.3 "RoPE Position Shift": keys are
// cached without rotation and rotated at their current logical position.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace skv {

// Rotate 8 bf16 pairs in fp32 and emit them as fp16: a holds elements x_e..x_{e+7},
// b their partners x_{e+d/2}..; cs[k] = (cos, sin) of element e+k.  The rotated
// Q and K feed an fp16 x fp16 tensor-core product (3 more significand bits
// than bf16); values are clamped to the finite fp16 range.
// t[w] = (cos, sin) of elements 2w and 2w+1 of the chunk.
__device__ __forceinline__ void rotate_pairs4(uint4& a, uint4& b, const float4 (&t)[4]) {
  uint32_t* pa = reinterpret_cast<uint32_t*>(&a);
  uint32_t* pb = reinterpret_cast<uint32_t*>(&b);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float x0 = bf16_lo(pa[w]), x1 = bf16_hi(pa[w]);
    const float y0 = bf16_lo(pb[w]), y1 = bf16_hi(pb[w]);
    pa[w] = pack_f16x2_sat(x0 * t[w].x - y0 * t[w].y, x1 * t[w].z - y1 * t[w].w);
    pb[w] = pack_f16x2_sat(y0 * t[w].x + x0 * t[w].y, y1 * t[w].z + x1 * t[w].w);
  }
}

__device__ __forceinline__ void rotate_pairs(uint4& a, uint4& b, const float2* __restrict__ cs) {
  const float4* c4 = reinterpret_cast<const float4*>(cs);
  float4 t[4];
#pragma unroll
  for (int w = 0; w < 4; ++w) t[w] = __ldg(c4 + w);
  rotate_pairs4(a, b, t);
}

// Logical position of physical key row r and how many rows from r on (r
// included) continue with consecutive positions: the rest of the prefix, of
// the ring frame, or the tail.
__device__ __forceinline__ void key_pos_run(const Geom& g, const int* __restrict__ heads, int r, int& pos,
                                            int& run) {
  const int u = r - g.P;
  if (u < 0) {
    pos = r;
    run = g.P - r;
    return;
  }
  if (u >= g.ring_rows()) {
    pos = r;
    run = 1 << 30;
    return;
  }
  const int FT = g.F * g.T;
  const int v = u / FT;
  const int rem = u - v * FT;
  const int sl = rem / g.T;
  const int t = rem - sl * g.T;
  int f = sl - heads[v];
  if (f < 0) f += g.F;
  pos = g.P + v * FT + f * g.T + t;
  run = g.T - t;
}

__device__ __forceinline__ void advance_angles(float4 (&cs)[4], const float4 (&st)[4]) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float4 c = cs[w];
    cs[w] = make_float4(c.x * st[w].x - c.y * st[w].y, c.y * st[w].x + c.x * st[w].y,
                        c.z * st[w].z - c.w * st[w].w, c.w * st[w].z + c.z * st[w].w);
  }
}

}  // namespace skv

namespace skv {

// Load n_tiles query tiles of 128 rows into shared memory, rotated at their
// positions and stored as fp16 in the 128-byte-swizzled K-major layout
// (tile t at dst + t*tile_bytes, 64-column halves half_bytes apart).  The
// (row, 8-pair chunk) items are spread over the 128 calling threads and
// fetched two at a time, so the global and table loads overlap.
// row_src(r) returns the pre-RoPE bf16 row of tile row r (nullptr for a
// padding row, which is zero-filled) and its position.
template <int D, typename RowSrc>
__device__ __forceinline__ void load_rotate_q(uint8_t* dst, int n_tiles, int tile_bytes, int half_bytes,
                                              const float2* __restrict__ rope, int tid128, RowSrc row_src) {
  constexpr int HALF = D / 2;
  constexpr int NCH = HALF / 8;
  constexpr int BATCH = 2;
  const int n_items = n_tiles * 128 * NCH;
  for (int i0 = tid128 * BATCH; i0 < n_items; i0 += 128 * BATCH) {
    uint4 xa[BATCH], xb[BATCH];
    float4 t[BATCH][4];
    int rr[BATCH], cc[BATCH];
    bool live[BATCH];
#pragma unroll
    for (int q = 0; q < BATCH; ++q) {
      const int it = i0 + q;
      rr[q] = it / NCH;
      cc[q] = it % NCH;
      live[q] = false;
      if (it < n_items) {
        int pos;
        const uint16_t* src = row_src(rr[q], pos);
        if (src) {
          live[q] = true;
          xa[q] = *reinterpret_cast<const uint4*>(src + cc[q] * 8);
          xb[q] = *reinterpret_cast<const uint4*>(src + HALF + cc[q] * 8);
          const float4* c4 = reinterpret_cast<const float4*>(rope + (size_t)pos * HALF + cc[q] * 8);
#pragma unroll
          for (int w = 0; w < 4; ++w) t[q][w] = __ldg(c4 + w);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < BATCH; ++q) {
      if (i0 + q >= n_items) continue;
      if (live[q]) {
        rotate_pairs4(xa[q], xb[q], t[q]);
      } else {
        xa[q] = make_uint4(0, 0, 0, 0);
        xb[q] = xa[q];
      }
      const int tile = rr[q] / 128, row = rr[q] % 128;
      const int ea = cc[q] * 8, eb = HALF + cc[q] * 8;
      uint8_t* base = dst + tile * tile_bytes;
      *reinterpret_cast<uint4*>(base + (ea / 64) * half_bytes + row * 128 + ((((ea % 64) / 8) ^ (row & 7)) << 4)) = xa[q];
      *reinterpret_cast<uint4*>(base + (eb / 64) * half_bytes + row * 128 + ((((eb % 64) / 8) ^ (row & 7)) << 4)) = xb[q];
    }
  }
}

}  // namespace skv
