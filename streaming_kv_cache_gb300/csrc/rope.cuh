// Device helpers shared by the attention kernels for the rotary embedding
// applied on the fly: rotate-half rotation of bf16 pairs into fp16, logical
// positions of physical key rows, the angle step R(p+1) = R(p) R(1), and the
// in-place rotation of a thread's rows of a key tile.
//
// FlashDrive blog walkthrough, section 3.3 "RoPE Position Shift": keys are
// cached without rotation and rotated at their current logical position.
#pragma once

#include <stdint.h>

#include "common.cuh"
#include "tc.cuh"

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

// Logical position of physical key row r and how many rows from r on (r
// included) continue with consecutive positions: the rest of the prefix, of
// the ring frame, or the tail.  With a table row per key (rope_steps 0) the
// run is always 1, so that every row reads its own angles.
__device__ __forceinline__ void key_pos_run(const Geom& g, const int* __restrict__ heads, int r, int& pos,
                                            int& run) {
  const int u = r - g.P;
  if (u < 0) {
    pos = r;
    run = g.rope_steps ? g.P - r : 1;
    return;
  }
  if (u >= g.ring_rows()) {
    pos = r;
    run = g.rope_steps ? 1 << 30 : 1;
    return;
  }
  const int FT = g.F * g.T;
  int rem, t;
  const int v = fastdiv(u, FT, g.ft_m, rem);
  const int sl = fastdiv(rem, g.T, g.t_m, t);
  int f = sl - heads[v];
  if (f < 0) f += g.F;
  pos = g.P + v * FT + f * g.T + t;
  run = g.rope_steps ? g.T - t : 1;
}

// The (cos, sin) of the 8 frequencies of one chunk as packed fp32 pairs:
// c[w] = cosines of frequencies 2w and 2w+1, s[w] their sines.
struct Ang8 {
  uint64_t c[4], s[4];
};

// From table entries t[w] = (cos f_2w, sin f_2w, cos f_2w+1, sin f_2w+1).
__device__ __forceinline__ Ang8 ang8_from(const float4 (&t)[4]) {
  Ang8 a;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    a.c[w] = f2_pack(t[w].x, t[w].z);
    a.s[w] = f2_pack(t[w].y, t[w].w);
  }
  return a;
}

// R(p+1) = R(p) R(1) per frequency: r = R(1) of the chunk.
__device__ __forceinline__ void ang8_step(Ang8& a, const Ang8& r) {
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint64_t c = a.c[w], s = a.s[w];
    a.c[w] = f2_sub(f2_mul(c, r.c[w]), f2_mul(s, r.s[w]));
    a.s[w] = f2_fma(c, r.s[w], f2_mul(s, r.c[w]));
  }
}

// rotate_pairs4 on packed fp32 pairs: x' = x cos - y sin, y' = y cos + x sin
// for the 8 (x, y) = (a, b) element pairs, fp16 out clamped to the finite range.
__device__ __forceinline__ void rotate8(uint4& a, uint4& b, const Ang8& t) {
  uint32_t* pa = reinterpret_cast<uint32_t*>(&a);
  uint32_t* pb = reinterpret_cast<uint32_t*>(&b);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const uint64_t x = f2_pack(bf16_lo(pa[w]), bf16_hi(pa[w]));
    const uint64_t y = f2_pack(bf16_lo(pb[w]), bf16_hi(pb[w]));
    const uint64_t xr = f2_sub(f2_mul(x, t.c[w]), f2_mul(y, t.s[w]));
    const uint64_t yr = f2_fma(x, t.s[w], f2_mul(y, t.c[w]));
    float x0, x1, y0, y1;
    f2_unpack(xr, x0, x1);
    f2_unpack(yr, y0, y1);
    pa[w] = pack_f16x2_sat(x0, x1);
    pb[w] = pack_f16x2_sat(y0, y1);
  }
}

// Rotate rows r0 .. r0+NPT-1 (tile rows row_base ..) of a key tile in shared
// memory, this thread's 8-frequency chunk (a half at off_a/chunk ca, b half at
// off_b/chunk cb); rows at or past row_lim are left as they are.  pos/run and
// first describe row r0 (its logical position, the rows from it on with
// consecutive positions, its table angles).  Inside one run the angles step
// by R(1); rows are loaded two at a time before they are rotated.
// TABLE: compiled for a table row per key (rope_mode 1); the kernels that
// take it are instantiated for that mode alone, so the stepping path of the
// others keeps its registers.
template <int NPT, bool TABLE = false>
__device__ __forceinline__ void rotate_key_rows(uint8_t* kt, uint32_t off_a, uint32_t off_b, int ca, int cb,
                                                int row_base, int r0, int row_lim, int pos, int run,
                                                const float4 (&first)[4], const Ang8& step, const Geom& g,
                                                const int* heads, const float4* rope4, int ea, int half) {
  if (run >= NPT && r0 + NPT <= row_lim) {
    // two rows in flight at a time (registers)
    constexpr int IF = NPT >= 2 ? 2 : 1;
    Ang8 ang = ang8_from(first);
#pragma unroll
    for (int k0 = 0; k0 < NPT; k0 += IF) {
      uint4 xa[IF], xb[IF];
#pragma unroll
      for (int k = 0; k < IF; ++k) {
        xa[k] = *reinterpret_cast<const uint4*>(kt + off_a + tc::sw128_off(row_base + k0 + k, ca));
        xb[k] = *reinterpret_cast<const uint4*>(kt + off_b + tc::sw128_off(row_base + k0 + k, cb));
      }
#pragma unroll
      for (int k = 0; k < IF; ++k) {
        if (k0 + k > 0) ang8_step(ang, step);
        rotate8(xa[k], xb[k], ang);
        *reinterpret_cast<uint4*>(kt + off_a + tc::sw128_off(row_base + k0 + k, ca)) = xa[k];
        *reinterpret_cast<uint4*>(kt + off_b + tc::sw128_off(row_base + k0 + k, cb)) = xb[k];
      }
    }
    return;
  }
  if (TABLE && !g.rope_steps && r0 + NPT <= row_lim) {
    // a table row per key (no stepping): the loads of every row after the
    // first go out together, then the rows are rotated
    float4 t[NPT > 1 ? NPT - 1 : 1][4];
#pragma unroll
    for (int k = 1; k < NPT; ++k) {
      int pk, rk;
      key_pos_run(g, heads, r0 + k, pk, rk);
#pragma unroll
      for (int w4 = 0; w4 < 4; ++w4) t[k - 1][w4] = __ldg(rope4 + ((size_t)pk * half + ea) / 2 + w4);
    }
#pragma unroll
    for (int k = 0; k < NPT; ++k) {
      uint4* pa = reinterpret_cast<uint4*>(kt + off_a + tc::sw128_off(row_base + k, ca));
      uint4* pb = reinterpret_cast<uint4*>(kt + off_b + tc::sw128_off(row_base + k, cb));
      uint4 xa = *pa, xb = *pb;
      rotate8(xa, xb, k == 0 ? ang8_from(first) : ang8_from(t[k > 0 ? k - 1 : 0]));
      *pa = xa;
      *pb = xb;
    }
    return;
  }
  // a run boundary or the end of the keys inside this thread's rows
  Ang8 ang = ang8_from(first);
#pragma unroll 1
  for (int k = 0; k < NPT; ++k) {
    const int r = r0 + k;
    if (r >= row_lim) break;
    if (k > 0) {
      if (run > 1) {
        --run;
        ++pos;
        ang8_step(ang, step);
      } else {
        key_pos_run(g, heads, r, pos, run);
        float4 t[4];
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) t[w4] = __ldg(rope4 + ((size_t)pos * half + ea) / 2 + w4);
        ang = ang8_from(t);
      }
    }
    uint4* pa = reinterpret_cast<uint4*>(kt + off_a + tc::sw128_off(row_base + k, ca));
    uint4* pb = reinterpret_cast<uint4*>(kt + off_b + tc::sw128_off(row_base + k, cb));
    uint4 xa = *pa, xb = *pb;
    rotate8(xa, xb, ang);
    *pa = xa;
    *pb = xb;
  }
}

}  // namespace skv
