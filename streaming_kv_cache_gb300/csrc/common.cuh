// Shared device-side helpers of libskv: cache geometry, logical-index
// arithmetic and bf16 conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "skv.h"

namespace skv {

// n / d and n % d by multiply-high for n < 2^31, d >= 1, with m =
// floor((2^32 - 1) / d): the first quotient is floor(n/d) or one less
// (n m / 2^32 undershoots n / d by less than 2n / 2^32 < 1), so a single
// correction step makes it exact.
__host__ __device__ __forceinline__ uint32_t fastdiv_m(uint32_t d) { return 0xFFFFFFFFu / d; }
__device__ __forceinline__ int fastdiv(int n, int d, uint32_t m, int& rem) {
  uint32_t q = __umulhi((uint32_t)n, m);
  uint32_t r = (uint32_t)n - q * (uint32_t)d;
  if (r >= (uint32_t)d) {
    ++q;
    r -= (uint32_t)d;
  }
  rem = (int)r;
  return (int)q;
}

// Plain-value copy of the cache geometry that kernels receive by value.
struct Geom {
  int C, V, F, T, P, tail_cap, Hkv, d, row_cap, rope_len;
  uint32_t ft_m, t_m;   // fastdiv multipliers of F*T and T
  int rope_steps;       // 1: table row = position, angles step along runs; 0: a table row per key
  __host__ __device__ int ring_rows() const { return V * F * T; }
  __host__ __device__ int n_visual() const { return P + V * F * T; }
};

inline Geom geom_of(const skv_cache& c) {
  Geom g;
  g.C = c.n_cache; g.V = c.n_view; g.F = c.n_frame; g.T = c.frame_len; g.P = c.prefix_len;
  g.tail_cap = c.tail_cap; g.Hkv = c.n_kv_head; g.d = c.head_dim; g.row_cap = c.row_cap;
  g.rope_len = c.rope_len;
  g.rope_steps = c.rope_mode == 0;
  g.ft_m = fastdiv_m((uint32_t)(g.F * g.T > 0 ? g.F * g.T : 1));
  g.t_m = fastdiv_m((uint32_t)(g.T > 0 ? g.T : 1));
  return g;
}

// Logical index of token t of view v's newest frame (the new-frame queries).
__host__ __device__ __forceinline__ int new_frame_index(const Geom& g, int v, int t) {
  return g.P + v * g.F * g.T + (g.F - 1) * g.T + t;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Round two floats to bf16 (nearest, ties to even) and pack lo | hi << 16.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Round two floats to fp16 (nearest even), saturating to +-65504 instead of
// overflowing, packed lo | hi << 16 (the convert takes the upper half first).
__device__ __forceinline__ uint32_t pack_f16x2_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Packed fp32 pairs (Blackwell f32x2 arithmetic): lo in the low word.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// three-input maximum
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void set_status(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace skv
