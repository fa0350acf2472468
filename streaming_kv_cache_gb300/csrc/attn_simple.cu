// Straightforward streaming attention on CUDA cores (fp32): one warp per
// query row, 32-key tiles staged in shared memory with the rotary embedding
// applied as they are loaded.  Serves both the new-frame prefill and the
// verify block.
//
// FlashDrive blog walkthrough, sections 3.2-3.3: a query sees a key iff the
// key's logical index is at most its own; keys are cached pre-RoPE and
// rotated at their current logical position when used.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace skv {

namespace {

constexpr int TK = 32;       // keys per tile (one per lane)
constexpr int ROWS = 8;      // query rows (warps) per CTA

template <int D>
__global__ void __launch_bounds__(ROWS * 32) attn_simple_kernel(
    Geom g, int Hq, int mode, int n_tok, const uint16_t* __restrict__ q, uint16_t* __restrict__ out,
    float* __restrict__ lse, const int32_t* __restrict__ tail_len, const uint16_t* __restrict__ k,
    const uint16_t* __restrict__ vt, const float2* __restrict__ rope,
    const int32_t* __restrict__ head, float scale_log2, int32_t* __restrict__ status) {
  __shared__ float sk[TK][D + 1];
  __shared__ float sv[TK][D + 1];
  __shared__ float sq[ROWS][D];
  __shared__ int sidx[TK];
  __shared__ int s_ok;

  constexpr int HALF = D / 2;
  const int n_chunk = (n_tok + ROWS - 1) / ROWS;
  int bid = blockIdx.x;
  const int chunk = bid % n_chunk;  bid /= n_chunk;
  const int hq = bid % Hq;          bid /= Hq;
  const int c = bid;
  const int G = Hq / g.Hkv;
  const int hk = hq / G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* head_c = head + (size_t)c * g.V;

  // validity of the ring heads (and of the tail in verify mode)
  if (threadIdx.x == 0) {
    int ok = 1;
    for (int v = 0; v < g.V; ++v)
      if (head_c[v] < 0 || head_c[v] >= g.F) ok = 0;
    if (!ok) set_status(status, SKV_DEV_BAD_HEAD);
    if (mode == 1) {
      const int tl = tail_len[c];
      if (tl < 0 || tl + n_tok > g.tail_cap) ok = 0;  // reported by the tail write
    }
    s_ok = ok;
  }
  __syncthreads();
  if (!s_ok) return;

  const int tl = mode == 1 ? tail_len[c] : 0;
  const int tok = chunk * ROWS + warp;
  const bool row_ok = tok < n_tok;
  int q_idx = -1;
  if (row_ok) {
    if (mode == 0) q_idx = new_frame_index(g, tok / g.T, tok % g.T);
    else q_idx = g.n_visual() + tl + tok;
  }
  // keys needed by the CTA: up to the largest query index in it
  const int last_tok = min(n_tok, (chunk + 1) * ROWS) - 1;
  const int row_end = mode == 0 ? g.P + (last_tok / g.T + 1) * g.F * g.T
                                : g.n_visual() + tl + last_tok + 1;

  // rotated query row
  if (row_ok) {
    const uint16_t* qr = q + (((size_t)c * n_tok + tok) * Hq + hq) * D;
    const float2* cs = rope + (size_t)q_idx * HALF;
    for (int i = lane; i < HALF; i += 32) {
      const float x1 = __uint_as_float((uint32_t)qr[i] << 16);
      const float x2 = __uint_as_float((uint32_t)qr[i + HALF] << 16);
      const float2 t = cs[i];
      sq[warp][i] = x1 * t.x - x2 * t.y;
      sq[warp][i + HALF] = x2 * t.x + x1 * t.y;
    }
  }

  float m = -INFINITY, l = 0.f;
  float o[D / 32];
#pragma unroll
  for (int j = 0; j < D / 32; ++j) o[j] = 0.f;

  const uint16_t* kc = k + ((size_t)c * g.Hkv + hk) * g.row_cap * D;
  const uint16_t* vc = vt + ((size_t)c * g.Hkv + hk) * D * (size_t)g.row_cap;

  for (int r0 = 0; r0 < row_end; r0 += TK) {
    __syncthreads();
    if (threadIdx.x < TK) {
      const int r = r0 + threadIdx.x;
      sidx[threadIdx.x] = r < row_end ? key_index(g, head_c, r) : 0x7FFFFFFF;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < TK * HALF; e += ROWS * 32) {
      const int kk = e / HALF, i = e - kk * HALF;
      const int r = r0 + kk;
      float a = 0.f, b = 0.f;
      if (r < row_end) {
        const float x1 = __uint_as_float((uint32_t)kc[(size_t)r * D + i] << 16);
        const float x2 = __uint_as_float((uint32_t)kc[(size_t)r * D + i + HALF] << 16);
        const float2 t = rope[(size_t)sidx[kk] * HALF + i];
        a = x1 * t.x - x2 * t.y;
        b = x2 * t.x + x1 * t.y;
      }
      sk[kk][i] = a;
      sk[kk][i + HALF] = b;
    }
    for (int e = threadIdx.x; e < TK * D; e += ROWS * 32) {
      const int dim = e / TK, kk = e - dim * TK;
      const int r = r0 + kk;
      sv[kk][dim] = r < row_end ? __uint_as_float((uint32_t)vc[(size_t)dim * g.row_cap + r] << 16) : 0.f;
    }
    __syncthreads();
    if (!row_ok) continue;
    float s = 0.f;
#pragma unroll 8
    for (int i = 0; i < D; ++i) s += sq[warp][i] * sk[lane][i];
    s = (sidx[lane] <= q_idx) ? s * scale_log2 : -INFINITY;
    float mt = s;
#pragma unroll
    for (int off = 16; off; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
    const float m_new = fmaxf(m, mt);
    if (m_new == -INFINITY) continue;  // nothing visible yet in this row
    const float alpha = exp2f(m - m_new);
    const float p = exp2f(s - m_new);
    float ps = p;
#pragma unroll
    for (int off = 16; off; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    l = l * alpha + ps;
    m = m_new;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) o[j] *= alpha;
    for (int kk = 0; kk < TK; ++kk) {
      const float pk = __shfl_sync(0xffffffffu, p, kk);
#pragma unroll
      for (int j = 0; j < D / 32; ++j) o[j] += pk * sv[kk][lane + 32 * j];
    }
  }

  if (row_ok) {
    const float inv = 1.f / l;
    uint16_t* orow = out + (((size_t)c * n_tok + tok) * Hq + hq) * D;
#pragma unroll
    for (int j = 0; j < D / 32; ++j) {
      const __nv_bfloat16 b = __float2bfloat16_rn(o[j] * inv);
      orow[lane + 32 * j] = *reinterpret_cast<const uint16_t*>(&b);
    }
    if (lse && lane == 0)
      lse[((size_t)c * Hq + hq) * n_tok + tok] = (m + log2f(l)) * 0.69314718055994531f;
  }
}

}  // namespace

cudaError_t launch_attn_simple(const Geom& g, int Hq, int mode, int n_tok, const void* q,
                               void* out, float* lse, const int32_t* tail_len, const void* k,
                               const void* vt, const float* rope, const int32_t* head,
                               float sm_scale, int32_t* status, cudaStream_t st) {
  const long long blocks = (long long)g.C * Hq * ((n_tok + ROWS - 1) / ROWS);
  if (blocks <= 0) return cudaSuccess;
  const float scale_log2 = sm_scale * 1.4426950408889634f;
  auto* qq = static_cast<const uint16_t*>(q);
  auto* oo = static_cast<uint16_t*>(out);
  auto* kk = static_cast<const uint16_t*>(k);
  auto* vv = static_cast<const uint16_t*>(vt);
  auto* rr = reinterpret_cast<const float2*>(rope);
  if (g.d == 128)
    attn_simple_kernel<128><<<(unsigned)blocks, ROWS * 32, 0, st>>>(
        g, Hq, mode, n_tok, qq, oo, lse, tail_len, kk, vv, rr, head, scale_log2, status);
  else
    attn_simple_kernel<64><<<(unsigned)blocks, ROWS * 32, 0, st>>>(
        g, Hq, mode, n_tok, qq, oo, lse, tail_len, kk, vv, rr, head, scale_log2, status);
  return cudaGetLastError();
}

}  // namespace skv
