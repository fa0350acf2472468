// stream_attn_prefill on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// FlashDrive blog walkthrough, section 3.2 "View-Major Ordering" and 3.3
// "RoPE Position Shift"; paper summary, "Streaming Inference": only the
// newest frame of each view becomes queries; it sees the system prefix, the
// earlier views, its own view's older frames and its own frame causally;
// keys are cached pre-RoPE and rotated at their current logical position.
//
// One CTA = one (cache, kv head, view, chunk of 2*TQ new-frame tokens).  Its
// 2 x 128 query rows pack TQ = 128/G tokens x the G query heads that share
// the kv head (GQA), so every K/V tile feeds 256 rows.  Key tiles of 128
// rows stream through a 2-stage TMA ring in physical (ring) order; softmax
// is order-free, so only positions and the mask need logical indices.
//
//   warps 0-3   softmax + epilogue of query tile 0 (TMEM lanes = rows)
//   warps 4-7   softmax + epilogue of query tile 1
//   warp  8     TMA producer (K tile, V^T tile) and TMEM allocator
//   warp  9     MMA issuer: S_i = Q_i K^T (smem x smem, fp16 rotated
//               operands), O_i += P_i V (bf16 P from TMEM, bf16 V^T from smem)
//   warps 10-13 RoPE: rotate Q once, then every K tile in shared memory
//               between the TMA landing and the MMA
//
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [384,384+D);
// P_i (bf16 pairs) overwrites the first 64 columns of S_i.
// Online softmax in the exp2 domain with lazy rescaling: O and l are only
// rescaled when a row's running max grows by more than 8 (factor 256).
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace skv {

namespace {

constexpr int BM = 128;          // rows per query tile
constexpr int BN = 128;          // keys per tile
constexpr int NSTAGE = 2;
constexpr int NTHREADS = 448;
constexpr int WARP_TMA = 8, WARP_MMA = 9, WARP_ROPE = 10;
constexpr int MAX_TILES = 1024;
constexpr float RESCALE_THRESHOLD = 8.0f;
constexpr uint64_t DRAIN_NS = 500000000ull;  // bounded wait for own in-flight copies/MMAs

template <int D>
struct Layout {
  static constexpr int QT = BM * D * 2;   // bytes of one query tile
  static constexpr int KT = BN * D * 2;   // bytes of one K tile
  static constexpr int VT = D * BN * 2;   // bytes of one V^T tile
  static constexpr int HALF_Q = BM * 128; // bytes of one 64-column half of a Q/K tile
  static constexpr int HALF_V = D * 128;  // bytes of one 64-key half of a V^T tile
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + 2 * QT;
  static constexpr int V_OFF = K_OFF + NSTAGE * KT;
  static constexpr int BAR_OFF = V_OFF + NSTAGE * VT;
  static constexpr int NBAR = 18;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int TILE_OFF = MISC_OFF + 64;
  static constexpr int BYTES = TILE_OFF + MAX_TILES * 4;
  static constexpr int ALLOC = BYTES + 1024;   // slack for 1024-byte alignment
};

// barrier slots
enum {
  B_QFULL = 0, B_KFULL = 1, B_KROT = 3, B_KEMPTY = 5, B_VFULL = 7, B_VEMPTY = 9,
  B_SFULL = 11, B_PFULL = 13, B_ODONE = 15, B_DRAIN = 17, B_COUNT = 18
};
static_assert(Layout<128>::NBAR == B_COUNT && Layout<64>::NBAR == B_COUNT, "barrier slots");

struct PrefillParams {
  Geom g;
  int Hq, G, TQ, chunks;   // chunks of 2*TQ tokens per view
  const uint16_t* q;
  uint16_t* out;
  float* lse;
  const float2* rope;
  const int32_t* head;
  int32_t* status;
  float scale_log2;
  uint64_t wait_ns;
};

// Rotate 8 bf16 pairs in fp32 and emit them as fp16: a holds elements x_e..x_{e+7},
// b their partners x_{e+d/2}..; cs[k] = (cos, sin) of element e+k.  The rotated
// Q and K feed an fp16 x fp16 tensor-core product (3 more significand bits
// than bf16); values are clamped to the finite fp16 range.
__device__ __forceinline__ void rotate_pairs(uint4& a, uint4& b, const float2* __restrict__ cs) {
  uint32_t* pa = reinterpret_cast<uint32_t*>(&a);
  uint32_t* pb = reinterpret_cast<uint32_t*>(&b);
  const float4* c4 = reinterpret_cast<const float4*>(cs);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const float4 t = __ldg(c4 + w);   // (cos, sin) of elements 2w and 2w+1
    const float x0 = bf16_lo(pa[w]), x1 = bf16_hi(pa[w]);
    const float y0 = bf16_lo(pb[w]), y1 = bf16_hi(pb[w]);
    pa[w] = pack_f16x2_sat(x0 * t.x - y0 * t.y, x1 * t.z - y1 * t.w);
    pb[w] = pack_f16x2_sat(y0 * t.x + x0 * t.y, y1 * t.z + x1 * t.w);
  }
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const PrefillParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  int* s_ntiles = reinterpret_cast<int*>(smem + L::MISC_OFF + 8);
  int* s_tiles = reinterpret_cast<int*>(smem + L::TILE_OFF);

  const Geom& g = p.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // work item: views in descending order (later views have more keys)
  int w = blockIdx.x;
  const int chunk = w % p.chunks;  w /= p.chunks;
  const int h = w % g.Hkv;         w /= g.Hkv;
  const int c = w % g.C;           w /= g.C;
  const int vq = g.V - 1 - w;
  const int t0 = chunk * 2 * p.TQ;                 // first token (within the view's newest frame)
  const int t_max = min(g.T, t0 + 2 * p.TQ) - 1;   // last valid token of the CTA
  const int32_t* head_c = p.head + (size_t)c * g.V;
  const int FT = g.F * g.T;
  const int row_end = g.P + (vq + 1) * FT;         // keys beyond are later views / tail
  const int zc = c * g.Hkv + h;                    // (cache, kv head) plane of the tensor maps
  const uint64_t wait_ns = p.wait_ns;

  if (tid == 0) {
    for (int i = 0; i < L::NBAR; ++i) {
      const bool many = i == B_QFULL || i == B_KROT || i == B_KROT + 1 || i == B_PFULL || i == B_PFULL + 1;
      tc::mbar_init(bar(i), many ? 128 : 1);   // 128 = one arrival per thread of a warpgroup
    }
    *s_abort = 0;
    // tile list over physical key rows [0, row_end), skipping tiles made only
    // of newest-frame rows that no query of this CTA may see
    int ok = 1;
    for (int v = 0; v <= vq; ++v) {
      const int hv = head_c[v];
      if (hv < 0 || hv >= g.F) ok = 0;
    }
    int n = 0;
    if (ok) {
      const int s_new = (head_c[vq] + g.F - 1) % g.F;
      const int ns0 = g.P + (vq * g.F + s_new) * g.T;
      const int inv_lo = ns0 + t_max + 1, inv_hi = ns0 + g.T;
      for (int r0 = 0; r0 < row_end && n < MAX_TILES; r0 += BN) {
        const int r1 = min(r0 + BN, row_end);
        if (r0 >= inv_lo && r1 <= inv_hi) continue;
        s_tiles[n++] = r0;
      }
    } else {
      set_status(p.status, SKV_DEV_BAD_HEAD);
    }
    *s_ntiles = n;
    tc::fence_barrier_init();
  }
  if (warp == WARP_TMA) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int nt = *s_ntiles;

  if (warp == WARP_TMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nt > 0) {
      tc::prefetch_tmap(&tmap_k);
      tc::prefetch_tmap(&tmap_v);
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int s = j & 1, u = j >> 1, r0 = s_tiles[j];
        if (j >= NSTAGE && !tc::mbar_wait(bar(B_KEMPTY + s), (u - 1) & 1, wait_ns, s_abort)) break;
        tc::mbar_arrive_expect_tx(bar(B_KFULL + s), L::KT);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          tc::tma_load_3d(sbase + L::K_OFF + s * L::KT + hf * L::HALF_Q, &tmap_k, bar(B_KFULL + s), hf * 64, r0, zc);
        if (j >= NSTAGE && !tc::mbar_wait(bar(B_VEMPTY + s), (u - 1) & 1, wait_ns, s_abort)) {
          issued = j + 1;   // the K load of tile j is in flight
          break;
        }
        tc::mbar_arrive_expect_tx(bar(B_VFULL + s), L::VT);
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
          tc::tma_load_3d(sbase + L::V_OFF + s * L::VT + hf * L::HALF_V, &tmap_v, bar(B_VFULL + s), r0 + hf * 64, 0, zc);
        issued = j + 1;
      }
      if (*s_abort) {
        set_status(p.status, SKV_DEV_TIMEOUT);
        // let the copies this thread started land before the CTA exits
        for (int j = max(0, issued - NSTAGE); j < issued; ++j) {
          const int s = j & 1, u = j >> 1;
          volatile int never = 0;
          tc::mbar_wait(bar(B_KFULL + s), u & 1, DRAIN_NS, &never);
          tc::mbar_wait(bar(B_VFULL + s), u & 1, DRAIN_NS, &never);
        }
      }
    }
  } else if (warp == WARP_MMA) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idesc_qk = tc::idesc_f16(BM, BN);
      constexpr uint32_t idesc_pv = tc::idesc_bf16(BM, D);
      auto issue_qk = [&](int i, int s) {
        const uint32_t qa = sbase + L::Q_OFF + i * L::QT;
        const uint32_t kb = sbase + L::K_OFF + s * L::KT;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::HALF_Q + (kk & 3) * 32;
          tc::mma_ss(tmem + i * 128, tc::sdesc_sw128(qa + off), tc::sdesc_sw128(kb + off), idesc_qk, kk > 0);
        }
      };
      auto issue_pv = [&](int i, int s, bool acc) {
        const uint32_t vb = sbase + L::V_OFF + s * L::VT;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::HALF_V + (kk & 3) * 32;
          tc::mma_ts(tmem + 256 + i * 128, tmem + i * 128 + kk * 8, tc::sdesc_sw128(vb + off), idesc_pv,
                     (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = tc::mbar_wait(bar(B_QFULL), 0, wait_ns, s_abort);
      if (ok) ok = tc::mbar_wait(bar(B_KROT), 0, wait_ns, s_abort);
      if (ok) {
        tc::tc_fence_after();
        issue_qk(0, 0);
        tc::mma_commit(bar(B_SFULL));
        issue_qk(1, 0);
        tc::mma_commit(bar(B_SFULL + 1));
        tc::mma_commit(bar(B_KEMPTY));
      }
      for (int j = 0; ok && j < nt; ++j) {
        const int s = j & 1, u = j >> 1;
        const int s2 = (j + 1) & 1, u2 = (j + 1) >> 1;
        if (!(ok = tc::mbar_wait(bar(B_VFULL + s), u & 1, wait_ns, s_abort))) break;
        if (!(ok = tc::mbar_wait(bar(B_PFULL), j & 1, wait_ns, s_abort))) break;
        tc::tc_fence_after();
        issue_pv(0, s, j > 0);
        tc::mma_commit(bar(B_ODONE));
        if (j + 1 < nt) {
          if (!(ok = tc::mbar_wait(bar(B_KROT + s2), u2 & 1, wait_ns, s_abort))) break;
          tc::tc_fence_after();
          issue_qk(0, s2);
          tc::mma_commit(bar(B_SFULL));
        }
        if (!(ok = tc::mbar_wait(bar(B_PFULL + 1), j & 1, wait_ns, s_abort))) break;
        tc::tc_fence_after();
        issue_pv(1, s, j > 0);
        tc::mma_commit(bar(B_ODONE + 1));
        tc::mma_commit(bar(B_VEMPTY + s));
        if (j + 1 < nt) {
          issue_qk(1, s2);
          tc::mma_commit(bar(B_SFULL + 1));
          tc::mma_commit(bar(B_KEMPTY + s2));
        }
      }
      if (!ok) set_status(p.status, SKV_DEV_TIMEOUT);
      // every MMA this thread issued completes before TMEM is released
      tc::mma_commit(bar(B_DRAIN));
      volatile int never = 0;
      tc::mbar_wait(bar(B_DRAIN), 0, DRAIN_NS, &never);
    }
  } else if (warp >= WARP_ROPE) {
    // ----------------------------------------------------------------- RoPE
    const int rt = tid - WARP_ROPE * 32;   // 0..127: row of the tile
    constexpr int HALF = D / 2;
    // query tiles: rotate each row at its logical position and store it in
    // the 128-byte-swizzled K-major layout the MMA reads
#pragma unroll 1
    for (int i = 0; i < 2; ++i) {
      const int tok = t0 + i * p.TQ + rt / p.G;
      const int gq = rt % p.G;
      uint8_t* qt = smem + L::Q_OFF + i * L::QT;
      if (tok < g.T) {
        const int pos = g.P + vq * FT + (g.F - 1) * g.T + tok;
        const uint16_t* qrow = p.q + (((size_t)c * (g.V * g.T) + vq * g.T + tok) * p.Hq + h * p.G + gq) * D;
        const float2* cs = p.rope + (size_t)pos * HALF;
#pragma unroll
        for (int ch = 0; ch < HALF / 8; ++ch) {
          uint4 a = *reinterpret_cast<const uint4*>(qrow + ch * 8);
          uint4 b = *reinterpret_cast<const uint4*>(qrow + HALF + ch * 8);
          rotate_pairs(a, b, cs + ch * 8);
          const int ca = (ch * 8) / 64, cb = (HALF + ch * 8) / 64;
          *reinterpret_cast<uint4*>(qt + ca * L::HALF_Q + tc::sw128_off(rt, (ch * 8 % 64) / 8)) = a;
          *reinterpret_cast<uint4*>(qt + cb * L::HALF_Q + tc::sw128_off(rt, ((HALF + ch * 8) % 64) / 8)) = b;
        }
      } else {
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int ch = 0; ch < D / 8; ++ch)
          *reinterpret_cast<uint4*>(qt + (ch / 8) * L::HALF_Q + tc::sw128_off(rt, ch % 8)) = z;
      }
    }
    tc::fence_proxy_async_smem();
    tc::mbar_arrive(bar(B_QFULL));
    // key tiles: rotate in place once TMA has landed them
#pragma unroll 1
    for (int j = 0; j < nt; ++j) {
      const int s = j & 1, u = j >> 1;
      if (!tc::mbar_wait(bar(B_KFULL + s), u & 1, wait_ns, s_abort)) {
        set_status(p.status, SKV_DEV_TIMEOUT);
        break;
      }
      const int r = s_tiles[j] + rt;
      if (r < row_end) {
        const int pos = key_index(g, head_c, r);
        const float2* cs = p.rope + (size_t)pos * HALF;
        uint8_t* kt = smem + L::K_OFF + s * L::KT;
#pragma unroll
        for (int ch = 0; ch < HALF / 8; ++ch) {
          const int ea = ch * 8, eb = HALF + ch * 8;
          uint4* pa = reinterpret_cast<uint4*>(kt + (ea / 64) * L::HALF_Q + tc::sw128_off(rt, (ea % 64) / 8));
          uint4* pb = reinterpret_cast<uint4*>(kt + (eb / 64) * L::HALF_Q + tc::sw128_off(rt, (eb % 64) / 8));
          uint4 a = *pa, b = *pb;
          rotate_pairs(a, b, cs + ea);
          *pa = a;
          *pb = b;
        }
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(bar(B_KROT + s));
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    const int i = warp >> 2;            // query tile
    const int lg = warp & 3;            // TMEM lane group of this warp
    const int row = lg * 32 + lane;
    const int tok = t0 + i * p.TQ + row / p.G;
    const int gq = row % p.G;
    const bool valid = tok < g.T;
    const uint32_t t_lane = (uint32_t)(lg * 32) << 16;
    const uint32_t tS = tmem + t_lane + i * 128;
    const uint32_t tO = tmem + t_lane + 256 + i * 128;
    int ns0 = 0;
    if (nt > 0) {
      const int s_new = (head_c[vq] + g.F - 1) % g.F;
      ns0 = g.P + (vq * g.F + s_new) * g.T;
    }
    const int inv_a = ns0 + min(tok, g.T - 1) + 1, inv_b = ns0 + g.T;   // rows this query may not see
    const float sl = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
#pragma unroll 1
    for (int j = 0; j < nt; ++j) {
      // tcgen05.ld/st below are warp-collective: every branch around them is warp-uniform
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(B_SFULL + i), j & 1, wait_ns, s_abort));
      if (!ok) break;
      tc::tc_fence_after();
      const int r0 = s_tiles[j];
      const int a = inv_a - r0, b = inv_b - r0, e = row_end - r0;
      const bool full = (a >= BN || b <= 0 || a >= b) && e >= BN;
      const uint32_t span = (uint32_t)max(b - a, 0);
      // pass 1: row max of the scaled scores
      float mx = -INFINITY;
#pragma unroll
      for (int cb = 0; cb < BN / 32; ++cb) {
        uint32_t v[32];
        tc::tmem_ld32(tS + cb * 32, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int kk = cb * 32 + k;
          const bool vis = full || ((uint32_t)(kk - a) >= span && kk < e);
          mx = fmaxf(mx, vis ? __uint_as_float(v[k]) * sl : -INFINITY);
        }
      }
      const bool grow = j > 0 && mx > m_used + RESCALE_THRESHOLD;
      if (j == 0) {
        m_used = (mx == -INFINITY) ? 0.f : mx;
      } else if (__any_sync(0xffffffffu, grow)) {
        // O_i holds tiles < j, all complete: S_i(j) was committed after PV_i(j-1).
        // Rows whose max did not grow past the threshold keep theirs (alpha = 1).
        const float m_new = grow ? mx : m_used;
        const float alpha = tc::ex2(m_used - m_new);
        l *= alpha;
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t o[32];
          tc::tmem_ld32(tO + cb * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tc::tmem_st32(tO + cb * 32, o);
        }
        tc::tmem_wait_st();
        m_used = m_new;
      }
      // pass 2: P = 2^(s*scale - m), bf16 pairs into the first 64 columns of S_i
#pragma unroll
      for (int cb = 0; cb < BN / 32; ++cb) {
        uint32_t v[32];
        tc::tmem_ld32(tS + cb * 32, v);
        tc::tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const int kk = cb * 32 + k;
          const bool v0 = full || ((uint32_t)(kk - a) >= span && kk < e);
          const bool v1 = full || ((uint32_t)(kk + 1 - a) >= span && kk + 1 < e);
          const float p0 = v0 ? tc::ex2(fmaf(__uint_as_float(v[k]), sl, -m_used)) : 0.f;
          const float p1 = v1 ? tc::ex2(fmaf(__uint_as_float(v[k + 1]), sl, -m_used)) : 0.f;
          l += p0 + p1;
          pk[k >> 1] = pack_bf16x2(p0, p1);
        }
        tc::tmem_st16(tS + cb * 16, pk);
      }
      tc::tmem_wait_st();
      tc::tc_fence_before();
      tc::mbar_arrive(bar(B_PFULL + i));
    }
    if (!ok) set_status(p.status, SKV_DEV_TIMEOUT);
    bool done = ok && nt > 0;
    if (done) done = __all_sync(0xffffffffu, tc::mbar_wait(bar(B_ODONE + i), (nt - 1) & 1, wait_ns, s_abort));
    if (done) {
      tc::tc_fence_after();
      const float inv_l = 1.f / l;
      const size_t tok_row = (size_t)c * (g.V * g.T) + vq * g.T + tok;
      uint16_t* orow = p.out + (tok_row * p.Hq + h * p.G + gq) * D;
#pragma unroll 1
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t o[32];
        tc::tmem_ld32(tO + cb * 32, o);
        tc::tmem_wait_ld();
        if (valid) {
          uint4 pk[4];
          uint32_t* pw = reinterpret_cast<uint32_t*>(pk);
#pragma unroll
          for (int k = 0; k < 16; ++k)
            pw[k] = pack_bf16x2(__uint_as_float(o[2 * k]) * inv_l, __uint_as_float(o[2 * k + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(orow + cb * 32);
#pragma unroll
          for (int k = 0; k < 4; ++k) dst[k] = pk[k];
        }
      }
      if (valid && p.lse)
        p.lse[((size_t)c * p.Hq + h * p.G + gq) * (g.V * g.T) + vq * g.T + tok] =
            (m_used + __log2f(l)) * 0.69314718055994531f;
    } else if (nt > 0 && *s_abort) {
      set_status(p.status, SKV_DEV_TIMEOUT);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == WARP_TMA) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

}  // namespace

// K: [C*Hkv][row_cap][d] -> boxes of 64 dims x 128 rows; V^T: [C*Hkv][d][row_cap]
// -> boxes of 64 keys x d rows.  Both with the 128-byte swizzle.
cudaError_t make_kv_tmaps(const Geom& g, const void* k, const void* vt, CUtensorMap* tk, CUtensorMap* tv) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t planes = (cuuint64_t)g.C * g.Hkv;
  {
    cuuint64_t dims[3] = {(cuuint64_t)g.d, (cuuint64_t)g.row_cap, planes};
    cuuint64_t strides[2] = {(cuuint64_t)g.d * 2, (cuuint64_t)g.row_cap * g.d * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (fn(tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)g.row_cap, (cuuint64_t)g.d, planes};
    cuuint64_t strides[2] = {(cuuint64_t)g.row_cap * 2, (cuuint64_t)g.row_cap * g.d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)g.d, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (fn(tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(vt), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

cudaError_t launch_prefill_tc(const Geom& g, int Hq, const void* q, void* out, float* lse, const void* k,
                              const void* vt, const float* rope, const int32_t* head, float sm_scale,
                              int32_t* status, uint64_t wait_ns, cudaStream_t st) {
  if ((g.row_cap + BN - 1) / BN > MAX_TILES) return cudaErrorInvalidValue;
  CUtensorMap tk, tv;
  cudaError_t e = make_kv_tmaps(g, k, vt, &tk, &tv);
  if (e != cudaSuccess) return e;
  PrefillParams p;
  p.g = g;
  p.Hq = Hq;
  p.G = Hq / g.Hkv;
  p.TQ = BM / p.G;
  p.chunks = (g.T + 2 * p.TQ - 1) / (2 * p.TQ);
  p.q = static_cast<const uint16_t*>(q);
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.rope = reinterpret_cast<const float2*>(rope);
  p.head = head;
  p.status = status;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.wait_ns = wait_ns ? wait_ns : 2000000000ull;
  const long long blocks = (long long)g.C * g.Hkv * g.V * p.chunks;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  if (g.d == 128) {
    const int smem = Layout<128>::ALLOC;
    e = cudaFuncSetAttribute(prefill_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<128><<<(unsigned)blocks, NTHREADS, smem, st>>>(tk, tv, p);
  } else {
    const int smem = Layout<64>::ALLOC;
    e = cudaFuncSetAttribute(prefill_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<64><<<(unsigned)blocks, NTHREADS, smem, st>>>(tk, tv, p);
  }
  return cudaGetLastError();
}

}  // namespace skv
