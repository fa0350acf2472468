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
//   warps 10-11 idle (complete the third warpgroup)
//   warps 12-15 RoPE: rotate Q once, then every K tile in shared memory
//               between the TMA landing and the MMA
// Registers are re-split per warpgroup with setmaxnreg: the softmax threads
// hold a whole 128-score row (192 registers), the others shrink.
//
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [384,384+D);
// P_i (bf16 pairs) overwrites the first 64 columns of S_i.
// Online softmax in the exp2 domain with lazy rescaling: O and l are only
// rescaled when a row's running max grows by more than 8 (factor 256).
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "rope.cuh"
#include "tc.cuh"

namespace skv {

namespace {

constexpr int BM = 128;          // rows per query tile
constexpr int BN = 128;          // keys per tile
constexpr int NSTAGE = 2;
constexpr int NTHREADS = 512;
constexpr int WARP_TMA = 8, WARP_MMA = 9, WARP_ROPE = 12;
// register split (launch: 512 threads x 128): 2 x 128 x 176 + 128 x 56 + 128 x 104 = 65536
constexpr int REG_SOFTMAX = 176, REG_CTRL = 56, REG_ROPE = 104;
static_assert(256 * REG_SOFTMAX + 128 * REG_CTRL + 128 * REG_ROPE == 65536, "register split");
constexpr int MAX_TILES = 1024;
constexpr int MAX_VIEWS = 64;
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
  static constexpr int HEAD_OFF = MISC_OFF + 64;     // ring heads of this cache (<= MAX_VIEWS)
  static constexpr int TILE_OFF = HEAD_OFF + MAX_VIEWS * 4;
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
  int* s_head = reinterpret_cast<int*>(smem + L::HEAD_OFF);

  const Geom& g = p.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // work item: the V x chunks CTAs of one (cache, kv head) are adjacent, so
  // they run together and share that plane's K/V tiles through L2; inside a
  // plane the later (heavier) views come first
  int w = blockIdx.x;
  const int chunk = w % p.chunks;  w /= p.chunks;
  const int vq = g.V - 1 - (w % g.V);  w /= g.V;
  const int h = w % g.Hkv;         w /= g.Hkv;
  const int c = w;
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
      s_head[v] = hv;
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

  if (warp >= 8 && warp < WARP_ROPE) {
    tc::setmaxnreg_dec<REG_CTRL>();
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
      // descriptors advance by adding (byte offset >> 4) to the start-address field
      const uint64_t dq0 = tc::sdesc_sw128(sbase + L::Q_OFF);
      const uint64_t dk0 = tc::sdesc_sw128(sbase + L::K_OFF);
      const uint64_t dv0 = tc::sdesc_sw128(sbase + L::V_OFF);
      auto issue_qk = [&](int i, int s) {
        const uint64_t dq = dq0 + ((uint32_t)(i * L::QT) >> 4);
        const uint64_t dk = dk0 + ((uint32_t)(s * L::KT) >> 4);
#pragma unroll 1
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::HALF_Q + (kk & 3) * 32) >> 4;
          tc::mma_ss(tmem + i * 128, dq + off, dk + off, idesc_qk, kk > 0);
        }
      };
      auto issue_pv = [&](int i, int s, bool acc) {
        const uint64_t dv = dv0 + ((uint32_t)(s * L::VT) >> 4);
#pragma unroll 1
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::HALF_V + (kk & 3) * 32) >> 4;
          tc::mma_ts(tmem + 256 + i * 128, tmem + i * 128 + kk * 8, dv + off, idesc_pv,
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
  }
  } else if (warp >= WARP_ROPE) {
    // ----------------------------------------------------------------- RoPE
    tc::setmaxnreg_dec<REG_ROPE>();
    const int rt = tid - WARP_ROPE * 32;   // 0..127: row of the tile
    constexpr int HALF = D / 2;
    // query tiles: row r of tile i = (token t0 + i*TQ + r/G, head r%G), rotated
    // at its logical position (fp16, swizzled K-major)
    load_rotate_q<D>(smem + L::Q_OFF, 2, L::QT, L::HALF_Q, p.rope, rt, [&](int rr, int& pos) -> const uint16_t* {
      const int i = rr / 128, r = rr % 128;
      const int tok = t0 + i * p.TQ + r / p.G;
      pos = g.P + vq * FT + (g.F - 1) * g.T + tok;
      if (tok >= g.T) return nullptr;
      return p.q + (((size_t)c * (g.V * g.T) + vq * g.T + tok) * p.Hq + h * p.G + r % p.G) * D;
    });
    tc::fence_proxy_async_smem();
    tc::mbar_arrive(bar(B_QFULL));
    // key tiles, rotated in place once TMA has landed them.  Thread (warp wr,
    // lane ln) takes chunk ch = ln % NCH (8 frequencies) of NCH consecutive
    // rows; inside a frame consecutive rows have consecutive positions, so
    // their (cos, sin) advance by one complex multiplication with R(1)
    // instead of a table load.  The first row's table entries of the next
    // tile are fetched while the current tile is rotated.
    constexpr int NCH = HALF / 8;
    const int wr = rt >> 5, ln = rt & 31;
    const int ch = ln % NCH;
    const int row_base = wr * 32 + (ln / NCH) * NCH;
    const int ea = ch * 8, eb = HALF + ch * 8;
    const uint32_t off_a = (ea / 64) * L::HALF_Q, off_b = (eb / 64) * L::HALF_Q;
    const int ca = (ea % 64) / 8, cb = (eb % 64) / 8;
    const float4* rope4 = reinterpret_cast<const float4*>(p.rope);
    float4 step[4];
#pragma unroll
    for (int w4 = 0; w4 < 4; ++w4) step[w4] = __ldg(rope4 + (HALF + ea) / 2 + w4);   // R(1)
    int pf_pos = -1, pf_run = 0;
    float4 pf[4];
    auto fetch = [&](int jj) {
      const int r = s_tiles[jj] + row_base;
      pf_pos = -1;
      if (r < row_end) {
        key_pos_run(g, s_head, r, pf_pos, pf_run);
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) pf[w4] = __ldg(rope4 + ((size_t)pf_pos * HALF + ea) / 2 + w4);
      }
    };
    if (nt > 0) fetch(0);
#pragma unroll 1
    for (int j = 0; j < nt; ++j) {
      const int s = j & 1, u = j >> 1;
      if (!tc::mbar_wait(bar(B_KFULL + s), u & 1, wait_ns, s_abort)) {
        set_status(p.status, SKV_DEV_TIMEOUT);
        break;
      }
      if (pf_pos >= 0) {
        uint8_t* kt = smem + L::K_OFF + s * L::KT;
        const int r0 = s_tiles[j] + row_base;
        int pos = pf_pos, run = pf_run;
        float4 cs[4] = {pf[0], pf[1], pf[2], pf[3]};
#pragma unroll
        for (int k = 0; k < NCH; ++k) {
          const int r = r0 + k;
          if (r >= row_end) break;
          if (k > 0) {
            if (run > 1) {
              --run;
              ++pos;
              advance_angles(cs, step);
            } else {
              key_pos_run(g, s_head, r, pos, run);
#pragma unroll
              for (int w4 = 0; w4 < 4; ++w4) cs[w4] = __ldg(rope4 + ((size_t)pos * HALF + ea) / 2 + w4);
            }
          }
          const int row = row_base + k;
          uint4* pa = reinterpret_cast<uint4*>(kt + off_a + tc::sw128_off(row, ca));
          uint4* pb = reinterpret_cast<uint4*>(kt + off_b + tc::sw128_off(row, cb));
          uint4 xa = *pa, xb = *pb;
          rotate_pairs4(xa, xb, cs);
          *pa = xa;
          *pb = xb;
        }
      }
      if (j + 1 < nt) fetch(j + 1);
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(bar(B_KROT + s));
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    tc::setmaxnreg_inc<REG_SOFTMAX>();
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
      // the whole 128-score row in one TMEM round trip
      uint32_t v[BN];
#pragma unroll
      for (int cb = 0; cb < BN / 32; ++cb)
        tc::tmem_ld32(tS + cb * 32, *reinterpret_cast<uint32_t(*)[32]>(v + cb * 32));
      const int r0 = s_tiles[j];
      const int a = inv_a - r0, b = inv_b - r0, e = row_end - r0;
      const bool full = (a >= BN || b <= 0 || a >= b) && e >= BN;
      tc::tmem_wait_ld();
      if (!__all_sync(0xffffffffu, full)) {
        const uint32_t span = (uint32_t)max(b - a, 0);
#pragma unroll
        for (int k = 0; k < BN; ++k)
          if (!((uint32_t)(k - a) >= span && k < e)) v[k] = __float_as_uint(-INFINITY);
      }
      // row max with 8 independent chains
      float m8[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) m8[q] = __uint_as_float(v[q]);
#pragma unroll
      for (int k = 8; k < BN; ++k) m8[k & 7] = fmaxf(m8[k & 7], __uint_as_float(v[k]));
      float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                       fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
      mx *= sl;
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
      // P = 2^(s*scale - m) as bf16 pairs into the first 64 columns of S_i
      const float nm = -m_used;
      float l8[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) l8[q] = 0.f;
#pragma unroll
      for (int cb = 0; cb < BN / 32; ++cb) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const float p0 = tc::ex2(fmaf(__uint_as_float(v[cb * 32 + k]), sl, nm));
          const float p1 = tc::ex2(fmaf(__uint_as_float(v[cb * 32 + k + 1]), sl, nm));
          l8[(k >> 1) & 7] += p0 + p1;
          pk[k >> 1] = pack_bf16x2(p0, p1);
        }
        tc::tmem_st16(tS + cb * 16, pk);
      }
      l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
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

// Raise the kernel's dynamic shared-memory limit once per device.
template <typename K>
cudaError_t set_smem_once(K kernel, int bytes, int variant) {
  static int done[64][2];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev][variant]) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev][variant] = 1;
  return e;
}

}  // namespace

// K: [C*Hkv][row_cap][d] -> boxes of 64 dims x k_box_rows rows; V^T:
// [C*Hkv][d][row_cap] -> boxes of 64 keys x d rows.  Both with the 128-byte
// swizzle.
cudaError_t make_kv_tmaps(const Geom& g, const void* k, const void* vt, int k_box_rows, CUtensorMap* tk,
                          CUtensorMap* tv) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t planes = (cuuint64_t)g.C * g.Hkv;
  {
    cuuint64_t dims[3] = {(cuuint64_t)g.d, (cuuint64_t)g.row_cap, planes};
    cuuint64_t strides[2] = {(cuuint64_t)g.d * 2, (cuuint64_t)g.row_cap * g.d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)k_box_rows, 1};
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
  cudaError_t e = make_kv_tmaps(g, k, vt, BN, &tk, &tv);
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
    if ((e = set_smem_once(prefill_tc_kernel<128>, smem, 0)) != cudaSuccess) return e;
    prefill_tc_kernel<128><<<(unsigned)blocks, NTHREADS, smem, st>>>(tk, tv, p);
  } else {
    const int smem = Layout<64>::ALLOC;
    if ((e = set_smem_once(prefill_tc_kernel<64>, smem, 1)) != cudaSuccess) return e;
    prefill_tc_kernel<64><<<(unsigned)blocks, NTHREADS, smem, st>>>(tk, tv, p);
  }
  return cudaGetLastError();
}

}  // namespace skv
