// stream_attn_verify on the tensor cores: split-K attention of a drafted
// block over the streaming cache, HBM-bound, plus the combine of the splits.
//
// FlashDrive blog walkthrough, section 4.2: the target model checks a whole
// drafted block in one forward pass; VFlash "03 · Generalist decoding": the
// block holds one accepted anchor plus the proposals.  Block token j of
// cache c sits at logical index P + V*F*T + tail_len[c] + j and sees every
// key up to its own index (the block is causal within itself).
//
// One CTA = one (cache, kv head, key split).  Its 128-row query tile holds
// the blk x G block rows of the kv head's query group (zero-padded), so the
// MMA is M=128 with most rows idle: the kernel is bound by streaming K and
// V^T from HBM, not by the tensor cores.  64-key tiles flow through 2-stage
// TMA rings for K and V^T; RoPE is applied to each K tile in shared memory
// (fp16 out), S double-buffers in TMEM so QK of tile j+1 overlaps the
// softmax of tile j, and P (bf16) overwrites its S buffer for the PV MMA.
// Each split leaves an unnormalised fp32 partial (O, running max m, sum l)
// in the workspace; the last split of a (cache, kv head) to finish merges
// them (read back from L2) and writes the bf16 output.  With a single split
// the kernel writes the output directly.
//
//   warps 0-1  softmax + epilogue (TMEM lanes 0-63 = block rows)
//   warp  2    K producer, TMEM allocator
//   warp  3    V^T producer
//   warp  4    MMA issuer
//   warps 5-8  RoPE (query block once, then every K tile)
#include <cudaTypedefs.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"
#include "rope.cuh"
#include "tc.cuh"

namespace skv {

namespace {

constexpr int BM = 128;     // query-tile rows (block rows, zero-padded)
constexpr int BN = 64;      // keys per tile
constexpr int NTHREADS = 288;
constexpr int WARP_KTMA = 2, WARP_VTMA = 3, WARP_MMA = 4, WARP_ROPE = 5;
constexpr int SOFTMAX_THREADS = 64;
constexpr int MAX_VIEWS = 64;
constexpr int MAX_SPLITS = 64;
constexpr float RESCALE_THRESHOLD = 8.0f;
// pairs of every 16 in a 32-score chunk whose exponentials run on the FMA pipe
constexpr int FMA_EXP_PAIRS = 0;
constexpr uint64_t DRAIN_NS = 500000000ull;

template <int D>
struct VLayout {
  static constexpr int QT = BM * D * 2;
  static constexpr int KT = BN * D * 2;   // 64 rows x D
  static constexpr int VT = D * BN * 2;   // D rows x 64 keys (one 128-byte-swizzled box)
  static constexpr int HALF_Q = BM * 128;
  static constexpr int HALF_K = BN * 128;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + QT;
  static constexpr int V_OFF = K_OFF + 2 * KT;
  static constexpr int BAR_OFF = V_OFF + 2 * VT;
  static constexpr int NBAR = 18;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int HEAD_OFF = MISC_OFF + 32;
  static constexpr int BYTES = HEAD_OFF + MAX_VIEWS * 4;
  static constexpr int ALLOC = BYTES + 1024;
};

enum {
  V_QFULL = 0, V_KFULL = 1, V_KROT = 3, V_KEMPTY = 5, V_VFULL = 7, V_VEMPTY = 9,
  V_SFULL = 11, V_PFULL = 13, V_PVDONE = 15, V_ODONE = 16, V_DRAIN = 17, V_COUNT = 18
};
static_assert(VLayout<128>::NBAR == V_COUNT, "barrier slots");
// the merge keeps 128 block rows x MAX_SPLITS weights in the K and V stages
static_assert(2 * VLayout<64>::KT + 2 * VLayout<64>::VT >= 128 * MAX_SPLITS * 4, "merge scratch");

struct VerifyParams {
  Geom g;
  int Hq, G, blk, R;          // R = blk * G block rows per kv head
  int splits, per;            // key splits per (cache, kv head), tiles per split
  const int32_t* tail_len;
  const uint16_t* q;          // [C][blk][Hq][D]
  uint16_t* out;              // [C][blk][Hq][D]
  float* ws_o;                // [C*Hkv*splits][R][D]
  float* ws_ml;               // [C*Hkv*splits][R][2]
  int* ws_count;              // [C*Hkv] arrival counters, zero between calls
  const float2* rope;
  const int32_t* head;
  int32_t* status;
  float scale_log2;
  uint64_t wait_ns;
};

// Arrival of a split whose partial is stored (called by the 64 softmax
// threads): the last split of the (cache, kv head) to arrive is told to merge
// and leaves the counter at zero for the next call.
__device__ __forceinline__ void arrive_split(const VerifyParams& p, int unit, int tid, int* s_flag) {
  asm volatile("bar.sync 1, %0;" ::"r"(SOFTMAX_THREADS) : "memory");
  if (tid == 0) {
    __threadfence();
    const int prev = atomicAdd(&p.ws_count[unit], 1);
    const int last = prev == p.splits - 1;
    if (last) {
      p.ws_count[unit] = 0;
      __threadfence();
    }
    s_flag[3] = last;
  }
}

// O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s over the splits of one
// (cache, kv head), bf16 into the block rows; all threads of the CTA, with
// wts (shared memory, R x splits floats) for the per-row split weights.
template <int D>
__device__ __noinline__ void merge_splits(const VerifyParams& p, int unit, int c, int h, int tid, float* wts) {
  const size_t base = (size_t)unit * p.splits;
  const int S = p.splits;
  for (int row = tid; row < p.R; row += NTHREADS) {
    float M = -INFINITY;
#pragma unroll 8
    for (int sp = 0; sp < S; ++sp) M = fmaxf(M, __ldcg(p.ws_ml + ((base + sp) * p.R + row) * 2));
    float den = 0.f;
#pragma unroll 8
    for (int sp = 0; sp < S; ++sp) {
      const float m = __ldcg(p.ws_ml + ((base + sp) * p.R + row) * 2);
      const float w = m == -INFINITY ? 0.f : exp2f(m - M);
      wts[row * S + sp] = w;
      den += w * __ldcg(p.ws_ml + ((base + sp) * p.R + row) * 2 + 1);
    }
    const float inv = 1.f / den;
    for (int sp = 0; sp < S; ++sp) wts[row * S + sp] *= inv;
  }
  __syncthreads();
  for (int e = tid; e < p.R * (D / 4); e += NTHREADS) {
    const int row = e / (D / 4), d4 = e % (D / 4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int sp = 0; sp < S; ++sp) {
      const float w = wts[row * S + sp];
      const float4 o = __ldcg(reinterpret_cast<const float4*>(p.ws_o + ((base + sp) * p.R + row) * D) + d4);
      if (w != 0.f) {
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
      }
    }
    const int jt = row / p.G, gq = row % p.G;
    uint2 pk;
    pk.x = pack_bf16x2(acc.x, acc.y);
    pk.y = pack_bf16x2(acc.z, acc.w);
    *reinterpret_cast<uint2*>(p.out + (((size_t)c * p.blk + jt) * p.Hq + h * p.G + gq) * D + d4 * 4) = pk;
  }
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 2)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const VerifyParams p) {
  using L = VLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  // nt, tile0, tail_len, merge flag, epilogue flags of the two softmax warps
  int* s_info = reinterpret_cast<int*>(smem + L::MISC_OFF + 8);
  int* s_head = reinterpret_cast<int*>(smem + L::HEAD_OFF);

  const Geom& g = p.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x % p.splits;
  const int unit = blockIdx.x / p.splits;       // c * Hkv + h
  const int h = unit % g.Hkv, c = unit / g.Hkv;
  const int32_t* head_c = p.head + (size_t)c * g.V;
  const uint64_t wait_ns = p.wait_ns;
  const size_t pidx = (size_t)unit * p.splits + split;

  if (tid == 0) {
    for (int i = 0; i < L::NBAR; ++i) {
      // warp-wide events arrive once per warp (after __syncwarp)
      const bool many = i == V_QFULL || i == V_KROT || i == V_KROT + 1;
      const bool soft = i == V_PFULL || i == V_PFULL + 1;
      tc::mbar_init(bar(i), many ? 4 : soft ? SOFTMAX_THREADS / 32 : 1);
    }
    *s_abort = 0;
    int ok = 1;
    for (int v = 0; v < g.V; ++v) {
      const int hv = head_c[v];
      if (hv < 0 || hv >= g.F) ok = 0;
      s_head[v] = hv;
    }
    if (!ok) set_status(p.status, SKV_DEV_BAD_HEAD);
    const int tl = p.tail_len[c];
    if (tl < 0 || tl + p.blk > g.tail_cap) ok = 0;   // reported by the tail write
    int nt = 0, tile0 = 0;
    if (ok) {
      const int n_keys = g.n_visual() + tl + p.blk;
      const int nt_unit = (n_keys + BN - 1) / BN;
      tile0 = split * p.per;
      nt = max(0, min(p.per, nt_unit - tile0));
    }
    s_info[0] = ok ? nt : -1;
    s_info[1] = tile0;
    s_info[2] = ok ? tl : 0;
    s_info[3] = 0;
    tc::fence_barrier_init();
  }
  if (warp == WARP_KTMA) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), 256);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int nt = max(s_info[0], 0);
  const bool unit_ok = s_info[0] >= 0;
  const int tile0 = s_info[1];
  const int tl = s_info[2];
  const int q_base = g.n_visual() + tl;    // logical index of block token 0

  if (warp == WARP_KTMA || warp == WARP_VTMA) {
    // ------------------------------------------------------------ producers
    const bool is_k = warp == WARP_KTMA;
    if (lane == 0 && nt > 0) {
      tc::prefetch_tmap(is_k ? &tmap_k : &tmap_v);
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int s = j & 1, u = j >> 1, r0 = (tile0 + j) * BN;
        const int zc = c * g.Hkv + h;
        if (j >= 2 && !tc::mbar_wait(bar((is_k ? V_KEMPTY : V_VEMPTY) + s), (u - 1) & 1, wait_ns, s_abort))
          break;
        if (is_k) {
          tc::mbar_arrive_expect_tx(bar(V_KFULL + s), L::KT);
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf)
            tc::tma_load_3d(sbase + L::K_OFF + s * L::KT + hf * L::HALF_K, &tmap_k, bar(V_KFULL + s), hf * 64, r0, zc);
        } else {
          tc::mbar_arrive_expect_tx(bar(V_VFULL + s), L::VT);
          tc::tma_load_3d(sbase + L::V_OFF + s * L::VT, &tmap_v, bar(V_VFULL + s), r0, 0, zc);
        }
        issued = j + 1;
      }
      if (*s_abort) {
        set_status(p.status, SKV_DEV_TIMEOUT);
        for (int j = max(0, issued - 2); j < issued; ++j) {
          volatile int never = 0;
          tc::mbar_wait(bar((is_k ? V_KFULL : V_VFULL) + (j & 1)), (j >> 1) & 1, DRAIN_NS, &never);
        }
      }
    }
  } else if (warp == WARP_MMA) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idesc_qk = tc::idesc_f16(BM, BN);
      constexpr uint32_t idesc_pv = tc::idesc_bf16(BM, D);
      const uint64_t dq0 = tc::sdesc_sw128(sbase + L::Q_OFF);
      const uint64_t dk0 = tc::sdesc_sw128(sbase + L::K_OFF);
      const uint64_t dv0 = tc::sdesc_sw128(sbase + L::V_OFF);
      auto issue_qk = [&](int j) {
        const uint64_t dk = tc::opaque(dk0 + ((uint32_t)((j & 1) * L::KT) >> 4));
        const uint64_t dq = tc::opaque(dq0);
        const uint32_t d_tmem = tmem + (j & 1) * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offq = ((kk >> 2) * L::HALF_Q + (kk & 3) * 32) >> 4;
          const uint32_t offk = ((kk >> 2) * L::HALF_K + (kk & 3) * 32) >> 4;
          tc::mma_ss(d_tmem, dq + offq, dk + offk, idesc_qk, kk > 0);
        }
      };
      bool ok = true;
      auto issue_pv = [&](int t) {
        const int vs = t & 1, vu = t >> 1;
        if (!(ok = tc::mbar_wait(bar(V_VFULL + vs), vu & 1, wait_ns, s_abort))) return;
        if (!(ok = tc::mbar_wait(bar(V_PFULL + (t & 1)), (t >> 1) & 1, wait_ns, s_abort))) return;
        tc::tc_fence_after();
        const uint64_t dv = tc::opaque(dv0 + ((uint32_t)(vs * L::VT) >> 4));
        const uint32_t a_tmem = tmem + (t & 1) * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          tc::mma_ts(tmem + 128, a_tmem + kk * 8, dv + (((kk & 3) * 32) >> 4), idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(bar(V_PVDONE));
        tc::mma_commit(bar(V_VEMPTY + vs));
      };
      ok = tc::mbar_wait(bar(V_QFULL), 0, wait_ns, s_abort);
      for (int j = 0; ok && j < nt; ++j) {
        const int ks = j & 1, ku = j >> 1;
        if (!(ok = tc::mbar_wait(bar(V_KROT + ks), ku & 1, wait_ns, s_abort))) break;
        tc::tc_fence_after();
        issue_qk(j);
        tc::mma_commit(bar(V_SFULL + (j & 1)));
        tc::mma_commit(bar(V_KEMPTY + ks));
        if (j >= 1) issue_pv(j - 1);
      }
      if (ok) issue_pv(nt - 1);
      if (ok) tc::mma_commit(bar(V_ODONE));
      if (!ok) set_status(p.status, SKV_DEV_TIMEOUT);
      tc::mma_commit(bar(V_DRAIN));
      volatile int never = 0;
      tc::mbar_wait(bar(V_DRAIN), 0, DRAIN_NS, &never);
    }
  } else if (warp >= WARP_ROPE) {
    // ----------------------------------------------------------------- RoPE
    const int rt = tid - WARP_ROPE * 32;   // 0..127
    constexpr int HALF = D / 2;
    if (nt > 0) {
      // query block: row n = (token n / G, head n % G) of this kv head's group
      load_rotate_q<D>(smem + L::Q_OFF, 1, L::QT, L::HALF_Q, p.rope, rt, [&](int rr, int& pos) -> const uint16_t* {
        const int jt = rr / p.G;
        pos = q_base + (rr < p.R ? jt : 0);
        if (rr >= p.R) return nullptr;
        return p.q + (((size_t)c * p.blk + jt) * p.Hq + h * p.G + rr % p.G) * D;
      });
    }
    tc::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar(V_QFULL));
    // key tiles: chunk ch (8 frequencies) of NPT consecutive rows per thread
    constexpr int NCH = HALF / 8;
    constexpr int NPT = BN * NCH / 128;   // rows per thread
    const int wr = rt >> 5, ln = rt & 31;
    const int ch = ln % NCH;
    const int row_base = wr * 16 + (ln / NCH) * NPT;
    const int ea = ch * 8, eb = HALF + ch * 8;
    const uint32_t off_a = (ea / 64) * L::HALF_K, off_b = (eb / 64) * L::HALF_K;
    const int ca = (ea % 64) / 8, cb = (eb % 64) / 8;
    const float4* rope4 = reinterpret_cast<const float4*>(p.rope);
    float4 step[4];
#pragma unroll
    for (int w4 = 0; w4 < 4; ++w4) step[w4] = __ldg(rope4 + (HALF + ea) / 2 + w4);   // R(1)
    const int row_lim = q_base + p.blk;   // rows at or beyond are not keys of this pass
    // the first row's (cos, sin) of the next tile is fetched while the current one is rotated
    int pf_pos = -1, pf_run = 0;
    float4 pf[4];
    auto fetch = [&](int jj) {
      const int r = (tile0 + jj) * BN + row_base;
      pf_pos = -1;
      if (r < row_lim) {
        key_pos_run(g, s_head, r, pf_pos, pf_run);
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) pf[w4] = __ldg(rope4 + ((size_t)pf_pos * HALF + ea) / 2 + w4);
      }
    };
    if (nt > 0) fetch(0);
#pragma unroll 1
    for (int j = 0; j < nt; ++j) {
      const int s = j & 1, u = j >> 1;
      if (!tc::mbar_wait(bar(V_KFULL + s), u & 1, wait_ns, s_abort)) {
        set_status(p.status, SKV_DEV_TIMEOUT);
        break;
      }
      if (pf_pos >= 0) {
        const int r0 = (tile0 + j) * BN + row_base;
        uint8_t* kt = smem + L::K_OFF + s * L::KT;
        int pos = pf_pos, run = pf_run;
        float4 cs[4] = {pf[0], pf[1], pf[2], pf[3]};
#pragma unroll
        for (int k = 0; k < NPT; ++k) {
          const int r = r0 + k;
          if (r >= row_lim) break;
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
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar(V_KROT + s));
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    const int row = warp * 32 + lane;            // TMEM lane = block row (warps 0, 1)
    const uint32_t t_lane = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tmem + t_lane + 128;
    const bool valid = row < p.R;
    const int jt = valid ? row / p.G : 0;
    const int lim = q_base + jt;                 // largest key index this row may see
    const float sl = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
#pragma unroll 1
    for (int j = 0; j < nt; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(V_SFULL + sb), (j >> 1) & 1, wait_ns, s_abort));
      if (!ok) break;
      tc::tc_fence_after();
      const uint32_t tS = tmem + t_lane + sb * BN;
      uint32_t v[BN];
#pragma unroll
      for (int cb = 0; cb < BN / 32; ++cb)
        tc::tmem_ld32(tS + cb * 32, *reinterpret_cast<uint32_t(*)[32]>(v + cb * 32));
      const int r0 = (tile0 + j) * BN;
      tc::tmem_wait_ld();
      if (!__all_sync(0xffffffffu, r0 + BN - 1 <= lim)) {
#pragma unroll
        for (int k = 0; k < BN; ++k)
          if (r0 + k > lim) v[k] = __float_as_uint(-INFINITY);
      }
      // row max: four chains of three-input maxima
      float m4[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) m4[q] = fmaxf(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
#pragma unroll
      for (int k = 8; k < BN; k += 2)
        m4[(k >> 1) & 3] = fmax3(m4[(k >> 1) & 3], __uint_as_float(v[k]), __uint_as_float(v[k + 1]));
      float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      mx *= sl;
      const bool grow = j > 0 && mx > m_used + RESCALE_THRESHOLD;
      if (j == 0) {
        m_used = (mx == -INFINITY) ? 0.f : mx;
      } else if (__any_sync(0xffffffffu, grow)) {
        // PV(j-1) must have landed in O before it is rescaled
        ok = __all_sync(0xffffffffu, tc::mbar_wait(bar(V_PVDONE), (j - 1) & 1, wait_ns, s_abort));
        if (!ok) break;
        tc::tc_fence_after();
        const float m_new = grow ? mx : m_used;
        const float alpha = tc::ex2(m_used - m_new);
        l *= alpha;
#pragma unroll 1
        for (int cb = 0; cb < D / 16; ++cb) {   // 16 columns at a time: the score row stays live
          uint32_t o[16];
          tc::tmem_ld16(tO + cb * 16, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tc::tmem_st16(tO + cb * 16, o);
        }
        tc::tmem_wait_st();
        m_used = m_new;
      }
      // scale-and-shift runs on packed fp32 pairs
      const uint64_t sl2 = f2_pack(sl, sl), nm2 = f2_pack(-m_used, -m_used);
      float l8[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) l8[q] = 0.f;
#pragma unroll
      for (int cb = 0; cb < BN / 32; ++cb) {
        uint32_t pk[16];
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(v[cb * 32 + k]), __uint_as_float(v[cb * 32 + k + 1])), sl2, nm2),
                    x0, x1);
          float p0, p1;
          if (fma_exp_pair(k >> 1, FMA_EXP_PAIRS)) {
            exp2_fma_x2(x0, x1, p0, p1);
          } else {
            p0 = tc::ex2(x0);
            p1 = tc::ex2(x1);
          }
          l8[(k >> 1) & 7] += p0 + p1;
          pk[k >> 1] = pack_bf16x2(p0, p1);
        }
        tc::tmem_st16(tS + cb * 16, pk);
      }
      l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar(V_PFULL + sb));
    }
    if (!ok) set_status(p.status, SKV_DEV_TIMEOUT);
    bool done = ok && nt > 0;
    if (done) done = __all_sync(0xffffffffu, tc::mbar_wait(bar(V_ODONE), 0, wait_ns, s_abort));
    // both softmax warps take the same epilogue path (the merge below syncs them)
    if (lane == 0) s_info[4 + warp] = done;
    asm volatile("bar.sync 1, %0;" ::"r"(SOFTMAX_THREADS) : "memory");
    done = s_info[4] && s_info[5];
    if (done) {
      tc::tc_fence_after();
      const int gq = valid ? row % p.G : 0;
      if (p.splits == 1) {
        const float inv_l = 1.f / l;
        uint16_t* orow = p.out + (((size_t)c * p.blk + jt) * p.Hq + h * p.G + gq) * D;
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
#pragma unroll
            for (int k = 0; k < 4; ++k) reinterpret_cast<uint4*>(orow + cb * 32)[k] = pk[k];
          }
        }
      } else {
        float* orow = p.ws_o + (pidx * p.R + row) * D;
#pragma unroll 1
        for (int cb = 0; cb < D / 32; ++cb) {
          uint32_t o[32];
          tc::tmem_ld32(tO + cb * 32, o);
          tc::tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              reinterpret_cast<uint4*>(orow + cb * 32)[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
          }
        }
        if (valid) {
          p.ws_ml[(pidx * p.R + row) * 2] = m_used;
          p.ws_ml[(pidx * p.R + row) * 2 + 1] = l;
        }
        arrive_split(p, unit, tid, s_info);
      }
    } else if (nt == 0 && unit_ok && p.splits > 1) {
      // a split past the unit's keys contributes nothing
      if (valid) {
        p.ws_ml[(pidx * p.R + row) * 2] = -INFINITY;
        p.ws_ml[(pidx * p.R + row) * 2 + 1] = 0.f;
      }
      arrive_split(p, unit, tid, s_info);
    } else if (nt > 0 && *s_abort) {
      set_status(p.status, SKV_DEV_TIMEOUT);
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == WARP_KTMA) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 256);
  }
  if (s_info[3]) {
    __threadfence();
    // the K/V stages are idle now: they hold the split weights
    merge_splits<D>(p, unit, c, h, tid, reinterpret_cast<float*>(smem + L::K_OFF));
  }
}

int g_num_sms[64];

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!g_num_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
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

// Split plan.  Two CTAs are resident per SM, so the grid runs in waves of
// 2 * SMs CTAs.  A split of n key tiles costs about n + 3 tile times (set-up,
// pipeline fill and the partial), and merging S splits about 2 + S/2; the
// plan takes the split count with the smallest (number of waves) x (cost of
// one split) + merge.  Fewer splits win ties.  At most MAX_SPLITS splits, so
// the merge weights (block rows x splits floats) fit in the idle K/V stages.
void verify_plan(const Geom& g, int Hq, int blk, int* splits, int* per) {
  (void)Hq;
  (void)blk;
  const long long units = (long long)g.C * g.Hkv;
  const int tiles_max = (g.n_visual() + g.tail_cap + BN - 1) / BN;
  const long long wave = 2LL * num_sms();
  long long best_s = 1, best_cost = -1;
  for (long long s = 1; s <= tiles_max; ++s) {
    const long long pr = (tiles_max + s - 1) / s;
    const long long sp = (tiles_max + pr - 1) / pr;
    if (sp != s) continue;
    if (sp > MAX_SPLITS) continue;
    const long long waves = (units * sp + wave - 1) / wave;
    const long long cost = waves * (pr + 3) + (sp > 1 ? 2 + sp / 2 : 0);   // + the merge
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_s = s;
    }
  }
  const int pr = (int)((tiles_max + best_s - 1) / best_s);
  *per = pr;
  *splits = (tiles_max + pr - 1) / pr;
}

// Workspace: [units] int32 counters (256-byte aligned block), then the fp32
// partial O rows and the (m, l) pairs.
size_t verify_ws_bytes(const Geom& g, int Hq, int blk) {
  int splits, per;
  verify_plan(g, Hq, blk, &splits, &per);
  if (splits <= 1) return 0;
  const size_t units = (size_t)g.C * g.Hkv;
  const size_t rows = units * splits * blk * (Hq / g.Hkv);
  return (units * 4 + 255) / 256 * 256 + rows * (g.d + 2) * sizeof(float);
}

cudaError_t make_kv_tmaps(const Geom& g, const void* k, const void* vt, int k_box_rows, int v_box_rows,
                          CUtensorMap* tk, CUtensorMap* tv);

cudaError_t launch_verify_tc(const Geom& g, int Hq, int blk, const int32_t* tail_len, const void* q, void* out,
                             const void* k, const void* vt, const float* rope, const int32_t* head,
                             void* ws, size_t ws_bytes, float sm_scale, int32_t* status, uint64_t wait_ns,
                             cudaStream_t st) {
  if (g.V > MAX_VIEWS) return cudaErrorNotSupported;
  CUtensorMap tk, tv;
  cudaError_t e = make_kv_tmaps(g, k, vt, BN, g.d, &tk, &tv);
  if (e != cudaSuccess) return e;
  VerifyParams p;
  p.g = g;
  p.Hq = Hq;
  p.G = Hq / g.Hkv;
  p.blk = blk;
  p.R = blk * p.G;
  verify_plan(g, Hq, blk, &p.splits, &p.per);
  p.tail_len = tail_len;
  p.q = static_cast<const uint16_t*>(q);
  p.out = static_cast<uint16_t*>(out);
  const size_t need = verify_ws_bytes(g, Hq, blk);
  if (ws_bytes < need || (need && !ws)) return cudaErrorInvalidValue;
  const size_t units = (size_t)g.C * g.Hkv;
  const size_t n_rows = units * p.splits * p.R;
  p.ws_count = static_cast<int*>(ws);
  p.ws_o = need ? reinterpret_cast<float*>(static_cast<char*>(ws) + (units * 4 + 255) / 256 * 256) : nullptr;
  p.ws_ml = need ? p.ws_o + n_rows * g.d : nullptr;
  p.rope = reinterpret_cast<const float2*>(rope);
  p.head = head;
  p.status = status;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.wait_ns = wait_ns ? wait_ns : 2000000000ull;
  const long long blocks = (long long)g.C * g.Hkv * p.splits;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  if (g.d == 128) {
    const int smem = VLayout<128>::ALLOC;
    if ((e = set_smem_once(verify_tc_kernel<128>, smem, 0)) != cudaSuccess) return e;
    verify_tc_kernel<128><<<(unsigned)blocks, NTHREADS, smem, st>>>(tk, tv, p);
  } else {
    const int smem = VLayout<64>::ALLOC;
    if ((e = set_smem_once(verify_tc_kernel<64>, smem, 1)) != cudaSuccess) return e;
    verify_tc_kernel<64><<<(unsigned)blocks, NTHREADS, smem, st>>>(tk, tv, p);
  }
  return cudaGetLastError();
}

}  // namespace skv
