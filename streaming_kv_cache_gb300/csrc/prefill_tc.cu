// stream_attn_prefill on the 5th-generation tensor cores (tcgen05 + TMEM),
// CTA pairs with M = 256 pair MMAs.
//
// FlashDrive blog walkthrough, section 3.2 "View-Major Ordering" and 3.3
// "RoPE Position Shift"; paper summary, "Streaming Inference": only the
// newest frame of each view becomes queries; it sees the system prefix, the
// earlier views, its own view's older frames and its own frame causally;
// keys are cached pre-RoPE and rotated at their current logical position.
// The same kernel takes the other query sets of the method, as segments of
// consecutive logical positions: the trajectory / text tokens after the views
// (section 3.2: they see every view and are causal among themselves) and
// every token of the window (section 11: the first window only fills the
// cache).  A query sees exactly the keys whose logical index is not above its
// own; in physical rows that is a prefix of the rows minus, for a frame of a
// view, the rest of that view's ring after the query (at most two runs).
//
// A cluster of two CTAs handles one (cache, kv head, segment, 4*TQ tokens);
// each CTA owns 2 x 128 query rows that pack TQ = 128/G tokens x the
// G query heads sharing the kv head (GQA).  Both CTAs walk the same list of
// 128-key tiles in physical (ring) order -- softmax does not depend on key
// order, so only positions and the mask need logical indices.  Each CTA
// loads and rotates HALF of every tile: K rows [64*rank, 64*rank + 64) and
// V^T dimension rows [D/2*rank, D/2*(rank+1)).  The even CTA issues the pair
// MMAs (tcgen05.mma.cta_group::2, M = 256): S_i = Q_i K^T takes A = each
// CTA's own query tile and B = the two K halves; O_i += P_i V takes A = each
// CTA's P (TMEM) and B = the two V^T halves.  Commits reach the barriers of
// both CTAs; the odd CTA's arrivals reach the even CTA's barriers across
// the cluster.
//
//   warps 0-3   softmax + epilogue of query tile 0 (TMEM lanes = rows)
//   warps 4-7   softmax + epilogue of query tile 1
//   warp  8     K producer (TMA) and TMEM allocator
//   warp  9     MMA issuer (even CTA only)
//   warp  10    forwards "V half landed" to the even CTA
//   warp  11    V^T producer (TMA)
//   warps 12-15 RoPE: rotate Q once, then this CTA's half of every K tile
//               in shared memory between the TMA landing and the MMA
// Registers are re-split per warpgroup with setmaxnreg: the softmax threads
// hold a whole 128-score row (184 registers), the others shrink.
//
// TMEM (512 columns per CTA): S0 [0,128) S1 [128,256) O0 [256,256+D)
// O1 [384,384+D); P_i (bf16 pairs) overwrites the first 64 columns of S_i.
// Online softmax in the exp2 domain with a lagging max: the row max is taken
// on a query's first tile only, and O and l are rescaled only when a later
// tile's probability sum passes 2^20.
#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "rope.cuh"
#include "tc.cuh"

namespace skv {

namespace {

constexpr int BM = 128;          // rows per query tile (per CTA)
constexpr int BN = 128;          // keys per tile (pair)
constexpr int HN = BN / 2;       // keys per tile loaded by one CTA
constexpr int NST = 3;           // K and V stages (three ran faster than four: a smaller carve-out, more L1)
constexpr int NTHREADS = 512;
constexpr int WARP_KTMA = 8, WARP_MMA = 9, WARP_VFWD = 10, WARP_VTMA = 11, WARP_ROPE = 12;
// register split (launch: 512 threads x 128): 2 x 128 x 184 + 128 x 48 + 128 x 96 = 65536
// (measured: 184/48/96 0.8% faster than 176/56/104; 192/40/88 and 168/72/104 slower).
// With the insert fused the control warps also transpose V: 176/56/104 there.
template <bool FUSED> struct RegSplit {
  static constexpr int SOFTMAX = FUSED ? 176 : 184, CTRL = FUSED ? 56 : 48, ROPE = FUSED ? 104 : 96;
  static_assert(256 * SOFTMAX + 128 * CTRL + 128 * ROPE == 65536, "register split");
};
constexpr int MAX_TILES = 1024;
constexpr int BAR_TILES = 4;    // named barrier: the set-up warp -> the two producers
constexpr int MAX_VIEWS = 64;
constexpr float LAG_LIMIT = 1048576.0f;   // 2^20: a tile's probability sum that triggers a rescale
constexpr uint64_t DRAIN_NS = 500000000ull;  // bounded wait for own in-flight copies/MMAs

template <int D>
struct Layout {
  static constexpr int QT = BM * D * 2;     // bytes of one query tile
  static constexpr int HALF_Q = BM * 128;   // one 64-column half of a query tile
  static constexpr int KST = HN * D * 2;    // this CTA's K rows of a tile: 64 x D
  static constexpr int HALF_K = HN * 128;   // one 64-column half of them
  static constexpr int VST = (D / 2) * BN * 2;  // this CTA's V^T rows: D/2 x 128 keys
  static constexpr int HALF_V = (D / 2) * 128;  // one 64-key half of them
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + 2 * QT;
  static constexpr int V_OFF = K_OFF + NST * KST;
  static constexpr int BAR_OFF = V_OFF + NST * VST;
  static constexpr int NBAR = 32;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int HEAD_OFF = MISC_OFF + 64;     // ring heads of this cache (<= MAX_VIEWS)
  static constexpr int TILE_OFF = HEAD_OFF + MAX_VIEWS * 4;
  // per softmax row: the second run of its mask (a2, n2), its output row
  // (-1: none) and its LSE index
  static constexpr int MASK_OFF = TILE_OFF + MAX_TILES * 4;
  // per tile, with the insert fused: bit b set = rows [r0 + 64b, r0 + 64b + 64)
  // are a new frame, read from the step's input instead of the ring
  static constexpr int SRC_OFF = MASK_OFF + 4 * 2 * BM * 4;
  static constexpr int BYTES = SRC_OFF + MAX_TILES;
  static constexpr int ALLOC = BYTES + 1024;   // slack for 1024-byte alignment
};

// barrier slots.  "even" = lives in the even CTA only and counts the
// arrivals of both CTAs; "pair" = completed by a pair-MMA commit in both.
enum {
  B_QFULL = 0,                 // even: 2 x 8 softmax warps (query tiles rotated)
  B_QLOAD = 1,                 // local: this CTA's query tiles landed (TMA)
  B_KFULL = 2,                 // local: this CTA's K half landed (TMA)
  B_KROT = B_KFULL + NST,      // even: 2 x 4 RoPE warps (K halves rotated) + 2 forwarders (V^T halves landed)
  B_KEMPTY = B_KROT + NST,     // pair: K stage free
  B_VFULL = B_KEMPTY + NST,    // local: this CTA's V^T half landed (TMA)
  B_VEMPTY = B_VFULL + NST,    // pair: V stage free
  B_SFULL = B_VEMPTY + NST,    // pair: S_i ready
  B_PFULL = B_SFULL + 2,       // even: 2 x 4 softmax warps (P_i ready)
  B_ODONE = B_PFULL + 2,       // pair: PV_i issued so far complete
  B_DRAIN = B_ODONE + 2,       // pair: every MMA complete
  B_COUNT = B_DRAIN + 1
};
static_assert(Layout<128>::NBAR >= B_COUNT && Layout<64>::NBAR >= B_COUNT, "barrier slots");

struct PrefillParams {
  Geom g;
  int Hq, G, TQ;
  // query segments of every cache and the work items they make (blocks of
  // 4*TQ tokens, one CTA pair each), in the order the items of a (cache, kv
  // head) plane run: the tail block, the views' frames, the prefix
  int nbt, n_tail;        // tail blocks and tail query tokens
  int nf, nbf;            // frames per view that are queries (0, 1 = newest, F) and blocks per frame
  int nbp;                // prefix blocks (0: the prefix is not queried)
  int items;              // items per plane: nbt + V*nf*nbf + nbp
  int NQ;                 // query tokens per cache in q / out / lse
  int q_view0, q_tail0;   // a cache's first query token of the view frames and of the tail block
  const int32_t* tail_len;  // [C] tail rows the tail block follows
  const uint16_t* q;
  uint16_t* out;
  float* lse;
  const float2* rope;
  const int32_t* head;
  int32_t* status;
  float scale_log2;
  uint64_t wait_ns;
  // the insert fused into the new-frame prefill: the ring heads still name
  // the oldest frames, each view's new frame is read from the step's input
  // and written into that slot by the CTA pair of its last query block, and
  // the last CTA of a cache to start advances the heads (counter in sync)
  int32_t* head_w;        // heads to advance (fused only)
  int32_t* sync;          // [C][V] zeroed counters; [c][0] counts the CTAs of cache c
  uint16_t* ring_k;       // the cache's k and vt, written with the new frames
  uint16_t* ring_vt;
};

// SW: compiled for a wait limit under the suspend hint (see tc::bounded_wait)
// Keys of view v's ring that a query at logical frame f, token t (frame f in
// ring slot `slot`) may not see: the later tokens of its own frame and the
// view's later frames, a cyclic run of the ring starting just after the
// query's row, returned as at most two runs of physical rows [a1, a1 + n1)
// and [a2, a2 + n2).
__device__ __forceinline__ void ring_hole(const Geom& g, int v, int f, int slot, int t, int& a1, int& n1,
                                          int& a2, int& n2) {
  const int FT = g.F * g.T, base = g.P + v * FT;
  const int o = slot * g.T + t + 1;                        // 1 .. FT
  const int len = (g.F - 1 - f) * g.T + (g.T - 1 - t);
  n1 = min(len, FT - o);
  a1 = base + o;
  n2 = len - n1;
  a2 = base;
}

// FUSED: the frame insert is done by this launch (see PrefillParams): the new
// frames' K and V come from the step's input through tmap_kn / tmap_vn.
// TABLE: rope_mode 1 (a table row per key), see rotate_key_rows.
template <int D, bool SW, bool FUSED, bool TABLE = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_kn,
                  const __grid_constant__ CUtensorMap tmap_vn, const PrefillParams p) {
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
  int* s_mask = reinterpret_cast<int*>(smem + L::MASK_OFF);
  int* s_wrap = reinterpret_cast<int*>(smem + L::MISC_OFF + 12);   // 1: some row's mask has a second run
  uint8_t* s_src = smem + L::SRC_OFF;

  const Geom& g = p.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = tc::cluster_ctarank();       // 0 = even CTA (issues the MMAs)
  // barriers in the even CTA, addressed across the cluster
  auto bar_even = [&](int i) { return tc::map_to_cta(bar(i), 0); };

  // work item: the items of one (cache, kv head) are adjacent, so they run
  // together and share that plane's K/V tiles through L2; inside a plane the
  // heavier items come first: the tail block (it sees the whole window),
  // then the frames, later views and frames first, then the prefix
  int w = blockIdx.x >> 1;
  const int it = w % p.items;      w /= p.items;
  const int h = w % g.Hkv;
  const int c = w / g.Hkv;
  const int FT = g.F * g.T;
  int pc, n_seg, qoff, pos0, vq = -1, fq = 0, vmax = -1, bad = 0;
  if (it < p.nbt) {                                // tail block
    pc = it;
    n_seg = p.n_tail;
    qoff = p.q_tail0;
    const int tl = p.tail_len[c];
    bad = tl < 0 ? SKV_DEV_BAD_TAIL : (tl + p.n_tail > g.tail_cap ? SKV_DEV_TAIL_OVERFLOW : 0);
    pos0 = g.n_visual() + max(tl, 0);
    vmax = g.V - 1;
  } else if (it < p.nbt + g.V * p.nf * p.nbf) {    // one frame of one view
    int j = it - p.nbt;
    pc = j % p.nbf;  j /= p.nbf;
    const int fi = j % p.nf;
    vq = g.V - 1 - j / p.nf;
    fq = g.F - 1 - fi;
    n_seg = g.T;
    qoff = p.q_view0 + (vq * p.nf + (p.nf - 1 - fi)) * g.T;
    pos0 = g.P + vq * FT + fq * g.T;
    vmax = vq;
  } else {                                         // prefix
    pc = it - p.nbt - g.V * p.nf * p.nbf;
    n_seg = g.P;
    qoff = 0;
    pos0 = 0;
  }
  const int t0 = (pc * 2 + (int)rank) * 2 * p.TQ;      // first token of this CTA
  const int t_max = min(n_seg, (pc + 1) * 4 * p.TQ) - 1;  // last token of the pair (shared tile list)
  const int32_t* head_c = p.head + (size_t)c * g.V;
  // keys beyond are never visible to the item: later views and the tail for
  // a frame; for the prefix and the tail (physical row = logical index) the
  // rows after the item's last token
  const int row_end = vq >= 0 ? g.P + (vq + 1) * FT : pos0 + t_max + 1;
  const int zc = c * g.Hkv + h;                    // (cache, kv head) plane of the tensor maps
  const uint64_t wait_ns = p.wait_ns;

  // The copies of a key tile (first row r0, new-frame flags src) into stage
  // s: this CTA's 64 K rows (K producer) or its D/2 V^T rows of the 128 keys
  // (V producer).  A 64-row block of a view's new frame comes from the
  // step's input [C][V][T][Hkv][d] when the insert is fused: K rows as they
  // are, V token-major (an MN-major operand for the PV product); every other
  // block from the ring.
  auto issue_rows = [&](bool is_k, int s, int r0, uint32_t src) {
    auto new_block = [&](int r, int& t_in, int& cv) {
      const int u = r - g.P, v = u / FT;
      t_in = u % FT % g.T;
      cv = c * g.V + v;
    };
    if (is_k) {
      tc::mbar_arrive_expect_tx(bar(B_KFULL + s), L::KST);
      if (FUSED && (src >> rank) & 1u) {
        int t_in, cv;
        new_block(r0 + HN * (int)rank, t_in, cv);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          tc::tma_load_4d(sbase + L::K_OFF + s * L::KST + hf * L::HALF_K, &tmap_kn, bar(B_KFULL + s), hf * 64, h,
                          t_in, cv);
      } else {
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          tc::tma_load_3d(sbase + L::K_OFF + s * L::KST + hf * L::HALF_K, &tmap_k, bar(B_KFULL + s), hf * 64,
                          r0 + HN * (int)rank, zc);
      }
    } else {
      tc::mbar_arrive_expect_tx(bar(B_VFULL + s), L::VST);
#pragma unroll
      for (int kh = 0; kh < 2; ++kh) {
        if (FUSED && (src >> kh) & 1u) {
          int t_in, cv;
          new_block(r0 + kh * 64, t_in, cv);
          tc::tma_load_4d(sbase + L::V_OFF + s * L::VST + kh * L::HALF_V, &tmap_vn, bar(B_VFULL + s),
                          (D / 2) * (int)rank, h, t_in, cv);
        } else {
          tc::tma_load_3d(sbase + L::V_OFF + s * L::VST + kh * L::HALF_V, &tmap_v, bar(B_VFULL + s), r0 + kh * 64,
                          (D / 2) * (int)rank, zc);
        }
      }
    }
  };
  auto issue_tile = [&](bool is_k, int j) { issue_rows(is_k, j % NST, s_tiles[j], FUSED ? s_src[j] : 0u); };

  // With a prefix of at least one key tile, every item's first tile is rows
  // [0, BN): prefix keys, which every query sees (no hole reaches them) and
  // no new frame holds.  Its copies start at entry too, with the queries'.
  const bool early0 = g.P >= BN;

  // RoPE warps: R(1) of their chunk and, with early0, the first-row angles of
  // tile 0 (a prefix row: its position is its row), loaded at entry
  float4 e_step4[4], e_pf[4];
  if (warp >= WARP_ROPE) {
    const int rt = tid - WARP_ROPE * 32, ln = rt & 31;
    constexpr int HALF = D / 2, NCH = HALF / 8, NPT = HN * NCH / 128;
    const int ea = (ln % NCH) * 8;
    const int row0 = HN * (int)rank + (rt >> 5) * (HN / 4) + (ln / NCH) * NPT;
    const float4* rope4 = reinterpret_cast<const float4*>(p.rope);
#pragma unroll
    for (int w4 = 0; w4 < 4; ++w4) e_step4[w4] = __ldg(rope4 + (HALF + ea) / 2 + w4);
    if (early0) {
#pragma unroll
      for (int w4 = 0; w4 < 4; ++w4) e_pf[w4] = __ldg(rope4 + ((size_t)row0 * HALF + ea) / 2 + w4);
    }
  }

  // The query tiles depend on nothing the set-up computes: their copy starts
  // at entry (its barrier is initialised here, the others below).  Both
  // tiles: rows (token, head) of kv head h, 64 columns per box.
  if ((warp == WARP_KTMA || warp == WARP_VTMA) && lane == 0 && early0) {
    const bool is_k = warp == WARP_KTMA;
    tc::mbar_init(bar(is_k ? B_KFULL : B_VFULL), 1);
    tc::fence_barrier_init();
    tc::fence_proxy_async_smem();
    tc::prefetch_tmap(is_k ? &tmap_k : &tmap_v);
    issue_rows(is_k, 0, 0, 0u);
  }
  if (warp == WARP_KTMA && lane == 0) {
    tc::mbar_init(bar(B_QLOAD), 1);
    tc::fence_barrier_init();
    tc::fence_proxy_async_smem();
    tc::prefetch_tmap(&tmap_q);
    const int z0 = c * p.NQ + qoff + t0;
    tc::mbar_arrive_expect_tx(bar(B_QLOAD), 2 * L::QT);
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int hf = 0; hf < D / 64; ++hf)
        tc::tma_load_3d(sbase + L::Q_OFF + i * L::QT + hf * L::HALF_Q, &tmap_q, bar(B_QLOAD), hf * 64, h * p.G,
                        z0 + i * p.TQ);
  }

  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < B_COUNT; ++i) {
        if (i == B_QLOAD || (early0 && (i == B_KFULL || i == B_VFULL))) continue;
        // warpgroup-wide events arrive once per warp (after __syncwarp)
        int count = 1;
        if (i == B_PFULL || i == B_PFULL + 1) count = 8;      // 2 CTAs x 4 warps
        if (i >= B_KROT && i < B_KROT + NST) count = 10;      // 2 x 4 RoPE warps + 2 forwarders
        if (i == B_QFULL) count = 16;                         // 2 CTAs x 8 softmax warps
        tc::mbar_init(bar(i), count);
      }
      *s_abort = 0;
    }
    // ring heads of the views whose rows the item reads, one lane per view
    // (with the insert fused: the heads as they are once it is done)
    bool ok = bad == 0;
    for (int v = lane; v <= vmax; v += 32) {
      const int hv = head_c[v];
      ok = ok && hv >= 0 && hv < g.F;
      s_head[v] = FUSED ? (hv + 1) % g.F : hv;
    }
    ok = __all_sync(0xffffffffu, ok);
    __syncwarp();
    // tile list over physical key rows [0, row_end), skipping tiles made only
    // of ring rows that no query of the pair may see (the hole of its last
    // token lies inside every other token's); 32 tiles per step
    int n = 0, wrap = 0;
    if (ok) {
      int a1 = 0, n1 = 0, a2 = 0, n2 = 0;
      if (vq >= 0) {
        const int slot = (s_head[vq] + fq) % g.F;
        ring_hole(g, vq, fq, slot, t_max, a1, n1, a2, n2);
        // the first token's hole holds every other token's: if it has no
        // second run, no row's mask has one
        int u1, m1, u2, m2;
        ring_hole(g, vq, fq, slot, pc * 4 * p.TQ, u1, m1, u2, m2);
        wrap = m2 > 0;
      }
      const int n_all = (row_end + BN - 1) / BN;
      for (int k0 = 0; k0 < n_all; k0 += 32) {
        const int k = k0 + lane, r0 = k * BN, r1 = min(r0 + BN, row_end);
        const bool keep = k < n_all && !(r0 >= a1 && r1 <= a1 + n1) && !(r0 >= a2 && r1 <= a2 + n2);
        const uint32_t ball = __ballot_sync(0xffffffffu, keep);
        if (keep) {
          const int slot_j = n + __popc(ball & ((1u << lane) - 1));
          s_tiles[slot_j] = r0;
          if (FUSED) {
            // which 64-row block of the tile is a view's new frame (bits 0-1),
            // and which of those this pair writes into the ring (bits 2-3): the
            // pair of a view's last query block sees all of its new frame
            uint32_t f = 0;
            for (int b = 0; b < 2; ++b) {
              const int u = r0 + 64 * b - g.P;
              if (u < 0 || u >= g.ring_rows() || r0 + 64 * b >= row_end) continue;
              const int v = u / FT, sl = (u % FT) / g.T;
              if (sl != (s_head[v] + g.F - 1) % g.F) continue;
              f |= 1u << b;
              if (v == vq && pc == p.nbf - 1) f |= 4u << b;
            }
            s_src[slot_j] = (uint8_t)f;
          }
        }
        n += __popc(ball);
      }
    } else if (rank == 0 && lane == 0) {
      set_status(p.status, bad ? bad : SKV_DEV_BAD_HEAD);
    }
    if (lane == 0) {
      *s_ntiles = n;
      *s_wrap = wrap;
      tc::fence_barrier_init();
    }
    // the tile list and the local barriers are ready: the producers may start
    tc::bar_arrive_n(BAR_TILES, 96);
  }
  if (warp == WARP_KTMA || warp == WARP_VTMA) {
    // the first NST tiles need no free stage: their copies start before the
    // TMEM allocation and the cluster barrier
    tc::bar_sync_n(BAR_TILES, 96);
    if (lane == 0) {
      const int n0 = *s_ntiles;
      tc::prefetch_tmap(warp == WARP_KTMA ? &tmap_k : &tmap_v);
      for (int j = early0 ? 1 : 0; j < n0 && j < NST; ++j) issue_tile(warp == WARP_KTMA, j);
    }
  }
  if (warp == WARP_KTMA) {
    tc::tmem_alloc_pair(tc::smem_u32(s_tmem), 512);
    tc::tmem_relinquish_pair();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();          // barriers of both CTAs initialised before any cross-CTA arrival
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int nt = *s_ntiles;
  if (FUSED && tid == 0) {
    // every CTA of the cache reads the heads in its set-up, before this
    // arrival; the last to arrive advances them (a head out of range stays,
    // as the insert leaves it) and leaves the counter at zero
    __threadfence();
    const int per_cache = 2 * g.Hkv * p.items;
    if (atomicAdd(p.sync + (size_t)c * g.V, 1) == per_cache - 1) {
      for (int v = 0; v < g.V; ++v) {
        const int hv = p.head_w[(size_t)c * g.V + v];
        if (hv >= 0 && hv < g.F) p.head_w[(size_t)c * g.V + v] = (hv + 1) % g.F;
      }
      p.sync[(size_t)c * g.V] = 0;
      __threadfence();
    }
  }

  if (warp >= 8 && warp < WARP_ROPE) {
    tc::setmaxnreg_dec<RegSplit<FUSED>::CTRL>();
    if (warp == WARP_KTMA || warp == WARP_VTMA) {
      // -------------------------------------- producers of this CTA's halves
      const bool is_k = warp == WARP_KTMA;
      if (lane == 0) {
        // tiles [0, NST) were issued before the cluster barrier (tile 0 at
        // entry with early0, even for an item that then has no tiles)
        int issued = max(min(nt, NST), early0 ? 1 : 0);
        for (int j = NST; j < nt; ++j) {
          const int s = j % NST, u = j / NST;
          if (!tc::mbar_wait_cluster<SW>(bar((is_k ? B_KEMPTY : B_VEMPTY) + s), (u - 1) & 1, wait_ns, s_abort))
            break;
          issue_tile(is_k, j);
          issued = j + 1;
        }
        if (*s_abort) set_status(p.status, SKV_DEV_TIMEOUT);
        // the copies this thread started land before the CTA exits, whether or
        // not their consumers (which may have given up) waited for them (the
        // query tiles are copied for every item, even one without key tiles)
        if (is_k) {
          volatile int never = 0;
          tc::mbar_wait<SW>(bar(B_QLOAD), 0, DRAIN_NS, &never);
        }
        for (int j = max(0, issued - NST); j < issued; ++j) {
          volatile int never = 0;
          tc::mbar_wait<SW>(bar((is_k ? B_KFULL : B_VFULL) + j % NST), (j / NST) & 1, DRAIN_NS, &never);
        }
      }
    } else if (warp == WARP_VFWD) {
      // ------------------- tell the even CTA when this CTA's V^T half landed
      // (one barrier per stage with the K rotation: a key tile is ready for
      // both of its MMAs at once, so the MMA issuer waits once per tile).
      // With the insert fused, a new-frame block this pair writes into the
      // ring (token-major in shared memory) goes out transposed first.
      if (nt > 0) {
        for (int j = 0; j < nt; ++j) {
          const int s = j % NST, u = j / NST;
          const bool ok = __all_sync(0xffffffffu, tc::mbar_wait<SW>(bar(B_VFULL + s), u & 1, wait_ns, s_abort));
          if (!ok) {
            if (lane == 0) set_status(p.status, SKV_DEV_TIMEOUT);
            break;
          }
          if (FUSED) {
            const uint32_t src = s_src[j];
#pragma unroll 1
            for (int kh = 0; kh < 2; ++kh) {
              if (!((src >> (2 + kh)) & 1u)) continue;
              // 64 keys x 64 dimensions, one key per 128-byte swizzled row;
              // lane: dimensions lane and lane + 32, 8 keys per 16-byte store
              const uint8_t* box = smem + L::V_OFF + s * L::VST + kh * L::HALF_V;
              uint16_t* dst = p.ring_vt + ((size_t)zc * D + (D / 2) * rank) * g.row_cap + s_tiles[j] + 64 * kh;
#pragma unroll
              for (int dh = 0; dh < 2; ++dh) {
                const int dd = lane + 32 * dh;
#pragma unroll 1
                for (int i = 0; i < 8; ++i) {
                  uint32_t w[4];
#pragma unroll
                  for (int e = 0; e < 8; e += 2) {
                    const int k0 = 8 * i + e;
                    const uint16_t lo = *reinterpret_cast<const uint16_t*>(
                        box + k0 * 128 + (((dd >> 3) ^ (k0 & 7)) << 4) + (dd & 7) * 2);
                    const uint16_t hi = *reinterpret_cast<const uint16_t*>(
                        box + (k0 + 1) * 128 + (((dd >> 3) ^ ((k0 + 1) & 7)) << 4) + (dd & 7) * 2);
                    w[e / 2] = (uint32_t)lo | ((uint32_t)hi << 16);
                  }
                  *reinterpret_cast<uint4*>(dst + (size_t)dd * g.row_cap + 8 * i) = make_uint4(w[0], w[1], w[2], w[3]);
                }
              }
            }
            __syncwarp();
          }
          tc::mbar_arrive_cluster_cta_if(bar_even(B_KROT + s), lane == 0);
        }
      }
    } else if (warp == WARP_MMA) {
      // ------------------------------------------ MMA issuer (even CTA only)
      if (lane == 0 && nt > 0 && rank == 0) {
        constexpr uint32_t idesc_qk = tc::idesc_f16(2 * BM, BN);
        constexpr uint32_t idesc_pv = tc::idesc_bf16(2 * BM, D);
        constexpr uint32_t idesc_pv_mn = tc::idesc_bf16_bmn(2 * BM, D);
        // descriptors advance by adding (byte offset >> 4) to the start-address field;
        // each CTA's operands sit at the same offsets in its own shared memory.
        // The k-steps are unrolled (one thread must stay ahead of the tensor
        // cores); each issue re-materialises its base descriptors (opaque
        // move) so the compiler does not hoist every descriptor of the loop
        // into registers.
        const uint64_t dq0 = tc::sdesc_sw128(sbase + L::Q_OFF);
        const uint64_t dk0 = tc::sdesc_sw128(sbase + L::K_OFF);
        const uint64_t dv0 = tc::sdesc_sw128(sbase + L::V_OFF);
        auto issue_qk = [&](int i, int s) {
          const uint64_t dq = tc::opaque(dq0 + ((uint32_t)(i * L::QT) >> 4));
          const uint64_t dk = tc::opaque(dk0 + ((uint32_t)(s * L::KST) >> 4));
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t oq = ((kk >> 2) * L::HALF_Q + (kk & 3) * 32) >> 4;
            const uint32_t ok = ((kk >> 2) * L::HALF_K + (kk & 3) * 32) >> 4;
            tc::mma_ss_pair(tmem + i * 128, dq + oq, dk + ok, idesc_qk, kk > 0);
          }
        };
        // mn: bit kh set = key block kh of the tile holds token-major values
        // (a new frame read from the step's input), an MN-major operand: 8
        // keys of 128 bytes per 1024-byte group, 16 keys = 2048 bytes per k-step
        auto issue_pv = [&](int i, int s, bool acc, uint32_t mn) {
          const uint64_t dv = tc::opaque(dv0 + ((uint32_t)(s * L::VST) >> 4));
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const bool bmn = FUSED && ((mn >> (kk >> 2)) & 1u);
            const uint32_t ov = ((kk >> 2) * L::HALF_V + (kk & 3) * (bmn ? 2048 : 32)) >> 4;
            tc::mma_ts_pair(tmem + 256 + i * 128, tmem + i * 128 + kk * 8, dv + ov, bmn ? idesc_pv_mn : idesc_pv,
                            (acc || kk > 0) ? 1u : 0u);
          }
        };
        bool ok = tc::mbar_wait_short<SW>(bar(B_QFULL), 0, wait_ns, s_abort);
        if (ok) ok = tc::mbar_wait_short<SW>(bar(B_KROT), 0, wait_ns, s_abort);
        if (ok) {
          tc::tc_fence_after();
          issue_qk(0, 0);
          tc::mma_commit_pair(bar(B_SFULL));
          issue_qk(1, 0);
          tc::mma_commit_pair(bar(B_SFULL + 1));
          tc::mma_commit_pair(bar(B_KEMPTY));
        }
        for (int j = 0; ok && j < nt; ++j) {
          const int s = j % NST;
          const int s2 = (j + 1) % NST, u2 = (j + 1) / NST;
          if (!(ok = tc::mbar_wait_short<SW>(bar(B_PFULL), j & 1, wait_ns, s_abort))) break;
          tc::tc_fence_after();
          const uint32_t mn = FUSED ? (uint32_t)s_src[j] & 3u : 0u;
          issue_pv(0, s, j > 0, mn);
          tc::mma_commit_pair(bar(B_ODONE));
          if (j + 1 < nt) {
            if (!(ok = tc::mbar_wait_short<SW>(bar(B_KROT + s2), u2 & 1, wait_ns, s_abort))) break;
            tc::tc_fence_after();
            issue_qk(0, s2);
            tc::mma_commit_pair(bar(B_SFULL));
          }
          if (!(ok = tc::mbar_wait_short<SW>(bar(B_PFULL + 1), j & 1, wait_ns, s_abort))) break;
          tc::tc_fence_after();
          issue_pv(1, s, j > 0, mn);
          tc::mma_commit_pair(bar(B_ODONE + 1));
          tc::mma_commit_pair(bar(B_VEMPTY + s));
          if (j + 1 < nt) {
            issue_qk(1, s2);
            tc::mma_commit_pair(bar(B_SFULL + 1));
            tc::mma_commit_pair(bar(B_KEMPTY + s2));
          }
        }
        if (!ok) set_status(p.status, SKV_DEV_TIMEOUT);
        // every MMA issued completes (in both CTAs' TMEM) before TMEM is released
        tc::mma_commit_pair(bar(B_DRAIN));
      }
      if (lane == 0 && nt > 0) {
        volatile int never = 0;
        tc::mbar_wait_cluster<SW>(bar(B_DRAIN), 0, DRAIN_NS, &never);
      }
    }
  } else if (warp >= WARP_ROPE) {
    // ----------------------------------------------------------------- RoPE
    tc::setmaxnreg_dec<RegSplit<FUSED>::ROPE>();
    const int rt = tid - WARP_ROPE * 32;   // 0..127
    constexpr int HALF = D / 2;
    // this CTA's 64 rows of every key tile, rotated in place once TMA has
    // landed them.  Thread (warp wr, lane ln) takes chunk ch = ln % NCH (8
    // frequencies) of NPT consecutive rows; inside a frame consecutive rows
    // have consecutive positions, so their (cos, sin) advance by one complex
    // multiplication with R(1) instead of a table load.  The first row's
    // table entries of the next tile are fetched while the current tile is
    // rotated.
    constexpr int NCH = HALF / 8;
    constexpr int NPT = HN * NCH / 128;   // rows per thread
    const int wr = rt >> 5, ln = rt & 31;
    const int ch = ln % NCH;
    const int row_base = wr * (HN / 4) + (ln / NCH) * NPT;
    const int ea = ch * 8, eb = HALF + ch * 8;
    const uint32_t off_a = (ea / 64) * L::HALF_K, off_b = (eb / 64) * L::HALF_K;
    const int ca = (ea % 64) / 8, cb = (eb % 64) / 8;
    const float4* rope4 = reinterpret_cast<const float4*>(p.rope);
    const Ang8 step = ang8_from(e_step4);             // R(1), loaded at entry
    const int row0 = HN * (int)rank + row_base;       // this thread's first row inside a tile
    int pf_pos = -1, pf_run = 0;
    float4 pf[4];
    auto fetch = [&](int jj) {
      const int r = s_tiles[jj] + row0;
      pf_pos = -1;
      if (r < row_end) {
        key_pos_run(g, s_head, r, pf_pos, pf_run);
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) pf[w4] = __ldg(rope4 + ((size_t)pf_pos * HALF + ea) / 2 + w4);
      }
    };
    if (nt > 0) {
      if (early0 && row0 < row_end) {
        // tile 0 is rows [0, BN) of the prefix: position = row, the rest of
        // the prefix is its run
        pf_pos = row0;
        pf_run = g.rope_steps ? g.P - row0 : 1;
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4) pf[w4] = e_pf[w4];
      } else {
        fetch(0);
      }
    }
#pragma unroll 1
    for (int j = 0; j < nt; ++j) {
      const int s = j % NST, u = j / NST;
      bool ok = tc::mbar_wait<SW>(bar(B_KFULL + s), u & 1, wait_ns, s_abort);
      const uint32_t src = FUSED ? (uint32_t)s_src[j] : 0u;
      if (FUSED && ((src >> (2 + rank)) & 1u)) {
        // this CTA's K block is a new frame of the pair's own view: it goes
        // into the ring slot of the oldest frame (pre-RoPE, by TMA) before it
        // is rotated in place.  (Barriers here see all four RoPE warps take
        // the same path: the predicate is the AND of every thread's wait.)
        ok = tc::bar_and(3, 128, ok);
        if (ok && rt == 0) {
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf)
            tc::tma_store_3d(&tmap_k, sbase + L::K_OFF + s * L::KST + hf * L::HALF_K, hf * 64,
                             s_tiles[j] + HN * (int)rank, zc);
          tc::tma_store_commit_wait_read();
        }
        tc::bar_and(3, 128, true);
      }
      if (!ok) {
        set_status(p.status, SKV_DEV_TIMEOUT);
        break;
      }
      if (pf_pos >= 0)
        rotate_key_rows<NPT, TABLE>(smem + L::K_OFF + s * L::KST, off_a, off_b, ca, cb, row_base, s_tiles[j] + row0,
                             row_end, pf_pos, pf_run, pf, step, g, s_head, rope4, ea, HALF);
      tc::fence_proxy_async();
      __syncwarp();
      tc::mbar_arrive_cluster_cta_if(bar_even(B_KROT + s), lane == 0);
      // after the arrive, whose release would otherwise wait for these loads
      if (j + 1 < nt) fetch(j + 1);
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    tc::setmaxnreg_inc<RegSplit<FUSED>::SOFTMAX>();
    const int i = warp >> 2;            // query tile
    const int lg = warp & 3;            // TMEM lane group of this warp
    const int row = lg * 32 + lane;
    const int tok = t0 + i * p.TQ + row / p.G;
    const int gq = row % p.G;
    const bool valid = tok < n_seg;
    const uint32_t t_lane = (uint32_t)(lg * 32) << 16;
    const uint32_t tS = tmem + t_lane + i * 128;
    const uint32_t tO = tmem + t_lane + 256 + i * 128;
    // the keys this query sees: rows [0, row_end) minus [a1, a1 + n1) and
    // [a2, a2 + n2) (rows past the segment's end act as its last token); the
    // second run, when the ring has turned, waits in shared memory
    int* my_mask = s_mask + i * BM + row;
    const uint32_t mask_sa = sbase + L::MASK_OFF + 4u * (i * BM + row);
    int a1 = 0, n1 = 0;
    const bool wrap = *s_wrap != 0;
    // Query rotation, part 1: the table entries of the thread's rows, loaded
    // first (they depend only on the rows' positions, so their latency runs
    // under the mask set-up and the queries' copy).  Query tiles as TMA
    // landed them: bf16 row r of tile qi = (token t0 + qi*TQ + r/G, head
    // r%G); thread tid takes chunk ch (8 frequencies) of NCH consecutive rows.
    // Rows of one token (its G heads) share one load; the rows that reuse
    // the previous row's entries (bit q of dup) take them once they landed.
    constexpr int HALF = D / 2, NCH = HALF / 8;
    const int ch = tid % NCH, rr0 = (tid / NCH) * NCH;
    const int ea = ch * 8, eb = HALF + ch * 8;
    float4 cs[NCH][4];
    uint32_t dup = 0;
    if (nt > 0) {
      const float4* rope4 = reinterpret_cast<const float4*>(p.rope);
      int prev_tok = -1;
#pragma unroll
      for (int q = 0; q < NCH; ++q) {
        const int rr = rr0 + q, qi = rr >> 7, r = rr & 127;
        const int qtok = min(t0 + qi * p.TQ + r / p.G, n_seg - 1);
        if (q > 0 && qtok == prev_tok) {
          dup |= 1u << q;
        } else {
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) cs[q][w4] = __ldg(rope4 + ((size_t)(pos0 + qtok) * HALF + ea) / 2 + w4);
        }
        prev_tok = qtok;
      }
    }
    if (nt > 0) {
      const int tq = min(tok, n_seg - 1);
      int a2 = 0, n2 = 0;
      if (vq < 0) {
        a1 = pos0 + tq + 1;         // the later tokens of a prefix / tail span
        n1 = row_end - a1;
      } else {
        ring_hole(g, vq, fq, (s_head[vq] + fq) % g.F, tq, a1, n1, a2, n2);
      }
      my_mask[0] = a2;
      my_mask[2 * BM] = n2;
      // output row (token, head) and LSE entry; both below 2^31 (checked at launch)
      const int tok_row = c * p.NQ + qoff + tok;
      my_mask[4 * BM] = valid ? tok_row * p.Hq + h * p.G + gq : -1;
      my_mask[6 * BM] = (c * p.Hq + h * p.G + gq) * p.NQ + qoff + tok;
    }
    const float sl = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    if (nt > 0) {
      // part 2: rotate in place, at each token's logical position, into fp16,
      // four rows at a time
      const uint32_t off_a = (ea / 64) * L::HALF_Q, off_b = (eb / 64) * L::HALF_Q;
      const int ca = (ea % 64) / 8, cb = (eb % 64) / 8;
      ok = __all_sync(0xffffffffu, tc::mbar_wait<SW>(bar(B_QLOAD), 0, wait_ns, s_abort));
      if (ok) {
#pragma unroll
        for (int q = 1; q < NCH; ++q)
          if ((dup >> q) & 1u) {
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) cs[q][w4] = cs[q - 1][w4];
          }
#pragma unroll
        for (int b4 = 0; b4 < NCH; b4 += 4) {
          uint4 xa[4], xb[4];
          uint8_t* rp[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int rr = rr0 + b4 + q, qi = rr >> 7, r = rr & 127;
            rp[q] = smem + L::Q_OFF + qi * L::QT;
            xa[q] = *reinterpret_cast<const uint4*>(rp[q] + off_a + tc::sw128_off(r, ca));
            xb[q] = *reinterpret_cast<const uint4*>(rp[q] + off_b + tc::sw128_off(r, cb));
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int r = (rr0 + b4 + q) & 127;
            rotate_pairs4(xa[q], xb[q], cs[b4 + q]);
            *reinterpret_cast<uint4*>(rp[q] + off_a + tc::sw128_off(r, ca)) = xa[q];
            *reinterpret_cast<uint4*>(rp[q] + off_b + tc::sw128_off(r, cb)) = xb[q];
          }
        }
        tc::fence_proxy_async();
      }
      __syncwarp();
      tc::mbar_arrive_cluster_cta_if(bar_even(B_QFULL), lane == 0 && ok);
    }
#pragma unroll 1
    for (int j = 0; ok && j < nt; ++j) {
      // tcgen05.ld/st below are warp-collective: every branch around them is warp-uniform
      ok = __all_sync(0xffffffffu, tc::mbar_wait_cluster<SW>(bar(B_SFULL + i), j & 1, wait_ns, s_abort));
      if (!ok) break;
      tc::tc_fence_after();
      // the whole 128-score row in one TMEM round trip
      uint32_t v[BN];
#pragma unroll
      for (int cb = 0; cb < BN / 32; ++cb)
        tc::tmem_ld32(tS + cb * 32, *reinterpret_cast<uint32_t(*)[32]>(v + cb * 32));
      const int r0 = s_tiles[j];
      const int a = a1 - r0, e = row_end - r0;
      const bool full = (n1 == 0 || a >= BN || a + n1 <= 0) && e >= BN;
      tc::tmem_wait_ld();
      if (!__all_sync(0xffffffffu, full)) {
#pragma unroll
        for (int k = 0; k < BN; ++k)
          if (!((uint32_t)(k - a) >= (uint32_t)n1 && k < e)) v[k] = __float_as_uint(-INFINITY);
      }
      if (wrap) {
        // the second run of a hole that wraps around the end of the ring
        const int b2 = tc::ld_shared_s32(mask_sa) - r0;
        const uint32_t n2 = (uint32_t)tc::ld_shared_s32(mask_sa + 2 * BM * 4);
        if (!__all_sync(0xffffffffu, n2 == 0 || b2 >= BN || b2 + (int)n2 <= 0)) {
#pragma unroll
          for (int k = 0; k < BN; ++k)
            if ((uint32_t)(k - b2) < n2) v[k] = __float_as_uint(-INFINITY);
        }
      }
      // The row max is taken on a query's first tile only; later tiles keep
      // the running max m_used.  A larger score then gives a probability above
      // 1, which costs nothing while the tile's sum stays under LAG_LIMIT (bf16
      // P and fp32 O and l keep their relative precision at any scale); a
      // larger sum (or an infinite one) sends the warp through the rescale:
      // the tile's own max, O and l scaled down to it, P again.
      auto row_max = [&]() {
        float m4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) m4[q] = fmaxf(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
#pragma unroll
        for (int k = 8; k < BN; k += 2)
          m4[(k >> 1) & 3] = fmax3(m4[(k >> 1) & 3], __uint_as_float(v[k]), __uint_as_float(v[k + 1]));
        return fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl;
      };
      // P = 2^(s*scale - m) as bf16 pairs into the first 64 columns of S_i;
      // scale-and-shift and the row sum run on packed fp32 pairs
      auto p_pass = [&]() {
        const uint64_t sl2 = f2_pack(sl, sl), nm2 = f2_pack(-m_used, -m_used);
        uint64_t l2[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) l2[q] = 0ull;
#pragma unroll
        for (int cb = 0; cb < BN / 32; ++cb) {
          uint32_t pk[16];
#pragma unroll
          for (int k = 0; k < 32; k += 2) {
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(v[cb * 32 + k]), __uint_as_float(v[cb * 32 + k + 1])), sl2, nm2),
                      x0, x1);
            const float p0 = tc::ex2(x0), p1 = tc::ex2(x1);
            l2[(k >> 1) & 3] = f2_add(l2[(k >> 1) & 3], f2_pack(p0, p1));
            pk[k >> 1] = pack_bf16x2(p0, p1);
          }
          tc::tmem_st16(tS + cb * 16, pk);
        }
        const uint64_t s2 = f2_add(f2_add(l2[0], l2[1]), f2_add(l2[2], l2[3]));
        float s0, s1;
        f2_unpack(s2, s0, s1);
        return s0 + s1;
      };
      if (j == 0) {
        const float mx = row_max();
        m_used = (mx == -INFINITY) ? 0.f : mx;
      }
      float ts = p_pass();
      if (__any_sync(0xffffffffu, !(ts <= LAG_LIMIT))) {
        // O_i holds tiles < j, all complete: S_i(j) was committed after PV_i(j-1).
        // Rows whose max did not grow keep theirs (alpha = 1) and write the same P again.
        tc::tmem_wait_st();
        const float mx = row_max();
        const float m_new = mx > m_used ? mx : m_used;
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
        m_used = m_new;
        ts = p_pass();
      }
      l += ts;
      tc::tmem_wait_st();
      tc::tc_fence_before();
      __syncwarp();
      tc::mbar_arrive_cluster_cta_if(bar_even(B_PFULL + i), lane == 0);
    }
    if (!ok) set_status(p.status, SKV_DEV_TIMEOUT);
    bool done = ok && nt > 0;
    if (done) done = __all_sync(0xffffffffu, tc::mbar_wait_cluster<SW>(bar(B_ODONE + i), (nt - 1) & 1, wait_ns, s_abort));
    if (done) {
      tc::tc_fence_after();
      const float inv_l = 1.f / l;
      const int o_row = my_mask[4 * BM];
      uint16_t* orow = p.out + (size_t)max(o_row, 0) * D;
#pragma unroll 1
      for (int cb = 0; cb < D / 32; ++cb) {
        uint32_t o[32];
        tc::tmem_ld32(tO + cb * 32, o);
        tc::tmem_wait_ld();
        if (o_row >= 0) {
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
      if (o_row >= 0 && p.lse)
        p.lse[my_mask[6 * BM]] =
            (m_used + __log2f(l)) * 0.69314718055994531f;
    } else if (nt > 0 && *s_abort) {
      set_status(p.status, SKV_DEV_TIMEOUT);
    }
  }

  // no cross-CTA traffic (arrivals, pair MMAs into this CTA's TMEM) after this point
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();
  if (warp == WARP_KTMA) {
    tc::tc_fence_after();
    tc::tmem_dealloc_pair(tmem, 512);
  }
}

// Raise the kernel's dynamic shared-memory limit once per device, and ask
// for the smallest shared-memory carve-out that holds it: the rest of the
// SM's 256 KB stays L1, which serves the rotary-table loads (measured: the
// largest carve-out made the 36-layer call 3% slower).
template <typename K>
cudaError_t set_smem_once(K kernel, int bytes, int variant) {
  static std::atomic<int> done[64][7];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev][variant].load(std::memory_order_relaxed)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxL1);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev][variant].store(1, std::memory_order_relaxed);
  return e;
}

}  // namespace

// K: [C*Hkv][row_cap][d] -> boxes of 64 dims x k_box_rows rows; V^T:
// [C*Hkv][d][row_cap] -> boxes of 64 keys x v_box_rows dimension rows.  Both
// with the 128-byte swizzle.
// cuTensorMapEncodeTiled from the driver, looked up once (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> cached{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 fn = cached.load(std::memory_order_relaxed);
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
      cached.store(fn, std::memory_order_relaxed);
    }
  }
  return fn;
}

cudaError_t make_kv_tmaps(const Geom& g, const void* k, const void* vt, int k_box_rows, int v_box_rows,
                          CUtensorMap* tk, CUtensorMap* tv) {
  auto fn = tmap_encode_fn();
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
    cuuint32_t box[3] = {64, (cuuint32_t)v_box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (fn(tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(vt), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

bool prefill_insert_fusable(const Geom& g) { return g.d == 128 && g.P % 64 == 0 && g.T % 64 == 0; }

cudaError_t launch_prefill_tc(const Geom& g, int Hq, const PrefillQuery& qs, const void* q, void* out, float* lse,
                              const void* k, const void* vt, const float* rope, int32_t* head,
                              float sm_scale, int32_t* status, uint64_t wait_ns, cudaStream_t st,
                              const void* k_new, const void* v_new, int32_t* sync) {
  if ((g.row_cap + BN - 1) / BN > MAX_TILES || g.V > MAX_VIEWS) return cudaErrorNotSupported;
  const bool fused = k_new != nullptr;
  if (fused && (!prefill_insert_fusable(g) || qs.nf != 1 || qs.n_tail || qs.prefix || !v_new || !sync))
    return cudaErrorInvalidValue;
  // output rows (token, head) and LSE entries are indexed in 32 bits
  if ((long long)g.C * qs.NQ * Hq > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  CUtensorMap tk, tv, tq;
  cudaError_t e = make_kv_tmaps(g, k, vt, HN, g.d / 2, &tk, &tv);
  if (e != cudaSuccess) return e;
  {
    // queries [C * NQ tokens][Hq][d] bf16: a box is 64 columns of the G
    // heads of one kv head for TQ tokens, i.e. 128 rows (token, head) of 128 B
    const int G = Hq / g.Hkv;
    cuuint64_t dims[3] = {(cuuint64_t)g.d, (cuuint64_t)Hq, (cuuint64_t)g.C * qs.NQ};
    cuuint64_t strides[2] = {(cuuint64_t)g.d * 2, (cuuint64_t)Hq * g.d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(BM / G)};
    cuuint32_t es[3] = {1, 1, 1};
    auto fn = tmap_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    if (fn(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // the step's new frames [C][V][T][Hkv][d]: boxes of 64 columns x 64 tokens
  // of one (cache, view, kv head), as the ring's K boxes and as token-major V
  CUtensorMap tkn = tk, tvn = tv;
  if (fused) {
    auto fn = tmap_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[4] = {(cuuint64_t)g.d, (cuuint64_t)g.Hkv, (cuuint64_t)g.T, (cuuint64_t)g.C * g.V};
    cuuint64_t strides[3] = {(cuuint64_t)g.d * 2, (cuuint64_t)g.Hkv * g.d * 2, (cuuint64_t)g.T * g.Hkv * g.d * 2};
    cuuint32_t box[4] = {64, 1, 64, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    for (int i = 0; i < 2; ++i)
      if (fn(i ? &tvn : &tkn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(i ? v_new : k_new), dims,
             strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
  }
  PrefillParams p;
  p.g = g;
  p.Hq = Hq;
  p.G = Hq / g.Hkv;
  p.TQ = BM / p.G;
  const int blk_tok = 4 * p.TQ;                    // tokens of one CTA pair
  p.n_tail = qs.n_tail;
  p.nbt = (qs.n_tail + blk_tok - 1) / blk_tok;
  p.nf = qs.nf;
  p.nbf = (g.T + blk_tok - 1) / blk_tok;
  p.nbp = qs.prefix ? (g.P + blk_tok - 1) / blk_tok : 0;
  p.items = p.nbt + g.V * p.nf * p.nbf + p.nbp;
  p.NQ = qs.NQ;
  p.q_view0 = qs.q_view0;
  p.q_tail0 = qs.q_tail0;
  p.tail_len = qs.tail_len;
  p.q = static_cast<const uint16_t*>(q);
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.rope = reinterpret_cast<const float2*>(rope);
  p.head = head;
  p.head_w = head;
  p.sync = sync;
  p.ring_k = static_cast<uint16_t*>(const_cast<void*>(k));
  p.ring_vt = static_cast<uint16_t*>(const_cast<void*>(vt));
  p.status = status;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.wait_ns = wait_ns ? wait_ns : 2000000000ull;
  if (p.nbt > 0 && !qs.tail_len) return cudaErrorInvalidValue;
  const long long blocks = 2LL * g.C * g.Hkv * p.items;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  const bool sw = p.wait_ns < tc::kSuspendHintNs;
  auto launch = [&](auto kernel, int smem, int variant) -> cudaError_t {
    cudaError_t err = set_smem_once(kernel, smem, variant);
    if (err != cudaSuccess) return err;
    kernel<<<(unsigned)blocks, NTHREADS, smem, st>>>(tk, tv, tq, tkn, tvn, p);
    return cudaSuccess;
  };
  if (fused)
    e = sw ? launch(prefill_tc_kernel<128, true, true>, Layout<128>::ALLOC, 5)
           : launch(prefill_tc_kernel<128, false, true>, Layout<128>::ALLOC, 4);
  else if (g.d == 128 && !sw && !g.rope_steps)
    e = launch(prefill_tc_kernel<128, false, false, true>, Layout<128>::ALLOC, 6);
  else if (g.d == 128)
    e = sw ? launch(prefill_tc_kernel<128, true, false>, Layout<128>::ALLOC, 2)
           : launch(prefill_tc_kernel<128, false, false>, Layout<128>::ALLOC, 0);
  else
    e = sw ? launch(prefill_tc_kernel<64, true, false>, Layout<64>::ALLOC, 3)
           : launch(prefill_tc_kernel<64, false, false>, Layout<64>::ALLOC, 1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace skv
