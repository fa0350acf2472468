// stream_attn_verify on the tensor cores: attention of a drafted block over
// the streaming cache, HBM-bound, with the key range of all caches spread
// evenly over one wave of CTAs.
//
// FlashDrive blog walkthrough, section 4.2: the target model checks a whole
// drafted block in one forward pass; VFlash "03 · Generalist decoding": the
// block holds one accepted anchor plus the proposals.  Block token j of
// cache c sits at logical index P + V*F*T + tail_len[c] + j and sees every
// key up to its own index (the block is causal within itself).
//
// Work units are (cache, kv head) planes of TM key tiles of 64 keys each.
// The units' tiles form one sequence of units x TM tiles; CTA b takes tiles
// [b*W, (b+1)*W) of it, so one wave of CTAs (two per SM) gets equal shares
// (a split in the manner of stream-K).  A CTA's share falls into pieces at
// unit boundaries; a unit that one piece covers is written straight to the
// output, otherwise every piece leaves an unnormalised fp32 partial (O,
// running max m, sum l) in the workspace.  With few pieces per unit the
// piece that arrives last merges them after its CTA's key loop; with many
// (small batches) the launch is cooperative, every CTA meets at a grid
// barrier once its partials are out, and all warps of the grid merge.
//
// Per piece the query buffer holds the unit's blk x G block rows in its 64
// rows (the WIDE form below: 128); the M=128 MMA reads rows past them from
// whatever shared memory follows, and their S and O rows (TMEM lanes) are
// never read.  Most MMA rows are idle: the kernel is bound by streaming K and
// V^T from HBM, not by the tensor cores.  The query block lands by TMA and is rotated in place;
// 64-key tiles flow through a 3-stage TMA ring for K (a stage is held while
// its tile is rotated) and a 2-stage one for V^T; RoPE is applied to each K
// tile in shared memory (fp16 out), S double-buffers in TMEM so QK of tile
// j+1 overlaps the softmax of tile j, and P (bf16) overwrites its S buffer
// for the PV MMA.
//
//   warps 0-1  softmax + epilogue (TMEM lanes 0-63 = block rows)
//   warp  2    K producer, TMEM allocator
//   warp  3    V^T producer
//   warp  4    MMA issuer
//   warps 5-8  RoPE (query block of every piece, then its K tiles)
// The WIDE form (blocks of more than 64 rows per kv head, one CTA per SM):
//   warps 0-3  softmax + epilogue (TMEM lanes 0-127)
//   warps 4-6  K producer, V^T producer, MMA issuer; warp 7 idle
//   warps 8-15 RoPE
#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "rope.cuh"
#include "tc.cuh"

namespace skv {

namespace {

constexpr int BM = 128;     // query-tile rows (block rows; the rest unused)
constexpr int BN = 64;      // keys per tile
constexpr int MAX_VIEWS = 64;
constexpr int MAX_PIECES = 16;   // pieces of one CTA's share
constexpr int MAX_SPLITS = 64;   // pieces of one unit
constexpr int MIN_SHARE = 4;     // key tiles per CTA at least
// When a unit may be cut into this many pieces or more (P_max), the units
// that pieces share are merged by every CTA after a grid barrier (a
// cooperative launch); with fewer, by each unit's last piece to arrive,
// which overlaps the merge with the other CTAs' key loops (measured: the
// barrier costs more than it saves at two pieces per unit, and saves a third
// of a batch-one call).
constexpr int COOP_MIN_PIECES = 4;
constexpr float RESCALE_THRESHOLD = 8.0f;
constexpr uint64_t DRAIN_NS = 500000000ull;

// Two forms of the kernel.  NARROW: units of up to 64 block rows, two
// softmax warps (TMEM lanes 0-63), four RoPE warps, two CTAs per SM.  WIDE,
// for blocks of more than 64 rows per kv head (17 tokens x 4 heads, say):
// units of up to 128 rows, four softmax warps (lanes 0-127), eight RoPE
// warps and one CTA per SM, so that a plane's keys stream once for all of
// its block rows.
template <bool WIDE>
struct VCfg {
  static constexpr int ROWS = WIDE ? 128 : 64;     // block rows of a unit at most
  static constexpr int SM_WARPS = ROWS / 32;       // softmax warps: TMEM lanes [0, ROWS)
  static constexpr int WARP_KTMA = SM_WARPS, WARP_VTMA = SM_WARPS + 1, WARP_MMA = SM_WARPS + 2;
  static constexpr int WARP_ROPE = WIDE ? 8 : 5;   // (WIDE: warp 7 has no role)
  static constexpr int ROPE_WARPS = WIDE ? 8 : 4;
  // RoPE groups: the RoPE warps split into RG groups that rotate alternate
  // key tiles (all of them rotate each piece's query block)
  static constexpr int RG = WIDE ? 2 : 1;
  static constexpr int NT = (WARP_ROPE + ROPE_WARPS) * 32;
  static constexpr int CTAS_PER_SM = WIDE ? 1 : 2;
  // K stages (a K tile is held through its rotation) and V^T stages: one
  // CTA per SM keeps as many bytes in flight as two of the narrow form
  static constexpr int KST = WIDE ? 6 : 3;
  static constexpr int VST = WIDE ? 4 : 2;
  // S buffers in TMEM (BN columns each; O follows them): the MMA issuer runs
  // QK up to NS - 1 tiles ahead of PV
  static constexpr int NS = WIDE ? 4 : 2;
  static constexpr int TMEM_COLS = WIDE ? 512 : 256;
};

// mbarrier slots for KST K stages and VST V^T stages
template <int KST, int VST, int NS>
struct VBars {
  enum : int {
    QLOAD = 0,                  // query block landed (TMA)
    QFULL = 1,                  // RoPE warps: query block rotated
    QEMPTY = 2,                 // MMA commit: the piece's QK MMAs are done with it
    KFULL = 3,                  // K tile landed
    KROT = KFULL + KST,         // RoPE warps: K tile rotated
    KEMPTY = KROT + KST,        // MMA commit: K stage free
    VFULL = KEMPTY + KST,       // V^T tile landed
    VEMPTY = VFULL + VST,       // MMA commit: V^T stage free
    SFULL = VEMPTY + VST,       // MMA commit: S buffer ready (NS)
    PFULL = SFULL + NS,         // softmax warps: P in the S buffer (NS)
    PVDONE = PFULL + NS,        // MMA commit: the PV of a tile landed in O (NS: one per S buffer)
    ODONE = PVDONE + NS,        // MMA commit: the piece's last PV landed
    OFREE = ODONE + 1,          // softmax warps: O read out
    DRAIN = OFREE + 1,          // MMA commit: everything issued is complete
    COUNT = DRAIN + 1
  };
};

template <int D, bool WIDE>
struct VLayout {
  static constexpr int QROWS = VCfg<WIDE>::ROWS;   // query rows kept in shared memory (block rows)
  static constexpr int QT = QROWS * D * 2;
  static constexpr int KT = BN * D * 2;   // 64 rows x D
  static constexpr int VT = D * BN * 2;   // D rows x 64 keys (one 128-byte-swizzled box)
  static constexpr int HALF_Q = QROWS * 128;
  static constexpr int HALF_K = BN * 128;
  static constexpr int Q_OFF = 0;
  static constexpr int K_OFF = Q_OFF + QT;
  static constexpr int KST = VCfg<WIDE>::KST, VST = VCfg<WIDE>::VST;
  static constexpr int V_OFF = K_OFF + KST * KT;
  // the merge keeps (m, l) of ROWS block rows x MAX_SPLITS pieces in the K
  // and V stages (extended where they are smaller)
  static constexpr int SCRATCH = 2 * QROWS * MAX_SPLITS * 4;
  static constexpr int BAR_OFF = (V_OFF + VST * VT > K_OFF + SCRATCH ? V_OFF + VST * VT : K_OFF + SCRATCH);
  static constexpr int NBAR = (VBars<KST, VST, VCfg<WIDE>::NS>::COUNT + 1) / 2 * 2;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int PIECE_OFF = MISC_OFF + 64;                 // MAX_PIECES x 8 ints
  static constexpr int MERGE_OFF = PIECE_OFF + MAX_PIECES * 32;   // units to merge
  static constexpr int HEAD_OFF = MERGE_OFF + MAX_PIECES * 4;     // per RoPE warp: MAX_VIEWS heads
  static constexpr int R64_OFF = HEAD_OFF + VCfg<WIDE>::ROPE_WARPS * MAX_VIEWS * 4;  // per RoPE warp: R(BN) of every chunk
  static constexpr int BYTES = R64_OFF + VCfg<WIDE>::ROPE_WARPS * (D / 16) * 64;
  static constexpr int ALLOC = BYTES + 1024;
};

// the rotation tables are read as float4
static_assert(VLayout<128, false>::R64_OFF % 16 == 0 && VLayout<64, false>::R64_OFF % 16 == 0 &&
                  VLayout<128, true>::R64_OFF % 16 == 0 && VLayout<64, true>::R64_OFF % 16 == 0,
              "R64 alignment");

// One piece of a CTA's share: tiles [ta, ta + nt) of unit u, piece k of the
// unit's n, whose cache has tl tail tokens; g0 = the CTA's tiles before it.
enum { PC_U = 0, PC_TA, PC_NT, PC_TL, PC_K, PC_N, PC_OK, PC_G0 };

struct VerifyParams {
  Geom g;
  int Hq, G, blk, R;          // R = blk * G block rows per kv head
  int RH, RU, TQH;            // row units per kv head (ROWS block rows each), rows per unit at most, tokens per query box
  int TM, W, P_max;           // tiles per unit, tiles per CTA, pieces per unit at most
  int units;
  const int32_t* tail_len;
  uint16_t* out;              // [C][blk][Hq][D]
  float* ws_o;                // [units * P_max][R][D]
  float* ws_ml;               // [units * P_max][R][2]
  int* ws_count;              // [units] arrival counters, zero between calls
  int coop;                   // 1: cooperative launch, the merge runs after a grid barrier on every CTA
  uint32_t* bar_count;        // grid barrier: arrivals (zero between calls) and generation
  uint32_t* bar_gen;
  const float2* rope;
  const int32_t* head;
  int32_t* status;
  float scale_log2;
  uint64_t wait_ns;
};

__host__ __device__ __forceinline__ int first_cta(long long u, int TM, int W) { return (int)(u * TM / W); }
__host__ __device__ __forceinline__ int last_cta(long long u, int TM, int W) { return (int)(((u + 1) * TM - 1) / W); }

// O = sum_k 2^(m_k - M) O_k / sum_k 2^(m_k - M) l_k over the n pieces of
// unit u, bf16 into the block rows; all threads of the CTA, with wts
// (shared memory, 2 x R x n floats) for the pieces' (m, l), then the per-row
// weights.  The partials are read from L2 with many loads in flight: this
// runs once the CTA's keys are done, on the kernel's tail.
template <int D, bool WIDE>
__device__ __noinline__ void merge_pieces(const VerifyParams& p, int u, int n, int tid, float* wts) {
  constexpr int NTHREADS = VCfg<WIDE>::NT;
  const size_t base = (size_t)u * p.P_max;
  const int plane = u / p.RH, rh = u % p.RH;
  const int c = plane / p.g.Hkv, h = plane % p.g.Hkv;
  const int row0 = rh * VCfg<WIDE>::ROWS;            // first block row of this unit
  const int R = min(p.RU, p.R - row0);               // its rows
  const int RS = p.RU;                               // row stride of the workspace
  float* wm = wts;           // [n][R]: m, then the weight
  float* wl = wts + n * R;   // [n][R]: l
  // every (piece, row) (m, l), four pairs per thread in flight
  for (int i0 = tid; i0 < n * R; i0 += 4 * NTHREADS) {
    float2 ml[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = i0 + q * NTHREADS;
      ml[q] = i < n * R ? __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + (base + i / R) * RS + i % R)
                        : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = i0 + q * NTHREADS;
      if (i < n * R) {
        wm[i] = ml[q].x;
        wl[i] = ml[q].y;
      }
    }
  }
  __syncthreads();
  for (int row = tid; row < R; row += NTHREADS) {
    float M = -INFINITY;
    for (int k = 0; k < n; ++k) M = fmaxf(M, wm[k * R + row]);
    float den = 0.f;
    for (int k = 0; k < n; ++k) {
      const float m = wm[k * R + row];
      const float w = m == -INFINITY ? 0.f : exp2f(m - M);
      wm[k * R + row] = w;
      den += w * wl[k * R + row];
    }
    const float inv = 1.f / den;
    for (int k = 0; k < n; ++k) wm[k * R + row] *= inv;
  }
  __syncthreads();
  // (row, 4 columns) items, two of them per thread and four pieces at a time in flight
  constexpr int D4 = D / 4;
  constexpr int IT = 2;
  const int n_items = R * D4;
  for (int e0 = tid; e0 < n_items; e0 += IT * NTHREADS) {
    float4 acc[IT];
#pragma unroll
    for (int q = 0; q < IT; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < n; k0 += 4) {
      float4 t[IT][4];
      float w[IT][4];
#pragma unroll
      for (int q = 0; q < IT; ++q) {
        const int e = e0 + q * NTHREADS, row = e < n_items ? e / D4 : 0, d4 = e % D4;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int k = k0 + kk;
          w[q][kk] = (e < n_items && k < n) ? wm[k * R + row] : 0.f;
          t[q][kk] = w[q][kk] != 0.f ? __ldcg(reinterpret_cast<const float4*>(p.ws_o + ((base + k) * RS + row) * D) + d4)
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int q = 0; q < IT; ++q)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          acc[q].x += w[q][kk] * t[q][kk].x;
          acc[q].y += w[q][kk] * t[q][kk].y;
          acc[q].z += w[q][kk] * t[q][kk].z;
          acc[q].w += w[q][kk] * t[q][kk].w;
        }
    }
#pragma unroll
    for (int q = 0; q < IT; ++q) {
      const int e = e0 + q * NTHREADS;
      if (e >= n_items) continue;
      const int row = e / D4, d4 = e % D4;
      const int jt = (row0 + row) / p.G, gq = (row0 + row) % p.G;
      uint2 pk;
      pk.x = pack_bf16x2(acc[q].x, acc[q].y);
      pk.y = pack_bf16x2(acc[q].z, acc[q].w);
      *reinterpret_cast<uint2*>(p.out + (((size_t)c * p.blk + jt) * p.Hq + h * p.G + gq) * D + d4 * 4) = pk;
    }
  }
  __syncthreads();
}

// The merge of every unit that more than one piece shares, spread over all
// warps of a cooperative launch once every piece has left its partial: warp
// gw of n_w takes (unit, row) pairs gw, gw + n_w, ...; lane k holds the (m, l)
// of pieces k and k + 32, the row max and the weights go round by shuffles,
// and lane i sums columns 4i .. 4i+3 over the pieces (eight loads in flight).
// A row whose pieces all left l = 0 belongs to a skipped cache and is not
// written.
template <int D, bool WIDE>
__device__ __noinline__ void merge_all(const VerifyParams& p, int gw, int n_w, int lane) {
  constexpr int D4 = D / 4;
  constexpr uint32_t FULL = 0xffffffffu;
  static_assert(MAX_SPLITS <= 64, "two pieces per lane");
  const float4* ws_o4 = reinterpret_cast<const float4*>(p.ws_o);
  const float2* ws_ml2 = reinterpret_cast<const float2*>(p.ws_ml);
  const long long pairs = (long long)p.units * p.RU;
  for (long long e = gw; e < pairs; e += n_w) {
    const int u = (int)(e / p.RU), row = (int)(e - (long long)u * p.RU);
    const int plane = u / p.RH, row0 = (u % p.RH) * VCfg<WIDE>::ROWS;
    if (row >= p.R - row0) continue;
    const int f = first_cta(u, p.TM, p.W), n = last_cta(u, p.TM, p.W) - f + 1;
    if (n <= 1) continue;                      // its one piece wrote the output
    const size_t base = (size_t)u * p.P_max;
    float mk[2], lk[2], M = -INFINITY;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int k = lane + 32 * q;
      const float2 ml = k < n ? __ldcg(ws_ml2 + (base + k) * p.RU + row) : make_float2(-INFINITY, 0.f);
      mk[q] = ml.x;
      lk[q] = ml.y;
      M = fmaxf(M, ml.x);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
    float wk[2], den = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      wk[q] = mk[q] == -INFINITY ? 0.f : exp2f(mk[q] - M);
      den += wk[q] * lk[q];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(FULL, den, o);
    if (!(den > 0.f)) continue;
    const float inv = 1.f / den;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k0 = 0; k0 < n; k0 += 8) {
      float w[8];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int k = k0 + kk;
        const float w0 = __shfl_sync(FULL, wk[0], k & 31), w1 = __shfl_sync(FULL, wk[1], k & 31);
        w[kk] = k < n ? (k < 32 ? w0 : w1) * inv : 0.f;
      }
      float4 t[8];
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        t[kk] = (lane < D4 && w[kk] != 0.f) ? __ldcg(ws_o4 + ((base + k0 + kk) * p.RU + row) * D4 + lane)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        acc.x += w[kk] * t[kk].x;
        acc.y += w[kk] * t[kk].y;
        acc.z += w[kk] * t[kk].z;
        acc.w += w[kk] * t[kk].w;
      }
    }
    if (lane < D4) {
      const int c = plane / p.g.Hkv, h = plane % p.g.Hkv;
      const int brow = row0 + row, jt = brow / p.G, gq = brow % p.G;
      uint2 pk;
      pk.x = pack_bf16x2(acc.x, acc.y);
      pk.y = pack_bf16x2(acc.z, acc.w);
      *reinterpret_cast<uint2*>(p.out + (((size_t)c * p.blk + jt) * p.Hq + h * p.G + gq) * D + lane * 4) = pk;
    }
  }
}

// SW: compiled for a wait limit under the suspend hint (see tc::bounded_wait)
// TABLE: rope_mode 1 (a table row per key), see rotate_key_rows.
template <int D, bool SW, bool WIDE, bool TABLE = false>
__global__ void __launch_bounds__(VCfg<WIDE>::NT, VCfg<WIDE>::CTAS_PER_SM)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                 const __grid_constant__ CUtensorMap tmap_q, const VerifyParams p) {
  using L = VLayout<D, WIDE>;
  using C = VCfg<WIDE>;
  constexpr int WARP_KTMA = C::WARP_KTMA, WARP_VTMA = C::WARP_VTMA, WARP_MMA = C::WARP_MMA;
  constexpr int WARP_ROPE = C::WARP_ROPE;
  constexpr int SOFTMAX_THREADS = C::ROWS;
  constexpr int NRT = C::ROPE_WARPS * 32;   // RoPE threads
  constexpr int KST = C::KST, VST = C::VST, NS = C::NS;
  using VB = VBars<KST, VST, NS>;
  constexpr int V_QLOAD = VB::QLOAD, V_QFULL = VB::QFULL, V_QEMPTY = VB::QEMPTY, V_KFULL = VB::KFULL;
  constexpr int V_KROT = VB::KROT, V_KEMPTY = VB::KEMPTY, V_VFULL = VB::VFULL, V_VEMPTY = VB::VEMPTY;
  constexpr int V_SFULL = VB::SFULL, V_PFULL = VB::PFULL, V_PVDONE = VB::PVDONE, V_ODONE = VB::ODONE;
  constexpr int V_OFREE = VB::OFREE, V_DRAIN = VB::DRAIN, V_COUNT = VB::COUNT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = tc::smem_u32(smem);
  auto bar = [&](int i) { return sbase + L::BAR_OFF + 8u * i; };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 4);
  // [0] piece count, [1] units to merge, [2..] the softmax warps' verdicts
  volatile int* s_info = reinterpret_cast<volatile int*>(smem + L::MISC_OFF + 8);
  int* s_piece = reinterpret_cast<int*>(smem + L::PIECE_OFF);
  int* s_merge = reinterpret_cast<int*>(smem + L::MERGE_OFF);

  const Geom& g = p.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t wait_ns = p.wait_ns;

  if (warp == 0) {
    if (lane == 0) {
      for (int i = 0; i < V_COUNT; ++i) {
        int count = 1;
        if (i == V_QFULL) count = C::ROPE_WARPS;
        if (i >= V_KROT && i < V_KROT + KST) count = C::ROPE_WARPS / C::RG;
        if ((i >= V_PFULL && i < V_PFULL + NS) || i == V_OFREE) count = C::SM_WARPS;
        tc::mbar_init(bar(i), count);
      }
      *s_abort = 0;
      s_info[1] = 0;
    }
    // this CTA's share [g0, g1) of the units' tile sequence, cut at unit
    // boundaries: piece l is unit u0 + l (its first tile ta, tiles before tb),
    // one lane per piece, so that the pieces' checks load together
    const long long g0 = (long long)blockIdx.x * p.W;
    const long long g1 = min(g0 + p.W, (long long)p.units * p.TM);
    const int u0 = (int)(g0 / p.TM);
    const int n = g1 > g0 ? min(MAX_PIECES, (int)((g1 - 1) / p.TM) - u0 + 1) : 0;
    int nt = 0;
    if (lane < n) {
      const int u = u0 + lane;
      const int ta = lane == 0 ? (int)(g0 - (long long)u0 * p.TM) : 0;
      const int tb = (int)min((long long)p.TM, g1 - (long long)u * p.TM);
      const int c = u / p.RH / g.Hkv;
      // unit checks: ring heads in range, tail within its capacity
      const int tl = p.tail_len[c];
      bool head_ok = true;
#pragma unroll 4
      for (int v = 0; v < g.V; ++v) {
        const int hv = p.head[(size_t)c * g.V + v];
        head_ok = head_ok && hv >= 0 && hv < g.F;
      }
      const bool ok = head_ok && tl >= 0 && tl + p.blk <= g.tail_cap;
      const int nt_unit = (g.n_visual() + tl + p.blk + BN - 1) / BN;
      nt = ok ? max(0, min(tb, nt_unit) - ta) : 0;
      int* pc = s_piece + lane * 8;
      pc[PC_U] = u;
      pc[PC_TA] = ta;
      pc[PC_NT] = nt;
      pc[PC_TL] = ok ? tl : 0;
      pc[PC_K] = (int)blockIdx.x - first_cta(u, p.TM, p.W);
      pc[PC_N] = last_cta(u, p.TM, p.W) - first_cta(u, p.TM, p.W) + 1;
      pc[PC_OK] = ok;
      // the tail's own checks are reported by the tail write
      if (!head_ok && ta == 0) set_status(p.status, SKV_DEV_BAD_HEAD);
    }
    // tiles of the pieces before each (exclusive prefix sum over the lanes)
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane < n) s_piece[lane * 8 + PC_G0] = incl - nt;
    if (lane == 0) {
      s_info[0] = n;
      tc::fence_barrier_init();
    }
  }
  if (warp == WARP_KTMA) {
    tc::tmem_alloc(tc::smem_u32(s_tmem), C::TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int n_pieces = s_info[0];
  // every role walks the same pieces; tiles are counted CTA-wide (stages and
  // S buffers), pieces with work are counted for the per-piece barriers
  auto P = [&](int i, int f) { return s_piece[i * 8 + f]; };

  if (warp == WARP_KTMA || warp == WARP_VTMA) {
    // ------------------------------------------------------------ producers
    const bool is_k = warp == WARP_KTMA;
    const int nst = is_k ? KST : VST;
    if (lane == 0) {
      tc::prefetch_tmap(is_k ? &tmap_k : &tmap_v);
      int gt = 0;
      bool ok = true, tail_ready = false;
      for (int pi = 0; ok && pi < n_pieces; ++pi) {
        const int nt = P(pi, PC_NT), ta = P(pi, PC_TA), zc = P(pi, PC_U) / p.RH;
        for (int j = 0; j < nt; ++j) {
          const int s = gt % nst, u = gt / nst, r0 = (ta + j) * BN;
          if (!tail_ready && r0 + BN > g.n_visual()) {
            // rows of the tail: the block's K/V are written by the kernel before this one
            asm volatile("griddepcontrol.wait;" ::: "memory");
            tail_ready = true;
          }
          if (gt >= nst && !(ok = tc::mbar_wait<SW>(bar((is_k ? V_KEMPTY : V_VEMPTY) + s), (u - 1) & 1, wait_ns, s_abort)))
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
          ++gt;
        }
      }
      if (!ok) set_status(p.status, SKV_DEV_TIMEOUT);
      // the copies this thread started land before the CTA exits, whether or
      // not their consumers (which may have given up) waited for them
      for (int j = max(0, gt - nst); j < gt; ++j) {
        volatile int never = 0;
        tc::mbar_wait<SW>(bar((is_k ? V_KFULL : V_VFULL) + j % nst), (j / nst) & 1, DRAIN_NS, &never);
      }
    }
  } else if (warp == WARP_MMA) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc::idesc_f16(BM, BN);
      constexpr uint32_t idesc_pv = tc::idesc_bf16(BM, D);
      const uint64_t dq0 = tc::sdesc_sw128(sbase + L::Q_OFF);
      const uint64_t dk0 = tc::sdesc_sw128(sbase + L::K_OFF);
      const uint64_t dv0 = tc::sdesc_sw128(sbase + L::V_OFF);
      auto issue_qk = [&](int gg) {
        const uint64_t dk = tc::opaque(dk0 + ((uint32_t)((gg % KST) * L::KT) >> 4));
        const uint64_t dq = tc::opaque(dq0);
        const uint32_t d_tmem = tmem + (gg % NS) * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offq = ((kk >> 2) * L::HALF_Q + (kk & 3) * 32) >> 4;
          const uint32_t offk = ((kk >> 2) * L::HALF_K + (kk & 3) * 32) >> 4;
          tc::mma_ss(d_tmem, dq + offq, dk + offk, idesc_qk, kk > 0);
        }
      };
      bool ok = true;
      int a = 0;   // pieces with work so far
      // PV of the CTA's tile gg; `first` = the piece's first, which starts O afresh
      auto issue_pv = [&](int gg, bool first) {
        const int vs = gg % VST, vu = gg / VST;
        if (!(ok = tc::mbar_wait_short<SW>(bar(V_VFULL + vs), vu & 1, wait_ns, s_abort))) return;
        if (!(ok = tc::mbar_wait_short<SW>(bar(V_PFULL + gg % NS), (gg / NS) & 1, wait_ns, s_abort))) return;
        // the softmax warps have read the previous piece's O out
        if (first && a > 0 && !(ok = tc::mbar_wait_short<SW>(bar(V_OFREE), (a - 1) & 1, wait_ns, s_abort))) return;
        tc::tc_fence_after();
        const uint64_t dv = tc::opaque(dv0 + ((uint32_t)(vs * L::VT) >> 4));
        const uint32_t a_tmem = tmem + (gg % NS) * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          tc::mma_ts(tmem + NS * BN, a_tmem + kk * 8, dv + (((kk & 3) * 32) >> 4), idesc_pv,
                     (!first || kk > 0) ? 1u : 0u);
        tc::mma_commit(bar(V_PVDONE + gg % NS));
        tc::mma_commit(bar(V_VEMPTY + vs));
      };
      int gt = 0;
      for (int pi = 0; ok && pi < n_pieces; ++pi) {
        const int nt = P(pi, PC_NT);
        if (nt == 0) continue;
        if (!(ok = tc::mbar_wait_short<SW>(bar(V_QFULL), a & 1, wait_ns, s_abort))) break;
        // step j: QK of the piece's tile j, then PV of its tile j - (NS - 1)
        // (S buffer of tile j is free: the PV of tile j - NS went out a step
        // earlier, and the tensor pipe runs in issue order)
        for (int j = 0; ok && j < nt + NS - 1; ++j) {
          const int gg = gt + j;
          if (j < nt) {
            if (!(ok = tc::mbar_wait_short<SW>(bar(V_KROT + gg % KST), (gg / KST) & 1, wait_ns, s_abort))) break;
            tc::tc_fence_after();
            issue_qk(gg);
            tc::mma_commit(bar(V_SFULL + gg % NS));
            tc::mma_commit(bar(V_KEMPTY + gg % KST));
            if (j == nt - 1) tc::mma_commit(bar(V_QEMPTY));
          }
          if (j >= NS - 1) issue_pv(gg - (NS - 1), j == NS - 1);
        }
        if (ok) tc::mma_commit(bar(V_ODONE));
        gt += nt;
        ++a;
      }
      if (!ok) set_status(p.status, SKV_DEV_TIMEOUT);
      // every MMA issued completes before TMEM is released
      tc::mma_commit(bar(V_DRAIN));
      volatile int never = 0;
      tc::mbar_wait<SW>(bar(V_DRAIN), 0, DRAIN_NS, &never);
    }
  } else if (warp >= WARP_ROPE) {
    // ----------------------------------------------------------------- RoPE
    const int rt = tid - WARP_ROPE * 32;   // 0 .. NRT-1
    const int wr = rt >> 5, ln = rt & 31;
    constexpr int HALF = D / 2;
    constexpr int NCH = HALF / 8;
    constexpr int RG = C::RG, RW = C::ROPE_WARPS / RG;   // groups of RW warps, alternate tiles
    constexpr int NPT = BN * NCH / (RW * 32);           // key rows per thread
    const int grp = wr / RW;
    int* s_head = reinterpret_cast<int*>(smem + L::HEAD_OFF) + wr * MAX_VIEWS;   // this warp's copy
    const int ch = ln % NCH;
    const int row_base = (wr % RW) * (BN / RW) + (ln / NCH) * NPT;
    const int ea = ch * 8, eb = HALF + ch * 8;
    const uint32_t off_a = (ea / 64) * L::HALF_K, off_b = (eb / 64) * L::HALF_K;
    const int ca = (ea % 64) / 8, cb = (eb % 64) / 8;
    const float4* rope4 = reinterpret_cast<const float4*>(p.rope);
    float4 step4[4];
#pragma unroll
    for (int w4 = 0; w4 < 4; ++w4) step4[w4] = __ldg(rope4 + (HALF + ea) / 2 + w4);   // R(1)
    const Ang8 step = ang8_from(step4);
    // R(RG BN) of every chunk in this warp's shared memory: a thread's first
    // row of its group's next tile, RG BN rows on inside the same run, is
    // this tile's first row turned by R(RG BN), no table load
    float4* s_r64 = reinterpret_cast<float4*>(smem + L::R64_OFF) + wr * NCH * 4;
    // (a table of at most RG BN rows has no run longer than that to turn along)
    if (ln < NCH * 4 && g.rope_len > RG * BN)
      s_r64[ln] = __ldg(rope4 + ((size_t)(RG * BN) * HALF + (ln / 4) * 8) / 2 + ln % 4);
    __syncwarp();
    int gt = 0, a = 0;
    bool ok = true, q_in_flight = false;
    for (int pi = 0; ok && pi < n_pieces; ++pi) {
      const int nt = P(pi, PC_NT);
      if (nt == 0) continue;
      const int u = P(pi, PC_U), ta = P(pi, PC_TA);
      const int plane = u / p.RH, c = plane / g.Hkv, h = plane % g.Hkv;
      const int row0 = (u % p.RH) * C::ROWS, R_u = min(p.RU, p.R - row0);   // this unit's block rows
      const int q_base = g.n_visual() + P(pi, PC_TL);   // logical index of block token 0
      for (int v = ln; v < g.V; v += 32) s_head[v] = p.head[(size_t)c * g.V + v];
      __syncwarp();
      // the query block of this piece: rows n = (token n / G, head n % G),
      // by TMA once the previous piece's QK MMAs are done with the buffer
      if (a > 0 && !(ok = tc::mbar_wait<SW>(bar(V_QEMPTY), (a - 1) & 1, wait_ns, s_abort))) break;
      if (rt == 0) {
        tc::mbar_arrive_expect_tx(bar(V_QLOAD), p.TQH * p.G * 128 * (D / 64));
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          tc::tma_load_3d(sbase + L::Q_OFF + hf * L::HALF_Q, &tmap_q, bar(V_QLOAD), hf * 64, h * p.G,
                          c * p.blk + row0 / p.G);
        q_in_flight = true;
      }
      if (!(ok = tc::mbar_wait<SW>(bar(V_QLOAD), a & 1, wait_ns, s_abort))) break;
      q_in_flight = false;
      // rotate the block rows in place at their tokens' positions (fp16 out)
      for (int it = rt; it < R_u * NCH; it += NRT) {
        const int n = it / NCH, cq = it % NCH;
        const int qa = cq * 8, qb = HALF + cq * 8;
        uint4* pa = reinterpret_cast<uint4*>(smem + L::Q_OFF + (qa / 64) * L::HALF_Q + tc::sw128_off(n, (qa % 64) / 8));
        uint4* pb = reinterpret_cast<uint4*>(smem + L::Q_OFF + (qb / 64) * L::HALF_Q + tc::sw128_off(n, (qb % 64) / 8));
        float4 cs[4];
#pragma unroll
        for (int w4 = 0; w4 < 4; ++w4)
          cs[w4] = __ldg(rope4 + ((size_t)(q_base + (row0 + n) / p.G) * HALF + qa) / 2 + w4);
        uint4 xa = *pa, xb = *pb;
        rotate_pairs4(xa, xb, cs);
        *pa = xa;
        *pb = xb;
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (ln == 0) tc::mbar_arrive(bar(V_QFULL));
      // key tiles: chunk ch (8 frequencies) of NPT consecutive rows per thread
      const int row_lim = q_base + p.blk;   // rows at or beyond are not keys of this pass
      // the first row's (cos, sin) of the next tile is fetched while the current one is rotated
      int pf_pos = -1, pf_run = 0;
      float4 pf[4];
      auto fetch = [&](int jj) {
        const int r = (ta + jj) * BN + row_base;
        pf_pos = -1;
        if (r < row_lim) {
          key_pos_run(g, s_head, r, pf_pos, pf_run);
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) pf[w4] = __ldg(rope4 + ((size_t)pf_pos * HALF + ea) / 2 + w4);
        }
      };
      // this group's tiles of the piece: j = j0, j0 + RG, ... (tile gg of the
      // CTA belongs to group gg mod RG)
      const int j0 = (grp - gt % RG + RG) % RG;
      if (j0 < nt) fetch(j0);
#pragma unroll 1
      for (int j = j0; j < nt; j += RG) {
        const int gg = gt + j, s = gg % KST;
        if (!(ok = tc::mbar_wait<SW>(bar(V_KFULL + s), (gg / KST) & 1, wait_ns, s_abort))) break;
        if (pf_pos >= 0)
          rotate_key_rows<NPT, TABLE>(smem + L::K_OFF + s * L::KT, off_a, off_b, ca, cb, row_base, (ta + j) * BN + row_base,
                               row_lim, pf_pos, pf_run, pf, step, g, s_head, rope4, ea, HALF);
        if (j + RG < nt) {
          if (pf_pos >= 0 && pf_run > RG * BN && (ta + j + RG) * BN + row_base < row_lim) {
            const float4* r = s_r64 + ch * 4;
#pragma unroll
            for (int w4 = 0; w4 < 4; ++w4) {
              const float4 c = pf[w4], t = r[w4];
              pf[w4] = make_float4(c.x * t.x - c.y * t.y, c.y * t.x + c.x * t.y,
                                   c.z * t.z - c.w * t.w, c.w * t.z + c.z * t.w);
            }
            pf_pos += RG * BN;
            pf_run -= RG * BN;
          } else {
            fetch(j + RG);
          }
        }
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (ln == 0) tc::mbar_arrive(bar(V_KROT + s));
      }
      gt += nt;
      ++a;
    }
    if (!ok) {
      set_status(p.status, SKV_DEV_TIMEOUT);
      if (q_in_flight) {
        // let the query copy this thread started land before the CTA exits
        volatile int never = 0;
        tc::mbar_wait<SW>(bar(V_QLOAD), a & 1, DRAIN_NS, &never);
      }
    }
  } else if (warp < C::SM_WARPS) {
    // ------------------------------------------------- softmax + epilogue
    const int row = warp * 32 + lane;            // TMEM lane = the unit's block row
    const uint32_t t_lane = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tmem + t_lane + NS * BN;
    const float sl = p.scale_log2;
    int gt = 0, a = 0;
    bool alive = true;
    for (int pi = 0; alive && pi < n_pieces; ++pi) {
      if (!P(pi, PC_OK)) {
        // a skipped cache: without a grid barrier no piece of its units
        // arrives; with one, the merge finds l = 0 in every piece and skips it
        if (p.coop && P(pi, PC_N) > 1 && (P(pi, PC_U) % p.RH) * C::ROWS + row < p.R) {
          const size_t sl = (size_t)P(pi, PC_U) * p.P_max + P(pi, PC_K);
          p.ws_ml[(sl * p.RU + row) * 2] = -INFINITY;
          p.ws_ml[(sl * p.RU + row) * 2 + 1] = 0.f;
        }
        continue;
      }
      const int nt = P(pi, PC_NT), u = P(pi, PC_U), n_unit = P(pi, PC_N);
      const int plane = u / p.RH, c = plane / g.Hkv, h = plane % g.Hkv;
      const int brow = (u % p.RH) * C::ROWS + row;   // block row of this lane
      const bool valid = brow < p.R;
      const int jt = valid ? brow / p.G : 0;
      const int gq = valid ? brow % p.G : 0;
      const bool multi = n_unit > 1;
      const size_t slot = (size_t)u * p.P_max + P(pi, PC_K);
      const int lim = g.n_visual() + P(pi, PC_TL) + jt;   // largest key index this row may see
      float m_used = -INFINITY, l = 0.f;
      bool ok = true;
#pragma unroll 1
      for (int j = 0; j < nt; ++j) {
        const int gg = gt + j, sb = gg % NS;
        // tcgen05.ld/st below are warp-collective: every branch around them is warp-uniform
        ok = __all_sync(0xffffffffu, tc::mbar_wait<SW>(bar(V_SFULL + sb), (gg / NS) & 1, wait_ns, s_abort));
        if (!ok) break;
        tc::tc_fence_after();
        const uint32_t tS = tmem + t_lane + sb * BN;
        uint32_t v[BN];
#pragma unroll
        for (int cb = 0; cb < BN / 32; ++cb)
          tc::tmem_ld32(tS + cb * 32, *reinterpret_cast<uint32_t(*)[32]>(v + cb * 32));
        const int r0 = (P(pi, PC_TA) + j) * BN;
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
        // (rows past the block hold no query: they never ask for a rescale)
        const bool grow = valid && j > 0 && mx > m_used + RESCALE_THRESHOLD;
        if (j == 0) {
          m_used = (mx == -INFINITY) ? 0.f : mx;
        } else if (__any_sync(0xffffffffu, grow)) {
          // PV of the previous tile must have landed in O before it is rescaled
          // (one barrier per S buffer: up to NS - 1 PVs may be in flight, but
          // only the one of tile gg - 1 on its buffer's barrier)
          ok = __all_sync(0xffffffffu, tc::mbar_wait<SW>(bar(V_PVDONE + (gg - 1) % NS), ((gg - 1) / NS) & 1,
                                                          wait_ns, s_abort));
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
        // the row sum in four packed fp32 pairs: one add per pair of probabilities
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
        {
          const uint64_t s2 = f2_add(f2_add(l2[0], l2[1]), f2_add(l2[2], l2[3]));
          float s0, s1;
          f2_unpack(s2, s0, s1);
          l += s0 + s1;
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(V_PFULL + sb));
      }
      if (ok && nt > 0) ok = __all_sync(0xffffffffu, tc::mbar_wait<SW>(bar(V_ODONE), a & 1, wait_ns, s_abort));
      // every softmax warp takes the same path from here (named barriers below)
      if (lane == 0) s_info[2 + warp] = ok;
      asm volatile("bar.sync 1, %0;" ::"r"(SOFTMAX_THREADS) : "memory");
#pragma unroll
      for (int w2 = 0; w2 < C::SM_WARPS; ++w2) ok = ok && s_info[2 + w2];
      asm volatile("bar.sync 1, %0;" ::"r"(SOFTMAX_THREADS) : "memory");
      if (!ok) {
        alive = false;
        break;
      }
      if (nt > 0) {
        tc::tc_fence_after();
        if (!multi) {
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
          float* orow = p.ws_o + (slot * p.RU + row) * D;
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
        }
        // O is read out: the next piece's first PV may overwrite it
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(V_OFREE));
      }
      if (multi) {
        // this piece's share (empty when it lies past the unit's keys)
        if (valid) {
          p.ws_ml[(slot * p.RU + row) * 2] = nt > 0 ? m_used : -INFINITY;
          p.ws_ml[(slot * p.RU + row) * 2 + 1] = nt > 0 ? l : 0.f;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(SOFTMAX_THREADS) : "memory");
        if (tid == 0 && !p.coop) {
          __threadfence();
          const int prev = atomicAdd(&p.ws_count[u], 1);
          if (prev == n_unit - 1) {
            // the last piece of unit u: merge it once this CTA's keys are done
            p.ws_count[u] = 0;
            __threadfence();
            s_merge[s_info[1]] = u;
            s_info[1] = s_info[1] + 1;
          }
        }
      }
      gt += nt;
      if (nt > 0) ++a;
    }
    if (!alive) set_status(p.status, SKV_DEV_TIMEOUT);
  }

  tc::tc_fence_before();
  __syncthreads();
  if (warp == WARP_KTMA) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (p.coop) {
    // every CTA's partials are in the workspace once all have arrived here;
    // then all warps of the grid merge the units that pieces share
    if (tc::grid_barrier(p.bar_count, p.bar_gen, gridDim.x, wait_ns, s_info + 12))
      merge_all<D, WIDE>(p, (int)blockIdx.x * (C::NT / 32) + warp, (int)gridDim.x * (C::NT / 32), lane);
    else if (tid == 0)
      set_status(p.status, SKV_DEV_TIMEOUT);
    return;
  }
  // units whose last piece this CTA held: the K/V stages are idle now and hold
  // the merge weights
  const int n_merge = s_info[1];
  if (n_merge > 0 && !*s_abort) {
    __threadfence();
    for (int i = 0; i < n_merge; ++i) {
      const int u = s_merge[i];
      merge_pieces<D, WIDE>(p, u, last_cta(u, p.TM, p.W) - first_cta(u, p.TM, p.W) + 1, tid,
                            reinterpret_cast<float*>(smem + L::K_OFF));
    }
  }
}

// SM count per device ordinal, asked once (threads that race store the same value)
std::atomic<int> g_num_sms[64];

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = g_num_sms[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_num_sms[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// Raise the kernel's dynamic shared-memory limit once per device and return
// how many of its CTAs one SM holds (asked once per device as well).
template <typename K>
cudaError_t set_smem_once(K kernel, int bytes, int threads, int variant, int* per_sm) {
  static std::atomic<int> occ[64][10];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && (*per_sm = occ[dev][variant].load(std::memory_order_relaxed)) > 0)
    return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  int n = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, bytes);
  if (e != cudaSuccess) return e;
  *per_sm = n;
  if (dev >= 0 && dev < 64 && n > 0) occ[dev][variant].store(n, std::memory_order_relaxed);
  return cudaSuccess;
}

struct VerifyPlan {
  int TM, W, n_cta, P_max;
};

// Partition.  Two CTAs (WIDE: one) are resident per SM.  When the units alone fill more
// than half of that wave, each CTA takes one whole unit; otherwise the
// units' tiles are spread over at most one wave, each CTA taking at least
// MIN_SHARE tiles and at most MAX_PIECES - 2 whole units' worth (so its
// share has at most MAX_PIECES pieces), every unit in at most MAX_SPLITS
// pieces, no CTA empty.
VerifyPlan verify_plan(const Geom& g, int RH, bool wide) {
  VerifyPlan pl;
  const long long units = (long long)g.C * g.Hkv * RH;
  pl.TM = (g.n_visual() + g.tail_cap + BN - 1) / BN;
  const long long total = units * pl.TM;
  const long long slots = (long long)(wide ? VCfg<true>::CTAS_PER_SM : VCfg<false>::CTAS_PER_SM) * num_sms();
  if (units <= slots && 2 * units > slots) {
    // one whole unit per CTA already fills most of the wave: no partials
    pl.W = pl.TM;
    pl.n_cta = (int)units;
    pl.P_max = 1;
    return pl;
  }
  long long n = min(slots, (total + MIN_SHARE - 1) / MIN_SHARE);
  n = max(n, (units + MAX_PIECES - 3) / (MAX_PIECES - 2));
  n = min(n, total / max(1LL, (long long)((pl.TM + MAX_SPLITS - 2) / (MAX_SPLITS - 1))));
  n = max(n, 1LL);
  const long long W = (total + n - 1) / n;
  n = (total + W - 1) / W;
  pl.W = (int)W;
  pl.n_cta = (int)n;
  pl.P_max = (int)((pl.TM + W - 1) / W + 1);
  return pl;
}

// True when every unit lies inside one CTA's share (no partials to merge).
bool all_single(const VerifyPlan& pl, long long units) {
  if (pl.W % pl.TM != 0) return false;
  (void)units;
  return true;
}

}  // namespace

// The WIDE form serves blocks of more than 64 rows per kv head.
bool verify_wide(int Hq, int Hkv, int blk) { return blk * (Hq / Hkv) > VCfg<false>::ROWS; }

// Block rows per kv head in units of at most ROWS of the form: each (cache,
// kv head, row unit) is one work unit that streams the plane's keys.
int row_halves(int Hq, int Hkv, int blk) {
  const int rows = verify_wide(Hq, Hkv, blk) ? VCfg<true>::ROWS : VCfg<false>::ROWS;
  return (blk * (Hq / Hkv) + rows - 1) / rows;
}

// Workspace: [units] int32 arrival counters and the grid barrier's two words
// (a 256-byte aligned block), then the fp32 partial O rows and the (m, l)
// pairs of units x P_max piece slots, each slot holding a unit's (at most
// ROWS of the form) rows.
size_t ws_header_bytes(size_t units) { return ((units + 2) * 4 + 255) / 256 * 256; }

size_t verify_ws_bytes(const Geom& g, int Hq, int blk) {
  const bool wide = verify_wide(Hq, g.Hkv, blk);
  const int RH = row_halves(Hq, g.Hkv, blk);
  const VerifyPlan pl = verify_plan(g, RH, wide);
  const size_t units = (size_t)g.C * g.Hkv * RH;
  if (units == 0 || all_single(pl, (long long)units)) return 0;
  const size_t rows = units * pl.P_max * min(blk * (Hq / g.Hkv), wide ? VCfg<true>::ROWS : VCfg<false>::ROWS);
  return ws_header_bytes(units) + rows * (g.d + 2) * sizeof(float);
}

cudaError_t make_kv_tmaps(const Geom& g, const void* k, const void* vt, int k_box_rows, int v_box_rows,
                          CUtensorMap* tk, CUtensorMap* tv);
PFN_cuTensorMapEncodeTiled_v12000 tmap_encode_fn();

cudaError_t launch_verify_tc(const Geom& g, int Hq, int blk, const int32_t* tail_len, const void* q, void* out,
                             const void* k, const void* vt, const float* rope, const int32_t* head,
                             void* ws, size_t ws_bytes, float sm_scale, int32_t* status, uint64_t wait_ns,
                             cudaStream_t st) {
  const bool wide = verify_wide(Hq, g.Hkv, blk);
  const int ROWS = wide ? VCfg<true>::ROWS : VCfg<false>::ROWS;
  if (g.V > MAX_VIEWS || Hq / g.Hkv > VCfg<false>::ROWS) return cudaErrorNotSupported;
  const int RH = row_halves(Hq, g.Hkv, blk);
  const size_t units = (size_t)g.C * g.Hkv * RH;
  if (units == 0) return cudaSuccess;
  CUtensorMap tk, tv, tq;
  cudaError_t e = make_kv_tmaps(g, k, vt, BN, g.d, &tk, &tv);
  if (e != cudaSuccess) return e;
  {
    // block queries [C * blk tokens][Hq][d] bf16: a box is 64 columns of the
    // G heads of one kv head for the tokens of one row half, i.e. its block
    // rows (token, head)
    const int G = Hq / g.Hkv;
    const int box_tok = RH > 1 ? ROWS / G : blk;
    cuuint64_t dims[3] = {(cuuint64_t)g.d, (cuuint64_t)Hq, (cuuint64_t)g.C * blk};
    cuuint64_t strides[2] = {(cuuint64_t)g.d * 2, (cuuint64_t)Hq * g.d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)box_tok};
    cuuint32_t es[3] = {1, 1, 1};
    auto fn = tmap_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    if (fn(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const VerifyPlan pl = verify_plan(g, RH, wide);
  VerifyParams p;
  p.g = g;
  p.Hq = Hq;
  p.G = Hq / g.Hkv;
  p.blk = blk;
  p.R = blk * p.G;
  p.RH = RH;
  p.RU = min(p.R, ROWS);
  p.TQH = RH > 1 ? ROWS / p.G : blk;
  p.TM = pl.TM;
  p.W = pl.W;
  p.P_max = pl.P_max;
  p.units = (int)units;
  p.tail_len = tail_len;
  p.out = static_cast<uint16_t*>(out);
  const size_t need = verify_ws_bytes(g, Hq, blk);
  if (ws_bytes < need || (need && !ws)) return cudaErrorInvalidValue;
  const size_t n_rows = units * p.P_max * p.RU;
  p.ws_count = static_cast<int*>(ws);
  p.ws_o = need ? reinterpret_cast<float*>(static_cast<char*>(ws) + ws_header_bytes(units)) : nullptr;
  p.ws_ml = need ? p.ws_o + n_rows * g.d : nullptr;
  p.bar_count = need ? reinterpret_cast<uint32_t*>(ws) + units : nullptr;
  p.bar_gen = need ? p.bar_count + 1 : nullptr;
  p.rope = reinterpret_cast<const float2*>(rope);
  p.head = head;
  p.status = status;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.wait_ns = wait_ns ? wait_ns : 2000000000ull;
  // When pieces share units and the grid fits on the GPU at once, the launch
  // is cooperative: every CTA waits at a grid barrier for all partials, then
  // all of them merge.  Otherwise the last piece of a unit to arrive merges
  // it, and the launch is a programmatic dependent of the tail write before
  // it (set-up, query blocks and visual key tiles overlap that kernel, whose
  // writes the producers wait for before they load a tile that reaches the
  // tail).
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3((unsigned)pl.n_cta);
  const int n_threads = wide ? VCfg<true>::NT : VCfg<false>::NT;
  cfg.blockDim = dim3(n_threads);
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool sw = p.wait_ns < tc::kSuspendHintNs;
  auto launch = [&](auto kernel, int smem, int variant) -> cudaError_t {
    int per_sm = 0;
    cudaError_t err = set_smem_once(kernel, smem, n_threads, variant, &per_sm);
    if (err != cudaSuccess) return err;
    p.coop = need > 0 && pl.P_max >= COOP_MIN_PIECES && (long long)pl.n_cta <= (long long)per_sm * num_sms();
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.numAttrs = p.coop ? 2 : 1;
    cfg.dynamicSmemBytes = smem;
    cudaError_t le = cudaLaunchKernelEx(&cfg, kernel, tk, tv, tq, p);
    if (le != cudaSuccess && p.coop) {
      // a driver that refuses the pair of attributes: a cooperative launch
      // alone (the refusal is a launch-argument error, cleared here)
      cudaGetLastError();
      attr[0] = attr[1];
      cfg.numAttrs = 1;
      le = cudaLaunchKernelEx(&cfg, kernel, tk, tv, tq, p);
    }
    return le;
  };
  const bool table = g.d == 128 && !sw && !g.rope_steps;
  if (table) {
    e = wide ? launch(verify_tc_kernel<128, false, true, true>, VLayout<128, true>::ALLOC, 9)
             : launch(verify_tc_kernel<128, false, false, true>, VLayout<128, false>::ALLOC, 8);
  } else if (wide) {
    if (g.d == 128)
      e = sw ? launch(verify_tc_kernel<128, true, true>, VLayout<128, true>::ALLOC, 6)
             : launch(verify_tc_kernel<128, false, true>, VLayout<128, true>::ALLOC, 4);
    else
      e = sw ? launch(verify_tc_kernel<64, true, true>, VLayout<64, true>::ALLOC, 7)
             : launch(verify_tc_kernel<64, false, true>, VLayout<64, true>::ALLOC, 5);
  } else if (g.d == 128) {
    e = sw ? launch(verify_tc_kernel<128, true, false>, VLayout<128, false>::ALLOC, 2)
           : launch(verify_tc_kernel<128, false, false>, VLayout<128, false>::ALLOC, 0);
  } else {
    e = sw ? launch(verify_tc_kernel<64, true, false>, VLayout<64, false>::ALLOC, 3)
           : launch(verify_tc_kernel<64, false, false>, VLayout<64, false>::ALLOC, 1);
  }
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace skv
