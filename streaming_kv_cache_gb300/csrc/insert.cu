// Writing token-major K/V into the cache: the frame insert of a streaming
// step (evict the oldest slot of each view's ring, advance its head), the
// placement of prefix/tail rows, and the verify block's tail write.
//
// FlashDrive blog walkthrough, section 3.1: each step evicts every view's
// oldest frame, keeps the other frames and only adds the newest one.  Here
// the ring never moves data: the new frame overwrites the slot of the oldest
// frame and the view's head advances by one (mod F).
//
// One CTA copies a chunk of CH tokens of one (cache, group, kv head): the K
// rows are straight 16-byte copies into [row][d]; the V rows go through
// shared memory and are written transposed into [d][row], one coalesced run
// of CH tokens per dimension.  In a full chunk every thread has all of its
// 16-byte loads in flight before its first store.
//
// The verify block's tail write also computes the greedy accept length (it
// needs only the token ids) and lets the attention kernel that follows launch
// early: that kernel waits for this one's writes only before it reads tail rows.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace skv {

namespace {

constexpr int CH = 32;        // tokens per CTA
constexpr int THREADS = 128;

enum WriteMode { MODE_ROWS = 0, MODE_INSERT = 1, MODE_TAIL = 2 };

// Token ids of a verify block and the accept outputs (all null: none).
struct AcceptArgs {
  const int32_t* target;
  const int32_t* draft;
  int32_t* accept_len;
  int32_t* next_token;
};

// TAIL: the instance that serves the verify block's tail writes, which asks
// for its own shared-memory carve-out (below); the code is the same.
template <int D, bool TAIL>
__global__ void __launch_bounds__(THREADS) write_rows_kernel(
    Geom g, uint16_t* __restrict__ k, uint16_t* __restrict__ vt,
    const uint16_t* __restrict__ k_src, const uint16_t* __restrict__ v_src, int n_group,
    int n_tok, int mode, int row0, int32_t* __restrict__ head, int32_t* __restrict__ sync,
    const int32_t* __restrict__ tail_len, int32_t* __restrict__ status, AcceptArgs acc) {
  __shared__ __align__(16) uint16_t sv[CH][D + 2];
  __shared__ int s_base;
  // the attention kernel after a tail write may start its own set-up now
  if (mode == MODE_TAIL) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int n_chunk = (n_tok + CH - 1) / CH;
  int bid = blockIdx.x;
  const int chunk = bid % n_chunk;  bid /= n_chunk;
  const int h = bid % g.Hkv;        bid /= g.Hkv;
  const int grp = bid % n_group;    bid /= n_group;
  const int c = bid;
  const int t0 = chunk * CH;
  const int nt = min(CH, n_tok - t0);

  if (threadIdx.x == 0) {
    int base = -1;
    if (mode == MODE_ROWS) {
      base = row0;
    } else if (mode == MODE_INSERT) {
      const int s = head[c * g.V + grp];
      if (s >= 0 && s < g.F) base = g.P + (grp * g.F + s) * g.T;
      else if (h == 0 && chunk == 0) set_status(status, SKV_DEV_BAD_HEAD);
    } else {
      const int tl = tail_len[c];
      if (tl < 0) {
        if (h == 0 && chunk == 0) set_status(status, SKV_DEV_BAD_TAIL);
      } else if (tl + n_tok > g.tail_cap) {
        if (h == 0 && chunk == 0) set_status(status, SKV_DEV_TAIL_OVERFLOW);
      } else {
        base = g.n_visual() + tl;
      }
    }
    s_base = base;
  }
  __syncthreads();
  const int base = s_base;

  if (base >= 0) {
    // K: token-major source rows -> [c][h][row][d]; 16-byte vectors.
    constexpr int VEC = D / 8;
    const size_t src_tok_stride = (size_t)g.Hkv * D;
    const uint16_t* ks = k_src + (((size_t)c * n_group + grp) * n_tok + t0) * src_tok_stride + (size_t)h * D;
    const uint16_t* vs = v_src + (((size_t)c * n_group + grp) * n_tok + t0) * src_tok_stride + (size_t)h * D;
    uint16_t* kd = k + (((size_t)c * g.Hkv + h) * g.row_cap + base + t0) * D;
    constexpr int PER = CH * VEC / THREADS;   // vectors per thread of a full chunk
    if (nt == CH) {
      // a full chunk: every load of this thread in flight before its stores
      uint4 kv[PER], vv[PER];
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int i = threadIdx.x + q * THREADS, t = i / VEC, j = i - t * VEC;
        kv[q] = *reinterpret_cast<const uint4*>(ks + t * src_tok_stride + j * 8);
        vv[q] = *reinterpret_cast<const uint4*>(vs + t * src_tok_stride + j * 8);
      }
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        const int i = threadIdx.x + q * THREADS, t = i / VEC, j = i - t * VEC;
        *reinterpret_cast<uint4*>(kd + (size_t)t * D + j * 8) = kv[q];
        const uint16_t* pv = reinterpret_cast<const uint16_t*>(&vv[q]);
#pragma unroll
        for (int e = 0; e < 8; ++e) sv[t][j * 8 + e] = pv[e];
      }
    } else {
      for (int i = threadIdx.x; i < nt * VEC; i += THREADS) {
        const int t = i / VEC, j = i - t * VEC;
        const uint4 val = *reinterpret_cast<const uint4*>(ks + t * src_tok_stride + j * 8);
        *reinterpret_cast<uint4*>(kd + (size_t)t * D + j * 8) = val;
        const uint4 vv = *reinterpret_cast<const uint4*>(vs + t * src_tok_stride + j * 8);
        const uint16_t* pv = reinterpret_cast<const uint16_t*>(&vv);
#pragma unroll
        for (int e = 0; e < 8; ++e) sv[t][j * 8 + e] = pv[e];
      }
    }
    __syncthreads();
    // V: transposed write, one run of nt tokens per dimension.
    uint16_t* vd = vt + ((size_t)c * g.Hkv + h) * D * (size_t)g.row_cap + base + t0;
    for (int i = threadIdx.x; i < D * CH; i += THREADS) {
      const int dim = i / CH, t = i - dim * CH;
      if (t < nt) vd[(size_t)dim * g.row_cap + t] = sv[t][dim];
    }
  }

  if (mode == MODE_TAIL && acc.target && h == 0 && chunk == 0 && threadIdx.x == 0) {
    // greedy longest prefix: the largest k <= n_tok-1 with draft[i] == target[i-1]
    // for 1 <= i <= k; the target's own token at k comes next
    const int32_t* t = acc.target + (size_t)c * n_tok;
    const int32_t* dr = acc.draft + (size_t)c * n_tok;
    int kk = 0;
    while (kk + 1 < n_tok && dr[kk + 1] == t[kk]) ++kk;
    acc.accept_len[c] = kk;
    acc.next_token[c] = t[kk];
  }

  if (mode == MODE_INSERT) {
    // The last CTA of this (cache, view) to finish advances the head; every
    // CTA has read the head before it arrives here, and the counter is left
    // at zero for the next step.
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      const int per_view = g.Hkv * n_chunk;
      const int done = atomicAdd(&sync[c * g.V + grp], 1);
      if (done == per_view - 1) {
        if (base >= 0) head[c * g.V + grp] = (head[c * g.V + grp] + 1) % g.F;
        sync[c * g.V + grp] = 0;
        __threadfence();
      }
    }
  }
}

}  // namespace

cudaError_t launch_write_rows(const Geom& g, void* k, void* vt, const void* k_src,
                              const void* v_src, int n_group, int n_tok, int mode, int row0,
                              int32_t* head, int32_t* sync, const int32_t* tail_len,
                              int32_t* status, cudaStream_t st, const int32_t* target,
                              const int32_t* draft, int32_t* accept_len, int32_t* next_token) {
  const AcceptArgs acc{target, draft, accept_len, next_token};
  if (n_tok <= 0 || g.C <= 0) return cudaSuccess;
  const long long blocks = (long long)g.C * n_group * g.Hkv * ((n_tok + CH - 1) / CH);
  if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
  auto* kk = static_cast<uint16_t*>(k);
  auto* vv = static_cast<uint16_t*>(vt);
  auto* ks = static_cast<const uint16_t*>(k_src);
  auto* vs = static_cast<const uint16_t*>(v_src);
  if (mode == MODE_TAIL) {
    // the same shared-memory carve-out as the attention kernel that may
    // follow as a programmatic dependent, so that its CTAs can land on SMs
    // that still run this kernel's (the other writes keep the default: the
    // frame insert ran 14% slower with it)
    static std::atomic<int> done[64];
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64 && !done[dev].load(std::memory_order_relaxed)) {
      cudaFuncSetAttribute(write_rows_kernel<128, true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
      cudaFuncSetAttribute(write_rows_kernel<64, true>, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
      done[dev].store(1, std::memory_order_relaxed);
    }
  }
  auto launch = [&](auto kernel) {
    kernel<<<(unsigned)blocks, THREADS, 0, st>>>(g, kk, vv, ks, vs, n_group, n_tok, mode, row0, head, sync, tail_len,
                                                 status, acc);
  };
  if (g.d == 128)
    mode == MODE_TAIL ? launch(write_rows_kernel<128, true>) : launch(write_rows_kernel<128, false>);
  else
    mode == MODE_TAIL ? launch(write_rows_kernel<64, true>) : launch(write_rows_kernel<64, false>);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Rotary table: tab[p][i] = (cos, sin)(p * theta^(-2i/d)), angles in fp64.

__global__ void rope_table_kernel(float2* __restrict__ tab, int n_pos, int half, int d,
                                  double theta) {
  const long long n = (long long)n_pos * half;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(e / half), i = (int)(e - (long long)p * half);
    const double inv_freq = pow(theta, -2.0 * i / d);
    double s, c;
    sincos((double)p * inv_freq, &s, &c);
    tab[e] = make_float2((float)c, (float)s);
  }
}

cudaError_t launch_rope_table(float* tab, int n_pos, int d, double theta, cudaStream_t st) {
  const long long n = (long long)n_pos * (d / 2);
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  rope_table_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(reinterpret_cast<float2*>(tab), n_pos,
                                                             d / 2, d, theta);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Multi-section rotary table: row n = the angles of the token at logical
// index n.  A camera token tau of a frame whose first token is at b has the
// position triple (b, b + tau / W, b + tau % W), every other token (n, n, n);
// frequency i turns by the component its mask bits name.

__global__ void mrope_table_kernel(float2* __restrict__ tab, int n_pos, int half, int d, double theta,
                                   MRopeGeom m) {
  const long long n_all = (long long)n_pos * half;
  const long long vis_end = (long long)m.P + (long long)m.V * m.F * m.T;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n_all;
       e += (long long)gridDim.x * blockDim.x) {
    const int n = (int)(e / half), i = (int)(e - (long long)n * half);
    long long pt = n, ph = n, pw = n;
    if (n >= m.P && n < vis_end) {
      const int tau = (n - m.P) % m.T;
      const long long b = n - tau;
      pt = b;
      ph = b + tau / m.W;
      pw = b + tau % m.W;
    }
    const long long comp = ((m.h_mask >> i) & 1ull) ? ph : (((m.w_mask >> i) & 1ull) ? pw : pt);
    const double inv_freq = pow(theta, -2.0 * i / d);
    double s, c;
    sincos((double)comp * inv_freq, &s, &c);
    tab[e] = make_float2((float)c, (float)s);
  }
}

cudaError_t launch_mrope_table(float* tab, int n_pos, int d, double theta, const MRopeGeom& m, cudaStream_t st) {
  const long long n = (long long)n_pos * (d / 2);
  const int blocks = (int)((n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096);
  mrope_table_kernel<<<blocks > 0 ? blocks : 1, 256, 0, st>>>(reinterpret_cast<float2*>(tab), n_pos, d / 2, d,
                                                              theta, m);
  return cudaGetLastError();
}

}  // namespace skv
