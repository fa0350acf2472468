// Host-side launchers of the libskv kernels (internal to the library).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace skv {

// mode 0: rows at row0; 1: frame insert (ring slot, head advance); 2: verify
// block into the tail, with the accept length when target/draft are given.
cudaError_t launch_write_rows(const Geom& g, void* k, void* vt, const void* k_src,
                              const void* v_src, int n_group, int n_tok, int mode, int row0,
                              int32_t* head, int32_t* sync, const int32_t* tail_len,
                              int32_t* status, cudaStream_t st, const int32_t* target = nullptr,
                              const int32_t* draft = nullptr, int32_t* accept_len = nullptr,
                              int32_t* next_token = nullptr);

cudaError_t launch_rope_table(float* tab, int n_pos, int d, double theta, cudaStream_t st);

// Geometry and frequency map of the multi-section rotary table.
struct MRopeGeom {
  int P, V, F, T, W;
  uint64_t h_mask, w_mask;   // frequency i turns by h (bit i of h_mask), w (of w_mask), else t
};
cudaError_t launch_mrope_table(float* tab, int n_pos, int d, double theta, const MRopeGeom& m, cudaStream_t st);

// The query tokens of one prefill launch, the same for every cache; a
// cache's rows of q / out / lse hold NQ tokens.
struct PrefillQuery {
  int nf;                   // frames per view that are queries: 0, 1 (the newest) or F (all)
  bool prefix;              // the prefix tokens are queries
  int n_tail;               // tail tokens that are queries (they follow tail_len[c] tail rows)
  const int32_t* tail_len;  // [C] on the device; needed when n_tail > 0
  int NQ;                   // query tokens per cache
  int q_view0;              // token of view 0's first queried frame; view v, queried frame i at
                            // q_view0 + (v * nf + i) * T
  int q_tail0;              // token of the first tail query; prefix token j at j
};

// With k_new / v_new ([C][V][T][Hkv][d]) and sync given, the launch also does
// the frame insert (new-frame queries only; prefill_insert_fusable geometry):
// heads still name the oldest frames when it starts and are advanced by it.
cudaError_t launch_prefill_tc(const Geom& g, int Hq, const PrefillQuery& qs, const void* q, void* out, float* lse,
                              const void* k, const void* vt, const float* rope, int32_t* head,
                              float sm_scale, int32_t* status, uint64_t wait_ns, cudaStream_t st,
                              const void* k_new = nullptr, const void* v_new = nullptr, int32_t* sync = nullptr);
bool prefill_insert_fusable(const Geom& g);

cudaError_t launch_verify_tc(const Geom& g, int Hq, int blk, const int32_t* tail_len, const void* q, void* out,
                             const void* k, const void* vt, const float* rope, const int32_t* head,
                             void* ws, size_t ws_bytes, float sm_scale, int32_t* status, uint64_t wait_ns,
                             cudaStream_t st);
size_t verify_ws_bytes(const Geom& g, int Hq, int blk);

int check_insert_args(const skv_cache* cache, const void* k_new, const void* v_new);
int record_cuda_error(cudaError_t e);

}  // namespace skv
