/*
 * skv.h -- C ABI of libskv: streaming view-major KV-cache attention on GB300
 * (sm_103a).
 *
 * The operation (FlashDrive, Flash Vision-Language-Action Inference for
 * Autonomous Driving; blog walkthrough section 3 "Encode & Prefill: Streaming
 * Inference" and paper summary "Streaming Inference"): a VLA model looks at a
 * sliding window of F frames from each of V camera views.  Every step the
 * window advances by one frame per view, so only the newest frame is new.
 * The cache keeps the keys WITHOUT rotary embedding (pre-RoPE) and rotates
 * each key at its current logical position inside the attention kernel,
 * because that position moves as older frames are evicted (blog section 3.3
 * "RoPE Position Shift").  Tokens are ordered view-major -- the system prefix,
 * then view 0's frames oldest to newest, view 1's, ..., then the reasoning
 * tail (blog section 3.2 "View-Major Ordering") -- and a query sees a key iff
 * the key's logical index is at most its own.
 *
 * Conventions shared by every call:
 *  - All pointers named "device" are CUDA device pointers owned by the
 *    caller, in memory of the device that is current when the call is made
 *    (the kernels launch there; the library does not check where a pointer
 *    lives).  The library never allocates, never frees and never keeps a
 *    pointer after a call returns.
 *  - bf16 tensors are raw 16-bit brain-float arrays, C-contiguous, in the
 *    layout stated beside them; every device pointer must be 16-byte
 *    aligned.
 *  - `stream` is a cudaStream_t passed as void*.  Calls only enqueue work on
 *    it, never synchronise and never copy to or from the host, so they may
 *    be captured into a CUDA graph.
 *  - The attention calls rotate Q and K in fp32 and hand the tensor cores
 *    fp16 operands (11 significant bits, 3 more than bf16).  fp16's largest
 *    finite value is 65504: a rotated component beyond it is clamped to
 *    +-65504, with no status bit.  The rotation keeps the length of every
 *    (x_i, x_{i+d/2}) pair, so Q and K whose components all lie within
 *    +-46000 (65504 / sqrt 2) never reach the clamp.  Components under
 *    2^-14 in magnitude are fp16 subnormals and keep fewer bits.  The softmax
 *    scale is applied in fp32 after the product, so large K with a small
 *    sm_scale stays exact up to that rounding.
 *  - A call returns SKV_OK after enqueueing, or a negative SKV_ERR_* code
 *    and enqueues nothing.  Errors found on the device while the kernels run
 *    (a bounded wait that gave up, a ring head out of range, a tail that
 *    would overflow) are OR-ed into the int32 device word cache->status as
 *    SKV_DEV_* bits; the caller reads it when it wants to.
 */
#ifndef SKV_H_
#define SKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SKV_VERSION 1

/* host-side return codes */
#define SKV_OK 0
#define SKV_ERR_INVALID (-1)     /* null/misaligned pointer, bad shape or argument */
#define SKV_ERR_UNSUPPORTED (-2) /* no sm_103 device current, or shape outside what the kernels cover */
#define SKV_ERR_CUDA (-3)        /* a CUDA runtime/driver call failed; see skv_last_cuda_error() */
#define SKV_ERR_TOO_LARGE (-4)   /* shape exceeds the fixed scratch of kv_stream_insert_noalloc */

/* device status bits (OR-ed into *cache->status) */
#define SKV_DEV_TIMEOUT 1        /* a bounded wait inside a kernel gave up; outputs are undefined */
#define SKV_DEV_BAD_HEAD 2       /* a ring head was outside [0, F); that cache was skipped */
#define SKV_DEV_TAIL_OVERFLOW 4  /* tail_len + blk > tail_cap in verify; that cache was skipped */
#define SKV_DEV_BAD_TAIL 8       /* tail_len < 0 in verify; that cache was skipped */

/*
 * One set of C independent caches (model layers x batch) of identical
 * geometry.  Per cache c and kv head h there are row_cap key rows:
 *
 *   rows [0, P)                      system prefix, logical index = row
 *   rows [P, P + V*F*T)              the ring: view v, slot s, token t at
 *                                    row P + (v*F + s)*T + t
 *   rows [P + V*F*T, ... + tail_cap) reasoning-token tail, index = row
 *
 * The ring of view v holds its F frames in F slots; head[c][v] is the slot
 * of the oldest frame, so logical frame f (0 = oldest) sits in slot
 * (head + f) mod F and a ring key's logical index is P + v*F*T + f*T + t.
 * Inserting a frame overwrites the oldest slot and advances the head; no
 * data moves.
 *
 * k   device bf16 [C][Hkv][row_cap][d]  pre-RoPE keys, one row per token
 * vt  device bf16 [C][Hkv][d][row_cap]  values, stored transposed (dimension-
 *                                       major) so that both tensor-core
 *                                       products read K-major operands
 * head    device int32 [C][V]   ring heads (0 for an empty cache)
 * sync    device int32 [C][V]   zero-initialised counters used by
 *                               kv_stream_insert; the call leaves them at 0.
 *                               No other call reads them: those accept NULL
 * rope    device fp32 [rope_len][d/2][2]  rotary angles, read as rope_mode says;
 *                               rope_len must cover every logical index
 *                               (P + V*F*T + tail_cap)
 *   rope_mode 0: row p holds (cos, sin) of p*theta^(-2i/d) (filled by
 *                skv_build_rope_table): a token's position is its logical
 *                index, and the kernels step the angles along runs of
 *                consecutive positions (one table read per run);
 *   rope_mode 1: row n holds the angles of the token at logical index n
 *                under any per-token positions (filled, for the
 *                multi-section reading, by skv_build_mrope_table): the
 *                kernels read the row of every key and query.
 * status  device int32 [1]      SKV_DEV_* bits, OR-ed in by the kernels
 *
 * Every row of k and vt must hold finite values (allocate them zeroed):
 * masked keys still pass through the tensor cores with weight 0.
 */
typedef struct skv_cache {
  int32_t n_cache;    /* C */
  int32_t n_view;     /* V >= 1 */
  int32_t n_frame;    /* F >= 1 */
  int32_t frame_len;  /* T >= 1 */
  int32_t prefix_len; /* P >= 0 */
  int32_t tail_cap;   /* rows reserved for reasoning tokens, >= 0 */
  int32_t n_kv_head;  /* Hkv >= 1 */
  int32_t head_dim;   /* d: 64 or 128 */
  int32_t row_cap;    /* >= P + V*F*T + tail_cap, multiple of 8 */
  int32_t rope_len;   /* rows of the rope table */
  void* k;
  void* vt;
  int32_t* head;
  int32_t* sync;
  const float* rope;
  int32_t* status;
  uint64_t wait_ns;   /* limit of every bounded wait in a kernel; 0 = 2 s */
  int32_t rope_mode;  /* 0 or 1, see rope above */
  int32_t reserved;   /* 0 */
} skv_cache;

/* Library version (SKV_VERSION). */
int skv_version(void);

/* Human-readable text for an SKV_* return code or SKV_DEV_* bit set. */
const char* skv_status_string(int code);

/* The cudaError_t of the last call that returned SKV_ERR_CUDA on this host
 * thread (0 if none). */
int skv_last_cuda_error(void);

/* Smallest valid row_cap for a geometry (rounded up to a multiple of 128). */
int32_t skv_row_cap(int32_t P, int32_t V, int32_t F, int32_t T, int32_t tail_cap);

/*
 * Fill the rotary table used by every attention call:
 * tab[p][i] = (cos(p * theta^(-2i/d)), sin(...)) for p < n_pos, i < d/2,
 * angles formed and reduced in fp64 on the device, rounded once to fp32.
 * tab: device fp32 [n_pos][d/2][2].  Pairs (i, i + d/2) of a head vector
 * rotate together (rotate-half form).
 */
int skv_build_rope_table(float* tab, int32_t n_pos, int32_t head_dim, double theta,
                         void* stream);

/*
 * Fill a rotary table for rope_mode 1 with the multi-section reading of the
 * positions (FlashDrive's backbone is a Qwen3-VL model, whose vision tokens
 * carry temporal, height and width positions; the pages print no rotary
 * formula, so this is a stated reading, not the pages' text):
 *  - a token that is not a camera token (prefix, tail, verify block) at
 *    logical index n has the position triple (t, h, w) = (n, n, n);
 *  - the T tokens of a frame form rows of grid_w tokens in raster order;
 *    token tau of a frame whose first token sits at logical index b has
 *    (t, h, w) = (b, b + tau / grid_w, b + tau % grid_w);
 *  - frequency i (i < d/2) turns by the height component when bit i of
 *    h_mask is set, by the width component when bit i of w_mask is set,
 *    else by the temporal one: angle = component * theta^(-2i/d).
 * Row n of tab holds (cos, sin) of those angles for the token at logical
 * index n (n < n_pos); angles in fp64, rounded once to fp32.  The rows of
 * tokens that are not camera tokens equal skv_build_rope_table's.
 * tab: device fp32 [n_pos][d/2][2].  Needs head_dim/2 <= 64, T % grid_w == 0
 * and no bit set in both masks (else SKV_ERR_INVALID).
 */
int skv_build_mrope_table(float* tab, int32_t n_pos, int32_t head_dim, double theta, int32_t P,
                          int32_t V, int32_t F, int32_t T, int32_t grid_w, uint64_t h_mask,
                          uint64_t w_mask, void* stream);

/*
 * Write n_rows token-major K/V rows into rows [row0, row0 + n_rows) of every
 * cache and kv head, as they are (pre-RoPE).  Used to place the system
 * prefix and reasoning-tail tokens; the ring is written by kv_stream_insert.
 * k_src, v_src: device bf16 [C][n_rows][Hkv][d].  Bit-exact copy.
 */
int kv_write_rows(const skv_cache* cache, int32_t row0, int32_t n_rows, const void* k_src,
                  const void* v_src, void* stream);

/*
 * kv_stream_insert -- one streaming step of the window (blog section 3.1:
 * evict each view's oldest frame, keep the rest, add only the newest).
 * For every cache c and view v: s = head[c][v]; the new frame's K/V are
 * written into slot s (evicting the oldest frame); then head[c][v] =
 * (s + 1) mod F.  Prefix, tail and every other slot are untouched.
 * k_new, v_new: device bf16 [C][V][T][Hkv][d], token-major, pre-RoPE.
 * Bit-exact.  The initial fill of an empty cache is F calls; attention is
 * defined once the window is full (the first window only fills the cache).
 * A head outside [0, F) sets SKV_DEV_BAD_HEAD and that (c, v) is skipped.
 */
int kv_stream_insert(const skv_cache* cache, const void* k_new, const void* v_new,
                     void* stream);

/*
 * kv_stream_insert_noalloc -- kv_stream_insert for callers that cannot
 * allocate device memory.  Some callers of this library may not call
 * cudaMalloc at all: an inference runtime that hands its plug-ins only the
 * buffers it planned ahead of time, a real-time control loop that must
 * never block in the allocator, or code running where allocation is
 * forbidden after start-up.  Such a caller cannot provide the scratch
 * counters kv_stream_insert needs in cache->sync.  The pages have no
 * counterpart to this call; it only changes where that scratch lives.
 *
 * Same inputs, outputs and results as kv_stream_insert; cache->sync is
 * ignored and may be NULL.  The per-(cache, view) arrival counters live in
 * one file-scope static device array of SKV_NOALLOC_MAX_CACHE_VIEWS int32
 * (64 KiB), which every GPU that loads libskv holds until the process
 * exits.  n_cache * n_view above that limit returns SKV_ERR_TOO_LARGE and
 * enqueues nothing.
 *
 * The first call on a device looks up the array's device address, with
 * that device current; make that first call before any stream capture.
 * The address is kept for the life of the process: after a
 * cudaDeviceReset of that device it is stale, so do not call this again
 * in a process that reset the device.
 * Every call first clears the counters it uses with an asynchronous memset
 * on `stream`; it calls no cudaMalloc, cudaFree or allocating library
 * routine.  All calls on one device share the one array and it keeps what
 * the last call left, so calls that overlap on that GPU (for instance on
 * two streams) race: serialise them.
 */
#define SKV_NOALLOC_MAX_CACHE_VIEWS 16384
int kv_stream_insert_noalloc(const skv_cache* cache, const void* k_new, const void* v_new,
                             void* stream);

/*
 * stream_attn_prefill -- attention of the newest frame's tokens over the
 * window (blog sections 3.2-3.3).  Call it after kv_stream_insert, so the
 * newest frame is in the cache.  Query token j = (view j / T, token j mod T
 * of that view's newest frame) sits at logical index
 * P + v*F*T + (F-1)*T + t and sees every key whose logical index is at most
 * its own: the prefix, all earlier views, its own view's older frames and
 * its own frame causally; never later views nor the tail.  Queries and keys
 * are rotated (rotate-half RoPE from cache->rope) at their logical
 * positions inside the kernel; query head h reads kv head h / (Hq/Hkv).
 *
 * q_new: device bf16 [C][V*T][Hq][d], pre-RoPE.
 * out:   device bf16 [C][V*T][Hq][d]: softmax(sm_scale * q.k) v, fp32
 *        accumulation, rounded to nearest even once.
 * lse:   device fp32 [C][Hq][V*T] natural-log sum of exp of the scaled
 *        scores, or NULL.
 * Needs Hq % Hkv == 0 and 128 % (Hq/Hkv) == 0.  The kernel covers V <= 64,
 * row_cap <= 131072 and C * (query tokens) * Hq < 2^31; outside that the
 * call returns SKV_ERR_UNSUPPORTED and enqueues nothing (the same limits
 * hold for stream_attn_prefill_tail and stream_attn_window).
 */
int stream_attn_prefill(const skv_cache* cache, int32_t n_q_head, const void* q_new, void* out,
                        float* lse, float sm_scale, void* stream);

/*
 * stream_attn_prefill_insert -- kv_stream_insert of the step's new frames
 * followed by stream_attn_prefill of their queries, as one call (blog
 * section 3.1: each step evicts the oldest frame and prefills only the
 * newest; the insert is folded into the prefill so that the new frames are
 * read from the input once, by the attention kernel itself).  Same inputs,
 * results and status bits as the two calls: the ring holds the new frames
 * bit for bit and the heads are advanced afterwards.
 *
 * k_new, v_new: device bf16 [C][V][T][Hkv][d] (as kv_stream_insert);
 * q_new, out, lse as stream_attn_prefill.  cache->sync is needed (zeroed
 * counters, left at 0).
 *
 * With head_dim 128 and P and T multiples of 64 it is one kernel launch: the
 * new frames' K/V tiles come straight from k_new / v_new, the CTA pair of
 * each view's last query block writes that frame into the ring slot of the
 * oldest frame, and the last CTA of a cache to start advances its heads.
 * Otherwise the call enqueues the insert and then the prefill.
 */
int stream_attn_prefill_insert(const skv_cache* cache, int32_t n_q_head, const void* k_new,
                               const void* v_new, const void* q_new, void* out, float* lse,
                               float sm_scale, void* stream);

/*
 * stream_attn_prefill_tail -- the trajectory / text tokens that follow the
 * views, as queries (blog section 3.2: they see every view and are causal
 * among themselves; with the newest frames they are a step's only new
 * queries).  Runs on the same tensor-core kernel as stream_attn_prefill.
 *
 * Tail token j (j < n_tok) of cache c sits at logical index
 * P + V*F*T + tail_len[c] + j.  The call
 *  1. writes the tokens' pre-RoPE K/V into tail rows tail_len[c] + j;
 *  2. attends each token over the prefix, all frames, the tail
 *     [0, tail_len[c]) and tokens 0..j of its own span.
 * The caller then advances tail_len[c] by n_tok.
 *
 * tail_len: device int32 [C], tokens already in the tail (0 at the start of
 *           a step).
 * q_tail:   device bf16 [C][n_tok][Hq][d]; k_tail, v_tail: [C][n_tok][Hkv][d].
 * out:      device bf16 [C][n_tok][Hq][d].
 * lse:      device fp32 [C][Hq][n_tok] or NULL.
 * Needs 1 <= n_tok <= tail_cap, Hq % Hkv == 0 and 128 % (Hq/Hkv) == 0, and
 * the shape limits of stream_attn_prefill (checked before anything is
 * written).  tail_len[c] < 0 sets SKV_DEV_BAD_TAIL, tail_len[c] + n_tok > tail_cap sets
 * SKV_DEV_TAIL_OVERFLOW; that cache is then neither written nor attended.
 */
int stream_attn_prefill_tail(const skv_cache* cache, int32_t n_q_head, int32_t n_tok,
                             const int32_t* tail_len, const void* q_tail, const void* k_tail,
                             const void* v_tail, void* out, float* lse, float sm_scale,
                             void* stream);

/*
 * stream_attn_window -- every token of the window as a query: the first
 * window of a stream, which only fills the cache (blog section 11), or a
 * full re-encode.  Call it once the window is full (F inserts).
 *
 * Window token i (i < N = P + V*F*T) is the token at logical index i: the
 * prefix, then view 0's frames oldest to newest, then view 1's, ...  It sees
 * every key whose logical index is at most i (never the tail); queries and
 * keys are rotated at their logical positions in the kernel.  The ring may
 * have any head: frame f of view v is read from slot (head + f) mod F.
 *
 * q_win: device bf16 [C][N][Hq][d], pre-RoPE, in logical order.
 * out:   device bf16 [C][N][Hq][d].
 * lse:   device fp32 [C][Hq][N] or NULL.
 * Needs Hq % Hkv == 0 and 128 % (Hq/Hkv) == 0, and the shape limits of
 * stream_attn_prefill.
 */
int stream_attn_window(const skv_cache* cache, int32_t n_q_head, const void* q_win, void* out,
                       float* lse, float sm_scale, void* stream);

/* Bytes of device workspace stream_attn_verify needs for this geometry. */
size_t skv_verify_workspace_bytes(const skv_cache* cache, int32_t n_q_head, int32_t blk);

/*
 * stream_attn_verify -- one speculative-verify pass (blog section 4.2,
 * steps 1-4; VFlash "03 · Generalist decoding": the target checks a drafted
 * block in one pass and keeps the longest matching prefix plus its own next
 * token).
 *
 * Block token j (j < blk; token 0 = the last accepted token, 1.. = drafts)
 * of cache c sits at logical index P + V*F*T + tail_len[c] + j.  The call
 *  1. writes the block's pre-RoPE K/V into tail rows tail_len[c] + j;
 *  2. attends each block query over the prefix, all frames, the tail
 *     [0, tail_len[c]) and block tokens 0..j (causal within the block);
 *  3. if target_ids and draft_ids are both non-NULL, sets accept_len[c] =
 *     the largest k <= blk-1 with draft[c][i] == target[c][i-1] for all
 *     1 <= i <= k, and next_token[c] = target[c][accept_len[c]].
 * The caller then advances tail_len[c] by accept_len[c] + 1.
 *
 * tail_len: device int32 [C], tokens already in the tail.
 * q_blk:    device bf16 [C][blk][Hq][d]; k_blk, v_blk: [C][blk][Hkv][d].
 * out:      device bf16 [C][blk][Hq][d].
 * target_ids, draft_ids: device int32 [C][blk] or NULL.
 * accept_len, next_token: device int32 [C] (unused when ids are NULL).
 * ws: device workspace of ws_bytes >= skv_verify_workspace_bytes(); it must
 *     be zero-filled before its first use, the call leaves it ready for the
 *     next one (re-zero it after a call that set a device status bit).
 *     Calls that may run at the same time (other streams) need workspaces
 *     of their own: the arrival counters in it are per call.
 * Small batches spread each (cache, kv head)'s keys over many CTAs; when
 * four or more share one and the grid fits on the GPU at once, the call is
 * a cooperative launch whose CTAs meet once at a grid barrier (its wait is
 * bounded by cache->wait_ns and ends in SKV_DEV_TIMEOUT); such a launch
 * starts only when the whole grid can be resident.
 * Needs 1 <= blk <= tail_cap, V <= 64 and Hq/Hkv <= 64 (else
 * SKV_ERR_UNSUPPORTED).  A block of up to 128 rows per kv head
 * (blk * Hq/Hkv) streams the keys once; a larger one is taken 128 rows at a
 * time, which needs Hq/Hkv to divide 128.  tail_len + blk > tail_cap sets
 * SKV_DEV_TAIL_OVERFLOW and skips that cache.
 */
int stream_attn_verify(const skv_cache* cache, int32_t n_q_head, int32_t blk,
                       const int32_t* tail_len, const void* q_blk, const void* k_blk,
                       const void* v_blk, void* out, const int32_t* target_ids,
                       const int32_t* draft_ids, int32_t* accept_len, int32_t* next_token,
                       void* ws, size_t ws_bytes, float sm_scale, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SKV_H_ */
