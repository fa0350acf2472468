"""Oracle for streaming view-major KV-cache attention -- TEST INFRASTRUCTURE.

Only the tests, the package's smoke check and the benchmark's CPU-baseline
leg may import this module.  The product path never calls it; it shares no
code, table or helper with the CUDA library.

It is a plain, slow, fp64 NumPy restatement of what the FlashDrive pages
describe for one attention layer with given K/V:

* [FD-blog] = "FlashDrive: Flash Vision-Language-Action Inference for Autonomous
  Driving", blog walkthrough (jjl357.github.io);
* [FD-summary] = the same title, paper summary page (m.montaan.com);
* [VFlash] = "VFlash: Enabling System-1 VLMs for Physical AI".

For one layer whose cached K/V are given, streaming attention is exactly
causal attention over the full logical window, kept for the new rows; the
approximation the pages discuss ([FD-blog] 3.4) only appears across the
layers of a model, because cached K/V were produced under an older context.
So every function here computes the plain definition by full recompute:
logical window -> positions -> RoPE on every key and query -> dense mask ->
fp64 softmax -> P V.

bf16 tensors are passed in as uint16 bit patterns and widened exactly to fp64.

Parity status: every function below is pinned by the CPU tests (closed forms,
invariants, brute force, a library SDPA and the pages' worked examples); none
is "parity unpinned".
"""
from __future__ import annotations

import collections

import numpy as np


# ---------------------------------------------------------------------------
# number formats

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# rotary position embedding ([FD-blog] 3.3 "RoPE Position Shift"; the page's
# formula was lost in extraction -- this is the rotate-half form with pairs
# (i, i + d/2) and frequency theta^(-2i/d), angles in fp64)

def rope_rotate(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """Rotate rows of x (shape [..., n, d], fp64) by R(pos[n]).

    For i < d/2 the pair (x_i, x_{i+d/2}) turns by angle pos * theta^(-2i/d):
    y_i = x_i cos - x_{i+d/2} sin,  y_{i+d/2} = x_{i+d/2} cos + x_i sin.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    inv_freq = float(theta) ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ---------------------------------------------------------------------------
# multi-section rotary: a stated reading.  [FD-news] names a Qwen3-VL
# backbone, whose vision tokens carry (temporal, height, width) positions,
# and [FD-blog] 3.3 lost the rotary formula, so this form is not printed on
# the pages.  Reading: a token has a position triple (t, h, w).  Tokens that
# are not camera tokens (prefix, tail, blocks) have t = h = w = their logical
# index n, so they rotate exactly as in rope_rotate.  The T tokens of a frame
# form rows of W tokens in raster order; token tau of a frame whose first
# token sits at logical index b has t = b, h = b + (tau // W), w = b + (tau %
# W).  Frequency i (of the d/2) turns by the component sec[i] (0 = t, 1 = h,
# 2 = w) times theta^(-2i/d).  Positions still shift as frames age, because b
# is a logical index.

def interleaved_sections(d: int, n_h: int, n_w: int) -> np.ndarray:
    """Frequency -> component map: the d/2 frequencies are dealt to t, h, w
    in turn (frequency i gets component i mod 3) while h and w still have
    frequencies left of their shares n_h and n_w; every other frequency
    belongs to t."""
    sec = np.zeros(d // 2, dtype=np.int64)
    for i in range(d // 2):
        c, k = i % 3, i // 3
        if (c == 1 and k < n_h) or (c == 2 and k < n_w):
            sec[i] = c
    return sec


class MRope:
    """The multi-section reading for one window geometry: P prefix tokens,
    V views of F frames of T tokens in rows of W, and the frequency map sec."""

    def __init__(self, P, V, F, T, W, sec):
        assert T % W == 0
        self.P, self.V, self.F, self.T, self.W = P, V, F, T, W
        self.sec = np.asarray(sec, dtype=np.int64)

    def triples(self, idx) -> np.ndarray:
        """Position triples [n][3] (t, h, w) of the tokens at logical
        indices idx."""
        out = []
        for n in np.asarray(idx, dtype=np.int64).reshape(-1):
            n = int(n)
            if self.P <= n < self.P + self.V * self.F * self.T:
                tau = (n - self.P) % self.T
                b = n - tau
                out.append((b, b + tau // self.W, b + tau % self.W))
            else:
                out.append((n, n, n))
        return np.array(out, dtype=np.int64).reshape(-1, 3)


def rope_rotate_sections(x: np.ndarray, triples: np.ndarray, theta: float, sec: np.ndarray) -> np.ndarray:
    """Rotate rows of x ([..., n, d], fp64) by position triples [n][3]: the
    pair (x_i, x_{i+d/2}) turns by triples[n, sec[i]] * theta^(-2i/d), in the
    rotate-half form of rope_rotate."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    i = np.arange(d // 2, dtype=np.float64)
    freq = np.power(float(theta), -2.0 * i / d)                     # theta^(-2i/d)
    comp = np.asarray(triples, dtype=np.float64)[:, np.asarray(sec, dtype=np.int64)]   # [n][d/2]
    ang = comp * freq[None, :]
    cos, sin = np.cos(ang), np.sin(ang)
    lo, hi = x[..., : d // 2], x[..., d // 2:]
    return np.concatenate([lo * cos - hi * sin, hi * cos + lo * sin], axis=-1)


def _rotate(x, pos, theta, mrope):
    """rope_rotate at logical positions, or the multi-section rotation of
    the tokens at those logical indices when a reading is given."""
    if mrope is None:
        return rope_rotate(x, pos, theta)
    return rope_rotate_sections(x, mrope.triples(pos), theta, mrope.sec)


# ---------------------------------------------------------------------------
# the logical sliding window ([FD-blog] 3.1 and 3.2; [FD-summary] "Streaming
# Inference")

class StreamWindow:
    """Logical state of one cache: system prefix, V views of up to F frames
    each (a deque per view, oldest first) and the reasoning-token tail.

    The logical token order is view-major: the prefix, then view 0's frames
    oldest to newest, then view 1's, ..., then the tail ([FD-blog] 3.2).
    A token's position is its logical index in that order (1-D positions).
    All K/V are kept pre-RoPE, as bf16 bits [tokens][Hkv][d].
    """

    def __init__(self, P, V, F, T, Hkv, d, prefix_k, prefix_v):
        self.P, self.V, self.F, self.T, self.Hkv, self.d = P, V, F, T, Hkv, d
        self.prefix_k = np.asarray(prefix_k, dtype=np.uint16).reshape(P, Hkv, d)
        self.prefix_v = np.asarray(prefix_v, dtype=np.uint16).reshape(P, Hkv, d)
        self.views = [collections.deque() for _ in range(V)]
        self.tail_k = np.zeros((0, Hkv, d), np.uint16)
        self.tail_v = np.zeros((0, Hkv, d), np.uint16)
        self.n_inserts = 0

    def insert(self, k_frame, v_frame):
        """One streaming step for every view: evict the view's oldest frame
        once the window is full, then append the new frame as the newest
        ([FD-blog] 3.1: evict oldest, move the rest forward, only the newest
        frame is new).  k_frame/v_frame: [V][T][Hkv][d] bits."""
        k_frame = np.asarray(k_frame, dtype=np.uint16).reshape(self.V, self.T, self.Hkv, self.d)
        v_frame = np.asarray(v_frame, dtype=np.uint16).reshape(self.V, self.T, self.Hkv, self.d)
        for v in range(self.V):
            dq = self.views[v]
            if len(dq) == self.F:
                dq.popleft()
            dq.append((k_frame[v].copy(), v_frame[v].copy()))
        self.n_inserts += 1

    @property
    def full(self) -> bool:
        return all(len(dq) == self.F for dq in self.views)

    def set_tail(self, k, v):
        self.tail_k = np.asarray(k, dtype=np.uint16).reshape(-1, self.Hkv, self.d).copy()
        self.tail_v = np.asarray(v, dtype=np.uint16).reshape(-1, self.Hkv, self.d).copy()

    @property
    def n_visual(self) -> int:
        return self.P + self.V * self.F * self.T

    def logical_kv(self, with_tail: bool = True):
        """K and V bits in logical order, shape [N][Hkv][d]."""
        assert self.full, "attention is defined once the window is full"
        ks, vs = [self.prefix_k], [self.prefix_v]
        for dq in self.views:
            for fk, fv in dq:
                ks.append(fk)
                vs.append(fv)
        if with_tail:
            ks.append(self.tail_k)
            vs.append(self.tail_v)
        return np.concatenate(ks, axis=0), np.concatenate(vs, axis=0)

    def new_frame_index(self, v: int, t: int) -> int:
        """Logical index (= position) of token t of view v's newest frame."""
        return self.P + v * self.F * self.T + (self.F - 1) * self.T + t

    def ring_expected(self):
        """Physical ring contents a head-pointer ring must hold.

        The ring keeps the F frames of a view in F slots and never moves
        data: after n inserts the head (the slot of the oldest frame) is
        n mod F and logical frame f lives in slot (head + f) mod F -- the
        page's "move the rest forward" becomes a change of head.
        Returns (head [V], k [V][F][T][Hkv][d], v [V][F][T][Hkv][d]).
        """
        assert self.full
        head = self.n_inserts % self.F
        k = np.zeros((self.V, self.F, self.T, self.Hkv, self.d), np.uint16)
        v = np.zeros_like(k)
        for vi, dq in enumerate(self.views):
            for f, (fk, fv) in enumerate(dq):
                s = (head + f) % self.F
                k[vi, s] = fk
                v[vi, s] = fv
        return np.full(self.V, head, np.int32), k, v


# ---------------------------------------------------------------------------
# attention ([FD-blog] 3.2: standard attention with mask M; a query sees a key
# iff the key's logical index is at most the query's)

def attention_rows(q_bits, q_pos, k_bits, v_bits, k_pos, theta, sm_scale, mrope=None):
    """Masked softmax attention of selected query rows over a key sequence.

    q_bits [n][Hq][d] pre-RoPE queries at logical positions q_pos [n];
    k_bits, v_bits [N][Hkv][d] pre-RoPE keys / values at positions k_pos [N].
    Query head h uses key/value head floor(h / (Hq/Hkv)).
    Score = <R(q_pos) q, R(k_pos) k> * sm_scale, kept iff k_pos <= q_pos.
    With mrope (an MRope reading) the rotation is the multi-section one of
    the tokens at those logical indices; the mask stays on logical indices.
    Returns O [n][Hq][d] (fp64) and the natural-log LSE [n][Hq] of the
    scaled scores.
    """
    q = bf16_to_f64(q_bits)
    k = bf16_to_f64(k_bits)
    v = bf16_to_f64(v_bits)
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    q_pos = np.asarray(q_pos, dtype=np.int64)
    k_pos = np.asarray(k_pos, dtype=np.int64)
    visible = k_pos[None, :] <= q_pos[:, None]                     # [n][N]
    kr = _rotate(np.transpose(k, (1, 0, 2)), k_pos, theta, mrope)  # [Hkv][N][d]
    vt = np.transpose(v, (1, 0, 2))                                # [Hkv][N][d]
    qr = _rotate(np.transpose(q, (1, 0, 2)), q_pos, theta, mrope)  # [Hq][n][d]
    out = np.zeros((Hq, n, d))
    lse = np.zeros((Hq, n))
    for h in range(Hq):
        kh = h // G
        s = (qr[h] @ kr[kh].T) * sm_scale
        s = np.where(visible, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        out[h] = (p / l) @ vt[kh]
        lse[h] = (m + np.log(l))[:, 0]
    return np.transpose(out, (1, 0, 2)), lse.T


# ---------------------------------------------------------------------------
# the three steps of the path

def stream_prefill(win: StreamWindow, q_new, theta, sm_scale, rows=None, mrope=None):
    """New-frame queries against the full window ([FD-blog] 3.2, 3.3).

    q_new [V*T][Hq][d] pre-RoPE bits, token j = (view j // T, token j % T) of
    that view's newest frame.  Only these tokens are queries; keys are the
    prefix and every view's frames (the tail lies after all of them and is
    never visible).  `rows` optionally restricts the computation to a subset
    of query tokens (each row is independent).  Returns (O, LSE) for the
    selected rows.
    """
    q_new = np.asarray(q_new, dtype=np.uint16)
    nq = win.V * win.T
    rows = np.arange(nq) if rows is None else np.asarray(rows)
    q_pos = np.array([win.new_frame_index(int(j) // win.T, int(j) % win.T) for j in rows])
    k_bits, v_bits = win.logical_kv(with_tail=False)
    k_pos = np.arange(k_bits.shape[0])
    return attention_rows(q_new[rows], q_pos, k_bits, v_bits, k_pos, theta, sm_scale, mrope)


def _block_after_tail(win: StreamWindow, blk_q, blk_k, blk_v, theta, sm_scale, mrope=None):
    """Tokens appended after the window's tail, as queries: token j sits at
    logical index n_visual + tail_len + j and sees the prefix, all frames, the
    whole tail and block tokens 0..j.  blk_q [n][Hq][d], blk_k/blk_v
    [n][Hkv][d].  Returns (O [n][Hq][d], LSE [n][Hq])."""
    k_bits, v_bits = win.logical_kv(with_tail=True)
    base = k_bits.shape[0]
    blk = np.asarray(blk_q).shape[0]
    k_all = np.concatenate([k_bits, np.asarray(blk_k, np.uint16)], axis=0)
    v_all = np.concatenate([v_bits, np.asarray(blk_v, np.uint16)], axis=0)
    k_pos = np.arange(k_all.shape[0])
    q_pos = base + np.arange(blk)
    return attention_rows(np.asarray(blk_q, np.uint16), q_pos, k_all, v_all, k_pos,
                          theta, sm_scale, mrope)


def stream_verify(win: StreamWindow, blk_q, blk_k, blk_v, theta, sm_scale, mrope=None):
    """Speculative-verify block ([FD-blog] 4.2 steps 1-2; [VFlash] "03 ·
    Generalist decoding": the target checks a whole drafted block in one
    pass).

    The block's tokens follow the tail: block token j sits at logical index
    n_visual + tail_len + j and sees the prefix, all frames, the whole tail
    and block tokens 0..j.  blk_q [blk][Hq][d], blk_k/blk_v [blk][Hkv][d].
    Returns (O [blk][Hq][d], LSE [blk][Hq]).
    """
    return _block_after_tail(win, blk_q, blk_k, blk_v, theta, sm_scale, mrope)


def stream_prefill_tail(win: StreamWindow, tail_q, tail_k, tail_v, theta, sm_scale, mrope=None):
    """Trajectory / text tokens after the views as queries ([FD-blog] 3.2
    "View-Major Ordering": the trailing trajectory and text tokens see every
    view and are causal among themselves; with the newest frames they are the
    only new queries of a step).

    The n tokens follow the window's current tail: token j sits at logical
    index n_visual + tail_len + j and sees everything before it plus tokens
    0..j of its own span -- the same rows a verify block of n tokens computes.
    tail_q [n][Hq][d], tail_k/tail_v [n][Hkv][d].  Returns (O, LSE).  The
    caller appends tail_k/tail_v to the window's tail afterwards.
    """
    return _block_after_tail(win, tail_q, tail_k, tail_v, theta, sm_scale, mrope)


def stream_window(win: StreamWindow, q_win, theta, sm_scale, rows=None, mrope=None):
    """Every token of the window as a query: the first window of a stream,
    which only fills the cache ([FD-blog] 11 "Implementation Map": the first
    streaming window returns no trajectory), or a full re-encode.

    q_win [N][Hq][d] pre-RoPE bits in logical order -- the prefix, then view
    0's frames oldest to newest, then view 1's, ... -- N = P + V*F*T.  Token i
    sits at position i and sees keys 0..i ([FD-blog] 3.2: the prefix is seen
    by every frame, a view sees the earlier views, its own older frames and
    its own frame causally).  The tail follows the window and is not
    visible.  `rows` optionally restricts the computation to a subset of
    tokens.  Returns (O, LSE) for the selected rows.
    """
    q_win = np.asarray(q_win, dtype=np.uint16)
    k_bits, v_bits = win.logical_kv(with_tail=False)
    n = k_bits.shape[0]
    rows = np.arange(n) if rows is None else np.asarray(rows)
    return attention_rows(q_win[rows], rows, k_bits, v_bits, np.arange(n), theta, sm_scale, mrope)


def accept_length(target_ids, draft_ids):
    """Greedy longest-prefix acceptance ([FD-blog] 4.2 steps 3-4; [VFlash]
    "keeps the longest matching prefix plus its own next token").

    Block slot 0 holds the last accepted token; slots 1..blk-1 hold drafts.
    target_ids[i] is the target's choice for the token after block slot i.
    Draft i is accepted while draft[i] == target[i-1] for every earlier i.
    Returns (accept_len, next_token): the number of accepted drafts and the
    target's token at the first rejected (or the bonus) position.
    """
    target = [int(x) for x in target_ids]
    draft = [int(x) for x in draft_ids]
    k = 0
    for i in range(1, len(draft)):
        if draft[i] != target[i - 1]:
            break
        k += 1
    return k, target[k]
