"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs.  Ring heads, cache bytes and accept lengths are compared
bit for bit; attention outputs within max-abs 1e-2 and mean-abs 1e-3."""
import numpy as np
import pytest
import torch

from oracle import skv_oracle as O
from streaming_kv_cache_gb300 import skv, synth

from gpu_harness import LSE_TOL, Pair, assert_close, assert_lse, bf16_dev_to_f64, from_dev, to_dev

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_kv_cache_gb300 import build
    build.build()


def _prefill_check(pair, step_tag, rows=None, watch=None, lse_tol=LSE_TOL, rel=0.0, max_abs=1e-2):
    w = pair.w
    q = synth.frame_q(w, pair.n_inserts - 1, pair.tag + step_tag)
    out, lse = skv.stream_attn_prefill(pair.cache, to_dev(q), w.sm_scale, lse=True)
    got = bf16_dev_to_f64(out)
    got_lse = lse.cpu().numpy()
    for c in (pair.watch if watch is None else watch):
        want, wl = O.stream_prefill(pair.win[c], q[c], w.theta, w.sm_scale, rows=rows)
        sel = slice(None) if rows is None else rows
        assert_close(got[c][sel], want, "%s cache %d" % (w.name, c), rel=rel, max_abs=max_abs)
        assert_lse(got_lse[c][:, sel].T, wl, lse_tol, "%s cache %d" % (w.name, c))
    assert pair.cache.device_status() == 0
    return got


def test_insert_and_prefill_tiny():
    pair = Pair(W["tiny"], "t0")
    pair.fill()
    pair.check_ring()
    for s in range(W["tiny"].steps):
        pair.insert()
        pair.check_ring()
        _prefill_check(pair, "s%d" % s)


def test_prefill_alpamayo_step():
    pair = Pair(W["alpamayo_step"], "a0")
    pair.fill()
    pair.insert()
    pair.check_ring()
    _prefill_check(pair, "x")


def test_alpamayo_20_streaming_steps():
    """Ring wraps 5 times; positions shift each step; every step's cache and
    outputs against a full-window recompute."""
    w = W["alpamayo_20steps"]
    pair = Pair(w, "s20")
    pair.fill()
    for s in range(w.steps):
        pair.insert()
        pair.check_ring()
        _prefill_check(pair, "s%d" % s)


def test_prefill_scaleup_36_layers():
    """The scale-up workload in the launch the bench times (36 layer caches
    in one call): every query row and head of the first and the last layer
    cache element by element, and sampled rows (tile edges, frame edges,
    random rows) of every one of the 36."""
    w = W["scaleup_36L"]
    pair = Pair(w, "big")
    pair.fill()
    pair.insert()
    pair.check_ring()
    q = synth.frame_q(w, pair.n_inserts - 1, pair.tag + "x")
    out, lse = skv.stream_attn_prefill(pair.cache, to_dev(q), w.sm_scale, lse=True)
    got = bf16_dev_to_f64(out)
    got_lse = lse.cpu().numpy()
    assert pair.cache.device_status() == 0
    rng = np.random.default_rng(5)
    sampled = np.array(sorted(set([0, 1, 127, 128, w.T - 1, w.T, 2 * w.T + 7, w.n_new - 1]
                                  + list(rng.integers(0, w.n_new, 8)))))
    for c in range(w.C):
        whole = c in (0, w.C - 1)
        # whole caches in chunks of rows, to bound the oracle's memory
        chunks = np.array_split(np.arange(w.n_new), 6) if whole else [sampled]
        for rows in chunks:
            want, wl = O.stream_prefill(pair.win[c], q[c], w.theta, w.sm_scale, rows=rows)
            assert_close(got[c][rows], want, "scale-up cache %d rows %d..%d" % (c, rows[0], rows[-1]))
            assert_lse(got_lse[c][:, rows].T, wl, LSE_TOL, "scale-up cache %d" % c)


def test_prefill_peaky_queries():
    """Q x 4: sharper softmax, larger logits.  Outputs then reach |o| > 4,
    where rounding to bf16 alone costs up to 2^-8 |o|; that bound is added
    to the absolute one."""
    w = W["alpamayo_step"].with_(q_scale=4.0 / np.sqrt(128), C=2)
    pair = Pair(w, "peak")
    pair.fill()
    pair.insert()
    _prefill_check(pair, "x", rel=2.0 ** -8, lse_tol=4 * LSE_TOL)


def test_prefill_dominant_late_keys():
    """A few keys of the newest frames, 30x larger than the rest, dominate
    the rows that may see them: their tiles come late in the key loop, so
    the running max jumps and O and l are rescaled.  A wrong rescale costs
    O(1); the 30x scores themselves carry 30x the rounding of the fp16
    rotated operands (2^-11 relative), so the max bound is 5e-2 here."""
    w = W["alpamayo_step"].with_(C=1)
    pair = Pair(w, "dom")
    pair.fill()
    k, v = synth.frame_kv(w, pair.n_inserts, pair.tag)
    kf = O.bf16_to_f64(k).astype(np.float32)
    for view, tok in ((1, 30), (2, 5), (3, 170)):
        kf[:, view, tok] *= 30.0
    pair.insert(synth.f32_to_bf16_bits(kf), v)
    _prefill_check(pair, "x", max_abs=5e-2, lse_tol=30 * LSE_TOL)


@pytest.mark.parametrize("half", [0, 1])
def test_prefill_dominant_key_in_either_half_of_a_tile(half):
    """One key of view 1's newest frame, 30x larger than the rest, placed at
    an offset of its 128-key tile in the first (0-63) or the second (64-127)
    half: the running max of every row that sees it jumps on that tile, and
    the rescale must cover the tile's keys on both sides of the large one."""
    w = W["alpamayo_step"].with_(C=1)
    pair = Pair(w, "domh%d" % half)
    pair.fill()
    view = 1
    slot = int(pair.cache.head.cpu().numpy()[0][view])      # the slot the next insert writes
    row0 = w.P + (view * w.F + slot) * w.T
    # the first token of the frame whose row offset in its tile lies in the half
    tok = next(t for t in range(w.T) if ((row0 + t) % 128) // 64 == half and (row0 + t) % 64 >= 8)
    k, v = synth.frame_kv(w, pair.n_inserts, pair.tag)
    kf = O.bf16_to_f64(k).astype(np.float32)
    kf[:, view, tok] *= 30.0
    pair.insert(synth.f32_to_bf16_bits(kf), v)
    _prefill_check(pair, "x", max_abs=5e-2, lse_tol=30 * LSE_TOL)


@pytest.mark.parametrize("B", synth.VERIFY_BATCHES)
def test_verify_alpamayo_batches(B):
    w = W["alpamayo_verify"].with_(C=B)
    pair = Pair(w, "v%d" % B)
    pair.fill()
    pair.insert()
    pair.set_tail(w.tail_len)
    q, k, v = synth.verify_block(w, pair.tag)
    target, draft, planted = synth.planted_ids(B, w.blk, pair.tag)
    tail = torch.full((B,), w.tail_len, dtype=torch.int32, device="cuda")
    out, acc, nxt = skv.stream_attn_verify(
        pair.cache, tail, to_dev(q), to_dev(k), to_dev(v), w.sm_scale,
        target_ids=torch.from_numpy(target).cuda(), draft_ids=torch.from_numpy(draft).cuda())
    got = bf16_dev_to_f64(out)
    acc, nxt = acc.cpu().numpy(), nxt.cpu().numpy()
    kk = from_dev(pair.cache.k)
    vt = from_dev(pair.cache.vt)
    base = pair.cache.n_visual + w.tail_len
    for c in range(B):
        want, _ = O.stream_verify(pair.win[c], q[c], k[c], v[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "verify B=%d cache %d" % (B, c))
        a, n = O.accept_length(target[c], draft[c])
        assert acc[c] == a == planted[c] and nxt[c] == n
        # the block's K/V landed in the tail rows, bit-exact
        np.testing.assert_array_equal(kk[c][:, base:base + w.blk].transpose(1, 0, 2), k[c])
        np.testing.assert_array_equal(vt[c][:, :, base:base + w.blk].transpose(2, 0, 1), v[c])
    assert pair.cache.device_status() == 0


@pytest.mark.parametrize("B,blk", [(1, 9), (8, 9), (1, 17)])
def test_verify_merge_after_grid_barrier_repeats_and_captures(B, blk):
    """Small batches spread each unit over many pieces, and the partials are
    merged by every CTA after a grid barrier (a cooperative launch).  Three
    calls on one workspace (the barrier's words go back to their start state
    after each) and a CUDA-graph replay of the same call give bit-identical
    outputs, within the tolerance of the oracle."""
    w = W["alpamayo_verify"].with_(C=B, blk=blk)
    watch = list(range(B)) if B <= 2 else [0, 3, 7]
    pair = Pair(w, "vg%d_%d" % (B, blk), watch=watch)
    pair.fill()
    pair.insert()
    pair.set_tail(w.tail_len)
    q, k, v = synth.verify_block(w, pair.tag)
    tail = torch.full((B,), w.tail_len, dtype=torch.int32, device="cuda")
    dq, dk, dv = to_dev(q), to_dev(k), to_dev(v)
    ws = skv.verify_workspace(pair.cache, w.Hq, w.blk)
    assert ws.numel() > 0                       # pieces share units
    outs = []
    for _ in range(3):
        out, _, _ = skv.stream_attn_verify(pair.cache, tail, dq, dk, dv, w.sm_scale, ws=ws)
        outs.append(out.clone())
    for o in outs[1:]:
        assert torch.equal(o, outs[0])
    got = bf16_dev_to_f64(outs[0])
    for c in watch:
        want, _ = O.stream_verify(pair.win[c], q[c], k[c], v[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "verify B=%d blk %d cache %d" % (B, blk, c))
    # captured into a graph and replayed twice
    gout = torch.empty_like(outs[0])
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(g):
            skv.stream_attn_verify(pair.cache, tail, dq, dk, dv, w.sm_scale, ws=ws, out=gout)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        gout.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(gout, outs[0])
    assert pair.cache.device_status() == 0


def test_verify_full_block_rows_uneven_tails():
    """64 block rows per kv head (blk 16, 4 query heads per kv head) and a
    different tail length per cache: units end at different key tiles, so
    some shares hold pieces past a unit's keys, and units span several
    shares whose partials are merged."""
    w = W["alpamayo_verify"].with_(C=6, blk=16)
    tails = [0, 5, 16, 33, 60, 100]
    pair = Pair(w, "vr")
    pair.fill()
    pair.insert()
    tk, tv = synth.tail_kv(w, max(tails), pair.tag)
    skv.kv_write_rows(pair.cache, pair.cache.n_visual, to_dev(tk), to_dev(tv))
    for c in range(w.C):
        pair.win[c].set_tail(tk[c][:tails[c]], tv[c][:tails[c]])
    q, k, v = synth.verify_block(w, pair.tag)
    tail = torch.tensor(tails, dtype=torch.int32, device="cuda")
    out, _, _ = skv.stream_attn_verify(pair.cache, tail, to_dev(q), to_dev(k), to_dev(v), w.sm_scale)
    got = bf16_dev_to_f64(out)
    for c in range(w.C):
        want, _ = O.stream_verify(pair.win[c], q[c], k[c], v[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "verify blk 16 cache %d (tail %d)" % (c, tails[c]))
    assert pair.cache.device_status() == 0


@pytest.mark.parametrize("B", [8, 64])
def test_verify_large_tail_capacity_uneven_tails(B):
    """A tail capacity of 1024 rows with tails of 0 to 700 tokens in use: the
    shares are planned for the capacity and each piece skips the key tiles
    past its tail in use; every block row against the oracle on a spread of
    caches."""
    w = W["alpamayo_verify"].with_(C=B, tail_cap=1024)
    tails = [(37 * c * c + 11 * c) % 701 for c in range(B)]
    watch = list(range(B)) if B <= 8 else [0, 1, 2, 17, 40, 63]
    pair = Pair(w, "vcap%d" % B, watch=watch)
    pair.fill()
    pair.insert()
    tk, tv = synth.tail_kv(w, max(tails), pair.tag)
    skv.kv_write_rows(pair.cache, pair.cache.n_visual, to_dev(tk), to_dev(tv))
    for c in watch:
        pair.win[c].set_tail(tk[c][:tails[c]], tv[c][:tails[c]])
    q, k, v = synth.verify_block(w, pair.tag)
    tail = torch.tensor(tails, dtype=torch.int32, device="cuda")
    out, _, _ = skv.stream_attn_verify(pair.cache, tail, to_dev(q), to_dev(k), to_dev(v), w.sm_scale)
    got = bf16_dev_to_f64(out)
    for c in watch:
        want, _ = O.stream_verify(pair.win[c], q[c], k[c], v[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "verify tail_cap 1024 B=%d cache %d (tail %d)" % (B, c, tails[c]))
    assert pair.cache.device_status() == 0


@pytest.mark.parametrize("B", [1, 8, 64])
def test_verify_17_query_block(B):
    """A 17-query block (the last accepted token + 16 drafts): 68 block rows
    per kv head, one unit of the 128-row form that streams each plane's keys
    once; accept lengths up to 16."""
    w = W["alpamayo_verify"].with_(C=B, blk=17)
    watch = list(range(B)) if B <= 8 else [0, 1, 31, 62, 63]
    pair = Pair(w, "b17_%d" % B, watch=watch)
    pair.fill()
    pair.insert()
    pair.set_tail(w.tail_len)
    q, k, v = synth.verify_block(w, pair.tag)
    target, draft, planted = synth.planted_ids(B, w.blk, pair.tag)
    tail = torch.full((B,), w.tail_len, dtype=torch.int32, device="cuda")
    out, acc, nxt = skv.stream_attn_verify(
        pair.cache, tail, to_dev(q), to_dev(k), to_dev(v), w.sm_scale,
        target_ids=torch.from_numpy(target).cuda(), draft_ids=torch.from_numpy(draft).cuda())
    got = bf16_dev_to_f64(out)
    acc, nxt = acc.cpu().numpy(), nxt.cpu().numpy()
    for c in watch:
        want, _ = O.stream_verify(pair.win[c], q[c], k[c], v[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "17-query verify B=%d cache %d" % (B, c))
    for c in range(B):
        a, n = O.accept_length(target[c], draft[c])
        assert acc[c] == a == planted[c] and nxt[c] == n
    assert pair.cache.device_status() == 0


# Degenerate and ragged geometries: no prefix, one view of one frame,
# one-token frames, MHA (G = 1), eight query heads per kv head (a 9-query
# block is then 72 rows: one unit of the 128-row form), frames and prefixes
# that fill no tile evenly.
DEGENERATE = [
    # name, P, V, F, T, Hq, Hkv, d
    ("no_prefix", 0, 2, 3, 40, 8, 2, 64),
    ("one_view_one_frame", 16, 1, 1, 64, 8, 8, 128),
    ("mha_ragged", 7, 3, 2, 33, 4, 4, 128),
    ("gqa8", 12, 2, 2, 50, 64, 8, 128),
    ("one_token_frames", 5, 3, 4, 1, 8, 2, 64),
]


@pytest.mark.parametrize("geo", DEGENERATE, ids=[g[0] for g in DEGENERATE])
def test_degenerate_geometries(geo):
    name, P, V, F, T, Hq, Hkv, d = geo
    w = synth.Workload(name, P=P, V=V, F=F, T=T, Hq=Hq, Hkv=Hkv, d=d, theta=1e4, C=2,
                       sm_scale=1.0 / np.sqrt(d), tail_cap=32, tail_len=5, blk=9)
    pair = Pair(w, "dg")
    pair.fill()
    for _ in range(2):          # the ring wraps (F = 1: every insert replaces the frame)
        pair.insert()
    pair.check_ring()
    _prefill_check(pair, "dg")
    pair.set_tail(w.tail_len)
    q, k, v = synth.verify_block(w, pair.tag)
    tail = torch.full((w.C,), w.tail_len, dtype=torch.int32, device="cuda")
    out, _, _ = skv.stream_attn_verify(pair.cache, tail, to_dev(q), to_dev(k), to_dev(v), w.sm_scale)
    got = bf16_dev_to_f64(out)
    for c in range(w.C):
        want, _ = O.stream_verify(pair.win[c], q[c], k[c], v[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "%s verify cache %d" % (name, c))
    assert pair.cache.device_status() == 0


WIDE_BLOCKS = [
    # name, Hq, Hkv, d, blk: rows per kv head = blk * Hq / Hkv
    ("d64_68_rows", 8, 2, 64, 17),       # head_dim 64: one key row per RoPE thread
    ("g8_136_rows", 64, 8, 128, 17),     # two units of the 128-row form per plane
    ("g4_128_rows", 32, 8, 128, 32),     # exactly one full unit
]


@pytest.mark.parametrize("geo", WIDE_BLOCKS, ids=[g[0] for g in WIDE_BLOCKS])
def test_verify_blocks_of_more_than_64_rows(geo):
    """Blocks of more than 64 rows per kv head run on the 128-row form of the
    verify kernel; uneven tails, every block row against the oracle."""
    name, Hq, Hkv, d, blk = geo
    w = synth.Workload(name, P=12, V=2, F=2, T=50, Hq=Hq, Hkv=Hkv, d=d, theta=1e4, C=3,
                       sm_scale=1.0 / np.sqrt(d), tail_cap=96, tail_len=5, blk=blk)
    pair = Pair(w, "wd")
    pair.fill()
    pair.insert()
    tails = [0, 23, 51]
    tk, tv = synth.tail_kv(w, max(tails), pair.tag)
    skv.kv_write_rows(pair.cache, pair.cache.n_visual, to_dev(tk), to_dev(tv))
    for c in range(w.C):
        pair.win[c].set_tail(tk[c][:tails[c]], tv[c][:tails[c]])
    q, k, v = synth.verify_block(w, pair.tag)
    target, draft, planted = synth.planted_ids(w.C, w.blk, pair.tag)
    tail = torch.tensor(tails, dtype=torch.int32, device="cuda")
    out, acc, nxt = skv.stream_attn_verify(
        pair.cache, tail, to_dev(q), to_dev(k), to_dev(v), w.sm_scale,
        target_ids=torch.from_numpy(target).cuda(), draft_ids=torch.from_numpy(draft).cuda())
    got = bf16_dev_to_f64(out)
    acc, nxt = acc.cpu().numpy(), nxt.cpu().numpy()
    for c in range(w.C):
        want, _ = O.stream_verify(pair.win[c], q[c], k[c], v[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "%s verify cache %d (tail %d)" % (name, c, tails[c]))
        a, n = O.accept_length(target[c], draft[c])
        assert acc[c] == a == planted[c] and nxt[c] == n
    assert pair.cache.device_status() == 0


def test_verify_tiny_and_tail_advance():
    """Two verify rounds; the caller advances tail_len by accept_len + 1."""
    w = W["tiny"].with_(C=3, blk=9)
    pair = Pair(w, "vt")
    pair.fill()
    tail = torch.zeros((w.C,), dtype=torch.int32, device="cuda")
    tail_host = np.zeros(w.C, np.int64)
    tk = {c: np.zeros((0, w.Hkv, w.d), np.uint16) for c in range(w.C)}
    tv = {c: np.zeros((0, w.Hkv, w.d), np.uint16) for c in range(w.C)}
    for rnd in range(2):
        q, k, v = synth.verify_block(w, "r%d" % rnd)
        target, draft, _ = synth.planted_ids(w.C, w.blk, "r%d" % rnd)
        out, acc, nxt = skv.stream_attn_verify(
            pair.cache, tail, to_dev(q), to_dev(k), to_dev(v), w.sm_scale,
            target_ids=torch.from_numpy(target).cuda(), draft_ids=torch.from_numpy(draft).cuda())
        got = bf16_dev_to_f64(out)
        acc_h = acc.cpu().numpy()
        for c in range(w.C):
            pair.win[c].set_tail(tk[c], tv[c])
            want, _ = O.stream_verify(pair.win[c], q[c], k[c], v[c], w.theta, w.sm_scale)
            assert_close(got[c], want, "tiny verify round %d cache %d" % (rnd, c))
            keep = int(acc_h[c]) + 1
            tk[c] = np.concatenate([tk[c], k[c][:keep]])
            tv[c] = np.concatenate([tv[c], v[c][:keep]])
            tail_host[c] += keep
        tail += acc + 1
        np.testing.assert_array_equal(tail.cpu().numpy(), tail_host)


def test_verify_tail_overflow_sets_status():
    w = W["tiny"].with_(C=2, blk=9)
    pair = Pair(w, "ovf")
    pair.fill()
    before_k = from_dev(pair.cache.k)
    tail = torch.tensor([w.tail_cap - 8, 0], dtype=torch.int32, device="cuda")
    q, k, v = synth.verify_block(w, "ovf")
    out = torch.zeros((w.C, w.blk, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    skv.stream_attn_verify(pair.cache, tail, to_dev(q), to_dev(k), to_dev(v), w.sm_scale, out=out)
    assert pair.cache.device_status() & skv.SKV_DEV_TAIL_OVERFLOW
    after_k = from_dev(pair.cache.k)
    np.testing.assert_array_equal(after_k[0], before_k[0])      # cache 0 skipped entirely
    assert (from_dev(out)[0] == 0).all()
    want, _ = O.stream_verify(pair.win[1], q[1], k[1], v[1], w.theta, w.sm_scale)
    assert_close(bf16_dev_to_f64(out)[1], want, "cache 1 unaffected")


def test_bad_head_sets_status():
    w = W["tiny"].with_(C=2)
    pair = Pair(w, "bh")
    pair.fill()
    pair.cache.head[1, 0] = w.F + 3
    k, v = synth.frame_kv(w, 99, "bh")
    skv.kv_stream_insert(pair.cache, to_dev(k), to_dev(v))
    assert pair.cache.device_status() & skv.SKV_DEV_BAD_HEAD
    heads = pair.cache.head.cpu().numpy()
    assert heads[1, 0] == w.F + 3 and (heads[0] == 1).all() and heads[1, 1] == 1


def test_untouched_rows_keep_their_bytes():
    """Finite poison in the tail and padding rows survives inserts."""
    w = W["alpamayo_step"].with_(C=2)
    pair = Pair(w, "poison")
    nv = pair.cache.n_visual
    pair.cache.k[:, :, nv:] = 1536.0
    pair.cache.vt[:, :, :, nv:] = -77.0
    pair.fill()
    pair.insert()
    pair.insert()
    pair.check_ring()
    assert (pair.cache.k[:, :, nv:] == 1536.0).all()
    assert (pair.cache.vt[:, :, :, nv:] == -77.0).all()
    _prefill_check(pair, "p")


def test_checkpoint_resume_mid_stream():
    """Copy the cache state to the host mid-stream, restore it into a fresh
    cache, and continue: identical bytes and outputs."""
    w = W["tiny"].with_(C=2)
    a = Pair(w, "ckpt")
    a.fill()
    a.insert()
    saved = {n: getattr(a.cache, n).cpu() for n in ("k", "vt", "head", "sync")}
    b = skv.StreamCache(w.C, w.P, w.V, w.F, w.T, w.Hkv, w.d, w.theta, tail_cap=w.tail_cap)
    for n, t in saved.items():
        getattr(b, n).copy_(t)
    k, v = synth.frame_kv(w, a.n_inserts, a.tag)
    q = synth.frame_q(w, a.n_inserts, a.tag)
    a.insert()
    skv.kv_stream_insert(b, to_dev(k), to_dev(v))
    oa = skv.stream_attn_prefill(a.cache, to_dev(q), w.sm_scale)
    ob = skv.stream_attn_prefill(b, to_dev(q), w.sm_scale)
    assert torch.equal(a.cache.k, b.k) and torch.equal(a.cache.vt, b.vt)
    assert torch.equal(a.cache.head, b.head)
    assert torch.equal(oa, ob)


def test_empty_cache_set_is_a_no_op():
    w = W["tiny"].with_(C=0)
    cache = skv.StreamCache(0, w.P, w.V, w.F, w.T, w.Hkv, w.d, w.theta, tail_cap=w.tail_cap)
    e = torch.empty((0, w.V, w.T, w.Hkv, w.d), dtype=torch.bfloat16, device="cuda")
    skv.kv_stream_insert(cache, e, e)
    q = torch.empty((0, w.n_new, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    out = skv.stream_attn_prefill(cache, q, w.sm_scale)
    assert out.numel() == 0


def test_calls_are_graph_capturable():
    """insert + prefill + verify captured into one CUDA graph and replayed
    give the same bytes as the same calls made eagerly on a twin cache."""
    w = W["tiny"].with_(C=2, blk=9)
    twins = [Pair(w, "graph"), Pair(w, "graph")]
    for t in twins:
        t.fill()
    k, v = synth.frame_kv(w, w.F, "graph")
    q = synth.frame_q(w, w.F, "graph")
    bq, bk, bv = synth.verify_block(w, "graph")
    tgt, drf, _ = synth.planted_ids(w.C, w.blk, "graph")
    dev = {n: to_dev(x) for n, x in dict(k=k, v=v, q=q, bq=bq, bk=bk, bv=bv).items()}
    ids = (torch.from_numpy(tgt).cuda(), torch.from_numpy(drf).cuda())
    outs = []
    for n, t in enumerate(twins):
        tail = torch.zeros((w.C,), dtype=torch.int32, device="cuda")
        po = torch.empty_like(dev["q"])
        vo = torch.empty_like(dev["bq"])
        acc = torch.empty((w.C,), dtype=torch.int32, device="cuda")
        nxt = torch.empty((w.C,), dtype=torch.int32, device="cuda")
        ws = skv.verify_workspace(t.cache, w.Hq, w.blk)

        def step():
            skv.kv_stream_insert(t.cache, dev["k"], dev["v"])
            skv.stream_attn_prefill(t.cache, dev["q"], w.sm_scale, out=po)
            skv.stream_attn_verify(t.cache, tail, dev["bq"], dev["bk"], dev["bv"], w.sm_scale,
                                   target_ids=ids[0], draft_ids=ids[1], ws=ws, out=vo,
                                   accept_len=acc, next_token=nxt)
        if n == 0:
            step()
        else:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                with torch.cuda.graph(g):
                    step()
            torch.cuda.current_stream().wait_stream(side)
            g.replay()
        torch.cuda.synchronize()
        outs.append((po.clone(), vo.clone(), acc.clone(), t.cache.k.clone(), t.cache.head.clone()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    assert twins[1].cache.device_status() == 0
