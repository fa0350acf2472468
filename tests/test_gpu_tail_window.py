"""GPU parity of the two other query sets of the streaming step against the
fp64 oracle: the trajectory / text tokens after the views
(stream_attn_prefill_tail) and every window token (stream_attn_window, the
first window).  Both run on the tensor-core prefill kernel.  Tail rows are
compared bit for bit; outputs within max-abs 1e-2 and mean-abs 1e-3, LSE
within 1e-2."""
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


def _set_tails(pair, tails):
    """Different tail lengths per cache, written to the cache and the oracle."""
    w = pair.w
    n = max(tails)
    tk, tv = synth.tail_kv(w, n, pair.tag)
    if n:
        skv.kv_write_rows(pair.cache, pair.cache.n_visual, to_dev(tk), to_dev(tv))
    for c, win in pair.win.items():
        win.set_tail(tk[c][:tails[c]], tv[c][:tails[c]])
    return torch.tensor(tails, dtype=torch.int32, device="cuda")


def _tail_check(pair, tail, n, tag):
    """One stream_attn_prefill_tail call against the oracle; appends the
    tokens to the oracle windows' tails."""
    w = pair.w
    q, k, v = synth.tail_block(w, n, pair.tag + tag)
    tails = tail.cpu().numpy()
    out, lse = skv.stream_attn_prefill_tail(pair.cache, tail, to_dev(q), to_dev(k), to_dev(v),
                                            w.sm_scale, lse=True)
    got, got_lse = bf16_dev_to_f64(out), lse.cpu().numpy()
    kk, vt = from_dev(pair.cache.k), from_dev(pair.cache.vt)
    for c, win in pair.win.items():
        want, wl = O.stream_prefill_tail(win, q[c], k[c], v[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "%s tail n=%d cache %d" % (w.name, n, c))
        assert_lse(got_lse[c].T, wl, LSE_TOL, "%s tail cache %d" % (w.name, c))
        base = pair.cache.n_visual + int(tails[c])
        np.testing.assert_array_equal(kk[c][:, base:base + n].transpose(1, 0, 2), k[c])
        np.testing.assert_array_equal(vt[c][:, :, base:base + n].transpose(2, 0, 1), v[c])
        win.set_tail(np.concatenate([win.tail_k, k[c]]), np.concatenate([win.tail_v, v[c]]))
    assert pair.cache.device_status() == 0


@pytest.mark.parametrize("n", [1, 9, 32])
def test_tail_prefill_tiny(n):
    w = W["tiny"].with_(C=2)
    pair = Pair(w, "tt%d" % n)
    pair.fill()
    pair.insert()
    tail = torch.zeros((w.C,), dtype=torch.int32, device="cuda")
    _tail_check(pair, tail, n, "a")


@pytest.mark.parametrize("n", [9, 100, 128])
def test_tail_prefill_alpamayo_uneven_tails(n):
    """Tail tokens after a different number of existing tail rows per cache;
    n = 100 and 128 (the whole tail) span several query tiles with a ragged
    end."""
    w = W["alpamayo_step"].with_(C=3)
    pair = Pair(w, "ta%d" % n)
    pair.fill()
    pair.insert()
    tails = [0, 16, 28][: w.C] if n < 128 else [0, 0, 0]
    tail = _set_tails(pair, tails)
    _tail_check(pair, tail, n, "a")


def test_streaming_step_views_then_tail_then_verify():
    """One whole step: insert the new frames, prefill their queries, prefill
    20 trajectory / text tokens after the views, then verify a 9-token block
    after them; every stage against the oracle."""
    w = W["alpamayo_step"].with_(C=2, blk=9)
    pair = Pair(w, "step")
    pair.fill()
    pair.insert()
    q = synth.frame_q(w, pair.n_inserts - 1, "step")
    got = bf16_dev_to_f64(skv.stream_attn_prefill(pair.cache, to_dev(q), w.sm_scale))
    for c, win in pair.win.items():
        want, _ = O.stream_prefill(win, q[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "step prefill cache %d" % c)
    tail = torch.zeros((w.C,), dtype=torch.int32, device="cuda")
    _tail_check(pair, tail, 20, "tx")
    tail += 20
    bq, bk, bv = synth.verify_block(w, "step")
    out, _, _ = skv.stream_attn_verify(pair.cache, tail, to_dev(bq), to_dev(bk), to_dev(bv), w.sm_scale)
    got = bf16_dev_to_f64(out)
    for c, win in pair.win.items():
        want, _ = O.stream_verify(win, bq[c], bk[c], bv[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "step verify cache %d" % c)
    assert pair.cache.device_status() == 0


def test_tail_prefill_overflow_sets_status():
    w = W["tiny"].with_(C=2)
    pair = Pair(w, "tov")
    pair.fill()
    before_k = from_dev(pair.cache.k)
    tail = torch.tensor([w.tail_cap - 4, 0], dtype=torch.int32, device="cuda")
    q, k, v = synth.tail_block(w, 9, "tov")
    out = torch.zeros((w.C, 9, w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    skv.stream_attn_prefill_tail(pair.cache, tail, to_dev(q), to_dev(k), to_dev(v), w.sm_scale, out=out)
    assert pair.cache.device_status() & skv.SKV_DEV_TAIL_OVERFLOW
    np.testing.assert_array_equal(from_dev(pair.cache.k)[0], before_k[0])   # cache 0 skipped
    assert (from_dev(out)[0] == 0).all()
    want, _ = O.stream_prefill_tail(pair.win[1], q[1], k[1], v[1], w.theta, w.sm_scale)
    assert_close(bf16_dev_to_f64(out)[1], want, "cache 1 unaffected")


def _window_check(pair, tag, rows=None):
    w = pair.w
    q = synth.window_q(w, pair.tag + tag)
    out, lse = skv.stream_attn_window(pair.cache, to_dev(q), w.sm_scale, lse=True)
    got, got_lse = bf16_dev_to_f64(out), lse.cpu().numpy()
    sel = slice(None) if rows is None else rows
    for c, win in pair.win.items():
        want, wl = O.stream_window(win, q[c], w.theta, w.sm_scale, rows=rows)
        assert_close(got[c][sel], want, "%s window cache %d" % (w.name, c))
        assert_lse(got_lse[c][:, sel].T, wl, LSE_TOL, "%s window cache %d" % (w.name, c))
    assert pair.cache.device_status() == 0


@pytest.mark.parametrize("extra", [0, 1, 3])
def test_window_tiny(extra):
    """extra = 0: the first window (every head 0); 1 and 3: the ring has
    turned, so a frame's hole (its view's later frames) wraps around the end
    of the ring."""
    w = W["tiny"].with_(C=2)
    pair = Pair(w, "wt%d" % extra)
    pair.fill()
    for _ in range(extra):
        pair.insert()
    _window_check(pair, "a")


@pytest.mark.parametrize("extra", [0, 2])
def test_window_alpamayo(extra):
    w = W["alpamayo_step"].with_(C=1)
    pair = Pair(w, "wa%d" % extra)
    pair.fill()
    for _ in range(extra):
        pair.insert()
    _window_check(pair, "a")


def test_window_scaleup_sampled_rows():
    """The scale-up geometry (prefix 512, 6 views x 8 frames x 256 tokens)
    with a turned ring; rows from the prefix, every view's first, middle and
    last frames, tile edges and the last token."""
    w = W["scaleup_36L"].with_(C=2)
    pair = Pair(w, "ws", watch=[1])
    pair.fill()
    pair.insert()
    FT = w.F * w.T
    rows = [0, 1, 127, 128, w.P - 1]
    for v in range(w.V):
        for f in (0, 3, w.F - 1):
            b = w.P + v * FT + f * w.T
            rows += [b, b + 127, b + 128, b + w.T - 1]
    rows = np.array(sorted(set(rows + [w.n_window - 1])))
    _window_check(pair, "a", rows=rows)


def test_window_scaleup_whole_cache():
    """Every one of the 12,800 window tokens of one scale-up cache (turned
    ring), all heads, element by element; the oracle works through the rows
    in chunks to bound its memory."""
    w = W["scaleup_36L"].with_(C=2)
    pair = Pair(w, "wsw", watch=[0])
    pair.fill()
    pair.insert()
    q = synth.window_q(w, pair.tag + "a")
    out, lse = skv.stream_attn_window(pair.cache, to_dev(q), w.sm_scale, lse=True)
    got, got_lse = bf16_dev_to_f64(out), lse.cpu().numpy()
    assert pair.cache.device_status() == 0
    win = pair.win[0]
    for rows in np.array_split(np.arange(w.n_window), 16):
        want, wl = O.stream_window(win, q[0], w.theta, w.sm_scale, rows=rows)
        assert_close(got[0][rows], want, "scale-up window rows %d..%d" % (rows[0], rows[-1]))
        assert_lse(got_lse[0][:, rows].T, wl, LSE_TOL, "scale-up window")


WINDOW_GEOMETRIES = [
    # name, P, V, F, T, Hq, Hkv, d
    ("no_prefix", 0, 2, 3, 40, 8, 2, 64),
    ("mha_ragged", 7, 3, 2, 33, 4, 4, 128),
    ("gqa8_long_prefix", 300, 2, 2, 50, 64, 8, 128),
    ("one_token_frames", 5, 3, 4, 1, 8, 2, 64),
]


@pytest.mark.parametrize("geo", WINDOW_GEOMETRIES, ids=[g[0] for g in WINDOW_GEOMETRIES])
def test_window_and_tail_degenerate_geometries(geo):
    name, P, V, F, T, Hq, Hkv, d = geo
    w = synth.Workload(name, P=P, V=V, F=F, T=T, Hq=Hq, Hkv=Hkv, d=d, theta=1e4, C=2,
                       sm_scale=1.0 / np.sqrt(d), tail_cap=48)
    pair = Pair(w, "wd")
    pair.fill()
    pair.insert()
    _window_check(pair, "a")
    tail = _set_tails(pair, [3, 0])
    _tail_check(pair, tail, 45, "b")


def test_streams_at_different_phases_in_one_launch():
    """Several independent streams (vehicles) in one launch of each call:
    every cache's ring has turned a different number of times (its own head)
    and its tail holds a different number of tokens.  Insert, prefill of the
    new frames, the whole window, tail tokens and a verify block are each one
    launch over all caches and match the oracle cache by cache."""
    w = W["alpamayo_step"].with_(C=4, blk=9)
    pair = Pair(w, "phase")
    pair.fill()
    heads = [(3 * c) % w.F for c in range(w.C)]
    pair.cache.head.copy_(torch.tensor(heads, dtype=torch.int32)[:, None].expand(w.C, w.V).contiguous().cuda())
    for c, win in pair.win.items():
        for dq in win.views:
            dq.rotate(-heads[c])     # logical frame f now lives in slot (head + f) mod F
    pair.insert()
    got_heads = pair.cache.head.cpu().numpy()
    np.testing.assert_array_equal(got_heads[:, 0], [(h + 1) % w.F for h in heads])
    q = synth.frame_q(w, pair.n_inserts - 1, "phase")
    got = bf16_dev_to_f64(skv.stream_attn_prefill(pair.cache, to_dev(q), w.sm_scale))
    for c, win in pair.win.items():
        want, _ = O.stream_prefill(win, q[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "prefill, stream %d (head %d)" % (c, heads[c]))
    rows = np.array([0, 255, 256, w.P + 5, w.P + w.T + 3, w.n_window // 2, w.n_window - 1])
    _window_check(pair, "w", rows=rows)
    tail = _set_tails(pair, [0, 7, 30, 64])
    _tail_check(pair, tail, 12, "t")
    tail += 12
    bq, bk, bv = synth.verify_block(w, "phase")
    out, _, _ = skv.stream_attn_verify(pair.cache, tail, to_dev(bq), to_dev(bk), to_dev(bv), w.sm_scale)
    got = bf16_dev_to_f64(out)
    for c, win in pair.win.items():
        want, _ = O.stream_verify(win, bq[c], bk[c], bv[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "verify, stream %d" % c)
    assert pair.cache.device_status() == 0
