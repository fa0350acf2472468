"""GPU parity of the multi-section rotary reading (rope_mode 1): the table
builder against the oracle's position triples, and insert, prefill of the new
frames, tail tokens, the whole window and verify against the oracle run with
the same reading.  Outputs within max-abs 1e-2 and mean-abs 1e-3."""
import numpy as np
import pytest
import torch

from oracle import skv_oracle as O
from streaming_kv_cache_gb300 import skv, synth

from gpu_harness import LSE_TOL, Pair, assert_close, assert_lse, bf16_dev_to_f64, to_dev

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_kv_cache_gb300 import build
    build.build()


def _reading(w, grid_w):
    """The oracle's reading and the cache argument for it: frequencies dealt
    in turn, the height and width shares 5/16 of the d/2 each."""
    n_hw = (w.d // 2) * 5 // 16
    sec = O.interleaved_sections(w.d, n_hw, n_hw)
    return O.MRope(w.P, w.V, w.F, w.T, grid_w, sec), (grid_w, sec)


@pytest.mark.parametrize("name,grid_w", [("tiny", 4), ("alpamayo_step", 15)])
def test_mrope_table_is_the_reading(name, grid_w):
    """Row n of the table holds cos / sin of the angles of the token at
    logical index n: the triple's component of each frequency times
    theta^(-2i/d), rounded once from fp64.  The rows of the prefix and the
    tail (t = h = w = n) are the 1-D table's, bit for bit."""
    w = W[name]
    m, arg = _reading(w, grid_w)
    n_pos = w.n_window + w.tail_cap
    tab = torch.empty((n_pos, w.d // 2, 2), dtype=torch.float32, device="cuda")
    skv.skv_build_mrope_table(tab, w.theta, w.P, w.V, w.F, w.T, grid_w, arg[1])
    got = tab.cpu().numpy().astype(np.float64)
    tr = m.triples(np.arange(n_pos))
    inv = float(w.theta) ** (-2.0 * np.arange(w.d // 2) / w.d)
    ang = tr[:, m.sec].astype(np.float64) * inv[None, :]
    np.testing.assert_allclose(got[..., 0], np.cos(ang), atol=2e-7, rtol=0)
    np.testing.assert_allclose(got[..., 1], np.sin(ang), atol=2e-7, rtol=0)
    one_d = torch.empty_like(tab)
    skv.skv_build_rope_table(one_d, w.theta)
    assert torch.equal(tab[:w.P], one_d[:w.P])
    assert torch.equal(tab[w.n_window:], one_d[w.n_window:])
    assert not torch.equal(tab[w.P:w.n_window], one_d[w.P:w.n_window])


def _mrope_step(w, grid_w, tag, window_rows=None):
    m, arg = _reading(w, grid_w)
    pair = Pair(w, tag, mrope=arg)
    pair.fill()
    pair.insert()                      # the ring has turned: positions have shifted
    pair.check_ring()
    # new frames
    q = synth.frame_q(w, pair.n_inserts - 1, tag)
    out, lse = skv.stream_attn_prefill(pair.cache, to_dev(q), w.sm_scale, lse=True)
    got, got_lse = bf16_dev_to_f64(out), lse.cpu().numpy()
    for c, win in pair.win.items():
        want, wl = O.stream_prefill(win, q[c], w.theta, w.sm_scale, mrope=m)
        assert_close(got[c], want, "%s mrope prefill cache %d" % (w.name, c))
        assert_lse(got_lse[c].T, wl, LSE_TOL)
        one_d, _ = O.stream_prefill(win, q[c], w.theta, w.sm_scale)
        assert np.abs(one_d - want).max() > 2e-2      # the reading changes these results
    # the whole window, some rows
    qw = synth.window_q(w, tag)
    outw = bf16_dev_to_f64(skv.stream_attn_window(pair.cache, to_dev(qw), w.sm_scale))
    sel = slice(None) if window_rows is None else window_rows
    for c, win in pair.win.items():
        want, _ = O.stream_window(win, qw[c], w.theta, w.sm_scale, rows=window_rows, mrope=m)
        assert_close(outw[c][sel], want, "%s mrope window cache %d" % (w.name, c))
    # tail tokens after the views, then a verify block after them
    n_tail = 7
    tq, tk, tv = synth.tail_block(w, n_tail, tag)
    tail = torch.zeros((w.C,), dtype=torch.int32, device="cuda")
    tout = bf16_dev_to_f64(skv.stream_attn_prefill_tail(pair.cache, tail, to_dev(tq), to_dev(tk), to_dev(tv),
                                                        w.sm_scale))
    for c, win in pair.win.items():
        want, _ = O.stream_prefill_tail(win, tq[c], tk[c], tv[c], w.theta, w.sm_scale, mrope=m)
        assert_close(tout[c], want, "%s mrope tail cache %d" % (w.name, c))
        win.set_tail(tk[c], tv[c])
    tail += n_tail
    bq, bk, bv = synth.verify_block(w, tag)
    vout, _, _ = skv.stream_attn_verify(pair.cache, tail, to_dev(bq), to_dev(bk), to_dev(bv), w.sm_scale)
    vout = bf16_dev_to_f64(vout)
    for c, win in pair.win.items():
        want, _ = O.stream_verify(win, bq[c], bk[c], bv[c], w.theta, w.sm_scale, mrope=m)
        assert_close(vout[c], want, "%s mrope verify cache %d" % (w.name, c))
    assert pair.cache.device_status() == 0


def test_mrope_tiny_streaming_step():
    _mrope_step(W["tiny"].with_(C=2), 4, "mr_t")


def test_mrope_alpamayo_streaming_step():
    """Frames of 180 tokens in 12 rows of 15; prefill of all 720 new-frame
    queries, window rows at frame and row edges, tail tokens and a verify
    block, two caches."""
    w = W["alpamayo_step"].with_(C=2)
    FT = w.F * w.T
    rows = [0, 255, 256, 270, 271, w.P + FT - 1]
    for v in range(w.V):
        for f in (0, w.F - 1):
            b = w.P + v * FT + f * w.T
            rows += [b, b + 14, b + 15, b + 100, b + w.T - 1]
    _mrope_step(w, 15, "mr_a", window_rows=np.array(sorted(set(rows))))


def test_mrope_17_token_verify_block():
    """The multi-section reading on the 128-row form of the verify kernel
    (17 tokens x 4 heads = 68 block rows), two caches after a ring turn."""
    w = W["alpamayo_step"].with_(C=2, blk=17)
    m, arg = _reading(w, 15)
    pair = Pair(w, "mr17", mrope=arg)
    pair.fill()
    pair.insert()
    bq, bk, bv = synth.verify_block(w, pair.tag)
    tail = torch.zeros((w.C,), dtype=torch.int32, device="cuda")
    vout, _, _ = skv.stream_attn_verify(pair.cache, tail, to_dev(bq), to_dev(bk), to_dev(bv), w.sm_scale)
    vout = bf16_dev_to_f64(vout)
    for c, win in pair.win.items():
        win.set_tail(np.zeros((0, w.Hkv, w.d), np.uint16), np.zeros((0, w.Hkv, w.d), np.uint16))
        want, _ = O.stream_verify(win, bq[c], bk[c], bv[c], w.theta, w.sm_scale, mrope=m)
        assert_close(vout[c], want, "mrope 17-token verify cache %d" % c)
    assert pair.cache.device_status() == 0
