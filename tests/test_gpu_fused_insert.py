"""GPU parity of stream_attn_prefill_insert: the frame insert and the
new-frame prefill as one call.  On twin caches it must leave the ring bytes,
heads and insert counters exactly as kv_stream_insert followed by
stream_attn_prefill does, over several streaming steps (the ring wraps), and
its outputs must match the oracle within max-abs 1e-2 / mean-abs 1e-3.  The
one-kernel form runs where head_dim is 128 and the prefix and frames are
multiples of 64 tokens; the Alpamayo-shaped frames (180 tokens) take the
two-launch form."""
import numpy as np
import pytest
import torch

from oracle import skv_oracle as O
from streaming_kv_cache_gb300 import skv, synth

from gpu_harness import LSE_TOL, MEASURED, Pair, assert_close, assert_lse, bf16_dev_to_f64, to_dev

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_kv_cache_gb300 import build
    build.build()


def _twin_steps(w, tag, steps, rows=None, watch=None):
    """Fill two twin caches, then run `steps` streaming steps: the first by
    insert + prefill, the second by the fused call; compare after each."""
    a = Pair(w, tag, watch=watch)
    b = Pair(w, tag, watch=[])
    a.fill()
    b.fill()
    same_out = True
    for st in range(steps):
        k, v = synth.frame_kv(w, a.n_inserts, tag)
        q = synth.frame_q(w, a.n_inserts, tag)
        a.insert(k, v)
        oa, la = skv.stream_attn_prefill(a.cache, to_dev(q), w.sm_scale, lse=True)
        ob, lb = skv.stream_attn_prefill_insert(b.cache, to_dev(k), to_dev(v), to_dev(q), w.sm_scale, lse=True)
        torch.cuda.synchronize()
        assert torch.equal(a.cache.k, b.cache.k), "ring K after step %d" % st
        assert torch.equal(a.cache.vt, b.cache.vt), "ring V after step %d" % st
        assert torch.equal(a.cache.head, b.cache.head), "heads after step %d" % st
        assert (b.cache.sync == 0).all()
        assert b.cache.device_status() == 0
        same_out = same_out and torch.equal(oa, ob) and torch.equal(la, lb)
        got, got_lse = bf16_dev_to_f64(ob), lb.cpu().numpy()
        for c, win in a.win.items():
            want, wl = O.stream_prefill(win, q[c], w.theta, w.sm_scale, rows=rows)
            sel = slice(None) if rows is None else rows
            assert_close(got[c][sel], want, "%s fused step %d cache %d" % (w.name, st, c))
            assert_lse(got_lse[c][:, sel].T, wl, LSE_TOL)
    a.check_ring()
    return same_out


def test_fused_one_kernel_small_aligned_geometry():
    """Prefix 64, 3 views x 3 frames x 64 tokens, GQA 4, d = 128: five steps
    (the ring wraps), every row against the oracle, results equal to the
    two calls."""
    w = synth.Workload("aligned_small", P=64, V=3, F=3, T=64, Hq=8, Hkv=2, d=128, theta=1e6, C=2,
                       sm_scale=1.0 / np.sqrt(128), tail_cap=64)
    same = _twin_steps(w, "fz_s", 5)
    MEASURED.setdefault("test_fused_one_kernel_small_aligned_geometry", {})["bit_equal_to_two_calls"] = float(same)


def test_fused_one_kernel_scaleup_geometry():
    """The scale-up geometry (prefix 512, 6 views x 8 frames x 256 tokens),
    three layer caches, two steps; sampled rows against the oracle."""
    w = W["scaleup_36L"].with_(C=3)
    rows = np.array(sorted({0, 1, 127, 128, 255, 256, 511, 700, 1023, 1024, 1279, 1280, 1535}))
    same = _twin_steps(w, "fz_b", 2, rows=rows, watch=[0, 2])
    MEASURED.setdefault("test_fused_one_kernel_scaleup_geometry", {})["bit_equal_to_two_calls"] = float(same)


def test_fused_call_on_frames_of_180_tokens():
    """Frames of 180 tokens cannot be cut into 64-token blocks: the call
    enqueues the insert and the prefill; the same checks hold."""
    w = W["alpamayo_step"].with_(C=2)
    rows = np.arange(0, w.n_new, 37)
    assert _twin_steps(w, "fz_a", 2, rows=rows)
