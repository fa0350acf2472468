"""Failure detection without a GPU fault.

Every barrier wait of the attention kernels is bounded by the cache's
`wait_ns`.  With a 1 ns limit the first wait that is not already satisfied
gives up: the kernel sets SKV_DEV_TIMEOUT in the caller's status word, lets
the copies and MMAs its own threads started land, frees its tensor memory
and returns.  The test then shows that the context and the cache still work:
the same calls with the normal limit match the oracle."""
import numpy as np
import pytest
import torch

from oracle import skv_oracle as O
from streaming_kv_cache_gb300 import skv, synth

from gpu_harness import Pair, assert_close, bf16_dev_to_f64, to_dev

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_kv_cache_gb300 import build
    build.build()


@pytest.mark.parametrize("name,blk", [("tiny", 9), ("alpamayo_step", 9), ("alpamayo_step", 17)])
def test_wait_timeout_sets_status_and_context_survives(name, blk):
    """blk 17 at four query heads per kv head is 68 block rows: the 128-row
    form of the verify kernel."""
    w = W[name] if name == "tiny" else W[name].with_(C=2)
    pair = Pair(w, "to")
    pair.fill()
    cache = pair.cache
    q = synth.frame_q(w, pair.n_inserts - 1, "to")
    wv = w.with_(blk=blk)
    qb, kb, vb = synth.verify_block(wv, "to")
    tail = torch.zeros((w.C,), dtype=torch.int32, device="cuda")
    ws = skv.verify_workspace(cache, w.Hq, blk)

    # 1 ns: the kernels give up at their first wait that is not already met
    cache.wait_ns = 1
    skv.stream_attn_prefill(cache, to_dev(q), w.sm_scale)
    torch.cuda.synchronize()
    assert cache.device_status() & skv.SKV_DEV_TIMEOUT
    cache.status.zero_()
    skv.stream_attn_verify(cache, tail, to_dev(qb), to_dev(kb), to_dev(vb), w.sm_scale, ws=ws)
    torch.cuda.synchronize()
    assert cache.device_status() & skv.SKV_DEV_TIMEOUT

    # the normal limit again: same cache, same context, results match the oracle.
    # A call that set a status bit may leave workspace counters behind: re-zero.
    cache.wait_ns = 0
    cache.status.zero_()
    ws.zero_()
    out = skv.stream_attn_prefill(cache, to_dev(q), w.sm_scale)
    got = bf16_dev_to_f64(out)
    for c in pair.watch:
        want, _ = O.stream_prefill(pair.win[c], q[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "%s prefill after a timeout, cache %d" % (name, c))
    out = skv.stream_attn_verify(cache, tail, to_dev(qb), to_dev(kb), to_dev(vb), w.sm_scale, ws=ws)[0]
    got = bf16_dev_to_f64(out)
    for c in pair.watch:
        pair.win[c].set_tail(np.zeros((0, w.Hkv, w.d), np.uint16), np.zeros((0, w.Hkv, w.d), np.uint16))
        want, _ = O.stream_verify(pair.win[c], qb[c], kb[c], vb[c], w.theta, w.sm_scale)
        assert_close(got[c], want, "%s verify after a timeout, cache %d" % (name, c))
    assert cache.device_status() == 0


@pytest.mark.parametrize("blk", [9, 17])
def test_short_limit_path_matches_the_oracle(blk):
    """A wait limit under a millisecond selects the kernels' polling
    instantiations (no suspend hint, the clock read at every poll); with a
    limit no wait reaches (0.9 ms) they give the same results as the normal
    ones, for both forms of the verify kernel."""
    w = W["alpamayo_step"].with_(C=2, blk=blk)
    pair = Pair(w, "sl%d" % blk, wait_ns=900000)
    pair.fill()
    pair.insert()
    q = synth.frame_q(w, pair.n_inserts - 1, pair.tag)
    out = bf16_dev_to_f64(skv.stream_attn_prefill(pair.cache, to_dev(q), w.sm_scale))
    for c in pair.watch:
        want, _ = O.stream_prefill(pair.win[c], q[c], w.theta, w.sm_scale)
        assert_close(out[c], want, "short-limit prefill cache %d" % c)
    qb, kb, vb = synth.verify_block(w, pair.tag)
    tail = torch.zeros((w.C,), dtype=torch.int32, device="cuda")
    vout = bf16_dev_to_f64(skv.stream_attn_verify(pair.cache, tail, to_dev(qb), to_dev(kb), to_dev(vb),
                                                  w.sm_scale)[0])
    for c in pair.watch:
        want, _ = O.stream_verify(pair.win[c], qb[c], kb[c], vb[c], w.theta, w.sm_scale)
        assert_close(vout[c], want, "short-limit verify blk %d cache %d" % (blk, c))
    assert pair.cache.device_status() == 0
