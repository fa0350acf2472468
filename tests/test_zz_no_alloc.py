"""kv_stream_insert_noalloc: the insert for callers that cannot allocate
device memory (its scratch counters live in a static device array inside
the library).  Called through the C ABI and compared with kv_stream_insert
on two calls in a row.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from streaming_kv_cache_gb300 import skv, synth

pytestmark = pytest.mark.gpu


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def test_noalloc_insert_matches_insert_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_kv_cache_gb300 import build
    build.build()
    L = skv.lib()
    w = synth.WORKLOADS["alpamayo_step"].with_(C=3)
    caches = [skv.StreamCache(w.C, w.P, w.V, w.F, w.T, w.Hkv, w.d, w.theta, tail_cap=w.tail_cap)
              for _ in range(2)]
    pk, pv = synth.prefix_kv(w, "na")
    for c in caches:
        skv.kv_write_rows(c, 0, _dev(pk), _dev(pv))
    ref, new = caches
    # a sentinel in the cache's own counter tensor: the descriptor handed to
    # the no-alloc call carries no sync pointer, so these must stay untouched
    new.sync.fill_(0x5A5A)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for i in range(w.F + 2):          # fills the window, then two streaming steps
        k, v = synth.frame_kv(w, i, "na")
        kd, vd = _dev(k), _dev(v)
        skv.kv_stream_insert(ref, kd, vd)
        desc = new.desc()
        desc.sync = None                 # the caller provides no scratch
        rc = L.kv_stream_insert_noalloc(ctypes.byref(desc), ctypes.c_void_p(kd.data_ptr()),
                                        ctypes.c_void_p(vd.data_ptr()), stream)
        assert rc == skv.SKV_OK, skv.status_string(rc)
        torch.cuda.synchronize()
        # insert is a bit-exact copy: compare bytes, heads and status
        assert torch.equal(ref.k, new.k), i
        assert torch.equal(ref.vt, new.vt), i
        assert torch.equal(ref.head, new.head), i
        assert new.device_status() == 0 and ref.device_status() == 0
    assert (new.sync == 0x5A5A).all()    # the cache's own counters were never touched


def test_noalloc_insert_rejects_too_many_counters():
    L = skv.lib() if torch.cuda.is_available() else pytest.skip("no CUDA device")
    d = skv.skv_cache(n_cache=skv.SKV_NOALLOC_MAX_CACHE_VIEWS // 4 + 1, n_view=4, n_frame=4,
                      frame_len=180, prefix_len=256, tail_cap=128, n_kv_head=8, head_dim=128,
                      row_cap=3328, rope_len=3264, k=0x10000, vt=0x20000, head=0x30000, sync=None,
                      rope=0x40000, status=0x50000, wait_ns=0)
    assert L.kv_stream_insert_noalloc(ctypes.byref(d), ctypes.c_void_p(0x10000),
                                      ctypes.c_void_p(0x10000), None) == skv.SKV_ERR_TOO_LARGE
