"""Guard bands around the caller's buffers.  Every output a call writes
(attention output, LSE, accept length, next token) and the verify
workspace sit inside a larger allocation between two 8 KiB guard bands
filled with a fixed bit pattern; a float output starts as NaN, an int32 one
as a value it can never take.
After the call the guards must hold their bytes (no write past either end),
the outputs must hold no NaN (every element written), and the results must
be bit-identical to the same call on plain buffers.  The guards lie inside
the same allocation, so a stray write lands in them instead of faulting."""
import math

import numpy as np
import pytest
import torch

from streaming_kv_cache_gb300 import skv, synth

from gpu_harness import Pair, to_dev

pytestmark = pytest.mark.gpu

GUARD_BYTES = 8192
# bit patterns (as the signed integer type of the same width): guards, and
# what the buffer starts with (NaN for the float outputs, a value the int32
# results cannot take, zero for the workspace)
BITS = {torch.bfloat16: (torch.int16, -0x5B, 0x7FC1),            # 0xFFA5 / 0x7FC1
        torch.float32: (torch.int32, -0x5A5A5A5B, 0x7FC00001),   # 0xA5A5A5A5 / quiet NaN
        torch.int32: (torch.int32, 0x5A5A5A5A, -0x7FFFFFFF),
        torch.uint8: (torch.uint8, 0xA5, 0)}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from streaming_kv_cache_gb300 import build
    build.build()


class Guarded:
    """A buffer of `shape` with guard bands on both sides in one allocation."""

    def __init__(self, shape, dtype):
        itype, self.guard_bits, poison = BITS[dtype]
        esize = torch.empty((), dtype=dtype).element_size()
        self.g = GUARD_BYTES // esize
        self.n = math.prod(shape)
        self.raw = torch.empty((2 * self.g + self.n,), dtype=dtype, device="cuda")
        self.bits = self.raw.view(itype)
        self.bits.fill_(self.guard_bits)
        self.bits[self.g:self.g + self.n].fill_(poison)
        self.t = self.raw[self.g:self.g + self.n].view(shape)
        assert self.t.data_ptr() % 16 == 0

    def guards_intact(self):
        head, tail = self.bits[:self.g], self.bits[self.g + self.n:]
        return bool((head == self.guard_bits).all()) and bool((tail == self.guard_bits).all())


def _check_out(gd: Guarded, plain: torch.Tensor, what: str):
    assert gd.guards_intact(), "%s: a guard band was written" % what
    if gd.t.dtype.is_floating_point:
        assert not torch.isnan(gd.t).any(), "%s: some elements were never written" % what
    assert torch.equal(gd.t.view(torch.int16) if gd.t.dtype == torch.bfloat16 else gd.t,
                       plain.view(torch.int16) if plain.dtype == torch.bfloat16 else plain), \
        "%s: differs from the same call on a plain buffer" % what


@pytest.mark.parametrize("name", ["tiny", "alpamayo_step"])
def test_prefill_window_and_tail_write_only_their_outputs(name):
    w = synth.WORKLOADS[name].with_(C=2)
    pair = Pair(w, "guard")
    pair.fill()
    pair.insert()
    C, Hq = w.C, w.Hq

    q = to_dev(synth.frame_q(w, pair.n_inserts - 1, "guard"))
    out_g, lse_g = Guarded(q.shape, torch.bfloat16), Guarded((C, Hq, w.n_new), torch.float32)
    skv.stream_attn_prefill(pair.cache, q, w.sm_scale, out=out_g.t, lse=lse_g.t)
    out_p, lse_p = skv.stream_attn_prefill(pair.cache, q, w.sm_scale, lse=True)
    torch.cuda.synchronize()
    _check_out(out_g, out_p, "prefill out")
    _check_out(lse_g, lse_p, "prefill lse")

    qw = to_dev(synth.window_q(w, "guard"))
    out_g, lse_g = Guarded(qw.shape, torch.bfloat16), Guarded((C, Hq, w.n_window), torch.float32)
    skv.stream_attn_window(pair.cache, qw, w.sm_scale, out=out_g.t, lse=lse_g.t)
    out_p, lse_p = skv.stream_attn_window(pair.cache, qw, w.sm_scale, lse=True)
    torch.cuda.synchronize()
    _check_out(out_g, out_p, "window out")
    _check_out(lse_g, lse_p, "window lse")

    n = 13
    tq, tk, tv = (to_dev(x) for x in synth.tail_block(w, n, "guard"))
    tail = torch.tensor([0, 5], dtype=torch.int32, device="cuda")
    out_g, lse_g = Guarded(tq.shape, torch.bfloat16), Guarded((C, Hq, n), torch.float32)
    skv.stream_attn_prefill_tail(pair.cache, tail, tq, tk, tv, w.sm_scale, out=out_g.t, lse=lse_g.t)
    out_p, lse_p = skv.stream_attn_prefill_tail(pair.cache, tail, tq, tk, tv, w.sm_scale, lse=True)
    torch.cuda.synchronize()
    _check_out(out_g, out_p, "tail out")
    _check_out(lse_g, lse_p, "tail lse")
    assert pair.cache.device_status() == 0


@pytest.mark.parametrize("name,B,blk", [("tiny", 3, 9), ("alpamayo_verify", 8, 9), ("alpamayo_verify", 8, 17),
                                         ("alpamayo_verify", 1, 17)])
def test_verify_writes_only_its_outputs_and_workspace(name, B, blk):
    """blk 17 at four query heads per kv head runs on the 128-row form, whose
    workspace rows per piece slot differ."""
    w = synth.WORKLOADS[name].with_(C=B, blk=blk)
    pair = Pair(w, "guardv", watch=[])
    pair.fill()
    pair.set_tail(w.tail_len)
    q, k, v = (to_dev(x) for x in synth.verify_block(w, "guardv"))
    tgt, drf, planted = synth.planted_ids(B, w.blk, "guardv")
    tgt, drf = torch.from_numpy(tgt).cuda(), torch.from_numpy(drf).cuda()
    tail = torch.full((B,), w.tail_len, dtype=torch.int32, device="cuda")
    ws_n = max(16, skv.skv_verify_workspace_bytes(pair.cache, w.Hq, w.blk))
    ws_g = Guarded((ws_n,), torch.uint8)       # the workspace itself starts zeroed
    out_g = Guarded(q.shape, torch.bfloat16)
    acc_g, nxt_g = Guarded((B,), torch.int32), Guarded((B,), torch.int32)
    for _ in range(2):                         # the workspace is reused as the call leaves it
        skv.stream_attn_verify(pair.cache, tail, q, k, v, w.sm_scale, target_ids=tgt, draft_ids=drf,
                               ws=ws_g.t, out=out_g.t, accept_len=acc_g.t, next_token=nxt_g.t)
        out_p, acc_p, nxt_p = skv.stream_attn_verify(pair.cache, tail, q, k, v, w.sm_scale,
                                                     target_ids=tgt, draft_ids=drf)
        torch.cuda.synchronize()
        _check_out(out_g, out_p, "verify out")
        _check_out(acc_g, acc_p, "accept_len")
        _check_out(nxt_g, nxt_p, "next_token")
        assert ws_g.guards_intact(), "verify workspace: a guard band was written"
        np.testing.assert_array_equal(acc_g.t.cpu().numpy(), planted)
    assert pair.cache.device_status() == 0


def test_fused_insert_prefill_writes_only_its_outputs():
    """The fused insert + prefill on two caches filled alike: one writes into
    guarded output and LSE buffers, the other into plain ones; the guards
    hold, every element is written, and both give the same bits."""
    w = synth.WORKLOADS["alpamayo_step"].with_(C=2)
    pa, pb = Pair(w, "guardf", watch=[]), Pair(w, "guardf", watch=[])
    pa.fill()
    pb.fill()
    k, v = (to_dev(x) for x in synth.frame_kv(w, pa.n_inserts, "guardf"))
    q = to_dev(synth.frame_q(w, pa.n_inserts, "guardf"))
    out_g, lse_g = Guarded(q.shape, torch.bfloat16), Guarded((w.C, w.Hq, w.n_new), torch.float32)
    skv.stream_attn_prefill_insert(pa.cache, k, v, q, w.sm_scale, out=out_g.t, lse=lse_g.t)
    out_p, lse_p = skv.stream_attn_prefill_insert(pb.cache, k, v, q, w.sm_scale, lse=True)
    torch.cuda.synchronize()
    _check_out(out_g, out_p, "fused prefill out")
    _check_out(lse_g, lse_p, "fused prefill lse")
    assert torch.equal(pa.cache.k, pb.cache.k) and torch.equal(pa.cache.vt, pb.cache.vt)
    assert torch.equal(pa.cache.head, pb.cache.head)
    assert pa.cache.device_status() == 0 and pb.cache.device_status() == 0
