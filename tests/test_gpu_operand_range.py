"""Range of the rotated operands.

The attention kernels rotate Q and K in fp32 and hand the tensor cores fp16
values, whose largest finite magnitude is 65504.  The header states the
behaviour: a rotated component beyond that is clamped to +-65504 (no status
bit), and inputs whose components all lie within +-46000 never reach the
clamp, because the rotation keeps the length of every (x_i, x_{i+d/2}) pair.

Inside the range the kernels must match the oracle at the usual tolerance
even with very large keys and queries (the softmax scale is applied after
the product, in fp32).  Outside it they must match the oracle's attention
computed on rotated operands clamped to +-65504.
"""
import numpy as np
import pytest
import torch

from oracle import skv_oracle as O
from streaming_kv_cache_gb300 import skv, synth

from gpu_harness import LSE_TOL, Pair, assert_close, assert_lse, bf16_dev_to_f64, to_dev

FP16_MAX = 65504.0


def attention_clamped(q_bits, q_pos, k_bits, v_bits, k_pos, theta, sm_scale, clamp):
    """The oracle's masked attention (plain fp64: rotate every key and query
    at its position, dense mask idx(k) <= idx(q), softmax, P V), with the
    rotated Q and K components clamped to [-clamp, clamp] before the
    product: the documented behaviour of the kernels outside fp16's range."""
    q = O.bf16_to_f64(q_bits)
    k = O.bf16_to_f64(k_bits)
    v = O.bf16_to_f64(v_bits)
    n, Hq, d = q.shape
    G = Hq // k.shape[1]
    qr = np.clip(O.rope_rotate(np.transpose(q, (1, 0, 2)), q_pos, theta), -clamp, clamp)
    kr = np.clip(O.rope_rotate(np.transpose(k, (1, 0, 2)), k_pos, theta), -clamp, clamp)
    vt = np.transpose(v, (1, 0, 2))
    visible = np.asarray(k_pos)[None, :] <= np.asarray(q_pos)[:, None]
    out = np.zeros((Hq, n, d))
    lse = np.zeros((Hq, n))
    for h in range(Hq):
        s = np.where(visible, (qr[h] @ kr[h // G].T) * sm_scale, -np.inf)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        out[h] = (p / l) @ vt[h // G]
        lse[h] = (m + np.log(l))[:, 0]
    return np.transpose(out, (1, 0, 2)), lse.T


def test_clamped_reference_without_clamp_is_the_oracle():
    """Pin of the reference above: with a clamp no value reaches, it is the
    oracle's attention_rows."""
    rng = np.random.default_rng(3)
    n, N, Hq, Hkv, d = 5, 23, 4, 2, 8
    bits = lambda *s: synth.f32_to_bf16_bits(rng.standard_normal(s).astype(np.float32))
    q, k, v = bits(n, Hq, d), bits(N, Hkv, d), bits(N, Hkv, d)
    q_pos = np.array([3, 9, 14, 20, 22])
    k_pos = np.arange(N)
    want = O.attention_rows(q, q_pos, k, v, k_pos, 1e4, 0.3)
    got = attention_clamped(q, q_pos, k, v, k_pos, 1e4, 0.3, np.inf)
    np.testing.assert_allclose(got[0], want[0], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got[1], want[1], rtol=1e-12, atol=1e-12)
    # and a clamp that bites changes the result
    assert np.abs(attention_clamped(q, q_pos, k, v, k_pos, 1e4, 0.3, 0.5)[0] - want[0]).max() > 1e-3


def _scaled(bits, target_max):
    """bf16 bits scaled so that the largest magnitude is target_max."""
    x = O.bf16_to_f64(bits)
    return synth.f32_to_bf16_bits((x * (target_max / np.abs(x).max())).astype(np.float32))


def _large_key_pair(tag, k_max):
    w = synth.WORKLOADS["tiny"].with_(C=2, blk=9)
    pair = Pair(w, tag)
    for i in range(w.F + 1):
        k, v = synth.frame_kv(w, i, tag)
        pair.insert(_scaled(k, k_max), v)
    return pair


@pytest.mark.gpu
@pytest.mark.parametrize("q_max", [4.0, 30000.0])
def test_large_operands_inside_the_fp16_range(q_max):
    """Keys up to +-45,000 (and queries up to +-30,000): every rotated
    component stays under 65504, so prefill and verify match the oracle at
    the usual tolerance; sm_scale brings the logits back to order one."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    k_max = 45000.0
    pair = _large_key_pair("rng_in%d" % int(q_max), k_max)
    w = pair.w
    # frame keys ~ N(0, (k_max/4)^2), queries ~ N(0, (q_max/4)^2)
    sm_scale = 1.0 / (np.sqrt(w.d) * (k_max / 4.0) * (q_max / 4.0))
    q = _scaled(synth.frame_q(w, w.F, pair.tag), q_max)
    out, lse = skv.stream_attn_prefill(pair.cache, to_dev(q), sm_scale, lse=True)
    got, got_lse = bf16_dev_to_f64(out), lse.cpu().numpy()
    for c, win in pair.win.items():
        want, wl = O.stream_prefill(win, q[c], w.theta, sm_scale)
        assert_close(got[c], want, "large operands prefill cache %d" % c)
        assert_lse(got_lse[c].T, wl, LSE_TOL)
    bq, bk, bv = synth.verify_block(w, pair.tag)
    bq = _scaled(bq, q_max)
    bk = _scaled(bk, k_max)
    tail = torch.zeros((w.C,), dtype=torch.int32, device="cuda")
    vout, _, _ = skv.stream_attn_verify(pair.cache, tail, to_dev(bq), to_dev(bk), to_dev(bv), sm_scale)
    got = bf16_dev_to_f64(vout)
    for c, win in pair.win.items():
        want, _ = O.stream_verify(win, bq[c], bk[c], bv[c], w.theta, sm_scale)
        assert_close(got[c], want, "large operands verify cache %d" % c)
    assert pair.cache.device_status() == 0


@pytest.mark.gpu
def test_keys_beyond_the_fp16_range_are_clamped():
    """Keys up to +-300,000: most rotated components pass 65504 and are
    clamped to +-65504, as the header states; prefill and verify match the
    oracle's attention on clamped rotated operands (and not the unclamped
    oracle, which shows that the clamp is what decides these results)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    k_max = 300000.0
    pair = _large_key_pair("rng_out", k_max)
    w = pair.w
    sm_scale = 1.0 / (np.sqrt(w.d) * FP16_MAX)
    q = synth.frame_q(w, w.F, pair.tag)
    out = skv.stream_attn_prefill(pair.cache, to_dev(q), sm_scale)
    got = bf16_dev_to_f64(out)
    for c, win in pair.win.items():
        kb, vb = win.logical_kv(with_tail=False)
        q_pos = np.array([win.new_frame_index(j // w.T, j % w.T) for j in range(w.n_new)])
        want, _ = attention_clamped(q[c], q_pos, kb, vb, np.arange(kb.shape[0]), w.theta, sm_scale,
                                    FP16_MAX)
        assert_close(got[c], want, "clamped prefill cache %d" % c)
        unclamped, _ = O.stream_prefill(win, q[c], w.theta, sm_scale)
        assert np.abs(unclamped - want).max() > 5e-2
    bq, bk, bv = synth.verify_block(w, pair.tag)
    bk = _scaled(bk, k_max)
    tail = torch.zeros((w.C,), dtype=torch.int32, device="cuda")
    vout, _, _ = skv.stream_attn_verify(pair.cache, tail, to_dev(bq), to_dev(bk), to_dev(bv), sm_scale)
    got = bf16_dev_to_f64(vout)
    for c, win in pair.win.items():
        kb, vb = win.logical_kv(with_tail=True)
        k_all = np.concatenate([kb, bk[c]])
        v_all = np.concatenate([vb, bv[c]])
        q_pos = kb.shape[0] + np.arange(w.blk)
        want, _ = attention_clamped(bq[c], q_pos, k_all, v_all, np.arange(k_all.shape[0]), w.theta,
                                    sm_scale, FP16_MAX)
        assert_close(got[c], want, "clamped verify cache %d" % c)
    assert pair.cache.device_status() == 0
