"""Pins for the oracle: closed forms, invariants, brute force, a library SDPA
and the pages' worked examples.  Each pin is chosen so that a plausible slip
in the oracle (a dropped term, a wrong sign or index, a transposed operand)
fails at least one of them.  CPU only."""
import cmath
import json
import math
import os

import numpy as np
import pytest

from oracle import skv_oracle as O
from streaming_kv_cache_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _bits(shape, seed, scale=1.0):
    return synth.normal_bf16(shape, "pin", seed, scale=scale)


# --------------------------------------------------------------------------
# number format

def test_bf16_widening_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0001, 0x7F7F, 0x8000], np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 2.0 ** -133, (2 - 2.0 ** -7) * 2.0 ** 127, -0.0]
    got = O.bf16_to_f64(bits)
    assert got.dtype == np.float64
    assert list(got) == want


def test_generator_rounds_to_nearest_even():
    # 1 + 2^-8 is a tie between 1 and 1+2^-7 -> even (1.0); 1 + 3*2^-9 rounds up.
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -9, 1 + 2.0 ** -7 + 2.0 ** -8], np.float32)
    b = synth.f32_to_bf16_bits(x)
    assert list(O.bf16_to_f64(b)) == [1.0, 1 + 2.0 ** -7, 1 + 2.0 ** -6]


# --------------------------------------------------------------------------
# RoPE

def test_rope_identity_at_position_zero():
    x = O.bf16_to_f64(_bits((5, 64), 1))
    np.testing.assert_array_equal(O.rope_rotate(x, np.zeros(5), 1e4), x)


def test_rope_hand_values_d4():
    # d=4, theta=16: pair 0 turns at rate 16^0 = 1, pair 1 at 16^(-2/4) = 1/4.
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    y = O.rope_rotate(x, np.array([4]), 16.0)[0]
    a0, a1 = 4.0, 1.0
    want = [1 * math.cos(a0) - 3 * math.sin(a0), 2 * math.cos(a1) - 4 * math.sin(a1),
            3 * math.cos(a0) + 1 * math.sin(a0), 4 * math.cos(a1) + 2 * math.sin(a1)]
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-14)


def test_rope_d2_is_complex_rotation():
    # d = 2: the one pair turns by angle = position (theta^0 = 1).
    x = np.array([[0.3, -1.7]] * 4)
    pos = np.array([0, 1, 7, 12345])
    y = O.rope_rotate(x, pos, 1e6)
    for i, p in enumerate(pos):
        z = complex(0.3, -1.7) * cmath.exp(1j * p)
        assert abs(y[i, 0] - z.real) < 1e-12 and abs(y[i, 1] - z.imag) < 1e-12


def test_rope_preserves_pair_norms():
    x = O.bf16_to_f64(_bits((7, 128), 2))
    pos = np.array([0, 3, 179, 3135, 3160, 12799, 99999])
    y = O.rope_rotate(x, pos, 1e6)
    n0 = x[:, :64] ** 2 + x[:, 64:] ** 2
    n1 = y[:, :64] ** 2 + y[:, 64:] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12, atol=1e-12)


def test_rope_relativity():
    # <R(m) q, R(n) k> depends on m - n only.
    q = O.bf16_to_f64(_bits((1, 64), 3))
    k = O.bf16_to_f64(_bits((1, 64), 4))
    for m, n in [(10, 3), (3135, 256), (700, 700)]:
        base = float((O.rope_rotate(q, [m], 1e4) @ O.rope_rotate(k, [n], 1e4).T)[0, 0])
        for c in (1, 97, 5000):
            sh = float((O.rope_rotate(q, [m + c], 1e4) @ O.rope_rotate(k, [n + c], 1e4).T)[0, 0])
            assert abs(sh - base) < 1e-9 * max(1.0, abs(base))


# --------------------------------------------------------------------------
# attention core

def _brute_attention(q, qp, k, v, kp, theta, scale):
    """Scalar triple loop; RoPE through complex numbers."""
    n, Hq, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    half = d // 2

    def rot(vec, p):
        out = [0.0] * d
        for i in range(half):
            z = complex(vec[i], vec[i + half]) * cmath.exp(1j * p * theta ** (-2.0 * i / d))
            out[i], out[i + half] = z.real, z.imag
        return out

    res = np.zeros((n, Hq, d))
    for a in range(n):
        for h in range(Hq):
            qa = rot(list(q[a, h]), qp[a])
            scores = []
            for b in range(k.shape[0]):
                if kp[b] <= qp[a]:
                    kb = rot(list(k[b, h // G]), kp[b])
                    scores.append((sum(x * y for x, y in zip(qa, kb)) * scale, b))
            mx = max(s for s, _ in scores)
            w = [(math.exp(s - mx), b) for s, b in scores]
            tot = sum(x for x, _ in w)
            for x, b in w:
                for j in range(d):
                    res[a, h, j] += x / tot * v[b, h // G, j]
    return res


def test_attention_matches_brute_force_tiny():
    Hq, Hkv, d, N = 4, 2, 8, 11
    qb, kb, vb = _bits((3, Hq, d), 5), _bits((N, Hkv, d), 6), _bits((N, Hkv, d), 7)
    qp = np.array([4, 7, 10])
    kp = np.arange(N)
    got, _ = O.attention_rows(qb, qp, kb, vb, kp, 100.0, 0.35)
    want = _brute_attention(O.bf16_to_f64(qb), qp, O.bf16_to_f64(kb), O.bf16_to_f64(vb), kp,
                            100.0, 0.35)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_attention_rows_sum_to_one_and_uniform_v():
    Hq, Hkv, d, N = 4, 2, 16, 40
    qb, kb = _bits((6, Hq, d), 8), _bits((N, Hkv, d), 9)
    ones = np.full((N, Hkv, d), 0x3F80, np.uint16)  # every value 1.0
    out, _ = O.attention_rows(qb, np.arange(6) * 7, kb, ones, np.arange(N), 1e4, 0.25)
    np.testing.assert_allclose(out, 1.0, rtol=0, atol=1e-12)
    one_v = _bits((1, Hkv, d), 10)
    vb = np.repeat(one_v, N, axis=0)
    out, _ = O.attention_rows(qb, np.arange(6) * 7, kb, vb, np.arange(N), 1e4, 0.25)
    want = O.bf16_to_f64(one_v)[0][np.arange(Hq) // 2]
    np.testing.assert_allclose(out, np.broadcast_to(want, out.shape), rtol=1e-12, atol=1e-12)


def test_attention_single_dominant_key():
    # With zero RoPE influence (all positions 0 -> all visible) and q = 40*k_j,
    # the softmax is dominated by key j.
    d, N = 16, 9
    kb = _bits((N, 1, d), 11)
    k = O.bf16_to_f64(kb)
    j = 5
    q = synth.f32_to_bf16_bits((40 * k[j]).astype(np.float32)[None])
    vb = _bits((N, 1, d), 12)
    out, _ = O.attention_rows(q, [0], kb, vb, np.zeros(N, int), 1e4, 1.0)
    np.testing.assert_allclose(out[0, 0], O.bf16_to_f64(vb)[j, 0], atol=1e-6)


def test_lse_is_log_sum_exp():
    d, N = 8, 5
    qb, kb, vb = _bits((1, 1, d), 13), _bits((N, 1, d), 14), _bits((N, 1, d), 15)
    _, lse = O.attention_rows(qb, [N - 1], kb, vb, np.arange(N), 1e4, 0.5)
    q = O.rope_rotate(O.bf16_to_f64(qb)[:, 0], [N - 1], 1e4)[0]
    kr = O.rope_rotate(O.bf16_to_f64(kb)[:, 0], np.arange(N), 1e4)
    want = math.log(sum(math.exp(0.5 * float(q @ kr[i])) for i in range(N)))
    assert abs(lse[0, 0] - want) < 1e-12


def test_masked_keys_do_not_matter():
    Hq, Hkv, d, N = 2, 1, 16, 30
    qb, kb, vb = _bits((4, Hq, d), 16), _bits((N, Hkv, d), 17), _bits((N, Hkv, d), 18)
    qp = np.array([3, 10, 11, 20])
    a, _ = O.attention_rows(qb, qp, kb, vb, np.arange(N), 1e4, 0.3)
    kb2, vb2 = kb.copy(), vb.copy()
    kb2[21:] = _bits((N - 21, Hkv, d), 19)
    vb2[21:] = _bits((N - 21, Hkv, d), 20)
    b, _ = O.attention_rows(qb, qp, kb2, vb2, np.arange(N), 1e4, 0.3)
    np.testing.assert_array_equal(a, b)
    # a key that IS visible does matter
    vb2[2] = synth.f32_to_bf16_bits(O.bf16_to_f64(vb2[2]).astype(np.float32) + 1.0)
    c, _ = O.attention_rows(qb, qp, kb2, vb2, np.arange(N), 1e4, 0.3)
    assert np.abs(c - a).max() > 1e-6


def _rope_complex(x, pos, theta):
    d = x.shape[-1]
    half = d // 2
    z = x[..., :half] + 1j * x[..., half:]
    w = np.exp(1j * np.asarray(pos, float)[:, None] * theta ** (-np.arange(half) * 2.0 / d))
    zr = z * w
    return np.concatenate([zr.real, zr.imag], axis=-1)


def _sdpa(qr, kr, v, mask, scale):
    """torch SDPA in fp64 on CPU: qr [n][Hq][d], kr/v [N][Hkv][d], mask [n][N]."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as Fn
    q = torch.from_numpy(np.ascontiguousarray(np.transpose(qr, (1, 0, 2))))[None]
    k = torch.from_numpy(np.ascontiguousarray(np.transpose(kr, (1, 0, 2))))[None]
    vv = torch.from_numpy(np.ascontiguousarray(np.transpose(v, (1, 0, 2))))[None]
    m = torch.from_numpy(mask)[None, None]
    o = Fn.scaled_dot_product_attention(q, k, vv, attn_mask=m, scale=scale, enable_gqa=True)
    return np.transpose(o[0].numpy(), (1, 0, 2))


def test_attention_vs_torch_sdpa_gqa():
    Hq, Hkv, d, N = 8, 2, 32, 70
    qb, kb, vb = _bits((9, Hq, d), 21), _bits((N, Hkv, d), 22), _bits((N, Hkv, d), 23)
    qp = np.array([0, 5, 17, 30, 31, 44, 60, 68, 69])
    kp = np.arange(N)
    got, _ = O.attention_rows(qb, qp, kb, vb, kp, 1e4, 0.2)
    qr = np.stack([_rope_complex(O.bf16_to_f64(qb)[:, h], qp, 1e4) for h in range(Hq)], 1)
    kr = np.stack([_rope_complex(O.bf16_to_f64(kb)[:, h], kp, 1e4) for h in range(Hkv)], 1)
    want = _sdpa(qr, kr, O.bf16_to_f64(vb), kp[None, :] <= qp[:, None], 0.2)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def test_mha_is_the_gqa_special_case():
    d, N = 16, 12
    qb, kb, vb = _bits((3, 2, d), 24), _bits((N, 1, d), 25), _bits((N, 1, d), 26)
    qp = [4, 8, 11]
    gqa, _ = O.attention_rows(qb, qp, kb, vb, np.arange(N), 1e4, 0.3)
    mha, _ = O.attention_rows(qb, qp, np.repeat(kb, 2, 1), np.repeat(vb, 2, 1),
                              np.arange(N), 1e4, 0.3)
    np.testing.assert_array_equal(gqa, mha)


# --------------------------------------------------------------------------
# window, ring and ordering

def _label_window(P, V, F, T):
    """A window whose K carries readable labels: K[...,0] = view, [...,1] =
    the frame's insert number, [...,2] = token; prefix tokens carry -1."""
    def enc(vals):
        return synth.f32_to_bf16_bits(np.asarray(vals, np.float32))
    pk = np.zeros((P, 1, 4), np.float32)
    pk[:, 0, :] = [-1, -1, -1, 0]
    win = O.StreamWindow(P, V, F, T, 1, 4, enc(pk), enc(pk))
    return win, enc


def _insert_labelled(win, enc, n):
    V, T = win.V, win.T
    k = np.zeros((V, T, 1, 4), np.float32)
    for v in range(V):
        for t in range(T):
            k[v, t, 0] = [v, n, t, 0]
    win.insert(enc(k), enc(k))


def test_view_major_order_matches_page_listing():
    g = _gold("view_major_order.json")
    V, F, T, P = g["views"], g["frames"], 2, 1
    win, enc = _label_window(P, V, F, T)
    for n in range(F):
        _insert_labelled(win, enc, n)
    k, _ = win.logical_kv(with_tail=False)
    lab = O.bf16_to_f64(k)[:, 0, :3]
    got = ["sys"]
    for row in range(P, k.shape[0], T):
        v, f, _ = lab[row]
        got.append("Camera %d: f%d" % (v + 1, f))
    got.append("tail")
    assert got == g["order"]
    # the new frame of view v sits in that view's last slot, not at the end
    for v in range(V):
        idx = win.new_frame_index(v, 0)
        assert int(lab[idx, 0]) == v and int(lab[idx, 1]) == F - 1


def test_sliding_window_example():
    g = _gold("sliding_window.json")
    F, V = g["frames"], g["views"]
    win, enc = _label_window(1, V, F, 1)
    names = {}
    for n in range(F):                       # frames t-3 .. t
        _insert_labelled(win, enc, n)
        names[n] = g["window_t"][n]
    before = [int(f) for f in O.bf16_to_f64(win.logical_kv(False)[0])[1:1 + F, 0, 1]]
    assert [names[f] for f in before] == g["window_t"]
    _insert_labelled(win, enc, F)           # frame t+1
    names[F] = "t+1"
    for v in range(V):
        rows = O.bf16_to_f64(win.logical_kv(False)[0])[1 + v * F:1 + (v + 1) * F, 0, 1]
        assert [names[int(f)] for f in rows] == g["window_t_plus_1"]
    kept = len(set(g["window_t"]) & set(g["window_t_plus_1"])) / F
    assert kept == g["unchanged_fraction"] == (F - 1) / F
    assert g["images_per_step_before"] == V * F and g["images_new_per_step"] == V


def test_streamed_window_equals_rebuild_and_ring_closed_form():
    P, V, F, T, H, d = 3, 3, 4, 5, 2, 8
    pk, pv = _bits((P, H, d), 30), _bits((P, H, d), 31)
    frames = [(_bits((V, T, H, d), 100 + i), _bits((V, T, H, d), 200 + i)) for i in range(11)]
    win = O.StreamWindow(P, V, F, T, H, d, pk, pv)
    for i, (k, v) in enumerate(frames):
        win.insert(k, v)
        if i + 1 < F:
            continue
        fresh = O.StreamWindow(P, V, F, T, H, d, pk, pv)
        for k2, v2 in frames[i + 1 - F:i + 1]:
            fresh.insert(k2, v2)
        a, b = win.logical_kv(), fresh.logical_kv()
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])
        # a physical ring written slot-by-slot (slot = insert number mod F)
        ring_k = np.zeros((V, F, T, H, d), np.uint16)
        for j in range(i + 1):
            ring_k[:, j % F] = frames[j][0]
        head, rk, _ = win.ring_expected()
        np.testing.assert_array_equal(rk, ring_k)
        assert (head == (i + 1) % F).all()


# --------------------------------------------------------------------------
# prefill: the mask rules of the page, read off through one-hot values

def test_prefill_mask_follows_page_rules():
    """[FD-blog] 3.2 mask bullets: a newest frame sees the system tokens, the
    earlier views, its own view's history frames, and its own frame
    causally; it does not see later views."""
    P, V, F, T = 2, 3, 3, 4
    N = P + V * F * T
    d = 64 if N <= 64 else 128
    win = O.StreamWindow(P, V, F, T, 1, d, np.zeros((P, 1, d), np.uint16),
                         np.zeros((P, 1, d), np.uint16))
    for i in range(F):
        win.insert(np.zeros((V, T, 1, d), np.uint16), np.zeros((V, T, 1, d), np.uint16))
    # value of logical key j = one-hot e_j; all keys equal -> weights uniform on visible set
    onehot = np.zeros((N, 1, d), np.float32)
    onehot[np.arange(N), 0, np.arange(N)] = 1.0
    vb = synth.f32_to_bf16_bits(onehot)
    win.prefix_v = vb[:P]
    r = P
    for dq in win.views:
        for f in range(len(dq)):
            dq[f] = (dq[f][0], vb[r:r + T])
            r += T
    q = np.zeros((V * T, 1, d), np.uint16)
    out, _ = O.stream_prefill(win, q, 1e4, 1.0)
    for j in range(V * T):
        vq, tq = divmod(j, T)
        seen = set(np.nonzero(out[j, 0, :N] > 0)[0].tolist())
        want = set(range(P))                                         # system tokens
        for v in range(V):
            for f in range(F):
                for t in range(T):
                    key = P + v * F * T + f * T + t
                    if v < vq:                                       # earlier views
                        want.add(key)
                    elif v == vq and f < F - 1:                      # own history frames
                        want.add(key)
                    elif v == vq and f == F - 1 and t <= tq:         # own frame, causal
                        want.add(key)
        assert seen == want, j
        np.testing.assert_allclose(out[j, 0, sorted(want)], 1.0 / len(want), rtol=1e-12)


def _tiny_window(w, n_inserts, tag):
    pk, pv = synth.prefix_kv(w, tag)
    win = O.StreamWindow(w.P, w.V, w.F, w.T, w.Hkv, w.d, pk[0], pv[0])
    for i in range(n_inserts):
        k, v = synth.frame_kv(w, i, tag)
        win.insert(k[0], v[0])
    return win


def _full_sequence_sdpa(win, q_rows, q_pos, extra_k=None, extra_v=None, scale=1.0, theta=1e4):
    k, v = win.logical_kv(with_tail=True)
    if extra_k is not None:
        k = np.concatenate([k, extra_k])
        v = np.concatenate([v, extra_v])
    kp = np.arange(k.shape[0])
    kf, vf, qf = O.bf16_to_f64(k), O.bf16_to_f64(v), O.bf16_to_f64(q_rows)
    kr = np.stack([_rope_complex(kf[:, h], kp, theta) for h in range(kf.shape[1])], 1)
    qr = np.stack([_rope_complex(qf[:, h], q_pos, theta) for h in range(qf.shape[1])], 1)
    return _sdpa(qr, kr, vf, kp[None, :] <= np.asarray(q_pos)[:, None], scale)


def test_prefill_tiny_vs_sdpa_on_full_window():
    w = synth.WORKLOADS["tiny"]
    win = _tiny_window(w, w.F + 2, "sdpa")
    q = synth.frame_q(w, w.F + 1, "sdpa")[0]
    got, _ = O.stream_prefill(win, q, w.theta, w.sm_scale)
    # queries placed at the rows of each view's newest frame in the listing
    q_pos = [w.P + v * w.F * w.T + (w.F - 1) * w.T + t for v in range(w.V) for t in range(w.T)]
    want = _full_sequence_sdpa(win, q, q_pos, scale=w.sm_scale, theta=w.theta)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def test_prefill_row_subset_equals_full():
    w = synth.WORKLOADS["tiny"]
    win = _tiny_window(w, w.F, "rows")
    q = synth.frame_q(w, w.F - 1, "rows")[0]
    full, lf = O.stream_prefill(win, q, w.theta, w.sm_scale)
    rows = np.array([0, 5, 17, 31])
    part, lp = O.stream_prefill(win, q, w.theta, w.sm_scale, rows=rows)
    # equal up to BLAS blocking of the row count
    np.testing.assert_allclose(part, full[rows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lp, lf[rows], rtol=1e-13, atol=1e-14)


def test_tail_is_invisible_to_prefill():
    w = synth.WORKLOADS["tiny"]
    win = _tiny_window(w, w.F, "tail")
    q = synth.frame_q(w, w.F - 1, "tail")[0]
    a, _ = O.stream_prefill(win, q, w.theta, w.sm_scale)
    tk, tv = synth.tail_kv(w, 5, "tail")
    win.set_tail(tk[0], tv[0])
    b, _ = O.stream_prefill(win, q, w.theta, w.sm_scale)
    np.testing.assert_array_equal(a, b)


# --------------------------------------------------------------------------
# verify

def test_verify_vs_sdpa_with_tail():
    w = synth.WORKLOADS["tiny"].with_(blk=9)
    win = _tiny_window(w, w.F + 1, "ver")
    tk, tv = synth.tail_kv(w, 6, "ver")
    win.set_tail(tk[0], tv[0])
    q, k, v = (x[0] for x in synth.verify_block(w, "ver"))
    got, _ = O.stream_verify(win, q, k, v, w.theta, w.sm_scale)
    base = win.n_visual + 6
    want = _full_sequence_sdpa(win, q, base + np.arange(9), k, v, w.sm_scale, w.theta)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def test_verify_block_of_one_is_plain_decode():
    """A one-token block is decoding: the last token attends every key, so
    the mask drops out and an unmasked SDPA gives the answer."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as Fn
    w = synth.WORKLOADS["tiny"].with_(blk=1)
    win = _tiny_window(w, w.F, "dec")
    tk, tv = synth.tail_kv(w, 3, "dec")
    win.set_tail(tk[0], tv[0])
    q, k, v = (x[0] for x in synth.verify_block(w, "dec"))
    got, _ = O.stream_verify(win, q, k, v, w.theta, w.sm_scale)
    kk, vv = win.logical_kv()
    kk, vv = np.concatenate([kk, k]), np.concatenate([vv, v])
    pos = np.arange(kk.shape[0])
    kr = np.stack([_rope_complex(O.bf16_to_f64(kk)[:, h], pos, w.theta) for h in range(w.Hkv)], 1)
    qr = np.stack([_rope_complex(O.bf16_to_f64(q)[:, h], [pos[-1]], w.theta) for h in range(w.Hq)], 1)
    o = Fn.scaled_dot_product_attention(
        torch.from_numpy(np.transpose(qr, (1, 0, 2)).copy())[None],
        torch.from_numpy(np.transpose(kr, (1, 0, 2)).copy())[None],
        torch.from_numpy(np.transpose(O.bf16_to_f64(vv), (1, 0, 2)).copy())[None],
        scale=w.sm_scale, enable_gqa=True)
    np.testing.assert_allclose(got, np.transpose(o[0].numpy(), (1, 0, 2)), rtol=1e-10, atol=1e-12)


def test_verify_rows_are_causal_within_block():
    w = synth.WORKLOADS["tiny"].with_(blk=9)
    win = _tiny_window(w, w.F, "caus")
    q, k, v = (x[0] for x in synth.verify_block(w, "caus"))
    a, _ = O.stream_verify(win, q, k, v, w.theta, w.sm_scale)
    k2, v2 = k.copy(), v.copy()
    k2[5:] ^= np.uint16(0x0040)
    v2[5:] ^= np.uint16(0x0040)
    b, _ = O.stream_verify(win, q, k2, v2, w.theta, w.sm_scale)
    np.testing.assert_array_equal(a[:5], b[:5])
    assert np.abs(a[5:] - b[5:]).max() > 0


# --------------------------------------------------------------------------
# the whole window as queries (first window) and tail tokens as queries

def _causal_sdpa(q_bits, k_bits, v_bits, theta, scale):
    """torch SDPA fp64 with its own causal mask (is_causal): query i sees keys
    0..i of a sequence whose positions are 0..N-1."""
    torch = pytest.importorskip("torch")
    import torch.nn.functional as Fn
    pos = np.arange(k_bits.shape[0])
    qf, kf, vf = O.bf16_to_f64(q_bits), O.bf16_to_f64(k_bits), O.bf16_to_f64(v_bits)
    qr = np.stack([_rope_complex(qf[:, h], pos, theta) for h in range(qf.shape[1])], 0)
    kr = np.stack([_rope_complex(kf[:, h], pos, theta) for h in range(kf.shape[1])], 0)
    vr = np.transpose(vf, (1, 0, 2))
    o = Fn.scaled_dot_product_attention(torch.from_numpy(qr)[None], torch.from_numpy(kr)[None],
                                        torch.from_numpy(np.ascontiguousarray(vr))[None],
                                        is_causal=True, scale=scale, enable_gqa=True)
    return np.transpose(o[0].numpy(), (1, 0, 2))


@pytest.mark.parametrize("n_inserts", [2, 5])
def test_window_is_causal_attention_over_the_listing(n_inserts):
    """First window (n_inserts = F) and a rotated ring (F + 3): every token a
    query is plain causal attention over the logical sequence."""
    w = synth.WORKLOADS["tiny"]
    win = _tiny_window(w, n_inserts, "win%d" % n_inserts)
    q = synth.normal_bf16((win.n_visual, w.Hq, w.d), "winq", n_inserts)
    got, lse = O.stream_window(win, q, w.theta, w.sm_scale)
    k, v = win.logical_kv(with_tail=False)
    want = _causal_sdpa(q, k, v, w.theta, w.sm_scale)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)
    assert got.shape == (win.n_visual, w.Hq, w.d) and lse.shape == (win.n_visual, w.Hq)


def test_window_first_token_sees_only_itself():
    """Token 0 has a single visible key, so its output is that key's value
    exactly and its LSE is its own scaled score."""
    w = synth.WORKLOADS["tiny"]
    win = _tiny_window(w, w.F, "one")
    q = synth.normal_bf16((win.n_visual, w.Hq, w.d), "oneq")
    got, lse = O.stream_window(win, q, w.theta, w.sm_scale, rows=np.array([0]))
    G = w.Hq // w.Hkv
    v0 = O.bf16_to_f64(win.prefix_v[0])
    for h in range(w.Hq):
        np.testing.assert_array_equal(got[0, h], v0[h // G])
        s = float(O.bf16_to_f64(q[0, h]) @ O.bf16_to_f64(win.prefix_k[0, h // G])) * w.sm_scale
        assert abs(lse[0, h] - s) < 1e-12     # position 0: the rotation is the identity


def test_window_newest_frame_rows_equal_prefill():
    """The window's rows of each view's newest frame are the streaming
    prefill's rows: same positions, same visible keys."""
    w = synth.WORKLOADS["tiny"]
    win = _tiny_window(w, w.F + 1, "same")
    qn = synth.frame_q(w, w.F, "same")[0]
    q = synth.normal_bf16((win.n_visual, w.Hq, w.d), "sameq")
    rows = np.array([win.new_frame_index(v, t) for v in range(w.V) for t in range(w.T)])
    q[rows] = qn
    a, la = O.stream_window(win, q, w.theta, w.sm_scale, rows=rows)
    b, lb = O.stream_prefill(win, qn, w.theta, w.sm_scale)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(la, lb, rtol=1e-13, atol=1e-14)


def test_window_earlier_tokens_ignore_later_frames():
    """Changing view 1's newest frame leaves every token before it unchanged,
    bit for bit, and changes that frame's own rows."""
    w = synth.WORKLOADS["tiny"]
    win_a = _tiny_window(w, w.F, "late")
    win_b = _tiny_window(w, w.F, "late")
    k, v = win_b.views[1][-1]
    win_b.views[1][-1] = (k ^ np.uint16(0x0040), v ^ np.uint16(0x0040))
    q = synth.normal_bf16((win_a.n_visual, w.Hq, w.d), "lateq")
    a, _ = O.stream_window(win_a, q, w.theta, w.sm_scale)
    b, _ = O.stream_window(win_b, q, w.theta, w.sm_scale)
    first = win_a.new_frame_index(1, 0)
    np.testing.assert_array_equal(a[:first], b[:first])
    assert np.abs(a[first:] - b[first:]).max() > 0


def test_tail_prefill_vs_sdpa():
    w = synth.WORKLOADS["tiny"]
    win = _tiny_window(w, w.F + 2, "tp")
    tk, tv = synth.tail_kv(w, 4, "tp")
    win.set_tail(tk[0], tv[0])
    n = 11
    q = synth.normal_bf16((n, w.Hq, w.d), "tpq")
    k = synth.normal_bf16((n, w.Hkv, w.d), "tpk")
    v = synth.normal_bf16((n, w.Hkv, w.d), "tpv")
    got, _ = O.stream_prefill_tail(win, q, k, v, w.theta, w.sm_scale)
    base = win.n_visual + 4
    want = _full_sequence_sdpa(win, q, base + np.arange(n), k, v, w.sm_scale, w.theta)
    np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)


def test_tail_prefill_at_once_equals_token_by_token():
    """Causal within the span: n tokens in one call give the rows that n
    one-token calls give when each call's K/V is appended to the tail before
    the next."""
    w = synth.WORKLOADS["tiny"]
    win = _tiny_window(w, w.F, "inc")
    n = 6
    q = synth.normal_bf16((n, w.Hq, w.d), "incq")
    k = synth.normal_bf16((n, w.Hkv, w.d), "inck")
    v = synth.normal_bf16((n, w.Hkv, w.d), "incv")
    whole, lw = O.stream_prefill_tail(win, q, k, v, w.theta, w.sm_scale)
    for j in range(n):
        one, lo = O.stream_prefill_tail(win, q[j:j + 1], k[j:j + 1], v[j:j + 1], w.theta, w.sm_scale)
        np.testing.assert_allclose(one[0], whole[j], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lo[0], lw[j], rtol=1e-12, atol=1e-13)
        win.set_tail(np.concatenate([win.tail_k, k[j:j + 1]]), np.concatenate([win.tail_v, v[j:j + 1]]))


# --------------------------------------------------------------------------
# accept length

def test_accept_page_example():
    g = _gold("accept_example.json")
    words = {}

    def tok(s):
        return words.setdefault(s, len(words))

    draft = [tok(g["anchor"])] + [tok(s) for s in g["draft"]]
    n = g["target_agrees_first"]
    target = [tok(s) for s in g["draft"][:n]] + [tok(g["target_at_7"])]
    target += [tok("<t%d>" % i) for i in range(len(draft) - len(target))]
    k, nxt = O.accept_length(target, draft)
    assert k == g["expected_accept_len"] == 6
    assert nxt == tok(g["target_at_7"])


def test_accept_vflash_block_of_16():
    g = _gold("accept_example.json")
    blk = g["vflash_block"]
    target = list(range(100, 100 + blk))
    for k_plant in (0, 7, 15):
        draft = [1] + [target[i - 1] if i <= k_plant else 9999 for i in range(1, blk)]
        assert O.accept_length(target, draft) == (k_plant, target[k_plant])


def test_accept_planted_prefixes():
    target, draft, k = synth.planted_ids(64, 9, "pin")
    for b in range(64):
        got, nxt = O.accept_length(target[b], draft[b])
        assert got == k[b] and nxt == target[b, k[b]]


def test_accept_extremes():
    t = [5, 6, 7, 8, 9, 10, 11, 12, 13]
    assert O.accept_length(t, [0] + t[:8]) == (8, 13)       # all drafts accepted: bonus token
    assert O.accept_length(t, [0, 4] + t[1:8]) == (0, 5)    # first draft rejected
    assert O.accept_length(t, [t[0]] * 9) == (1, 6)         # slot 0 is never compared


# --------------------------------------------------------------------------
# multi-section rotary (a stated reading: position triples (t, h, w), the
# frequencies dealt to the components in turn)

def test_mrope_sections_are_dealt_in_turn():
    sec = O.interleaved_sections(128, 20, 20)
    assert len(sec) == 64
    assert list(sec[:9]) == [0, 1, 2, 0, 1, 2, 0, 1, 2]
    assert list(sec[60:]) == [0, 0, 0, 0]           # h and w shares used up: the rest is t
    assert (sec == 1).sum() == 20 and (sec == 2).sum() == 20 and (sec == 0).sum() == 24
    assert list(O.interleaved_sections(8, 1, 0)) == [0, 1, 0, 0]


def test_mrope_triples_of_a_small_geometry():
    """P=8, two views of two frames of 16 tokens in rows of 4: hand-listed."""
    m = O.MRope(8, 2, 2, 16, 4, O.interleaved_sections(8, 1, 1))
    want = {0: (0, 0, 0), 7: (7, 7, 7),              # prefix: t = h = w = n
            8: (8, 8, 8),                           # view 0, frame 0, token 0
            13: (8, 9, 9),                          # token 5: row 1, column 1
            35: (24, 26, 27),                       # frame 1 starts at 24; token 11: row 2, column 3
            40: (40, 40, 40),                       # view 1, frame 0, token 0
            71: (56, 59, 59),                       # last window token: frame at 56, token 15
            72: (72, 72, 72), 80: (80, 80, 80)}     # the tail after the window
    got = m.triples(list(want))
    for (n, tr), g in zip(want.items(), got):
        assert tuple(g) == tr, n


def test_mrope_equal_components_are_the_1d_rotation_bit_for_bit():
    x = O.bf16_to_f64(_bits((2, 7, 64), 30))
    pos = np.array([0, 1, 5, 99, 1000, 3137, 12799])
    sec = O.interleaved_sections(64, 10, 10)
    got = O.rope_rotate_sections(x, np.stack([pos, pos, pos], 1), 1e6, sec)
    assert np.array_equal(got, O.rope_rotate(x, pos, 1e6))


def test_mrope_hand_values():
    """d = 6: three frequencies, one per component (t, h, w).  A unit vector
    along pair i turns by the angle p_{sec(i)} * 16^(-2i/6)."""
    sec = O.interleaved_sections(6, 1, 1)
    assert list(sec) == [0, 1, 2]
    tr = np.array([[2, 5, 7]])
    for i in range(3):
        x = np.zeros((1, 6))
        x[0, i] = 1.0
        y = O.rope_rotate_sections(x, tr, 16.0, sec)[0]
        a = tr[0, i] * 16.0 ** (-2.0 * i / 6)
        want = np.zeros(6)
        want[i], want[i + 3] = math.cos(a), math.sin(a)
        np.testing.assert_allclose(y, want, atol=1e-15)


def test_mrope_a_component_moves_only_its_frequencies():
    x = O.bf16_to_f64(_bits((1, 64), 31))
    sec = O.interleaved_sections(64, 10, 10)
    a = O.rope_rotate_sections(x, np.array([[40, 43, 45]]), 1e4, sec)[0]
    b = O.rope_rotate_sections(x, np.array([[40, 43, 46]]), 1e4, sec)[0]     # only w moved
    moved = np.abs(a - b) > 1e-12
    pair = np.concatenate([sec, sec]) == 2
    assert moved[pair].all() and not moved[~pair].any()


def test_mrope_is_relative_in_every_component():
    """Shifting both triples by the same (c_t, c_h, c_w) leaves the score."""
    q = O.bf16_to_f64(_bits((1, 64), 32))
    k = O.bf16_to_f64(_bits((1, 64), 33))
    sec = O.interleaved_sections(64, 10, 10)
    m, n = np.array([[300, 304, 311]]), np.array([[120, 121, 129]])
    base = float((O.rope_rotate_sections(q, m, 1e4, sec) @ O.rope_rotate_sections(k, n, 1e4, sec).T)[0, 0])
    for c in ([5, 0, 0], [0, 9, 0], [0, 0, 3], [7, 2, 11]):
        c = np.array([c])
        sh = float((O.rope_rotate_sections(q, m + c, 1e4, sec) @ O.rope_rotate_sections(k, n + c, 1e4, sec).T)[0, 0])
        assert abs(sh - base) < 1e-9 * max(1.0, abs(base))


def _brute_attention_mrope(q, qt, k, v, kt, q_idx, k_idx, sec, theta, scale):
    """Scalar loop over rows, heads and keys; each frequency turns its pair
    through a complex multiplication by its component of the triple; the
    mask is on logical indices."""
    n, Hq, d = q.shape
    G = Hq // k.shape[1]
    half = d // 2

    def rot(vec, tr):
        out = [0.0] * d
        for i in range(half):
            z = complex(vec[i], vec[i + half]) * cmath.exp(1j * tr[sec[i]] * theta ** (-2.0 * i / d))
            out[i], out[i + half] = z.real, z.imag
        return out

    res = np.zeros((n, Hq, d))
    for a in range(n):
        for h in range(Hq):
            qa = rot(list(q[a, h]), qt[a])
            scores = [(sum(x * y for x, y in zip(qa, rot(list(k[b, h // G]), kt[b]))) * scale, b)
                      for b in range(k.shape[0]) if k_idx[b] <= q_idx[a]]
            mx = max(s for s, _ in scores)
            w = [(math.exp(s - mx), b) for s, b in scores]
            tot = sum(x for x, _ in w)
            for x, b in w:
                res[a, h] += x / tot * v[b, h // G]
    return res


def test_mrope_attention_matches_brute_force():
    """Attention with the multi-section rotation over a small window: prefix
    of 3, two views of two frames of 6 tokens in rows of 3, two tail tokens."""
    m = O.MRope(3, 2, 2, 6, 3, O.interleaved_sections(8, 1, 1))
    N = 3 + 2 * 2 * 6 + 2
    qb, kb, vb = _bits((4, 4, 8), 34), _bits((N, 2, 8), 35), _bits((N, 2, 8), 36)
    q_idx = np.array([4, 13, 26, 28])
    k_idx = np.arange(N)
    got, _ = O.attention_rows(qb, q_idx, kb, vb, k_idx, 50.0, 0.4, mrope=m)
    want = _brute_attention_mrope(O.bf16_to_f64(qb), m.triples(q_idx), O.bf16_to_f64(kb), O.bf16_to_f64(vb),
                                  m.triples(k_idx), q_idx, k_idx, m.sec, 50.0, 0.4)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)
    # and it is not the 1-D rotation
    one_d, _ = O.attention_rows(qb, q_idx, kb, vb, k_idx, 50.0, 0.4)
    assert np.abs(one_d - got).max() > 1e-3
