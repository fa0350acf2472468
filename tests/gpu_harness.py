"""Shared set-up for the GPU parity tests: drive the CUDA path through the
binding and the oracle side by side on the same seeded inputs."""
from __future__ import annotations

import os

import numpy as np
import torch

from oracle import skv_oracle as O
from streaming_kv_cache_gb300 import skv, synth

# tolerance stated for the attention outputs (bf16 in, fp32 accumulate)
MAX_ABS = 1e-2
MEAN_ABS = 1e-3
# LSE (natural log) bound, set from the measured errors: the largest seen by
# any parity test on N(0,1)-scaled inputs is 7.9e-4 (the whole window of the
# 8-heads-per-kv-head geometry; the five workloads stay under 5e-4), and the
# bound keeps a margin of about 4x over it.  Tests whose scores are k times
# larger by construction scale it by k (the fp16 rounding of the rotated
# operands moves a score in proportion to its size).
LSE_TOL = 3e-3


def to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def from_dev(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_dev_to_f64(t: torch.Tensor) -> np.ndarray:
    return O.bf16_to_f64(from_dev(t))


# The largest errors each GPU test measured against the oracle, keyed by test:
# {test: {"max-abs": .., "mean-abs": .., "lse": ..}}; conftest prints them at
# the end of the run, so the tolerances can be read against measured values.
MEASURED = {}


def _note(kind: str, value: float):
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0].split("::")[-1]
    rec = MEASURED.setdefault(test, {})
    rec[kind] = max(rec.get(kind, 0.0), float(value))


def assert_close(got: np.ndarray, want: np.ndarray, what: str, max_abs=MAX_ABS, mean_abs=MEAN_ABS,
                 rel=0.0):
    """max |got - want| <= max_abs (+ rel * |want| when rel > 0) and mean <= mean_abs.

    rel = 2^-8 adds the bf16 output-rounding bound (half an ulp) for cases
    whose outputs grow past magnitude 1, e.g. a sharpened softmax."""
    err = np.abs(got - want)
    assert np.isfinite(got).all(), "%s: non-finite output" % what
    mn = float(err.mean())
    mx = float((err - rel * np.abs(want)).max()) if rel else float(err.max())
    _note("max-abs", mx)
    _note("mean-abs", mn)
    assert mx <= max_abs and mn <= mean_abs, "%s: max-abs %.3g mean-abs %.3g" % (what, mx, mn)
    return mx, mn


def assert_lse(got: np.ndarray, want: np.ndarray, tol: float, what: str = "lse"):
    """max |got - want| < tol for natural-log LSE values."""
    err = float(np.abs(got - want).max())
    _note("lse", err)
    assert err < tol, "%s: lse err %.3g" % (what, err)
    return err


class Pair:
    """A GPU StreamCache and oracle windows for a subset of its caches."""

    def __init__(self, w: synth.Workload, tag: str, watch=None, tail_cap=None, wait_ns=0, mrope=None):
        self.w, self.tag = w, tag
        self.watch = list(range(w.C)) if watch is None else list(watch)
        self.cache = skv.StreamCache(w.C, w.P, w.V, w.F, w.T, w.Hkv, w.d, w.theta,
                                     tail_cap=w.tail_cap if tail_cap is None else tail_cap,
                                     wait_ns=wait_ns, mrope=mrope)
        pk, pv = synth.prefix_kv(w, tag)
        if w.P:
            skv.kv_write_rows(self.cache, 0, to_dev(pk), to_dev(pv))
        self.win = {c: O.StreamWindow(w.P, w.V, w.F, w.T, w.Hkv, w.d, pk[c], pv[c]) for c in self.watch}
        self.n_inserts = 0

    def insert(self, k=None, v=None):
        if k is None:
            k, v = synth.frame_kv(self.w, self.n_inserts, self.tag)
        skv.kv_stream_insert(self.cache, to_dev(k), to_dev(v))
        for c, win in self.win.items():
            win.insert(k[c], v[c])
        self.n_inserts += 1

    def fill(self):
        while self.n_inserts < self.w.F:
            self.insert()

    def set_tail(self, n: int):
        tk, tv = synth.tail_kv(self.w, n, self.tag)
        if n:
            skv.kv_write_rows(self.cache, self.cache.n_visual, to_dev(tk), to_dev(tv))
        for c, win in self.win.items():
            win.set_tail(tk[c], tv[c])

    def check_ring(self):
        """Ring heads, ring slots and prefix rows bit-exact against the oracle."""
        w, cache = self.w, self.cache
        torch.cuda.synchronize()
        heads = cache.head.cpu().numpy()
        k = from_dev(cache.k)
        vt = from_dev(cache.vt)
        P, R = w.P, w.V * w.F * w.T
        for c, win in self.win.items():
            head, rk, rv = win.ring_expected()
            np.testing.assert_array_equal(heads[c], head)
            gk = k[c][:, P:P + R].reshape(w.Hkv, w.V, w.F, w.T, w.d).transpose(1, 2, 3, 0, 4)
            gv = vt[c][:, :, P:P + R].reshape(w.Hkv, w.d, w.V, w.F, w.T).transpose(2, 3, 4, 0, 1)
            np.testing.assert_array_equal(gk, rk)
            np.testing.assert_array_equal(gv, rv)
            np.testing.assert_array_equal(k[c][:, :P].transpose(1, 0, 2), win.prefix_k)
            np.testing.assert_array_equal(vt[c][:, :, :P].transpose(2, 0, 1), win.prefix_v)
        assert cache.device_status() == 0
