"""Mutation check of the oracle's pins.  Each entry below plants one
plausible slip in a copy of the oracle's source: a sign, an index, an
exponent, an operand, a dropped term.  The copy is loaded as a module, and
every pin of test_oracle_pins.py runs against it; at least one pin must fail
for each slip.  The unmodified oracle must pass them all under the same
harness.  CPU only; the real oracle module is never modified."""
import importlib.util
import os
import types

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE = os.path.join(os.path.dirname(HERE), "oracle", "skv_oracle.py")
PINS = os.path.join(HERE, "test_oracle_pins.py")

# (name, exact text in the oracle, the slip that replaces it)
MUTATIONS = [
    ("rotation sign",
     "x1 * c - x2 * s, x2 * c + x1 * s", "x1 * c + x2 * s, x2 * c - x1 * s"),
    ("frequency exponent",
     "(-2.0 * np.arange(half, dtype=np.float64) / d)", "(-1.0 * np.arange(half, dtype=np.float64) / d)"),
    ("interleaved instead of rotate-half pairs",
     "x1, x2 = x[..., :half], x[..., half:]", "x1, x2 = x[..., 0::2], x[..., 1::2]"),
    ("GQA head map",
     "kh = h // G", "kh = h % Hkv"),
    ("strict mask",
     "visible = k_pos[None, :] <= q_pos[:, None]", "visible = k_pos[None, :] < q_pos[:, None]"),
    ("dropped softmax scale",
     "s = (qr[h] @ kr[kh].T) * sm_scale", "s = (qr[h] @ kr[kh].T)"),
    ("unnormalised probabilities",
     "out[h] = (p / l) @ vt[kh]", "out[h] = p @ vt[kh]"),
    ("V from the query head",
     "out[h] = (p / l) @ vt[kh]", "out[h] = (p / l) @ vt[h % Hkv]"),
    ("LSE without the max",
     "lse[h] = (m + np.log(l))[:, 0]", "lse[h] = np.log(l)[:, 0]"),
    ("new-frame index without the view offset",
     "return self.P + v * self.F * self.T + (self.F - 1) * self.T + t",
     "return self.P + (self.F - 1) * self.T + t"),
    ("evicts the newest frame",
     "dq.popleft()", "dq.pop()"),
    ("views in reverse order",
     "        for dq in self.views:\n            for fk, fv in dq:",
     "        for dq in reversed(self.views):\n            for fk, fv in dq:"),
    ("ring slot turns the wrong way",
     "s = (head + f) % self.F", "s = (head - f) % self.F"),
    ("block positions off by one",
     "q_pos = base + np.arange(blk)", "q_pos = base + np.arange(blk) + 1"),
    ("block placed without the tail length",
     "base = k_bits.shape[0]", "base = win.n_visual"),
    ("window queries one position late",
     "attention_rows(q_win[rows], rows, k_bits", "attention_rows(q_win[rows], rows + 1, k_bits"),
    ("accept compares the same slot",
     "if draft[i] != target[i - 1]:", "if draft[i] != target[i]:"),
    ("next token one slot early",
     "return k, target[k]", "return k, target[k - 1]"),
    ("bf16 widening shift",
     "<< np.uint32(16)", "<< np.uint32(15)"),
    ("multi-section: rows and columns swapped",
     "out.append((b, b + tau // self.W, b + tau % self.W))",
     "out.append((b, b + tau % self.W, b + tau // self.W))"),
    ("multi-section: temporal component from the token",
     "out.append((b, b + tau // self.W, b + tau % self.W))",
     "out.append((n, b + tau // self.W, b + tau % self.W))"),
    ("multi-section: token offset without the prefix",
     "tau = (n - self.P) % self.T", "tau = n % self.T"),
    ("multi-section: frequencies not dealt in turn",
     "c, k = i % 3, i // 3", "c, k = (i // 3) % 3, i % 3"),
    ("multi-section: rotation sign",
     "lo * cos - hi * sin, hi * cos + lo * sin", "lo * cos + hi * sin, hi * cos - lo * sin"),
    ("multi-section: component order reversed",
     "[:, np.asarray(sec, dtype=np.int64)]", "[:, 2 - np.asarray(sec, dtype=np.int64)]"),
    ("multi-section: reading ignored by the attention",
     "return rope_rotate_sections(x, mrope.triples(pos), theta, mrope.sec)",
     "return rope_rotate(x, pos, theta)"),
]


def _module_from_source(src: str, name: str):
    mod = types.ModuleType(name)
    mod.__file__ = ORACLE
    exec(compile(src, "%s [%s]" % (ORACLE, name), "exec"), mod.__dict__)
    return mod


def _pin_calls():
    """The pin module (a private copy) and every test call in it, with the
    parametrized ones expanded."""
    spec = importlib.util.spec_from_file_location("pins_for_mutation_check", PINS)
    pins = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(pins)
    calls = []
    for name, fn in sorted(vars(pins).items()):
        if not (name.startswith("test_") and callable(fn)):
            continue
        params = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not params:
            calls.append((name, fn, {}))
            continue
        assert len(params) == 1, name
        argnames, argvalues = params[0].args[:2]
        names = [a.strip() for a in argnames.split(",")] if isinstance(argnames, str) else list(argnames)
        for vals in argvalues:
            vals = vals if len(names) > 1 else (vals,)
            calls.append(("%s%s" % (name, list(vals)), fn, dict(zip(names, vals))))
    return pins, calls


def _failing_pins(pins, calls, oracle_mod):
    saved = pins.O
    pins.O = oracle_mod
    failed = []
    try:
        for name, fn, kw in calls:
            try:
                fn(**kw)
            except Exception:          # an assertion or a crash: either way the slip is seen
                failed.append(name)
    finally:
        pins.O = saved
    return failed


@pytest.fixture(scope="module")
def harness():
    src = open(ORACLE).read()
    pins, calls = _pin_calls()
    assert len(calls) >= 30
    return src, pins, calls


def test_unmodified_oracle_passes_every_pin_under_the_harness(harness):
    src, pins, calls = harness
    assert _failing_pins(pins, calls, _module_from_source(src, "oracle_copy")) == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_each_planted_slip_fails_a_pin(harness, name, old, new):
    src, pins, calls = harness
    assert src.count(old) == 1, "the text to mutate must occur exactly once: %r" % old
    mutant = _module_from_source(src.replace(old, new), "oracle_mutant")
    failed = _failing_pins(pins, calls, mutant)
    assert failed, "no pin catches the slip '%s'" % name
