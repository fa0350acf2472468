"""Python binding of libskv (ctypes).

Argument marshalling only: every step of the streaming-attention path runs in
the library's CUDA kernels.  PyTorch provides device memory and the current
stream.  The functions carry the C entry points' names; see include/skv.h for
the full contract.
"""
from __future__ import annotations

import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libskv.so")

SKV_OK, SKV_ERR_INVALID, SKV_ERR_UNSUPPORTED, SKV_ERR_CUDA, SKV_ERR_TOO_LARGE = 0, -1, -2, -3, -4
SKV_NOALLOC_MAX_CACHE_VIEWS = 16384
SKV_DEV_TIMEOUT, SKV_DEV_BAD_HEAD, SKV_DEV_TAIL_OVERFLOW, SKV_DEV_BAD_TAIL = 1, 2, 4, 8

# every function the C header declares
EXPORTS = ("skv_version", "skv_status_string", "skv_last_cuda_error", "skv_row_cap",
           "skv_build_rope_table", "skv_build_mrope_table", "kv_write_rows", "kv_stream_insert", "kv_stream_insert_noalloc",
           "stream_attn_prefill", "stream_attn_prefill_insert", "stream_attn_prefill_tail",
           "stream_attn_window",
           "skv_verify_workspace_bytes", "stream_attn_verify")


class SkvError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        msg = "%s: %s" % (what, status_string(code)) if what else status_string(code)
        if code == SKV_ERR_CUDA:
            msg += " (cudaError %d)" % lib().skv_last_cuda_error()
        super().__init__(msg)


class skv_cache(ctypes.Structure):
    _fields_ = [("n_cache", ctypes.c_int32), ("n_view", ctypes.c_int32),
                ("n_frame", ctypes.c_int32), ("frame_len", ctypes.c_int32),
                ("prefix_len", ctypes.c_int32), ("tail_cap", ctypes.c_int32),
                ("n_kv_head", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("row_cap", ctypes.c_int32), ("rope_len", ctypes.c_int32),
                ("k", ctypes.c_void_p), ("vt", ctypes.c_void_p),
                ("head", ctypes.c_void_p), ("sync", ctypes.c_void_p),
                ("rope", ctypes.c_void_p), ("status", ctypes.c_void_p),
                ("wait_ns", ctypes.c_uint64), ("rope_mode", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_lib_handle = None


def lib():
    """Load libskv.so (built in-tree by streaming_kv_cache_gb300.build)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError("libskv.so is not built (%s); run streaming_kv_cache_gb300.build.build()"
                              % _LIB_PATH)
        L = ctypes.CDLL(_LIB_PATH)
        P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
        cp = ctypes.POINTER(skv_cache)
        sig = {
            "skv_version": ([], ctypes.c_int),
            "skv_status_string": ([ctypes.c_int], ctypes.c_char_p),
            "skv_last_cuda_error": ([], ctypes.c_int),
            "skv_row_cap": ([I32, I32, I32, I32, I32], I32),
            "skv_build_rope_table": ([P, I32, I32, ctypes.c_double, P], ctypes.c_int),
            "skv_build_mrope_table": ([P, I32, I32, ctypes.c_double, I32, I32, I32, I32, I32,
                                       ctypes.c_uint64, ctypes.c_uint64, P], ctypes.c_int),
            "kv_write_rows": ([cp, I32, I32, P, P, P], ctypes.c_int),
            "kv_stream_insert": ([cp, P, P, P], ctypes.c_int),
            "kv_stream_insert_noalloc": ([cp, P, P, P], ctypes.c_int),
            "stream_attn_prefill": ([cp, I32, P, P, P, ctypes.c_float, P], ctypes.c_int),
            "stream_attn_prefill_insert": ([cp, I32, P, P, P, P, P, ctypes.c_float, P], ctypes.c_int),
            "stream_attn_prefill_tail": ([cp, I32, I32, P, P, P, P, P, P, ctypes.c_float, P],
                                         ctypes.c_int),
            "stream_attn_window": ([cp, I32, P, P, P, ctypes.c_float, P], ctypes.c_int),
            "skv_verify_workspace_bytes": ([cp, I32, I32], SZ),
            "stream_attn_verify": ([cp, I32, I32, P, P, P, P, P, P, P, P, P, P, SZ,
                                    ctypes.c_float, P], ctypes.c_int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes, fn.restype = args, res
        _lib_handle = L
    return _lib_handle


def status_string(code: int) -> str:
    return lib().skv_status_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != SKV_OK:
        raise SkvError(rc, what)


def _stream():
    """The current torch stream of the current device: the library launches
    on the current device, so the tensors of a call must live there."""
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _need(t, shape, dtype, name):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.device.type != "cuda":
        raise ValueError("%s must be on a CUDA device" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def skv_row_cap(P, V, F, T, tail_cap) -> int:
    r = lib().skv_row_cap(P, V, F, T, tail_cap)
    if r < 0:
        raise SkvError(SKV_ERR_INVALID, "skv_row_cap")
    return r


def skv_build_rope_table(tab: torch.Tensor, theta: float):
    n_pos, half, two = tab.shape
    _need(tab, (n_pos, half, 2), torch.float32, "rope table")
    _check(lib().skv_build_rope_table(_ptr(tab), n_pos, 2 * half, float(theta), _stream()),
           "skv_build_rope_table")


def section_masks(sec) -> tuple:
    """(h_mask, w_mask) of a frequency -> component map (0 = t, 1 = h, 2 = w)."""
    h = sum(1 << i for i, c in enumerate(sec) if int(c) == 1)
    w = sum(1 << i for i, c in enumerate(sec) if int(c) == 2)
    return h, w


def skv_build_mrope_table(tab: torch.Tensor, theta: float, P: int, V: int, F: int, T: int,
                          grid_w: int, sec):
    """The multi-section rotary table (see include/skv.h): row n holds the
    angles of the token at logical index n; sec maps frequency i to its
    component (0 = temporal, 1 = height, 2 = width)."""
    n_pos, half, two = tab.shape
    _need(tab, (n_pos, half, 2), torch.float32, "rope table")
    if len(sec) != half:
        raise ValueError("sec must give a component for each of the %d frequencies" % half)
    h, w = section_masks(sec)
    _check(lib().skv_build_mrope_table(_ptr(tab), n_pos, 2 * half, float(theta), P, V, F, T, grid_w,
                                       h, w, _stream()), "skv_build_mrope_table")


class StreamCache:
    """C independent streaming caches of one geometry, in device memory.

    Tensors (all zero-initialised, owned by this object):
      k      bf16 [C][Hkv][row_cap][d]   pre-RoPE keys
      vt     bf16 [C][Hkv][d][row_cap]   values, dimension-major
      head   int32 [C][V]                ring heads
      sync   int32 [C][V]                insert counters
      rope   fp32 [rope_len][d/2][2]     (cos, sin) table
      status int32 [1]                   device status bits

    mrope=(grid_w, sec) selects the multi-section rotary reading (rope_mode 1):
    frames are rows of grid_w tokens and sec maps each of the d/2
    frequencies to its component (0 = temporal, 1 = height, 2 = width).
    """

    def __init__(self, C, P, V, F, T, Hkv, d, theta, tail_cap=128, device="cuda", wait_ns=0,
                 mrope=None):
        self.C, self.P, self.V, self.F, self.T = C, P, V, F, T
        self.Hkv, self.d, self.theta, self.tail_cap = Hkv, d, float(theta), tail_cap
        self.row_cap = skv_row_cap(P, V, F, T, tail_cap)
        self.rope_len = P + V * F * T + tail_cap
        dev = torch.device(device)
        self.k = torch.zeros((C, Hkv, self.row_cap, d), dtype=torch.bfloat16, device=dev)
        self.vt = torch.zeros((C, Hkv, d, self.row_cap), dtype=torch.bfloat16, device=dev)
        self.head = torch.zeros((C, V), dtype=torch.int32, device=dev)
        self.sync = torch.zeros((C, V), dtype=torch.int32, device=dev)
        self.rope = torch.empty((self.rope_len, d // 2, 2), dtype=torch.float32, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)
        self.wait_ns = int(wait_ns)
        self.rope_mode = 0 if mrope is None else 1
        with torch.cuda.device(dev):
            if mrope is None:
                skv_build_rope_table(self.rope, self.theta)
            else:
                skv_build_mrope_table(self.rope, self.theta, P, V, F, T, mrope[0], mrope[1])

    @property
    def n_visual(self):
        return self.P + self.V * self.F * self.T

    def desc(self) -> skv_cache:
        return skv_cache(self.C, self.V, self.F, self.T, self.P, self.tail_cap, self.Hkv, self.d,
                         self.row_cap, self.rope_len, self.k.data_ptr(), self.vt.data_ptr(),
                         self.head.data_ptr(), self.sync.data_ptr(), self.rope.data_ptr(),
                         self.status.data_ptr(), self.wait_ns, self.rope_mode, 0)

    def device_status(self) -> int:
        return int(self.status.item())


def kv_write_rows(cache: StreamCache, row0: int, k_src: torch.Tensor, v_src: torch.Tensor):
    n = k_src.shape[1]
    shp = (cache.C, n, cache.Hkv, cache.d)
    _need(k_src, shp, torch.bfloat16, "k_src")
    _need(v_src, shp, torch.bfloat16, "v_src")
    d = cache.desc()
    _check(lib().kv_write_rows(ctypes.byref(d), row0, n, _ptr(k_src), _ptr(v_src), _stream()),
           "kv_write_rows")


def kv_stream_insert(cache: StreamCache, k_new: torch.Tensor, v_new: torch.Tensor):
    shp = (cache.C, cache.V, cache.T, cache.Hkv, cache.d)
    _need(k_new, shp, torch.bfloat16, "k_new")
    _need(v_new, shp, torch.bfloat16, "v_new")
    d = cache.desc()
    _check(lib().kv_stream_insert(ctypes.byref(d), _ptr(k_new), _ptr(v_new), _stream()),
           "kv_stream_insert")


def kv_stream_insert_noalloc(cache: StreamCache, k_new: torch.Tensor, v_new: torch.Tensor):
    """kv_stream_insert without caller scratch: for callers that may not
    allocate device memory, the insert's counters live in a fixed static
    device array inside the library (cache.sync is not used)."""
    shp = (cache.C, cache.V, cache.T, cache.Hkv, cache.d)
    _need(k_new, shp, torch.bfloat16, "k_new")
    _need(v_new, shp, torch.bfloat16, "v_new")
    d = cache.desc()
    d.sync = None
    _check(lib().kv_stream_insert_noalloc(ctypes.byref(d), _ptr(k_new), _ptr(v_new), _stream()),
           "kv_stream_insert_noalloc")


def stream_attn_prefill(cache: StreamCache, q_new: torch.Tensor, sm_scale: float,
                        out: torch.Tensor | None = None, lse: torch.Tensor | bool | None = None):
    """Returns out (and lse when asked for) for the new-frame queries."""
    C, nq, Hq, d = q_new.shape
    _need(q_new, (cache.C, cache.V * cache.T, Hq, cache.d), torch.bfloat16, "q_new")
    if out is None:
        out = torch.empty_like(q_new)
    _need(out, q_new.shape, torch.bfloat16, "out")
    if lse is True:
        lse = torch.empty((C, Hq, nq), dtype=torch.float32, device=q_new.device)
    if isinstance(lse, torch.Tensor):
        _need(lse, (C, Hq, nq), torch.float32, "lse")
    else:
        lse = None
    dd = cache.desc()
    _check(lib().stream_attn_prefill(ctypes.byref(dd), Hq, _ptr(q_new), _ptr(out), _ptr(lse),
                                     float(sm_scale), _stream()), "stream_attn_prefill")
    return (out, lse) if lse is not None else out


def stream_attn_prefill_insert(cache: StreamCache, k_new: torch.Tensor, v_new: torch.Tensor,
                               q_new: torch.Tensor, sm_scale: float, out: torch.Tensor | None = None,
                               lse: torch.Tensor | bool | None = None):
    """kv_stream_insert(k_new, v_new) then stream_attn_prefill(q_new) as one
    call (one kernel where the geometry allows).  Returns out (and lse when
    asked for)."""
    shp = (cache.C, cache.V, cache.T, cache.Hkv, cache.d)
    _need(k_new, shp, torch.bfloat16, "k_new")
    _need(v_new, shp, torch.bfloat16, "v_new")
    C, nq, Hq, d = q_new.shape
    _need(q_new, (cache.C, cache.V * cache.T, Hq, cache.d), torch.bfloat16, "q_new")
    if out is None:
        out = torch.empty_like(q_new)
    _need(out, q_new.shape, torch.bfloat16, "out")
    lse = _lse_arg(lse, C, Hq, nq, q_new.device)
    dd = cache.desc()
    _check(lib().stream_attn_prefill_insert(ctypes.byref(dd), Hq, _ptr(k_new), _ptr(v_new), _ptr(q_new),
                                            _ptr(out), _ptr(lse), float(sm_scale), _stream()),
           "stream_attn_prefill_insert")
    return (out, lse) if lse is not None else out


def _lse_arg(lse, C, Hq, n, device):
    if lse is True:
        lse = torch.empty((C, Hq, n), dtype=torch.float32, device=device)
    if isinstance(lse, torch.Tensor):
        _need(lse, (C, Hq, n), torch.float32, "lse")
        return lse
    return None


def stream_attn_prefill_tail(cache: StreamCache, tail_len: torch.Tensor, q_tail: torch.Tensor,
                             k_tail: torch.Tensor, v_tail: torch.Tensor, sm_scale: float,
                             out: torch.Tensor | None = None,
                             lse: torch.Tensor | bool | None = None):
    """Writes the tokens' K/V after tail_len[c] tail rows and returns their
    attention output (and lse when asked for).  The caller advances
    tail_len by the number of tokens."""
    C, n, Hq, d = q_tail.shape
    _need(q_tail, (cache.C, n, Hq, cache.d), torch.bfloat16, "q_tail")
    _need(k_tail, (cache.C, n, cache.Hkv, cache.d), torch.bfloat16, "k_tail")
    _need(v_tail, (cache.C, n, cache.Hkv, cache.d), torch.bfloat16, "v_tail")
    _need(tail_len, (cache.C,), torch.int32, "tail_len")
    if out is None:
        out = torch.empty_like(q_tail)
    _need(out, q_tail.shape, torch.bfloat16, "out")
    lse = _lse_arg(lse, C, Hq, n, q_tail.device)
    dd = cache.desc()
    _check(lib().stream_attn_prefill_tail(ctypes.byref(dd), Hq, n, _ptr(tail_len), _ptr(q_tail),
                                          _ptr(k_tail), _ptr(v_tail), _ptr(out), _ptr(lse),
                                          float(sm_scale), _stream()), "stream_attn_prefill_tail")
    return (out, lse) if lse is not None else out


def stream_attn_window(cache: StreamCache, q_win: torch.Tensor, sm_scale: float,
                       out: torch.Tensor | None = None, lse: torch.Tensor | bool | None = None):
    """Every window token as a query (logical order: prefix, then each view's
    frames oldest to newest).  Returns out (and lse when asked for)."""
    C, n, Hq, d = q_win.shape
    _need(q_win, (cache.C, cache.n_visual, Hq, cache.d), torch.bfloat16, "q_win")
    if out is None:
        out = torch.empty_like(q_win)
    _need(out, q_win.shape, torch.bfloat16, "out")
    lse = _lse_arg(lse, C, Hq, n, q_win.device)
    dd = cache.desc()
    _check(lib().stream_attn_window(ctypes.byref(dd), Hq, _ptr(q_win), _ptr(out), _ptr(lse),
                                    float(sm_scale), _stream()), "stream_attn_window")
    return (out, lse) if lse is not None else out


def skv_verify_workspace_bytes(cache: StreamCache, n_q_head: int, blk: int) -> int:
    d = cache.desc()
    return int(lib().skv_verify_workspace_bytes(ctypes.byref(d), n_q_head, blk))


def verify_workspace(cache: StreamCache, n_q_head: int, blk: int) -> torch.Tensor:
    """A zero-filled workspace for stream_attn_verify."""
    n = max(16, skv_verify_workspace_bytes(cache, n_q_head, blk))
    return torch.zeros((n,), dtype=torch.uint8, device=cache.k.device)


def stream_attn_verify(cache: StreamCache, tail_len: torch.Tensor, q_blk: torch.Tensor,
                       k_blk: torch.Tensor, v_blk: torch.Tensor, sm_scale: float,
                       target_ids: torch.Tensor | None = None, draft_ids: torch.Tensor | None = None,
                       ws: torch.Tensor | None = None, out: torch.Tensor | None = None,
                       accept_len: torch.Tensor | None = None, next_token: torch.Tensor | None = None):
    """One verify pass.  Returns (out, accept_len, next_token); the last two
    are None when no ids are given."""
    C, blk, Hq, d = q_blk.shape
    _need(q_blk, (cache.C, blk, Hq, cache.d), torch.bfloat16, "q_blk")
    _need(k_blk, (cache.C, blk, cache.Hkv, cache.d), torch.bfloat16, "k_blk")
    _need(v_blk, (cache.C, blk, cache.Hkv, cache.d), torch.bfloat16, "v_blk")
    _need(tail_len, (cache.C,), torch.int32, "tail_len")
    if out is None:
        out = torch.empty_like(q_blk)
    _need(out, q_blk.shape, torch.bfloat16, "out")
    ids = target_ids is not None and draft_ids is not None
    if ids:
        _need(target_ids, (cache.C, blk), torch.int32, "target_ids")
        _need(draft_ids, (cache.C, blk), torch.int32, "draft_ids")
        if accept_len is None:
            accept_len = torch.empty((cache.C,), dtype=torch.int32, device=q_blk.device)
        if next_token is None:
            next_token = torch.empty((cache.C,), dtype=torch.int32, device=q_blk.device)
        _need(accept_len, (cache.C,), torch.int32, "accept_len")
        _need(next_token, (cache.C,), torch.int32, "next_token")
    if ws is None:
        ws = verify_workspace(cache, Hq, blk)
    dd = cache.desc()
    _check(lib().stream_attn_verify(
        ctypes.byref(dd), Hq, blk, _ptr(tail_len), _ptr(q_blk), _ptr(k_blk), _ptr(v_blk), _ptr(out),
        _ptr(target_ids) if ids else None, _ptr(draft_ids) if ids else None,
        _ptr(accept_len) if ids else None, _ptr(next_token) if ids else None,
        _ptr(ws), ws.numel(), float(sm_scale), _stream()), "stream_attn_verify")
    return out, (accept_len if ids else None), (next_token if ids else None)
