"""The C ABI on a machine without a GPU: the library builds, loads and exports
every declared symbol, and the host-side argument checks answer before any
device work is enqueued."""
import ctypes
import os
import re
import subprocess

import pytest

from streaming_kv_cache_gb300 import build as B
from streaming_kv_cache_gb300 import skv, synth

HEADER = os.path.join(B.ROOT, "include", "skv.h")


@pytest.fixture(scope="module")
def L():
    B.build()
    return skv.lib()


def _declared():
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\*?\s+\*?([a-z_0-9]+)\(", src, flags=re.M)))


def test_header_declares_the_binding_exports():
    assert sorted(skv.EXPORTS) == _declared()


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in _declared():
        assert name in syms, name
        assert getattr(L, name) is not None


def test_version_and_strings(L):
    assert L.skv_version() == 1
    for code in (0, -1, -2, -3, 1, 2, 4, 8, 6):
        assert len(skv.status_string(code)) > 0


def test_row_cap(L):
    assert skv.skv_row_cap(256, 4, 4, 180, 128) == 3328
    assert skv.skv_row_cap(512, 6, 8, 256, 128) == 12928
    assert skv.skv_row_cap(8, 2, 2, 16, 32) == 128
    assert L.skv_row_cap(-1, 1, 1, 1, 0) == -1
    assert L.skv_row_cap(0, 0, 1, 1, 0) == -1


FAKE = 0x10000  # never dereferenced: every case below fails validation first


def _desc(**kw):
    base = dict(n_cache=2, n_view=4, n_frame=4, frame_len=180, prefix_len=256, tail_cap=128,
                n_kv_head=8, head_dim=128, row_cap=3328, rope_len=3264, k=FAKE, vt=FAKE * 2,
                head=FAKE * 3, sync=FAKE * 4, rope=FAKE * 5, status=FAKE * 6, wait_ns=0)
    base.update(kw)
    return skv.skv_cache(**base)


@pytest.mark.parametrize("bad", [
    dict(head_dim=96), dict(head_dim=0), dict(n_view=0), dict(n_frame=0), dict(frame_len=0),
    dict(prefix_len=-1), dict(tail_cap=-1), dict(n_kv_head=0), dict(row_cap=3200),
    dict(row_cap=3330), dict(rope_len=3000), dict(k=0), dict(vt=0), dict(head=0),
    dict(rope=0), dict(status=0), dict(k=FAKE + 8), dict(vt=FAKE + 2), dict(head=FAKE + 2),
])
def test_bad_cache_descriptor_is_rejected(L, bad):
    d = _desc(**bad)
    p = ctypes.c_void_p
    assert L.kv_stream_insert(ctypes.byref(d), p(FAKE), p(FAKE), None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_prefill(ctypes.byref(d), 32, p(FAKE), p(FAKE), None, 1.0, None) == skv.SKV_ERR_INVALID


def test_sync_counters_are_needed_by_the_insert_only(L):
    """cache->sync holds the frame insert's arrival counters: kv_stream_insert
    rejects a null or misaligned one, every other call accepts a descriptor
    without it (here they get past every argument check and stop only at
    the missing GPU)."""
    p = ctypes.c_void_p
    for sync in (0, FAKE + 2):
        r = ctypes.byref(_desc(sync=sync))
        assert L.kv_stream_insert(r, p(FAKE), p(FAKE), None) == skv.SKV_ERR_INVALID
    r = ctypes.byref(_desc(sync=0))
    no_gpu = (skv.SKV_ERR_CUDA, skv.SKV_ERR_UNSUPPORTED)
    assert L.stream_attn_prefill(r, 32, p(FAKE), p(FAKE), None, 1.0, None) in no_gpu
    assert L.stream_attn_window(r, 32, p(FAKE), p(FAKE), None, 1.0, None) in no_gpu
    assert L.stream_attn_prefill_tail(r, 32, 9, *[p(FAKE)] * 5, None, 1.0, None) in no_gpu
    assert L.kv_write_rows(r, 0, 8, p(FAKE), p(FAKE), None) in no_gpu
    ws = L.skv_verify_workspace_bytes(r, 32, 9)
    assert ws > 0
    assert L.stream_attn_verify(r, 32, 9, *[p(FAKE)] * 5, None, None, None, None, p(FAKE), ws, 1.0,
                                None) in no_gpu


def test_null_descriptor(L):
    assert L.kv_stream_insert(None, None, None, None) == skv.SKV_ERR_INVALID
    assert L.skv_verify_workspace_bytes(None, 32, 9) == 0


def test_call_arguments_are_checked(L):
    d = _desc()
    p = ctypes.c_void_p
    r = ctypes.byref(d)
    # misaligned / null tensors
    assert L.kv_stream_insert(r, p(FAKE + 4), p(FAKE), None) == skv.SKV_ERR_INVALID
    assert L.kv_stream_insert(r, None, p(FAKE), None) == skv.SKV_ERR_INVALID
    # query heads not a multiple of kv heads; group size not dividing 128
    assert L.stream_attn_prefill(r, 30, p(FAKE), p(FAKE), None, 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_prefill(r, 24, p(FAKE), p(FAKE), None, 1.0, None) == skv.SKV_ERR_UNSUPPORTED
    assert L.stream_attn_prefill(r, 32, p(FAKE), p(FAKE), None, 0.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_prefill(r, 32, p(FAKE), p(FAKE), p(FAKE + 2), 1.0, None) == skv.SKV_ERR_INVALID
    # rows outside the cache
    assert L.kv_write_rows(r, 3300, 29, p(FAKE), p(FAKE), None) == skv.SKV_ERR_INVALID
    assert L.kv_write_rows(r, -1, 2, p(FAKE), p(FAKE), None) == skv.SKV_ERR_INVALID
    ws = L.skv_verify_workspace_bytes(r, 32, 9)
    args = [p(FAKE)] * 5
    # block too large for the tail; more than 64 query heads per kv head; a
    # block of more than 128 rows per kv head whose group size does not divide
    # 128 (rows are taken 128 at a time, whole tokens each); ids half given
    assert L.stream_attn_verify(r, 32, 129, *args, None, None, None, None, p(FAKE), ws, 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_verify(r, 1024, 9, *args, None, None, None, None, p(FAKE), ws, 1.0, None) == skv.SKV_ERR_UNSUPPORTED
    assert L.stream_attn_verify(r, 24, 43, *args, None, None, None, None, p(FAKE), ws, 1.0, None) == skv.SKV_ERR_UNSUPPORTED
    assert L.stream_attn_verify(r, 24, 42, *args, None, None, None, None, p(FAKE), ws, 1.0, None) != skv.SKV_ERR_UNSUPPORTED
    assert L.stream_attn_verify(r, 24, 22, *args, None, None, None, None, p(FAKE), ws, 1.0, None) != skv.SKV_ERR_UNSUPPORTED
    assert L.stream_attn_verify(r, 32, 9, *args, p(FAKE), p(FAKE), None, p(FAKE), p(FAKE), ws, 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_verify(r, 32, 0, *args, None, None, None, None, p(FAKE), ws, 1.0, None) == skv.SKV_ERR_INVALID


def test_tail_and_window_arguments(L):
    d = _desc()
    p = ctypes.c_void_p
    r = ctypes.byref(d)
    t = [p(FAKE)] * 4            # tail_len, q, k, v
    # token count outside [1, tail_cap]; group size; scale; misaligned tensors / lse
    assert L.stream_attn_prefill_tail(r, 32, 0, *t, p(FAKE), None, 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_prefill_tail(r, 32, 129, *t, p(FAKE), None, 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_prefill_tail(r, 30, 9, *t, p(FAKE), None, 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_prefill_tail(r, 24, 9, *t, p(FAKE), None, 1.0, None) == skv.SKV_ERR_UNSUPPORTED
    assert L.stream_attn_prefill_tail(r, 32, 9, *t, p(FAKE), None, -1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_prefill_tail(r, 32, 9, *t[:3], p(FAKE + 8), p(FAKE), None, 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_prefill_tail(r, 32, 9, None, *t[1:], p(FAKE), None, 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_prefill_tail(r, 32, 9, *t, p(FAKE), p(FAKE + 2), 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_window(r, 30, p(FAKE), p(FAKE), None, 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_window(r, 24, p(FAKE), p(FAKE), None, 1.0, None) == skv.SKV_ERR_UNSUPPORTED
    assert L.stream_attn_window(r, 32, p(FAKE + 8), p(FAKE), None, 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_window(r, 32, p(FAKE), None, None, 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_window(r, 32, p(FAKE), p(FAKE), None, float("nan"), None) == skv.SKV_ERR_INVALID
    bad = _desc(head_dim=96)
    assert L.stream_attn_window(ctypes.byref(bad), 32, p(FAKE), p(FAKE), None, 1.0, None) == skv.SKV_ERR_INVALID
    assert L.stream_attn_prefill_tail(ctypes.byref(bad), 32, 9, *t, p(FAKE), None, 1.0, None) == skv.SKV_ERR_INVALID


def test_rope_mode_and_multi_section_table_arguments(L):
    p = ctypes.c_void_p
    bad = _desc(rope_mode=2)
    assert L.stream_attn_prefill(ctypes.byref(bad), 32, p(FAKE), p(FAKE), None, 1.0, None) == skv.SKV_ERR_INVALID
    ok = _desc(rope_mode=1)
    assert L.stream_attn_prefill(ctypes.byref(ok), 32, p(FAKE), p(FAKE), None, 1.0, None) in (
        skv.SKV_ERR_CUDA, skv.SKV_ERR_UNSUPPORTED)          # past every argument check
    f = L.skv_build_mrope_table
    assert f(p(FAKE), 10, 128, 1e6, 256, 4, 4, 180, 16, 0, 0, None) == skv.SKV_ERR_INVALID   # 180 % 16
    assert f(p(FAKE), 10, 128, 1e6, 256, 4, 4, 180, 15, 3, 6, None) == skv.SKV_ERR_INVALID   # bit 1 in both
    assert f(p(FAKE), 10, 256, 1e6, 256, 4, 4, 180, 15, 0, 0, None) == skv.SKV_ERR_INVALID   # d/2 > 64
    assert f(None, 10, 128, 1e6, 256, 4, 4, 180, 15, 0, 0, None) == skv.SKV_ERR_INVALID
    assert f(p(FAKE), 10, 128, 1e6, 256, 4, 4, 180, 15, 2, 4, None) in (skv.SKV_ERR_CUDA, skv.SKV_ERR_UNSUPPORTED)
    h, w = skv.section_masks([0, 1, 2, 0, 1, 2, 0])
    assert (h, w) == (0b0010010, 0b0100100)


def test_rope_table_arguments(L):
    p = ctypes.c_void_p
    assert L.skv_build_rope_table(None, 10, 128, 1e4, None) == skv.SKV_ERR_INVALID
    assert L.skv_build_rope_table(p(FAKE), 0, 128, 1e4, None) == skv.SKV_ERR_INVALID
    assert L.skv_build_rope_table(p(FAKE), 10, 127, 1e4, None) == skv.SKV_ERR_INVALID
    assert L.skv_build_rope_table(p(FAKE), 10, 128, -1.0, None) == skv.SKV_ERR_INVALID
    assert L.skv_build_rope_table(p(FAKE + 4), 10, 128, 1e4, None) == skv.SKV_ERR_INVALID


def test_header_compiles_as_c_and_struct_layout_matches_the_binding(L, tmp_path):
    """A C99 program built against the header and linked with the library:
    the header is plain C, the no-GPU answers hold from C, and the size and
    every field offset of skv_cache agree with the ctypes structure the
    Python binding passes."""
    exe = str(tmp_path / "abi_check")
    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "abi_check.c")
    lib_dir = os.path.dirname(B.LIB)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-I",
                        os.path.join(B.ROOT, "include"), src, "-L", lib_dir, "-lskv",
                        "-Wl,-rpath," + lib_dir, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    layout = dict(line.split() for line in r.stdout.splitlines() if not line.startswith("FAIL"))
    assert int(layout["size"]) == ctypes.sizeof(skv.skv_cache)
    for name, _ in skv.skv_cache._fields_:
        assert int(layout[name]) == getattr(skv.skv_cache, name).offset, name
    assert layout["fails"] == "0"


def _shape_desc(**kw):
    """A descriptor with a consistent geometry (row_cap and rope_len derived)."""
    g = dict(n_cache=2, n_view=4, n_frame=4, frame_len=180, prefix_len=256, tail_cap=128,
             n_kv_head=8, head_dim=128)
    g.update(kw)
    need = g["prefix_len"] + g["n_view"] * g["n_frame"] * g["frame_len"] + g["tail_cap"]
    return _desc(**g, row_cap=skv.skv_row_cap(g["prefix_len"], g["n_view"], g["n_frame"],
                                              g["frame_len"], g["tail_cap"]), rope_len=need)


def _prefill_family(L, d, Hq=32):
    p = ctypes.c_void_p
    r = ctypes.byref(d)
    return (L.stream_attn_prefill(r, Hq, p(FAKE), p(FAKE), None, 1.0, None),
            L.stream_attn_prefill_tail(r, Hq, 9, p(FAKE), p(FAKE), p(FAKE), p(FAKE), p(FAKE), None, 1.0,
                                       None),
            L.stream_attn_window(r, Hq, p(FAKE), p(FAKE), None, 1.0, None))


def test_prefill_shape_limits_are_checked_before_anything_is_enqueued(L):
    """Outside the kernel's tables (more than 64 views, more than 1024 key
    tiles of 128 rows) the calls answer SKV_ERR_UNSUPPORTED on the host --
    for the tail prefill before its rows are written -- while verify, which
    has no tile table, only limits the views."""
    assert _prefill_family(L, _shape_desc(n_view=65, n_frame=1, frame_len=1, prefix_len=0)) == \
        (skv.SKV_ERR_UNSUPPORTED,) * 3
    # the ring holds 4 x 4 x 180 = 2880 rows and the tail 128
    big = _shape_desc(prefix_len=131072 - 2880 - 128 + 1, n_cache=1)    # 131,073 rows: 1025 tiles
    assert (big.row_cap + 127) // 128 == 1025
    assert _prefill_family(L, big) == (skv.SKV_ERR_UNSUPPORTED,) * 3
    ok = _shape_desc(prefix_len=131072 - 2880 - 128, n_cache=0)         # 131,072 rows: 1024 tiles
    assert (ok.row_cap + 127) // 128 == 1024
    assert _prefill_family(L, ok) == (skv.SKV_OK,) * 3
    p = ctypes.c_void_p
    v65 = _shape_desc(n_view=65, n_frame=1, frame_len=1, prefix_len=0)
    ws = L.skv_verify_workspace_bytes(ctypes.byref(v65), 32, 9)
    assert L.stream_attn_verify(ctypes.byref(v65), 32, 9, *[p(FAKE)] * 5, None, None, None, None,
                                p(FAKE), ws, 1.0, None) == skv.SKV_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_every_workload_geometry_is_within_the_kernels(L, name):
    """The shape checks accept every workload's geometry (an empty cache set
    returns SKV_OK once every shape check has passed)."""
    w = synth.WORKLOADS[name]
    d = _shape_desc(n_cache=0, n_view=w.V, n_frame=w.F, frame_len=w.T, prefix_len=w.P,
                    tail_cap=w.tail_cap, n_kv_head=w.Hkv, head_dim=w.d)
    assert _prefill_family(L, d, Hq=w.Hq) == (skv.SKV_OK,) * 3


def test_host_shape_limits_match_the_kernels():
    """The host-side limits in api.cu are the kernels' own table sizes."""
    csrc = os.path.join(B.ROOT, "streaming_kv_cache_gb300", "csrc")

    def const(fname, name):
        src = open(os.path.join(csrc, fname)).read()
        m = re.search(r"constexpr\s+(?:int|long long)\s+%s\s*=\s*(\d+)" % name, src)
        assert m, (fname, name)
        return int(m.group(1))

    assert const("api.cu", "kMaxViews") == const("prefill_tc.cu", "MAX_VIEWS") == const("verify_tc.cu", "MAX_VIEWS")
    assert const("api.cu", "kPrefillMaxKeyTiles") == const("prefill_tc.cu", "MAX_TILES")
    assert const("api.cu", "kPrefillKeyTile") == const("prefill_tc.cu", "BN")


def _sm_count():
    """The SM count the library plans for: the device's, or 148 without one."""
    try:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.get_device_properties(0).multi_processor_count
    except Exception:
        pass
    return 148


def _verify_plan(C, Hkv, G, blk, d, n_visual, tail_cap, n_sm):
    """The verify partition, restated: the row form (64 or 128 block rows per
    unit), the units' tiles of 64 keys spread over at most one wave (two CTAs
    per SM for the 64-row form, one for the 128-row form), at least 4 tiles and
    at most 14 whole units' worth per CTA, at most 64 pieces per unit.
    Returns (tiles per unit, tiles per CTA, CTAs, pieces per unit at most,
    units, rows per unit, workspace bytes)."""
    R = blk * G
    rows = 128 if R > 64 else 64
    RH = -(-R // rows)
    units = C * Hkv * RH
    TM = -(-(n_visual + tail_cap) // 64)
    total = units * TM
    slots = (1 if rows == 128 else 2) * n_sm
    if units <= slots < 2 * units:
        W, n, P = TM, units, 1
    else:
        n = min(slots, -(-total // 4))
        n = max(n, -(-units // 14))
        n = min(n, total // max(1, (TM + 62) // 63))
        n = max(n, 1)
        W = -(-total // n)
        n = -(-total // W)
        P = -(-TM // W) + 1
    RU = min(R, rows)
    ws = 0 if W % TM == 0 else ((units + 2) * 4 + 255) // 256 * 256 + units * P * RU * (d + 2) * 4
    return TM, W, n, P, units, RU, ws


@pytest.mark.parametrize("blk", [1, 9, 16, 17, 32, 33])
@pytest.mark.parametrize("Hq", [8, 32, 64])
def test_verify_plan_bounds_and_workspace(L, blk, Hq):
    """Over batches, tail capacities and window sizes: every unit is cut into
    at most 64 pieces and every CTA's share into at most 16 (the kernel's
    tables), the one-wave rule holds, and the library's workspace size is the
    plan's.  Whenever a unit may be cut into four pieces or more (the plans
    that ask for the merge after a grid barrier, a cooperative launch), the
    grid fits one wave of the form's CTAs per SM."""
    Hkv, d, n_sm = 8, 128, _sm_count()
    G = Hq // Hkv
    for C in (1, 3, 8, 32, 64, 200, 1000):
        for tail_cap, frames in ((64, (16, 1, 1, 32)), (128, (256, 4, 4, 180)), (1024, (512, 6, 8, 256))):
            if blk > tail_cap:
                continue
            P, V, F, T = frames
            TM, W, n, Pm, units, RU, ws = _verify_plan(C, Hkv, G, blk, d, P + V * F * T, tail_cap, n_sm)
            assert Pm <= 64, (C, blk, Hq, tail_cap)
            assert (W - 1) // TM + 2 <= 16 or Pm == 1, (C, blk, Hq, tail_cap)
            assert n * W >= units * TM > (n - 1) * W
            if Pm >= 4:
                assert n <= (1 if blk * G > 64 else 2) * n_sm, (C, blk, Hq, tail_cap)
            desc = _shape_desc(n_cache=C, n_view=V, n_frame=F, frame_len=T, prefix_len=P, tail_cap=tail_cap,
                               n_kv_head=Hkv, head_dim=d)
            assert L.skv_verify_workspace_bytes(ctypes.byref(desc), Hq, blk) == ws, (C, blk, Hq, tail_cap)
