"""streaming_kv_cache_gb300 -- streaming view-major KV-cache attention on GB300.

A C-ABI library (libskv.so, hand-written CUDA for sm_103a) with three calls
on the streaming path -- kv_stream_insert, stream_attn_prefill and
stream_attn_verify -- plus the tail-token and whole-window prefills, and a
thin ctypes binding.  Build it with streaming_kv_cache_gb300.build.build().
"""
from . import synth  # noqa: F401
from .skv import (EXPORTS, SkvError, StreamCache, kv_stream_insert,  # noqa: F401
                  kv_stream_insert_noalloc, kv_write_rows,
                  lib, skv_build_rope_table, skv_row_cap, skv_verify_workspace_bytes,
                  skv_build_mrope_table, status_string, stream_attn_prefill,
                  stream_attn_prefill_insert, stream_attn_prefill_tail, stream_attn_verify,
                  stream_attn_window, verify_workspace)
