"""The oracle: plain fp64 CPU restatement of streaming view-major KV-cache
attention, used only by the tests, the smoke check and the benchmark's
CPU-baseline leg.  It is test infrastructure, not part of the product."""
from .skv_oracle import (StreamWindow, accept_length, attention_rows, bf16_to_f64,  # noqa: F401
                         rope_rotate, stream_prefill, stream_verify)
