"""GB300 (sm_103a) chunked KDA prefill and decode.

The compute lives in ``libkda_gb300.so`` (hand-written CUDA kernels behind the
C ABI of ``include/kda.h``); this package is its thin binding.
"""
from .api import (KdaDesc, KdaError, chunk_prefill, chunk_prefill_act, decode, decode_draft, load,
                  make_desc, prefill_min_workspace_size, prefill_path, prefill_workspace_size,
                  read_device_status)

__all__ = ["KdaDesc", "KdaError", "chunk_prefill", "chunk_prefill_act", "decode", "decode_draft",
           "load", "make_desc", "prefill_min_workspace_size", "prefill_path",
           "prefill_workspace_size", "read_device_status"]
