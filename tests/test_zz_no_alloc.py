"""kda_chunk_prefill_noalloc: the prefill for callers that cannot allocate.

Plug-in hosts whose device allocator belongs to someone else, and real-time paths that
forbid allocation after start-up, cannot hand the prefill a freshly allocated workspace.  This entry point takes its scratch from a
fixed array in the library's own device memory instead.  These tests call it through
the C ABI and check it against kda_chunk_prefill (which gets a caller workspace) on
two calls in a row, so the second call also shows that leftovers from the first in
the shared array do not leak into its result.  The file is named to be collected
last.
"""
import ctypes

import pytest
import torch

import linear_attention_prefill_chunked_gb300 as kda
from linear_attention_prefill_chunked_gb300 import synthetic
from tests._util import to_dev

MAX_SEQS = 16384  # KDA_NOALLOC_MAX_SEQS in include/kda.h


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc_call(lib, d, pool, o):
    """One kda_chunk_prefill_noalloc call in pool mode on the current stream."""
    desc = kda.make_desc(num_seqs=d["cu_seqlens"].numel() - 1, total_tokens=d["q"].shape[0],
                         Hk=d["q"].shape[1], Hv=d["v"].shape[1], K=d["q"].shape[2],
                         V=d["v"].shape[2], qkv_dtype=d["q"].dtype, state_dtype=pool.dtype,
                         num_slots=pool.shape[0])
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.kda_chunk_prefill_noalloc(
        ctypes.byref(desc), _ptr(d["q"]), _ptr(d["k"]), _ptr(d["v"]), _ptr(d["g"]),
        _ptr(d["beta"]), _ptr(d["cu_seqlens"]), _ptr(pool), _ptr(d["state_indices"]), None,
        _ptr(o), stream)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_noalloc_matches_workspace_entry_point_twice(dtype):
    lib = kda.load()
    # bf16 runs the tensor-core kernel, fp32 the CUDA-core kernel
    workloads = [synthetic.make([70, 1, 129, 64], Hk=2, Hv=4, K=128, V=128, dtype=dtype,
                                seed=31 + i, state="pool", num_slots=9, last_index_pad=True)
                 for i in range(2)]
    for w in workloads:  # two calls in a row, different inputs
        d = to_dev(w)
        pool_ref = d["state"].clone()
        o_ref, _ = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                     state=pool_ref, state_indices=d["state_indices"])
        pool = d["state"].clone()
        o = torch.full_like(o_ref, float("nan"))
        rc = _noalloc_call(lib, d, pool, o)
        assert rc == 0, lib.kda_status_string(rc)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: bit-identical, so that a stale value left in
        # the shared array by the call before (an order, a counter) cannot hide in a tolerance
        assert torch.equal(o, o_ref), "o (no-alloc vs workspace)"
        assert torch.equal(pool, pool_ref), "pool (no-alloc vs workspace)"


def test_noalloc_rejects_batches_beyond_its_scratch():
    lib = kda.load()
    fake = ctypes.c_void_p(1 << 20)  # never dereferenced: the call must return first
    desc = kda.make_desc(num_seqs=MAX_SEQS + 1, total_tokens=MAX_SEQS + 1, Hk=1, Hv=1, K=128,
                         V=128, qkv_dtype=torch.bfloat16)
    rc = lib.kda_chunk_prefill_noalloc(ctypes.byref(desc), fake, fake, fake, fake, fake, fake,
                                       None, None, None, fake, None)
    assert rc == 3  # KDA_ERR_WORKSPACE_TOO_SMALL
