"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol include/kda.h declares, the descriptor layout matches, and
host-checkable errors return before anything is enqueued."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import linear_attention_prefill_chunked_gb300 as kda
from linear_attention_prefill_chunked_gb300 import api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    lib = kda.load()
    names = _declared()
    assert set(names) == set(api.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", api.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r" T (kda_\w+)", out))
    assert set(names) <= exported


def test_descriptor_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    fields = [f for f, _ in api.KdaDesc._fields_]
    body = "\n".join(f'  printf("{f} %zu\\n", offsetof(kda_desc_t, {f}));' for f in fields)
    src.write_text(f"""#include <stddef.h>
#include <stdio.h>
#include "kda.h"
int main(void) {{
  printf("size %zu\\n", sizeof(kda_desc_t));
{body}
  return 0;
}}
""")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), "-I",
                    "/usr/local/cuda/include", str(src), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    assert int(got["size"]) == ctypes.sizeof(api.KdaDesc)
    for f in fields:
        assert int(got[f]) == getattr(api.KdaDesc, f).offset, f


def _desc(**kw):
    base = dict(num_seqs=3, total_tokens=100, Hk=2, Hv=4, K=128, V=128, qkv_dtype=torch.bfloat16)
    base.update(kw)
    return kda.make_desc(**base)


def test_workspace_queries_and_path_selection():
    assert kda.prefill_workspace_size(_desc()) >= 256
    lib = kda.load()
    assert lib.kda_decode_workspace_size(ctypes.byref(_desc())) >= 256
    bad = [_desc(K=96), _desc(Hv=3), _desc(Hk=0)]
    d = _desc()
    d.chunk_size = 32
    bad.append(d)
    d = _desc()
    d.flags = 16                                             # no such flag
    bad.append(d)
    for b in bad:
        assert kda.prefill_workspace_size(b) == 0
        assert kda.prefill_path(b) == -1
    assert kda.prefill_path(_desc(qkv_dtype=torch.float32)) == 0
    assert kda.prefill_path(_desc()) == 1                    # bf16, 128x128 heads
    d = _desc()
    d.flags = 1                                              # KDA_FLAG_CUDA_CORE_PATH
    assert kda.prefill_path(d) == 0
    assert kda.prefill_path(_desc(K=64)) == 0
    d = _desc()
    d.flags = 8                                              # KDA_FLAG_STATE_VK: same path
    assert kda.prefill_path(d) == 1
    # the least workspace (no long sequence cut) is below the full size
    assert 256 <= kda.prefill_min_workspace_size(_desc()) < kda.prefill_workspace_size(_desc())
    d = _desc()
    d.flags = 2                                              # KDA_FLAG_SCALAR_GATE
    assert kda.prefill_path(d) == (1 if d.num_v_heads % 8 == 0 else 0)
    d = _desc(Hv=4, Hk=4)
    d.flags = 2                                              # heads staged in groups of 8
    assert kda.prefill_path(d) == 0


def test_host_checked_errors_return_before_any_launch():
    lib = kda.load()
    P = ctypes.c_void_p
    fake = P(1 << 20)  # aligned dummy address: never dereferenced by these calls
    d = _desc()
    call = lambda desc, ws=fake, nws=0, **kw: lib.kda_chunk_prefill(
        ctypes.byref(desc) if desc is not None else None, kw.get("q", fake), fake, fake, fake,
        fake, kw.get("cu", fake), kw.get("state", None), kw.get("idx", None),
        kw.get("final", None), fake, ws, nws, None)
    assert call(None) == 1                                   # null descriptor
    assert call(d, cu=None) == 1                             # null cu_seqlens
    assert call(d, q=None) == 1                              # null q with T > 0
    assert call(d, q=P((1 << 20) + 2)) == 1                  # misaligned q
    assert call(_desc(K=96)) == 2                            # unsupported head dim
    assert call(d, idx=fake) == 1                            # pool mode without a pool
    d_pool = _desc(num_slots=8)
    assert call(d_pool, idx=fake, state=fake, final=P(2 << 20)) == 1  # final != pool
    assert call(d, ws=P((1 << 20) + 64)) == 1                # misaligned workspace
    assert call(d, nws=16) == 3                              # workspace too small
    dd = _desc(num_slots=8)
    dd.total_tokens = 5                                      # decode needs T == N
    assert lib.kda_decode(ctypes.byref(dd), fake, fake, fake, fake, fake, fake, None, fake, fake,
                          4096, None) == 1
    assert lib.kda_status_string(3) == b"workspace too small"


def test_oracle_library_builds():
    from oracle import kda_oracle
    assert os.path.exists(kda_oracle.build())


def test_pipeline_wait_limit_is_bounded():
    """The watchdog bound of the tensor-core prefill's waits: 0 restores the 2 s default, more
    than 2 s is refused (host only; the GPU test makes the waits run out)."""
    from linear_attention_prefill_chunked_gb300 import api
    with pytest.raises(api.KdaError):
        api.set_pipeline_wait_limit(3_000_000_000)
    api.set_pipeline_wait_limit(2_000_000_000)
    api.set_pipeline_wait_limit(0)
