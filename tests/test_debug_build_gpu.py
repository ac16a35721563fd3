"""The bounds-checked debug build (KDA_DEBUG=1 selects libkda_gb300_debug.so, compiled with
-DKDA_DEBUG): every kernel checks its computed global and shared-memory indices, skips an
access that would leave its buffer and reports KDA_DEVICE_DEBUG_BOUNDS in the device status
word -- never a trap.  The small configurations of every entry point run in that build in a
child process; each call must leave a clean status word and give the normal build's results
bit for bit (the checks guard accesses, they change no arithmetic)."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, torch
sys.path.insert(0, sys.argv[1])
import linear_attention_prefill_chunked_gb300 as kda
from linear_attention_prefill_chunked_gb300 import api, synthetic
from tests._util import to_dev
mode = sys.argv[2]
assert api.debug_build() == (mode == "debug")
out = {}
def run(name, fn):
    r = fn()
    ws = r[-1]
    bits = kda.read_device_status(ws)
    assert bits == 0, (name, bits)
    out[name] = [x.cpu() for x in r[:-1]]
def prefill(w, **kw):
    d = to_dev(w)
    st = d["state"]
    o, fin = kda.chunk_prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], state=st,
                               state_indices=d["state_indices"], **kw)
    return o, (st if d["state_indices"] is not None else fin), kda.chunk_prefill.last_workspace
run("pool_fp32", lambda: prefill(synthetic.pool_varlen()))
run("pool_bf16", lambda: prefill(synthetic.pool_varlen(state_dtype=torch.bfloat16)))
run("tiny_fp32", lambda: prefill(synthetic.tiny_varlen()))
run("cut", lambda: prefill(synthetic.make([3000, 100, 37], Hk=2, Hv=4, K=128, V=128, seed=41,
                                          state="pool", num_slots=5)))
run("cut_vk", lambda: prefill(synthetic.make([1500, 63, 130], Hk=2, Hv=4, K=128, V=128, seed=7,
                                             state="pool", num_slots=6), state_layout="vk"))
run("many_short", lambda: prefill(synthetic.make(([0, 1, 5, 63, 64, 65, 130, 17] * 40), Hk=1, Hv=2,
                                                 K=128, V=128, seed=77, state="pool", num_slots=330)))
w = synthetic.make([1] * 200, Hk=4, Hv=8, K=128, V=128, seed=2, state="pool", num_slots=260)
d = to_dev(w)
def dec(layout):
    pool = d["state"].clone()
    o = kda.decode(d["q"], d["k"], d["v"], d["g"], d["beta"], pool, d["state_indices"], state_layout=layout)
    return o, pool, kda.decode.last_workspace
run("decode", lambda: dec("kv"))
run("decode_vk", lambda: dec("vk"))
torch.save(out, sys.argv[3])
print("ok", sorted(out))
'''


def _child(mode, path):
    env = dict(os.environ)
    env.pop("KDA_DEBUG", None)
    if mode == "debug":
        env["KDA_DEBUG"] = "1"
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, mode, path], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]


def test_debug_build_clean_and_bit_identical(tmp_path):
    import torch
    _child("release", str(tmp_path / "release.pt"))
    _child("debug", str(tmp_path / "debug.pt"))
    a, b = torch.load(tmp_path / "release.pt"), torch.load(tmp_path / "debug.pt")
    assert sorted(a) == sorted(b)
    for name in a:
        for x, y in zip(a[name], b[name]):
            assert torch.equal(x, y), name
