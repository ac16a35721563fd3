"""Benchmark of the chunked KDA prefill (tokens/s) on the throughput workload.

Workload: 32768 packed tokens in 16 sequences (lengths log-uniform in [64, 8192],
rescaled), Hk = Hv = 32, K = V = 128, bf16 q/k/v, fp32 g/beta, fp32 state pool of
256 slots updated in place.  One step = one kda_chunk_prefill call over the whole
batch.  Inputs (1.68 GB per step) are larger than L2, so no flush is needed.

Prints one JSON line.  --impl reference times the fp64 CPU oracle instead.
Multi-GPU (torchrun): every rank runs the same workload on its own GPU
(replicas, no collective on the data path); value = tokens of all ranks / max time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "KDA prefill tokens/s at Hv=32,K=V=128 (1 GB300); % of HBM/tensor roofline"
# The oracle runs the whole workload (every sequence and v-head, ~2 s on 16 host threads,
# ~35 core-seconds); a smaller head count can be passed to cpu_baseline for quick runs.
SAMPLE_HEADS = 32


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def _traffic_from_profile(summary="kda_prefill_tc_traffic.txt", source="kda_prefill_tc.cu"):
    """DRAM bytes per launch from a committed ncu summary, or None if the kernel
    source changed since those counters were taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", summary)
    src = os.path.join(ROOT, "linear_attention_prefill_chunked_gb300", "csrc", source)
    if not (os.path.exists(p) and os.path.exists(src)):
        return None
    kv = {}
    with open(p) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                a, b = line.split(":", 1)
                kv[a.strip()] = b.strip()
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    if kv.get("kernel_sha256_prefix") != sha:
        return None
    return int(kv["bytes_per_launch"])


def algorithmic_bytes(w, gate_act=False, scalar_gate=False):
    """Bytes the path must move once: q, k, v, g (or the gate pre-activation a with A_log and
    dt_bias), beta in; o out; pool rows in and out."""
    T, Hk, K = w.q.shape
    Hv, V = w.v.shape[1], w.v.shape[2]
    e = w.q.element_size()
    se = w.state.element_size() if w.state is not None else 4
    if scalar_gate:
        gate = T * Hv * 4
    else:
        gate = (T * Hv * K * e + Hv * 4 + Hv * K * 4) if gate_act else T * Hv * K * 4
    return (T * Hk * K * e * 2 + T * Hv * V * e + gate + T * Hv * 4 + T * Hv * V * e
            + w.N * Hv * K * V * se * 2)


def algorithmic_flops(w):
    """MMA FLOPs of the chunked form, counting triangles, exact for partial chunks."""
    K, V, Hv = w.q.shape[2], w.v.shape[2], w.v.shape[1]
    tot = 0
    for L in w.lens:
        for c0 in range(0, L, 64):
            c = min(64, L - c0)
            tri_s, tri = c * (c - 1) // 2, c * (c + 1) // 2
            tot += (2 * tri_s * K + 2 * tri * (K + V + K + V) + c ** 3 // 3 + 3 * 2 * c * K * V)
    return tot * Hv


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        # raw samples: KDA_BENCH_CLOCKS_DIR if set, else the system temporary directory
        d = os.environ.get("KDA_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"kda_bench_clocks_rank{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        return dist, ws, rank, local
    return None, 1, 0, local


def max_over_ranks(dist, x):
    """Largest of the ranks' x (x itself without a process group).  Every rank must call it.
    NCCL reduces a tensor on the rank's GPU, gloo one in host memory."""
    if not dist:
        return x
    dev = (torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl"
           else torch.device("cpu"))
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(ws, units_per_rank, ms):
    """Whole-job throughput: the units all ws replicas processed over the slowest one's time."""
    return ws * units_per_rank / (ms * 1e-3)


def cpu_baseline(w, num_threads=0, heads=SAMPLE_HEADS):
    """Time the fp64 oracle on a bounded sample: all sequences, v-heads 0..heads-1."""
    from oracle import kda_oracle
    H = min(heads, w.v.shape[1])
    hk = max(1, H * w.q.shape[1] // w.v.shape[1])
    kda_oracle.build()
    args = (w.q[:, :hk].contiguous(), w.k[:, :hk].contiguous(), w.v[:, :H].contiguous(),
            w.g[:, :H].contiguous(), w.beta[:, :H].contiguous(), w.cu_seqlens)
    t0 = time.perf_counter()
    kda_oracle.recurrence(*args, scale=w.scale, state=w.state[:, :H].contiguous(),
                          state_indices=w.state_indices, num_threads=num_threads)
    dt = time.perf_counter() - t0
    cores = num_threads if num_threads > 0 else (os.cpu_count() or 1)
    frac = H / w.v.shape[1]
    return {"value": w.T * frac / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": (f"the whole workload: all {w.N} sequences ({w.T} tokens) and all {H} v-heads, "
                       f"fp64 token-by-token, {dt:.2f} s" if frac == 1 else
                       f"all {w.N} sequences ({w.T} tokens), v-heads 0-{H - 1} of {w.v.shape[1]} "
                       f"({frac:.3f} of the work), fp64 token-by-token, {dt:.2f} s; value scaled "
                       f"to full-width tokens")}


def per_core_rate(w, tokens=4096):
    """The oracle on one core: one (sequence, v-head) pair of ``tokens`` tokens (the first
    tokens of the longest sequence, head 0), in tokens per second per core."""
    from oracle import kda_oracle
    n = max(range(w.N), key=lambda i: w.lens[i])
    a = int(w.cu_seqlens[n])
    L = min(tokens, w.lens[n])
    sl = slice(a, a + L)
    t0 = time.perf_counter()
    kda_oracle.recurrence(w.q[sl, :1], w.k[sl, :1], w.v[sl, :1], w.g[sl, :1], w.beta[sl, :1],
                          [0, L], scale=w.scale, num_threads=1)
    dt = time.perf_counter() - t0
    return {"value": L / dt, "unit": "tokens/s per core (one v-head)",
            "sample": f"one (sequence, v-head) pair of {L} tokens on 1 thread, {dt:.3f} s"}


def config_parity(dev):
    """Each workload configuration once more on the GPU from fresh inputs, against the oracle
    (wall time and host threads of the oracle, relative L2 of o and of the final states over
    the whole tensor).  The decode configuration runs 512 of its rows on a 1024-slot pool;
    the test suite compares all 4032 of them."""
    import numpy as np

    import linear_attention_prefill_chunked_gb300 as kda
    from linear_attention_prefill_chunked_gb300 import synthetic
    from oracle import kda_oracle

    def rel(x, ref):
        x = x.detach().cpu().double().numpy() if hasattr(x, "detach") else np.asarray(x)
        return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))

    t = lambda x: None if x is None else x.to(dev).contiguous()
    out = {}
    cases = [("tiny_varlen", synthetic.tiny_varlen(), False),
             ("pool_varlen_fp32_pool", synthetic.pool_varlen(), True),
             ("pool_varlen_bf16_pool", synthetic.pool_varlen(state_dtype=torch.bfloat16), True),
             ("large_decay", synthetic.large_decay(), True),
             ("throughput", synthetic.throughput(), True)]
    for name, w, pool_mode in cases:
        st = t(w.state)
        o, fin = kda.chunk_prefill(t(w.q), t(w.k), t(w.v), t(w.g), t(w.beta), t(w.cu_seqlens),
                                   state=st, state_indices=t(w.state_indices) if pool_mode else None)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        o_ref, s_ref = kda_oracle.recurrence(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens,
                                             scale=w.scale, state=w.state,
                                             state_indices=w.state_indices if pool_mode else None)
        dt = time.perf_counter() - t0
        if pool_mode:  # the written rows
            sl = torch.where(w.state_indices >= 0, w.state_indices,
                             torch.full_like(w.state_indices, w.state.shape[0] - 1)).long()
            e_s = rel(st[sl.to(dev)], s_ref[sl.numpy()])
        else:
            e_s = rel(fin, s_ref)
        out[name] = {"rel_l2_o": rel(o, o_ref), "rel_l2_state": e_s,
                     "finite": bool(torch.isfinite(o).all()), "oracle_s": round(dt, 3),
                     "oracle_threads": os.cpu_count()}
    w = synthetic.decode_batch(num_rows=512, num_pad=8, num_slots=1024, pool_device=dev)
    real = np.flatnonzero(w.state_indices.numpy() >= 0)
    slots = w.state_indices[real].long()
    before = w.state[slots.to(dev)].cpu()
    o = kda.decode(t(w.q), t(w.k), t(w.v), t(w.g), t(w.beta), w.state, t(w.state_indices))
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    o_ref, s_ref = kda_oracle.recurrence(w.q[real], w.k[real], w.v[real], w.g[real], w.beta[real],
                                         np.arange(real.size + 1), scale=w.scale, state=before)
    dt = time.perf_counter() - t0
    out["decode_512_rows"] = {"rel_l2_o": rel(o[torch.from_numpy(real).to(dev)], o_ref),
                              "rel_l2_state": rel(w.state[slots.to(dev)], s_ref),
                              "finite": bool(torch.isfinite(o).all()), "oracle_s": round(dt, 3),
                              "oracle_threads": os.cpu_count()}
    return out


def e2e_pipelined(w, dev, stream, pool, ws_t, act, act_dev, steps):
    """End to end through the public API (chunk_prefill / chunk_prefill_act) from pinned host
    memory: every step copies its inputs host -> device and reads its output o back.  Steps
    run as a pipeline over two device input sets: the copy-in of step i+1 (on one copy stream)
    and the read-back of step i-1 (on another) overlap the prefill of step i, each stream
    waiting on events only.  Returns (ms per step, host->device and device->host bytes per
    step); the time runs from the first copy-in to the end of the last read-back."""
    import linear_attention_prefill_chunked_gb300 as kda
    host = [x.contiguous().pin_memory() for x in
            (w.q, w.k, w.v, act_dev[0] if act else w.g, w.beta, w.cu_seqlens, w.state_indices)]
    h_out = [torch.empty((w.T, 32, 128), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    sets = [[torch.empty_like(x, device=dev) for x in host] for _ in range(2)]
    outs = [torch.empty((w.T, 32, 128), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in host)
    d2h = h_out[0].numel() * h_out[0].element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=False)

    def run(n):
        e_in, e_done, e_out = [None] * n, [None] * n, [None] * n
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(e_done[i - 2])   # set b no longer read by step i-2
                for d, h in zip(sets[b], host):
                    d.copy_(h, non_blocking=True)
                e_in[i] = ev()
                e_in[i].record(s_in)
            stream.wait_event(e_in[i])
            if i >= 2:
                stream.wait_event(e_out[i - 2])      # out b read back
            dq, dk, dv, dg, db, dcu, didx = sets[b]
            if act:
                kda.chunk_prefill_act(dq, dk, dv, dg, act_dev[1], act_dev[2], db, dcu, state=pool,
                                      state_indices=didx, out=outs[b], workspace=ws_t,
                                      stream=stream)
            else:
                kda.chunk_prefill(dq, dk, dv, dg, db, dcu, state=pool, state_indices=didx,
                                  out=outs[b], workspace=ws_t, stream=stream)
            e_done[i] = ev()
            e_done[i].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(e_done[i])
                h_out[b].copy_(outs[b], non_blocking=True)
                e_out[i] = ev()
                e_out[i].record(s_out)
        return e_out[n - 1]

    run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    last = run(steps)
    s_in.wait_event(last)
    e1.record(s_in)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, h2d, d2h


def run_reference(args, dist, ws, rank):
    from linear_attention_prefill_chunked_gb300 import synthetic
    if rank != 0:
        return
    w = synthetic.throughput()
    times = []
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline(w)
        if i >= args.warmup:
            times.append(cb)
    val = statistics.median(t["value"] for t in times)
    ms = w.T / val * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "tokens": w.T, "num_seqs": w.N, "Hk": 32, "Hv": 32,
                       "K": 128, "V": 128,
                       "parallelism": "host threads over (sequence, head); rank 0 only"},
            "cpu_baseline": {k: times[-1][k] for k in ("kind", "cores", "sample")} | {"value": val,
                                                                                      "unit": "tokens/s"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def run_decode(args, dist, ws, rank, local):
    """Decode of 4096 one-token rows (64 padding rows on the sentinel) on an 8192-slot fp32
    pool (16 GiB, resident): real rows per second, against the HBM roofline of streaming
    each row's state tile in and out once (4,243,584 bytes per real row)."""
    import linear_attention_prefill_chunked_gb300 as kda
    from linear_attention_prefill_chunked_gb300 import synthetic

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kda.load()
    if args.workload == "decode_small":  # 512 rows on a 2 GiB pool: small enough for an ncu capture
        w = synthetic.decode_batch(num_rows=512, num_pad=8, num_slots=1024, pool_device=dev)
    else:
        w = synthetic.decode_batch(pool_device=dev)
    t = lambda x: x.to(dev).contiguous()
    q, k, v, g, beta, idx = (t(x) for x in (w.q, w.k, w.v, w.g, w.beta, w.state_indices))
    pool = w.state
    out = torch.empty_like(v)
    stream = torch.cuda.current_stream(dev)
    step = lambda: kda.decode(q, k, v, g, beta, pool, idx, out=out, stream=stream)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        for i in range(args.steps):
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in ev]
    ms = max_over_ranks(dist, statistics.median(per))
    if rank != 0:
        return
    real = int((w.state_indices >= 0).sum())
    Hv, K, V = w.v.shape[1], w.q.shape[2], w.v.shape[2]
    row_bytes = 2 * Hv * K * V * 4 + Hv * (2 * K * 2 + V * 2 + K * 4 + 4 + V * 2)
    hbm, _, src = _peaks()
    achieved = real * row_bytes / (ms * 1e-3) / 1e9
    print(json.dumps({
        "metric": f"KDA decode rows/s ({w.N} one-token rows, Hv=32, K=V=128, fp32 pool)",
        "value": job_rate(ws, real, ms), "unit": "rows/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "real_rows": real, "padding_rows": w.N - real,
                   "pool": f"fp32 [{pool.shape[0]}, 32, 128, 128], resident",
                   "l2": f"state tiles ({pool.numel() * 4 / 2**30:.0f} GiB pool) larger than L2, no flush"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm,
                     "traffic": (_traffic_from_profile("kda_decode_traffic.txt", "kda_decode.cu")
                                 if args.workload == "decode" else None),
                     "peak_source": src,
                     "algorithmic_bytes_per_launch": real * row_bytes},
        "clocks": clk.summary(), "gpu_launches": args.steps}), flush=True)


def run_ours(args, dist, ws, rank, local):
    import linear_attention_prefill_chunked_gb300 as kda
    from linear_attention_prefill_chunked_gb300 import synthetic

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    kda.load()
    if args.workload == "profile":
        w = synthetic.make([1024] * 8, Hk=32, Hv=32, K=128, V=128, seed=5, state="pool",
                           num_slots=16, name="profile_8x1024_Hv32_K128")
    elif args.workload == "many_short":  # 8192 prompts of 1..8 tokens: the work-list order step
        gen = torch.Generator().manual_seed(8192)
        lens = torch.randint(1, 9, (8192,), generator=gen).tolist()
        w = synthetic.make(lens, Hk=32, Hv=32, K=128, V=128, gen=gen, state="pool",
                           num_slots=8193, name="many_short_8192seq_Hv32_K128")
    else:
        w = synthetic.throughput()
    act = args.gate == "act"
    if args.gate == "scalar":  # one log-decay per (token, head): the GDN form
        w.g = synthetic.scalar_gate_inputs(w.T, 32, seed=0)
        w.name += "_scalar_gate"
    if act:  # the kernel computes the gate from a bf16 pre-activation
        a_h, A_log_h, dtb_h = synthetic.gate_act_inputs(w.T, 32, 128, seed=0)
        w.name += "_gate_act"
    t = lambda x: x.to(dev).contiguous()
    q, k, v, g, beta, cu, idx = (t(x) for x in (w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens,
                                                 w.state_indices))
    if act:
        a_d, A_log_d, dtb_d = t(a_h), t(A_log_h), t(dtb_h)
    pool = t(w.state)
    out = torch.empty((w.T, 32, 128), dtype=torch.bfloat16, device=dev)
    desc = kda.make_desc(num_seqs=w.N, total_tokens=w.T, Hk=32, Hv=32, K=128, V=128,
                         qkv_dtype=torch.bfloat16, num_slots=pool.shape[0])
    path = kda.prefill_path(desc)
    ws_t = torch.empty(kda.prefill_workspace_size(desc), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        if act:
            kda.chunk_prefill_act(q, k, v, a_d, A_log_d, dtb_d, beta, cu, state=pool,
                                  state_indices=idx, out=out, workspace=ws_t, stream=stream,
                                  qk_l2norm=args.qk_l2norm)
        else:
            kda.chunk_prefill(q, k, v, g, beta, cu, state=pool, state_indices=idx, out=out,
                              workspace=ws_t, stream=stream, qk_l2norm=args.qk_l2norm)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        # untimed calls for about a second with the clock sampler running, so that its record
        # covers the GPU under sustained load right up to (and through) the timed steps
        soak = 0
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < args.clock_soak_s:
            for _ in range(10):
                step()
            soak += 10
            torch.cuda.synchronize()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    per = [a.elapsed_time(b) for a, b in ev]  # ms, one launch sequence each
    total_ms = max_over_ranks(dist, sum(per))
    if dist:
        dist.barrier()
    bits = kda.read_device_status(ws_t)

    e2e_ms, h2d, d2h = None, 0, 0
    if not args.no_e2e:
        e2e_ms, h2d, d2h = e2e_pipelined(w, dev, stream, pool, ws_t, act,
                                         (a_h, A_log_d, dtb_d) if act else None, args.e2e_steps)
        e2e_ms = max_over_ranks(dist, e2e_ms)

    if rank != 0:
        return
    hbm, bf16, src = _peaks()
    ms = total_ms / args.steps  # mean over the timed steps, used for value and roofline alike
    value = job_rate(ws, w.T, ms)
    nbytes = algorithmic_bytes(w, act, args.gate == "scalar")
    flops = algorithmic_flops(w)
    kern_ms = ms
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    t_roof = max(nbytes / (hbm * 1e9), flops / (bf16 * 1e12))
    traffic = _traffic_from_profile() if path == 1 else None
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.T, "num_seqs": w.N, "Hk": 32, "Hv": 32,
                   "K": 128, "V": 128, "chunk": 64, "state_pool": "fp32, 256 slots, in place",
                   "kernel_path": "tcgen05 fused" if path == 1 else "CUDA-core fp32",
                   "gate": ("in-kernel activation of a bf16 pre-activation" if act
                            else "fp32 log-decay per token and head (scalar, GDN)"
                            if args.gate == "scalar" else "fp32 log-decay input"),
                   "qk_l2norm": "in kernel" if args.qk_l2norm else "by the caller",
                   "l2": f"inputs larger than L2 ({nbytes / 1e9:.2f} GB per step), no flush",
                   "parallelism": f"replicas x{ws}" if ws > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else src,
                     "algorithmic_bytes_per_launch": nbytes, "algorithmic_flops_per_launch": flops,
                     "roofline_time_ms": t_roof * 1e3, "frac_of_roofline_time": t_roof * 1e3 / kern_ms},
        "clocks": clk.summary() | {"window": f"{soak} untimed calls over ~{args.clock_soak_s:g} s of "
                                             f"sustained load, then the {args.steps} timed steps"},
        "e2e": {"value": job_rate(ws, w.T, e2e_ms) if e2e_ms else None, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": f"each step copies its pinned host q/k/v/{'a' if act else 'g'}/beta/cu_seqlens/"
                        "indices in and reads o back; steps are pipelined over two device input "
                        "sets (copies of step i+1 and the read-back of step i-1 overlap the "
                        "prefill of step i); the state pool stays resident on the device"},
        # tensor-core path: planning + prefill + combine (the combine returns at once when
        # nothing was cut); CUDA-core path: the prefill
        "gpu_launches": args.steps * (3 if path == 1 else 1),
        "device_status": bits, "wall_s": wall,
    }
    if ws == 1 and not args.no_cpu_baseline:
        if act:  # the oracle gets the gate its own activation computes from a
            from oracle import kda_oracle
            w.g = torch.from_numpy(kda_oracle.gate_activation(a_h, A_log_h, dtb_h)).float()
        line["cpu_baseline"] = cpu_baseline(w)
        line["cpu_baseline"]["per_core"] = per_core_rate(w)
        if not args.no_parity and args.workload == "throughput" and args.gate == "given" \
                and not args.qk_l2norm:
            line["parity"] = config_parity(dev)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--no-parity", action="store_true",
                    help="skip the per-configuration oracle comparison of the default run")
    ap.add_argument("--clock-soak-s", type=float, default=1.0,
                    help="seconds of untimed calls, clock sampler running, before the timed steps")
    ap.add_argument("--gate", default="given", choices=["given", "act", "scalar"],
                    help="act: the gate computed in the kernel from a bf16 pre-activation "
                         "(kda_chunk_prefill_act); scalar: one log-decay per token and head")
    ap.add_argument("--qk-l2norm", action="store_true",
                    help="normalise q and k inside the kernel (KDA_FLAG_QK_L2NORM)")
    ap.add_argument("--workload", default="throughput",
                    choices=["throughput", "profile", "many_short", "decode", "decode_small"],
                    help="profile: 8 x 1024 tokens, Hv=32; decode_small: 512 decode rows on a "
                         "2 GiB pool (smaller cases for ncu captures); many_short: 8192 "
                         "sequences of 1 to 8 tokens")
    args = ap.parse_args()
    dist, ws, rank, local = _dist()
    try:
        if args.impl == "reference":
            run_reference(args, dist, ws, rank)
        else:
            (run_decode if args.workload.startswith("decode") else run_ours)(args, dist, ws, rank, local)
    finally:
        if dist:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
