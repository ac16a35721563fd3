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
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(local) as clk:
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

    # End to end through the public API from pinned host buffers (copies inside).
    e2e_ms, h2d, d2h = None, 0, 0
    if not args.no_e2e:
        hq, hk, hv, hg, hb, hcu, hidx = (x.contiguous().pin_memory() for x in
                                         (w.q, w.k, w.v, a_h if act else w.g, w.beta,
                                          w.cu_seqlens, w.state_indices))
        h_out = torch.empty((w.T, 32, 128), dtype=torch.bfloat16).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hg, hb, hcu, hidx))
        d2h = h_out.numel() * h_out.element_size()

        def e2e_step():
            dq, dk, dv, dg, db, dcu, didx = (x.to(dev, non_blocking=True) for x in
                                             (hq, hk, hv, hg, hb, hcu, hidx))
            if act:
                o, _ = kda.chunk_prefill_act(dq, dk, dv, dg, A_log_d, dtb_d, db, dcu, state=pool,
                                             state_indices=didx, workspace=ws_t, stream=stream)
            else:
                o, _ = kda.chunk_prefill(dq, dk, dv, dg, db, dcu, state=pool, state_indices=didx,
                                         workspace=ws_t, stream=stream)
            h_out.copy_(o, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e2e_steps = max(2, min(args.steps, 5))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(dist, e0.elapsed_time(e1) / e2e_steps)

    if rank != 0:
        return
    hbm, bf16, src = _peaks()
    ms = total_ms / args.steps
    value = job_rate(ws, w.T, ms)
    nbytes = algorithmic_bytes(w, act, args.gate == "scalar")
    flops = algorithmic_flops(w)
    kern_ms = statistics.median(per)
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
        "clocks": clk.summary(),
        "e2e": {"value": job_rate(ws, w.T, e2e_ms) if e2e_ms else None, "unit": "tokens/s",
                "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": f"pinned host q/k/v/{'a' if act else 'g'}/beta/cu_seqlens/indices copied in, "
                        "o copied out each step; the state pool stays resident on the device"},
        "gpu_launches": args.steps * (2 if path == 1 else 1),
        "device_status": bits, "wall_s": wall,
    }
    if ws == 1 and not args.no_cpu_baseline:
        if act:  # the oracle gets the gate its own activation computes from a
            from oracle import kda_oracle
            w.g = torch.from_numpy(kda_oracle.gate_activation(a_h, A_log_h, dtb_h)).float()
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
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
