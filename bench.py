"""Benchmark of the ParisKV decode step on GB300.

One step = one decode step of one layer of the Llama-3.1-8B-shaped workload:
paris_append_decode (new token per KV head, flush every 128 steps),
paris_retrieve (32 query heads over a 131072-token context) and
paris_sparse_attend.  Layer contexts are rotated so the working set is far
larger than L2.  Prints one JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "keys scanned/s & µs per decode step (frac. of HBM peak); recall@k vs exact top-k"
UNIT = "keys/s"

WORKLOADS = {
    # Llama-3.1-8B-shaped decode layer: batch 1, 32 q / 8 KV heads, d = 128,
    # 131072-token bf16 context, sink 16, local 512, update buffer 128,
    # B = 16 (m = 8), rho = 4, candidates 5%, k = 1024.
    "llama8b-128k": dict(batch=1, n_kv_heads=8, n_q_heads=32, head_dim=128, n_sub=16, rho=4, sink=16, local=512,
                         update_buf=128, topk=1024, cand_bp=500, context=131072, layers=8),
    # the same layer shape, 32 layer contexts: one captured graph steps a token
    # through every layer (the whole model's decode-time retrieval and attention)
    "llama8b-128k-32l": dict(batch=1, n_kv_heads=8, n_q_heads=32, head_dim=128, n_sub=16, rho=4, sink=16,
                             local=512, update_buf=128, topk=1024, cand_bp=500, context=131072, layers=32),
    # the 32 layers with each layer's Retrieval-zone K/V in pinned host memory (UVA, ~17 GB pinned in all)
    "llama8b-128k-32l-uva": dict(batch=1, n_kv_heads=8, n_q_heads=32, head_dim=128, n_sub=16, rho=4, sink=16,
                                 local=512, update_buf=128, topk=1024, cand_bp=500, context=131072, layers=32,
                                 retrieval_on_host=1),
    # the small case the oracle finishes in seconds
    "tiny-4k": dict(batch=1, n_kv_heads=1, n_q_heads=1, head_dim=128, n_sub=16, rho=4, sink=0, local=0,
                    update_buf=128, topk=64, cand_bp=1000, context=4096, layers=64),
    # Qwen3-8B-shaped long generation: batch 8, 32768-token prompt, decode keys
    # drifting by 0.02 sigma per 256 steps, the Update Buffer flushed every 128
    "qwen3-8b-drift": dict(batch=8, n_kv_heads=8, n_q_heads=32, head_dim=128, n_sub=16, rho=4, sink=16,
                           local=512, update_buf=128, topk=1024, cand_bp=500, context=32768, layers=8, drift=0.02),
    # 1M-token context, Retrieval-zone K/V in pinned host memory read through UVA
    "1m-uva": dict(batch=1, n_kv_heads=8, n_q_heads=32, head_dim=128, n_sub=16, rho=4, sink=16, local=512,
                   update_buf=128, topk=2048, cand_bp=500, context=1048576, layers=2, retrieval_on_host=1),
    # the 128K-token layer with its Retrieval-zone K/V in pinned host memory (UVA)
    "llama8b-128k-uva": dict(batch=1, n_kv_heads=8, n_q_heads=32, head_dim=128, n_sub=16, rho=4, sink=16,
                             local=512, update_buf=128, topk=1024, cand_bp=500, context=131072, layers=8,
                             retrieval_on_host=1),
    # the same 1M-token context with the whole cache in HBM (it fits: ~4 GiB per layer of 280 GB)
    "1m-hbm": dict(batch=1, n_kv_heads=8, n_q_heads=32, head_dim=128, n_sub=16, rho=4, sink=16, local=512,
                   update_buf=128, topk=2048, cand_bp=500, context=1048576, layers=2, retrieval_on_host=0),
    # one point of the 256K batch-5 sweep (candidate fraction, rho and k from the command line)
    "sweep-256k": dict(batch=5, n_kv_heads=8, n_q_heads=32, head_dim=128, n_sub=16, rho=4, sink=16, local=512,
                       update_buf=128, topk=1024, cand_bp=500, context=262144, layers=4),
}
DESCRIPTION = {
    "llama8b-128k": "Llama-3.1-8B-shaped decode layer, 131072-token context",
    "tiny-4k": "one KV head, 4096 float32 keys",
    "llama8b-128k-32l": "Llama-3.1-8B-shaped decode, 32 layers of 131072-token context",
    "llama8b-128k-32l-uva": "Llama-3.1-8B-shaped decode, 32 layers of 131072-token context, "
                            "Retrieval-zone K/V in pinned host memory (UVA)",
    "qwen3-8b-drift": "Qwen3-8B-shaped long generation, batch 8, 32768-token prompt, drifting decode keys",
    "1m-uva": "1M-token context, Retrieval-zone K/V in pinned host memory (UVA)",
    "1m-hbm": "1M-token context, the whole cache in HBM",
    "llama8b-128k-uva": "Llama-3.1-8B-shaped decode layer, 131072-token context, Retrieval-zone K/V in pinned host memory (UVA)",
    "sweep-256k": "256K-token context, batch 5 (one point of the candidate-fraction x rho x k sweep)",
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


TRAFFIC_SOURCES = {  # each kernel's source file and the headers it includes
    "decode": ["kernels_decode.cu", "paris_device.cuh", "paris_internal.cuh"],
    "dense": ["kernels_dense.cu", "paris_device.cuh", "paris_internal.cuh"],
}


TRAFFIC_WORKLOAD = "llama8b-128k"  # the workload the committed counters were taken on


def traffic_record(kernel: str, args):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when the kernel's source changed since the counters were taken or
    the run is not the one they were taken on (its workload at its own
    parameters, top-k best first: the bytes of a launch depend on them)."""
    if args.workload != TRAFFIC_WORKLOAD or args.cand_bp or args.rho or args.topk or args.topk_order != "score":
        return None
    import hashlib
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path) or kernel not in TRAFFIC_SOURCES:
        return None
    src = b"".join(open(os.path.join(ROOT, "long_context_kv_gb300", "csrc", f), "rb").read()
                   for f in TRAFFIC_SOURCES[kernel])
    sha = hashlib.sha1(src).hexdigest()[:12]
    for line in open(path):
        parts = line.split()
        if len(parts) >= 3 and not line.startswith("#") and parts[0] == kernel and parts[1] == sha:
            return float(parts[2])
    return None


# ---------------------------------------------------------------------------
# ranks (one process per GPU; every rank runs its own replica of the workload)
# ---------------------------------------------------------------------------
def rank_seed(rank: int, layer: int) -> int:
    """Seed of a rank's layer context: ranks draw disjoint synthetic inputs."""
    return 20260202 + 1 + 1000 * rank + layer


def rank_barrier(dist: bool) -> None:
    if dist:
        import torch.distributed as tdist
        tdist.barrier()


def max_over_ranks_of(x: float, dist: bool, device: str) -> float:
    """The largest x over all ranks (the job's time is its slowest rank's)."""
    if not dist:
        return x
    import torch
    import torch.distributed as tdist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(keys_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job keys per second: every rank scans its own keys_per_rank in
    the timed region, and the job takes the slowest rank's ms_max."""
    return keys_per_rank * world / (ms_max / 1e3)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_config(args, world) -> dict:
    """The JSON line's config: the workload with the parameters it runs at."""
    w = workload_of(args)
    nl = args.layers or w["layers"]
    return {"workload": DESCRIPTION[args.workload], "batch": w["batch"], "n_q_heads": w["n_q_heads"],
            "n_kv_heads": w["n_kv_heads"], "head_dim": w["head_dim"], "context": w["context"], "sink": w["sink"],
            "local": w["local"], "update_buf": w["update_buf"], "n_sub": w["n_sub"], "rho": w["rho"],
            "cand_pct": w["cand_bp"] / 100, "topk": w["topk"], "topk_order": args.topk_order,
            "retrieval_on_host": w.get("retrieval_on_host", 0), "drift_sigma_per_256_steps": w.get("drift", 0.0),
            "kv_dtype": "f32" if args.workload == "tiny-4k" else "bf16", "layers_rotated": nl,
            "l2": f"inputs larger than L2: {nl} layer contexts rotated, each revisited after "
                  f"{nl - 1} other layers' steps", "parallelism": f"replicas x{world}"}


def run_ours(args, rank, world):
    import numpy as np
    import torch

    from long_context_kv_gb300 import build as B
    from long_context_kv_gb300 import paris as P
    from long_context_kv_gb300 import synth

    dev = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev)
    B.build()
    P.load()
    w = workload_of(args)
    nl = args.layers or w["layers"]
    ctxlen, d = w["context"], w["head_dim"]
    b, hkv, hq, S = w["batch"], w["n_kv_heads"], w["n_q_heads"], w["sink"]
    # inputs per layer: every timed and untimed step below, plus up to one
    # Update Buffer's worth of steps to bring each layer to a flushing append
    per_layer_steps = (args.warmup + 8 * args.steps + 64 + nl - 1) // nl + w["update_buf"] + 4
    max_ctx = ctxlen + per_layer_steps + 8
    fdt = torch.bfloat16 if args.workload != "tiny-4k" else torch.float32
    gen = torch.Generator(device="cuda")
    layers = []
    keep_keys = None
    t_setup = time.time()
    for li in range(nl):
        seed = rank_seed(rank, li)
        cfg = P.make_config(batch=b, n_kv_heads=hkv, n_q_heads=hq, head_dim=d, n_sub=w["n_sub"], rho=w["rho"],
                            sink=S, local=w["local"], update_buf=w["update_buf"], topk=w["topk"],
                            cand_bp=w["cand_bp"], max_ctx=max_ctx, retrieval_on_host=w.get("retrieval_on_host", 0),
                            topk_order=P.PARIS_TOPK_BY_POSITION if args.topk_order == "position" else P.PARIS_TOPK_BY_SCORE)
        ctx = P.Context(cfg, synth.srht_signs(seed, d))
        scale = torch.from_numpy(synth.channel_scale(seed, hkv, d)).cuda()
        gen.manual_seed(seed)
        K = (torch.randn((b, hkv, ctxlen, d), generator=gen, device="cuda") * scale[None, :, None, :]).to(fdt)
        V = torch.randn((b, hkv, ctxlen, d), generator=gen, device="cuda").to(fdt)
        ctx.paris_encode_prefill(K, V, ctxlen)
        st = ctx.paris_get_state()
        N0 = st["N"]
        # per decode step of this layer: new token and the query (a Retrieval-zone key + N(0, 0.5^2))
        kn = torch.randn((per_layer_steps, b, hkv, d), generator=gen, device="cuda") * scale[None, None]
        if w.get("drift"):
            # mu(t) = rate (t / 256) delta s, delta a fixed random +-1 vector per KV head
            delta = torch.randint(0, 2, (hkv, d), generator=gen, device="cuda").float() * 2 - 1
            t = torch.arange(per_layer_steps, device="cuda", dtype=torch.float32) * nl + li
            kn = kn + w["drift"] * (t / 256.0)[:, None, None, None] * (delta * scale)[None, None]
        kn = kn.to(fdt)
        vn = torch.randn((per_layer_steps, b, hkv, d), generator=gen, device="cuda").to(fdt)
        pos = torch.randint(S, S + N0, (per_layer_steps, b, hq), generator=gen, device="cuda")
        kvh_of = torch.arange(hq, device="cuda") // (hq // hkv)
        picked = K[torch.arange(b, device="cuda")[None, :, None], kvh_of[None, None, :], pos].float()
        qs = (picked + 0.5 * torch.randn(picked.shape, generator=gen, device="cuda")).to(fdt).contiguous()
        if li == 0:
            keep_keys = K  # layer 0 keys, for recall
        del K, V, picked
        idx = torch.empty((b, hq, w["topk"]), dtype=torch.int32, device="cuda")
        sc = torch.empty((b, hq, w["topk"]), dtype=torch.float32, device="cuda")
        out = torch.empty((b, hq, d), dtype=torch.bfloat16, device="cuda")
        layers.append(dict(ctx=ctx, kn=kn, vn=vn, qs=qs, idx=idx, sc=sc, out=out, step=0, N0=N0))
    torch.cuda.synchronize()
    log(f"[rank {rank}] setup {time.time() - t_setup:.1f}s, {nl} layer contexts, "
        f"{torch.cuda.memory_allocated() / 2**30:.1f} GiB allocated by torch")

    def step_layer(L):
        j = L["step"]
        L["step"] = j + 1
        L["ctx"].paris_decode_step(L["kn"][j], L["vn"][j], L["qs"][j], L["idx"], L["sc"], L["out"])

    def step(i):
        step_layer(layers[i % nl])

    if args.profile_case:
        # the decode steps, then as many standalone sparse-attention calls
        # (over each layer's last top-k), dense-attention calls and GQA-shared
        # attention calls on the same caches
        for i in range(args.warmup + args.steps):
            step(i)
        for i in range(args.warmup + args.steps):
            L = layers[i % nl]
            L["ctx"].paris_sparse_attend(L["qs"][0], L["idx"], L["out"])
        for i in range(args.warmup + args.steps):
            L = layers[i % nl]
            L["ctx"].paris_dense_attend(L["qs"][0], L["out"])
        for i in range(args.warmup + args.steps):
            L = layers[i % nl]
            L["ctx"].paris_sparse_attend_gqa(L["qs"][0], L["idx"], L["out"])
        torch.cuda.synchronize()
        return {"profile_case": DESCRIPTION[args.workload], "layers": nl, "steps": args.warmup + args.steps}

    dist = world > 1

    def barrier():
        torch.cuda.synchronize()
        rank_barrier(dist)

    def max_over_ranks(x):
        return max_over_ranks_of(x, dist, "cuda")

    i = 0
    for _ in range(args.warmup):
        step(i)
        i += 1
    stream = torch.cuda.current_stream()

    def timed(fn):
        barrier()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(torch.cuda.current_stream())
        fn()
        z.record(torch.cuda.current_stream())
        barrier()
        return max_over_ranks(a.elapsed_time(z))

    # eager: every step launched from Python through the ABI
    def eager_steps():
        nonlocal i
        for _ in range(args.steps):
            step(i)
            i += 1
    ms_eager = timed(eager_steps)

    # graph: the same K decode steps captured once (positions, flushes and
    # all) and replayed; replays repeat identical, idempotent work, so the
    # replay time is the device time of those K steps without host gaps
    def capture(profile=False):
        nonlocal i
        keys = []
        cs = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        if profile:
            for L in layers:
                L["ctx"].paris_profile_begin(64 * args.steps)
        c0 = [L["ctx"].paris_launch_counts() for L in layers]
        with torch.cuda.graph(g, stream=cs):
            for _ in range(args.steps):
                keys.append(layers[i % nl]["ctx"].paris_get_state()["N"] * b * hkv)
                step(i)
                i += 1
        c1 = [L["ctx"].paris_launch_counts() for L in layers]
        n = sum(c1[li][k] - c0[li][k] for li in range(nl) for k in c1[li])
        return g, keys, n

    g_main, keys_per_step, launches = capture()
    g_main.replay()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        t_end = time.time() + 1.0
        while time.time() < t_end:  # load before the timed replay so the clock samples see it
            g_main.replay()
            torch.cuda.synchronize()
        ms = timed(g_main.replay)
        for _ in range(3):
            g_main.replay()
        torch.cuda.synchronize()
    value = job_throughput(sum(keys_per_step), world, ms)

    # the calls of the path one by one (paris_retrieve, paris_sparse_attend,
    # paris_append_decode), each as K captured calls replayed like the step
    def timed_calls(call):
        nonlocal i
        cs = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            for _ in range(args.steps):
                call(layers[i % nl], i)
                i += 1
        g.replay()
        torch.cuda.synchronize()
        return timed(g.replay) / args.steps

    def call_retrieve(L, _):
        L["ctx"].paris_retrieve(L["qs"][L["step"]], L["idx"], L["sc"])

    def call_attend(L, _):
        L["ctx"].paris_sparse_attend(L["qs"][L["step"]], L["idx"], L["out"])

    def call_append(L, _):
        j = L["step"]
        L["step"] = j + 1
        L["ctx"].paris_append_decode(L["kn"][j], L["vn"][j])

    def call_dense(L, _):
        L["ctx"].paris_dense_attend(L["qs"][L["step"]], L["out"])

    def call_gqa(L, _):
        L["ctx"].paris_sparse_attend_gqa(L["qs"][L["step"]], L["idx"], L["out"])

    keys_retrieve = sum(L["ctx"].paris_get_state()["N"] * b * hkv for L in layers) / nl
    ms_retrieve = timed_calls(call_retrieve)
    ms_attend = timed_calls(call_attend)
    ms_dense = timed_calls(call_dense)
    ms_gqa = timed_calls(call_gqa)
    # rows the GQA-shared attention reads per KV head (the union of its query heads' top-k), layer 0
    G = hq // hkv
    st0 = layers[0]["ctx"].paris_get_state()
    k_eff0 = int(st0["k_eff"])
    idx0 = layers[0]["idx"][:, :, :k_eff0].reshape(b, hkv, G * k_eff0)
    union_rows = sum(int(torch.unique(idx0[s_, h_]).numel()) for s_ in range(b) for h_ in range(hkv)) / (b * hkv)
    tokens_dense = sum(L["ctx"].paris_get_state()["T"] for L in layers) / nl
    ms_append = timed_calls(call_append)

    # a decode step whose append fills the Update Buffer: the append, the
    # flush (Local's oldest tokens join the Retrieval zone and the touched
    # chunks' index is rebuilt), then retrieval and attention.  Each layer is
    # first brought (eagerly, untimed) to the step before its next flush;
    # then one flushing step per layer is captured and replayed (idempotent:
    # the same token, the same rebuilt index, the same zones).
    U = w["update_buf"]
    for L in layers:
        while L["ctx"].paris_get_state()["n_buf"] != U - 1:
            step_layer(L)
    torch.cuda.synchronize()
    cs_f = torch.cuda.Stream()
    g_flush = torch.cuda.CUDAGraph()
    f0 = [L["ctx"].paris_launch_counts() for L in layers]
    with torch.cuda.graph(g_flush, stream=cs_f):
        for L in layers:
            step_layer(L)
    f1 = [L["ctx"].paris_launch_counts() for L in layers]
    flush_launches = {k: sum(f1[li][k] - f0[li][k] for li in range(nl)) for k in f1[0]}
    assert all(L["ctx"].paris_get_state()["n_buf"] == 0 for L in layers), "every captured step must flush"
    g_flush.replay()
    torch.cuda.synchronize()
    ms_flush = timed(g_flush.replay) / nl
    del g_flush

    # per-step device time distribution: events around each eager step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(64)]
    barrier()
    for e0, e1 in ev:
        e0.record(stream)
        step(i)
        i += 1
        e1.record(stream)
    torch.cuda.synchronize()
    step_us = sorted(1e3 * e0.elapsed_time(e1) for e0, e1 in ev)
    pct = lambda p_: step_us[min(len(step_us) - 1, int(p_ * len(step_us)))]

    # per-kernel device time: a second capture with events around every kernel
    g_prof, _, _ = capture(profile=True)
    g_prof.replay()
    torch.cuda.synchronize()
    prof = {}
    for L in layers:
        for k, (t, n) in L["ctx"].paris_profile_end().items():
            a = prof.setdefault(k, [0.0, 0])
            a[0] += t
            a[1] += n
    del g_prof
    kernels = {k: {"us_per_launch": 1e3 * v[0] / v[1], "launches": v[1],
                   "timing": "CUDA events around each launch in a second captured replay (includes the events' cost)"}
               for k, v in prof.items() if v[1]}
    us_decode = 1e3 * prof.get("decode", [0.0, 0])[0] / args.steps

    # roofline of the dominant kernel (algorithmic bytes per launch)
    Nmean = sum(keys_per_step) / len(keys_per_step) / (b * hkv)
    nch = -(-int(Nmean) // 16384)
    C = max((w["cand_bp"] * int(Nmean) + 9999) // 10000, min(w["topk"], int(Nmean)))
    keff = min(w["topk"], C)
    nwin = S + w["local"] + w["update_buf"] // 2
    # Algorithmic bytes of one decode-step launch (one layer), per unit of
    # work: 16 B of bucket ids per Retrieval key and (sequence, KV head) --
    # the full scan a flat layout streams; 128 B of codes and w per candidate
    # and (sequence, query head); 8 B per top-k output; the top-k K and V
    # rows (2 x 256 B) per query head, and the window's rows (Sink, Local,
    # Buffer) once per KV head.  The kernel itself reads only the rho hot
    # bucket lists of each subspace (2 B per entry), so it moves fewer bytes
    # than this for the ids; "design_bytes" counts what it does read.
    alg = {
        "decode": b * hkv * 16 * Nmean + b * hq * (C * 128 + keff * 8 + keff * 4 * d) + b * hkv * nwin * 4 * d,
    }
    design = {
        "decode": b * hq * (2 * w["rho"] * w["n_sub"] * Nmean / 256 + C * 128 + keff * 4 * d + keff * 8)
                  + b * hkv * (nch * 16 * 264 * 4 + nwin * 4 * d),
    }
    dom = max(kernels, key=lambda k: kernels[k]["us_per_launch"] * kernels[k]["launches"])
    peak, peak_src = hbm_peak()
    roof = None
    if dom in alg:
        # When every timed step is exactly one launch of the dominant kernel
        # (no flush among them), its duration is the graph-replayed step time
        # itself; otherwise the mean of the event-bracketed launches of the
        # second capture (events add a little to each launch).
        one_per_step = launches == args.steps and kernels[dom]["launches"] == args.steps
        us_dom = 1e3 * ms / args.steps if one_per_step else kernels[dom]["us_per_launch"]
        ach = alg[dom] / (us_dom * 1e-6) / 1e9
        tr = traffic_record(dom, args)
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "peak_source": peak_src, "traffic": tr,
                "traffic_source": "profiles/dram_traffic.txt (ncu capture of these kernel sources)" if tr else None,
                "us_per_launch": us_dom,
                "time_source": ("graph replay of the timed steps, one launch per step" if one_per_step else
                                "CUDA events around each launch in a second captured replay"),
                "algorithmic_bytes": alg[dom], "design_bytes": design[dom]}
    # paris_retrieve alone (one decode-kernel launch per call, no attention):
    # 16 B of ids per Retrieval key and (sequence, KV head), 128 B of codes
    # and w per candidate and (sequence, query head), 8 B per top-k output
    Nr = keys_retrieve / (b * hkv)
    Cr = max((w["cand_bp"] * int(Nr) + 9999) // 10000, min(w["topk"], int(Nr)))
    alg_r = b * hkv * 16 * Nr + b * hq * (Cr * 128 + min(w["topk"], Cr) * 8)
    ach_r = alg_r / (ms_retrieve * 1e-3) / 1e9
    roof_r = {"kernel": "decode (paris_retrieve: no attention)", "bound": "hbm", "achieved": round(ach_r, 1),
              "peak": peak, "unit": "GB/s", "frac": round(ach_r / peak, 4), "peak_source": peak_src,
              "us_per_launch": 1e3 * ms_retrieve, "time_source": "graph replay of K paris_retrieve calls",
              "algorithmic_bytes": alg_r}

    # end to end through the public API with host buffers: each step's inputs
    # (q, k, v packed in one pinned buffer) go up in one copy, the step runs,
    # and its outputs (top-k positions and estimates, attention output, packed
    # in one device buffer) come back in one copy.  The copies run on a stream
    # of their own with three device buffers each way: the next step's inputs
    # go up while a step runs and its outputs come back during the next one,
    # so no copy sits between two decode steps on the compute stream.  The
    # timed region ends when the last outputs are in host memory.
    L0 = layers[0]

    def packed(parts, device, pinned=False):
        sizes = [t.numel() * t.element_size() for t in parts]
        offs = [sum(sizes[:j]) for j in range(len(sizes))]
        buf = torch.empty(sum(sizes), dtype=torch.uint8, device=device, pin_memory=pinned)
        views = [buf[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts, offs, sizes)]
        return buf, views

    h_in, (h_q, h_k, h_v) = packed([L0["qs"][0], L0["kn"][0], L0["vn"][0]], "cpu", pinned=True)
    h_q.copy_(L0["qs"][0])
    h_k.copy_(L0["kn"][0])
    h_v.copy_(L0["vn"][0])
    nbuf = 3
    d_ins = [packed([L0["qs"][0], L0["kn"][0], L0["vn"][0]], "cuda") for _ in range(nbuf)]
    d_ress = [packed([L0["idx"], L0["sc"], L0["out"]], "cuda") for _ in range(nbuf)]
    h_ress = [torch.empty_like(d_ress[0][0], device="cpu", pin_memory=True) for _ in range(nbuf)]
    copy_stream = torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]   # inputs of buffer j are on the device
    ev_run = [torch.cuda.Event() for _ in range(nbuf)]  # the step using buffer j is done
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]  # outputs of buffer j are in host memory
    for j in range(nbuf):
        ev_run[j].record(stream)
        ev_out[j].record(stream)

    def inputs_up(s_):
        j = s_ % nbuf
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_run[j])  # the step that last read buffer j is done
            d_ins[j][0].copy_(h_in, non_blocking=True)
            ev_in[j].record(copy_stream)

    # the keys each step scans, from each layer's zone state: an append fills
    # the Update Buffer, and the append that fills it moves update_buf tokens
    # into the Retrieval zone before the step's retrieval (checked below
    # against the library's own state)
    zone = [L["ctx"].paris_get_state() for L in layers]
    zN = [z_["N"] for z_ in zone]
    zbuf = [z_["n_buf"] for z_ in zone]
    barrier()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    keys_e2e = 0
    e2.record(stream)
    inputs_up(0)
    for s_ in range(args.steps):
        j = s_ % nbuf
        if s_ + 1 < args.steps:
            inputs_up(s_ + 1)
        li = i % nl
        L = layers[li]
        zbuf[li] += 1
        if zbuf[li] == w["update_buf"]:
            zN[li] += w["update_buf"]
            zbuf[li] = 0
        keys_e2e += zN[li] * b * hkv
        _, (d_q, d_k, d_v) = d_ins[j]
        d_res, (d_idx, d_sc, d_out) = d_ress[j]
        stream.wait_event(ev_in[j])
        stream.wait_event(ev_out[j])  # buffer j's last outputs are in host memory
        L["ctx"].paris_decode_step(d_k, d_v, d_q, d_idx, d_sc, d_out)
        ev_run[j].record(stream)
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(ev_run[j])
            h_ress[j].copy_(d_res, non_blocking=True)
            ev_out[j].record(copy_stream)
        i += 1
    for j in range(nbuf):
        stream.wait_event(ev_out[j])
    e3.record(stream)
    barrier()
    ms_e2e = max_over_ranks(e2.elapsed_time(e3))
    for li, L in enumerate(layers):
        st_ = L["ctx"].paris_get_state()
        assert (st_["N"], st_["n_buf"]) == (zN[li], zbuf[li]), "zone bookkeeping of the end-to-end loop"
    h2d = h_in.numel()
    d2h = h_ress[0].numel()

    # recall@k on layer 0 against the exact float64 top-k of <k, q>
    recall = None
    if keep_keys is not None and rank == 0:
        ctx = L0["ctx"]
        st = ctx.paris_get_state()
        N0 = L0["N0"]
        gen.manual_seed(777)
        rs = []
        for t in range(4):
            pos = torch.randint(S, S + N0, (b, hq), generator=gen, device="cuda")
            kvh_of = torch.arange(hq, device="cuda") // (hq // hkv)
            picked = keep_keys[torch.arange(b, device="cuda")[:, None], kvh_of[None, :], pos].float()
            q = (picked + 0.5 * torch.randn(picked.shape, generator=gen, device="cuda")).to(fdt).contiguous()
            k_eff = ctx.paris_retrieve(q, L0["idx"], L0["sc"])
            torch.cuda.synchronize()
            for s_ in range(b):
                for h in range(hq):
                    Kz = keep_keys[s_, h // (hq // hkv), S:S + min(N0, st["N"])].double()
                    ex = torch.topk(Kz @ q[s_, h].double(), k_eff).indices + S
                    got = L0["idx"][s_, h, :k_eff].long()
                    rs.append(torch.isin(got, ex).float().mean().item())
        recall = sum(rs) / len(rs)

    res = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": run_config(args, world),
        "us_per_decode_step": 1e3 * ms / args.steps,
        # one token through all rotated layers: the graph launches the layers' steps back to back
        "us_per_token_all_layers": 1e3 * ms / args.steps * nl,
        "us_per_decode_step_eager": 1e3 * ms_eager / args.steps,
        "us_decode_kernel": us_decode,
        "us_per_decode_step_eager_p10_p50_p90": [round(pct(0.1), 2), round(pct(0.5), 2), round(pct(0.9), 2)],
        "us_retrieve": 1e3 * ms_retrieve, "keys_per_s_retrieve": job_throughput(keys_retrieve, world, ms_retrieve),
        "us_sparse_attend": 1e3 * ms_attend, "us_append": 1e3 * ms_append,
        # the step whose append flushes (once every update_buf steps per layer) and the mean step
        "us_flush_step": 1e3 * ms_flush, "flush_step_launches": {k: v for k, v in flush_launches.items() if v},
        "us_per_step_amortised": 1e3 * ((U - 1) * ms / args.steps + ms_flush) / U,
        # GQA-shared variant: the union of a KV head's query heads' top-k, each row read once per KV head
        "gqa_shared_attention": {
            "us_per_step": 1e3 * ms_gqa, "us_per_head_sparse_attention": 1e3 * ms_attend,
            "union_rows_per_kv_head": union_rows, "per_head_rows_per_kv_head": G * k_eff0,
        },
        # the full-attention comparator on the same cache: every K/V row once per step
        "dense_attention": {
            "us_per_step": 1e3 * ms_dense,
            "decode_step_speedup": ms_dense / (ms / args.steps),
            "hbm_gbs": b * hkv * tokens_dense * 4 * d / (ms_dense * 1e-3) / 1e9,
            "hbm_frac": round(b * hkv * tokens_dense * 4 * d / (ms_dense * 1e-3) / 1e9 / peak, 4),
            "traffic": traffic_record("dense", args),
        },
        "recall_at_k": recall,
        "kernels": kernels,
        "roofline": roof,
        "roofline_retrieve": roof_r,
        "e2e": {"value": job_throughput(keys_e2e, world, ms_e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    return res


SWEEP_BP = (200, 500, 1000, 2000)
SWEEP_RHO = (1, 2, 4, 8)
SWEEP_K = (256, 512, 1024, 2048, 4096)


def run_sweep(args):
    """The 256K batch-5 sweep: candidate fraction x rho x k (80 points), one
    JSON line per point with recall@k against the exact float64 top-k and the
    decode-step and paris_retrieve times (graph replay over rotated layer
    contexts, as the main benchmark).  Every point builds fresh contexts from
    the same synthetic K/V."""
    import torch

    from long_context_kv_gb300 import build as B
    from long_context_kv_gb300 import paris as P
    from long_context_kv_gb300 import synth

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
    B.build()
    P.load()
    w = dict(WORKLOADS["sweep-256k"])
    nl = args.layers or 2
    b, hkv, hq, d, S = w["batch"], w["n_kv_heads"], w["n_q_heads"], w["head_dim"], w["sink"]
    T = w["context"]
    G = hq // hkv
    steps = args.steps
    per_layer = (args.warmup + 2 * steps + nl - 1) // nl + 2
    gen = torch.Generator(device="cuda")
    data = []
    for li in range(nl):
        seed = rank_seed(0, li)
        scale = torch.from_numpy(synth.channel_scale(seed, hkv, d)).cuda()
        gen.manual_seed(seed)
        K = (torch.randn((b, hkv, T, d), generator=gen, device="cuda") * scale[None, :, None, :]).to(torch.bfloat16)
        V = torch.randn((b, hkv, T, d), generator=gen, device="cuda").to(torch.bfloat16)
        kn = (torch.randn((per_layer, b, hkv, d), generator=gen, device="cuda") * scale[None, None]).to(torch.bfloat16)
        vn = torch.randn((per_layer, b, hkv, d), generator=gen, device="cuda").to(torch.bfloat16)
        N0 = T - S - w["local"]
        pos = torch.randint(S, S + N0, (per_layer + 4, b, hq), generator=gen, device="cuda")
        kvh_of = torch.arange(hq, device="cuda") // G
        picked = K[torch.arange(b, device="cuda")[None, :, None], kvh_of[None, None, :], pos].float()
        qs = (picked + 0.5 * torch.randn(picked.shape, generator=gen, device="cuda")).to(torch.bfloat16).contiguous()
        data.append(dict(K=K, V=V, kn=kn, vn=vn, qs=qs, seed=seed))
        del picked
    torch.cuda.synchronize()

    def timed(fn):
        torch.cuda.synchronize()
        a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(torch.cuda.current_stream())
        fn()
        z.record(torch.cuda.current_stream())
        torch.cuda.synchronize()
        return a.elapsed_time(z)

    for bp in SWEEP_BP:
        for rho in SWEEP_RHO:
            for k in SWEEP_K:
                layers = []
                for li, dat in enumerate(data):
                    cfg = P.make_config(batch=b, n_kv_heads=hkv, n_q_heads=hq, head_dim=d, n_sub=16, rho=rho, sink=S,
                                        local=w["local"], update_buf=w["update_buf"], topk=k, cand_bp=bp,
                                        max_ctx=T + per_layer + 8, retrieval_on_host=0)
                    ctx = P.Context(cfg, synth.srht_signs(dat["seed"], d))
                    ctx.paris_encode_prefill(dat["K"], dat["V"], T)
                    layers.append(dict(ctx=ctx, dat=dat, step=0,
                                       idx=torch.empty((b, hq, k), dtype=torch.int32, device="cuda"),
                                       sc=torch.empty((b, hq, k), dtype=torch.float32, device="cuda"),
                                       out=torch.empty((b, hq, d), dtype=torch.bfloat16, device="cuda")))

                def one(i, retrieve_only=False):
                    L = layers[i % nl]
                    dat, j = L["dat"], L["step"]
                    if retrieve_only:
                        L["ctx"].paris_retrieve(dat["qs"][j], L["idx"], L["sc"])
                        return
                    L["step"] = j + 1
                    L["ctx"].paris_decode_step(dat["kn"][j], dat["vn"][j], dat["qs"][j], L["idx"], L["sc"], L["out"])

                for i in range(args.warmup):
                    one(i)
                res = {}
                for name, ro in (("step", False), ("retrieve", True)):
                    g = torch.cuda.CUDAGraph()
                    cs = torch.cuda.Stream()
                    with torch.cuda.graph(g, stream=cs):
                        for i in range(steps):
                            one(args.warmup + i, ro)
                    g.replay()
                    torch.cuda.synchronize()
                    res[name] = 1e3 * timed(g.replay) / steps
                    del g
                # recall@k on layer 0 against the exact float64 top-k of <k, q>
                L0 = layers[0]
                st = L0["ctx"].paris_get_state()
                N = int(st["N"])
                rs = []
                for t in range(2):
                    q = L0["dat"]["qs"][per_layer + t]
                    k_eff = L0["ctx"].paris_retrieve(q, L0["idx"], L0["sc"])
                    for s_ in range(b):
                        for kvh in range(hkv):
                            Kz = L0["dat"]["K"][s_, kvh, S:S + N].double()
                            ex_all = torch.topk(Kz @ q[s_, kvh * G:(kvh + 1) * G].double().T, k_eff, dim=0).indices
                            for gi in range(G):
                                got = L0["idx"][s_, kvh * G + gi, :k_eff].long()
                                rs.append(torch.isin(got, ex_all[:, gi] + S).float().mean().item())
                keys = b * hkv * N
                print(json.dumps({"sweep_point": {"cand_pct": bp / 100, "rho": rho, "topk": k},
                                  "recall_at_k": sum(rs) / len(rs), "us_per_decode_step": res["step"],
                                  "us_retrieve": res["retrieve"], "keys_per_s_step": keys / (res["step"] * 1e-6),
                                  "C": int(st["C"]), "k_eff": int(st["k_eff"]), "N": N,
                                  "workload": DESCRIPTION["sweep-256k"], "layers_rotated": nl,
                                  "timing": "graph replay, layers rotated"}), flush=True)
                for L in layers:
                    L["ctx"].close()
                del layers
                torch.cuda.synchronize()


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    return ln.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _oracle_process(args, procs: int):
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-sample", "--workload", args.workload,
           "--cand-bp", str(args.cand_bp), "--rho", str(args.rho), "--topk", str(args.topk),
           "--steps", str(args.cpu_steps), "--warmup", str(args.warmup if args.impl == "reference" else 0),
           "--oracle-procs", str(procs)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        log(r.stderr[-2000:])
        return None
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(args):
    """The oracle as it stands, timed on the host cores in fresh processes:
    one process per core (each on its own KV head's decode steps, started
    together), and once single-threaded.  No CUDA work in either."""
    procs = max(1, min(host_cores(), args.oracle_procs_max))
    many = _oracle_process(args, procs)
    one = _oracle_process(args, 1) if procs > 1 else many
    if many is None or one is None:
        return None
    res = dict(many)
    res["cpu_model"] = cpu_model()
    res["single_thread"] = {"value": one["value"], "unit": one["unit"], "cores": 1, "seconds": one["seconds"],
                            "sample": one["sample"]}
    return res


def workload_of(args) -> dict:
    """The workload's parameters, with the sweep point's overrides applied."""
    w = dict(WORKLOADS[args.workload])
    for key in ("cand_bp", "rho", "topk"):
        v = getattr(args, key, None)
        if v:
            w[key] = v
    return w


def _bf16_values(x):
    """float32 array -> the float32 values of its bf16 rounding (round to
    nearest even; inputs are finite): what the library stores for K and V."""
    import numpy as np
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def _oracle_setup(args, head: int, room: int):
    """Prefill (untimed) of one KV head of the workload for the oracle: the
    head's keys and values (bf16-valued where the workload is bf16) with
    room for `room` decode tokens, its zones and its encoded Retrieval zone."""
    import numpy as np

    from long_context_kv_gb300 import synth
    from oracle import pariskv as o

    w = workload_of(args)
    d, S, L, U = w["head_dim"], w["sink"], w["local"], w["update_buf"]
    T = w["context"]
    seed = 20260202 + 1
    scale = synth.channel_scale(seed, head + 1, d)  # row `head` is this head's scale
    K = np.empty((T + room, d), dtype=np.float32)
    V = np.empty((T + room, d), dtype=np.float32)
    K[:T] = synth.key_rows(seed, 0, head, 0, T, d, scale)
    V[:T] = synth.value_rows(seed, 0, head, 0, T, d)
    bf = args.workload != "tiny-4k"
    if bf:
        K[:T] = _bf16_values(K[:T])
        V[:T] = _bf16_values(V[:T])
    signs = synth.srht_signs(seed, d)
    lev, thr = o.rsq_levels_f32(8)
    z = o.Zones(S, L, U)
    z.prefill(T)
    enc = o.encode_contract(K[S:S + z.N], signs, 16, lev, thr)
    return dict(w=w, K=K, V=V, z=z, enc=enc, signs=signs, lev=lev, thr=thr, scale=scale[head], bf=bf,
                rng=np.random.default_rng(seed + 7919 * head))


def _oracle_steps(st, n_steps: int) -> int:
    """n_steps decode steps of one KV head (its G query heads): append the
    step's token, then retrieval and sparse attention per query head.
    Returns the Retrieval-zone keys scanned."""
    import numpy as np

    from oracle import pariskv as o

    w, z, enc, rng, K, V = st["w"], st["z"], st["enc"], st["rng"], st["K"], st["V"]
    d, S = w["head_dim"], w["sink"]
    G = w["n_q_heads"] // w["n_kv_heads"]
    keys = 0
    for _ in range(n_steps):
        kn = rng.standard_normal(d).astype(np.float32) * st["scale"]
        vn = rng.standard_normal(d).astype(np.float32)
        t = z.T
        K[t] = _bf16_values(kn) if st["bf"] else kn
        V[t] = _bf16_values(vn) if st["bf"] else vn
        lo, hi = z.append()
        if hi > lo:  # a flush moved Local's oldest tokens into the Retrieval zone: encode them
            e1 = o.encode_contract(K[lo:hi], st["signs"], 16, st["lev"], st["thr"])
            for key in enc:
                enc[key] = np.concatenate([enc[key], e1[key]])
        N = z.N
        for _h in range(G):
            q = K[S + rng.integers(0, N)] + 0.5 * rng.standard_normal(d).astype(np.float32)
            r = o.retrieve_contract(enc, q.astype(np.float32), st["signs"], 16, w["rho"], w["cand_bp"], w["topk"],
                                    st["lev"])
            rows = np.concatenate([z.sink(), z.local(), z.buffer(), S + r["top_idx"]])
            o.attention(q, K[rows], V[rows])
        keys += N
    return keys


def _oracle_worker(args, head, barrier, queue):
    st = _oracle_setup(args, head, args.warmup + max(1, args.steps))
    _oracle_steps(st, args.warmup)
    barrier.wait()
    t0 = time.perf_counter()
    keys = _oracle_steps(st, max(1, args.steps))
    queue.put((head, keys, time.perf_counter() - t0))


def oracle_sample(args):
    """Decode steps of the workload run by the oracle as it stands; keys
    scanned = N per step and KV head.  With --oracle-procs P > 1, P processes
    (spawned, one per core) each run their own KV head's steps, released
    together by a barrier; the rate is all their keys over the wall time
    from the barrier to the last one's end."""
    steps = max(1, args.steps)
    w = workload_of(args)
    G = w["n_q_heads"] // w["n_kv_heads"]
    P = max(1, args.oracle_procs)
    if P == 1:
        st = _oracle_setup(args, 0, args.warmup + steps)
        _oracle_steps(st, args.warmup)
        t0 = time.perf_counter()
        keys = _oracle_steps(st, steps)
        dt = time.perf_counter() - t0
        print(json.dumps({"value": keys / dt, "unit": UNIT, "cores": 1, "kind": "oracle", "seconds": dt,
                          "sample": f"{steps} decode steps of 1 KV head ({G} query heads) of the "
                                    f"{DESCRIPTION[args.workload]}, single thread"}))
        return
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(P + 1)
    queue = ctx.Queue()
    ps = [ctx.Process(target=_oracle_worker, args=(args, h, barrier, queue)) for h in range(P)]
    for p_ in ps:
        p_.start()
    barrier.wait(timeout=600)
    t0 = time.perf_counter()
    res = [queue.get(timeout=600) for _ in range(P)]
    dt = time.perf_counter() - t0
    for p_ in ps:
        p_.join()
    keys = sum(r[1] for r in res)
    print(json.dumps({"value": keys / dt, "unit": UNIT, "cores": P, "kind": "oracle", "seconds": dt,
                      "sample": f"{steps} decode steps of each of {P} KV heads ({G} query heads each) of the "
                                f"{DESCRIPTION[args.workload]}, one process per core"}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama8b-128k", choices=sorted(WORKLOADS))
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--cand-bp", dest="cand_bp", type=int, default=0, help="candidates in basis points (sweep point)")
    ap.add_argument("--rho", type=int, default=0, help="hot centroids per subspace (sweep point)")
    ap.add_argument("--topk", type=int, default=0, help="k (sweep point)")
    ap.add_argument("--topk-order", dest="topk_order", default="score", choices=["score", "position"],
                    help="top-k lists best first (the contract's order) or in ascending position (no sort)")
    ap.add_argument("--cpu-steps", type=int, default=60)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-sample", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--oracle-procs", dest="oracle_procs", type=int, default=1, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-procs-max", dest="oracle_procs_max", type=int, default=64,
                    help="most processes of the multi-core oracle baseline")
    ap.add_argument("--sweep", action="store_true",
                    help="with --workload sweep-256k: all 80 points (candidate fraction x rho x k), one JSON line each")
    ap.add_argument("--profile-case", action="store_true",
                    help="only set up the workload and run warmup + steps decode steps, untimed (for ncu)")
    args = ap.parse_args()
    if args.oracle_sample:
        oracle_sample(args)
        return
    if args.sweep:
        if args.workload != "sweep-256k" or args.impl != "ours":
            ap.error("--sweep runs the sweep-256k workload of our arm")
        run_sweep(args)
        return
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        if rank != 0:
            return
        args.cpu_steps = max(1, args.steps)
        cb = cpu_baseline(args)
        if cb is None:
            print(json.dumps({"impl": "reference", "unavailable": "oracle run failed"}))
            return
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": run_config(args, world),
            "cpu_baseline": {"value": cb["value"], "unit": UNIT, "cores": cb["cores"], "kind": "oracle",
                             "sample": cb["sample"], "cpu_model": cb["cpu_model"],
                             "single_thread": cb["single_thread"]},
            "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }))
        return
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        tdist.init_process_group("nccl")
    cb = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.profile_case:
        cb = cpu_baseline(args)  # before any CUDA work in this process
    res = run_ours(args, rank, world)
    if rank == 0:
        if not args.profile_case:
            res["cpu_baseline"] = cb
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


if __name__ == "__main__":
    main()
