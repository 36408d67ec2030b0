"""Benchmark of the drift-scoring / sparse-refresh step through libpolestar.

A step is one pass of the whole path over one batch of synthetic input: for
every layer, spherical k-means (warm-started), NVFP4 residuals, centroid keys
+ proxy attention + KL drift, top-k drifting clusters and the sparse K/V
refresh; then the commit over the current block.  Default workload: the
32-layer stress configuration (batch 32, window 4096, d 4096, 32 heads x 128,
C 256, 15 k-means iterations, top-k 16, commit over 64 x 126464 logits), each
layer with its own window, queries, weights and state; the LLaDA-8B-shaped
layer (batch 1, window 1024) follows under "extra".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl polestar|reference]

Timing: device-side CUDA events on the launching stream around a CUDA-graph
replay of the whole step; between steps the inputs drift in place and L2 is
flushed (512 MB write), outside the timed events; W >= 3 warm-up steps; for N
> 1 (torchrun) every rank runs an independent replica, the timed region is
bracketed by barriers and the slowest rank's time counts.  `--impl
reference` times the CPU oracle on one (window, layer) slice of the same
workload per step and extrapolates to the whole step (rank 0 only).
"""

import argparse
import hashlib
import glob
import json
import re
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "drift-refresh steps/s and window tokens/s; achieved HBM GB/s vs ~8 TB/s peak"
DEFAULT_WORKLOAD = "stress_b32_n4096_l32"
EXTRA_WORKLOAD = "llada8b_layer_n1024"
L2_FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="polestar", choices=["polestar", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--layers", type=int, default=0,
                    help="layers per step (0: the workload's own, 32 for the 32-layer ones)")
    ap.add_argument("--extra", default=EXTRA_WORKLOAD,
                    help="a second workload measured after the first and reported under "
                         "'extra' ('none' to skip)")
    ap.add_argument("--op", choices=["kmeans", "nvfp4", "proxy", "topk", "refresh", "commit"],
                    help="profiling mode: build one layer of the workload (--batch windows), "
                         "then run this op --reps times on it and exit, printing nothing but a "
                         "one-line summary (for a profiler to capture the op's kernels)")
    ap.add_argument("--batch", type=int, default=0, help="windows per layer in --op mode")
    ap.add_argument("--reps", type=int, default=3, help="calls of the op in --op mode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-overlap", action="store_true",
                    help="skip the latency-hiding measurement (the drift step of one layer on "
                         "a side stream behind a synthetic main forward)")
    ap.add_argument("--decode", action="store_true",
                    help="also time the decode loop under the refresh schedule and report it "
                         "under 'decode' (one layer: tau_upd 4, every 4th refresh full; "
                         "multi-layer workloads: every layer refreshed at every step)")
    ap.add_argument("--ablation", action="store_true",
                    help="also compare the drift signals (KL, cosine, entropy) on the "
                         "workload's planted drift and time the scoring pass")
    ap.add_argument("--offload", action="store_true",
                    help="quantised clusters in a pinned host store, refresh from the "
                         "reconstruction of the selected clusters (Polestar 2.C)")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    return 6800.0, 1900.0, "fallback"


def source_hash():
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "drift_aware_kv_spherical_gb300", "csrc", "*"))):
        h.update(open(f, "rb").read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm = [float(r[1]) for r in self.rows if len(r) >= 9 and r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if len(r) >= 9 and r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows if len(r) >= 9
                          for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(sm)}


def world_max(x, dev):
    """Max of a per-rank number over all ranks (the identity on one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_steps_per_s(world, steps, max_total_ms):
    """Whole-job throughput: every rank ran `steps` steps; the slowest rank's
    time counts."""
    return world * steps / (max_total_ms / 1000.0)


def graph_kernel_count(g):
    """Kernel nodes in a captured step (cudaGraphGetNodes through the CUDA
    runtime that torch loaded); None if the runtime cannot be reached."""
    import ctypes
    import torch
    try:
        raw = g.raw_cuda_graph()
    except Exception:
        return None
    rt = None
    cands = ["libcudart.so.13", "libcudart.so.12", "libcudart.so"]
    base = os.path.dirname(torch.__file__)
    cands += glob.glob(os.path.join(base, "lib", "libcudart*.so*"))
    cands += glob.glob(os.path.join(os.path.dirname(base), "nvidia", "cu*", "lib",
                                    "libcudart.so*"))
    for name in cands:
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            pass
    if rt is None:
        return None
    n = ctypes.c_size_t(0)
    if rt.cudaGraphGetNodes(ctypes.c_void_p(raw), None, ctypes.byref(n)) != 0:
        return None
    nodes = (ctypes.c_void_p * n.value)()
    if rt.cudaGraphGetNodes(ctypes.c_void_p(raw), nodes, ctypes.byref(n)) != 0:
        return None
    kind = ctypes.c_int(0)
    count = 0
    for k in range(n.value):
        if rt.cudaGraphNodeGetType(ctypes.c_void_p(nodes[k]), ctypes.byref(kind)) == 0 \
                and kind.value == 0:          # cudaGraphNodeTypeKernel
            count += 1
    return count


def op_work(w, npos_mean):
    """Algorithmic bytes and flops of each op for one window batch."""
    esz = 4 if w.dtype == "f32" else 2
    B, N, d, C = w.B, w.N, w.d, w.C
    H = B * N * d * esz
    nkv = w.Hkv * w.dh
    M = npos_mean * B
    return {
        "kmeans": ((w.iters + 1) * H, 2.0 * (w.iters + 1) * B * N * C * d),
        "nvfp4": (H + B * N * d // 2 + B * N * d // 16, 0.0),
        "proxy_kl": (d * nkv * esz + B * C * d * 4 + B * N * w.Hq * w.dh * esz + 2 * B * N * C * 4,
                     2.0 * B * C * d * nkv + 2.0 * B * N * w.Hq * C * w.dh),
        "topk": (B * N * 13, 0.0),
        "refresh": (2 * d * nkv * esz + M * d * esz + 2 * M * nkv * esz, 4.0 * M * d * nkv),
        "commit": (B * w.P * w.V * (2 if w.logits == "bf16" else 4), 0.0),
    }


# kernel trace names (the library's kernels, as the CUDA runtime names them)
# -> what they compute
KERNEL_KEYS = [("GramClusterEpi", "gram_gemm"), ("k_km_gram", "kmeans_passes"),
               ("KmAssign", "kmeans_assign"), ("KmFastEpi", "kmeans_assign"),
               ("k_km_recheck", "kmeans_recheck"), ("k_km_rho", "kmeans_rho"),
               ("k_km_fin_stats", "kmeans_fin_stats"), ("k_km_fin_chat", "kmeans_final"),
               ("k_km_argmax", "kmeans_argmax"),
               ("k_km_prep", "kmeans_prep"),
               ("k_kpp_gram", "kpp_gram"), ("k_kpp_pick", "kpp_pick"),
               ("k_kpp_weights", "kpp_weights"),
               ("k_drift_score", "drift_score"), ("k_assign", "kmeans_assign"),
               ("k_fp4_amax", "nvfp4_amax"), ("k_fp4_quant", "nvfp4_quant"),
               ("Ckeys", "centroid_keys"), ("k_ckeys", "centroid_keys"),
               ("k_split_f32", "proxy_split"), ("Proxy", "proxy_attn"),
               ("k_proxy", "proxy_attn"), ("k_topk", "topk"), ("k_gather_rows", "refresh_gather"),
               ("Refresh", "refresh_gemm"), ("k_refresh", "refresh_gemm"),
               ("k_commit_scan", "commit_scan"), ("k_commit_rule", "commit_rule"),
               ("k_pack_clusters", "offload_pack"), ("k_fetch_dequant", "offload_fetch")]


def kernel_key(name):
    if "k_cluster_scan" in name:  # first template flag: the final pass (C_hat only)
        m = re.search(r"k_cluster_scanI(?:13__nv_bfloat16|f)Lb([01])E", name)
        return "kmeans_final" if m and m.group(1) == "1" else "kmeans_update"
    for pat, key in KERNEL_KEYS:
        if pat in name:
            return key
    return name[:48]


def kernel_work(key, w, npos_mean):
    """Algorithmic bytes and flops of one launch of a kernel, or None."""
    esz = 4 if w.dtype == "f32" else 2
    B, N, d, C = w.B, w.N, w.d, w.C
    nkv = w.Hkv * w.dh
    H = B * N * d * esz
    M = npos_mean * B
    # Gram form (bf16, N <= 1024): 24-bit Gram slabs of R = 16 ceil(N / 256)
    # rows per CTA over Z = ceil(N / R) CTAs; pass 0's cosines in the GEMM when
    # 2C <= 128
    R = 16 * -(-N // 256)
    slab = B * -(-N // R) * N * R * 3
    fused0 = 2 * C <= 128
    return {
        "gram_gemm": (H + slab + (B * N * C * 4 if fused0 else 0),
                      B * (float(N) * (N + 1) * d + (2.0 * N * C * d if fused0 else 0.0))),
        "kmeans_passes": (slab + 2 * B * N * C * 4 + B * N * 12, 0.0),
        "kmeans_assign": (H + B * C * d * 2, 2.0 * B * N * C * d),
        "kmeans_rho": (H + B * N * 8, 2.0 * B * N * d),
        "kmeans_update": (H + B * C * d * 4, 0.0),
        "kmeans_fin_stats": (B * N * 12, 0.0),
        "kmeans_final": (B * N * 4 + 2 * B * C * d * 4, 0.0),
        "nvfp4_amax": (H, 0.0),
        "nvfp4_quant": (H + B * N * d // 2 + B * N * d // 16, 0.0),
        "centroid_keys": (d * nkv * esz + B * C * d * 4, 2.0 * B * C * d * nkv),
        "proxy_attn": (B * N * w.Hq * w.dh * esz + 2 * B * N * C * 4,
                       2.0 * B * N * w.Hq * C * w.dh),
        "topk": (B * N * 13, 0.0),
        "refresh_gather": (2 * M * d * esz, 0.0),
        "refresh_gemm": (2 * d * nkv * esz + M * d * esz + 2 * M * nkv * esz, 4.0 * M * d * nkv),
        "commit_scan": (B * w.P * w.V * (2 if w.logits == "bf16" else 4), 0.0),
    }.get(key)


def measure_overlap(w, dev, reps=20):
    """Latency hiding (the pages overlap the drift work with the main forward
    on CUDA streams), through Pipeline.step_overlapped on one layer: the
    main stream runs a synthetic forward of a transformer layer over the
    window (bf16 GEMMs: x W_qkv, W_o, a gated MLP of width 3.5 d: W_up to 2
    widths, W_down back; activations left out) that produces the layer's
    inputs, the layer's drift work forks onto a drift stream behind it, and
    the main stream goes on with the next layer's forward (the same GEMMs,
    in the slot step_overlapped gives the rest of the model).  Each
    arrangement is captured as a CUDA graph: the two forwards alone, the
    drift step alone, both through step_overlapped.  hidden = (t_main +
    t_drift - t_both) / t_drift, the share of the drift step's time the
    overlap hides."""
    import torch
    from drift_aware_kv_spherical_gb300.pipeline import Pipeline
    from drift_aware_kv_spherical_gb300 import workloads as wl
    M, d = w.B * w.N, w.d
    ff = int(3.5 * d) // 256 * 256
    g = torch.Generator(device=dev)
    g.manual_seed(20260717)

    def rnd(*shape):
        return (torch.randn(*shape, generator=g, device=dev) * 0.02).to(torch.bfloat16)

    X, Wqkv, Wo, Wup, Wdown = rnd(M, d), rnd(d, 3 * d), rnd(d, d), rnd(d, 2 * ff), rnd(ff, d)
    L = wl.make_layer(w, 0, dev)
    H, Wq, Wk, Wv = L["H"], L["Wq"], L["Wk"], L["Wv"]
    del L
    Q = wl.make_queries(w, H, Wq)
    u = wl.make_uniforms(w, 0, dev)
    logits = wl.make_logits(w, 0, dev).to(wl.logits_dtype(w))
    pipe = Pipeline(w, layers=1, device=dev)
    pipe.step([H], [Q], [Wk], [Wv], logits, init_us=[u], first=True)
    sm, sd = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def forward(l, s):
        with torch.cuda.stream(s):
            qkv = X @ Wqkv
            o = qkv[:, :d] @ Wo
            up = o @ Wup
            up[:, :ff] @ Wdown

    def capture(fn):
        torch.cuda.synchronize()
        for _ in range(2):
            fn()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=sm):
            fn()
        return graph

    def drift_only():
        sd.wait_stream(sm)
        pipe.step([H], [Q], [Wk], [Wv], logits, stream=sd)
        sm.wait_stream(sd)

    def both():
        pipe.step_overlapped([H], [Q], [Wk], [Wv], logits, sm, sd, forward=forward)

    gm = capture(lambda: (forward(0, sm), forward(1, sm)))
    gd = capture(drift_only)
    gb = capture(both)
    flops = 2 * 2.0 * M * d * (3 * d + d + 2 * ff + ff)

    def timed(graph):
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream(dev)
        a.record(cur)
        for _ in range(reps):
            graph.replay()
        b.record(cur)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3 / reps

    t_main, t_drift, t_both = timed(gm), timed(gd), timed(gb)
    return {"api": "Pipeline.step_overlapped (main stream: the forward; drift stream: "
                   "clustering, quantisation, proxy attention, top-k, refresh, commit)",
            "main_forward": f"bf16 GEMMs of two layers over {M} rows (d {d}, MLP {ff}): the "
                            f"layer whose drift is computed and the next, "
                            f"{flops / 1e12:.2f} TFLOP, captured graph",
            "main_us": t_main, "drift_us": t_drift, "both_us": t_both,
            "main_tflops": flops / (t_main * 1e-6) / 1e12,
            "hidden_fraction": (t_main + t_drift - t_both) / t_drift}


def measure_decode(w, L, Hs, Qs, logits, u, dev, steps=64, warm=8, tau_upd=4, full_period=4,
                   layers=1):
    """The decode loop under the refresh schedule, eager, on the workload's
    layer.  Wall pace: the host reads every step's outcome (tokens
    committed, block decided) to take the schedule's decision, as a decode
    loop must.  Device time by step kind: a second run in which a device-side
    spin before each step lets the host enqueue the whole step first, so the
    events time the kernels.  The re-init step's kernels: the library trace
    of one such step."""
    import torch
    from drift_aware_kv_spherical_gb300 import polestar as ps
    from drift_aware_kv_spherical_gb300.pipeline import Pipeline
    pipe = Pipeline(w, layers=layers, device=dev)
    stream = torch.cuda.current_stream(dev)
    marks, tokens, timing = [], [0], [False]
    plain = pipe.block_progress

    def progress(stream=None):
        c, done = plain(stream)
        tokens[0] += c
        return c, done

    pipe.block_progress = progress

    def inputs(t, block_start):
        if timing[0]:  # long enough for the host to enqueue the whole step behind it
            torch.cuda._sleep(2_000_000 * layers)
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(stream)
            marks.append([ev, None])
        n = layers  # every layer takes the workload's layer (one set of weights)
        return ([Hs[t % 4]] * n, [Qs[t % 4]] * n, [L["Wk"]] * n, [L["Wv"]] * n,
                logits[t % 4], [u] * n)

    def on_step(t, act):
        if timing[0]:
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(stream)
            marks[-1][1] = ev

    def run(n, graphs=False):
        return pipe.decode(ps.Schedule(tau_upd, full_period, w.P), inputs, n, on_step=on_step,
                           graphs=graphs)

    run(warm)
    torch.cuda.synchronize()
    tokens[0] = 0
    t0 = time.perf_counter()
    acts = run(steps)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    ntok = tokens[0]
    # the same loop through CUDA graphs (captured during the warm-up run)
    run(warm + 16, graphs=True)
    torch.cuda.synchronize()
    tokens[0] = 0
    t0 = time.perf_counter()
    acts_g = run(steps, graphs=True)
    torch.cuda.synchronize()
    wall_g = time.perf_counter() - t0
    ntok_g = tokens[0]
    timing[0] = True
    acts_t = run(steps)
    torch.cuda.synchronize()
    ps.ps_check()
    kinds = {"reuse": [], "refresh": [], "full": [], "reinit": []}
    for (a, b), act in zip(marks, acts_t):
        k = ("reinit" if act & ps.SCHED_REINIT else "full" if act & ps.SCHED_FULL
             else "refresh" if act & ps.SCHED_REFRESH else "reuse")
        kinds[k].append(a.elapsed_time(b))
    # the kernels of one re-init step (k-means++ seeding, full refresh)
    timing[0] = False
    Hs0, Qs0, Wk0, Wv0, lg0, us0 = inputs(0, 0)
    ps.ps_trace_enable(True)
    torch.cuda._sleep(20_000_000 * layers)  # the step's launches enqueued before it runs
    pipe.decode_step(ps.SCHED_REFRESH | ps.SCHED_FULL | ps.SCHED_REINIT | ps.SCHED_SLIDE,
                     Hs0, Qs0, Wk0, Wv0, lg0, us0)
    torch.cuda.synchronize()
    rec = ps.ps_trace_records()
    ps.ps_trace_enable(False)
    by = {}
    for name, ms in rec:
        key = kernel_key(name) or name[:40]
        n, tot = by.get(key, (0, 0.0))
        by[key] = (n + 1, tot + ms)
    return {"layers": layers, "tau_upd": tau_upd, "full_period": full_period, "steps": steps,
            "blocks_finished": sum(bool(a & 4) for a in acts),
            "wall_ms_per_step": wall * 1e3 / steps, "tokens_per_s": ntok / wall,
            "tokens": ntok, "graph_wall_ms_per_step": wall_g * 1e3 / steps,
            "graph_tokens_per_s": ntok_g / wall_g,
            "graph_refresh_frac": sum(bool(a & 1) for a in acts_g) / steps, "refresh_frac": sum(bool(a & 1) for a in acts) / steps,
            "full_frac": sum(bool(a & 2) and not a & 8 for a in acts) / steps,
            "reinit_frac": sum(bool(a & 8) for a in acts) / steps,
            "device_ms_by_step_kind": {k: (statistics.mean(v) if v else None)
                                       for k, v in kinds.items()},
            "reinit_step_kernels": {k: {"launches": n, "us": round(t * 1e3, 1)}
                                    for k, (n, t) in sorted(by.items(), key=lambda x: -x[1][1])},
            "timing": "wall: eager loop (graph_*: the loop through CUDA graphs) with one host "
                      "read per step; device: CUDA events around each eager step, enqueued "
                      "ahead behind a device-side spin"}


def measure_ablation(w, L, Hs, Qs, logits, u, dev, steps=3, reps=50):
    """The drift signals side by side on synthetic data: for each scorer, a
    window build and `steps` drifted steps of the workload's layer; the rows
    whose hidden state moved are the truth, and the top-k refresh positions
    the selection.  Reports precision and recall of the selection (summed
    over the steps) and the scoring pass's device time on the proxy
    distributions (ps_drift_score; KL is fused into the proxy on the default
    path)."""
    import torch
    from drift_aware_kv_spherical_gb300 import polestar as ps
    from drift_aware_kv_spherical_gb300.pipeline import Pipeline
    names = {ps.SCORER_KL: "kl", ps.SCORER_COSINE: "cosine", ps.SCORER_ENTROPY: "entropy"}
    out = {}
    for scorer, name in names.items():
        pipe = Pipeline(w, layers=1, device=dev, scorer=scorer)
        pipe.step([Hs[0]], [Qs[0]], [L["Wk"]], [L["Wv"]], logits[0], init_us=[u], first=True)
        tp = sel = truth = 0
        for t in range(1, steps + 1):
            pipe.step([Hs[t]], [Qs[t]], [L["Wk"]], [L["Wv"]], logits[t])
            moved = (Hs[t] != Hs[t - 1]).any(dim=-1)
            picked = pipe.state[0].posmask.bool()
            tp += int((moved & picked).sum())
            sel += int(picked.sum())
            truth += int(moved.sum())
        st = pipe.state[0]
        cur, prev = st.A[(pipe.t + 1) % 2], st.A[pipe.t % 2]
        D = torch.empty_like(st.D)
        for _ in range(5):
            ps.ps_drift_score(cur, prev, scorer, D)
        ps.ps_trace_enable(True)
        torch.cuda._sleep(10_000_000)  # the launches enqueued before they run
        for _ in range(reps):
            ps.ps_drift_score(cur, prev, scorer, D)
        torch.cuda.synchronize()
        rec = ps.ps_trace_records()
        ps.ps_trace_enable(False)
        ps.ps_check()
        us = statistics.mean(ms for _, ms in rec) * 1e3
        nbytes = cur.numel() * 4 * (1 if scorer == ps.SCORER_ENTROPY else 2) + D.numel() * 4
        out[name] = {"precision": tp / max(sel, 1), "recall": tp / max(truth, 1),
                     "selected_rows": sel, "moved_rows": truth,
                     "score_pass_us": us, "score_pass_gbs": nbytes / (us * 1e-6) / 1e9}
    out["note"] = ("truth: rows whose hidden state changed between steps (the current block "
                   "and a seeded share of the others); selection: the top-k clusters' rows; "
                   "score pass: the library trace's events around each launch, L2-resident")
    return out


def offload_rates(records, nsteps, w, npos_mean):
    """Host-link traffic of the offload kernels: the store they write (every
    row's record, by the GPU into pinned host memory) and read (the selected
    clusters' records), GB/s over each kernel's own duration."""
    rec = (w.d // 2 + 15) // 16 * 16 + (w.d // 16 + 15) // 16 * 16
    out = {"record_bytes": rec}
    for key, nbytes in (("offload_pack", w.B * w.N * rec), ("offload_fetch", npos_mean * w.B * rec)):
        ms = [m for name, m in records if kernel_key(name) == key]
        if ms:
            t = sum(ms) / len(ms)
            out[key] = {"bytes_per_launch": nbytes, "us_per_launch": 1e3 * t,
                        "host_link_gbs": nbytes / (t * 1e-3) / 1e9,
                        "launches_per_step": len(ms) / nsteps}
    return out


# kernels whose launches take no work for windows whose k-means passes have
# settled (the faster Lloyd passes skip them)
EARLY_EXIT = ("kmeans_assign", "kmeans_update", "kmeans_recheck")


def kernel_rooflines(records, nsteps, w, npos_mean, hbm, tf):
    """Per kernel: launches and time per step, average launch time and its
    algorithmic roofline fraction.  For the k-means kernels with an early
    exit, the per-launch work and time are those of the launches that did
    work: a launch under a tenth of the kernel's longest one in the trace took
    no tile (its windows had settled) and is counted apart; a launch whose
    windows had partly settled counts as whole, so the fraction errs low."""
    agg = {}
    for name, ms in records:
        k = kernel_key(name)
        a = agg.setdefault(k, [0, 0.0, []])
        a[0] += 1
        a[1] += ms
        a[2].append(ms)
    out = {}
    for k, (n, ms, each) in agg.items():
        row = {"launches_per_step": n / nsteps, "us_per_step": 1e3 * ms / nsteps,
               "us_per_launch": 1e3 * ms / n}
        if k in EARLY_EXIT:
            busy = [x for x in each if x >= 0.1 * max(each)]
            row["working_launches_per_step"] = len(busy) / nsteps
            row["us_per_working_launch"] = 1e3 * sum(busy) / len(busy)
            n, ms = len(busy), sum(busy)
        work = kernel_work(k, w, npos_mean)
        if work is not None:
            by, fl = work
            sec = ms / n * 1e-3
            tensor = fl / (tf * 1e12) > by / (hbm * 1e9)
            ach = fl / sec / 1e12 if tensor else by / sec / 1e9
            row.update({"bound": "tensor" if tensor else "hbm", "achieved": ach,
                        "peak": tf if tensor else hbm, "unit": "TFLOP/s" if tensor else "GB/s",
                        "frac": ach / (tf if tensor else hbm), "alg_bytes": by,
                        "alg_flops": fl})
        out[k] = {kk: (round(v, 6) if isinstance(v, float) else v) for kk, v in row.items()}
    return out


def run_reference(args):
    """The CPU oracle, as it stands, on this host's cores: each step is one
    (window, layer) slice of the workload -- a1-a6 on one window of one
    layer, warm-started from its previous step -- and the commit of one
    sequence; the whole-workload step is extrapolated linearly as B x layers
    slices plus B commits (exact for one window of one layer)."""
    import numpy as np
    import oracle
    from drift_aware_kv_spherical_gb300 import workloads as wl

    w = wl.BY_NAME[args.workload]
    layers = getattr(args, "layers", 0) or w.layers
    L = wl.make_layer(w, 0, "cpu", B=1)
    H0 = L["H"]
    Wk, Wv = L["Wk"].float().numpy(), L["Wv"].float().numpy()
    Hs = [H0]
    for t in range(1, 4):
        Hs.append(wl.drift_rows(w, Hs[-1], t))
    Qs = [wl.make_queries(w, H, L["Wq"]).float().numpy()[0] for H in Hs]
    Hn = [H.float().numpy()[0] for H in Hs]
    # the logits as they arrive (bf16 values are exact in the oracle's fp64)
    logits = [wl.make_logits(w, t, B=1).to(wl.logits_dtype(w)).float().numpy()[0]
              for t in range(4)]
    u = wl.make_uniforms(w, B=1).numpy()[0]
    mu = oracle.kmeanspp_init(Hn[0], w.C, u)[0]
    st = dict(mu=mu, chat=None, A=None, s=np.zeros(w.P, np.float32),
              n=np.zeros(w.P, np.int32), p=np.zeros(w.P, np.float32),
              u=np.ones(w.P, np.uint8))
    role = np.zeros(w.P, np.uint8)
    params = oracle.CommitParams(w.tau_s, w.alpha, w.ratio, w.mode, 1)
    Kc = np.zeros((w.N, w.Hkv * w.dh), np.float32)

    def step(t):
        i = t % 4
        t0 = time.perf_counter()
        r = oracle.kmeans_spherical(Hn[i], st["mu"], w.iters, st["chat"])
        st["mu"], st["chat"] = r["mu"], r["chat"]
        oracle.nvfp4_residual(Hn[i], r["mu"].astype(np.float32), r["assign"],
                              r["rho"].astype(np.float32))
        Kt = oracle.centroid_keys(r["chat"], Wk)
        A, D = oracle.proxy_attn_kl(Qs[i], Kt, w.Hq, w.Hkv, w.dh, st["A"])
        st["A"] = A
        sel = oracle.topk_drift(D.astype(np.float32), r["assign"], r["counts"], w.k)
        oracle.refresh_kv(Hn[i], sel[2], sel[3], Wk, Wv, Kc, Kc, 0, w.dtype == "bf16")
        t1 = time.perf_counter()
        c = oracle.commit_rule(logits[i], role, st["u"],
                               D[w.blk_start:w.blk_start + w.P].astype(np.float32),
                               st["s"], st["n"], st["p"], None, params)
        st["s"], st["n"], st["p"], st["u"] = c["d_sum"], c["d_cnt"], c["d_prev"], c["undecided"]
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1

    for t in range(args.warmup):
        step(t)
    times = [step(args.warmup + t) for t in range(args.steps)]
    t_slice = statistics.mean(a for a, _ in times)
    t_commit = statistics.mean(b for _, b in times)
    sec = w.B * layers * t_slice + w.B * t_commit
    sps = 1.0 / sec
    cores = _blas_threads()
    scale = w.B * layers
    sample = (f"one (window, layer) slice of {w.name} per step: a1-a6 on one window of one "
              f"layer ({t_slice * 1e3:.1f} ms) and a7 on one sequence ({t_commit * 1e3:.1f} ms), "
              f"fp64 numpy; " +
              ("exact: one window of one layer" if scale == 1 else
               f"extrapolated linearly to the step's {w.B} x {layers} slices and {w.B} commits"))
    line = {"impl": "reference", "metric": METRIC, "value": sps, "unit": "steps/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * sec, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, layers),
            "window_tokens_per_s": sps * w.B * w.N,
            "cpu_baseline": {"value": sps, "unit": "steps/s", "cores": cores,
                             "kind": "oracle", "sample": sample,
                             "extrapolated": scale > 1},
            "e2e": {"value": sps, "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info()]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def workload_config(w, layers=None):
    layers = w.layers if layers is None else layers
    return {"workload": w.name, "B": w.B, "N": w.N, "d": w.d, "Hq": w.Hq, "Hkv": w.Hkv,
            "dh": w.dh, "C": w.C, "iters": w.iters, "k": w.k, "P": w.P, "V": w.V,
            "layers": layers, "logits": w.logits,
            "weights": "per layer (seeded per layer)",
            "l2": ("flushed between steps (512 MB write)" if layers == 1 else
                   "inputs larger than L2 (every layer's window and queries are read each "
                   "step); also flushed between steps (512 MB write)")}


def cpu_baseline(w, layers, budget_s=20.0):
    """The oracle on one (window, layer) slice of the workload, extrapolated
    to the whole step (run_reference), a few samples within the budget."""
    import io
    import contextlib
    samples = 3
    ns = argparse.Namespace(steps=samples, warmup=0, workload=w.name, gpus=1, layers=layers)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        run_reference(ns)
    line = json.loads(buf.getvalue())
    cb = line["cpu_baseline"]
    cb["sample"] += f", {samples} samples"
    return cb


def one_layer_inputs(w, dev):
    """One layer's inputs for the optional one-layer measurements: the
    layer, four steps of drifted hidden states and their queries, four sets
    of logits, the k-means++ draws."""
    from drift_aware_kv_spherical_gb300 import workloads as wl
    L = wl.make_layer(w, 0, dev)
    Hs = [L["H"]]
    for t in range(1, 4):
        Hs.append(wl.drift_rows(w, Hs[-1], t))
    Qs = [wl.make_queries(w, H, L["Wq"]) for H in Hs]
    logits = [wl.make_logits(w, t, dev).to(wl.logits_dtype(w)) for t in range(4)]
    return L, Hs, Qs, logits, wl.make_uniforms(w, 0, dev)


def bench_workload(w, layers, args, dev, world, local, trace_steps=None):
    """Every measurement of one workload: the device-timed step (CUDA-graph
    replay, inputs resident), the per-op breakdown, the library trace, the
    end-to-end run through the public API; returns the JSON line's fields."""
    import torch
    import torch.distributed as dist
    from drift_aware_kv_spherical_gb300 import polestar as ps
    from drift_aware_kv_spherical_gb300 import workloads as wl
    from drift_aware_kv_spherical_gb300.pipeline import Pipeline

    # every layer's own inputs in fixed device buffers (graph replay needs
    # fixed addresses); between steps they drift in place, outside the timed
    # events
    ins = []
    for l in range(layers):
        L = wl.make_layer(w, l, dev)
        Q = wl.make_queries(w, L["H"], L["Wq"])
        ins.append(dict(H=L["H"], Q=Q, Wq=L["Wq"], Wk=L["Wk"], Wv=L["Wv"],
                        u=wl.make_uniforms(w, l, dev)))
        del L
    torch.cuda.empty_cache()
    Hs, Qs = [x["H"] for x in ins], [x["Q"] for x in ins]
    Wks, Wvs, us = [x["Wk"] for x in ins], [x["Wv"] for x in ins], [x["u"] for x in ins]
    # the logits in the dtype the workload states (else the model's own)
    logits = [wl.make_logits(w, t, dev).to(wl.logits_dtype(w)) for t in range(2)]
    dL = torch.empty_like(logits[0])
    pipe = Pipeline(w, layers=layers, device=dev, offload=args.offload)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    step_no = 0

    def advance():
        """The next step's inputs: every layer drifts, new logits."""
        nonlocal step_no
        step_no += 1
        for l in range(layers):
            wl.drift_inplace(w, Hs[l], Qs[l], ins[l]["Wq"], step_no, l)
        dL.copy_(logits[step_no % 2])

    # window build: k-means++ seeding, first distributions
    dL.copy_(logits[0])
    pipe.step(Hs, Qs, Wks, Wvs, dL, init_us=us, first=True)
    torch.cuda.synchronize()
    ps.ps_check()
    ops = ["kmeans", "nvfp4", "proxy_kl", "topk", "refresh", "commit"]

    def op_calls(parity, ev=None):
        """One step, layer by layer, events between the ops (summed per op)."""
        pipe.t = parity
        for l in range(layers):
            st = pipe.state[l]
            cur, prev = st.A[parity], st.A[1 - parity]
            rec = (lambda j: ev[l][j].record()) if ev is not None else (lambda j: None)
            rec(0)
            ps.ps_kmeans_spherical(Hs[l], st.mu, st.assign, st.rho, st.chat, st.counts,
                                   w.iters, objective=st.obj, ws=pipe.ws[ps.OP_KMEANS])
            rec(1)
            ps.ps_nvfp4_residual(Hs[l], st.mu, st.assign, st.rho, st.codes, st.scales, st.S,
                                 ws=pipe.ws[ps.OP_NVFP4])
            if pipe.offload:  # the store in host memory
                ps.ps_nvfp4_pack_clusters(st.codes, st.scales, st.assign, w.C, st.store,
                                          st.order, st.cl_off)
            rec(2)
            ps.ps_proxy_attn_kl(Qs[l], st.chat, Wks[l], prev, cur, st.D, w.Hkv,
                                ws=pipe.ws[ps.OP_PROXY_KL])
            rec(3)
            ps.ps_topk_drift(st.D, st.assign, st.counts, w.k, st.sel, st.sel_score, st.pos,
                             st.npos, st.posmask)
            rec(4)
            src = Hs[l]
            if pipe.offload:  # the selected clusters' rows from the host store
                ps.ps_nvfp4_fetch_dequant(st.store, st.order, st.cl_off, st.sel, st.mu, st.rho,
                                          st.S, st.Ht)
                src = st.Ht
            ps.ps_refresh_kv(src, st.pos, st.npos, Wks[l], Wvs[l], st.Kc, st.Vc, w.Hkv, w.dh,
                             ws=pipe.ws[ps.OP_REFRESH])
            rec(5)
        if ev is not None:
            ev[layers][0].record()
        pipe.commit_step(dL)
        if ev is not None:
            ev[layers][1].record()

    for t in range(args.warmup):                    # eager warm-up
        advance()
        op_calls(step_no % 2)
    torch.cuda.synchronize()
    ps.ps_check()

    # one graph per A ping-pong parity: the pipeline's step with the ops off
    # the critical path (NVFP4, commit) on side streams
    def concurrent_step(parity):
        pipe.t = parity          # A[parity] is this step's distribution
        pipe.step(Hs, Qs, Wks, Wvs, dL, concurrent=True)

    for t in range(2):           # side streams warmed up eagerly
        advance()
        concurrent_step(step_no % 2)
    torch.cuda.synchronize()
    ps.ps_check()
    graphs = []
    cap = torch.cuda.Stream(dev)
    for parity in (0, 1):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            concurrent_step(parity)
        graphs.append(g)
    launches = graph_kernel_count(graphs[0])       # None if the runtime is unreachable
    for t in range(args.warmup):                    # graph warm-up
        advance()
        graphs[step_no % 2].replay()
    torch.cuda.synchronize()
    ps.ps_check()

    # timed region: K graph replays; the inputs drift and L2 is flushed
    # between them, outside the timed events
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    for t in range(args.steps):
        advance()
        flush.zero_()
        gev[t][0].record(stream)
        graphs[step_no % 2].replay()
        gev[t][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    ps.ps_check()
    total_ms = world_max(sum(a.elapsed_time(b) for a, b in gev), dev)
    ms_step = total_ms / args.steps
    steps_per_s = aggregate_steps_per_s(world, args.steps, total_ms)
    del graphs

    # per-op breakdown: eager steps, events between the calls; a device-side
    # spin before each step lets the host enqueue the whole step first, so
    # the events time the kernels and not the host's launch pace
    nops = min(args.steps, 3)
    mk = lambda n: [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    events = [[mk(6) for _ in range(layers)] + [mk(2)] for _ in range(nops)]
    for t in range(nops):
        advance()
        flush.zero_()
        torch.cuda._sleep(4_000_000 * layers)
        op_calls(step_no % 2, events[t])
    torch.cuda.synchronize()
    ps.ps_check()
    npos_mean = float(torch.stack([st.npos.float().mean() for st in pipe.state]).mean())
    per_op = {op: [sum(ev[l][j].elapsed_time(ev[l][j + 1]) for l in range(layers))
                   for ev in events] for j, op in enumerate(ops[:5])}
    per_op["commit"] = [ev[layers][0].elapsed_time(ev[layers][1]) for ev in events]
    eager_ms = statistics.mean(ev[0][0].elapsed_time(ev[layers][1]) for ev in events)

    # per kernel: the library's own trace (CUDA events around each of its
    # launches, on the launching stream) over eager steps
    ntrace = trace_steps or (3 if layers == 1 else 1)
    ps.ps_trace_enable(True)
    for t in range(ntrace):
        advance()
        flush.zero_()
        torch.cuda._sleep(4_000_000 * layers)
        op_calls(step_no % 2)
    torch.cuda.synchronize()
    trace = ps.ps_trace_records()
    ps.ps_trace_enable(False)
    ps.ps_check()
    lib_launches = round(len(trace) / ntrace)       # every launch of its calls is traced

    # end to end through the public API (the pipeline's layer and commit
    # calls, eager): every step copies every layer's window and queries and
    # the block's logits from pinned host memory and reads its results
    # back.  Layer l's copy for a step runs on a copy stream as soon as the
    # previous step's layer l has finished reading its buffers, so copies
    # overlap the compute of the layers before; every copy and kernel lies
    # inside the timed interval.
    hH = [Hs[0].cpu().pin_memory(), None]
    hQ = [Qs[0].cpu().pin_memory(), None]
    wl.drift_inplace(w, Hs[0], Qs[0], ins[0]["Wq"], step_no + 1, 0)
    hH[1], hQ[1] = Hs[0].cpu().pin_memory(), Qs[0].cpu().pin_memory()
    hL = [x.cpu().pin_memory() for x in logits]
    last = pipe.state[-1]
    out = [torch.empty(pipe.token.shape, dtype=torch.int32).pin_memory(),
           torch.empty(pipe.conf.shape).pin_memory(),
           torch.empty(pipe.commit.shape, dtype=torch.uint8).pin_memory(),
           torch.empty(last.D.shape).pin_memory()]
    # a layer's window and queries go on two copy streams (two copy engines)
    cs, cq = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    done = [None] * (layers + 1)

    def e2e_run(n):
        ev = torch.cuda.Event
        t0 = ev(enable_timing=True)
        t0.record(stream)
        for i in range(n):
            for l in range(layers):
                after = done[l] if done[l] is not None else t0
                cs.wait_event(after)
                cq.wait_event(after)
                with torch.cuda.stream(cs):
                    Hs[l].copy_(hH[(i + l) % 2], non_blocking=True)
                with torch.cuda.stream(cq):
                    Qs[l].copy_(hQ[(i + l) % 2], non_blocking=True)
                stream.wait_event(cs.record_event())
                stream.wait_event(cq.record_event())
                joins = []
                pipe.layer_step(l, Hs[l], Qs[l], Wks[l], Wvs[l], stream=stream,
                                concurrent=True, joins=joins)
                for e in joins:
                    stream.wait_event(e)
                done[l] = stream.record_event()
            cs.wait_event(done[layers] if done[layers] is not None else t0)
            with torch.cuda.stream(cs):
                dL.copy_(hL[i % 2], non_blocking=True)
            stream.wait_event(cs.record_event())
            pipe.commit_step(dL, stream)
            done[layers] = stream.record_event()
            pipe.t += 1
            out[0].copy_(pipe.token, non_blocking=True)
            out[1].copy_(pipe.conf, non_blocking=True)
            out[2].copy_(pipe.commit, non_blocking=True)
            out[3].copy_(last.D, non_blocking=True)
        t1 = ev(enable_timing=True)
        t1.record(stream)
        return t0, t1

    e2e_run(max(1, args.warmup // 2))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    a, b = e2e_run(args.steps)
    torch.cuda.synchronize()
    ps.ps_check()
    e2e_ms = world_max(a.elapsed_time(b), dev)
    h2d = layers * (hH[0].numel() * hH[0].element_size() + hQ[0].numel() * hQ[0].element_size()) \
        + hL[0].numel() * hL[0].element_size()
    d2h = sum(x.numel() * x.element_size() for x in out)

    # rooflines: each op's algorithmic work against its measured time, and
    # every kernel's from the trace
    hbm, tf, src = peaks()
    work = op_work(w, npos_mean)
    rows = {}
    for op in ops:
        ms = statistics.mean(per_op[op])
        by, fl = work[op]
        if op != "commit":
            by, fl = by * layers, fl * layers
        bound = "tensor" if fl / (tf * 1e12) > by / (hbm * 1e9) else "hbm"
        ach = (fl / (ms * 1e-3) / 1e12) if bound == "tensor" else (by / (ms * 1e-3) / 1e9)
        peak = tf if bound == "tensor" else hbm
        rows[op] = {"ms": ms, "bound": bound, "achieved": ach, "peak": peak,
                    "unit": "TFLOP/s" if bound == "tensor" else "GB/s", "frac": ach / peak,
                    "alg_bytes": by, "alg_flops": fl}
    kernels = kernel_rooflines(trace, ntrace, w, npos_mean, hbm, tf)
    # the dominant kernel: most device time per step among those with a
    # stated algorithmic workload
    top = max((k for k in kernels if "frac" in kernels[k]),
              key=lambda k: kernels[k]["us_per_step"])
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        tj = json.load(open(tpath))
        per = tj.get("per_launch_bytes", {}).get(w.name, {})
        if tj.get("source_hash") == source_hash() and top in per:
            traffic = per[top]
    r = kernels[top]
    res = {
        "value": steps_per_s, "ms_per_step": ms_step, "dtype": w.dtype,
        "config": workload_config(w, layers),
        "window_tokens_per_s": steps_per_s * w.B * w.N,
        "e2e": {"value": aggregate_steps_per_s(world, args.steps, e2e_ms), "unit": "steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "timing": "eager calls of the public pipeline API; every layer's window and "
                          "queries and the logits copied from pinned host memory each step "
                          "(layer l's window and queries on two copy streams once the previous "
                          "step's layer l is done), results read back; one interval over the "
                          "steps"},
        "roofline": {"bound": r["bound"], "achieved": r["achieved"], "peak": r["peak"],
                     "unit": r["unit"], "frac": r["frac"], "traffic": traffic,
                     "kernel": top, "us_per_launch": r["us_per_launch"],
                     "launches_per_step": r["launches_per_step"],
                     "alg_bytes_per_launch": r["alg_bytes"],
                     "alg_flops_per_launch": r["alg_flops"], "peak_source": src},
        "kernels": kernels,
        "ops": {op: {k: (round(v, 6) if isinstance(v, float) else v) for k, v in rows[op].items()}
                for op in ops},
        "clocks": clk,
        "gpu_launches": lib_launches * args.steps,
        "graph_kernel_nodes": launches,
        "eager_ms_per_step": eager_ms,
        "timing": "CUDA-graph replay of the whole step (every layer, then the commit) per "
                  "timed step",
    }
    if args.offload:
        res["config"]["offload"] = "NVFP4 clusters in pinned host memory, fetched per step"
        res["offload"] = offload_rates(trace, ntrace, w, npos_mean)
    return res


def run_op(args):
    """--op mode: one layer of the workload with `--batch` windows; the
    window is clustered from centroids drawn from its own rows (no k-means++
    rounds, so few launches precede the captured ones), one whole step runs,
    then the chosen op runs --reps times on the layer's state, each call
    doing the work of a drifted step (k-means restarts from the same warm
    centroids each time)."""
    import dataclasses
    import torch
    from drift_aware_kv_spherical_gb300 import polestar as ps
    from drift_aware_kv_spherical_gb300 import workloads as wl
    from drift_aware_kv_spherical_gb300.pipeline import Pipeline
    w = wl.BY_NAME[args.workload]
    if args.batch:
        w = dataclasses.replace(w, B=args.batch)
    dev = torch.device("cuda", 0)
    L = wl.make_layer(w, 0, dev)
    H, Wk, Wv = L["H"], L["Wk"], L["Wv"]
    Q = wl.make_queries(w, H, L["Wq"])
    logits = wl.make_logits(w, 0, dev).to(wl.logits_dtype(w))
    pipe = Pipeline(w, layers=1, device=dev)
    st = pipe.state[0]
    g = torch.Generator(device=dev).manual_seed(7)
    rows = torch.randint(0, w.N, (w.B, w.C), generator=g, device=dev)
    seed = torch.gather(H.float(), 1, rows[..., None].expand(-1, -1, w.d))
    st.mu.copy_(seed / seed.norm(dim=2, keepdim=True))
    pipe.t = 1
    pipe.step([H], [Q], [Wk], [Wv], logits)       # A[1] and the clustering
    wl.drift_inplace(w, H, Q, L["Wq"], 1)
    pipe.t = 0
    pipe.step([H], [Q], [Wk], [Wv], logits)       # A[0]: a previous distribution exists
    torch.cuda.synchronize()
    ps.ps_check()
    mu0 = st.mu.clone()
    cur, prev = st.A[1], st.A[0]
    # each call timed with CUDA events on the current stream (the first is
    # a warm-up when there are several)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.reps + 1)]
    ev[0].record()
    for rep in range(args.reps):
        if args.op == "kmeans":
            st.mu.copy_(mu0)
            ps.ps_kmeans_spherical(H, st.mu, st.assign, st.rho, st.chat, st.counts, w.iters,
                                   objective=st.obj, ws=pipe.ws[ps.OP_KMEANS])
        elif args.op == "nvfp4":
            ps.ps_nvfp4_residual(H, st.mu, st.assign, st.rho, st.codes, st.scales, st.S,
                                 ws=pipe.ws[ps.OP_NVFP4])
        elif args.op == "proxy":
            ps.ps_proxy_attn_kl(Q, st.chat, Wk, prev, cur, st.D, w.Hkv,
                                ws=pipe.ws[ps.OP_PROXY_KL])
        elif args.op == "topk":
            ps.ps_topk_drift(st.D, st.assign, st.counts, w.k, st.sel, st.sel_score, st.pos,
                             st.npos, st.posmask)
        elif args.op == "refresh":
            ps.ps_refresh_kv(H, st.pos, st.npos, Wk, Wv, st.Kc, st.Vc, w.Hkv, w.dh,
                             ws=pipe.ws[ps.OP_REFRESH])
        else:
            pipe.commit_step(logits)
        ev[rep + 1].record()
    torch.cuda.synchronize()
    ps.ps_check()
    us = [ev[i].elapsed_time(ev[i + 1]) * 1e3 for i in range(args.reps)]
    print(json.dumps({"op": args.op, "workload": w.name, "B": w.B, "reps": args.reps,
                      "npos": int(st.npos.sum()),
                      "us_per_call": statistics.median(us[1:] if len(us) > 1 else us)}))


def main():
    args = parse()
    if args.op:
        run_op(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    assert args.warmup >= 3, "at least 3 warm-up steps"

    import torch
    import torch.distributed as dist
    from drift_aware_kv_spherical_gb300 import workloads as wl

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl")
    w = wl.BY_NAME[args.workload]
    layers = args.layers or w.layers
    res = bench_workload(w, layers, args, dev, world, local)
    torch.cuda.empty_cache()
    line = {"metric": METRIC, "value": res.pop("value"), "unit": "steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res.pop("ms_per_step"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": res.pop("dtype"), "data": "synthetic", "config": res.pop("config")}
    line.update(res)
    line["parallelism"] = f"replicas x{world}"
    if not args.no_overlap:
        line["overlap"] = measure_overlap(w, dev, reps=20 if layers == 1 else 5)
        torch.cuda.empty_cache()
    if args.ablation or args.decode:
        L, Hs1, Qs1, logits1, u1 = one_layer_inputs(w, dev)
        if args.ablation:
            line["ablation"] = measure_ablation(w, L, Hs1, Qs1, logits1, u1, dev)
        if args.decode:
            if w.layers > 1:  # the multi-layer loop refreshes every layer at every step
                line["decode"] = measure_decode(w, L, Hs1, Qs1, logits1, u1, dev, steps=48,
                                                warm=4, tau_upd=0, full_period=0,
                                                layers=w.layers)
            else:
                line["decode"] = measure_decode(w, L, Hs1, Qs1, logits1, u1, dev)
        del L, Hs1, Qs1, logits1
        torch.cuda.empty_cache()
    if args.extra and args.extra != "none" and args.extra != w.name:
        xw = wl.BY_NAME[args.extra]
        xr = bench_workload(xw, xw.layers, args, dev, world, local)
        line["extra"] = {xw.name: {
            "value": xr["value"], "unit": "steps/s", "ms_per_step": xr["ms_per_step"],
            "window_tokens_per_s": xr["window_tokens_per_s"], "config": xr["config"],
            "e2e": xr["e2e"], "roofline": xr["roofline"], "kernels": xr["kernels"],
            "clocks": xr["clocks"], "gpu_launches": xr["gpu_launches"]}}
        if not args.no_overlap:
            line["extra"][xw.name]["overlap"] = measure_overlap(xw, dev)
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, layers)
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
