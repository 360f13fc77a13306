"""Benchmark: draft-tree builds per second at the Qwen3-4B shape (B=64).

One step = one whole round of the hot path (LM head + Top-M, the 15-depth
batched expansion, global Top-B, tree + mask) on one batch of synthetic input,
replayed as one CUDA graph through the C ABI.  Inputs are resident in HBM when
the timed region starts; the LM head streams 778 MB of weights per round, more
than the 129 MB L2, so no explicit L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(no data-path collective); value = rounds of all ranks / max elapsed.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
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
sys.path.insert(0, ROOT)

METRIC = "draft-tree builds/sec & us/round (Qwen3-4B shape, B=64); HBM GB/s vs peak"
WORKLOAD = "qwen3_4b"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _tensor_peak():
    """Dense bf16 TFLOP/s for a kernel timed alone (the burst figure)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def gemm_flops(cfg):
    """Tensor work of one LM-head launch: every H row of the block (the swap-AB
    N dimension) against the vocabulary rows and the W1_H rows."""
    return 2.0 * cfg.n_req * cfg.block * cfg.d * (cfg.V + cfg.r)


def _config_dict(cfg, n_inputs):
    lm_mb = cfg.V * cfg.d * 2 / 1e6
    return {
        "workload": f"{cfg.name}: d={cfg.d} V={cfg.V} block={cfg.block} g={cfg.g} r={cfg.r} "
                    f"M={cfg.M} K={cfg.K} W={cfg.W} B={cfg.B} beta={cfg.beta} T={cfg.T} n_req={cfg.n_req}",
        "n_req": cfg.n_req, "depth": cfg.block - 1, "B": cfg.B, "distinct_inputs": n_inputs,
        "l2": f"inputs larger than L2 ({lm_mb:.0f} MB LM head streamed per round), no flush",
    }


GEMM_NAME = "k_gemm_tc (LM head + W1_H, tcgen05/TMA)"
GEMM_NAME_FUSED = "k_gemm_tc + k_topm_merge (LM head + W1_H with the Top-M in the epilogue, tcgen05/TMA; merge)"


def algorithmic_bytes(cfg):
    """HBM bytes one launch of the LM-head GEMM and one whole round must move
    (weights read once, gathered rows, hidden states; the roofline numerators).
    The logits are not counted: the method needs only their Top-M."""
    D = cfg.block - 1
    lm = cfg.V * cfg.d * 2
    w1h = cfg.r * cfg.d * 2
    h = cfg.n_req * cfg.block * cfg.d * 2
    kernel = lm + w1h + h
    round_bytes = kernel + chain_bytes(cfg)
    return kernel, round_bytes


def _live_counts(cfg):
    """Live branches entering each depth: L_0 = 1, L_i = min(W, L_{i-1} K)."""
    L, out = 1, []
    for _ in range(cfg.block - 1):
        out.append(L)
        L = min(cfg.W, L * cfg.K)
    return out


def chain_bytes(cfg):
    """HBM bytes of the depth chain: the GRU hidden weights and the S-half of
    W1 once, the W2 rows of every depth's candidates, the GRU-input rows of
    the root and of every surviving child (fp32 table rows of 3g)."""
    D = cfg.block - 1
    w_hh = 3 * cfg.g * cfg.g * 2
    w1s = cfg.r * cfg.g * 2
    w2 = cfg.n_req * D * cfg.M * cfg.r * 2
    xrows = cfg.n_req * (1 + sum(min(cfg.W, L * cfg.K) for L in _live_counts(cfg)[:-1])) * 3 * cfg.g * 4
    return w_hh + w1s + w2 + xrows


def chain_flops(cfg):
    """Multiply-add work of the depth chain (2 FLOP each): per live branch the
    projection of its state through [W_hh | W1_S] and its correction over the
    M candidates."""
    per = sum(2 * L * (cfg.g * (3 * cfg.g + cfg.r) + cfg.r * cfg.M) for L in _live_counts(cfg))
    return cfg.n_req * per


def topm_bytes(cfg):
    """HBM bytes of Top-M over materialised logits: every logit read once."""
    return cfg.n_req * (cfg.block - 1) * cfg.V * 4


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def walk_bytes(cfg):
    """HBM bytes one acceptance walk must move: the target logits of every tree
    slot once, the trees, the outputs."""
    S, D = cfg.B + 1, cfg.block - 1
    return cfg.n_req * (S * cfg.V * 4 + 2 * S * 4 + (D + 2) * 4)


def time_accept_walk(builder, cfg, trees, stream, peak, n_launch=200):
    """The acceptance walk (dt_accept_walk) over the round's own trees, timed
    alone with CUDA events around graph replays on the current stream;
    distinct target-logit buffers rotate so that their total exceeds L2."""
    import numpy as np
    import torch
    from workloads import make_target_logits
    per = cfg.n_req * (cfg.B + 1) * cfg.V * 4
    n_in = int(min(8, max(2, -(-4 * 129e6 // per))))
    Zs, TPs = [], []
    for j in range(n_in):
        t = trees[j % len(trees)]
        tok, par = t["tok"].cpu().numpy(), t["parent"].cpu().numpy()
        Z = np.stack([make_target_logits(tok[q], par[q], cfg.V, 7000 + 100 * j + q, follow=0.8)
                      for q in range(cfg.n_req)])
        Zs.append(torch.from_numpy(Z).cuda())
        TPs.append((t["tok"], t["parent"]))
    D = cfg.block - 1
    acc = torch.empty(cfg.n_req, D, dtype=torch.int32, device="cuda")
    alen = torch.empty(cfg.n_req, dtype=torch.int32, device="cuda")
    bon = torch.empty(cfg.n_req, dtype=torch.int32, device="cuda")
    lens = []
    for j in range(n_in):
        builder.accept_walk(Zs[j], *TPs[j], accepted=acc, accept_len=alen, bonus=bon)
        lens += alen.cpu().tolist()
    torch.cuda.synchronize()
    # one CUDA graph of n_in launches (one per input), so that host-side call
    # overhead does not starve a kernel of a few microseconds
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for j in range(n_in):
                builder.accept_walk(Zs[j], *TPs[j], accepted=acc, accept_len=alen, bonus=bon, stream=side)
    stream.wait_stream(side)
    reps = max(1, n_launch // n_in)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * n_in)
    nb = walk_bytes(cfg)
    del Zs
    return {"kernel": "k_accept (row argmax + walk, one launch)", "us_per_launch": us,
            "algorithmic_bytes_per_launch": nb, "achieved": nb / (us * 1e-6) / 1e9, "peak": peak,
            "unit": "GB/s", "frac": nb / (us * 1e-6) / 1e9 / peak, "distinct_inputs": n_in,
            "mean_accept_len": float(np.mean(lens)),
            "inputs": "target logits N(0,1) per slot, the draft followed at 80 % of slots (synthetic)"}


def time_two_streams(builder, cfg, wd, Hs, roots, n_rounds):
    """Throughput mode: independent rounds alternate between two contexts on two
    streams, so that one round's kernels may overlap the other's; timed with
    CUDA events from a common start to the end of both streams."""
    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    b2 = DraftTreeBuilder(cfg, wd)
    try:
        streams = (torch.cuda.Stream(), torch.cuda.Stream())
        builders = (builder, b2)
        outs = [[b.new_tree() for _ in range(len(Hs))] for b in builders]
        for k in range(2 * len(Hs)):  # capture every pointer set of both contexts first
            j = k % len(Hs)
            builders[k % 2].build_round(Hs[j], roots[j], outs[k % 2][j], stream=streams[k % 2])
        torch.cuda.synchronize()
        main = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_wall = time.perf_counter()
        e0.record(main)
        for st in streams:
            st.wait_stream(main)
        for k in range(n_rounds):
            j = k % len(Hs)
            builders[k % 2].build_round(Hs[j], roots[j], outs[k % 2][j], stream=streams[k % 2])
            if k == 7:
                # a first chunk far slower than a round means the contexts do not
                # share the GPU well: stop there rather than time the rest
                torch.cuda.synchronize()
                if time.perf_counter() - t_wall > 0.5:
                    n_rounds = 8
                    break
        for st in streams:
            main.wait_stream(st)
        e1.record(main)
        torch.cuda.synchronize()
        status = b2.device_status()
    finally:
        b2.close()
    us = e0.elapsed_time(e1) * 1e3 / n_rounds
    return {"value": 1e6 / us, "unit": "builds/s", "us_per_round": us, "streams": 2, "contexts": 2,
            "rounds": n_rounds, "device_status": status,
            "note": "independent rounds alternating over two contexts and streams; latency mode is the headline"}


def time_stages(builder, cfg, H, root, stream, n=50):
    """The stages of the round timed alone, each captured in a CUDA graph of
    one call and replayed n times between CUDA events on the launching stream:
    the LM-head GEMM writing the logits (dt_base_logits); with the Top-M in the
    GEMM's epilogue, that GEMM and the merge of its lists as a round runs them
    (dt_base_topm, key lm_head_topm), else the Top-M kernel (dt_topm); and the
    expansion with its Top-B/tree tail (dt_expand_prune)."""
    import torch
    out = builder.new_tree()
    side = torch.cuda.Stream()
    calls = {"lm_head": lambda st: builder.base_logits(H, stream=st)}
    if "epilogue" in builder.plan():
        calls["lm_head_topm"] = lambda st: builder.base_topm(H, stream=st)
    else:
        calls["topm"] = lambda st: builder.topm(stream=st)
    calls["chain"] = lambda st: builder.expand_prune(root, out, stream=st)
    res = {}
    for name, fn in calls.items():
        side.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            fn(side)  # warm (and leaves the workspace in the state the next stage reads)
            with torch.cuda.graph(g, stream=side):
                fn(side)
        stream.wait_stream(side)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        res[name] = e0.elapsed_time(e1) * 1e3 / n
    return res


def kernel_rooflines(cfg, us, peak, peak_kind, tpeak, tpeak_kind):
    """One roofline entry per kernel of the round (bytes or FLOPs per launch
    over its CUDA-event time), largest time first."""
    kb, _ = algorithmic_bytes(cfg)
    ents = []
    gf = gemm_flops(cfg)
    fused = "lm_head_topm" in us
    t = (us["lm_head_topm"] if fused else us["lm_head"]) * 1e-6
    hbm, ten = kb / t / 1e9, gf / t / 1e12
    ent = {"kernel": GEMM_NAME_FUSED if fused else GEMM_NAME, "us_per_launch": t * 1e6,
           "bound": "hbm" if hbm / peak >= ten / tpeak else "tensor",
           "algorithmic_bytes_per_launch": kb, "hbm_gbs": hbm, "hbm_frac": hbm / peak,
           "algorithmic_flops_per_launch": gf, "tflops": ten, "tensor_frac": ten / tpeak}
    if fused:
        ent["note"] = ("the LM-head GEMM with the Top-M in its epilogue and the merge kernel, timed together as "
                       "a round runs them; the GEMM alone, writing the logits: %.1f us" % us["lm_head"])
    ents.append(ent)
    if not fused:
        tb = topm_bytes(cfg)
        t = us["topm"] * 1e-6
        ents.append({"kernel": "k_topm (Top-M + rest log-partition over the logits)", "us_per_launch": us["topm"],
                     "bound": "hbm", "algorithmic_bytes_per_launch": tb, "hbm_gbs": tb / t / 1e9,
                     "hbm_frac": tb / t / 1e9 / peak})
    cb, cf = chain_bytes(cfg), chain_flops(cfg)
    t = us["chain"] * 1e-6
    ents.append({"kernel": "depth chain (all depths + Top-B + tree/mask)", "us_per_launch": us["chain"],
                 "bound": "hbm", "algorithmic_bytes_per_launch": cb, "hbm_gbs": cb / t / 1e9,
                 "hbm_frac": cb / t / 1e9 / peak, "algorithmic_flops_per_launch": cf,
                 "tflops": cf / t / 1e12, "tensor_frac": cf / t / 1e12 / tpeak,
                 "note": "latency-bound: a sequence of dependent depths, each a few MFLOP"})
    for e in ents:
        e["peak_hbm_gbs"] = peak
        e["peak_source"] = f"{peak_kind} hbm_gbs; {tpeak_kind} bf16_tflops"
    ents.sort(key=lambda e: -e["us_per_launch"])
    return ents


def replica_seeds(rank, n_inputs):
    """Round seeds of one replica: every rank builds trees of its own inputs."""
    return [rank * 100000 + s for s in range(n_inputs)]


def job_throughput(dist, elapsed_s, e2e_s, steps, e2e_steps, world, device="cpu"):
    """Whole-job rates of N independent replicas: the slowest rank's times
    (max over ranks) divide the rounds of all ranks."""
    import torch
    if dist is not None:
        t = torch.tensor([elapsed_s, e2e_s], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed_s, e2e_s = float(t[0]), float(t[1])
    return steps * world / elapsed_s, e2e_steps * world / e2e_s, elapsed_s, e2e_s


def oracle_round(orc, cfg, H, root):
    """One round of the oracle of the workload's builder."""
    if getattr(cfg, "builder", "dartree") == "best_first":
        from oracle.besttree import build_best_first
        return [build_best_first(orc, H[q], int(root[q])) for q in range(H.shape[0])]
    return orc.build_round(H, root)


def run_oracle_rounds(cfg, w, seeds):
    from oracle.dartree import Oracle
    from workloads import make_round_inputs
    orc = Oracle(w, cfg)
    trees, times = [], []
    for s in seeds:
        H, root = make_round_inputs(cfg, s)
        t0 = time.perf_counter()
        trees.append(oracle_round(orc, cfg, H, root))
        times.append(time.perf_counter() - t0)
    return orc, trees, times


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def bench_reference(args):
    """The fp64 oracle as it stands, on the host cores, same workload and metric."""
    from workloads import get_config, make_weights
    cfg = get_config(args.workload)
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = make_weights(cfg)
    # warm-up and timed rounds are bounded samples: the whole run stays within
    # a few minutes whatever K and W are
    run_oracle_rounds(cfg, w, range(1000, 1000 + min(args.warmup, 3)))
    from oracle.dartree import Oracle
    from workloads import make_round_inputs
    orc = Oracle(w, cfg)
    times = []
    t_start = time.perf_counter()
    for s in range(args.steps):
        H, root = make_round_inputs(cfg, s)
        t0 = time.perf_counter()
        oracle_round(orc, cfg, H, root)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > args.cpu_seconds * 8:
            break
    total = sum(times)
    value = len(times) / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "builds/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config_dict(cfg, args.steps),
        "cpu_baseline": {"value": value, "unit": "builds/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"{len(times)} whole rounds (seeds 0..{len(times) - 1}) of the fp64 oracle, "
                                   f"at most {args.cpu_seconds * 8:.0f} s"},
        "e2e": {"value": value, "unit": "builds/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bench_gpu(args):
    import numpy as np
    import torch

    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder, bf16_tensor
    from conditional_draft_tree_lm_gb300.build import build_library
    from workloads import get_config, make_round_inputs, make_weights

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    build_library()
    cfg = get_config(args.workload)
    w = make_weights(cfg)
    wd = {k: bf16_tensor(v) for k, v in w.items()}
    torch.cuda.synchronize()
    t_create = time.perf_counter()
    builder = DraftTreeBuilder(cfg, wd)
    torch.cuda.synchronize()
    create_ms = (time.perf_counter() - t_create) * 1e3
    n_inputs = args.inputs
    seeds = replica_seeds(rank, n_inputs)
    Hs, roots = [], []
    for s in seeds:
        H, root = make_round_inputs(cfg, s)
        Hs.append(bf16_tensor(H))
        roots.append(torch.from_numpy(root.astype(np.int32)).cuda())
    outs = [builder.new_tree() for _ in range(n_inputs)]
    stream = torch.cuda.current_stream()

    def step(k):
        j = k % n_inputs
        builder.build_round(Hs[j], roots[j], outs[j])

    for k in range(args.warmup):
        step(k)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for k in range(args.steps):
        step(k)
    ev1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ms = ev0.elapsed_time(ev1)
    # per-round latency distribution (one event pair per round)
    lat = []
    for k in range(min(args.steps, 200)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step(k)
        b.record(stream)
        b.synchronize()
        lat.append(a.elapsed_time(b) * 1e3)
    # every kernel of the round timed alone (graph replays, events on the stream)
    stage_us = time_stages(builder, cfg, Hs[0], roots[0], stream, n=max(20, min(args.steps, 100)))
    lm_ms = stage_us.get("lm_head_topm", stage_us["lm_head"]) / 1e3
    peak, peak_kind = _peaks()
    walk = time_accept_walk(builder, cfg, outs, stream, peak) if not args.no_walk else None
    thr = time_two_streams(builder, cfg, wd, Hs, roots, max(10, min(args.steps, 200))) \
        if args.throughput else None
    clk = clocks.stop()
    # end to end through the public API with host buffers (pinned)
    Hh = [torch.from_numpy(np.ascontiguousarray(make_round_inputs(cfg, s)[0]).view(np.int16))
          .view(torch.bfloat16).pin_memory() for s in seeds[:4]]
    rh = [torch.from_numpy(make_round_inputs(cfg, s)[1].astype(np.int32)).pin_memory() for s in seeds[:4]]
    nh = len(Hh)
    out_h = {k: v.cpu().pin_memory() for k, v in builder.new_tree().items()}
    for k in range(3):
        builder.build_round_host(Hh[k % nh], rh[k % nh], out_h)
    n_e2e = max(10, min(args.steps, 200))
    t0 = time.perf_counter()
    for k in range(n_e2e):
        builder.build_round_host(Hh[k % nh], rh[k % nh], out_h)
    e2e_s = time.perf_counter() - t0
    h2d = Hh[0].numel() * 2 + rh[0].numel() * 4
    d2h = sum(v.numel() * v.element_size() for v in out_h.values())

    status = builder.device_status()
    value, e2e_value, elapsed, e2e_s = job_throughput(dist, ms / 1e3, e2e_s, args.steps, n_e2e, world,
                                                      device="cuda" if dist is not None and
                                                      dist.get_backend() == "nccl" else "cpu")
    kbytes, rbytes = algorithmic_bytes(cfg)
    achieved = kbytes / (lm_ms / 1e3) / 1e9
    tpeak, tpeak_kind = _tensor_peak()
    tflops = gemm_flops(cfg) / (lm_ms / 1e3) / 1e12
    kernels = kernel_rooflines(cfg, stage_us, peak, peak_kind, tpeak, tpeak_kind)
    traffic = None
    prof = os.path.join(ROOT, "profiles", f"lm_head_gemm_{cfg.name}_traffic.json")
    if os.path.exists(prof):
        try:
            with open(prof) as f:
                pj = json.load(f)
            if pj.get("kernel_source_hash") == _kernel_hash():
                traffic = pj.get("dram_bytes_per_launch")
        except Exception:
            traffic = None
    us_round = 1e6 * elapsed / args.steps
    top = kernels[0]
    gname = GEMM_NAME_FUSED if "lm_head_topm" in stage_us else GEMM_NAME
    if top["kernel"].startswith("k_gemm_tc"):
        roofline = None  # filled below (the GEMM's own object, with its ncu traffic)
    else:
        roofline = {"bound": "hbm", "kernel": top["kernel"], "achieved": top["hbm_gbs"], "peak": peak,
                    "unit": "GB/s", "frac": top["hbm_frac"], "peak_source": f"{peak_kind} hbm_gbs",
                    "traffic": None, "algorithmic_bytes_per_launch": top["algorithmic_bytes_per_launch"],
                    "avg_launch_us": top["us_per_launch"], "tensor_frac": top.get("tensor_frac"),
                    "note": top.get("note")}
    line = {
        "metric": METRIC, "value": value, "unit": "builds/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / args.steps, "us_per_round": us_round,
        "us_per_round_note": "mean of back-to-back graph replays (pipelined rounds), the figure the "
                             "60 % HBM target is stated for; isolated_round_us_* are single synchronised rounds",
        "isolated_round_us_p10_p50_p90": [float(np.percentile(lat, q)) for q in (10, 50, 90)],
        "isolated_round_hbm_frac_p50": rbytes / (float(np.percentile(lat, 50)) * 1e-6) / 1e9 / peak,
        "round_hbm_gbs": rbytes / (us_round * 1e-6) / 1e9,
        "round_hbm_frac": rbytes / (us_round * 1e-6) / 1e9 / peak,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1/fan_in) weights, N(0,1) hidden states)",
        "config": _config_dict(cfg, n_inputs),
        "kernels": kernels,
        "create": {"ms": create_ms, "gru_input_table_bytes": cfg.V * 3 * cfg.g * 4,
                   "note": "dt_create: workspace + GRU input table X = E W_ih^T + b_ih (one tcgen05 GEMM)"},
        "roofline": roofline if roofline is not None else ({"bound": "hbm", "kernel": gname,
                      "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                      "peak_source": f"{peak_kind} hbm_gbs", "traffic": traffic,
                      "algorithmic_bytes_per_launch": kbytes, "avg_launch_us": lm_ms * 1e3,
                      "tensor_frac": tflops / tpeak}
                     if achieved / peak >= tflops / tpeak else
                     {"bound": "tensor", "kernel": gname,
                      "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s", "frac": tflops / tpeak,
                      "peak_source": f"{tpeak_kind} bf16_tflops (burst)", "traffic": traffic,
                      "algorithmic_flops_per_launch": gemm_flops(cfg), "avg_launch_us": lm_ms * 1e3,
                      "hbm_frac": achieved / peak}),
        "e2e": {"value": e2e_value, "unit": "builds/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": builder.round_kernel_count() * args.steps,
        "plan": builder.plan(),
        "accept_walk": walk,
        "throughput_mode": thr,
        "clocks": clk,
        "device_status": status,
    }
    if rank == 0 and not args.no_cpu_baseline:
        t_budget = args.cpu_seconds
        seeds_cpu, times = [], []
        from oracle.dartree import Oracle
        orc = Oracle(w, cfg)
        t_start = time.perf_counter()
        k = 0
        while time.perf_counter() - t_start < t_budget and k < 16:
            H, root = make_round_inputs(cfg, seeds[k % n_inputs])
            t0 = time.perf_counter()
            oracle_round(orc, cfg, H, root)
            times.append(time.perf_counter() - t0)
            seeds_cpu.append(seeds[k % n_inputs])
            k += 1
        line["cpu_baseline"] = {"value": len(times) / sum(times), "unit": "builds/s", "cores": cpu_cores(),
                                "kind": "oracle",
                                "sample": f"{len(times)} whole rounds of the fp64 oracle (~{t_budget:.0f} s budget)"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    builder.close()
    if dist:
        dist.destroy_process_group()


def _kernel_hash():
    import hashlib
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "common.cuh", "topm_fused.cuh"):
        with open(os.path.join(ROOT, "conditional_draft_tree_lm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=WORKLOAD, help="a named workload of workloads/configs.py")
    ap.add_argument("--inputs", type=int, default=16)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-walk", action="store_true", help="skip the acceptance-walk measurement")
    ap.add_argument("--throughput", action="store_true",
                    help="also measure throughput mode (two contexts on two streams)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_gpu(args)


if __name__ == "__main__":
    main()
