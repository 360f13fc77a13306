"""Per-depth phase breakdown of the clustered depth chain (a profiling tool).

Builds an instrumented copy of libdtree (``-DDT_DCHAIN_TIMING``,
``-DDT_TOPM_TIMING``, ``-DDT_GEMM_TIMING``: thread 0 of CTA 0 and of the last
CTA record ``clock64()`` at every phase boundary of every depth) beside the
normal library, replays whole rounds of a workload through it, and prints the
mean cycles of each phase: X (waiting for and gathering the previous depth's
states), A1 (W1_S projection and z), A2 (partial correction), A3 (W_hh projection), R (the cluster
reduction of the correction), B (corrected log-probs and top-K: B.sel; the
children: B.out; the block barrier: B.bar), top-W, C (GRU update,
publication), and the kernel's prologue and tail.  Every CTA also records the
global timer when it has published a depth's states and when it holds all of
them, which shows the spread of the publications and the exchange latency.
It also prints the Top-M's phases (row 0) and the LM-head GEMM's tiles (CTA 0).
The normal library is not touched; the instrumented one is only loaded by this
process.

    python -m conditional_draft_tree_lm_gb300.chain_timing [--workload qwen3_4b] [--rounds 20]
"""
from __future__ import annotations

import argparse
import ctypes
import os
import sys

import numpy as np

# phase k runs from stamp k to stamp k+1 of the same depth (the last one to
# the next depth's stamp 0); the last depth ends at stamp LAST_END
PHASES = ["X", "A1", "A2", "A3", "R", "B.sel", "B.out", "B.bar", "topW", "C", "next"]
SLOTS = 66          # kMaxDepth + 2
NPH = 20
XCTAS = 128         # CTAs with exchange stamps
LAST_END = 8


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="qwen3_4b")
    ap.add_argument("--rounds", type=int, default=20)
    ap.add_argument("--mhz", type=float, default=0.0, help="SM clock for the microsecond column "
                                                           "(default 2070, the GB300's maximum)")
    ap.add_argument("--save", default="", help="also save the raw stamps (numpy .npy) here")
    args = ap.parse_args()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import torch

    from . import dtree
    from .build import LIB_DIR, build_library
    from workloads import get_config, make_round_inputs, make_weights

    path = build_library(force=True, extra_flags=["-DDT_DCHAIN_TIMING", "-DDT_TOPM_TIMING", "-DDT_GEMM_TIMING",
                                                  "-DDT_CHAIN_TIMING"],
                         lib_path=os.path.join(LIB_DIR, "libdtree_timing.so"))
    dtree._lib = None
    lib = dtree.load_library(path)
    dtree._lib = lib  # the builder below runs on the instrumented copy
    lib.dt_dchain_stamps.restype = ctypes.c_int
    lib.dt_dchain_stamps.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.dt_dchain_xstamps.restype = ctypes.c_int
    lib.dt_dchain_xstamps.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.dt_topm_stamps.restype = ctypes.c_int
    lib.dt_topm_stamps.argtypes = [ctypes.c_void_p, ctypes.c_int]
    lib.dt_gemm_stamps.restype = ctypes.c_int
    lib.dt_gemm_stamps.argtypes = [ctypes.c_void_p, ctypes.c_int]

    torch.cuda.set_device(0)
    cfg = get_config(args.workload)
    w = make_weights(cfg)
    wd = {k: dtree.bf16_tensor(v) for k, v in w.items()}
    b = dtree.DraftTreeBuilder(cfg, wd)
    print("plan:", b.plan())
    if "clustered depth chain on" not in b.plan():
        grid_chain_report(lib, b, cfg, args)
        return
    D = cfg.block - 1
    buf = np.zeros(2 * SLOTS * NPH, dtype=np.uint64)
    xbuf = np.zeros(2 * SLOTS * XCTAS, dtype=np.uint64)
    tbuf = np.zeros(2 * 64 * 16, dtype=np.uint64)
    gbuf = np.zeros(17 * 8, dtype=np.uint64)
    acc, xacc, tacc, gacc, tbacc = [], [], [], [], []
    lib.dt_dchain_topb_stamps.restype = ctypes.c_int
    lib.dt_dchain_topb_stamps.argtypes = [ctypes.c_void_p, ctypes.c_int]
    tbb = np.zeros(8, dtype=np.uint64)
    for s in range(args.rounds + 3):
        H, r = make_round_inputs(cfg, s)
        Hd = dtree.bf16_tensor(H)
        rd = torch.from_numpy(r.astype(np.int32)).cuda()
        b.build_round(Hd, rd)
        torch.cuda.synchronize()
        n = lib.dt_dchain_stamps(buf.ctypes.data, buf.size)
        if n != buf.size:
            raise SystemExit("dt_dchain_stamps failed")
        if lib.dt_dchain_xstamps(xbuf.ctypes.data, xbuf.size) != xbuf.size:
            raise SystemExit("dt_dchain_xstamps failed")
        if lib.dt_topm_stamps(tbuf.ctypes.data, tbuf.size) != tbuf.size:
            raise SystemExit("dt_topm_stamps failed")
        if lib.dt_gemm_stamps(gbuf.ctypes.data, gbuf.size) != gbuf.size:
            raise SystemExit("dt_gemm_stamps failed")
        if s >= 3:
            acc.append(buf.reshape(2, SLOTS, NPH).astype(np.int64).copy())
            xacc.append(xbuf.reshape(2, SLOTS, XCTAS).astype(np.int64).copy())
            tacc.append(tbuf.reshape(2, 64, 16).astype(np.int64).copy())
            gacc.append(gbuf.reshape(17, 8).astype(np.int64).copy())
            lib.dt_dchain_topb_stamps(tbb.ctypes.data, tbb.size)
            tbacc.append(tbb.astype(np.int64).copy())
    st = np.stack(acc)  # [rounds, cta, slot, phase]
    if args.save:
        np.save(args.save, st)
    mhz = args.mhz or 2070.0
    us = 1.0 / mhz
    print(f"{len(acc)} rounds of {cfg.name}; cycles (us at {mhz:.0f} MHz), mean over rounds")
    for c, name in ((0, "CTA 0"), (1, "last CTA")):
        k = st[:, c]
        pro = (k[:, 0, 4] - k[:, 0, 0]).mean()
        gw = (k[:, 0, 5] - k[:, 0, 4]).mean()
        first = (k[:, 1, 0] - k[:, 0, 5]).mean()
        loop = (k[:, 0, 1] - k[:, 1, 0]).mean()
        print(f"\n{name}: prologue {pro:.0f} ({pro * us:.2f}), wait for the previous kernel {gw:.0f} "
              f"({gw * us:.2f}), to depth 1 {first:.0f} ({first * us:.2f}), depth loop {loop:.0f} "
              f"({loop * us:.2f})" + (f", tail {(k[:, 0, 2] - k[:, 0, 1]).mean() * us:.2f} us (last nodes "
                                       f"{(k[:, 0, 6] - k[:, 0, 1]).mean() * us:.2f}, Top-B "
                                       f"{(k[:, 0, 7] - k[:, 0, 6]).mean() * us:.2f}, tree/mask "
                                       f"{(k[:, 0, 2] - k[:, 0, 7]).mean() * us:.2f})" if c == 0 else ""))
        print("depth " + " ".join(f"{p:>7s}" for p in PHASES) + "    total(us)")
        nph = len(PHASES)
        tot = np.zeros(nph)
        for i in range(1, D + 1):
            row = []
            for ph in range(nph):
                if i == D and ph >= LAST_END:
                    row.append(0.0)  # the last depth ends after its node arrays
                    continue
                if i == D and ph == LAST_END - 1:
                    nxt = k[:, 0, 1]
                elif ph + 1 < nph:
                    nxt = k[:, i, ph + 1]
                else:
                    nxt = k[:, i + 1, 0]
                row.append((nxt - k[:, i, ph]).mean())
            tot += np.array(row)
            end = k[:, i + 1, 0] if i < D else k[:, 0, 1]
            print(f"{i:5d} " + " ".join(f"{v:7.0f}" for v in row) + f"  {(end - k[:, i, 0]).mean() * us:8.2f}")
        print("mean  " + " ".join(f"{v / D:7.0f}" for v in tot) + "  (cycles per depth)")
        print("us    " + " ".join(f"{v / D * us:7.2f}" for v in tot))
        # finer split of three phases (depths 2..D-1), from the extra stamps
        mid = slice(2, D)
        sub = lambda a, b: (k[:, mid, b] - k[:, mid, a]).mean()
        print(f"  A1: loads + MMAs {sub(1, 11):.0f}, partial sums {sub(11, 12):.0f}, barrier {sub(12, 13):.0f}, "
              f"z {sub(13, 2):.0f};  B.sel: operands {sub(5, 15):.0f}, top-K rounds + log-partition {sub(15, 6):.0f};  "
              f"topW: rounds {sub(8, 14):.0f}, survivor order {sub(14, 9):.0f};  "
              f"X: loads issued {sub(0, 16):.0f}, poll {sub(16, 17):.0f}, barrier + copies {sub(17, 1):.0f}")
    tb = np.stack(tbacc).mean(axis=0)
    t6 = st[:, 0, 0, 6].mean()  # before Top-B
    print("  tail (cycles from the Top-B's start): keys %.0f, histogram %.0f, bound %.0f, candidates %.0f, ranks + "
          "order %.0f | tree slots %.0f, parents %.0f, ancestors %.0f, mask to the end %.0f" % (
              tb[0] - t6, tb[1] - tb[0], tb[2] - tb[1], tb[3] - tb[2], tb[4] - tb[3], tb[5] - tb[4], tb[6] - tb[5],
              tb[7] - tb[6], st[:, 0, 0, 2].mean() - tb[7]))
    exchange_report(np.stack(xacc), D, b.plan())
    topm_report(np.stack(tacc))
    gemm_report(np.stack(gacc), 1.0 / mhz)
    b.close()


GRID_PHASES = ["A", "bar1", "B", "bar2", "C", "bar3"]


def grid_chain_report(lib, b, cfg, args):
    """The grid-barrier chain (several requests, or many branches): per depth,
    phase A (projections; its waits for state blocks shown apart), the
    barrier after it, phase B (selections; with one request also phase C), the
    barrier before the all-request phase C, phase C, and the depth's last
    barrier, for CTA 0 and the last CTA; phase B is split further (scoring,
    the top-W)."""
    import torch

    from . import dtree
    from workloads import make_round_inputs
    lib.dt_chain_stamps.restype = ctypes.c_int
    lib.dt_chain_stamps.argtypes = [ctypes.c_void_p, ctypes.c_int]
    D = cfg.block - 1
    buf = np.zeros(2 * SLOTS * 20, dtype=np.uint64)
    lib.dt_chain_tcstamps.restype = ctypes.c_int
    lib.dt_chain_tcstamps.argtypes = [ctypes.c_void_p, ctypes.c_int]
    tcb = np.zeros(3 * 128, dtype=np.uint64)
    acc, tacc = [], []
    for s in range(args.rounds + 3):
        H, r = make_round_inputs(cfg, s)
        Hd = dtree.bf16_tensor(H)
        rd = torch.from_numpy(np.asarray(r).astype(np.int32)).cuda()
        b.build_round(Hd, rd)
        torch.cuda.synchronize()
        if lib.dt_chain_stamps(buf.ctypes.data, buf.size) != buf.size:
            raise SystemExit("dt_chain_stamps failed")
        if s >= 3:
            acc.append(buf.reshape(2, SLOTS, 20).astype(np.int64).copy())
            lib.dt_chain_tcstamps(tcb.ctypes.data, tcb.size)
            tacc.append(tcb.reshape(3, 128).astype(np.int64).copy())
    st = np.stack(acc)
    us = 1.0 / (args.mhz or 2070.0)
    print(f"{len(acc)} rounds of {cfg.name}; grid-barrier chain; cycles, mean over rounds")
    for c, name in ((0, "CTA 0"), (1, "last CTA")):
        k = st[:, c]
        print(f"\n{name}")
        print("depth " + " ".join(f"{p:>8s}" for p in GRID_PHASES) + "  blk-wait  total(us)")
        tot = np.zeros(len(GRID_PHASES) + 1)
        for i in range(1, D + 1):
            t = k[:, i]
            # stamp 4 exists only with several requests; stamp 6 not at the last depth
            s4 = np.where(t[:, 4] > 0, t[:, 4], t[:, 3])
            s6 = t[:, 6] if i < D else t[:, 5]
            row = [(t[:, 1] - t[:, 0]).mean(), (t[:, 2] - t[:, 1]).mean(), (t[:, 3] - t[:, 2]).mean(),
                   (s4 - t[:, 3]).mean(), (t[:, 5] - s4).mean(), (s6 - t[:, 5]).mean(), t[:, 7].mean()]
            tot += np.array(row)
            print(f"{i:5d} " + " ".join(f"{v:8.0f}" for v in row) + f"  {(s6 - t[:, 0]).mean() * us:8.2f}")
        print("us    " + " ".join(f"{v / D * us:8.2f}" for v in tot))
        if c == 0 and D >= 2:
            t = np.stack(tacc).mean(axis=0)
            n = int((t[1] > 0).sum())
            if n:
                t0 = t[0, 0]
                lat = t[1, :n] - t[0, :n]
                print(f"  tcgen05 phase A, depth 2 ({n} chunks; cycles from the first copy): copy latency "
                      f"mean {lat.mean():.0f} (min {lat.min():.0f}, max {lat.max():.0f}); data landed at "
                      + ", ".join(f"{v - t0:.0f}" for v in t[1, :min(n, 12)]) + f" ...; last {t[1, n - 1] - t0:.0f}; "
                      f"products issued {t[2, 0] - t0:.0f}")
        mid = k[:, 2:D]
        if (mid[:, :, 8] > 0).all():
            sub = lambda a, b: (mid[:, :, b] - mid[:, :, a]).mean() * us
            print(f"  B (branches spread): scoring {sub(2, 8):.2f} [to the branch {sub(2, 12):.2f}, z {sub(12, 13):.2f}, "
                  f"logits {sub(13, 14):.2f}, log-partition + keys {sub(14, 15):.2f}, K best {sub(15, 16):.2f}, "
                  f"children: token order {sub(16, 19):.2f}, writes {sub(19, 18):.2f}, + {sub(18, 8):.2f}], barrier {sub(8, 9):.2f}, children read back "
                  f"{sub(9, 10):.2f}, top-W {sub(10, 11):.2f} [threshold {sub(10, 17):.2f}], the rest {sub(11, 3):.2f} us")
        elif (mid[:, :, 10] > 0).all():
            sub = lambda a, b: (mid[:, :, b] - mid[:, :, a]).mean() * us
            print(f"  B: selections {sub(2, 10):.2f}, top-W {sub(10, 11):.2f}, the rest {sub(11, 3):.2f} us")


def gemm_report(gs, us):
    """CTA 0 of the LM-head GEMM, tile by tile (us from the MMA warp's first tile)."""
    g = gs.mean(axis=0)
    t0 = g[0, 0]
    n = int((gs[0, :16, 1] > 0).sum())
    print(f"\nLM-head GEMM, CTA 0 ({n} tiles; us from its first MMA, mean over rounds)")
    print("tile   MMA start   MMA end   epilogue has it   appended    ranked   epilogue done")
    for t in range(n):
        print(f"{t:4d}  {(g[t, 0] - t0) * us:9.2f}  {(g[t, 1] - t0) * us:8.2f}  {(g[t, 2] - t0) * us:16.2f}  "
              f"{(g[t, 4] - t0) * us:9.2f}  {(g[t, 5] - t0) * us:8.2f}  {(g[t, 3] - t0) * us:14.2f}")
    print(f"final pass: sums reduced {(g[16, 3] - t0) * us:.2f}, epilogue end {(g[16, 0] - t0) * us:.2f}")


def topm_report(ts):
    """Top-M of row 0 by the global timer: the chunk CTAs' phases and the merge."""
    part, mrg = ts[:, 0], ts[:, 1, 0]  # [rounds, split, k], [rounds, k]
    S = int((part[0, :, 1] > 0).sum())
    m = lambda a, b: (mrg[:, b] - mrg[:, a]).mean()
    if S == 0:
        # the Top-M ran in the LM-head GEMM's epilogue: only the merge kernel
        print("\nTop-M in the LM-head GEMM's epilogue; the merge kernel, row 0 (ns, mean over rounds): "
              f"entries + range {m(0, 10):.0f}, histogram {m(10, 11):.0f}, bin {m(11, 12):.0f}, "
              f"gather {m(12, 13):.0f}, rank {m(13, 14):.0f}, winners {m(1, 2):.0f}, their ranks {m(2, 3):.0f}, "
              f"rest + writes {m(3, 4):.0f}; total {m(0, 4):.0f}")
        return
    part = part[:, :S]
    t1 = part[:, :, 1].min(axis=1)  # the earliest chunk CTA past the wait
    d = lambda a, b: (part[:, :, b] - part[:, :, a]).mean()
    print(f"\nTop-M, row 0 ({S} chunk CTAs; ns, mean over CTAs and rounds)")
    print(f"chunk CTAs: stats {d(1, 2):.0f}, rung {d(2, 3):.0f}, collect {d(3, 4):.0f}, M-th key [range {d(4, 10):.0f}, "
          f"histogram {d(10, 11):.0f}, bin {d(11, 12):.0f}, gather {d(12, 13):.0f}, rank {d(13, 14):.0f}], "
          f"losers {d(7, 8):.0f}, winners {d(8, 9):.0f}, their ranks {d(9, 5):.0f}, rest + arrival {d(5, 6):.0f}")
    print(f"chunk CTAs past the wait: last {(part[:, :, 1] - t1[:, None]).max(axis=1).mean():.0f} ns after the first; "
          f"arrivals: first {(part[:, :, 6].min(axis=1) - t1).mean():.0f}, last "
          f"{(part[:, :, 6].max(axis=1) - t1).mean():.0f}")
    print(f"merge: starts {(mrg[:, 0] - t1).mean():.0f}; entries + range {m(0, 10):.0f}, histogram {m(10, 11):.0f}, "
          f"bin {m(11, 12):.0f}, gather {m(12, 13):.0f}, rank {m(13, 14):.0f}, winners {m(1, 2):.0f}, "
          f"their ranks {m(2, 3):.0f}, rest + writes {m(3, 4):.0f}; ends {(mrg[:, 4] - t1).mean():.0f}")


def exchange_report(xs, D, plan):
    """The state exchange seen by the global timer: for each depth, the spread
    of the CTAs' publication times and how long after the last publication
    each CTA held every state."""
    import re
    m = re.search(r"on (\d+) CTAs", plan)
    G = min(int(m.group(1)), XCTAS) if m else XCTAS
    pub, got = xs[:, 0, :, :G], xs[:, 1, :, :G]  # [rounds, depth, cta]
    print(f"\nexchange (global timer, ns; {G} CTAs, mean over rounds)")
    print("depth  pub spread  last-pub CTA (mode)  got - last pub: min / median / max")
    spreads, lat_med, lat_max = [], [], []
    for i in range(1, D):
        p, q = pub[:, i], got[:, i]
        last = p.max(axis=1)
        spread = (last - p.min(axis=1)).mean()
        lat = q - last[:, None]
        who = np.bincount(p.argmax(axis=1), minlength=G).argmax()
        spreads.append(spread)
        lat_med.append(np.median(lat, axis=1).mean())
        lat_max.append(lat.max(axis=1).mean())
        print(f"{i:5d}  {spread:10.0f}  {who:19d}  {lat.min(axis=1).mean():7.0f} / {lat_med[-1]:7.0f} / "
              f"{lat_max[-1]:7.0f}")
    print(f"mean   {np.mean(spreads):10.0f}  {'':19s}  {'':7s}   {np.mean(lat_med):7.0f} / {np.mean(lat_max):7.0f}")
    # the publication order: mean lateness of each CTA against the first one
    late = (pub[:, 1:D] - pub[:, 1:D].min(axis=2, keepdims=True)).mean(axis=(0, 1))
    order = np.argsort(-late)
    print("latest publishers (CTA: mean ns after the first): " +
          ", ".join(f"{c}: {late[c]:.0f}" for c in order[:8]))
    print("earliest publishers: " + ", ".join(f"{c}: {late[c]:.0f}" for c in order[-4:]))
    d = np.diff(np.sort(np.unique(pub[0, 1:D].ravel())))
    if d.size:
        print(f"timer step (smallest nonzero difference seen): {d[d > 0].min() if (d > 0).any() else 0} ns")


if __name__ == "__main__":
    main()
