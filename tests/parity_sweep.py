"""Parity sweep: many seeded rounds through the CUDA path against the fp64 oracle.

Reports what the parity bar asks for ("near-tie exclusion" reading R9): the
rounds that match bit for bit, the mismatching rounds the oracle excuses by an
outcome-relevant near-tie (a selection boundary within 1e-3 whose single flip
changes the emitted tree), the unexcused mismatches (must be 0), the fraction
of rounds with any literal near-tie at a selection boundary, the fraction with
an outcome-relevant one (on a subsample, each needs one oracle re-run per
recorded tie), and the largest cumulative-score error of the matching rounds.

Needs a GPU.  Usage:
    python -m tests.parity_sweep --workload qwen3_4b --rounds 200 --relevance 30 --out sweep.json
"""
from __future__ import annotations

import argparse
import json
import time

import numpy as np


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="qwen3_4b")
    ap.add_argument("--rounds", type=int, default=200)
    ap.add_argument("--first-seed", type=int, default=0)
    ap.add_argument("--relevance", type=int, default=30, help="rounds whose near-ties are re-run for relevance")
    ap.add_argument("--T", type=float, default=None, help="override the workload's temperature")
    ap.add_argument("--beta", type=float, default=None, help="override the workload's depth penalty")
    ap.add_argument("--out", default=None)
    args = ap.parse_args()

    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    from oracle.besttree import best_first_tie_report, build_best_first
    from oracle.dartree import Oracle, base_logits, near_tie_report
    from tests.parity import TIE_TOL, to_np, tree_matches, upload_round, upload_weights
    from workloads import get_config, make_round_inputs, make_weights

    torch.cuda.set_device(0)
    over = {k: v for k, v in (("T", args.T), ("beta", args.beta)) if v is not None}
    cfg = get_config(args.workload, **over)
    best_first = getattr(cfg, "builder", "dartree") == "best_first"

    def oracle_tree(Hq, rq, ell, rec=None):
        if best_first:
            return build_best_first(orc, Hq, rq, ell=ell, rec=rec, tol=TIE_TOL if rec is not None else None)
        return orc.build_request(Hq, rq, ell=ell, rec=rec, tol=TIE_TOL if rec is not None else None)

    def relevant_tie(Hq, rq, ell):
        rep_ = (best_first_tie_report if best_first else near_tie_report)(orc, Hq, rq, tol=TIE_TOL, ell=ell)
        return rep_["relevant"]

    w = make_weights(cfg)
    b = DraftTreeBuilder(cfg, upload_weights(w))
    orc = Oracle(w, cfg)
    res = dict(workload=cfg.name, T=cfg.T, beta=cfg.beta, rounds=0, requests=0, match=0, excused=0,
               unexcused=0, literal_tie=0, relevance_sample=0, relevant_tie=0, max_score_err_matching=0.0,
               unexcused_details=[])
    t0 = time.time()
    try:
        for s in range(args.first_seed, args.first_seed + args.rounds):
            H, root = make_round_inputs(cfg, s)
            out = to_np(b.build_round(*upload_round(H, root)))
            res["rounds"] += 1
            for q in range(cfg.n_req):
                res["requests"] += 1
                ell = base_logits(H[q][1:], w["lm_head"])
                rec = []
                t = oracle_tree(H[q], int(root[q]), ell, rec=rec)
                literal = bool(rec)
                res["literal_tie"] += int(literal)
                ok, why = tree_matches(out, q, t)
                sampled = res["relevance_sample"] < args.relevance
                relevant = None
                if (not ok or sampled) and literal:
                    relevant = relevant_tie(H[q], int(root[q]), ell)
                if sampled:
                    res["relevance_sample"] += 1
                    res["relevant_tie"] += int(bool(relevant))
                if ok:
                    res["match"] += 1
                    err = float(np.max(np.abs(out["logp_cum"][q].astype(np.float64) - t.logp_cum)))
                    res["max_score_err_matching"] = max(res["max_score_err_matching"], err)
                elif relevant:
                    res["excused"] += 1
                else:
                    res["unexcused"] += 1
                    res["unexcused_details"].append(dict(seed=s, request=q, why=why))
        res["device_status"] = b.device_status()
    finally:
        b.close()
    n = max(1, res["requests"])
    res["excused_fraction"] = res["excused"] / n
    res["literal_tie_fraction"] = res["literal_tie"] / n
    res["relevant_tie_fraction_sampled"] = res["relevant_tie"] / max(1, res["relevance_sample"])
    res["seconds"] = time.time() - t0
    line = json.dumps(res)
    print(line)
    if args.out:
        with open(args.out, "w") as f:
            f.write(line + "\n")


if __name__ == "__main__":
    main()
