"""Write the stored oracle trees used as regression fixtures.

The pages print no worked numeric example, so the fixtures here are written
by this script from the fp64 oracle alone (``oracle/``) on the tiny workload
(fp32 weights, root token id 0) and are pinned by the oracle's own pin tests.
Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle.dartree import Oracle  # noqa: E402
from workloads import get_config, make_weights, make_round_inputs  # noqa: E402


def main():
    cfg = get_config("tiny")
    w = make_weights(cfg)
    orc = Oracle(w, cfg)
    out = {"workload": cfg.as_dict(), "source": "fp64 oracle (oracle/dartree.py)", "rounds": []}
    for seed in range(3):
        H, root = make_round_inputs(cfg, seed)
        t = orc.build_request(H[0], int(root[0]))
        out["rounds"].append({
            "seed": seed,
            "root": int(root[0]),
            "cand_tok": t.cand_tok.tolist(),
            "rest_lse": [round(float(x), 12) for x in t.rest_lse],
            "node_tok": t.node_tok.tolist(),
            "node_parent": t.node_parent.tolist(),
            "node_score": [round(float(x), 12) for x in t.node_score],
            "sel": t.sel.tolist(),
            "tok": t.tok.tolist(),
            "parent": t.parent.tolist(),
            "depth": t.depth.tolist(),
            "logp_cum": [round(float(x), 12) for x in t.logp_cum],
        })
    with open(os.path.join(HERE, "tiny_fp32_rounds.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
