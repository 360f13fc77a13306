"""Helpers shared by the GPU parity tests, smoke() and the bench's checks.

They upload seeded workloads, run the CUDA path through the C ABI, and compare
its results with the fp64 oracle: token / parent / depth / mask bit-exact,
log-probabilities within 2e-3 absolute; a mismatching round is excused only
when the oracle shows an outcome-relevant near-tie (a selection boundary
within 1e-3 whose single flip changes the emitted tree).
"""
from __future__ import annotations

import numpy as np

LOGP_TOL = 2e-3     # absolute, node log-probs and cumulative scores
TIE_TOL = 1e-3      # near-tie window of the exclusion rule


def upload_weights(w: dict, device="cuda"):
    from conditional_draft_tree_lm_gb300 import bf16_tensor
    return {k: bf16_tensor(v, device) for k, v in w.items()}


def upload_round(H_bits, root, device="cuda"):
    import torch
    from conditional_draft_tree_lm_gb300 import bf16_tensor
    return bf16_tensor(H_bits, device), torch.from_numpy(np.ascontiguousarray(root, dtype=np.int32)).to(device)


def to_np(out: dict) -> dict:
    return {k: v.cpu().numpy() for k, v in out.items()}


def tree_matches(gpu: dict, q: int, t) -> tuple[bool, str]:
    """Compare request q of a GPU tree dict with an oracle Tree."""
    if not np.array_equal(gpu["tok"][q], t.tok):
        return False, "tok"
    if not np.array_equal(gpu["parent"][q], t.parent):
        return False, "parent"
    if not np.array_equal(gpu["depth"][q], t.depth):
        return False, "depth"
    if not np.array_equal(gpu["mask"][q], t.mask):
        return False, "mask"
    err = np.max(np.abs(gpu["logp_cum"][q].astype(np.float64) - t.logp_cum))
    if err > LOGP_TOL:
        return False, f"logp_cum err {err:.3g}"
    return True, ""


def check_round(orc, gpu: dict, H_bits, root, beta=None, T=None, ells=None):
    """Per-request verdicts: list of (status, detail) with status in
    {"match", "excused", "MISMATCH"}."""
    from oracle.dartree import near_tie_report
    res = []
    for q in range(H_bits.shape[0]):
        ell = None if ells is None else ells[q]
        t = orc.build_request(H_bits[q], int(root[q]), beta=beta, T=T, ell=ell)
        ok, why = tree_matches(gpu, q, t)
        if ok:
            res.append(("match", ""))
            continue
        rep = near_tie_report(orc, H_bits[q], int(root[q]), tol=TIE_TOL, beta=beta, T=T, ell=ell)
        if rep["relevant"]:
            res.append(("excused", why + f" ({len(rep['relevant_ties'])} relevant near-ties)"))
        else:
            res.append(("MISMATCH", why))
    return res


def report_counts(label: str, counts: dict, details=None) -> str:
    """One line with a test's round verdicts (printed, and used in assertion
    messages, so the number of bit-exact rounds shows in every run)."""
    line = (f"{label}: {counts.get('match', 0)} bit-exact, {counts.get('excused', 0)} excused, "
            f"{counts.get('MISMATCH', 0)} mismatched")
    print(line, flush=True)
    if details:
        bad = [d for d in details if "match" not in d]
        if bad:
            line += f" {bad}"
    return line
