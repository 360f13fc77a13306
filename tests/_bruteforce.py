"""Independent restatement of one path's score, built from torch library layers.

Used to pin the oracle: for a token path root -> t_1 -> ... -> t_k it re-runs
the GRU from the root along that path with ``torch.nn.GRUCell`` (PyTorch gate
order, the hidden bias set to zero), the correction with ``torch.nn.Linear`` +
``torch.nn.functional.silu``, restricts the correction to the Top-M base
logits of each depth (``torch.sort``, stable, so ties keep the lower token id)
and takes ``torch.log_softmax`` over the whole vocabulary.  Nothing here is
shared with the oracle's code.
"""
from __future__ import annotations

import numpy as np
import torch

from workloads import bf16_bits_to_f32


def _t(x):
    x = np.asarray(x)
    if x.dtype == np.uint16:
        x = bf16_bits_to_f32(x)
    return torch.from_numpy(np.ascontiguousarray(x).astype(np.float64))


class PathScorer:
    def __init__(self, weights, cfg, T=None):
        self.cfg = cfg
        self.T = cfg.T if T is None else T
        d, g, r, V = cfg.d, cfg.g, cfg.r, cfg.V
        self.gru = torch.nn.GRUCell(d, g, bias=True, dtype=torch.float64)
        self.lin1 = torch.nn.Linear(d + g, r, bias=False, dtype=torch.float64)
        self.lin2 = torch.nn.Linear(r, V, bias=False, dtype=torch.float64)
        self.head = torch.nn.Linear(d, V, bias=False, dtype=torch.float64)
        with torch.no_grad():
            self.gru.weight_ih.copy_(_t(weights["w_ih"]))
            self.gru.bias_ih.copy_(_t(weights["b_ih"]))
            self.gru.weight_hh.copy_(_t(weights["w_hh"]))
            self.gru.bias_hh.zero_()
            self.lin1.weight.copy_(_t(weights["w1"]))
            self.lin2.weight.copy_(_t(weights["w2"]))
            self.head.weight.copy_(_t(weights["lm_head"]))
        self.emb = _t(weights["emb"])

    @torch.no_grad()
    def depth_logprobs(self, H, i, h):
        """Full-vocabulary corrected log-probs at depth i given the state h."""
        Hi = _t(H[i])
        base = self.head(Hi)
        order = torch.sort(base, descending=True, stable=True).indices
        cand = order[: self.cfg.M]
        dL = self.lin2(torch.nn.functional.silu(self.lin1(torch.cat([Hi, h]))))
        full = base.clone()
        full[cand] = full[cand] + dL[cand]
        return torch.log_softmax(full / self.T, dim=0), cand

    @torch.no_grad()
    def root_state(self, root_tok):
        g = self.cfg.g
        return self.gru(self.emb[root_tok][None], torch.zeros(1, g, dtype=torch.float64))[0]

    @torch.no_grad()
    def path_score(self, H, root_tok, path):
        h = self.root_state(root_tok)
        s = 0.0
        for i, t in enumerate(path, start=1):
            lp, _ = self.depth_logprobs(H, i, h)
            s += float(lp[t])
            h = self.gru(self.emb[t][None], h[None])[0]
        return s

    @torch.no_grad()
    def children(self, H, root_tok, path, K):
        """Top-K children tokens of the node reached by ``path`` (ties -> lower id)."""
        h = self.root_state(root_tok)
        for t in path:
            h = self.gru(self.emb[t][None], h[None])[0]
        i = len(path) + 1
        lp, cand = self.depth_logprobs(H, i, h)
        vals = lp[cand].numpy()
        ids = cand.numpy()
        order = np.lexsort((ids, -vals))[:K]
        return sorted(int(ids[j]) for j in order)


def node_path(node_tok, node_parent, v):
    path = []
    while v > 0:
        path.append(int(node_tok[v]))
        v = int(node_parent[v])
    return tuple(reversed(path))
