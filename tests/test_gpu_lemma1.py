"""Lemma 1 on the GPU's own super-tree, at the wide-tree workload.

"DARTree: Speculative Diffusion Decoding with Autoregressive Draft Trees",
Metodología, 2. Poda Diferida, Equivalencia Teórica: with beta <= 0 the
global Top-B over score + beta * depth selects the same node set as
sequential max-heap best-first over the same super-tree.

The round runs through the step API (base logits, Top-M, the 15 depths one
launch each, then dt_prune_topB); the test then runs an independent max-heap
(pop the largest key, ties to the lower node index, push the popped node's
children) over the node arrays the GPU itself wrote, and requires the GPU's
selection to equal it exactly, and to be ancestor-closed, for
beta in {0, -0.25, -1} (M = 256, K = 32, W = 64, B = 512: 27 680 nodes).
As a negative control, at beta = +5 (DT_FLAG_POSITIVE_BETA) the two part on
some seed while the Top-B is still exactly the B largest keys.
"""
import heapq

import numpy as np
import pytest

from tests.parity import upload_round, upload_weights
from workloads import get_config, make_round_inputs, make_weights

pytestmark = pytest.mark.gpu


def _heap(parent, key, B):
    kids = [[] for _ in range(parent.size)]
    for v in range(1, parent.size):
        kids[int(parent[v])].append(v)
    h = [(-float(key[c]), c) for c in kids[0]]
    heapq.heapify(h)
    out = []
    while h and len(out) < B:
        _, v = heapq.heappop(h)
        out.append(v)
        for c in kids[v]:
            heapq.heappush(h, (-float(key[c]), c))
    return sorted(out)


@pytest.fixture(scope="module")
def wide_weights():
    import torch
    torch.cuda.set_device(0)
    cfg = get_config("wide")
    return upload_weights(make_weights(cfg))


def _gpu_super_tree(b, cfg, seed):
    """One round's super-tree through the step API, then dt_prune_topB: the
    GPU's node arrays (parent, score), node depths and selection."""
    import torch
    D = cfg.block - 1
    H, root = make_round_inputs(cfg, seed)
    Hd, rd = upload_round(H, root)
    b.base_logits(Hd)
    b.topm()
    nodes = b.new_nodes()
    for i in range(1, D + 1):
        b.expand_depth(i, rd, nodes["node_tok"], nodes["node_parent"], nodes["node_logp"], nodes["node_score"])
    sel = torch.empty(cfg.n_req, cfg.B, dtype=torch.int32, device="cuda")
    b.prune_topB(nodes["node_score"], sel)
    torch.cuda.synchronize()
    parent = nodes["node_parent"][0].cpu().numpy().astype(np.int64)
    score = nodes["node_score"][0].cpu().numpy()
    depth = np.zeros(parent.size, dtype=np.int64)
    off, n = 1, cfg.K
    for i in range(1, D + 1):
        depth[off:off + n] = i
        off += n
        n = min(cfg.W, n) * cfg.K
    return parent, score, depth, sel[0].cpu().numpy().tolist()


def test_gpu_top_b_differs_from_heap_at_positive_beta(wide_weights):
    """The negative control (beta = +5, DT_FLAG_POSITIVE_BETA): Lemma 1 needs
    beta <= 0, and with a depth bonus the GPU's global Top-B and a max-heap
    over the same GPU super-tree part on some seed; the Top-B itself is still
    exactly the B largest keys (ties to the lower node index)."""
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    cfg = get_config("wide", beta=5.0, positive_beta=True)
    b = DraftTreeBuilder(cfg, wide_weights)
    try:
        differs = 0
        for seed in range(2):
            parent, score, depth, got = _gpu_super_tree(b, cfg, seed)
            key = (score + np.float32(5.0) * depth.astype(np.float32)).astype(np.float32)
            order = np.lexsort((np.arange(1, key.size), -key[1:].astype(np.float64))) + 1
            assert got == sorted(order[:cfg.B].tolist()), seed
            differs += got != _heap(parent, key, cfg.B)
        assert differs > 0, "beta > 0 never parted the global Top-B from the heap: the Lemma 1 check is vacuous"
    finally:
        b.close()


@pytest.mark.parametrize("beta", [0.0, -0.25, -1.0])
def test_gpu_top_b_equals_heap_over_gpu_nodes(wide_weights, beta):
    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    cfg = get_config("wide", beta=beta)
    D = cfg.block - 1
    b = DraftTreeBuilder(cfg, wide_weights)
    try:
        for seed in range(2):
            H, root = make_round_inputs(cfg, seed)
            Hd, rd = upload_round(H, root)
            b.base_logits(Hd)
            b.topm()
            nodes = b.new_nodes()
            for i in range(1, D + 1):
                b.expand_depth(i, rd, nodes["node_tok"], nodes["node_parent"], nodes["node_logp"],
                               nodes["node_score"])
            sel = torch.empty(cfg.n_req, cfg.B, dtype=torch.int32, device="cuda")
            b.prune_topB(nodes["node_score"], sel)
            torch.cuda.synchronize()
            parent = nodes["node_parent"][0].cpu().numpy().astype(np.int64)
            score = nodes["node_score"][0].cpu().numpy()
            # node depth from the depth-major numbering (n_1 = K, n_i = min(W, n_{i-1}) K)
            depth = np.zeros(parent.size, dtype=np.int64)
            off, n = 1, cfg.K
            for i in range(1, D + 1):
                depth[off:off + n] = i
                off += n
                n = min(cfg.W, n) * cfg.K
            assert off == parent.size
            assert np.all(parent[1:] < np.arange(1, parent.size))
            assert np.all(depth[1:] == depth[parent[1:]] + 1)
            # the key as the GPU forms it: fp32 score + beta * depth, in fp32
            key = (score + np.float32(beta) * depth.astype(np.float32)).astype(np.float32)
            got = sel[0].cpu().numpy().tolist()
            assert got == _heap(parent, key, cfg.B), (seed, beta)
            chosen = set(got) | {0}
            assert all(int(parent[v]) in chosen for v in got), (seed, beta)
        assert b.device_status() == 0
    finally:
        b.close()
