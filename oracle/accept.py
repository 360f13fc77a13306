"""CPU oracle of greedy tree verification: the acceptance walk over an emitted tree.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference arm of ``bench.py`` may import or run this module.
The CUDA library never calls it and shares no code with it.

What it computes.  The target model scores every slot of the emitted tree in
one forward pass with the ancestor-only mask ("Resumen Técnico: DominoTree",
Metodología, 5. Verificación; "DARTree: Speculative Diffusion Decoding with
Autoregressive Draft Trees", Metodología, 2. Poda Diferida, Verificación).
Its logits at slot a predict the token that follows the path root..a.  With
greedy verification the walk is lossless: it commits exactly the tokens that
serial greedy decoding of the target would produce (same page, Resultados
Experimentales, Ausencia de Pérdida).  Steps, per request:

1. y_a = argmax_v Z[a, v] for every slot a of the tree (the target's token
   after slot a).  Reading: equal maxima go to the lower token id.
2. From the root, move to the child c of the current slot a whose draft token
   equals y_a, while one exists (siblings carry distinct tokens, so there is at
   most one).  The slots moved into are the accepted drafts.
3. The target's token at the last accepted slot (the root when none) is the
   bonus token; tau = accepted + 1 tokens are committed this round.

Pins (``tests/test_oracle_accept.py``): brute-force row maxima with explicit
ties, the deepest slot whose every edge matches (found without walking),
serial greedy decoding of a target defined by a next-token function of the
prefix, a hand-worked example in ``tests/golden/``, and planted mistakes.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class WalkResult:
    target_tok: np.ndarray  # [S] int64: y_a per slot
    accepted: list           # accepted slots in path order (root excluded)
    bonus: int               # the target's token at the last accepted slot
    tau: int                 # accepted + 1


def target_argmax(Z: np.ndarray) -> np.ndarray:
    """Per row of Z [S, V]: the index of the largest value, lower index on ties
    (numpy's argmax returns the first occurrence of the maximum)."""
    return np.argmax(np.asarray(Z), axis=1).astype(np.int64)


def accept_walk(tok, parent, Z) -> WalkResult:
    """Greedy verification of one tree.  tok, parent: [S] with parent[0] = -1
    and parent[c] < c; Z: [S, V] target logits per slot."""
    tok = np.asarray(tok, dtype=np.int64)
    parent = np.asarray(parent, dtype=np.int64)
    y = target_argmax(Z)
    S = tok.size
    children = [[] for _ in range(S)]
    for c in range(1, S):
        children[int(parent[c])].append(c)
    accepted = []
    a = 0
    while True:
        nxt = [c for c in children[a] if tok[c] == y[a]]
        if not nxt:
            break
        if len(nxt) > 1:
            raise ValueError("siblings share a token")
        a = nxt[0]
        accepted.append(a)
    return WalkResult(target_tok=y, accepted=accepted, bonus=int(y[a]), tau=len(accepted) + 1)


def accept_walk_rounds(tok, parent, Z):
    """accept_walk over [n_req, S] trees and [n_req, S, V] logits."""
    return [accept_walk(tok[q], parent[q], Z[q]) for q in range(np.asarray(tok).shape[0])]
