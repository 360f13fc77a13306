"""Pins of the acceptance-walk oracle (``oracle/accept.py``), no GPU.

Greedy tree verification ("Resumen Técnico: DominoTree", Metodología, 5.
Verificación; Resultados Experimentales, Ausencia de Pérdida) is pinned by:

* row maxima against a plain loop with explicit ties (lower token id wins);
* the accepted path against the deepest slot whose every edge matches the
  target's token at its parent, found by checking each slot's ancestor chain
  (no walk);
* losslessness: with target logits whose maximum follows a next-token function
  of the prefix, the committed tokens equal serial greedy decoding of that
  function;
* a hand-worked example (``tests/golden/accept_walk_small.json``);
* planted mistakes in the oracle, each caught by one of the pins above.
"""
import json
import os

import numpy as np
import pytest

import oracle.accept as oa
from workloads import make_target_logits, make_tree

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accept_walk_small.json")


def _loop_argmax(row):
    best, arg = -np.inf, -1
    for v, x in enumerate(row):
        if x > best:  # strict: the first (lowest) index keeps a tie
            best, arg = x, v
    return arg


def _pin_argmax():
    rng = np.random.default_rng(7)
    Z = rng.integers(0, 4, size=(40, 23)).astype(np.float32)  # many exact ties
    got = oa.target_argmax(Z)
    want = [_loop_argmax(r) for r in Z]
    assert got.tolist() == want


def _pin_golden():
    g = json.load(open(GOLDEN))
    v = oa.accept_walk(np.array(g["tok"]), np.array(g["parent"]), np.array(g["Z"], dtype=np.float32))
    assert v.target_tok.tolist() == g["target_tok"]
    assert v.accepted == g["accepted"]
    assert v.bonus == g["bonus"]
    assert v.tau == g["tau"]


def _pin_bruteforce(seeds=range(40)):
    for s in seeds:
        S, V, D = 30, 12, 6
        tok, parent, _ = make_tree(S, V, D, s)
        Z = make_target_logits(tok, parent, V, s, follow=0.9, tie=(s % 3 == 0))
        y = [_loop_argmax(r) for r in Z]
        # slots whose every edge from the root matches the target's token at the parent
        ok = []
        for c in range(1, S):
            a, good = c, True
            while a != 0:
                if tok[a] != y[parent[a]]:
                    good = False
                    break
                a = parent[a]
            if good:
                ok.append(c)
        deepest = 0
        for c in ok:
            depth_c = 0
            a = c
            while a != 0:
                a, depth_c = parent[a], depth_c + 1
            depth_d = 0
            a = deepest
            while a != 0:
                a, depth_d = parent[a], depth_d + 1
            if depth_c > depth_d:
                deepest = c
        path = []
        a = deepest
        while a != 0:
            path.append(a)
            a = parent[a]
        path.reverse()
        assert sorted(path) == sorted(ok), "matching slots form one chain"
        v = oa.accept_walk(tok, parent, Z)
        assert v.accepted == path, s
        assert v.bonus == y[deepest] and v.tau == len(path) + 1, s


def _next_token(prefix, V):
    h = 17
    for t in prefix:
        h = (h * 1000003 + int(t) + 1) % 2147483647
    return h % V


def _pin_lossless(seeds=range(25)):
    for s in seeds:
        S, V, D = 40, 9, 8
        tok, parent, _ = make_tree(S, V, D, 100 + s)
        tok = tok.copy()
        # retokenise each child to the target's next token where no sibling has it yet
        rng = np.random.default_rng([9, s])
        path_toks = {0: (int(tok[0]),)}
        for c in range(1, S):
            p = int(parent[c])
            want = _next_token(path_toks[p], V)
            sib = [int(tok[k]) for k in range(1, c) if parent[k] == p]
            if rng.random() < 0.8 and want not in sib:
                tok[c] = want
            elif int(tok[c]) in sib:
                tok[c] = next(t for t in range(V) if t not in sib)
            path_toks[c] = path_toks[p] + (int(tok[c]),)
        Z = rng.standard_normal((S, V)).astype(np.float32)
        for a in range(S):
            Z[a, _next_token(path_toks[a], V)] = 10.0
        v = oa.accept_walk(tok, parent, Z)
        committed = [int(tok[c]) for c in v.accepted] + [v.bonus]
        # serial greedy decoding of the target from the root
        prefix = (int(tok[0]),)
        serial = []
        for _ in range(v.tau):
            t = _next_token(prefix, V)
            serial.append(t)
            prefix = prefix + (t,)
        assert committed == serial, s
        # and the walk stopped because the tree has no continuation
        last = v.accepted[-1] if v.accepted else 0
        nxt = _next_token(path_toks[last], V)
        assert not any(parent[c] == last and tok[c] == nxt for c in range(1, S))


def test_argmax_ties_to_lower_id():
    _pin_argmax()


def test_golden_hand_worked():
    _pin_golden()


def test_walk_is_deepest_matching_chain():
    _pin_bruteforce()


def test_walk_is_lossless():
    _pin_lossless()


def test_generator_trees_are_valid():
    for s in range(10):
        tok, parent, depth = make_tree(65, 151936, 15, s)
        assert parent[0] == -1 and all(0 <= parent[c] < c for c in range(1, 65))
        assert depth.max() <= 15
        for a in range(65):
            sib = tok[1:][parent[1:] == a]
            assert len(set(sib.tolist())) == sib.size


def _planted(name):
    real_walk, real_argmax = oa.accept_walk, oa.target_argmax
    if name == "ties_to_higher_id":
        def f(Z):
            Z = np.asarray(Z)
            return (Z.shape[1] - 1 - np.argmax(Z[:, ::-1], axis=1)).astype(np.int64)
        return {"target_argmax": f}
    if name == "no_bonus":
        def w(tok, parent, Z):
            v = real_walk(tok, parent, Z)
            v.tau = len(v.accepted)
            return v
        return {"accept_walk": w}
    if name == "child_own_logits":
        def w(tok, parent, Z):
            y = oa.target_argmax(Z)
            S = len(tok)
            acc, a = [], 0
            while True:
                nxt = [c for c in range(1, S) if parent[c] == a and tok[c] == y[c]]
                if not nxt:
                    break
                a = nxt[0]
                acc.append(a)
            return oa.WalkResult(y, acc, int(y[a]), len(acc) + 1)
        return {"accept_walk": w}
    if name == "one_step_only":
        def w(tok, parent, Z):
            v = real_walk(tok, parent, Z)
            acc = v.accepted[:1]
            last = acc[-1] if acc else 0
            return oa.WalkResult(v.target_tok, acc, int(v.target_tok[last]), len(acc) + 1)
        return {"accept_walk": w}
    if name == "bonus_from_root":
        def w(tok, parent, Z):
            v = real_walk(tok, parent, Z)
            v.bonus = int(v.target_tok[0])
            return v
        return {"accept_walk": w}
    raise KeyError(name)


@pytest.mark.parametrize("name", ["ties_to_higher_id", "no_bonus", "child_own_logits", "one_step_only",
                                  "bonus_from_root"])
def test_planted_mistakes_are_caught(monkeypatch, name):
    for attr, fn in _planted(name).items():
        monkeypatch.setattr(oa, attr, fn)
    caught = 0
    for pin in (_pin_argmax, _pin_golden, _pin_bruteforce, _pin_lossless):
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught >= 1, name
