"""Pins of the near-tie excusal rule (the only divergence the GPU parity tests
may forgive).

The rule ("Resumen Técnico: DominoTree", Resultados Experimentales, Ausencia
de Pérdida: bit-identical trees up to ties): a GPU round that differs from the
oracle is excused only when some selection boundary of the oracle's own build
has a gap within the window AND flipping that single decision, then re-running
the rest of the round, changes the emitted tokens, parents or depths.

Both report functions (``oracle.dartree.near_tie_report`` for the depth-batched
build, ``oracle.besttree.best_first_tie_report`` for the best-first heap) are
pinned on hand-built base logits under marginal scoring, where every
selection key is a function of those logits alone, so the test knows which
decisions are near-ties and which flips matter:

* a Top-M boundary near-tie between two tokens far below every branch's top-K
  is recorded but is NOT outcome-relevant (swapping them cannot change any
  child);
* a top-K boundary near-tie at the root's expansion IS outcome-relevant (the
  swapped token is a child that the emitted tree keeps).

Planted mistakes (each must fail one of these pins): every recorded tie
called relevant; the swap never applied in the re-run; the re-run rebuilding
the base logits from H instead of the ones it was given.
"""
import numpy as np
import pytest

import oracle.besttree as ob
import oracle.dartree as od
from oracle.besttree import best_first_tie_report
from oracle.dartree import Oracle, near_tie_report
from workloads import get_config, make_round_inputs, make_weights

TOL = 1e-3
GAP = 1e-4  # the planted near-ties


def _spacing(i):
    # per-depth spacing of the candidate logits, chosen so that sums of
    # spacings over a path never coincide within the window
    return 1.7 + 0.31 * i + 0.0137 * i * i


def _logits(cfg, planted):
    """Hand-built base logits [D, V].  planted: "M" puts a near-tie between the
    M-th and (M+1)-th candidates of depth 3; "K" puts one between the K-th and
    (K+1)-th candidates of depth 1 (the root's expansion)."""
    D, V, M, K = cfg.block - 1, cfg.V, cfg.M, cfg.K
    ell = np.empty((D, V))
    for i in range(1, D + 1):
        rng = np.random.default_rng([9, i])
        order = rng.permutation(V)
        c = _spacing(i)
        vals = 12.0 - c * np.arange(M + 1)
        vals[M] = vals[M - 1] - (GAP if (planted == "M" and i == 3) else 1.0)
        if planted == "K" and i == 1:
            # the root's K children are nearly as likely as each other, so
            # every one of them is kept in the emitted tree
            vals[:K + 1] = 12.0 - 0.07 * np.arange(K + 1)
            vals[K] = vals[K - 1] - GAP
            vals[K + 1:] = vals[K] - 2.0 - c * np.arange(M - K)
        row = vals[M] - 3.0 - np.abs(rng.standard_normal(V))
        row[order[:M + 1]] = vals
        ell[i - 1] = row
    return ell, order


@pytest.fixture(scope="module")
def setup():
    cfg = get_config("tiny", marginal=True)
    w = make_weights(cfg)
    H, root = make_round_inputs(cfg, 0)
    return cfg, w, H, int(root[0])


def _depth_report(cfg, w, H, root, planted):
    ell, _ = _logits(cfg, planted)
    return near_tie_report(Oracle(w, cfg), H[0], root, tol=TOL, ell=ell)


def _best_report(cfg, w, H, root, planted):
    ell, _ = _logits(cfg.with_(builder="best_first"), planted)
    return best_first_tie_report(Oracle(w, cfg), H[0], root, tol=TOL, ell=ell)


# ---------------------------------------------------------------------------
# the pins
# ---------------------------------------------------------------------------
def _pin_not_relevant(rep):
    m_ties = [t for t in rep["ties"] if t["stage"] == "M"]
    assert rep["literal"] and m_ties, "the planted Top-M near-tie was not recorded"
    assert all(abs(t["gap"] - GAP) < 1e-9 for t in m_ties)
    assert not rep["relevant"], rep["relevant_ties"]


def _pin_relevant(rep):
    k_ties = [t for t in rep["relevant_ties"] if t["stage"] == "K"]
    assert rep["relevant"] and k_ties, "the planted top-K near-tie was not found outcome-relevant"
    assert all(abs(t["gap"] - GAP) < 1e-9 for t in k_ties)


def test_depth_batched_not_relevant_tie(setup):
    _pin_not_relevant(_depth_report(*setup, "M"))


def test_depth_batched_relevant_tie(setup):
    _pin_relevant(_depth_report(*setup, "K"))


def test_best_first_not_relevant_tie(setup):
    _pin_not_relevant(_best_report(*setup, "M"))


def test_best_first_relevant_tie(setup):
    _pin_relevant(_best_report(*setup, "K"))


def test_only_planted_ties_are_recorded(setup):
    """No boundary other than the planted one comes within the window, so the
    pins above test exactly the planted decision."""
    for fn in (_depth_report, _best_report):
        for planted, stage in (("M", "M"), ("K", "K")):
            rep = fn(*setup, planted)
            assert [t["stage"] for t in rep["ties"]] == [stage], (fn.__name__, planted, rep["ties"])


# ---------------------------------------------------------------------------
# planted mistakes: each must fail at least one pin
# ---------------------------------------------------------------------------
def _all_relevant(monkeypatch):
    monkeypatch.setattr(od, "_same_tree", lambda a, b: False)


def _swap_ignored(monkeypatch):
    orig_d, orig_b = od.Oracle.build_request, ob.build_best_first

    def d(self, *a, swaps=None, **kw):
        return orig_d(self, *a, **kw)

    def b(*a, swaps=None, **kw):
        return orig_b(*a, **kw)
    monkeypatch.setattr(od.Oracle, "build_request", d)
    monkeypatch.setattr(ob, "build_best_first", b)


def _ell_ignored_on_rerun(monkeypatch):
    orig_d, orig_b = od.Oracle.build_request, ob.build_best_first

    def d(self, *a, swaps=None, ell=None, **kw):
        return orig_d(self, *a, swaps=swaps, ell=None if swaps else ell, **kw)

    def b(*a, swaps=None, ell=None, **kw):
        return orig_b(*a, swaps=swaps, ell=None if swaps else ell, **kw)
    monkeypatch.setattr(od.Oracle, "build_request", d)
    monkeypatch.setattr(ob, "build_best_first", b)


PINS = [
    (_depth_report, "M", _pin_not_relevant), (_depth_report, "K", _pin_relevant),
    (_best_report, "M", _pin_not_relevant), (_best_report, "K", _pin_relevant),
]


@pytest.mark.parametrize("plant", [_all_relevant, _swap_ignored, _ell_ignored_on_rerun])
@pytest.mark.parametrize("builder", ["depth", "best"])
def test_planted_mistakes_are_caught(setup, monkeypatch, plant, builder):
    plant(monkeypatch)
    fn = _depth_report if builder == "depth" else _best_report
    caught = False
    for f, planted, pin in PINS:
        if f is not fn:
            continue
        try:
            pin(f(*setup, planted))
        except Exception:  # a failed pin, or a re-run that cannot apply its flip
            caught = True
    assert caught, f"planted mistake {plant.__name__} passed every pin of the {builder} report"
