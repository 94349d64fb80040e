"""The oracle's pins catch the mistakes they are there to catch.

Each mutant is the oracle with one plausible mistake planted around it, on
the CPU: a dropped term, a wrong index, a missing bias, a flipped sign, the
wrong tie-break, swapped gate/up halves, a missing routing probability, the
wrong order inside an expert's group.  Every pin listed for a mutant must
pass on the oracle itself and fail on the mutant.
"""
import numpy as np
import pytest

from tests import test_oracle as pins


class Mutant:
    """The oracle with some of its functions replaced."""

    def __init__(self, base, **replace):
        self._base = base
        for name, make in replace.items():
            setattr(self, name, make(base))

    def __getattr__(self, name):
        return getattr(self._base, name)


def _swap_halves(w13_bits, I):
    w = np.array(w13_bits, copy=True)
    w[:, :I], w[:, I:] = w13_bits[:, I:], w13_bits[:, :I]
    return w


def _topk_ties_to_highest(base):
    def topk(scores, k):
        s = np.ascontiguousarray(np.asarray(scores)[:, ::-1])
        ids, wts = base.topk(s, k)
        return (s.shape[1] - 1 - ids).astype(np.int32), wts
    return topk


def _group_slot_before_token(base):
    def permute(ids, E):
        off, _ = base.permute(ids, E)
        flat = np.asarray(ids).reshape(-1)
        k = np.asarray(ids).shape[1]
        order = sorted(range(flat.size), key=lambda p: (flat[p], p % k, p // k))
        return off, np.array(order, np.int32)
    return permute


MUTANTS = {
    "router drops the last k term": (
        dict(router=lambda b: lambda x, w, bias=None: b.router(np.asarray(x)[:, :-1],
                                                              np.asarray(w)[:, :-1], bias)),
        [pins.test_router_exact_integer_case]),
    "router reads the rows of W in reverse": (
        dict(router=lambda b: lambda x, w, bias=None: b.router(x, np.asarray(w)[::-1], bias)),
        [pins.test_router_exact_integer_case, pins.test_router_one_hot_closed_form]),
    "router leaves out the bias": (
        dict(router=lambda b: lambda x, w, bias=None: b.router(x, w, None)),
        [pins.test_router_exact_integer_case, pins.test_router_one_hot_closed_form]),
    "sigmoid of the negated score": (
        dict(sigmoid=lambda b: lambda v: b.sigmoid(-np.asarray(v))),
        [pins.test_sigmoid_closed_forms]),
    "top-k breaks ties to the highest index": (
        dict(topk=_topk_ties_to_highest),
        [pins.test_topk_special_rows]),
    "MoE with the gate and up halves swapped": (
        dict(moe=lambda b: lambda x, ids, wts, w13, w2, E, I: b.moe(x, ids, wts, _swap_halves(w13, I),
                                                                    w2, E, I)),
        [pins.test_moe_hand_worked_example, pins.test_moe_reduces_to_dense_swiglu]),
    "MoE without the routing probability": (
        dict(moe=lambda b: lambda x, ids, wts, w13, w2, E, I: b.moe(x, ids, np.ones_like(wts), w13,
                                                                    w2, E, I)),
        [pins.test_moe_hand_worked_example, pins.test_moe_invariants]),
    "grouping by slot before token inside an expert": (
        dict(permute=_group_slot_before_token),
        [pins.test_permute_matches_stable_sort]),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_planted_mistake(oracle_mod, name):
    replace, pin_tests = MUTANTS[name]
    mutant = Mutant(oracle_mod, **replace)
    for pin in pin_tests:
        pin(oracle_mod)
        with pytest.raises(AssertionError):
            pin(mutant)


def test_brute_force_pin_catches_wrong_tie_break(oracle_mod):
    """The brute-force top-k pin (rows full of exact ties) fails on the
    mutant that breaks ties to the highest index."""
    mutant = Mutant(oracle_mod, topk=_topk_ties_to_highest)
    pins.test_topk_brute_force(oracle_mod, 5, 2)
    with pytest.raises(AssertionError):
        pins.test_topk_brute_force(mutant, 5, 2)
