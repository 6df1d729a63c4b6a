"""Planted mistakes in the oracle (CPU only): each deliberately broken copy of
the naive single-head attention must fail at least one pin.  This is what
makes the pins worth trusting: a dropped term, a wrong sign or index, a
transposed operand or a wrong alignment would not slip through."""

import math

import numpy as np
import pytest

from oracle_pins import ALL_CHECKS


def _make(mut):
    def fn(q, k, v, scale, causal):
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
        Lq, Lk = q.shape[0], k.shape[0]
        sc = {"no_scale": 1.0, "scale_squared": scale * scale}.get(mut, scale)
        S = sc * (q @ k.T) if mut != "transposed" else sc * (k @ q.T)  # S_ij = q_j . k_i
        i = np.arange(Lq)[:, None]
        j = np.arange(Lk)[None, :]
        if causal:
            if mut == "strict_causal":
                vis = j < i + (Lk - Lq)
            elif mut == "top_left_causal":
                vis = j <= i
            elif mut == "causal_flipped":
                vis = j >= i + (Lk - Lq)
            else:
                vis = j <= i + (Lk - Lq)
        else:
            vis = np.ones((Lq, Lk), dtype=bool)
        Sm = np.where(vis, S, -np.inf)
        anyv = vis.any(axis=1)
        m = np.where(anyv, Sm.max(axis=1, initial=-np.inf), 0.0)
        E = np.where(vis, np.exp(Sm - m[:, None]), 0.0)
        if mut == "drop_last_key":
            E[:, -1] = 0.0
        l = E.sum(axis=1)
        if mut == "softmax_wrong_axis":
            col = E.sum(axis=0, keepdims=True)
            P = E / np.where(col == 0, 1.0, col)
        elif mut == "unnormalised":
            P = E
        else:
            P = E / np.where(anyv, l, 1.0)[:, None]
        O = P @ (k[:, : v.shape[1]] if (mut == "uses_k" and k.shape[1] >= v.shape[1]) else v)
        O = np.where(anyv[:, None], O, 0.0)
        if mut == "lse_without_max":
            lse = np.log(np.where(anyv, l, 1.0))
        elif mut == "lse_log2":
            lse = m + np.log2(np.where(anyv, l, 1.0))
        elif mut == "lse_unmasked":
            mm = S.max(axis=1)
            lse = mm + np.log(np.exp(S - mm[:, None]).sum(axis=1))
        else:
            lse = m + np.log(np.where(anyv, l, 1.0))
        lse = np.where(anyv, lse, -np.inf) if mut != "lse_unmasked" else lse
        return O, lse

    return fn


MUTANTS = [
    "no_scale", "scale_squared", "transposed", "strict_causal", "top_left_causal",
    "causal_flipped", "drop_last_key", "softmax_wrong_axis", "unnormalised", "uses_k",
    "lse_without_max", "lse_log2", "lse_unmasked",
]


@pytest.mark.parametrize("mut", MUTANTS)
def test_mutant_is_caught(mut):
    fn = _make(mut)
    failed = []
    for check in ALL_CHECKS:
        try:
            check(fn)
        except Exception:  # an assertion or a shape error both count as caught
            failed.append(check.__name__)
    assert failed, f"mutant {mut} passed every pin"


def test_unmutated_copy_passes():
    """The harness itself is sound: the copy with no mutation passes all."""
    fn = _make("none")
    for check in ALL_CHECKS:
        check(fn)
