"""The validity rule the GPU tests apply to sequences left out of the bit-exact
comparison (tests/gpu_util.check_decision_validity), checked on the CPU: decisions the
oracle takes pass, decisions that break the sampler's rule fail."""
import numpy as np
import pytest

import oracle
from gpu_util import check_decision_validity

MASK = 3


def _oracle_case(conf_vals, gamma, steps=0, T=16, decoded=()):
    """Logits rows whose confidences are exactly conf_vals (two-valued rows: the top
    logit a, every other id 0, conf = e^a / (e^a + V - 2) with the mask id removed),
    and the oracle's step on them."""
    S, V = len(conf_vals), 64
    ids = np.full(S, MASK, np.int64)
    for p in decoded:
        ids[p] = 40
    lg = np.zeros((S, V))
    for i, c in enumerate(conf_vals):
        a = np.log(c * (V - 2) / (1.0 - c))
        lg[i, 10 + i] = a
    r = oracle.unmask_step(lg, ids, steps, MASK, gamma, T)
    return ids, r


def _check(ids0, r, ids_g, com, gamma, kind=0, band=1e-5):
    check_decision_validity(ids_g, com, ids0, r["tok"], r["conf"], MASK, kind, gamma, r["k_min"],
                            band * r["conf"])


def test_oracle_decision_is_valid():
    ids0, r = _oracle_case([0.9, 0.5, 0.85, 0.2], 0.8)
    _check(ids0, r, r["ids"], r["commit"], 0.8)


def test_floor_decision_is_valid():
    ids0, r = _oracle_case([0.3, 0.5, 0.6, 0.2], 0.8)
    assert r["commit"].tolist() == [0, 0, 1, 0]
    _check(ids0, r, r["ids"], r["commit"], 0.8)


@pytest.mark.parametrize("plant", ["skip_above", "take_below", "wrong_token", "no_remask",
                                   "floor_wrong_one", "floor_too_many", "commit_decoded"])
def test_invalid_decisions_fail(plant):
    gamma = 0.8
    if plant.startswith("floor"):
        ids0, r = _oracle_case([0.3, 0.5, 0.6, 0.2], gamma)
    elif plant == "commit_decoded":
        ids0, r = _oracle_case([0.9, 0.5, 0.85, 0.2], gamma, decoded=(1,))
    else:
        ids0, r = _oracle_case([0.9, 0.5, 0.85, 0.2], gamma)
    ids, com = r["ids"].copy(), r["commit"].astype(bool).copy()
    if plant == "skip_above":          # a position clearly above gamma left masked
        com[2] = False
        ids[2] = MASK
    elif plant == "take_below":        # a position clearly below gamma committed
        com[1] = True
        ids[1] = r["tok"][1]
    elif plant == "wrong_token":
        ids[0] = r["tok"][0] + 1
    elif plant == "no_remask":         # an uncommitted position not set back to the mask id
        ids[3] = 7
    elif plant == "floor_wrong_one":   # the floor takes a less confident position
        com[:] = False
        com[1] = True
        ids = ids0.copy()
        ids[1] = r["tok"][1]
    elif plant == "floor_too_many":
        com[1] = True
        ids[1] = r["tok"][1]
    elif plant == "commit_decoded":
        com[1] = True
    with pytest.raises(AssertionError):
        _check(ids0, r, ids, com, gamma)


def test_band_admits_either_side_of_gamma():
    """A confidence within the band of gamma may be committed or not."""
    gamma = 0.8
    ids0, r = _oracle_case([0.9, 0.8 + 2e-6, 0.1], gamma)
    _check(ids0, r, r["ids"], r["commit"], gamma)           # oracle: commits position 1
    ids, com = r["ids"].copy(), r["commit"].astype(bool).copy()
    com[1] = False
    ids[1] = MASK
    _check(ids0, r, ids, com, gamma)                         # kernel may leave it masked


def test_predict_noise_and_mock_ar():
    ids0, r = _oracle_case([0.3, 0.5, 0.6, 0.2], 0.8)
    # predict-and-noise with k = 2 most confident: positions 1 and 2
    com = np.array([False, True, True, False])
    ids = ids0.copy()
    ids[com] = r["tok"][com]
    r2 = dict(r, k_min=2)
    check_decision_validity(ids, com, ids0, r["tok"], r["conf"], MASK, 2, 0.8, 2, 1e-5 * r["conf"])
    with pytest.raises(AssertionError):
        bad = np.array([True, False, True, False])
        ids_b = ids0.copy()
        ids_b[bad] = r["tok"][bad]
        check_decision_validity(ids_b, bad, ids0, r["tok"], r["conf"], MASK, 2, 0.8, r2["k_min"],
                                1e-5 * r["conf"])
    # mock-AR: the leftmost masked position only
    left = np.array([True, False, False, False])
    ids_l = ids0.copy()
    ids_l[0] = r["tok"][0]
    check_decision_validity(ids_l, left, ids0, r["tok"], r["conf"], MASK, 1, 0.8, 1, 0.0)
    with pytest.raises(AssertionError):
        wrong = np.array([False, False, True, False])
        ids_w = ids0.copy()
        ids_w[2] = r["tok"][2]
        check_decision_validity(ids_w, wrong, ids0, r["tok"], r["conf"], MASK, 1, 0.8, 1, 0.0)
