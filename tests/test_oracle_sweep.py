"""The oracle against the brute-force proposal over many random tiny configurations
(the generator and the check live with the other pins, in ``oracle_pins.py``)."""
import numpy as np
import pytest

from oracle import dspark_oracle as O
from oracle_pins import check_sweep_case, sweep_case


@pytest.mark.parametrize("seed", range(120))
def test_oracle_matches_brute_force(seed):
    check_sweep_case(seed)


def test_sweep_reaches_ties_and_threshold_equality():
    # the sweep is only worth its name if ties and conf == conf_min actually occur in it
    ties = equal = 0
    for seed in range(120):
        c = sweep_case(seed)
        ifp = 0 if c["sfa"] else 1
        N = c["L_in"] - ifp
        z = O.base_logits(c["hidden"], c["W"], c["bias"], ifp, N)
        for row in z.reshape(-1, c["V"]):
            ties += int(np.sum(row == row.max()) > 1)
        conf = O.confidence(c["hidden"], c["w_conf"], c["b_conf"], ifp, N)
        equal += int(np.any(conf == c["conf_min"]))
    assert ties >= 10 and equal >= 3, (ties, equal)
