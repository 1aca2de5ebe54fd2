"""The greedy-choice comparison the GPU parity tests use: a unique oracle
choice must be matched, a near-tie may take any token within the bound."""
import numpy as np

from tests.gpu_util import greedy_choice_check


def test_unique_positions_must_match_and_ties_stay_within_the_bound():
    ref = np.array([[0.0, 1.0, 0.5],      # unique: argmax 1 (gap 0.5)
                    [0.0, 1.0, 0.99],     # near-tie between 1 and 2
                    [2.0, 0.0, 1.0]])     # unique: argmax 0
    assert greedy_choice_check(ref, [1, 2, 0]) == (2, 2, 1, 0)
    assert greedy_choice_check(ref, [1, 1, 2]) == (1, 2, 1, 0)      # a unique position missed
    assert greedy_choice_check(ref, [1, 0, 0]) == (2, 2, 1, 1)      # a near-tie answered outside the bound
    assert greedy_choice_check(ref, [1, 2, 0], tol=1e-3) == (2, 3, 0, 0)   # a tighter bound: no tie left
