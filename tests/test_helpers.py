"""CPU checks of the GPU tests' own helpers."""
import numpy as np

from tests.helpers import near_tie_tokens


def test_near_tie_tokens_flags_ties_that_decide_set_or_order():
    R = 2
    l = np.array([[10.0, 5.0, 1.0, 0.0],            # clear: gaps 5 and 4
                  [10.0, 5.0, 5.0 - 1e-4, 0.0],     # the 2nd / 3rd pair: which experts
                  [10.0, 10.0 - 1e-4, 5.0, 0.0],    # the 1st / 2nd pair: slot order
                  [10.0, 5.0, 1.0, 1.0 - 1e-4]])    # a tie below the selection: irrelevant
    assert near_tie_tokens(l, R).tolist() == [False, True, True, False]
    # R = E: only the order of all experts can flip
    assert near_tie_tokens(l[:, :2], 2).tolist() == [False, False, True, False]
