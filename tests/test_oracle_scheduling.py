"""Pins of the oracle's scheduling rules on hand-worked sequences.

"33. Removing overhead", §Async scheduling (placeholder ids replaced on the device by the previous step's
sampled ids) and "19. Fast decode", §Host synchronizations (stop ids checked every check_every steps, the
output cut after each request's first stop id).
"""
import numpy as np
import pytest

import oracle


def test_gather_reads_the_previous_steps_row_or_the_host_id():
    # step N sampled [50, 51, 52] for its rows 0..2; step N+1 packs a 2-token prompt chunk (host ids 7, 8)
    # then three decode rows: its row of request 0 -> previous row 0, request 1's id already known (99),
    # request 2 -> previous row 2
    got = oracle.gather_input_ids([7, 8, -1, 99, -1], [-1, -1, 0, -1, 2], [50, 51, 52])
    np.testing.assert_array_equal(got, [7, 8, 50, 99, 52])
    # rows may be permuted and repeated
    np.testing.assert_array_equal(oracle.gather_input_ids([0, 0, 0], [2, 0, 2], [5, 6, 7]), [7, 5, 7])
    # nothing gathered: the host's ids
    np.testing.assert_array_equal(oracle.gather_input_ids([3, 4], [-1, -1], []), [3, 4])
    with pytest.raises(ValueError):
        oracle.gather_input_ids([0], [1], [5])          # row 1 of a 1-row previous step
    with pytest.raises(ValueError):
        oracle.gather_input_ids([0], [-2], [5])


def test_stop_trim_hand_worked():
    toks = np.array([[10, 11, 2, 13, 14, 15, 16, 17],
                     [20, 21, 22, 23, 24, 3, 26, 27],
                     [30, 31, 32, 33, 34, 35, 36, 37]])
    # stop ids {2, 3}: request 0 stops at step 3, request 1 at step 6, request 2 never -> all 8 steps run
    out, lens, n = oracle.stop_trim(toks, [2, 3], check_every=4)
    assert n == 8
    np.testing.assert_array_equal(lens, [3, 6, 8])
    np.testing.assert_array_equal(out[0], [10, 11, 2, -1, -1, -1, -1, -1])
    np.testing.assert_array_equal(out[1], [20, 21, 22, 23, 24, 3, -1, -1])
    np.testing.assert_array_equal(out[2], toks[2])
    # with 37 also a stop id, request 2 stops at step 8; every request has stopped only at the check after
    # step 8
    out, lens, n = oracle.stop_trim(toks, [2, 3, 37], check_every=4)
    assert n == 8 and list(lens) == [3, 6, 8]
    # with 32 a stop id the last request stops at step 3: the checks come after steps 4 and 8, so the loop
    # ends after step 8 (request 1 stops at step 6); with checks every 2 steps it ends after step 6
    _, lens, n = oracle.stop_trim(toks, [2, 3, 32], check_every=4)
    assert n == 8 and list(lens) == [3, 6, 3]
    _, lens, n = oracle.stop_trim(toks, [2, 3, 32], check_every=2)
    assert n == 6 and list(lens) == [3, 6, 3]
    # checks every step end the loop at the last first-stop
    assert oracle.stop_trim(toks, [2, 3, 32], check_every=1)[2] == 6
    # a stop id found only after max_steps does not count
    out, lens, n = oracle.stop_trim(toks, [3], check_every=3, max_steps=5)
    assert n == 5 and list(lens) == [5, 5, 5]
    assert (out[:, 5:] == -1).all() and out.shape == (3, 5)
    # the last group is cut at max_steps
    assert oracle.stop_trim(toks[:1], [17], check_every=3, max_steps=7)[2] == 7
    # no stop ids: every step runs
    _, lens, n = oracle.stop_trim(toks, [], check_every=3)
    assert n == 8 and (lens == 8).all()


def test_stop_trim_single_request_equals_first_stop_rounded_up_to_a_check():
    rng = np.random.default_rng(3)
    for _ in range(200):
        n, every = int(rng.integers(1, 30)), int(rng.integers(1, 9))
        t = rng.integers(0, 6, size=(1, n))
        out, lens, steps = oracle.stop_trim(t, [0], check_every=every)
        hits = np.flatnonzero(t[0] == 0)
        if hits.size == 0:
            assert steps == n and lens[0] == n
        else:
            f = int(hits[0]) + 1
            assert lens[0] == f and steps == min(n, -(-f // every) * every)
            assert out[0, f - 1] == 0 and (out[0, f:] == -1).all()
