"""The packed-sequence piece plan's rule (tests/plan_rule.py, the restatement the GPU tests read
the device's plan against) pinned on hand-worked batches and on invariants of any plan.

Lengths are in tokens, 64 to a chunk; H heads on 152 SMs give cap = 152 // H entries of H chains
per phase and e_max = 256 // H pieces past the first ones."""
import numpy as np

from plan_rule import expected_plan


def test_pages_lengths_are_not_cut():
    # 29, 24, 32, 19 and 13 chunks at H = 16 (cap 9): X = 8 and 9 need 11 entries per phase;
    # X = 10 fits (3, 3, 4, 2, 2 pieces: 9 entries, 18 in the two phases) but takes
    # 2 * 10 + 2 + 14 = 36 chunk times against the 32 of the longest sequence run whole
    counts, k = expected_plan((1800, 1500, 2000, 1200, 800), 16, 152)
    assert counts == [5, 0, 0, 32, 0] and k == [1] * 5


def test_long_sequence_batch():
    # 256, 128, 64, ... 2 chunks at H = 16: X = 64 cuts the first into 4 pieces and the second
    # into 2 (A = 4 entries per phase, U = 6 whole, 5 of them fit the first phase beside 4
    # entries), 2 * 64 + 2 + 14 = 144 < 256; every X from 57 to 63 makes 5, 3 and 2 pieces
    # (A = 7, 2A + U = 19 > 18) and a longer X costs more
    lens = (16384, 8192, 4096, 2048, 1024, 512, 256, 128)
    counts, k = expected_plan(lens, 16, 152)
    assert k == [4, 2, 1, 1, 1, 1, 1, 1]
    assert counts == [8, 2, 4 + 1, 64, 1]   # 2 summaries, 4 pieces + 1 whole, X, 1 scan job


def test_one_long_sequence_among_short_ones():
    # 64, 2, 5, 1 chunks at H = 4 (cap 38): X = 8 gives 8 pieces (A = 7), time 16 + 6 + 14 = 36;
    # X = 9 still 8 pieces, 38
    counts, k = expected_plan((4096, 100, 300, 64), 4, 152)
    assert k == [8, 1, 1, 1] and counts == [4, 6, 7, 8, 1]


def test_whole_sequences_move_to_the_second_phase():
    # 79, 19, 18, 16, 15, 13, 11, 0 chunks at H = 16 (cap 9): X = 16 gives 5, 2, 2 pieces
    # (A = 6, U = 5): 3 whole sequences fit the first phase, 2 move to the second (6 + 2
    # entries); time 32 + 3 + 14 = 49 < 79
    counts, k = expected_plan((5000, 1200, 1100, 1000, 900, 800, 700, 0), 16, 152)
    assert k == [5, 2, 2, 1, 1, 1, 1, 1] and counts == [8, 3, 8, 16, 1]


def test_no_plan_without_one_wave_or_length():
    # more chains than SMs (20 sequences x 16 heads), or a longest sequence under 16 chunks
    counts, k = expected_plan([8192] + [64] * 19, 16, 152)
    assert counts == [20, 0, 0, 128, 0] and k == [1] * 20
    counts, k = expected_plan((960, 100), 2, 152)
    assert counts == [2, 0, 0, 15, 0]


def test_invariants_of_any_plan():
    # on seeded random batches: a cut keeps both phases within cap entries and the pieces
    # within e_max, beats the longest sequence run whole, and its counts agree with its pieces
    rng = np.random.default_rng(0x6D6E0100)
    for trial in range(300):
        H = int(rng.choice([1, 2, 4, 8, 16, 32]))
        cap, e_max = 152 // H, max(1, 256 // H)
        nseq = int(rng.integers(1, min(cap, 12) + 1))
        lens = [int(x) for x in rng.integers(0, 40000, size=nseq)]
        counts, k = expected_plan(lens, H, 152)
        n = [(ln + 63) // 64 for ln in lens]
        assert counts[0] == nseq and len(k) == nseq
        A, U = sum(x - 1 for x in k), sum(x == 1 for x in k)
        if counts[2] == 0:   # nothing cut
            assert k == [1] * nseq and counts[3] == max(n)
            continue
        X = counts[3]
        assert k == [max(1, -(-m // X)) for m in n]
        assert A <= cap and 2 * A + U <= 2 * cap and A <= e_max
        assert counts[1] == sum(max(0, x - 2) for x in k)
        assert counts[4] == sum(x >= 3 for x in k)
        assert counts[2] == A + max(0, U - (cap - A)) <= cap   # the second phase, one wave
        assert A + min(U, cap - A) <= cap                       # the first phase, one wave
        assert 2 * X + max(0, max(k) - 2) + 14 < max(n)
