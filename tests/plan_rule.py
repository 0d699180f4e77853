"""The packed-sequence piece plan restated from its rule, for the tests: the library makes the
plan on the device (gdn_varlen.cu, in the block that checks cu_seqlens) and writes it into the
workspace, where tests/test_gpu_varlen.py reads it back; tests/test_plan_rule.py pins this
restatement on hand-worked batches. Test infrastructure only."""


def expected_plan(lens, H, sms):
    """The piece plan restated from its rule (the library makes it on the device, in the
    length-check block): piece lengths X = 8 chunks, then each an eighth longer, below the
    longest sequence; both phases in one wave of sms // H entries of H chains (A = the pieces
    past the first ones, one entry per phase each; U = the sequences left whole, one entry in
    either phase), A at most 256 // H; time 2 X + the most scan steps + 14 chunk times, the
    smallest (then the shortest X) taken when it beats the longest sequence run whole.
    Returns the counts (entries of the first phase, summaries, second-phase entries, X, scan
    jobs) and each sequence's piece count."""
    n = [(ln + 63) // 64 for ln in lens]
    cap, e_max, maxn = sms // H, max(1, 256 // H), max(n)

    def pieces(x):
        return [max(1, -(-m // x)) for m in n]

    best = (maxn, maxn)
    if len(n) <= cap and len(n) <= 256 and maxn >= 16:
        x = 8
        while x < maxn:
            k = pieces(x)
            A, U = sum(kk - 1 for kk in k), sum(kk == 1 for kk in k)
            cost = 2 * x + max(0, max(kk - 2 for kk in k)) + 14
            if A <= cap and 2 * A + U <= 2 * cap and A <= e_max and (cost, x) < best:
                best = (cost, x)
            x += max(1, x // 8)
    X = best[1]
    if X >= maxn:
        return [len(n), 0, 0, maxn, 0], [1] * len(n)
    k = pieces(X)
    A, U = sum(kk - 1 for kk in k), sum(kk == 1 for kk in k)
    room1 = cap - A
    return [len(n), sum(max(0, kk - 2) for kk in k), A + max(0, U - room1), X,
            sum(kk >= 3 for kk in k)], k
