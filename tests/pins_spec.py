"""Checks that pin the speculative-verification oracle to facts fixed outside it.

The rule (lecture notes "Decoding: Sampling, Beam Search and Speculative
Decoding", section 5.2, after Leviathan et al. 2023 and Chen et al. 2023):
accept the draft token x with probability min(1, p(x)/q(x)); at the first
rejection draw from norm(max(0, p - q)) and stop; after G acceptances draw one
more token from the target at position G.  The notes prove that the output
token is then distributed exactly as p, and that the acceptance rate is
sum(min(p, q)) = 1 - TV(p, q).  Those two facts are what the main check here
evaluates exactly, by integrating the oracle's decisions over every uniform on
the 2^-24 grid it uses; the others are special cases with a known answer and
Philox frequencies.

Each check takes an oracle library handle ``L`` and raises AssertionError when
the oracle disagrees.
"""
import numpy as np

import oracle

GRID = 1 << 24


def _dist(rng, V, support):
    w = np.zeros(V)
    ids = rng.choice(V, size=support, replace=False)
    w[ids] = rng.gamma(0.7, size=support) + 1e-3
    return (w / w.sum()).astype(np.float32)


def _first_k(pred, lo=0, hi=GRID):
    """Smallest k in [lo, hi] with pred(k) true, for pred monotone false -> true
    (hi when none in [lo, hi) is)."""
    while lo < hi:
        mid = (lo + hi) // 2
        if pred(mid):
            hi = mid
        else:
            lo = mid + 1
    return lo


def _exact_first_token_law(p, q, L):
    """Exact law of the first output token for G = 1, over the oracle's own
    uniform grid: P(accept d) is counted by bisection on u_acc (the decision
    is monotone in u), the residual draw's law by bisection on u_res (the
    inverse CDF is nondecreasing in u).  Returns (law, acceptance rate)."""
    V = p.shape[1]
    law = np.zeros(V)
    alpha = 0.0
    res_law = None
    for d in range(V):
        if q[0, d] <= 0:
            continue

        def rejects(k, d=d):
            r = oracle.spec_verify_u(p, q, [d], [k / GRID], [0.0, 0.0], L=L)
            assert r["status"] == 0, r
            return r["n_accepted"] == 0

        k_rej = _first_k(rejects)
        acc = k_rej / GRID
        law[d] += q[0, d] * acc
        alpha += q[0, d] * acc
        if acc < 1.0:
            if res_law is None:
                res_law = np.zeros(V)

                def tok(k, d=d):
                    r = oracle.spec_verify_u(p, q, [d], [(GRID - 1) / GRID], [k / GRID, 0.0],
                                             L=L)
                    assert r["status"] == 0 and r["n_accepted"] == 0, r
                    return int(r["tokens"][0])

                prev = 0
                for x in range(V):
                    nxt = _first_k(lambda k: tok(k) > x, lo=prev)
                    res_law[x] = (nxt - prev) / GRID
                    prev = nxt
                assert prev == GRID
            law += q[0, d] * (1.0 - acc) * res_law
    return law, alpha


def check_spec_output_law(L=None):
    """The output token is distributed exactly as the target p, and the
    acceptance rate is sum(min(p, q)) = 1 - TV(p, q) (notes, section 5.2)."""
    rng = np.random.Generator(np.random.PCG64(21))
    cases = []
    for _ in range(5):
        V = 7
        cases.append((_dist(rng, V, 5), _dist(rng, V, 5)))
    # draft much wider than the target, and the reverse
    cases.append((_dist(rng, 6, 2), _dist(rng, 6, 6)))
    cases.append((_dist(rng, 6, 6), _dist(rng, 6, 2)))
    for pt, qd in cases:
        p = np.stack([pt, pt])  # row G = 1 (the bonus row) is unused when G = 1 rejects
        q = qd[None, :]
        law, alpha = _exact_first_token_law(p, q, L)
        pd, qdd = pt.astype(np.float64), qd.astype(np.float64)
        assert np.max(np.abs(law - pd)) < 2e-6, (law, pd)
        assert abs(alpha - np.minimum(pd, qdd).sum()) < 2e-6, (alpha, np.minimum(pd, qdd).sum())
        tv = 0.5 * np.abs(pd - qdd).sum()
        assert abs(alpha - (1.0 - tv)) < 2e-6


def _inverse_cdf(w, u):
    """Brute-force interval lookup in id order: the id whose interval
    [C(x-1), C(x)) of the cumulative weights contains u * sum(w)."""
    c = np.cumsum(np.asarray(w, dtype=np.float64))
    return int(np.searchsorted(c, u * c[-1], side="right"))


def check_spec_special_cases(L=None):
    """Cases whose outcome is fixed by the rule without any arithmetic doubt."""
    rng = np.random.Generator(np.random.PCG64(22))
    V, G = 9, 3
    ps = [_dist(rng, V, 6) for _ in range(G + 1)]
    d = [int(np.argmax(ps[i])) for i in range(G)]
    # q == p at every position: every draft is accepted (u < 1 = p/q), and the
    # bonus token is the inverse CDF of p_G at the last position's u_res.
    for u_last in (0.0, 0.3, 0.77, 1 - 2.0 ** -24):
        r = oracle.spec_verify_u(np.stack(ps), np.stack(ps[:G]), d, [1 - 2.0 ** -24] * G,
                                 [0.9, 0.1, 0.5, u_last], L=L)
        assert r["status"] == 0 and r["n_accepted"] == G
        assert list(r["tokens"][:G]) == d
        assert r["tokens"][G] == _inverse_cdf(ps[G], u_last), (r, u_last)
    # position 1's target has no mass at the draft token: the draft at 0 is
    # accepted (q0 = p0), the one at 1 is rejected whatever u is, and since
    # the draft's support there is disjoint from the target's, the residual
    # is p_1 itself; the draw uses position 1's u_res.
    p1 = np.zeros(V, np.float32)
    p1[:4] = [0.125, 0.375, 0.25, 0.25]
    q1 = np.zeros(V, np.float32)
    q1[6:] = [0.5, 0.25, 0.25]
    p = np.stack([ps[0], p1, ps[2], ps[3]])
    q = np.stack([ps[0], q1, ps[2]])
    for u1 in (0.0, 0.1, 0.126, 0.49, 0.5, 0.76, 0.99):
        r = oracle.spec_verify_u(p, q, [d[0], 6, d[2]], [0.5, 0.0, 0.5], [0.9, u1, 0.2, 0.3],
                                 L=L)
        assert r["status"] == 0 and r["n_accepted"] == 1, r
        assert r["tokens"][0] == d[0] and r["tokens"][2] == -1 and r["tokens"][3] == -1
        assert r["tokens"][1] == _inverse_cdf(p1, u1), (u1, r)
    # an exact switch point: u * S equals a cumulative weight (dyadic values),
    # and the draw takes the first id whose cumulative weight EXCEEDS it
    r = oracle.spec_verify_u(p, q, [d[0], 6, d[2]], [0.5, 0.0, 0.5], [0.9, 0.5, 0.2, 0.3], L=L)
    assert r["tokens"][1] == 2 and r["margin"] == 0.0, r
    # two rejections in a row: the first one ends the step
    p0 = np.zeros(V, np.float32)
    p0[:2] = [0.5, 0.5]
    q0 = np.zeros(V, np.float32)
    q0[5] = 1.0
    r = oracle.spec_verify_u(np.stack([p0, p1, ps[2], ps[3]]), np.stack([q0, q1, ps[2]]),
                             [5, 6, d[2]], [0.3, 0.3, 0.3], [0.75, 0.1, 0.2, 0.3], L=L)
    assert r["status"] == 0 and r["n_accepted"] == 0
    assert list(r["tokens"]) == [1, -1, -1, -1], r
    # acceptance is u * q < p: with p = q / 2, u = 0.5 - 2^-24 accepts and
    # u = 0.5 rejects
    qh = np.zeros(V, np.float32)
    qh[:2] = [0.5, 0.5]
    ph = np.zeros(V, np.float32)
    ph[:3] = [0.25, 0.25, 0.5]
    for u, acc in ((0.5 - 2.0 ** -24, 1), (0.5, 0)):
        r = oracle.spec_verify_u(np.stack([ph, ps[1]]), qh[None, :], [0], [u], [0.1, 0.1], L=L)
        assert r["status"] == 0 and r["n_accepted"] == acc, (u, r)
        if not acc:
            assert r["tokens"][0] == 2  # the residual is all at id 2
    # G = 0: one draw from p_0
    for u in (0.0, 0.45, 0.99):
        r = oracle.spec_verify_u(ps[0][None, :], np.zeros((0, V), np.float32), [], [], [u], L=L)
        assert r["status"] == 0 and r["n_accepted"] == 0
        assert r["tokens"][0] == _inverse_cdf(ps[0], u)


def check_spec_status(L=None):
    """Statuses: a draft token outside [0, V) or a read probability outside
    [0, 1] (or NaN) is invalid; a rejection whose residual has no mass is
    empty; outputs of such a sequence are all -1."""
    V = 6
    p = np.full((2, V), 1.0 / V, np.float32)
    q = np.full((1, V), 1.0 / V, np.float32)
    assert oracle.spec_verify_u(p, q, [V], [0.5], [0.5, 0.5], L=L)["status"] == 3
    assert oracle.spec_verify_u(p, q, [-1], [0.5], [0.5, 0.5], L=L)["status"] == 3
    assert oracle.spec_verify_u(p, q, [V - 1], [0.5], [0.5, 0.5], L=L)["status"] == 0
    pb = p.copy()
    pb[1, 3] = np.nan  # in the drawn bonus row
    r = oracle.spec_verify_u(pb, q, [0], [0.5], [0.5, 0.5], L=L)
    assert r["status"] == 3 and list(r["tokens"]) == [-1, -1] and r["n_accepted"] == 0
    pb = p.copy()
    pb[1, 0] = 1.5
    assert oracle.spec_verify_u(pb, q, [0], [0.5], [0.5, 0.5], L=L)["status"] == 3
    qb = q.copy()
    qb[0, 2] = -0.25  # the draft token's own probability
    assert oracle.spec_verify_u(p, qb, [2], [0.5], [0.5, 0.5], L=L)["status"] == 3
    # p_0 <= q_0 everywhere, rejection at d: no residual mass
    pe = np.stack([np.full(V, 0.5 / V, np.float32), p[1]])
    r = oracle.spec_verify_u(pe, q, [1], [0.9], [0.5, 0.5], L=L)
    assert r["status"] == 1 and list(r["tokens"]) == [-1, -1], r
    # the same inputs accepted (u small): the bonus row decides
    r = oracle.spec_verify_u(pe, q, [1], [0.1], [0.5, 0.5], L=L)
    assert r["status"] == 0 and r["n_accepted"] == 1


def check_spec_philox_frequencies(L=None, n=60000):
    """With Philox uniforms over consecutive offsets, the first output token
    follows p and the acceptance rate is sum(min(p, q)) within binomial noise;
    the residual draw uses a word of the block independent of the acceptance
    test's."""
    p0 = np.array([0.05, 0.30, 0.05, 0.35, 0.25], np.float32)
    q0 = np.array([0.40, 0.05, 0.35, 0.10, 0.10], np.float32)
    p = np.broadcast_to(np.stack([p0, p0])[None], (n, 2, 5)).copy()
    q = np.broadcast_to(q0[None, None, :], (n, 1, 5)).copy()
    rng = np.random.Generator(np.random.PCG64(23))
    d = rng.choice(5, size=(n, 1), p=q0.astype(np.float64) / q0.sum()).astype(np.int32)
    r = oracle.spec_verify(p, q, d, np.full(n, 7, np.uint64),
                           np.arange(n, dtype=np.uint64) * 2, L=L)
    assert np.all(r["status"] == 0)
    pd = p0.astype(np.float64)
    freq = np.bincount(r["tokens"][:, 0], minlength=5) / n
    sd = np.sqrt(pd * (1 - pd) / n)
    assert np.all(np.abs(freq - pd) <= 5 * sd), (freq, pd)
    alpha = np.minimum(pd, q0.astype(np.float64)).sum()
    acc = r["n_accepted"].mean()
    assert abs(acc - alpha) <= 5 * np.sqrt(alpha * (1 - alpha) / n), (acc, alpha)


def check_spec_fx_agrees(L=None, n=300):
    """The labelled fixed-point variant takes the same decisions as the rule
    over the reals wherever u * S lies more than 1e-6 of S from a switch point
    (its weights are floor(w * 2^42) of binary32 differences: together they
    move a prefix by far less than that), and nearly every draw is that far."""
    rng = np.random.Generator(np.random.PCG64(29))
    far = 0
    for t in range(n):
        V = int(rng.choice([5, 60, 700, 5000]))
        G = int(rng.integers(0, 4))
        p = np.stack([_dist(rng, V, int(rng.integers(1, V + 1))) for _ in range(G + 1)])
        q = np.stack([_dist(rng, V, int(rng.integers(1, V + 1))) for _ in range(G)]) if G else None
        d = [int(rng.choice(V, p=q[i].astype(np.float64) / q[i].sum())) for i in range(G)]
        ua = rng.integers(0, GRID, size=G) / GRID
        ur = rng.integers(0, GRID, size=G + 1) / GRID
        qq = q if G else np.zeros((0, V), np.float32)
        r = oracle.spec_verify_u(p, qq, d, ua, ur, L=L)
        f = oracle.spec_verify_u(p, qq, d, ua, ur, L=L, fixed=True)
        assert r["status"] == f["status"] and r["n_accepted"] == f["n_accepted"], (t, r, f)
        if r["status"] == 0 and r["margin"] > 1e-6:
            far += 1
            assert list(r["tokens"]) == list(f["tokens"]), (t, r, f)
    assert far >= 0.95 * n, far


SPEC_CHECKS = [check_spec_special_cases, check_spec_status, check_spec_output_law,
               check_spec_philox_frequencies, check_spec_fx_agrees]
