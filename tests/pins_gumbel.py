"""Checks that pin the Gumbel-max oracle.

The lecture notes (section 3.2) state the identity behind it: the argmax of
z_i + g_i, with g_i = -log(-log(u_i)) independent Gumbel noise, is a draw
from softmax(z).  The frequency check compares many draws with the exact
softmax of the kept set, computed here from the logits; the others check
greedy rows, statuses and the uniform's range.  Each check takes an oracle
library handle ``L``.
"""
import numpy as np

import oracle


def check_gumbel_frequencies(L=None, n=200000):
    x = np.array([[2.0, 0.5, 1.5, -1.0, 1.0, 0.0, 3.0]], dtype=np.float32)
    V = x.shape[1]
    kept = np.array([[0b0010111]], dtype=np.uint32)  # ids 0, 1, 2 and 4
    t = np.float32(0.8)
    xs = np.repeat(x, n, axis=0)
    r = oracle.gumbel_sample(xs, "f32", V, np.full(n, t, np.float32), np.full(n, 3, np.uint64),
                             np.arange(n, dtype=np.uint64), kept_mask=np.repeat(kept, n, axis=0),
                             L=L)
    assert np.all(r["status"] == 0)
    z = (x[0] / t).astype(np.float64)
    ids = [0, 1, 2, 4]
    p = np.zeros(V)
    p[ids] = np.exp(z[ids] - z[ids].max())
    p /= p.sum()
    freq = np.bincount(r["token"], minlength=V) / n
    sd = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(freq - p) <= 5 * sd + 1e-12), (freq, p)


def check_gumbel_greedy_and_status(L=None):
    x = np.array([[1.0, 3.0, 3.0, -np.inf, 2.0],
                  [np.nan, 1.0, 2.0, 0.0, 0.5],
                  [-np.inf] * 5,
                  [1.0, 2.0, 3.0, 4.0, 5.0],
                  [1.0, np.inf, 0.0, 0.0, 0.0]], dtype=np.float32)
    B, V = x.shape
    kept = np.array([[0b11111], [0b11110], [0b11111], [0b00111], [0b11101]], dtype=np.uint32)
    seed = np.zeros(B, np.uint64)
    off = np.arange(B, dtype=np.uint64)
    r = oracle.gumbel_sample(x, "f32", V, np.zeros(B, np.float32), seed, off, kept_mask=kept, L=L)
    # greedy: first maximum; a NaN outside the kept set is ignored; no
    # candidate; the mask limits the argmax; +inf outside the kept set
    assert list(r["status"]) == [0, 0, 1, 0, 0], r
    assert list(r["token"]) == [1, 2, -1, 2, 0], r
    r = oracle.gumbel_sample(x, "f32", V, np.full(B, 1.0, np.float32), seed, off, L=L)
    assert list(r["status"][[1, 2, 4]]) == [oracle.ORC_NONFINITE, oracle.ORC_EMPTY,
                                            oracle.ORC_NONFINITE]
    r = oracle.gumbel_sample(x[:1], "f32", V, np.array([-1.0], np.float32), seed[:1], off[:1],
                             L=L)
    assert r["status"][0] == oracle.ORC_INVALID and r["token"][0] == -1


def check_gumbel_uniforms(L=None, n=40000):
    u = np.array([oracle.gumbel_uniform(9, 77, i, L=L) for i in range(n)])
    assert u.min() > 0.0 and u.max() < 1.0
    # the four words of a block are used in turn: no repeats inside a block
    assert np.all(np.diff(u.reshape(-1, 4), axis=1) != 0)
    hist = np.bincount(np.minimum((u * 20).astype(int), 19), minlength=20)
    chi2 = ((hist - n / 20) ** 2 / (n / 20)).sum()
    assert chi2 < 60.0, chi2  # 19 degrees of freedom


GUMBEL_CHECKS = [check_gumbel_greedy_and_status, check_gumbel_uniforms, check_gumbel_frequencies]


def check_top_logprobs(L=None):
    """Top logprobs of a worked row: p = (0.5, 0.2, 0.2, 0.1) at logits ln p
    (T = 1, top-k 3, top-p 1): the kept set is the first three, renormalised
    to (5/9, 2/9, 2/9); ranked by logit with the smaller id first among the
    tied pair; a fourth slot is empty.  Over a whole kept set the
    probabilities sum to one."""
    p = np.array([0.5, 0.2, 0.2, 0.1])
    x = np.log(p).astype(np.float32)[None]
    r = oracle.run_batch(x, "f32", 4, temperature=[1.0], top_k=[3], top_p=[1.0],
                         want_probs=True, L=L)
    kept = r["probs"] > 0
    ids, lps = oracle.top_logprobs(x, kept, r["probs"], r["status"], 4)
    assert list(ids[0]) == [0, 1, 2, -1], ids
    want = np.log(np.array([5 / 9, 2 / 9, 2 / 9]))
    assert np.allclose(lps[0, :3], want, rtol=0, atol=1e-6) and lps[0, 3] == -np.inf, lps
    rng = np.random.Generator(np.random.PCG64(33))
    xs = (rng.standard_normal((3, 50)) * 2).astype(np.float32)
    r = oracle.run_batch(xs, "f32", 50, temperature=[0.7] * 3, top_k=[10, 50, 30],
                         top_p=[0.9, 0.8, 1.0], want_probs=True, L=L)
    kept = r["probs"] > 0
    ids, lps = oracle.top_logprobs(xs, kept, r["probs"], r["status"], 32)
    for b in range(3):
        m = ids[b] >= 0
        assert m.sum() == min(32, kept[b].sum())
        if kept[b].sum() <= 32:
            assert abs(np.exp(lps[b, m]).sum() - 1.0) < 1e-9
        assert np.all(np.diff(xs[b, ids[b, m]]) <= 0)


GUMBEL_CHECKS.append(check_top_logprobs)
