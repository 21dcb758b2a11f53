"""Checks that pin the CPU oracle to facts fixed outside it.

Each check takes an oracle library handle ``L`` (``oracle.lib()`` or a mutant
built by the mutation test) and raises AssertionError when the oracle disagrees
with the pages' worked examples, exact rationals, library routines (numpy,
torch, cuRAND) or brute force from definitions written here independently of
the oracle's code.
"""
import ctypes
import math
import os
from fractions import Fraction

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "worked_examples.txt")


# --------------------------------------------------------------------------
# Golden worked examples
# --------------------------------------------------------------------------

def load_golden():
    cases, cur = [], None
    with open(GOLDEN) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            key, val = key.strip(), val.strip()
            if key == "case":
                cur = {"name": val, "temperature": Fraction(1), "mask": None,
                       "exact_boundary": 0}
                cases.append(cur)
            elif key in ("probs", "expect_probs"):
                cur[key] = [Fraction(v) for v in val.split()]
            elif key in ("expect_kept", "mask"):
                cur[key] = [int(v) for v in val.split()]
            elif key in ("top_p", "temperature"):
                cur[key] = Fraction(val)
            else:
                cur[key] = int(val)
    return cases


def exact_contract(probs, temperature, top_k, top_p, mask):
    """The contract on exact rationals (test-side restatement, no sorting
    helpers shared with the oracle): temperature as p^(1/T) for T = 1/n,
    mask, top-k, renormalise, top-p with '>=', renormalise."""
    n = len(probs)
    inv_t = 1 / temperature
    assert inv_t.denominator == 1, "exact path supports T = 1/integer only"
    w = [p ** int(inv_t) for p in probs]
    legal = [mask is None or i in mask for i in range(n)]
    w = [w[i] if legal[i] else Fraction(0) for i in range(n)]
    ids = [i for i in range(n) if legal[i]]
    ids.sort(key=lambda i: (-w[i], i))
    k = min(top_k, len(ids))
    sk = ids[:k]
    mk = sum(w[i] for i in sk)
    q = {i: w[i] / mk for i in sk}
    sp, cum = [], Fraction(0)
    for i in sk:
        sp.append(i)
        cum += q[i]
        if cum >= top_p:
            break
    mp = sum(q[i] for i in sp)
    return sorted(sp), {i: q[i] / mp for i in sp}


def check_worked_examples(L=None):
    for c in load_golden():
        kept_x, prob_x = exact_contract(c["probs"], c["temperature"], c["top_k"], c["top_p"],
                                        c["mask"])
        # The page's printed answer follows from the contract on exact rationals.
        assert kept_x == c["expect_kept"], (c["name"], kept_x)
        assert [prob_x[i] for i in kept_x] == c["expect_probs"], c["name"]
        n = len(c["probs"])
        x = np.log(np.array([float(p) for p in c["probs"]]))
        z = x / float(c["temperature"])
        legal = np.array([c["mask"] is None or i in c["mask"] for i in range(n)], dtype=np.uint8)
        r = oracle.select_core(x, z, legal, c["top_k"], float(c["top_p"]), 0.5, L=L)
        assert r["status"] == oracle.ORC_OK, c["name"]
        if c["exact_boundary"]:
            # fp cannot settle mass == p: the oracle must flag the row and keep
            # either the page's prefix or one more.
            assert r["flags"] & oracle.FLAG_TOPP_BOUNDARY, c["name"]
            got = list(np.nonzero(r["kept"])[0])
            assert got[:len(kept_x)] == kept_x and len(got) - len(kept_x) in (0, 1), c["name"]
            continue
        assert list(np.nonzero(r["kept"])[0]) == kept_x, (c["name"], r["kept"])
        for i in kept_x:
            assert abs(r["prob"][i] - float(prob_x[i])) < 1e-12, (c["name"], i, r["prob"][i])
        assert abs(r["prob"].sum() - 1.0) < 1e-12


def check_dyadic_boundary(L=None):
    """Exact top-p boundary where double arithmetic is exact: probabilities
    (1/2, 1/4, 1/8, 1/32, 1/32, 1/32, 1/32) and p = 7/8.  The cumulative mass
    of the first three is exactly 7/8: '>=' keeps three, '>' would keep four."""
    libm = ctypes.CDLL("libm.so.6")
    libm.exp.restype = ctypes.c_double
    libm.exp.argtypes = [ctypes.c_double]
    k = [0, 1, 2, 4, 4, 4, 4]
    x = np.array([math.log(2.0 ** -j) for j in k])
    # precondition: the C library's exp returns the dyadic weights exactly
    assert all(libm.exp(float(v)) == 2.0 ** -j for v, j in zip(x, k))
    r = oracle.select_core(x, x, np.ones(7, np.uint8), 7, 0.875, 0.1, L=L)
    assert list(np.nonzero(r["kept"])[0]) == [0, 1, 2], r["kept"]
    assert r["prob"][0] == 4 / 7 and r["prob"][1] == 2 / 7 and r["prob"][2] == 1 / 7


def check_order_negative_controls():
    """The KB note's section 03 contrasts: the other orders give other sets."""
    pr = [Fraction(2, 5), Fraction(3, 10), Fraction(1, 5), Fraction(1, 10)]
    # top-p on the full distribution first, then top-k = 2: keeps {A, B}
    cum, sp = Fraction(0), []
    for i in range(4):
        sp.append(i)
        cum += pr[i]
        if cum >= Fraction(1, 2):
            break
    assert sorted(set(sp) & {0, 1}) == [0, 1]
    # top-k = 2 before a C/D-only constraint: empty
    assert set([0, 1]) & {2, 3} == set()


# --------------------------------------------------------------------------
# Front end: greedy ties, masks, status codes
# --------------------------------------------------------------------------

def _bits_f32(rows):
    return np.ascontiguousarray(np.array(rows, dtype=np.float32))


def check_greedy_tie(L=None):
    """Lecture 9 answer 1: greedy picks the earlier vocabulary id on a tie."""
    x = _bits_f32([[0.1, 0.4, 0.4, 0.1, -1.0]])
    r = oracle.run_batch(x, "f32", 5, temperature=[0.0], top_k=[5], top_p=[1.0], L=L)
    assert r["status"][0] == 0 and r["token"][0] == 1 and r["kept_count"][0] == 1
    assert r["kept_mask"][0, 0] == (1 << 1)
    r = oracle.run_batch(x, "f32", 5, mode="argmax", L=L)
    assert r["token"][0] == 1


def check_mask_bit_order(L=None):
    """Bit j%32 of word j/32 allows token j.  Only tokens 33 and 40 allowed."""
    V = 48
    x = _bits_f32([np.arange(V, dtype=np.float32)[::-1]])  # token 0 is the largest
    mask = np.zeros((1, 2), dtype=np.uint32)
    mask[0, 1] = (1 << 1) | (1 << 8)
    r = oracle.run_batch(x, "f32", V, temperature=[0.0], bitmask=mask, L=L)
    assert r["status"][0] == 0 and r["token"][0] == 33, r["token"]
    r = oracle.run_batch(x, "f32", V, temperature=[1.0], top_k=[V], top_p=[1.0],
                         bitmask=mask, L=L)
    assert r["kept_count"][0] == 2 and r["kept_mask"][0, 1] == mask[0, 1]
    assert r["kept_mask"][0, 0] == 0


def check_status_codes(L=None):
    V = 8
    base = np.linspace(-1, 1, V, dtype=np.float32)
    rows = np.stack([base] * 8)
    rows[1, 3] = np.nan                       # NaN in a legal slot
    rows[2, :] = -np.inf                      # everything -inf
    rows[3, 5] = np.inf                       # +inf in a legal slot
    rows[4, 2] = np.nan                       # NaN, but masked out below
    mask = np.full((8, 1), 0xFF, dtype=np.uint32)
    mask[4, 0] = 0xFF & ~(1 << 2)
    mask[5, 0] = 0                            # nothing allowed
    t = [1.0, 1.0, 1.0, 1.0, 1.0, 1.0, -0.5, 1.0]
    k = [3, 3, 3, 3, 3, 3, 3, 0]
    p = [0.9] * 8
    r = oracle.run_batch(rows, "f32", V, temperature=t, top_k=k, top_p=p, bitmask=mask, L=L)
    want = [0, 2, 1, 2, 0, 1, 3, 3]
    assert list(r["status"]) == want, r["status"]
    for i, s in enumerate(want):
        if s:
            assert r["token"][i] == -1 and r["kept_count"][i] == 0
            assert not r["kept_mask"][i].any()
    for bad_p in (0.0, 1.5, float("nan")):
        r = oracle.run_batch(rows[:1], "f32", V, temperature=[1.0], top_k=[2], top_p=[bad_p], L=L)
        assert r["status"][0] == 3


# --------------------------------------------------------------------------
# Decoders and Philox
# --------------------------------------------------------------------------

def check_decoders(L=None):
    L = L or oracle.lib()
    bits = np.arange(65536, dtype=np.uint16)
    ref16 = bits.view(np.float16).astype(np.float32)  # numpy's IEEE binary16 decode
    refbf = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    mine16 = np.array([L.orc_f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    minebf = np.array([L.orc_bf16_to_f32(int(b)) for b in bits], dtype=np.float32)
    for mine, ref in ((mine16, ref16), (minebf, refbf)):
        nan_m, nan_r = np.isnan(mine), np.isnan(ref)
        assert (nan_m == nan_r).all()
        assert (mine[~nan_m].view(np.uint32) == ref[~nan_r].view(np.uint32)).all()


def curand_blocks(seed, n_blocks):
    """First n_blocks Philox4x32-10 blocks of cuRAND's host generator, or None
    when libcurand is not available."""
    for path in ("/usr/local/cuda/lib64/libcurand.so", "libcurand.so", "libcurand.so.10"):
        try:
            cr = ctypes.CDLL(path)
            break
        except OSError:
            cr = None
    if cr is None:
        return None
    gen = ctypes.c_void_p()
    if cr.curandCreateGeneratorHost(ctypes.byref(gen), 161) != 0:  # PHILOX4_32_10
        return None
    try:
        assert cr.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        buf = (ctypes.c_uint * (4 * n_blocks))()
        assert cr.curandGenerate(gen, buf, 4 * n_blocks) == 0
        return np.array(buf[:], dtype=np.uint32).reshape(n_blocks, 4)
    finally:
        cr.curandDestroyGenerator(gen)


def check_philox_vs_curand(L=None):
    """cuRAND's host Philox4x32-10 generator emits block i of seed s as the
    block function at counter (0, 0, i, 0), key (lo32 s, hi32 s)."""
    any_run = False
    for seed in (0, 1, 12345, (1 << 40) + 7, (1 << 64) - 1):
        ref = curand_blocks(seed, 64)
        if ref is None:
            return False
        any_run = True
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for i in range(64):
            got = oracle.philox4x32_10([0, 0, i, 0], key, L=L)
            assert (got == ref[i]).all(), (seed, i)
    return any_run


def check_uniformity(L=None, n=200000):
    """u over consecutive offsets: mean, variance and a 64-bin chi-square."""
    u = np.array([oracle.uniform(9, o, L=L) for o in range(n)])
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 4 * math.sqrt(1 / 12 / n)
    assert abs(u.var() - 1 / 12) < 0.002
    h, _ = np.histogram(u, bins=64, range=(0, 1))
    e = n / 64
    chi2 = ((h - e) ** 2 / e).sum()
    assert chi2 < 63 + 6 * math.sqrt(2 * 63), chi2  # ~6 sigma for 63 dof
    # granularity 2^-24: u * 2^24 is an integer
    assert np.all(np.floor(u * 2**24) == u * 2**24)


# --------------------------------------------------------------------------
# Brute force from definitions (O(V^2) ranks, interval sampling)
# --------------------------------------------------------------------------

def brute_row(x32, legal, t, k, p, u):
    """Contract from definitions, for tiny V.  Returns (status, token, kept
    set, probs dict, boundary) with boundary=True when a top-p or CDF decision
    sits within 1e-9 of its threshold (float-order dependent)."""
    V = len(x32)
    ids = [i for i in range(V) if legal[i]]
    if any(math.isnan(float(x32[i])) or math.isinf(float(x32[i])) for i in ids):
        return 2, -1, set(), {}, False
    if not ids:
        return 1, -1, set(), {}, False
    if t == 0.0:
        mx = max(float(x32[i]) for i in ids)
        tok = min(i for i in ids if float(x32[i]) == mx)
        return 0, tok, {tok}, {tok: 1.0}, False
    z = {i: float(np.float32(x32[i]) / np.float32(t)) for i in ids}
    rank = {i: sum(1 for j in ids if x32[j] > x32[i] or (x32[j] == x32[i] and j < i))
            for i in ids}
    K = min(k, V, len(ids))
    sk = [i for i in ids if rank[i] < K]
    m = max(z[i] for i in ids)
    w = {i: math.exp(z[i] - m) for i in ids}
    mk = math.fsum(w[i] for i in sk)
    q = {i: w[i] / mk for i in sk}
    boundary = False
    if p >= 1.0:
        sp = sk
    else:
        sp = []
        for i in sk:
            above = math.fsum(q[j] for j in sk if rank[j] < rank[i])
            if abs(above - p) < 1e-9:
                boundary = True
            if above < p:
                sp.append(i)
    mp = math.fsum(q[i] for i in sp)
    r = {i: q[i] / mp for i in sp}
    tok, cum = max(sp), 0.0
    acc = []
    for i in sorted(sp):
        acc.append(r[i])
        cum = math.fsum(acc)
        if abs(cum - u) < 1e-9:
            boundary = True
        if cum > u:
            tok = i
            break
    return 0, tok, set(sp), r, boundary


def check_bruteforce(L=None, seeds=range(6), V=12, B=160):
    rng = np.random.Generator(np.random.PCG64(1234))
    for s in seeds:
        x = rng.integers(-2, 2, size=(B, V)).astype(np.float32)   # 4-level grid: ties
        x[rng.random((B, V)) < 0.05] = -np.inf
        allowed = rng.random((B, V)) < rng.uniform(0.2, 1.0, size=(B, 1))
        mask = np.zeros((B, 1), dtype=np.uint32)
        for b in range(B):
            for j in range(V):
                if allowed[b, j]:
                    mask[b, 0] |= np.uint32(1 << j)
        t = rng.choice(np.array([0.0, 0.5, 0.7, 1.0, 2.0], np.float32), size=B)
        k = rng.choice(np.array([1, 2, 3, 5, 8, 12, 40], np.int32), size=B)
        p = rng.choice(np.array([0.2, 0.5, 0.75, 0.9, 1.0], np.float32), size=B)
        seed = rng.integers(0, 2**63, size=B, dtype=np.uint64)
        off = rng.integers(0, 2**63, size=B, dtype=np.uint64)
        r = oracle.run_batch(x, "f32", V, temperature=t, top_k=k, top_p=p, seed=seed,
                             offset=off, bitmask=mask, want_probs=True, L=L)
        for b in range(B):
            legal = [bool(allowed[b, j]) and not (np.isinf(x[b, j]) and x[b, j] < 0)
                     for j in range(V)]
            st, tok, kept, probs, bnd = brute_row(x[b], legal, float(t[b]), int(k[b]),
                                                   float(p[b]), r["u"][b])
            assert r["status"][b] == st, (s, b)
            if st:
                continue
            if bnd:
                continue
            got = {j for j in range(V) if (r["kept_mask"][b, 0] >> j) & 1}
            assert got == kept, (s, b, got, kept, t[b], k[b], p[b])
            assert r["token"][b] == tok, (s, b)
            for j in kept:
                assert abs(r["probs"][b, j] - probs[j]) < 1e-12


def check_exhaustive_masks(L=None, V=10):
    """Every mask over V=10 tokens, on tie-heavy logits, several parameter sets."""
    x_row = np.array([1, 3, 3, 0, 2, 3, 1, 2, 0, 3], dtype=np.float32)
    masks = np.arange(1 << V, dtype=np.uint32).reshape(-1, 1)
    B = masks.shape[0]
    x = np.repeat(x_row[None, :], B, axis=0)
    for (t, k, p) in ((1.0, 3, 1.0), (0.7, 4, 0.6), (2.0, 10, 0.9), (0.0, 3, 0.5), (1.0, 1, 1.0)):
        off = np.arange(B, dtype=np.uint64)
        r = oracle.run_batch(x, "f32", V, temperature=[t] * B, top_k=[k] * B, top_p=[p] * B,
                             seed=[5] * B, offset=off, bitmask=masks, L=L)
        for b in range(B):
            legal = [bool((int(masks[b, 0]) >> j) & 1) for j in range(V)]
            st, tok, kept, _, bnd = brute_row(x_row, legal, t, k, p, r["u"][b])
            assert r["status"][b] == st
            if st or bnd:
                continue
            got = {j for j in range(V) if (r["kept_mask"][b, 0] >> j) & 1}
            assert got == kept and r["token"][b] == tok, (b, t, k, p, got, kept)


# --------------------------------------------------------------------------
# Sampler: inverse CDF in id order, frequencies, Gumbel-max
# --------------------------------------------------------------------------

def check_sampler_intervals(L=None):
    """For a fixed kept distribution, the token for u is the id whose CDF
    interval (in id order) contains u."""
    probs = np.array([0.1, 0.05, 0.4, 0.25, 0.2])
    x = np.log(probs)
    for u in np.linspace(0.0005, 0.9995, 97):
        r = oracle.select_core(x, x, np.ones(5, np.uint8), 5, 1.0, u, L=L)
        cdf = np.cumsum(probs)
        want = int(np.searchsorted(cdf, u, side="right"))
        assert r["token"] == want, (u, r["token"], want)


def check_frequencies_and_gumbel(L=None, n=200000):
    """Draws over consecutive offsets follow the kept distribution, and so do
    Gumbel-max draws (lecture 9, section 3.2) on the same logits."""
    V = 6
    x = np.array([[2.0, 0.5, 1.5, -1.0, 1.0, 0.0]], dtype=np.float32)
    xs = np.repeat(x, n, axis=0)
    r = oracle.run_batch(xs, "f32", V, temperature=[0.8] * n, top_k=[4] * n, top_p=[0.95] * n,
                         seed=[11] * n, offset=np.arange(n, dtype=np.uint64), want_probs=False,
                         L=L)
    single = oracle.run_batch(x, "f32", V, temperature=[0.8], top_k=[4], top_p=[0.95],
                              want_probs=True, L=L)
    ptrue = single["probs"][0]
    freq = np.bincount(r["token"], minlength=V) / n
    sd = np.sqrt(ptrue * (1 - ptrue) / n)
    assert np.all(np.abs(freq - ptrue) <= 5 * sd + 1e-12), (freq, ptrue)
    # Gumbel-max on the kept logits: argmax(z_i + g_i) over the kept set.
    kept = ptrue > 0
    z = (x[0].astype(np.float64) / np.float32(0.8))
    rng = np.random.Generator(np.random.PCG64(5))
    g = -np.log(-np.log(rng.random((n, V))))
    zz = np.where(kept[None, :], z[None, :] + g, -np.inf)
    gfreq = np.bincount(zz.argmax(axis=1), minlength=V) / n
    assert np.all(np.abs(gfreq - ptrue) <= 5 * sd + 1e-12), (gfreq, ptrue)


def check_temperature_limit(L=None):
    """As T -> 0 the distribution collapses onto the argmax (lecture 9, 3.3):
    with two kept logits 1 apart, the ratio is exp(-1/T)."""
    x = np.array([[3.0, 2.0, -5.0]], dtype=np.float32)
    for t in (1.0, 0.5, 0.25, 0.1):
        r = oracle.run_batch(x, "f32", 3, temperature=[t], top_k=[2], top_p=[1.0],
                             want_probs=True, L=L)
        pr = r["probs"][0]
        z0 = float(np.float32(3.0) / np.float32(t))
        z1 = float(np.float32(2.0) / np.float32(t))
        assert abs(pr[1] / pr[0] - math.exp(z1 - z0)) < 1e-12
        assert abs(pr[0] - 1 / (1 + math.exp(z1 - z0))) < 1e-12


ALL_CHECKS = [check_worked_examples, check_dyadic_boundary, check_greedy_tie,
              check_mask_bit_order, check_status_codes, check_decoders,
              check_philox_vs_curand, check_uniformity, check_bruteforce,
              check_exhaustive_masks, check_sampler_intervals,
              check_frequencies_and_gumbel, check_temperature_limit]
