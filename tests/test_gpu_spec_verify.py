"""Speculative-decoding verification: the CUDA path (through the C ABI)
against the CPU oracle, sequence by sequence.

The oracle is the rule over the reals (lecture notes, section 5.2): residual
max(0, p - q) in double, compensated sums.  Statuses and accepted counts are
exact (the acceptance test u * q < p is exact in double on both sides).  The
drawn token must equal the oracle's wherever u * S lies more than 1e-6 of S
from a switch point of the draw; the sequences closer than that are counted,
reported and bounded.  A second, labelled check compares every token with the
oracle's fixed-point variant, which takes the draw in the integer precision
the library states (floor(w * 2^42) of binary32 differences)."""
import numpy as np
import pytest
import torch

import oracle
from top_selection_stats_gb300 import binding, workloads
import gpu_helpers as H

pytestmark = pytest.mark.gpu


def run_both(c, V=None):
    V = c["V"] if V is None else V
    B, G = c["B"], c["G"]
    s = H.sampler()
    dev = torch.device("cuda", 0)
    p = c["p"].to(dev)
    q = c["q"].to(dev) if G else None
    d = c["d"].to(dev) if G else None
    g = s.spec_verify(p, q, d, c["seed"].to(dev), c["offset"].to(dev), V=V)
    torch.cuda.synchronize()
    g = {k: v.cpu().numpy() for k, v in g.items()}
    args = (c["p"].numpy(), c["q"].numpy() if G else None, c["d"].numpy() if G else None,
            c["seed"].numpy().view(np.uint64), c["offset"].numpy().view(np.uint64))
    r = oracle.spec_verify(*args, V=V, n_threads=oracle.host_cores())
    r["fixed"] = oracle.spec_verify(*args, V=V, n_threads=oracle.host_cores(), fixed=True)
    return g, r


MARGIN = 1e-6


def compare(g, r):
    bad = np.nonzero(g["status"] != r["status"])[0]
    assert bad.size == 0, ("status", bad[:8], g["status"][bad[:8]], r["status"][bad[:8]])
    bad = np.nonzero(g["n_accepted"] != r["n_accepted"])[0]
    assert bad.size == 0, ("n_accepted", bad[:8], g["n_accepted"][bad[:8]],
                           r["n_accepted"][bad[:8]])
    far = r["margin"] > MARGIN
    bad = np.nonzero(far & (g["tokens"] != r["tokens"]).any(axis=1))[0]
    assert bad.size == 0, ("tokens", bad[:8], g["tokens"][bad[:4]], r["tokens"][bad[:4]])
    near = int((~far & (r["status"] == 0)).sum())
    print(f"spec_verify: {near} of {len(far)} sequences within {MARGIN:g} of a switch point")
    assert near <= 0.1 * len(far) + 2, near
    f = r["fixed"]
    bad = np.nonzero((g["tokens"] != f["tokens"]).any(axis=1))[0]
    assert bad.size == 0, ("tokens vs fixed-point variant", bad[:8])
    return near


@pytest.mark.parametrize("B,G,V", [(32, 4, 1000), (16, 1, 5), (8, 0, 300), (20, 31, 2000),
                                   (12, 2, 1), (12, 2, 3), (40, 4, 4099), (24, 3, 17000),
                                   (16, 4, 70001)])
def test_random_cases(B, G, V):
    c = workloads.verify_case(B * 1000 + G * 10 + V % 97, B, G, V, ld=(V + 3) // 4 * 4,
                              support=(1, min(V, 300)), wide_frac=0.2,
                              wide=(min(V, 2000), min(V, 20000)))
    compare(*run_both(c))


def test_padded_rows_ignore_entries_past_v():
    V, ld = 4099, 4104
    c = workloads.verify_case(77, 24, 3, V, ld=ld, support=(1, 300), wide_frac=0.3,
                              wide=(2000, 4000))
    c["p"][:, :, V:] = float("nan")  # past V: never read as a probability
    c["q"][:, :, V:] = float("nan")
    compare(*run_both(c, V=V))


def test_wide_rows_and_eight_cta_clusters():
    V = 1 << 20
    c = workloads.verify_case(78, 4, 2, V, support=(1000, 5000), wide_frac=0.5,
                              wide=(100000, 400000))
    g, r = run_both(c)
    compare(g, r)
    assert np.all(g["status"] == 0)


def test_medium_batch():
    c = workloads.verify_case(79, 64, 4, 32000, wide_frac=0.15, wide=(5000, 20000))
    compare(*run_both(c))


def test_full_size_workload():
    c = workloads.make_verify("verify256x4x128256_f32")
    g, r = run_both(c)
    compare(g, r)
    assert np.all(g["status"] == 0)
    # both outcomes occur: some sequences draw after a rejection, some get a
    # bonus token
    assert (g["n_accepted"] < c["G"]).any() and (g["n_accepted"] == c["G"]).any()


def _edge_case():
    V, G, B = 257, 3, 8
    c = workloads.verify_case(80, B, G, V, ld=260, support=(3, 40))
    p, q, d = c["p"], c["q"], c["d"]
    # 0: draft equals target everywhere (drafts on the target's support): all
    #    accepted, bonus from p_G
    q[0] = p[0, :G]
    d[0] = p[0, :G].argmax(dim=1).to(torch.int32)
    # 1: target puts no mass where the draft drew at position 0 and the
    #    supports are disjoint there: rejection, residual = p_0
    p[1, 0] = 0.0
    p[1, 0, :4] = torch.tensor([0.125, 0.375, 0.25, 0.25])
    q[1, 0] = 0.0
    q[1, 0, 10] = 1.0
    d[1, 0] = 10
    # 2: draft token out of range
    d[2, 1] = V
    # 3: NaN in the drawn residual row (position 0 rejects: p = 0 at d)
    p[3, 0] = 0.0
    p[3, 0, 5] = 1.0
    q[3, 0] = 0.0
    q[3, 0, 6] = 1.0
    d[3, 0] = 6
    p[3, 0, 100] = float("nan")
    # 4: probability above 1 at a draft token
    q[4, 2, d[4, 2]] = 1.5
    # 5: residual with no mass: p_0 <= q_0 everywhere, p_0(d) = 0
    q[5, 0] = 0.0
    q[5, 0, :8] = 0.125
    p[5, 0] = 0.0
    p[5, 0, :4] = 0.0625
    d[5, 0] = 6
    # 6: negative entry in the bonus row of a sequence that accepts all
    q[6] = p[6, :G]
    d[6] = p[6, :G].argmax(dim=1).to(torch.int32)
    p[6, G, 7] = -0.5
    return c


def test_edge_cases():
    c = _edge_case()
    g, r = run_both(c)
    compare(g, r)
    assert g["n_accepted"][0] == c["G"]
    assert g["status"][1] == 0 and g["n_accepted"][1] == 0
    assert list(g["status"][2:7]) == [3, 3, 3, 1, 3]
    assert np.all(g["tokens"][2:7] == -1)


def test_repeated_calls_and_offsets():
    c = workloads.verify_case(81, 48, 4, 9000, wide_frac=0.2, wide=(2000, 8000))
    for step in range(3):
        c["offset"] = c["offset"] + step * (c["G"] + 1) * c["B"]
        compare(*run_both(c))


def test_consumes_kept_sets_of_the_sampler():
    """The step downstream of the kept-set API: target and draft probabilities
    come from smp_topk_topp_mask (probs_out) on two logits batches; every
    output respects the rule's supports."""
    s = H.sampler()
    B, G, V = 16, 3, 32000
    rng = np.random.Generator(np.random.PCG64(82))
    x_t = workloads.head_rows(rng, B * (G + 1), V, 2.0, np.full(B * (G + 1), 200), 3.0, 10.0)
    x_d = x_t[: B * (G + 1)].reshape(B, G + 1, V)[:, :G].reshape(B * G, V).copy()
    x_d += rng.standard_normal(x_d.shape, dtype=np.float32) * np.float32(1.0)
    dev = torch.device("cuda", 0)

    def probs(x, n):
        t = torch.full((n,), 1.0, device=dev)
        k = torch.full((n,), 50, dtype=torch.int32, device=dev)
        pp = torch.full((n,), 0.9, device=dev)
        out = s.topk_topp_mask(torch.as_tensor(x).to(dev), t, k, pp, want_probs=True)
        assert int(out["status"].abs().sum()) == 0
        return out["probs"]

    pt = probs(x_t, B * (G + 1)).view(B, G + 1, V)
    qd = probs(x_d, B * G).view(B, G, V)
    # drafts drawn from q on the host
    qn = qd.cpu().numpy().astype(np.float64)
    d = np.zeros((B, G), np.int32)
    for b in range(B):
        for i in range(G):
            d[b, i] = rng.choice(V, p=qn[b, i] / qn[b, i].sum())
    seed = torch.full((B,), 5, dtype=torch.int64, device=dev)
    off = torch.arange(B, dtype=torch.int64, device=dev) * (G + 1)
    out = s.spec_verify(pt.contiguous(), qd.contiguous(), torch.as_tensor(d).to(dev), seed, off)
    torch.cuda.synchronize()
    st, n, tok = (out[k].cpu().numpy() for k in ("status", "n_accepted", "tokens"))
    P, Q = pt.cpu().numpy(), qd.cpu().numpy()
    assert np.all(st == 0)
    for b in range(B):
        j = n[b]
        assert list(tok[b, :j]) == list(d[b, :j])
        assert np.all(P[b, np.arange(j), d[b, :j]] > 0)
        x = tok[b, j]
        if j < G:
            assert P[b, j, x] > Q[b, j, x]
        else:
            assert P[b, G, x] > 0
        assert np.all(tok[b, j + 1:] == -1)


def test_call_level_errors():
    s = H.sampler()
    dev = torch.device("cuda", 0)
    L = s.lib
    p = torch.zeros((2, 3, 64), device=dev)
    q = torch.zeros((2, 2, 64), device=dev)
    d = torch.zeros((2, 2), dtype=torch.int32, device=dev)
    sd = torch.zeros(2, dtype=torch.int64, device=dev)
    o = torch.empty((2, 3), dtype=torch.int32, device=dev)
    n = torch.empty(2, dtype=torch.int32, device=dev)
    st = torch.empty(2, dtype=torch.int32, device=dev)
    P = binding._ptr

    def call(pp, G, V, ld, qq=q):
        return L.smp_spec_verify(s.h, pp, P(qq), P(d), 2, G, V, ld, P(sd), P(sd), P(o), P(n),
                                 P(st), None)

    assert call(P(p), 2, 64, 64) == 0
    torch.cuda.synchronize()
    assert call(ctypes_offset(p, 1), 2, 60, 60) == 3      # base not 16-byte aligned
    assert call(P(p), 2, 62, 62) == 3                       # ld not a multiple of 4
    assert call(P(p), 2, 65, 64) == 3                       # ld < V
    assert call(P(p), 32, 64, 64) == 6                      # G above 31
    assert call(P(p), 2, 64, 64, qq=None) == 3              # NULL draft probabilities
    assert L.smp_spec_verify(s.h, P(p), None, None, 0, 2, 64, 64, None, None, None, None, None,
                             None) == 0                     # B = 0: nothing to do


def ctypes_offset(t, elems):
    import ctypes
    return ctypes.c_void_p(t.data_ptr() + 4 * elems)
