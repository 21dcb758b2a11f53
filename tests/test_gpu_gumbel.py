"""Gumbel-max sampling: the CUDA path (through the C ABI) against the CPU
oracle.  The decision is an argmax of fp32 values whose noise comes from
CUDA's logf / log1pf on the device and from double-precision log in the
oracle, so tokens must be equal wherever the oracle's best perturbed value
leads the second by at least 1e-4 (the fp32 evaluation of z + g is within
about 1e-5 of the double one for |z| < 100); closer rows are counted, not
compared.  Greedy rows and statuses are exact."""
import numpy as np
import pytest
import torch

import oracle
from top_selection_stats_gb300 import workloads
import gpu_helpers as H

pytestmark = pytest.mark.gpu

MARGIN = 1e-4


def run_both(case, kept):
    s = H.sampler()
    d = H.to_dev(case)
    km = None if kept is None else torch.as_tensor(kept.view(np.int32)).cuda()
    g = s.gumbel_sample(d["logits"], d["temperature"], d["seed"], d["offset"], kept_mask=km)
    torch.cuda.synchronize()
    r = oracle.gumbel_sample(workloads.bits_numpy(case["logits"]), case["dtype"], case["V"],
                             case["temperature"].numpy(), case["seed"].numpy().view(np.uint64),
                             case["offset"].numpy().view(np.uint64), kept_mask=kept,
                             n_threads=oracle.host_cores())
    return g["tokens"].cpu().numpy(), g["status"].cpu().numpy(), r


def compare(tok, st, r):
    assert np.array_equal(st, r["status"]), (np.nonzero(st != r["status"])[0][:8])
    ok = (r["status"] == 0) & (r["margin"] >= MARGIN)
    bad = np.nonzero(ok & (tok != r["token"]))[0]
    assert bad.size == 0, (bad[:8], tok[bad[:8]], r["token"][bad[:8]], r["margin"][bad[:8]])
    assert np.all(tok[r["status"] != 0] == -1)
    return int(ok.sum()), int(((r["status"] == 0) & ~ok).sum())


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("V", [1, 7, 1000, 32000, 70001])
def test_random_rows_with_kept_sets(dtype, V):
    case = workloads.random_case(V * 5 + len(dtype), 32, V, dtype=dtype, mask_frac=0.3,
                                 neg_inf_frac=0.01 if V > 8 else 0.0)
    # kept sets from the oracle's top-k / top-p (the inputs a caller would pass)
    r0 = H.oracle_run(case)
    kept = r0["kept_mask"]
    tok, st, r = run_both(case, kept)
    checked, close = compare(tok, st, r)
    assert checked >= close


def test_full_legal_set_and_greedy_rows():
    case = workloads.random_case(31, 48, 20000, dtype="bf16", temps=(0.0, 0.5, 1.0, 1.3),
                                 mask_frac=0.0, neg_inf_frac=0.02)
    tok, st, r = run_both(case, None)
    compare(tok, st, r)
    greedy = (case["temperature"].numpy() == 0) & (st == 0)
    assert greedy.any() and np.array_equal(tok[greedy], r["token"][greedy])


def test_bench_workload_with_kept_sets():
    case = workloads.make("mixed256x128256_bf16")
    r0 = H.oracle_run(case)
    tok, st, r = run_both(case, r0["kept_mask"])
    checked, close = compare(tok, st, r)
    assert checked > 200


def test_statuses():
    x = np.array([[1.0, 2.0, 3.0, 4.0], [np.nan, 1.0, 2.0, 3.0], [-np.inf] * 4, [1.0, 2.0, 0.5, 0.0]],
                 dtype=np.float32)
    case = dict(name="status", B=4, V=4, dtype="f32", logits=torch.from_numpy(x),
                temperature=torch.tensor([1.0, 1.0, 1.0, -1.0]),
                seed=torch.zeros(4, dtype=torch.int64), offset=torch.arange(4, dtype=torch.int64))
    tok, st, r = run_both(case, None)
    assert list(st) == [0, 2, 1, 3] and list(st) == list(r["status"])
    kept = np.array([[0b1111], [0b1110], [0b1111], [0b1111]], dtype=np.uint32)
    tok, st, r = run_both(case, kept)  # the NaN is outside row 1's kept set
    assert list(st) == [0, 0, 1, 3] and list(st) == list(r["status"])


def test_gumbel_draws_follow_the_kept_distribution():
    """Draws over many offsets follow the oracle's final probabilities, as
    the inverse-CDF sampler's do (the two sampler families agree)."""
    s = H.sampler()
    x = (np.random.Generator(np.random.PCG64(41)).standard_normal(4000) * 2).astype(np.float32)
    x[:6] += np.array([6.0, 5.5, 5.0, 4.5, 4.0, 3.0], np.float32)
    B, n_calls = 4096, 12
    xs = torch.from_numpy(np.repeat(x[None], B, axis=0)).cuda()
    t = torch.full((B,), 0.9, device="cuda")
    k = torch.full((B,), 8, dtype=torch.int32, device="cuda")
    p = torch.full((B,), 0.95, device="cuda")
    seed = torch.full((B,), 17, dtype=torch.int64, device="cuda")
    m = s.topk_topp_mask(xs, t, k, p)
    counts_g = np.zeros(4000)
    counts_s = np.zeros(4000)
    for c in range(n_calls):
        off = torch.arange(B, dtype=torch.int64, device="cuda") + c * B
        g = s.gumbel_sample(xs, t, seed, off, kept_mask=m["kept_mask"])
        q = s.sample(xs, t, k, p, seed, off)
        counts_g += np.bincount(g["tokens"].cpu().numpy(), minlength=4000)
        counts_s += np.bincount(q["tokens"].cpu().numpy(), minlength=4000)
    n = B * n_calls
    r = oracle.run_batch(x[None], "f32", 4000, temperature=[0.9], top_k=[8], top_p=[0.95],
                         want_probs=True)
    pr = r["probs"][0]
    sd = np.sqrt(pr * (1 - pr) / n)
    for counts in (counts_g, counts_s):
        f = counts / n
        assert np.all(np.abs(f - pr) <= 5 * sd + 1e-12), (f[:10], pr[:10])
