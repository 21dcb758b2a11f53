"""CUDA path (through the C ABI) against the CPU oracle, element by element."""
import numpy as np
import pytest
import torch

import oracle
from top_selection_stats_gb300 import workloads
import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["board", "split"])
def kernel(request):
    """Every parity case runs on both sampler kernels (smp_set_kernel)."""
    s = H.sampler()
    s.set_kernel(request.param)
    yield request.param
    s.set_kernel("board")


def run_and_compare(case, modes=("sample", "mask"), check_probs=True, rows=None):
    r = H.oracle_run(case, want_probs=True, rows=rows)
    out = {}
    for mode in modes:
        g = H.gpu_run(case, mode=mode, want_probs=check_probs)
        out[mode] = H.compare(case, g, r, mode=mode, rows=rows,
                              check_probs=check_probs and mode == "mask")
    return out


def test_tiny_mixed_f32():
    run_and_compare(workloads.make("tiny4x1024_f32"))


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("V", [1, 7, 31, 33, 1000, 2049, 5003, 32000, 70001])
def test_random_shapes(dtype, V):
    case = workloads.random_case(V * 7 + len(dtype), 24, V, dtype=dtype, mask_frac=0.3,
                                 neg_inf_frac=0.01 if V > 8 else 0.0)
    run_and_compare(case)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ties_on_integer_grid(dtype):
    case = workloads.random_case(11, 32, 4096, dtype=dtype, grid=6, mask_frac=0.2,
                                 topks=(1, 3, 40, 700, 2000, 4096), topps=(0.5, 0.9, 1.0))
    run_and_compare(case)


def test_full_row_fallback_paths(kernel):
    """Large k beyond the candidate buffer and flat rows under top-p force the
    exact refinement path; it must agree with the oracle too."""
    case = workloads.random_case(5, 32, 60000, dtype="bf16", sigma=0.5, n_head=(0, 4),
                                 temps=(1.0, 2.0), topks=(5000, 20000, 60000),
                                 topps=(0.5, 0.9, 0.99, 1.0), mask_frac=0.25)
    g = H.gpu_run(case, mode="sample", row_info=True)
    r = H.oracle_run(case, want_probs=True)
    H.compare(case, g, r)
    paths = g["row_info"][:, 0]
    assert (paths == 4).any(), paths  # the refinement path ran


def test_topk_only_f32_full():
    case = workloads.make("topk64x32000_f32")
    out = run_and_compare(case)
    assert out["sample"]["token_checked"] > 50


def test_mixed_bf16_full():
    case = workloads.make("mixed256x128256_bf16")
    run_and_compare(case, check_probs=True)


def test_ties_masks_bf16_full():
    case = workloads.make("ties512x151936_bf16")
    r = H.oracle_run(case, want_probs=False)
    assert (r["status"] == 1).sum() == 1  # the row with an empty mask
    g = H.gpu_run(case, mode="sample")
    H.compare(case, g, r)


def _rows_cpu(case, rows):
    """The given rows of a (device) case, on the host, as a case of their own."""
    idx = torch.as_tensor(rows, device=case["logits"].device)
    out = {k: (v.index_select(0, idx.to(v.device)).cpu() if torch.is_tensor(v) else v)
           for k, v in case.items()}
    out["B"] = len(rows)
    return out


def test_decode_loop_f16():
    """The repeated decode loop: 200 steps of 1024 x 256000 fp16 logits, fresh
    each step, the Philox offsets advanced by the B blocks each step consumes,
    kept masks returned.  Every row is compared at steps 0, 1, 2, 99 and 199,
    32 random rows at every other step."""
    rng = np.random.default_rng(0)
    full = {0, 1, 2, 99, 199}
    tot = dict(rows=0, topp_boundary=0, cdf_boundary=0, token_checked=0)
    for step in range(200):
        case = workloads.make("decode1024x256000_f16", step=step, device="cuda")
        B = case["B"]
        rows = np.arange(B) if step in full else np.sort(rng.choice(B, size=32, replace=False))
        g = H.gpu_run(case, mode="sample")
        r = H.oracle_run(_rows_cpu(case, rows))
        st = H.compare(case, g, r, rows=rows)
        for k in tot:
            tot[k] += st[k]
    H.record_boundaries("decode1024x256000_f16 (200 steps)", tot, bounded=True)


def test_topk_covering_a_sparse_legal_set():
    """Rows whose top_k exceeds a sparse legal set (30 % -inf, grammar masks)
    and top_p = 1 keep every legal token, also when the legal set is larger
    than a slice's candidate list (found by a randomised sweep)."""
    case = workloads.random_case(752032311, 33, 70001, dtype="f16", mask_frac=0.8,
                                 neg_inf_frac=0.3, sigma=4.0, n_head=(0, 500),
                                 temps=(0.0, 0.5, 1.0, 1.3, 2.0))
    run_and_compare(case)


def test_far_negative_logits_keep_the_sigma_path(kernel):
    """A penalised decode input: 16 legal logits per row pushed to -60000.
    The results still match the oracle, and on the board kernel the
    sigma-truncated list still serves the rows it serves on the clean input
    (the deviation estimate leaves far-negative values out)."""
    case = workloads.make("decode1024x256000_f16", step=3, device="cuda", rows=64)
    clean = H.gpu_run(case, mode="sample", row_info=True)
    rng = np.random.default_rng(7)
    x = case["logits"].clone()
    for b in range(case["B"]):
        ids = torch.as_tensor(rng.choice(case["V"], size=16, replace=False), device=x.device)
        x[b, ids] = -60000.0
    pen = dict(case, logits=x, name="decode_penalised")
    g = H.gpu_run(pen, mode="sample", row_info=True)
    r = H.oracle_run({k: (v.cpu() if torch.is_tensor(v) else v) for k, v in pen.items()})
    H.compare(pen, g, r)
    if kernel == "board":
        n_clean = int((clean["row_info"][:, 0] == 3).sum())
        n_pen = int((g["row_info"][:, 0] == 3).sum())
        assert n_clean > 0 and n_pen >= n_clean - 2, (n_clean, n_pen)


def test_argmax_matches_oracle():
    for name in ("tiny4x1024_f32", "topk64x32000_f32"):
        case = workloads.make(name)
        g = H.gpu_run(case, mode="argmax")
        r = H.oracle_run(case, mode="argmax")
        H.compare(case, g, r, mode="argmax")
    case = workloads.random_case(3, 64, 3001, dtype="bf16", grid=3, mask_frac=0.5,
                                 neg_inf_frac=0.05)
    H.compare(case, H.gpu_run(case, mode="argmax"), H.oracle_run(case, mode="argmax"),
              mode="argmax")


def test_error_rows():
    V = 300
    x = np.random.default_rng(1).standard_normal((6, V)).astype(np.float32)
    x[1, 5] = np.nan
    x[2, :] = -np.inf
    x[3, 7] = np.inf
    allowed = np.ones((6, V), bool)
    allowed[4] = False
    case = dict(name="errors", B=6, V=V, dtype="f32", logits=torch.from_numpy(x),
                bitmask=torch.from_numpy(workloads.mask_from_allowed(allowed).view(np.int32)),
                temperature=torch.tensor([1, 1, 1, 1, 1, -1.0], dtype=torch.float32),
                top_k=torch.tensor([5] * 6, dtype=torch.int32),
                top_p=torch.tensor([0.9] * 6, dtype=torch.float32),
                seed=torch.zeros(6, dtype=torch.int64), offset=torch.arange(6))
    g = H.gpu_run(case)
    assert list(g["status"]) == [0, 2, 1, 2, 1, 3]
    H.compare(case, g, H.oracle_run(case))


def test_strided_and_unaligned_rows():
    """ld > V (padded rows) and rows that are not 16-byte aligned (plain loads)."""
    for dtype, V, ld in (("bf16", 1003, 1011), ("f32", 5001, 5003), ("f16", 4096, 4100)):
        base = workloads.random_case(V + ld, 16, ld, dtype=dtype, topps=(0.9, 1.0))
        full = base["logits"]
        case = dict(base)
        case["V"] = V
        # oracle sees [B, ld] storage, V columns
        x = workloads.bits_numpy(full)
        p = {k: base[k].numpy() for k in ("temperature", "top_k", "top_p", "seed", "offset")}
        p["top_k"] = np.minimum(p["top_k"], V)
        r = oracle.run_batch(x, dtype, V, ld=ld, n_threads=4, **p)
        s = H.sampler()
        d = {k: torch.as_tensor(v).cuda() for k, v in p.items()}
        lg = full.cuda()
        out = s.sample(lg, d["temperature"], d["top_k"], d["top_p"], d["seed"], d["offset"],
                       V=V, want_mask=True)
        torch.cuda.synchronize()
        g = {k: v.cpu().numpy() for k, v in out.items()}
        g["kept_mask"] = g["kept_mask"].view(np.uint32)
        case["B"] = 16
        case["name"] = f"strided-{dtype}"
        H.compare(case, g, r)


def test_determinism_repeated_calls():
    case = workloads.make("mixed256x128256_bf16")
    a = H.gpu_run(case, mode="sample")
    for _ in range(5):
        b = H.gpu_run(case, mode="sample")
        assert (a["tokens"] == b["tokens"]).all()
        assert (a["kept_mask"] == b["kept_mask"]).all()


def test_sampling_frequencies_tv():
    """10^6 draws of one row (replicated, distinct offsets) against the
    oracle's exact probabilities: total variation within the noise floor."""
    V = 2000
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(V) * 2).astype(np.float32)
    x[rng.choice(V, 30, replace=False)] += 6
    n_per, calls = 4096, 245
    case1 = dict(name="tv", B=1, V=V, dtype="f32", logits=torch.from_numpy(x[None, :].copy()),
                 bitmask=None, temperature=torch.tensor([0.9]), top_k=torch.tensor([50], dtype=torch.int32),
                 top_p=torch.tensor([0.9]), seed=torch.tensor([3]), offset=torch.tensor([0]))
    r = H.oracle_run(case1, want_probs=True)
    p = r["probs"][0]
    s = H.sampler()
    lg = torch.from_numpy(np.repeat(x[None, :], n_per, axis=0)).cuda()
    t = torch.full((n_per,), 0.9, device="cuda")
    k = torch.full((n_per,), 50, dtype=torch.int32, device="cuda")
    pp = torch.full((n_per,), 0.9, device="cuda")
    sd = torch.full((n_per,), 3, dtype=torch.int64, device="cuda")
    counts = torch.zeros(V, dtype=torch.int64, device="cuda")
    for c in range(calls):
        off = torch.arange(n_per, device="cuda", dtype=torch.int64) + c * n_per
        out = s.sample(lg, t, k, pp, sd, off)
        counts += torch.bincount(out["tokens"].long(), minlength=V)
    n = n_per * calls
    freq = counts.cpu().numpy() / n
    tv = 0.5 * np.abs(freq - p).sum()
    floor = 0.5 * np.sum(np.sqrt(2 * p * (1 - p) / (np.pi * n)))
    assert tv <= max(0.01, 3 * floor), (tv, floor)
    assert tv <= 0.01


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_tie_groups_beyond_list_capacity(dtype):
    """Rows of three values only: every boundary value has ~17k copies, more than
    the candidate list holds, so the earliest-id tie quota is resolved by ranking
    the copies in id order over the whole row."""
    case = workloads.random_case(17 + len(dtype), 24, 50000, dtype=dtype, grid=3,
                                 temps=(0.5, 1.0, 3.0), topks=(5000, 20000, 40000, 50000),
                                 topps=(0.2, 0.6, 0.95, 1.0), mask_frac=0.2,
                                 mask_density=(0.5, 0.9))
    g = H.gpu_run(case, mode="sample", row_info=True)
    r = H.oracle_run(case, want_probs=True)
    H.compare(case, g, r)
    gm = H.gpu_run(case, mode="mask", want_probs=True)
    H.compare(case, gm, r, mode="mask", check_probs=True)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_tie_groups_of_hundreds_at_the_boundary(dtype):
    """A value with 300-2040 copies holds the top-k or top-p boundary, so the
    earliest-id quota ranks hundreds of tied ids: spread over the row (ranked
    within one bin of consecutive ids) or packed into consecutive ids (a bin
    with more copies than threads takes the radix ranking)."""
    V, B = 128256, 16
    rng = np.random.default_rng(31)
    x = np.clip(rng.standard_normal((B, V)), -6.0, 3.5).astype(np.float32)
    T = np.empty(B, np.float32)
    K = np.empty(B, np.int32)
    P = np.empty(B, np.float32)
    for r_ in range(B):
        m = (300, 700, 1500, 2040)[r_ % 4]
        topk_row = (r_ // 4) % 2 == 0
        ids = (np.arange(1024, 1024 + m) if r_ >= 8 else rng.choice(V - 8, size=m, replace=False))
        x[r_, ids] = 4.0
        head = np.setdiff1d(np.arange(V - 8, V), ids)[:5]
        x[r_, head] = 6.0 + 0.5 * np.arange(5)
        T[r_] = 1.0 if r_ % 3 else 0.7
        xv = workloads.to_dtype(x[r_], dtype).float().numpy().astype(np.float64)
        w = np.exp((xv - xv.max()) / T[r_])
        if topk_row:
            K[r_], P[r_] = 5 + m // 2, 1.0
        else:
            w4 = np.exp((4.0 - xv.max()) / T[r_])
            K[r_] = V
            P[r_] = np.float32((w[xv > 4.0].sum() + (m // 2 + 0.5) * w4) / w.sum())
    case = dict(name="tiegroups", B=B, V=V, dtype=dtype, logits=workloads.to_dtype(x, dtype),
                bitmask=None, temperature=torch.from_numpy(T), top_k=torch.from_numpy(K),
                top_p=torch.from_numpy(P), seed=torch.full((B,), 3, dtype=torch.int64),
                offset=torch.arange(B))
    run_and_compare(case)


def test_few_legal_tokens_take_the_whole_legal_set():
    """Grammar masks that leave a handful of tokens: the list takes every legal
    token, k beyond the legal count keeps them all."""
    V = 151936
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((12, V)) * 2).astype(np.float32)
    allowed = np.zeros((12, V), bool)
    for r_ in range(12):
        allowed[r_, rng.choice(V, size=int(rng.integers(1, 3000)), replace=False)] = True
    case = dict(name="fewlegal", B=12, V=V, dtype="bf16", logits=workloads.to_dtype(x, "bf16"),
                bitmask=torch.from_numpy(workloads.mask_from_allowed(allowed).view(np.int32)),
                temperature=torch.tensor([0.8, 1.0, 1.3] * 4, dtype=torch.float32),
                top_k=torch.tensor([40, 1000, 4096, V] * 3, dtype=torch.int32),
                top_p=torch.tensor([0.95, 1.0, 0.5, 0.9] * 3, dtype=torch.float32),
                seed=torch.full((12,), 9, dtype=torch.int64), offset=torch.arange(12))
    run_and_compare(case)


def check_logprobs(case):
    """smp_sample_logprob: the same tokens as smp_sample, and the log of each
    drawn token's final probability within the probabilities' tolerance
    (|d log r| = |dr| / r <= 1e-5); greedy rows 0, error rows NaN."""
    r = H.oracle_run(case, want_probs=True)
    s = H.sampler()
    d = H.to_dev(case)
    args = (d["logits"], d["temperature"], d["top_k"], d["top_p"], d["seed"], d["offset"])
    g = s.sample(*args, bitmask=d["bitmask"], want_logprob=True)
    plain = s.sample(*args, bitmask=d["bitmask"])
    torch.cuda.synchronize()
    tok, st, lp = (g[k].cpu().numpy() for k in ("tokens", "status", "logprobs"))
    ptok, pst = plain["tokens"].cpu().numpy(), plain["status"].cpu().numpy()
    bad = np.nonzero((tok != ptok) | (st != pst))[0]
    assert bad.size == 0, (case["name"], bad[:8], tok[bad[:8]], ptok[bad[:8]], st[bad[:8]],
                           pst[bad[:8]], r["token"][bad[:8]], r["flags"][bad[:8]])
    assert np.array_equal(st, r["status"])
    assert np.all(np.isnan(lp[st != 0]))
    greedy = (st == 0) & (case["temperature"].cpu().numpy() == 0)
    assert np.all(lp[greedy] == 0.0)
    ok = (st == 0) & (tok == r["token"]) & ((r["flags"] & oracle.FLAG_TOPP_BOUNDARY) == 0)
    rows = np.nonzero(ok)[0]
    want = np.log(r["probs"][rows, tok[rows]])
    err = np.abs(lp[rows].astype(np.float64) - want)
    assert err.max(initial=0.0) <= H.PROB_RTOL, (case["name"], rows[err.argmax()], err.max())
    return len(rows)


@pytest.mark.parametrize("name", ["tiny4x1024_f32", "topk64x32000_f32"])
def test_logprobs_named(name):
    assert check_logprobs(workloads.make(name)) > 0


def test_logprobs_bench_workload():
    # every row class of the bench workload: greedy, keep-all, lists, flat top-p
    assert check_logprobs(workloads.make("mixed256x128256_bf16")) > 200


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_logprobs_random(dtype):
    case = workloads.random_case(4242 + len(dtype), 48, 20000, dtype=dtype, mask_frac=0.3,
                                 neg_inf_frac=0.01)
    assert check_logprobs(case) > 0


def test_logprobs_ties_and_masks():
    assert check_logprobs(workloads.make("ties512x151936_bf16", rows=96)) > 0


def test_interleaved_launches_repeat_bit_for_bit():
    """Launches of different batch sizes and row mixes, interleaved in varying
    orders and with the optional outputs on and off, give the same results
    for the same inputs every time.  Rows that share passes over the job
    board depend on timing between CTAs; this checks that no result does (a
    missing barrier there once turned a stale claim into an expired wait)."""
    cases = [workloads.make("mixed256x128256_bf16"),
             workloads.random_case(4245, 48, 20000, dtype="f32", mask_frac=0.3, neg_inf_frac=0.01),
             workloads.random_case(4246, 48, 20000, dtype="bf16", mask_frac=0.3,
                                   neg_inf_frac=0.01),
             workloads.random_case(501, 96, 70001, dtype="bf16", topks=(20, 1000, 6666, 70001),
                                   topps=(0.8, 0.95, 1.0))]
    s = H.sampler()
    devc = [H.to_dev(c) for c in cases]

    def run(i, lp):
        d = devc[i]
        out = s.sample(d["logits"], d["temperature"], d["top_k"], d["top_p"], d["seed"],
                       d["offset"], bitmask=d["bitmask"], want_mask=True, want_logprob=lp)
        return tuple(out[k].cpu().numpy().copy() for k in ("tokens", "status", "kept_mask",
                                                            "kept_count"))

    first = [run(i, False) for i in range(len(cases))]
    for i in range(len(cases)):
        assert not first[i][1].any(), (cases[i]["name"], np.nonzero(first[i][1])[0][:8])
    rng = np.random.Generator(np.random.PCG64(99))
    for rep in range(24):
        i = int(rng.integers(0, len(cases)))
        got = run(i, bool(rep % 2))
        for a, b, what in zip(first[i], got, ("tokens", "status", "kept_mask", "kept_count")):
            bad = np.nonzero((a != b).reshape(a.shape[0], -1).any(axis=1))[0]
            assert bad.size == 0, (cases[i]["name"], rep, what, bad[:8])


def check_top_logprobs(case, n):
    """smp_top_logprobs on smp_sample_logprob's outputs: the n best kept
    tokens by logit (smallest id first among equal logits) equal the
    oracle's, and their logprobs are within the probabilities' tolerance of
    the log of the oracle's final probabilities (2e-5: the drawn token's own
    logprob plus a difference of two fp32 scaled logits)."""
    r = H.oracle_run(case, want_probs=True)
    s = H.sampler()
    d = H.to_dev(case)
    g = s.sample(d["logits"], d["temperature"], d["top_k"], d["top_p"], d["seed"], d["offset"],
                 bitmask=d["bitmask"], want_mask=True, want_logprob=True)
    t = s.top_logprobs(d["logits"], d["temperature"], g["kept_mask"], g["tokens"], g["logprobs"],
                       n)
    torch.cuda.synchronize()
    gi, gl = t["ids"].cpu().numpy(), t["logprobs"].cpu().numpy()
    st, tok = g["status"].cpu().numpy(), g["tokens"].cpu().numpy()
    x = workloads.bits_numpy(case["logits"])
    xv = x if case["dtype"] == "f32" else torch.from_numpy(x.view(np.int16)).view(
        torch.bfloat16 if case["dtype"] == "bf16" else torch.float16).float().numpy()
    wi, wl = oracle.top_logprobs(xv, r["probs"] > 0, r["probs"], r["status"], n)
    ok = (st == 0) & (r["status"] == 0) & (tok == r["token"]) & (r["flags"] == 0)
    rows = np.nonzero(ok)[0]
    assert np.array_equal(gi[rows], wi[rows]), rows[(gi[rows] != wi[rows]).any(axis=1)][:5]
    fin = np.isfinite(wl[rows])
    err = np.abs(gl[rows][fin].astype(np.float64) - wl[rows][fin])
    assert err.max(initial=0.0) <= 2e-5, err.max()
    assert np.all(gl[rows][~fin] == -np.inf)
    bad = st != 0
    assert np.all(gi[bad] == -1) and np.all(np.isnan(gl[bad]))
    return len(rows)


@pytest.mark.parametrize("n", [1, 5, 32])
def test_top_logprobs_bench_workload(n):
    assert check_top_logprobs(workloads.make("mixed256x128256_bf16"), n) > 200


@pytest.mark.parametrize("dtype", ["f32", "f16"])
def test_top_logprobs_random_and_ties(dtype):
    case = workloads.random_case(5150 + len(dtype), 40, 9000, dtype=dtype, mask_frac=0.3,
                                 neg_inf_frac=0.01)
    assert check_top_logprobs(case, 20) > 0
    ties = workloads.random_case(12, 32, 4096, dtype=dtype, grid=6, mask_frac=0.2,
                                 topks=(3, 40, 700, 4096), topps=(0.5, 0.9, 1.0))
    assert check_top_logprobs(ties, 32) > 0
    # rows of 9001 tokens: not 16-byte aligned past row 0, and a partial last word
    odd = workloads.random_case(5170 + len(dtype), 24, 9001, dtype=dtype, mask_frac=0.2)
    assert check_top_logprobs(odd, 7) > 0
