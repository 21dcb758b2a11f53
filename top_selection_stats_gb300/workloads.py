"""Seeded synthetic inputs for batched top-k / top-p sampling.

This module only draws inputs: logits, legal-token bitmasks and per-row
sampling parameters.  It holds none of the selection arithmetic, and both the
CUDA path and the CPU oracle consume what it produces.

The workloads stand in for the serving runs measured in the Qrita paper notes
(four models on WikiText-2, vocabularies 128,256 to 262,208): logits are a
Gaussian background plus a small shifted head, the shape that paper's
sigma-truncation assumes (key design 1).  Values are drawn in float32 with
numpy's PCG64 and cast to bf16 / fp16 with round-to-nearest-even by torch.

Named workloads:
  tiny4x1024_f32      B=4    V=1024   f32  -- small mixed-parameter case
  topk64x32000_f32    B=64   V=32000  f32  -- pure top-k (k=50, p=1)
  mixed256x128256_bf16 B=256 V=128256 bf16 -- mixed per-row parameters
  ties512x151936_bf16 B=512  V=151936 bf16 -- quantised head (ties) + grammar masks
  decode1024x256000_f16 B=1024 V=256000 fp16 -- repeated decode, drawn on the device
  verify256x4x128256_f32 B=256 sequences, G=4 draft tokens, V=128256 -- inputs of
                      speculative-decoding verification (see verify_case)
  verify64x4x128256_f32  the same with B=64 (small case for profiling)
"""
import numpy as np
import torch

WORKLOADS = {
    "tiny4x1024_f32": dict(B=4, V=1024, dtype="f32", seed=0),
    "topk64x32000_f32": dict(B=64, V=32000, dtype="f32", seed=1),
    "mixed256x128256_bf16": dict(B=256, V=128256, dtype="bf16", seed=2),
    "ties512x151936_bf16": dict(B=512, V=151936, dtype="bf16", seed=3),
    "decode1024x256000_f16": dict(B=1024, V=256000, dtype="f16", seed=4),
}

VERIFY_WORKLOADS = {
    "verify256x4x128256_f32": dict(B=256, G=4, V=128256, seed=5),
    "verify64x4x128256_f32": dict(B=64, G=4, V=128256, seed=6),
}

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def n_words(V):
    return (V + 31) // 32


def to_dtype(x_f32, dtype):
    """float32 numpy/torch -> torch tensor of the workload dtype (RNE cast)."""
    t = torch.as_tensor(x_f32, dtype=torch.float32)
    return t.to(TORCH_DTYPE[dtype])


def bits_numpy(t):
    """Host numpy view of a logits tensor: float32 values or uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def mask_from_allowed(allowed_bool):
    """bool [B, V] -> uint32 [B, ceil(V/32)]: bit j%32 of word j/32 = token j allowed."""
    B, V = allowed_bool.shape
    W = n_words(V)
    padded = np.zeros((B, W * 32), dtype=np.uint64)
    padded[:, :V] = allowed_bool
    padded = padded.reshape(B, W, 32)
    weights = (np.uint64(1) << np.arange(32, dtype=np.uint64))
    return (padded * weights).sum(axis=2).astype(np.uint32)


def head_rows(rng, B, V, sigma, n_head, lo, hi):
    """Gaussian background N(0, sigma^2) plus n_head[r] distinct ids per row shifted
    by U(lo, hi)."""
    x = rng.standard_normal((B, V), dtype=np.float32) * np.float32(sigma)
    for r in range(B):
        ids = rng.choice(V, size=int(n_head[r]), replace=False)
        x[r, ids] += rng.uniform(lo, hi, size=ids.shape[0]).astype(np.float32)
    return x


def _params(B, temperature, top_k, top_p, seed_value, base_offset=0):
    return dict(
        temperature=torch.as_tensor(np.asarray(temperature, dtype=np.float32)),
        top_k=torch.as_tensor(np.asarray(top_k, dtype=np.int32)),
        top_p=torch.as_tensor(np.asarray(top_p, dtype=np.float32)),
        seed=torch.full((B,), int(seed_value), dtype=torch.int64),
        offset=torch.arange(B, dtype=torch.int64) + int(base_offset),
    )


def make(name, step=0, device="cpu", rows=None):
    """Build a named workload.

    Returns a dict: logits (torch [B, V] of the workload dtype), bitmask (torch
    int32 [B, W] holding uint32 bit patterns, or None), temperature / top_k /
    top_p / seed / offset (torch, length B), and B, V, dtype, name.
    ``rows`` optionally keeps only the first ``rows`` rows (small parity cases).
    ``step`` selects the decode step (fresh logits, offsets advanced by B).
    """
    cfg = WORKLOADS[name]
    B, V, dtype, seed = cfg["B"], cfg["V"], cfg["dtype"], cfg["seed"]
    bitmask = None
    if name == "tiny4x1024_f32":
        rng = np.random.Generator(np.random.PCG64(seed))
        x = head_rows(rng, B, V, 1.0, np.full(B, 8), 4.0, 8.0)
        t = [1.0, 0.0, 0.7, 1.0]
        k = [50, V, 1024, 2]
        p = [0.9, 1.0, 0.8, 0.5]
        par = _params(B, t, k, p, 0)
        logits = to_dtype(x, dtype)
    elif name == "topk64x32000_f32":
        rng = np.random.Generator(np.random.PCG64(seed))
        x = head_rows(rng, B, V, 2.0, np.full(B, 200), 5.0, 15.0)
        par = _params(B, np.ones(B), np.full(B, 50), np.ones(B), 1)
        logits = to_dtype(x, dtype)
    elif name == "mixed256x128256_bf16":
        rng = np.random.Generator(np.random.PCG64(seed))
        n_head = rng.integers(50, 501, size=B)
        x = head_rows(rng, B, V, 2.0, n_head, 3.0, 12.0)
        t = rng.choice(np.array([0.0, 0.7, 1.0, 1.3], dtype=np.float32), size=B)
        k = rng.choice(np.array([1, 20, 50, 1000, V], dtype=np.int32), size=B)
        p = rng.choice(np.array([0.8, 0.9, 0.95, 1.0], dtype=np.float32), size=B)
        par = _params(B, t, k, p, 2)
        logits = to_dtype(x, dtype)
    elif name == "ties512x151936_bf16":
        rng = np.random.Generator(np.random.PCG64(seed))
        n_head = rng.integers(50, 501, size=B)
        x = head_rows(rng, B, V, 2.0, n_head, 3.0, 12.0)
        for r in range(B):
            q = np.float32(np.percentile(x[r], 99.9))
            mx = np.float32(x[r].max())
            levels = to_dtype(np.linspace(q, mx, 64, dtype=np.float32), "bf16").float().numpy()
            levels = np.unique(levels)
            sel = x[r] >= q
            v = x[r, sel]
            idx = np.abs(v[:, None] - levels[None, :]).argmin(axis=1)
            x[r, sel] = levels[idx]
        allowed = np.ones((B, V), dtype=bool)
        perm = rng.permutation(B)
        n30, n5 = int(round(0.30 * B)), int(round(0.05 * B))
        for r in perm[:n30]:
            allowed[r] = False
            allowed[r, rng.choice(V, size=int(0.05 * V), replace=False)] = True
        for r in perm[n30:n30 + n5]:
            allowed[r] = False
            allowed[r, rng.choice(V, size=int(rng.integers(2, 5)), replace=False)] = True
        allowed[perm[n30 + n5]] = False  # exactly one row allows nothing
        bitmask = torch.as_tensor(mask_from_allowed(allowed).view(np.int32))
        par = _params(B, np.full(B, 0.8), np.full(B, 40), np.full(B, 0.95), 3)
        logits = to_dtype(x, dtype)
    elif name == "decode1024x256000_f16":
        dev = torch.device(device)
        g = torch.Generator(device=dev)
        g.manual_seed(seed * 1000003 + step)
        x = torch.randn((B, V), generator=g, device=dev, dtype=torch.float32) * 1.5
        ids = torch.rand((B, V), generator=g, device=dev).argsort(dim=1)[:, :1000]
        shift = torch.rand((B, 1000), generator=g, device=dev) * 8.0 + 2.0
        x.scatter_add_(1, ids, shift)
        logits = x.to(torch.float16)
        rng = np.random.Generator(np.random.PCG64(seed))
        k = rng.choice(np.array([50, 4096], dtype=np.int32), size=B)
        p = rng.choice(np.array([0.9, 1.0], dtype=np.float32), size=B)
        par = _params(B, np.ones(B), k, p, 4, base_offset=step * B)
    else:  # pragma: no cover
        raise KeyError(name)
    out = dict(name=name, B=B, V=V, dtype=dtype, logits=logits, bitmask=bitmask, **par)
    if rows is not None and rows < B:
        out = {k2: (v[:rows] if torch.is_tensor(v) else v) for k2, v in out.items()}
        out["B"] = rows
    if device != "cpu":
        out = {k2: (v.to(device) if torch.is_tensor(v) else v) for k2, v in out.items()}
    return out


def random_case(seed, B, V, dtype="f32", sigma=2.0, n_head=(0, 64), head=(2.0, 10.0),
                grid=None, temps=(0.0, 0.5, 0.7, 1.0, 1.3), topks=None, topps=None,
                mask_frac=0.0, mask_density=(0.02, 0.6), neg_inf_frac=0.0):
    """Small random batch for parity tests.

    grid: if given, logits are drawn from this many integer levels (forces ties).
    mask_frac: fraction of rows given a random legal-token mask.
    neg_inf_frac: fraction of entries set to -inf (also illegal by the contract).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    if grid is not None:
        x = rng.integers(0, grid, size=(B, V)).astype(np.float32)
    else:
        nh = rng.integers(n_head[0], n_head[1] + 1, size=B)
        x = head_rows(rng, B, V, sigma, np.minimum(nh, V), head[0], head[1])
    if neg_inf_frac > 0:
        x[rng.random((B, V)) < neg_inf_frac] = -np.inf
    if topks is None:
        topks = (1, 2, 5, 50, max(1, V // 3), V, V + 7)
    if topps is None:
        topps = (0.3, 0.5, 0.8, 0.9, 0.95, 1.0)
    t = rng.choice(np.array(temps, dtype=np.float32), size=B)
    k = rng.choice(np.array(topks, dtype=np.int32), size=B)
    p = rng.choice(np.array(topps, dtype=np.float32), size=B)
    bitmask = None
    if mask_frac > 0:
        allowed = np.ones((B, V), dtype=bool)
        for r in range(B):
            if rng.random() < mask_frac:
                dens = rng.uniform(*mask_density)
                allowed[r] = rng.random(V) < dens
        bitmask = torch.as_tensor(mask_from_allowed(allowed).view(np.int32))
    par = _params(B, t, k, p, int(rng.integers(0, 2**31)))
    return dict(name=f"random{seed}", B=B, V=V, dtype=dtype, logits=to_dtype(x, dtype),
                bitmask=bitmask, **par)


def verify_case(seed, B, G, V, ld=None, support=(50, 500), wide_frac=0.1, wide=(20000, 50000),
                overlap=0.7, noise=0.5):
    """Inputs of speculative-decoding verification: per sequence, G draft
    positions with a draft distribution q_i and a draft token drawn from it,
    and G+1 target distributions p_i (the last one for the bonus token).

    Each p_i is a normalised distribution on a random support (UniformInt
    ``support`` ids, or ``wide`` ids for a ``wide_frac`` share of positions),
    the shape of the kept sets that top-k / top-p leave.  q_i shares
    ``overlap`` of p_i's support with weights perturbed by a log-normal factor
    (sigma ``noise``) and puts the rest of its mass on ids of its own.  Values
    are normalised in float64 and stored as float32; draft tokens are drawn
    from the stored q_i with numpy.  Rows are padded with zeros to ``ld``.
    Returns torch CPU tensors p [B, G+1, ld], q [B, G, ld], d int32 [B, G],
    seed / offset int64 [B] (offsets G+1 apart), and B, G, V, ld.
    """
    ld = V if ld is None else ld
    rng = np.random.Generator(np.random.PCG64(seed))
    p = np.zeros((B, G + 1, ld), dtype=np.float32)
    q = np.zeros((B, max(G, 1), ld), dtype=np.float32)
    d = np.zeros((B, max(G, 1)), dtype=np.int32)

    def support_size():
        lo, hi = wide if rng.random() < wide_frac else support
        return int(min(V, rng.integers(lo, hi + 1)))

    for s in range(B):
        for i in range(G + 1):
            n = support_size()
            ids = rng.choice(V, size=n, replace=False)
            w = rng.gamma(0.6, size=n) + 1e-4
            p[s, i, ids] = (w / w.sum()).astype(np.float32)
            if i == G:
                continue
            n_sh = int(round(overlap * n))
            wq = np.zeros(V)
            wq[ids[:n_sh]] = w[:n_sh] * np.exp(noise * rng.standard_normal(n_sh))
            n_own = max(1, n - n_sh)
            own = rng.choice(V, size=n_own, replace=False)
            wq[own] += rng.gamma(0.6, size=n_own) + 1e-4
            qi = (wq / wq.sum()).astype(np.float32)
            q[s, i, :V] = qi
            c = np.cumsum(qi.astype(np.float64))
            d[s, i] = min(int(np.searchsorted(c, rng.random() * c[-1], side="right")), V - 1)
            while qi[d[s, i]] == 0.0:  # land on a support id
                d[s, i] -= 1
    return dict(B=B, G=G, V=V, ld=ld, p=torch.from_numpy(p),
                q=torch.from_numpy(q[:, :G]), d=torch.from_numpy(d[:, :G]),
                seed=torch.full((B,), int(seed) * 7919 + 1, dtype=torch.int64),
                offset=torch.arange(B, dtype=torch.int64) * (G + 1))


def rank_shard(case, rank, world):
    """Rank `rank`'s batch of a job run on `world` ranks: the job is `world`
    consecutive copies of the case's B rows, copy r drawing with its Philox
    offsets advanced by r * B (so no two ranks repeat a draw), and each rank's
    batch is its own contiguous block of B rows -- one GPU's batch is its
    shard, with no exchange between ranks.  world = 1 returns the case."""
    if world <= 1:
        return case
    out = dict(case)
    out["offset"] = case["offset"] + int(rank) * int(case["B"])
    out["name"] = f"{case['name']}[shard {rank}/{world}]"
    return out


def global_job(case, world):
    """The whole job that rank_shard splits: its `world` shards' rows,
    concatenated in rank order (host tensors)."""
    parts = [rank_shard(case, r, world) for r in range(world)]
    out = dict(case)
    for k, v in case.items():
        if torch.is_tensor(v):
            out[k] = torch.cat([p[k] for p in parts], dim=0)
    out["B"] = case["B"] * world
    out["name"] = f"{case['name']}[x{world}]"
    return out


def make_verify(name):
    cfg = VERIFY_WORKLOADS[name]
    out = verify_case(cfg["seed"], cfg["B"], cfg["G"], cfg["V"])
    out["name"] = name
    return out
