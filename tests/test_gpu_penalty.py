"""Repetition penalty (in place, CTRL rule): the CUDA path (through the C ABI)
against the CPU oracle, bit for bit on the stored logits, and chained with
the sampler."""
import numpy as np
import pytest
import torch

import oracle
from top_selection_stats_gb300 import binding, workloads
import gpu_helpers as H

pytestmark = pytest.mark.gpu


def history(rng, B, V, Hn, pad_frac=0.1):
    h = rng.integers(0, V, size=(B, Hn)).astype(np.int32)
    if Hn:
        h[:, Hn // 2:] = h[:, :Hn - Hn // 2][:, :Hn // 2]  # repeats
        pad = rng.random((B, Hn)) < pad_frac
        h[pad] = rng.choice(np.array([-1, -7, V, V + 3], dtype=np.int32), size=int(pad.sum()))
    return h


def run_both(case, hist, pen):
    V, dt = case["V"], case["dtype"]
    s = H.sampler()
    dev = torch.device("cuda", 0)
    lg = case["logits"].to(dev).contiguous()
    st = s.repetition_penalty(lg, torch.as_tensor(hist).to(dev), torch.as_tensor(pen).to(dev),
                              V=V)
    torch.cuda.synchronize()
    got = workloads.bits_numpy(lg)
    want, wst = oracle.repetition_penalty(workloads.bits_numpy(case["logits"]), dt, V, hist, pen)
    return got, st.cpu().numpy(), want, wst


def assert_same(got, want, dtype):
    if dtype == "f32":
        both_nan = np.isnan(got) & np.isnan(want)
        gb, wb = got.view(np.uint32), want.view(np.uint32)
    else:
        exp_mask = 0x7c00 if dtype == "f16" else 0x7f80
        man_mask = 0x03ff if dtype == "f16" else 0x007f

        def isnan16(b):
            return ((b & exp_mask) == exp_mask) & ((b & man_mask) != 0)
        both_nan = isnan16(got) & isnan16(want)
        gb, wb = got, want
    bad = np.argwhere((gb != wb) & ~both_nan)
    assert bad.size == 0, (dtype, bad[:5], gb[tuple(bad[0])], wb[tuple(bad[0])])


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("V,Hn", [(1, 4), (33, 40), (1000, 300), (32000, 1024), (128256, 512)])
def test_bit_exact(dtype, V, Hn):
    rng = np.random.Generator(np.random.PCG64(V + Hn + len(dtype)))
    B = 24
    case = workloads.random_case(V * 3 + Hn, B, V, dtype=dtype, neg_inf_frac=0.02 if V > 8 else 0)
    hist = history(rng, B, V, Hn)
    pen = rng.choice(np.array([1.0, 1.1, 1.3, 2.0, 0.7, 0.0, -1.0, np.nan, np.inf],
                              dtype=np.float32), size=B)
    got, st, want, wst = run_both(case, hist, pen)
    assert np.array_equal(st, wst)
    assert_same(got, want, dtype)
    # invalid penalties leave the row unchanged
    orig = workloads.bits_numpy(case["logits"])
    for r in np.nonzero(wst)[0]:
        assert np.array_equal(got[r].view(np.uint8), orig[r].view(np.uint8))


def test_padded_rows_nan_and_empty_history():
    rng = np.random.Generator(np.random.PCG64(5))
    B, V, ld = 8, 5000, 5008
    x = (rng.standard_normal((B, ld)) * 3).astype(np.float32)
    x[:, 100] = np.nan
    x[:, 101] = -np.inf
    x[:, 102] = 0.0
    x[:, 103] = -0.0
    case = dict(V=V, dtype="f32", logits=torch.from_numpy(x))
    hist = history(rng, B, V, 200)
    hist[:, :4] = [100, 101, 102, 103]
    hist[:, 4] = V + 2  # inside the padded row, but past V: padding
    pen = np.full(B, 1.25, np.float32)
    got, st, want, wst = run_both(case, hist, pen)
    assert np.all(st == 0) and np.all(wst == 0)
    assert_same(got, want, "f32")
    assert np.array_equal(got[:, V:].view(np.uint32), x[:, V:].view(np.uint32))
    # H = 0: statuses only, nothing changes
    got, st, want, wst = run_both(case, np.zeros((B, 0), np.int32), pen)
    assert np.all(st == 0) and np.array_equal(got.view(np.uint32), x.view(np.uint32))


def test_largest_vocabulary():
    rng = np.random.Generator(np.random.PCG64(6))
    B, V = 3, 1 << 20
    case = workloads.random_case(77, B, V, dtype="bf16", n_head=(0, 8))
    hist = history(rng, B, V, 4096)
    got, st, want, wst = run_both(case, hist, np.array([1.2, 1.5, 3.0], np.float32))
    assert np.all(st == 0)
    assert_same(got, want, "bf16")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_penalty_then_sample_matches_oracle(dtype):
    """The processor's place in the pipeline: penalty, then the sampler, on
    both sides."""
    rng = np.random.Generator(np.random.PCG64(7 + len(dtype)))
    case = workloads.random_case(900 + len(dtype), 32, 20000, dtype=dtype, mask_frac=0.2,
                                 temps=(0.0, 0.7, 1.0), topks=(1, 20, 50, 1000, 20000),
                                 topps=(0.8, 0.95, 1.0))
    # the history holds the head: the penalty moves the kept sets
    x = workloads.bits_numpy(case["logits"])
    xv = x if dtype == "f32" else torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().numpy()
    top = np.argsort(-xv, axis=1)[:, :64].astype(np.int32)
    hist = np.concatenate([top, history(rng, 32, 20000, 64)], axis=1)
    pen = np.full(32, 1.5, np.float32)
    s = H.sampler()
    d = H.to_dev(case)
    st = s.repetition_penalty(d["logits"], torch.as_tensor(hist).cuda(), torch.as_tensor(pen).cuda())
    torch.cuda.synchronize()
    assert int(st.abs().sum()) == 0
    pen_bits, _ = oracle.repetition_penalty(x, dtype, 20000, hist, pen)
    pcase = dict(case)
    pcase["logits"] = d["logits"].cpu()
    assert np.array_equal(workloads.bits_numpy(pcase["logits"]).view(np.uint8),
                          pen_bits.view(np.uint8))
    g = H.gpu_run(pcase, mode="sample")
    r = H.oracle_run(pcase)
    H.compare(pcase, g, r, mode="sample")


def test_call_level_errors():
    s = H.sampler()
    L = s.lib
    dev = torch.device("cuda", 0)
    lg = torch.zeros((2, 64), device=dev)
    hist = torch.zeros((2, 4), dtype=torch.int32, device=dev)
    pen = torch.ones(2, device=dev)
    st = torch.empty(2, dtype=torch.int32, device=dev)
    P = binding._ptr
    assert L.smp_repetition_penalty(s.h, P(lg), 0, 2, 64, 64, P(hist), 4, 4, P(pen), P(st),
                                    None) == 0
    torch.cuda.synchronize()
    assert L.smp_repetition_penalty(s.h, P(lg), 0, 2, 64, 63, P(hist), 4, 4, P(pen), P(st),
                                    None) == 3              # ld < V
    assert L.smp_repetition_penalty(s.h, P(lg), 0, 2, 64, 64, None, 4, 4, P(pen), P(st),
                                    None) == 3              # NULL history with H > 0
    assert L.smp_repetition_penalty(s.h, P(lg), 0, 2, 64, 64, P(hist), 4, 3, P(pen), P(st),
                                    None) == 3              # history_ld < H
    assert L.smp_repetition_penalty(s.h, P(lg), 7, 2, 64, 64, P(hist), 4, 4, P(pen), P(st),
                                    None) == 3              # unknown dtype
    assert L.smp_repetition_penalty(s.h, P(lg), 0, 2, 64, 64, P(hist), 4, 4, P(pen), None,
                                    None) == 3              # NULL row_status
