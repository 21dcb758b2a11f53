"""Checks that pin the repetition-penalty oracle and its float encoders.

The rule (a reading: the "Sampling system design" post leaves the formula
open and names positive and negative logits as the point where frameworks
differ) is the CTRL rule of Keskar et al. 2019: for every distinct token of
the history, x / theta if x > 0, else x * theta.  The checks use worked
values with closed forms, duplicates and padding in the history, invalid
penalties, and the encoders against numpy / torch casts (both round to
nearest, ties to even).  Each check takes an oracle library handle ``L``.
"""
import numpy as np
import torch

import oracle


def _bits_to_f32(bits):
    return np.asarray(bits, dtype=np.uint32).view(np.float32)


def check_encoders(L=None, n=60000):
    rng = np.random.Generator(np.random.PCG64(31))
    bits = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    # values near the rounding points of both formats, the f16 range edges
    # and its subnormals
    extra = np.array([1.0, -1.0, 0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e-8, 2.0**-24,
                      2.0**-25, 3 * 2.0**-26, 2.0**-14, 2.0**-14 - 2.0**-25, 6.1e-5, np.inf,
                      -np.inf, 1.00390625, 1.001953125, 1.0009765625, 1.00048828125],
                     dtype=np.float32)
    halves = (rng.integers(0, 2**16, size=4000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000
    vals = np.concatenate([_bits_to_f32(bits), extra, _bits_to_f32(halves)])
    want_bf = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    with np.errstate(over="ignore"):  # values past the f16 range become infinities
        want_h = vals.astype(np.float16).view(np.uint16)
    for v, wb, wh in zip(vals, want_bf, want_h):
        gb = oracle.f32_to_bf16(v, L=L)
        gh = oracle.f32_to_f16(v, L=L)
        if np.isnan(v):
            assert (gb & 0x7fff) > 0x7f80 and (gh & 0x7fff) > 0x7c00, (v, gb, gh)
            continue
        assert gb == wb, (float(v), hex(gb), hex(wb))
        assert gh == wh, (float(v), hex(gh), hex(wh))


def check_penalty_worked_values(L=None):
    V = 8
    x = np.array([[2.0, -2.0, 0.0, -np.inf, 3.0, 8.0, -0.5, 1.5]], dtype=np.float32)
    hist = np.array([[0, 1, 2, 3, 5, 5, 5, -1, 8, 6]], dtype=np.int32)
    out, st = oracle.repetition_penalty(x, "f32", V, hist, [2.0], L=L)
    assert st[0] == 0
    # positive logits are divided, the others multiplied; 5 appears three times
    # and is penalised once; -1 and 8 (= V) are padding; 4 and 7 are not in
    # the history
    want = np.array([1.0, -4.0, 0.0, -np.inf, 3.0, 4.0, -1.0, 1.5], dtype=np.float32)
    assert np.array_equal(out[0], want), out
    # a penalty of 1 changes nothing
    out, st = oracle.repetition_penalty(x, "f32", V, hist, [1.0], L=L)
    assert np.array_equal(out, x) and st[0] == 0
    # invalid penalties leave the row unchanged and mark it
    for bad in (0.0, -1.5, np.nan, np.inf):
        out, st = oracle.repetition_penalty(x, "f32", V, hist, [bad], L=L)
        assert st[0] == oracle.ORC_INVALID and np.array_equal(out, x)


def check_penalty_vs_numpy(L=None):
    """Random rows in the three storage formats against numpy float32
    arithmetic and numpy / torch round-to-nearest-even casts."""
    rng = np.random.Generator(np.random.PCG64(32))
    B, V, H = 6, 300, 80
    x = (rng.standard_normal((B, V)) * 4).astype(np.float32)
    hist = rng.integers(-5, V + 5, size=(B, H)).astype(np.int32)
    pen = np.array([1.0, 1.1, 1.3, 2.0, 0.8, 1.05], dtype=np.float32)
    for dtype in ("f32", "bf16", "f16"):
        if dtype == "f32":
            stored = x
            vals = x.copy()
        elif dtype == "bf16":
            t = torch.from_numpy(x).to(torch.bfloat16)
            stored = t.view(torch.int16).numpy().view(np.uint16)
            vals = t.float().numpy()
        else:
            h = x.astype(np.float16)
            stored = h.view(np.uint16)
            vals = h.astype(np.float32)
        out, st = oracle.repetition_penalty(stored, dtype, V, hist, pen, L=L)
        assert np.all(st == 0)
        want = vals.copy()
        for r in range(B):
            ids = np.unique(hist[r][(hist[r] >= 0) & (hist[r] < V)])
            v = vals[r, ids]
            want[r, ids] = np.where(v > 0, v / pen[r], v * pen[r]).astype(np.float32)
        if dtype == "f32":
            got = out
        elif dtype == "bf16":
            want = torch.from_numpy(want).to(torch.bfloat16).view(torch.int16).numpy()
            got = out.view(np.int16)
        else:
            want = want.astype(np.float16).view(np.uint16)
            got = out
        assert np.array_equal(got, want), dtype


PENALTY_CHECKS = [check_penalty_worked_values, check_penalty_vs_numpy, check_encoders]
