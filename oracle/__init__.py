"""CPU oracle for batched top-k / top-p truncation and sampling.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA library (``top_selection_stats_gb300``) and never imports it.

The arithmetic lives in ``oracle.c`` (plain C, double precision after the fp32
temperature division); this module only marshals numpy arrays.

Parity status of each function (what pins it is listed in the tests):
  * orc_select_core  -- pinned: worked examples of the KB note (section 02-03),
                        lecture exercises 7 and 8, O(V^2) brute force.
  * orc_batch        -- pinned through orc_select_core plus decoder and
                        front-end tests (greedy ties, masks, status codes).
  * orc_philox4x32_10 -- pinned against cuRAND's host Philox4x32-10 generator
                        where libcurand is present, and by uniformity tests.
  * orc_repetition_penalty, orc_f32_to_bf16, orc_f32_to_f16 -- pinned by
                        worked values of the CTRL rule, duplicates and padding
                        in the history, and the encoders against numpy / torch
                        round-to-nearest-even casts over many values.
  * top_logprobs (numpy, on the oracle's outputs) -- pinned by a worked
                        example and the normalisation of a whole kept set.
  * orc_gumbel_sample -- pinned by its frequencies against the exact softmax
                        of the kept set (the lecture's Gumbel-max identity),
                        greedy at T = 0, statuses and the uniform's range.
  * orc_spec_verify_u / orc_spec_verify -- the rule over the reals (double
                        residual, compensated sums); pinned by the exact
                        output distribution (it equals the target's, the
                        identity of the lecture notes' section 5.2), the
                        acceptance rate sum(min(p, q)), special cases (p == q,
                        disjoint supports) and Philox frequencies.
  * orc_spec_verify_fx_u (fixed=True) -- a second, labelled variant in the
                        CUDA library's stated integer precision; pinned by
                        agreement with the real-number rule wherever u * S
                        lies more than 1e-9 of S from a switch point.
"""
import ctypes
import os

import numpy as np

from . import build as _build

ORC_OK, ORC_EMPTY, ORC_NONFINITE, ORC_INVALID = 0, 1, 2, 3
ORC_F32, ORC_BF16, ORC_F16 = 0, 1, 2
FLAG_TOPP_BOUNDARY, FLAG_CDF_BOUNDARY = 1, 2

_lib = None


def load(path):
    """Load an oracle shared library from ``path`` and declare its signatures."""
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    L.orc_bf16_to_f32.restype = ctypes.c_float
    L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_f16_to_f32.restype = ctypes.c_float
    L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_philox4x32_10.restype = None
    L.orc_philox4x32_10.argtypes = [P, P, P]
    L.orc_uniform.restype = ctypes.c_double
    L.orc_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
    L.orc_select_core.restype = ctypes.c_int
    L.orc_select_core.argtypes = [ctypes.c_int, P, P, P, ctypes.c_int32, ctypes.c_double,
                                  ctypes.c_double, P, P, P, P, P, P]
    L.orc_batch.restype = ctypes.c_int
    L.orc_batch.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, P,
                            P, P, P, P, P, ctypes.c_int, P, P, P, P, P, P, P, ctypes.c_int]
    L.orc_spec_verify_u.restype = ctypes.c_int
    L.orc_spec_verify_u.argtypes = [ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int64, P, P, P,
                                    P, P, P]
    L.orc_spec_verify_fx_u.restype = ctypes.c_int
    L.orc_spec_verify_fx_u.argtypes = [ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int64, P, P,
                                       P, P, P]
    L.orc_spec_verify.restype = ctypes.c_int
    L.orc_spec_verify.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                                  ctypes.c_int64, P, P, P, P, P, P, P, ctypes.c_int,
                                  ctypes.c_int]
    L.orc_f32_to_bf16.restype = ctypes.c_uint16
    L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
    L.orc_f32_to_f16.restype = ctypes.c_uint16
    L.orc_f32_to_f16.argtypes = [ctypes.c_float]
    L.orc_repetition_penalty.restype = ctypes.c_int
    L.orc_repetition_penalty.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int64, P, ctypes.c_int, ctypes.c_int64, P, P]
    L.orc_gumbel_uniform.restype = ctypes.c_double
    L.orc_gumbel_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int]
    L.orc_gumbel_sample.restype = ctypes.c_int
    L.orc_gumbel_sample.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                    P, P, P, P, P, P, P, ctypes.c_int]
    return L


def lib():
    """The oracle library, built from source on first use."""
    global _lib
    if _lib is None:
        _lib = load(_build.build())
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def philox4x32_10(ctr, key, L=None):
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    (L or lib()).orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed, offset, L=None):
    return (L or lib()).orc_uniform(int(seed) & (2**64 - 1), int(offset) & (2**64 - 1))


def select_core(x, z, legal, top_k, top_p, u, L=None):
    """Core selection on double arrays (used by the pins)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    z = np.ascontiguousarray(z, dtype=np.float64)
    legal = np.ascontiguousarray(legal, dtype=np.uint8)
    n = x.shape[0]
    kept = np.zeros(n, dtype=np.uint8)
    prob = np.zeros(n, dtype=np.float64)
    tok = np.zeros(1, dtype=np.int32)
    ntk = np.zeros(1, dtype=np.int32)
    nkp = np.zeros(1, dtype=np.int32)
    fl = np.zeros(1, dtype=np.int32)
    st = (L or lib()).orc_select_core(n, _ptr(x), _ptr(z), _ptr(legal), int(top_k),
                                      float(top_p), float(u), _ptr(kept), _ptr(prob),
                                      _ptr(tok), _ptr(ntk), _ptr(nkp), _ptr(fl))
    return dict(status=st, kept=kept.astype(bool), prob=prob, token=int(tok[0]),
                n_topk=int(ntk[0]), n_kept=int(nkp[0]), flags=int(fl[0]))


_DT = {"f32": ORC_F32, "bf16": ORC_BF16, "f16": ORC_F16}


def run_batch(logits_bits, dtype, V, temperature=None, top_k=None, top_p=None, seed=None,
              offset=None, bitmask=None, mode="sample", want_mask=True, want_probs=False,
              n_threads=1, ld=None, L=None):
    """Run the oracle over a batch.

    logits_bits: numpy array [B, ld] -- float32 for "f32", uint16 bit patterns
    for "bf16" / "f16".  bitmask: uint32 [B, ceil(V/32)] or None.
    Returns a dict of numpy arrays.
    """
    dt = _DT[dtype]
    arr = np.ascontiguousarray(logits_bits)
    if dt == ORC_F32:
        assert arr.dtype == np.float32
    else:
        assert arr.dtype == np.uint16
    B = arr.shape[0]
    ld = arr.shape[1] if ld is None else ld
    W = (V + 31) // 32
    m = 1 if mode == "argmax" else 0

    def arrf(a, dtp, default):
        if a is None:
            return np.full(B, default, dtype=dtp)
        return np.ascontiguousarray(a, dtype=dtp)

    t = arrf(temperature, np.float32, 1.0)
    k = arrf(top_k, np.int32, V)
    p = arrf(top_p, np.float32, 1.0)
    s = arrf(seed, np.uint64, 0)
    o = arrf(offset, np.uint64, 0)
    bm = None if bitmask is None else np.ascontiguousarray(bitmask, dtype=np.uint32)
    status = np.zeros(B, dtype=np.int32)
    token = np.zeros(B, dtype=np.int32)
    count = np.zeros(B, dtype=np.int32)
    flags = np.zeros(B, dtype=np.int32)
    u = np.zeros(B, dtype=np.float64)
    kmask = np.zeros((B, W), dtype=np.uint32) if want_mask else None
    probs = np.zeros((B, V), dtype=np.float64) if want_probs else None
    (L or lib()).orc_batch(_ptr(arr), dt, B, V, ld, _ptr(bm), _ptr(t), _ptr(k), _ptr(p),
                           _ptr(s), _ptr(o), m, _ptr(status), _ptr(token), _ptr(count),
                           _ptr(kmask), _ptr(probs), _ptr(flags), _ptr(u), int(n_threads))
    return dict(status=status, token=token, kept_count=count, kept_mask=kmask, probs=probs,
                flags=flags, u=u)


def spec_verify_u(p, q, d, u_acc, u_res, L=None, fixed=False):
    """One sequence with explicit uniforms.  p: float32 [G+1, V], q: float32
    [G, V], d: int [G], u_acc: [G], u_res: [G+1].  fixed: the labelled
    fixed-point variant instead of the real-number rule.  Returns a dict."""
    p = np.ascontiguousarray(p, dtype=np.float32)
    G1, V = p.shape
    G = G1 - 1
    q = np.ascontiguousarray(q if G else np.zeros((1, V)), dtype=np.float32)
    d = np.ascontiguousarray(d if G else [0], dtype=np.int32)
    ua = np.ascontiguousarray(u_acc if G else [0.0], dtype=np.float64)
    ur = np.ascontiguousarray(u_res, dtype=np.float64)
    out = np.zeros(G + 1, dtype=np.int32)
    n = np.zeros(1, dtype=np.int32)
    mg = np.zeros(1, dtype=np.float64)
    if fixed:
        st = (L or lib()).orc_spec_verify_fx_u(G, V, _ptr(p), _ptr(q), V, _ptr(d), _ptr(ua),
                                               _ptr(ur), _ptr(out), _ptr(n))
        mg[0] = np.inf
    else:
        st = (L or lib()).orc_spec_verify_u(G, V, _ptr(p), _ptr(q), V, _ptr(d), _ptr(ua),
                                            _ptr(ur), _ptr(out), _ptr(n), _ptr(mg))
    return dict(status=st, tokens=out, n_accepted=int(n[0]), margin=float(mg[0]))


def spec_verify(p, q, d, seed, offset, V=None, n_threads=1, L=None, fixed=False):
    """Batch with Philox uniforms.  p: float32 [B, G+1, ld], q: float32
    [B, G, ld], d: int32 [B, G]; seed, offset: uint64 [B]; V <= ld (default
    ld).  fixed: the labelled fixed-point variant (margin = inf)."""
    p = np.ascontiguousarray(p, dtype=np.float32)
    B, G1, ld = p.shape
    G = G1 - 1
    V = ld if V is None else V
    q = np.ascontiguousarray(q if G else np.zeros((B, 1, ld)), dtype=np.float32)
    d = np.ascontiguousarray(d if G else np.zeros((B, 1)), dtype=np.int32)
    s = np.ascontiguousarray(seed, dtype=np.uint64)
    o = np.ascontiguousarray(offset, dtype=np.uint64)
    out = np.zeros((B, G + 1), dtype=np.int32)
    n = np.zeros(B, dtype=np.int32)
    st = np.zeros(B, dtype=np.int32)
    mg = np.zeros(B, dtype=np.float64)
    (L or lib()).orc_spec_verify(B, G, V, _ptr(p), _ptr(q), ld, _ptr(d), _ptr(s), _ptr(o),
                                 _ptr(out), _ptr(n), _ptr(st), _ptr(mg), int(bool(fixed)),
                                 int(n_threads))
    return dict(status=st, tokens=out, n_accepted=n, margin=mg)


def repetition_penalty(logits_bits, dtype, V, history, penalty, L=None):
    """Returns a penalised copy of logits_bits (float32 values or uint16
    bit patterns, [B, ld]) and the per-row statuses.  history: int32 [B, H]
    (entries outside [0, V) are padding); penalty: float32 [B]."""
    out = np.array(logits_bits, copy=True, order="C")
    B, ld = out.shape
    h = np.ascontiguousarray(history, dtype=np.int32)
    H = h.shape[1] if h.ndim == 2 else 0
    pen = np.ascontiguousarray(penalty, dtype=np.float32)
    st = np.zeros(B, dtype=np.int32)
    (L or lib()).orc_repetition_penalty(_ptr(out), _DT[dtype], B, V, ld, _ptr(h), H, H,
                                        _ptr(pen), _ptr(st))
    return out, st


def f32_to_bf16(x, L=None):
    return (L or lib()).orc_f32_to_bf16(float(x))


def f32_to_f16(x, L=None):
    return (L or lib()).orc_f32_to_f16(float(x))


def gumbel_uniform(seed, offset, i, L=None):
    return (L or lib()).orc_gumbel_uniform(int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                           int(i))


def gumbel_sample(logits_bits, dtype, V, temperature, seed, offset, kept_mask=None, ld=None,
                  n_threads=1, L=None):
    """Gumbel-max draw per row; returns dict(token, status, margin)."""
    arr = np.ascontiguousarray(logits_bits)
    B = arr.shape[0]
    ld = arr.shape[1] if ld is None else ld
    km = None if kept_mask is None else np.ascontiguousarray(kept_mask, dtype=np.uint32)
    t = np.ascontiguousarray(temperature, dtype=np.float32)
    s = np.ascontiguousarray(seed, dtype=np.uint64)
    o = np.ascontiguousarray(offset, dtype=np.uint64)
    tok = np.zeros(B, dtype=np.int32)
    st = np.zeros(B, dtype=np.int32)
    mg = np.zeros(B, dtype=np.float64)
    (L or lib()).orc_gumbel_sample(_ptr(arr), _DT[dtype], B, V, ld, _ptr(km), _ptr(t), _ptr(s),
                                   _ptr(o), _ptr(tok), _ptr(st), _ptr(mg), int(n_threads))
    return dict(token=tok, status=st, margin=mg)


def top_logprobs(x, kept, probs, status, n):
    """The n most likely tokens of each row's final kept set and their
    log-probabilities, from the oracle's own outputs: x float [B, V] (the
    logits as values), kept bool [B, V], probs [B, V] (final probabilities),
    status [B].  Ranked by logit descending, smallest id first among equal
    logits; slots past the kept set get id -1 and -inf, error rows -1 and
    NaN."""
    B, V = x.shape
    ids = np.full((B, n), -1, dtype=np.int32)
    lps = np.full((B, n), -np.inf)
    for r in range(B):
        if status[r] != ORC_OK:
            lps[r] = np.nan
            continue
        cand = np.nonzero(kept[r])[0]
        order = cand[np.lexsort((cand, -x[r, cand].astype(np.float64)))][:n]
        ids[r, :len(order)] = order
        lps[r, :len(order)] = np.log(probs[r, order])
    return ids, lps


def bf16_to_f32(bits):
    return lib().orc_bf16_to_f32(int(bits))


def f16_to_f32(bits):
    return lib().orc_f16_to_f32(int(bits))


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
