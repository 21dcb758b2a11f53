"""Bounded device waits that run out (smp_set_wait_limit with a bound far
below a copy's latency): every row either completes exactly as it does
without the bound or returns SMP_ERR_TIMEOUT with token -1 and count 0 -- no
substituted token -- and the next call on the same handle, and a call of the
no-allocation entry point, are bit-exact again.  No wait is made to hang:
each one gives up after its bound and the kernel reports the status."""
import numpy as np
import pytest
import torch

from top_selection_stats_gb300 import Sampler, workloads, binding

pytestmark = pytest.mark.gpu

ST_OK, ST_TIMEOUT = 0, 4


def _run(s, d, **kw):
    out = s.sample(d["logits"], d["temperature"], d["top_k"], d["top_p"], d["seed"],
                   d["offset"], bitmask=d["bitmask"], want_mask=True, **kw)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy().copy() for k, v in out.items() if torch.is_tensor(v)}


@pytest.mark.parametrize("kernel", ["board", "split"])
def test_expired_waits_report_timeouts_and_the_next_call_is_clean(kernel):
    s = Sampler(0, max_batch=4096, max_vocab=1 << 20)
    try:
        s.set_kernel(kernel)
        d = workloads.make("mixed256x128256_bf16", device="cuda")
        ref = _run(s, d)
        assert np.all(ref["status"] == ST_OK)
        s.set_wait_limit(200)  # SM cycles: far below a staged copy's latency
        got = _run(s, d)
        st = got["status"]
        assert set(np.unique(st).tolist()) <= {ST_OK, ST_TIMEOUT}, np.unique(st)
        n_to = int((st == ST_TIMEOUT).sum())
        print(f"{kernel}: {n_to} of {len(st)} rows timed out")
        if kernel == "board":
            assert n_to > 0  # the waits for other CTAs' chunks cannot finish in time
        # (the split kernel waits only for its own copies, and the hardware
        # parks its first poll for up to a microsecond, so few or none expire)
        to = st == ST_TIMEOUT
        assert np.all(got["tokens"][to] == -1) and np.all(got["kept_count"][to] == 0)
        ok = ~to
        assert np.array_equal(got["tokens"][ok], ref["tokens"][ok])
        assert np.array_equal(got["kept_count"][ok], ref["kept_count"][ok])
        assert np.array_equal(got["kept_mask"][ok], ref["kept_mask"][ok])
        # the default bound again: the same handle is clean
        s.set_wait_limit(0)
        for _ in range(2):
            again = _run(s, d)
            for k in ("status", "tokens", "kept_count", "kept_mask"):
                assert np.array_equal(again[k], ref[k]), k
        if kernel == "board":
            # the no-allocation entry point (its own board, default bound)
            B, V = d["B"], d["V"]
            tok = torch.empty(B, dtype=torch.int32, device="cuda")
            sta = torch.empty(B, dtype=torch.int32, device="cuda")
            km = torch.empty((B, (V + 31) // 32), dtype=torch.int32, device="cuda")
            kc = torch.empty(B, dtype=torch.int32, device="cuda")
            binding.sample_noalloc(d["logits"], d["temperature"], d["top_k"], d["top_p"],
                                   d["seed"], d["offset"], tok, sta, kept_mask=km,
                                   kept_count=kc)
            torch.cuda.synchronize()
            assert np.array_equal(tok.cpu().numpy(), ref["tokens"])
            assert np.array_equal(sta.cpu().numpy(), ref["status"])
            assert np.array_equal(kc.cpu().numpy(), ref["kept_count"])
    finally:
        s.close()


def test_wait_limit_setter_rejects_no_handle():
    s = Sampler(0, max_batch=8, max_vocab=1024)
    try:
        assert s.lib.smp_set_wait_limit(None, 5) == binding.SMP_ERR_INVALID_PARAM
        s.set_wait_limit(-3)  # restores the default
        s.set_wait_limit(0)
    finally:
        s.close()
