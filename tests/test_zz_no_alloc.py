"""smp_sample_noalloc, the sampling call that allocates nothing, against smp_sample.

Some callers may not call cudaMalloc. One example is a plugin inside a serving
runtime that has reserved the device's memory for its own pool. For them the
library offers one sampling call whose scratch (the job board) is a static
device array rather than a handle's workspace. This file's name makes pytest
collect it last, so a failure here never stops a run before the other tests.
"""
import os
import shutil

import pytest
import torch

from top_selection_stats_gb300 import Sampler, SmpError, binding, workloads
from top_selection_stats_gb300.binding import SMP_ERR_CAPACITY, SMP_ERR_INVALID_PARAM


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    from top_selection_stats_gb300 import build
    build.build()
    return binding.load_library()


def test_noalloc_rejects_bad_arguments_before_any_device_work(lib):
    # every check below returns before the first CUDA call, so no GPU is needed
    assert lib.smp_sample_noalloc(None, 1, 1, 8, 8, None, None, None, None, None, None,
                                  None) == SMP_ERR_INVALID_PARAM
    params = binding.RowParams(1, 1, 1, 1, 1)
    assert lib.smp_sample_noalloc(1, 7, 1, 8, 8, None, params, 1, 1, None, None,
                                  None) == SMP_ERR_INVALID_PARAM
    assert lib.smp_sample_noalloc(1, 1, 1, 8, 4, None, params, 1, 1, None, None,
                                  None) == SMP_ERR_INVALID_PARAM


def _outputs(B, V, dev):
    W = workloads.n_words(V)
    return dict(tokens=torch.full((B,), -7, dtype=torch.int32, device=dev),
                status=torch.full((B,), -7, dtype=torch.int32, device=dev),
                kept_mask=torch.full((B, W), -7, dtype=torch.int32, device=dev),
                kept_count=torch.full((B,), -7, dtype=torch.int32, device=dev))


def _noalloc(case, out):
    return binding.sample_noalloc(case["logits"], case["temperature"], case["top_k"],
                                  case["top_p"], case["seed"], case["offset"], out["tokens"],
                                  out["status"], bitmask=case["bitmask"],
                                  kept_mask=out["kept_mask"], kept_count=out["kept_count"])


@pytest.mark.gpu
def test_noalloc_matches_smp_sample_on_two_calls_in_a_row():
    # The mixed batch has flat top-p rows whose second pass goes through the
    # job board; the second call (another shape, grammar masks, ties) must
    # find the board as the first call left it: cleared.
    dev = torch.device("cuda", 0)
    cases = [workloads.make("mixed256x128256_bf16", device="cuda"),
             workloads.make("ties512x151936_bf16", device="cuda")]
    got = []
    for case in cases:  # two calls in a row, before any handle exists
        out = _outputs(case["B"], case["V"], dev)
        _noalloc(case, out)
        got.append(out)
    torch.cuda.synchronize()
    s = Sampler(0, max_batch=4096, max_vocab=1 << 20)
    for case, out in zip(cases, got):
        ref = s.sample(case["logits"], case["temperature"], case["top_k"], case["top_p"],
                       case["seed"], case["offset"], bitmask=case["bitmask"], want_mask=True)
        torch.cuda.synchronize()
        # same kernel, same inputs: integer outputs agree exactly
        for k in ("status", "tokens", "kept_count", "kept_mask"):
            assert torch.equal(out[k], ref[k]), (case["name"], k)
        assert (out["status"] == 0).sum().item() >= case["B"] - 1, case["name"]
    s.close()


@pytest.mark.gpu
def test_noalloc_rejects_vocabulary_beyond_its_scratch():
    # one more token than 128 staging chunks of bf16; the buffers are real and
    # large enough, but the call must refuse before launching anything
    V = 128 * 12288 + 1
    dev = torch.device("cuda", 0)
    case = dict(logits=torch.zeros((1, V), dtype=torch.bfloat16, device=dev), bitmask=None,
                temperature=torch.ones(1, device=dev),
                top_k=torch.full((1,), 50, dtype=torch.int32, device=dev),
                top_p=torch.full((1,), 0.9, device=dev),
                seed=torch.zeros(1, dtype=torch.int64, device=dev),
                offset=torch.zeros(1, dtype=torch.int64, device=dev))
    out = _outputs(1, V, dev)
    with pytest.raises(SmpError) as e:
        _noalloc(case, out)
    assert e.value.code == SMP_ERR_CAPACITY
    torch.cuda.synchronize()
    assert out["status"].item() == -7 and out["tokens"].item() == -7
