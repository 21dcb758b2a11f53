"""The CPU oracle against facts fixed outside it (no GPU needed)."""
import numpy as np
import pytest

import oracle
import pins


def test_worked_examples():
    pins.check_worked_examples()


def test_dyadic_exact_boundary():
    pins.check_dyadic_boundary()


def test_order_negative_controls():
    pins.check_order_negative_controls()


def test_greedy_tie_earliest_id():
    pins.check_greedy_tie()


def test_mask_bit_order():
    pins.check_mask_bit_order()


def test_status_codes():
    pins.check_status_codes()


def test_decoders_all_patterns():
    pins.check_decoders()


def test_philox_matches_curand_host_generator():
    if not pins.check_philox_vs_curand():
        pytest.skip("libcurand not available")


def test_uniformity():
    pins.check_uniformity()


def test_bruteforce_tiny_vocab():
    pins.check_bruteforce()


def test_exhaustive_masks():
    pins.check_exhaustive_masks()


def test_sampler_intervals():
    pins.check_sampler_intervals()


def test_frequencies_and_gumbel_max():
    pins.check_frequencies_and_gumbel()


def test_temperature_limit():
    pins.check_temperature_limit()


def test_invariants_random_rows():
    """Kept top-k count = min(k, |L|) when p = 1, kept set is a rank prefix,
    probabilities sum to 1."""
    from top_selection_stats_gb300 import workloads
    case = workloads.random_case(3, 64, 300, topps=(1.0,), temps=(0.7, 1.0), mask_frac=0.3)
    x = workloads.bits_numpy(case["logits"])
    bm = None if case["bitmask"] is None else case["bitmask"].numpy().view(np.uint32)
    r = oracle.run_batch(x, "f32", 300, temperature=case["temperature"].numpy(),
                         top_k=case["top_k"].numpy(), top_p=case["top_p"].numpy(),
                         bitmask=bm, want_probs=True)
    for b in range(64):
        legal = np.ones(300, bool) if bm is None else np.array(
            [(bm[b, j >> 5] >> (j & 31)) & 1 for j in range(300)], bool)
        legal &= ~(np.isinf(x[b]) & (x[b] < 0))
        nl = int(legal.sum())
        assert r["kept_count"][b] == min(int(case["top_k"][b]), nl)
        kept = np.array([(r["kept_mask"][b, j >> 5] >> (j & 31)) & 1 for j in range(300)], bool)
        if kept.any():
            lo = x[b][kept].min()
            assert not np.any(legal & ~kept & (x[b] > lo))
        assert abs(r["probs"][b].sum() - 1.0) < 1e-12


