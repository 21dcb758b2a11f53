"""The Gumbel-max oracle against facts fixed outside it (no GPU needed)."""
import pins_gumbel


def test_gumbel_frequencies_follow_softmax_of_kept_set():
    pins_gumbel.check_gumbel_frequencies()


def test_gumbel_greedy_and_status():
    pins_gumbel.check_gumbel_greedy_and_status()


def test_gumbel_uniforms():
    pins_gumbel.check_gumbel_uniforms()


def test_top_logprobs_worked_example():
    pins_gumbel.check_top_logprobs()
