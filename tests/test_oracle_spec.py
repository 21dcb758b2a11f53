"""The speculative-verification oracle against facts fixed outside it (no GPU
needed): the exact output law and acceptance rate of the lecture notes'
section 5.2, special cases and Philox frequencies."""
import pins_spec


def test_spec_special_cases():
    pins_spec.check_spec_special_cases()


def test_spec_status_codes():
    pins_spec.check_spec_status()


def test_spec_output_law_is_target():
    pins_spec.check_spec_output_law()


def test_spec_philox_frequencies():
    pins_spec.check_spec_philox_frequencies()
