"""The repetition-penalty oracle and its float encoders against facts fixed
outside it (no GPU needed)."""
import pins_penalty


def test_penalty_worked_values():
    pins_penalty.check_penalty_worked_values()


def test_penalty_against_numpy():
    pins_penalty.check_penalty_vs_numpy()


def test_encoders_against_numpy_and_torch():
    pins_penalty.check_encoders()
