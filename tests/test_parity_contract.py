"""The parity contract itself (tests/parity.py), on hand-made rows: the output-unit term of
the forward check admits exactly the final rounding of O and nothing else."""
import numpy as np
import pytest

from parity import check_rows


def test_final_rounding_of_a_large_output_is_admitted():
    # 5.0155 lies in [4, 8), where bf16 values are 2^-5 apart: its nearest bf16 value is 5.0,
    # 0.0155 away, which is more than the 1e-2 bound but within half a unit of the output
    ref = np.array([[5.0155, 0.25, -0.5, 0.125]])
    got = np.array([[5.0, 0.25, -0.5, 0.125]])
    lse = np.zeros(1)
    with pytest.raises(AssertionError):
        check_rows(got, lse, ref, lse, "no output type")
    check_rows(got, lse, ref, lse, "bf16 output", dtype="bf16")
    # fp16 is 2^-8 apart there: half a unit is 0.002, so the same output fails
    with pytest.raises(AssertionError):
        check_rows(got, lse, ref, lse, "fp16 output", dtype="f16")


def test_errors_beyond_the_rounding_still_fail():
    ref = np.array([[0.3, 0.25, -0.5, 0.125]])
    got = ref + np.array([[0.0, 0.011, 0.0, 0.0]])
    lse = np.zeros(1)
    with pytest.raises(AssertionError):
        check_rows(got, lse, ref, lse, "bf16 output", dtype="bf16")
    got = ref.copy()
    with pytest.raises(AssertionError):
        check_rows(got, lse + 2e-3, ref, lse, "LSE", dtype="bf16")
    check_rows(got, lse + 5e-4, ref, lse, "LSE", dtype="bf16")


def test_rows_without_keys_must_be_exact():
    ref = np.zeros((1, 4))
    lse_ref = np.array([-np.inf])
    check_rows(ref, lse_ref, ref, lse_ref, "empty row", dtype="bf16")
    with pytest.raises(AssertionError):
        check_rows(ref + 1e-9, lse_ref, ref, lse_ref, "empty row", dtype="bf16")
    with pytest.raises(AssertionError):
        check_rows(ref, np.array([0.0]), ref, lse_ref, "empty row", dtype="bf16")
