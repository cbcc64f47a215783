"""The parity comparison's own rules, on the CPU (no GPU, no oracle)."""
import numpy as np
import pytest
import torch

from tests.parity_util import P_ROUND, compare, half_ulp_bf16


def _bf16(x):
    return torch.tensor(x, dtype=torch.float64).to(torch.bfloat16)


def test_bound_accepts_weight_rounding_and_rejects_more():
    # O_ref = 0.5 with sum_j w_j |v_j| = 5 (dominant weights on large |v| of
    # opposite signs): the weight rounding allows 1/2 ulp + P_ROUND * 5 =
    # 0.0227, beyond 1e-2 raw.  GPU values below sit on the bf16 grid
    # (spacing 2^-8 in [0.5, 1)).
    o_ref = np.array([[0.5]])
    lse_ref = np.array([3.0])
    st = compare(_bf16([[0.5 + 3 * 2.0 ** -8]]), torch.tensor([3.0]), o_ref, lse_ref, "within",
                 absv_ref=np.array([[5.0]]))
    assert st["o_max_over_bound"] <= 0.0 and st["o_max_abs"] > 1e-2
    # With sum_j w_j |v_j| = 0.5 the bound is 1/2 ulp + P_ROUND / 2 = 0.0040:
    # an error of 2 grid steps (0.0078) passes the 1e-2 rules but not the
    # bound.
    with pytest.raises(AssertionError):
        compare(_bf16([[0.5 + 2 * 2.0 ** -8]]), torch.tensor([3.0]), o_ref, lse_ref, "beyond",
                absv_ref=np.array([[0.5]]))


def test_without_bound_raw_rule_applies_below_two():
    # |O_ref| in [1, 2): an error of 0.0116 is within 1/2 ulp (0.0039) + 1e-2
    # but not within 1e-2 raw.
    o_ref = np.array([[1.004]])
    lse_ref = np.array([0.0])
    with pytest.raises(AssertionError):
        compare(_bf16([[1.015625]]), torch.tensor([0.0]), o_ref, lse_ref, "raw")
    compare(_bf16([[1.0078125]]), torch.tensor([0.0]), o_ref, lse_ref, "raw ok")


def test_masked_rows_must_be_plus_zero_and_minus_inf():
    o_ref = np.zeros((1, 2))
    lse_ref = np.array([-np.inf])
    compare(torch.zeros((1, 2), dtype=torch.bfloat16), torch.tensor([-np.inf]), o_ref, lse_ref)
    with pytest.raises(AssertionError):
        compare(torch.tensor([[-0.0, 0.0]], dtype=torch.bfloat16), torch.tensor([-np.inf]),
                o_ref, lse_ref)


def test_bound_takes_the_ulp_of_the_rounded_output():
    # An exact value just below 2 whose kernel value (within P_ROUND * 0.5
    # of it) rounds up to the bf16 grid above 2, where the spacing doubles:
    # the rounding may move it by half an ulp of [2, 4), 2^-8, not of [1, 2).
    o_ref = np.array([[1.9990]])
    st = compare(_bf16([[2.0078125]]), torch.tensor([1.0]), o_ref, np.array([1.0]), "crossing",
                 absv_ref=np.array([[0.5]]))
    assert st["o_max_over_bound"] <= 0.0
