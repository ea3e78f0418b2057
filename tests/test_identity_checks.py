"""The whole-tensor checks the full-size GPU tests apply to every head (exact zero rows, and the
identities sum_t dV_t = sum_r dO_r and sum_t dK_t = sm_scale sum_r (dO_r . (O*_r - O_r)) q_r
within their derived tolerances) are themselves checked on the CPU: the oracle's gradients,
rounded to bf16 as the library returns them, pass them; the same gradients with one kv block's
rows dropped or doubled, or a padded row written, fail them."""
import numpy as np
import pytest
import torch

from block_sparse_video_tok_gb300 import workloads as wl
from tests.parity import (bf16_round, check_zero_rows_and_identities, f64, oracle_backward,
                          oracle_forward)


@pytest.fixture(scope="module")
def oracle_case(oracle):
    case = wl.make_case(1, 2, 64, 16, vbs="ragged33", seed=71, kv_pool=list(range(60)))
    o64, lse64 = oracle_forward(case)
    o_b = bf16_round(o64)
    dq64, dk64, dv64 = oracle_backward(case, f64(o_b), lse64.astype(np.float32).astype(np.float64))
    from oracle import oracle as orc
    _, k2q_num, _ = orc.invert(case["q2k_idx"], case["q2k_num"], case["nb"])
    return case, o_b, bf16_round(dk64), bf16_round(dv64), torch.from_numpy(k2q_num)


def test_oracle_gradients_pass(oracle_case):
    case, o_b, dk, dv, k2q_num = oracle_case
    rdv, rdk = check_zero_rows_and_identities(case, k2q_num, case["q"], case["do"], o_b, dk, dv)
    assert rdv < 0.5 and rdk < 0.5


@pytest.mark.parametrize("mistake", ["drop_dv_block", "double_dk_block", "padded_row_written",
                                     "unselected_block_written"])
def test_planted_mistakes_fail(oracle_case, mistake):
    case, o_b, dk, dv, k2q_num = oracle_case
    dk, dv = dk.clone(), dv.clone()
    j = 5                                       # a selected block
    assert int(k2q_num[0, 1, j]) > 0
    rows = slice(64 * j, 64 * j + int(case["vbs"][j]))
    if mistake == "drop_dv_block":
        dv[0, 1, rows] = 0
    elif mistake == "double_dk_block":
        dk[0, 1, rows] *= 2
    elif mistake == "padded_row_written":
        jj = int(np.flatnonzero(case["vbs"] < 64)[0])
        dv[0, 0, 64 * jj + 63] = dv[0, 0, 64 * jj]
    else:
        dk[0, 0, 64 * 61] = 1.0                 # blocks 60-63 are selected by no q block
    with pytest.raises(AssertionError):
        check_zero_rows_and_identities(case, k2q_num, case["q"], case["do"], o_b, dk, dv)
