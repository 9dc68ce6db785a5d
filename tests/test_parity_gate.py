"""The forward parity gate itself (tests/parity.py), on hand-made values:
what it accepts and what it rejects, so that a change to it that loosens the
target's tolerance shows up here."""
import numpy as np
import pytest
import torch

from tests.parity import compare, round_to, ulp, workload_rows

BF, FP = torch.bfloat16, torch.float16


def run(g, r, dtype=BF):
    # padded with exact elements so that only the max-abs part of the gate is
    # exercised (the mean-abs part has its own test)
    pad = np.full(10000, 0.25)
    g = np.concatenate([np.asarray(g, np.float64), pad])
    r = np.concatenate([np.asarray(r, np.float64), pad])
    return compare(g, r, None, None, dtype, "t")


def test_within_the_flat_gate_passes():
    st = run([0.5, -1.25], [0.5 + 0.009, -1.25 - 0.0099])
    assert st["n_over_gate"] == 0


def test_flat_gate_applies_below_two_in_bf16():
    # half an ulp at 1.5 is 2^-8: no allowance, 0.0101 fails
    with pytest.raises(AssertionError):
        run([1.5], [1.5 + 0.0101])


def test_output_rounding_allowance_at_bf16_four_to_eight():
    # exact 4.0 + 0.0155 rounds to 4.0 (spacing 2^-5 there): an exact kernel
    # delivers 4.0, 0.0155 away from the oracle, which the allowance explains
    r = 4.0 + 0.0155
    assert round_to(np.array([r]), BF)[0] == 4.0
    st = run([4.0], [r])
    assert st["n_over_gate"] == 1


def test_allowance_rejects_errors_beyond_rounding():
    # 4.03125 is the next bf16 above 4.0; the oracle at 4.0 + 0.0001 is
    # 0.031 away from it: no value within 1e-2 of the oracle rounds there
    with pytest.raises(AssertionError):
        run([4.03125], [4.0001])
    # two ulps from the rounded oracle at [2, 4) (spacing 2^-6)
    with pytest.raises(AssertionError):
        run([2.0 + 3 * 2 ** -6], [2.0 + 2 ** -6 + 0.004])


def test_fp16_allowance_starts_at_sixteen():
    with pytest.raises(AssertionError):
        run([8.0], [8.0105], FP)
    st = run([16.0], [16.0 + 0.0155], FP)
    assert st["n_over_gate"] == 1


def test_mean_gate():
    g = np.full(100, 0.5)
    compare(g + 0.0009, g, None, None, BF, "mean")
    with pytest.raises(AssertionError):
        compare(g + 0.002, g, None, None, BF, "mean")


def test_lse_gate():
    o = np.zeros(4)
    compare(o, o, np.zeros(4) + 9e-4, np.zeros(4), BF, "lse")
    with pytest.raises(AssertionError):
        compare(o, o, np.zeros(4) + 1.1e-3, np.zeros(4), BF, "lse")


def test_ulp_values():
    assert ulp(np.array([1.0]), BF)[0] == 2.0 ** -7
    assert ulp(np.array([3.0]), BF)[0] == 2.0 ** -6
    assert ulp(np.array([1.0]), FP)[0] == 2.0 ** -10
    assert ulp(np.array([0.0]), FP)[0] == 2.0 ** -24


def test_workload_rows_plan():
    bh, rows = workload_rows(2, 3, 100, 10, 5)
    # every row of heads 0 and 5, ten distinct rows of each of heads 1..4
    for h in (0, 5):
        assert sorted(rows[bh == h].tolist()) == list(range(100))
    for h in range(1, 5):
        r = rows[bh == h]
        assert len(r) == 10 and len(set(r.tolist())) == 10
    assert rows.min() >= 0 and rows.max() < 100
