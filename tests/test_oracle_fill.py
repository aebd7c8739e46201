"""Pins of the residual-fill oracle (oracle/residual_fill.py).

The bf16 rounding is pinned against a library routine that rounds the same way
(torch's fp32 -> bfloat16 conversion, round to nearest even) on fp32-exact values and
against hand-worked halfway cases; the product is pinned by its definition on one-hot
rows, by linearity, and by a small hand-computed case.
"""
import numpy as np
import torch

from oracle.residual_fill import bf16_round, residual_rows, residual_rows_bf16, rounding_bound


def test_bf16_round_matches_torch_on_fp32_values():
    g = torch.Generator().manual_seed(4)
    v32 = torch.cat([torch.randn(20000, generator=g) * 10 ** torch.randint(-8, 8, (20000,), generator=g).float(),
                     torch.tensor([1.0, -1.0, 0.0, 3.0, 255.0, 257.0, 1e-30])])
    want = v32.to(torch.bfloat16).to(torch.float64).numpy()
    got = bf16_round(v32.to(torch.float64).numpy())
    assert np.array_equal(got, want)


def test_bf16_round_halfway_cases_go_to_even():
    # bf16 keeps 8 significant bits: between 1 and 2 the spacing is 2^-7
    assert bf16_round(np.array([1 + 2 ** -8]))[0] == 1.0                  # halfway, 1.0 is even
    assert bf16_round(np.array([1 + 3 * 2 ** -8]))[0] == 1 + 2 ** -6      # halfway, round up to even
    assert bf16_round(np.array([1 + 2 ** -8 + 2 ** -40]))[0] == 1 + 2 ** -7  # just above halfway
    assert bf16_round(np.array([-(1 + 3 * 2 ** -8)]))[0] == -(1 + 2 ** -6)
    assert bf16_round(np.array([257.0]))[0] == 256.0                      # 257 = 256 + half of 2
    assert bf16_round(np.array([0.0]))[0] == 0.0


def test_residual_rows_one_hot_and_hand_case():
    rng = np.random.default_rng(2)
    A = rng.standard_normal((3, 2, 16, 10))
    x = np.eye(10)[[4, 7]]                                  # tokens pick hidden units 4 and 7
    R = residual_rows(x, A)
    assert R.shape == (3, 2, 2, 16)
    assert np.array_equal(R[:, 0], A[:, :, :, 4]) and np.array_equal(R[:, 1], A[:, :, :, 7])
    x = np.array([[1.0, 2.0]])
    A = np.zeros((1, 2, 16, 2))
    A[0, 0, 0] = [3.0, 4.0]                                 # k row 0: 1*3 + 2*4
    A[0, 1, 5] = [-1.0, 0.5]                                # v row 5: -1 + 1
    R = residual_rows(x, A)
    assert R[0, 0, 0, 0] == 11.0 and R[0, 0, 1, 5] == 0.0 and np.count_nonzero(R) == 1


def test_residual_rows_linear_and_bound_covers_rounding():
    rng = np.random.default_rng(3)
    x1 = rng.integers(-4, 5, (5, 24)).astype(np.float64)
    x2 = rng.integers(-4, 5, (5, 24)).astype(np.float64)
    A = rng.integers(-3, 4, (2, 2, 16, 24)).astype(np.float64)
    assert np.array_equal(residual_rows(x1 + x2, A), residual_rows(x1, A) + residual_rows(x2, A))
    exact = residual_rows(x1, A)
    nz = exact != 0
    assert np.all(np.abs(residual_rows_bf16(x1, A) - exact)[nz] <= rounding_bound(x1, A, exact)[nz])
