"""Residual rows from hidden states: the oracle of the residual fill and of the fused
decode append (test infrastructure only: imported by tests/, never by the package).

ForkKV L2 section 2 Q2: a LoRA projection of hidden state x is x W + x A B, so the
cache can keep x A (rank r = 16) per adapter instead of the full projection; section
3, Figure 6: an agent forked from a prefix fills its own residual pages with the x A
rows of every prefix token.  With A stored as PEFT stores lora_A.weight ([r][hidden]),
residual row k of token t is  sum_i x[t][i] * A[k][i].

The oracle evaluates that sum in fp64 and rounds once to bf16, round to nearest with
ties to even (the storage format of the cache rows); the rounding is written out from
the format's definition (8 significant bits), not through an fp32 intermediate, so no
double rounding enters.
"""
from __future__ import annotations

import numpy as np


def bf16_round(v: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 value (ties to even), returned as fp64.  Normal range only
    (|v| >= 2^-126, finite, below the bf16 overflow threshold) or exact zero."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)                    # v = m * 2^e, 0.5 <= |m| < 1
    q = np.rint(np.ldexp(m, 8))           # 8 significant bits; rint rounds half to even
    return np.ldexp(q, e - 8)


def residual_rows(x: np.ndarray, A: np.ndarray) -> np.ndarray:
    """x [n_tok][hidden], A [n_agents][2][16][hidden] -> [n_agents][n_tok][2][16] fp64 sums."""
    x = np.asarray(x, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    return np.einsum("ti,akri->atkr", x, A)


def residual_rows_bf16(x: np.ndarray, A: np.ndarray) -> np.ndarray:
    return bf16_round(residual_rows(x, A))


def rounding_bound(x: np.ndarray, A: np.ndarray, exact: np.ndarray) -> np.ndarray:
    """Largest |device - exact| a correct device result can have: half a bf16 unit in the last
    place of the exact value, plus the fp32 accumulation error of a length-`hidden` sum of
    products (products of two bf16 values are exact in fp32; each of at most `hidden` fp32
    additions adds at most 2^-24 of the running magnitude, bounded by sum |x_i A_i|), doubled
    for the rounding of that error into the bf16 grid."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    A = np.abs(np.asarray(A, dtype=np.float64))
    hidden = x.shape[-1]
    mag = np.einsum("ti,akri->atkr", x, A)
    _, e = np.frexp(np.abs(exact))
    half_ulp = np.ldexp(np.ones_like(exact), e - 9)
    return half_ulp + 2.0 * hidden * 2.0 ** -24 * mag
