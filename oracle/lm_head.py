"""LM head of the verify step, fp64 on the CPU (test infrastructure).

Page 2 §1.2 argues that decoding is bound by the weights and logit rows it
moves; the verify step's logits are an LM head's output: for each new row r
with hidden state h_r (the last hidden layer's output, any normalisation
already applied) and the head's weight matrix W (one row of H weights per
vocabulary entry), z[r, v] = sum_k h_r[k] * W[v, k].  The oracle is that
definition in fp64 from the given (bf16-valued) inputs.

Pinned by tests/test_oracle_lm_head.py against closed forms (one-hot hidden
states select weight columns, a hand-computed 2 x 3 case, linearity).
"""
from __future__ import annotations

import numpy as np


def oracle_lm_head(hidden: np.ndarray, weight: np.ndarray) -> np.ndarray:
    """z[..., v] = sum_k hidden[..., k] * weight[v, k], fp64."""
    h = np.asarray(hidden, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    return np.einsum("...k,vk->...v", h, w)
