"""Pins for the oracle's router logits (CPU only): fp32(sum_h x[t,h] wr[e,h])
of bf16 inputs, the router GEMM in front of the routing step.

Hand cases with exact results fix the operand roles (a transposed router
matrix or a shifted index gives another answer); Python's math.fsum (an
exactly rounded sum) recomputes random cases independently.
"""
import math

import numpy as np
import torch

import oracle


def _bf16(values):
    return torch.tensor(np.asarray(values, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)


def _f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_constant_rows_give_exact_multiples():
    H, Eg = 64, 6
    x = _bf16(np.ones((2, H)))
    wr = _bf16(np.repeat((np.arange(Eg) + 1)[:, None] / 8.0, H, axis=1))
    lg = oracle.router_logits(x, wr)
    np.testing.assert_array_equal(lg, np.tile((np.arange(Eg) + 1) * H / 8.0, (2, 1)).astype(np.float32))


def test_permutation_router_selects_one_hidden_element():
    H, Eg, T = 32, 10, 3
    rng = np.random.default_rng(1)
    xv = rng.normal(size=(T, H))
    x = _bf16(xv)
    w = np.zeros((Eg, H))
    for e in range(Eg):
        w[e, (3 * e + 1) % H] = 1.0
    lg = oracle.router_logits(x, _bf16(w))
    xf = _f64(x)
    expected = np.stack([[xf[t, (3 * e + 1) % H] for e in range(Eg)] for t in range(T)]).astype(np.float32)
    np.testing.assert_array_equal(lg, expected)
    # the negated router negates every logit exactly
    np.testing.assert_array_equal(oracle.router_logits(x, _bf16(-w)), -expected)


def test_random_logits_equal_the_exactly_rounded_sum():
    T, H, Eg = 3, 96, 5
    rng = np.random.default_rng(2)
    x = _bf16(rng.normal(size=(T, H)))
    wr = _bf16(rng.normal(scale=0.1, size=(Eg, H)))
    lg = oracle.router_logits(x, wr)
    xf, wf = _f64(x), _f64(wr)
    for t in range(T):
        for e in range(Eg):
            assert lg[t, e] == np.float32(math.fsum(xf[t] * wf[e])), (t, e)
