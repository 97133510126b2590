"""The GPU tests' parity checks reject planted errors (CPU only).

The checks that compare the CUDA path with the oracle are only as strong as what they refuse.
Here each one is given the oracle's own result, which it must accept, and then that result with
one planted error, which it must refuse: a single element off by more than the tolerance, two
heads swapped, a small error spread over a whole row (inside the element bound, caught by the
cosine), an LSE shifted or made infinite, a non-finite output.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle.workload_oracle import oracle_decode
from test_gpu_fp8_q import assert_fp8_parity
from test_gpu_parity import assert_parity


@pytest.fixture(scope="module")
def case():
    w = W.small_variant(W.WORKLOADS[2], num_requests=2, ctx_lo=300, ctx_hi=500, topk=128)
    ref = oracle_decode(W.make_problem(w))
    out = torch.from_numpy(ref["out"]).to(torch.bfloat16)
    lse = torch.from_numpy(ref["lse"]).to(torch.float32)
    return ref, out, lse


def _planted(out, lse, kind):
    o, l = out.clone(), lse.clone()
    if kind == "one element":
        o[1, 7, 300] += 0.05
    elif kind == "heads swapped":
        o[0, [3, 4]] = o[0, [4, 3]]
    elif kind == "spread over a row":  # the row of smallest norm, +-0.006 on every element
        t, h = np.unravel_index(int(torch.linalg.vector_norm(o.float(), dim=-1).argmin()), o.shape[:2])
        g = torch.Generator().manual_seed(1)
        o[t, h] = (o[t, h].float() + 0.006 * torch.sign(torch.randn(512, generator=g))).to(torch.bfloat16)
    elif kind == "lse shifted":
        l[0, 5] += 2e-3
    elif kind == "lse infinite":
        l[1, 2] = float("-inf")
    elif kind == "non-finite output":
        o[0, 0, 0] = float("nan")
    return o, l


KINDS = ["one element", "heads swapped", "spread over a row", "lse shifted", "lse infinite", "non-finite output"]


def test_parity_check_accepts_the_oracle(case):
    ref, out, lse = case
    assert_parity(out, lse, ref)


@pytest.mark.parametrize("kind", KINDS)
def test_parity_check_refuses_a_planted_error(case, kind):
    ref, out, lse = case
    o, l = _planted(out, lse, kind)
    if kind == "spread over a row":  # inside the element bound: only the cosine can see it
        assert np.abs(o.double().numpy() - ref["out"]).max() <= 1e-2
    with pytest.raises(AssertionError):
        assert_parity(o, l, ref)


@pytest.mark.parametrize("kind", ["heads swapped", "lse shifted", "lse infinite", "non-finite output"])
def test_fp8_parity_check_refuses_a_planted_error(case, kind):
    # the FP8-q check bounds errors by 0.14 max|v| (E4M3 weights) and keeps the cosine and LSE
    ref, out, lse = case
    vmax = float(np.abs(ref["out"]).max())
    assert_fp8_parity(out, lse, ref, vmax)
    o, l = _planted(out, lse, kind)
    with pytest.raises(AssertionError):
        assert_fp8_parity(o, l, ref, vmax)
