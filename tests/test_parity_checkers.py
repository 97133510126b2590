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


# ----------------------------------------------------------------------------- indexer


@pytest.fixture(scope="module")
def ix_case():
    from oracle import indexer_oracle as IX
    import oracle as O
    g = np.random.default_rng(3)
    q = g.integers(0, 256, (64, 128), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0  # no NaN codes
    kc = g.integers(0, 256, (600, 128), dtype=np.uint8)
    kc[(kc & 0x7F) == 0x7F] = 0
    keys = O.e4m3_decode(kc)
    sc = 2.0 ** g.integers(-10, -4, 600).astype(np.float64)
    wt = g.standard_normal(64) / 8
    ref = IX.logits_of_token(q, wt, keys, sc)
    bound = np.abs(wt) @ (np.abs(O.e4m3_decode(q)) @ np.abs(keys).T) * sc[None, :]
    return ref, np.asarray(bound).reshape(-1), IX.topk_set(ref, 100)


def test_logits_check_accepts_the_oracle_and_refuses_planted_errors(ix_case):
    from test_gpu_indexer import _check_logits
    ref, bound, _ = ix_case
    row = torch.from_numpy(np.concatenate([ref, np.zeros(40)])).to(torch.float32)  # slots past n are not read
    _check_logits(row, ref, bound)
    for planted in ("off", "nan"):
        bad = row.clone()
        k = int(np.argmax(bound))
        bad[k] = float("nan") if planted == "nan" else bad[k] + 3e-4 * float(bound[k])
        with pytest.raises(AssertionError):
            _check_logits(bad, ref, bound)


@pytest.mark.parametrize("planted", ["duplicate", "a low value", "descending", "past the row", "short row padding"])
def test_topk_check_accepts_the_oracle_and_refuses_planted_errors(ix_case, planted):
    from test_gpu_indexer import _check_topk_valid
    ref, bound, sel = ix_case
    K = 100
    _check_topk_valid(torch.from_numpy(sel.astype(np.int32)), ref, bound, K)
    bad = sel.astype(np.int32).copy()
    rr, bb = ref, bound
    if planted == "duplicate":
        bad[5] = bad[4]
    elif planted == "a low value":
        bad[np.argmax(ref[bad])] = int(np.argmin(ref))
        bad.sort()
    elif planted == "descending":
        bad = bad[::-1].copy()
    elif planted == "past the row":
        bad[-1] = ref.shape[0]
    elif planted == "short row padding":  # 60 visible slots: all of them, then -1 (here one slot missed)
        rr, bb = ref[:60], bound[:60]
        _check_topk_valid(torch.from_numpy(np.concatenate([np.arange(60), -np.ones(40)]).astype(np.int32)), rr, bb, K)
        bad = np.concatenate([np.arange(59), -np.ones(41)]).astype(np.int32)
    with pytest.raises(AssertionError):
        _check_topk_valid(torch.from_numpy(bad), rr, bb, K)


# ----------------------------------------------------------------------------- operand range


@pytest.mark.parametrize("planted", ["none", "row scaled by 0.97", "spread over a row", "lse shifted"])
def test_scale_free_check_sees_errors_at_small_magnitudes(case, planted):
    # outputs of keys scaled by 1e-5 are compared after dividing by the gain: errors far below
    # the absolute tolerance of unscaled outputs must still be refused
    from test_gpu_operand_range import _assert_close
    ref, out, lse = case
    gain = 1e-5
    small = {"out": ref["out"] * gain, "lse": ref["lse"]}
    o = (torch.from_numpy(ref["out"]) * gain).to(torch.bfloat16)
    l = lse.clone()
    if planted == "row scaled by 0.97":
        o[1, 3] = (o[1, 3].double() * 0.97).to(torch.bfloat16)
    elif planted == "spread over a row":
        t, h = np.unravel_index(int(np.linalg.norm(ref["out"], axis=-1).argmin()), ref["out"].shape[:2])
        g = torch.Generator().manual_seed(2)
        o[t, h] = (o[t, h].double() + 0.006 * gain * torch.sign(torch.randn(512, generator=g))).to(torch.bfloat16)
    elif planted == "lse shifted":
        l[1, 1] -= 2e-3
    if planted == "none":
        _assert_close(o, l, small, out_scale=gain)
    else:
        assert np.abs(o.double().numpy() - small["out"]).max() < 1e-6  # invisible to an absolute bound
        with pytest.raises(AssertionError):
            _assert_close(o, l, small, out_scale=gain)
