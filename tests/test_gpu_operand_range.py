"""Operand range of the decode kernels, through the C ABI, against the float64 oracle.

The kernels feed 16-bit MMAs. q is normalised per row by a power of two, so any finite
bf16 q must give the oracle's result; the test scales q by 1e5 or 3e-6 (outside f16's
range) and divides sm_scale by the same gain, which leaves the softmax unchanged, so the
usual tolerances apply. Keys are scaled per slot; the output scales with them, so it is
compared after dividing by the gain (a scale-free metric), with the cosine taken over
every row. The 16-head kernel folds block scales into fp32 and serves any scale; the
tensor-core kernel (64+ heads, fp8_ds) serves block scales inside the f16 window
[2^-15, 2^7] and flags the others with SMLA_DEVERR_RANGE; RoPE values beyond f16's range
make its outputs non-finite.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import sparse_mla_decode_smla_gb300 as smla
import workloads as W
from oracle.workload_oracle import oracle_decode
from sparse_mla_decode_smla_gb300.runner import DeviceDecode

pytestmark = pytest.mark.gpu

OUT_ATOL, COS_MIN, LSE_ATOL = 1e-2, 0.9999, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    smla.lib()


def _case(heads, fmt="fp8_ds", **gains):
    base = W.small_variant(W.WORKLOADS[2], num_requests=2, ctx_lo=400, ctx_hi=700, topk=384)
    w = base.replace(num_heads=heads, kv_format=fmt, name=f"range_H{heads}_{fmt}", **gains)
    if fmt == "fp8_tensor":
        w = w.replace(kv_scale=2.0 ** -6)
    return w


def _assert_close(out, lse, ref, out_scale=1.0):
    o = out.double().cpu().numpy() / out_scale
    r = ref["out"] / out_scale
    assert np.isfinite(o).all()
    err = np.abs(o - r).max()
    assert err <= OUT_ATOL, f"max abs err {err} (after dividing by {out_scale})"
    cos = (o * r).sum(-1) / (np.linalg.norm(o, axis=-1) * np.linalg.norm(r, axis=-1))
    assert cos.min() >= COS_MIN, f"min cosine {cos.min()}"
    lerr = np.abs(lse.double().cpu().numpy() - ref["lse"]).max()
    assert lerr <= LSE_ATOL, f"lse err {lerr}"


def _run(w, scale_mode=smla.SMLA_SCALE_POW2, splits=0):
    p = W.make_problem(w)
    dd = DeviceDecode(p, scale_mode=scale_mode, num_splits=splits)
    out, lse = dd.run()
    bits = smla.read_error(dd.desc, dd.workspace)
    ref = oracle_decode(p, scale_mode=O.SCALE_FP32 if scale_mode == smla.SMLA_SCALE_FP32 else O.SCALE_POW2)
    return out, lse, ref, bits, dd


@pytest.mark.parametrize("heads", [16, 64, 128])
@pytest.mark.parametrize("fmt", ["fp8_ds", "fp8_tensor"])
@pytest.mark.parametrize("gain", [1e5, 3e-6])
def test_q_beyond_f16_range_is_exact(heads, fmt, gain):
    w = _case(heads, fmt, q_gains=(gain,))
    w = w.replace(sm_scale=float(np.float32(W.SM_SCALE_576 / gain)))
    out, lse, ref, bits, _ = _run(w, splits=1 if heads == 128 else 0)
    _assert_close(out, lse, ref)
    assert bits == 0


@pytest.mark.parametrize("heads", [16, 128])
def test_q_rows_spanning_many_octaves(heads):
    # within every row, dims alternate between x1e3 and x1e-3 (2^20 apart)
    w = _case(heads, q_dim_gains=(1e3, 1e-3))
    w = w.replace(sm_scale=float(np.float32(W.SM_SCALE_576 / 1e3)))
    out, lse, ref, bits, _ = _run(w)
    _assert_close(out, lse, ref)
    assert bits == 0


# key gains inside the window: block amax of ~3.5 x gain over 448 gives POW2 scales of
# 2^-15 (gain 0.004) and 2^7 (gain 1e4); FP32 scales of ~1.6e-4 (gain 0.02) and ~78 (1e4)
@pytest.mark.parametrize("heads", [16, 64, 128])
@pytest.mark.parametrize("mode,gain", [(smla.SMLA_SCALE_POW2, 0.004), (smla.SMLA_SCALE_POW2, 1e4),
                                       (smla.SMLA_SCALE_FP32, 0.02), (smla.SMLA_SCALE_FP32, 1e4)])
def test_key_scales_inside_the_window(heads, mode, gain):
    w = _case(heads, latent_gains=(gain,), rope_gains=(gain,))
    w = w.replace(sm_scale=float(np.float32(W.SM_SCALE_576 / gain)))
    out, lse, ref, bits, _ = _run(w, scale_mode=mode)
    _assert_close(out, lse, ref, out_scale=gain)
    assert bits == 0


@pytest.mark.parametrize("heads", [64, 128])
def test_mixed_slot_magnitudes_inside_the_window(heads):
    # neighbouring slots 10^4 apart in magnitude; sm_scale keeps the largest slots' scores
    # of order one, and the error is measured against the largest values' scale
    w = _case(heads, latent_gains=(0.01, 1.0, 100.0), rope_gains=(0.01, 1.0, 100.0))
    w = w.replace(sm_scale=float(np.float32(W.SM_SCALE_576 / 100.0)))
    out, lse, ref, bits, _ = _run(w, splits=3)
    _assert_close(out, lse, ref, out_scale=100.0)
    assert bits == 0


@pytest.mark.parametrize("mode,gain", [(smla.SMLA_SCALE_POW2, 1e-5), (smla.SMLA_SCALE_POW2, 1e5),
                                       (smla.SMLA_SCALE_FP32, 0.004)])
def test_key_scales_outside_the_window(mode, gain):
    # 16 heads (block scales folded in fp32): exact. 64 and 128 heads (f16 operands):
    # the call reports SMLA_DEVERR_RANGE, and smla_read_error SMLA_ERR_OPERAND_RANGE.
    w = _case(16, latent_gains=(gain,), rope_gains=(gain,))
    w = w.replace(sm_scale=float(np.float32(W.SM_SCALE_576 / gain)))
    out, lse, ref, bits, _ = _run(w, scale_mode=mode)
    _assert_close(out, lse, ref, out_scale=gain)
    assert bits == 0
    for heads in (64, 128):
        p = W.make_problem(w.replace(num_heads=heads))
        dd = DeviceDecode(p, scale_mode=mode)
        dd.run()
        v = ctypes.c_int32(0)
        st = smla.lib().smla_read_error(ctypes.byref(dd.desc), ctypes.c_void_p(dd.workspace.data_ptr()),
                                        dd.workspace.numel() * 4, ctypes.byref(v), None)
        assert v.value == smla.SMLA_DEVERR_RANGE and st == 10


def test_rope_beyond_f16_range():
    # RoPE values of 1e5: the 16-head kernel multiplies them as bf16 and stays exact; the
    # tensor-core kernel's f16 operands cannot hold them, and its outputs turn non-finite
    # (visible to the caller, as the header states) instead of silently wrong
    w = _case(16, rope_gains=(1e5,)).replace(sm_scale=float(np.float32(W.SM_SCALE_576 / 1e5)))
    out, lse, ref, bits, _ = _run(w)
    assert bits == 0
    _assert_close(out, lse, ref)
    p = W.make_problem(w.replace(num_heads=128))
    out, _ = DeviceDecode(p).run()
    assert not torch.isfinite(out.float()).all()
