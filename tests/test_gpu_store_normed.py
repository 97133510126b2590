"""GPU parity of the cache write fused with RMSNorm and RoPE (smla_store_kv_normed) against the
float64 oracle, through the C ABI.

Where fp32 and float64 compute the same values (power-of-two row magnitudes, eps = 0, rotations
by 0, +-1 and +-0.5) the stored rows must equal the oracle's bit for bit in every format. On
general inputs the kernel's fp32 norm may round to the neighbouring bf16 value where the exact
result sits near a rounding midpoint: every stored bf16 value must be within one bf16 step of the
oracle's, at least 99.9% of them equal, and the FP8 rows must be the oracle packer's rows of the
kernel's own normed values.
"""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_mla_decode_smla_gb300 as smla
import workloads as W
from oracle.workload_oracle import oracle_decode
from sparse_mla_decode_smla_gb300.runner import DeviceDecode

pytestmark = pytest.mark.gpu

FMTS = {"bf16": (smla.SMLA_KV_BF16, 1152), "fp8_ds": (smla.SMLA_KV_FP8_DS, 656),
        "fp8_tensor": (smla.SMLA_KV_FP8_TENSOR, 576)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    smla.lib()


def _bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _store(fmt, x, eps, slots, num_slots, scale_mode=smla.SMLA_SCALE_POW2, kv_scale=1.0, err=None):
    kvf, rb = FMTS[fmt]
    kv = torch.full((num_slots, rb), 0xAB, dtype=torch.uint8, device="cuda")
    smla.store_kv_normed(kvf, x.latent.cuda(), x.rope.cuda(), x.weight.cuda(), eps, x.positions.cuda(),
                         x.cos_sin.cuda(), slots.cuda(), kv, num_slots, scale_mode=scale_mode,
                         kv_scale=kv_scale, error_word=err)
    torch.cuda.synchronize()
    return kv.cpu().numpy()


def _oracle(fmt, x, eps, scale_mode=O.SCALE_POW2, kv_scale=None):
    cs = x.cos_sin.double().numpy()[x.positions.numpy()]
    return O.store_normed_rows(_bits(x.latent), _bits(x.rope), _bits(x.weight), eps, cs[:, :32], cs[:, 32:],
                               fmt, scale_mode, kv_scale)


def _exact_inputs(n, seed):
    g = torch.Generator().manual_seed(seed)
    mag = torch.exp2(torch.randint(-4, 5, (n, 1), generator=g).float())
    sign = torch.where(torch.rand(n, 512, generator=g) < 0.5, -1.0, 1.0)
    x = W.make_store_inputs(n, seed, max_position=64)
    x.latent = (mag * sign).to(torch.bfloat16)
    pick = torch.tensor([0.0, 1.0, -1.0, 0.5, -0.5])
    x.cos_sin = pick[torch.randint(0, 5, (64, 64), generator=g)].to(torch.float32)
    return x


@pytest.mark.parametrize("fmt", list(FMTS))
def test_bit_exact_where_fp32_is_exact(fmt):
    n = 700
    x = _exact_inputs(n, 3)
    slots = torch.randperm(900)[:n].to(torch.int64)
    slots[7] = -1    # not stored
    slots[8] = 905   # beyond the cache's 900 rows: not stored
    got = _store(fmt, x, 0.0, slots, 900, kv_scale=2.0 ** -3)
    ref = _oracle(fmt, x, 0.0, kv_scale=2.0 ** -3)
    m = slots.numpy()
    ok = (m >= 0) & (m < 900)
    assert np.array_equal(got[m[ok]], ref[ok])
    # every other row of the cache keeps its bytes
    assert (got[np.setdiff1d(np.arange(900), m[ok])] == 0xAB).all()


# a power-of-two scale takes the kernel's exact reciprocal, any other one its division
@pytest.mark.parametrize("fmt,mode,kv_scale", [("bf16", 0, 1.0), ("fp8_ds", smla.SMLA_SCALE_POW2, 1.0),
                                               ("fp8_ds", smla.SMLA_SCALE_FP32, 1.0), ("fp8_tensor", 0, 2.0 ** -4),
                                               ("fp8_tensor", 0, 0.0371)])
def test_general_inputs_within_one_bf16_step(fmt, mode, kv_scale):
    n = 3000
    x = W.make_store_inputs(n, 11)
    slots = torch.randperm(4000)[:n].to(torch.int64)
    got = _store(fmt, x, 1e-6, slots, 4000, scale_mode=mode, kv_scale=kv_scale)[slots.numpy()]
    # the oracle's normed, rotated bf16 values
    cs = x.cos_sin.double().numpy()[x.positions.numpy()]
    lat = O.rms_norm_bf16(_bits(x.latent), _bits(x.weight), 1e-6)
    rope = O.rope_bf16(_bits(x.rope), cs[:, :32], cs[:, 32:])
    if fmt == "bf16":
        vals = O.bf16_bits_to_f64(got.view("<u2").reshape(n, 576))
        ref = np.concatenate([lat, rope], axis=1)
        # one bf16 step, plus the fp32 rounding of a c - b s where it cancels
        r = O.bf16_bits_to_f64(_bits(x.rope))
        a, b, c, s = np.abs(r[:, 0::2]), np.abs(r[:, 1::2]), np.abs(cs[:, :32]), np.abs(cs[:, 32:])
        terms = np.repeat(a * c + b * s, 2, axis=1) * 2.0 ** -22
        tol = np.abs(ref) * 2.0 ** -7 + np.concatenate([np.zeros((n, 512)), terms], axis=1)
        assert (np.abs(vals - ref) <= tol + 1e-38).all()
        assert (vals == ref).mean() >= 0.999
        return
    # FP8 rows: the kernel's rows must be the oracle packer's rows of values within one bf16
    # step of the oracle's; rows whose normed values agree exactly must agree byte for byte
    ref_rows = _oracle(fmt, x, 1e-6, scale_mode=mode, kv_scale=kv_scale)
    same = (got == ref_rows).all(axis=1)
    assert same.mean() >= 0.99
    deq_got = O.dequant_rows(got, fmt, kv_scale if fmt == "fp8_tensor" else None)
    deq_ref = O.dequant_rows(ref_rows, fmt, kv_scale if fmt == "fp8_tensor" else None)
    # one E4M3 step of the value, or one subnormal step of a block whose scale moved
    amax = np.abs(deq_ref).max(axis=1, keepdims=True)
    tol = np.maximum(np.abs(deq_ref), np.abs(deq_got)) * 2.0 ** -3 + amax * 2.0 ** -8
    assert (np.abs(deq_got - deq_ref) <= tol).all()


def test_out_of_range_position_is_flagged_and_skipped():
    x = W.make_store_inputs(8, 5, max_position=32)
    x.positions[3] = 40
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = torch.arange(8, dtype=torch.int64)
    got = _store("fp8_ds", x, 1e-6, slots, 8, err=err)
    assert err.item() == smla.SMLA_DEVERR_INDEX
    assert (got[3] == 0xAB).all()  # not written
    ok = [i for i in range(8) if i != 3]
    x.positions[3] = 0
    ref = _oracle("fp8_ds", x, 1e-6)
    assert (got[ok] == ref[ok]).all(axis=1).mean() >= 0.85


def test_normed_cache_feeds_the_decode():
    # a cache written by the fused store, decoded with 128 heads, against the oracle decode of
    # the oracle's own rows
    w = W.small_variant(W.WORKLOADS[2], num_requests=2, ctx_lo=600, ctx_hi=600, topk=256)
    p = W.make_problem(w)
    n = p.num_slots
    x = W.make_store_inputs(n, 21)
    slots = torch.arange(n, dtype=torch.int64)
    rows = _store("fp8_ds", x, 1e-6, slots, n)
    ref_rows = _oracle("fp8_ds", x, 1e-6)
    kv = torch.from_numpy(rows).cuda()
    dd = DeviceDecode(p, kv=kv)
    out, lse = dd.run()
    torch.cuda.synchronize()

    class Cache:  # the oracle's own normed rows, by physical slot
        def fetch(self, phys):
            return ref_rows[np.asarray(phys, dtype=np.int64)]

    ref = oracle_decode(p, cache=Cache())
    assert np.abs(out.double().cpu().numpy() - ref["out"]).max() <= 1e-2
    assert np.abs(lse.double().cpu().numpy() - ref["lse"]).max() <= 1e-3
