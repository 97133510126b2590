"""GPU parity of FP8 q (E4M3 codes with a per-tensor q_scale) against the per-tensor FP8 cache,
the FP8-operand tensor-core kernel, through the C ABI.

The oracle decodes exactly, on the same E4M3 q and cache codes. The kernel multiplies the codes
on the tensor cores with fp32 accumulation, and takes its probabilities into PV as E4M3 values,
each within 2^-4 relative of its exact value, then normalises by their sum. So every output is a
convex combination of the selected values whose weights move by at most 2 * 2^-4 / (1 - 2^-4)
in total: |out - ref| <= 0.14 * max |v| * kv_scale (plus the bf16 rounding of out). The LSE uses
the weights before rounding and keeps the usual 1e-3.
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

BOUND = 0.14      # times max |v| * kv_scale, from the E4M3 rounding of the weights
COS_MIN = 0.999   # per (token, head), measured typical agreement
LSE_ATOL = 1e-3
QS = W.Q_SCALE_FP8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    smla.lib()


def run_fp8_q(problem, num_splits=0, q_scale=QS, topk=None, req_id=None):
    """The FP8-q decode of a problem on the per-tensor cache: (out, lse, E4M3 q, error word)."""
    w = problem.w
    dd = DeviceDecode(problem, num_splits=num_splits)
    q8 = W.q_to_e4m3(problem.q, q_scale)
    dd.q = q8.cuda().contiguous()
    dd.desc.q_format, dd.desc.q_scale = smla.SMLA_Q_FP8_E4M3, q_scale
    if topk is not None:
        dd.topk = topk.to(device="cuda", dtype=torch.int32).contiguous()
    dd.req_id = req_id
    ws = smla.workspace_size(dd.desc)
    dd.workspace = torch.zeros((ws + 255) // 256 * 256 // 4, dtype=torch.int32, device="cuda")
    out, lse = dd.run()
    torch.cuda.synchronize()
    err = int(dd.workspace[0].item())
    return out, lse, q8, err


def max_abs_value(problem):
    """max |v| * kv_scale over the cache (a bound on every token's selected values)."""
    w = problem.w
    lat, _ = problem.raw_pages(range(problem.num_pages))
    codes = O.pack_fp8_tensor(lat.view(torch.int16).numpy().view(np.uint16),
                              np.zeros((lat.shape[0], 64), dtype=np.uint16), w.kv_scale)
    return float(np.abs(O.dequant_rows(codes, "fp8_tensor", w.kv_scale)[:, :512]).max())


def assert_fp8_parity(out, lse, ref, vmax, tokens=None):
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    if tokens is not None:
        o, l = o[tokens], l[tokens]
    r, rl = ref["out"], ref["lse"]
    assert np.isfinite(o).all()
    err = np.abs(o - r)
    assert (err <= BOUND * vmax + np.abs(r) * 2.0 ** -8 + 1e-6).all(), f"max err {err.max()} vs {BOUND * vmax}"
    num = (o * r).sum(-1)
    den = np.linalg.norm(o, axis=-1) * np.linalg.norm(r, axis=-1)
    nz = den > 0
    cos = num[nz] / den[nz]
    assert cos.min() >= COS_MIN, f"min cosine {cos.min()}"
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))
    fin = np.isfinite(rl)
    if fin.any():
        assert np.abs(l[fin] - rl[fin]).max() <= LSE_ATOL
    return err.max(), cos.min()


SMALL = [
    W.small_variant(W.EXTRA_WORKLOADS[1], num_requests=2, ctx_lo=700, ctx_hi=700, topk=448),   # 128 heads, sink
    W.small_variant(W.EXTRA_WORKLOADS[2], num_requests=2, ctx_lo=300, ctx_hi=900, topk=256),   # MTP, next_n 4
    W.small_variant(W.EXTRA_WORKLOADS[0], num_requests=3, ctx_lo=100, ctx_hi=900, topk=320),   # 64 heads, padding
]


@pytest.mark.parametrize("wi", range(len(SMALL)))
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_fp8_q_matches_oracle(wi, splits):
    p = W.make_problem(SMALL[wi])
    out, lse, q8, err = run_fp8_q(p, num_splits=splits)
    assert err == 0
    ref = oracle_decode(p, q_e4m3=q8, q_scale=QS)
    e, c = assert_fp8_parity(out, lse, ref, max_abs_value(p))
    print(f"{SMALL[wi].name} splits={splits}: max abs err {e:.4g}, min cos {c:.6f}")


@pytest.mark.parametrize("heads", [64, 96])
def test_fp8_q_head_counts_and_many_splits(heads):
    # 96 heads: the second head group holds 32 real heads; 16 splits merge in the merge kernel
    w = SMALL[0].replace(num_heads=heads, topk=1024, ctx_lo=2000, ctx_hi=2000)
    p = W.make_problem(w)
    for splits in (0, 16):
        out, lse, q8, err = run_fp8_q(p, num_splits=splits)
        assert err == 0
        assert_fp8_parity(out, lse, oracle_decode(p, q_e4m3=q8, q_scale=QS), max_abs_value(p))


def test_fp8_q_scale_and_kv_scale():
    # a q_scale and a kv_scale that are not powers of two
    w = SMALL[1].replace(kv_scale=0.0137)
    p = W.make_problem(w)
    out, lse, q8, err = run_fp8_q(p, q_scale=0.0291)
    assert err == 0
    assert_fp8_parity(out, lse, oracle_decode(p, q_e4m3=q8, q_scale=0.0291), max_abs_value(p))


def test_fp8_q_identical_values_give_the_value():
    # every selected slot of token 0 is the same slot: the weights sum to 1 whatever their
    # rounding, so the output is that slot's value (up to fp32 sums and the bf16 output)
    w = SMALL[0]
    p = W.make_problem(w)
    topk = p.topk.clone()
    topk[0, :] = 5
    out, lse, q8, err = run_fp8_q(p, topk=topk)
    assert err == 0
    p.topk = topk
    ref = oracle_decode(p, tokens=[0], q_e4m3=q8, q_scale=QS)
    o = out[0].double().cpu().numpy()
    assert np.abs(o - ref["out"][0]).max() <= np.abs(ref["out"][0]).max() * 2.0 ** -7
    assert np.abs(lse[0].double().cpu().numpy() - ref["lse"][0]).max() <= LSE_ATOL


def test_fp8_q_invalid_entries_are_masked_and_flagged():
    w = SMALL[1]
    p = W.make_problem(w)
    topk = p.topk.clone()
    topk[1, 7] = 10 ** 6  # outside the page table
    out, lse, q8, err = run_fp8_q(p, topk=topk)
    assert err == smla.SMLA_DEVERR_INDEX
    p.topk = topk
    assert_fp8_parity(out, lse, oracle_decode(p, q_e4m3=q8, q_scale=QS), max_abs_value(p))


def test_fp8_q_full_size_mtp_sampled():
    # the MTP batch at full size on the per-tensor cache, in the bench's launch configuration
    w = W.EXTRA_WORKLOADS[2]
    p = W.make_problem(w, device="cuda")
    out, lse, q8, err = run_fp8_q(p)
    assert err == 0
    ctx = p.ctx
    tokens = sorted({0, 77, 130, 255, 4 * int(ctx.argmin()), 4 * int(ctx.argmax()) + 3})
    ref = oracle_decode(p, tokens=tokens, q_e4m3=q8, q_scale=QS)
    vmax = 6.0  # N(0, 1) values in E4M3 at kv_scale 1 stay below this over any sample of the pool
    assert_fp8_parity(out, lse, ref, vmax, tokens=tokens)


@pytest.mark.parametrize("splits", [1, 3, 16])
def test_fp8_q_outputs_stay_inside_their_buffers(splits):
    # out and lse between guard bands: one split, splits merged in the cluster, and splits
    # through the merge kernel (16 of 64 entries); lse = NULL gives the same output bits
    w = SMALL[0].replace(num_heads=128, topk=1024, ctx_lo=1500, ctx_hi=1500)
    p = W.make_problem(w)
    dd = DeviceDecode(p, num_splits=splits)
    dd.q = W.q_to_e4m3(p.q, QS).cuda().contiguous()
    dd.desc.q_format, dd.desc.q_scale = smla.SMLA_Q_FP8_E4M3, QS
    want_out, want_lse = [x.clone() for x in dd.run()]
    T, H, G = w.num_tokens, w.num_heads, 4096
    ob = torch.full((G + T * H * 512 + G,), 0x3039, dtype=torch.int16, device="cuda")
    lb = torch.full((G + T * H + G,), -7.0, dtype=torch.float32, device="cuda")
    dd.out = ob[G:G + T * H * 512].view(torch.bfloat16).view(T, H, 512)
    dd.lse = lb[G:G + T * H].view(T, H)
    out, lse = dd.run()
    torch.cuda.synchronize()
    assert (ob[:G] == 0x3039).all() and (ob[G + T * H * 512:] == 0x3039).all()
    assert (lb[:G] == -7.0).all() and (lb[G + T * H:] == -7.0).all()
    assert torch.equal(out.view(torch.int16), want_out.view(torch.int16)) and torch.equal(lse, want_lse)
    dd.lse = None
    out, _ = dd.run()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), want_out.view(torch.int16))
    assert smla.read_error(dd.desc, dd.workspace) == 0
