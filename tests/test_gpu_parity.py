"""GPU parity of the CUDA path against the float64 oracle, through the C ABI.

Tolerances (bf16 output, fp32 LSE): max |out - ref| <= 1e-2, per-(token, head)
cosine >= 0.9999, |lse - ref| <= 1e-3; cache packing and gather/dequant are
bit-exact. Inputs come from the seeded workload generator; the oracle packs
its own cache rows from the same source values.
"""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_mla_decode_smla_gb300 as smla
import workloads as W
from oracle.workload_oracle import OracleCache, oracle_decode
from sparse_mla_decode_smla_gb300.runner import DeviceDecode, pack_problem_cache

pytestmark = pytest.mark.gpu

OUT_ATOL, COS_MIN, LSE_ATOL = 1e-2, 0.9999, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    smla.lib()
    torch.cuda.init()


def _bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def assert_parity(out, lse, ref, tokens=None, lse_atol=LSE_ATOL):
    o = out.double().cpu().numpy()
    l = lse.double().cpu().numpy()
    if tokens is not None:
        o, l = o[tokens], l[tokens]
    r, rl = ref["out"], ref["lse"]
    assert np.isfinite(o).all()
    err = np.abs(o - r).max()
    assert err <= OUT_ATOL, f"max abs err {err}"
    num = (o * r).sum(-1)
    den = np.linalg.norm(o, axis=-1) * np.linalg.norm(r, axis=-1)
    big = np.linalg.norm(r, axis=-1) > 1e-3
    if big.any():
        cos = num[big] / den[big]
        assert cos.min() >= COS_MIN, f"min cosine {cos.min()}"
    assert np.array_equal(np.isneginf(l), np.isneginf(rl))
    fin = np.isfinite(rl)
    if fin.any():
        lerr = np.abs(l[fin] - rl[fin]).max()
        assert lerr <= lse_atol, f"lse err {lerr}"


SMALL = [
    W.WORKLOADS[0],
    W.small_variant(W.WORKLOADS[1], num_requests=3, ctx_lo=100, ctx_hi=900, topk=320),
    W.small_variant(W.WORKLOADS[2], num_requests=2, ctx_lo=700, ctx_hi=700, topk=448),
    W.small_variant(W.WORKLOADS[3], num_requests=2, ctx_lo=300, ctx_hi=500, topk=256),
    W.small_variant(W.WORKLOADS[4], num_requests=4, ctx_lo=400, ctx_hi=1000, topk=320, tail_pad=64),
]


@pytest.fixture(scope="module")
def small_cases():
    cases = {}
    for w in SMALL:
        p = W.make_problem(w)
        cases[w.name] = (p, oracle_decode(p))
    return cases


# ------------------------------------------------------------------ pack / gather


def _pack_inputs(n, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, 512, generator=g)
    x = x * (2.0 ** torch.randint(-30, 30, (n, 4, 1), generator=g)).repeat_interleave(128, 2).view(n, 512)
    x[0, :128] = 0.0
    x[1, 128:256] = 56.0
    x[2, :] = torch.tensor([1e-40, -3e38, 65504.0, -0.0] * 128)
    rope = torch.randn(n, 64, generator=g)
    return x.to(torch.bfloat16), rope.to(torch.bfloat16)


@pytest.mark.parametrize("mode", [smla.SMLA_SCALE_POW2, smla.SMLA_SCALE_FP32])
def test_pack_fp8_bit_exact(mode):
    n, slots = 3000, 4000
    lat, rope = _pack_inputs(n, 1 + mode)
    mapping = torch.randperm(slots)[:n].to(torch.int64)
    mapping[5] = -1
    mapping[6] = slots + 10  # out of range: skipped
    kv = torch.full((slots, 656), 0xAB, dtype=torch.uint8, device="cuda")
    smla.pack_kv(smla.SMLA_KV_FP8_DS, mode, lat.cuda(), rope.cuda(), mapping.cuda(), kv, slots)
    got = kv.cpu().numpy()
    ref = O.pack_fp8_ds(_bits(lat), _bits(rope), mode)
    m = mapping.numpy()
    ok = (m >= 0) & (m < slots)
    assert np.array_equal(got[m[ok]], ref[ok])
    untouched = np.setdiff1d(np.arange(slots), m[ok])
    assert (got[untouched] == 0xAB).all()


def test_pack_bf16_bit_exact():
    lat, rope = _pack_inputs(500, 7)
    mapping = torch.arange(499, -1, -1, dtype=torch.int64)
    kv = torch.zeros((500, 1152), dtype=torch.uint8, device="cuda")
    smla.pack_kv(smla.SMLA_KV_BF16, 0, lat.cuda(), rope.cuda(), mapping.cuda(), kv, 500)
    ref = O.pack_bf16(_bits(lat), _bits(rope))
    assert np.array_equal(kv.cpu().numpy()[mapping.numpy()], ref)


@pytest.mark.parametrize("wi", [0, 1, 4])
def test_gather_dequant_bit_exact(wi):
    w = SMALL[wi]
    p = W.make_problem(w)
    kv = pack_problem_cache(p)
    topk = p.topk.clone()
    topk[0, 1] = 10 ** 6  # beyond the page table: invalid, flagged
    d = smla.make_desc(w.num_tokens, w.num_heads, w.topk, w.num_requests, w.page_size, p.num_pages,
                       w.page_table_stride, smla.runner.FMT[w.kv_format], w.sm_scale, next_n=w.next_n)
    rows = torch.full((w.num_tokens, w.topk, 576), 7.0, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    smla.gather_dequant(d, kv, p.page_table.cuda(), topk.cuda(), None, rows, err)
    cache = OracleCache(p)
    ref = O.gather_dequant(cache.fetch, w.kv_format, p.page_table.numpy(), topk.numpy(), w.page_size,
                           p.num_pages, next_n=w.next_n)
    got = rows.cpu().double().numpy()
    assert np.array_equal(got, ref)
    assert err.item() == smla.SMLA_DEVERR_INDEX


@pytest.mark.parametrize("wi", [2, 4])
def test_decode_fp32_block_scales(wi):
    # fp8_ds rows packed with fp32 block scales (amax / 448, not powers of two). The
    # 16-head path folds the scale into fp32 partial scores; the tensor-core path rounds
    # code * scale to its f16 MMA operand (within 2^-11 relative). Both meet every
    # tolerance.
    w = SMALL[wi]
    p = W.make_problem(w)
    out, lse = DeviceDecode(p, scale_mode=smla.SMLA_SCALE_FP32).run()
    ref = oracle_decode(p, scale_mode=O.SCALE_FP32)
    assert_parity(out, lse, ref)


# ------------------------------------------------------------------ per-tensor FP8 cache

TENSOR = W.EXTRA_WORKLOADS[0]  # fp8tensor_T32_H64_K2048_ctx1k-32k


@pytest.mark.parametrize("kv_scale", [1.0, 2.0 ** -6, 0.0137])
def test_pack_fp8_tensor_bit_exact(kv_scale):
    n, slots = 2000, 2500
    g = torch.Generator().manual_seed(5)
    lat = (torch.randn(n, 512, generator=g) * 4).to(torch.bfloat16)
    rope = (torch.randn(n, 64, generator=g) * 4).to(torch.bfloat16)
    lat[0, :8] = 1e4  # saturates at +-448
    mapping = torch.randperm(slots, generator=g)[:n].to(torch.int64)
    mapping[3] = -1
    kv = torch.full((slots, 576), 0xAB, dtype=torch.uint8, device="cuda")
    smla.pack_kv_fp8_tensor(lat.cuda(), rope.cuda(), mapping.cuda(), kv, slots, kv_scale)
    ref = O.pack_fp8_tensor(_bits(lat), _bits(rope), kv_scale)
    m = mapping.numpy()
    ok = m >= 0
    assert np.array_equal(kv.cpu().numpy()[m[ok]], ref[ok])


def test_gather_dequant_fp8_tensor_bit_exact():
    w = W.small_variant(TENSOR, num_requests=3, ctx_lo=100, ctx_hi=900, topk=320).replace(kv_scale=0.0137)
    p = W.make_problem(w)
    kv = pack_problem_cache(p)
    d = smla.make_desc(w.num_tokens, w.num_heads, w.topk, w.num_requests, w.page_size, p.num_pages,
                       w.page_table_stride, smla.SMLA_KV_FP8_TENSOR, w.sm_scale, kv_scale=w.kv_scale)
    rows = torch.full((w.num_tokens, w.topk, 576), 7.0, device="cuda")
    smla.gather_dequant(d, kv, p.page_table.cuda(), p.topk.cuda(), None, rows)
    ref = O.gather_dequant(OracleCache(p).fetch, "fp8_tensor", p.page_table.numpy(), p.topk.numpy(),
                           w.page_size, p.num_pages, kv_scale=w.kv_scale)
    assert np.array_equal(rows.cpu().double().numpy(), ref)


@pytest.mark.parametrize("heads,sink,kv_scale", [(16, False, 1.0), (64, False, 1.0), (128, True, 2.0 ** -6),
                                                 (64, True, 0.0137)])
@pytest.mark.parametrize("splits", [1, 3])
def test_decode_fp8_tensor_matches_oracle(heads, sink, kv_scale, splits):
    w = W.small_variant(TENSOR, num_requests=3, ctx_lo=200, ctx_hi=800, topk=448).replace(
        num_heads=heads, sink=sink, kv_scale=kv_scale, name=f"fp8tensor_H{heads}")
    p = W.make_problem(w)
    out, lse = DeviceDecode(p, num_splits=splits).run()
    assert_parity(out, lse, oracle_decode(p))


# ------------------------------------------------------------------ decode parity


@pytest.mark.parametrize("wi", range(len(SMALL)))
@pytest.mark.parametrize("splits", [0, 1, 3])
def test_decode_matches_oracle(small_cases, wi, splits):
    p, ref = small_cases[SMALL[wi].name]
    dd = DeviceDecode(p, num_splits=splits)
    out, lse = dd.run()
    torch.cuda.synchronize()
    assert_parity(out, lse, ref)
    assert smla.read_error(dd.desc, dd.workspace) == 0


@pytest.mark.parametrize("heads", [32, 48, 80, 96, 112])
def test_decode_other_head_counts(heads):
    # head counts between the workloads' 16/64/128: the 80..112 cases leave part of a warp's
    # 32 TMEM lanes without a head in the tensor-core kernel
    w = W.small_variant(W.WORKLOADS[2], num_requests=2, ctx_lo=500, ctx_hi=900, topk=320).replace(
        num_heads=heads, name=f"fp8_H{heads}")
    p = W.make_problem(w)
    for splits in (1, 2):
        out, lse = DeviceDecode(p, num_splits=splits).run()
        assert_parity(out, lse, oracle_decode(p))


@pytest.mark.parametrize("wi", [1, 2, 4])
def test_split_count_invariance(small_cases, wi):
    p, ref = small_cases[SMALL[wi].name]
    dd = DeviceDecode(p)
    for s in (1, 2, 4, 5, 8):
        dd2 = DeviceDecode(p, kv=dd.kv, num_splits=s)
        out, lse = dd2.run()
        assert_parity(out, lse, ref)


@pytest.mark.parametrize("heads", [16, 64])
def test_duplicated_indices_count_per_position(heads):
    # A slot listed at several positions counts once per position (the plain sum over the
    # list): positions 200..259 repeat the slots at 0..59, across the two splits.
    w = W.small_variant(W.WORKLOADS[1], num_requests=2, ctx_lo=600, ctx_hi=600, topk=320).replace(
        num_heads=heads, name=f"fp8_dup_H{heads}")
    p = W.make_problem(w)
    tk = p.topk.clone()
    assert bool((tk[:, :60] >= 0).all())
    tk[:, 200:260] = tk[:, 0:60]
    p.topk = tk
    out, lse = DeviceDecode(p, num_splits=2).run()
    assert_parity(out, lse, oracle_decode(p))


@pytest.mark.parametrize("wi", [1, 2, 4])  # 64 and 128 heads (tensor-core kernel), 16 heads
def test_unselected_rows_are_never_read(small_cases, wi):
    # Overwrite every cache row no valid index selects with NaN codes: output is bitwise unchanged.
    p, _ = small_cases[SMALL[wi].name]
    dd = DeviceDecode(p, num_splits=2)
    out0, lse0 = [x.clone() for x in dd.run()]
    P = p.w.page_size
    pt = p.page_table.numpy()
    used = set()
    for t in range(p.w.num_tokens):
        for i in p.topk[t].tolist():
            if i >= 0:
                used.add(int(pt[t // p.w.next_n, i // P]) * P + i % P)
    mask = torch.ones(p.num_slots, dtype=torch.bool)
    mask[list(used)] = False
    dd.kv[mask.cuda()] = 0x7F
    out1, lse1 = dd.run()
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


@pytest.mark.parametrize("wi", [1, 2, 4])
def test_index_order_does_not_change_the_result(small_cases, wi):
    # the result depends on the selected entries, not their order: permuting every token's
    # top-k row changes only the order of the sums
    p, ref = small_cases[SMALL[wi].name]
    dd = DeviceDecode(p)
    out0, lse0 = [x.clone() for x in dd.run()]
    g = torch.Generator().manual_seed(11)
    perm = torch.stack([torch.randperm(p.w.topk, generator=g) for _ in range(p.w.num_tokens)])
    dd.topk = torch.gather(p.topk.cpu().to(torch.int64), 1, perm).to(torch.int32).to(dd.topk.device).contiguous()
    out1, lse1 = dd.run()
    assert_parity(out1, lse1, ref)
    assert (out1.float() - out0.float()).abs().max().item() <= OUT_ATOL
    fin = torch.isfinite(lse0)
    assert torch.equal(fin, torch.isfinite(lse1))
    assert (lse1[fin] - lse0[fin]).abs().max().item() <= 1e-4


@pytest.mark.parametrize("wi,topk,splits", [(1, 320, 1), (2, 448, 3), (1, 1024, 16), (4, 320, 0), (4, 320, 3)])
def test_outputs_stay_inside_their_buffers(wi, topk, splits):
    # out and lse lie between guard bands of a sentinel pattern: the decode writes nothing
    # outside its [T, H, 512] and [T, H] elements, with one split, splits merged inside the
    # cluster, splits through the merge kernel (16 of 64 entries), and the mma.sync kernel
    w = W.small_variant(W.WORKLOADS[wi], num_requests=2, ctx_lo=topk + 100, ctx_hi=topk + 400, topk=topk)
    p = W.make_problem(w)
    dd = DeviceDecode(p, num_splits=splits)
    want_out, want_lse = [x.clone() for x in dd.run()]
    T, H, G = w.num_tokens, w.num_heads, 4096  # G guard elements on each side (16-byte multiples)
    ob = torch.full((G + T * H * 512 + G,), 0x3039, dtype=torch.int16, device="cuda")
    lb = torch.full((G + T * H + G,), -7.0, dtype=torch.float32, device="cuda")
    dd.out = ob[G:G + T * H * 512].view(torch.bfloat16).view(T, H, 512)
    dd.lse = lb[G:G + T * H].view(T, H)
    out, lse = dd.run()
    torch.cuda.synchronize()
    assert (ob[:G] == 0x3039).all() and (ob[G + T * H * 512:] == 0x3039).all()
    assert (lb[:G] == -7.0).all() and (lb[G + T * H:] == -7.0).all()
    assert torch.equal(out, want_out) and torch.equal(lse, want_lse)


def test_page_relabel_is_bitwise_invariant(small_cases):
    p, _ = small_cases[SMALL[1].name]
    dd = DeviceDecode(p, num_splits=1)
    out0, lse0 = [x.clone() for x in dd.run()]
    P = p.w.page_size
    perm = torch.randperm(p.num_pages, generator=torch.Generator().manual_seed(5))  # page q -> perm[q]
    kv2 = torch.empty_like(dd.kv).view(p.num_pages, P, -1)
    kv2[perm.cuda()] = dd.kv.view(p.num_pages, P, -1)
    pt2 = torch.where(p.page_table >= 0, perm[p.page_table.clamp(min=0).long()].to(torch.int32), p.page_table)
    dd.kv = kv2.view(p.num_slots, -1)
    dd.page_table = pt2.cuda()
    out1, lse1 = dd.run()
    assert torch.equal(out0, out1) and torch.equal(lse0, lse1)


def test_padding_placement_and_empty_rows():
    w = W.small_variant(W.WORKLOADS[2], num_requests=3, ctx_lo=300, ctx_hi=300, topk=256)
    p = W.make_problem(w)
    rng = np.random.default_rng(0)
    topk = p.topk.numpy().copy()
    # token 0: 100 valid scattered between -1; token 1: nothing selected; token 2 unchanged
    row = np.full(256, -1, np.int32)
    row[np.sort(rng.permutation(256)[:100])] = topk[0, :100]
    topk[0] = row
    topk[1] = -1
    p.topk = torch.from_numpy(topk)
    ref = oracle_decode(p)
    for s in (1, 3):
        dd = DeviceDecode(p, num_splits=s)
        out, lse = dd.run()
        assert_parity(out, lse, ref)
        assert (out[1] == 0).all()
        assert torch.equal(lse[1].cpu(), p.sink.cpu())  # empty selection: lse = sigma


def test_invalid_entries_are_masked_and_flagged():
    w = W.small_variant(W.WORKLOADS[4], num_requests=2, ctx_lo=500, ctx_hi=500, topk=128)
    p = W.make_problem(w)
    topk = p.topk.clone()
    topk[0, 3] = -7               # negative, not padding
    topk[1, 5] = 64 * 100         # beyond the request's page table
    pt = p.page_table.clone()
    pt[1, -1] = p.num_pages + 3   # a page entry out of range
    topk[1, 9] = 64 * (w.page_table_stride - 1) + 2
    p.topk, p.page_table = topk, pt
    ref = oracle_decode(p)
    assert ref["n_invalid"][0] == 1 and ref["n_invalid"][1] >= 2
    dd = DeviceDecode(p, num_splits=1)
    out, lse = dd.run()
    assert_parity(out, lse, ref)
    err = smla.read_error(dd.desc, dd.workspace)
    assert err == smla.SMLA_DEVERR_INDEX | smla.SMLA_DEVERR_PAGE
    assert smla.read_error(dd.desc, dd.workspace) == 0  # cleared


def test_req_id_per_token():
    w = W.small_variant(W.WORKLOADS[1], num_requests=3, ctx_lo=200, ctx_hi=700, topk=192)
    p = W.make_problem(w)
    # tokens served in reverse request order through an explicit mapping
    req = torch.tensor([2, 1, 0], dtype=torch.int32)
    p2 = W.Problem(**{**p.__dict__, "topk": p.topk[[2, 1, 0]].contiguous(), "q": p.q[[2, 1, 0]].contiguous()})
    dd = DeviceDecode(p2)
    dd.req_id = req.cuda()
    out, lse = dd.run()
    ref = oracle_decode(p)
    order = [2, 1, 0]
    assert_parity(out[order], lse[order], ref)


def test_kernel_events_bracket_the_decode_kernel():
    # the measurement hook records its events around the decode kernel only: the interval
    # is positive and no longer than the whole call (decode + split merge)
    w = W.small_variant(W.WORKLOADS[2], num_requests=2, ctx_lo=2048, ctx_hi=2048, topk=2048)
    dd = DeviceDecode(W.make_problem(w), num_splits=4)
    s = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in evs:
        e.record(s)
    dd.run()
    ref_out = dd.out.clone()
    smla.set_kernel_events(evs[1], evs[2])
    evs[0].record(s)
    dd.run()
    evs[3].record(s)
    smla.set_kernel_events()
    torch.cuda.synchronize()
    k_ms, all_ms = evs[1].elapsed_time(evs[2]), evs[0].elapsed_time(evs[3])
    assert 0.0 < k_ms <= all_ms
    assert torch.equal(dd.out, ref_out)


@pytest.mark.parametrize("wi", [1, 2])
def test_mixed_batch_one_call(wi):
    # one call over requests that contribute 5, 1 and 3 query tokens (a prefill chunk, a
    # decode token, a speculative run), each token with its own causal index set: every
    # token is its own work item, mapped to its request by req_id_per_token, so nothing is
    # padded to the longest request
    w = W.small_variant(W.WORKLOADS[wi], num_requests=3, ctx_lo=300, ctx_hi=700, topk=256).replace(next_n=5)
    p = W.make_problem(w)
    sel = [0, 1, 2, 3, 4, 9, 12, 13, 14]
    req = torch.tensor([0, 0, 0, 0, 0, 1, 2, 2, 2], dtype=torch.int32)
    # buffers sized for 9 tokens; the page table keeps its 3 request rows
    p2 = W.Problem(**{**p.__dict__, "topk": p.topk[sel].contiguous(), "q": p.q[sel].contiguous(),
                      "w": w.replace(num_requests=len(sel), next_n=1)})
    dd = DeviceDecode(p2)
    dd.desc.num_requests = 3
    dd.req_id = req.cuda()
    out, lse = dd.run()
    sink = None if p.sink is None else p.sink.cpu().double().numpy()
    ref = O.decode(_bits(p.q[sel]), OracleCache(p).fetch, w.kv_format, p.page_table.cpu().numpy(),
                   p.topk[sel].cpu().numpy(), w.page_size, p.num_pages, w.sm_scale, sink=sink,
                   req_id_per_token=req.numpy())
    assert_parity(out, lse, ref)


@pytest.mark.parametrize("page_size", [1, 16, 256])
def test_decode_other_page_sizes(page_size):
    w = W.small_variant(W.WORKLOADS[2], num_requests=2, ctx_lo=600, ctx_hi=900, topk=320).replace(
        page_size=page_size, name=f"fp8_P{page_size}")
    p = W.make_problem(w)
    assert_parity(*DeviceDecode(p).run(), oracle_decode(p))


@pytest.mark.parametrize("wi,splits", [(1, 0), (1, 8), (4, 0), (2, 5), (1, 12), (2, 12)])
def test_decode_long_index_rows(wi, splits):
    # 8192 entries per row: more than one split's 2048-entry index list, so at least 4 splits.
    # Up to 8 splits of the tensor-core kernel merge inside a thread-block cluster; 12 take
    # the partials through global memory and the merge kernel.
    w = W.small_variant(W.WORKLOADS[wi], num_requests=1, ctx_lo=9000, ctx_hi=9000, topk=8192,
                        tail_pad=1000 if wi == 4 else 0)
    p = W.make_problem(w)
    assert_parity(*DeviceDecode(p, num_splits=splits).run(), oracle_decode(p))


@pytest.mark.parametrize("wi", [1, 2, 4])  # 64 and 128 heads (tensor-core kernel), 16 heads
@pytest.mark.parametrize("topk", [4, 60, 68])
def test_decode_index_rows_shorter_than_a_tile(wi, topk):
    # fewer entries than one 64-slot tile, and one tile plus a ragged 4; a 40-slot context
    # leaves some rows shorter still, padded with -1
    w = W.small_variant(W.WORKLOADS[wi], num_requests=3, ctx_lo=40, ctx_hi=500, topk=topk)
    p = W.make_problem(w)
    ref = oracle_decode(p)
    for splits in (0, 2):
        assert_parity(*DeviceDecode(p, num_splits=splits).run(), ref)


@pytest.mark.parametrize("wi", [1, 4])
def test_decode_longest_index_row(wi):
    # the largest top-k the library takes, 64 splits of 2048 entries: every split lane of the
    # merge kernel (f16 partials from the tensor-core kernel, fp32 from the mma.sync one)
    w = W.small_variant(W.WORKLOADS[wi], num_requests=1, ctx_lo=131072, ctx_hi=131072, topk=131072)
    p = W.make_problem(w)
    dd = DeviceDecode(p)
    assert smla.plan_launches(dd.desc, 152).num_splits == 64
    assert_parity(*dd.run(), oracle_decode(p))
    assert smla.read_error(dd.desc, dd.workspace) == 0


def test_decode_largest_page_size():
    w = W.small_variant(W.WORKLOADS[2], num_requests=2, ctx_lo=5000, ctx_hi=9000, topk=320).replace(
        page_size=4096, name="fp8_P4096")
    p = W.make_problem(w)
    assert_parity(*DeviceDecode(p).run(), oracle_decode(p))


@pytest.mark.parametrize("heads", [64, 128])
def test_decode_bf16_cache_many_heads(heads):
    w = W.WORKLOADS[0].replace(num_heads=heads, name=f"bf16_H{heads}")
    p = W.make_problem(w)
    for splits in (1, 2):
        assert_parity(*DeviceDecode(p, num_splits=splits).run(), oracle_decode(p))


@pytest.mark.parametrize("wi", [1, 2])
def test_decode_two_tokens_per_request(wi):
    w = W.small_variant(W.WORKLOADS[wi], num_requests=2, ctx_lo=300, ctx_hi=700, topk=256).replace(next_n=2)
    p = W.make_problem(w)
    assert_parity(*DeviceDecode(p).run(), oracle_decode(p))


def test_bounded_wait_runs_out_and_reports():
    # a wait that nothing completes gives up after its limit, sets the timeout bit and
    # returns; the context stays usable for the next decode
    import time
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    smla.selftest_wait_timeout(err, 2000)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert err.item() == smla.SMLA_DEVERR_TIMEOUT
    assert 0.002 <= dt < 1.0
    p = W.make_problem(SMALL[1])
    assert_parity(*DeviceDecode(p).run(), oracle_decode(p))


def test_read_error_status_per_bit():
    # smla_read_error: SMLA_ERR_TIMEOUT (9) whenever the timeout bit is set, else
    # SMLA_ERR_INDEX_RANGE (7) for index/page bits, else SMLA_ERR_OPERAND_RANGE (10)
    import ctypes
    d = smla.make_desc(1, 16, 64, 1, 64, 4, 4, smla.SMLA_KV_FP8_DS, 1 / 24)
    ws = torch.zeros(64, dtype=torch.int32, device="cuda")
    L = smla.lib()

    def status():
        v = ctypes.c_int32(0)
        st = L.smla_read_error(ctypes.byref(d), ctypes.c_void_p(ws.data_ptr()), 256, ctypes.byref(v), None)
        return st, v.value

    smla.selftest_wait_timeout(ws, 1000)
    assert status() == (9, smla.SMLA_DEVERR_TIMEOUT)
    assert status() == (0, 0)  # read clears the word
    for word, st in [(1, 7), (2, 7), (5, 9), (8, 10), (9, 7), (12, 9)]:
        ws[0] = word
        assert status() == (st, word)


@pytest.mark.parametrize("heads,fmt,elem", [(128, smla.SMLA_KV_FP8_DS, 2), (64, smla.SMLA_KV_FP8_TENSOR, 2),
                                            (16, smla.SMLA_KV_FP8_DS, 4), (64, smla.SMLA_KV_BF16, 4)])
def test_workspace_holds_partials_at_their_element_size(heads, fmt, elem):
    # 12 splits merge in the merge kernel: the tensor-core kernel writes f16 partial rows,
    # the mma.sync kernel fp32 ones; the workspace is the error word, the LSEs and the rows
    T, S = 3, 12
    d = smla.make_desc(T, heads, S * 256, T, 64, 64, 64, fmt, 1 / 24, num_splits=S)
    rows = T * S * heads
    assert smla.workspace_size(d) == 256 + (rows * 4 + 255) // 256 * 256 + rows * 512 * elem


def test_plan_query_agrees_with_the_device_workspace():
    # the host-only plan query, given this device's SM count, asks for the workspace the
    # device-side query asks for
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for w in list(W.WORKLOADS) + list(W.EXTRA_WORKLOADS):
        fmt = {"bf16": smla.SMLA_KV_BF16, "fp8_ds": smla.SMLA_KV_FP8_DS, "fp8_tensor": smla.SMLA_KV_FP8_TENSOR}[w.kv_format]
        for splits in (0, 3, 12):
            d = smla.make_desc(w.num_tokens, w.num_heads, w.topk, w.num_requests, w.page_size, 1024, 64, fmt,
                               1 / 24, next_n=w.next_n, num_splits=splits)
            assert smla.plan_launches(d, sms).workspace_bytes == smla.workspace_size(d), (w.name, splits)


# ------------------------------------------------------------------ full-size, sampled


@pytest.mark.parametrize("name", [w.name for w in W.WORKLOADS[1:]] + [w.name for w in W.EXTRA_WORKLOADS])
def test_full_size_sampled_tokens(name):
    w = W.BY_NAME[name]
    p = W.make_problem(w, device="cuda")
    dd = DeviceDecode(p)  # the launch configuration the bench times (library-chosen splits)
    out, lse = dd.run()
    torch.cuda.synchronize()
    T = w.num_tokens
    # a token in every eighth of the batch (so in every wave of CTAs), the last token, and
    # the first and last tokens of the requests with the shortest and longest contexts
    ctx = p.ctx.cpu()
    lo, hi = int(ctx.argmin()), int(ctx.argmax())
    tokens = set(range(0, T, max(1, T // 8))) | {T - 1}
    tokens |= {lo * w.next_n, lo * w.next_n + w.next_n - 1, hi * w.next_n, hi * w.next_n + w.next_n - 1}
    tokens = sorted(tokens)
    ref = oracle_decode(p, tokens=tokens)
    assert_parity(out, lse, ref, tokens=tokens)
    assert torch.isfinite(out.float()).all()
    assert smla.read_error(dd.desc, dd.workspace) == 0
    del dd, p
    torch.cuda.empty_cache()


def test_tail_wave_split_launch():
    # (token, head group) items filling one wave of SMs plus 8: the library runs the last 8
    # items as a second launch of two splits each, merged in their cluster; every token,
    # those of the tail included, against the oracle
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = (sms + 8 + 1) // 2
    w = W.small_variant(W.WORKLOADS[2], num_requests=T, ctx_lo=600, ctx_hi=600, topk=512)
    p = W.make_problem(w)
    dd = DeviceDecode(p)
    out, lse = dd.run()
    torch.cuda.synchronize()
    assert int(dd.workspace[0].item()) == 0
    assert_parity(out, lse, oracle_decode(p))
    # the second launch may start while the first drains: calls back to back on one stream, with
    # another batch's call in between into other buffers, give the same bits
    ref_out, ref_lse = out.clone(), lse.clone()
    w2 = W.small_variant(W.WORKLOADS[2], num_requests=T, ctx_lo=900, ctx_hi=900, topk=512)
    dd2 = DeviceDecode(W.make_problem(w2))
    for _ in range(3):
        dd.run()
        dd2.run()
    torch.cuda.synchronize()
    assert torch.equal(dd.out.view(torch.int16), ref_out.view(torch.int16))
    assert torch.equal(dd.lse, ref_lse)
    out2, lse2 = dd2.out.clone(), dd2.lse.clone()
    dd2.run()
    torch.cuda.synchronize()
    assert torch.equal(dd2.out.view(torch.int16), out2.view(torch.int16)) and torch.equal(dd2.lse, lse2)


@pytest.mark.parametrize("wi,topk,splits", [(1, 320, 1), (2, 448, 3), (1, 1024, 16), (4, 320, 3)])
def test_lse_is_optional(wi, topk, splits):
    # lse = NULL: the output is the same, bit for bit, with one split, splits merged in the
    # cluster, splits through the merge kernel, and the mma.sync kernel
    w = W.small_variant(W.WORKLOADS[wi], num_requests=2, ctx_lo=topk + 100, ctx_hi=topk + 400, topk=topk)
    p = W.make_problem(w)
    want = DeviceDecode(p, num_splits=splits).run()[0].clone()
    dd = DeviceDecode(p, num_splits=splits, with_lse=False)
    out, lse = dd.run()
    torch.cuda.synchronize()
    assert lse is None and torch.equal(out.view(torch.int16), want.view(torch.int16))
    assert smla.read_error(dd.desc, dd.workspace) == 0


def test_decode_on_a_side_stream():
    # the library launches on the caller's stream: on a non-default stream, with the whole-wave
    # and tail launches of the head-group kernel, the result equals the default stream's
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = (sms + 8 + 1) // 2
    w = W.small_variant(W.WORKLOADS[2], num_requests=T, ctx_lo=600, ctx_hi=600, topk=512)
    p = W.make_problem(w)
    dd = DeviceDecode(p)
    assert smla.plan_launches(dd.desc, sms).num_launches == 2
    ref_out, ref_lse = [x.clone() for x in dd.run()]
    torch.cuda.synchronize()
    dd.out.zero_()
    dd.lse.zero_()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        dd.run(side)
    side.synchronize()
    assert torch.equal(dd.out.view(torch.int16), ref_out.view(torch.int16)) and torch.equal(dd.lse, ref_lse)
