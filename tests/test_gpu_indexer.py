"""GPU parity of the indexer (FP8 paged MQA logits + top-k) against the float64 oracle,
through the C ABI.

Logits: the oracle's values are exact up to the final weighted sum; the kernel accumulates
dot products and the head sum in fp32, so each logit must lie within 1e-4 of the sum of the
absolute values of its terms (sum_h |w_h| |scale| sum_d |q_hd k_d|). Top-k: given the same
fp32 logits, the kernel's index set must equal the oracle's bit for bit (both take the lowest
indices at a tie); on the kernel's own logits, every selected slot must be within that bound
of the K-th largest oracle logit, and every slot clearly above it must be selected.
"""
import numpy as np
import pytest
import torch

import oracle as O
import sparse_mla_decode_smla_gb300 as smla
import workloads as W
from oracle import indexer_oracle as IX
from oracle.workload_oracle import oracle_decode
from sparse_mla_decode_smla_gb300.runner import DeviceDecode

pytestmark = pytest.mark.gpu

REL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    smla.lib()


class Indexer:
    """Device buffers and calls of one indexer batch."""

    def __init__(self, problem, heads=W.INDEX_HEADS, topk=None, logits_stride=None, ctx=None):
        w = problem.w
        self.p = problem
        self.ix = W.make_indexer_inputs(problem, heads=heads, device="cuda")
        if ctx is not None:
            self.ix.ctx = torch.tensor(ctx, dtype=torch.int32, device="cuda")
        self.stride = logits_stride or w.page_table_stride * w.page_size
        self.K = topk or w.topk
        self.desc = smla.make_indexer_desc(w.num_requests, w.next_n, heads, w.page_size, problem.num_pages,
                                           w.page_table_stride, self.stride, self.K)
        self.pt = problem.page_table.to(device="cuda", dtype=torch.int32).contiguous()
        self.logits = torch.full((w.num_tokens, self.stride), float("nan"), device="cuda")
        self.topk = torch.full((w.num_tokens, self.K), -7, dtype=torch.int32, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(self):
        smla.indexer_logits(self.desc, self.ix.q, self.ix.weights, self.ix.cache, self.pt, self.ix.ctx,
                            self.logits, self.err)
        smla.indexer_topk(self.desc, self.logits, self.ix.ctx, self.topk)
        torch.cuda.synchronize()
        return self.logits, self.topk

    def oracle(self, tokens=None):
        """(logits, absolute-term bounds) of the listed tokens, float64."""
        w = self.p.w
        ctx = self.ix.ctx.cpu().numpy()
        q = self.ix.q.cpu().numpy()
        wt = self.ix.weights.cpu().double().numpy()
        tokens = range(w.num_tokens) if tokens is None else tokens
        pt = self.p.page_table.cpu().numpy()
        cache = self.ix.cache
        out = {}
        for t in tokens:
            r, i = divmod(t, w.next_n)
            n = IX.visible_len(ctx[r], w.next_n, i)
            pages = sorted({int(pt[r][s // w.page_size]) for s in range(0, n, w.page_size)})
            host = {pg: cache[pg].cpu().numpy() for pg in pages}
            keys = np.zeros((n, 128))
            sc = np.zeros(n)
            for s0 in range(0, n, w.page_size):
                codes, scales = IX.page_keys(host[int(pt[r][s0 // w.page_size])], w.page_size)
                m = min(w.page_size, n - s0)
                keys[s0:s0 + m] = O.e4m3_decode(codes[:m])
                sc[s0:s0 + m] = scales[:m]
            lg = IX.logits_of_token(q[t], wt[t], keys, sc)
            qa = np.abs(O.e4m3_decode(q[t]))
            bound = np.abs(wt[t]) @ (qa @ np.abs(keys).T) * np.abs(sc)[None, :] if n else np.zeros(0)
            out[t] = (lg, np.asarray(bound).reshape(-1))
        return out


def _check_logits(gpu_row, ref, bound):
    n = ref.shape[0]
    g = gpu_row[:n].double().cpu().numpy()
    assert np.isfinite(g).all()
    err = np.abs(g - ref)
    assert (err <= REL * bound + 1e-30).all(), f"max err / bound {np.max(err / np.maximum(bound, 1e-30))}"


def _check_topk_valid(sel, ref, bound, K):
    n = ref.shape[0]
    sel = sel.cpu().numpy()
    if n <= K:
        assert np.array_equal(sel, np.concatenate([np.arange(n), -np.ones(K - n, dtype=np.int64)]))
        return
    assert len(set(sel.tolist())) == K and sel.min() >= 0 and sel.max() < n
    assert np.all(np.diff(sel) > 0)  # ascending
    tau = np.sort(ref)[-K]
    tol = REL * bound.max()
    assert (ref[sel] >= tau - 2 * tol).all()
    chosen = np.zeros(n, dtype=bool)
    chosen[sel] = True
    assert chosen[ref > tau + 2 * tol].all()


SMALL = [
    (W.small_variant(W.WORKLOADS[2], num_requests=3, ctx_lo=300, ctx_hi=2600, topk=512), 64),
    (W.small_variant(W.WORKLOADS[3], num_requests=2, ctx_lo=1500, ctx_hi=3000, topk=256), 64),  # next_n = 4
    (W.small_variant(W.WORKLOADS[3], num_requests=3, ctx_lo=200, ctx_hi=1100, topk=256), 32),
]


@pytest.mark.parametrize("wi", range(len(SMALL)))
def test_logits_and_topk_match_oracle(wi):
    w, heads = SMALL[wi]
    ix = Indexer(W.make_problem(w), heads=heads)
    logits, topk = ix.run()
    assert ix.err.item() == 0
    for t, (ref, bound) in ix.oracle().items():
        _check_logits(logits[t], ref, bound)
        _check_topk_valid(topk[t], ref, bound, ix.K)


@pytest.mark.parametrize("page_size", [16, 32, 128])
def test_other_page_sizes(page_size):
    w = W.small_variant(W.WORKLOADS[3], num_requests=2, ctx_lo=700, ctx_hi=1300, topk=256).replace(
        page_size=page_size)
    ix = Indexer(W.make_problem(w))
    logits, topk = ix.run()
    assert ix.err.item() == 0
    for t, (ref, bound) in ix.oracle().items():
        _check_logits(logits[t], ref, bound)
        _check_topk_valid(topk[t], ref, bound, ix.K)


def test_topk_bit_exact_on_given_logits_with_ties():
    # the same fp32 logits on both sides: many ties, some rows shorter than K
    w = W.small_variant(W.WORKLOADS[3], num_requests=3, ctx_lo=100, ctx_hi=5000, topk=300)
    p = W.make_problem(w)
    ix = Indexer(p)
    g = torch.Generator().manual_seed(4)
    stride = ix.stride
    vals = torch.randint(-40, 40, (w.num_tokens, stride), generator=g).float() / 4  # heavy ties
    vals[1] = torch.randn(stride, generator=g)                                     # distinct values
    vals[2, :] = 1.5                                                               # all equal
    ix.logits.copy_(vals.cuda())
    smla.indexer_topk(ix.desc, ix.logits, ix.ix.ctx, ix.topk)
    torch.cuda.synchronize()
    ctx = ix.ix.ctx.cpu().numpy()
    for t in range(w.num_tokens):
        r, i = divmod(t, w.next_n)
        n = IX.visible_len(ctx[r], w.next_n, i)
        ref = IX.topk_set(vals[t, :n].double().numpy(), ix.K)
        want = np.concatenate([ref, -np.ones(ix.K - len(ref), dtype=np.int64)])
        assert np.array_equal(ix.topk[t].cpu().numpy(), want), t


def test_short_empty_and_overlong_contexts():
    w = W.small_variant(W.WORKLOADS[3], num_requests=3, ctx_lo=600, ctx_hi=600, topk=512)
    p = W.make_problem(w)
    # request 0: 2 slots (its 4 query rows see 0, 0, 1 and 2 of them), request 1: 300 (fewer
    # than K), request 2: longer than its page table (served up to stride * P, flagged)
    ix = Indexer(p, ctx=[2, 300, 5000])
    logits, topk = ix.run()
    assert ix.err.item() == smla.SMLA_DEVERR_INDEX
    assert (topk[0:2] == -1).all()
    assert topk[2, 0].item() == 0 and (topk[2, 1:] == -1).all()
    assert topk[3, :2].tolist() == [0, 1] and (topk[3, 2:] == -1).all()
    assert topk[4, :297].tolist() == list(range(297)) and (topk[4, 297:] == -1).all()
    for t, (ref, bound) in ix.oracle(tokens=[4, 5, 6, 7]).items():
        _check_logits(logits[t], ref, bound)


def test_invalid_page_entry_is_flagged():
    w = W.small_variant(W.WORKLOADS[3], num_requests=2, ctx_lo=900, ctx_hi=900, topk=256)
    p = W.make_problem(w)
    ix = Indexer(p)
    ix.pt[1, 3] = 10 ** 7  # a page the visible context needs, outside the pool
    ix.run()
    assert ix.err.item() == smla.SMLA_DEVERR_PAGE
    # request 0 is untouched
    for t, (ref, bound) in ix.oracle(tokens=[0, 3]).items():
        _check_logits(ix.logits[t], ref, bound)


def test_full_size_mtp_batch_sampled():
    # the MTP decode batch's shape: 64 requests x 4 query rows, 4k-128k contexts, top-k 2048
    w = W.WORKLOADS[3]
    p = W.make_problem(w, device="cuda")
    ix = Indexer(p)
    logits, topk = ix.run()
    assert ix.err.item() == 0
    ctx = ix.ix.ctx.cpu()
    lo, hi = int(ctx.argmin()), int(ctx.argmax())
    tokens = sorted({0, 77, 130, 255, 4 * lo, 4 * hi + 3})
    for t, (ref, bound) in ix.oracle(tokens=tokens).items():
        _check_logits(logits[t], ref, bound)
        _check_topk_valid(topk[t], ref, bound, ix.K)


def test_indexer_topk_feeds_the_decode():
    # the decode consumes the indexer's top-k as its index rows; its output against the oracle
    # decode on those same indices
    w = W.small_variant(W.WORKLOADS[3], num_requests=2, ctx_lo=1200, ctx_hi=2500, topk=512)
    p = W.make_problem(w)
    ix = Indexer(p)
    _, topk = ix.run()
    p.topk = topk.cpu()
    dd = DeviceDecode(p)
    out, lse = dd.run()
    torch.cuda.synchronize()
    ref = oracle_decode(p)
    o = out.double().cpu().numpy()
    assert np.abs(o - ref["out"]).max() <= 1e-2
    assert np.abs(lse.double().cpu().numpy() - ref["lse"]).max() <= 1e-3


def test_topk_threshold_bin_at_and_over_the_shared_buffer():
    # 20,003 visible slots a token. The kernel gathers the keys of the threshold's 12-bit bin into
    # a shared-memory buffer of 12,288; with more, its last two radix passes read global memory.
    # Token 0: every key in one bin (values in [1, 1.125): one sign, exponent and top three
    # mantissa bits). Token 1: exactly 12,288 keys in that bin, the rest below it. Token 2: one
    # more. Given fp32 logits, each index set must equal the oracle's bit for bit.
    w = W.small_variant(W.WORKLOADS[3], num_requests=3, ctx_lo=20003, ctx_hi=20003, topk=2048).replace(next_n=1)
    p = W.make_problem(w)
    ix = Indexer(p)
    g = torch.Generator().manual_seed(11)
    n = ix.stride
    vals = 1.0 + torch.randint(0, 1 << 20, (w.num_tokens, n), generator=g).float() * 2.0 ** -23
    vals[:, ::7] = 1.0  # ties at the bottom of the bin
    vals[1, 12288:] = 0.25
    vals[2, 12289:] = 0.25
    ix.logits.copy_(vals.cuda())
    smla.indexer_topk(ix.desc, ix.logits, ix.ix.ctx, ix.topk)
    torch.cuda.synchronize()
    ctx = ix.ix.ctx.cpu().numpy()
    for t in range(w.num_tokens):
        vis = IX.visible_len(ctx[t], 1, 0)
        assert vis == 20003
        ref = IX.topk_set(vals[t, :vis].double().numpy(), ix.K)
        assert np.array_equal(ix.topk[t].cpu().numpy(), ref), t
    # all keys equal (more than the buffer holds): the lowest K indices
    ix.logits.fill_(2.5)
    smla.indexer_topk(ix.desc, ix.logits, ix.ix.ctx, ix.topk)
    torch.cuda.synchronize()
    for t in range(w.num_tokens):
        assert np.array_equal(ix.topk[t].cpu().numpy(), np.arange(ix.K)), t


@pytest.mark.parametrize("extra", [1, 3])
def test_topk_rows_at_every_alignment(extra):
    # a logits row stride that is not a multiple of four floats puts successive rows at each
    # 4-byte offset from a 16-byte boundary (the kernel reads the aligned body 16 bytes at a time
    # and the ends one key at a time); given fp32 logits the index sets must equal the oracle's
    w = W.small_variant(W.WORKLOADS[3], num_requests=3, ctx_lo=2500, ctx_hi=9000, topk=512)
    p = W.make_problem(w)
    ix = Indexer(p, logits_stride=w.page_table_stride * w.page_size + extra)
    g = torch.Generator().manual_seed(5)
    vals = torch.randint(-30, 30, (w.num_tokens, ix.stride), generator=g).float() / 8  # ties
    vals[1::3] = torch.randn(ix.stride, generator=g)                                   # distinct values
    ix.logits.copy_(vals.cuda())
    smla.indexer_topk(ix.desc, ix.logits, ix.ix.ctx, ix.topk)
    torch.cuda.synchronize()
    ctx = ix.ix.ctx.cpu().numpy()
    offsets = set()
    for t in range(w.num_tokens):
        r, i = divmod(t, w.next_n)
        n = IX.visible_len(ctx[r], w.next_n, i)
        offsets.add((t * ix.stride) % 4)
        ref = IX.topk_set(vals[t, :n].double().numpy(), ix.K)
        want = np.concatenate([ref, -np.ones(ix.K - len(ref), dtype=np.int64)])
        assert np.array_equal(ix.topk[t].cpu().numpy(), want), t
    assert offsets == {0, 1, 2, 3}


def test_topk_signed_zeros_are_one_value():
    # -0.0 and +0.0 are the same value: where the K-th largest logit is zero, the zeros of either
    # sign tie and the lowest indices are taken (the oracle's stable sort on values)
    w = W.small_variant(W.WORKLOADS[3], num_requests=2, ctx_lo=1500, ctx_hi=4000, topk=300)
    p = W.make_problem(w)
    ix = Indexer(p)
    g = torch.Generator().manual_seed(9)
    shape = (w.num_tokens, ix.stride)
    zeros = torch.where(torch.rand(shape, generator=g) < 0.5, torch.tensor(-0.0), torch.tensor(0.0))
    vals = torch.where(torch.rand(shape, generator=g) < 0.03, torch.tensor(1.0), zeros)
    vals[:, 7] = -1.0
    assert (torch.signbit(vals) & (vals == 0)).any()
    ix.logits.copy_(vals.cuda())
    smla.indexer_topk(ix.desc, ix.logits, ix.ix.ctx, ix.topk)
    torch.cuda.synchronize()
    ctx = ix.ix.ctx.cpu().numpy()
    for t in range(w.num_tokens):
        r, i = divmod(t, w.next_n)
        n = IX.visible_len(ctx[r], w.next_n, i)
        ref = IX.topk_set(vals[t, :n].double().numpy(), ix.K)
        assert (vals[t, :n] == 1.0).sum() < ix.K  # the threshold is zero
        assert np.array_equal(ix.topk[t].cpu().numpy(), ref), t


def test_topk_more_tokens_than_sms_longest_first():
    # more tokens than SMs: the kernel takes the longest rows first (CTA b serves the token with
    # the b-th longest row); every token's index set must still equal the oracle's, given the
    # same fp32 logits
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    w = W.small_variant(W.WORKLOADS[3], num_requests=sms + 48, ctx_lo=2100, ctx_hi=9000, topk=2048).replace(next_n=1)
    p = W.make_problem(w)
    ix = Indexer(p)
    g = torch.Generator().manual_seed(13)
    vals = torch.randint(-200, 200, (w.num_tokens, ix.stride), generator=g).float() / 16  # ties
    ix.logits.copy_(vals.cuda())
    smla.indexer_topk(ix.desc, ix.logits, ix.ix.ctx, ix.topk)
    torch.cuda.synchronize()
    ctx = ix.ix.ctx.cpu().numpy()
    assert w.num_tokens > sms and len(set(ctx.tolist())) > 1
    got = ix.topk.cpu().numpy()
    for t in range(w.num_tokens):
        n = IX.visible_len(ctx[t], 1, 0)
        ref = IX.topk_set(vals[t, :n].double().numpy(), ix.K)
        want = np.concatenate([ref, -np.ones(ix.K - len(ref), dtype=np.int64)])
        assert np.array_equal(got[t], want), t
