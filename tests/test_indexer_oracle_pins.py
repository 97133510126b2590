"""Pins of the indexer oracle (FP8 paged MQA logits + top-k) against hand-worked values,
closed forms, brute force and library routines. CPU only."""
import numpy as np
import pytest
import torch

import oracle as O
from oracle import indexer_oracle as IX

P = 4  # page size of the hand-built caches


def _page(codes: np.ndarray, scales) -> np.ndarray:
    """One cache page: P x 128 codes (slot-major), then P fp32 scales (little-endian)."""
    out = np.zeros(P * 132, dtype=np.uint8)
    out[:P * 128] = np.asarray(codes, dtype=np.uint8).reshape(-1)
    out[P * 128:] = np.asarray(scales, dtype="<f4").view(np.uint8)
    return out


ONE, TWO, HALF, NEG_THREE = 0x38, 0x40, 0x30, 0xC4  # E4M3FN codes of 1, 2, 0.5, -3


def test_e4m3_codes_used_here():
    assert O.e4m3_decode(np.array([ONE, TWO, HALF, NEG_THREE])).tolist() == [1.0, 2.0, 0.5, -3.0]


def test_visible_length_per_query_row():
    # a request of context 10 with next_n = 4 rows: rows see 7, 8, 9, 10 slots
    assert [IX.visible_len(10, 4, i) for i in range(4)] == [7, 8, 9, 10]
    assert [IX.visible_len(5, 1, 0), IX.visible_len(2, 4, 0)] == [5, 0]


def test_page_keys_reads_codes_then_scales():
    codes = np.zeros((P, 128), dtype=np.uint8)
    codes[2, 5] = TWO
    page = _page(codes, [1.0, 0.25, 8.0, 0.5])
    c, s = IX.page_keys(page, P)
    assert c[2, 5] == TWO and c.sum() == TWO and s.tolist() == [1.0, 0.25, 8.0, 0.5]


def test_single_head_closed_form_with_relu():
    # q = e_0 (value 1), key dim 0 = 2 or -3: logit = w * max(0, scale * k_0)
    q = np.zeros((1, 128), dtype=np.uint8)
    q[0, 0] = ONE
    keys = np.zeros((2, 128))
    keys[0, 0], keys[1, 0] = 2.0, -3.0
    lg = IX.logits_of_token(q, np.array([1.5]), keys, np.array([0.25, 4.0]))
    assert lg.tolist() == [1.5 * 0.5, 0.0]


def test_logits_match_brute_force_loops():
    rng = np.random.default_rng(3)
    H, n = 3, 5
    q = rng.integers(0, 0x7F, size=(H, 128)).astype(np.uint8)  # finite codes, both signs below
    q[:, ::2] |= 0x80
    keys_codes = rng.integers(0, 0x7F, size=(n, 128)).astype(np.uint8)
    keys_codes[1::2] |= 0x80
    keys = O.e4m3_decode(keys_codes)
    sc = np.array([0.5, 1.0, 2.0 ** -6, 3.0, 0.125])
    w = np.array([0.3, -1.25, 2.0])
    qv = O.e4m3_decode(q)
    brute = []
    for s in range(n):
        tot = 0.0
        for h in range(H):
            dot = 0.0
            for d in range(128):
                dot += float(qv[h, d]) * float(keys[s, d])
            tot += w[h] * max(0.0, sc[s] * dot)
        brute.append(tot)
    np.testing.assert_allclose(IX.logits_of_token(q, w, keys, sc), brute, rtol=1e-13, atol=0)


def test_logits_match_torch_float8_decode():
    g = torch.Generator().manual_seed(9)
    q8 = torch.randn(64, 128, generator=g).to(torch.float8_e4m3fn)
    k8 = (torch.randn(40, 128, generator=g) * 32).to(torch.float8_e4m3fn)
    sc = torch.exp2(torch.randint(-10, -3, (40,), generator=g).double())
    w = torch.randn(64, generator=g, dtype=torch.float64) / 8
    ref = (w[:, None] * torch.relu((q8.double() @ k8.double().T) * sc[None, :])).sum(0)
    got = IX.logits_of_token(q8.view(torch.uint8).numpy(), w.numpy(), k8.double().numpy(), sc.numpy())
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_logits_follow_the_page_table():
    # request pages [1, 0]: slots 0..3 in physical page 1, slots 4..7 in page 0
    p0 = np.zeros((P, 128), dtype=np.uint8)
    p1 = np.zeros((P, 128), dtype=np.uint8)
    p0[:, 0] = TWO       # slots 4..7: key dim 0 = 2
    p1[:, 0] = HALF      # slots 0..3: key dim 0 = 0.5
    cache = np.stack([_page(p0, [1.0] * P), _page(p1, [2.0] * P)])
    q = np.zeros((1, 1, 128), dtype=np.uint8)
    q[0, 0, 0] = ONE
    lg = IX.indexer_logits(q, np.ones((1, 1)), cache, np.array([[1, 0]]), ctx=[7], next_n=1, page_size=P)[0]
    assert lg.tolist() == [1.0] * 4 + [2.0] * 3  # 0.5 * scale 2, then 2 * scale 1; 7 visible


def test_next_n_rows_see_their_causal_prefix():
    cache = np.stack([_page(np.full((P, 128), ONE, dtype=np.uint8), [1.0] * P)] * 3)
    q = np.zeros((3, 1, 128), dtype=np.uint8)
    q[:, 0, 0] = ONE
    lg = IX.indexer_logits(q, np.ones((3, 1)), cache, np.array([[0, 1, 2]]), ctx=[10], next_n=3, page_size=P)
    assert [len(x) for x in lg] == [8, 9, 10]


def test_topk_set_distinct_values_match_argpartition():
    rng = np.random.default_rng(1)
    x = rng.permutation(1000).astype(np.float64)
    got = IX.topk_set(x, 37)
    ref = np.sort(np.argpartition(-x, 37)[:37])
    assert np.array_equal(got, ref)


def test_topk_set_ties_and_short_rows():
    assert IX.topk_set(np.array([1.0, 3.0, 3.0, 2.0]), 2).tolist() == [1, 2]
    assert IX.topk_set(np.array([3.0, 1.0, 3.0]), 1).tolist() == [0]  # lower index first at a tie
    assert IX.topk_set(np.array([5.0, -1.0]), 4).tolist() == [0, 1]   # fewer than k: all
