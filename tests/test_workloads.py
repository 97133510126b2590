"""Host checks of the seeded workload generator (CPU)."""
import torch

import workloads as W


def test_tiny_workload_shapes_and_indices():
    w = W.WORKLOADS[0]
    p = W.make_problem(w)
    assert p.q.shape == (2, 16, 576) and p.q.dtype == torch.bfloat16
    assert p.kv_bf16.shape == (4, 64, 576)
    assert p.page_table.shape == (2, 4)
    for r in range(2):
        assert sorted(p.page_table[r].tolist()) == [0, 1, 2, 3]
    for t in range(2):
        row = p.topk[t]
        assert (row >= 0).all() and len(set(row.tolist())) == 128 and row.max() < 256


def test_padded_tail_and_distinct():
    w = W.small_variant(W.WORKLOADS[4], num_requests=3, ctx_lo=300, ctx_hi=900, topk=256, tail_pad=51)
    p = W.make_problem(w)
    for t in range(p.topk.shape[0]):
        row = p.topk[t].tolist()
        valid = [x for x in row if x != -1]
        assert row[len(valid):] == [-1] * (256 - len(valid))
        assert len(valid) == 205 and len(set(valid)) == 205
        assert max(valid) < int(p.ctx[t])


def test_mtp_causal_prefix_and_page_pool():
    w = W.small_variant(W.WORKLOADS[3], num_requests=2, ctx_lo=100, ctx_hi=130, topk=160)
    p = W.make_problem(w)
    assert p.topk.shape == (8, 160)
    for t in range(8):
        r, i = divmod(t, 4)
        visible = int(p.ctx[r]) - 3 + i
        valid = [x for x in p.topk[t].tolist() if x != -1]
        assert len(valid) == min(visible, 160) and max(valid) < visible
    used = [x for x in p.page_table.flatten().tolist() if x != -1]
    assert sorted(used) == list(range(p.num_pages))


def test_raw_chunk_is_reproducible():
    w = W.small_variant(W.WORKLOADS[1], num_requests=2, ctx_lo=200, ctx_hi=300, topk=64)
    a = W.make_problem(w)
    b = W.make_problem(w)
    la, ra = a.raw_chunk(0)
    lb, rb = b.raw_chunk(0)
    assert torch.equal(la, lb) and torch.equal(ra, rb)
    pages = [0, 2]
    lat, rope = a.raw_pages(pages)
    assert torch.equal(lat[64:128], la[128:192]) and torch.equal(rope[:64], ra[:64])


def test_per_tensor_fp8_workload_shape():
    w = W.BY_NAME["fp8tensor_T32_H64_K2048_ctx1k-32k"]
    assert w.kv_format == "fp8_tensor" and w.row_bytes == 576 and w.kv_scale == 1.0
    small = W.small_variant(w, num_requests=2, ctx_lo=100, ctx_hi=300, topk=128)
    p = W.make_problem(small)
    assert p.topk.shape == (2, 128) and p.q.shape == (2, 64, 576)


def test_magnitude_gains_multiply_the_draw_before_rounding():
    base = W.small_variant(W.WORKLOADS[2], num_requests=2, ctx_lo=300, ctx_hi=300, topk=64)
    w = base.replace(q_gains=(1e5, 1.0), q_dim_gains=(1.0, 1e-3), latent_gains=(1e-4, 2.0, 3.0),
                     rope_gains=(7.0,))
    p0, p1 = W.make_problem(base), W.make_problem(w)
    q0, q1 = p0.q.float(), p1.q.float()
    # same draw: q1 = bf16(q_f32 * gain); compare against the bf16 rounding of the gained draw
    assert torch.equal(torch.sign(q0), torch.sign(q1))
    assert torch.allclose(q1[:, 0, 0], q0[:, 0, 0] * 1e5, rtol=1e-2)
    assert torch.allclose(q1[:, 1, 1], q0[:, 1, 1] * 1e-3, rtol=1e-2)
    lat0, rope0 = p0.raw_chunk(0)
    lat1, rope1 = p1.raw_chunk(0)
    assert torch.allclose(lat1[0].float(), lat0[0].float() * 1e-4, rtol=1e-2)
    assert torch.allclose(lat1[4].float(), lat0[4].float() * 2.0, rtol=1e-2)
    assert torch.allclose(rope1[5].float(), rope0[5].float() * 7.0, rtol=1e-2)


def test_oracle_cache_fetches_the_row_of_each_physical_slot():
    # the oracle's cache of a problem returns, for physical slot s, the packed source row of
    # page s // P at position s % P, whatever the order the slots are asked in
    import numpy as np

    import oracle as O
    from oracle.workload_oracle import OracleCache

    w = W.small_variant(W.WORKLOADS[2], num_requests=2, ctx_lo=300, ctx_hi=700, topk=128)
    p = W.make_problem(w)
    cache = OracleCache(p)
    P = w.page_size
    pages = sorted({int(x) for x in p.page_table.flatten().tolist() if 0 <= x < p.num_pages})
    g = np.random.default_rng(5)
    slots = np.array([pg * P + int(g.integers(P)) for pg in g.permutation(pages)[:12]], dtype=np.int64)
    got = cache.fetch(slots)
    for k, s in enumerate(slots.tolist()):
        lat, rope = p.raw_pages([s // P])
        bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
        want = O.pack_fp8_ds(bits(lat[s % P:s % P + 1]), bits(rope[s % P:s % P + 1]))
        assert np.array_equal(got[k], want[0]), s
