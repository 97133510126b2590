"""Pins for the float64 oracle: each checks it against something other than itself.

Library routines (torch's float8_e4m3fn and bfloat16 casts, torch SDPA in
float64, numpy's IEEE float32 division, np.logaddexp), closed forms of
softmax attention, hand-derived addressing examples and invariances that the
definition implies. CPU only.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O


def _bits(t_bf16: torch.Tensor) -> np.ndarray:
    return t_bf16.contiguous().view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------- e4m3

def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_e4m3_decode_spec_points():
    # OCP 8-bit floating point specification, E4M3 table: max normal 448 = S.1111.110,
    # min normal 2^-6 = S.0001.000, max subnormal 0.875 * 2^-6, min subnormal 2^-9,
    # NaN = S.1111.111, 1.0 = S.0111.000.
    v = O.e4m3_decode(np.array([0x7E, 0x08, 0x07, 0x01, 0x38, 0x80, 0xFE], dtype=np.uint8))
    assert v.tolist() == [448.0, 2.0 ** -6, 0.875 * 2.0 ** -6, 2.0 ** -9, 1.0, -0.0, -448.0]
    assert np.signbit(v[5])
    assert np.isnan(O.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_e4m3_encode_roundtrips_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(O.e4m3_encode_rne_satfinite(O.e4m3_decode(codes)), codes)


def test_e4m3_encode_ties_go_to_even_code():
    pos = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2  # exact in float64
    got = O.e4m3_encode_rne_satfinite(mids).astype(int)
    lo = np.arange(0x7E)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, expect)
    # just off the midpoint goes to the nearer neighbour
    eps = np.ldexp(1.0, -30)
    assert np.array_equal(O.e4m3_encode_rne_satfinite(mids - eps).astype(int), lo)
    assert np.array_equal(O.e4m3_encode_rne_satfinite(mids + eps).astype(int), lo + 1)


def test_e4m3_encode_matches_torch_in_range():
    g = torch.Generator().manual_seed(7)
    x = torch.cat([torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = x.clamp(-448, 448).to(torch.float32)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode_rne_satfinite(x.to(torch.float64).numpy())
    assert np.array_equal(got, ref)


def test_e4m3_encode_saturates_and_keeps_zero_sign():
    big = np.array([448.0, 449.0, 463.99, 464.0, 500.0, 1e30, np.inf])
    assert (O.e4m3_encode_rne_satfinite(big) == 0x7E).all()
    assert (O.e4m3_encode_rne_satfinite(-big) == 0xFE).all()
    assert O.e4m3_encode_rne_satfinite(np.array([-0.0, -1e-9, 1e-9]))[:3].tolist() == [0x80, 0x80, 0x00]
    assert O.e4m3_encode_rne_satfinite(np.array([np.nan]))[0] == 0x7F


def test_bf16_decode_matches_torch():
    bits = np.random.default_rng(1).integers(0, 1 << 16, 5000, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = O.bf16_bits_to_f64(bits)
    both = ~np.isnan(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[both], ref[both])


# ----------------------------------------------------------------------------- pack

def _rand_latent(n, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, 512, generator=g)
    x = x * (2.0 ** torch.randint(-20, 20, (n, 4, 1), generator=g)).repeat_interleave(128, 2).view(n, 512)
    x[0, :128] = 0.0  # an all-zero block
    x[1, 128:256] = 448.0 * 2.0 ** -3  # a block whose amax/448 is an exact power of two
    return x.to(torch.bfloat16)


def test_pack_pow2_scales_and_bound():
    lat = _rand_latent(64)
    rope = torch.randn(64, 64).to(torch.bfloat16)
    rows = O.pack_fp8_ds(_bits(lat), _bits(rope), O.SCALE_POW2)
    assert rows.shape == (64, 656)
    sc = rows[:, 512:528].copy().view("<f4").astype(np.float64)
    x = lat.to(torch.float64).numpy().reshape(64, 4, 128)
    amax = np.abs(x).max(axis=2)
    m, _ = np.frexp(sc)
    assert (m == 0.5).all()  # powers of two
    nz = amax > 0
    # smallest power of two with amax / scale <= 448
    assert (amax[nz] / sc[nz] <= 448).all() and (amax[nz] / sc[nz] > 224).all()
    assert (sc[~nz] == 1.0).all()
    assert sc[1, 1] == 2.0 ** -3  # amax/448 exactly a power of two -> that power
    codes = rows[:, :512]
    assert not np.isnan(O.e4m3_decode(codes)).any()
    deq = O.e4m3_decode(codes).reshape(64, 4, 128) * sc[:, :, None]
    # RNE into e4m3: half an ulp, i.e. 2^-4 relative in the normal range, 2^-10*scale below it
    err = np.abs(deq - x)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * sc[:, :, None])
    assert (err <= bound).all()
    assert np.array_equal(rows[:, 528:].copy().view("<u2"), _bits(rope))


def test_pack_fp32_scale_is_ieee_quotient():
    lat = _rand_latent(32, seed=3)
    rows = O.pack_fp8_ds(_bits(lat), _bits(torch.zeros(32, 64, dtype=torch.bfloat16)), O.SCALE_FP32)
    sc = rows[:, 512:528].copy().view("<f4")
    amax = np.abs(lat.to(torch.float32).numpy().reshape(32, 4, 128)).max(axis=2).astype(np.float32)
    expect = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0))  # numpy IEEE fp32 divide
    assert np.array_equal(sc, expect)
    # codes are RNE(fp32 quotient) with saturation, checked through torch's cast
    q = (lat.to(torch.float32).view(32, 4, 128) / torch.from_numpy(sc.copy())[:, :, None]).clamp(-448, 448)
    ref = q.to(torch.float8_e4m3fn).view(torch.uint8).view(32, 512).numpy()
    assert np.array_equal(rows[:, :512], ref)


def test_pack_bf16_layout():
    lat = torch.randn(5, 512).to(torch.bfloat16)
    rope = torch.randn(5, 64).to(torch.bfloat16)
    rows = O.pack_bf16(_bits(lat), _bits(rope))
    assert rows.shape == (5, 1152)
    back = rows.view("<u2").reshape(5, 576)
    assert np.array_equal(back[:, :512], _bits(lat)) and np.array_equal(back[:, 512:], _bits(rope))


@pytest.mark.parametrize("kv_scale", [1.0, 2.0 ** -6, 0.0137])
def test_pack_fp8_tensor_matches_torch_cast(kv_scale):
    # codes are torch's float8_e4m3fn cast of the fp32 quotient x / kv_scale (in range)
    g = torch.Generator().manual_seed(21)
    lat = torch.randn(200, 512, generator=g).to(torch.bfloat16)
    rope = torch.randn(200, 64, generator=g).to(torch.bfloat16)
    rows = O.pack_fp8_tensor(_bits(lat), _bits(rope), kv_scale)
    assert rows.shape == (200, 576) and rows.dtype == np.uint8
    x = torch.cat([lat, rope], 1).to(torch.float32)
    quot = (x / torch.tensor(kv_scale, dtype=torch.float32))
    assert quot.abs().max() < 448
    ref = quot.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(rows, ref)


def test_pack_fp8_tensor_saturates_and_scales_by_powers_of_two():
    lat = torch.full((2, 512), 3.0).to(torch.bfloat16)
    lat[1, :] = -1000.0
    rope = torch.zeros(2, 64).to(torch.bfloat16)
    rows = O.pack_fp8_tensor(_bits(lat), _bits(rope), 1.0)
    assert (rows[1, :512] == 0xFE).all() and (rows[:, 512:] == 0).all()
    # x / s with s a power of two is exact: scaling x and s together leaves the codes
    x = torch.randn(50, 576, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    a = O.pack_fp8_tensor(_bits(x[:, :512]), _bits(x[:, 512:]), 2.0 ** -4)
    xb = (x.to(torch.float32) * 8).to(torch.bfloat16)
    b = O.pack_fp8_tensor(_bits(xb[:, :512]), _bits(xb[:, 512:]), 2.0 ** -1)
    assert np.array_equal(a, b)


def test_dequant_fp8_tensor_matches_torch():
    codes = np.random.default_rng(9).integers(0, 256, (300, 576), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x3C  # no NaN codes
    for s in (1.0, 0.0137, 2.0 ** -9):
        got = O.dequant_rows(codes, "fp8_tensor", s)
        assert np.array_equal(got, _torch_tensor_keys(codes, s).numpy())


def test_dequant_rows_fp8_is_fp32_product():
    lat = _rand_latent(16, seed=5)
    rows = O.pack_fp8_ds(_bits(lat), _bits(torch.randn(16, 64).to(torch.bfloat16)), O.SCALE_FP32)
    k = O.dequant_rows(rows, "fp8_ds")
    codes = torch.from_numpy(rows[:, :512].copy()).view(torch.float8_e4m3fn).to(torch.float32)
    sc = torch.from_numpy(rows[:, 512:528].copy().view("<f4").copy()).repeat_interleave(128, 1)
    assert np.array_equal(k[:, :512], (codes * sc).to(torch.float64).numpy())  # torch fp32 multiply


# ----------------------------------------------------------------------------- addressing

def test_physical_slots_hand_example():
    # page size 4, request pages [2, 0, 1]; index 5 -> page 0 slot 1; 0 -> page 2 slot 0;
    # 11 -> page 1 slot 3.  Physical = page * 4 + offset.
    keep, phys, bad = O.physical_slots(np.array([5, -1, 0, 11]), np.array([2, 0, 1]), 4, 3)
    assert keep == [0, 2, 3] and phys.tolist() == [1, 8, 7] and bad == 0


def test_request_of_token_hand_example_next_n():
    # next_n = 4 query rows per request (MTP): tokens 0-3 -> request 0, 4-7 -> 1, 8-11 -> 2.
    assert [O.request_of_token(t, 4, None) for t in range(12)] == [0] * 4 + [1] * 4 + [2] * 4
    # next_n = 1: every token is its own request
    assert [O.request_of_token(t, 1, None) for t in range(5)] == [0, 1, 2, 3, 4]
    # next_n = 3 with a ragged last request: tokens 6, 7 -> request 2
    assert [O.request_of_token(t, 3, None) for t in range(8)] == [0, 0, 0, 1, 1, 1, 2, 2]


def test_request_of_token_explicit_map_overrides_next_n():
    # a mixed batch: a 3-token chunk of request 2, one decode token of request 0 and two
    # speculative rows of request 1; the explicit map wins over t // next_n
    req = np.array([2, 2, 2, 0, 1, 1], dtype=np.int32)
    assert [O.request_of_token(t, 1, req) for t in range(6)] == [2, 2, 2, 0, 1, 1]
    assert [O.request_of_token(t, 4, req) for t in range(6)] == [2, 2, 2, 0, 1, 1]


def test_decode_routes_tokens_to_their_request_page_table():
    # Two requests over one pool of 4 pages of 4 slots; request 0 maps its pages to
    # physical [3, 1], request 1 to [0, 2]. With next_n = 2, tokens 0, 1 read request 0's
    # slots and tokens 2, 3 request 1's: check each token against attend() on the rows
    # picked out by hand (physical slot = page * 4 + offset).
    g = torch.Generator().manual_seed(5)
    P, H = 4, 2
    lat = torch.randn(16, 512, generator=g).to(torch.bfloat16)
    rope = torch.randn(16, 64, generator=g).to(torch.bfloat16)
    rows = O.pack_bf16(_bits(lat), _bits(rope))
    q = torch.randn(4, H, 576, generator=g).to(torch.bfloat16)
    pt = np.array([[3, 1], [0, 2]], dtype=np.int32)
    topk = np.array([[0, 5, -1], [7, 2, 1], [0, 5, -1], [7, 2, 1]], dtype=np.int32)
    by_hand = {0: [12, 5], 1: [7, 14, 13], 2: [0, 9], 3: [11, 2, 1]}
    res = O.decode(_bits(q), lambda ph: rows[ph], "bf16", pt, topk, P, 4, 0.05, next_n=2)
    for t, slots in by_hand.items():
        keys = O.dequant_rows(rows[slots], "bf16")
        o, l, _ = O.attend(O.bf16_bits_to_f64(_bits(q)[t]), keys, 0.05, None)
        assert np.array_equal(res["out"][t], o) and np.array_equal(res["lse"][t], l)
    # an explicit map that swaps the requests: token 2 now reads request 0's slots
    res2 = O.decode(_bits(q), lambda ph: rows[ph], "bf16", pt, topk, P, 4, 0.05, next_n=2,
                    req_id_per_token=np.array([1, 1, 0, 0], dtype=np.int32))
    o, _, _ = O.attend(O.bf16_bits_to_f64(_bits(q)[2]), O.dequant_rows(rows[[12, 5]], "bf16"), 0.05, None)
    assert np.array_equal(res2["out"][2], o)


def test_physical_slots_invalid_entries_dropped_and_counted():
    keep, phys, bad = O.physical_slots(np.array([-5, 12, 4, 0, -1]), np.array([2, -1, 1]), 4, 3)
    # -5: negative non-padding; 12: beyond stride*P; 4: page entry -1; 0: page 2 -> slot 8
    assert keep == [3] and phys.tolist() == [8] and bad == 3
    # a page entry equal to num_pages is one past the pool: 13 -> page entry 3 of a 3-page pool
    keep, phys, bad = O.physical_slots(np.array([13, 9]), np.array([2, -1, 1, 3]), 4, 3)
    assert keep == [1] and phys.tolist() == [5] and bad == 1


# ----------------------------------------------------------------------------- attention

TENSOR_SCALE = 2.0 ** -5  # per-tensor scale of the fp8_tensor pins (N(0,1) values stay in range)


def _torch_tensor_keys(rows: np.ndarray, kv_scale: float) -> torch.Tensor:
    """Keys of per-tensor FP8 rows through torch's own float8 decode and an fp32 multiply."""
    codes = torch.from_numpy(np.ascontiguousarray(rows[:, :576])).view(torch.float8_e4m3fn)
    return (codes.to(torch.float32) * torch.tensor(kv_scale, dtype=torch.float32)).to(torch.float64)


def _problem(n_pages=3, P=64, H=4, fmt="fp8_ds", seed=0, sink=False):
    g = torch.Generator().manual_seed(seed)
    n = n_pages * P
    lat = torch.randn(n, 512, generator=g).to(torch.bfloat16)
    rope = torch.randn(n, 64, generator=g).to(torch.bfloat16)
    if fmt == "fp8_ds":
        rows = O.pack_fp8_ds(_bits(lat), _bits(rope))
    elif fmt == "fp8_tensor":
        rows = O.pack_fp8_tensor(_bits(lat), _bits(rope), TENSOR_SCALE)
    else:
        rows = O.pack_bf16(_bits(lat), _bits(rope))
    q = torch.randn(1, H, 576, generator=g).to(torch.bfloat16)
    pt = torch.randperm(n_pages, generator=g).numpy()[None, :].astype(np.int32)
    sig = torch.randn(H, generator=g, dtype=torch.float64).numpy() if sink else None
    return rows, q, pt, sig


@pytest.mark.parametrize("fmt", ["fp8_ds", "bf16", "fp8_tensor"])
@pytest.mark.parametrize("sink", [False, True])
def test_full_context_topk_equals_dense_sdpa(fmt, sink):
    P, n_pages, H = 64, 3, 4
    rows, q, pt, sig = _problem(n_pages, P, H, fmt, seed=11, sink=sink)
    ctx = n_pages * P
    perm = np.random.default_rng(2).permutation(ctx).astype(np.int32)
    sm = 1.0 / 24
    kvs = TENSOR_SCALE if fmt == "fp8_tensor" else None
    res = O.decode(_bits(q), lambda s: rows[s], fmt, pt, perm[None, :], P, n_pages, sm, sink=sig,
                   kv_scale=kvs)
    # dense reference: all keys of the request in logical order, by page table lookup
    logical_rows = np.concatenate([rows[p * P:(p + 1) * P] for p in pt[0]])
    if fmt == "fp8_tensor":  # keys decoded by torch, not by the oracle
        keys = _torch_tensor_keys(logical_rows, TENSOR_SCALE)
    else:
        keys = torch.from_numpy(O.dequant_rows(logical_rows, fmt))
    qf = torch.from_numpy(O.bf16_bits_to_f64(_bits(q[0])))  # [H, 576]
    if sig is None:
        out = torch.nn.functional.scaled_dot_product_attention(
            qf[None, :, None, :], keys.expand(1, H, ctx, 576), keys[:, :512].expand(1, H, ctx, 512), scale=sm)
    else:  # sink as an extra key that scores sigma_h and carries a zero value
        qa = torch.cat([qf, torch.ones(H, 1, dtype=torch.float64)], 1)
        ka = torch.cat([keys, torch.zeros(ctx, 1, dtype=torch.float64)], 1).expand(H, ctx, 577)
        ks = torch.zeros(H, 1, 577, dtype=torch.float64)
        ks[:, 0, 576] = torch.from_numpy(sig) / sm
        kk = torch.cat([ka, ks], 1)
        vv = torch.cat([keys[:, :512].expand(H, ctx, 512), torch.zeros(H, 1, 512, dtype=torch.float64)], 1)
        out = torch.nn.functional.scaled_dot_product_attention(qa[None, :, None, :], kk[None], vv[None], scale=sm)
    np.testing.assert_allclose(res["out"][0], out[0, :, 0].numpy(), rtol=1e-12, atol=1e-13)
    scores = sm * (qf @ keys.T)
    if sig is not None:
        scores = torch.cat([scores, torch.from_numpy(sig)[:, None]], 1)
    np.testing.assert_allclose(res["lse"][0], torch.logsumexp(scores, 1).numpy(), rtol=0, atol=1e-12)


def test_single_index_closed_form():
    rows, q, pt, _ = _problem(1, 64, 3, "fp8_ds", seed=4)
    idx = np.full((1, 16), -1, dtype=np.int32)
    idx[0, 7] = 9
    res = O.decode(_bits(q), lambda s: rows[s], "fp8_ds", pt, idx, 64, 1, 0.125)
    k = O.dequant_rows(rows[[pt[0, 0] * 64 + 9]], "fp8_ds")[0]
    assert np.array_equal(res["out"][0], np.broadcast_to(k[:512], (3, 512)))
    qf = O.bf16_bits_to_f64(_bits(q[0]))
    s = [0.125 * math.fsum(qf[h] * k) for h in range(3)]
    np.testing.assert_allclose(res["lse"][0], s, rtol=0, atol=1e-12)


def test_sink_single_index_closed_form_and_limits():
    rows, q, pt, _ = _problem(1, 64, 2, "bf16", seed=5)
    idx = np.array([[3, -1, -1, -1]], dtype=np.int32)
    sig = np.array([0.3, -2.0])
    fetch = lambda s: rows[s]  # noqa: E731
    res = O.decode(_bits(q), fetch, "bf16", pt, idx, 64, 1, 0.05, sink=sig)
    k = O.dequant_rows(rows[[pt[0, 0] * 64 + 3]], "bf16")[0]
    qf = O.bf16_bits_to_f64(_bits(q[0]))
    s = 0.05 * (qf @ k)
    w = 1.0 / (1.0 + np.exp(sig - s))  # e^s / (e^s + e^sigma)
    np.testing.assert_allclose(res["out"][0], w[:, None] * k[None, :512], rtol=1e-14, atol=0)
    np.testing.assert_allclose(res["lse"][0], np.logaddexp(s, sig), rtol=0, atol=1e-14)
    np.testing.assert_allclose(res["lse_nosink"][0], s, rtol=0, atol=1e-14)
    # sigma -> -inf is no sink; sigma -> +inf drives the output to zero
    lo = O.decode(_bits(q), fetch, "bf16", pt, idx, 64, 1, 0.05, sink=np.array([-1e30, -1e30]))
    no = O.decode(_bits(q), fetch, "bf16", pt, idx, 64, 1, 0.05, sink=None)
    assert np.array_equal(lo["out"], no["out"]) and np.array_equal(lo["lse"], no["lse"])
    hi = O.decode(_bits(q), fetch, "bf16", pt, idx, 64, 1, 0.05, sink=np.array([800.0, 800.0]))
    assert np.abs(hi["out"]).max() < 1e-300


def test_identical_values_closed_form():
    # every selected slot holds the same row: all scores equal, out = v * n e^s / (n e^s + e^sigma)
    rows, q, pt, _ = _problem(1, 64, 2, "fp8_ds", seed=6)
    rows = np.repeat(rows[:1], 64, axis=0)
    idx = np.arange(10, dtype=np.int32)[None, :]
    sig = np.array([1.5, -0.5])
    res = O.decode(_bits(q), lambda s: rows[s], "fp8_ds", pt, idx, 64, 1, 0.1, sink=sig)
    k = O.dequant_rows(rows[:1], "fp8_ds")[0]
    s = 0.1 * (O.bf16_bits_to_f64(_bits(q[0])) @ k)
    frac = 10 * np.exp(s) / (10 * np.exp(s) + np.exp(sig))
    np.testing.assert_allclose(res["out"][0], frac[:, None] * k[None, :512], rtol=1e-13, atol=1e-15)


def test_empty_selection():
    rows, q, pt, _ = _problem(1, 64, 2, "fp8_ds", seed=7)
    idx = np.full((1, 8), -1, dtype=np.int32)
    res = O.decode(_bits(q), lambda s: rows[s], "fp8_ds", pt, idx, 64, 1, 0.1)
    assert (res["out"] == 0).all() and np.isneginf(res["lse"]).all()
    sig = np.array([0.25, -3.0])
    res = O.decode(_bits(q), lambda s: rows[s], "fp8_ds", pt, idx, 64, 1, 0.1, sink=sig)
    assert (res["out"] == 0).all() and np.array_equal(res["lse"][0], sig)


def test_padding_placement_and_removal_invariance():
    rows, q, pt, sig = _problem(2, 64, 4, "fp8_ds", seed=8, sink=True)
    rng = np.random.default_rng(3)
    valid = rng.permutation(128)[:40].astype(np.int32)
    tail = np.concatenate([valid, np.full(24, -1, np.int32)])
    inter = np.full(64, -1, np.int32)
    inter[np.sort(rng.permutation(64)[:40])] = valid
    f = lambda s: rows[s]  # noqa: E731
    a = O.decode(_bits(q), f, "fp8_ds", pt, tail[None], 64, 2, 0.1, sink=sig)
    b = O.decode(_bits(q), f, "fp8_ds", pt, inter[None], 64, 2, 0.1, sink=sig)
    c = O.decode(_bits(q), f, "fp8_ds", pt, valid[None], 64, 2, 0.1, sink=sig)
    for r in (b, c):
        assert np.array_equal(a["out"], r["out"]) and np.array_equal(a["lse"], r["lse"])
    # the order of valid indices changes only rounding
    d = O.decode(_bits(q), f, "fp8_ds", pt, valid[::-1][None].copy(), 64, 2, 0.1, sink=sig)
    np.testing.assert_allclose(a["out"], d["out"], rtol=1e-12, atol=1e-14)


def test_page_relabel_invariance_bitwise():
    rows, q, pt, _ = _problem(4, 64, 4, "fp8_ds", seed=9)
    idx = np.random.default_rng(4).permutation(256)[:100].astype(np.int32)[None]
    a = O.decode(_bits(q), lambda s: rows[s], "fp8_ds", pt, idx, 64, 4, 0.1)
    relabel = np.array([3, 0, 2, 1])  # physical page p moves to relabel[p]
    rows2 = np.empty_like(rows)
    for p in range(4):
        rows2[relabel[p] * 64:(relabel[p] + 1) * 64] = rows[p * 64:(p + 1) * 64]
    pt2 = relabel[pt]
    b = O.decode(_bits(q), lambda s: rows2[s], "fp8_ds", pt2, idx, 64, 4, 0.1)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])


def test_brute_force_scalar_loops():
    rows, q, pt, sig = _problem(1, 64, 2, "fp8_ds", seed=10, sink=True)
    idx = np.array([[5, 60, -1, 17, 33]], dtype=np.int32)
    res = O.decode(_bits(q), lambda s: rows[s], "fp8_ds", pt, idx, 64, 1, 0.07, sink=sig)
    qf = O.bf16_bits_to_f64(_bits(q[0]))
    P0 = int(pt[0, 0])
    for h in range(2):
        ks, ss = [], []
        for i in (5, 60, 17, 33):
            r = rows[P0 * 64 + i]
            scl = [float(np.frombuffer(r[512 + 4 * b:516 + 4 * b].tobytes(), "<f4")[0]) for b in range(4)]
            kv = [float(np.float32(float(O.e4m3_decode(np.array([r[d]], np.uint8))[0]) * scl[d // 128]))
                  for d in range(512)]
            kv += [float(np.frombuffer((r[528 + 2 * e:530 + 2 * e].tobytes() + b"").rjust(4, b"\0"), "<f4")[0])
                   for e in range(64)]
            ks.append(kv)
            ss.append(0.07 * math.fsum(qf[h, d] * kv[d] for d in range(576)))
        den = math.fsum([math.exp(s) for s in ss] + [math.exp(sig[h])])
        for c in (0, 100, 511):
            o = math.fsum(math.exp(s) * k[c] for s, k in zip(ss, ks)) / den
            assert abs(o - res["out"][0, h, c]) < 1e-13
        assert abs(math.log(den) - res["lse"][0, h]) < 1e-13


def test_gather_dequant_rows_and_padding():
    rows, q, pt, _ = _problem(2, 64, 1, "fp8_ds", seed=12)
    idx = np.array([[70, -1, 3]], dtype=np.int32)
    g = O.gather_dequant(lambda s: rows[s], "fp8_ds", pt, idx, 64, 2)
    assert g.shape == (1, 3, 576)
    assert (g[0, 1] == 0).all()
    np.testing.assert_array_equal(g[0, 0], O.dequant_rows(rows[[pt[0, 1] * 64 + 6]], "fp8_ds")[0])
    np.testing.assert_array_equal(g[0, 2], O.dequant_rows(rows[[pt[0, 0] * 64 + 3]], "fp8_ds")[0])


# ----------------------------------------------------------------------------- fused store

def test_bf16_rne_matches_torch_rounding():
    x = np.random.default_rng(5).normal(size=4000) * 7.3
    got = O.bf16_rne(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()  # torch rounds f64 -> bf16
    assert np.array_equal(got, ref)
    # ties to even: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7
    assert O.bf16_rne(np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8])).tolist() == [1.0, 1 + 2 * 2.0 ** -7]


def test_rms_norm_closed_forms():
    # a constant row c: mean(x^2) = c^2, so y = w * c / sqrt(c^2 + eps); with eps = 0, y = w * sign(c)
    c = np.full((1, 512), -3.0)
    w = np.linspace(0.5, 2.0, 512)
    y = O.rms_norm_bf16(_bits(torch.tensor(c).to(torch.bfloat16)), _bits(torch.tensor(w).to(torch.bfloat16)), 0.0)
    wq = torch.tensor(w).to(torch.bfloat16).double().numpy()
    assert np.array_equal(y[0], O.bf16_rne(-wq))
    # scaling x by any positive factor leaves the eps = 0 norm unchanged
    g = torch.Generator().manual_seed(2)
    x = torch.randn(3, 512, generator=g).to(torch.bfloat16)
    wb = torch.ones(512).to(torch.bfloat16)
    a = O.rms_norm_bf16(_bits(x), _bits(wb), 0.0)
    b = O.rms_norm_bf16(_bits((x.double() * 4).to(torch.bfloat16)), _bits(wb), 0.0)
    assert np.array_equal(a, b)
    # eps counts: a row of ones with eps = 3 gives y = w / sqrt(1 + 3) = w / 2, exactly
    ones = np.ones((1, 512))
    y = O.rms_norm_bf16(_bits(torch.tensor(ones).to(torch.bfloat16)), _bits(torch.tensor(w).to(torch.bfloat16)), 3.0)
    assert np.array_equal(y[0], wq / 2)


def test_rms_norm_matches_torch_float64():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(16, 512, generator=g).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(512, generator=g)).to(torch.bfloat16)
    for eps in (1e-6, 0.5):  # the second is of the order of mean(x^2), so it moves every output
        ref = torch.nn.functional.rms_norm(x.double(), (512,), w.double(), eps=float(np.float32(eps)))
        got = O.rms_norm_bf16(_bits(x), _bits(w), eps)
        assert np.array_equal(got, O.bf16_rne(ref.numpy()))


def test_rope_rotation_special_angles_and_complex_product():
    g = torch.Generator().manual_seed(8)
    r = torch.randn(4, 64, generator=g).to(torch.bfloat16)
    rv = r.double().numpy()
    one, zero = np.ones((4, 32)), np.zeros((4, 32))
    assert np.array_equal(O.rope_bf16(_bits(r), one, zero), rv)            # angle 0: identity
    quarter = O.rope_bf16(_bits(r), zero, one)                               # angle pi/2: (-b, a)
    assert np.array_equal(quarter[:, 0::2], -rv[:, 1::2]) and np.array_equal(quarter[:, 1::2], rv[:, 0::2])
    # general angles: the complex product (a + ib) e^{i theta}, by torch
    th = torch.rand(4, 32, generator=g, dtype=torch.float64) * 6.28
    cos, sin = torch.cos(th).float().double(), torch.sin(th).float().double()
    z = torch.view_as_complex(r.double().reshape(4, 32, 2).contiguous()) * torch.complex(cos, sin)
    ref = torch.view_as_real(z).reshape(4, 64).numpy()
    assert np.array_equal(O.rope_bf16(_bits(r), cos.numpy(), sin.numpy()), O.bf16_rne(ref))


def test_store_normed_rows_is_norm_rope_then_the_packer():
    g = torch.Generator().manual_seed(9)
    lat = torch.randn(5, 512, generator=g).to(torch.bfloat16)
    rope = torch.randn(5, 64, generator=g).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(512, generator=g)).to(torch.bfloat16)
    eps = 0.25
    # the norm by torch in float64, rounded to bf16 by torch
    normed = torch.nn.functional.rms_norm(lat.double(), (512,), w.double(), eps=eps).to(torch.bfloat16)
    # a quarter turn maps each pair (a, b) to (-b, a), exactly
    turned = torch.stack([-rope[:, 1::2], rope[:, 0::2]], dim=2).reshape(5, 64)
    cos, sin = np.zeros((5, 32)), np.ones((5, 32))
    rows = O.store_normed_rows(_bits(lat), _bits(rope), _bits(w), eps, cos, sin, "fp8_ds")
    assert np.array_equal(rows, O.pack_fp8_ds(_bits(normed), _bits(turned)))
    rows = O.store_normed_rows(_bits(lat), _bits(rope), _bits(w), eps, cos, sin, "bf16")
    assert np.array_equal(rows, O.pack_bf16(_bits(normed), _bits(turned)))


# ----------------------------------------------------------------------------- FP8 q

def test_q_values_e4m3_matches_torch_decode_times_scale():
    codes = np.arange(256, dtype=np.uint8)
    finite = ~np.isin(codes, [0x7F, 0xFF])
    for qs in (1.0, 2.0 ** -3, 0.37):
        got = O.q_values(codes[finite], "e4m3", qs)
        ref = torch.from_numpy(codes[finite]).view(torch.float8_e4m3fn).to(torch.float64) * float(np.float32(qs))
        assert np.array_equal(got, ref.numpy())
    with pytest.raises(ValueError):
        O.q_values(codes, "e4m3", None)


@pytest.mark.parametrize("sink", [False, True])
def test_decode_fp8_q_equals_dense_sdpa(sink):
    # E4M3 q (torch's cast) against the per-tensor FP8 cache: the full context as top-k equals
    # dense float64 SDPA on q and keys decoded by torch
    P, n_pages, H = 64, 3, 4
    rows, q, pt, sig = _problem(n_pages, P, H, "fp8_tensor", seed=13, sink=sink)
    qs = 2.0 ** -2
    q8 = (q.float() / qs).to(torch.float8_e4m3fn)
    ctx = n_pages * P
    perm = np.random.default_rng(3).permutation(ctx).astype(np.int32)
    sm = 1.0 / 24
    res = O.decode(q8.view(torch.uint8).numpy(), lambda s: rows[s], "fp8_tensor", pt, perm[None, :], P, n_pages,
                   sm, sink=sig, kv_scale=TENSOR_SCALE, q_format="e4m3", q_scale=qs)
    logical_rows = np.concatenate([rows[p * P:(p + 1) * P] for p in pt[0]])
    keys = _torch_tensor_keys(logical_rows, TENSOR_SCALE)
    qf = q8[0].to(torch.float64) * qs
    scores = sm * (qf @ keys.T)
    if sig is not None:
        scores = torch.cat([scores, torch.from_numpy(sig)[:, None]], 1)
    w = torch.softmax(scores, 1)[:, :ctx]
    np.testing.assert_allclose(res["out"][0], (w @ keys[:, :512]).numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(res["lse"][0], torch.logsumexp(scores, 1).numpy(), rtol=0, atol=1e-12)


def test_decode_fp8_q_scale_folds_into_the_scores():
    # bmm1_scale = sm_scale * q_scale * kv_scale: scaling q by q_scale is scaling sm_scale by it
    P, n_pages, H = 64, 2, 3
    rows, q, pt, _ = _problem(n_pages, P, H, "fp8_tensor", seed=17)
    q8 = q.float().to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    idx = np.random.default_rng(4).permutation(n_pages * P)[:100].astype(np.int32)[None, :]
    qs = float(np.float32(0.37))
    a = O.decode(q8, lambda s: rows[s], "fp8_tensor", pt, idx, P, n_pages, 0.05, kv_scale=TENSOR_SCALE,
                 q_format="e4m3", q_scale=qs)
    b = O.decode(q8, lambda s: rows[s], "fp8_tensor", pt, idx, P, n_pages, 0.05 * qs, kv_scale=TENSOR_SCALE,
                 q_format="e4m3", q_scale=1.0)
    np.testing.assert_allclose(a["out"], b["out"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(a["lse"], b["lse"], rtol=0, atol=1e-12)
