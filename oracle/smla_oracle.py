"""Float64 CPU oracle for DeepSeek-style sparse MLA decode.

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's CPU
baseline may import this module; the library never does. It shares no code
with the CUDA path and takes its inputs from the seeded `workloads` module.

Sources (the vLLM / SGLang review pages for DeepSeek-V4 sparse MLA):
* "vLLM PR #43477, 关键源码片段" (forward_mqa): request-local top-k indices are
  turned into physical cache slots through req_id_per_token, the block table
  and the block size; the output is [num_tokens, num_heads, kv_lora_rank=512]
  and has q's dtype; the cache is the fp8_ds_mla layout with one shared latent
  per slot (num_kv_heads == 1).
* "SGLang PR #24692, 实现拆解 2-3" (_gather_and_dequant, _sm120_sparse_decode_fwd,
  _merge_partial_attn, _apply_attn_sink): gather with in-page addressing,
  dequantise, softmax attention over the gathered rows, per-head sink logit.
* "vLLM PR #43827, 功能与动机 / 关键源码片段": the "UE8M0 paged" FlashMLA layout
  (power-of-two block scales) next to contiguous BF16 / FP8 caches; the
  softmax scale multiplies the QK product (bmm1 scale).

Readings where the pages are silent (all listed with reasons in the design
notes): the 656-byte row is [512 e4m3 | 4 fp32 scales | 64 bf16 RoPE];
scale b covers latent dims [128b, 128b+128); e4m3 is OCP E4M3FN; a
dequantised latent element is fl32(e4m3 * scale); LSE is the natural log of
the softmax denominator including the sink term; the sink adds exp(sigma_h)
to the denominator only; only -1 means padding.

Every function here is a plain definition evaluated in float64: there is no
online softmax, no tiling and no split-K. Each one is pinned by
tests/test_oracle_pins.py against something other than itself (closed forms,
torch's number formats, dense float64 attention, brute force), so none is
parity unpinned; tests/test_oracle_planted_mistakes.py plants plausible slips in
a copy of this module and requires a pin to fail for each.
"""
from __future__ import annotations

import math
from typing import Callable

import numpy as np

LATENT = 512
ROPE = 64
DIM = LATENT + ROPE
BLOCK = 128  # latent dims per fp32 scale
FP8_ROW_BYTES = LATENT + 4 * 4 + ROPE * 2  # 656
BF16_ROW_BYTES = DIM * 2  # 1152
FP8_TENSOR_ROW_BYTES = DIM  # 576
E4M3_MAX = 448.0

SCALE_POW2 = 0
SCALE_FP32 = 1

# --------------------------------------------------------------------------- #
# Number formats
# --------------------------------------------------------------------------- #


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values (bf16 is the top half of fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    # Widening a signalling-NaN pattern quietens it, which NumPy reports as an
    # invalid-value warning; the value stays NaN either way.
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """OCP E4M3FN code -> float64 value.

    1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent field 0 is
    subnormal (2^-6 * m/8); S.1111.111 is NaN; there is no infinity; the
    largest finite magnitude is 448 (code 0x7e).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    val = np.where(s == 1, -mag, mag)
    return np.where((e == 15) & (m == 7), np.nan, val)


_E4M3_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))  # codes 0..126, ascending, 0 .. 448


def e4m3_encode_rne_satfinite(x: np.ndarray) -> np.ndarray:
    """float64 (holding fp32 values) -> E4M3FN code, round-to-nearest-even, saturating.

    Finite magnitudes above 448, and infinities, become +-448; NaN becomes
    0x7f. The sign of zero is kept (a negative value that rounds to zero gives
    0x80).
    """
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    hi = np.searchsorted(_E4M3_POS, a, side="left")  # first table value >= a
    hi = np.clip(hi, 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    d_hi = _E4M3_POS[hi] - a
    d_lo = a - _E4M3_POS[lo]
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(a >= E4M3_MAX, 126, code)  # saturate (also +-inf)
    code = np.where(np.isnan(x), 0x7F, code | np.where(neg, 0x80, 0))
    return code.astype(np.uint8)


def f32(x) -> np.ndarray:
    """Round float64 values to the nearest fp32 (RNE), returned as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


# --------------------------------------------------------------------------- #
# Cache format
# --------------------------------------------------------------------------- #


def pow2_ceil_f32(v: np.ndarray) -> np.ndarray:
    """Smallest power of two >= v, for positive fp32 values v (exact)."""
    m, e = np.frexp(np.asarray(v, dtype=np.float64))  # v = m * 2^e, m in [0.5, 1)
    return np.where(m == 0.5, v, np.ldexp(1.0, e))


def block_scales(latent: np.ndarray, scale_mode: int = SCALE_POW2) -> np.ndarray:
    """Per-128 block scale of [N, 512] float64 latents (exact fp32 values) -> [N, 4].

    amax = max |x| over the block. POW2 (the "UE8M0" reading of the FlashMLA
    layout): the smallest power of two >= fl32(amax / 448). FP32: fl32(amax / 448).
    A block of zeros gets scale 1.
    """
    amax = np.abs(latent.reshape(latent.shape[0], 4, BLOCK)).max(axis=2)
    ratio = f32(amax / E4M3_MAX)
    sc = pow2_ceil_f32(np.where(ratio > 0, ratio, 1.0)) if scale_mode == SCALE_POW2 else ratio
    return np.where(amax == 0, 1.0, sc)


def pack_fp8_ds(latent_bits: np.ndarray, rope_bits: np.ndarray,
                scale_mode: int = SCALE_POW2) -> np.ndarray:
    """Quantise bf16 latent [N,512] + bf16 RoPE [N,64] (uint16 bit patterns) into 656-byte rows.

    Row = 512 E4M3 codes of fl32(x / scale_b) | 4 fp32 scales (little-endian) |
    64 bf16 RoPE values (little-endian), as read from the fp8_ds_mla cache.
    """
    lat = bf16_bits_to_f64(latent_bits).reshape(-1, LATENT)
    n = lat.shape[0]
    sc = block_scales(lat, scale_mode)  # [N, 4]
    q = f32(lat / np.repeat(sc, BLOCK, axis=1))
    codes = e4m3_encode_rne_satfinite(q)
    out = np.empty((n, FP8_ROW_BYTES), dtype=np.uint8)
    out[:, :LATENT] = codes
    out[:, LATENT:LATENT + 16] = sc.astype("<f4").view(np.uint8).reshape(n, 16)
    out[:, LATENT + 16:] = np.asarray(rope_bits, dtype="<u2").reshape(n, ROPE).view(np.uint8)
    return out


def pack_fp8_tensor(latent_bits: np.ndarray, rope_bits: np.ndarray, kv_scale: float) -> np.ndarray:
    """Quantise bf16 latent [N,512] + bf16 RoPE [N,64] into 576-byte per-tensor FP8 rows.

    The contiguous FP8 cache of FlashInfer's DeepSeek-V4 path (vLLM PR #43827,
    "实现拆解 4" and "关键源码片段": the compressor's store_full_fp8 writes a
    per-tensor FP8 cache with one fp8 scale; _resolve_dsv4_kv_cache_dtype gives it
    dtype float8_e4m3fn): all 576 values [latent 512 | RoPE 64] are E4M3 codes of
    fl32(x / kv_scale), round-to-nearest-even, saturating at +-448.
    """
    lat = bf16_bits_to_f64(latent_bits).reshape(-1, LATENT)
    rope = bf16_bits_to_f64(rope_bits).reshape(-1, ROPE)
    x = np.concatenate([lat, rope], axis=1)
    q = f32(x / float(f32(kv_scale)))
    return e4m3_encode_rne_satfinite(q).astype(np.uint8).reshape(-1, FP8_TENSOR_ROW_BYTES)


def pack_bf16(latent_bits: np.ndarray, rope_bits: np.ndarray) -> np.ndarray:
    """bf16 cache row: 576 bf16 values [latent 512 | rope 64] (little-endian) = 1152 bytes."""
    n = np.asarray(latent_bits).reshape(-1, LATENT).shape[0]
    row = np.concatenate([np.asarray(latent_bits, dtype="<u2").reshape(n, LATENT),
                          np.asarray(rope_bits, dtype="<u2").reshape(n, ROPE)], axis=1)
    return row.view(np.uint8).reshape(n, BF16_ROW_BYTES)


def dequant_rows(rows: np.ndarray, kv_format: str, kv_scale: float | None = None) -> np.ndarray:
    """Cache rows [n, R] uint8 -> [n, 576] float64 key vectors.

    fp8_ds: latent element d = fl32(e4m3(code_d) * scale[d // 128]) -- the
    float64 product of a 4-bit and a 24-bit significand is exact, so rounding
    it once to fp32 is the fp32 multiply; RoPE is bf16, exact.
    fp8_tensor: every element d = fl32(e4m3(code_d) * kv_scale), the per-tensor
    scale of the FlashInfer path (vLLM PR #43827: bmm1_scale = scale * q_scale *
    kv_scale, bmm2_scale = kv_scale, i.e. keys and values both carry kv_scale).
    bf16: the 576 bf16 values, exact.
    """
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    if kv_format == "bf16":
        return bf16_bits_to_f64(rows.view("<u2").reshape(n, DIM))
    if kv_format == "fp8_tensor":
        if kv_scale is None:
            raise ValueError("fp8_tensor rows need kv_scale")
        return f32(e4m3_decode(rows[:, :DIM]) * float(f32(kv_scale)))
    codes = rows[:, :LATENT]
    sc = rows[:, LATENT:LATENT + 16].copy().view("<f4").reshape(n, 4).astype(np.float64)
    lat = f32(e4m3_decode(codes) * np.repeat(sc, BLOCK, axis=1))
    rope = bf16_bits_to_f64(rows[:, LATENT + 16:].copy().view("<u2").reshape(n, ROPE))
    return np.concatenate([lat, rope], axis=1)


# --------------------------------------------------------------------------- #
# Addressing
# --------------------------------------------------------------------------- #


def request_of_token(t: int, next_n: int, req_id_per_token) -> int:
    """Token -> request: req_id_per_token[t] when given, else t // next_n (next_n query rows per request)."""
    if req_id_per_token is not None:
        return int(req_id_per_token[t])
    return t // next_n


def physical_slots(idx_row: np.ndarray, pt_row: np.ndarray, page_size: int, num_pages: int):
    """Request-local top-k indices -> (positions kept, physical slot ids).

    phys = page_table[r, idx // P] * P + idx % P (vLLM PR #43477, forward_mqa:
    triton_convert_req_index_to_global_index). -1 is padding. Any other index
    outside [0, stride*P), or one whose page entry is outside [0, num_pages),
    is invalid: it is dropped as well and counted in `n_invalid`.
    """
    stride = len(pt_row)
    keep, phys, n_invalid = [], [], 0
    for j, idx in enumerate(np.asarray(idx_row, dtype=np.int64).tolist()):
        if idx == -1:
            continue
        if idx < 0 or idx >= stride * page_size:
            n_invalid += 1
            continue
        page = int(pt_row[idx // page_size])
        if page < 0 or page >= num_pages:
            n_invalid += 1
            continue
        keep.append(j)
        phys.append(page * page_size + idx % page_size)
    return keep, np.asarray(phys, dtype=np.int64), n_invalid


# --------------------------------------------------------------------------- #
# Attention
# --------------------------------------------------------------------------- #


def attend(q: np.ndarray, keys: np.ndarray, sm_scale: float, sink: np.ndarray | None):
    """Softmax attention of H query rows over n shared key/value rows, float64.

    q [H, 576], keys [n, 576]; values are keys[:, :512] (MLA: V is the latent).
    s[h, j] = sm_scale * <q_h, k_j>;
    out_h = sum_j e^{s_hj} v_j / (sum_j e^{s_hj} + [sink] e^{sigma_h});
    lse_h = log(sum_j e^{s_hj} + [sink] e^{sigma_h}) (natural log).
    Returns (out [H,512], lse [H], lse_without_sink [H]). With no rows the
    output is 0, lse is -inf without a sink and sigma_h with one.
    """
    H = q.shape[0]
    n = keys.shape[0]
    sig = None if sink is None else np.asarray(sink, dtype=np.float64)
    if n == 0:
        lse0 = np.full(H, -np.inf)
        lse = lse0.copy() if sig is None else sig.copy()
        return np.zeros((H, LATENT)), lse, lse0
    s = float(sm_scale) * (q @ keys.T)  # [H, n]
    m = s.max(axis=1, keepdims=True)
    if sig is not None:
        m = np.maximum(m, sig[:, None])
    e = np.exp(s - m)
    denom = e.sum(axis=1)
    m0 = s.max(axis=1)
    lse0 = m0 + np.log(np.exp(s - m0[:, None]).sum(axis=1))
    if sig is not None:
        denom = denom + np.exp(sig - m[:, 0])
    out = (e @ keys[:, :LATENT]) / denom[:, None]
    lse = m[:, 0] + np.log(denom)
    return out, lse, lse0


def q_values(q, q_format: str = "bf16", q_scale: float | None = None) -> np.ndarray:
    """q of one token as float64 values: bf16 bit patterns, or E4M3 codes times the per-tensor
    q_scale (the FP8-Q path of vLLM PR #43827, "关键源码片段": bmm1_scale = scale * q_scale *
    kv_scale; the product of a 4-bit significand and an fp32 scale is exact in float64)."""
    if q_format == "bf16":
        return bf16_bits_to_f64(q)
    if q_format == "e4m3":
        if q_scale is None:
            raise ValueError("E4M3 q needs q_scale")
        return e4m3_decode(q) * float(np.float32(q_scale))
    raise ValueError(q_format)


def decode(q_bits: np.ndarray, fetch_rows: Callable[[np.ndarray], np.ndarray], kv_format: str,
           page_table: np.ndarray, topk: np.ndarray, page_size: int, num_pages: int,
           sm_scale: float, sink=None, next_n: int = 1, req_id_per_token=None, tokens=None,
           kv_scale: float | None = None, q_format: str = "bf16", q_scale: float | None = None):
    """Sparse MLA decode of the listed tokens (all by default), float64.

    q_bits [T, H, 576] bf16 bit patterns (q_format "bf16") or E4M3 codes (q_format "e4m3",
    values code * q_scale); fetch_rows(phys_slots) -> [n, R] uint8 cache rows; page_table
    [B, stride]; topk [T, K] request-local indices.
    Returns dict(out [t,H,512], lse [t,H], lse_nosink [t,H], n_invalid [t]).
    """
    q_bits = np.asarray(q_bits)
    T, H, _ = q_bits.shape
    tokens = list(range(T)) if tokens is None else list(tokens)
    outs, lses, lse0s, bad = [], [], [], []
    for t in tokens:
        r = request_of_token(t, next_n, req_id_per_token)
        _, phys, n_invalid = physical_slots(topk[t], page_table[r], page_size, num_pages)
        rows = fetch_rows(phys) if len(phys) else np.zeros((0, 1), dtype=np.uint8)
        keys = dequant_rows(rows, kv_format, kv_scale) if len(phys) else np.zeros((0, DIM))
        o, l, l0 = attend(q_values(q_bits[t], q_format, q_scale), keys, sm_scale, sink)
        outs.append(o)
        lses.append(l)
        lse0s.append(l0)
        bad.append(n_invalid)
    return dict(out=np.stack(outs), lse=np.stack(lses), lse_nosink=np.stack(lse0s),
                n_invalid=np.asarray(bad))


def gather_dequant(fetch_rows, kv_format: str, page_table, topk, page_size: int, num_pages: int,
                   next_n: int = 1, req_id_per_token=None, kv_scale: float | None = None) -> np.ndarray:
    """The gathered, dequantised key rows: [T, K, 576] as fp32 values (float64 array).

    Row (t, j) is dequant(row at the physical slot of topk[t, j]); padding and
    invalid entries give a zero row. Every value is an exact fp32 number
    (fl32 products for the FP8 latent, exact bf16 otherwise).
    """
    T, K = topk.shape
    out = np.zeros((T, K, DIM))
    for t in range(T):
        r = request_of_token(t, next_n, req_id_per_token)
        keep, phys, _ = physical_slots(topk[t], page_table[r], page_size, num_pages)
        if keep:
            out[t, keep] = dequant_rows(fetch_rows(phys), kv_format, kv_scale)
    return out


# --------------------------------------------------------------------------- #
# Quantise-on-write store fused with the latent's norm and the key's RoPE
# --------------------------------------------------------------------------- #
# The compressor's store of the vLLM PR #43827 page ("实现拆解 4-6":
# SparseAttnCompressNormRopeStoreFullC4Kernel with store_full_kv / store_full_fp8, and the
# fused "qnorm rope kv insert" test): normalise the latent, rotate the RoPE part, quantise and
# store the row. The page names the steps, not their formulas; the readings are: RMSNorm over
# the 512 latent dims with a per-dim weight, y = x / sqrt(mean(x^2) + eps) * w; the rotation
# turns adjacent pairs (2j, 2j+1) of the 64 RoPE dims by the angle whose cosine and sine the
# caller's table holds for the row's position; both results are rounded to bf16 (the values
# an unfused pipeline would store), then packed exactly as pack_fp8_ds / pack_fp8_tensor /
# pack_bf16 pack them.


def bf16_rne(x) -> np.ndarray:
    """float64 -> nearest bf16 value (round half to even, 8 significant bits), as float64.
    Finite inputs of normal bf16 magnitude (the only ones used here)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2^e, |m| in [0.5, 1)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def f64_to_bf16_bits(x) -> np.ndarray:
    """bf16 values (exactly representable) -> uint16 bit patterns."""
    return (np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def rms_norm_bf16(latent_bits: np.ndarray, weight_bits: np.ndarray, eps: float) -> np.ndarray:
    """[n, 512] bf16 latents (bit patterns) -> bf16 values of x / sqrt(mean(x^2) + eps) * w (float64)."""
    x = bf16_bits_to_f64(latent_bits).reshape(-1, LATENT)
    w = bf16_bits_to_f64(weight_bits).reshape(LATENT)
    r = 1.0 / np.sqrt((x * x).mean(axis=1, keepdims=True) + float(np.float32(eps)))
    return bf16_rne(x * r * w[None, :])


def rope_bf16(rope_bits: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """[n, 64] bf16 RoPE values -> bf16 values of the pairs (2j, 2j+1) rotated by the angle with
    cosine cos[:, j] and sine sin[:, j] ([n, 32] each, fp32 values): (a c - b s, a s + b c)."""
    r = bf16_bits_to_f64(rope_bits).reshape(-1, ROPE)
    a, b = r[:, 0::2], r[:, 1::2]
    c, s = np.asarray(cos, dtype=np.float64), np.asarray(sin, dtype=np.float64)
    out = np.empty_like(r)
    out[:, 0::2] = a * c - b * s
    out[:, 1::2] = a * s + b * c
    return bf16_rne(out)


def store_normed_rows(latent_bits, rope_bits, weight_bits, eps, cos, sin, kv_format: str,
                      scale_mode: int = SCALE_POW2, kv_scale: float | None = None) -> np.ndarray:
    """Cache rows of the fused store: norm + rotation (bf16), then the format's packer."""
    lat = f64_to_bf16_bits(rms_norm_bf16(latent_bits, weight_bits, eps))
    rope = f64_to_bf16_bits(rope_bf16(rope_bits, cos, sin))
    if kv_format == "bf16":
        return pack_bf16(lat, rope)
    if kv_format == "fp8_tensor":
        return pack_fp8_tensor(lat, rope, kv_scale)
    return pack_fp8_ds(lat, rope, scale_mode)
