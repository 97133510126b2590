"""Float64 CPU oracle for the sparse-attention indexer (FP8 paged MQA logits + top-k).

TEST INFRASTRUCTURE ONLY. Only the tests, the smoke check and the bench's CPU
baseline may import this module; the library never does. It shares no code with
the CUDA path and takes its inputs from the seeded `workloads` module.

What the pages give (the vLLM PR #52164 page, "功能与动机" and "实现拆解 1-5"; the
SGLang PR #24692 page, "实现拆解 5" and "关键文件"): the indexer runs before the
sparse decode and chooses each query token's top-k slots; its kernel is the FP8
paged MQA logits kernel (fp8_paged_mqa_logits), scheduled from the requests'
context lengths; with next_n query rows per request (MTP) the native path hands
the kernel all next_n rows of a request at once, so each key tile is read once
instead of next_n times (flattening); the result feeds the decode's
topk_indices. The pages do not print the logit formula, the cache bytes or the
tie rule. The readings taken here (each one listed in the design notes):

* logit[t, s] = sum_h w[t, h] * max(0, scale_s * <q[t, h], k_s>): "MQA" logits of
  H_I query heads against one shared key per slot, combined over heads by the
  per-(token, head) weights the caller passes, after a ReLU (the DeepSeek-V3.2
  indexer form the kernel's name and its weights argument point to);
* q holds E4M3 codes (FP8 q); a key is 128 E4M3 codes with one fp32 scale;
* a page of the key cache is P x 128 codes (slot-major) followed by P fp32 scales;
* query row i (0-based) of a request with next_n rows and context length ctx sees
  slots [0, ctx - next_n + 1 + i) (the causal prefix the decode workloads use);
* top-k = the indices of the K largest logits among the visible slots, as a set
  (any order); with fewer than K visible slots all of them, then -1 padding; at a
  tie on the K-th value any choice among the tied slots is correct.

Every function is a plain definition in float64: products of E4M3 values are exact
in float64 and so is a sum of 128 of them, so the only rounding is in the final
weighted sum over heads. tests/test_indexer_oracle_pins.py pins every function
(hand-built pages, closed forms, scalar loops, torch's float8 decode, argpartition),
and tests/test_oracle_planted_mistakes.py requires those pins to catch plausible
slips planted in a copy of this module.
"""
from __future__ import annotations

import numpy as np

from .smla_oracle import e4m3_decode

INDEX_DIM = 128


def visible_len(ctx: int, next_n: int, i: int) -> int:
    """Slots query row i of a request (next_n rows, context ctx) sees: ctx - next_n + 1 + i, at least 0."""
    return max(0, int(ctx) - int(next_n) + 1 + int(i))


def page_keys(cache_page: np.ndarray, page_size: int):
    """One cache page (bytes) -> (codes [P, 128] uint8, scales [P] float64)."""
    cache_page = np.ascontiguousarray(cache_page, dtype=np.uint8)
    codes = cache_page[:page_size * INDEX_DIM].reshape(page_size, INDEX_DIM)
    scales = cache_page[page_size * INDEX_DIM:page_size * (INDEX_DIM + 4)].copy().view("<f4")
    return codes, scales.astype(np.float64)


def request_keys(cache: np.ndarray, pt_row: np.ndarray, n: int, page_size: int):
    """Keys of request-local slots 0..n-1: (values [n, 128] float64, scales [n] float64).

    Slot s lives in physical page pt_row[s // P] at in-page position s % P.
    """
    vals = np.zeros((n, INDEX_DIM))
    sc = np.zeros(n)
    for s0 in range(0, n, page_size):
        codes, scales = page_keys(cache[int(pt_row[s0 // page_size])], page_size)
        m = min(page_size, n - s0)
        vals[s0:s0 + m] = e4m3_decode(codes[:m])
        sc[s0:s0 + m] = scales[:m]
    return vals, sc


def logits_of_token(q_codes: np.ndarray, weights: np.ndarray, keys: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """logit[s] = sum_h w[h] * max(0, scale_s * <q_h, k_s>) for one query token, float64.

    q_codes [H_I, 128] E4M3 codes, weights [H_I], keys [n, 128] values, scales [n].
    """
    q = e4m3_decode(q_codes)                 # [H_I, 128], exact
    dots = q @ keys.T                        # [H_I, n], exact in float64
    act = np.maximum(0.0, dots * scales[None, :])
    return np.asarray(weights, dtype=np.float64) @ act


def indexer_logits(q_codes, weights, cache, page_table, ctx, next_n: int, page_size: int, tokens=None):
    """Logits of the listed tokens (all by default): list of float64 arrays, one per token,
    each of the token's visible length (slots beyond it are outside the result)."""
    q_codes = np.asarray(q_codes)
    T = q_codes.shape[0]
    tokens = range(T) if tokens is None else tokens
    out = []
    for t in tokens:
        r, i = divmod(int(t), next_n)
        n = visible_len(ctx[r], next_n, i)
        keys, sc = request_keys(cache, page_table[r], n, page_size)
        out.append(logits_of_token(q_codes[t], weights[t], keys, sc))
    return out


def topk_set(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest entries (all of them when there are fewer), by a stable sort:
    at a tie the lower index goes first. One correct answer among several at ties."""
    n = logits.shape[0]
    if n <= k:
        return np.arange(n)
    order = np.argsort(-logits, kind="stable")
    return np.sort(order[:k])
