"""Oracle-side set-up of a seeded decode batch (test infrastructure only).

Packs the cache rows the oracle needs with the oracle's own packer, from the
seeded source values in `workloads`, and runs the float64 decode. Nothing
here comes from the CUDA path.
"""
from __future__ import annotations

import numpy as np
import torch

from . import smla_oracle as O


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


class OracleCache:
    """Packed cache rows of the pages a set of requests uses, keyed by physical page."""

    def __init__(self, problem, requests=None, scale_mode: int = O.SCALE_POW2):
        w = problem.w
        P = w.page_size
        self.P = P
        pt = problem.page_table.cpu().numpy()
        reqs = range(w.num_requests) if requests is None else sorted(set(requests))
        pages = sorted({int(x) for r in reqs for x in pt[r] if 0 <= x < problem.num_pages})
        self.index = {p: i for i, p in enumerate(pages)}
        if w.kv_format == "bf16":
            kv = problem.kv_bf16.cpu().reshape(problem.num_pages, P, 576)
            sel = kv[pages].reshape(-1, 576)
            self.rows = O.pack_bf16(_bits(sel[:, :512]), _bits(sel[:, 512:]))
        elif w.kv_format == "fp8_tensor":
            lat, rope = problem.raw_pages(pages)
            self.rows = O.pack_fp8_tensor(_bits(lat), _bits(rope), w.kv_scale)
        else:
            lat, rope = problem.raw_pages(pages)
            self.rows = O.pack_fp8_ds(_bits(lat), _bits(rope), scale_mode)

    def fetch(self, phys: np.ndarray) -> np.ndarray:
        phys = np.asarray(phys, dtype=np.int64)
        loc = np.array([self.index[int(s) // self.P] for s in phys], dtype=np.int64)
        return self.rows[loc * self.P + phys % self.P]


def oracle_decode(problem, tokens=None, scale_mode: int = O.SCALE_POW2, cache: OracleCache | None = None,
                  q_e4m3: torch.Tensor | None = None, q_scale: float | None = None):
    """Float64 decode of the listed tokens (all by default) of a seeded problem; with q_e4m3
    ([T, H, 576] uint8 E4M3 codes) and q_scale, of that FP8 q instead of the problem's bf16 q."""
    w = problem.w
    T = w.num_tokens
    tokens = list(range(T)) if tokens is None else list(tokens)
    if cache is None:
        cache = OracleCache(problem, [t // w.next_n for t in tokens], scale_mode)
    sink = None if problem.sink is None else problem.sink.cpu().double().numpy()
    q = _bits(problem.q) if q_e4m3 is None else q_e4m3.cpu().numpy()
    return O.decode(q, cache.fetch, w.kv_format, problem.page_table.cpu().numpy(),
                    problem.topk.cpu().numpy(), w.page_size, problem.num_pages, w.sm_scale,
                    sink=sink, next_n=w.next_n, tokens=tokens,
                    kv_scale=w.kv_scale if w.kv_format == "fp8_tensor" else None,
                    q_format="bf16" if q_e4m3 is None else "e4m3", q_scale=q_scale)
