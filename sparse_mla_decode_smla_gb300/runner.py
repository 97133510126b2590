"""Device-side set-up of a decode batch: cache packing, buffers and the decode call.

Used by the tests and the bench. Every step of the decode itself runs in the
library; this module only allocates torch tensors and calls the binding.
"""
from __future__ import annotations

import torch

from . import (SMLA_KV_BF16, SMLA_KV_FP8_DS, SMLA_KV_FP8_TENSOR, SMLA_SCALE_POW2, decode,
               make_desc, pack_kv, pack_kv_fp8_tensor, workspace_size)

FMT = {"bf16": SMLA_KV_BF16, "fp8_ds": SMLA_KV_FP8_DS, "fp8_tensor": SMLA_KV_FP8_TENSOR}


def pack_problem_cache(problem, scale_mode: int = SMLA_SCALE_POW2, device="cuda") -> torch.Tensor:
    """The problem's whole cache as a device byte tensor [num_slots, R], written by smla_pack_kv."""
    w = problem.w
    R = w.row_bytes
    kv = torch.empty((problem.num_slots, R), dtype=torch.uint8, device=device)
    if w.kv_format == "bf16":
        src = problem.kv_bf16.reshape(-1, 576).to(device)
        lat, rope = src[:, :512].contiguous(), src[:, 512:].contiguous()
        slots = torch.arange(problem.num_slots, dtype=torch.int64, device=device)
        pack_kv(SMLA_KV_BF16, scale_mode, lat, rope, slots, kv, problem.num_slots)
        return kv
    from workloads import CHUNK_SLOTS
    for c in range(problem.num_chunks):
        lat, rope = problem.raw_chunk(c)
        lat, rope = lat.to(device), rope.to(device)
        lo = c * CHUNK_SLOTS
        slots = torch.arange(lo, lo + lat.shape[0], dtype=torch.int64, device=device)
        if w.kv_format == "fp8_tensor":
            pack_kv_fp8_tensor(lat, rope, slots, kv, problem.num_slots, w.kv_scale)
        else:
            pack_kv(SMLA_KV_FP8_DS, scale_mode, lat, rope, slots, kv, problem.num_slots)
        del lat, rope, slots
    return kv


class DeviceDecode:
    """All device buffers of one decode batch, and the call that decodes it."""

    def __init__(self, problem, kv: torch.Tensor | None = None, scale_mode: int = SMLA_SCALE_POW2,
                 num_splits: int = 0, device="cuda", with_lse: bool = True):
        w = problem.w
        self.problem = problem
        self.kv = kv if kv is not None else pack_problem_cache(problem, scale_mode, device)
        self.q = problem.q.to(device).contiguous()
        self.page_table = problem.page_table.to(device=device, dtype=torch.int32).contiguous()
        self.topk = problem.topk.to(device=device, dtype=torch.int32).contiguous()
        self.sink = None if problem.sink is None else problem.sink.to(device).contiguous()
        self.req_id = None
        T, H = w.num_tokens, w.num_heads
        self.desc = make_desc(T, H, w.topk, w.num_requests, w.page_size, problem.num_pages,
                              w.page_table_stride, FMT[w.kv_format], w.sm_scale, next_n=w.next_n,
                              num_splits=num_splits, kv_scale=w.kv_scale)
        ws = workspace_size(self.desc)
        self.workspace = torch.zeros((ws + 255) // 256 * 256 // 4, dtype=torch.int32, device=device)
        self.out = torch.empty((T, H, 512), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((T, H), dtype=torch.float32, device=device) if with_lse else None
        # the decode kernel the library dispatches to for this batch (the FP8 caches with 64
        # or more heads take the tensor-core head-group kernel)
        fp8 = w.kv_format in ("fp8_ds", "fp8_tensor")
        self.kernel_name = "decode_hg_kernel" if fp8 and H >= 64 else "decode_mma_kernel"

    def run(self, stream=None):
        decode(self.desc, self.q, self.kv, self.page_table, self.topk, self.req_id, self.sink,
               self.out, self.lse, self.workspace, stream)
        return self.out, self.lse
