"""smla_decode_noalloc: the workspace-free entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc -- a plugin inside another serving engine that has
reserved the GPU's memory, or a binding that only receives the engine's buffers. This
entry point keeps its split partials in a scratch array inside the library. Its output
must match smla_decode's (which takes a caller-allocated workspace) within the parity
tolerances, call after call, and it must refuse work that does not fit its scratch.
Collected last on purpose; it depends on no other test.
"""
import numpy as np
import pytest
import torch

import sparse_mla_decode_smla_gb300 as smla
import workloads as W
from sparse_mla_decode_smla_gb300.runner import DeviceDecode

pytestmark = pytest.mark.gpu

OUT_ATOL, COS_MIN, LSE_ATOL = 1e-2, 0.9999, 1e-3


def _close(out, lse, out_ref, lse_ref):
    o, r = out.double().cpu().numpy(), out_ref.double().cpu().numpy()
    assert np.isfinite(o).all()
    assert np.abs(o - r).max() <= OUT_ATOL
    den = np.linalg.norm(o, axis=-1) * np.linalg.norm(r, axis=-1)
    big = np.linalg.norm(r, axis=-1) > 1e-3
    assert ((o * r).sum(-1)[big] / den[big]).min() >= COS_MIN
    l, lr = lse.double().cpu().numpy(), lse_ref.double().cpu().numpy()
    assert np.array_equal(np.isneginf(l), np.isneginf(lr))
    fin = np.isfinite(lr)
    assert np.abs(l[fin] - lr[fin]).max() <= LSE_ATOL


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    # (workload, splits, whether the partials go through the scratch): up to 8 splits of the
    # tensor-core kernel merge inside the kernel and need none; 11 splits of it, and the
    # mma.sync kernel's splits, keep real partials in the scratch
    cases = [
        (W.small_variant(W.WORKLOADS[1], num_requests=3, ctx_lo=100, ctx_hi=900, topk=320), 3, False),
        (W.small_variant(W.WORKLOADS[4], num_requests=3, ctx_lo=400, ctx_hi=900, topk=320), 3, True),
        (W.small_variant(W.WORKLOADS[2], num_requests=2, ctx_lo=900, ctx_hi=900, topk=704), 12, True),
    ]
    for w, splits, partials in cases:
        p = W.make_problem(w)
        dd = DeviceDecode(p, num_splits=splits)
        assert (smla.workspace_size(dd.desc) > 256) == partials
        out_ref, lse_ref = [x.clone() for x in dd.run()]
        for _ in range(2):
            out = torch.full_like(dd.out, float("nan"))
            lse = torch.full_like(dd.lse, float("nan"))
            smla.decode_noalloc(dd.desc, dd.q, dd.kv, dd.page_table, dd.topk, None, dd.sink, out, lse)
            torch.cuda.synchronize()
            _close(out, lse, out_ref, lse_ref)


def test_noalloc_rejects_work_beyond_its_scratch():
    w = W.small_variant(W.WORKLOADS[2], num_requests=64, ctx_lo=300, ctx_hi=300, topk=2048)
    # 16 splits: more than a cluster merges, so they need partials beyond the 16 MiB scratch
    d = smla.make_desc(w.num_tokens, w.num_heads, w.topk, w.num_requests, w.page_size, 320,
                       w.page_table_stride, smla.SMLA_KV_FP8_DS, w.sm_scale, num_splits=16)
    assert smla.workspace_size(d) > smla.NOALLOC_SCRATCH_BYTES
    dummy = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(smla.SmlaError) as e:
        smla.decode_noalloc(d, dummy, dummy, dummy, dummy, None, None, dummy, None)
    assert e.value.status == 5  # SMLA_ERR_WORKSPACE, nothing launched


def test_noalloc_reports_device_errors_until_read():
    # The scratch holds the device error word too: it collects the bits of every call until
    # smla_noalloc_read_error reads and clears it, so an invalid entry is never lost.
    w = W.small_variant(W.WORKLOADS[2], num_requests=2, ctx_lo=500, ctx_hi=500, topk=256)
    p = W.make_problem(w)
    dd = DeviceDecode(p)
    out, lse = torch.empty_like(dd.out), torch.empty_like(dd.lse)
    smla.noalloc_read_error()  # whatever an earlier caller left
    smla.decode_noalloc(dd.desc, dd.q, dd.kv, dd.page_table, dd.topk, None, dd.sink, out, lse)
    assert smla.noalloc_read_error() == 0
    bad = dd.topk.clone()
    bad[1, 7] = 10 ** 6  # beyond the request's page table: masked and flagged
    for _ in range(2):
        smla.decode_noalloc(dd.desc, dd.q, dd.kv, dd.page_table, bad, None, dd.sink, out, lse)
    smla.decode_noalloc(dd.desc, dd.q, dd.kv, dd.page_table, dd.topk, None, dd.sink, out, lse)
    assert smla.noalloc_read_error() == smla.SMLA_DEVERR_INDEX  # kept across the clean call
    assert smla.noalloc_read_error() == 0  # and cleared by the read
