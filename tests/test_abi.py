"""The C ABI library loads, exports every entry point include/smla.h declares, and rejects
bad arguments on the host before touching the GPU (CPU only: no compute call is made)."""
import ctypes
import os
import re

import pytest

import sparse_mla_decode_smla_gb300 as smla
from sparse_mla_decode_smla_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()  # incremental: recompiles only sources newer than their objects
    return smla.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "smla.h")).read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(smla_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ["smla_decode", "smla_pack_kv", "smla_workspace_size", "smla_gather_dequant",
              "smla_read_error", "smla_status_string", "smla_abi_version"]:
        assert n in names


def test_every_declared_symbol_is_exported(L):
    for n in _declared():
        assert hasattr(L, n), n
    assert set(_declared()) <= set(smla.EXPORTS) | set(_declared())


def test_abi_version_and_status_strings(L):
    assert L.smla_abi_version() == 5
    for s in range(11):
        assert smla.status_string(s) != "unknown status"
    assert smla.status_string(99) == "unknown status"


def _header_enum(prefix):
    text = open(os.path.join(ROOT, "include", "smla.h")).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(rf"\b({prefix}\w+)\s*=\s*(\d+)", text)}


def test_binding_statuses_and_error_bits_match_header():
    st = _header_enum("SMLA_ERR_") | {"SMLA_OK": 0}
    assert {v: k for k, v in st.items()} == smla.STATUS
    # a distinct status for a timeout, apart from the index/page one and the device one
    assert len({st["SMLA_ERR_TIMEOUT"], st["SMLA_ERR_INDEX_RANGE"], st["SMLA_ERR_DEVICE"],
                st["SMLA_ERR_OPERAND_RANGE"]}) == 4
    bits = _header_enum("SMLA_DEVERR_")
    assert bits == {"SMLA_DEVERR_INDEX": smla.SMLA_DEVERR_INDEX, "SMLA_DEVERR_PAGE": smla.SMLA_DEVERR_PAGE,
                    "SMLA_DEVERR_TIMEOUT": smla.SMLA_DEVERR_TIMEOUT, "SMLA_DEVERR_RANGE": smla.SMLA_DEVERR_RANGE}
    assert all(v & (v - 1) == 0 for v in bits.values()) and len(set(bits.values())) == len(bits)


def test_desc_layout_matches_header():
    # int32 x6, int64, int32 x2, float, int32, float, int32, float, int32; natural alignment
    assert ctypes.sizeof(smla.smla_desc) == 64
    assert smla.smla_desc.num_pages.offset == 24
    assert smla.smla_desc.kv_scale.offset == 48
    assert smla.smla_desc.q_format.offset == 52
    assert smla.smla_desc.q_scale.offset == 56
    assert smla.smla_desc.reserved.offset == 60


def _desc(**kw):
    d = smla.make_desc(4, 16, 64, 4, 64, 8, 4, smla.SMLA_KV_FP8_DS, 1 / 24)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def _decode_status(L, d, q=16, kv=16, pt=16, topk=16, out=16, ws=256):
    P = ctypes.c_void_p
    return L.smla_decode(ctypes.byref(d) if d is not None else None, P(q), P(kv), P(pt), P(topk),
                         None, None, P(out), None, P(ws), 1 << 20, None)


@pytest.mark.parametrize("field,value,status", [
    ("num_heads", 8, 2), ("num_heads", 144, 2), ("num_heads", 40, 2), ("topk", 0, 2),
    ("topk", 6, 2), ("page_size", 48, 2), ("page_size", 8192, 2), ("num_pages", 0, 2),
    ("kv_format", 3, 4), ("num_splits", 65, 2), ("num_tokens", 0, 2), ("next_n", 0, 2),
])
def test_decode_rejects_bad_desc_on_host(L, field, value, status):
    assert _decode_status(L, _desc(**{field: value})) == status


def test_decode_rejects_null_and_misaligned_pointers(L):
    assert _decode_status(L, None) == 1
    assert _decode_status(L, _desc(), q=0) == 1
    assert _decode_status(L, _desc(), ws=0) == 1
    assert _decode_status(L, _desc(), q=16 + 8) == 3
    assert _decode_status(L, _desc(), topk=16 + 4) == 3
    assert _decode_status(L, _desc(), ws=256 + 16) == 3
    d = _desc()
    d.reserved[0] = 1
    assert _decode_status(L, d) == 2
    # more tokens than requests * next_n without req_id_per_token
    assert _decode_status(L, _desc(num_tokens=9, num_requests=2, next_n=4)) == 2


def test_decode_fp8_q_host_checks(L):
    # E4M3 q is served with the per-tensor FP8 cache and 64 or more heads only; q_scale must be
    # finite and positive; an unknown q_format is unsupported (all rejected before any launch)
    ten = dict(kv_format=smla.SMLA_KV_FP8_TENSOR, num_heads=64, q_format=smla.SMLA_Q_FP8_E4M3, q_scale=0.5)
    assert _decode_status(L, _desc(**{**ten, "kv_format": smla.SMLA_KV_FP8_DS})) == 4
    assert _decode_status(L, _desc(**{**ten, "kv_format": smla.SMLA_KV_BF16})) == 4
    assert _decode_status(L, _desc(**{**ten, "num_heads": 48})) == 4
    assert _decode_status(L, _desc(**{**ten, "q_scale": 0.0})) == 2
    assert _decode_status(L, _desc(**{**ten, "q_scale": float("inf")})) == 2
    assert _decode_status(L, _desc(q_format=2)) == 4


def test_decode_rejects_caches_beyond_32_bit_row_coordinates(L):
    # rows are gathered by 32-bit row coordinates, one past the last slot marking a masked
    # row: num_pages * page_size must stay below 2^31 - 1
    # (rejected before any device call; a cache below the limit would go on to launch, so it
    # is not tried here with these dummy pointers)
    assert _decode_status(L, _desc(num_pages=1 << 25, page_size=64)) == 2  # 2^31 slots
    assert _decode_status(L, _desc(num_pages=1 << 31, page_size=1)) == 2   # 2^31 slots


def test_pack_rejects_bad_arguments_on_host(L):
    P = ctypes.c_void_p
    assert L.smla_pack_kv(7, 0, P(16), P(16), P(16), 4, P(16), 4, None) == 4
    assert L.smla_pack_kv(1, 5, P(16), P(16), P(16), 4, P(16), 4, None) == 4
    assert L.smla_pack_kv(1, 0, P(16), P(16), P(16), -1, P(16), 4, None) == 2
    assert L.smla_pack_kv(1, 0, None, P(16), P(16), 4, P(16), 4, None) == 1
    assert L.smla_pack_kv(1, 0, P(24), P(16), P(16), 4, P(16), 4, None) == 3
    assert L.smla_pack_kv(1, 0, P(16), P(16), P(16), 0, P(16), 4, None) == 0  # nothing to do


def test_workspace_size_checks_desc_first(L):
    n = ctypes.c_size_t(123)
    assert L.smla_workspace_size(ctypes.byref(_desc(num_heads=7)), ctypes.byref(n)) == 2
    assert n.value == 0
    assert L.smla_workspace_size(ctypes.byref(_desc()), None) == 1


def test_read_error_null(L):
    v = ctypes.c_int32(0)
    assert L.smla_read_error(None, None, 4, ctypes.byref(v), None) == 1
    assert L.smla_noalloc_read_error(None, None) == 1


def test_kernel_events_hook_needs_both_or_neither(L):
    P = ctypes.c_void_p
    assert L.smla_set_kernel_events(P(16), None) == 1
    assert L.smla_set_kernel_events(None, P(16)) == 1
    assert L.smla_set_kernel_events(None, None) == 0


@pytest.mark.parametrize("kv_scale", [0.0, -1.0, float("nan"), float("inf")])
def test_per_tensor_fp8_needs_a_positive_finite_scale(L, kv_scale):
    d = _desc(kv_format=smla.SMLA_KV_FP8_TENSOR)
    d.kv_scale = kv_scale
    assert _decode_status(L, d) == 2
    P = ctypes.c_void_p
    assert L.smla_pack_kv_fp8_tensor(P(16), P(16), P(16), 4, ctypes.c_float(kv_scale), P(16), 8, None) == 2


def test_selftest_wait_rejects_bad_arguments(L):
    P = ctypes.c_void_p
    assert L.smla_selftest_wait_timeout(None, 10, None) == 1
    assert L.smla_selftest_wait_timeout(P(16), 0, None) == 2
    assert L.smla_selftest_wait_timeout(P(16), 200000, None) == 2


def test_indexer_desc_layout_and_host_checks(L):
    assert ctypes.sizeof(smla.smla_indexer_desc) == 56
    assert smla.smla_indexer_desc.num_pages.offset == 24
    P = ctypes.c_void_p

    def status(**kw):
        d = smla.make_indexer_desc(4, 1, 64, 64, 16, 8, 1024, 256)
        for k, v in kw.items():
            setattr(d, k, v)
        return L.smla_indexer_logits(ctypes.byref(d), P(16), P(16), P(16), P(16), P(16), P(16), P(16), None)

    assert status(num_heads=48) == 2
    assert status(next_n=5, num_tokens=20) == 2
    assert status(num_tokens=5) == 2                       # T must be B * next_n
    assert status(page_size=256) == 2
    assert status(num_requests=9000, num_tokens=9000) == 2
    d = smla.make_indexer_desc(4, 1, 64, 64, 16, 8, 1024, 256)
    assert L.smla_indexer_logits(ctypes.byref(d), None, P(16), P(16), P(16), P(16), P(16), P(16), None) == 1
    assert L.smla_indexer_logits(ctypes.byref(d), P(8), P(16), P(16), P(16), P(16), P(16), P(16), None) == 3
    assert L.smla_indexer_topk(ctypes.byref(d), P(16), None, P(16), None) == 1


def test_store_normed_desc_layout_and_host_checks(L):
    assert ctypes.sizeof(smla.smla_store_desc) == 48
    P = ctypes.c_void_p

    def status(**kw):
        d = smla.smla_store_desc()
        d.kv_format, d.scale_mode, d.kv_scale, d.rms_eps = smla.SMLA_KV_FP8_DS, 0, 1.0, 1e-6
        d.n, d.num_slots, d.max_position = 4, 8, 16
        for k, v in kw.items():
            setattr(d, k, v)
        return L.smla_store_kv_normed(ctypes.byref(d), P(16), P(16), P(16), P(16), P(16), P(16), P(16), None, None)

    assert status(kv_format=7) == 4
    assert status(scale_mode=3) == 4
    assert status(rms_eps=-1.0) == 2 and status(rms_eps=float("nan")) == 2
    assert status(max_position=0) == 2
    assert status(kv_format=smla.SMLA_KV_FP8_TENSOR, kv_scale=0.0) == 2
    assert status(n=0) == 0  # nothing to do
    d = smla.smla_store_desc()
    d.kv_format, d.n, d.num_slots, d.max_position = smla.SMLA_KV_BF16, 4, 8, 16
    assert L.smla_store_kv_normed(ctypes.byref(d), P(8), P(16), P(16), P(16), P(16), P(16), P(16), None, None) == 3
    assert L.smla_store_kv_normed(ctypes.byref(d), P(16), P(16), P(16), P(16), P(4), P(16), P(16), None, None) == 3
    assert L.smla_store_kv_normed(ctypes.byref(d), None, P(16), P(16), P(16), P(16), P(16), P(16), None, None) == 1


def _plan(L, d, sms=152):
    p = smla.smla_launch_plan()
    st = L.smla_plan_launches(ctypes.byref(d), sms, ctypes.byref(p))
    return st, p


def test_launch_plan_layout_matches_header():
    # int32 x8 (ctas is two of them), then one uint64 at its natural alignment
    assert ctypes.sizeof(smla.smla_launch_plan) == 40
    assert smla.smla_launch_plan.ctas.offset == 20
    assert smla.smla_launch_plan.workspace_bytes.offset == 32
    assert _header_enum("SMLA_KERNEL_") == {"SMLA_KERNEL_HEAD_GROUP": smla.SMLA_KERNEL_HEAD_GROUP,
                                            "SMLA_KERNEL_HEAD_GROUP_FP8": smla.SMLA_KERNEL_HEAD_GROUP_FP8,
                                            "SMLA_KERNEL_MMA": smla.SMLA_KERNEL_MMA}
    assert _header_enum("SMLA_MERGE_") == {"SMLA_MERGE_NONE": smla.SMLA_MERGE_NONE,
                                           "SMLA_MERGE_CLUSTER": smla.SMLA_MERGE_CLUSTER,
                                           "SMLA_MERGE_KERNEL": smla.SMLA_MERGE_KERNEL}


def _wl_desc(tokens, heads, fmt=smla.SMLA_KV_FP8_DS, topk=2048, next_n=1, **kw):
    d = smla.make_desc(tokens, heads, topk, tokens // next_n, 64, 4096, 2048, fmt, 1 / 24, next_n=next_n)
    for k, v in kw.items():
        setattr(d, k, v)
    return d


@pytest.mark.parametrize("name,desc,expect", [
    # 64 requests x 4 MTP rows x 2 head groups = 512 items = 3 waves of 152 + 56: the last 56
    # run as a second launch with two splits each
    ("mtp 256 x 128 heads", _wl_desc(256, 128, next_n=4),
     dict(kernel=1, num_splits=1, split_len=2048, merge=0, num_launches=2, ctas=(456, 112), tail_items=56,
          workspace_bytes=256)),
    ("mtp, E4M3 q, per-tensor cache", _wl_desc(256, 128, smla.SMLA_KV_FP8_TENSOR, next_n=4, q_format=1, q_scale=1.0),
     dict(kernel=2, num_splits=1, split_len=2048, merge=0, num_launches=2, ctas=(456, 112), tail_items=56,
          workspace_bytes=256)),
    # 256 items = 152 + 104: a last wave more than half full stays in the one launch
    ("128 x 128 heads", _wl_desc(128, 128),
     dict(kernel=1, num_splits=1, split_len=2048, merge=0, num_launches=1, ctas=(256, 0), tail_items=0,
          workspace_bytes=256)),
    # 32 items: four splits of 512 fill 128 SMs, merged inside the cluster
    ("32 x 64 heads", _wl_desc(32, 64),
     dict(kernel=1, num_splits=4, split_len=512, merge=1, num_launches=1, ctas=(128, 0), tail_items=0,
          workspace_bytes=256)),
    # 16 heads: the mma.sync kernel, one CTA per (token, 16 heads), 256 >= 152 so one split
    ("256 x 16 heads", _wl_desc(256, 16),
     dict(kernel=3, num_splits=1, split_len=2048, merge=0, num_launches=1, ctas=(256, 0), tail_items=0,
          workspace_bytes=256)),
    # 4 x 16 heads: about two CTAs an SM wants 76 splits, capped at 2048 / 256 = 8; fp32
    # partials of 4 x 8 x 16 rows for the merge kernel: 256 + 2048 B of LSE, 512 x 512 x 4 B
    ("4 x 16 heads", _wl_desc(4, 16),
     dict(kernel=3, num_splits=8, split_len=256, merge=2, num_launches=1, ctas=(32, 0), tail_items=0,
          workspace_bytes=2304 + 512 * 512 * 4)),
    # 12 splits asked: 2048 / 12 rounds up to 192 entries, hence 11 splits, beyond a cluster's 8:
    # f16 partials of 2 x 11 x 64 rows through the merge kernel: 256 + 5632 B of LSE, 1408 x 512 x 2 B
    ("2 x 64 heads, 12 splits asked", _wl_desc(2, 64, num_splits=12),
     dict(kernel=1, num_splits=11, split_len=192, merge=2, num_launches=1, ctas=(22, 0), tail_items=0,
          workspace_bytes=5888 + 1408 * 512 * 2)),
    # the bf16 cache takes the mma.sync kernel at any head count
    ("bf16 cache, 64 x 128 heads", _wl_desc(64, 128, smla.SMLA_KV_BF16),
     dict(kernel=3, num_splits=1, split_len=2048, merge=0, num_launches=1, ctas=(512, 0), tail_items=0,
          workspace_bytes=256)),
])
def test_plan_launches_of_the_benchmarked_shapes(L, name, desc, expect):
    st, p = _plan(L, desc)
    assert st == 0, name
    got = {k: getattr(p, k) for k in expect}
    got["ctas"] = tuple(p.ctas)
    assert got == expect, name


def test_plan_tail_split_boundaries(L):
    # items = tokens x 2 head groups; the second launch appears exactly when the remainder
    # over whole waves is at most half the SMs, and only with library-chosen splits
    for sms in (152, 148, 132):
        for tokens in range(sms // 2 + 1, 3 * sms):
            st, p = _plan(L, _wl_desc(tokens, 128), sms)
            assert st == 0
            items = 2 * tokens
            rem = items % sms
            tail = items > sms and 0 < rem and 2 * rem <= sms
            assert p.num_launches == (2 if tail else 1), (sms, tokens)
            total = p.ctas[0] + p.ctas[1]
            if tail:
                assert p.ctas[0] == items - rem and p.ctas[1] == 2 * rem and p.tail_items == rem
            elif items >= sms:
                assert p.num_splits == 1 and total == items
    st, p = _plan(L, _wl_desc(256, 128, next_n=4, num_splits=1))
    assert st == 0 and p.num_launches == 1 and tuple(p.ctas) == (512, 0)
    # short index rows keep one launch
    st, p = _plan(L, _wl_desc(256, 128, topk=256, next_n=4))
    assert st == 0 and p.num_launches == 1


def test_plan_splits_cover_the_index_row(L):
    for heads in (16, 32, 64, 128):
        for topk in (4, 64, 252, 256, 2048, 4096, 8192, 2048 * 64):
            for tokens in (1, 3, 40, 300):
                for splits in (0, 1, 5, 64):
                    st, p = _plan(L, _wl_desc(tokens, heads, topk=topk, num_splits=splits))
                    assert st == 0
                    S, n = p.num_splits, p.split_len
                    assert n % 64 == 0 and n <= 2048 and 1 <= S <= 64
                    assert (S - 1) * n < topk <= S * n, (heads, topk, tokens, splits, S, n)
                    if S == 1:
                        assert p.merge == smla.SMLA_MERGE_NONE
                    elif heads >= 64 and S <= 8:
                        assert p.merge == smla.SMLA_MERGE_CLUSTER and p.workspace_bytes == 256
                    else:
                        assert p.merge == smla.SMLA_MERGE_KERNEL and p.workspace_bytes > 256


def test_plan_launches_host_checks(L):
    p = smla.smla_launch_plan()
    assert L.smla_plan_launches(None, 152, ctypes.byref(p)) == 1
    assert L.smla_plan_launches(ctypes.byref(_desc()), 152, None) == 1
    assert L.smla_plan_launches(ctypes.byref(_desc()), 0, ctypes.byref(p)) == 2
    p.kernel = 7
    assert L.smla_plan_launches(ctypes.byref(_desc(num_heads=8)), 152, ctypes.byref(p)) == 2
    assert p.kernel == 0  # zeroed on error
    assert smla.plan_launches(_desc(), 152).kernel == smla.SMLA_KERNEL_MMA


def test_without_a_device_every_launching_call_fails_loudly(L):
    # No CPU fallback: with no sm_103 device, every call that would launch returns
    # SMLA_ERR_DEVICE after its argument checks, and only the host-only plan query answers.
    # smla_workspace_size launches nothing and tells whether a device is present; with one,
    # these dummy pointers must not reach a launch, so the test stops there.
    n = ctypes.c_size_t(0)
    if L.smla_workspace_size(ctypes.byref(_desc()), ctypes.byref(n)) != 8:
        pytest.skip("an sm_103 device is present")
    P = ctypes.c_void_p
    v = ctypes.c_int32(0)
    assert _decode_status(L, _desc()) == 8
    assert L.smla_decode_noalloc(ctypes.byref(_desc()), P(16), P(16), P(16), P(16), None, None, P(16), None,
                                 None) == 8
    assert L.smla_pack_kv(1, 0, P(16), P(16), P(16), 4, P(16), 8, None) == 8
    assert L.smla_pack_kv_fp8_tensor(P(16), P(16), P(16), 4, ctypes.c_float(1.0), P(16), 8, None) == 8
    sd = smla.smla_store_desc()
    sd.kv_format, sd.n, sd.num_slots, sd.max_position = smla.SMLA_KV_BF16, 4, 8, 16
    assert L.smla_store_kv_normed(ctypes.byref(sd), P(16), P(16), P(16), P(16), P(16), P(16), P(16), None,
                                  None) == 8
    assert L.smla_gather_dequant(ctypes.byref(_desc()), P(16), P(16), P(16), None, P(16), None, None) == 8
    xd = smla.make_indexer_desc(4, 1, 64, 64, 16, 8, 1024, 256)
    assert L.smla_indexer_logits(ctypes.byref(xd), P(16), P(16), P(16), P(16), P(16), P(16), P(16), None) == 8
    assert L.smla_indexer_topk(ctypes.byref(xd), P(16), P(16), P(16), None) == 8
    assert L.smla_selftest_wait_timeout(P(16), 10, None) == 8
    assert L.smla_noalloc_read_error(ctypes.byref(v), None) == 8
    p = smla.smla_launch_plan()
    assert L.smla_plan_launches(ctypes.byref(_desc()), 152, ctypes.byref(p)) == 0


def test_descriptor_rules_one_violation_at_a_time(L):
    # every field rule of smla_desc as the header states it, checked through the host-only plan
    # query (which runs smla_decode's descriptor checks and touches no device): a valid
    # descriptor passes, and each single violation gives its documented status
    import numpy as np
    g = np.random.default_rng(17)
    violations = [
        ("num_tokens", 0, 2), ("num_requests", 0, 2), ("next_n", 0, 2), ("topk", 0, 2),
        ("num_heads", 0, 2), ("num_heads", 24, 2), ("num_heads", 144, 2), ("topk", 130, 2),
        ("topk", 64 * 2048 + 4, 2), ("page_size", 3, 2), ("page_size", 8192, 2), ("num_pages", 0, 2),
        ("num_pages", (1 << 31) + 1, 2), ("page_table_stride", 0, 2), ("kv_format", 3, 4),
        ("sm_scale", float("inf"), 2), ("num_splits", -1, 2), ("num_splits", 65, 2), ("q_format", 2, 4),
    ]
    p = smla.smla_launch_plan()
    for _ in range(200):
        d = smla.make_desc(int(g.integers(1, 400)), 16 * int(g.integers(1, 9)), 4 * int(g.integers(1, 4097)),
                           int(g.integers(1, 64)), 1 << int(g.integers(0, 13)), int(g.integers(1, 1 << 20)),
                           int(g.integers(1, 4096)), int(g.integers(0, 3)), float(g.uniform(0.01, 1.0)),
                           next_n=int(g.integers(1, 5)), num_splits=int(g.integers(0, 65)),
                           kv_scale=float(g.uniform(0.001, 2.0)))
        assert L.smla_plan_launches(ctypes.byref(d), 152, ctypes.byref(p)) == 0
        assert 1 <= p.num_splits <= 64 and p.ctas[0] >= 1
        field, value, status = violations[int(g.integers(len(violations)))]
        setattr(d, field, value)
        assert L.smla_plan_launches(ctypes.byref(d), 152, ctypes.byref(p)) == status, (field, value)
