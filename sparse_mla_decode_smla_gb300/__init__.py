"""Python binding of libsmla.so (GB300 sparse MLA decode).

Argument marshalling only: every step of the decode runs in the library's CUDA
kernels. The functions mirror the C ABI in include/smla.h and take torch
tensors for device memory and the current torch stream. There is no fallback:
importing fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

from ._build import LIB as LIB_PATH

SMLA_KV_BF16 = 0
SMLA_KV_FP8_DS = 1
SMLA_KV_FP8_TENSOR = 2
SMLA_SCALE_POW2 = 0
SMLA_SCALE_FP32 = 1
SMLA_Q_BF16 = 0
SMLA_Q_FP8_E4M3 = 1
SMLA_DEVERR_INDEX = 1
SMLA_DEVERR_PAGE = 2
SMLA_DEVERR_TIMEOUT = 4
SMLA_DEVERR_RANGE = 8
SMLA_KERNEL_HEAD_GROUP = 1
SMLA_KERNEL_HEAD_GROUP_FP8 = 2
SMLA_KERNEL_MMA = 3
SMLA_MERGE_NONE = 0
SMLA_MERGE_CLUSTER = 1
SMLA_MERGE_KERNEL = 2

STATUS = {0: "SMLA_OK", 1: "SMLA_ERR_NULL", 2: "SMLA_ERR_SHAPE", 3: "SMLA_ERR_ALIGN",
          4: "SMLA_ERR_UNSUPPORTED", 5: "SMLA_ERR_WORKSPACE", 6: "SMLA_ERR_CUDA",
          7: "SMLA_ERR_INDEX_RANGE", 8: "SMLA_ERR_DEVICE", 9: "SMLA_ERR_TIMEOUT",
          10: "SMLA_ERR_OPERAND_RANGE"}
DEVICE_ERROR_STATUSES = (0, 7, 9, 10)  # statuses that report device error bits
EXPORTS = ["smla_status_string", "smla_abi_version", "smla_workspace_size", "smla_decode",
           "smla_pack_kv", "smla_gather_dequant", "smla_read_error", "smla_decode_noalloc",
           "smla_set_kernel_events", "smla_pack_kv_fp8_tensor", "smla_selftest_wait_timeout",
           "smla_noalloc_read_error", "smla_indexer_logits", "smla_indexer_topk", "smla_store_kv_normed",
           "smla_plan_launches"]
NOALLOC_SCRATCH_BYTES = 16 << 20


class SmlaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({status_string(status)})")


class smla_desc(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("num_requests", ctypes.c_int32),
                ("next_n", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int64), ("page_table_stride", ctypes.c_int32),
                ("kv_format", ctypes.c_int32), ("sm_scale", ctypes.c_float),
                ("num_splits", ctypes.c_int32), ("kv_scale", ctypes.c_float),
                ("q_format", ctypes.c_int32), ("q_scale", ctypes.c_float),
                ("reserved", ctypes.c_int32 * 1)]


class smla_launch_plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("num_splits", ctypes.c_int32),
                ("split_len", ctypes.c_int32), ("merge", ctypes.c_int32),
                ("num_launches", ctypes.c_int32), ("ctas", ctypes.c_int32 * 2),
                ("tail_items", ctypes.c_int32), ("workspace_bytes", ctypes.c_uint64)]


class smla_indexer_desc(ctypes.Structure):
    _fields_ = [("num_tokens", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("num_requests", ctypes.c_int32), ("next_n", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("page_table_stride", ctypes.c_int32),
                ("num_pages", ctypes.c_int64), ("logits_stride", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("reserved", ctypes.c_int32 * 4)]


class smla_store_desc(ctypes.Structure):
    _fields_ = [("kv_format", ctypes.c_int32), ("scale_mode", ctypes.c_int32),
                ("kv_scale", ctypes.c_float), ("rms_eps", ctypes.c_float), ("n", ctypes.c_int64),
                ("num_slots", ctypes.c_int64), ("max_position", ctypes.c_int64),
                ("reserved", ctypes.c_int32 * 2)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libsmla.so (raises when it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with sparse_mla_decode_smla_gb300._build.build()")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        D = ctypes.POINTER(smla_desc)
        L.smla_status_string.restype = ctypes.c_char_p
        L.smla_status_string.argtypes = [I32]
        L.smla_abi_version.restype = I32
        L.smla_abi_version.argtypes = []
        L.smla_workspace_size.restype = I32
        L.smla_workspace_size.argtypes = [D, ctypes.POINTER(SZ)]
        L.smla_plan_launches.restype = I32
        L.smla_plan_launches.argtypes = [D, I32, ctypes.POINTER(smla_launch_plan)]
        L.smla_decode.restype = I32
        L.smla_decode.argtypes = [D, P, P, P, P, P, P, P, P, P, SZ, P]
        L.smla_pack_kv.restype = I32
        L.smla_pack_kv.argtypes = [I32, I32, P, P, P, I64, P, I64, P]
        L.smla_pack_kv_fp8_tensor.restype = I32
        L.smla_pack_kv_fp8_tensor.argtypes = [P, P, P, I64, ctypes.c_float, P, I64, P]
        L.smla_gather_dequant.restype = I32
        L.smla_gather_dequant.argtypes = [D, P, P, P, P, P, P, P]
        L.smla_decode_noalloc.restype = I32
        L.smla_decode_noalloc.argtypes = [D, P, P, P, P, P, P, P, P, P]
        L.smla_set_kernel_events.restype = I32
        L.smla_set_kernel_events.argtypes = [P, P]
        L.smla_selftest_wait_timeout.restype = I32
        L.smla_selftest_wait_timeout.argtypes = [P, ctypes.c_uint32, P]
        L.smla_read_error.restype = I32
        L.smla_read_error.argtypes = [D, P, SZ, ctypes.POINTER(I32), P]
        L.smla_noalloc_read_error.restype = I32
        L.smla_noalloc_read_error.argtypes = [ctypes.POINTER(I32), P]
        XD = ctypes.POINTER(smla_indexer_desc)
        L.smla_indexer_logits.restype = I32
        L.smla_indexer_logits.argtypes = [XD, P, P, P, P, P, P, P, P]
        L.smla_indexer_topk.restype = I32
        L.smla_indexer_topk.argtypes = [XD, P, P, P, P]
        L.smla_store_kv_normed.restype = I32
        L.smla_store_kv_normed.argtypes = [ctypes.POINTER(smla_store_desc), P, P, P, P, P, P, P, P, P]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().smla_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return ctypes.c_void_p(int(getattr(stream, "cuda_stream", stream)))  # a torch stream or a handle


def _check(fn: str, status: int):
    if status != 0:
        raise SmlaError(fn, status)


def make_desc(num_tokens, num_heads, topk, num_requests, page_size, num_pages, page_table_stride,
              kv_format, sm_scale, next_n=1, num_splits=0, kv_scale=1.0, q_format=0,
              q_scale=1.0) -> smla_desc:
    d = smla_desc()
    d.num_tokens, d.num_heads, d.topk = num_tokens, num_heads, topk
    d.num_requests, d.next_n, d.page_size = num_requests, next_n, page_size
    d.num_pages, d.page_table_stride = num_pages, page_table_stride
    d.kv_format, d.sm_scale, d.num_splits = kv_format, sm_scale, num_splits
    d.kv_scale = kv_scale
    d.q_format, d.q_scale = q_format, q_scale
    return d


def workspace_size(desc: smla_desc) -> int:
    n = ctypes.c_size_t(0)
    _check("smla_workspace_size", lib().smla_workspace_size(ctypes.byref(desc), ctypes.byref(n)))
    return n.value


def plan_launches(desc: smla_desc, num_sms: int) -> smla_launch_plan:
    """The launches smla_decode makes for desc on a device with num_sms SMs (host-only)."""
    p = smla_launch_plan()
    _check("smla_plan_launches", lib().smla_plan_launches(ctypes.byref(desc), int(num_sms), ctypes.byref(p)))
    return p


def decode(desc, q, kv_cache, page_table, topk, req_id_per_token, sink, out, lse, workspace,
           stream=None):
    _check("smla_decode", lib().smla_decode(
        ctypes.byref(desc), _ptr(q), _ptr(kv_cache), _ptr(page_table), _ptr(topk),
        _ptr(req_id_per_token), _ptr(sink), _ptr(out), _ptr(lse), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def decode_noalloc(desc, q, kv_cache, page_table, topk, req_id_per_token, sink, out, lse,
                   stream=None):
    """smla_decode with the library's own scratch array instead of a workspace.

    For callers that cannot allocate device memory. Calls share one scratch array per
    device, so overlapping calls race; the first call on a device must precede any
    stream capture.
    """
    _check("smla_decode_noalloc", lib().smla_decode_noalloc(
        ctypes.byref(desc), _ptr(q), _ptr(kv_cache), _ptr(page_table), _ptr(topk),
        _ptr(req_id_per_token), _ptr(sink), _ptr(out), _ptr(lse), _stream(stream)))


def set_kernel_events(start=None, stop=None):
    """Record `start` / `stop` (torch.cuda.Event, already created) around the decode kernel
    of every later decode call from this thread; no arguments turns recording off."""
    def handle(ev):
        if ev is None:
            return None
        h = int(ev.cuda_event)
        if h == 0:
            raise ValueError("the event has not been created yet: record it once first")
        return ctypes.c_void_p(h)
    _check("smla_set_kernel_events", lib().smla_set_kernel_events(handle(start), handle(stop)))


def pack_kv(kv_format, scale_mode, latent, rope, slot_mapping, kv_cache, num_slots, stream=None):
    _check("smla_pack_kv", lib().smla_pack_kv(
        kv_format, scale_mode, _ptr(latent), _ptr(rope), _ptr(slot_mapping), latent.shape[0],
        _ptr(kv_cache), num_slots, _stream(stream)))


def pack_kv_fp8_tensor(latent, rope, slot_mapping, kv_cache, num_slots, kv_scale, stream=None):
    _check("smla_pack_kv_fp8_tensor", lib().smla_pack_kv_fp8_tensor(
        _ptr(latent), _ptr(rope), _ptr(slot_mapping), latent.shape[0], float(kv_scale),
        _ptr(kv_cache), num_slots, _stream(stream)))


def gather_dequant(desc, kv_cache, page_table, topk, req_id_per_token, rows, error_word=None,
                   stream=None):
    _check("smla_gather_dequant", lib().smla_gather_dequant(
        ctypes.byref(desc), _ptr(kv_cache), _ptr(page_table), _ptr(topk), _ptr(req_id_per_token),
        _ptr(rows), _ptr(error_word), _stream(stream)))


def selftest_wait_timeout(error_word, limit_us: int, stream=None):
    """Run the bounded-wait self-test: error_word (device int32) gets SMLA_DEVERR_TIMEOUT."""
    _check("smla_selftest_wait_timeout", lib().smla_selftest_wait_timeout(
        _ptr(error_word), int(limit_us), _stream(stream)))


def read_error(desc, workspace, stream=None) -> int:
    """Synchronises, returns and clears the device error word (SMLA_DEVERR_* bits)."""
    v = ctypes.c_int32(0)
    st = lib().smla_read_error(ctypes.byref(desc), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), ctypes.byref(v),
                               _stream(stream))
    if st not in DEVICE_ERROR_STATUSES:
        raise SmlaError("smla_read_error", st)
    return v.value


def noalloc_read_error(stream=None) -> int:
    """Synchronises, returns and clears the error word of decode_noalloc (SMLA_DEVERR_* bits)."""
    v = ctypes.c_int32(0)
    st = lib().smla_noalloc_read_error(ctypes.byref(v), _stream(stream))
    if st not in DEVICE_ERROR_STATUSES:
        raise SmlaError("smla_noalloc_read_error", st)
    return v.value


def make_indexer_desc(num_requests, next_n, num_heads, page_size, num_pages, page_table_stride,
                      logits_stride, topk) -> smla_indexer_desc:
    d = smla_indexer_desc()
    d.num_tokens, d.num_heads, d.num_requests = num_requests * next_n, num_heads, num_requests
    d.next_n, d.page_size, d.page_table_stride = next_n, page_size, page_table_stride
    d.num_pages, d.logits_stride, d.topk = num_pages, logits_stride, topk
    return d


def indexer_logits(desc, q, weights, k_cache, page_table, context_lens, logits, error_word,
                   stream=None):
    """FP8 paged MQA logits (smla_indexer_logits): logits[t, s] for every visible slot."""
    _check("smla_indexer_logits", lib().smla_indexer_logits(
        ctypes.byref(desc), _ptr(q), _ptr(weights), _ptr(k_cache), _ptr(page_table),
        _ptr(context_lens), _ptr(logits), _ptr(error_word), _stream(stream)))


def indexer_topk(desc, logits, context_lens, topk, stream=None):
    """Top-k slots of every token's visible logits (smla_indexer_topk), ascending, -1 padded."""
    _check("smla_indexer_topk", lib().smla_indexer_topk(
        ctypes.byref(desc), _ptr(logits), _ptr(context_lens), _ptr(topk), _stream(stream)))


def store_kv_normed(kv_format, latent, rope, norm_weight, eps, positions, cos_sin, slot_mapping, kv_cache,
                    num_slots, scale_mode=SMLA_SCALE_POW2, kv_scale=1.0, error_word=None, stream=None):
    """The cache write fused with RMSNorm and RoPE (smla_store_kv_normed)."""
    d = smla_store_desc()
    d.kv_format, d.scale_mode, d.kv_scale, d.rms_eps = kv_format, scale_mode, kv_scale, eps
    d.n, d.num_slots, d.max_position = latent.shape[0], num_slots, cos_sin.shape[0]
    _check("smla_store_kv_normed", lib().smla_store_kv_normed(
        ctypes.byref(d), _ptr(latent), _ptr(rope), _ptr(norm_weight), _ptr(positions), _ptr(cos_sin),
        _ptr(slot_mapping), _ptr(kv_cache), _ptr(error_word), _stream(stream)))
