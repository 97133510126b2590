// C ABI of libsmla.so: argument checks, split planning and kernel dispatch.
// Nothing here allocates device memory or synchronises (except smla_read_error).
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>

#include "../../include/smla.h"
#include "indexer.h"
#include "kernels.h"

namespace {

constexpr size_t kWsAlign = 256;
constexpr int kMaxDevices = 64;

// Per-device facts, looked up on first use. Several host threads may look them up at
// once; they store the same values, through atomics.
struct DevInfo {
  std::atomic<int> ok{-1};  // -1 unknown, 0 unusable, 1 sm_103
  std::atomic<int> num_sms{0};
};
DevInfo g_dev[kMaxDevices];

// Events of smla_set_kernel_events, per host thread (NULL: no recording).
thread_local cudaEvent_t t_ev_start = nullptr;
thread_local cudaEvent_t t_ev_stop = nullptr;

smla_status current_device(int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return SMLA_ERR_DEVICE;
  }
  DevInfo* di = dev < kMaxDevices ? &g_dev[dev] : nullptr;
  int ok = di ? di->ok.load(std::memory_order_acquire) : -1;
  int sms = di ? di->num_sms.load(std::memory_order_relaxed) : 0;
  if (ok < 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return SMLA_ERR_DEVICE;
    }
    ok = (major == 10 && minor == 3) ? 1 : 0;
    if (di) {
      di->num_sms.store(sms, std::memory_order_relaxed);
      di->ok.store(ok, std::memory_order_release);
    }
  }
  if (ok != 1) return SMLA_ERR_DEVICE;
  *num_sms = sms;
  return SMLA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

smla_status check_desc(const smla_desc* d) {
  if (!d) return SMLA_ERR_NULL;
  if (d->num_tokens < 1 || d->num_requests < 1 || d->next_n < 1 || d->topk < 1)
    return SMLA_ERR_SHAPE;
  if (d->num_heads < 16 || d->num_heads > 128 || d->num_heads % 16 != 0) return SMLA_ERR_SHAPE;
  if (d->topk % 4 != 0) return SMLA_ERR_SHAPE;
  if (!is_pow2(d->page_size) || d->page_size > 4096) return SMLA_ERR_SHAPE;
  if (d->num_pages < 1 || d->page_table_stride < 1) return SMLA_ERR_SHAPE;
  if (d->num_pages > (int64_t(1) << 31)) return SMLA_ERR_SHAPE;
  if (d->kv_format != SMLA_KV_BF16 && d->kv_format != SMLA_KV_FP8_DS &&
      d->kv_format != SMLA_KV_FP8_TENSOR)
    return SMLA_ERR_UNSUPPORTED;
  if (!isfinite(d->sm_scale)) return SMLA_ERR_SHAPE;
  if (d->kv_format == SMLA_KV_FP8_TENSOR && !(isfinite(d->kv_scale) && d->kv_scale > 0.f))
    return SMLA_ERR_SHAPE;
  if (d->num_splits < 0 || d->num_splits > smla::kMaxSplits) return SMLA_ERR_SHAPE;
  if (d->topk > smla::kMaxSplits * smla::kMaxSplitLen) return SMLA_ERR_SHAPE;
  if (d->reserved[0] != 0) return SMLA_ERR_SHAPE;
  if (d->q_format != SMLA_Q_BF16 && d->q_format != SMLA_Q_FP8_E4M3) return SMLA_ERR_UNSUPPORTED;
  if (d->q_format == SMLA_Q_FP8_E4M3) {
    if (!(isfinite(d->q_scale) && d->q_scale > 0.f)) return SMLA_ERR_SHAPE;
    // E4M3 q runs on the FP8-operand tensor-core kernel only
    if (d->kv_format != SMLA_KV_FP8_TENSOR || d->num_heads < smla::kHgMinHeads) return SMLA_ERR_UNSUPPORTED;
  }
  return SMLA_OK;
}

struct Plan {
  int num_splits;
  int split_len;
  bool cluster_merge;  // the tensor-core kernel merges its splits inside a thread-block cluster
  size_t lse_off, o_off, bytes;
};

// The FP8 caches with 64 or more heads take the tensor-core head-group kernel.
bool use_hg(const smla_desc* d) {
  return (d->kv_format == SMLA_KV_FP8_DS || d->kv_format == SMLA_KV_FP8_TENSOR) &&
         d->num_heads >= smla::kHgMinHeads;
}

Plan make_plan(const smla_desc* d, int num_sms) {
  int S = d->num_splits;
  if (S == 0) {
    S = 1;
    if (use_hg(d)) {
      // one CTA per (token, split, group of 64 heads), one per SM: fill one wave at most,
      // with splits that fit one cluster (merged in the kernel)
      const int units = d->num_tokens * ((d->num_heads + 63) / 64);
      if (units < num_sms) S = std::min(num_sms / units, smla::kMaxClusterMerge);
    } else {
      const int units = d->num_tokens * (d->num_heads / 16);
      if (units < num_sms) S = (2 * num_sms + units - 1) / units;
    }
    const int cap = d->topk / 256 > 1 ? d->topk / 256 : 1;  // at least 256 slots per split
    if (S > cap) S = cap;
  }
  const int min_splits = (d->topk + smla::kMaxSplitLen - 1) / smla::kMaxSplitLen;
  if (S < min_splits) S = min_splits;
  if (S > smla::kMaxSplits) S = smla::kMaxSplits;
  int len = (d->topk + S - 1) / S;
  len = (len + smla::kTile - 1) / smla::kTile * smla::kTile;
  S = (d->topk + len - 1) / len;
  Plan p;
  p.num_splits = S;
  p.split_len = len;
  p.cluster_merge = use_hg(d) && S > 1 && S <= smla::kMaxClusterMerge;
  p.lse_off = kWsAlign;
  size_t bytes = kWsAlign;
  if (S > 1 && !p.cluster_merge) {  // split partials in global memory, for the merge kernel
    const size_t rows = size_t(d->num_tokens) * S * d->num_heads;
    bytes = round_up(p.lse_off + rows * 4, kWsAlign);
    p.o_off = bytes;
    // the tensor-core kernel writes f16 partial rows, the mma.sync kernel fp32 ones
    bytes += rows * 512 * (use_hg(d) ? 2 : 4);
  } else {
    p.o_off = bytes;
  }
  p.bytes = bytes;
  return p;
}

// Tail split (head-group kernels, library-chosen splits): when the (token, head group) items
// fill whole waves of one CTA per SM plus a remainder of at most half a wave, the remainder
// runs as a second launch with two splits an item, merged inside their cluster, so the last
// wave takes about half a CTA's time instead of a whole one.
struct Tail {
  bool on;
  int units;     // (token, head group) items
  int rem;       // items of the second launch
  int split_len; // index entries per split of the second launch
};

Tail plan_tail(const smla_desc* d, const Plan& plan, int num_sms) {
  Tail t;
  t.units = d->num_tokens * ((d->num_heads + 63) / 64);
  t.rem = t.units % num_sms;
  t.on = use_hg(d) && d->num_splits == 0 && plan.num_splits == 1 && d->topk >= 512 && t.units > num_sms &&
         t.rem > 0 && 2 * t.rem <= num_sms;
  t.split_len = ((d->topk + 1) / 2 + smla::kTile - 1) / smla::kTile * smla::kTile;
  return t;
}

int ilog2(int x) {
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

smla::DecodeArgs make_args(const smla_desc* d, const void* q, const void* kv,
                           const int32_t* pt, const int32_t* topk, const int32_t* req,
                           const float* sink) {
  smla::DecodeArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.kv = static_cast<const uint8_t*>(kv);
  a.page_table = pt;
  a.topk = topk;
  a.req_id = req;
  a.sink = sink;
  a.T = d->num_tokens;
  a.H = d->num_heads;
  a.K = d->topk;
  a.B = d->num_requests;
  a.next_n = d->next_n;
  a.stride = d->page_table_stride;
  a.log2_page = ilog2(d->page_size);
  a.kv_format = d->kv_format;
  a.num_pages = d->num_pages;
  a.c2 = d->sm_scale * 1.4426950408889634f;
  a.kv_scale = d->kv_format == SMLA_KV_FP8_TENSOR ? d->kv_scale : 1.f;
  a.q_fp8 = d->q_format == SMLA_Q_FP8_E4M3 ? 1 : 0;
  a.q_scale = a.q_fp8 ? d->q_scale : 1.f;
  return a;
}

smla_status check_indexer_desc(const smla_indexer_desc* d) {
  if (!d) return SMLA_ERR_NULL;
  if (d->num_requests < 1 || d->num_requests > smla::kIxMaxRequests || d->next_n < 1 || d->next_n > 4)
    return SMLA_ERR_SHAPE;
  if (int64_t(d->num_tokens) != int64_t(d->num_requests) * d->next_n) return SMLA_ERR_SHAPE;
  if (d->num_heads != 32 && d->num_heads != 64) return SMLA_ERR_SHAPE;
  if (d->num_heads * d->next_n > 256) return SMLA_ERR_SHAPE;
  if (d->page_size != 16 && d->page_size != 32 && d->page_size != 64 && d->page_size != 128) return SMLA_ERR_SHAPE;
  if (d->page_table_stride < 1 || d->num_pages < 1 || d->num_pages >= (int64_t(1) << 31)) return SMLA_ERR_SHAPE;
  if (d->logits_stride < 1 || d->topk < 1) return SMLA_ERR_SHAPE;
  for (int i = 0; i < 4; ++i)
    if (d->reserved[i] != 0) return SMLA_ERR_SHAPE;
  return SMLA_OK;
}

smla::IndexerArgs make_indexer_args(const smla_indexer_desc* d, const int32_t* ctx) {
  smla::IndexerArgs a;
  memset(&a, 0, sizeof(a));
  a.ctx = ctx;
  a.T = d->num_tokens;
  a.H = d->num_heads;
  a.B = d->num_requests;
  a.next_n = d->next_n;
  a.stride = d->page_table_stride;
  a.log2_page = ilog2(d->page_size);
  a.logits_stride = d->logits_stride;
  a.K = d->topk;
  a.num_pages = d->num_pages;
  return a;
}

// The status smla_read_error reports for a device error word: a timeout first (every
// output of the call is invalid), then invalid entries, then operands outside the f16 window.
smla_status error_status(int32_t v) {
  if (v & SMLA_DEVERR_TIMEOUT) return SMLA_ERR_TIMEOUT;
  if (v & (SMLA_DEVERR_INDEX | SMLA_DEVERR_PAGE)) return SMLA_ERR_INDEX_RANGE;
  if (v & SMLA_DEVERR_RANGE) return SMLA_ERR_OPERAND_RANGE;
  return SMLA_OK;
}

}  // namespace

extern "C" {

const char* smla_status_string(int32_t s) {
  switch (s) {
    case SMLA_OK: return "ok";
    case SMLA_ERR_NULL: return "null pointer";
    case SMLA_ERR_SHAPE: return "size out of range";
    case SMLA_ERR_ALIGN: return "misaligned pointer";
    case SMLA_ERR_UNSUPPORTED: return "unsupported combination";
    case SMLA_ERR_WORKSPACE: return "workspace too small";
    case SMLA_ERR_CUDA: return "CUDA error";
    case SMLA_ERR_INDEX_RANGE: return "invalid index or page entry met on the device";
    case SMLA_ERR_DEVICE: return "no sm_103 device";
    case SMLA_ERR_TIMEOUT: return "a pipeline wait on the device gave up (outputs invalid)";
    case SMLA_ERR_OPERAND_RANGE: return "a block scale or RoPE value outside the f16 window met on the device";
    default: return "unknown status";
  }
}

int32_t smla_abi_version(void) { return 5; }

smla_status smla_workspace_size(const smla_desc* d, size_t* bytes) {
  if (!bytes) return SMLA_ERR_NULL;
  *bytes = 0;
  smla_status st = check_desc(d);
  if (st != SMLA_OK) return st;
  int sms = 0;
  st = current_device(&sms);
  if (st != SMLA_OK) return st;
  *bytes = make_plan(d, sms).bytes;
  return SMLA_OK;
}

smla_status smla_plan_launches(const smla_desc* d, int32_t num_sms, smla_launch_plan* p) {
  if (!p) return SMLA_ERR_NULL;
  memset(p, 0, sizeof(*p));
  smla_status st = check_desc(d);
  if (st != SMLA_OK) return st;
  if (num_sms < 1) return SMLA_ERR_SHAPE;
  const Plan plan = make_plan(d, num_sms);
  const Tail tail = plan_tail(d, plan, num_sms);
  p->kernel = d->q_format == SMLA_Q_FP8_E4M3 ? SMLA_KERNEL_HEAD_GROUP_FP8
              : use_hg(d)                    ? SMLA_KERNEL_HEAD_GROUP
                                             : SMLA_KERNEL_MMA;
  p->num_splits = plan.num_splits;
  p->split_len = plan.split_len;
  p->merge = plan.num_splits == 1 ? SMLA_MERGE_NONE : plan.cluster_merge ? SMLA_MERGE_CLUSTER : SMLA_MERGE_KERNEL;
  if (!use_hg(d)) {
    p->num_launches = 1;
    p->ctas[0] = d->num_tokens * plan.num_splits * (d->num_heads / 16);
  } else if (tail.on) {
    p->num_launches = 2;
    p->ctas[0] = (tail.units - tail.rem) * plan.num_splits;
    p->ctas[1] = tail.rem * 2;
    p->tail_items = tail.rem;
  } else {
    p->num_launches = 1;
    p->ctas[0] = tail.units * plan.num_splits;
  }
  p->workspace_bytes = plan.bytes;
  return SMLA_OK;
}

smla_status smla_decode(const smla_desc* d, const void* q, const void* kv_cache,
                        const int32_t* page_table, const int32_t* topk,
                        const int32_t* req_id_per_token, const float* sink, void* out,
                        float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  smla_status st = check_desc(d);
  if (st != SMLA_OK) return st;
  // rows are gathered by 32-bit row coordinates (one past the last slot marks a masked row)
  if (d->num_pages * d->page_size >= smla::kMaxGatherSlots) return SMLA_ERR_SHAPE;
  if (!q || !kv_cache || !page_table || !topk || !out || !workspace) return SMLA_ERR_NULL;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(topk, 16) || !aligned(out, 16) ||
      !aligned(page_table, 4) || !aligned(workspace, kWsAlign) ||
      (req_id_per_token && !aligned(req_id_per_token, 4)) || (sink && !aligned(sink, 4)) ||
      (lse && !aligned(lse, 4)))
    return SMLA_ERR_ALIGN;
  if (!req_id_per_token && (d->num_tokens - 1) / d->next_n >= d->num_requests)
    return SMLA_ERR_SHAPE;
  int sms = 0;
  st = current_device(&sms);
  if (st != SMLA_OK) return st;
  const Plan plan = make_plan(d, sms);
  if (workspace_bytes < plan.bytes) return SMLA_ERR_WORKSPACE;
  smla::DecodeArgs a = make_args(d, q, kv_cache, page_table, topk, req_id_per_token, sink);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.out = out;
  a.lse = lse;
  a.err = reinterpret_cast<int32_t*>(ws);
  a.lse_part = reinterpret_cast<float*>(ws + plan.lse_off);
  a.o_part = reinterpret_cast<float*>(ws + plan.o_off);
  a.num_splits = plan.num_splits;
  a.split_len = plan.split_len;
  // the tensor-core kernel's keys, hence its normalised partials, lie within f16's range;
  // up to a cluster's worth of its splits merge inside the kernel
  a.part_f16 = use_hg(d) ? 1 : 0;
  a.cluster_merge = plan.cluster_merge ? 1 : 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto launch = [&](const smla::DecodeArgs& x) {
    return x.q_fp8 ? smla::launch_decode_hg_f8(x, s)
                   : use_hg(d) ? smla::launch_decode_hg(x, s) : smla::launch_decode_mma(x, sms, s);
  };
  const Tail tail = plan_tail(d, plan, sms);
  if (t_ev_start && cudaEventRecord(t_ev_start, s) != cudaSuccess) return SMLA_ERR_CUDA;
  cudaError_t e;
  if (tail.on) {
    smla::DecodeArgs full = a, last = a;
    full.nitems = tail.units - tail.rem;
    last.item0 = tail.units - tail.rem;
    last.nitems = tail.rem;
    last.num_splits = 2;
    last.split_len = tail.split_len;
    last.cluster_merge = 1;
    // the remainder's items are independent of the whole waves': its CTAs take SMs as the last
    // wave's CTAs leave, with no launch gap in between
    last.overlap_prev = 1;
    e = launch(full);
    if (e == cudaSuccess) e = launch(last);
  } else {
    e = launch(a);
  }
  if (e != cudaSuccess) return SMLA_ERR_CUDA;
  if (t_ev_stop && cudaEventRecord(t_ev_stop, s) != cudaSuccess) return SMLA_ERR_CUDA;
  if (plan.num_splits > 1 && !a.cluster_merge && smla::launch_merge(a, s) != cudaSuccess) return SMLA_ERR_CUDA;
  return SMLA_OK;
}

smla_status smla_set_kernel_events(void* start, void* stop) {
  if ((start == nullptr) != (stop == nullptr)) return SMLA_ERR_NULL;
  t_ev_start = static_cast<cudaEvent_t>(start);
  t_ev_stop = static_cast<cudaEvent_t>(stop);
  return SMLA_OK;
}

smla_status smla_pack_kv(int32_t kv_format, int32_t scale_mode, const void* latent,
                         const void* rope, const int64_t* slot_mapping, int64_t n,
                         void* kv_cache, int64_t num_slots, void* stream) {
  if (kv_format != SMLA_KV_BF16 && kv_format != SMLA_KV_FP8_DS) return SMLA_ERR_UNSUPPORTED;
  if (scale_mode != SMLA_SCALE_POW2 && scale_mode != SMLA_SCALE_FP32) return SMLA_ERR_UNSUPPORTED;
  if (n < 0 || num_slots < 0) return SMLA_ERR_SHAPE;
  if (n == 0) return SMLA_OK;
  if (!latent || !rope || !slot_mapping || !kv_cache) return SMLA_ERR_NULL;
  if (!aligned(latent, 16) || !aligned(rope, 16) || !aligned(kv_cache, 16) ||
      !aligned(slot_mapping, 8))
    return SMLA_ERR_ALIGN;
  if (n > (int64_t(1) << 36)) return SMLA_ERR_SHAPE;
  int sms = 0;
  smla_status st = current_device(&sms);
  if (st != SMLA_OK) return st;
  if (smla::launch_pack(kv_format, scale_mode, 1.f, latent, rope, slot_mapping, n, kv_cache, num_slots,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SMLA_ERR_CUDA;
  return SMLA_OK;
}

smla_status smla_pack_kv_fp8_tensor(const void* latent, const void* rope,
                                    const int64_t* slot_mapping, int64_t n, float kv_scale,
                                    void* kv_cache, int64_t num_slots, void* stream) {
  if (!(isfinite(kv_scale) && kv_scale > 0.f)) return SMLA_ERR_SHAPE;
  if (n < 0 || num_slots < 0) return SMLA_ERR_SHAPE;
  if (n == 0) return SMLA_OK;
  if (!latent || !rope || !slot_mapping || !kv_cache) return SMLA_ERR_NULL;
  if (!aligned(latent, 16) || !aligned(rope, 16) || !aligned(kv_cache, 16) ||
      !aligned(slot_mapping, 8))
    return SMLA_ERR_ALIGN;
  if (n > (int64_t(1) << 36)) return SMLA_ERR_SHAPE;
  int sms = 0;
  smla_status st = current_device(&sms);
  if (st != SMLA_OK) return st;
  if (smla::launch_pack(SMLA_KV_FP8_TENSOR, SMLA_SCALE_FP32, kv_scale, latent, rope, slot_mapping, n,
                        kv_cache, num_slots, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SMLA_ERR_CUDA;
  return SMLA_OK;
}

smla_status smla_store_kv_normed(const smla_store_desc* d, const void* latent, const void* rope,
                                 const void* norm_weight, const int64_t* positions, const float* cos_sin,
                                 const int64_t* slot_mapping, void* kv_cache, int32_t* error_word,
                                 void* stream) {
  if (!d) return SMLA_ERR_NULL;
  if (d->kv_format != SMLA_KV_BF16 && d->kv_format != SMLA_KV_FP8_DS && d->kv_format != SMLA_KV_FP8_TENSOR)
    return SMLA_ERR_UNSUPPORTED;
  if (d->kv_format == SMLA_KV_FP8_DS && d->scale_mode != SMLA_SCALE_POW2 && d->scale_mode != SMLA_SCALE_FP32)
    return SMLA_ERR_UNSUPPORTED;
  if (d->kv_format == SMLA_KV_FP8_TENSOR && !(isfinite(d->kv_scale) && d->kv_scale > 0.f)) return SMLA_ERR_SHAPE;
  if (!(isfinite(d->rms_eps) && d->rms_eps >= 0.f)) return SMLA_ERR_SHAPE;
  if (d->n < 0 || d->num_slots < 0 || d->max_position < 1 || d->n > (int64_t(1) << 36)) return SMLA_ERR_SHAPE;
  for (int i = 0; i < 2; ++i)
    if (d->reserved[i] != 0) return SMLA_ERR_SHAPE;
  if (d->n == 0) return SMLA_OK;
  if (!latent || !rope || !norm_weight || !positions || !cos_sin || !slot_mapping || !kv_cache) return SMLA_ERR_NULL;
  if (!aligned(latent, 16) || !aligned(rope, 16) || !aligned(norm_weight, 16) || !aligned(kv_cache, 16) ||
      !aligned(positions, 8) || !aligned(slot_mapping, 8) || !aligned(cos_sin, 16) ||
      (error_word && !aligned(error_word, 4)))
    return SMLA_ERR_ALIGN;
  int sms = 0;
  smla_status st = current_device(&sms);
  if (st != SMLA_OK) return st;
  if (smla::launch_store_normed(d->kv_format, d->scale_mode, d->kv_format == SMLA_KV_FP8_TENSOR ? d->kv_scale : 1.f,
                                latent, rope, norm_weight, d->rms_eps, positions, cos_sin, d->max_position,
                                slot_mapping, d->n, kv_cache, d->num_slots, error_word,
                                static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SMLA_ERR_CUDA;
  return SMLA_OK;
}

smla_status smla_gather_dequant(const smla_desc* d, const void* kv_cache,
                                const int32_t* page_table, const int32_t* topk,
                                const int32_t* req_id_per_token, float* rows,
                                int32_t* error_word, void* stream) {
  smla_status st = check_desc(d);
  if (st != SMLA_OK) return st;
  if (!kv_cache || !page_table || !topk || !rows) return SMLA_ERR_NULL;
  if (!aligned(kv_cache, 16) || !aligned(rows, 16) || !aligned(topk, 4) ||
      !aligned(page_table, 4) || (error_word && !aligned(error_word, 4)))
    return SMLA_ERR_ALIGN;
  if (!req_id_per_token && (d->num_tokens - 1) / d->next_n >= d->num_requests)
    return SMLA_ERR_SHAPE;
  int sms = 0;
  st = current_device(&sms);
  if (st != SMLA_OK) return st;
  smla::DecodeArgs a = make_args(d, nullptr, kv_cache, page_table, topk, req_id_per_token, nullptr);
  a.err = error_word;
  if (smla::launch_gather_dequant(a, rows, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SMLA_ERR_CUDA;
  return SMLA_OK;
}

smla_status smla_indexer_logits(const smla_indexer_desc* d, const void* q, const float* weights,
                                const void* k_cache, const int32_t* page_table, const int32_t* context_lens,
                                float* logits, int32_t* error_word, void* stream) {
  smla_status st = check_indexer_desc(d);
  if (st != SMLA_OK) return st;
  if (!q || !weights || !k_cache || !page_table || !context_lens || !logits || !error_word) return SMLA_ERR_NULL;
  if (!aligned(q, 16) || !aligned(weights, 16) || !aligned(k_cache, 16) || !aligned(page_table, 4) ||
      !aligned(context_lens, 4) || !aligned(logits, 4) || !aligned(error_word, 4))
    return SMLA_ERR_ALIGN;
  int sms = 0;
  st = current_device(&sms);
  if (st != SMLA_OK) return st;
  smla::IndexerArgs a = make_indexer_args(d, context_lens);
  a.q = static_cast<const uint8_t*>(q);
  a.weights = weights;
  a.cache = static_cast<const uint8_t*>(k_cache);
  a.page_table = page_table;
  a.logits = logits;
  a.err = error_word;
  if (smla::launch_indexer_logits(a, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess) return SMLA_ERR_CUDA;
  return SMLA_OK;
}

smla_status smla_indexer_topk(const smla_indexer_desc* d, const float* logits, const int32_t* context_lens,
                              int32_t* topk, void* stream) {
  smla_status st = check_indexer_desc(d);
  if (st != SMLA_OK) return st;
  if (!logits || !context_lens || !topk) return SMLA_ERR_NULL;
  if (!aligned(logits, 4) || !aligned(context_lens, 4) || !aligned(topk, 4)) return SMLA_ERR_ALIGN;
  int sms = 0;
  st = current_device(&sms);
  if (st != SMLA_OK) return st;
  smla::IndexerArgs a = make_indexer_args(d, context_lens);
  a.logits = const_cast<float*>(logits);
  a.topk = topk;
  // one CTA a token and an SM: with more tokens than SMs, the longest rows go first
  a.longest_first = d->num_tokens > sms && d->num_tokens <= smla::kTkRankMax ? 1 : 0;
  if (smla::launch_indexer_topk(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return SMLA_ERR_CUDA;
  return SMLA_OK;
}

smla_status smla_selftest_wait_timeout(int32_t* error_word, uint32_t limit_us, void* stream) {
  if (!error_word) return SMLA_ERR_NULL;
  if (!aligned(error_word, 4)) return SMLA_ERR_ALIGN;
  if (limit_us < 1 || limit_us > 100000) return SMLA_ERR_SHAPE;
  int sms = 0;
  smla_status st = current_device(&sms);
  if (st != SMLA_OK) return st;
  if (smla::launch_selftest_wait(error_word, uint64_t(limit_us) * 1000u, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return SMLA_ERR_CUDA;
  return SMLA_OK;
}

smla_status smla_read_error(const smla_desc* d, void* workspace, size_t workspace_bytes,
                            int32_t* error_word, void* stream) {
  (void)d;
  if (!workspace || !error_word) return SMLA_ERR_NULL;
  if (workspace_bytes < sizeof(int32_t)) return SMLA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(workspace, 0, sizeof(v), s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return SMLA_ERR_CUDA;
  *error_word = v;
  return error_status(v);
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Workspace-free entry point: the scratch lives in this file-scope device array.
// ---------------------------------------------------------------------------------------
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[SMLA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch, looked up once per device with that device current
// (concurrent first calls store the same address).
std::atomic<void*> g_noalloc_addr[kMaxDevices];

smla_status noalloc_scratch(void** ptr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return SMLA_ERR_DEVICE;
  }
  void* p = g_noalloc_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return SMLA_ERR_CUDA;
    }
    g_noalloc_addr[dev].store(p, std::memory_order_release);
  }
  *ptr = p;
  return SMLA_OK;
}

}  // namespace

extern "C" smla_status smla_decode_noalloc(const smla_desc* d, const void* q, const void* kv_cache,
                                           const int32_t* page_table, const int32_t* topk,
                                           const int32_t* req_id_per_token, const float* sink,
                                           void* out, float* lse, void* stream) {
  smla_status st = check_desc(d);
  if (st != SMLA_OK) return st;
  if (!q || !kv_cache || !page_table || !topk || !out) return SMLA_ERR_NULL;
  int sms = 0;
  st = current_device(&sms);
  if (st != SMLA_OK) return st;
  if (make_plan(d, sms).bytes > SMLA_NOALLOC_SCRATCH_BYTES) return SMLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != SMLA_OK) return st;
  // The error word (the array's first 4 bytes, zero when the library loads) accumulates
  // the device error bits of every call until smla_noalloc_read_error reads and clears it.
  // smla_decode checks every argument before it launches anything.
  return smla_decode(d, q, kv_cache, page_table, topk, req_id_per_token, sink, out, lse, scratch,
                     SMLA_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" smla_status smla_noalloc_read_error(int32_t* error_word, void* stream) {
  if (!error_word) return SMLA_ERR_NULL;
  int sms = 0;
  smla_status st = current_device(&sms);
  if (st != SMLA_OK) return st;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != SMLA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(scratch, 0, sizeof(v), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return SMLA_ERR_CUDA;
  *error_word = v;
  return error_status(v);
}
