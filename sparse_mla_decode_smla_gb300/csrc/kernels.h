// Internal launchers of the sparse MLA decode library (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/smla.h"

namespace smla {

constexpr int kMaxSplits = 64;
constexpr int kTile = 64;       // split lengths are multiples of this
constexpr int kMaxSplitLen = 2048;  // index entries of one split staged in shared memory

struct DecodeArgs {
  const void* q;
  const uint8_t* kv;
  const int32_t* page_table;
  const int32_t* topk;
  const int32_t* req_id;
  const float* sink;
  void* out;
  float* lse;
  float* o_part;    // [T, S, H, 512] fp32, or f16 when part_f16 (S > 1)
  float* lse_part;  // [T, S, H] fp32 (S > 1)
  int32_t* err;     // device error word
  int32_t T, H, K, B, next_n, stride, log2_page, kv_format;
  int64_t num_pages;
  int32_t num_splits, split_len;
  float c2;  // sm_scale * log2(e)
  float kv_scale;  // per-tensor scale (SMLA_KV_FP8_TENSOR)
  int32_t part_f16;  // the decode kernel writes o_part as f16 (values within f16's range)
  // The split CTAs of a (token, head group) form one thread-block cluster (cluster size =
  // num_splits) and merge their partials through distributed shared memory; no o_part.
  int32_t cluster_merge;
  int32_t q_fp8;   // q holds E4M3 codes (SMLA_Q_FP8_E4M3), times q_scale
  float q_scale;
  // head-group kernels: this launch serves the (token, head group) items [item0, item0 +
  // nitems), nitems = 0 meaning all T x ceil(H / 64) of them
  int32_t item0, nitems;
  // launched with programmatic stream serialisation: its CTAs may start while the previous
  // kernel on the stream drains (nothing here reads what that kernel writes)
  int32_t overlap_prev;
};
// Largest cluster the in-kernel split merge uses (the portable cluster size).
constexpr int kMaxClusterMerge = 8;

cudaError_t launch_decode_mma(const DecodeArgs& a, int num_sms, cudaStream_t s);
// One CTA per (token, split, group of 64 heads); FP8 caches.
cudaError_t launch_decode_hg(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_merge(const DecodeArgs& a, cudaStream_t s);
// The FP8-operand head-group kernel: E4M3 q against the per-tensor FP8 cache, 64+ heads.
cudaError_t launch_decode_hg_f8(const DecodeArgs& a, cudaStream_t s);

// Row gathers (TMA tile::gather4) address the cache by 32-bit row coordinates, and one past
// the last slot marks a masked row: caches must hold fewer slots than this.
constexpr int64_t kMaxGatherSlots = (int64_t(1) << 31) - 1;
int kv_row_bytes(int32_t kv_format);
// The driver's cuTensorMapEncodeTiled, looked up once (no link against the driver library).
cudaError_t tensor_map_encoder(PFN_cuTensorMapEncodeTiled_v12000* out);
// Tensor map of the cache as [slots, row bytes / 8] 8-byte words with one-row boxes.
cudaError_t kv_gather_map(const DecodeArgs& a, CUtensorMap* out);
// Tensor map of q as [T H rows, 576] bf16 with [64 rows x 64 dims] boxes, 128-byte swizzle.
cudaError_t q_tile_map(const DecodeArgs& a, CUtensorMap* out);
// Tensor maps of E4M3 q as [T H rows, 576] bytes: [64 rows x 128 B] boxes with 128-byte
// swizzle (latent) and [64 rows x 32 B] boxes with 32-byte swizzle (RoPE).
cudaError_t q_e4m3_maps(const DecodeArgs& a, CUtensorMap* map128, CUtensorMap* map32);

// The tensor-core head-group kernel serves the FP8 caches with at least this many heads.
constexpr int kHgMinHeads = 64;
cudaError_t launch_pack(int32_t kv_format, int32_t scale_mode, float kv_scale, const void* latent,
                        const void* rope, const int64_t* slot_mapping, int64_t n, void* kv,
                        int64_t num_slots, cudaStream_t s);
cudaError_t launch_gather_dequant(const DecodeArgs& a, float* rows, cudaStream_t s);
// The quantise-on-write store fused with the latent's RMSNorm and the RoPE rotation.
cudaError_t launch_store_normed(int32_t kv_format, int32_t scale_mode, float kv_scale, const void* latent,
                                const void* rope, const void* weight, float eps, const int64_t* positions,
                                const float* cos_sin, int64_t max_position, const int64_t* slot_mapping,
                                int64_t n, void* kv, int64_t num_slots, int32_t* err, cudaStream_t s);

cudaError_t launch_selftest_wait(int32_t* err, uint64_t limit_ns, cudaStream_t s);

}  // namespace smla
