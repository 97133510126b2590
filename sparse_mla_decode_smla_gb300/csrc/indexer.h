// Internal launchers of the sparse-attention indexer (not part of the C ABI).
#pragma once

#include "kernels.h"

namespace smla {

// Requests an indexer call may hold (the logits kernel keeps their schedule prefix in
// shared memory).
constexpr int kIxMaxRequests = 8192;

struct IndexerArgs {
  const uint8_t* q;         // [T, H, 128] E4M3 codes
  const float* weights;     // [T, H] fp32
  const uint8_t* cache;     // [num_pages, P * 132]: P x 128 E4M3 codes, then P fp32 scales
  const int32_t* page_table;
  const int32_t* ctx;       // [B] context lengths
  float* logits;            // [T, logits_stride] fp32
  int32_t* topk;            // [T, K] int32
  int32_t* err;             // device error word
  int32_t T, H, B, next_n, stride, log2_page, logits_stride, K;
  int64_t num_pages;
  // top-k: CTA b takes the token with the b-th longest visible row (ties by index) instead of
  // token b; worth it when the tokens take more than one wave of CTAs
  int32_t longest_first;
};
cudaError_t launch_indexer_logits(const IndexerArgs& a, int num_sms, cudaStream_t s);
cudaError_t launch_indexer_topk(const IndexerArgs& a, cudaStream_t s);
// Batches up to this many tokens may take the top-k's longest-row-first order (each CTA ranks
// every row's length, so the cost grows with the square of the batch).
constexpr int kTkRankMax = 512;

}  // namespace smla
