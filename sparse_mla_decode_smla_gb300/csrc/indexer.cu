// Sparse-attention indexer on sm_103a: FP8 paged MQA logits and their top-k, the step that
// chooses each query token's top-k slots for the sparse decode (the vLLM PR #52164 page,
// "功能与动机" and "实现拆解 1-5": fp8_paged_mqa_logits, scheduled from the requests' context
// lengths, with the next_n query rows of a request handled natively; the SGLang PR #24692
// page, "实现拆解 5": fp8_paged_mqa_logits for the indexer).
//
// What it computes, per query token t (row i of request r, next_n rows per request) and visible
// slot s < ctx_r - next_n + 1 + i:
//     logit[t, s] = sum_h w[t, h] * max(0, scale_s * <q[t, h], k_s>)
// with q and k_s E4M3 (128 dims) and one fp32 scale per key; then the indices of the K largest
// logits of each token.
//
// indexer_logits_kernel: persistent, one CTA per SM. Every CTA derives the same schedule from the
// context lengths (a block-wide scan of the requests' 1024-slot chunk counts) and takes a
// contiguous, balanced range of (request, chunk) items, so its q and weights change rarely.
//  * producer (warp 0, one thread): per 128-slot tile, one 3-D TMA load per key page (P x 128
//    codes, 128-byte swizzle: the K-major operand layout as it lands) and one bulk copy of the
//    page's P scales, into a 4-stage ring; q of the item's request (next_n x H_I rows of 128
//    codes) and its weights when the request changes.
//  * MMA (warp 1, one thread): D[128 slots, N] = K_tile x q^T with N = H_I x next_n, four
//    tcgen05.mma kind::f8f6f4 (K = 32 each), into one of two TMEM accumulators. The next_n query
//    rows of a request share every key tile: it is read once, not next_n times.
//  * epilogue (warps 2-9): thread = slot; each warp pair of a TMEM lane quarter splits the
//    request's query rows; ReLU and the weighted sum over heads in fp32 in four independent
//    chains, the key's scale applied once (max(0, s d) = |s| max(0, sgn(s) d)); coalesced
//    stores of the visible logits.
// Every wait is bounded; a wait that gives up sets SMLA_DEVERR_TIMEOUT.
//
// indexer_topk_kernel: one CTA of 1024 threads per token, radix select over the token's visible
// logits (keys made order-preserving as unsigned 32-bit integers, -0 equal to +0) to the K-th
// largest value. The row is read 16 bytes at a time, but for up to three keys at each end:
//  * pass 0 histograms bits [31:20] of every key and finds the bin holding the K-th largest by
//    a scan across the whole block;
//  * pass 1 has each warp read its contiguous segment: it counts the keys above that bin and
//    gathers the bin's keys, with their indices, into shared memory;
//  * bits [19:10] and [9:0] are then selected among the gathered keys, whose counts above and
//    equal to the threshold join their segments' counts (when the bin holds more keys than the
//    buffer, these two passes and the counts read global memory instead);
//  * the counts are scanned across warps, and each warp writes every index above the threshold
//    and, among indices equal to it, the lowest ones up to K: the top-k set in ascending index
//    order (when no tie is cut, simply every key at or above the threshold).
// Three passes over a token's logits, not five.
//
// The producer warp prefetches the next item's page-table entries into shared memory by
// cp.async and issues each tile's copies with one lane per page, and the epilogue hands a
// stage back as soon as it has read the stage's key scales.
#include <math_constants.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "indexer.h"
#include "tcgen05.cuh"

namespace smla {
namespace {

// Tensor map of the index-key cache as [num_pages][P][128] bytes with [1 x P x 128] boxes,
// 128-byte swizzle; of q as [T H rows, 128] bytes with [H next_n x 128] boxes, 128-byte swizzle.
cudaError_t index_key_map(const IndexerArgs& a, CUtensorMap* out) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (tensor_map_encoder(&encode) != cudaSuccess) return cudaErrorNotSupported;
  const cuuint64_t P = cuuint64_t(1) << a.log2_page;
  const cuuint64_t dims[3] = {128, P, cuuint64_t(a.num_pages)};
  const cuuint64_t strides[2] = {128, P * 132};
  const cuuint32_t box[3] = {128, cuuint32_t(P), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(a.cache), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t index_q_map(const IndexerArgs& a, CUtensorMap* out) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (tensor_map_encoder(&encode) != cudaSuccess) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {128, cuuint64_t(a.T) * a.H};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, cuuint32_t(a.H * a.next_n)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.q), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}


constexpr int kIxDim = 128;              // index dims (bytes of E4M3 per key or q row)
constexpr int kIxTile = 128;             // slots per tile (the MMA's M)
constexpr int kIxChunk = 1024;           // slots per scheduled item
constexpr int kIxStages = 6;
constexpr int kIxEpiWarps = 8;
constexpr int kIxFirstEpi = 2;
constexpr int kIxThreads = 32 * (kIxFirstEpi + kIxEpiWarps);
constexpr int kIxMaxN = 256;             // H_I x next_n

constexpr size_t kIxOffQ = 0;                                   // [N rows x 128 B], 128-byte swizzle
constexpr size_t kIxOffK = kIxOffQ + size_t(kIxMaxN) * kIxDim;  // [stage][128 x 128 B]
constexpr size_t kIxStageK = size_t(kIxTile) * kIxDim;
constexpr size_t kIxOffSc = kIxOffK + kIxStages * kIxStageK;    // [stage][128] fp32 scales
constexpr size_t kIxOffW = kIxOffSc + kIxStages * kIxTile * 4;  // [N] fp32 weights
constexpr size_t kIxOffPre = kIxOffW + kIxMaxN * 4;             // [kIxMaxReq + 1] item prefix
constexpr size_t kIxOffPg = kIxOffPre + size_t(kIxMaxRequests + 1) * 4;  // [2][64] page entries
constexpr size_t kIxOffTm = kIxOffPg + 2 * 64 * 4;
constexpr size_t kIxOffBars = (kIxOffTm + 16 + 7) / 8 * 8;
enum { X_FULL = 0, X_EMPTY = X_FULL + kIxStages, X_DFULL = X_EMPTY + kIxStages, X_DEMPTY = X_DFULL + 2,
       X_QFULL = X_DEMPTY + 2, X_QFREE, X_DRAIN, X_COUNT };
constexpr size_t kIxSmem = kIxOffBars + X_COUNT * 8 + 1024;
static_assert(kIxOffK % 1024 == 0 && kIxStageK % 1024 == 0 && kIxOffSc % 16 == 0 && kIxOffW % 16 == 0,
              "swizzle atoms, bulk copies, weight vectors");
static_assert(kIxSmem <= 232448, "shared memory budget");

// Four fp32 from shared memory (16-byte aligned).
__device__ __forceinline__ float4 lds_f32x4(uint32_t addr) {
  const uint4 v = lds128(addr);
  return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
}

// sum_h w[h] * max(0, sgn * d[h]) over H heads (d: the row's TMEM words), in four independent
// chains. H is a compile-time constant so the weight loads (shared memory, the same address in
// every lane) are all issued before the first is used.
template <int H, bool POS>
__device__ __forceinline__ float head_sum(const uint32_t (&d)[64], uint32_t w_row, float sgn) {
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int e = 0; e < H; e += 4) {
    const float4 w4 = lds_f32x4(w_row + uint32_t(e) * 4u);
    const float x0 = __uint_as_float(d[e]), x1 = __uint_as_float(d[e + 1]);
    const float x2 = __uint_as_float(d[e + 2]), x3 = __uint_as_float(d[e + 3]);
    a0 = fmaf(w4.x, fmaxf(0.f, POS ? x0 : sgn * x0), a0);
    a1 = fmaf(w4.y, fmaxf(0.f, POS ? x1 : sgn * x1), a1);
    a2 = fmaf(w4.z, fmaxf(0.f, POS ? x2 : sgn * x2), a2);
    a3 = fmaf(w4.w, fmaxf(0.f, POS ? x3 : sgn * x3), a3);
  }
  return (a0 + a1) + (a2 + a3);
}

// TMA load of box (x, y, z) of a 3-D tensor map into dst, counting the box bytes on bar.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];\n" ::"r"(dst),
      "l"(tmap), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

struct Item {
  int r, c;  // request, chunk
};

__global__ void __launch_bounds__(kIxThreads, 1)
    indexer_logits_kernel(const IndexerArgs p, const __grid_constant__ CUtensorMap kmap,
                          const __grid_constant__ CUtensorMap qmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  auto bar = [&](int k) -> uint32_t { return sb + uint32_t(kIxOffBars) + 8u * k; };
  int32_t* pre = reinterpret_cast<int32_t*>(sm + kIxOffPre);  // pre[r] = items of requests < r
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {  // the TMA descriptors, fetched before their first use
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&qmap);
  }
  const int N = p.H * p.next_n;
  const int P = 1 << p.log2_page;

  // a request's context as served: at most its page table's capacity and the logits row
  auto ctx_of = [&](int r) -> int {
    return min(__ldg(p.ctx + r), min(p.stride << p.log2_page, p.logits_stride));
  };
  // ---- schedule: a block-wide scan of the requests' chunk counts (their largest visible
  // length is ctx_r: the last query row sees the whole context)
  auto nchunks = [&](int r) -> int {
    const int ctx = ctx_of(r);
    return ctx > 0 ? (ctx + kIxChunk - 1) / kIxChunk : 0;
  };
  {
    int* wsum = reinterpret_cast<int*>(sm + kIxOffW);  // scratch before the weights are loaded
    int carry = 0;
    for (int base = 0; base < p.B; base += kIxThreads) {
      const int r = base + tid;
      const int v = r < p.B ? nchunks(r) : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wsum[warp] = x;
      __syncthreads();
      int before = carry;
      for (int w2 = 0; w2 < warp; ++w2) before += wsum[w2];
      if (r < p.B) pre[r] = before + x - v;
      int tot = 0;
      for (int w2 = 0; w2 < kIxThreads / 32; ++w2) tot += wsum[w2];
      __syncthreads();
      carry += tot;
    }
    if (tid == 0) pre[p.B] = carry;
    if (blockIdx.x == 0)  // a context longer than the page table or the logits row is cut and flagged
      for (int r = tid; r < p.B; r += kIxThreads)
        if (__ldg(p.ctx + r) > ctx_of(r)) atomicOr(p.err, SMLA_DEVERR_INDEX);
    if (tid == 0) {
      mbar_init(bar(X_QFULL), 1);
      mbar_init(bar(X_QFREE), 1 + kIxEpiWarps);
      mbar_init(bar(X_DRAIN), 1);
      for (int s = 0; s < kIxStages; ++s) {
        mbar_init(bar(X_FULL + s), 1);
        mbar_init(bar(X_EMPTY + s), 1 + kIxEpiWarps);  // the MMAs' commit + the epilogue (scales)
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(bar(X_DFULL + b), 1);
        mbar_init(bar(X_DEMPTY + b), kIxEpiWarps);
      }
      tc::fence_mbarrier_init_cluster();
    }
    if (warp == 1) tc::alloc(sb + uint32_t(kIxOffTm), 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
  }
  const uint32_t tm = *reinterpret_cast<volatile uint32_t*>(sm + kIxOffTm);
  const int total = pre[p.B];
  const int G = gridDim.x;
  const int it0 = int((int64_t(total) * blockIdx.x) / G), it1 = int((int64_t(total) * (blockIdx.x + 1)) / G);
  // the item at flat index `it`: the request whose prefix range holds it
  auto item_at = [&](int it, int hint) -> Item {
    int r = hint;
    while (r + 1 < p.B && pre[r + 1] <= it) ++r;
    return Item{r, it - pre[r]};
  };
  int r_first = 0;
  {
    int lo = 0, hi = p.B - 1;  // last r with pre[r] <= it0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= it0) lo = mid; else hi = mid - 1;
    }
    r_first = lo;
  }
  auto tiles_of = [&](const Item& x) -> int {
    const int ctx = ctx_of(x.r);
    const int s0 = x.c * kIxChunk;
    return (min(ctx, s0 + kIxChunk) - s0 + kIxTile - 1) / kIxTile;
  };

  bool ok = true;
  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    // The warp prefetches the next item's page-table entries (1024 / P pages, two per lane) by
    // 4-byte cp.async into a two-item shared ring while lane 0 issues the current item's
    // copies, so no tile waits on a dependent page-table load.
    const int ppi = kIxChunk >> p.log2_page;  // pages per item
    const int npg = kIxTile >> p.log2_page;   // pages per tile (P <= 128)
    int32_t* spg = reinterpret_cast<int32_t*>(sm + kIxOffPg);
    auto prefetch = [&](const Item& x, int buf) {
      const int32_t* pt_row = p.page_table + int64_t(x.r) * p.stride;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int li = lane + 32 * k, lp = x.c * ppi + li;
        if (li < ppi && lp < p.stride)
          cp_async4(smem_u32(spg + buf * 64 + li), pt_row + lp);
        else
          spg[buf * 64 + li] = -1;
      }
      cp_async_commit();
    };
    if (it0 < it1) prefetch(item_at(it0, r_first), 0);
    int u = 0, qloads = 0, rq = -1, r = r_first;
    for (int it = it0; it < it1 && ok; ++it) {
      const Item x = item_at(it, r);
      r = x.r;
      const int buf = (it - it0) & 1;
      if (it + 1 < it1)
        prefetch(item_at(it + 1, r), buf ^ 1);
      else
        cp_async_commit();  // an empty group keeps the count of groups in flight at one
      cp_async_wait<1>();   // this item's entries have landed
      __syncwarp();
      if (lane == 0 && x.r != rq) {  // q and weights of the request, once the previous ones are unused
        if (qloads > 0 && !mbar_wait(bar(X_QFREE), (qloads - 1) & 1)) ok = false;
        if (ok) {
          mbar_arrive_expect_tx(bar(X_QFULL), uint32_t(N) * kIxDim + uint32_t(N) * 4u);
          tma_load_2d(sb + uint32_t(kIxOffQ), &qmap, 0, x.r * N, bar(X_QFULL));
          bulk_g2s(sb + uint32_t(kIxOffW), p.weights + int64_t(x.r) * N, uint32_t(N) * 4u, bar(X_QFULL));
          ++qloads;
          rq = x.r;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      qloads = __shfl_sync(0xffffffffu, qloads, 0);
      rq = __shfl_sync(0xffffffffu, rq, 0);
      // The whole warp issues a tile's copies: lane g checks page g of the tile and, when it is
      // valid, issues its 3-D load and its scales' copy, all in one instruction each.
      const int ctx = ctx_of(x.r);
      const int nt = tiles_of(x);
      for (int j = 0; j < nt && ok; ++j, ++u) {
        const int st = u % kIxStages;
        if (!__all_sync(0xffffffffu, mbar_wait(bar(X_EMPTY + st), ((u / kIxStages) & 1) ^ 1))) {
          ok = false;
          break;
        }
        // pages outside the request's table or the pool are not fetched: their rows keep
        // stale bytes, which only feed logits beyond the visible range or flagged ones
        const int li = j * npg + lane;
        const int32_t pg = lane < npg ? spg[buf * 64 + li] : -1;
        const bool valid = lane < npg && pg >= 0 && pg < p.num_pages;
        if (lane < npg && !valid && ((x.c * ppi + li) << p.log2_page) < ctx)  // a page the visible context needs
          atomicOr(p.err, SMLA_DEVERR_PAGE);
        const uint32_t mask = __ballot_sync(0xffffffffu, valid);
        if (lane == 0) mbar_arrive_expect_tx(bar(X_FULL + st), uint32_t(__popc(mask)) * uint32_t(P) * (kIxDim + 4));
        __syncwarp();
        if (valid) {
          tma_load_3d(sb + uint32_t(kIxOffK + st * kIxStageK) + uint32_t(lane * P * kIxDim), &kmap, 0, 0, pg,
                      bar(X_FULL + st));
          bulk_g2s(sb + uint32_t(kIxOffSc) + uint32_t(st * kIxTile * 4 + lane * P * 4),
                   p.cache + int64_t(pg) * P * (kIxDim + 4) + int64_t(P) * kIxDim, uint32_t(P) * 4u,
                   bar(X_FULL + st));
        }
      }
    }
    cp_async_wait<0>();
    // no copy may land after the CTA has left
    if (lane == 0) {
      for (int v = max(0, u - kIxStages); v < u; ++v)
        if (!mbar_wait(bar(X_FULL + v % kIxStages), (v / kIxStages) & 1)) break;
      if (qloads > 0) mbar_wait(bar(X_QFULL), (qloads - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_e4m3_f32(128, N);
      int u = 0, qloads = 0, rq = -1, r = r_first;
      for (int it = it0; it < it1 && ok; ++it) {
        const Item x = item_at(it, r);
        r = x.r;
        if (x.r != rq) {
          if (!mbar_wait(bar(X_QFULL), qloads & 1)) { ok = false; break; }
          ++qloads;
          rq = x.r;
        }
        const int nt = tiles_of(x);
        for (int j = 0; j < nt; ++j, ++u) {
          const int st = u % kIxStages, b = u & 1;
          if (!mbar_wait(bar(X_FULL + st), (u / kIxStages) & 1)) { ok = false; break; }
          if (u >= 2 && !mbar_wait(bar(X_DEMPTY + b), ((u >> 1) - 1) & 1)) { ok = false; break; }
          tc::fence_after();
          const uint32_t ka = sb + uint32_t(kIxOffK + st * kIxStageK);
#pragma unroll
          for (int k = 0; k < kIxDim / 32; ++k)
            tc::mma_ss_f8(tm + uint32_t(b * N), tc::sdesc_sw128(ka + 32 * k, 16, 1024),
                   tc::sdesc_sw128(sb + uint32_t(kIxOffQ) + 32 * k, 16, 1024), idesc, k > 0);
          tc::commit(bar(X_EMPTY + st));
          tc::commit(bar(X_DFULL + b));
        }
        // the last item of this request: q and weights may be replaced once its MMAs are done
        const bool last_of_req = it + 1 >= it1 || item_at(it + 1, r).r != x.r;
        if (last_of_req && ok) tc::commit(bar(X_QFREE));
      }
      // every MMA issued has completed before the tensor memory is released
      tc::commit(bar(X_DRAIN));
      if (!mbar_wait(bar(X_DRAIN), 0)) ok = false;
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    const int ew = warp - kIxFirstEpi;
    const int quarter = warp & 3, half = ew >> 2;
    const int row = 32 * quarter + lane;  // slot within the tile
    const uint32_t lrow = tm + (uint32_t(32 * quarter) << 16);
    // the two warps of a lane quarter split the request's query rows
    const int nn = p.next_n, i_lo = half ? (nn + 1) / 2 : 0, i_hi = half ? nn : (nn + 1) / 2;
    const uint32_t wsm = sb + uint32_t(kIxOffW);
    int u = 0, r = r_first, rq = -1, qloads = 0;
    for (int it = it0; it < it1 && ok; ++it) {
      const Item x = item_at(it, r);
      r = x.r;
      if (x.r != rq) {
        if (!mbar_wait(bar(X_QFULL), qloads & 1)) { ok = false; break; }
        ++qloads;
        rq = x.r;
      }
      const int ctx = ctx_of(x.r);
      const int nt = tiles_of(x);
      for (int j = 0; j < nt; ++j, ++u) {
        const int st = u % kIxStages, b = u & 1;
        if (!mbar_wait(bar(X_DFULL + b), (u >> 1) & 1)) { ok = false; break; }
        tc::fence_after();
        const int s = x.c * kIxChunk + j * kIxTile + row;
        const float sc = lds_f32(sb + uint32_t(kIxOffSc) + uint32_t(st * kIxTile + row) * 4);
        // the scale is in a register: the stage goes back to the producer (its codes were
        // consumed by the MMAs, whose commit is the stage's other arrival)
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(X_EMPTY + st));
        // max(0, sc * d) = |sc| * max(0, sgn * d), sgn the sign of sc: the scale leaves the sum,
        // and with every lane's scale non-negative (quantisation scales) the sign does too
        const bool pos = __all_sync(0xffffffffu, !(sc < 0.f));
        const float sgn = sc < 0.f ? -1.f : 1.f, asc = fabsf(sc);
        for (int i = i_lo; i < i_hi; ++i) {
          uint32_t v[64];  // the row's 64 (or 32) head scores, both loads before one wait
          tc::ld32(lrow + uint32_t(b * N + i * p.H), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          if (p.H > 32) tc::ld32(lrow + uint32_t(b * N + i * p.H + 32), *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          tc::wait_ld();
          const uint32_t w_row = wsm + uint32_t(i * p.H) * 4u;
          const float hs = p.H == 64 ? (pos ? head_sum<64, true>(v, w_row, sgn) : head_sum<64, false>(v, w_row, sgn))
                                     : (pos ? head_sum<32, true>(v, w_row, sgn) : head_sum<32, false>(v, w_row, sgn));
          const int vis = ctx - nn + 1 + i;
          const int t = x.r * nn + i;
          if (s < vis) p.logits[int64_t(t) * p.logits_stride + s] = asc * hs;
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(X_DEMPTY + b));
      }
      const bool last_of_req = it + 1 >= it1 || item_at(it + 1, r).r != x.r;
      if (last_of_req && ok) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(X_QFREE));
      }
    }
  }
  if (!ok && lane == 0) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after();
    tc::dealloc(tm, 512);
  }
}

// ------------------------------------------------------------------------------ top-k

constexpr int kTkThreads = 1024;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkUnroll = 8;  // independent 4-byte loads in flight per thread (global fallback passes)
constexpr int kTkVec = 4;     // independent 16-byte loads in flight per thread
constexpr int kTkCand = 12288;  // keys of the threshold bin held in shared memory (with their indices)
constexpr size_t kTkSmem = size_t(kTkCand) * 8;  // dynamic shared memory of the top-k kernel

// Order-preserving unsigned key of a float: the sign bit set for positive values, every bit
// flipped for negative ones. -0 is taken as +0 first (x + 0 rounds -0 to +0 and changes no other
// value), so equal values have equal keys.
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(__fadd_rn(f, 0.f));
  return u ^ (uint32_t(int32_t(u) >> 31) | 0x80000000u);
}

__global__ void __launch_bounds__(kTkThreads) indexer_topk_kernel(const IndexerArgs p) {
  __shared__ uint32_t hist[4096];
  __shared__ uint32_t s_need, s_sel, s_ncand;
  __shared__ uint32_t wgt[kTkWarps], weq[kTkWarps], wsum[kTkWarps];
  extern __shared__ uint32_t tk_dyn[];
  uint32_t* cand_key = tk_dyn;                                     // [kTkCand]
  int32_t* cand_idx = reinterpret_cast<int32_t*>(tk_dyn + kTkCand);  // [kTkCand]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cap = min(p.stride << p.log2_page, p.logits_stride);
  auto visible = [&](int tt) {
    const int rr = tt / p.next_n;
    return max(0, min(__ldg(p.ctx + rr), cap) - p.next_n + 1 + (tt - rr * p.next_n));
  };
  // Longest rows first (when the tokens take more than one wave of CTAs): CTA b takes the
  // token whose visible length ranks b-th (ties by index), so the rows that take longest start
  // in the first wave and the short ones fill in behind them. Each CTA ranks the lengths in the
  // shared memory the candidate buffer uses later.
  int t = blockIdx.x;
  if (p.longest_first && p.T <= kTkRankMax) {
    int* len = reinterpret_cast<int*>(tk_dyn);
    for (int k = tid; k < p.T; k += kTkThreads) len[k] = visible(k);
    __syncthreads();
    for (int k = tid; k < p.T; k += kTkThreads) {
      const int lk = len[k];
      int rank = 0;
      for (int j = 0; j < p.T; ++j) {
        const int lj = len[j];
        rank += (lj > lk || (lj == lk && j < k)) ? 1 : 0;
      }
      if (rank == int(blockIdx.x)) s_sel = uint32_t(k);
    }
    __syncthreads();
    t = int(s_sel);
    __syncthreads();  // s_sel is reused below
  }
  const int vis = visible(t);
  int32_t* out = p.topk + int64_t(t) * p.K;
  const float* lg = p.logits + int64_t(t) * p.logits_stride;
  if (vis <= p.K) {  // every visible slot, then padding
    for (int j = tid; j < p.K; j += kTkThreads) out[j] = j < vis ? j : -1;
    return;
  }
  // The visible row in three parts: `head` keys before the first 16-byte boundary, `nv` groups
  // of four read as one 16-byte load each, and the tail after them. Warp w's segment is the
  // contiguous index range [seg_lo(w), seg_lo(w + 1)): body groups [w gs, (w + 1) gs), with the
  // head in warp 0's segment and the tail in the last warp's.
  const int head = min(vis, int(((16u - (uint32_t(reinterpret_cast<uintptr_t>(lg)) & 15u)) & 15u) >> 2));
  const int nv = (vis - head) >> 2;
  const int body_end = head + 4 * nv;
  const int gs = max(1, (nv + kTkWarps - 1) / kTkWarps);
  const float4* lgv = reinterpret_cast<const float4*>(lg + head);
  auto seg_lo = [&](int w) { return w == 0 ? 0 : (w >= kTkWarps ? vis : head + 4 * min(nv, w * gs)); };
  auto owner = [&](int s) {
    return s < head ? 0 : (s >= body_end ? kTkWarps - 1 : min(kTkWarps - 1, ((s - head) >> 2) / gs));
  };
  const int v_lo = min(nv, warp * gs), v_hi = min(nv, (warp + 1) * gs);  // my body groups

  // The bin of hist[0, nb) holding the need-th largest key, counted from the top: s_sel, and
  // s_need = how many keys of that bin complete the set. Thread j sums the nb / 1024 bins
  // just below nb - (nb / 1024) j, the sums are scanned across the block in thread order, and
  // the one thread whose bins hold the need-th key walks them.
  auto find_bin = [&](int nb, uint32_t need) {
    const int per = nb / kTkThreads;
    const int top = nb - 1 - per * tid;
    uint32_t c = 0;
    for (int k = 0; k < per; ++k) c += hist[top - k];
    uint32_t x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      const uint32_t v = wsum[lane];
      uint32_t z = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, z, o);
        if (lane >= o) z += y;
      }
      wsum[lane] = z - v;  // the warps before, exclusive
    }
    __syncthreads();
    uint32_t acc = wsum[warp] + (x - c);
    if (acc < need && acc + c >= need) {
      for (int k = 0; k < per; ++k) {
        const uint32_t h = hist[top - k];
        if (acc + h >= need) {
          s_sel = uint32_t(top - k);
          s_need = need - acc;
          break;
        }
        acc += h;
      }
    }
    __syncthreads();
  };
  // Histogram of the keys' bits [sh, sh + width) among those whose higher bits equal prefix,
  // then find_bin. `key_at(j)` gives key j of `count`.
  auto select = [&](auto key_at, int count, uint32_t prefix, int sh, int width, uint32_t need) {
    const int nb = 1 << width;
    const uint32_t hmask = sh + width >= 32 ? 0u : (0xffffffffu << (sh + width));
    for (int k = tid; k < nb; k += kTkThreads) hist[k] = 0;
    __syncthreads();
    for (int s0 = tid; s0 < count; s0 += kTkThreads * kTkUnroll) {
      uint32_t key[kTkUnroll];
#pragma unroll
      for (int k = 0; k < kTkUnroll; ++k) {
        const int s = s0 + k * kTkThreads;
        key[k] = s < count ? key_at(s) : 0u;
      }
#pragma unroll
      for (int k = 0; k < kTkUnroll; ++k)
        if (s0 + k * kTkThreads < count && (key[k] & hmask) == prefix) atomicAdd(&hist[(key[k] >> sh) & (nb - 1)], 1u);
    }
    __syncthreads();
    find_bin(nb, need);
  };
  auto global_key = [&](int s) { return order_key(__ldg(lg + s)); };

  // pass 0: bits [31:20] of every visible key
  for (int k = tid; k < 4096; k += kTkThreads) hist[k] = 0;
  __syncthreads();
  for (int v0 = tid; v0 < nv; v0 += kTkThreads * kTkVec) {
    float4 f[kTkVec];
#pragma unroll
    for (int k = 0; k < kTkVec; ++k) {
      const int v = v0 + k * kTkThreads;
      f[k] = v < nv ? __ldg(lgv + v) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kTkVec; ++k)
      if (v0 + k * kTkThreads < nv) {
        atomicAdd(&hist[order_key(f[k].x) >> 20], 1u);
        atomicAdd(&hist[order_key(f[k].y) >> 20], 1u);
        atomicAdd(&hist[order_key(f[k].z) >> 20], 1u);
        atomicAdd(&hist[order_key(f[k].w) >> 20], 1u);
      }
  }
  if (tid < head) atomicAdd(&hist[global_key(tid) >> 20], 1u);
  if (tid < vis - body_end) atomicAdd(&hist[global_key(body_end + tid) >> 20], 1u);
  __syncthreads();
  find_bin(4096, uint32_t(p.K));
  const uint32_t sel0 = s_sel;
  uint32_t need = s_need;
  // pass 1 over each warp's segment: count the keys above the threshold bin, and gather the
  // bin's keys (and their indices) into shared memory
  if (tid == 0) s_ncand = 0;
  __syncthreads();
  const uint32_t bin_lo = sel0 << 20, bin_hi = bin_lo | 0xfffffu;
  uint32_t ngt = 0;  // this lane's keys above the bin, summed over the warp after the pass
  auto visit1 = [&](uint32_t key, int s, bool in) {
    ngt += (in && key > bin_hi) ? 1u : 0u;
    if (in && key - bin_lo <= 0xfffffu) {
      const uint32_t c = atomicAdd(&s_ncand, 1u);
      if (c < uint32_t(kTkCand)) {
        cand_key[c] = key;
        cand_idx[c] = s;
      }
    }
  };
  if (warp == 0) visit1(lane < head ? global_key(lane) : 0u, lane, lane < head);
  for (int g0 = v_lo; g0 < v_hi; g0 += 32 * kTkVec) {
    float4 f[kTkVec];
#pragma unroll
    for (int k = 0; k < kTkVec; ++k) {
      const int g = g0 + 32 * k + lane;
      f[k] = g < v_hi ? __ldg(lgv + g) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kTkVec; ++k) {
      const int g = g0 + 32 * k + lane;
      const bool in = g < v_hi;
      const int s = head + 4 * g;
      visit1(order_key(f[k].x), s, in);
      visit1(order_key(f[k].y), s + 1, in);
      visit1(order_key(f[k].z), s + 2, in);
      visit1(order_key(f[k].w), s + 3, in);
    }
  }
  if (warp == kTkWarps - 1) {
    const int s = body_end + lane;
    visit1(s < vis ? global_key(s) : 0u, s, s < vis);
  }
  ngt = __reduce_add_sync(0xffffffffu, ngt);
  __syncthreads();
  const int ncand = int(s_ncand);
  uint32_t prefix = sel0 << 20;
  uint32_t neq = 0;
  if (ncand <= kTkCand) {
    // passes 2 and 3 on the gathered keys of the bin
    auto cand_key_at = [&](int c) { return cand_key[c]; };
    select(cand_key_at, ncand, prefix, 10, 10, need);
    prefix |= s_sel << 10;
    need = s_need;
    select(cand_key_at, ncand, prefix, 0, 10, need);
    prefix |= s_sel;
    need = s_need;
    // the bin's keys above and equal to the threshold, into their warp segment's counts
    if (tid < kTkWarps) {
      wgt[tid] = 0;
      weq[tid] = 0;
    }
    __syncthreads();
    for (int c = tid; c < ncand; c += kTkThreads) {
      const uint32_t key = cand_key[c];
      const int w = owner(cand_idx[c]);
      if (key > prefix) atomicAdd(&wgt[w], 1u);
      else if (key == prefix) atomicAdd(&weq[w], 1u);
    }
    __syncthreads();
    ngt += wgt[warp];
    neq = weq[warp];
    __syncthreads();
  } else {
    // more keys in the bin than the buffer holds: passes 2 and 3 over global memory, then the
    // segments' counts
    select(global_key, vis, prefix, 10, 10, need);
    prefix |= s_sel << 10;
    need = s_need;
    select(global_key, vis, prefix, 0, 10, need);
    prefix |= s_sel;
    need = s_need;
    ngt = 0;
    const int a0 = seg_lo(warp), a1 = seg_lo(warp + 1);
    for (int s0 = a0; s0 < a1; s0 += 32 * kTkUnroll) {
      uint32_t key[kTkUnroll];
#pragma unroll
      for (int k = 0; k < kTkUnroll; ++k) {
        const int s = s0 + 32 * k + lane;
        key[k] = s < a1 ? global_key(s) : 0u;
      }
#pragma unroll
      for (int k = 0; k < kTkUnroll; ++k) {
        const bool in = s0 + 32 * k + lane < a1;
        ngt += __popc(__ballot_sync(0xffffffffu, in && key[k] > prefix));
        neq += __popc(__ballot_sync(0xffffffffu, in && key[k] == prefix));
      }
    }
  }
  // prefix is the K-th largest key; `need` keys equal to it complete the set (the lowest
  // indices among them). The segments' counts are scanned across warps, and then every warp
  // writes its selected indices in order (ballots within each chunk of 32 lanes).
  if (lane == 0) {
    wgt[warp] = ngt;
    weq[warp] = neq;
  }
  __syncthreads();
  uint32_t bg = 0, be = 0, eq_all = 0;
  for (int w2 = 0; w2 < kTkWarps; ++w2) {
    if (w2 < warp) {
      bg += wgt[w2];
      be += weq[w2];
    }
    eq_all += weq[w2];
  }
  const uint32_t below = (1u << lane) - 1u;
  if (eq_all == need) {
    // every key equal to the threshold is admitted (no tie is cut): the set is the keys at or
    // above it. A lane's count of selected keys (0 to 4) is spread over three ballots, one a
    // bit, so the lanes below are counted with three popcounts.
    uint32_t base = bg + be;
    if (warp == 0) {
      const bool sel = lane < head && global_key(lane) >= prefix;
      const uint32_t m = __ballot_sync(0xffffffffu, sel);
      if (sel) out[base + __popc(m & below)] = lane;
      base += __popc(m);
    }
    for (int g0 = v_lo; g0 < v_hi; g0 += 32 * kTkVec) {
      float4 f[kTkVec];
#pragma unroll
      for (int k = 0; k < kTkVec; ++k) {
        const int g = g0 + 32 * k + lane;
        f[k] = g < v_hi ? __ldg(lgv + g) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < kTkVec; ++k) {
        const int g = g0 + 32 * k + lane;
        const bool in = g < v_hi;
        const bool s0 = in && order_key(f[k].x) >= prefix, s1 = in && order_key(f[k].y) >= prefix;
        const bool s2 = in && order_key(f[k].z) >= prefix, s3 = in && order_key(f[k].w) >= prefix;
        const uint32_t c = uint32_t(s0) + uint32_t(s1) + uint32_t(s2) + uint32_t(s3);
        const uint32_t b0 = __ballot_sync(0xffffffffu, c & 1u), b1 = __ballot_sync(0xffffffffu, c & 2u);
        const uint32_t b2 = __ballot_sync(0xffffffffu, c & 4u);
        uint32_t pos = base + __popc(b0 & below) + 2u * __popc(b1 & below) + 4u * __popc(b2 & below);
        const int s = head + 4 * g;
        if (s0) out[pos++] = s;
        if (s1) out[pos++] = s + 1;
        if (s2) out[pos++] = s + 2;
        if (s3) out[pos] = s + 3;
        base += __popc(b0) + 2u * __popc(b1) + 4u * __popc(b2);
      }
    }
    if (warp == kTkWarps - 1) {
      const int s = body_end + lane;
      const bool sel = s < vis && global_key(s) >= prefix;
      const uint32_t m = __ballot_sync(0xffffffffu, sel);
      if (sel) out[base + __popc(m & below)] = s;
    }
    return;
  }
  // one key a lane (the head and the tail): "above" keys go after the admitted "equal" ones
  // before them; the first `need` equal keys in index order are admitted
  auto emit1 = [&](uint32_t key, int s, bool in) {
    const bool gt = in && key > prefix, eq = in && key == prefix;
    const uint32_t mg = __ballot_sync(0xffffffffu, gt), me = __ballot_sync(0xffffffffu, eq);
    const uint32_t rg = bg + __popc(mg & below), re = be + __popc(me & below);
    if (gt) out[rg + min(re, need)] = s;
    if (eq && re < need) out[rg + re] = s;
    bg += __popc(mg);
    be += __popc(me);
  };
  if (warp == 0) emit1(lane < head ? global_key(lane) : 0u, lane, lane < head);
  for (int g0 = v_lo; g0 < v_hi; g0 += 32 * kTkVec) {
    float4 f[kTkVec];
#pragma unroll
    for (int k = 0; k < kTkVec; ++k) {
      const int g = g0 + 32 * k + lane;
      f[k] = g < v_hi ? __ldg(lgv + g) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < kTkVec; ++k) {
      // four keys a lane, lane-major: the keys before (lane, j) are every key of the lanes
      // below and this lane's keys before j
      const int g = g0 + 32 * k + lane;
      const bool in = g < v_hi;
      const uint32_t key[4] = {order_key(f[k].x), order_key(f[k].y), order_key(f[k].z), order_key(f[k].w)};
      bool gt[4], eq[4];
      uint32_t rg = bg, re = be, tg = 0, te = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        gt[j] = in && key[j] > prefix;
        eq[j] = in && key[j] == prefix;
        const uint32_t mg = __ballot_sync(0xffffffffu, gt[j]), me = __ballot_sync(0xffffffffu, eq[j]);
        rg += __popc(mg & below);
        re += __popc(me & below);
        tg += __popc(mg);
        te += __popc(me);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int s = head + 4 * g + j;
        if (gt[j]) out[rg + min(re, need)] = s;
        if (eq[j] && re < need) out[rg + re] = s;
        rg += gt[j] ? 1u : 0u;
        re += eq[j] ? 1u : 0u;
      }
      bg += tg;
      be += te;
    }
  }
  if (warp == kTkWarps - 1) {
    const int s = body_end + lane;
    emit1(s < vis ? global_key(s) : 0u, s, s < vis);
  }
}
}  // namespace

cudaError_t launch_indexer_logits(const IndexerArgs& a, int num_sms, cudaStream_t s) {
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t(1) << dev) : 0;
  if (!(configured.load(std::memory_order_acquire) & bit) || !bit) {
    const cudaError_t e =
        cudaFuncSetAttribute(indexer_logits_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kIxSmem));
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_release);
  }
  alignas(64) CUtensorMap kmap;
  alignas(64) CUtensorMap qmap;
  cudaError_t e = index_key_map(a, &kmap);
  if (e == cudaSuccess) e = index_q_map(a, &qmap);
  if (e != cudaSuccess) return e;
  indexer_logits_kernel<<<num_sms, kIxThreads, kIxSmem, s>>>(a, kmap, qmap);
  return cudaGetLastError();
}

cudaError_t launch_indexer_topk(const IndexerArgs& a, cudaStream_t s) {
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t(1) << dev) : 0;
  if (!(configured.load(std::memory_order_acquire) & bit) || !bit) {
    const cudaError_t e =
        cudaFuncSetAttribute(indexer_topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kTkSmem));
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_release);
  }
  indexer_topk_kernel<<<a.T, kTkThreads, kTkSmem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace smla
