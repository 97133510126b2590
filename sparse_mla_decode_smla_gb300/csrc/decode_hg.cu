// Sparse MLA decode on the 5th-generation tensor cores (tcgen05, TMEM accumulators) for the
// FP8 caches (fp8_ds: 656-byte rows with per-128 scales and bf16 RoPE; per-tensor FP8: 576
// E4M3 codes with one scale, vLLM PR #43827), one CTA per (query token, top-k split, group of
// 64 heads). Up to 8 splits of a (token, head group) form one thread-block cluster and merge
// their partials through distributed shared memory.
//
// What it computes is the sparse decode of vLLM PR #43477 "关键源码片段" (forward_mqa) with
// the sink and split merge of SGLang PR #24692 "关键文件": out_h = softmax over the selected
// slots of sm_scale * <q_h, k_j>, applied to v_j = k_j[0:512].
//
// Why one CTA holds 64 heads: the fp32 output of 64 heads x 512 dims is 128 KB, half of
// an SM's tensor memory, if the two halves of each head's 512 dims are stacked on the 128
// TMEM lanes: lane l < 64 holds head l's dims [0, 256), lane 64 + l its dims [256, 512), in
// 256 columns. q is stacked the same way (lane l < 64: dims [0, 256) of head l; lane 64 + l:
// dims [256, 512)), so QK needs no exchange between SMs:
//  * QK of a 64-slot tile: B stacks the same slots twice, rows 0-63 with dims [0, 256) and
//    rows 64-127 with dims [256, 512). Lane l < 64, columns 0-63 of the M128 N128 result are
//    the low partial scores of head l; lane 64 + l, columns 64-127, the high ones (the other
//    two quadrants are unused). The 64 RoPE dims are split the same way, with q's RoPE part
//    as an A operand in shared memory. 18 x M128 N128 K16 per tile: the cost of these MMAs
//    barely depends on N, so a wide tile halves the QK cost per slot.
//  * The two partial rows of a head meet in shared memory: the warp of lane quarter w and
//    the warp of quarter w ^ 2 hold heads 32(w & 1) .. 32(w & 1) + 31, low and high. The low
//    warp finishes slots 0-31 and the high warp slots 32-63; they swap their maxima, so both
//    take the same running max and rescale factor.
//  * PV: A = [P; 0] against the latent dims [0, 256) of the tile and A = [0; P] against dims
//    [256, 512), both into the same 256 TMEM columns, so lanes 0-63 accumulate the low
//    output dims and lanes 64-127 the high ones. 8 x M128 N256 K16 per tile.
// Half of each MMA's rows or columns are unused: 64 heads fill only half of an M = 128
// tile. In exchange a group of 64 heads needs one SM, not two, and no traffic between SMs.
//
// The MMAs run on f16 operands with fp32 accumulation: an E4M3 code converts to f16 exactly,
// and the block scale applies with one f16 multiply (exact for power-of-two scales, within
// 2^-11 otherwise); q converts from bf16 exactly. Dequantised keys and q must stay within
// f16's range (+-65504).
//
// Per CTA (480 threads):
//  * start-up: one thread initialises the barriers and issues q as nine TMA boxes of
//    [64 heads x 64 dims] (128-byte swizzle), which land while the producers prime their rings.
//  * warps 12-13, producers: index entries five tiles ahead and page-table entries three
//    tiles ahead by 4-byte cp.async, then the selected rows by TMA gathers of four rows each
//    (tile::gather4 on a tensor map of the cache) into a ring of four 16-row stages, a whole
//    tile; a masked slot gets a row outside the tensor, which the TMA fills with zeros
//    without reading memory. One gather per four rows keeps the TMA engine, which serialises
//    its operations, off the critical path. Warp 12 fills stages 0 and 2 of every tile,
//    warp 13 stages 1 and 3.
//  * warps 4-11, dequant: e4m3 (* scale) -> f16 into the latent K tile (two buffers): four
//    128-byte-swizzled blocks of [64 slots x 64 low dims | 64 slots x 64 high dims], which
//    are B of QK (K-major) and B of PV (MN-major). A 16-row quarter of a buffer is rewritten
//    as soon as PV has finished reading it. The RoPE dims go to one 64-byte-swizzled block
//    once QK of the previous tile has completed.
//  * warp 14, MMA issuer (one thread): QK of tile i+1 runs while the softmax of tile i does;
//    of the two, whichever is ready is issued first (PV of tile i when its P is written).
//  * warps 0-3, softmax and epilogue: base-2 online softmax with lazy rescaling (the running
//    max moves only when it grows by more than 8, as in FlashAttention-4).
//  * split merge (more than one split, at most 8): after a cluster barrier the softmax
//    threads store their normalised f16 rows and LSEs into the shared memory of the cluster
//    CTA that merges their head; after a second barrier every CTA merges its share of the
//    heads from its own shared memory. More splits go through global memory and the merge
//    kernel.
// Every wait is bounded in time; a wait that gives up sets SMLA_DEVERR_TIMEOUT. The two
// warps of a head pair meet at named barriers that also AND their status, so both leave the
// tile loop at the same barrier and neither waits for a partner that has left.
#include <math_constants.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace smla {
namespace {

constexpr int kHgN = 64;                 // slots per tile
constexpr int kHgSub = 16;               // rows per raw-ring stage (a quarter tile)
constexpr int kHgFirstDequant = 4;       // warps 0..3: softmax
constexpr int kHgDequantWarps = 8;
constexpr int kHgFirstProducer = kHgFirstDequant + kHgDequantWarps;
constexpr int kHgProducers = 2;
constexpr int kHgMmaWarp = kHgFirstProducer + kHgProducers;
// fp8_ds: the block scales of every raw stage are checked against the f16 window by a warp
// of their own, so the dequant warps, which set the tile period, do no extra work for it
constexpr int kHgCheckWarp = kHgMmaWarp + 1;
constexpr int kHgThreads = 32 * (kHgCheckWarp + 1);
constexpr int kHgDequantThreads = 32 * kHgDequantWarps;
// Named barrier of every warp but the producers, once q is placed (ids 1-10 belong to the
// softmax warp pairs, 0 to __syncthreads)
constexpr int kHgBarQPlaced = 11;
// Named barrier of the softmax and dequant warps between the two passes of q placement
constexpr int kHgBarQMax = 12;
constexpr int kHgRawStages = 4;  // a whole tile
constexpr int kHgGroup = 2688;              // four gathered rows (<= 4 x 656 B), 128-byte aligned
constexpr int kHgRawStage = 4 * kHgGroup;   // 16 rows
constexpr int kHgPairBlk = 2 * kHgN * 128;  // [64 slots x 64 low dims | same slots, high dims]
constexpr int kHgKLat = 4 * kHgPairBlk;     // latent K tile (two buffers)
constexpr int kHgRopeBlk = 2 * kHgN * 64;   // [64 slots x RoPE 0..31 | same slots, 32..63]
constexpr int kHgPBlk = 64 * kHgN * 2;      // 64 rows x 64 slots f16, 128-byte swizzle
constexpr int kHgQrope = 128 * 64;          // q RoPE, [128 rows x 32 dims] f16
constexpr int kHgXRow = 80;                 // 16 fp32 + padding (conflict-free rows)
constexpr int kHgIdxAhead = 5, kHgIdxRing = 6;
constexpr int kHgAhead = 3, kHgPageRing = 4;
constexpr int kHgMetaRing = 8;
constexpr float kHgRescaleThreshold = 8.f;  // log2 units
static_assert(kHgIdxAhead <= 2 * kHgAhead && kHgIdxRing > kHgIdxAhead && kHgPageRing > kHgAhead,
              "index and page rings");

// TMEM columns (512 allocated)
constexpr uint32_t kHgTmO = 0;    // O [128 lanes x 256] fp32, lanes 64.. = high dims
constexpr uint32_t kHgTmQ = 256;  // q latent [128 lanes x 256 dims] f16: 128 columns
constexpr uint32_t kHgTmS = 384;  // scores [128 lanes x 128] fp32

constexpr size_t kHgOffK = 0;
constexpr size_t kHgOffRope = kHgOffK + 2 * size_t(kHgKLat);
constexpr size_t kHgOffP = kHgOffRope + kHgRopeBlk;  // [0 | P | 0]
constexpr size_t kHgOffQr = kHgOffP + 3 * size_t(kHgPBlk);
constexpr size_t kHgOffRaw = kHgOffQr + kHgQrope;
constexpr size_t kHgOffXs = kHgOffRaw + size_t(kHgRawStages) * kHgRawStage;
constexpr size_t kHgOffXm = kHgOffXs + 128 * size_t(kHgXRow);
constexpr size_t kHgOffIdx = kHgOffXm + 128 * 4;
constexpr size_t kHgOffPages = kHgOffIdx + size_t(kHgIdxRing) * kHgN * 4;
constexpr size_t kHgOffMeta = kHgOffPages + size_t(kHgPageRing) * kHgN * 4;
constexpr size_t kHgOffTmem = kHgOffMeta + kHgMetaRing * 8;
constexpr size_t kHgOffBars = kHgOffTmem + 16;
// mbarrier indices, laid out from the raw ring's stage count
enum {
  H_RAW_FULL = 0,
  H_RAW_EMPTY = H_RAW_FULL + kHgRawStages,
  H_K_FULL = H_RAW_EMPTY + kHgRawStages,  // [buffer]
  H_K_FREE = H_K_FULL + 2,                 // [buffer][16-slot chunk]
  H_ROPE_FULL = H_K_FREE + 8,
  H_S_FULL, H_S_FREE, H_P_READY, H_PV_DONE, H_Q, H_DRAIN, H_COUNT
};
static_assert(H_RAW_EMPTY == kHgRawStages && H_K_FULL == 2 * kHgRawStages && H_COUNT == 2 * kHgRawStages + 17,
              "one mbarrier per ring stage and buffer, none shared");
constexpr size_t kSmemHg = kHgOffBars + H_COUNT * 8 + 1024;  // + alignment slack
static_assert(kSmemHg <= 232448, "shared memory budget");
static_assert(kHgOffK % 1024 == 0 && kHgKLat % 1024 == 0 && kHgOffP % 1024 == 0 && kHgOffRope % 512 == 0 &&
                  kHgOffQr % 512 == 0 && kHgOffRaw % 128 == 0 && kHgOffBars % 8 == 0 && kHgGroup % 128 == 0 &&
                  kHgGroup >= 4 * kFp8RowBytes,
              "swizzle atoms: 1024-byte (128-byte swizzle) and 512-byte (64-byte swizzle) aligned");
// q staging at start-up, in the K-tile area (first written by the pipeline after the
// start-up barriers): nine 128-byte-swizzled boxes of [64 heads x 64 dims] bf16
constexpr uint32_t kHgQBox = 64 * 128;
constexpr uint32_t kHgQBytes = 9 * kHgQBox;
static_assert(kHgQBytes <= kHgOffRope, "q staging fits in the K-tile area");

template <bool TENS>
__global__ void __launch_bounds__(kHgThreads, 1)
    decode_hg_kernel(const DecodeArgs p, const __grid_constant__ CUtensorMap kv_map,
                     const __grid_constant__ CUtensorMap q_map) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  auto bar = [&](int k) -> uint32_t { return sb + uint32_t(kHgOffBars) + 8u * k; };
  // Split-merge buffer in the K-tile area, filled by the cluster's CTAs once their pipelines
  // are done: the f16 partial rows of the heads this CTA merges, row s hp + k for split s and
  // head k of its range (16-byte chunk c of row r at chunk c ^ (r & 7)), at most 72 rows;
  // then the rows' LSEs and the merge weights.
  auto mrow_addr = [&](int r, int c) -> uint32_t {
    return sb + uint32_t(kHgOffK) + uint32_t(r) * 1024u + uint32_t((c ^ (r & 7)) << 4);
  };
  const uint32_t mlse = sb + uint32_t(kHgOffK) + 72u * 1024u;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the two TMA descriptors, fetched before their first use (q's load, the first row gathers)
  if (tid == 0) prefetch_tensormap(&q_map);
  if (tid == 32 * kHgFirstProducer) prefetch_tensormap(&kv_map);

  // Per-tensor FP8 codes go into the K tile unscaled (exact in f16); kv_scale is applied in
  // fp32 to the scores (bmm1_scale = sm_scale * kv_scale) and to O (bmm2_scale = kv_scale),
  // the scale algebra of vLLM PR #43827 "关键源码片段".
  constexpr bool tens = TENS;
  const float c2 = tens ? p.c2 * p.kv_scale : p.c2;
  const int G = (p.H + 63) >> 6;  // groups of 64 heads, one CTA each
  // the splits of a (token, head group) are consecutive CTAs: with the in-kernel merge they
  // form one cluster, and the split is the CTA's rank in it
  const int split = blockIdx.x % p.num_splits;
  const int item = p.item0 + int(blockIdx.x) / p.num_splits;
  const int g = item % G;
  const int t = item / G;
  const int r = p.req_id ? __ldg(p.req_id + t) : t / p.next_n;
  const bool req_ok = r >= 0 && r < p.B;
  const int32_t* pt_row = p.page_table + int64_t(req_ok ? r : 0) * p.stride;
  const int32_t* idx_row = p.topk + int64_t(t) * p.K;
  const int j0 = split * p.split_len;
  const int j1 = min(p.K, j0 + p.split_len);
  const int nidx = max(0, j1 - j0);
  const int ntiles = req_ok ? (nidx + kHgN - 1) / kHgN : 0;
  const int h0 = 64 * g;
  const int gheads = min(64, p.H - h0);  // heads of this group
  const int nq = req_ok ? gheads : 0;     // q rows to load
  const int mhp = (gheads + p.num_splits - 1) / p.num_splits;  // heads each split merges (cluster merge)

  // Producer lanes 0-15 of warp 12 + pw own slots 16q + lane for q in {pw, pw + 2} of every
  // tile. They fetch each slot's index kHgIdxAhead tiles ahead and, once it has landed, its
  // page-table entry kHgAhead tiles ahead. Every ring step commits one cp.async group
  // {indices of tile i + kHgIdxAhead, page entries of tile i + kHgAhead}; the steps before
  // tile 0 prime the rings before the set-up.
  const bool producer = warp >= kHgFirstProducer && warp < kHgMmaWarp;
  const int pw = warp - kHgFirstProducer;
  const bool act = lane < kHgSub;
  int32_t* sidx = reinterpret_cast<int32_t*>(sm + kHgOffIdx);
  int32_t* spage = reinterpret_cast<int32_t*>(sm + kHgOffPages);
  auto in_split = [&](int tile, int q) {
    return act && tile < ntiles && tile * kHgN + kHgSub * q + lane < nidx;
  };
  auto idx_of = [&](int tile, int q) -> int32_t {
    return in_split(tile, q) ? sidx[(tile % kHgIdxRing) * kHgN + kHgSub * q + lane] : -1;
  };
  auto ring_step = [&](int i) {
    cp_async_wait<kHgIdxAhead - kHgAhead - 1>();  // the group that fetched indices i + kHgAhead
    const int tp = i + kHgAhead;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int q = pw + 2 * k;
      if (tp >= 0) {
        const int32_t idx = idx_of(tp, q);
        if (idx >= 0 && (idx >> p.log2_page) < p.stride)
          cp_async4(smem_u32(spage + (tp % kHgPageRing) * kHgN + kHgSub * q + lane), pt_row + (idx >> p.log2_page));
      }
      const int ti = i + kHgIdxAhead;
      if (in_split(ti, q))
        cp_async4(smem_u32(sidx + (ti % kHgIdxRing) * kHgN + kHgSub * q + lane),
                  idx_row + j0 + ti * kHgN + kHgSub * q + lane);
    }
    cp_async_commit();
  };
  if (producer)
    for (int i = -kHgIdxAhead; i < 0; ++i) ring_step(i);

  // ------------------------------------------------------------------ set-up
  {
    // masked slots of the first tiles dequantise zeros, and the P buffer's zero blocks stay 0
    uint4* z = reinterpret_cast<uint4*>(sm + kHgOffRaw);
    for (int k = tid; k < kHgRawStages * kHgRawStage / 16; k += kHgThreads) z[k] = make_uint4(0, 0, 0, 0);
    uint4* zp = reinterpret_cast<uint4*>(sm + kHgOffP);
    for (int k = tid; k < 3 * kHgPBlk / 16; k += kHgThreads) zp[k] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
      for (int s = 0; s < kHgRawStages; ++s) {
        mbar_init(bar(H_RAW_FULL + s), 1);  // the expect_tx arrival of the stage's producer warp
        mbar_init(bar(H_RAW_EMPTY + s), kHgDequantWarps + (tens ? 0 : 1));  // + the check warp
      }
      for (int b = 0; b < 2; ++b) mbar_init(bar(H_K_FULL + b), kHgDequantWarps);
      for (int c = 0; c < 8; ++c) mbar_init(bar(H_K_FREE + c), 1);
      mbar_init(bar(H_ROPE_FULL), kHgDequantWarps);
      mbar_init(bar(H_S_FULL), 1);
      mbar_init(bar(H_S_FREE), 4);
      mbar_init(bar(H_P_READY), 4);
      mbar_init(bar(H_PV_DONE), 1);
      mbar_init(bar(H_Q), 1);
      mbar_init(bar(H_DRAIN), 1);
      tc::fence_mbarrier_init_cluster();
      if (!req_ok && split == 0 && g == 0) atomicOr(p.err, SMLA_DEVERR_INDEX);
      // the group's q rows [t H + h0, + 64) as nine 64-dim boxes; they land while the
      // producers prime their index and page rings (rows past the group are not used)
      if (nq > 0) {
        mbar_arrive_expect_tx(bar(H_Q), kHgQBytes);
        for (int bx = 0; bx < 9; ++bx)
          tma_load_2d(sb + uint32_t(kHgOffK) + bx * kHgQBox, &q_map, 64 * bx, t * p.H + h0, bar(H_Q));
      }
    }
    if (warp == kHgMmaWarp) tc::alloc(sb + uint32_t(kHgOffTmem), 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
  }
  const uint32_t tm = *reinterpret_cast<volatile uint32_t*>(sm + kHgOffTmem);

  // The softmax and dequant warps place q: lane l < 64 gets dims [0, 256) of head h0 + l,
  // lane 64 + l dims [256, 512), as f16 in TMEM (A of QK); the RoPE dims go to shared memory,
  // rows 0-63 dims 512..543 and rows 64-127 dims 544..575 (64-byte swizzle). Box b of the
  // staged q holds dims [64b, 64b+64) of the 64 heads, 16-byte chunk c of head row r at
  // chunk c ^ (r & 7). Warp w serves TMEM lane quarter w % 4 and part w / 4 of each row:
  // 32-dim chunks {0, 1, 2}, {3, 4, 5} or {6, 7} and the row's 32 RoPE dims.
  //
  // Each row gets a power-of-two normaliser: its largest |q| over the 288 dims it holds
  // (256 latent + 32 RoPE) is brought into [1, 2), and the factor 2^f goes back into the
  // fp32 scores. So any finite bf16 q is exact in f16 (elements below 2^-17 of the row's
  // largest keep 2^-25 of it in absolute error), whatever its magnitude. The three parts'
  // maxima meet in shared memory (the score-exchange rows, unused until the tile loop).
  if (warp < kHgFirstProducer) {
    const int quarter = warp & 3, part = warp >> 2;
    const int half = quarter >> 1;
    const int hl = 32 * (quarter & 1) + lane;
    const int row = 32 * quarter + lane;
    const uint32_t lrow = tm + (uint32_t(32 * quarter) << 16);
    const uint32_t qs = sb + uint32_t(kHgOffK) + uint32_t(hl) * 128;
    auto qchunk = [&](int dim) -> uint32_t {  // 8 dims [dim, dim + 8) of head hl
      return qs + (dim >> 6) * kHgQBox + ((((dim >> 3) & 7) ^ (hl & 7)) << 4);
    };
    const int ch0 = 3 * part, ch1 = min(8, ch0 + 3);  // this part's 32-dim latent chunks
    const bool rope = part == 2;
    const bool got = nq == 0 || mbar_wait(bar(H_Q), 0);
    if (!got && lane == 0 && part == 0) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
    const bool have = got && hl < nq;
    uint32_t m4[4] = {0, 0, 0, 0};  // bf16x2 magnitudes, four independent running maxima
    if (have) {
      for (int k = 4 * ch0; k < 4 * ch1 + (rope ? 4 : 0); ++k) {  // 8-dim chunks; RoPE last
        const uint4 v = lds128(qchunk(k < 4 * ch1 ? 256 * half + 8 * k : kLatent + 32 * half + 8 * (k - 4 * ch1)));
        m4[0] = bf16x2_max(m4[0], v.x & 0x7fff7fffu);
        m4[1] = bf16x2_max(m4[1], v.y & 0x7fff7fffu);
        m4[2] = bf16x2_max(m4[2], v.z & 0x7fff7fffu);
        m4[3] = bf16x2_max(m4[3], v.w & 0x7fff7fffu);
      }
    }
    const uint32_t mx = bf16x2_hmax_bits(bf16x2_max(bf16x2_max(m4[0], m4[1]), bf16x2_max(m4[2], m4[3])));
    const uint32_t pmax = sb + uint32_t(kHgOffXs);  // [part][row] u32
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(pmax + uint32_t(128 * part + row) * 4), "r"(mx) : "memory");
    named_bar(kHgBarQMax, 32 * kHgFirstProducer);
    const uint32_t rmax = max(max(lds_u32(pmax + uint32_t(row) * 4), lds_u32(pmax + uint32_t(128 + row) * 4)),
                              lds_u32(pmax + uint32_t(256 + row) * 4));
    const int qf = pow2_exponent_of_bf16(rmax);
    const float qdown = exp2_int(-qf);
    auto cvt = [&](uint32_t w) { return pack_f16x2(bf16_lo(w) * qdown, bf16_hi(w) * qdown); };
#pragma unroll 1
    for (int ch = ch0; ch < ch1; ++ch) {
      uint32_t wv[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (have) v = lds128(qchunk(256 * half + 32 * ch + 8 * k));
        wv[4 * k] = cvt(v.x); wv[4 * k + 1] = cvt(v.y);
        wv[4 * k + 2] = cvt(v.z); wv[4 * k + 3] = cvt(v.w);
      }
      tc::st16(lrow + kHgTmQ + 16 * ch, wv);
    }
    tc::wait_st();
    if (rope) {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (have) v = lds128(qchunk(kLatent + 32 * half + 8 * c));
        const uint32_t dst = sb + uint32_t(kHgOffQr) + row * 64 + ((c ^ ((row >> 1) & 3)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(cvt(v.x)), "r"(cvt(v.y)),
                     "r"(cvt(v.z)), "r"(cvt(v.w))
                     : "memory");
      }
      fence_proxy_async_smem();  // read by the tensor core
    }
    // the factor of this row, read by the softmax warps of both halves of the head after
    // the barrier below; the slot is next written in the tile loop, after both warps of a
    // pair have met at a barrier
    if (part == 0)
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(sb + uint32_t(kHgOffXm) + uint32_t(row) * 4), "f"(exp2_int(qf))
                   : "memory");
  }
  // q is in place for the MMA warp, and its staging copy in the K-tile area has been read
  // before the dequant warps write there. The producer warps write only their own rings and
  // start gathering without waiting for it.
  if (!producer && warp != kHgCheckWarp) {
    tc::fence_before();
    named_bar(kHgBarQPlaced, kHgThreads - 32 * (kHgProducers + 1));
    tc::fence_after();
  }

  bool ok = true;
  // cluster merge: the softmax threads' final row factor and LSE (without the sink)
  float cm_f = 0.f, cm_lse = -CUDART_INF_F;
  // ------------------------------------------------------------------ producer
  if (producer) {
    uint16_t* meta = reinterpret_cast<uint16_t*>(sm + kHgOffMeta);
    const uint32_t rowbytes = tens ? uint32_t(kFp8TensorRowBytes) : uint32_t(kFp8RowBytes);
    // a row the tensor map does not hold: its gather reads nothing and fills zeros
    const int32_t oob_row = int32_t(p.num_pages << p.log2_page);
    for (int i = 0; i < ntiles && ok; ++i) {
      ring_step(i);
#pragma unroll 1
      for (int k = 0; k < 2 && ok; ++k) {
        const int q = pw + 2 * k;
        const int u = 4 * i + q, st = u % kHgRawStages;
        if (!mbar_wait(bar(H_RAW_EMPTY + st), ((u / kHgRawStages) & 1) ^ 1)) {
          ok = false;
          break;
        }
        const int32_t idx = idx_of(i, q);
        int64_t phys = -1;
        if (idx != -1) {
          if (idx < 0 || (idx >> p.log2_page) >= p.stride) {
            atomicOr(p.err, SMLA_DEVERR_INDEX);
          } else {
            const int32_t pg = spage[(i % kHgPageRing) * kHgN + kHgSub * q + lane];
            if (pg < 0 || pg >= p.num_pages)
              atomicOr(p.err, SMLA_DEVERR_PAGE);
            else
              phys = (int64_t(pg) << p.log2_page) + (idx & ((1 << p.log2_page) - 1));
          }
        }
        const uint32_t vm = __ballot_sync(0xffffffffu, phys >= 0);
        // lane g < 4 gathers rows 4g..4g+3 of the stage, unless none of them is selected
        const int32_t y = phys >= 0 ? int32_t(phys) : oob_row;
        const int32_t y0 = __shfl_sync(0xffffffffu, y, 4 * (lane & 3));
        const int32_t y1 = __shfl_sync(0xffffffffu, y, 4 * (lane & 3) + 1);
        const int32_t y2 = __shfl_sync(0xffffffffu, y, 4 * (lane & 3) + 2);
        const int32_t y3 = __shfl_sync(0xffffffffu, y, 4 * (lane & 3) + 3);
        uint32_t groups = 0;
#pragma unroll
        for (int gq = 0; gq < 4; ++gq) groups |= ((vm >> (4 * gq)) & 15u) ? (1u << gq) : 0u;
        if (lane == 0) {
          meta[(i % kHgMetaRing) * 4 + q] = uint16_t(vm);
          mbar_arrive_expect_tx(bar(H_RAW_FULL + st), uint32_t(__popc(groups)) * 4u * rowbytes);
        }
        __syncwarp();
        if (lane < 4 && ((groups >> lane) & 1u))
          tma_gather4(sb + uint32_t(kHgOffRaw) + uint32_t(st * kHgRawStage + lane * kHgGroup), &kv_map, 0, y0, y1,
                      y2, y3, bar(H_RAW_FULL + st));
      }
    }
    cp_async_wait<0>();
    // no copy may land after the CTA has left: wait for this warp's stages among the last
    // ring's worth
    const int total = 4 * ntiles;
    for (int u = max(0, total - kHgRawStages); u < total; ++u)
      if ((u & 1) == pw && !mbar_wait(bar(H_RAW_FULL + u % kHgRawStages), (u / kHgRawStages) & 1)) break;
  }
  // ------------------------------------------------------------------ MMA issuer
  else if (warp == kHgMmaWarp) {
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t kIdQK = tc::idesc_f16_f32(128, 128, false, false);
      constexpr uint32_t kIdPV = tc::idesc_f16_f32(128, 256, false, true);
      const uint32_t qr = sb + uint32_t(kHgOffQr);
      const uint32_t rope = sb + uint32_t(kHgOffRope);
      const uint32_t d = tm + kHgTmS;
      // QK of tile i once its K tile and RoPE block are written and the scores of tile i-1
      // have been read
      auto qk_ready = [&](int i) {
        return mbar_test_wait(bar(H_K_FULL + (i & 1)), (i >> 1) & 1) &&
               (i == 0 || mbar_test_wait(bar(H_S_FREE), (i - 1) & 1)) && mbar_test_wait(bar(H_ROPE_FULL), i & 1);
      };
      auto qk = [&](int i) {
        tc::fence_after();
        const uint32_t kt = sb + uint32_t(kHgOffK) + uint32_t((i & 1) * kHgKLat);
#pragma unroll
        for (int j = 0; j < 16; ++j)
          tc::mma_ts(d, tm + kHgTmQ + 8 * j, tc::sdesc_sw128(kt + (j >> 2) * kHgPairBlk + (j & 3) * 32, 16, 1024),
                     kIdQK, j > 0);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tc::mma_ss(d, tc::sdesc_sw64(qr + 32 * j, 16, 512), tc::sdesc_sw64(rope + 32 * j, 16, 512), kIdQK, 1);
        tc::commit(bar(H_S_FULL));
      };
      auto pv = [&](int i) {
        tc::fence_after();
        const uint32_t kt = sb + uint32_t(kHgOffK) + uint32_t((i & 1) * kHgKLat);
        const uint32_t pa = sb + uint32_t(kHgOffP) + uint32_t(kHgPBlk);  // P rows
#pragma unroll
        for (int s = 0; s < 4; ++s) {  // 16 slots per MMA
          // [P; 0] x latent dims [0, 256) -> lanes 0-63; [0; P] x dims [256, 512) -> lanes 64-127
          tc::mma_ss(tm + kHgTmO, tc::sdesc_sw128(pa + 32 * s, 16, 1024),
                     tc::sdesc_sw128(kt + 2048 * s, kHgPairBlk, 1024), kIdPV, (i > 0 || s > 0));
          tc::mma_ss(tm + kHgTmO, tc::sdesc_sw128(pa - kHgPBlk + 32 * s, 16, 1024),
                     tc::sdesc_sw128(kt + 8192 + 2048 * s, kHgPairBlk, 1024), kIdPV, 1);
          tc::commit(bar(H_K_FREE + 4 * (i & 1) + s));  // rows [16s, 16s+16) of the K tile are free
        }
        tc::commit(bar(H_PV_DONE));
      };
      // Issue whichever is ready first: PV of the oldest scored tile, or QK of the next one
      // (the barriers allow QK at most one tile ahead of PV). PV goes first, so a K buffer
      // never waits behind a QK whose tile is still being dequantised.
      int nqk = 0, npv = 0;
      uint64_t t0 = globaltimer_ns();
      for (uint32_t it = 0; npv < ntiles; ++it) {
        if (npv < nqk && mbar_test_wait(bar(H_P_READY), npv & 1)) {
          pv(npv++);
        } else if (nqk < ntiles && nqk <= npv + 1 && qk_ready(nqk)) {
          qk(nqk++);
        } else {
          if ((it & 255u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
            ok = false;
            break;
          }
          continue;
        }
        t0 = globaltimer_ns();
      }
      // every MMA issued has completed before the tensor memory is released
      tc::commit(bar(H_DRAIN));
      if (!mbar_wait(bar(H_DRAIN), 0)) ok = false;
    }
    __syncwarp();
  }
  // ------------------------------------------------------------------ f16 window check
  else if (warp == kHgCheckWarp) {
    if (!tens) {
      // lane l reads row l % 16 of each raw stage, block scales 2h and 2h+1 (h = l / 16).
      // Rows of the stage that were not gathered this time hold bytes checked when they
      // were (or zeros), so they never raise a false flag. Running extremes of the scales'
      // bit patterns (branch-free integer ops, so a stage goes back to the producers soon
      // after it lands) are compared with the window once, at the end: the largest scale
      // (inf and NaN count as the largest), the smallest non-zero power-of-two scale and
      // the smallest other scale. Only the 16 scale bytes of a row are read here: the
      // kernel's shared-memory traffic sets its pace.
      const int r = lane & 15, hh = lane >> 4;
      uint32_t smax = 0, smin_p2 = ~0u, smin_other = ~0u;
      for (int i = 0; i < ntiles && ok; ++i) {
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          const int u = 4 * i + q, st = u % kHgRawStages;
          if (!mbar_wait(bar(H_RAW_FULL + st), (u / kHgRawStages) & 1)) {
            ok = false;
            break;
          }
          const uint32_t row = sb + uint32_t(kHgOffRaw) + uint32_t(st * kHgRawStage) +
                               uint32_t((r >> 2) * kHgGroup + (r & 3) * kFp8RowBytes);
          const uint2 sc2 = lds64(row + kScaleOff + 8 * hh);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint32_t a = (e ? sc2.y : sc2.x) & 0x7fffffffu;
            const bool p2 = (a & 0x7fffffu) == 0;
            smax = max(smax, a);
            smin_p2 = min(smin_p2, (p2 && a != 0) ? a : ~0u);
            smin_other = min(smin_other, p2 ? ~0u : a);
          }
          // both loaded scales have been used: the stage may be overwritten
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(H_RAW_EMPTY + st));
        }
      }
      // window: power-of-two scales in [2^-15, 2^7], others in [2^-14, 2^7]
      const bool out_of_window = smax > 0x43000000u || smin_p2 < 0x38000000u || smin_other < 0x38800000u;
      if (__any_sync(0xffffffffu, out_of_window) && lane == 0) atomicOr(p.err, SMLA_DEVERR_RANGE);
    }
  }
  // ------------------------------------------------------------------ dequant
  else if (warp >= kHgFirstDequant) {
    const int dtid = tid - 32 * kHgFirstDequant;
    constexpr int rstride = tens ? kFp8TensorRowBytes : kFp8RowBytes;  // gathered rows, 4 per group
    auto raw_row = [&](uint32_t stage, int slot) -> uint32_t {
      return stage + uint32_t((slot >> 2) * kHgGroup + (slot & 3) * rstride);
    };
    // Jobs are placed so that every access phase of a warp (8 lanes for 16-byte accesses, 16 for
    // 8-byte ones) meets distinct bank groups. Gathered rows sit four to a 128-byte aligned group
    // at a 656- or 576-byte pitch, so a slot's bank offset is 16 (slot & 3) or 64 (slot & 1) bytes.
    // Latent jobs: bytes [16ch, 16ch+16) of a slot, two per thread (k = 0, 1).
    //  fp8_ds: slot lslot, ch = lch + k. A phase takes four slots whose slot & 3 and
    //  (slot & 7) >> 1 both differ ({0,3,5,6} or {1,2,4,7}, + 8), each with two chunks 64 bytes
    //  apart. The lanes of the upper chunk (hi) store their two 16-byte halves in the other
    //  order, so the swizzled K-tile stores stay distinct as well. Both chunks of a thread lie in
    //  one 128-dim block: one scale load.
    //  per-tensor: slot lslot + 8k, ch = lch. A phase takes two slots of opposite parity, each
    //  with four consecutive chunks.
    // RoPE jobs: dims [8rc, 8rc+8) of slot 16q + rslot, q = rq0 + k for k = 0, 1, placed the same
    // way for their loads (16 or 8 bytes) and their stores into the 64-byte swizzled RoPE block.
    int lslot, lch, hi = 0, rslot, rc;
    if constexpr (tens) {
      lslot = 2 * (lane >> 3) + ((lane >> 2) & 1);
      lch = 4 * (dtid >> 5) + (lane & 3);
      rslot = 2 * ((dtid >> 4) & 7) + ((dtid >> 2) & 1);
      rc = (dtid & 3) + 4 * ((dtid >> 3) & 1);
    } else {
      const int dw = dtid >> 5, ph = lane >> 3, jj = lane & 3;
      hi = (lane >> 2) & 1;
      lslot = 8 * (ph >> 1) + (((jj << 1) | (__popc(jj) & 1)) ^ (ph & 1));
      lch = 8 * (dw >> 1) + 2 * (dw & 1) + 4 * hi;
      rslot = dtid & 15;
      rc = ((dtid >> 4) & 3) + 4 * (((dtid >> 2) ^ (dtid >> 6)) & 1);
    }
    const int rq0 = 2 * (dtid >> 7);
    for (int i = 0; i < ntiles && ok; ++i) {
      const int b = i & 1;
      const uint32_t kt = sb + uint32_t(kHgOffK) + uint32_t(b * kHgKLat);
      uint4 rv0 = make_uint4(0, 0, 0, 0), rv1 = rv0;  // (two names keep them in registers)
#pragma unroll 1
      for (int q = 0; q < 4 && ok; ++q) {
        const int u = 4 * i + q, st = u % kHgRawStages;
        if (!mbar_wait(bar(H_RAW_FULL + st), (u / kHgRawStages) & 1)) { ok = false; break; }
        // convert the stage's codes into registers first: the raw stage goes back to the
        // producers at once, and only the stores wait for PV(i-2) to release the K rows
        const uint32_t raw = sb + uint32_t(kHgOffRaw) + uint32_t(st * kHgRawStage);
        uint32_t o[2][8];
        const float sc = tens ? 1.f : lds_f32(raw_row(raw, lslot) + kScaleOff + 4 * (lch >> 3));
        const __half2 s2 = __float2half2_rn(sc);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int slot = tens ? lslot + 8 * k : lslot, ch = tens ? lch : lch + k;
          uint4 v = lds128(raw_row(raw, slot) + 16 * ch);
          if (hi) v = make_uint4(v.z, v.w, v.x, v.y);  // o[k][0..3] then holds the upper half
          const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint32_t lo, hi;
            e4m3x4_to_f16x4(wv[e], lo, hi);  // exact
            if constexpr (tens) {  // the scale comes later, in fp32
              o[k][2 * e] = lo;
              o[k][2 * e + 1] = hi;
            } else {  // code * scale in f16 (exact for power-of-two scales in f16's range)
              __half2 x = __hmul2(*reinterpret_cast<const __half2*>(&lo), s2);
              __half2 y = __hmul2(*reinterpret_cast<const __half2*>(&hi), s2);
              o[k][2 * e] = *reinterpret_cast<uint32_t*>(&x);
              o[k][2 * e + 1] = *reinterpret_cast<uint32_t*>(&y);
            }
          }
        }
        if ((q & ~1) == rq0) {  // this thread's RoPE chunk of the stage, kept in registers
          uint4 v;
          if constexpr (tens) {  // eight E4M3 codes -> f16 (exact; the scale comes later in fp32)
            const uint2 cw = lds64(raw_row(raw, rslot) + kLatent + 8 * rc);
            uint32_t hh[4];
            e4m3x4_to_f16x4(cw.x, hh[0], hh[1]);
            e4m3x4_to_f16x4(cw.y, hh[2], hh[3]);
            v = make_uint4(hh[0], hh[1], hh[2], hh[3]);
          } else {  // bf16 RoPE -> f16
            const uint4 x = lds128(raw_row(raw, rslot) + kRopeOffFp8 + 16 * rc);
            v = make_uint4(bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y), bf16x2_to_f16x2(x.z),
                           bf16x2_to_f16x2(x.w));
          }
          if (q & 1)
            rv1 = v;
          else
            rv0 = v;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(H_RAW_EMPTY + st));
        // rows [16q, 16q+16) of the K buffer are free once that chunk of PV(i-2) is done
        if (i >= 2 && !mbar_wait(bar(H_K_FREE + 4 * b + q), ((i - 2) >> 1) & 1)) { ok = false; break; }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int slot = tens ? lslot + 8 * k : lslot, ch = tens ? lch : lch + k;
          // dims [16ch, 16ch+16): block ch/4 mod 4, low rows for ch < 16, high rows after
          const int rr = kHgN * (ch >> 4) + kHgSub * q + slot;
          const uint32_t row = kt + ((ch >> 2) & 3) * kHgPairBlk + rr * 128;
          const int c0 = 2 * (ch & 3);
          const uint32_t sw = rr & 7;
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(row + (((c0 + hi) ^ sw) << 4)), "r"(o[k][0]),
                       "r"(o[k][1]), "r"(o[k][2]), "r"(o[k][3]) : "memory");
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(row + (((c0 + 1 - hi) ^ sw) << 4)),
                       "r"(o[k][4]), "r"(o[k][5]), "r"(o[k][6]), "r"(o[k][7]) : "memory");
        }
      }
      if (!ok) break;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(H_K_FULL + b));
      // the single RoPE block is free once QK of the previous tile has completed
      if (i >= 1 && !mbar_wait(bar(H_S_FULL), (i - 1) & 1)) { ok = false; break; }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int rr = kHgN * (rc >> 2) + kHgSub * (rq0 + k) + rslot, c = rc & 3;
        const uint32_t dst = sb + uint32_t(kHgOffRope) + rr * 64 + ((c ^ ((rr >> 1) & 3)) << 4);
        const uint4 v = k ? rv1 : rv0;
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                     : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(H_ROPE_FULL));
    }
    // all K tiles are dequantised: the split merge, if one follows, may start launching
    if (dtid == 0) pdl_trigger();
  }
  // ------------------------------------------------------------------ softmax + epilogue
  else {
    const int half = warp >> 1;  // 0: lanes 0-63 (low dims), 1: lanes 64-127 (high dims)
    const int pr = warp & 1;     // head pair: warps pr (low) and pr + 2 (high)
    const int hl = 32 * pr + lane;
    const int h = h0 + hl;
    const uint32_t lrow = tm + (uint32_t(32 * warp) << 16);
    const uint64_t* meta = reinterpret_cast<const uint64_t*>(sm + kHgOffMeta);  // 64 slot bits per tile
    const uint32_t xmine = sb + uint32_t(kHgOffXs) + uint32_t(32 * warp + lane) * kHgXRow;
    const uint32_t xpart = sb + uint32_t(kHgOffXs) + uint32_t(32 * (warp ^ 2) + lane) * kHgXRow;
    const uint32_t mmine = sb + uint32_t(kHgOffXm) + uint32_t(32 * warp + lane) * 4;
    const uint32_t mpart = sb + uint32_t(kHgOffXm) + uint32_t(32 * (warp ^ 2) + lane) * 4;
    const int bar_x = 1 + pr;                     // both warps of the pair have written
    const int bar_mine = 3 + 2 * pr + half;       // the partner has read my row
    const int bar_part = 3 + 2 * pr + (half ^ 1); // I have read the partner's row
    const int bar_max = 7 + pr;                   // both maxima are written
    const int bar_x2 = 9 + pr;                    // both second halves are written
    float m = -CUDART_INF_F, l = 0.f;
    bool good = true;
    // the scores' factors: sm_scale * log2(e) times the q normaliser of my row and of the
    // partner's row (my partial and the partner's partial of the same head)
    const float c2m = c2 * lds_f32(mmine), c2p = c2 * lds_f32(mpart);

    // rescale this thread's O lane (256 columns) by a; PV of the previous tile is complete.
    // The TMEM loads and stores are warp-wide: the whole warp calls this when any lane
    // needs it.
    auto correct_o = [&](float a) {
#pragma unroll 1
      for (int k = 0; k < 16; ++k) {
        uint32_t v[16];
        tc::ld16(lrow + kHgTmO + 16 * k, v);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * a);
        tc::st16(lrow + kHgTmO + 16 * k, v);
      }
      tc::wait_st();
    };

    bool loop_ok = true;
    for (int i = 0; i < ntiles; ++i) {
      // my partial scores of all 64 slots: columns 64 * half of the score block
      float v[64];
      const bool got = good && mbar_wait(bar(H_S_FULL), i & 1);
      if (got) {
        tc::fence_after();
        uint32_t w0[32], w1[32];
        tc::ld32(lrow + kHgTmS + 64 * half, w0);
        tc::ld32(lrow + kHgTmS + 64 * half + 32, w1);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          v[e] = __uint_as_float(w0[e]);
          v[32 + e] = __uint_as_float(w1[e]);
        }
        tc::fence_before();
      } else {
#pragma unroll
        for (int e = 0; e < 64; ++e) v[e] = 0.f;
      }
      __syncwarp();
      if (lane == 0 && got) mbar_arrive(bar(H_S_FREE));
      // the low warp finishes slots 0-31 and sends its partials of slots 32-63; the high warp
      // the other way round (selects keep the arrays in registers)
      float own[32], send[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        own[e] = half ? v[32 + e] : v[e];
        send[e] = half ? v[e] : v[32 + e];
      }
      // the partner's partials of my 32 slots, in two rounds of 16 through one row each
      if (i > 0) named_bar(bar_mine, 64);  // the partner has read my previous row
#pragma unroll
      for (int k = 0; k < 4; ++k)
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(xmine + 16 * k), "r"(__float_as_uint(send[4 * k])),
                     "r"(__float_as_uint(send[4 * k + 1])), "r"(__float_as_uint(send[4 * k + 2])),
                     "r"(__float_as_uint(send[4 * k + 3])) : "memory");
      if (!named_bar_and(bar_x, 64, got)) {
        loop_ok = false;
        break;
      }
      float x[32];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 xv = lds128(xpart + 16 * k);
        x[4 * k] = __uint_as_float(xv.x); x[4 * k + 1] = __uint_as_float(xv.y);
        x[4 * k + 2] = __uint_as_float(xv.z); x[4 * k + 3] = __uint_as_float(xv.w);
      }
      named_bar_arrive(bar_part, 64);
      named_bar(bar_mine, 64);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(xmine + 16 * k),
                     "r"(__float_as_uint(send[16 + 4 * k])), "r"(__float_as_uint(send[16 + 4 * k + 1])),
                     "r"(__float_as_uint(send[16 + 4 * k + 2])), "r"(__float_as_uint(send[16 + 4 * k + 3]))
                     : "memory");
      named_bar(bar_x2, 64);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 xv = lds128(xpart + 16 * k);
        x[16 + 4 * k] = __uint_as_float(xv.x); x[16 + 4 * k + 1] = __uint_as_float(xv.y);
        x[16 + 4 * k + 2] = __uint_as_float(xv.z); x[16 + 4 * k + 3] = __uint_as_float(xv.w);
      }
      const uint32_t msk = uint32_t(meta[i % kHgMetaRing] >> (32 * half));
      float s[32];
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float sv = ((msk >> j) & 1u) ? fmaf(own[j], c2m, x[j] * c2p) : -CUDART_INF_F;
        s[j] = sv;
        mx = fmaxf(mx, sv);
      }
      named_bar_arrive(bar_part, 64);
      // both warps of the pair take the max over all 64 slots
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(mmine), "f"(mx) : "memory");
      named_bar(bar_max, 64);
      mx = fmaxf(mx, lds_f32(mpart));
      float a = 1.f;
      const float mn = fmaxf(m, mx);
      if (m == -CUDART_INF_F ? mn != -CUDART_INF_F : mn > m + kHgRescaleThreshold) {
        a = exp2f(m - mn);  // 0 when m was -inf
        m = mn;
      }
      const float base = m == -CUDART_INF_F ? 0.f : m;
      float sum = 0.f;
      uint32_t pw2[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float p0 = exp2f(s[2 * j] - base), p1 = exp2f(s[2 * j + 1] - base);
        sum += p0 + p1;
        pw2[j] = pack_f16x2(p0, p1);
      }
      l = l * a + sum;
      // the P block and O are free once PV of the previous tile is complete
      if (i >= 1 && !mbar_wait(bar(H_PV_DONE), (i - 1) & 1)) good = false;
      tc::fence_after();
      if (good && i > 0 && __any_sync(0xffffffffu, a != 1.f)) correct_o(a);
      if (good) {
        const uint32_t prow = sb + uint32_t(kHgOffP) + uint32_t(kHgPBlk) + uint32_t(hl) * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = 4 * half + k;
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(prow + ((c ^ (hl & 7)) << 4)),
                       "r"(pw2[4 * k]), "r"(pw2[4 * k + 1]), "r"(pw2[4 * k + 2]), "r"(pw2[4 * k + 3])
                       : "memory");
        }
        fence_proxy_async_smem();  // read by the tensor core
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0 && good) mbar_arrive(bar(H_P_READY));
    }

    // ---- epilogue: both row halves' sums, final row factor, then O lane -> output
    ok = loop_ok;
    if (ok) {
      if (ntiles > 0) named_bar(bar_mine, 64);  // the partner has read my last row
      bool fin = good;
      if (fin && ntiles > 0) {
        fin = mbar_wait(bar(H_PV_DONE), (ntiles - 1) & 1);
        tc::fence_after();
      }
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(xmine), "f"(l) : "memory");
      ok = named_bar_and(bar_x, 64, fin);
      if (ok) l += lds_f32(xpart);  // my half's sum + the other half's: same value in both warps
    }
    if (ok) {
      const int S = p.num_splits;
      const bool real = hl < gheads;
      const float lse0 = l > 0.f ? (m + log2f(l)) * kLn2 : -CUDART_INF_F;
      float lse_out = lse0;
      float f = l > 0.f ? (tens ? p.kv_scale : 1.f) / l : 0.f;
      if (S == 1 && p.sink && real) {
        const float sg = __ldg(p.sink + h);
        lse_out = fmaxf(lse0, sg) + log1pf(expf(-fabsf(lse0 - sg)));
        f *= expf(lse0 - lse_out);
      }
      if (real && half == 0) {
        if (S == 1) {
          if (p.lse) p.lse[int64_t(t) * p.H + h] = lse_out;
        } else if (!p.cluster_merge) {
          p.lse_part[(int64_t(t) * S + split) * p.H + h] = lse0;
        }
      }
      cm_f = f;
      cm_lse = lse0;
      const int64_t orow_g = S == 1 ? int64_t(t) * p.H + h : (int64_t(t) * S + split) * p.H + h;
      // four 16-column loads in flight per wait; every lane loads, only real heads store
      // (with the cluster merge the rows go out after the cluster barrier, at the teardown)
#pragma unroll 1
      for (int k4 = 0; k4 < 4 && !p.cluster_merge; ++k4) {
        uint32_t v4[4][16];
        if (ntiles > 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j) tc::ld16(lrow + kHgTmO + 64 * k4 + 16 * j, v4[j]);
          tc::wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 16; ++e) v4[j][e] = 0u;
        }
        if (!real) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t* vv = v4[j];
          const int col = 256 * half + 64 * k4 + 16 * j;
          if (S == 1) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow_g * kLatent + col);
            uint32_t o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o[e] = pack_bf16x2(__uint_as_float(vv[2 * e]) * f, __uint_as_float(vv[2 * e + 1]) * f);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
          } else {  // f16 partial: a convex combination of keys, so within f16's range
            uint32_t o[8];
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o[e] = pack_f16x2(__uint_as_float(vv[2 * e]) * f, __uint_as_float(vv[2 * e + 1]) * f);
            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__half*>(p.o_part) + orow_g * kLatent + col);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  if (!ok && lane == 0) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
  // the softmax threads' final row factors, for the warps that help push the rows (the P
  // block is free: every MMA has completed)
  const uint32_t cmf = sb + uint32_t(kHgOffP);
  if (p.cluster_merge && warp < 4) asm volatile("st.shared.f32 [%0], %1;" ::"r"(cmf + 4 * tid), "f"(cm_f) : "memory");
  tc::fence_before();
  __syncthreads();
  if (p.cluster_merge) {
    // Split merge inside the cluster (SGLang PR #24692 "关键文件": _merge_partial_attn, then
    // _apply_attn_sink). Rank r merges heads [r hp, r hp + hp) of the group.
    //  1. Cluster barrier: every CTA's pipeline is done, so its K-tile area is free.
    //  2. The softmax and dequant warps store the normalised f16 partial rows (O / l), and
    //     the softmax warps the LSEs, into the shared memory of the CTA that merges the head;
    //     remote stores do not stall.
    //  3. Cluster barrier: every row has landed. Each CTA merges from its own shared memory,
    //     and no CTA touches another's memory after this point.
    tc::cluster_arrive();
    tc::cluster_wait();
    if (warp < kHgFirstProducer) {
      // warp w reads TMEM lane quarter w % 4 (32 rows) and pushes its part w / 4 of the 16
      // 16-column chunks of each row: chunks [0, 6), [6, 11), [11, 16)
      const int qw = warp & 3, part = warp >> 2;
      const int half = qw >> 1, hl = 32 * (qw & 1) + lane;
      const uint32_t lrow = tm + (uint32_t(32 * qw) << 16);
      const bool real = hl < gheads;
      const int mr = split * mhp + hl % mhp;
      const uint32_t owner = uint32_t(hl / mhp);
      const float f = lds_f32(cmf + 4 * (32 * qw + lane));
      if (real && half == 0 && part == 0) tc::st_dsmem_f32(tc::mapa(mlse + mr * 4, owner), cm_lse);
      tc::fence_after();
      const int cb = part == 0 ? 0 : 1 + 5 * part, ce = 6 + 5 * part;
#pragma unroll 1
      for (int c = cb; c < ce; c += 2) {
        const bool two = c + 1 < ce;
        uint32_t v2[2][16];
        __syncwarp();  // the TMEM loads are warp-wide
        if (ntiles > 0) {
          tc::ld16(lrow + kHgTmO + 16 * c, v2[0]);
          if (two) tc::ld16(lrow + kHgTmO + 16 * (c + 1), v2[1]);
          tc::wait_ld();
        } else {
#pragma unroll
          for (int j = 0; j < 2; ++j)
#pragma unroll
            for (int e = 0; e < 16; ++e) v2[j][e] = 0u;
        }
        if (!real) continue;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (j == 1 && !two) break;
          uint32_t o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            o[e] = pack_f16x2(__uint_as_float(v2[j][2 * e]) * f, __uint_as_float(v2[j][2 * e + 1]) * f);
          const int c0 = 32 * half + 2 * (c + j);  // 16-byte chunk of the 1024-byte merge row
          if (owner == uint32_t(split)) {  // a head this CTA merges: its own shared memory
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(mrow_addr(mr, c0)), "r"(o[0]), "r"(o[1]),
                         "r"(o[2]), "r"(o[3]) : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(mrow_addr(mr, c0 + 1)), "r"(o[4]),
                         "r"(o[5]), "r"(o[6]), "r"(o[7]) : "memory");
          } else {
            tc::st_dsmem_v4(tc::mapa(mrow_addr(mr, c0), owner), o[0], o[1], o[2], o[3]);
            tc::st_dsmem_v4(tc::mapa(mrow_addr(mr, c0 + 1), owner), o[4], o[5], o[6], o[7]);
          }
        }
      }
    }
    tc::cluster_arrive();
    tc::cluster_wait();
    const int S = p.num_splits;
    const int hs = split * mhp, nk = max(0, min(gheads, hs + mhp) - hs);
    const uint32_t wtab = mlse + 512;  // [head - hs][8] merge weights (times the final factor)
    for (int k = tid; k < nk; k += kHgThreads) {
      float ls[kMaxClusterMerge];
      float M = -CUDART_INF_F;
#pragma unroll
      for (int s = 0; s < kMaxClusterMerge; ++s) {
        ls[s] = s < S ? lds_f32(mlse + (s * mhp + k) * 4) : -CUDART_INF_F;
        M = fmaxf(M, ls[s]);
      }
      float W = 0.f;
#pragma unroll
      for (int s = 0; s < kMaxClusterMerge; ++s) {
        ls[s] = (M == -CUDART_INF_F || ls[s] == -CUDART_INF_F) ? 0.f : expf(ls[s] - M);
        W += ls[s];
      }
      const float lse0 = W > 0.f ? M + logf(W) : -CUDART_INF_F;
      float lse = lse0, f = W > 0.f ? 1.f / W : 0.f;
      if (p.sink) {
        const float sg = __ldg(p.sink + h0 + hs + k);
        lse = fmaxf(lse0, sg) + log1pf(expf(-fabsf(lse0 - sg)));
        f *= expf(lse0 - lse);
      }
      if (p.lse) p.lse[int64_t(t) * p.H + h0 + hs + k] = lse;
#pragma unroll
      for (int s = 0; s < kMaxClusterMerge; ++s)
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(wtab + (k * kMaxClusterMerge + s) * 4), "f"(ls[s] * f)
                     : "memory");
    }
    __syncthreads();
    for (int j = tid; j < nk * 64; j += kHgThreads) {  // 8 output dims per job
      const int k = j >> 6, c = j & 63;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
      for (int s = 0; s < kMaxClusterMerge; ++s) {
        if (s >= S) break;
        const float w = lds_f32(wtab + (k * kMaxClusterMerge + s) * 4);
        const uint4 v = lds128(mrow_addr(s * mhp + k, c));
        const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&vw[e]));
          acc[2 * e] = fmaf(w, x.x, acc[2 * e]);
          acc[2 * e + 1] = fmaf(w, x.y, acc[2 * e + 1]);
        }
      }
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                            (int64_t(t) * p.H + h0 + hs + k) * kLatent + 8 * c);
      *dst = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                        pack_bf16x2(acc[6], acc[7]));
    }
  }
  if (warp == kHgMmaWarp) {
    tc::fence_after();
    tc::dealloc(tm, 512);
  }
}

}  // namespace

cudaError_t launch_decode_hg(const DecodeArgs& a, cudaStream_t s) {
  // devices (below 64) whose kernel attributes are set; concurrent first calls set them twice
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t(1) << dev) : 0;
  if (!(configured.load(std::memory_order_acquire) & bit) || !bit) {
    cudaError_t e = cudaFuncSetAttribute(decode_hg_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemHg));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_hg_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemHg));
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_release);
  }
  alignas(64) CUtensorMap map;
  alignas(64) CUtensorMap qmap;
  cudaError_t e = kv_gather_map(a, &map);
  if (e == cudaSuccess) e = q_tile_map(a, &qmap);
  if (e != cudaSuccess) return e;
  const int64_t items = a.nitems > 0 ? a.nitems : int64_t(a.T) * ((a.H + 63) / 64);
  const int64_t grid = items * a.num_splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kHgThreads);
  cfg.dynamicSmemBytes = kSmemHg;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (a.cluster_merge) {  // the splits of a (token, head group) share one cluster
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(a.num_splits);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (a.overlap_prev) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = na;
  if (a.kv_format == SMLA_KV_FP8_TENSOR) return cudaLaunchKernelEx(&cfg, decode_hg_kernel<true>, a, map, qmap);
  return cudaLaunchKernelEx(&cfg, decode_hg_kernel<false>, a, map, qmap);
}

}  // namespace smla

