// Sparse MLA decode on the 5th-generation tensor cores (tcgen05, TMEM accumulators),
// for the FP8 caches (fp8_ds: 656-byte rows with per-128 scales and bf16 RoPE; per-tensor
// FP8: 576 E4M3 codes with one scale, vLLM PR #43827) and 64..128 heads. One CTA pair
// (cluster of 2) per (query token, top-k split).
//
// What it computes is the sparse decode of vLLM PR #43477 "关键源码片段" (forward_mqa)
// with the sink and split merge of SGLang PR #24692 "关键文件": out_h = softmax over the
// selected slots of sm_scale * <q_h, k_j>, applied to v_j = k_j[0:512].
//
// Why a pair: the fp32 output of 128 heads x 512 dims fills one SM's whole tensor memory
// (512 columns). CTA c of the pair owns latent dims [256c, 256c+256) and RoPE dims
// [32c, 32c+32): it gathers only those bytes of each row, scores all 128 heads over its 288
// dims, and accumulates its 256 output dims. The two partial score rows of a head are
// summed by the CTA that owns the head (heads [64c, 64c+64)), which runs the softmax and
// sends the probabilities back, so both halves of PV use identical P.
//
// The MMAs run on f16 operands with fp32 accumulation. An E4M3 code converts to f16
// exactly in one instruction, and the block scale applies with one f16 multiply: exact for
// power-of-two scales and within 2^-11 otherwise, finer than bf16's 2^-8. q converts from
// bf16 exactly. The price is f16's range: dequantised keys and q must stay within
// +-65504 (for power-of-two block scales, a block's largest magnitude within 57344).
//
// Per CTA (416 threads):
//  * warps 8-11, producers (16 slots of every tile each): the split's index list by one
//    bulk copy, page-table entries four tiles ahead by 4-byte cp.async, then this CTA's
//    half of each valid row (256 latent bytes, the 4 scales, 32 RoPE values = 336 bytes)
//    as two bulk copies into a 3-stage ring. Bulk copies issued by one warp serialise on
//    the TMA engine; four issuing warps keep the gather near the per-SM limit.
//  * warps 0-3, dequant: e4m3 * scale -> f16, written as the swizzled K tile [64 slots x
//    288 dims]: four 128-byte-swizzled latent panels and a 64-byte-swizzled RoPE panel
//    (two buffers). The same bytes serve as B of QK (K-major) and
//    as B of PV (MN-major view of the 256 latent dims).
//  * warp 12, MMA issuer (one thread): QK = 18 x tcgen05.mma M128 N64 K16 with q (f16) as
//    the A operand in TMEM; PV = 4 x tcgen05.mma M128 N256 K16 with P from shared memory.
//    QK of tile i+1 is issued before PV of tile i, so scores are ready when softmax needs them.
//  * warps 4-7, softmax: thread h owns TMEM lane h (head h). Non-owners send their partial
//    score row to the peer (st.async into the peer's shared memory, counted by its
//    mbarrier); owners add the peer's row, mask, run a base-2 online softmax with lazy
//    rescaling (the running max moves only when it grows by more than 8, as in
//    FlashAttention-4), write P locally and into the peer, and rescale their O row in TMEM
//    when the max moved. Non-owners apply the same factor to their O row.
//  * epilogue: O * (1/l) (and the sink factor) -> bf16 out, or fp32 split partials.
// Every wait is bounded in time; a wait that gives up sets SMLA_DEVERR_TIMEOUT and the CTA
// falls through to the teardown, which both CTAs of the pair reach.
#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

// Optional timeline of the first cluster's pipeline events (compiled in with -DSMLA_TRACE;
// read back with smla_trace_read). Off in normal builds: the macro expands to nothing.
#ifdef SMLA_TRACE
__device__ unsigned long long g_trace[2][64][12];
__device__ unsigned long long g_span[4096][2];
#define TRACE(ev, tile)                                                                    \
  do {                                                                                     \
    if (blockIdx.x < 2 && (tile) < 64) g_trace[blockIdx.x][(tile)][(ev)] = globaltimer_ns(); \
  } while (0)
#else
#define TRACE(ev, tile) \
  do {                  \
  } while (0)
#endif

namespace smla {
namespace {

constexpr int kProducersTc = 4;   // warps 8..11; bulk copies from one warp serialise
constexpr int kMmaWarp = 8 + kProducersTc;
constexpr int kThreadsTc = 32 * (kMmaWarp + 1);
constexpr int kN = 64;             // slots per tile
constexpr int kStagesTc = 3;       // raw half-row ring
constexpr int kHalfRow = 336;      // 256 latent + 16 scales + 64 RoPE bytes
constexpr int kPanel = kN * 128;   // one 64-dim 128-byte-swizzled panel of a tile: 8 KB
constexpr int kRopePanel = kN * 64;  // the CTA's 32 RoPE dims, 64-byte swizzle: 4 KB
constexpr int kKtile = 4 * kPanel + kRopePanel;  // 4 latent panels + the RoPE panel
constexpr int kPtile = 128 * 128;  // P [128 heads x 64 slots] f16
constexpr int kXsRow = 272;        // 64 fp32 + padding (conflict-free row reads)
constexpr int kXs = 64 * kXsRow;
constexpr int kMetaRing = 8;
constexpr int kAheadTc = 4;        // page-table look-ahead (tiles)
constexpr int kPageRingTc = 6;
constexpr int kIdxAhead = 8;       // index look-ahead (tiles)
constexpr int kIdxRing = 16;
constexpr float kRescaleThreshold = 8.f;  // log2 units

// TMEM columns (512 allocated)
constexpr uint32_t kTmO = 0;    // O_c [128 x 256] fp32
constexpr uint32_t kTmQ = 256;  // q_c [128 x 288] f16: 144 columns
constexpr uint32_t kTmS = 448;  // S [128 x 64] fp32

constexpr size_t kOffKtile = 0;
constexpr size_t kOffPtile = kOffKtile + 2 * size_t(kKtile);
constexpr size_t kOffRaw = kOffPtile + 2 * size_t(kPtile);
constexpr size_t kOffXs = kOffRaw + size_t(kStagesTc) * kN * kHalfRow;
constexpr size_t kOffIdx = kOffXs + 2 * size_t(kXs);
constexpr size_t kOffPages = kOffIdx + size_t(kIdxRing) * kN * 4;
constexpr size_t kOffMeta = kOffPages + size_t(kPageRingTc) * kN * 4;
constexpr size_t kOffAlpha = kOffMeta + kMetaRing * 8;
constexpr size_t kOffFin = kOffAlpha + 2 * 64 * 4;
constexpr size_t kOffPhys = kOffFin + 64 * 4;
constexpr size_t kOffTmem = kOffPhys + 64 * 8;
constexpr size_t kOffBars = kOffTmem + 16;
enum {
  B_RAW_FULL = 0, B_RAW_EMPTY = 3, B_K_FULL = 6, B_K_FREE = 8, B_S_FULL = 10, B_S_FREE = 11,
  B_XS_FULL = 12, B_RP_FULL = 14, B_P_READY = 16, B_FIN = 18, B_IDX = 19, B_Q = 20, B_COUNT = 21
};
constexpr size_t kSmemTc = kOffBars + B_COUNT * 8 + 1024;  // + alignment slack
static_assert(kSmemTc <= 232448, "shared memory budget");
// q staging at start-up: 128 rows of 576 bytes (+16 for conflict-free 16-byte reads) in the
// K-tile and P-tile area, which the pipeline first writes after the start-up barrier
constexpr uint32_t kQRow = 592;
static_assert(128 * kQRow <= kOffRaw, "q staging fits below the raw ring");

__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// TENS: per-tensor FP8 rows (576 B, one scale) instead of fp8_ds rows (656 B, 4 block
// scales).
template <bool TENS>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreadsTc, 1)
    decode_tc_kernel(const DecodeArgs p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  auto bar = [&](int k) -> uint32_t { return sb + uint32_t(kOffBars) + 8u * k; };
  const uint32_t crank = tc::cluster_rank();
  const uint32_t peer = crank ^ 1u;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

#ifdef SMLA_TRACE
  if (threadIdx.x == 0 && blockIdx.x < 4096) g_span[blockIdx.x][0] = globaltimer_ns();
#endif
  // Per-tensor FP8 codes go into the K tile unscaled (exact in f16) and kv_scale is
  // applied in fp32 to the scores (bmm1_scale = sm_scale * kv_scale) and to O (bmm2_scale =
  // kv_scale), the scale algebra of vLLM PR #43827 "关键源码片段".
  constexpr bool tens = TENS;
  const float c2 = tens ? p.c2 * p.kv_scale : p.c2;
  const int item = blockIdx.x >> 1;
  const int split = item % p.num_splits;
  const int t = item / p.num_splits;
  const int r = p.req_id ? __ldg(p.req_id + t) : t / p.next_n;
  const bool req_ok = r >= 0 && r < p.B;
  const int32_t* pt_row = p.page_table + int64_t(req_ok ? r : 0) * p.stride;
  const int32_t* idx_row = p.topk + int64_t(t) * p.K;
  const int j0 = split * p.split_len;
  const int j1 = min(p.K, j0 + p.split_len);
  const int nidx = max(0, j1 - j0);
  const int ntiles = req_ok ? (nidx + kN - 1) / kN : 0;

  // Producer lanes (warps 8..11, slots [16 pw, 16 pw + 16) of every tile) fetch their slot's
  // index kIdxAhead tiles ahead and, once that has landed, its page-table entry kAheadTc
  // tiles ahead, both by 4-byte cp.async. Every ring step commits one group {index of tile
  // i+kIdxAhead, page entry of tile i+kAheadTc}; the steps before tile 0 only prime the two
  // rings, and they run first thing, so the first dependent round trips overlap the set-up.
  const bool producer = warp >= 8 && warp < kMmaWarp;
  const int pw = warp - 8;
  const bool act = lane < kN / kProducersTc;
  const int myslot = (kN / kProducersTc) * pw + lane;
  int32_t* sidx = reinterpret_cast<int32_t*>(sm + kOffIdx);    // index ring
  int32_t* spage = reinterpret_cast<int32_t*>(sm + kOffPages);  // page-table entry ring
  auto in_split = [&](int tile) { return act && tile < ntiles && tile * kN + myslot < nidx; };
  auto idx_of = [&](int tile) -> int32_t {
    return in_split(tile) ? sidx[(tile % kIdxRing) * kN + myslot] : -1;
  };
  auto ring_step = [&](int i) {
    cp_async_wait<kIdxAhead - kAheadTc - 1>();  // the group that fetched index i+kAheadTc
    const int tp = i + kAheadTc;
    if (tp >= 0) {
      const int32_t idx = idx_of(tp);
      if (idx >= 0 && (idx >> p.log2_page) < p.stride)
        cp_async4(smem_u32(spage + (tp % kPageRingTc) * kN + myslot), pt_row + (idx >> p.log2_page));
    }
    const int ti = i + kIdxAhead;
    if (in_split(ti))
      cp_async4(smem_u32(sidx + (ti % kIdxRing) * kN + myslot), idx_row + j0 + ti * kN + myslot);
    cp_async_commit();
  };
  if (producer)
    for (int i = -kIdxAhead; i < 0; ++i) ring_step(i);

  // ------------------------------------------------------------------ set-up
  {
    uint4* z = reinterpret_cast<uint4*>(sm + kOffRaw);
    for (int k = tid; k < kStagesTc * kN * kHalfRow / 16; k += kThreadsTc) z[k] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
      for (int s = 0; s < kStagesTc; ++s) {
        mbar_init(bar(B_RAW_FULL + s), kProducersTc);  // one expect_tx arrival per producer warp
        mbar_init(bar(B_RAW_EMPTY + s), 4);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(bar(B_K_FULL + b), 4);
        mbar_init(bar(B_K_FREE + b), 1);
        mbar_init(bar(B_XS_FULL + b), 1);
        mbar_init(bar(B_RP_FULL + b), 1);
        mbar_init(bar(B_P_READY + b), 4);
      }
      mbar_init(bar(B_S_FULL), 1);
      mbar_init(bar(B_S_FREE), 4);
      mbar_init(bar(B_FIN), 1);
      mbar_init(bar(B_IDX), 1);
      mbar_init(bar(B_Q), 1);
      tc::fence_mbarrier_init_cluster();
      if (!req_ok && crank == 0 && split == 0) atomicOr(p.err, SMLA_DEVERR_INDEX);
    }
    if (warp == kMmaWarp) tc::alloc(sb + uint32_t(kOffTmem), 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
  }
  const uint32_t tm = *reinterpret_cast<volatile uint32_t*>(sm + kOffTmem);

  // softmax warps place q_c in TMEM (A operand of QK): lane h = head h, 144 columns. The
  // 576 bytes of each head's row this CTA needs (latent dims [256c, 256c+256), RoPE dims
  // [32c, 32c+32)) arrive by two bulk copies into the (still idle) K/P-tile area, one
  // round trip for all heads, then go from shared memory into TMEM.
  if (warp >= 4 && warp < 8) {
    const int q4 = warp & 3;
    const int h = 32 * q4 + lane;
    const uint32_t lrow = tm + (uint32_t(32 * q4) << 16) + kTmQ;
    const int nheads = req_ok ? min(p.H, 128) : 0;
    const bool have = h < nheads;
    const uint32_t qs = sb + uint32_t(kOffKtile) + uint32_t(h) * kQRow;
    if (h == 0 && nheads > 0) mbar_arrive_expect_tx(bar(B_Q), uint32_t(nheads) * 576u);
    if (have) {
      const uint8_t* qrow = reinterpret_cast<const uint8_t*>(p.q) + (int64_t(t) * p.H + h) * (2 * kDim);
      bulk_g2s(qs, qrow + 512 * crank, 512, bar(B_Q));
      bulk_g2s(qs + 512, qrow + 1024 + 64 * crank, 64, bar(B_Q));
    }
    const bool got = nheads == 0 || mbar_wait(bar(B_Q), 0);
    if (!got && lane == 0) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
#pragma unroll 1
    for (int ch = 0; ch < 9; ++ch) {
      uint32_t wv[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (have && got) v = lds128(qs + 16 * (4 * ch + k));
        // the MMAs run on f16 operands: bf16 -> f16 (exact within f16's range)
        wv[4 * k] = bf16x2_to_f16x2(v.x); wv[4 * k + 1] = bf16x2_to_f16x2(v.y);
        wv[4 * k + 2] = bf16x2_to_f16x2(v.z); wv[4 * k + 3] = bf16x2_to_f16x2(v.w);
      }
      tc::st16(lrow + 16 * ch, wv);
    }
    tc::wait_st();
  }
  if (tid == 0) mbar_arrive_expect_tx(bar(B_FIN), 64 * 4);  // peer's final row factors
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  tc::cluster_arrive();  // the peer's barriers exist before any remote store lands
  tc::cluster_wait();

  bool ok = true;
  // ------------------------------------------------------------------ producer
  if (producer) {
    uint16_t* meta = reinterpret_cast<uint16_t*>(sm + kOffMeta);
    int issued = 0;
    for (int i = 0; i < ntiles && ok; ++i) {
      ring_step(i);
      const int st = i % kStagesTc;
      if (!mbar_wait(bar(B_RAW_EMPTY + st), ((i / kStagesTc) & 1) ^ 1)) {
        ok = false;
        break;
      }
      const int32_t idx = idx_of(i);
      int64_t phys = -1;
      if (idx != -1) {
        if (idx < 0 || (idx >> p.log2_page) >= p.stride) {
          atomicOr(p.err, SMLA_DEVERR_INDEX);
        } else {
          const int32_t pg = spage[(i % kPageRingTc) * kN + myslot];
          if (pg < 0 || pg >= p.num_pages)
            atomicOr(p.err, SMLA_DEVERR_PAGE);
          else
            phys = (int64_t(pg) << p.log2_page) + (idx & ((1 << p.log2_page) - 1));
        }
      }
      if (lane == 0) TRACE(0, i);
      const uint32_t vm = __ballot_sync(0xffffffffu, phys >= 0);
      if (lane == 0) {
        meta[(i % kMetaRing) * kProducersTc + pw] = uint16_t(vm);
        mbar_arrive_expect_tx(bar(B_RAW_FULL + st), uint32_t(__popc(vm)) * (tens ? 288u : uint32_t(kHalfRow)));
      }
      __syncwarp();
      if (tens && phys >= 0) {
        // latent [256c, 256c+256) and the RoPE codes [32c, 32c+32)
        const uint8_t* src = p.kv + phys * kFp8TensorRowBytes;
        const uint32_t dst = sb + uint32_t(kOffRaw) + uint32_t((st * kN + myslot) * kHalfRow);
        bulk_g2s(dst, src + 256 * crank, 256, bar(B_RAW_FULL + st));
        bulk_g2s(dst + 256, src + kLatent + 32 * crank, 32, bar(B_RAW_FULL + st));
      } else if (phys >= 0) {
        const uint8_t* src = p.kv + phys * kFp8RowBytes;
        const uint32_t dst = sb + uint32_t(kOffRaw) + uint32_t((st * kN + myslot) * kHalfRow);
        if (crank == 0) {
          bulk_g2s(dst, src, 256, bar(B_RAW_FULL + st));              // latent [0, 256)
          bulk_g2s(dst + 256, src + 512, 80, bar(B_RAW_FULL + st));   // scales + RoPE [0, 32)
        } else {
          bulk_g2s(dst, src + 256, 272, bar(B_RAW_FULL + st));        // latent [256, 512) + scales
          bulk_g2s(dst + 272, src + 592, 64, bar(B_RAW_FULL + st));   // RoPE [32, 64)
        }
      }
      issued = i + 1;
    }
    cp_async_wait<0>();
    for (int i = max(0, issued - kStagesTc); i < issued; ++i)
      if (!mbar_wait(bar(B_RAW_FULL + i % kStagesTc), (i / kStagesTc) & 1)) break;
  }
  // ------------------------------------------------------------------ MMA issuer
  else if (warp == kMmaWarp) {
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t kIdQK = tc::idesc_f16_f32(128, kN, false, false);
      constexpr uint32_t kIdPV = tc::idesc_f16_f32(128, 256, false, true);
      auto qk = [&](int i) -> bool {
        const int b = i & 1;
        if (!mbar_wait(bar(B_K_FULL + b), (i >> 1) & 1)) return false;
        if (i >= 1 && !mbar_wait(bar(B_S_FREE), (i - 1) & 1)) return false;
        tc::fence_after();
        const uint32_t kt = sb + uint32_t(kOffKtile) + uint32_t(b * kKtile);
#pragma unroll
        for (int s = 0; s < 18; ++s) {
          const uint64_t bdesc = s < 16 ? tc::sdesc_sw128(kt + (s >> 2) * kPanel + (s & 3) * 32, 16, 1024)
                                        : tc::sdesc_sw64(kt + 4 * kPanel + (s - 16) * 32, 16, 512);
          tc::mma_ts(tm + kTmS, tm + kTmQ + 8 * s, bdesc, kIdQK, s > 0);
        }
        tc::commit(bar(B_S_FULL));
        TRACE(3, i);
        return true;
      };
      auto pv = [&](int i) -> bool {
        const int b = i & 1;
        if (!mbar_wait(bar(B_P_READY + b), (i >> 1) & 1)) return false;
        tc::fence_after();
        const uint32_t pt = sb + uint32_t(kOffPtile) + uint32_t(b * kPtile);
        const uint32_t kt = sb + uint32_t(kOffKtile) + uint32_t(b * kKtile);
#pragma unroll
        for (int s = 0; s < 4; ++s)
          tc::mma_ss(tm + kTmO, tc::sdesc_sw128(pt + 32 * s, 16, 1024),
                     tc::sdesc_sw128(kt + 2048 * s, kPanel, 1024), kIdPV, (i > 0 || s > 0));
        tc::commit(bar(B_K_FREE + b));
        TRACE(4, i);
        return true;
      };
      ok = qk(0);
      for (int i = 0; i < ntiles && ok; ++i) {
        if (i + 1 < ntiles) ok = qk(i + 1);
        if (ok) ok = pv(i);
      }
      // MMAs still in flight must finish before the tensor memory is released
      const int last = ntiles - 1;
      mbar_wait(bar(B_K_FREE + (last & 1)), (last >> 1) & 1);
    }
    __syncwarp();
  }
  // ------------------------------------------------------------------ dequant
  else if (warp < 4) {
    for (int i = 0; i < ntiles && ok; ++i) {
      const int st = i % kStagesTc, b = i & 1;
      if (!mbar_wait(bar(B_RAW_FULL + st), (i / kStagesTc) & 1)) { ok = false; break; }
      if (tid == 0) TRACE(1, i);
      if (i >= 2 && !mbar_wait(bar(B_K_FREE + b), ((i - 2) >> 1) & 1)) { ok = false; break; }
      if (tid == 0) TRACE(2, i);
      const uint32_t raw = sb + uint32_t(kOffRaw) + uint32_t(st * kN * kHalfRow);
      const uint32_t kt = sb + uint32_t(kOffKtile) + uint32_t(b * kKtile);
#pragma unroll 4
      for (int k = 0; k < 8; ++k) {
        const int id = tid + 128 * k;
        const int ch = id >> 6, slot = id & 63;  // 16 latent bytes [16ch, 16ch+16) of slot
        const uint32_t rrow = raw + slot * kHalfRow;
        const uint4 v = lds128(rrow + 16 * ch);
        const float sc = tens ? 1.f : lds_f32(rrow + 256 + 4 * (2 * crank + (ch >> 3)));
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        uint32_t o[8];
        const __half2 s2 = __float2half2_rn(sc);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t lo, hi;
          e4m3x4_to_f16x4(wv[q], lo, hi);  // exact
          if constexpr (tens) {  // the scale comes later, in fp32
            o[2 * q] = lo;
            o[2 * q + 1] = hi;
          } else {  // code * scale in f16 (exact for power-of-two scales in f16's range)
            __half2 a = __hmul2(*reinterpret_cast<const __half2*>(&lo), s2);
            __half2 b = __hmul2(*reinterpret_cast<const __half2*>(&hi), s2);
            o[2 * q] = *reinterpret_cast<uint32_t*>(&a);
            o[2 * q + 1] = *reinterpret_cast<uint32_t*>(&b);
          }
        }
        const uint32_t row = kt + (ch >> 2) * kPanel + slot * 128;
        const int c0 = 2 * (ch & 3);
        const uint32_t sw = slot & 7;
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(row + ((c0 ^ sw) << 4)), "r"(o[0]),
                     "r"(o[1]), "r"(o[2]), "r"(o[3]) : "memory");
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(row + (((c0 + 1) ^ sw) << 4)), "r"(o[4]),
                     "r"(o[5]), "r"(o[6]), "r"(o[7]) : "memory");
      }
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int id = tid + 128 * k;
        const int rc = id >> 6, slot = id & 63;  // RoPE dims [8rc, 8rc+8) of slot
        uint4 v;
        if constexpr (tens) {  // eight E4M3 codes -> f16 (exact; the scale comes later in fp32)
          const uint2 cw = lds64(raw + slot * kHalfRow + 256 + 8 * rc);
          uint32_t h[4];
          e4m3x4_to_f16x4(cw.x, h[0], h[1]);
          e4m3x4_to_f16x4(cw.y, h[2], h[3]);
          v = make_uint4(h[0], h[1], h[2], h[3]);
        } else {  // bf16 RoPE -> f16
          const uint4 r = lds128(raw + slot * kHalfRow + 272 + 16 * rc);
          v = make_uint4(bf16x2_to_f16x2(r.x), bf16x2_to_f16x2(r.y), bf16x2_to_f16x2(r.z),
                         bf16x2_to_f16x2(r.w));
        }
        const uint32_t dst = kt + 4 * kPanel + slot * 64 + ((rc ^ ((slot >> 1) & 3)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v.x), "r"(v.y), "r"(v.z),
                     "r"(v.w) : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_K_FULL + b));
        mbar_arrive(bar(B_RAW_EMPTY + st));
      }
    }
    // all K tiles are dequantised: the split merge, if one follows, may start launching
    if (tid == 0) pdl_trigger();
  }
  // ------------------------------------------------------------------ softmax + epilogue
  else {
    const int q4 = warp & 3;
    const int h = 32 * q4 + lane;
    const bool owner = (h >> 6) == int(crank);
    const int orow = h - 64 * int(crank);  // row in my exchange buffers (owner)
    const int prow = h - 64 * int(peer);   // row in the peer's exchange buffers (non-owner)
    const uint32_t lrow = tm + (uint32_t(32 * q4) << 16);
    const uint64_t* meta = reinterpret_cast<const uint64_t*>(sm + kOffMeta);  // 4 x 16 slot bits per tile
    const bool xs_armer = owner && lane == 0 && (q4 & 1) == 0;       // first owner thread
    const bool rp_armer = !owner && lane == 0 && (q4 & 1) == 0;      // first non-owner thread
    float m = -CUDART_INF_F, l = 0.f;

    // rescale this thread's O row (256 columns) by a; waits for the previous PV first. The
    // TMEM loads and stores are warp-wide: the whole warp calls this when any lane needs
    // it (a = 1 leaves a row unchanged).
    auto correct_o = [&](int i, float a) -> bool {
      if (i > 0 && !mbar_wait(bar(B_K_FREE + ((i - 1) & 1)), ((i - 1) >> 1) & 1)) return false;
      tc::fence_after();
#pragma unroll 1
      for (int k = 0; k < 16; ++k) {
        uint32_t v[16];
        tc::ld16(lrow + kTmO + 16 * k, v);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = f2u(__uint_as_float(v[e]) * a);
        tc::st16(lrow + kTmO + 16 * k, v);
      }
      tc::wait_st();
      return true;
    };

    for (int i = 0; i < ntiles && ok; ++i) {
      const int b = i & 1;
      if (xs_armer) mbar_arrive_expect_tx(bar(B_XS_FULL + b), 64 * 256);
      if (rp_armer) mbar_arrive_expect_tx(bar(B_RP_FULL + b), 64 * 128 + 64 * 4);
      if (!mbar_wait(bar(B_S_FULL), i & 1)) { ok = false; break; }
      if (lane == 0 && q4 == 0) TRACE(5, i);
      tc::fence_after();
      float s[64];
      {
        uint32_t v[64];
        tc::ld64(lrow + kTmS, v);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 64; ++e) s[e] = __uint_as_float(v[e]);
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_S_FREE));
      const uint64_t msk = meta[i % kMetaRing];

      if (!owner) {
        const uint32_t rdst = tc::mapa(sb + uint32_t(kOffXs + b * kXs + prow * kXsRow), peer);
        const uint32_t rbar = tc::mapa(bar(B_XS_FULL + b), peer);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          tc::st_async_v4(rdst + 16 * k, f2u(s[4 * k]), f2u(s[4 * k + 1]), f2u(s[4 * k + 2]),
                          f2u(s[4 * k + 3]), rbar);
        if (!mbar_wait(bar(B_RP_FULL + b), (i >> 1) & 1)) { ok = false; break; }
        if (lane == 0) TRACE(6 + (q4 & 1) * 0, i);
        fence_proxy_async_smem();  // the peer's P rows are read by the tensor core
        const float a = reinterpret_cast<const float*>(sm + kOffAlpha)[b * 64 + prow];
        if (i > 0 && __any_sync(0xffffffffu, a != 1.f) && !correct_o(i, a)) { ok = false; break; }
      } else {
        if (!mbar_wait(bar(B_XS_FULL + b), (i >> 1) & 1)) { ok = false; break; }
        if (lane == 0) TRACE(7, i);
        const uint32_t xrow = sb + uint32_t(kOffXs + b * kXs + orow * kXsRow);
        float mx = -CUDART_INF_F;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint4 x = lds128(xrow + 16 * k);
          const float xs4[4] = {__uint_as_float(x.x), __uint_as_float(x.y), __uint_as_float(x.z),
                                __uint_as_float(x.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 4 * k + e;
            const float v = ((msk >> j) & 1ull) ? (s[j] + xs4[e]) * c2 : -CUDART_INF_F;
            s[j] = v;
            mx = fmaxf(mx, v);
          }
        }
        float a = 1.f;
        const float mn = fmaxf(m, mx);
        if (m == -CUDART_INF_F ? mn != -CUDART_INF_F : mn > m + kRescaleThreshold) {
          a = exp2f(m - mn);  // 0 when m was -inf
          m = mn;
        }
        const float base = m == -CUDART_INF_F ? 0.f : m;
        float sum = 0.f;
        uint32_t pw[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float p0 = exp2f(s[2 * j] - base), p1 = exp2f(s[2 * j + 1] - base);
          sum += p0 + p1;
          pw[j] = pack_f16x2(p0, p1);
        }
        l = l * a + sum;
        const uint32_t prow_l = sb + uint32_t(kOffPtile + b * kPtile + h * 128);
        const uint32_t prow_r = tc::mapa(prow_l, peer);
        const uint32_t rbar = tc::mapa(bar(B_RP_FULL + b), peer);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t off = uint32_t((k ^ (h & 7)) << 4);
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(prow_l + off), "r"(pw[4 * k]),
                       "r"(pw[4 * k + 1]), "r"(pw[4 * k + 2]), "r"(pw[4 * k + 3]) : "memory");
          tc::st_async_v4(prow_r + off, pw[4 * k], pw[4 * k + 1], pw[4 * k + 2], pw[4 * k + 3], rbar);
        }
        tc::st_async_b32(tc::mapa(sb + uint32_t(kOffAlpha + (b * 64 + orow) * 4), peer), f2u(a), rbar);
        fence_proxy_async_smem();  // my P rows are read by the tensor core
        if (lane == 0) TRACE(8, i);
        if (i > 0 && __any_sync(0xffffffffu, a != 1.f) && !correct_o(i, a)) { ok = false; break; }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_P_READY + b));
      if (lane == 0 && q4 == 3) TRACE(9, i);
    }

    // ---- epilogue: final row factor, then O row -> output
    if (ok) {
      float f = 0.f;
      const int S = p.num_splits;
      if (owner) {
        const float lse0 = l > 0.f ? (m + log2f(l)) * kLn2 : -CUDART_INF_F;
        float lse_out = lse0;
        f = l > 0.f ? (tens ? p.kv_scale : 1.f) / l : 0.f;
        if (S == 1 && p.sink && h < p.H) {
          const float sg = __ldg(p.sink + h);
          lse_out = fmaxf(lse0, sg) + log1pf(expf(-fabsf(lse0 - sg)));
          f *= expf(lse0 - lse_out);
        }
        if (h < p.H) {
          if (S == 1) {
            if (p.lse) p.lse[int64_t(t) * p.H + h] = lse_out;
          } else {
            p.lse_part[(int64_t(t) * S + split) * p.H + h] = lse0;
          }
        }
        tc::st_async_b32(tc::mapa(sb + uint32_t(kOffFin + orow * 4), peer), f2u(f), tc::mapa(bar(B_FIN), peer));
      } else {
        ok = mbar_wait(bar(B_FIN), 0);
        f = reinterpret_cast<const float*>(sm + kOffFin)[prow];
      }
      if (ok && ntiles > 0) {
        const int last = ntiles - 1;
        ok = mbar_wait(bar(B_K_FREE + (last & 1)), (last >> 1) & 1);
        tc::fence_after();
      }
      // TMEM loads are warp-wide: every lane takes part, only real heads store
      if (__all_sync(0xffffffffu, ok)) {
        const int64_t orow_g = S == 1 ? int64_t(t) * p.H + h : (int64_t(t) * S + split) * p.H + h;
        // four 16-column loads in flight per wait
#pragma unroll 1
        for (int k4 = 0; k4 < 4; ++k4) {
          uint32_t v4[4][16];
          if (ntiles > 0) {
#pragma unroll
            for (int j = 0; j < 4; ++j) tc::ld16(lrow + kTmO + 64 * k4 + 16 * j, v4[j]);
            tc::wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
              for (int e = 0; e < 16; ++e) v4[j][e] = 0u;
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t* v = v4[j];
            const int col = 256 * int(crank) + 64 * k4 + 16 * j;
            if (h >= p.H) {
            } else if (S == 1) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow_g * kLatent + col);
              uint32_t o[8];
#pragma unroll
              for (int e = 0; e < 8; ++e)
                o[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * f, __uint_as_float(v[2 * e + 1]) * f);
              dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
              dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
            } else {
              float4* dst = reinterpret_cast<float4*>(p.o_part + orow_g * kLatent + col);
#pragma unroll
              for (int e = 0; e < 4; ++e)
                dst[e] = make_float4(__uint_as_float(v[4 * e]) * f, __uint_as_float(v[4 * e + 1]) * f,
                                     __uint_as_float(v[4 * e + 2]) * f, __uint_as_float(v[4 * e + 3]) * f);
            }
          }
        }
      }
    }
  }

  // ------------------------------------------------------------------ teardown
  if (!ok && lane == 0) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
  tc::fence_before();
  __syncthreads();
  tc::cluster_arrive();  // no remote store may target a CTA that has left
  tc::cluster_wait();
  if (warp == kMmaWarp) {
    tc::fence_after();
    tc::dealloc(tm, 512);
  }
#ifdef SMLA_TRACE
  if (threadIdx.x == 0 && blockIdx.x < 4096) g_span[blockIdx.x][1] = globaltimer_ns();
#endif
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
  static int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemTc));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemTc));
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  const int64_t grid = int64_t(a.T) * a.num_splits * 2;
  if (a.kv_format == SMLA_KV_FP8_TENSOR)
    decode_tc_kernel<true><<<static_cast<unsigned>(grid), kThreadsTc, kSmemTc, s>>>(a);
  else
    decode_tc_kernel<false><<<static_cast<unsigned>(grid), kThreadsTc, kSmemTc, s>>>(a);
  return cudaGetLastError();
}

}  // namespace smla

#ifdef SMLA_TRACE
extern "C" int smla_trace_read(unsigned long long* host) {
  return int(cudaMemcpyFromSymbol(host, g_trace, sizeof(g_trace)));
}
extern "C" int smla_span_read(unsigned long long* host) {
  return int(cudaMemcpyFromSymbol(host, g_span, sizeof(g_span)));
}
#endif
