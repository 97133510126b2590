// Sparse MLA decode with FP8 operands on the 5th-generation tensor cores (tcgen05
// kind::f8f6f4): E4M3 q against the per-tensor FP8 cache (576 E4M3 codes a slot, one scale),
// the FP8-Q path of vLLM PR #43827 "关键源码片段" (bmm1_scale = scale * q_scale * kv_scale,
// bmm2_scale = kv_scale). One CTA per (query token, top-k split, group of 64 heads), with the
// same stacking as the 16-bit head-group kernel: lane l < 64 of the tensor memory holds head
// l's output dims [0, 256), lane 64 + l its dims [256, 512).
//
// What changes with 8-bit operands:
//  * q arrives as E4M3 codes: six TMA boxes stage it in shared memory, and the softmax warps
//    copy each row into TMEM, the A operand of QK (lane l < 64: head l's dims [0, 256) and
//    RoPE dims 512..543; lane 64 + l: dims [256, 512) and 544..575; four codes a column).
//  * The gathered cache rows are the MMA operands as they are: the copy warps only move each
//    16-byte chunk of a raw row to its place in the swizzled K tile (latent: two 16 KB pair
//    blocks [64 slots x 128 low dims | same slots x 128 high dims]; RoPE: [64 slots x 32 |
//    same slots x 32], 32-byte swizzle). A K tile is half the 16-bit one: three buffers, and
//    a raw ring of two tiles, fit.
//  * QK of a 64-slot tile is 9 M128 N128 K32 MMAs, PV 4 M128 N256 K32: half the tensor-pipe
//    time of the 16-bit kernel for the same work. What bounds the tile is shared-memory
//    bandwidth (gathers, the copy, the MMAs' operand reads, the score exchange), hence q in
//    TMEM and an MMA issuer that sleeps on its barriers instead of polling them.
//  * P is E4M3: p = 2^(s - m + 7), with the running max m moved whenever the max grows by more
//    than 1 (log2 units), so P <= 256 < 448 and values down to 2^-16 of the max survive. The
//    output is normalised by the sum of the E4M3 values PV accumulated (a convex combination
//    of the values); the LSE uses the sum before rounding.
//
// Per CTA (352 threads): warps 0-3 softmax and epilogue, warps 4-7 copy raw rows into the K
// tile, warps 8-9 producers (index and page rings, tile::gather4 row gathers, as in the 16-bit
// kernel), warp 10 MMA issuer. Every wait is bounded in time; a wait that gives up sets
// SMLA_DEVERR_TIMEOUT. Up to 8 splits merge inside a thread-block cluster.
#include <math_constants.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace smla {
namespace {

constexpr int kFN = 64;    // slots per tile
constexpr int kFSub = 16;  // rows per raw-ring stage (a quarter tile)
constexpr int kFFirstCopy = 4;  // warps 0..3: softmax
constexpr int kFCopyWarps = 4;
constexpr int kFFirstProducer = kFFirstCopy + kFCopyWarps;
constexpr int kFProducers = 2;
constexpr int kFMmaWarp = kFFirstProducer + kFProducers;
constexpr int kFThreads = 32 * (kFMmaWarp + 1);
constexpr int kFKBufs = 3;
constexpr int kFRawStages = 8;  // two tiles of gathered rows in flight
constexpr int kFGroup = 4 * kFp8TensorRowBytes;  // four gathered rows, 2304 B (128-byte multiple)
constexpr int kFRawStage = 4 * kFGroup;          // 16 rows
constexpr int kFPairBlk = 2 * kFN * 128;         // [64 slots x 128 low dims | same slots x 128 high dims]
constexpr int kFKLat = 2 * kFPairBlk;            // latent K tile, one buffer
constexpr int kFRopeBlk = 2 * kFN * 32;          // [64 slots x RoPE 0..31 | same slots x 32..63]
constexpr int kFPBlk = 64 * kFN;                 // 64 rows x 64 slots E4M3, 64-byte swizzle
constexpr int kFQAtom = 128 * 128;               // q latent atom: [128 rows x 128 dims]
constexpr int kFQRope = 128 * 32;                // q RoPE: [128 rows x 32 dims]
constexpr int kFXRow = 80;                       // 16 fp32 + padding (conflict-free rows)
constexpr int kFIdxAhead = 5, kFIdxRing = 6;
constexpr int kFAhead = 3, kFPageRing = 4;
constexpr int kFMetaRing = 8;
constexpr float kFRescaleThreshold = 1.f;  // log2 units: P stays below 2^(1 + kFPShift)
constexpr float kFPShift = 7.f;            // P = 2^(s - m + 7) <= 256 (E4M3 max 448)
static_assert(kFIdxAhead <= 2 * kFAhead && kFIdxRing > kFIdxAhead && kFPageRing > kFAhead, "index and page rings");
static_assert(kFGroup % 128 == 0, "gather destinations are 128-byte aligned");
// the producers run at most (K buffers + raw stages / 4 + 1) tiles ahead of the softmax
static_assert(kFMetaRing > kFKBufs + (kFRawStages + 3) / 4 + 1, "slot-mask ring");

// TMEM columns (512 allocated)
constexpr uint32_t kFTmO = 0;    // O [128 lanes x 256] fp32, lanes 64.. = high dims
constexpr uint32_t kFTmS = 256;  // scores [128 lanes x 128] fp32
constexpr uint32_t kFTmQ = 384;  // q [128 lanes x 288 codes]: 64 latent columns, then 8 RoPE

constexpr size_t kFOffK = 0;
constexpr size_t kFOffRope = kFOffK + size_t(kFKBufs) * kFKLat;
constexpr size_t kFOffP = kFOffRope + size_t(kFKBufs) * kFRopeBlk;  // [0 | P | 0]
// q is staged by TMA in the K-tile area (free until the copy warps' first write), then placed in
// TMEM: two 128-byte-swizzled latent atoms and a 32-byte-swizzled RoPE block
constexpr size_t kFOffQ = kFOffK;
constexpr size_t kFOffQr = kFOffQ + 2 * size_t(kFQAtom);
constexpr size_t kFOffRaw = kFOffP + 3 * size_t(kFPBlk);
constexpr size_t kFOffXs = kFOffRaw + size_t(kFRawStages) * kFRawStage;
constexpr size_t kFOffXm = kFOffXs + 128 * size_t(kFXRow);
constexpr size_t kFOffIdx = kFOffXm + 128 * 4;
constexpr size_t kFOffPages = kFOffIdx + size_t(kFIdxRing) * kFN * 4;
constexpr size_t kFOffMeta = kFOffPages + size_t(kFPageRing) * kFN * 4;
constexpr size_t kFOffTmem = kFOffMeta + kFMetaRing * 8;
constexpr size_t kFOffBars = kFOffTmem + 16;
enum {
  F_RAW_FULL = 0,
  F_RAW_EMPTY = F_RAW_FULL + kFRawStages,
  F_K_FULL = F_RAW_EMPTY + kFRawStages,  // [buffer]
  F_K_FREE = F_K_FULL + kFKBufs,         // [buffer]
  F_S_FULL = F_K_FREE + kFKBufs,
  F_S_FREE, F_P_READY, F_PV_DONE,
  F_Q,   // q's staging copy has landed
  F_QP,  // q is placed in TMEM (and its staging copy read)
  F_DRAIN, F_COUNT
};
static_assert(F_COUNT == 2 * kFRawStages + 2 * kFKBufs + 7, "one mbarrier per ring stage and buffer, none shared");
constexpr size_t kSmemF8 = kFOffBars + F_COUNT * 8 + 1024;  // + alignment slack
static_assert(kSmemF8 <= 232448, "shared memory budget");
static_assert(kFOffQr + kFQRope <= kFOffRope, "q staging fits in the K-tile area");
static_assert(kFOffK % 1024 == 0 && kFKLat % 1024 == 0 && kFOffQ % 1024 == 0 && kFOffRope % 256 == 0 &&
                  kFRopeBlk % 256 == 0 && kFOffQr % 256 == 0 && kFOffP % 512 == 0 && kFOffRaw % 128 == 0 &&
                  kFOffBars % 8 == 0,
              "swizzle atoms: 1024 B (128-byte swizzle), 512 B (64-byte), 256 B (32-byte)");
// the in-cluster split merge reuses the area below P (K tiles, RoPE blocks, q; free once every
// MMA has completed): 72 rows of 1024 B, LSEs, weights. P holds the final row factors then.
static_assert(kFOffP - kFOffK >= 72 * 1024 + 512 + 64 * kMaxClusterMerge * 4, "merge buffer");

// Wait for the phase of `bar` with the given parity, suspended for at most about hint_ns (the
// thread wakes as soon as the phase completes); true once it has completed. It spares the
// shared memory the polling of a test loop.
__device__ __forceinline__ bool mbar_try_wait_hint(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__global__ void __launch_bounds__(kFThreads, 1)
    decode_hg_f8_kernel(const DecodeArgs p, const __grid_constant__ CUtensorMap kv_map,
                        const __grid_constant__ CUtensorMap q_map128, const __grid_constant__ CUtensorMap q_map32) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(sm);
  auto bar = [&](int k) -> uint32_t { return sb + uint32_t(kFOffBars) + 8u * k; };
  // split-merge rows in the K-tile area (16-byte chunk c of row r at chunk c ^ (r & 7))
  auto mrow_addr = [&](int r, int c) -> uint32_t {
    return sb + uint32_t(kFOffK) + uint32_t(r) * 1024u + uint32_t((c ^ (r & 7)) << 4);
  };
  const uint32_t mlse = sb + uint32_t(kFOffK) + 72u * 1024u;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the TMA descriptors, fetched before their first use (q's loads, the first row gathers)
  if (tid == 0) {
    prefetch_tensormap(&q_map128);
    prefetch_tensormap(&q_map32);
  }
  if (tid == 32 * kFFirstProducer) prefetch_tensormap(&kv_map);

  // the codes' dot products take bmm1_scale = sm_scale * q_scale * kv_scale (times log2 e)
  const float c2 = p.c2 * p.q_scale * p.kv_scale;
  const int G = (p.H + 63) >> 6;
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
  const int ntiles = req_ok ? (nidx + kFN - 1) / kFN : 0;
  const int h0 = 64 * g;
  const int gheads = min(64, p.H - h0);
  const int mhp = (gheads + p.num_splits - 1) / p.num_splits;  // heads each split merges

  // Producer lanes 0-15 of warp kFFirstProducer + pw own slots 16q + lane, q in {pw, pw + 2}:
  // each slot's index kFIdxAhead tiles ahead, its page-table entry kFAhead tiles ahead.
  const bool producer = warp >= kFFirstProducer && warp < kFMmaWarp;
  const int pw = warp - kFFirstProducer;
  const bool act = lane < kFSub;
  int32_t* sidx = reinterpret_cast<int32_t*>(sm + kFOffIdx);
  int32_t* spage = reinterpret_cast<int32_t*>(sm + kFOffPages);
  auto in_split = [&](int tile, int q) {
    return act && tile < ntiles && tile * kFN + kFSub * q + lane < nidx;
  };
  auto idx_of = [&](int tile, int q) -> int32_t {
    return in_split(tile, q) ? sidx[(tile % kFIdxRing) * kFN + kFSub * q + lane] : -1;
  };
  auto ring_step = [&](int i) {
    cp_async_wait<kFIdxAhead - kFAhead - 1>();  // the group that fetched indices i + kFAhead
    const int tp = i + kFAhead;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int q = pw + 2 * k;
      if (tp >= 0) {
        const int32_t idx = idx_of(tp, q);
        if (idx >= 0 && (idx >> p.log2_page) < p.stride)
          cp_async4(smem_u32(spage + (tp % kFPageRing) * kFN + kFSub * q + lane), pt_row + (idx >> p.log2_page));
      }
      const int ti = i + kFIdxAhead;
      if (in_split(ti, q))
        cp_async4(smem_u32(sidx + (ti % kFIdxRing) * kFN + kFSub * q + lane),
                  idx_row + j0 + ti * kFN + kFSub * q + lane);
    }
    cp_async_commit();
  };
  if (producer)
    for (int i = -kFIdxAhead; i < 0; ++i) ring_step(i);

  // ------------------------------------------------------------------ set-up
  {
    // masked slots of the first tiles copy zeros, and the P buffer's zero blocks stay 0
    uint4* z = reinterpret_cast<uint4*>(sm + kFOffRaw);
    for (int k = tid; k < kFRawStages * kFRawStage / 16; k += kFThreads) z[k] = make_uint4(0, 0, 0, 0);
    uint4* zp = reinterpret_cast<uint4*>(sm + kFOffP);
    for (int k = tid; k < 3 * kFPBlk / 16; k += kFThreads) zp[k] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
      for (int s = 0; s < kFRawStages; ++s) {
        mbar_init(bar(F_RAW_FULL + s), 1);  // the expect_tx arrival of the stage's producer warp
        mbar_init(bar(F_RAW_EMPTY + s), kFCopyWarps);
      }
      for (int b = 0; b < kFKBufs; ++b) {
        mbar_init(bar(F_K_FULL + b), kFCopyWarps);
        mbar_init(bar(F_K_FREE + b), 1);
      }
      mbar_init(bar(F_S_FULL), 1);
      mbar_init(bar(F_S_FREE), 4);
      mbar_init(bar(F_QP), 4);  // the four softmax warps
      mbar_init(bar(F_P_READY), 4);
      mbar_init(bar(F_PV_DONE), 1);
      mbar_init(bar(F_Q), 1);
      mbar_init(bar(F_DRAIN), 1);
      tc::fence_mbarrier_init_cluster();
      if (!req_ok && split == 0 && g == 0) atomicOr(p.err, SMLA_DEVERR_INDEX);
      // the group's q rows [t H + h0, + 64): latent atom a holds dims [128a, +128) in rows
      // 0-63 and dims [256 + 128a, +128) in rows 64-127; RoPE dims 512.. / 544.. likewise
      if (ntiles > 0) {
        const int y = t * p.H + h0;
        const uint32_t qa = sb + uint32_t(kFOffQ), qr = sb + uint32_t(kFOffQr);
        mbar_arrive_expect_tx(bar(F_Q), 2 * kFQAtom + kFQRope);
        for (int a = 0; a < 2; ++a) {
          tma_load_2d(qa + a * kFQAtom, &q_map128, 128 * a, y, bar(F_Q));
          tma_load_2d(qa + a * kFQAtom + kFQAtom / 2, &q_map128, 256 + 128 * a, y, bar(F_Q));
        }
        tma_load_2d(qr, &q_map32, kLatent, y, bar(F_Q));
        tma_load_2d(qr + kFQRope / 2, &q_map32, kLatent + 32, y, bar(F_Q));
      }
    }
    if (warp == kFMmaWarp) tc::alloc(sb + uint32_t(kFOffTmem), 512);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
  }
  const uint32_t tm = *reinterpret_cast<volatile uint32_t*>(sm + kFOffTmem);

  bool ok = true;
  float cm_f = 0.f, cm_lse = -CUDART_INF_F;  // cluster merge: final row factor, LSE without the sink
  // ------------------------------------------------------------------ producer
  if (producer) {
    uint16_t* meta = reinterpret_cast<uint16_t*>(sm + kFOffMeta);
    constexpr uint32_t rowbytes = kFp8TensorRowBytes;
    const int32_t oob_row = int32_t(p.num_pages << p.log2_page);  // the TMA fills zeros
    for (int i = 0; i < ntiles && ok; ++i) {
      ring_step(i);
#pragma unroll 1
      for (int k = 0; k < 2 && ok; ++k) {
        const int q = pw + 2 * k;
        const int u = 4 * i + q, st = u % kFRawStages;
        if (!mbar_wait(bar(F_RAW_EMPTY + st), ((u / kFRawStages) & 1) ^ 1)) {
          ok = false;
          break;
        }
        const int32_t idx = idx_of(i, q);
        int64_t phys = -1;
        if (idx != -1) {
          if (idx < 0 || (idx >> p.log2_page) >= p.stride) {
            atomicOr(p.err, SMLA_DEVERR_INDEX);
          } else {
            const int32_t pg = spage[(i % kFPageRing) * kFN + kFSub * q + lane];
            if (pg < 0 || pg >= p.num_pages)
              atomicOr(p.err, SMLA_DEVERR_PAGE);
            else
              phys = (int64_t(pg) << p.log2_page) + (idx & ((1 << p.log2_page) - 1));
          }
        }
        const uint32_t vm = __ballot_sync(0xffffffffu, phys >= 0);
        const int32_t y = phys >= 0 ? int32_t(phys) : oob_row;
        const int32_t y0 = __shfl_sync(0xffffffffu, y, 4 * (lane & 3));
        const int32_t y1 = __shfl_sync(0xffffffffu, y, 4 * (lane & 3) + 1);
        const int32_t y2 = __shfl_sync(0xffffffffu, y, 4 * (lane & 3) + 2);
        const int32_t y3 = __shfl_sync(0xffffffffu, y, 4 * (lane & 3) + 3);
        uint32_t groups = 0;
#pragma unroll
        for (int gq = 0; gq < 4; ++gq) groups |= ((vm >> (4 * gq)) & 15u) ? (1u << gq) : 0u;
        if (lane == 0) {
          meta[(i % kFMetaRing) * 4 + q] = uint16_t(vm);
          mbar_arrive_expect_tx(bar(F_RAW_FULL + st), uint32_t(__popc(groups)) * 4u * rowbytes);
        }
        __syncwarp();
        if (lane < 4 && ((groups >> lane) & 1u))
          tma_gather4(sb + uint32_t(kFOffRaw) + uint32_t(st * kFRawStage + lane * kFGroup), &kv_map, 0, y0, y1, y2,
                      y3, bar(F_RAW_FULL + st));
      }
    }
    cp_async_wait<0>();
    // no copy may land after the CTA has left
    const int total = 4 * ntiles;
    for (int u = max(0, total - kFRawStages); u < total; ++u)
      if ((u & 1) == pw && !mbar_wait(bar(F_RAW_FULL + u % kFRawStages), (u / kFRawStages) & 1)) break;
  }
  // ------------------------------------------------------------------ MMA issuer
  else if (warp == kFMmaWarp) {
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t kIdQK = tc::idesc_e4m3_f32(128, 128, false, false);
      constexpr uint32_t kIdPV = tc::idesc_e4m3_f32(128, 256, false, true);
      // QK of tile i once its K tile is written and the scores of tile i-1 have been read
      auto qk_ready = [&](int i) {
        return mbar_test_wait(bar(F_K_FULL + i % kFKBufs), (i / kFKBufs) & 1) &&
               (i == 0 || mbar_test_wait(bar(F_S_FREE), (i - 1) & 1));
      };
      auto qk = [&](int i) {
        tc::fence_after();
        const int b = i % kFKBufs;
        const uint32_t kt = sb + uint32_t(kFOffK) + uint32_t(b * kFKLat);
        const uint32_t kr = sb + uint32_t(kFOffRope) + uint32_t(b * kFRopeBlk);
        const uint32_t d = tm + kFTmS;
#pragma unroll
        for (int j = 0; j < 8; ++j)  // 32 dims per MMA: q columns 8j.., K pair block j / 4, bytes 32 (j % 4)
          tc::mma_ts_f8(d, tm + kFTmQ + 8 * j, tc::sdesc_sw128(kt + (j >> 2) * kFPairBlk + (j & 3) * 32, 16, 1024),
                        kIdQK, j > 0);
        tc::mma_ts_f8(d, tm + kFTmQ + 64, tc::sdesc_sw32(kr, 16, 256), kIdQK, 1);
        tc::commit(bar(F_S_FULL));
      };
      auto pv = [&](int i) {
        tc::fence_after();
        const int b = i % kFKBufs;
        const uint32_t kt = sb + uint32_t(kFOffK) + uint32_t(b * kFKLat);
        const uint32_t pa = sb + uint32_t(kFOffP) + uint32_t(kFPBlk);  // P rows
#pragma unroll
        for (int s = 0; s < 2; ++s) {  // 32 slots per MMA
          // [P; 0] x latent dims [0, 256) -> lanes 0-63; [0; P] x dims [256, 512) -> lanes 64-127
          tc::mma_ss_f8(tm + kFTmO, tc::sdesc_sw64(pa + 32 * s, 16, 512),
                        tc::sdesc_sw128(kt + 4096 * s, kFPairBlk, 1024), kIdPV, (i > 0 || s > 0));
          tc::mma_ss_f8(tm + kFTmO, tc::sdesc_sw64(pa - kFPBlk + 32 * s, 16, 512),
                        tc::sdesc_sw128(kt + 8192 + 4096 * s, kFPairBlk, 1024), kIdPV, 1);
        }
        tc::commit(bar(F_K_FREE + b));
        tc::commit(bar(F_PV_DONE));
      };
      bool qok = mbar_wait(bar(F_QP), 0);
      if (!qok) ok = false;
      // PV of the oldest scored tile first when its P is ready, else QK of the next tile (at
      // most two tiles ahead of PV: two score buffers)
      int nqk = 0, npv = 0;
      uint64_t t0 = globaltimer_ns();
      for (uint32_t it = 0; qok && npv < ntiles; ++it) {
        if (npv < nqk && mbar_test_wait(bar(F_P_READY), npv & 1)) {
          pv(npv++);
        } else if (nqk < ntiles && nqk <= npv + 1 && qk_ready(nqk)) {
          qk(nqk++);
        } else {
          if ((it & 255u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
            ok = false;
            break;
          }
          // nothing to issue: sleep on the event that gates the next step (P of the oldest
          // scored tile, else the next K tile) rather than polling shared memory
          if (npv < nqk)
            mbar_try_wait_hint(bar(F_P_READY), npv & 1, 100);
          else if (nqk < ntiles)
            mbar_try_wait_hint(bar(F_K_FULL + nqk % kFKBufs), (nqk / kFKBufs) & 1, 100);
          continue;
        }
        t0 = globaltimer_ns();
      }
      // every MMA issued has completed before the tensor memory is released
      tc::commit(bar(F_DRAIN));
      if (!mbar_wait(bar(F_DRAIN), 0)) ok = false;
    }
    __syncwarp();
  }
  // ------------------------------------------------------------------ copy raw rows -> K tile
  else if (warp >= kFFirstCopy) {
    const int ctid = tid - 32 * kFFirstCopy;
    auto raw_row = [&](uint32_t stage, int slot) -> uint32_t {
      return stage + uint32_t((slot >> 2) * kFGroup + (slot & 3) * kFp8TensorRowBytes);
    };
    // a warp moves 16-byte chunks ch = lane of one row per step (conflict-free reads of 512
    // contiguous bytes and writes of 32 distinct chunks); threads 0-63 also move one RoPE chunk
    const int rslot = ctid >> 2, rc = ctid & 3;
    for (int i = 0; i < ntiles && ok; ++i) {
      const int b = i % kFKBufs;
      const uint32_t kt = sb + uint32_t(kFOffK) + uint32_t(b * kFKLat);
      const uint32_t kr = sb + uint32_t(kFOffRope) + uint32_t(b * kFRopeBlk);
      // the first K tile overwrites q's staging copy, read once q is placed in TMEM; later
      // ones wait for PV of tile i - kFKBufs to free their buffer
      if (i == 0 && !mbar_wait(bar(F_QP), 0)) {
        ok = false;
        break;
      }
      if (i >= kFKBufs && !mbar_wait(bar(F_K_FREE + b), ((i - kFKBufs) / kFKBufs) & 1)) {
        ok = false;
        break;
      }
#pragma unroll 1
      for (int q = 0; q < 4 && ok; ++q) {
        const int u = 4 * i + q, st = u % kFRawStages;
        if (!mbar_wait(bar(F_RAW_FULL + st), (u / kFRawStages) & 1)) {
          ok = false;
          break;
        }
        const uint32_t raw = sb + uint32_t(kFOffRaw) + uint32_t(st * kFRawStage);
        uint4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = lds128(raw_row(raw, (ctid >> 5) + 4 * k) + 16 * lane);
        uint4 rv = make_uint4(0, 0, 0, 0);
        if (ctid < 64) rv = lds128(raw_row(raw, rslot) + kLatent + 16 * rc);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(F_RAW_EMPTY + st));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // chunk lane = latent dims [16 lane, +16): half lane / 16, pair block (lane / 8) % 2
          const int slot = (ctid >> 5) + 4 * k;
          const int rr = kFN * (lane >> 4) + kFSub * q + slot;
          const uint32_t dst = kt + ((lane >> 3) & 1) * kFPairBlk + rr * 128 + (((lane & 7) ^ (rr & 7)) << 4);
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(v[k].x), "r"(v[k].y), "r"(v[k].z),
                       "r"(v[k].w) : "memory");
        }
        if (ctid < 64) {  // RoPE dims [16 rc, +16): half rc / 2, chunk rc % 2 of a 32-byte row
          const int rr = kFN * (rc >> 1) + kFSub * q + rslot;
          const uint32_t dst = kr + rr * 32 + (((rc & 1) ^ ((rr >> 2) & 1)) << 4);
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(dst), "r"(rv.x), "r"(rv.y), "r"(rv.z),
                       "r"(rv.w) : "memory");
        }
      }
      if (!ok) break;
      fence_proxy_async_smem();  // read by the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(F_K_FULL + b));
    }
    if (ctid == 0) pdl_trigger();
  }
  // ------------------------------------------------------------------ softmax + epilogue
  else {
    const int half = warp >> 1;  // 0: lanes 0-63 (low dims), 1: lanes 64-127 (high dims)
    const int pr = warp & 1;     // head pair: warps pr (low) and pr + 2 (high)
    const int hl = 32 * pr + lane;
    const int h = h0 + hl;
    const uint32_t lrow = tm + (uint32_t(32 * warp) << 16);
    const uint64_t* meta = reinterpret_cast<const uint64_t*>(sm + kFOffMeta);  // 64 slot bits per tile
    const uint32_t xmine = sb + uint32_t(kFOffXs) + uint32_t(32 * warp + lane) * kFXRow;
    const uint32_t xpart = sb + uint32_t(kFOffXs) + uint32_t(32 * (warp ^ 2) + lane) * kFXRow;
    const uint32_t mmine = sb + uint32_t(kFOffXm) + uint32_t(32 * warp + lane) * 4;
    const uint32_t mpart = sb + uint32_t(kFOffXm) + uint32_t(32 * (warp ^ 2) + lane) * 4;
    const int bar_x = 1 + pr;                      // both warps of the pair have written
    const int bar_mine = 3 + 2 * pr + half;        // the partner has read my row
    const int bar_part = 3 + 2 * pr + (half ^ 1);  // I have read the partner's row
    const int bar_max = 7 + pr;                    // both maxima are written
    const int bar_x2 = 9 + pr;                     // both second halves are written
    // m: running max (log2 units); lq: sum of the E4M3 weights PV accumulates, le: the same
    // weights before rounding (for the LSE), both in units of 2^kFPShift
    float m = -CUDART_INF_F, lq = 0.f, le = 0.f;
    bool good = true;

    auto correct_o = [&](float a) {  // warp-wide TMEM loads and stores
#pragma unroll 1
      for (int k = 0; k < 16; ++k) {
        uint32_t v[16];
        tc::ld16(lrow + kFTmO + 16 * k, v);
        tc::wait_ld();
#pragma unroll
        for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * a);
        tc::st16(lrow + kFTmO + 16 * k, v);
      }
      tc::wait_st();
    };

    // q placement: TMEM lane r = 32 warp + lane takes row r of the staged q (head r % 64, dims
    // [256 (r / 64), +256) and RoPE dims [512 + 32 (r / 64), +32)), four codes a column
    {
      const int qrow = 32 * warp + lane;
      bool have = ntiles > 0 && mbar_wait(bar(F_Q), 0);
      have = __all_sync(0xffffffffu, have);  // the TMEM stores are warp-wide
      if (ntiles > 0 && !have) {
        good = false;
        if (lane == 0) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
      }
      if (have) {
        const uint32_t qa = sb + uint32_t(kFOffQ), qr = sb + uint32_t(kFOffQr);
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int c = 4 * part + k;  // 16-byte chunk of the 128-byte atom row
              const uint4 v = lds128(qa + uint32_t(a * kFQAtom + qrow * 128 + ((c ^ (qrow & 7)) << 4)));
              w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
            }
            tc::st16(lrow + kFTmQ + 32 * a + 16 * part, w);
          }
        uint32_t rw[8];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const uint4 v = lds128(qr + uint32_t(qrow * 32 + ((c ^ ((qrow >> 2) & 1)) << 4)));
          rw[4 * c] = v.x; rw[4 * c + 1] = v.y; rw[4 * c + 2] = v.z; rw[4 * c + 3] = v.w;
        }
        tc::st8(lrow + kFTmQ + 64, rw);
        tc::wait_st();
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(F_QP));  // also: the staging copy has been read
    }

    bool loop_ok = true;
    for (int i = 0; i < ntiles; ++i) {
      float v[64];
      const uint32_t sbuf = kFTmS;  // column offset (lrow holds tm)
      const bool got = good && mbar_wait(bar(F_S_FULL), i & 1);
      if (got) {
        tc::fence_after();
        uint32_t w0[32], w1[32];
        tc::ld32(lrow + sbuf + 64 * half, w0);
        tc::ld32(lrow + sbuf + 64 * half + 32, w1);
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
      if (lane == 0 && got) mbar_arrive(bar(F_S_FREE));
      float own[32], send[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        own[e] = half ? v[32 + e] : v[e];
        send[e] = half ? v[e] : v[32 + e];
      }
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
      const uint32_t msk = uint32_t(meta[i % kFMetaRing] >> (32 * half));
      float s[32];
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float sv = ((msk >> j) & 1u) ? (own[j] + x[j]) * c2 : -CUDART_INF_F;
        s[j] = sv;
        mx = fmaxf(mx, sv);
      }
      named_bar_arrive(bar_part, 64);
      asm volatile("st.shared.f32 [%0], %1;" ::"r"(mmine), "f"(mx) : "memory");
      named_bar(bar_max, 64);
      mx = fmaxf(mx, lds_f32(mpart));
      float a = 1.f;
      const float mn = fmaxf(m, mx);
      if (m == -CUDART_INF_F ? mn != -CUDART_INF_F : mn > m + kFRescaleThreshold) {
        a = exp2f(m - mn);  // 0 when m was -inf
        m = mn;
      }
      const float base = m == -CUDART_INF_F ? 0.f : m - kFPShift;
      float sq = 0.f, se = 0.f;
      uint32_t pw4[8];  // 32 E4M3 codes
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float p0 = exp2f(s[4 * j] - base), p1 = exp2f(s[4 * j + 1] - base);
        const float p2 = exp2f(s[4 * j + 2] - base), p3 = exp2f(s[4 * j + 3] - base);
        se += (p0 + p1) + (p2 + p3);
        const uint32_t c01 = f32x2_to_e4m3x2(p0, p1), c23 = f32x2_to_e4m3x2(p2, p3);
        pw4[j] = c01 | (c23 << 16);
        uint32_t lo, hi;  // the E4M3 values back, exactly, as f16
        e4m3x4_to_f16x4(pw4[j], lo, hi);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&lo));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&hi));
        sq += (f01.x + f01.y) + (f23.x + f23.y);
      }
      lq = lq * a + sq;
      le = le * a + se;
      // the P block and O are free once PV of the previous tile is complete
      if (i >= 1 && !mbar_wait(bar(F_PV_DONE), (i - 1) & 1)) good = false;
      tc::fence_after();
      if (good && i > 0 && __any_sync(0xffffffffu, a != 1.f)) correct_o(a);
      if (good) {
        // row hl of P: 64 slot codes, 16-byte chunk c at c ^ ((hl >> 1) & 3); this warp's
        // slots are chunks 2 half, 2 half + 1
        const uint32_t prow = sb + uint32_t(kFOffP) + uint32_t(kFPBlk) + uint32_t(hl) * 64;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int c = 2 * half + k;
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(prow + ((c ^ ((hl >> 1) & 3)) << 4)),
                       "r"(pw4[4 * k]), "r"(pw4[4 * k + 1]), "r"(pw4[4 * k + 2]), "r"(pw4[4 * k + 3])
                       : "memory");
        }
        fence_proxy_async_smem();  // read by the tensor core
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0 && good) mbar_arrive(bar(F_P_READY));
    }

    // ---- epilogue: both row halves' sums, final row factor, then O lane -> output
    ok = loop_ok;
    if (ok) {
      if (ntiles > 0) named_bar(bar_mine, 64);  // the partner has read my last row
      bool fin = good;
      if (fin && ntiles > 0) {
        fin = mbar_wait(bar(F_PV_DONE), (ntiles - 1) & 1);
        tc::fence_after();
      }
      asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(xmine), "f"(lq), "f"(le) : "memory");
      ok = named_bar_and(bar_x, 64, fin);
      if (ok) {  // my half's sums + the other half's: the same values in both warps
        lq += lds_f32(xpart);
        le += lds_f32(xpart + 4);
      }
    }
    if (ok) {
      const int S = p.num_splits;
      const bool real = hl < gheads;
      const float lse0 = le > 0.f ? (m - kFPShift + log2f(le)) * kLn2 : -CUDART_INF_F;
      float lse_out = lse0;
      float f = lq > 0.f ? p.kv_scale / lq : 0.f;  // bmm2_scale = kv_scale
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
#pragma unroll 1
      for (int k4 = 0; k4 < 4 && !p.cluster_merge; ++k4) {
        uint32_t v4[4][16];
        if (ntiles > 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j) tc::ld16(lrow + kFTmO + 64 * k4 + 16 * j, v4[j]);
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
          uint32_t o[8];
          if (S == 1) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              o[e] = pack_bf16x2(__uint_as_float(vv[2 * e]) * f, __uint_as_float(vv[2 * e + 1]) * f);
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + orow_g * kLatent + col);
            dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
            dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
          } else {  // f16 partial: a convex combination of keys times kv_scale
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
  const uint32_t cmf = sb + uint32_t(kFOffP);  // final row factors (every MMA has completed)
  if (p.cluster_merge && warp < 4) asm volatile("st.shared.f32 [%0], %1;" ::"r"(cmf + 4 * tid), "f"(cm_f) : "memory");
  tc::fence_before();
  __syncthreads();
  if (p.cluster_merge) {
    // split merge inside the cluster (SGLang PR #24692 "关键文件": _merge_partial_attn, then
    // _apply_attn_sink): rank r merges heads [r hp, r hp + hp) of the group, from rows the
    // cluster's CTAs store into its shared memory between two cluster barriers
    tc::cluster_arrive();
    tc::cluster_wait();
    if (warp < kFFirstProducer) {
      // warp w reads TMEM lane quarter w % 4 and pushes half w / 4 of the 16 16-column chunks
      const int qw = warp & 3, part = warp >> 2;
      const int half = qw >> 1, hl = 32 * (qw & 1) + lane;
      const uint32_t lrow = tm + (uint32_t(32 * qw) << 16);
      const bool real = hl < gheads;
      const int mr = split * mhp + hl % mhp;
      const uint32_t owner = uint32_t(hl / mhp);
      const float f = lds_f32(cmf + 4 * (32 * qw + lane));
      if (real && half == 0 && part == 0) tc::st_dsmem_f32(tc::mapa(mlse + mr * 4, owner), cm_lse);
      tc::fence_after();
#pragma unroll 1
      for (int c = 8 * part; c < 8 * part + 8; c += 2) {
        uint32_t v2[2][16];
        __syncwarp();  // the TMEM loads are warp-wide
        if (ntiles > 0) {
          tc::ld16(lrow + kFTmO + 16 * c, v2[0]);
          tc::ld16(lrow + kFTmO + 16 * (c + 1), v2[1]);
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
          uint32_t o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            o[e] = pack_f16x2(__uint_as_float(v2[j][2 * e]) * f, __uint_as_float(v2[j][2 * e + 1]) * f);
          const int c0 = 32 * half + 2 * (c + j);  // 16-byte chunk of the 1024-byte merge row
          if (owner == uint32_t(split)) {
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
    for (int k = tid; k < nk; k += kFThreads) {
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
    for (int j = tid; j < nk * 64; j += kFThreads) {  // 8 output dims per job
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
          const float2 xx = __half22float2(*reinterpret_cast<const __half2*>(&vw[e]));
          acc[2 * e] = fmaf(w, xx.x, acc[2 * e]);
          acc[2 * e + 1] = fmaf(w, xx.y, acc[2 * e + 1]);
        }
      }
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                            (int64_t(t) * p.H + h0 + hs + k) * kLatent + 8 * c);
      *dst = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                        pack_bf16x2(acc[6], acc[7]));
    }
  }
  if (warp == kFMmaWarp) {
    tc::fence_after();
    tc::dealloc(tm, 512);
  }
}

}  // namespace

cudaError_t launch_decode_hg_f8(const DecodeArgs& a, cudaStream_t s) {
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t(1) << dev) : 0;
  if (!(configured.load(std::memory_order_acquire) & bit) || !bit) {
    const cudaError_t e =
        cudaFuncSetAttribute(decode_hg_f8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemF8));
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_release);
  }
  alignas(64) CUtensorMap map;
  alignas(64) CUtensorMap q128;
  alignas(64) CUtensorMap q32;
  cudaError_t e = kv_gather_map(a, &map);
  if (e == cudaSuccess) e = q_e4m3_maps(a, &q128, &q32);
  if (e != cudaSuccess) return e;
  const int64_t items = a.nitems > 0 ? a.nitems : int64_t(a.T) * ((a.H + 63) / 64);
  const int64_t grid = items * a.num_splits;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = kSmemF8;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (a.cluster_merge) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(a.num_splits);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (a.overlap_prev) {  // may start while the previous kernel drains (it reads none of its results)
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, decode_hg_f8_kernel, a, map, q128, q32);
}

}  // namespace smla
