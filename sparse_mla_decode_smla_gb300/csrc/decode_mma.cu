// Sparse MLA decode, warp-level tensor-core path (mma.sync m16n8k16). One CTA per
// (query token, top-k split, group of 16 heads); 4 consumer warps + 1 producer warp.
//
// What it computes (vLLM PR #43477 "关键源码片段", forward_mqa; SGLang PR #24692
// "实现拆解 2": tiled sparse decode with online softmax, split merge, sink): for each
// selected slot j, s_j = sm_scale * <q_h, k_j> over 576 dims, out_h = softmax-weighted
// sum of v_j = k_j[0:512].
//
// Producer warps (two): the split's index list is copied into shared memory (one bulk
// copy), then walked 32 slots at a time, each producer warp taking 16 slots of a stage.
// Page-table entries are fetched six stages ahead with 4-byte cp.async into a shared
// ring, so the dependent index -> page -> row chain never stalls the issue of row copies.
// Each valid slot's whole 656-byte row is one bulk copy (cp.async.bulk) into a 4-stage
// shared-memory ring; the stage's mbarrier counts the bytes. Bulk copies issued by one
// warp serialise on the TMA engine, so the copies of a stage come from two warps.
// Padding and invalid entries are never fetched.
//
// Consumer warps (warp w owns latent block w = dims [128w, 128w+128)):
//  * QK: warp w multiplies its 128 latent dims (+ RoPE dims [16w, 16w+16)) for the 32
//    slots of the stage. q sits in registers as A fragments (f16 for the latent, bf16 for
//    RoPE). B fragments are built from the staged E4M3 bytes with cvt.rn.f16x2.e4m3x2:
//    the k order inside an mma is permuted so each thread reads 16 contiguous bytes of a
//    row, and q is permuted the same way. The per-128 scale multiplies the fp32 partial
//    score of block w.
//  * The four partial scores meet in a double-buffered shared-memory array after one
//    barrier; every warp then sums all four and runs the masked base-2 online softmax for
//    all 32 slots (the same arithmetic in every warp, so all agree bit for bit). The
//    probabilities are then already in the registers of the PV B fragments.
//  * PV: O^T[dims, heads] = V^T P^T. Warp w accumulates its 128 output dims. A fragments
//    (V^T) come from the staged bytes of four rows, paired by prmt and converted; the
//    B fragments are p * scale_w[j] / r_w, with r_w the running maximum of scale_w over
//    the slots seen (keeps the f16 operand in [0, 1]).
//  * Epilogue: o = O * r_w / l, lse = (m + log2 l) * ln 2. With one split the sink is
//    applied here; otherwise fp32 partials go to the workspace for the merge kernel.
// Slots that are never fetched keep whatever finite bytes the ring held (it starts
// zeroed): their score is replaced by -inf, so their probability is exactly 0.
// All waits are mbarrier waits bounded in time; a wait that gives up sets
// SMLA_DEVERR_TIMEOUT and the CTA leaves after its copies in flight have landed.
#include <math_constants.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace smla {
namespace {

#ifndef SMLA_MMA_STAGES_FP8
#define SMLA_MMA_STAGES_FP8 4
#endif
#ifndef SMLA_MMA_MIN_BLOCKS
#define SMLA_MMA_MIN_BLOCKS 2
#endif
constexpr int kConsumerWarps = 4;
// Two producer warps, each issuing the bulk copies of half of every stage: bulk copies
// from a single warp serialise (about 14 GB/s per SM), several issuing warps do not.
constexpr int kProducerWarps = 2;
constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
constexpr int kSlots = 32;  // slots per stage
constexpr int kPageAhead = 6;  // page-table entries are fetched this many stages ahead
constexpr int kPageRing = 8;

template <int FMT>
struct Cfg {
  static constexpr bool kFp8 = FMT != SMLA_KV_BF16;          // e4m3 latent codes
  static constexpr bool kTensor = FMT == SMLA_KV_FP8_TENSOR;  // one scale, e4m3 RoPE too
  static constexpr int kRowBytes =
      kTensor ? kFp8TensorRowBytes : (kFp8 ? kFp8RowBytes : kBf16RowBytes);
  static constexpr int kStages = kFp8 ? SMLA_MMA_STAGES_FP8 : 3;
  static constexpr size_t kRing = size_t(kStages) * kSlots * kRowBytes;
  static constexpr size_t kRed = 2 * 4 * 4 * 32 * 16;  // partial scores [2][warp][nt][lane] float4
  static constexpr size_t kSmall = 16 * 4;               // stage valid masks
  static constexpr size_t kIdx = kMaxSplitLen * 4;       // the split's index list
  static constexpr size_t kPages = kPageRing * kSlots * 4;  // page-table entries in flight
  static constexpr size_t kBars = (2 * kStages + 2) * 8;
  static constexpr size_t kSmem = kRing + kRed + kSmall + kIdx + kPages + kBars;
};

__device__ __forceinline__ float fmax4(float a, float b, float c, float d) {
  return fmaxf(fmaxf(a, b), fmaxf(c, d));
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, SMLA_MMA_MIN_BLOCKS) decode_mma_kernel(const DecodeArgs p) {
  using C = Cfg<FMT>;
  constexpr bool kFp8 = C::kFp8;
  constexpr int RB = C::kRowBytes;
  constexpr int NST = C::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float4* red = reinterpret_cast<float4*>(smem + C::kRing);
  uint16_t* meta = reinterpret_cast<uint16_t*>(smem + C::kRing + C::kRed);  // [stage][producer]
  int32_t* sidx = reinterpret_cast<int32_t*>(smem + C::kRing + C::kRed + C::kSmall);
  int32_t* spage = sidx + kMaxSplitLen;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kRing + C::kRed + C::kSmall + C::kIdx + C::kPages);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + NST), cbar0 = smem_u32(bars + 2 * NST);
  const uint32_t idxbar = smem_u32(bars + 2 * NST + 1);
  const uint32_t ring_s = smem_u32(ring);

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5, g = lane >> 2, c = lane & 3;
  const int HG = p.H >> 4;
  int bid = blockIdx.x;
  const int hg = bid % HG;
  bid /= HG;
  const int split = bid % p.num_splits;
  const int t = bid / p.num_splits;
  const int h0 = hg * 16;

  const int r = p.req_id ? __ldg(p.req_id + t) : t / p.next_n;
  const bool req_ok = r >= 0 && r < p.B;
  const int32_t* pt_row = p.page_table + int64_t(req_ok ? r : 0) * p.stride;
  const int32_t* idx_row = p.topk + int64_t(t) * p.K;
  const int j0 = split * p.split_len;
  const int j1 = min(p.K, j0 + p.split_len);
  const int ntiles = req_ok ? max(0, (j1 - j0 + kSlots - 1) / kSlots) : 0;

  // ---- set-up: zeroed ring (never-fetched slots must hold finite bytes), barriers
  {
    uint4* z = reinterpret_cast<uint4*>(ring);
    for (size_t k = tid; k < C::kRing / 16; k += kThreads) z[k] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
    if (tid == 0) {
      for (int s = 0; s < NST; ++s) {
        mbar_init(full0 + 8 * s, kProducerWarps);  // one expect_tx arrival per producer warp
        mbar_init(empty0 + 8 * s, kConsumerWarps);
      }
      mbar_init(cbar0, kConsumerWarps);
      mbar_init(idxbar, 1);
      if (!req_ok) atomicOr(p.err, SMLA_DEVERR_INDEX);
    }
    __syncthreads();
  }

  // =================================================================== producer warp
  if (w >= kConsumerWarps) {
    const int pw = w - kConsumerWarps;          // producer warp: slots [16 pw, 16 pw + 16)
    const bool act = lane < kSlots / kProducerWarps;
    const int myslot = (kSlots / kProducerWarps) * pw + lane;
    // the split's index list, one bulk copy (16-byte aligned: K % 4 == 0, j0 % 64 == 0)
    const int nidx = j1 - j0;
    bool ok = true;
    if (ntiles > 0) {
      if (pw == 0 && lane == 0) {
        mbar_arrive_expect_tx(idxbar, uint32_t(nidx) * 4u);
        bulk_g2s(smem_u32(sidx), idx_row + j0, uint32_t(nidx) * 4u, idxbar);
      }
      ok = mbar_wait(idxbar, 0);
    }
    auto idx_of = [&](int tile) -> int32_t {
      const int j = tile * kSlots + myslot;
      return (act && tile < ntiles && j < nidx) ? sidx[j] : -1;
    };
    // page-table entries travel by 4-byte cp.async into a shared ring, kPageAhead stages
    // ahead of their use, so no lane ever waits on a dependent global load at issue time
    auto fetch_page = [&](int tile) {
      const int32_t idx = idx_of(tile);
      if (idx >= 0 && (idx >> p.log2_page) < p.stride)
        cp_async4(smem_u32(spage + (tile % kPageRing) * kSlots + myslot), pt_row + (idx >> p.log2_page));
      cp_async_commit();
    };
    if (ok)
      for (int d = 0; d < kPageAhead; ++d) fetch_page(d);
    int issued = 0;
    for (int i = 0; i < ntiles && ok; ++i) {
      fetch_page(i + kPageAhead);
      cp_async_wait<kPageAhead>();
      const int32_t idx_c = idx_of(i);
      const int st = i % NST;
      if (!mbar_wait(empty0 + 8 * st, ((i / NST) & 1) ^ 1)) {
        ok = false;
        break;
      }
      int64_t phys = -1;
      if (idx_c != -1) {
        if (idx_c < 0 || (idx_c >> p.log2_page) >= p.stride) {
          atomicOr(p.err, SMLA_DEVERR_INDEX);
        } else {
          const int32_t pg = spage[(i % kPageRing) * kSlots + myslot];
          if (pg < 0 || pg >= p.num_pages)
            atomicOr(p.err, SMLA_DEVERR_PAGE);
          else
            phys = (int64_t(pg) << p.log2_page) + (idx_c & ((1 << p.log2_page) - 1));
        }
      }
      const uint32_t vmask = __ballot_sync(0xffffffffu, phys >= 0);
      if (lane == 0) {
        meta[2 * st + pw] = uint16_t(vmask);
        mbar_arrive_expect_tx(full0 + 8 * st, uint32_t(__popc(vmask)) * RB);
      }
      __syncwarp();
      if (phys >= 0)
        bulk_g2s(ring_s + (st * kSlots + myslot) * RB, p.kv + phys * RB, RB, full0 + 8 * st);
      issued = i + 1;
    }
    cp_async_wait<0>();
    if (!ok && lane == 0) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
    // never leave while copies into this CTA's shared memory are in flight
    for (int i = max(0, issued - NST); i < issued; ++i)
      if (!mbar_wait(full0 + 8 * (i % NST), (i / NST) & 1)) break;
    return;
  }

  // =================================================================== consumer warps
  const __nv_bfloat16* qt =
      reinterpret_cast<const __nv_bfloat16*>(p.q) + (int64_t(t) * p.H + h0) * kDim;
  uint32_t qa[8][4];
  uint32_t qr[4];
  // FP8 caches: q enters the f16 MMAs scaled by a power-of-two normaliser per (head row,
  // 128-dim latent block) that brings the block's largest |q| into [1, 2); the factor goes
  // back into the block's fp32 partial score. So any finite bf16 q is exact in f16
  // (elements below 2^-17 of their block's largest keep 2^-25 of it in absolute error).
  // The per-tensor format's RoPE part (f16 too) gets its own normaliser per head row.
  float qf_g = 1.f, qf_g8 = 1.f, rf_g = 1.f, rf_g8 = 1.f;
  {
    const uint4* rg = reinterpret_cast<const uint4*>(qt + g * kDim + 128 * w + 32 * c);
    const uint4* rg8 = reinterpret_cast<const uint4*>(qt + (g + 8) * kDim + 128 * w + 32 * c);
    uint32_t a[16], b[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(rg + i), v8 = __ldg(rg8 + i);
      a[4 * i] = v.x; a[4 * i + 1] = v.y; a[4 * i + 2] = v.z; a[4 * i + 3] = v.w;
      b[4 * i] = v8.x; b[4 * i + 1] = v8.y; b[4 * i + 2] = v8.z; b[4 * i + 3] = v8.w;
    }
    // largest bf16 magnitude of rows g and g+8 over the warp's block (the quad's 4 x 32 dims)
    auto quad_max = [&](uint32_t m) {
      m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
      return max(m, __shfl_xor_sync(0xffffffffu, m, 2));
    };
    uint32_t ma = 0, mb = 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      ma = bf16x2_max(ma, a[i] & 0x7fff7fffu);
      mb = bf16x2_max(mb, b[i] & 0x7fff7fffu);
    }
    const int fa = pow2_exponent_of_bf16(quad_max(bf16x2_hmax_bits(ma)));
    const int fb = pow2_exponent_of_bf16(quad_max(bf16x2_hmax_bits(mb)));
    const float da = exp2_int(-fa), db = exp2_int(-fb);
    if (kFp8) {
      qf_g = exp2_int(fa);
      qf_g8 = exp2_int(fb);
    }
    auto cvt = [](uint32_t w, float d) { return pack_f16x2(bf16_lo(w) * d, bf16_hi(w) * d); };
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (kFp8) {
        qa[s][0] = cvt(a[2 * s], da);
        qa[s][1] = cvt(b[2 * s], db);
        qa[s][2] = cvt(a[2 * s + 1], da);
        qa[s][3] = cvt(b[2 * s + 1], db);
      } else {
        qa[s][0] = a[2 * s];
        qa[s][1] = b[2 * s];
        qa[s][2] = a[2 * s + 1];
        qa[s][3] = b[2 * s + 1];
      }
    }
    const uint2 rv = __ldg(reinterpret_cast<const uint2*>(qt + g * kDim + kLatent + 16 * w + 4 * c));
    const uint2 rv8 =
        __ldg(reinterpret_cast<const uint2*>(qt + (g + 8) * kDim + kLatent + 16 * w + 4 * c));
    qr[0] = rv.x; qr[1] = rv8.x; qr[2] = rv.y; qr[3] = rv8.y;
    if (C::kTensor) {  // the RoPE codes become f16 B fragments: q's RoPE part goes f16 too
      const uint32_t m1 = bf16x2_max(rv.x & 0x7fff7fffu, rv.y & 0x7fff7fffu);
      const uint32_t m2 = bf16x2_max(rv8.x & 0x7fff7fffu, rv8.y & 0x7fff7fffu);
      const int f1 = pow2_exponent_of_bf16(quad_max(bf16x2_hmax_bits(m1)));
      const int f2 = pow2_exponent_of_bf16(quad_max(bf16x2_hmax_bits(m2)));
      rf_g = exp2_int(f1);
      rf_g8 = exp2_int(f2);
      const float d1 = exp2_int(-f1), d2 = exp2_int(-f2);
      qr[0] = cvt(rv.x, d1); qr[1] = cvt(rv8.x, d2); qr[2] = cvt(rv.y, d1); qr[3] = cvt(rv8.y, d2);
    }
  }

  float O[8][2][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) O[i][j][e] = 0.f;
  // running max (base-2 logits) and row sum of heads g and g+8; every consumer warp
  // computes the same values for the whole stage, so no exchange is needed.
  float m_g = -CUDART_INF_F, m_g8 = -CUDART_INF_F, l_g = 0.f, l_g8 = 0.f;
  float r_w = 0.f;
  uint32_t n_done = 0;  // stages computed (cbar parity and partial-score buffer index)
  bool ok = true;
  // consumer-only barrier (bounded): each consumer warp arrives once, then all wait
  auto csync = [&](int k, uint32_t parity) -> bool {
    __syncwarp();
    if (lane == 0) mbar_arrive(cbar0 + 8 * k);
    const bool r = mbar_wait(cbar0 + 8 * k, parity & 1);
    __syncwarp();
    return r;
  };

  for (int i = 0; i < ntiles && ok; ++i) {
    const int st = i % NST;
    if (!mbar_wait(full0 + 8 * st, (i / NST) & 1)) {
      ok = false;
      break;
    }
    const uint32_t msk = uint32_t(meta[2 * st]) | (uint32_t(meta[2 * st + 1]) << 16);
    if (msk != 0u) {
      const uint32_t sb = ring_s + st * kSlots * RB;
      float4* rd = red + (n_done & 1) * (4 * 4 * 32);
      // ---- QK partial over latent block w (+ RoPE quarter w) for the 32 slots.
      // The four slot groups are independent accumulation chains; interleaving them
      // (k step outer) keeps four mma.sync in flight instead of one.
      float sc[4][2];
      float acc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
      if (kFp8) {
        uint32_t wd[4][8];
        float accr[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const uint32_t rb = sb + (8 * nt + g) * RB + 128 * w + 32 * c;
          const uint4 v0 = lds128(rb), v1 = lds128(rb + 16);
          wd[nt][0] = v0.x; wd[nt][1] = v0.y; wd[nt][2] = v0.z; wd[nt][3] = v0.w;
          wd[nt][4] = v1.x; wd[nt][5] = v1.y; wd[nt][6] = v1.z; wd[nt][7] = v1.w;
#pragma unroll
          for (int e = 0; e < 4; ++e) accr[nt][e] = 0.f;
          if (C::kTensor) {
            // RoPE codes of dims [16w + 4c, +4), one scale for everything
            const uint32_t rc = lds_u32(sb + (8 * nt + g) * RB + kLatent + 16 * w + 4 * c);
            uint32_t r0, r1;
            e4m3x4_to_f16x4(rc, r0, r1);
            mma_f16(accr[nt], qr, r0, r1);
            sc[nt][0] = p.kv_scale;
            sc[nt][1] = p.kv_scale;
          } else {
            const uint2 rv = lds64(sb + (8 * nt + g) * RB + kRopeOffFp8 + 2 * (16 * w + 4 * c));
            mma_bf16(accr[nt], qr, rv.x, rv.y);
            sc[nt][0] = lds_f32(sb + (8 * nt + 2 * c) * RB + kScaleOff + 4 * w);
            sc[nt][1] = lds_f32(sb + (8 * nt + 2 * c + 1) * RB + kScaleOff + 4 * w);
          }
        }
#pragma unroll
        for (int s = 0; s < 8; ++s)
#pragma unroll
          for (int nt = 0; nt < 4; ++nt) {
            uint32_t b0, b1;
            e4m3x4_to_f16x4(wd[nt][s], b0, b1);
            mma_f16(acc[nt], qa[s], b0, b1);
          }
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          if (C::kTensor) {  // the RoPE part carries the scale too (and q's RoPE normaliser)
            accr[nt][0] *= p.kv_scale * rf_g;
            accr[nt][1] *= p.kv_scale * rf_g;
            accr[nt][2] *= p.kv_scale * rf_g8;
            accr[nt][3] *= p.kv_scale * rf_g8;
          }
          // the block's scale and q's normaliser of rows g (elements 0, 1) and g+8 (2, 3)
          acc[nt][0] = fmaf(acc[nt][0], sc[nt][0] * qf_g, accr[nt][0]);
          acc[nt][1] = fmaf(acc[nt][1], sc[nt][1] * qf_g, accr[nt][1]);
          acc[nt][2] = fmaf(acc[nt][2], sc[nt][0] * qf_g8, accr[nt][2]);
          acc[nt][3] = fmaf(acc[nt][3], sc[nt][1] * qf_g8, accr[nt][3]);
        }
      } else {
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          const uint32_t rb = sb + (8 * nt + g) * RB;
          const uint32_t base = rb + 2 * (128 * w + 32 * c);
          uint32_t wd[16];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = lds128(base + 16 * k);
            wd[4 * k] = v.x; wd[4 * k + 1] = v.y; wd[4 * k + 2] = v.z; wd[4 * k + 3] = v.w;
          }
#pragma unroll
          for (int s = 0; s < 8; ++s) mma_bf16(acc[nt], qa[s], wd[2 * s], wd[2 * s + 1]);
          const uint2 rv = lds64(rb + 2 * kLatent + 2 * (16 * w + 4 * c));
          mma_bf16(acc[nt], qr, rv.x, rv.y);
          sc[nt][0] = 1.f;
          sc[nt][1] = 1.f;
        }
      }
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
        rd[(w * 4 + nt) * 32 + lane] = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
      if (!(ok = csync(0, n_done))) break;

      // ---- full scores of heads g, g+8 for all 32 slots (slot 8nt + 2c + {0,1})
      float sp[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const float4 a = rd[(0 * 4 + nt) * 32 + lane], b = rd[(1 * 4 + nt) * 32 + lane];
        const float4 cc = rd[(2 * 4 + nt) * 32 + lane], d = rd[(3 * 4 + nt) * 32 + lane];
        const int sl = 8 * nt + 2 * c;
        const bool v0 = (msk >> sl) & 1u, v1 = (msk >> (sl + 1)) & 1u;
        sp[nt][0] = v0 ? ((a.x + b.x) + (cc.x + d.x)) * p.c2 : -CUDART_INF_F;
        sp[nt][1] = v1 ? ((a.y + b.y) + (cc.y + d.y)) * p.c2 : -CUDART_INF_F;
        sp[nt][2] = v0 ? ((a.z + b.z) + (cc.z + d.z)) * p.c2 : -CUDART_INF_F;
        sp[nt][3] = v1 ? ((a.w + b.w) + (cc.w + d.w)) * p.c2 : -CUDART_INF_F;
      }
      float mg = fmax4(sp[0][0], sp[0][1], sp[1][0], sp[1][1]);
      mg = fmaxf(mg, fmax4(sp[2][0], sp[2][1], sp[3][0], sp[3][1]));
      float mg8 = fmax4(sp[0][2], sp[0][3], sp[1][2], sp[1][3]);
      mg8 = fmaxf(mg8, fmax4(sp[2][2], sp[2][3], sp[3][2], sp[3][3]));
      mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, 1));
      mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, 2));
      mg8 = fmaxf(mg8, __shfl_xor_sync(0xffffffffu, mg8, 1));
      mg8 = fmaxf(mg8, __shfl_xor_sync(0xffffffffu, mg8, 2));
      // ---- online softmax (base 2)
      const float ng = fmaxf(m_g, mg), ng8 = fmaxf(m_g8, mg8);
      const float bg = ng == -CUDART_INF_F ? 0.f : ng;
      const float bg8 = ng8 == -CUDART_INF_F ? 0.f : ng8;
      const float ag = exp2f(m_g - bg), ag8 = exp2f(m_g8 - bg8);
      float sum_g = 0.f, sum_g8 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        sp[nt][0] = exp2f(sp[nt][0] - bg);
        sp[nt][1] = exp2f(sp[nt][1] - bg);
        sp[nt][2] = exp2f(sp[nt][2] - bg8);
        sp[nt][3] = exp2f(sp[nt][3] - bg8);
        sum_g += sp[nt][0] + sp[nt][1];
        sum_g8 += sp[nt][2] + sp[nt][3];
      }
      sum_g += __shfl_xor_sync(0xffffffffu, sum_g, 1);
      sum_g += __shfl_xor_sync(0xffffffffu, sum_g, 2);
      sum_g8 += __shfl_xor_sync(0xffffffffu, sum_g8, 1);
      sum_g8 += __shfl_xor_sync(0xffffffffu, sum_g8, 2);
      l_g = l_g * ag + sum_g;
      l_g8 = l_g8 * ag8 + sum_g8;
      m_g = ng;
      m_g8 = ng8;
      // rescale factors of the O columns this thread holds (heads 2c, 2c+1, 2c+8, 2c+9),
      // computed by the lanes that own those heads' rows
      const float alpha[4] = {__shfl_sync(0xffffffffu, ag, 8 * c), __shfl_sync(0xffffffffu, ag, 8 * c + 4),
                              __shfl_sync(0xffffffffu, ag8, 8 * c), __shfl_sync(0xffffffffu, ag8, 8 * c + 4)};
      float tm = fmax4(sc[0][0], sc[0][1], sc[1][0], sc[1][1]);
      tm = fmaxf(tm, fmax4(sc[2][0], sc[2][1], sc[3][0], sc[3][1]));
      tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1));
      tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
      const float r_new = fmaxf(r_w, tm);
      const float rr = r_new > 0.f ? r_w / r_new : 1.f;
      r_w = r_new;
      const float inv_r = r_new > 0.f ? 1.f / r_new : 0.f;

      // ---- PV: O^T[128w.., heads] += V^T P^T
      // rescale only when some running maximum moved (rare after the first stages)
      const bool same = alpha[0] == 1.f && alpha[1] == 1.f && alpha[2] == 1.f && alpha[3] == 1.f && rr == 1.f;
      if (!__all_sync(0xffffffffu, same)) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) O[mt][nt][e] *= alpha[2 * nt + (e & 1)] * rr;
      }

#pragma unroll
      for (int kc = 0; kc < 2; ++kc) {
        const float f0 = sc[2 * kc][0] * inv_r, f1 = sc[2 * kc][1] * inv_r;
        const float f2 = sc[2 * kc + 1][0] * inv_r, f3 = sc[2 * kc + 1][1] * inv_r;
        const float* pa = sp[2 * kc];
        const float* pc = sp[2 * kc + 1];
        uint32_t bh0[2], bh1[2];
        if (kFp8) {
          bh0[0] = pack_f16x2(pa[0] * f0, pa[1] * f1);
          bh0[1] = pack_f16x2(pc[0] * f2, pc[1] * f3);
          bh1[0] = pack_f16x2(pa[2] * f0, pa[3] * f1);
          bh1[1] = pack_f16x2(pc[2] * f2, pc[3] * f3);
        } else {
          bh0[0] = pack_bf16x2(pa[0], pa[1]);
          bh0[1] = pack_bf16x2(pc[0], pc[1]);
          bh1[0] = pack_bf16x2(pa[2], pa[3]);
          bh1[1] = pack_bf16x2(pc[2], pc[3]);
        }
        const uint32_t r0 = sb + (16 * kc + 2 * c) * RB;
        if (kFp8) {
          const uint32_t off = 128 * w + 16 * g;
          const uint4 X = lds128(r0 + off), Y = lds128(r0 + RB + off);
          const uint4 Z = lds128(r0 + 8 * RB + off), U = lds128(r0 + 9 * RB + off);
          const uint32_t xs[4] = {X.x, X.y, X.z, X.w}, ys[4] = {Y.x, Y.y, Y.z, Y.w};
          const uint32_t zs[4] = {Z.x, Z.y, Z.z, Z.w}, us[4] = {U.x, U.y, U.z, U.w};
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t A[4], B[4];
            e4m3x4_to_f16x4(prmt(xs[q4], ys[q4], 0x5140), A[0], A[1]);
            e4m3x4_to_f16x4(prmt(xs[q4], ys[q4], 0x7362), B[0], B[1]);
            e4m3x4_to_f16x4(prmt(zs[q4], us[q4], 0x5140), A[2], A[3]);
            e4m3x4_to_f16x4(prmt(zs[q4], us[q4], 0x7362), B[2], B[3]);
            mma_f16(O[2 * q4][0], A, bh0[0], bh0[1]);
            mma_f16(O[2 * q4][1], A, bh1[0], bh1[1]);
            mma_f16(O[2 * q4 + 1][0], B, bh0[0], bh0[1]);
            mma_f16(O[2 * q4 + 1][1], B, bh1[0], bh1[1]);
          }
        } else {
          const uint32_t off = 2 * (128 * w + 16 * g);
          uint32_t xs[8], ys[8], zs[8], us[8];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const uint4 X = lds128(r0 + off + 16 * k), Y = lds128(r0 + RB + off + 16 * k);
            const uint4 Z = lds128(r0 + 8 * RB + off + 16 * k), U = lds128(r0 + 9 * RB + off + 16 * k);
            xs[4 * k] = X.x; xs[4 * k + 1] = X.y; xs[4 * k + 2] = X.z; xs[4 * k + 3] = X.w;
            ys[4 * k] = Y.x; ys[4 * k + 1] = Y.y; ys[4 * k + 2] = Y.z; ys[4 * k + 3] = Y.w;
            zs[4 * k] = Z.x; zs[4 * k + 1] = Z.y; zs[4 * k + 2] = Z.z; zs[4 * k + 3] = Z.w;
            us[4 * k] = U.x; us[4 * k + 1] = U.y; us[4 * k + 2] = U.z; us[4 * k + 3] = U.w;
          }
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint32_t A[4];
            A[0] = prmt(xs[k], ys[k], 0x5410);
            A[1] = prmt(xs[k], ys[k], 0x7632);
            A[2] = prmt(zs[k], us[k], 0x5410);
            A[3] = prmt(zs[k], us[k], 0x7632);
            mma_bf16(O[k][0], A, bh0[0], bh0[1]);
            mma_bf16(O[k][1], A, bh1[0], bh1[1]);
          }
        }
      }
      ++n_done;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
  }
  if (!ok) {
    if (lane == 0) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
    return;
  }

  // the main loop is over: the split merge, if one follows, may start launching
  if (tid == 0) pdl_trigger();
  // ---- epilogue: row sums and maxima of this thread's O columns come from their owners
  const float Lh[4] = {__shfl_sync(0xffffffffu, l_g, 8 * c), __shfl_sync(0xffffffffu, l_g, 8 * c + 4),
                       __shfl_sync(0xffffffffu, l_g8, 8 * c), __shfl_sync(0xffffffffu, l_g8, 8 * c + 4)};
  const float Mh[4] = {__shfl_sync(0xffffffffu, m_g, 8 * c), __shfl_sync(0xffffffffu, m_g, 8 * c + 4),
                       __shfl_sync(0xffffffffu, m_g8, 8 * c), __shfl_sync(0xffffffffu, m_g8, 8 * c + 4)};
  const int S = p.num_splits;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int h = (k >> 1) * 8 + 2 * c + (k & 1);
    const float L = Lh[k];
    const float lse0 = L > 0.f ? (Mh[k] + log2f(L)) * kLn2 : -CUDART_INF_F;
    float f = L > 0.f ? r_w / L : 0.f;
    float lse_out = lse0;
    if (S == 1 && p.sink) {
      const float sg = __ldg(p.sink + h0 + h);
      const float big = fmaxf(lse0, sg);
      lse_out = big + log1pf(expf(-fabsf(lse0 - sg)));
      f *= expf(lse0 - lse_out);
    }
    const int nt = k >> 1, par = k & 1;
    float v[16];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      v[2 * mt] = O[mt][nt][par] * f;
      v[2 * mt + 1] = O[mt][nt][par + 2] * f;
    }
    const int64_t row = int64_t(t) * p.H + h0 + h;
    if (S == 1) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + row * kLatent +
                                            128 * w + 16 * g);
      dst[0] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                          pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
      dst[1] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]),
                          pack_bf16x2(v[12], v[13]), pack_bf16x2(v[14], v[15]));
      if (w == 0 && g == 0 && p.lse) p.lse[row] = lse_out;
    } else {
      const int64_t prow = (int64_t(t) * S + split) * p.H + h0 + h;
      float4* dst = reinterpret_cast<float4*>(p.o_part + prow * kLatent + 128 * w + 16 * g);
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4)
        dst[k4] = make_float4(v[4 * k4], v[4 * k4 + 1], v[4 * k4 + 2], v[4 * k4 + 3]);
      if (w == 0 && g == 0) p.lse_part[prow] = lse0;
    }
  }
}

// Split merge (SGLang PR #24692 "关键文件": _merge_partial_attn, then _apply_attn_sink).
// One warp per (token, head, quarter of the 512 output dims): the lanes reduce
// M = max_s lse_s and W = sum_s e^{lse_s - M} (every quarter's warp the same way), then every
// lane accumulates 4 of the quarter's 128 dims over the splits, one load per split (fp32
// partials, or f16 ones from the tensor-core kernel).
// Four warps per row keep more loads in flight than one.
constexpr int kMergeWarps = 8;
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(const DecodeArgs p) {
  pdl_wait();  // the decode grid's partials are complete and visible
  const int lane = threadIdx.x & 31;
  const int64_t wid = int64_t(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  const int64_t row = wid >> 2;  // t * H + h
  const int quarter = int(wid & 3);
  if (row >= int64_t(p.T) * p.H) return;
  const int t = int(row / p.H), h = int(row % p.H);
  const int S = p.num_splits;
  const float* lp = p.lse_part + int64_t(t) * S * p.H + h;
  const float x0 = lane < S ? lp[int64_t(lane) * p.H] : -CUDART_INF_F;
  const float x1 = lane + 32 < S ? lp[int64_t(lane + 32) * p.H] : -CUDART_INF_F;
  float M = fmaxf(x0, x1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float w0 = (M == -CUDART_INF_F || x0 == -CUDART_INF_F) ? 0.f : expf(x0 - M);
  const float w1 = (M == -CUDART_INF_F || x1 == -CUDART_INF_F) ? 0.f : expf(x1 - M);
  float W = w0 + w1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
  const float lse0 = W > 0.f ? M + logf(W) : -CUDART_INF_F;
  float lse = lse0;
  float f = W > 0.f ? 1.f / W : 0.f;
  if (p.sink) {
    const float sg = __ldg(p.sink + h);
    lse = fmaxf(lse0, sg) + log1pf(expf(-fabsf(lse0 - sg)));
    f *= expf(lse0 - lse);
  }
  if (quarter == 0 && lane == 0 && p.lse) p.lse[row] = lse;

  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t e0 = (int64_t(t) * S * p.H + h) * kLatent + 128 * quarter + 4 * lane;  // first element
  const int64_t sstride = int64_t(p.H) * kLatent;                                     // elements between splits
#pragma unroll 4
  for (int s = 0; s < S; ++s) {
    const float wt = __shfl_sync(0xffffffffu, s < 32 ? w0 : w1, s & 31);
    if (wt == 0.f) continue;  // uniform across the warp
    float4 o;
    if (p.part_f16) {
      const uint2 v = __ldcs(reinterpret_cast<const uint2*>(reinterpret_cast<const __half*>(p.o_part) + e0 +
                                                            s * sstride));
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
      o = make_float4(a.x, a.y, b.x, b.y);
    } else {
      o = __ldcs(reinterpret_cast<const float4*>(p.o_part + e0 + s * sstride));
    }
    acc.x = fmaf(wt, o.x, acc.x);
    acc.y = fmaf(wt, o.y, acc.y);
    acc.z = fmaf(wt, o.z, acc.z);
    acc.w = fmaf(wt, o.w, acc.w);
  }
  uint2* dst = reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + row * kLatent + 128 * quarter) + lane;
  *dst = make_uint2(pack_bf16x2(acc.x * f, acc.y * f), pack_bf16x2(acc.z * f, acc.w * f));
}

template <int FMT>
cudaError_t launch_fmt(const DecodeArgs& a, cudaStream_t s) {
  const size_t smem = Cfg<FMT>::kSmem;
  // devices (below 64) whose kernel attribute is set; concurrent first calls set it twice
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaGetDevice(&dev);
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t(1) << dev) : 0;
  if (!(configured.load(std::memory_order_acquire) & bit) || !bit) {
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<FMT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_release);
  }
  const int64_t grid = int64_t(a.T) * a.num_splits * (a.H >> 4);
  decode_mma_kernel<FMT><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_mma(const DecodeArgs& a, int /*num_sms*/, cudaStream_t s) {
  if (a.kv_format == SMLA_KV_FP8_DS) return launch_fmt<SMLA_KV_FP8_DS>(a, s);
  if (a.kv_format == SMLA_KV_FP8_TENSOR) return launch_fmt<SMLA_KV_FP8_TENSOR>(a, s);
  return launch_fmt<SMLA_KV_BF16>(a, s);
}

cudaError_t launch_merge(const DecodeArgs& a, cudaStream_t s) {
  const int64_t rows = int64_t(a.T) * a.H;
  // launched with programmatic stream serialisation: its launch overlaps the decode grid's
  // tail, and the kernel waits (pdl_wait) for the decode results before reading them
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((4 * rows + kMergeWarps - 1) / kMergeWarps));
  cfg.blockDim = dim3(32 * kMergeWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel, a);
}

}  // namespace smla
