// Sparse MLA decode, warp-level tensor-core path (mma.sync m16n8k16). One CTA per
// (query token, top-k split, group of 16 heads); 4 consumer warps + 1 producer warp.
//
// What it computes (vLLM PR #43477 "关键源码片段", forward_mqa; SGLang PR #24692
// "实现拆解 2": tiled sparse decode with online softmax, split merge, sink): for each
// selected slot j, s_j = sm_scale * <q_h, k_j> over 576 dims, out_h = softmax-weighted
// sum of v_j = k_j[0:512].
//
// Producer warp: walks the split's top-k list 32 slots at a time. Index loads run two
// tiles ahead and page-table loads one tile ahead, so the dependent-load chain stays off
// the critical path. Each valid slot's whole 656-byte row is fetched with one bulk copy
// (cp.async.bulk, TMA engine) into a 4-stage shared-memory ring; the stage's mbarrier
// counts the bytes. Padding and invalid entries are never fetched.
//
// Consumer warps (warp w owns latent block w = dims [128w, 128w+128)):
//  * QK: warp w multiplies its 128 latent dims (+ RoPE dims [16w, 16w+16)) for the 32
//    slots of the stage. q sits in registers as A fragments (f16 for the latent, bf16 for
//    RoPE). B fragments are built from the staged E4M3 bytes with cvt.rn.f16x2.e4m3x2:
//    the k order inside an mma is permuted so each thread reads 16 contiguous bytes of a
//    row, and q is permuted the same way. The per-128 scale multiplies the fp32 partial
//    score of block w.
//  * The four partial scores are summed through shared memory; warp w then owns slots
//    [8w, 8w+8) of the stage for the masked base-2 online softmax.
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

#include "common.cuh"
#include "kernels.h"

namespace smla {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kSlots = 32;  // slots per stage

template <int FMT>
struct Cfg {
  static constexpr bool kFp8 = FMT == SMLA_KV_FP8_DS;
  static constexpr int kRowBytes = kFp8 ? kFp8RowBytes : kBf16RowBytes;
  static constexpr int kStages = kFp8 ? 4 : 3;
  static constexpr size_t kRing = size_t(kStages) * kSlots * kRowBytes;
  static constexpr size_t kRed = 4 * 4 * 32 * 16;  // partial scores [warp][nt][lane] float4
  static constexpr size_t kPbuf = 4 * 32 * 16;     // probabilities [nt][lane] float4
  static constexpr size_t kSmall = 64 * 4 + 64 * 4 + 16 * 4;  // maxima, row sums, stage masks
  static constexpr size_t kBars = (2 * kStages + 4) * 8;
  static constexpr size_t kSmem = kRing + kRed + kPbuf + kSmall + kBars;
};

__device__ __forceinline__ float fmax4(float a, float b, float c, float d) {
  return fmaxf(fmaxf(a, b), fmaxf(c, d));
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, 2) decode_mma_kernel(const DecodeArgs p) {
  using C = Cfg<FMT>;
  constexpr bool kFp8 = C::kFp8;
  constexpr int RB = C::kRowBytes;
  constexpr int NST = C::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float4* red = reinterpret_cast<float4*>(smem + C::kRing);
  float4* pbuf = reinterpret_cast<float4*>(smem + C::kRing + C::kRed);
  float* mx = reinterpret_cast<float*>(smem + C::kRing + C::kRed + C::kPbuf);
  float* lsum = mx + 64;
  uint32_t* meta = reinterpret_cast<uint32_t*>(lsum + 64);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kRing + C::kRed + C::kPbuf + C::kSmall);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + NST), cbar0 = smem_u32(bars + 2 * NST);
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
        mbar_init(full0 + 8 * s, 1);
        mbar_init(empty0 + 8 * s, kConsumerWarps);
      }
      for (int k = 0; k < 4; ++k) mbar_init(cbar0 + 8 * k, kConsumerWarps);
      if (!req_ok) atomicOr(p.err, SMLA_DEVERR_INDEX);
    }
    __syncthreads();
  }

  // =================================================================== producer warp
  if (w == kConsumerWarps) {
    auto idx_at = [&](int tile) -> int32_t {
      const int j = j0 + tile * kSlots + lane;
      return (tile < ntiles && j < j1) ? __ldg(idx_row + j) : -1;
    };
    auto page_of = [&](int32_t idx) -> int32_t {
      return (idx >= 0 && (idx >> p.log2_page) < p.stride) ? __ldg(pt_row + (idx >> p.log2_page)) : -1;
    };
    int32_t idx_a = idx_at(0), idx_b = idx_at(1);
    int32_t pg_a = page_of(idx_a);
    int issued = 0;
    bool ok = true;
    for (int i = 0; i < ntiles; ++i) {
      const int32_t idx_c = idx_a, pg_c = pg_a;
      idx_a = idx_b;
      idx_b = idx_at(i + 2);
      pg_a = page_of(idx_a);
      const int st = i % NST;
      if (!mbar_wait(empty0 + 8 * st, ((i / NST) & 1) ^ 1)) {
        ok = false;
        break;
      }
      int64_t phys = -1;
      if (idx_c != -1) {
        if (idx_c < 0 || (idx_c >> p.log2_page) >= p.stride) {
          atomicOr(p.err, SMLA_DEVERR_INDEX);
        } else if (pg_c < 0 || pg_c >= p.num_pages) {
          atomicOr(p.err, SMLA_DEVERR_PAGE);
        } else {
          phys = (int64_t(pg_c) << p.log2_page) + (idx_c & ((1 << p.log2_page) - 1));
        }
      }
      const uint32_t vmask = __ballot_sync(0xffffffffu, phys >= 0);
      if (lane == 0) {
        meta[st] = vmask;
        mbar_arrive_expect_tx(full0 + 8 * st, uint32_t(__popc(vmask)) * RB);
      }
      __syncwarp();
      if (phys >= 0)
        bulk_g2s(ring_s + (st * kSlots + lane) * RB, p.kv + phys * RB, RB, full0 + 8 * st);
      issued = i + 1;
    }
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
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (kFp8) {
        qa[s][0] = bf16x2_to_f16x2(a[2 * s]);
        qa[s][1] = bf16x2_to_f16x2(b[2 * s]);
        qa[s][2] = bf16x2_to_f16x2(a[2 * s + 1]);
        qa[s][3] = bf16x2_to_f16x2(b[2 * s + 1]);
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
  }

  float O[8][2][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) O[i][j][e] = 0.f;
  float m_g = -CUDART_INF_F, m_g8 = -CUDART_INF_F, l_g = 0.f, l_g8 = 0.f;
  float mo[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
  const int oh[4] = {2 * c, 2 * c + 1, 2 * c + 8, 2 * c + 9};
  float r_w = 0.f;
  uint32_t cb_phase = 0;  // sync points completed by the 4 consumer warps
  bool ok = true;
  // consumer-only barrier (bounded): every consumer warp arrives once, then all wait
  // cbar 0..2 complete once per computed stage (parity = cb_phase & 1); cbar 3 once.
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
    const uint32_t msk = meta[st];
    if (msk != 0u) {
      const uint32_t sb = ring_s + st * kSlots * RB;
      // ---- QK partial over latent block w (+ RoPE quarter w)
      float sc[4][2];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const uint32_t rb = sb + (8 * nt + g) * RB;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (kFp8) {
          float accr[4] = {0.f, 0.f, 0.f, 0.f};
          const uint4 v0 = lds128(rb + 128 * w + 32 * c);
          const uint4 v1 = lds128(rb + 128 * w + 32 * c + 16);
          const uint32_t wd[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
          const uint2 rv = lds64(rb + kRopeOffFp8 + 2 * (16 * w + 4 * c));
          mma_bf16(accr, qr, rv.x, rv.y);
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            uint32_t b0, b1;
            e4m3x4_to_f16x4(wd[s], b0, b1);
            mma_f16(acc, qa[s], b0, b1);
          }
          sc[nt][0] = lds_f32(sb + (8 * nt + 2 * c) * RB + kScaleOff + 4 * w);
          sc[nt][1] = lds_f32(sb + (8 * nt + 2 * c + 1) * RB + kScaleOff + 4 * w);
          acc[0] = fmaf(acc[0], sc[nt][0], accr[0]);
          acc[1] = fmaf(acc[1], sc[nt][1], accr[1]);
          acc[2] = fmaf(acc[2], sc[nt][0], accr[2]);
          acc[3] = fmaf(acc[3], sc[nt][1], accr[3]);
        } else {
          const uint32_t base = rb + 2 * (128 * w + 32 * c);
          uint32_t wd[16];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = lds128(base + 16 * k);
            wd[4 * k] = v.x; wd[4 * k + 1] = v.y; wd[4 * k + 2] = v.z; wd[4 * k + 3] = v.w;
          }
#pragma unroll
          for (int s = 0; s < 8; ++s) mma_bf16(acc, qa[s], wd[2 * s], wd[2 * s + 1]);
          const uint2 rv = lds64(rb + 2 * kLatent + 2 * (16 * w + 4 * c));
          mma_bf16(acc, qr, rv.x, rv.y);
          sc[nt][0] = 1.f;
          sc[nt][1] = 1.f;
        }
        red[(w * 4 + nt) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      }
      if (!(ok = csync(0, cb_phase))) break;

      // ---- scores of slots [8w, 8w+8): sum partials, scale, mask, stage max
      float s4[4];
      {
        const float4 a = red[(0 * 4 + w) * 32 + lane], b = red[(1 * 4 + w) * 32 + lane];
        const float4 cc = red[(2 * 4 + w) * 32 + lane], d = red[(3 * 4 + w) * 32 + lane];
        const int sl = 8 * w + 2 * c;
        const bool v0 = (msk >> sl) & 1u, v1 = (msk >> (sl + 1)) & 1u;
        s4[0] = v0 ? ((a.x + b.x) + (cc.x + d.x)) * p.c2 : -CUDART_INF_F;
        s4[1] = v1 ? ((a.y + b.y) + (cc.y + d.y)) * p.c2 : -CUDART_INF_F;
        s4[2] = v0 ? ((a.z + b.z) + (cc.z + d.z)) * p.c2 : -CUDART_INF_F;
        s4[3] = v1 ? ((a.w + b.w) + (cc.w + d.w)) * p.c2 : -CUDART_INF_F;
      }
      float mg = fmaxf(s4[0], s4[1]), mg8 = fmaxf(s4[2], s4[3]);
      mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, 1));
      mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, 2));
      mg8 = fmaxf(mg8, __shfl_xor_sync(0xffffffffu, mg8, 1));
      mg8 = fmaxf(mg8, __shfl_xor_sync(0xffffffffu, mg8, 2));
      if (c == 0) {
        mx[w * 16 + g] = mg;
        mx[w * 16 + g + 8] = mg8;
      }
      if (!(ok = csync(1, cb_phase))) break;

      // ---- online softmax (base 2) for the owned slots
      auto tmax = [&](int h) { return fmax4(mx[h], mx[16 + h], mx[32 + h], mx[48 + h]); };
      {
        const float ng = fmaxf(m_g, tmax(g)), ng8 = fmaxf(m_g8, tmax(g + 8));
        const float bg = ng == -CUDART_INF_F ? 0.f : ng;
        const float bg8 = ng8 == -CUDART_INF_F ? 0.f : ng8;
        const float p0 = exp2f(s4[0] - bg), p1 = exp2f(s4[1] - bg);
        const float p2 = exp2f(s4[2] - bg8), p3 = exp2f(s4[3] - bg8);
        l_g = l_g * exp2f(m_g - bg) + (p0 + p1);
        l_g8 = l_g8 * exp2f(m_g8 - bg8) + (p2 + p3);
        m_g = ng;
        m_g8 = ng8;
        pbuf[w * 32 + lane] = make_float4(p0, p1, p2, p3);
      }
      float alpha[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float n = fmaxf(mo[k], tmax(oh[k]));
        alpha[k] = exp2f(mo[k] - (n == -CUDART_INF_F ? 0.f : n));
        mo[k] = n;
      }
      float tm = fmax4(sc[0][0], sc[0][1], sc[1][0], sc[1][1]);
      tm = fmaxf(tm, fmax4(sc[2][0], sc[2][1], sc[3][0], sc[3][1]));
      tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1));
      tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
      const float r_new = fmaxf(r_w, tm);
      const float rr = r_new > 0.f ? r_w / r_new : 1.f;
      r_w = r_new;
      const float inv_r = r_new > 0.f ? 1.f / r_new : 0.f;
      if (!(ok = csync(2, cb_phase))) break;
      ++cb_phase;

      // ---- PV: O^T[128w.., heads] += V^T P^T
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) O[mt][nt][e] *= alpha[2 * nt + (e & 1)] * rr;

#pragma unroll
      for (int kc = 0; kc < 2; ++kc) {
        const float4 pa = pbuf[(2 * kc) * 32 + lane], pc = pbuf[(2 * kc + 1) * 32 + lane];
        const float f0 = sc[2 * kc][0] * inv_r, f1 = sc[2 * kc][1] * inv_r;
        const float f2 = sc[2 * kc + 1][0] * inv_r, f3 = sc[2 * kc + 1][1] * inv_r;
        uint32_t bh0[2], bh1[2];
        if (kFp8) {
          bh0[0] = pack_f16x2(pa.x * f0, pa.y * f1);
          bh0[1] = pack_f16x2(pc.x * f2, pc.y * f3);
          bh1[0] = pack_f16x2(pa.z * f0, pa.w * f1);
          bh1[1] = pack_f16x2(pc.z * f2, pc.w * f3);
        } else {
          bh0[0] = pack_bf16x2(pa.x, pa.y);
          bh0[1] = pack_bf16x2(pc.x, pc.y);
          bh1[0] = pack_bf16x2(pa.z, pa.w);
          bh1[1] = pack_bf16x2(pc.z, pc.w);
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
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
  }
  if (!ok) {
    if (lane == 0) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
    return;
  }

  // ---- epilogue
  l_g += __shfl_xor_sync(0xffffffffu, l_g, 1);
  l_g += __shfl_xor_sync(0xffffffffu, l_g, 2);
  l_g8 += __shfl_xor_sync(0xffffffffu, l_g8, 1);
  l_g8 += __shfl_xor_sync(0xffffffffu, l_g8, 2);
  if (c == 0) {
    lsum[w * 16 + g] = l_g;
    lsum[w * 16 + g + 8] = l_g8;
  }
  if (!csync(3, 0)) {
    if (lane == 0) atomicOr(p.err, SMLA_DEVERR_TIMEOUT);
    return;
  }
  const int S = p.num_splits;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int h = oh[k];
    const float L = (lsum[h] + lsum[16 + h]) + (lsum[32 + h] + lsum[48 + h]);
    const float lse0 = L > 0.f ? (mo[k] + log2f(L)) * kLn2 : -CUDART_INF_F;
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

// Merge of split partials by log-sum-exp, then the sink (SGLang PR #24692 "关键文件":
// _merge_partial_attn, _apply_attn_sink). One CTA per (token, 16 heads).
__global__ void __launch_bounds__(256) merge_kernel(const DecodeArgs p) {
  __shared__ float wts[16][kMaxSplits];
  __shared__ float fac[16];
  const int HG = p.H >> 4;
  const int t = blockIdx.x / HG, h0 = (blockIdx.x % HG) * 16;
  const int S = p.num_splits;
  if (threadIdx.x < 16) {
    const int h = h0 + threadIdx.x;
    const float* lp = p.lse_part + int64_t(t) * S * p.H + h;
    float M = -CUDART_INF_F;
    for (int s = 0; s < S; ++s) M = fmaxf(M, lp[int64_t(s) * p.H]);
    float W = 0.f;
    for (int s = 0; s < S; ++s) {
      const float x = lp[int64_t(s) * p.H];
      const float wt = (M == -CUDART_INF_F || x == -CUDART_INF_F) ? 0.f : expf(x - M);
      wts[threadIdx.x][s] = wt;
      W += wt;
    }
    const float lse0 = W > 0.f ? M + logf(W) : -CUDART_INF_F;
    float lse = lse0;
    float f = W > 0.f ? 1.f / W : 0.f;
    if (p.sink) {
      const float sg = __ldg(p.sink + h);
      lse = fmaxf(lse0, sg) + log1pf(expf(-fabsf(lse0 - sg)));
      f *= expf(lse0 - lse);
    }
    fac[threadIdx.x] = f;
    if (p.lse) p.lse[int64_t(t) * p.H + h] = lse;
  }
  __syncthreads();
  for (int e = threadIdx.x * 4; e < 16 * kLatent; e += blockDim.x * 4) {
    const int hl = e / kLatent, d = e % kLatent;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; ++s) {
      const float wt = wts[hl][s];
      if (wt == 0.f) continue;
      const float4 o = *reinterpret_cast<const float4*>(
          p.o_part + ((int64_t(t) * S + s) * p.H + h0 + hl) * kLatent + d);
      acc.x = fmaf(wt, o.x, acc.x);
      acc.y = fmaf(wt, o.y, acc.y);
      acc.z = fmaf(wt, o.z, acc.z);
      acc.w = fmaf(wt, o.w, acc.w);
    }
    const float f = fac[hl];
    uint2 pk = make_uint2(pack_bf16x2(acc.x * f, acc.y * f), pack_bf16x2(acc.z * f, acc.w * f));
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) +
                              (int64_t(t) * p.H + h0 + hl) * kLatent + d) = pk;
  }
}

template <int FMT>
cudaError_t launch_fmt(const DecodeArgs& a, cudaStream_t s) {
  const size_t smem = Cfg<FMT>::kSmem;
  static int configured_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<FMT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  const int64_t grid = int64_t(a.T) * a.num_splits * (a.H >> 4);
  decode_mma_kernel<FMT><<<static_cast<unsigned>(grid), kThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_mma(const DecodeArgs& a, int /*num_sms*/, cudaStream_t s) {
  return a.kv_format == SMLA_KV_FP8_DS ? launch_fmt<SMLA_KV_FP8_DS>(a, s)
                                       : launch_fmt<SMLA_KV_BF16>(a, s);
}

cudaError_t launch_merge(const DecodeArgs& a, cudaStream_t s) {
  merge_kernel<<<static_cast<unsigned>(a.T * (a.H >> 4)), 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace smla
