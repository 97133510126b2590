// Sparse MLA decode, warp-level tensor-core path (mma.sync m16n8k16), one CTA per
// (query token, top-k split, group of 16 heads).
//
// What it computes (vLLM PR #43477 "关键源码片段", forward_mqa; SGLang PR #24692
// "实现拆解 2": tiled sparse decode with online softmax, split merge, sink): for each
// selected slot j, s_j = sm_scale * <q_h, k_j> over 576 dims, out_h = softmax-weighted
// sum of v_j = k_j[0:512].
//
// Design (4 warps, warp w owns latent block w = dims [128w, 128w+128)):
//  * Gather: the top-k list of the split is walked in tiles of 64 slots. Threads 0..63
//    translate each slot's index through the page table one tile ahead of use; all 128
//    threads then copy whole rows into a 2-stage shared-memory ring with 16-byte
//    cp.async (zero-fill for padding: padded rows are never read from HBM).
//  * QK: warp w multiplies its 128 latent dims (+ RoPE dims [16w, 16w+16)) for all 64
//    slots. q is held in registers as A fragments (f16 for the latent, bf16 for RoPE).
//    B fragments are built straight from the staged E4M3 bytes with cvt.rn.f16x2.e4m3x2:
//    the k order inside an mma is permuted so that each thread reads 16 contiguous bytes
//    of one row, and q is permuted the same way. The per-128 scale multiplies the fp32
//    partial score of block w (exact for the fp32 product it replaces up to rounding).
//  * The four partial scores are summed through shared memory; warp w then owns slots
//    [16w, 16w+16) of the tile for the masked online softmax (base-2, running max).
//  * PV: O^T[dims, heads] = V^T P^T. Warp w accumulates its 128 output dims. A fragments
//    (V^T) come from the staged bytes of four rows, paired by prmt and converted; the
//    B fragments are the probabilities times scale_w[j] / r_w, where r_w is the running
//    maximum of scale_w over the slots seen (keeps the f16 operand in [0, 1]).
//  * Epilogue: o = O * r_w / l and lse = (m + log2 l) * ln 2. With one split the sink is
//    applied here and bf16 out / fp32 lse are written; otherwise the fp32 partials go to
//    the workspace and the merge kernel finishes.
#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace smla {
namespace {

constexpr int kThreads = 128;
constexpr int kStages = 2;  // 2 x 64-row stages: bf16 fits, and two CTAs per SM for fp8_ds
constexpr int kRing = kStages + 1;

template <int FMT>
struct Fmt {
  static constexpr int kRowBytes = FMT == SMLA_KV_FP8_DS ? kFp8RowBytes : kBf16RowBytes;
  static constexpr int kChunks = kRowBytes / 16;
};

template <int FMT>
constexpr size_t smem_bytes() {
  return size_t(kStages) * kTile * Fmt<FMT>::kRowBytes  // stage ring
         + 4 * 8 * 32 * 16                              // partial scores
         + 4 * 32 * 8 * 4                               // probabilities
         + 64 * 4 + 64 * 4                              // tile maxima, row sums
         + kRing * kTile * 8                            // physical slot ring
         + kRing * 2 * 4;                               // valid masks
}

__device__ __forceinline__ float fmax4(float a, float b, float c, float d) {
  return fmaxf(fmaxf(a, b), fmaxf(c, d));
}

template <int FMT>
__global__ void __launch_bounds__(kThreads) decode_mma_kernel(const DecodeArgs p) {
  constexpr bool kFp8 = FMT == SMLA_KV_FP8_DS;
  constexpr int RB = Fmt<FMT>::kRowBytes;
  constexpr int CH = Fmt<FMT>::kChunks;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stage = smem;
  float4* red = reinterpret_cast<float4*>(smem + size_t(kStages) * kTile * RB);
  float* pbuf = reinterpret_cast<float*>(red + 4 * 8 * 32);
  float* mx = pbuf + 4 * 32 * 8;
  float* lsum = mx + 64;
  int64_t* ring = reinterpret_cast<int64_t*>(lsum + 64);
  uint32_t* ring_mask = reinterpret_cast<uint32_t*>(ring + kRing * kTile);

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
  if (!req_ok && tid == 0 && hg == 0 && split == 0) atomicOr(p.err, SMLA_DEVERR_INDEX);
  const int32_t* pt_row = p.page_table + int64_t(req_ok ? r : 0) * p.stride;
  const int32_t* idx_row = p.topk + int64_t(t) * p.K;
  const int j0 = split * p.split_len;
  const int j1 = min(p.K, j0 + p.split_len);
  const int ntiles = req_ok ? max(0, (j1 - j0 + kTile - 1) / kTile) : 0;

  // ---- q fragments (registers for the whole kernel)
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

  // ---- slot bookkeeping
  auto load_idx = [&](int tile) -> int32_t {
    const int j = j0 + tile * kTile + tid;
    return (tile < ntiles && j < j1) ? __ldg(idx_row + j) : -1;
  };
  auto issue = [&](int tile) {
    const uint32_t st = smem_u32(stage + (tile % kStages) * kTile * RB);
    const int64_t* ph = ring + (tile % kRing) * kTile;
    for (int L = tid; L < kTile * CH; L += kThreads) {
      const int row = L / CH, ch = L - row * CH;
      const int64_t s = ph[row];
      const uint8_t* src = s >= 0 ? p.kv + s * RB + ch * 16 : p.kv;
      cp_async16(st + row * RB + ch * 16, src, s >= 0 ? 16 : 0);
    }
  };
  auto publish = [&](int tile, int64_t phys) {  // threads 0..63
    const int e = tile % kRing;
    ring[e * kTile + tid] = phys;
    const uint32_t m = __ballot_sync(0xffffffffu, phys >= 0);
    if (lane == 0) ring_mask[e * 2 + w] = m;
  };

  if (tid < kTile) {
#pragma unroll 1
    for (int s = 0; s < kStages; ++s)
      publish(s, translate_index(load_idx(s), pt_row, p.stride, p.log2_page, p.num_pages, p.err));
  }
  __syncthreads();
#pragma unroll 1
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < ntiles) issue(s);
    cp_async_commit();
  }
  int32_t idx_reg = tid < kTile ? load_idx(kStages) : -1;

  // ---- running state
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

#pragma unroll 1
  for (int i = 0; i < ntiles; ++i) {
    __syncthreads();  // stage (i-1) free, ring entry for tile i+kStages-1 visible
    if (i + kStages - 1 < ntiles) issue(i + kStages - 1);
    cp_async_commit();
    // look-ahead index translation for tile i+kStages: issue the page-table load now,
    // use it after this tile's compute.
    int32_t page_raw = -1;
    int32_t idx_cur = idx_reg;
    if (tid < kTile) {
      if (idx_cur >= 0 && (idx_cur >> p.log2_page) < p.stride)
        page_raw = __ldg(pt_row + (idx_cur >> p.log2_page));
      idx_reg = load_idx(i + kStages + 1);
    }
    cp_async_wait<kStages - 1>();
    __syncthreads();

    const int e_ring = i % kRing;
    const uint32_t msk0 = ring_mask[e_ring * 2], msk1 = ring_mask[e_ring * 2 + 1];
    if ((msk0 | msk1) != 0u) {
      const uint32_t st = smem_u32(stage + (i % kStages) * kTile * RB);
      // ---- QK partial over latent block w (+ RoPE quarter w)
      float sc[8][2];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const uint32_t rb = st + (8 * nt + g) * RB;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        if (kFp8) {
          float accr[4] = {0.f, 0.f, 0.f, 0.f};
          const uint4 v0 = lds128(rb + 128 * w + 32 * c);
          const uint4 v1 = lds128(rb + 128 * w + 32 * c + 16);
          const uint32_t wd[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            uint32_t b0, b1;
            e4m3x4_to_f16x4(wd[s], b0, b1);
            mma_f16(acc, qa[s], b0, b1);
          }
          const uint2 rv = lds64(rb + kRopeOffFp8 + 2 * (16 * w + 4 * c));
          mma_bf16(accr, qr, rv.x, rv.y);
          sc[nt][0] = lds_f32(st + (8 * nt + 2 * c) * RB + kScaleOff + 4 * w);
          sc[nt][1] = lds_f32(st + (8 * nt + 2 * c + 1) * RB + kScaleOff + 4 * w);
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
        red[(w * 8 + nt) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      }
      __syncthreads();

      // ---- scores of slots [16w, 16w+16): sum partials, scale, mask, tile max
      float s[2][4];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int nt = 2 * w + u;
        float4 a = red[(0 * 8 + nt) * 32 + lane];
        const float4 b = red[(1 * 8 + nt) * 32 + lane];
        const float4 cc = red[(2 * 8 + nt) * 32 + lane];
        const float4 d = red[(3 * 8 + nt) * 32 + lane];
        a.x = (a.x + b.x) + (cc.x + d.x);
        a.y = (a.y + b.y) + (cc.y + d.y);
        a.z = (a.z + b.z) + (cc.z + d.z);
        a.w = (a.w + b.w) + (cc.w + d.w);
        const int sl = 16 * w + 8 * u + 2 * c;
        const uint32_t mk = sl < 32 ? msk0 : msk1;
        const bool v0 = (mk >> (sl & 31)) & 1u, v1 = (mk >> ((sl + 1) & 31)) & 1u;
        s[u][0] = v0 ? a.x * p.c2 : -CUDART_INF_F;
        s[u][1] = v1 ? a.y * p.c2 : -CUDART_INF_F;
        s[u][2] = v0 ? a.z * p.c2 : -CUDART_INF_F;
        s[u][3] = v1 ? a.w * p.c2 : -CUDART_INF_F;
      }
      float mg = fmax4(s[0][0], s[0][1], s[1][0], s[1][1]);
      float mg8 = fmax4(s[0][2], s[0][3], s[1][2], s[1][3]);
      mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, 1));
      mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, 2));
      mg8 = fmaxf(mg8, __shfl_xor_sync(0xffffffffu, mg8, 1));
      mg8 = fmaxf(mg8, __shfl_xor_sync(0xffffffffu, mg8, 2));
      if (c == 0) {
        mx[w * 16 + g] = mg;
        mx[w * 16 + g + 8] = mg8;
      }
      __syncthreads();

      // ---- online softmax (base 2) for the owned slots; probabilities to shared memory
      auto tmax = [&](int h) { return fmax4(mx[h], mx[16 + h], mx[32 + h], mx[48 + h]); };
      {
        const float ng = fmaxf(m_g, tmax(g)), ng8 = fmaxf(m_g8, tmax(g + 8));
        const float bg = ng == -CUDART_INF_F ? 0.f : ng;
        const float bg8 = ng8 == -CUDART_INF_F ? 0.f : ng8;
        float pr[8];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          pr[4 * u + 0] = exp2f(s[u][0] - bg);
          pr[4 * u + 1] = exp2f(s[u][1] - bg);
          pr[4 * u + 2] = exp2f(s[u][2] - bg8);
          pr[4 * u + 3] = exp2f(s[u][3] - bg8);
        }
        l_g = l_g * exp2f(m_g - bg) + ((pr[0] + pr[1]) + (pr[4] + pr[5]));
        l_g8 = l_g8 * exp2f(m_g8 - bg8) + ((pr[2] + pr[3]) + (pr[6] + pr[7]));
        m_g = ng;
        m_g8 = ng8;
        float4* pb = reinterpret_cast<float4*>(pbuf + (w * 32 + lane) * 8);
        pb[0] = make_float4(pr[0], pr[1], pr[2], pr[3]);
        pb[1] = make_float4(pr[4], pr[5], pr[6], pr[7]);
      }
      float alpha[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float n = fmaxf(mo[k], tmax(oh[k]));
        alpha[k] = exp2f(mo[k] - (n == -CUDART_INF_F ? 0.f : n));
        mo[k] = n;
      }
      // running maximum of scale_w over the slots seen so far
      float tm = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) tm = fmax4(tm, sc[nt][0], sc[nt][1], 0.f);
      tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 1));
      tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 2));
      const float r_new = fmaxf(r_w, tm);
      const float rr = r_new > 0.f ? r_w / r_new : 1.f;
      r_w = r_new;
      const float inv_r = r_new > 0.f ? 1.f / r_new : 0.f;
      __syncthreads();

      // ---- PV: O^T[128w.., heads] += V^T P^T
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) O[mt][nt][e] *= alpha[2 * nt + (e & 1)] * rr;

#pragma unroll
      for (int kc = 0; kc < 4; ++kc) {
        const float4* pb = reinterpret_cast<const float4*>(pbuf + (kc * 32 + lane) * 8);
        const float4 pa = pb[0], pc = pb[1];
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
        const uint32_t r0 = st + (16 * kc + 2 * c) * RB;
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

    // publish the translated slots of tile i+kStages (used two iterations from now)
    if (tid < kTile) {
      int64_t phys = -1;
      if (idx_cur != -1) {
        if (idx_cur < 0 || (idx_cur >> p.log2_page) >= p.stride) {
          atomicOr(p.err, SMLA_DEVERR_INDEX);
        } else if (page_raw < 0 || page_raw >= p.num_pages) {
          atomicOr(p.err, SMLA_DEVERR_PAGE);
        } else {
          phys = (int64_t(page_raw) << p.log2_page) + (idx_cur & ((1 << p.log2_page) - 1));
        }
      }
      publish(i + kStages, phys);
    }
  }
  cp_async_wait<0>();

  // ---- epilogue
  l_g += __shfl_xor_sync(0xffffffffu, l_g, 1);
  l_g += __shfl_xor_sync(0xffffffffu, l_g, 2);
  l_g8 += __shfl_xor_sync(0xffffffffu, l_g8, 1);
  l_g8 += __shfl_xor_sync(0xffffffffu, l_g8, 2);
  __syncthreads();
  if (c == 0) {
    lsum[w * 16 + g] = l_g;
    lsum[w * 16 + g + 8] = l_g8;
  }
  __syncthreads();
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
  // 16 heads x 512 dims, 4 consecutive dims per thread step
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
  const size_t smem = smem_bytes<FMT>();
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
