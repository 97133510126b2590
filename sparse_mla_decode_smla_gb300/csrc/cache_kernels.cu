// Cache-row kernels: the quantise-on-write store (smla_pack_kv) and the gather +
// dequantise test hook (smla_gather_dequant).
//
// fp8_ds_mla row (656 B): 512 E4M3FN codes | 4 fp32 scales | 64 bf16 RoPE; scale b
// covers latent dims [128b, 128b+128) (vLLM PR #43477 "实现拆解 1": the fp8_ds_mla
// cache; vLLM PR #43827 "功能与动机": the "UE8M0 paged" FlashMLA layout, i.e. power-of-
// two block scales).
// Per-tensor FP8 row (576 B): 576 E4M3FN codes [latent 512 | RoPE 64] of x / kv_scale,
// one scale for the whole cache (vLLM PR #43827 "实现拆解 4": store_full_fp8).
#include <string.h>

#include "common.cuh"
#include "kernels.h"

namespace smla {

// The norm and rotation of the fused store (the compressor's store of vLLM PR #43827,
// "实现拆解 4-6": norm, RoPE and the cache write in one kernel). Inputs and outputs are bf16.
struct NormRope {
  const uint4* weight;     // [512] bf16 RMSNorm weight
  float eps;
  const int64_t* positions;  // [n] rotary positions
  const float* cos_sin;    // [max_position, 64] fp32: cos of the 32 pair angles, then their sin
  int64_t max_position;
  int32_t* err;            // rows whose position is outside [0, max_position) set SMLA_DEVERR_INDEX
};

__device__ __forceinline__ uint32_t bf16x2_pack_rn(float lo, float hi) { return pack_bf16x2(lo, hi); }

// x / scale for the E4M3 conversion. Where scale is a power of two in [2^-126, 2^126] its
// reciprocal is exact, so x * (1 / scale) is the same real number x / scale rounded once: the
// same fp32 value as the correctly rounded division, for every x. Otherwise divide.
struct ScaleDiv {
  float scale, inv;
  bool exact;
  __device__ __forceinline__ explicit ScaleDiv(float sc) : scale(sc) {
    const uint32_t b = __float_as_uint(sc);
    exact = (b & 0x007fffffu) == 0u && sc >= 0x1p-126f && sc <= 0x1p126f;
    inv = exact ? __frcp_rn(sc) : 0.f;
  }
  // E4M3 codes of x[0..2n) / scale, two per 16-bit word: one branch for the whole run
  template <int N>
  __device__ __forceinline__ void codes(const float* x, uint16_t* out) const {
    if (exact) {
#pragma unroll
      for (int i = 0; i < N; ++i) out[i] = f32x2_to_e4m3x2(__fmul_rn(x[2 * i], inv), __fmul_rn(x[2 * i + 1], inv));
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i)
        out[i] = f32x2_to_e4m3x2(__fdiv_rn(x[2 * i], scale), __fdiv_rn(x[2 * i + 1], scale));
    }
  }
};

// One warp per row. Lane l owns latent elements [16l, 16l+16); lanes 8b..8b+7 form block b.
// With NORM the row is first normalised (RMSNorm over the 512 latent dims: fp32 sum of
// squares in a fixed order, correctly rounded sqrt and divide, x * r * w rounded to bf16) and
// its RoPE pairs (2j, 2j+1) are rotated, (a c - b s, a s + b c) rounded to bf16.
// The kernel waits on one memory round trip per row, so its speed follows the rows in flight:
// the FP8 variants are held to 40 registers for six blocks per SM (measured faster than five,
// despite a few spilled words); the bf16 one at five blocks, 48 registers.
template <int FMT, bool NORM>
__global__ void __launch_bounds__(256, FMT == SMLA_KV_BF16 ? 5 : 6) pack_kernel(const uint4* __restrict__ latent,
                                                   const uint4* __restrict__ rope,
                                                   const int64_t* __restrict__ slot_mapping,
                                                   int64_t n, uint8_t* __restrict__ kv,
                                                   int64_t num_slots, int scale_mode,
                                                   float kv_scale, const NormRope nr) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (row >= n) return;
  // every load of the row is issued before the first one is used (all lie inside the row's
  // own inputs), so the warp waits for one memory round trip, not one per dependent load
  const int64_t slot = slot_mapping[row];
  uint4 x0 = latent[row * 64 + 2 * lane];
  uint4 x1 = latent[row * 64 + 2 * lane + 1];
  uint4 rp = lane < 8 ? rope[row * 8 + lane] : make_uint4(0, 0, 0, 0);  // RoPE dims [8 lane, +8)
  int64_t pos = 0;
  if constexpr (NORM) pos = nr.positions[row];
  if (slot < 0 || slot >= num_slots) return;
  if constexpr (NORM) {
    if (pos < 0 || pos >= nr.max_position) {  // the whole warp agrees: skip the row, flag it
      if (lane == 0 && nr.err) atomicOr(nr.err, SMLA_DEVERR_INDEX);
      return;
    }
    const uint4 g0 = nr.weight[2 * lane], g1 = nr.weight[2 * lane + 1];
    float4 c4 = make_float4(0.f, 0.f, 0.f, 0.f), s4 = c4;
    if (lane < 8) {  // cos and sin of the RoPE pairs 4 lane .. 4 lane + 3
      const float4* cs = reinterpret_cast<const float4*>(nr.cos_sin + pos * 64);
      c4 = cs[lane];
      s4 = cs[8 + lane];
    }
    uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(bf16_hi(w[i]), bf16_hi(w[i]), fmaf(bf16_lo(w[i]), bf16_lo(w[i]), ss));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float r = __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(ss, 1.f / kLatent), nr.eps)));  // 1/512: exact
    const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = bf16x2_pack_rn(__fmul_rn(__fmul_rn(bf16_lo(w[i]), r), bf16_lo(gw[i])),
                            __fmul_rn(__fmul_rn(bf16_hi(w[i]), r), bf16_hi(gw[i])));
    x0 = make_uint4(w[0], w[1], w[2], w[3]);
    x1 = make_uint4(w[4], w[5], w[6], w[7]);
    if (lane < 8) {  // pairs j = 4 lane .. 4 lane + 3, one per bf16 word
      const float cv[4] = {c4.x, c4.y, c4.z, c4.w}, sv[4] = {s4.x, s4.y, s4.z, s4.w};
      uint32_t rw[4] = {rp.x, rp.y, rp.z, rp.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float c = cv[k], sn = sv[k];
        const float a = bf16_lo(rw[k]), b = bf16_hi(rw[k]);
        rw[k] = bf16x2_pack_rn(__fsub_rn(__fmul_rn(a, c), __fmul_rn(b, sn)), __fadd_rn(__fmul_rn(a, sn), __fmul_rn(b, c)));
      }
      rp = make_uint4(rw[0], rw[1], rw[2], rw[3]);
    }
  }
  if (FMT == SMLA_KV_BF16) {
    uint4* dst = reinterpret_cast<uint4*>(kv + slot * kBf16RowBytes);
    dst[2 * lane] = x0;
    dst[2 * lane + 1] = x1;
    if (lane < 8) dst[64 + lane] = rp;
    return;
  }
  if (FMT == SMLA_KV_FP8_TENSOR) {
    uint8_t* dst = kv + slot * kFp8TensorRowBytes;
    const ScaleDiv dv(kv_scale);
    const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = bf16_lo(w[i]);
      v[2 * i + 1] = bf16_hi(w[i]);
    }
    uint16_t c[8];
    dv.codes<8>(v, c);
    *reinterpret_cast<uint4*>(dst + 16 * lane) =
        make_uint4(c[0] | (uint32_t(c[1]) << 16), c[2] | (uint32_t(c[3]) << 16), c[4] | (uint32_t(c[5]) << 16),
                   c[6] | (uint32_t(c[7]) << 16));
    if (lane < 8) {  // RoPE values [8 lane, 8 lane + 8)
      const uint32_t rw[4] = {rp.x, rp.y, rp.z, rp.w};
      float r[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        r[2 * i] = bf16_lo(rw[i]);
        r[2 * i + 1] = bf16_hi(rw[i]);
      }
      uint16_t rc[4];
      dv.codes<4>(r, rc);
      *reinterpret_cast<uint2*>(dst + kLatent + 8 * lane) =
          make_uint2(rc[0] | (uint32_t(rc[1]) << 16), rc[2] | (uint32_t(rc[3]) << 16));
    }
    return;
  }
  const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  float v[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = bf16_lo(w[i]);
    v[2 * i + 1] = bf16_hi(w[i]);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  float scale = 1.f;
  if (amax > 0.f) {
    const float ratio = __fdiv_rn(amax, 448.f);
    if (scale_mode == SMLA_SCALE_POW2) {
      int e;
      const float m = frexpf(ratio, &e);  // ratio = m * 2^e, m in [0.5, 1)
      scale = (m == 0.5f) ? ratio : ldexpf(1.f, e);
    } else {
      scale = ratio;
    }
  }
  uint16_t c[8];
  ScaleDiv(scale).codes<8>(v, c);
  uint8_t* dst = kv + slot * kFp8RowBytes;
  *reinterpret_cast<uint4*>(dst + 16 * lane) =
      make_uint4(c[0] | (uint32_t(c[1]) << 16), c[2] | (uint32_t(c[3]) << 16), c[4] | (uint32_t(c[5]) << 16),
                 c[6] | (uint32_t(c[7]) << 16));
  const float s1 = __shfl_sync(0xffffffffu, scale, 8);
  const float s2 = __shfl_sync(0xffffffffu, scale, 16);
  const float s3 = __shfl_sync(0xffffffffu, scale, 24);
  if (lane == 0) *reinterpret_cast<float4*>(dst + kScaleOff) = make_float4(scale, s1, s2, s3);
  if (lane < 8) *reinterpret_cast<uint4*>(dst + kRopeOffFp8 + 16 * lane) = rp;
}

template <bool NORM>
cudaError_t launch_pack_impl(int32_t kv_format, int32_t scale_mode, float kv_scale, const void* latent,
                             const void* rope, const int64_t* slot_mapping, int64_t n, void* kv,
                             int64_t num_slots, const NormRope& nr, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int64_t blocks = (n * 32 + 255) / 256;
  auto* L = static_cast<const uint4*>(latent);
  auto* R = static_cast<const uint4*>(rope);
  auto* K = static_cast<uint8_t*>(kv);
  if (kv_format == SMLA_KV_FP8_DS)
    pack_kernel<SMLA_KV_FP8_DS, NORM><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        L, R, slot_mapping, n, K, num_slots, scale_mode, kv_scale, nr);
  else if (kv_format == SMLA_KV_FP8_TENSOR)
    pack_kernel<SMLA_KV_FP8_TENSOR, NORM><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        L, R, slot_mapping, n, K, num_slots, scale_mode, kv_scale, nr);
  else
    pack_kernel<SMLA_KV_BF16, NORM><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        L, R, slot_mapping, n, K, num_slots, scale_mode, kv_scale, nr);
  return cudaGetLastError();
}

cudaError_t launch_pack(int32_t kv_format, int32_t scale_mode, float kv_scale, const void* latent,
                        const void* rope, const int64_t* slot_mapping, int64_t n, void* kv,
                        int64_t num_slots, cudaStream_t s) {
  NormRope none;
  memset(&none, 0, sizeof(none));
  return launch_pack_impl<false>(kv_format, scale_mode, kv_scale, latent, rope, slot_mapping, n, kv, num_slots,
                                 none, s);
}

cudaError_t launch_store_normed(int32_t kv_format, int32_t scale_mode, float kv_scale, const void* latent,
                                const void* rope, const void* weight, float eps, const int64_t* positions,
                                const float* cos_sin, int64_t max_position, const int64_t* slot_mapping,
                                int64_t n, void* kv, int64_t num_slots, int32_t* err, cudaStream_t s) {
  NormRope nr;
  nr.weight = static_cast<const uint4*>(weight);
  nr.eps = eps;
  nr.positions = positions;
  nr.cos_sin = cos_sin;
  nr.max_position = max_position;
  nr.err = err;
  return launch_pack_impl<true>(kv_format, scale_mode, kv_scale, latent, rope, slot_mapping, n, kv, num_slots, nr,
                                s);
}

// One warp per (token, top-k position). Lane l writes latent dims [16l, 16l+16) and
// RoPE dims [2l, 2l+2).
__global__ void __launch_bounds__(256) gather_dequant_kernel(DecodeArgs a, float* __restrict__ rows) {
  const int lane = threadIdx.x & 31;
  const int64_t item = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (item >= static_cast<int64_t>(a.T) * a.K) return;
  const int t = static_cast<int>(item / a.K);
  const int r = a.req_id ? a.req_id[t] : t / a.next_n;
  float* dst = rows + item * kDim;
  int64_t slot = -1;
  if (r >= 0 && r < a.B) {
    slot = translate_index(a.topk[item], a.page_table + static_cast<int64_t>(r) * a.stride,
                           a.stride, a.log2_page, a.num_pages, lane == 0 ? a.err : nullptr);
  } else if (lane == 0 && a.err) {
    atomicOr(a.err, SMLA_DEVERR_INDEX);
  }
  float v[16];
  float rp0 = 0.f, rp1 = 0.f;
  if (slot < 0) {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.f;
  } else if (a.kv_format == SMLA_KV_FP8_DS) {
    const uint8_t* src = a.kv + slot * kFp8RowBytes;
    const uint4 c = *reinterpret_cast<const uint4*>(src + 16 * lane);
    const float scale = reinterpret_cast<const float*>(src + kScaleOff)[lane >> 3];
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t lo, hi;
      e4m3x4_to_f16x4(w[i], lo, hi);
      const float2 f0 = __half22float2(*reinterpret_cast<__half2*>(&lo));
      const float2 f1 = __half22float2(*reinterpret_cast<__half2*>(&hi));
      v[4 * i] = __fmul_rn(f0.x, scale);
      v[4 * i + 1] = __fmul_rn(f0.y, scale);
      v[4 * i + 2] = __fmul_rn(f1.x, scale);
      v[4 * i + 3] = __fmul_rn(f1.y, scale);
    }
    const uint32_t rw = reinterpret_cast<const uint32_t*>(src + kRopeOffFp8)[lane];
    rp0 = bf16_lo(rw);
    rp1 = bf16_hi(rw);
  } else if (a.kv_format == SMLA_KV_FP8_TENSOR) {
    const uint8_t* src = a.kv + slot * kFp8TensorRowBytes;
    const uint4 c = *reinterpret_cast<const uint4*>(src + 16 * lane);
    const float scale = a.kv_scale;
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t lo, hi;
      e4m3x4_to_f16x4(w[i], lo, hi);
      const float2 f0 = __half22float2(*reinterpret_cast<__half2*>(&lo));
      const float2 f1 = __half22float2(*reinterpret_cast<__half2*>(&hi));
      v[4 * i] = __fmul_rn(f0.x, scale);
      v[4 * i + 1] = __fmul_rn(f0.y, scale);
      v[4 * i + 2] = __fmul_rn(f1.x, scale);
      v[4 * i + 3] = __fmul_rn(f1.y, scale);
    }
    // RoPE dims [2 lane, 2 lane + 2): two codes
    const uint32_t rc = reinterpret_cast<const uint16_t*>(src + kLatent)[lane];
    uint32_t lo, hi;
    e4m3x4_to_f16x4(rc, lo, hi);
    const float2 rf = __half22float2(*reinterpret_cast<__half2*>(&lo));
    rp0 = __fmul_rn(rf.x, scale);
    rp1 = __fmul_rn(rf.y, scale);
  } else {
    const uint8_t* src = a.kv + slot * kBf16RowBytes;
    const uint4 c0 = *reinterpret_cast<const uint4*>(src + 32 * lane);
    const uint4 c1 = *reinterpret_cast<const uint4*>(src + 32 * lane + 16);
    const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = bf16_lo(w[i]);
      v[2 * i + 1] = bf16_hi(w[i]);
    }
    const uint32_t rw = reinterpret_cast<const uint32_t*>(src + 2 * kLatent)[lane];
    rp0 = bf16_lo(rw);
    rp1 = bf16_hi(rw);
  }
  float4* d4 = reinterpret_cast<float4*>(dst + 16 * lane);
#pragma unroll
  for (int i = 0; i < 4; ++i) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  *reinterpret_cast<float2*>(dst + kLatent + 2 * lane) = make_float2(rp0, rp1);
}

// One warp waits, with the kernels' own bounded wait, on an mbarrier that nothing will
// complete; when the limit runs out it sets SMLA_DEVERR_TIMEOUT and returns, as a pipeline
// CTA does. Tests the timeout path without faulting or hanging anything.
__global__ void __launch_bounds__(32) selftest_wait_kernel(int32_t* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) mbar_init(b, 1);  // one arrival expected, none will come
  __syncwarp();
  if (!mbar_wait_for(b, 0, limit_ns) && threadIdx.x == 0) atomicOr(err, SMLA_DEVERR_TIMEOUT);
}

cudaError_t launch_selftest_wait(int32_t* err, uint64_t limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(err, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_gather_dequant(const DecodeArgs& a, float* rows, cudaStream_t s) {
  const int64_t items = static_cast<int64_t>(a.T) * a.K;
  const int64_t blocks = (items * 32 + 255) / 256;
  gather_dequant_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a, rows);
  return cudaGetLastError();
}

}  // namespace smla
