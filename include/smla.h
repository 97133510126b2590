/*
 * smla.h - C ABI of the GB300 sparse MLA decode library (libsmla.so).
 *
 * Sparse MLA decode, as the DeepSeek-V4 integration pages describe it
 * (vLLM PR #43477 "关键源码片段", forward_mqa; SGLang PR #24692 "实现拆解 2-3";
 * vLLM PR #43827 "关键源码片段"): for every query token, take the top-k
 * request-local slot indices chosen by the indexer, translate them through the
 * request's page table into physical cache slots, gather those rows of the
 * paged latent cache, dequantise them, score all heads over the 576 dims
 * (512 latent + 64 RoPE) against the one shared latent, apply a softmax with
 * an optional per-head sink logit and accumulate the 512-dim latent values.
 *
 * All tensor arguments are device pointers owned by the caller. The library
 * allocates no memory, never synchronises inside smla_decode / smla_pack_kv /
 * smla_gather_dequant, and returns a status instead of throwing. Argument
 * errors are found on the host before anything is launched; in that case
 * nothing is launched and no output is written. Streams are cudaStream_t
 * values passed as void* (NULL = the legacy default stream).
 */
#ifndef SMLA_H
#define SMLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum smla_status {
  SMLA_OK = 0,
  SMLA_ERR_NULL = 1,         /* a required pointer is NULL */
  SMLA_ERR_SHAPE = 2,        /* a size or count is outside the supported range */
  SMLA_ERR_ALIGN = 3,        /* a pointer breaks its alignment rule */
  SMLA_ERR_UNSUPPORTED = 4,  /* a valid combination this build does not serve */
  SMLA_ERR_WORKSPACE = 5,    /* workspace smaller than smla_workspace_size() */
  SMLA_ERR_CUDA = 6,         /* a CUDA runtime call or launch failed */
  SMLA_ERR_INDEX_RANGE = 7,  /* device met an invalid index or page entry (smla_read_error) */
  SMLA_ERR_DEVICE = 8,       /* no usable device, or not an sm_103 GPU */
  SMLA_ERR_TIMEOUT = 9,      /* a pipeline wait on the device gave up (smla_read_error) */
  SMLA_ERR_OPERAND_RANGE = 10 /* device met an operand outside the f16 window of the
                                 tensor-core path (SMLA_DEVERR_RANGE, smla_read_error) */
} smla_status;

/* Cache row formats. */
enum {
  /* 576 bf16 per slot, [latent 512 | RoPE 64] = 1152 bytes (the contiguous BF16
   * cache, vLLM PR #43477 "关键源码片段": (num_blocks, block_size, head_size)). */
  SMLA_KV_BF16 = 0,
  /* fp8_ds_mla: 656 bytes per slot = 512 E4M3FN latent codes | 4 fp32 scales
   * (little-endian; scale b covers latent dims [128b, 128b+128)) | 64 bf16 RoPE. */
  SMLA_KV_FP8_DS = 1,
  /* per-tensor FP8: 576 E4M3FN codes per slot, [latent 512 | RoPE 64] = 576 bytes, all
   * dequantised with the one fp32 scale smla_desc.kv_scale (the contiguous per-tensor FP8
   * cache of vLLM PR #43827 "实现拆解 4" / "关键源码片段": keys and values both carry
   * kv_scale, bmm1_scale = scale * q_scale * kv_scale, bmm2_scale = kv_scale; with
   * bf16 q, q_scale = 1; FP8 q: SMLA_Q_FP8_E4M3). */
  SMLA_KV_FP8_TENSOR = 2
};

/* Element type of q (smla_desc.q_format). */
enum {
  SMLA_Q_BF16 = 0,     /* [T, H, 576] bf16 */
  /* [T, H, 576] E4M3FN codes with one per-tensor scale smla_desc.q_scale: q = code * q_scale
   * (the FP8-Q path of vLLM PR #43827 "关键源码片段": bmm1_scale = scale * q_scale *
   * kv_scale, bmm2_scale = kv_scale). Served with SMLA_KV_FP8_TENSOR and 64 or more heads by
   * the FP8 tensor-core kernel, whose probabilities enter PV as E4M3 (see smla_decode). */
  SMLA_Q_FP8_E4M3 = 1
};

/* Block-scale rule of smla_pack_kv (amax = max |x| over the 128-dim block). */
enum {
  SMLA_SCALE_POW2 = 0, /* smallest power of two >= fl32(amax/448) ("UE8M0" layout) */
  SMLA_SCALE_FP32 = 1  /* fl32(amax/448) */
};

/* Bits of the device error word (smla_read_error). */
enum {
  SMLA_DEVERR_INDEX = 1, /* a top-k entry other than -1 outside [0, page_table_stride*page_size) */
  SMLA_DEVERR_PAGE = 2,  /* a page-table entry used by a valid index outside [0, num_pages) */
  SMLA_DEVERR_TIMEOUT = 4, /* an internal pipeline wait gave up (bounded waits; outputs invalid) */
  SMLA_DEVERR_RANGE = 8    /* fp8_ds with 64+ heads: a selected row holds a block scale outside
                              the f16 window [2^-15, 2^7] ([2^-14, 2^7] for scales that are not
                              powers of two); the outputs of that call may be inaccurate or
                              non-finite (see smla_decode) */
};

typedef struct smla_desc {
  int32_t num_tokens;        /* T >= 1: query tokens (requests x next_n) */
  int32_t num_heads;         /* H: multiple of 16, 16..128 */
  int32_t topk;              /* K >= 1, multiple of 4: entries per index row */
  int32_t num_requests;      /* B >= 1: rows of page_table */
  int32_t next_n;            /* >= 1: token t belongs to request t / next_n unless
                                req_id_per_token is given */
  int32_t page_size;         /* P: power of two, 1..4096 */
  int64_t num_pages;         /* physical pages in kv_cache (>= 1) */
  int32_t page_table_stride; /* entries per page_table row (>= 1) */
  int32_t kv_format;         /* SMLA_KV_* */
  float sm_scale;            /* softmax scale multiplying q.k (e.g. 1/sqrt(576)) */
  int32_t num_splits;        /* 0: the library chooses; n > 0: split the top-k list
                                into n contiguous parts merged by log-sum-exp */
  float kv_scale;            /* SMLA_KV_FP8_TENSOR: the cache's per-tensor scale (finite,
                                > 0); ignored by the other formats */
  int32_t q_format;          /* SMLA_Q_* (0: bf16) */
  float q_scale;             /* SMLA_Q_FP8_E4M3: q's per-tensor scale (finite, > 0);
                                ignored for bf16 q */
  int32_t reserved[1];       /* must be zero */
} smla_desc;

/* Human-readable name of a status (static string). */
const char* smla_status_string(int32_t status);

/* ABI version of this header (increments whenever the interface changes; 2 added kv_scale,
 * 3 added SMLA_ERR_TIMEOUT, SMLA_ERR_OPERAND_RANGE, SMLA_DEVERR_RANGE,
 * smla_noalloc_read_error, the indexer calls and smla_store_kv_normed; 4 added q_format and
 * q_scale in place of two reserved words; 5 added smla_plan_launches). */
int32_t smla_abi_version(void);

/*
 * Bytes of device workspace smla_decode needs for `d` on the current device: the
 * device error word, plus the split partials when the plan merges its splits in a
 * separate kernel (the tensor-core path merges up to 8 splits inside the decode kernel
 * and needs none). The caller allocates it (256-byte aligned) and zeroes it once before
 * first use; the library leaves the error word zeroed again after smla_read_error.
 * Writes 0 into *bytes on error.
 */
smla_status smla_workspace_size(const smla_desc* d, size_t* bytes);

/* Decode kernels (smla_launch_plan.kernel). */
enum {
  SMLA_KERNEL_HEAD_GROUP = 1,      /* tcgen05, 16-bit operands: FP8 caches, 64-128 heads */
  SMLA_KERNEL_HEAD_GROUP_FP8 = 2,  /* tcgen05, E4M3 operands: SMLA_Q_FP8_E4M3 */
  SMLA_KERNEL_MMA = 3              /* mma.sync: 16-48 heads, or the bf16 cache */
};

/* How the split partials of one work item are merged (smla_launch_plan.merge). */
enum {
  SMLA_MERGE_NONE = 0,     /* one split: the decode kernel writes the output */
  SMLA_MERGE_CLUSTER = 1,  /* inside the decode kernel, across its thread-block cluster */
  SMLA_MERGE_KERNEL = 2    /* partials in the workspace, then a separate merge kernel */
};

typedef struct smla_launch_plan {
  int32_t kernel;           /* SMLA_KERNEL_* */
  int32_t num_splits;       /* top-k splits of each work item in the first launch */
  int32_t split_len;        /* index entries a split covers (a multiple of 64; the last
                               split of an item takes what is left) */
  int32_t merge;            /* SMLA_MERGE_* of the first launch */
  int32_t num_launches;     /* decode launches: 1, or 2 when the last partial wave runs apart */
  int32_t ctas[2];          /* CTAs of each decode launch (ctas[1] = 0 with one launch) */
  int32_t tail_items;       /* work items of the second launch, two splits each, merged
                               across their cluster (0 with one launch) */
  uint64_t workspace_bytes; /* the value smla_workspace_size gives on such a device */
} smla_launch_plan;

/*
 * The launches smla_decode makes for `d` on a device with `num_sms` SMs (152 on GB300):
 * which kernel, how the top-k list is split, and the CTAs of each launch. A work item is
 * (token, group of 64 heads) for the head-group kernels and (token, 16 heads) for the
 * mma.sync kernel; a CTA takes one split of one item. When the head-group items with one
 * split fill whole waves of one CTA per SM plus a last wave at most half full, that last
 * wave runs as a second launch with two splits per item, so it takes about half a CTA's
 * time. Host-only: touches no device, launches nothing, and can be called without a GPU.
 * Status: SMLA_ERR_NULL for a NULL argument, SMLA_ERR_SHAPE for num_sms < 1, else the
 * status smla_decode's checks of `d` give; *plan is zeroed on error.
 */
smla_status smla_plan_launches(const smla_desc* d, int32_t num_sms, smla_launch_plan* plan);

/*
 * Sparse MLA decode (the hot path).
 *   q          [T, H, 576] bf16 (or E4M3 codes, q_format SMLA_Q_FP8_E4M3), 16-byte
 *              aligned; dims 0..511 pair with the latent, 512..575 with the RoPE part.
 *   kv_cache   [num_pages, P, R] bytes, R = 656 (FP8_DS), 576 (FP8_TENSOR) or 1152 (BF16),
 *              16-byte aligned. num_pages * P must stay below 2^31 - 1 (SMLA_ERR_SHAPE
 *              otherwise): rows are gathered by 32-bit row coordinates.
 *   page_table [B, page_table_stride] int32: request-local page -> physical page.
 *   topk       [T, K] int32, 16-byte aligned: request-local slot indices, -1 = padding.
 *              Index i of request r lives in physical slot
 *              page_table[r, i / P] * P + i % P.
 *   req_id_per_token [T] int32 or NULL (then request = t / next_n).
 *   sink       [H] fp32 or NULL: per-head sink logit sigma_h, adds e^sigma_h to the
 *              softmax denominator only.
 *   out        [T, H, 512] bf16, 16-byte aligned:
 *              out = sum_j e^{s_j} v_j / (sum_j e^{s_j} + [sink] e^{sigma_h}),
 *              s_j = sm_scale * <q, k_j>, v_j = k_j[0:512]. 0 when nothing is selected.
 *   lse        [T, H] fp32 or NULL: natural log of that denominator (-inf when it is
 *              empty and there is no sink).
 *   workspace  device memory of at least smla_workspace_size(d) bytes, 256-byte aligned.
 * Entries other than -1 that fall outside the request's page table, or whose page
 * entry lies outside [0, num_pages), are skipped like padding (never loaded) and set
 * a bit of the device error word, readable with smla_read_error. Duplicated indices
 * count once per occurrence. Rows skipped as padding are never read, so their bytes
 * may hold anything.
 *
 * Operand range. q may hold any finite bf16 values: every kernel brings each q row (or
 * row block) to [1, 2) by a power-of-two factor before its 16-bit MMAs and applies the
 * factor to the fp32 scores, so q is exact in f16 (elements below 2^-17 of their row's
 * largest keep 2^-25 of it in absolute error). For SMLA_KV_FP8_DS with 64 or more heads
 * the keys enter the tensor cores as f16 values code * scale: this is exact for
 * power-of-two block scales in [2^-15, 2^7] (every block amax in (0.0068, 57344] under
 * SMLA_SCALE_POW2), within two f16 roundings of 2^-11 each for other scales in
 * [2^-14, 2^7]. A selected row with a block scale outside that window sets
 * SMLA_DEVERR_RANGE, and the outputs of that call may be inaccurate or non-finite. The
 * bf16 RoPE values of such rows enter as f16 too: they must stay below 65504 in
 * magnitude (larger ones make the outputs of their heads non-finite; nothing flags them),
 * and values below 2^-17 keep 2^-25 in absolute error. Fewer than 64 heads,
 * SMLA_KV_FP8_TENSOR and SMLA_KV_BF16 apply scales in fp32 and have neither limit.
 *
 * FP8 q (q_format SMLA_Q_FP8_E4M3; only with SMLA_KV_FP8_TENSOR and 64 or more heads, else
 * SMLA_ERR_UNSUPPORTED): the codes of q and of the cache are the MMA operands (E4M3, fp32
 * accumulation); the scores take sm_scale * q_scale * kv_scale in fp32. The probabilities
 * enter PV as E4M3 values 2^(s - m + 7) (m within 1 of the running maximum), each within 2^-4
 * relative of its exact value (values below 2^-16 of the maximum weight are dropped), and the
 * output is normalised by the sum of those E4M3 values: every output is a convex combination
 * of the selected values times kv_scale, within 2^-3 * max |v_j| * kv_scale of the exact one.
 * The LSE uses the weights before rounding.
 */
smla_status smla_decode(const smla_desc* d, const void* q, const void* kv_cache,
                        const int32_t* page_table, const int32_t* topk,
                        const int32_t* req_id_per_token, const float* sink, void* out,
                        float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Measurement hook (the pages' interface has none): time the main decode kernel on its
 * own, apart from a split-merge kernel that may follow it (the tensor-core kernel merges up
 * to 8 splits itself, so its time includes that merge).
 *   start, stop  cudaEvent_t handles (passed as void*) created and destroyed by the
 *                caller; both NULL turns recording off, exactly one NULL is
 *                SMLA_ERR_NULL.
 * While set, every smla_decode / smla_decode_noalloc call made from this host thread
 * records `start` on its stream just before the decode kernel is launched and `stop`
 * just after it (before the merge kernel, when there is one). The setting belongs to
 * the calling host thread only. Recording failures make the decode call return
 * SMLA_ERR_CUDA.
 */
smla_status smla_set_kernel_events(void* start, void* stop);

/*
 * Write cache rows (the quantise-on-write store of the compressor, vLLM PR #43827
 * "实现拆解 4"): for each i < n with slot_mapping[i] >= 0, row slot_mapping[i] of
 * kv_cache receives latent[i] (512 bf16) and rope[i] (64 bf16).
 *   FP8_DS: per 128-dim block, scale by the SMLA_SCALE_* rule (an all-zero block gets
 *           scale 1); code = E4M3 round-to-nearest-even, saturating at +-448, of
 *           fl32(x / scale); RoPE is stored as given.
 *   BF16:   the 576 values are stored as given (scale_mode ignored).
 *   latent [n, 512] bf16 and rope [n, 64] bf16, 16-byte aligned; slot_mapping [n] int64;
 *   kv_cache holds num_slots rows. Entries of slot_mapping >= num_slots are skipped.
 * Status (all found before any launch): SMLA_ERR_UNSUPPORTED for another kv_format or
 * scale_mode, SMLA_ERR_SHAPE for n < 0, num_slots < 0 or n > 2^36, SMLA_ERR_NULL or
 * SMLA_ERR_ALIGN for a pointer (slot_mapping 8-byte aligned); n == 0 launches nothing.
 */
smla_status smla_pack_kv(int32_t kv_format, int32_t scale_mode, const void* latent,
                         const void* rope, const int64_t* slot_mapping, int64_t n,
                         void* kv_cache, int64_t num_slots, void* stream);

/*
 * Write rows of a per-tensor FP8 cache (SMLA_KV_FP8_TENSOR): for each i < n with
 * 0 <= slot_mapping[i] < num_slots, row slot_mapping[i] of kv_cache (576 bytes) receives
 * the E4M3 codes, round-to-nearest-even and saturating at +-448, of fl32(x / kv_scale)
 * for the 512 latent values latent[i] and the 64 RoPE values rope[i] (bf16). This is the
 * store_full_fp8 path of the compressor in vLLM PR #43827 "实现拆解 4-5".
 *   latent [n, 512] bf16 and rope [n, 64] bf16, 16-byte aligned; slot_mapping [n] int64;
 *   kv_scale finite and > 0 (SMLA_ERR_SHAPE otherwise).
 * Status: as smla_pack_kv; n == 0 launches nothing.
 */
smla_status smla_pack_kv_fp8_tensor(const void* latent, const void* rope,
                                    const int64_t* slot_mapping, int64_t n, float kv_scale,
                                    void* kv_cache, int64_t num_slots, void* stream);

/*
 * The cache write fused with the latent's normalisation and the key's RoPE (the compressor's
 * store of vLLM PR #43827, "实现拆解 4-6": SparseAttnCompressNormRopeStoreFullC4Kernel with
 * store_full_kv / store_full_fp8, tested as a fused "qnorm rope kv insert"). The page names
 * the steps; this library computes, for each row i with 0 <= slot_mapping[i] < num_slots:
 *   latent' = bf16(latent[i] * r * norm_weight), r = 1 / sqrt(mean(latent[i]^2) + rms_eps),
 *             in fp32 (sum of squares in a fixed order, correctly rounded sqrt and divide);
 *   rope'   = bf16 of the RoPE pairs (2j, 2j+1) = (a, b) turned to (a c - b s, a s + b c), with
 *             c = cos_sin[positions[i], j] and s = cos_sin[positions[i], 32 + j] (fp32);
 * and stores (latent', rope') exactly as smla_pack_kv (kv_format BF16 or FP8_DS with
 * scale_mode) or smla_pack_kv_fp8_tensor (kv_format FP8_TENSOR with kv_scale) would.
 *   latent [n, 512] and rope [n, 64] bf16, norm_weight [512] bf16: 16-byte aligned.
 *   positions [n] int64; cos_sin [max_position, 64] fp32, 16-byte aligned; slot_mapping [n] int64.
 *   error_word: device int32 or NULL; a row whose position is outside [0, max_position) is not
 *   written and sets SMLA_DEVERR_INDEX.
 * Status (before any launch): SMLA_ERR_UNSUPPORTED for another kv_format or scale_mode,
 * SMLA_ERR_SHAPE for a bad kv_scale, rms_eps, n, num_slots or max_position or a non-zero
 * reserved word, SMLA_ERR_NULL or SMLA_ERR_ALIGN for a pointer; n == 0 launches nothing.
 */
typedef struct smla_store_desc {
  int32_t kv_format;    /* SMLA_KV_* */
  int32_t scale_mode;   /* SMLA_SCALE_* (FP8_DS) */
  float kv_scale;       /* FP8_TENSOR: the per-tensor scale (finite, > 0) */
  float rms_eps;        /* >= 0 */
  int64_t n;            /* rows */
  int64_t num_slots;    /* rows of kv_cache */
  int64_t max_position; /* rows of cos_sin (>= 1) */
  int32_t reserved[2];  /* must be zero */
} smla_store_desc;

smla_status smla_store_kv_normed(const smla_store_desc* d, const void* latent, const void* rope,
                                 const void* norm_weight, const int64_t* positions,
                                 const float* cos_sin, const int64_t* slot_mapping, void* kv_cache,
                                 int32_t* error_word, void* stream);

/*
 * Test hook exposing the gather + dequantise steps of smla_decode
 * (the _gather_and_dequant reference path of SGLang PR #24692, "实现拆解 3"):
 * rows [T, K, 576] fp32 receives, for each (t, j), the dequantised key vector of the
 * slot topk[t, j] selects: latent element d = fl32(e4m3(code_d) * scale[d/128]) for
 * FP8_DS, the bf16 value otherwise; RoPE as bf16 values. Padding and invalid entries
 * give a zero row. error_word (device int32, may be NULL) receives SMLA_DEVERR_* bits.
 * The descriptor is checked as smla_decode checks it; kv_cache and rows 16-byte aligned.
 */
smla_status smla_gather_dequant(const smla_desc* d, const void* kv_cache,
                                const int32_t* page_table, const int32_t* topk,
                                const int32_t* req_id_per_token, float* rows,
                                int32_t* error_word, void* stream);

/*
 * Self-test of the failure path (the pages have no counterpart): launches one warp that
 * waits, with the same bounded mbarrier wait every pipeline stage of smla_decode uses, on
 * a barrier that nothing will complete. After limit_us microseconds (1..100000) the wait
 * gives up, sets SMLA_DEVERR_TIMEOUT in *error_word (a device int32) and the kernel returns,
 * as a stalled decode CTA would; the GPU context stays usable. Nothing faults or hangs.
 */
smla_status smla_selftest_wait_timeout(int32_t* error_word, uint32_t limit_us, void* stream);

/*
 * Synchronises `stream`, copies the device error word of `workspace` into
 * *error_word (SMLA_DEVERR_* bits accumulated since the last read) and clears it.
 * Returns SMLA_ERR_TIMEOUT when the timeout bit is set, else SMLA_ERR_INDEX_RANGE when
 * an index or page bit is set, else SMLA_ERR_OPERAND_RANGE when the range bit is set,
 * else SMLA_OK.
 */
smla_status smla_read_error(const smla_desc* d, void* workspace, size_t workspace_bytes,
                            int32_t* error_word, void* stream);

/*
 * ---------------------------------------------------------------------------------------
 * Sparse-attention indexer: the step before smla_decode that chooses each query token's
 * top-k slots (the vLLM PR #52164 page, "功能与动机" and "实现拆解 1-5": the FP8 paged MQA
 * logits kernel fp8_paged_mqa_logits, scheduled from the requests' context lengths, with the
 * next_n query rows of a request handled natively instead of flattened; the SGLang PR #24692
 * page, "实现拆解 5"). The pages give no formula; this library computes, for query row i of
 * request r (token t = r * next_n + i) and every slot s < ctx_r - next_n + 1 + i:
 *     logit[t, s] = sum_h weights[t, h] * max(0, scale_s * <q[t, h], k_s>)
 * with q[t, h] and k_s vectors of 128 E4M3 values and scale_s one fp32 per key, and then the
 * indices of each token's K largest logits.
 * ---------------------------------------------------------------------------------------
 */
typedef struct smla_indexer_desc {
  int32_t num_tokens;        /* T = num_requests * next_n */
  int32_t num_heads;         /* H_I: 32 or 64 index heads */
  int32_t num_requests;      /* B: 1..8192 */
  int32_t next_n;            /* query rows per request, 1..4, with H_I * next_n <= 256 */
  int32_t page_size;         /* P: 16, 32, 64 or 128 slots per page */
  int32_t page_table_stride; /* entries per page_table row (>= 1) */
  int64_t num_pages;         /* pages in k_cache (1 .. 2^31 - 1) */
  int32_t logits_stride;     /* floats per logits row (>= 1); contexts are served up to it */
  int32_t topk;              /* K of smla_indexer_topk (>= 1) */
  int32_t reserved[4];       /* must be zero */
} smla_indexer_desc;

/*
 * FP8 paged MQA logits of every query token over its visible context.
 *   q            [T, H_I, 128] E4M3 codes (uint8), 16-byte aligned.
 *   weights      [T, H_I] fp32, 16-byte aligned.
 *   k_cache      [num_pages, P * 132] bytes, 16-byte aligned: page p holds the P keys of its
 *                slots as P x 128 E4M3 codes (slot-major), followed by their P fp32 scales.
 *   page_table   [B, page_table_stride] int32: request-local page -> physical page.
 *   context_lens [B] int32: request r's slots are 0 .. ctx_r - 1 (slot s in page
 *                page_table[r, s / P] at position s % P); ctx_r above page_table_stride * P or
 *                logits_stride is served up to that bound and sets SMLA_DEVERR_INDEX.
 *   logits       [T, logits_stride] fp32: row t receives its visible slots; the rest of the
 *                row is not written.
 *   error_word   device int32 receiving SMLA_DEVERR_* bits: SMLA_DEVERR_PAGE for a page entry
 *                outside [0, num_pages) that a visible slot needs (those slots' logits are
 *                undefined), SMLA_DEVERR_INDEX as above, SMLA_DEVERR_TIMEOUT (outputs invalid).
 * All pointers are device memory owned by the caller; nothing is allocated or synchronised.
 * Argument errors return before anything is launched.
 */
smla_status smla_indexer_logits(const smla_indexer_desc* d, const void* q, const float* weights,
                                const void* k_cache, const int32_t* page_table,
                                const int32_t* context_lens, float* logits, int32_t* error_word,
                                void* stream);

/*
 * Top-k of the indexer logits: topk [T, K] int32 receives, for token t, the request-local
 * indices of its K largest visible logits in ascending index order; at a tie on the K-th
 * value the lowest indices are taken (-0 and +0 are one value). With fewer than K visible slots
 * the row is 0, 1, ..., visible - 1, then -1 padding: the topk_indices argument of smla_decode.
 *   logits [T, logits_stride] fp32 as smla_indexer_logits wrote them (only the visible
 *   part of each row is read); context_lens [B] int32 as given to that call.
 */
smla_status smla_indexer_topk(const smla_indexer_desc* d, const float* logits,
                              const int32_t* context_lens, int32_t* topk, void* stream);

/*
 * Size of the library-owned scratch array used by smla_decode_noalloc (16 MiB per device).
 */
#define SMLA_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * smla_decode without a caller-provided workspace. The pages have no counterpart for
 * this entry point: it exists for callers that cannot call cudaMalloc or own a device
 * allocator -- for example a plugin or callback running inside another serving engine
 * that has reserved the GPU's memory up front and forbids allocation on its hot path
 * (cudaMalloc synchronises the device and may fail once the pool is taken), or a
 * binding that only ever receives the engine's own input and output buffers.
 *
 * The split partials and the device error word live in a file-scope __device__ array
 * of SMLA_NOALLOC_SCRATCH_BYTES bytes inside libsmla.so. Every GPU that loads the
 * library holds that array until the process exits. The first call on a device looks
 * up the array's device address (cudaGetSymbolAddress) with that device current; make
 * that first call before any stream capture. The entry point itself calls no
 * cudaMalloc, cudaFree or allocating library routine.
 *
 * Arguments are those of smla_decode minus the workspace. A call whose split partials
 * would not fit in the array returns SMLA_ERR_WORKSPACE before launching anything
 * (choose num_splits = 1, which needs no partials, or fewer splits). All calls share
 * the one array, and its contents persist from call to call: calls that overlap on
 * the GPU (different streams, or different host threads) race on it and must be
 * serialised by the caller. The device error word lives in the array too: it starts at
 * zero when the library loads, collects the SMLA_DEVERR_* bits of every call, and is read
 * and cleared with smla_noalloc_read_error.
 */
smla_status smla_decode_noalloc(const smla_desc* d, const void* q, const void* kv_cache,
                                const int32_t* page_table, const int32_t* topk,
                                const int32_t* req_id_per_token, const float* sink, void* out,
                                float* lse, void* stream);

/*
 * The device error word of smla_decode_noalloc on the current device (its counterpart of
 * smla_read_error; the pages have none either). Synchronises `stream`, copies the SMLA_DEVERR_*
 * bits collected since the last read into *error_word (host memory) and clears them, with one
 * device-to-host copy and one memset on `stream` and no allocation. Returns the status
 * smla_read_error would give for the same bits. Serialise it with the decode calls, as
 * those calls are serialised among themselves.
 */
smla_status smla_noalloc_read_error(int32_t* error_word, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SMLA_H */
