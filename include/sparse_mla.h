/*
 * sparse_mla.h -- C ABI of libsparse_mla.so: sparse MLA decode attention over a paged FP8
 * KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The operation ("FlashMLA 与 DSA：内核、流水线和正确性边界", section 4.3, and "FlashMLA
 * Sparse Decode 完整计算过程详解", steps 1-19): for every query token t = (batch bi,
 * position si) and query head h,
 *
 *     J      = the top-k slots j of token t whose index is a valid physical token id
 *     K_j    = decoded 576-dim key of cache row indices[t][j] (512 dequantized NoPE dims,
 *              64 bf16 RoPE dims);  V_j = K_j[0:512]
 *     s_j    = sm_scale * <q[t][h], K_j>
 *     lse    = ln sum_{j in J} exp(s_j)
 *     out    = sum_{j in J} exp(s_j - lse) V_j
 *
 * with out = 0 and lse = +inf when J is empty.  MLA decodes as MQA: all h_q heads share
 * one latent KV head (h_kv = 1).
 *
 * Work is split in three calls, all asynchronous on the caller's CUDA stream:
 *   1. sparse_mla_sched_meta  -- greedy split-KV partition plan, computed on the GPU
 *   2. sparse_mla_decode_fwd  -- gather + dequant + QK^T + online softmax + PV
 *      (sparse_mla_decode_fwd_ex: with the attention sink, per-token top-k lengths, bf16
 *      split partials or a second KV cache)
 *   3. sparse_mla_combine     -- LSE-weighted merge of the split partial results
 * The steps that produce the index list are here too:
 *   sparse_mla_indexer_scores   -- the lightning-indexer scores over a paged FP8 key cache
 *   sparse_mla_topk_page_table  -- their exact top-k, emitted as physical cache ids
 *   sparse_mla_indexer_topk     -- the two chained, without the full score matrix
 *
 * Conventions shared by every entry point:
 *   - All buffers are owned by the caller.  The library allocates no memory and keeps no
 *     global state (except the fixed static scratch of sparse_mla_decode_static), and never
 *     synchronises a stream, except sparse_mla_read_device_status.
 *   - Pointers marked "device" must be device-accessible memory on the current device.
 *   - Arguments are validated before anything is launched; a bad argument returns an error
 *     and launches nothing.  The library never aborts the process and never prints.
 *   - A failed CUDA launch returns SMLA_ERR_CUDA (cudaGetLastError is read and cleared).
 *   - "stream" is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *   - The same smla_dims and num_sms must be used for the three decode calls of a problem.
 */
#ifndef SPARSE_MLA_H_
#define SPARSE_MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SMLA_OK = 0,
  SMLA_ERR_INVALID_ARG = 1, /* null pointer, negative size, size overflow */
  SMLA_ERR_UNSUPPORTED = 2, /* a shape outside h_q in {64,128}, d_qk = 576, d_v = 512,
                               page_block_size = 64 */
  SMLA_ERR_ALIGNMENT = 3,   /* a pointer below its required alignment */
  SMLA_ERR_WORKSPACE = 4,   /* a caller buffer smaller than sparse_mla_workspace_size says */
  SMLA_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  SMLA_ERR_TIMEOUT = 6,     /* device status: a bounded wait inside a kernel ran out */
  SMLA_ERR_DEVICE = 7       /* device status: a kernel reported bad data (see below) */
} smla_status;

/* Bits of the device status word (sparse_mla_read_device_status). */
#define SMLA_DEV_TIMEOUT 0x1u       /* a pipeline wait gave up; outputs are not valid */
#define SMLA_DEV_Q_RANGE 0x2u       /* |q| above 65504: not representable in the fp16 MMA */
#define SMLA_DEV_SCALE_RANGE 0x4u   /* a KV scale * 256 outside the fp16 normal range */
#define SMLA_DEV_TOPK_TABLE 0x8u    /* top-k: a selected position lies beyond the page table */
#define SMLA_DEV_NAN_INPUT 0x10u    /* a valid slot scored NaN or +inf: a NaN e4m3 code, scale or
                                       bf16 value (or bf16 +inf) in its row or in q, as the
                                       definition has it (every head of the token, or the heads
                                       scoring +inf, get out = NaN and lse = NaN), or a key
                                       value with |code * scale| * 256 above 65504, beyond the
                                       fp16 MMA's range (those heads are NaN; the definition's
                                       value is finite) */

/* Problem sizes.  Only d_qk = 576, d_v = 512, page_block_size = 64, h_q in {64, 128} are
 * supported ("FlashMLA 与 DSA", section 3.1: the 656-byte V3.2 row; section 6.1: h_q 64/128,
 * d_v 512).  topk may be any value >= 0; b or s_q = 0 is an empty problem.  extra_topk and
 * extra_num_blocks size the optional second cache and index list (smla_decode_opts); 0 when
 * it is not used.  The plan covers ceil(topk / 64) + ceil(extra_topk / 64) blocks per
 * request ("FlashMLA 与 DSA", section 3.2 counts topk + extra_topk). */
typedef struct {
  int32_t b;               /* batch (requests) */
  int32_t s_q;             /* query tokens per request */
  int32_t h_q;             /* query heads: 64 or 128 */
  int32_t d_qk;            /* 576 = 512 NoPE + 64 RoPE (SMLA_KV_V32), 512 (later formats) */
  int32_t d_v;             /* 512 */
  int32_t topk;            /* index slots per query token */
  int32_t page_block_size; /* 64 tokens per cache page */
  int64_t num_blocks;      /* pages in the KV cache pool; num_blocks * 64 <= 2^31 - 1 */
  int32_t extra_topk;      /* index slots per query token in the extra list (0: none) */
  int64_t extra_num_blocks; /* pages in the extra KV cache pool; * 64 <= 2^31 - 1 */
  int32_t kv_format;       /* SMLA_KV_*: layout of kv_cache (0, the 656-byte row, by default) */
  int32_t extra_kv_format; /* layout of the extra cache: SMLA_KV_V32 beside a V32 cache,
                              SMLA_KV_V41_FP4 beside a V41 cache (V4: no extra cache) */
} smla_dims;

/* KV-cache formats ("FlashMLA 与 DSA", sections 3.1, 2.1, 6.1 and 6.4; the second page, step
 * 2.3, maps d_qk = 576 to the V3.2 model and 512 to the later one).  The later formats store a
 * page of 64 tokens as structure-of-arrays: the 64 data rows, then the 64 scale rows; token id
 * t is row t % 64 of page t / 64, and with d_qk = d_v = 512 the value is the whole key.
 *   SMLA_KV_V32      656 bytes a token, one row: 512 e4m3 | 4 fp32 scales (per 128) | 64 bf16
 *                    RoPE; d_qk = 576, the value is the first 512 dims
 *   SMLA_KV_V4       584 bytes a token: data 448 e4m3 (NoPE) | 64 bf16 (RoPE); scales 7 e8m0
 *                    (per 64 NoPE dims) | 1 pad byte; d_qk = 512
 *   SMLA_KV_V41      528 bytes a token: data 512 e4m3; scales 16 e8m0 (per 32 dims); d_qk = 512
 *   SMLA_KV_V41_FP4  288 bytes a token: data 512 e2m1, two per byte (the even element in the
 *                    low nibble); scales 32 e4m3 (per 16 dims); only as the extra cache of a
 *                    V41 cache
 * The byte counts are the pages'; the split of each count into fields is the reading that
 * meets all of them.  e8m0 = 2^(e - 127) (0xFF is NaN).  The kernels multiply the dequantized
 * keys by 256 in fp16: an e8m0 scale outside [2^-22, 2^7] or an FP4 scale above 255 sets
 * SMLA_DEV_SCALE_RANGE. */
#define SMLA_KV_V32 0
#define SMLA_KV_V4 1
#define SMLA_KV_V41 2
#define SMLA_KV_V41_FP4 3

/*
 * sparse_mla_workspace_size -- sizes of the two caller-owned device buffers.
 *   num_sms      SMs the plan may use; <= 0 means "all SMs of the current device".
 *   sched_bytes  out: bytes for the partition plan (sparse_mla_sched_meta writes it).
 *   accum_bytes  out: bytes for the split-partial workspace: fp32 partial O [slots][s_q]
 *                [h_q][512], then (256-byte aligned) base-2 lse [slots][s_q][h_q], where
 *                slots = num_splits[r + 1] for the last request r that the plan splits.  0
 *                when the plan splits no request (the workspace pointer may then be NULL).
 *                The plan is a pure function of (b, topk, extra_topk, num_sms), walked here
 *                on the host in O(num_sm_parts).
 * Host-only; launches nothing.  Errors: SMLA_ERR_INVALID_ARG, SMLA_ERR_UNSUPPORTED,
 * SMLA_ERR_CUDA (device query failed).
 */
smla_status sparse_mla_workspace_size(const smla_dims* dims, int num_sms, size_t* sched_bytes,
                                      size_t* accum_bytes);

/*
 * sparse_mla_sched_meta -- the greedy split-KV plan ("FlashMLA Sparse Decode 完整计算过程
 * 详解", step 3; "FlashMLA 与 DSA", section 3.2).  One warp on the GPU computes:
 *   num_sm_parts = max(num_sms / s_q / 2, 1)        (one partition = one pair of SMs)
 *   blocks per request = ceil(topk / 64), overhead 5 per request,
 *   payload = ceil(sum(blocks + 5) / num_sm_parts) + 5,
 * then fills partitions left to right, splitting a request where it does not fit.
 *   sched_meta   device, 16-byte aligned, sched_bytes long (caller-owned, written here):
 *                int32 [num_sm_parts][8] {begin_req, end_req, begin_block, end_block
 *                (exclusive), begin_split_idx, is_first_req_splitted,
 *                is_last_req_splitted, 0}, then int32 num_splits prefix [b + 1], then the
 *                device status word (reset to 0 by this call).
 * Asynchronous on stream.  Errors: SMLA_ERR_INVALID_ARG, SMLA_ERR_UNSUPPORTED,
 * SMLA_ERR_ALIGNMENT, SMLA_ERR_WORKSPACE, SMLA_ERR_CUDA.
 */
smla_status sparse_mla_sched_meta(const smla_dims* dims, int num_sms, void* sched_meta,
                                  size_t sched_bytes, void* stream);

/*
 * sparse_mla_decode_fwd -- the split-KV attention pass ("FlashMLA Sparse Decode 完整计算过程
 * 详解", steps 5-15).  Each partition of the plan runs on a cluster of two CTAs: one gathers
 * and dequantizes the selected rows into an fp16 key tile, forms the scores with tcgen05 MMAs
 * and runs the online softmax; it streams P to the other, which gathers the value rows and
 * accumulates O = P V in tensor memory and writes it out.
 *   q          device bf16 [b][s_q][h_q][576], contiguous, 16-byte aligned
 *   kv_cache   device uint8 [num_blocks][64][1][656], contiguous, 16-byte aligned; row =
 *              512 e4m3 NoPE codes | 4 fp32 scales (dequant multipliers, one per 128 dims)
 *              | 64 bf16 RoPE values
 *   indices    device int32 [b][s_q][topk], contiguous, 4-byte aligned; value = physical
 *              token id page * 64 + offset; a value outside [0, num_blocks * 64) (for
 *              example -1) masks the slot; a repeated id counts once per slot
 *   sm_scale   softmax scale applied to q.K (for example 1/sqrt(576))
 *   sched_meta device, the plan written by sparse_mla_sched_meta for the same dims/num_sms
 *   workspace  device, >= accum_bytes, 16-byte aligned: split partials (read by combine);
 *              may be NULL when accum_bytes is 0
 *   out        device bf16 [b][s_q][h_q][512], 16-byte aligned; rows of unsplit requests
 *              are final after this call, split rows after sparse_mla_combine
 *   lse        device fp32 [b][h_q][s_q] (note the axis order), natural log, +inf for a
 *              row with no valid slot
 * Asynchronous on stream.  Errors: SMLA_ERR_INVALID_ARG, SMLA_ERR_UNSUPPORTED,
 * SMLA_ERR_ALIGNMENT, SMLA_ERR_WORKSPACE, SMLA_ERR_CUDA.  Device-side problems (a wait
 * that ran out, q or a scale outside the fp16 range) set bits of the status word.  The
 * kernels compute in fp16: q with |q| > 65504, a scale whose product with 256 leaves the
 * fp16 normal range, or a dequantized key beyond 65504 / 256 are UNSUPPORTED inputs, not
 * merely reported ones: out and lse are then not valid (SMLA_DEV_Q_RANGE,
 * SMLA_DEV_SCALE_RANGE or SMLA_DEV_NAN_INPUT tells the caller after the fact).
 */
smla_status sparse_mla_decode_fwd(const smla_dims* dims, int num_sms, const void* q,
                                  const void* kv_cache, const int32_t* indices, float sm_scale,
                                  const void* sched_meta, void* workspace,
                                  size_t workspace_bytes, void* out, float* lse, void* stream);

/*
 * sparse_mla_combine -- merge split partials ("FlashMLA Sparse Decode 完整计算过程详解",
 * step 16; "FlashMLA 与 DSA", section 3.2): per (token, head) with n > 1 splits,
 * M = max_j lse2_j, w_j = 2^(lse2_j - M), out = sum_j w_j o_j / sum_j w_j (bf16),
 * lse = (M + log2 sum_j w_j) ln 2; all splits empty gives out = 0, lse = +inf.  Rows of
 * unsplit requests are left untouched; when no request is split (see
 * sparse_mla_plan_has_splits) nothing is launched.
 *   sched_meta, workspace   as passed to sparse_mla_decode_fwd (read only)
 *   out, lse                as for sparse_mla_decode_fwd (written for split rows)
 * Asynchronous on stream; must follow sparse_mla_decode_fwd on the same stream.
 * Errors: as sparse_mla_decode_fwd.
 */
smla_status sparse_mla_combine(const smla_dims* dims, int num_sms, const void* sched_meta,
                               const void* workspace, size_t workspace_bytes, void* out,
                               float* lse, void* stream);

/*
 * Optional inputs of the decode variants ("FlashMLA 与 DSA：内核、流水线和正确性边界",
 * section 4.3, the reference semantics; "FlashMLA Sparse Decode 完整计算过程详解", step 13,
 * the attention sink inside the kernel).  A NULL field leaves its variant off; a NULL
 * smla_decode_opts pointer leaves all of them off.
 *   attn_sink    device fp32 [h_q], 4-byte aligned: one sink score per query head.  The
 *                output row becomes out * 1 / (1 + exp(attn_sink[h] - lse)): the sink acts
 *                as one more key with score attn_sink[h] and a zero value vector.  The
 *                returned lse is that of the real slots only (unchanged by the sink).  A row
 *                with no valid slot keeps out = 0, lse = +inf.
 *   topk_length  device int32 [b][s_q], 4-byte aligned: slot j of token t is masked when
 *                j >= topk_length[t], in addition to the index rule; a length above topk
 *                keeps every slot, a length <= 0 masks the whole row.  The plan still
 *                covers all topk slots (masked slots cost no cache reads, but their blocks
 *                still pass through the pipeline).
 *   extra_kv_cache, extra_indices, extra_topk_length
 *                the second cache ("FlashMLA 与 DSA", sections 3.2 and 6.1 name an extra_kv
 *                beside the main cache): device uint8 [extra_num_blocks][64][1][656] in the
 *                main cache's row format, 16-byte aligned; device int32
 *                [b][s_q][extra_topk] physical ids into it (masked outside [0,
 *                extra_num_blocks * 64)), 4-byte aligned; optional device int32 [b][s_q]
 *                lengths for that list (as topk_length).  The attention runs over the union
 *                of the main and the extra slots.  Required when dims->extra_topk > 0 (the
 *                cache pointer only when extra_num_blocks > 0).
 *   partials_bf16  nonzero: the split partials of O go through the workspace as bf16
 *                instead of fp32, halving their write and read traffic ("FlashMLA 与 DSA",
 *                section 5.6 reports this trade for a split kernel: partials are already
 *                normalised by their own exp-sum, so they are bounded by the largest value
 *                element).  Results stay within the library's tolerance but differ in the
 *                last bits from the fp32 path; the workspace size is unchanged.
 *   test_stall   test hook for the failure path, 0 in use: nonzero makes the MMA issuer of
 *                every partition's score CTA wait on a barrier that nothing arrives at.  Each
 *                waiting role gives up after its bounded wait (about 1 s), the kernel returns,
 *                the device status word gets SMLA_DEV_TIMEOUT and word 1 the first wait that
 *                ran out; the outputs of that call are not valid and the context stays usable.
 * The same options must be given to sparse_mla_decode_fwd_ex and sparse_mla_combine_ex of
 * one problem: the decode pass applies the sink to unsplit rows, the combine to split rows,
 * and both must agree on the partials' type.
 */
typedef struct {
  const float* attn_sink;
  const int32_t* topk_length;
  int32_t partials_bf16;
  const void* extra_kv_cache;
  const int32_t* extra_indices;
  const int32_t* extra_topk_length;
  int32_t test_stall;
} smla_decode_opts;

/* sparse_mla_decode_fwd with decode options (opts may be NULL: then identical to it).
 * Errors: as sparse_mla_decode_fwd; SMLA_ERR_ALIGNMENT for a misaligned option pointer. */
smla_status sparse_mla_decode_fwd_ex(const smla_dims* dims, int num_sms, const void* q,
                                     const void* kv_cache, const int32_t* indices,
                                     float sm_scale, const smla_decode_opts* opts,
                                     const void* sched_meta, void* workspace,
                                     size_t workspace_bytes, void* out, float* lse,
                                     void* stream);

/* sparse_mla_combine with decode options (opts may be NULL: then identical to it).  With
 * attn_sink set, a split row's merged output is divided by sum_j w_j + 2^(attn_sink[h]
 * log2(e) - M) instead of sum_j w_j (the same factor as above); topk_length is not read
 * here.  Errors: as sparse_mla_combine. */
smla_status sparse_mla_combine_ex(const smla_dims* dims, int num_sms,
                                  const smla_decode_opts* opts, const void* sched_meta,
                                  const void* workspace, size_t workspace_bytes, void* out,
                                  float* lse, void* stream);

/*
 * sparse_mla_decode_static -- sparse_mla_sched_meta, sparse_mla_decode_fwd and
 * sparse_mla_combine in one call, on scratch memory owned by the library instead of the
 * caller.  The pages describe no such call: it exists for callers that cannot provide
 * device buffers of their own, such as a plain C host program with no device allocator at
 * hand, or a latency-critical loop that may not call cudaMalloc (which can synchronise the
 * device) once it is running.
 *   dims, num_sms, q, kv_cache, indices, sm_scale, out, lse, stream
 *              as for sparse_mla_decode_fwd
 * Unlike every other entry point, this one uses library-owned state:
 *   - The scratch is one static device array of SMLA_STATIC_SCRATCH_BYTES (48 MiB) per
 *     device, created when the library's CUDA module loads; the call allocates nothing.
 *     A problem whose plan plus split partials (sparse_mla_workspace_size) exceed it is
 *     rejected with SMLA_ERR_WORKSPACE before anything is launched.  With num_sms = 152
 *     that admits, for example, b = 64, s_q = 1, h_q = 128 and b = 1, s_q = 4096,
 *     h_q = 128 (no request split: only the plan), b = 32, s_q = 1, h_q = 128 (every
 *     request split in two: 16 MB) and b = 128, s_q = 2, h_q = 64; use the three-call
 *     sequence with caller buffers beyond that.
 *   - The array belongs to the library's CUDA module, so every process that loads the
 *     module on a device holds its 48 MiB there until exit, whether or not it calls this
 *     entry point; under lazy module loading (the CUDA default) that happens on the first
 *     launch of any kernel of the library, under CUDA_MODULE_LOADING=EAGER when the library
 *     initialises CUDA on the device.
 *   - The first call on a device, made with that device current, looks up the array's
 *     device address (cudaGetSymbolAddress, which may load the CUDA module) and caches it
 *     for the current CUDA context; make that first call before any stream capture begins.
 *     A device reset (cudaDeviceReset, or a primary-context release and re-creation) ends
 *     the context the address belongs to: the next call sees the new context's id and
 *     looks the address up again, so that call too should come before any stream capture.
 *   - Every call on a device uses the same scratch, so two calls whose executions overlap
 *     on the GPU (different streams without an ordering between them, or host threads
 *     issuing at the same time) corrupt each other's results.  Order them, for example by
 *     issuing all of them on one stream.
 *   - The planner zeroes the status words at the start of every call and nothing else in
 *     the scratch needs an initial value.  The device status word of the last call (a wait
 *     that ran out, the input range flags) is read with sparse_mla_static_read_status.
 * Asynchronous on stream.  Errors: as sparse_mla_decode_fwd, plus SMLA_ERR_WORKSPACE for a
 * problem above the scratch size and SMLA_ERR_CUDA if the address lookup fails.
 */
#define SMLA_STATIC_SCRATCH_BYTES (((size_t)48) << 20)
smla_status sparse_mla_decode_static(const smla_dims* dims, int num_sms, const void* q,
                                     const void* kv_cache, const int32_t* indices,
                                     float sm_scale, void* out, float* lse, void* stream);

/*
 * sparse_mla_static_read_status -- the device status word of the last sparse_mla_decode_static
 * call on the current device with these dims and num_sms (the word lives in the plan, inside
 * the library's scratch).  Same results as sparse_mla_read_device_status: *code = the word,
 * SMLA_OK when it is 0, SMLA_ERR_TIMEOUT when SMLA_DEV_TIMEOUT is set, SMLA_ERR_DEVICE for
 * any other bit.  Synchronises stream (the read is ordered after the work issued on it).
 * The pages describe no such call.  Errors: as sparse_mla_decode_static before its launches.
 */
smla_status sparse_mla_static_read_status(const smla_dims* dims, int num_sms, int* code,
                                          void* stream);

/*
 * sparse_mla_plan_has_splits -- whether the plan of these sizes splits any request across
 * partitions (*has_splits = 1), that is whether sparse_mla_combine has work.  Host-only and
 * exact: every request has the same ceil(topk / 64) blocks, so the greedy plan of
 * sparse_mla_sched_meta splits a request in its first partition or nowhere.  When it returns
 * 0, sparse_mla_combine launches nothing.  Errors: SMLA_ERR_INVALID_ARG,
 * SMLA_ERR_UNSUPPORTED, SMLA_ERR_CUDA (device query for num_sms <= 0).
 */
smla_status sparse_mla_plan_has_splits(const smla_dims* dims, int num_sms, int* has_splits);

/*
 * sparse_mla_topk_page_table -- the step before the attention: for every query token, the
 * exact top-k of its index scores over its valid (causally visible) prefix, emitted as
 * physical cache ids ("FlashMLA 与 DSA", section 5.5: a two-stage filtered radix top-k whose
 * emit writes page_table[u / 64] * 64 + u % 64 directly; "sparse-attention co-design",
 * section 5, step five: a row with fewer than k valid tokens is padded with an invalid id,
 * never a repeated token).  The result is the `indices` input of sparse_mla_decode_fwd.
 *   dims->n_tok      query tokens (rows of scores); token t belongs to request t / s_q
 *   dims->s_q        query tokens per request (rows of the page table: ceil(n_tok / s_q))
 *   dims->topk       k, output slots per token (>= 1)
 *   dims->ld         row stride of scores in elements; ld * element size a multiple of 16
 *   dims->max_pages  columns of the page table
 *   dims->dtype      SMLA_SCORES_BF16 or SMLA_SCORES_FP32
 *   scores           device [n_tok][ld] bf16 or fp32, 16-byte aligned; finite or +-inf (NaN
 *                    is not ordered)
 *   valid_len        device int32 [n_tok]: token t scores positions [0, valid_len[t]) (clamped
 *                    to [0, ld])
 *   block_table      device int32 [ceil(n_tok / s_q)][max_pages]: page ids of each request
 *   out_indices      device int32 [n_tok][topk] (written): the selected ids in no particular
 *                    order, then -1 for the slots past min(k, valid_len[t]); ties at the k-th
 *                    largest value are broken arbitrarily (any k largest are a correct answer)
 *   status           optional device uint32 word: SMLA_DEV_TOPK_TABLE is or-ed in when a
 *                    selected position u has u / 64 >= max_pages (that slot gets -1)
 * Asynchronous on stream.  Errors: SMLA_ERR_INVALID_ARG, SMLA_ERR_UNSUPPORTED (dtype),
 * SMLA_ERR_ALIGNMENT, SMLA_ERR_CUDA.
 */
#define SMLA_SCORES_BF16 0
#define SMLA_SCORES_FP32 1
typedef struct {
  int32_t n_tok;
  int32_t s_q;
  int32_t topk;
  int32_t ld;
  int32_t max_pages;
  int32_t dtype;
} smla_topk_dims;
smla_status sparse_mla_topk_page_table(const smla_topk_dims* dims, const void* scores,
                                       const int32_t* valid_len, const int32_t* block_table,
                                       int32_t* out_indices, uint32_t* status, void* stream);

/*
 * sparse_mla_indexer_scores -- the lightning-indexer scores the top-k selects from ("FlashMLA 与
 * DSA", section 4.1: I[t, s] = sum_j w[t, j] ReLU(q[t, j] . k[s]) with e4m3 q and k and one key
 * per cached token shared by the 64 heads; section 5.3: the paged cache layout and the key
 * scale applied after the head sum; "sparse-attention co-design", section 5, steps one to
 * four: the query scale folded into w).  For every query token t and position s <
 * valid_len[t]:
 *     scores[t][s] = k_scale[s] * sum_{j < 64} w[t][j] * max(q8[t][j] . k8[s], 0)
 * computed with e4m3 x e4m3 tensor-core MMAs accumulated in fp32.
 *   dims->n_tok      query tokens; token t belongs to request t / s_q (n_tok % s_q == 0)
 *   dims->s_q        query tokens per request
 *   dims->heads      64;  dims->dim  128
 *   dims->max_pages  columns of the page table;  dims->num_pages  pages in the cache
 *   dims->ld         row stride of scores (valid_len is clamped to it)
 *   q8               device uint8 [n_tok][64][128] e4m3 codes, 16-byte aligned
 *   weights          device fp32 [n_tok][64] (the query scales and normalisations folded in)
 *   k_cache          device uint8 [num_pages][8448]: 64 x 128 e4m3 codes of a page's tokens,
 *                    then their 64 fp32 scales; 16-byte aligned
 *   block_table      device int32 [n_tok / s_q][max_pages]
 *   valid_len        device int32 [n_tok]
 *   scores           device fp32 [n_tok][ld] (written for s < min(valid_len[t], ld,
 *                    max_pages * 64) only); a page id outside [0, num_pages) scores 0
 *   status           optional device uint32 word (SMLA_DEV_TIMEOUT if a wait ran out)
 * num_sms <= 0 means all SMs of the current device.  Asynchronous on stream.  Errors:
 * SMLA_ERR_INVALID_ARG, SMLA_ERR_UNSUPPORTED, SMLA_ERR_ALIGNMENT, SMLA_ERR_CUDA.
 */
typedef struct {
  int32_t n_tok;
  int32_t s_q;
  int32_t heads;
  int32_t dim;
  int32_t max_pages;
  int32_t ld;
  int64_t num_pages;
  /* 0 normally.  Nonzero: the kernel's MMA issuer waits on a barrier nothing arrives at, so
   * that every bounded wait runs out (a test of the failure path: SMLA_DEV_TIMEOUT in status,
   * no score written, the context usable afterwards). */
  int32_t test_stall;
} smla_indexer_dims;
smla_status sparse_mla_indexer_scores(const smla_indexer_dims* dims, int num_sms, const void* q8,
                                      const float* weights, const void* k_cache,
                                      const int32_t* block_table, const int32_t* valid_len,
                                      float* scores, uint32_t* status, void* stream);

/*
 * sparse_mla_indexer_topk -- the two selection steps chained, without the [n_tok][ld] score
 * matrix ("FlashMLA 与 DSA", sections 4.1, 5.3 and 5.5; "sparse-attention co-design",
 * section 5, steps one to five, and its summary, which proposes fusing the indexer with the
 * top-k so that the full fp32 scores are neither written back nor read again).  For each run of query tokens whose scores fit `scratch`, the indexer scores
 * (as sparse_mla_indexer_scores) go into scratch and the exact top-k with the page-table emit
 * (as sparse_mla_topk_page_table on fp32 scores) reads them back, so the scores of at most
 * scratch_bytes / (L * 4) tokens exist at a time; with the scratch the size helper returns
 * (SMLA_SELECT_SCRATCH_BUDGET bytes or less) they stay in L2 between the two steps.
 * Positions considered for token t: s < min(valid_len[t], L), L = min(dims->ld,
 * dims->max_pages * 64).
 *   dims             as for sparse_mla_indexer_scores; dims->ld (a multiple of 4) bounds the
 *                    positions and no score matrix of that stride is needed
 *   topk             output slots per token (>= 1)
 *   q8, weights, k_cache, block_table, valid_len   as for sparse_mla_indexer_scores
 *   scratch          device buffer, 16-byte aligned, at least L * 4 bytes (one token's
 *                    scores); its contents on return are unspecified
 *   out_indices      device int32 [n_tok][topk] (written), as for sparse_mla_topk_page_table
 *   status           device uint32 word, required (SMLA_DEV_TIMEOUT, SMLA_DEV_TOPK_TABLE are
 *                    or-ed in): the top-k of a run reads the scores its indexer launch left,
 *                    so a wait that ran out in the indexer must be visible to the caller
 * Launches two kernels per run of tokens, all on stream, asynchronously.  Errors:
 * SMLA_ERR_INVALID_ARG, SMLA_ERR_UNSUPPORTED, SMLA_ERR_ALIGNMENT (also ld not a multiple of
 * 4), SMLA_ERR_WORKSPACE (scratch below one token's scores), SMLA_ERR_CUDA.
 *
 * sparse_mla_indexer_topk_scratch_size -- host only: the scratch bytes for dims: the scores
 * of min(n_tok, max(1, SMLA_SELECT_SCRATCH_BUDGET / (L * 4))) tokens.
 */
#define SMLA_SELECT_SCRATCH_BUDGET (48u << 20)
smla_status sparse_mla_indexer_topk_scratch_size(const smla_indexer_dims* dims, size_t* bytes);
smla_status sparse_mla_indexer_topk(const smla_indexer_dims* dims, int32_t topk, int num_sms,
                                    const void* q8, const float* weights, const void* k_cache,
                                    const int32_t* block_table, const int32_t* valid_len,
                                    void* scratch, size_t scratch_bytes, int32_t* out_indices,
                                    uint32_t* status, void* stream);

/* Human-readable name of a status code (static storage; never NULL). */
const char* sparse_mla_status_string(smla_status status);

/*
 * sparse_mla_read_device_status -- copy the device status word out of sched_meta into
 * *code (SMLA_DEV_* bits, 0 = clean).  Synchronises stream (the only call that does).
 * Returns SMLA_ERR_TIMEOUT if the TIMEOUT bit is set, SMLA_ERR_DEVICE for other bits,
 * SMLA_OK when clean; SMLA_ERR_INVALID_ARG / SMLA_ERR_CUDA on bad input or a CUDA error.
 */
smla_status sparse_mla_read_device_status(const smla_dims* dims, int num_sms,
                                          const void* sched_meta, int* code, void* stream);

/* Library build identifier (static storage). */
const char* sparse_mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_MLA_H_ */
