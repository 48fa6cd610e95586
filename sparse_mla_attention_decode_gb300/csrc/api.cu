// Host runtime of libsparse_mla.so: argument validation, buffer sizing and kernel launches
// behind the C ABI declared in include/sparse_mla.h.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/sparse_mla.h"
#include "smla_internal.h"

using namespace smla;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// The plan's slot count per request: the main list rounded up to whole 64-slot blocks, then the
// extra list (its blocks follow the main ones).
int64_t plan_topk(const smla_dims* d) {
  const int64_t nb_main = (static_cast<int64_t>(d->topk) + kPage - 1) / kPage;
  return nb_main * kPage + d->extra_topk;
}

smla_status check_dims(const smla_dims* d) {
  if (!d) return SMLA_ERR_INVALID_ARG;
  if (d->b < 0 || d->s_q < 0 || d->topk < 0 || d->num_blocks < 0 || d->extra_topk < 0 ||
      d->extra_num_blocks < 0)
    return SMLA_ERR_INVALID_ARG;
  if (d->h_q != 64 && d->h_q != 128) return SMLA_ERR_UNSUPPORTED;
  if (d->d_v != kDV || d->page_block_size != kPage) return SMLA_ERR_UNSUPPORTED;
  // the cache format fixes d_qk: 576 for the 656-byte rows, 512 for the later formats; the
  // extra cache is 656-byte beside a 656-byte cache and FP4 beside a V4.1 cache (V4: none)
  if (d->kv_format == SMLA_KV_V32) {
    if (d->d_qk != kDQk || d->extra_kv_format != SMLA_KV_V32) return SMLA_ERR_UNSUPPORTED;
  } else if (d->kv_format == SMLA_KV_V4) {
    if (d->d_qk != 512 || d->extra_topk != 0) return SMLA_ERR_UNSUPPORTED;
  } else if (d->kv_format == SMLA_KV_V41) {
    if (d->d_qk != 512 || (d->extra_topk != 0 && d->extra_kv_format != SMLA_KV_V41_FP4))
      return SMLA_ERR_UNSUPPORTED;
  } else {
    return SMLA_ERR_UNSUPPORTED;
  }
  if (d->num_blocks * static_cast<int64_t>(kPage) > INT32_MAX) return SMLA_ERR_UNSUPPORTED;
  if (d->extra_num_blocks * static_cast<int64_t>(kPage) > INT32_MAX) return SMLA_ERR_UNSUPPORTED;
  if (plan_topk(d) > INT32_MAX) return SMLA_ERR_UNSUPPORTED;
  const int64_t tokens = static_cast<int64_t>(d->b) * d->s_q;
  if (tokens > INT32_MAX / 128 || plan_topk(d) * tokens > (int64_t(1) << 40))
    return SMLA_ERR_UNSUPPORTED;
  if (d->s_q > 65535) return SMLA_ERR_UNSUPPORTED;  // grid.y
  return SMLA_OK;
}

// Option pointers are optional; those given must be 4-byte aligned (fp32 / int32 arrays).
smla_status check_opts(const smla_decode_opts* o) {
  if (o == nullptr) return SMLA_OK;
  if (!aligned(o->attn_sink, 4) || !aligned(o->topk_length, 4) || !aligned(o->extra_kv_cache, 16) ||
      !aligned(o->extra_indices, 4) || !aligned(o->extra_topk_length, 4))
    return SMLA_ERR_ALIGNMENT;
  return SMLA_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled from the driver, looked up once (no link-time dependency on libcuda).
EncodeTiledFn encode_tiled_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
    else
      cudaGetLastError();
  });
  return fn;
}

smla_status resolve_parts(const smla_dims* d, int num_sms, int* parts, int* sms_out = nullptr) {
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SMLA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SMLA_ERR_CUDA;
  }
  const int sq = d->s_q > 0 ? d->s_q : 1;
  int p = num_sms / sq / 2;
  *parts = p < 1 ? 1 : p;
  if (sms_out) *sms_out = num_sms;
  return SMLA_OK;
}

// Split slots the workspace must hold: the plan numbers the splits of request r from
// prefix[r] = r + (number of partitions that start inside an earlier request), so the last
// request that is split (one that a partition starts inside) ends at slot r_last + 1 +
// (partitions that start inside a request), and no slot past it is ever written.  0 when no
// request is split.  The same greedy walk as the planner kernel, one partition per step with
// the whole requests of a step taken at once: O(parts).
int64_t split_slots(int64_t b, int64_t topk, int parts) {
  const int64_t nb = (topk + kPage - 1) / kPage;
  if (b <= 0 || nb <= 0) return 0;
  const int64_t c = nb + kFixedOverhead;
  const int64_t P = (b * c + parts - 1) / parts + kFixedOverhead;
  int64_t req = 0, blk = 0, mid_starts = 0, last_split = -1;
  for (int p = 0; p < parts && req < b; ++p) {
    if (blk > 0) {  // this partition starts inside request req: req is split
      ++mid_starts;
      last_split = req;
    }
    int64_t remain = P;
    const int64_t left = nb - blk;
    if (left + kFixedOverhead <= remain) {  // the rest of the current request fits
      remain -= left + kFixedOverhead;
      ++req;
      blk = 0;
      if (remain > kFixedOverhead && req < b) {
        int64_t whole = remain / c;  // c > 5, so a request that fits leaves remain > 5 first
        if (whole > b - req) whole = b - req;
        remain -= whole * c;
        req += whole;
        if (req < b && remain > kFixedOverhead) blk = remain - kFixedOverhead;  // split here
      }
    } else {
      blk += remain - kFixedOverhead;  // take what fits and split the request here
    }
  }
  return last_split < 0 ? 0 : last_split + 1 + mid_starts;
}

AccumLayout workspace_layout(const smla_dims* d, int parts) {
  const int64_t slots = split_slots(d->b, plan_topk(d), parts);
  return accum_layout_slots(static_cast<int>(slots), d->s_q, d->h_q);
}

smla_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return SMLA_OK;
  (void)cudaGetLastError();
  return SMLA_ERR_CUDA;
}

}  // namespace

bool smla::encode_rows_map(CUtensorMap* map, const void* base, bool fp32, int64_t rows, int cols,
                           int box_cols, int box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  const cuuint64_t esize = fp32 ? 4 : 2;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * esize};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t elem[2] = {1, 1};
  return enc(map, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
             const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool smla::encode_bytes_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                            const uint64_t* strides, const uint32_t* box, bool swizzle128) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t bx[3], elem[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, static_cast<cuuint32_t>(rank),
             const_cast<void*>(base), d, st, bx, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
             swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

extern "C" {

const char* sparse_mla_version(void) { return "sparse_mla 0.1 sm_103a"; }

const char* sparse_mla_status_string(smla_status s) {
  switch (s) {
    case SMLA_OK: return "ok";
    case SMLA_ERR_INVALID_ARG: return "invalid argument";
    case SMLA_ERR_UNSUPPORTED: return "unsupported shape";
    case SMLA_ERR_ALIGNMENT: return "misaligned pointer";
    case SMLA_ERR_WORKSPACE: return "buffer too small";
    case SMLA_ERR_CUDA: return "CUDA error";
    case SMLA_ERR_TIMEOUT: return "device wait timed out";
    case SMLA_ERR_DEVICE: return "device reported bad data";
  }
  return "unknown status";
}

smla_status sparse_mla_workspace_size(const smla_dims* dims, int num_sms, size_t* sched_bytes,
                                      size_t* accum_bytes) {
  smla_status st = check_dims(dims);
  if (st != SMLA_OK) return st;
  if (!sched_bytes || !accum_bytes) return SMLA_ERR_INVALID_ARG;
  int parts = 0;
  if ((st = resolve_parts(dims, num_sms, &parts)) != SMLA_OK) return st;
  *sched_bytes = plan_layout(dims->b, parts).bytes;
  *accum_bytes = workspace_layout(dims, parts).bytes;
  return SMLA_OK;
}

smla_status sparse_mla_sched_meta(const smla_dims* dims, int num_sms, void* sched_meta,
                                  size_t sched_bytes, void* stream) {
  smla_status st = check_dims(dims);
  if (st != SMLA_OK) return st;
  if (!sched_meta) return SMLA_ERR_INVALID_ARG;
  if (!aligned(sched_meta, 16)) return SMLA_ERR_ALIGNMENT;
  int parts = 0;
  if ((st = resolve_parts(dims, num_sms, &parts)) != SMLA_OK) return st;
  const PlanLayout L = plan_layout(dims->b, parts);
  if (sched_bytes < L.bytes) return SMLA_ERR_WORKSPACE;
  uint8_t* base = static_cast<uint8_t*>(sched_meta);
  if (dims->b == 0) {  // empty problem: only the status word needs clearing
    return cuda_status(cudaMemsetAsync(base + L.status_off, 0, 16, static_cast<cudaStream_t>(stream)));
  }
  return cuda_status(launch_sched(dims->b, dims->s_q, static_cast<int>(plan_topk(dims)), parts,
                                  reinterpret_cast<int32_t*>(base + L.meta_off),
                                  reinterpret_cast<int32_t*>(base + L.prefix_off),
                                  reinterpret_cast<uint32_t*>(base + L.status_off),
                                  static_cast<cudaStream_t>(stream)));
}

smla_status sparse_mla_decode_fwd(const smla_dims* dims, int num_sms, const void* q,
                                  const void* kv_cache, const int32_t* indices, float sm_scale,
                                  const void* sched_meta, void* workspace, size_t workspace_bytes,
                                  void* out, float* lse, void* stream) {
  return sparse_mla_decode_fwd_ex(dims, num_sms, q, kv_cache, indices, sm_scale, nullptr,
                                  sched_meta, workspace, workspace_bytes, out, lse, stream);
}

smla_status sparse_mla_decode_fwd_ex(const smla_dims* dims, int num_sms, const void* q,
                                     const void* kv_cache, const int32_t* indices,
                                     float sm_scale, const smla_decode_opts* opts,
                                     const void* sched_meta, void* workspace,
                                     size_t workspace_bytes, void* out, float* lse,
                                     void* stream) {
  smla_status st = check_dims(dims);
  if (st != SMLA_OK) return st;
  const int64_t tokens = static_cast<int64_t>(dims->b) * dims->s_q;
  if (tokens == 0) return SMLA_OK;
  if (!q || !sched_meta || !out || !lse) return SMLA_ERR_INVALID_ARG;
  if (dims->topk > 0 && (!indices || (dims->num_blocks > 0 && !kv_cache))) return SMLA_ERR_INVALID_ARG;
  const bool extra = dims->extra_topk > 0;
  if (extra && (!opts || !opts->extra_indices ||
                (dims->extra_num_blocks > 0 && !opts->extra_kv_cache)))
    return SMLA_ERR_INVALID_ARG;
  if (!std::isfinite(sm_scale)) return SMLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(workspace, 16) ||
      !aligned(sched_meta, 16) || !aligned(indices, 4) || !aligned(lse, 4))
    return SMLA_ERR_ALIGNMENT;
  if ((st = check_opts(opts)) != SMLA_OK) return st;
  int parts = 0, sms = 0;
  if ((st = resolve_parts(dims, num_sms, &parts, &sms)) != SMLA_OK) return st;
  const AccumLayout A = workspace_layout(dims, parts);
  if (A.bytes > 0 && !workspace) return SMLA_ERR_INVALID_ARG;
  if (workspace_bytes < A.bytes) return SMLA_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (plan_topk(dims) == 0)
    return cuda_status(launch_fill_empty(static_cast<__nv_bfloat16*>(out), lse,
                                         tokens * dims->h_q, tokens * dims->h_q, s));
  const PlanLayout L = plan_layout(dims->b, parts);
  const uint8_t* plan = static_cast<const uint8_t*>(sched_meta);
  DecodeParams p;
  if (!encode_rows_map(&p.q_map, q, false, tokens * dims->h_q, dims->d_qk, 64, dims->h_q) ||
      !encode_rows_map(&p.out_map, out, false, tokens * dims->h_q, kDV, 64, dims->h_q))
    return SMLA_ERR_CUDA;
  if (A.max_splits > 0) {
    uint8_t* acc = static_cast<uint8_t*>(workspace) + A.o_off;
    const int64_t rows = static_cast<int64_t>(A.max_splits) * dims->s_q * dims->h_q;
    if (!encode_rows_map(&p.acc_map, acc, true, rows, kDV, 32, dims->h_q) ||
        !encode_rows_map(&p.acc16_map, acc, false, rows, kDV, 64, dims->h_q))
      return SMLA_ERR_CUDA;
  } else {  // no split slot: the kernel stores no partial, so these maps are never used
    p.acc_map = p.out_map;
    p.acc16_map = p.out_map;
  }
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kv = static_cast<const uint8_t*>(kv_cache);
  p.indices = indices;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.o_accum = A.max_splits > 0 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + A.o_off)
                               : nullptr;
  p.lse_accum = A.max_splits > 0
                    ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + A.lse_off)
                    : nullptr;
  p.meta = reinterpret_cast<const int32_t*>(plan + L.meta_off);
  p.nsplits = reinterpret_cast<const int32_t*>(plan + L.prefix_off);
  p.status = const_cast<uint32_t*>(reinterpret_cast<const uint32_t*>(plan + L.status_off));
  p.attn_sink = opts != nullptr ? opts->attn_sink : nullptr;
  p.topk_length = opts != nullptr ? opts->topk_length : nullptr;
  p.partials_bf16 = opts != nullptr && opts->partials_bf16 != 0 ? 1 : 0;
  p.test_stall = opts != nullptr && opts->test_stall != 0 ? 1 : 0;
  p.b = dims->b;
  p.s_q = dims->s_q;
  p.h_q = dims->h_q;
  p.topk = dims->topk;
  // one wave of 2-CTA clusters: with more query positions than clusters that fit (one
  // partition each then), every cluster walks several positions in one launch
  {
    const int fit = sms / (2 * parts);
    p.s_step = dims->s_q < fit ? dims->s_q : (fit < 1 ? 1 : fit);
  }
  p.extra_kv = extra ? static_cast<const uint8_t*>(opts->extra_kv_cache) : nullptr;
  p.extra_indices = extra ? opts->extra_indices : nullptr;
  p.extra_topk_length = extra ? opts->extra_topk_length : nullptr;
  p.extra_topk = dims->extra_topk;
  p.extra_rows = static_cast<int>(dims->extra_num_blocks * kPage);
  p.nb_main = (dims->topk + kPage - 1) / kPage;
  p.nb_total = static_cast<int>((plan_topk(dims) + kPage - 1) / kPage);
  p.num_rows = static_cast<int>(dims->num_blocks * kPage);
  p.kv_fmt = dims->kv_format == SMLA_KV_V4 ? FMT_V4 : dims->kv_format == SMLA_KV_V41 ? FMT_V41 : FMT_V32;
  p.q_chunks = dims->d_qk / 64;
  p.store32 = aligned(out, 32) && (A.max_splits == 0 || aligned(workspace, 32)) ? 1 : 0;
  p.score_scale_log2 = static_cast<float>(static_cast<double>(sm_scale) * 1.4426950408889634 / 256.0);
  return cuda_status(launch_decode(p, parts, s));
}

smla_status sparse_mla_combine(const smla_dims* dims, int num_sms, const void* sched_meta,
                               const void* workspace, size_t workspace_bytes, void* out, float* lse,
                               void* stream) {
  return sparse_mla_combine_ex(dims, num_sms, nullptr, sched_meta, workspace, workspace_bytes,
                               out, lse, stream);
}

smla_status sparse_mla_combine_ex(const smla_dims* dims, int num_sms,
                                  const smla_decode_opts* opts, const void* sched_meta,
                                  const void* workspace, size_t workspace_bytes, void* out,
                                  float* lse, void* stream) {
  smla_status st = check_dims(dims);
  if (st != SMLA_OK) return st;
  const int64_t tokens = static_cast<int64_t>(dims->b) * dims->s_q;
  if (tokens == 0 || plan_topk(dims) == 0) return SMLA_OK;
  if (!sched_meta || !out || !lse) return SMLA_ERR_INVALID_ARG;
  if (!aligned(out, 16) || !aligned(workspace, 16) || !aligned(sched_meta, 16) || !aligned(lse, 4))
    return SMLA_ERR_ALIGNMENT;
  if ((st = check_opts(opts)) != SMLA_OK) return st;
  int parts = 0;
  if ((st = resolve_parts(dims, num_sms, &parts)) != SMLA_OK) return st;
  const AccumLayout A = workspace_layout(dims, parts);
  if (A.bytes > 0 && !workspace) return SMLA_ERR_INVALID_ARG;
  if (workspace_bytes < A.bytes) return SMLA_ERR_WORKSPACE;
  // no request is split: the decode pass wrote every row, so nothing is launched
  if (A.max_splits == 0) return SMLA_OK;
  const PlanLayout L = plan_layout(dims->b, parts);
  CombineParams p;
  p.o_accum = reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + A.o_off);
  p.lse_accum = reinterpret_cast<const float*>(static_cast<const uint8_t*>(workspace) + A.lse_off);
  p.nsplits = reinterpret_cast<const int32_t*>(static_cast<const uint8_t*>(sched_meta) + L.prefix_off);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.attn_sink = opts != nullptr ? opts->attn_sink : nullptr;
  p.partials_bf16 = opts != nullptr && opts->partials_bf16 != 0 ? 1 : 0;
  p.b = dims->b;
  p.s_q = dims->s_q;
  p.h_q = dims->h_q;
  return cuda_status(launch_combine(p, static_cast<cudaStream_t>(stream)));
}

smla_status sparse_mla_topk_page_table(const smla_topk_dims* d, const void* scores,
                                       const int32_t* valid_len, const int32_t* block_table,
                                       int32_t* out_indices, uint32_t* status, void* stream) {
  if (!d) return SMLA_ERR_INVALID_ARG;
  if (d->n_tok < 0 || d->s_q < 1 || d->topk < 1 || d->ld < 0 || d->max_pages < 0)
    return SMLA_ERR_INVALID_ARG;
  if (d->dtype != SMLA_SCORES_BF16 && d->dtype != SMLA_SCORES_FP32) return SMLA_ERR_UNSUPPORTED;
  if (d->n_tok == 0) return SMLA_OK;
  if (!valid_len || !block_table || !out_indices || (d->ld > 0 && !scores))
    return SMLA_ERR_INVALID_ARG;
  const int esize = d->dtype == SMLA_SCORES_FP32 ? 4 : 2;
  if (!aligned(scores, 16) || (static_cast<int64_t>(d->ld) * esize) % 16 != 0 ||
      !aligned(valid_len, 4) || !aligned(block_table, 4) || !aligned(out_indices, 4) ||
      !aligned(status, 4))
    return SMLA_ERR_ALIGNMENT;
  if (static_cast<int64_t>(d->n_tok) * d->topk > INT32_MAX ||
      static_cast<int64_t>(d->max_pages) * kPage > INT32_MAX)
    return SMLA_ERR_UNSUPPORTED;
  return cuda_status(launch_topk(scores, d->dtype == SMLA_SCORES_FP32, valid_len, block_table,
                                 out_indices, status, d->n_tok, d->s_q, d->topk, d->ld,
                                 d->max_pages, static_cast<cudaStream_t>(stream)));
}

smla_status sparse_mla_indexer_scores(const smla_indexer_dims* d, int num_sms, const void* q8,
                                      const float* weights, const void* k_cache,
                                      const int32_t* block_table, const int32_t* valid_len,
                                      float* scores, uint32_t* status, void* stream) {
  if (!d) return SMLA_ERR_INVALID_ARG;
  if (d->n_tok < 0 || d->s_q < 1 || d->ld < 0 || d->max_pages < 0 || d->num_pages < 0)
    return SMLA_ERR_INVALID_ARG;
  if (d->heads != 64 || d->dim != 128) return SMLA_ERR_UNSUPPORTED;
  if (d->n_tok % d->s_q != 0) return SMLA_ERR_INVALID_ARG;
  if (d->n_tok == 0 || d->ld == 0) return SMLA_OK;
  if (!q8 || !weights || !block_table || !valid_len || !scores || (d->num_pages > 0 && !k_cache))
    return SMLA_ERR_INVALID_ARG;
  if (!aligned(q8, 16) || !aligned(k_cache, 16) || !aligned(weights, 4) ||
      !aligned(block_table, 4) || !aligned(valid_len, 4) || !aligned(scores, 4) ||
      !aligned(status, 4))
    return SMLA_ERR_ALIGNMENT;
  if (static_cast<int64_t>(d->n_tok) * 64 > INT32_MAX || d->num_pages > INT32_MAX ||
      static_cast<int64_t>(d->n_tok) * d->ld > (int64_t(1) << 40))
    return SMLA_ERR_UNSUPPORTED;
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return SMLA_ERR_CUDA;
    }
  }
  IndexerLaunch L;
  const int G = d->s_q < 4 ? d->s_q : 4;
  const uint64_t kd[3] = {128, 64, static_cast<uint64_t>(d->num_pages > 0 ? d->num_pages : 1)};
  const uint64_t ks[2] = {128, 8448};
  const uint32_t kb[3] = {128, 64, 1};
  const uint64_t qd[2] = {128, static_cast<uint64_t>(d->n_tok) * 64};
  const uint64_t qs[1] = {128};
  const uint32_t qb[2] = {128, static_cast<uint32_t>(64 * G)};
  // the key scales of a page: 256 bytes at offset 8192, one row per page
  const uint64_t sd[2] = {256, kd[2]};
  const uint64_t ss[1] = {8448};
  const uint32_t sb[2] = {256, 1};
  // with no page at all both maps point at q8 (its first 8192 bytes are readable) and the
  // kernel takes every key scale as 0
  const void* kbase = d->num_pages > 0 ? k_cache : q8;
  const void* sbase = d->num_pages > 0 ? static_cast<const void*>(static_cast<const uint8_t*>(k_cache) + 8192) : q8;
  if (!encode_bytes_map(&L.k_map, kbase, 3, kd, ks, kb) || !encode_bytes_map(&L.q_map, q8, 2, qd, qs, qb) ||
      !encode_bytes_map(&L.s_map, sbase, 2, sd, ss, sb, false))
    return SMLA_ERR_CUDA;
  L.w = weights;
  L.table = block_table;
  L.valid_len = valid_len;
  L.cache = static_cast<const uint8_t*>(k_cache);
  L.out = scores;
  L.status = status;
  L.n_tok = d->n_tok;
  L.s_q = d->s_q;
  L.max_pages = d->max_pages;
  L.ld = d->ld;
  L.num_sms = num_sms;
  L.num_pages = d->num_pages;
  L.test_stall = d->test_stall;
  return cuda_status(launch_indexer(L, static_cast<cudaStream_t>(stream)));
}

// Positions the chained selection considers: min(ld, max_pages * 64), or -1 if dims is bad.
static int64_t select_len(const smla_indexer_dims* d) {
  if (!d || d->n_tok < 0 || d->s_q < 1 || d->ld < 0 || d->max_pages < 0) return -1;
  const int64_t cap = static_cast<int64_t>(d->max_pages) * kPage;
  return d->ld < cap ? d->ld : cap;
}

smla_status sparse_mla_indexer_topk_scratch_size(const smla_indexer_dims* d, size_t* bytes) {
  const int64_t L = select_len(d);
  if (L < 0 || !bytes) return SMLA_ERR_INVALID_ARG;
  const int64_t row = L * 4;
  int64_t rows = row > 0 ? static_cast<int64_t>(SMLA_SELECT_SCRATCH_BUDGET) / row : d->n_tok;
  if (rows < 1) rows = 1;
  if (rows > d->n_tok) rows = d->n_tok;
  *bytes = static_cast<size_t>(rows * (row > 0 ? row : 16));
  return SMLA_OK;
}

smla_status sparse_mla_indexer_topk(const smla_indexer_dims* d, int32_t topk, int num_sms,
                                    const void* q8, const float* weights, const void* k_cache,
                                    const int32_t* block_table, const int32_t* valid_len,
                                    void* scratch, size_t scratch_bytes, int32_t* out_indices,
                                    uint32_t* status, void* stream) {
  const int64_t L = select_len(d);
  if (L < 0 || topk < 1) return SMLA_ERR_INVALID_ARG;
  if (d->heads != 64 || d->dim != 128) return SMLA_ERR_UNSUPPORTED;
  if (d->n_tok % d->s_q != 0) return SMLA_ERR_INVALID_ARG;
  if (d->n_tok == 0) return SMLA_OK;
  if (!scratch || !out_indices || !q8 || !weights || !block_table || !valid_len || !status)
    return SMLA_ERR_INVALID_ARG;
  if (d->ld % 4 != 0 || !aligned(scratch, 16)) return SMLA_ERR_ALIGNMENT;
  const int64_t row = L * 4;
  if (row > 0 && scratch_bytes < static_cast<size_t>(row)) return SMLA_ERR_WORKSPACE;
  const int64_t R = row > 0 ? static_cast<int64_t>(scratch_bytes / static_cast<size_t>(row)) : d->n_tok;
  const int n_req = d->n_tok / d->s_q;
  const uint8_t* q = static_cast<const uint8_t*>(q8);
  for (int64_t t = 0; t < d->n_tok;) {
    const int64_t r = t / d->s_q;
    int64_t n, sub_sq;
    if (d->s_q <= R) {  // whole requests
      int64_t reqs = R / d->s_q;
      if (reqs > n_req - r) reqs = n_req - r;
      n = reqs * d->s_q;
      sub_sq = d->s_q;
    } else {  // a run of one request's tokens, as a request of its own
      n = (r + 1) * d->s_q - t;
      if (n > R) n = R;
      sub_sq = n;
    }
    smla_indexer_dims ix = *d;
    ix.n_tok = static_cast<int32_t>(n);
    ix.s_q = static_cast<int32_t>(sub_sq);
    ix.ld = static_cast<int32_t>(L);
    const int32_t* table = block_table + r * d->max_pages;
    smla_status st = sparse_mla_indexer_scores(&ix, num_sms, q + t * 64 * 128, weights + t * 64,
                                               k_cache, table, valid_len + t,
                                               static_cast<float*>(scratch), status, stream);
    if (st != SMLA_OK) return st;
    smla_topk_dims tk;
    tk.n_tok = static_cast<int32_t>(n);
    tk.s_q = static_cast<int32_t>(sub_sq);
    tk.topk = topk;
    tk.ld = static_cast<int32_t>(L);
    tk.max_pages = d->max_pages;
    tk.dtype = SMLA_SCORES_FP32;
    st = sparse_mla_topk_page_table(&tk, scratch, valid_len + t, table, out_indices + t * topk,
                                    status, stream);
    if (st != SMLA_OK) return st;
    t += n;
  }
  return SMLA_OK;
}

smla_status sparse_mla_plan_has_splits(const smla_dims* dims, int num_sms, int* has_splits) {
  smla_status st = check_dims(dims);
  if (st != SMLA_OK) return st;
  if (!has_splits) return SMLA_ERR_INVALID_ARG;
  int parts = 0;
  if ((st = resolve_parts(dims, num_sms, &parts)) != SMLA_OK) return st;
  *has_splits = split_slots(dims->b, plan_topk(dims), parts) > 0 ? 1 : 0;
  return SMLA_OK;
}

smla_status sparse_mla_read_device_status(const smla_dims* dims, int num_sms,
                                          const void* sched_meta, int* code, void* stream) {
  smla_status st = check_dims(dims);
  if (st != SMLA_OK) return st;
  if (!sched_meta || !code) return SMLA_ERR_INVALID_ARG;
  int parts = 0;
  if ((st = resolve_parts(dims, num_sms, &parts)) != SMLA_OK) return st;
  const PlanLayout L = plan_layout(dims->b, parts);
  uint32_t word = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, static_cast<const uint8_t*>(sched_meta) + L.status_off, 4,
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return cuda_status(cudaErrorUnknown);
  if (cudaStreamSynchronize(s) != cudaSuccess) return cuda_status(cudaErrorUnknown);
  *code = static_cast<int>(word);
  if (word & SMLA_DEV_TIMEOUT) return SMLA_ERR_TIMEOUT;
  if (word) return SMLA_ERR_DEVICE;
  return SMLA_OK;
}

}  // extern "C"
