// Internal declarations shared by the host runtime and the kernels of libsparse_mla.so.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace smla {

constexpr int kDQk = 576, kDNope = 512, kDRope = 64, kDV = 512;
constexpr int kRowBytes = 656;  // 512 e4m3 + 4 x fp32 scale + 64 x bf16
constexpr int kPage = 64;
// KV-cache formats of the decode kernel: the 656-byte V3.2 row (d_qk 576) and the later
// structure-of-arrays pages (d_qk 512; the FP4 form only as the extra cache of a V4.1 cache)
enum : int { FMT_V32 = 0, FMT_V4 = 1, FMT_V41 = 2, FMT_V41_FP4 = 3 };
template <int kF>
struct FmtBytes {  // bytes of one token's data row and scale row
  static constexpr int kData = 0, kScale = 0;
};
template <>
struct FmtBytes<FMT_V4> {
  static constexpr int kData = 448 + 64 * 2, kScale = 8;
};
template <>
struct FmtBytes<FMT_V41> {
  static constexpr int kData = 512, kScale = 16;
};
constexpr int FP4_DATA = 256, FP4_SCALE = 32;
constexpr int kTopkBlock = 64;  // slots of the top-k list per pipeline block
constexpr int kFixedOverhead = 5;
constexpr int kMetaInts = 8;    // int32 fields per partition in the plan

// Layout of the caller's plan buffer.
struct PlanLayout {
  int parts;
  size_t meta_off, prefix_off, status_off, bytes;
};
inline PlanLayout plan_layout(int b, int parts) {
  PlanLayout L;
  L.parts = parts;
  L.meta_off = 0;
  L.prefix_off = static_cast<size_t>(parts) * kMetaInts * 4;
  size_t end = L.prefix_off + static_cast<size_t>(b + 1) * 4;
  L.status_off = (end + 15) & ~static_cast<size_t>(15);
  L.bytes = L.status_off + 64;
  return L;
}
// Layout of the split-partial workspace: o_accum fp32 [slots][s_q][h_q][512] then lse_accum
// fp32 [slots][s_q][h_q] (base-2 log-sum-exp), where slots is the number of split slots the
// plan numbers up to its last split request (split_slots); a plan that splits no request
// needs no workspace at all.
struct AccumLayout {
  int max_splits;
  size_t o_off, lse_off, bytes;
};
inline AccumLayout accum_layout_slots(int slots, int s_q, int h_q) {
  AccumLayout L;
  L.max_splits = slots;
  L.o_off = 0;
  size_t o_bytes = static_cast<size_t>(slots) * s_q * h_q * kDV * 4;
  L.lse_off = (o_bytes + 255) & ~static_cast<size_t>(255);
  L.bytes = slots > 0 ? L.lse_off + static_cast<size_t>(slots) * s_q * h_q * 4 : 0;
  return L;
}

struct DecodeParams {
  // Q as a 2-D tensor (rows = token * h_q + head, 576 bf16 columns), box 64 columns x h_q rows,
  // 128-byte swizzle: one box is one 64-dim chunk of a token's Q in the SW128 K-major layout.
  CUtensorMap q_map;    // (the type is 64-byte aligned)
  // out as rows (token * h_q + head) x 512 bf16, box 64 columns x h_q rows, 128-byte swizzle
  CUtensorMap out_map;
  // o_accum as rows ((split * s_q + s) * h_q + head) x 512 fp32, box 32 columns x h_q rows
  CUtensorMap acc_map;
  // the same rows as bf16 (partials_bf16), box 64 columns x h_q rows
  CUtensorMap acc16_map;
  const __nv_bfloat16* q;   // [b][s_q][h_q][576]
  const uint8_t* kv;        // [num_rows][656]
  const int32_t* indices;   // [b][s_q][topk]
  __nv_bfloat16* out;       // [b][s_q][h_q][512]
  float* lse;               // [b][h_q][s_q]
  float* o_accum;           // [max_splits][s_q][h_q][512]
  float* lse_accum;         // [max_splits][s_q][h_q]
  const int32_t* meta;      // [parts][8]
  const int32_t* nsplits;   // [b + 1]
  uint32_t* status;         // device status word
  const float* attn_sink;   // [h_q] or null
  const int32_t* topk_length;  // [b][s_q] or null
  const uint8_t* extra_kv;        // [extra_rows][656] or null
  const int32_t* extra_indices;   // [b][s_q][extra_topk] or null
  const int32_t* extra_topk_length;  // [b][s_q] or null
  int extra_topk, extra_rows;
  int nb_main, nb_total;    // blocks of the main list; of both lists (the plan's blocks)
  int b, s_q, h_q, topk;
  // clusters per partition: cluster y takes the query positions s = y, y + s_step, ... (< s_q)
  int s_step;
  int num_rows;             // num_blocks * 64
  float score_scale_log2;   // sm_scale * log2(e) / 256 (keys are dequantized scaled by 256)
  int kv_fmt;               // FMT_V32, FMT_V4 or FMT_V41 (the main cache)
  int q_chunks;             // 64-dim chunks of q and of the key: 9 (d_qk 576) or 8 (512)
  int store32;              // out and the workspace are 32-byte aligned (256-bit stores)
  int partials_bf16;        // split partials of O stored as bf16 rows (else fp32)
  int test_stall;           // failure-path test hook (see smla_decode_opts)
};

struct CombineParams {
  const float* o_accum;
  const float* lse_accum;
  const int32_t* nsplits;
  __nv_bfloat16* out;
  float* lse;
  const float* attn_sink;  // [h_q] or null
  int partials_bf16;       // o_accum holds bf16 rows (else fp32)
  int b, s_q, h_q;
};

// Encodes a 2-D row-major tensor map (rows x cols, 128-byte swizzle, box box_cols x box_rows)
// (host; false if the driver call is missing or fails).
bool encode_rows_map(CUtensorMap* map, const void* base, bool fp32, int64_t rows, int cols,
                     int box_cols, int box_rows);

// Kernel launchers (return the launch's cudaError_t).
cudaError_t launch_sched(int b, int s_q, int topk, int parts, int32_t* meta, int32_t* prefix,
                         uint32_t* status, cudaStream_t stream);
cudaError_t launch_decode(const DecodeParams& p, int parts, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream);
// Indexer scores (csrc/indexer.cu): the tensor maps are encoded by the host API.
struct IndexerLaunch {
  CUtensorMap k_map, q_map, s_map;
  const float* w;
  const int32_t* table;
  const int32_t* valid_len;
  const uint8_t* cache;
  float* out;
  uint32_t* status;
  int n_tok, s_q, max_pages, ld, num_sms;
  int64_t num_pages;
  int test_stall;
};
cudaError_t launch_indexer(const IndexerLaunch& L, cudaStream_t stream);
// Encodes a byte tensor map, with a 128-byte swizzle unless swizzle128 is false: dims /
// strides (bytes) / box, 2 or 3 dims.
bool encode_bytes_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides, const uint32_t* box, bool swizzle128 = true);
cudaError_t launch_topk(const void* scores, bool fp32, const int32_t* valid_len,
                        const int32_t* table, int32_t* out, uint32_t* status, int n_tok, int s_q,
                        int k, int ld, int max_pages, cudaStream_t stream);
cudaError_t launch_fill_empty(__nv_bfloat16* out, float* lse, int64_t rows_o, int64_t n_lse,
                              cudaStream_t stream);

}  // namespace smla
