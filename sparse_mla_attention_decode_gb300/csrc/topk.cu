// Exact top-k of index scores with the page-table emit: the step that turns a query token's
// scores over its visible context into the physical cache ids the sparse attention reads
// ("FlashMLA 与 DSA：内核、流水线和正确性边界", section 5.5; "sparse-attention co-design",
// section 5, step five).
//
// One CTA per query token (row).  Scores map to order-preserving unsigned keys (16-bit for
// bf16, 32-bit for fp32) and the k-th largest key is found 8 bits at a time, most significant
// first (a radix select):
//   pass 1   histogram of the top 8 key bits over the valid prefix of the row;
//   level 0  the threshold bin b is the one where the count of larger bins stops reaching k;
//            a second pass over the row emits every element of a larger bin, keeps the
//            positions of bin b as candidates in shared memory and builds the histogram of
//            their next 8 bits;
//   level l  the same on the candidates only, until every key bit is fixed; the elements left
//            then all equal the k-th largest key and fill the remaining slots by a countdown.
// If bin b holds more candidates than shared memory, the next levels re-read the row and
// filter it by the key prefix instead (slower, same result).  Elements are emitted as
// block_table[req][u / 64] * 64 + u % 64 directly into the output row, in no particular
// order; a row with at most k valid positions emits all of them and pads with -1.
#include <cstdint>

#include "../../include/sparse_mla.h"
#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int TK_THREADS = 1024;
constexpr int TK_CAP = 8192;  // candidate positions per buffer (two buffers)

struct TopkParams {
  const void* scores;
  const int32_t* valid_len;
  const int32_t* table;
  int32_t* out;
  uint32_t* status;
  int n_tok, s_q, k, ld, max_pages;
};

// Order-preserving keys: a larger score gives a larger unsigned key (negative values have
// all their bits flipped, non-negative ones only the sign bit).
template <bool kF32>
__device__ __forceinline__ uint32_t key_at(const TopkParams& p, const void* row, int u) {
  if (kF32) {
    const uint32_t x = __float_as_uint(reinterpret_cast<const float*>(row)[u]);
    return x ^ ((x >> 31) ? 0xFFFFFFFFu : 0x80000000u);
  }
  const uint32_t x = reinterpret_cast<const uint16_t*>(row)[u];
  return x ^ ((x & 0x8000u) ? 0xFFFFu : 0x8000u);
}

struct TopkShared {
  uint32_t hist[256];
  uint32_t n_out, n_cand, ties, overflow, bad;
  uint32_t bin, above;  // threshold bin of the current level and the count of larger bins
};

__device__ __forceinline__ void emit(const TopkParams& p, TopkShared& sh, int row, int req,
                                     int u) {
  const uint32_t pos = atomicAdd(&sh.n_out, 1u);
  if (pos >= static_cast<uint32_t>(p.k)) return;
  const int pg = u >> 6;
  int32_t id = -1;
  if (pg < p.max_pages) id = p.table[static_cast<size_t>(req) * p.max_pages + pg] * 64 + (u & 63);
  else sh.bad = 1u;
  p.out[static_cast<size_t>(row) * p.k + pos] = id;
}

// Threshold of one level: the bin b whose suffix count (bins >= b) first reaches `need`,
// and the count of the bins above it.  One warp; lane L owns bins 8 L .. 8 L + 7.
__device__ __forceinline__ void find_threshold(TopkShared& sh, uint32_t need) {
  const int lane = threadIdx.x & 31;
  uint32_t c[8], local = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    c[i] = sh.hist[8 * lane + i];
    local += c[i];
  }
  // count in the lanes above this one (bins above 8 lane + 7)
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += v;
  }
  uint32_t above = incl - local;
  if (above < need && incl >= need) {  // the threshold bin is in this lane
#pragma unroll
    for (int i = 7; i >= 0; --i) {
      if (above + c[i] >= need) {
        sh.bin = static_cast<uint32_t>(8 * lane + i);
        sh.above = above;
        break;
      }
      above += c[i];
    }
  }
}

template <bool kF32>
__global__ void __launch_bounds__(TK_THREADS) topk_kernel(const TopkParams p) {
  constexpr int kKeyBits = kF32 ? 32 : 16;
  constexpr int kLevels = kKeyBits / 8;
  constexpr int kVec = kF32 ? 4 : 8;  // elements per 16-byte load
  extern __shared__ uint32_t tk_smem[];
  __shared__ TopkShared sh;
  uint32_t* cand[2] = {tk_smem, tk_smem + TK_CAP};
  const int row = blockIdx.x, tid = threadIdx.x;
  const int req = row / p.s_q;
  int len = p.valid_len[row];
  len = len < 0 ? 0 : (len > p.ld ? p.ld : len);
  const uint8_t* rowp = static_cast<const uint8_t*>(p.scores) +
                        static_cast<size_t>(row) * p.ld * (kF32 ? 4 : 2);
  if (tid == 0) {
    sh.n_out = 0;
    sh.n_cand = 0;
    sh.ties = 0;
    sh.overflow = 0;
    sh.bad = 0;
  }
  if (len <= p.k) {  // every valid position is selected
    for (int u = tid; u < p.k; u += TK_THREADS) {
      int32_t id = -1;
      if (u < len) {
        const int pg = u >> 6;
        if (pg < p.max_pages) id = p.table[static_cast<size_t>(req) * p.max_pages + pg] * 64 + (u & 63);
        else atomicOr(p.status != nullptr ? p.status : &sh.bad, SMLA_DEV_TOPK_TABLE);
      }
      p.out[static_cast<size_t>(row) * p.k + u] = id;
    }
    return;
  }
  for (int i = tid; i < 256; i += TK_THREADS) sh.hist[i] = 0;
  __syncthreads();
  // pass 1: top 8 key bits over the valid prefix, 16 bytes per load
  const int nvec = len / kVec;
  for (int v = tid; v < nvec; v += TK_THREADS) {
    const uint4 w = *reinterpret_cast<const uint4*>(rowp + static_cast<size_t>(v) * 16);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
      uint32_t key;
      if (kF32) {
        const uint32_t x = ws[e];
        key = x ^ ((x >> 31) ? 0xFFFFFFFFu : 0x80000000u);
      } else {
        const uint32_t x = (ws[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
        key = x ^ ((x & 0x8000u) ? 0xFFFFu : 0x8000u);
      }
      atomicAdd(&sh.hist[key >> (kKeyBits - 8)], 1u);
    }
  }
  for (int u = nvec * kVec + tid; u < len; u += TK_THREADS)
    atomicAdd(&sh.hist[key_at<kF32>(p, rowp, u) >> (kKeyBits - 8)], 1u);
  __syncthreads();
  uint32_t need = static_cast<uint32_t>(p.k);
  uint32_t prefix = 0;  // key bits fixed so far (the top 8 * level bits)
  if (tid < 32) find_threshold(sh, need);
  __syncthreads();
  // Levels: at level l the threshold bin b of bits [kKeyBits - 8 (l + 1), kKeyBits - 8 l) is
  // known; one pass over the level's elements emits the larger bins, keeps bin b (the next
  // level's candidates) and builds the next level's histogram.
  int src = -1;  // -1: the whole row (filtered by prefix); 0 / 1: a candidate buffer
  for (int level = 0; level < kLevels; ++level) {
    const uint32_t b = sh.bin;
    const uint32_t above = sh.above;
    const int shift = kKeyBits - 8 * (level + 1);
    const bool last = level == kLevels - 1;
    const uint32_t take = need - above;  // of bin b, this many are selected
    const uint32_t n_src = src < 0 ? 0u : sh.n_cand;
    const bool all_of_bin = take == sh.hist[b];
    __syncthreads();
    if (tid == 0) sh.n_cand = 0;
    for (int i = tid; i < 256; i += TK_THREADS) sh.hist[i] = 0;
    __syncthreads();
    const int dst = src == 0 ? 1 : 0;
    auto visit = [&](int u, uint32_t key) {
      const uint32_t d = (key >> shift) & 0xFFu;
      if (d > b) {
        emit(p, sh, row, req, u);
      } else if (d == b) {
        if (last || all_of_bin) {
          // every element of bin b is selected, or the keys are fully fixed: fill by countdown
          if (all_of_bin || atomicAdd(&sh.ties, 1u) < take) emit(p, sh, row, req, u);
        } else {
          const uint32_t slot = atomicAdd(&sh.n_cand, 1u);
          if (slot < TK_CAP) cand[dst][slot] = static_cast<uint32_t>(u);
          else sh.overflow = 1u;
          atomicAdd(&sh.hist[(key >> (shift - 8)) & 0xFFu], 1u);
        }
      }
    };
    if (src < 0) {
      // the whole row: elements whose fixed key bits match the prefix
      const int pshift = kKeyBits - 8 * level;  // bits above this level
      for (int u = tid; u < len; u += TK_THREADS) {
        const uint32_t key = key_at<kF32>(p, rowp, u);
        if (level == 0 || (key >> pshift) == prefix) visit(u, key);
      }
    } else {
      for (uint32_t i = tid; i < n_src; i += TK_THREADS) {
        const int u = static_cast<int>(cand[src][i]);
        visit(u, key_at<kF32>(p, rowp, u));
      }
    }
    __syncthreads();
    if (last || all_of_bin) break;
    prefix = (prefix << 8) | b;
    need = take;
    src = sh.overflow ? -1 : dst;  // after an overflow the next levels re-read the row
    if (tid < 32) find_threshold(sh, need);
    __syncthreads();
  }
  if (tid == 0 && sh.bad && p.status != nullptr) atomicOr(p.status, SMLA_DEV_TOPK_TABLE);
}

}  // namespace

cudaError_t launch_topk(const void* scores, bool fp32, const int32_t* valid_len,
                        const int32_t* table, int32_t* out, uint32_t* status, int n_tok, int s_q,
                        int k, int ld, int max_pages, cudaStream_t stream) {
  TopkParams p{scores, valid_len, table, out, status, n_tok, s_q, k, ld, max_pages};
  const size_t smem = 2 * TK_CAP * sizeof(uint32_t);
  void (*kernel)(TopkParams) = fp32 ? topk_kernel<true> : topk_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kernel<<<n_tok, TK_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
