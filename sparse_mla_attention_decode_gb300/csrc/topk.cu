// Exact top-k of index scores with the page-table emit: the step that turns a query token's
// scores over its visible context into the physical cache ids the sparse attention reads
// ("FlashMLA 与 DSA：内核、流水线和正确性边界", section 5.5; "sparse-attention co-design",
// section 5, step five).
//
// One CTA per query token (row).  Scores map to order-preserving unsigned keys (16-bit for
// bf16, 32-bit for fp32) and the k-th largest key is found a few bits at a time, most
// significant first (a radix select):
//   pass 1   histogram of the top 12 key bits over the valid prefix of the row;
//   level 0  the threshold bin b is the one where the count of larger bins stops reaching k;
//            a second pass over the row emits every element of a larger bin, keeps the
//            positions of bin b as candidates in shared memory and builds the histogram of
//            their next bits;
//   level l  the same on the candidates only, until every key bit is fixed (bf16: 12 + 4
//            bits, fp32: 12 + 10 + 10); the elements left then all equal the k-th largest key
//            and fill the remaining slots by a countdown.
// The pages' kernel starts with 8 bits; 12 bits (an eighth of a binade per bin) keep the
// threshold bin of bell-shaped scores a few percent of the row instead of a quarter of it.
// If bin b holds more candidates than shared memory, the next levels re-read the row and
// filter it by the key prefix instead (slower, same result).  Emits and candidate pushes take
// one shared atomic per warp.  Elements are emitted as block_table[req][u / 64] * 64 + u % 64
// directly into the output row, in no particular order; a row with at most k valid positions
// emits all of them and pads with -1.
#include <cstdint>

#include "../../include/sparse_mla.h"
#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

#ifndef SMLA_TOPK_THREADS
#define SMLA_TOPK_THREADS 1024
#endif
#ifndef SMLA_TOPK_CAP
#define SMLA_TOPK_CAP 8192
#endif
#ifndef SMLA_TOPK_UNROLL
#define SMLA_TOPK_UNROLL 1
#endif
#ifndef SMLA_TOPK_MINB
#define SMLA_TOPK_MINB 2
#endif
constexpr int TK_THREADS = SMLA_TOPK_THREADS;
constexpr int TK_CAP = SMLA_TOPK_CAP;         // candidate positions of the first buffer
constexpr int TK_CAP1 = TK_CAP / 2;           // of the second (the later levels keep fewer)
constexpr int TK_UNROLL = SMLA_TOPK_UNROLL;   // 16-byte loads per thread in flight
constexpr int TK_BINS = 4096;  // the widest level (12 bits)

struct TopkParams {
  const void* scores;
  const int32_t* valid_len;
  const int32_t* table;
  int32_t* out;
  uint32_t* status;
  int n_tok, s_q, k, ld, max_pages;
};

// Key bits resolved by each level, most significant first.
template <bool kF32>
__device__ __forceinline__ constexpr int level_bits(int l) {
  return l == 0 ? 12 : (kF32 ? 10 : 4);
}
template <bool kF32>
__device__ __forceinline__ constexpr int levels() {
  return kF32 ? 3 : 2;
}

// Order-preserving keys: a larger score gives a larger unsigned key (negative values have
// all their bits flipped, non-negative ones only the sign bit).
template <bool kF32>
__device__ __forceinline__ uint32_t to_key(uint32_t x) {
  if (kF32) return x ^ ((x >> 31) ? 0xFFFFFFFFu : 0x80000000u);
  return x ^ ((x & 0x8000u) ? 0xFFFFu : 0x8000u);
}
template <bool kF32>
__device__ __forceinline__ uint32_t key_at(const uint8_t* row, int u) {
  if (kF32) return to_key<true>(__float_as_uint(reinterpret_cast<const float*>(row)[u]));
  return to_key<false>(reinterpret_cast<const uint16_t*>(row)[u]);
}
// Element e of a 16-byte vector (4 fp32 or 8 bf16) as a key.
template <bool kF32>
__device__ __forceinline__ uint32_t vec_key(const uint4& w, int e) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  if (kF32) return to_key<true>(ws[e]);
  return to_key<false>((ws[e >> 1] >> (16 * (e & 1))) & 0xFFFFu);
}

// Bit e set when element e of a 16-byte vector has a key of at least t (the full-width key of
// the sampled boundary).  Keys grow with the score, so when t lies in the upper half of the key
// range (a non-negative threshold) an element qualifies exactly when its bits, read as a signed
// integer, are at least t - 2^(n-1): negative scores never do.  `a` is that bound, for bf16
// shifted into the upper 16 bits (a bf16 in the upper half of a word is compared as the whole
// word, one in the lower half after a shift).  Other thresholds compare the keys.
template <bool kF32>
__device__ __forceinline__ uint32_t keep_mask(const uint4& w, bool fast, int32_t a, uint32_t t) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
  uint32_t m = 0;
  if (fast) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (kF32) {
        m |= static_cast<uint32_t>(static_cast<int32_t>(ws[i]) >= a) << i;
      } else {
        m |= static_cast<uint32_t>(static_cast<int32_t>(ws[i] << 16) >= a) << (2 * i);
        m |= static_cast<uint32_t>(static_cast<int32_t>(ws[i]) >= a) << (2 * i + 1);
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < (kF32 ? 4 : 8); ++e) m |= static_cast<uint32_t>(vec_key<kF32>(w, e) >= t) << e;
  }
  return m;
}

struct TopkShared {
  uint32_t n_out, n_cand, ties, overflow, bad;
  uint32_t bin, above;       // threshold bin of the current level and the count of larger bins
  uint32_t warp_sum[32], warp_above[32];
  uint32_t b_low;            // the sampled boundary bin (read by the peer of a CTA pair)
};

// Reads a 32-bit word of the peer CTA's shared memory (a shared::cluster address from mapa).
__device__ __forceinline__ uint32_t ld_peer_u32(uint32_t cluster_addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}

// Claims `take ? 1 : 0` consecutive slots of *counter for this lane with one atomic per warp;
// returns this lane's slot (meaningful when take).
__device__ __forceinline__ uint32_t warp_append(uint32_t* counter, bool take) {
  const unsigned mask = __activemask();
  const unsigned bal = __ballot_sync(mask, take);
  if (bal == 0u) return 0u;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(bal) - 1;
  uint32_t base = 0;
  if (lane == leader) base = atomicAdd(counter, static_cast<uint32_t>(__popc(bal)));
  base = __shfl_sync(mask, base, leader);
  return base + static_cast<uint32_t>(__popc(bal & ((1u << lane) - 1u)));
}

// Reserves `n` consecutive slots of *counter for this lane (warp scan of the counts, one
// atomic by the last active lane); returns this lane's first slot.
__device__ __forceinline__ uint32_t warp_reserve(uint32_t* counter, uint32_t n) {
  const unsigned mask = __activemask();
  const int lane = threadIdx.x & 31;
  uint32_t incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(mask, incl, o);
    if (lane >= o && ((mask >> (lane - o)) & 1u)) incl += v;
  }
  const int last = 31 - __clz(mask);
  uint32_t base = 0;
  if (lane == last && incl != 0u) base = atomicAdd(counter, incl);
  base = __shfl_sync(mask, base, last);
  return base + incl - n;
}

__device__ __forceinline__ void emit_at(const TopkParams& p, TopkShared& sh, int row, int req,
                                        uint32_t pos, int u) {
  if (pos >= static_cast<uint32_t>(p.k)) return;
  const int pg = u >> 6;
  int32_t id = -1;
  if (pg < p.max_pages) id = p.table[static_cast<size_t>(req) * p.max_pages + pg] * 64 + (u & 63);
  else sh.bad = 1u;
  p.out[static_cast<size_t>(row) * p.k + pos] = id;
}

// Threshold of one level over hist[0, nbins): the bin b whose suffix count (bins >= b) first
// reaches `need`, and the count of the bins above it.  Thread t owns bins [t * per, t * per +
// per); a block-wide suffix scan (shuffles, then the 32 warp totals) finds the owner.
__device__ void find_threshold(TopkShared& sh, const uint32_t* hist, int nbins, uint32_t need) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = nbins >= TK_THREADS ? nbins / TK_THREADS : 1;
  const int b0 = tid * per;
  uint32_t local = 0;
  if (b0 < nbins)
    for (int i = 0; i < per; ++i) local += hist[b0 + i];
  uint32_t incl = local;  // sum over this and the higher lanes of the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += v;
  }
  if (lane == 0) sh.warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const uint32_t w = lane < TK_THREADS / 32 ? sh.warp_sum[lane] : 0u;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_down_sync(0xffffffffu, wi, o);
      if (lane + o < 32) wi += v;
    }
    sh.warp_above[lane] = wi - w;  // the warps above this one
  }
  __syncthreads();
  incl += sh.warp_above[warp];
  uint32_t above = incl - local;
  if (b0 < nbins && above < need && incl >= need) {
    for (int i = per - 1; i >= 0; --i) {
      const uint32_t c = hist[b0 + i];
      if (above + c >= need) {
        sh.bin = static_cast<uint32_t>(b0 + i);
        sh.above = above;
        break;
      }
      above += c;
    }
  }
  __syncthreads();
}

// kPair: the row is split over a cluster of two CTAs (small batches, two SMs per row): each CTA
// takes the sampled pass and the candidate pass over half of the row's vectors (rank 1 also the
// tail); their histograms and candidates are then merged into rank 0 through distributed
// shared memory, and rank 0 alone runs the levels.  Both CTAs pass the same four cluster
// barriers on every path (a row with at most k valid positions takes none).
template <bool kF32, bool kPair>
__device__ __forceinline__ void topk_row(const TopkParams& p, TopkShared& sh, uint32_t* tk_smem,
                                         int row, uint32_t rank) {
  constexpr int kKeyBits = kF32 ? 32 : 16;
  constexpr int kVec = kF32 ? 4 : 8;  // elements per 16-byte load
  uint32_t* hist = tk_smem;                  // [TK_BINS]
  uint32_t* cand0 = tk_smem + TK_BINS;       // [TK_CAP]
  uint32_t* ckey0 = cand0 + TK_CAP;          // [TK_CAP] keys of the first candidates
  uint32_t* cand1 = ckey0 + TK_CAP;          // [TK_CAP1]
  const int tid = threadIdx.x;
  const int req = row / p.s_q;
  int len = p.valid_len[row];
  len = len < 0 ? 0 : (len > p.ld ? p.ld : len);
  const uint8_t* rowp = static_cast<const uint8_t*>(p.scores) +
                        static_cast<size_t>(row) * p.ld * (kF32 ? 4 : 2);
  if (len <= p.k) {  // every valid position is selected
    if (kPair && rank != 0) return;
    for (int u = tid; u < p.k; u += TK_THREADS) {
      int32_t id = -1;
      if (u < len) {
        const int pg = u >> 6;
        if (pg < p.max_pages) id = p.table[static_cast<size_t>(req) * p.max_pages + pg] * 64 + (u & 63);
        else if (p.status != nullptr) atomicOr(p.status, SMLA_DEV_TOPK_TABLE);
      }
      p.out[static_cast<size_t>(row) * p.k + u] = id;
    }
    return;
  }
  if (tid == 0) {
    sh.n_out = 0;
    sh.n_cand = 0;
    sh.ties = 0;
    sh.overflow = 0;
    sh.bad = 0;
    sh.bin = 0;    // stays 0 when a threshold search finds no bin (fewer elements than asked)
    sh.above = 0;
  }
  const int nvec = len / kVec;
  // this CTA's vectors [v_lo, v_hi) and tail (the positions past the whole vectors)
  const int v_lo = kPair && rank == 1 ? nvec / 2 : 0;
  const int v_hi = kPair && rank == 0 ? nvec / 2 : nvec;
  const bool own_tail = !kPair || rank == 1;
  // Sampled pass: the 12-bit histogram of every 16th vector picks a boundary bin b_low that
  // (from the sample) about 1.25 k + 256 elements reach; one full pass then keeps every element
  // of bin b_low or above as a candidate, with the exact histogram of the candidates.  The top
  // k are all among the candidates when there are at least k of them; with fewer, or more than
  // the buffer holds, the exact method below runs on the whole row instead.
  // the CTA's part of the row on its way into L2 (16 KB per request) while the sampled pass
  // runs, so that the full pass reads it from L2
  {
    const uint32_t bytes = static_cast<uint32_t>(v_hi - v_lo) * 16u;
    for (uint32_t c = static_cast<uint32_t>(tid); c * 16384u < bytes; c += TK_THREADS)
      bulk_prefetch_l2(rowp + static_cast<size_t>(v_lo) * 16 + c * 16384u,
                       bytes - c * 16384u < 16384u ? bytes - c * 16384u : 16384u);
  }
  for (int i = tid; i < TK_BINS; i += TK_THREADS) hist[i] = 0;
  __syncthreads();
  for (int v = v_lo + tid * 16; v < v_hi; v += TK_THREADS * 16) {
    const uint4 w = *reinterpret_cast<const uint4*>(rowp + static_cast<size_t>(v) * 16);
#pragma unroll
    for (int e = 0; e < kVec; ++e) atomicAdd(&hist[vec_key<kF32>(w, e) >> (kKeyBits - 12)], 1u);
  }
  __syncthreads();
  uint32_t b_low;
  if (kPair) {
    cluster_sync();  // (1) both sampled histograms are complete
    if (rank == 0) {
      const uint32_t peer = mapa(smem_u32(hist), 1);
      for (int i = tid; i < TK_BINS; i += TK_THREADS) hist[i] += ld_peer_u32(peer + 4u * i);
      __syncthreads();
      find_threshold(sh, hist, 1 << 12, static_cast<uint32_t>((5 * p.k) / 64 + 16));
      if (tid == 0)
        sh.b_low = sh.above + hist[sh.bin] >= static_cast<uint32_t>((5 * p.k) / 64 + 16) ? sh.bin : 0u;
    }
    cluster_sync();  // (2) rank 0 has merged the histograms and chosen the boundary
    b_low = rank == 0 ? sh.b_low : ld_peer_u32(mapa(smem_u32(&sh.b_low), 0));
  } else {
    find_threshold(sh, hist, 1 << 12, static_cast<uint32_t>((5 * p.k) / 64 + 16));
    b_low = sh.above + hist[sh.bin] >= static_cast<uint32_t>((5 * p.k) / 64 + 16) ? sh.bin : 0u;
  }
  __syncthreads();
  for (int i = tid; i < TK_BINS; i += TK_THREADS) hist[i] = 0;
  __syncthreads();
  // the candidate test as a compare on the raw bits when the boundary is non-negative
  const uint32_t t_low = b_low << (kKeyBits - 12);
  const bool fast = t_low >= (1u << (kKeyBits - 1));
  const int32_t a_fast = static_cast<int32_t>((t_low - (1u << (kKeyBits - 1))) << (32 - kKeyBits));
  // TK_UNROLL 16-byte loads per thread in flight, then the vectors in turn
  for (int v0 = v_lo + tid; v0 < v_hi; v0 += TK_UNROLL * TK_THREADS) {
    uint4 ws[TK_UNROLL];
#pragma unroll
    for (int j = 0; j < TK_UNROLL; ++j) {
      const int v = v0 + j * TK_THREADS;
      if (v < v_hi) ws[j] = *reinterpret_cast<const uint4*>(rowp + static_cast<size_t>(v) * 16);
    }
#pragma unroll
    for (int j = 0; j < TK_UNROLL; ++j) {
      const int v = v0 + j * TK_THREADS;
      if (v >= v_hi) break;  // the lanes still going are a prefix of the warp
      const uint4 w = ws[j];
      uint32_t m_keep = keep_mask<kF32>(w, fast, a_fast, t_low);
      const unsigned mask = __activemask();
      if (!__any_sync(mask, m_keep != 0u)) continue;
      uint32_t slot = warp_reserve(&sh.n_cand, __popc(m_keep));
      while (m_keep) {
        const int e = __ffs(m_keep) - 1;
        m_keep &= m_keep - 1u;
        const uint32_t key = vec_key<kF32>(w, e);
        if (slot < TK_CAP) {
          cand0[slot] = static_cast<uint32_t>(v * kVec + e);
          ckey0[slot] = key;
        }
        ++slot;
        atomicAdd(&hist[key >> (kKeyBits - 12)], 1u);
      }
    }
  }
  if (own_tail) {
    for (int u = nvec * kVec + tid; u < len; u += TK_THREADS) {
      const uint32_t key = key_at<kF32>(rowp, u);
      const bool keep = (key >> (kKeyBits - 12)) >= b_low;
      const uint32_t slot = warp_append(&sh.n_cand, keep);
      if (keep) {
        if (slot < TK_CAP) {
          cand0[slot] = static_cast<uint32_t>(u);
          ckey0[slot] = key;
        }
        atomicAdd(&hist[key >> (kKeyBits - 12)], 1u);
      }
    }
  }
  __syncthreads();
  if (kPair) {
    cluster_sync();  // (3) both candidate passes are done
    if (rank == 0) {  // append the peer's candidates and add its exact histogram
      const uint32_t n0 = sh.n_cand;
      const uint32_t n1 = ld_peer_u32(mapa(smem_u32(&sh.n_cand), 1));
      if (n0 <= static_cast<uint32_t>(TK_CAP) && n0 + n1 <= static_cast<uint32_t>(TK_CAP)) {
        const uint32_t pc = mapa(smem_u32(cand0), 1);
        const uint32_t pk = mapa(smem_u32(ckey0), 1);
        for (uint32_t i = tid; i < n1; i += TK_THREADS) {
          cand0[n0 + i] = ld_peer_u32(pc + 4u * i);
          ckey0[n0 + i] = ld_peer_u32(pk + 4u * i);
        }
      }
      const uint32_t ph = mapa(smem_u32(hist), 1);
      for (int i = tid; i < TK_BINS; i += TK_THREADS) hist[i] += ld_peer_u32(ph + 4u * i);
      __syncthreads();
      if (tid == 0) sh.n_cand = n0 + n1;  // above TK_CAP: the whole-row method below
    }
    cluster_sync();  // (4) rank 0 is done with the peer's shared memory
    if (rank != 0) return;
  }
  int src = 0;  // -1: the whole row (filtered by prefix); 0 / 1: a candidate buffer
  if (sh.n_cand < static_cast<uint32_t>(p.k) || sh.n_cand > static_cast<uint32_t>(TK_CAP)) {
    // the exact method on the whole row: the 12-bit histogram of every element
    __syncthreads();
    for (int i = tid; i < TK_BINS; i += TK_THREADS) hist[i] = 0;
    __syncthreads();
    for (int v = tid; v < nvec; v += TK_THREADS) {
      const uint4 w = *reinterpret_cast<const uint4*>(rowp + static_cast<size_t>(v) * 16);
#pragma unroll
      for (int e = 0; e < kVec; ++e) atomicAdd(&hist[vec_key<kF32>(w, e) >> (kKeyBits - 12)], 1u);
    }
    for (int u = nvec * kVec + tid; u < len; u += TK_THREADS)
      atomicAdd(&hist[key_at<kF32>(rowp, u) >> (kKeyBits - 12)], 1u);
    src = -1;
  }
  __syncthreads();
  uint32_t need = static_cast<uint32_t>(p.k);
  uint32_t prefix = 0;  // key bits fixed by the levels before this one
  int consumed = 0;     // how many
  find_threshold(sh, hist, 1 << 12, need);
  for (int level = 0; level < levels<kF32>(); ++level) {
    const int bits = level_bits<kF32>(level);
    const int shift = kKeyBits - consumed - bits;
    const bool last = level == levels<kF32>() - 1;
    const int nbits = last ? 0 : level_bits<kF32>(level + 1);
    const uint32_t b = sh.bin;
    const uint32_t take = need - sh.above;  // of bin b, this many are selected
    const bool all_of_bin = take == hist[b];
    const uint32_t n_src = src < 0 ? 0u : sh.n_cand;
    __syncthreads();
    if (tid == 0) sh.n_cand = 0;
    if (!last && !all_of_bin)
      for (int i = tid; i < (1 << nbits); i += TK_THREADS) hist[i] = 0;
    __syncthreads();
    uint32_t* dst = src == 0 ? cand1 : cand0;
    const uint32_t dcap = src == 0 ? static_cast<uint32_t>(TK_CAP1) : static_cast<uint32_t>(TK_CAP);
    const uint32_t* srcb = src == 0 ? cand0 : cand1;
    // the first candidates carry their keys (the later buffers hold positions only)
    const bool src_keys = src == 0 && level == 0;
    // one element: emit it (larger bin, or bin b when all of it or, at the last level, a tie
    // within the count), or keep it as a candidate of the next level
    auto visit = [&](bool in, int u, uint32_t key) {
      const uint32_t d = (key >> shift) & ((1u << bits) - 1u);
      bool out = in && d > b;
      const bool eq = in && d == b;
      bool keep = false;
      if (last || all_of_bin) {
        bool tie_ok = eq;
        if (!all_of_bin) {  // every lane takes part in the count (it is a warp collective)
          const uint32_t t = warp_append(&sh.ties, eq);
          tie_ok = eq && t < take;
        }
        out = out || tie_ok;
      } else {
        keep = eq;
      }
      const uint32_t pos = warp_append(&sh.n_out, out);
      if (out) emit_at(p, sh, row, req, pos, u);
      if (!last && !all_of_bin) {
        const uint32_t slot = warp_append(&sh.n_cand, keep);
        if (keep) {
          if (slot < dcap) dst[slot] = static_cast<uint32_t>(u);
          else sh.overflow = 1u;
          atomicAdd(&hist[(key >> (shift - nbits)) & ((1u << nbits) - 1u)], 1u);
        }
      }
    };
    if (src < 0 && consumed == 0 && !last && !all_of_bin) {
      // level 0 over the whole row (the common case): per 16-byte vector each lane marks its
      // larger-bin and bin-b elements in two bit masks, and one warp scan per mask reserves
      // their output and candidate slots
      for (int v = tid; v < nvec; v += TK_THREADS) {
        const uint4 w = *reinterpret_cast<const uint4*>(rowp + static_cast<size_t>(v) * 16);
        uint32_t m_out = 0, m_keep = 0;
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          const uint32_t d = vec_key<kF32>(w, e) >> shift;
          m_out |= static_cast<uint32_t>(d > b) << e;
          m_keep |= static_cast<uint32_t>(d == b) << e;
        }
        const unsigned mask = __activemask();
        if (!__any_sync(mask, (m_out | m_keep) != 0u)) continue;
        uint32_t pos = warp_reserve(&sh.n_out, __popc(m_out));
        uint32_t slot = warp_reserve(&sh.n_cand, __popc(m_keep));
        while (m_out) {
          const int e = __ffs(m_out) - 1;
          m_out &= m_out - 1u;
          emit_at(p, sh, row, req, pos++, v * kVec + e);
        }
        while (m_keep) {
          const int e = __ffs(m_keep) - 1;
          m_keep &= m_keep - 1u;
          if (slot < dcap) dst[slot] = static_cast<uint32_t>(v * kVec + e);
          else sh.overflow = 1u;
          ++slot;
          atomicAdd(&hist[(vec_key<kF32>(w, e) >> (shift - nbits)) & ((1u << nbits) - 1u)], 1u);
        }
      }
      for (int u = nvec * kVec + tid; u < len; u += TK_THREADS) visit(true, u, key_at<kF32>(rowp, u));
    } else if (src < 0) {
      // the whole row: elements whose fixed key bits match the prefix
      const int pshift = kKeyBits - consumed;
      for (int v = tid; v < nvec; v += TK_THREADS) {
        const uint4 w = *reinterpret_cast<const uint4*>(rowp + static_cast<size_t>(v) * 16);
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
          const uint32_t key = vec_key<kF32>(w, e);
          visit(consumed == 0 || (key >> pshift) == prefix, v * kVec + e, key);
        }
      }
      for (int u = nvec * kVec + tid; u < len; u += TK_THREADS) {
        const uint32_t key = key_at<kF32>(rowp, u);
        visit(consumed == 0 || (key >> pshift) == prefix, u, key);
      }
    } else {
      for (uint32_t i = tid; i < n_src; i += TK_THREADS) {
        const int u = static_cast<int>(srcb[i]);
        visit(true, u, src_keys ? ckey0[i] : key_at<kF32>(rowp, u));
      }
    }
    __syncthreads();
    if (last || all_of_bin) break;
    prefix = (prefix << bits) | b;
    consumed += bits;
    need = take;
    src = sh.overflow ? -1 : (src == 0 ? 1 : 0);  // after an overflow the levels re-read the row
    find_threshold(sh, hist, 1 << nbits, need);
  }
  if (tid == 0 && sh.bad && p.status != nullptr) atomicOr(p.status, SMLA_DEV_TOPK_TABLE);
}

template <bool kF32>
__global__ void __launch_bounds__(TK_THREADS, SMLA_TOPK_MINB) topk_kernel(const TopkParams p) {
  extern __shared__ uint32_t tk_smem[];
  __shared__ TopkShared sh;
  topk_row<kF32, false>(p, sh, tk_smem, blockIdx.x, 0);
}

// Two CTAs per row (cluster of two): small batches, where one CTA per row leaves SMs idle.
template <bool kF32>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TK_THREADS, 1)
    topk_pair_kernel(const TopkParams p) {
  extern __shared__ uint32_t tk_smem[];
  __shared__ TopkShared sh;
  topk_row<kF32, true>(p, sh, tk_smem, blockIdx.x >> 1, cluster_ctarank());
}

}  // namespace

cudaError_t launch_topk(const void* scores, bool fp32, const int32_t* valid_len,
                        const int32_t* table, int32_t* out, uint32_t* status, int n_tok, int s_q,
                        int k, int ld, int max_pages, cudaStream_t stream) {
  TopkParams p{scores, valid_len, table, out, status, n_tok, s_q, k, ld, max_pages};
  const size_t smem = (TK_BINS + 2 * TK_CAP + TK_CAP1) * sizeof(uint32_t);
  // fp32 rows run on a CTA pair when the SMs outnumber the rows twice over (measured at 64
  // rows of 32768: 20.3 -> 18.8 us; bf16 rows, half the bytes, lose more to the pair's
  // barriers and merges than they gain: 14.7 -> 16.6 us, so they keep one CTA)
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const bool pair = fp32 && 2 * static_cast<int64_t>(n_tok) <= sms;
  void (*kernel)(TopkParams) = pair ? (fp32 ? topk_pair_kernel<true> : topk_pair_kernel<false>)
                                    : (fp32 ? topk_kernel<true> : topk_kernel<false>);
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kernel<<<(pair ? 2 : 1) * n_tok, TK_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
