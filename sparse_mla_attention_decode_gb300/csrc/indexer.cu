// Lightning-indexer scores over a paged FP8 key cache: the scores the top-k selects from
// ("FlashMLA 与 DSA：内核、流水线和正确性边界", sections 4.1 and 5.3; "sparse-attention co-design",
// section 5, steps one to four):
//     I[t, s] = k_scale[s] * sum_{j < 64} w[t, j] * max(q8[t, j] . k8[s], 0)
// with e4m3 q8 [64 heads x 128] per query token and one shared e4m3 key k8 [128] per cached
// token, pages of 64 tokens laid out as 64 x 128 codes followed by their 64 fp32 scales.
//
// The product runs candidate-major on the tensor cores: A = a tile of 128 cached tokens
// (K-major, 128-byte swizzle: one 128-byte row per token), B = the e4m3 Q of up to four query
// tokens of one request (64 G rows), D = [128 tokens x 64 G] fp32 in tensor memory, four
// kind::f8f6f4 MMAs of K = 32 per tile.  A TMEM lane is one cached token, so the ReLU, the
// head weights and the 64-head sum stay inside one thread (no transpose, no cross-thread
// reduction), and the [tokens x heads] products never leave the SM.
//
// Work item = (query group of G <= 4 tokens of one request, chunk of up to 16 key tiles); the
// CTAs walk the items with a grid stride.  Warps 0-7: epilogue, two warpgroups (thread = TMEM
// lane = token; the even and the odd query tokens of the group); warp 8: TMA producer (Q once
// per item into one of two buffers, two page boxes per key tile, six stages); warp 9: MMA issuer (two TMEM
// accumulators of 256 columns).  Every wait is bounded (a second), after
// which the CTA raises SMLA_DEV_TIMEOUT and its roles leave.
#include <cstdint>

#include "../../include/sparse_mla.h"
#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int IX_THREADS = 320;  // warps 0-7 epilogue, 8 TMA producer, 9 MMA issuer
constexpr int IX_STAGES = 6;
constexpr int IX_TILE = 128;          // cached tokens per key tile (two pages)
constexpr int IX_CHUNK = 16;          // key tiles per work item
constexpr int IX_PAGE_BYTES = 8448;   // 64 x 128 codes + 64 x 4 scale bytes
constexpr int IX_STAGE_BYTES = IX_TILE * 128;
constexpr int IX_Q_BYTES = 256 * 128;
constexpr int IX_OFF_Q = IX_STAGES * IX_STAGE_BYTES;
constexpr int IX_OFF_BARS = IX_OFF_Q + 2 * IX_Q_BYTES;  // two Q buffers (items alternate)
enum IxBar {
  IB_K_FULL = 0,                          // [stages] expect-tx + the tile's bytes
  IB_K_EMPTY = IB_K_FULL + IX_STAGES,     // [stages] commit after the tile's MMAs
  IB_D_FULL = IB_K_EMPTY + IX_STAGES,     // [2] commit after the tile's MMAs
  IB_D_EMPTY = IB_D_FULL + 2,             // [2] 256 epilogue threads
  IB_Q_FULL = IB_D_EMPTY + 2,             // [2] expect-tx + Q's bytes
  IB_Q_FREE = IB_Q_FULL + 2,              // [2] commit after an item's last MMAs
  IB_DRAIN = IB_Q_FREE + 2,
  IB_COUNT
};
// [8 warps][256] head weights, 128-byte aligned (read as float4)
constexpr int IX_OFF_W = (IX_OFF_BARS + IB_COUNT * 8 + 127) & ~127;
static_assert(IX_OFF_W % 16 == 0, "float4 weight reads");
constexpr int IX_OFF_MISC = IX_OFF_W + 8 * 256 * 4;
// + TMEM slot, abort flag, alignment slack; at least 116 KB so that one CTA holds an SM (each
// CTA allocates all 512 tensor-memory columns)
constexpr int IX_SMEM_USED = IX_OFF_MISC + 32 + 1024;
constexpr int IX_SMEM = IX_SMEM_USED > 116 * 1024 ? IX_SMEM_USED : 116 * 1024;
constexpr uint64_t kIxWaitNs = 1000000000ull;

struct IndexerParams {
  CUtensorMap k_map;  // cache codes as (128 bytes, 64 rows, pages), box 128 x 64 x 1
  CUtensorMap q_map;  // q8 as (128 bytes, n_tok * 64 rows), box 128 x 64 G
  const float* w;
  const int32_t* table;
  const int32_t* valid_len;
  const uint8_t* cache;
  float* out;
  uint32_t* status;
  int n_tok, s_q, max_pages, ld, G, groups_per_req, n_groups, chunks, n_items;
  int64_t num_pages;
};

struct IxCtx {
  uint32_t sbase;
  volatile uint32_t* abort_flag;
  uint32_t* status;
  __device__ uint32_t bar(int i) const { return sbase + IX_OFF_BARS + 8u * i; }
  __device__ bool wait(int b, uint32_t parity) const {
    const uint32_t a = bar(b);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t deadline = globaltimer_ns() + kIxWaitNs;
    for (uint32_t i = 0;; ++i) {
      if (mbar_try_wait(a, parity)) return true;
      if ((i & 7u) == 7u) {
        if (*abort_flag) return false;
        if (globaltimer_ns() > deadline) {
          *abort_flag = 1u;
          if (status != nullptr) atomicOr(status, SMLA_DEV_TIMEOUT);
          return false;
        }
      }
    }
  }
  __device__ bool wait_warp(int b, uint32_t parity) const {
    return __all_sync(0xffffffffu, wait(b, parity));
  }
};

// The work item's query group and key-tile range (the same on every role).
struct IxItem {
  int req, t0, gs, tile0, tile1;  // tokens t0 .. t0 + gs - 1 of request req; tiles [tile0, tile1)
  int maxlen;
};
__device__ __forceinline__ IxItem item_of(const IndexerParams& p, int item) {
  IxItem it;
  const int g = item / p.chunks, c = item % p.chunks;
  it.req = g / p.groups_per_req;
  const int sg = g % p.groups_per_req;
  it.t0 = it.req * p.s_q + sg * p.G;
  it.gs = min(p.G, p.s_q - sg * p.G);
  int m = 0;
  for (int q = 0; q < it.gs; ++q) {
    int n = p.valid_len[it.t0 + q];
    n = n < 0 ? 0 : (n > p.ld ? p.ld : n);
    m = max(m, n);
  }
  it.maxlen = min(m, p.max_pages * 64);  // positions past the page table do not exist
  const int tiles = (m + IX_TILE - 1) / IX_TILE;
  it.tile0 = min(c * IX_CHUNK, tiles);
  it.tile1 = min(it.tile0 + IX_CHUNK, tiles);
  return it;
}

__device__ void ix_producer(const IndexerParams& p, const IxCtx& c) {
  uint32_t gt = 0, n = 0;
  for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
    const IxItem it = item_of(p, item);
    if (it.tile0 >= it.tile1) continue;
    const uint32_t qb = n & 1;  // the item two back used this Q buffer: its MMAs are done
    if (n >= 2 && !c.wait(IB_Q_FREE + qb, ((n >> 1) - 1) & 1)) return;
    mbar_arrive_expect_tx(c.bar(IB_Q_FULL + qb), static_cast<uint32_t>(p.G) * 64 * 128);
    tma_load_2d(c.sbase + IX_OFF_Q + qb * IX_Q_BYTES, &p.q_map, 0, it.t0 * 64, c.bar(IB_Q_FULL + qb));
    const int pages = (it.maxlen + 63) / 64;
    const int32_t* row = p.table + static_cast<size_t>(it.req) * p.max_pages;
    for (int tile = it.tile0; tile < it.tile1; ++tile, ++gt) {
      const uint32_t st = gt % IX_STAGES;
      if (gt >= IX_STAGES && !c.wait(IB_K_EMPTY + st, ((gt / IX_STAGES) - 1) & 1)) return;
      const int pa = row[2 * tile];
      const int pb = (2 * tile + 1 < pages) ? row[2 * tile + 1] : pa;  // past the end: ignored rows
      const uint32_t dst = c.sbase + st * IX_STAGE_BYTES;
      mbar_arrive_expect_tx(c.bar(IB_K_FULL + st), IX_STAGE_BYTES);
      tma_load_3d(dst, &p.k_map, 0, 0, pa, c.bar(IB_K_FULL + st));
      tma_load_3d(dst + IX_STAGE_BYTES / 2, &p.k_map, 0, 0, pb, c.bar(IB_K_FULL + st));
    }
    ++n;
  }
}

__device__ void ix_mma(const IndexerParams& p, const IxCtx& c, uint32_t tbase) {
  const uint32_t idesc = umma_idesc_f16(128, 64 * p.G, 0);  // e4m3 x e4m3 -> f32, K-major
  uint32_t gt = 0, n = 0;
  for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
    const IxItem it = item_of(p, item);
    if (it.tile0 >= it.tile1) continue;
    const uint32_t qb = n & 1;
    if (!c.wait(IB_Q_FULL + qb, (n >> 1) & 1)) return;
    const uint64_t bdesc = umma_desc(c.sbase + IX_OFF_Q + qb * IX_Q_BYTES, 16, 1024, 2);
    for (int tile = it.tile0; tile < it.tile1; ++tile, ++gt) {
      const uint32_t st = gt % IX_STAGES, db = gt & 1;
      if (!c.wait(IB_K_FULL + st, (gt / IX_STAGES) & 1)) return;
      if (gt >= 2 && !c.wait(IB_D_EMPTY + db, ((gt >> 1) - 1) & 1)) return;
      tc_fence_after();
      const uint64_t adesc = umma_desc(c.sbase + st * IX_STAGE_BYTES, 16, 1024, 2);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // 32 codes = 32 bytes of each row per MMA
        mma_ss_f8(tbase + db * 256, adesc + (kk * 32 >> 4), bdesc + (kk * 32 >> 4), idesc, kk > 0);
      mma_commit(c.bar(IB_K_EMPTY + st));
      mma_commit(c.bar(IB_D_FULL + db));
    }
    mma_commit(c.bar(IB_Q_FREE + qb));
    ++n;
  }
}

// Epilogue warpgroup `grp` (0: warps 0-3, 1: warps 4-7; thread i = TMEM lane = cached token)
// takes the group's query tokens q with q % 2 == grp.  Each warp stages the item's head
// weights in its own shared-memory slice (no barrier beyond the warp) and reads them four at a
// time; a token's 64 accumulator columns are loaded before one wait.
__device__ void ix_epilogue(const IndexerParams& p, const IxCtx& c, uint32_t tbase, int i,
                            int grp, float* wsm) {
  const uint32_t lane_base = static_cast<uint32_t>((i >> 5) * 32) << 16;
  const int lane = i & 31;
  uint32_t gt = 0;
  for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
    const IxItem it = item_of(p, item);
    if (it.tile0 >= it.tile1) continue;
    const int32_t* row = p.table + static_cast<size_t>(it.req) * p.max_pages;
    __syncwarp();
    for (int k = lane; k < it.gs * 64; k += 32) wsm[k] = __ldg(p.w + static_cast<size_t>(it.t0) * 64 + k);
    __syncwarp();
    // the key scale of this thread's token, one tile ahead (the page-table entry and then the
    // scale are two dependent loads; they overlap the wait for the tile's products)
    auto scale_of = [&](int tile) -> float {
      const int s = tile * IX_TILE + i;
      if (tile >= it.tile1 || s >= it.maxlen) return 0.f;
      const int page = row[s / 64];
      if (page < 0 || page >= p.num_pages) return 0.f;  // outside the cache: zero codes, score 0
      return __ldg(reinterpret_cast<const float*>(p.cache + static_cast<size_t>(page) * IX_PAGE_BYTES +
                                                  8192) + (s & 63));
    };
    float next_scale = scale_of(it.tile0);
    for (int tile = it.tile0; tile < it.tile1; ++tile, ++gt) {
      const uint32_t db = gt & 1;
      const float scale = next_scale;
      next_scale = scale_of(tile + 1);
      if (!c.wait_warp(IB_D_FULL + db, (gt >> 1) & 1)) return;
      tc_fence_after();
      const int s = tile * IX_TILE + i;  // this thread's cached token
      for (int q = grp; q < it.gs; q += 2) {
        uint32_t r[64];
#pragma unroll
        for (int jc = 0; jc < 4; ++jc) tmem_ld16(tbase + lane_base + db * 256 + q * 64 + jc * 16, r + 16 * jc);
        tmem_wait_ld();
        const float4* wq = reinterpret_cast<const float4*>(wsm + q * 64);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float4 wv = wq[e];
          acc[0] = fmaf(wv.x, fmaxf(__uint_as_float(r[4 * e]), 0.f), acc[0]);
          acc[1] = fmaf(wv.y, fmaxf(__uint_as_float(r[4 * e + 1]), 0.f), acc[1]);
          acc[2] = fmaf(wv.z, fmaxf(__uint_as_float(r[4 * e + 2]), 0.f), acc[2]);
          acc[3] = fmaf(wv.w, fmaxf(__uint_as_float(r[4 * e + 3]), 0.f), acc[3]);
        }
        int n = p.valid_len[it.t0 + q];
        n = n > p.ld ? p.ld : n;
        n = n > p.max_pages * 64 ? p.max_pages * 64 : n;
        if (s < n)
          p.out[static_cast<size_t>(it.t0 + q) * p.ld + s] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) * scale;
      }
      tc_fence_before();
      mbar_arrive(c.bar(IB_D_EMPTY + db));
    }
  }
}

__global__ void __launch_bounds__(IX_THREADS, 1) indexer_kernel(const __grid_constant__ IndexerParams p) {
  extern __shared__ uint8_t ix_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ix_smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  IxCtx c;
  c.sbase = smem_u32(sm);
  c.abort_flag = reinterpret_cast<volatile uint32_t*>(sm + IX_OFF_MISC + 16);
  c.status = p.status;
  if (threadIdx.x == 0) {
    *c.abort_flag = 0u;
    for (int b = 0; b < IX_STAGES; ++b) {
      mbar_init(c.bar(IB_K_FULL + b), 1);
      mbar_init(c.bar(IB_K_EMPTY + b), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.bar(IB_D_FULL + b), 1);
      mbar_init(c.bar(IB_D_EMPTY + b), 256);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.bar(IB_Q_FULL + b), 1);
      mbar_init(c.bar(IB_Q_FREE + b), 1);
    }
    mbar_init(c.bar(IB_DRAIN), 1);
    fence_mbar_init_cluster();
  }
  if (warp == 9) {
    tmem_alloc(c.sbase + IX_OFF_MISC, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(sm + IX_OFF_MISC);
  if (warp < 8) {
    ix_epilogue(p, c, tbase, threadIdx.x & 127, warp >> 2,
                reinterpret_cast<float*>(sm + IX_OFF_W) + warp * 256);
  } else if (warp == 8) {
    if (lane == 0) ix_producer(p, c);
  } else if (lane == 0) {
    ix_mma(p, c, tbase);
    mma_commit(c.bar(IB_DRAIN));  // every issued MMA has finished before TMEM is freed
    const uint64_t deadline = globaltimer_ns() + kIxWaitNs;
    while (!mbar_try_wait(c.bar(IB_DRAIN), 0) && globaltimer_ns() < deadline) {
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tbase, 512);
}

}  // namespace

cudaError_t launch_indexer(const IndexerLaunch& L, cudaStream_t stream) {
  IndexerParams p;
  p.k_map = L.k_map;
  p.q_map = L.q_map;
  p.w = L.w;
  p.table = L.table;
  p.valid_len = L.valid_len;
  p.cache = L.cache;
  p.out = L.out;
  p.status = L.status;
  p.n_tok = L.n_tok;
  p.s_q = L.s_q;
  p.max_pages = L.max_pages;
  p.ld = L.ld;
  p.num_pages = L.num_pages;
  p.G = L.s_q < 4 ? L.s_q : 4;
  p.groups_per_req = (L.s_q + p.G - 1) / p.G;
  p.n_groups = (L.n_tok / L.s_q) * p.groups_per_req;
  const int max_tiles = (L.ld + IX_TILE - 1) / IX_TILE;
  p.chunks = (max_tiles + IX_CHUNK - 1) / IX_CHUNK;
  if (p.chunks < 1) p.chunks = 1;
  p.n_items = p.n_groups * p.chunks;
  cudaError_t e = cudaFuncSetAttribute(indexer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, IX_SMEM);
  if (e != cudaSuccess) return e;
  int grid = p.n_items < L.num_sms ? p.n_items : L.num_sms;
  if (grid < 1) grid = 1;
  indexer_kernel<<<grid, IX_THREADS, IX_SMEM, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
