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
// Work item = (query group of G <= 4 tokens of one request, chunk of 16 key tiles); each CTA
// takes an equal contiguous range of the key tiles of all groups laid end to end, so
// consecutive items share their group's Q.  The first 4 NG warps: epilogue, NG warpgroups
// (thread = TMEM lane = token; NG = 2 at one query token per group, 3 above) taking the (tile,
// query token) units in turn; then the TMA producer (Q once per run of items of one group into
// one of two buffers; per key tile the two pages' codes and their key scales, as many stages
// as fit beside Q) and the MMA issuer (TMEM accumulators of 64 G columns: eight at G = 1,
// four at G = 2, two above).  A stage is
// released by the epilogue once it has read the tile's key scales (the MMAs are done by then),
// and the page ids, lengths and head weights of the next item load while the current one
// runs, so no global load sits on a role's critical path.  Every wait is bounded (a second),
// after which the CTA raises SMLA_DEV_TIMEOUT and its roles leave.
#include <cstdint>

#include "../../include/sparse_mla.h"
#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

// Warps [0, 4 NG): epilogue (NG warpgroups), 4 NG: TMA producer, 4 NG + 1: MMA issuer.  NG = 2
// at one query token per group, 3 when a group has several (the epilogue then sets the pace,
// and a third warpgroup hides more of its latency).
template <int NG>
struct IxWarps {
  static constexpr int kEpi = 4 * NG, kProducer = 4 * NG, kMma = 4 * NG + 1;
  static constexpr int kThreads = 32 * (4 * NG + 2);
};
constexpr int IX_MAX_STAGES = 12;
constexpr int IX_TILE = 128;          // cached tokens per key tile (two pages)
constexpr int IX_PAGE_BYTES = 8448;   // 64 x 128 codes + 64 x 4 scale bytes
constexpr int IX_STAGE_BYTES = IX_TILE * 128;
constexpr int IX_SC_BYTES = IX_TILE * 4;
enum IxBar {
  IB_K_FULL = 0,                            // [stages] expect-tx + the tile's bytes
  IB_K_EMPTY = IB_K_FULL + IX_MAX_STAGES,   // [stages] the 8 epilogue warps, scales read
  IB_D_FULL = IB_K_EMPTY + IX_MAX_STAGES,   // [8] commit after the tile's MMAs
  IB_D_EMPTY = IB_D_FULL + 8,               // [8] 256 epilogue threads
  IB_Q_FULL = IB_D_EMPTY + 8,               // [2] expect-tx + Q's bytes
  IB_Q_FREE = IB_Q_FULL + 2,                // [2] commit after an item's last MMAs
  IB_DRAIN = IB_Q_FREE + 2,
  IB_NEVER,                                 // nothing arrives (the failure-path test)
  IB_COUNT
};
// Shared memory (base 1024-aligned): barriers, [epilogue warps][256] head weights (read as
// float4), TMEM slot + abort flag, then the stages (codes, 16 KB each, 1024-aligned for the
// 128-byte swizzle), their key scales, and two Q buffers of 64 G x 128 bytes.  The number of
// stages is what fits beside the Q buffers: 12 at G = 1, 10, 9, 8 at G = 4.
constexpr int IX_OFF_BARS = 0;
constexpr int IX_OFF_W = 512;
static_assert(IB_COUNT * 8 <= IX_OFF_W, "barriers fit below the weights");
template <int NG>
struct IxLayout {
  static constexpr int kOffMisc = IX_OFF_W + IxWarps<NG>::kEpi * 256 * 4;
  static constexpr int kOffStages = (kOffMisc + 32 + 1023) / 1024 * 1024;
};
constexpr int IX_SMEM_MAX = 227 * 1024;
constexpr uint64_t kIxWaitNs = 1000000000ull;

struct IndexerParams {
  CUtensorMap k_map;  // cache codes as (128 bytes, 64 rows, pages), box 128 x 64 x 1
  CUtensorMap q_map;  // q8 as (128 bytes, n_tok * 64 rows), box 128 x 64 G
  CUtensorMap s_map;  // key scales as (256 bytes, pages), box 256 x 1, no swizzle
  const float* w;
  const int32_t* table;
  const int32_t* valid_len;
  const uint8_t* cache;
  float* out;
  uint32_t* status;
  int n_tok, s_q, max_pages, ld, G, groups_per_req, n_groups, chunks, n_items;
  int chunk;      // key tiles per work item
  int max_tiles;  // key tiles of a full row (ld / 128, rounded up)
  int nshift;  // 1 << nshift TMEM accumulators of 512 >> nshift columns
  int stages;  // key-tile stages
  uint32_t off_stages, off_sc, off_q, q_bytes;  // shared-memory offsets of the stages, their
                                                // scales and the Q buffers
  int test_stall;                   // the MMA issuer waits on IB_NEVER (bounded) and leaves
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

// A work item's query group and key-tile chunk, from its index alone (no load).
struct IxHead {
  int g, req, t0, gs, c;  // group g = tokens t0 .. t0 + gs - 1 of request req; key-tile chunk c
};
__device__ __forceinline__ IxHead head_of(const IndexerParams& p, int item) {
  IxHead h;
  const int g = item / p.chunks;
  h.g = g;
  h.c = item % p.chunks;
  h.req = g / p.groups_per_req;
  const int sg = g % p.groups_per_req;
  h.t0 = h.req * p.s_q + sg * p.G;
  h.gs = min(p.G, p.s_q - sg * p.G);
  return h;
}
// The valid lengths of the group's tokens (0 past the group or for an item that does not
// exist).  Every role loads them one item ahead, so the loads overlap the current item.
__device__ __forceinline__ void lens_load(const IndexerParams& p, const IxHead& h, bool live, int (&n)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) n[q] = (live && q < h.gs) ? p.valid_len[h.t0 + q] : 0;
}
// The CTA's share of the work: an equal contiguous range [v0, v1) of the key tiles of all
// query groups laid end to end (group g owns tiles [g * max_tiles, (g + 1) * max_tiles), split
// into items of `chunk` tiles), so the SMs get the same number of tiles to within one, and
// consecutive items share their group's Q (loaded once per run of items of one group).  The
// first and the last item of a share may be cut.
struct IxRange {
  int64_t v0, v1;  // tiles [v0, v1)
  int i0, i1;      // items [i0, i1)
};
__device__ __forceinline__ IxRange cta_range(const IndexerParams& p) {
  const int64_t total = static_cast<int64_t>(p.n_groups) * p.max_tiles;
  const int64_t per = total / gridDim.x, rem = total % gridDim.x;
  const int64_t b = blockIdx.x;
  IxRange r;
  r.v0 = b * per + (b < rem ? b : rem);
  r.v1 = r.v0 + per + (b < rem ? 1 : 0);
  auto item_at = [&](int64_t v) {  // the item holding end-to-end tile v
    const int64_t g = v / p.max_tiles;
    return static_cast<int>(g * p.chunks + (v - g * p.max_tiles) / p.chunk);
  };
  r.i0 = item_at(r.v0);
  r.i1 = r.v1 > r.v0 ? item_at(r.v1 - 1) + 1 : r.i0;
  return r;
}
// The work item's key-tile range within the CTA's share (the same on every role).
struct IxItem {
  int req, t0, gs, tile0, tile1;  // tiles [tile0, tile1)
  int base;                       // first tile of the item's chunk
  int maxlen;
};
__device__ __forceinline__ IxItem item_from(const IndexerParams& p, const IxHead& h, const int (&n)[4],
                                            int item, const IxRange& r) {
  IxItem it;
  it.req = h.req;
  it.t0 = h.t0;
  it.gs = h.gs;
  int m = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int v = n[q] < 0 ? 0 : (n[q] > p.ld ? p.ld : n[q]);
    m = max(m, v);
  }
  it.maxlen = min(m, p.max_pages * 64);  // positions past the page table do not exist
  const int tiles = (m + IX_TILE - 1) / IX_TILE;
  // the item's first tile end to end
  const int64_t v = static_cast<int64_t>(h.g) * p.max_tiles + static_cast<int64_t>(h.c) * p.chunk;
  const int jlo = static_cast<int>(r.v0 > v ? r.v0 - v : 0);
  const int jhi = static_cast<int>(r.v1 - v < p.chunk ? r.v1 - v : p.chunk);
  it.base = h.c * p.chunk;
  it.tile0 = min(it.base + jlo, tiles);
  it.tile1 = min(it.base + jhi, tiles);
  return it;
}

// The whole warp runs the loop: lane k holds page id k of the item's chunk (loaded one item
// ahead, one coalesced load per item); lane 0 waits and issues the copies.  If a wait runs out,
// lane 0 waits (bounded) for the copies it has issued to land before the warp leaves.
__device__ void ix_producer(const IndexerParams& p, const IxCtx& c, int lane) {
  auto ids_load = [&](const IxHead& h, bool live) -> int {
    const int k = 2 * h.c * p.chunk + lane;
    return (live && lane < 2 * p.chunk && k < p.max_pages)
               ? p.table[static_cast<size_t>(h.req) * p.max_pages + k] : -1;
  };
  uint32_t gt = 0, n = 0;  // key tiles and Q loads issued
  auto drain = [&]() {
    if (lane != 0) return;
    const uint64_t deadline = globaltimer_ns() + kIxWaitNs;
    const uint32_t S = static_cast<uint32_t>(p.stages);
    for (uint32_t k = 0; k < S && k < gt; ++k) {
      const uint32_t g = gt - 1 - k;  // the last tile issued into stage g % S
      while (!mbar_try_wait(c.bar(IB_K_FULL + g % S), (g / S) & 1) && globaltimer_ns() < deadline) {
      }
    }
    for (uint32_t k = 0; k < 2 && k < n; ++k) {
      const uint32_t g = n - 1 - k;
      while (!mbar_try_wait(c.bar(IB_Q_FULL + (g & 1)), (g >> 1) & 1) && globaltimer_ns() < deadline) {
      }
    }
  };
  uint32_t st = 0, ph = 0;  // stage of tile gt and (gt / stages) & 1
  const IxRange r = cta_range(p);
  const int i0 = r.i0, i1 = r.i1;
  int item = i0, cur_g = -1;  // cur_g: the group whose Q was loaded last
  IxHead h = head_of(p, item);
  int len[4];
  lens_load(p, h, item < i1, len);
  int ids = ids_load(h, item < i1);
  for (; item < i1; ++item) {
    const int nx = item + 1;
    const IxHead hn = head_of(p, nx);
    int len_n[4];
    lens_load(p, hn, nx < i1, len_n);
    const int ids_n = ids_load(hn, nx < i1);
    const IxItem it = item_from(p, h, len, item, r);
    if (it.tile0 < it.tile1) {
      const uint32_t qb = n & 1;  // the Q two loads back used this buffer: its MMAs are done
      int ok = 1;
      if (h.g != cur_g && lane == 0) {
        ok = (n < 2 || c.wait(IB_Q_FREE + qb, ((n >> 1) - 1) & 1)) ? 1 : 0;
        if (ok) {
          mbar_arrive_expect_tx(c.bar(IB_Q_FULL + qb), p.q_bytes);
          tma_load_2d(c.sbase + p.off_q + qb * p.q_bytes, &p.q_map, 0, it.t0 * 64, c.bar(IB_Q_FULL + qb));
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        drain();
        return;
      }
      if (h.g != cur_g) {
        ++n;
        cur_g = h.g;
      }
      const int pages = (it.maxlen + 63) / 64;
      for (int tile = it.tile0; tile < it.tile1; ++tile, ++gt) {
        const int j = 2 * (tile - it.base);
        const int pa = __shfl_sync(0xffffffffu, ids, j);
        const int pb_raw = __shfl_sync(0xffffffffu, ids, j + 1);
        const int pb = (2 * tile + 1 < pages) ? pb_raw : pa;  // past the end: ignored rows
        if (lane == 0) {
          ok = (gt < static_cast<uint32_t>(p.stages) || c.wait(IB_K_EMPTY + st, ph ^ 1u)) ? 1 : 0;
          if (ok) {
            const uint32_t dst = c.sbase + p.off_stages + st * IX_STAGE_BYTES;
            const uint32_t sdst = c.sbase + p.off_sc + st * IX_SC_BYTES;
            // a page id outside [0, num_pages) reads the fill value: zero codes and scales
            mbar_arrive_expect_tx(c.bar(IB_K_FULL + st), IX_STAGE_BYTES + IX_SC_BYTES);
            tma_load_3d(dst, &p.k_map, 0, 0, pa, c.bar(IB_K_FULL + st));
            tma_load_3d(dst + IX_STAGE_BYTES / 2, &p.k_map, 0, 0, pb, c.bar(IB_K_FULL + st));
            tma_load_2d(sdst, &p.s_map, 0, pa, c.bar(IB_K_FULL + st));
            tma_load_2d(sdst + 256, &p.s_map, 0, pb, c.bar(IB_K_FULL + st));
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          drain();
          return;
        }
        if (++st == static_cast<uint32_t>(p.stages)) {
          st = 0;
          ph ^= 1u;
        }
      }
    }
    h = hn;
    ids = ids_n;
#pragma unroll
    for (int q = 0; q < 4; ++q) len[q] = len_n[q];
  }
}

__device__ void ix_mma(const IndexerParams& p, const IxCtx& c, uint32_t tbase) {
  if (p.test_stall) {  // the failure-path test: a wait that runs out, before any MMA
    c.wait(IB_NEVER, 0);
    return;
  }
  const uint32_t idesc = umma_idesc_f16(128, 64 * p.G, 0);  // e4m3 x e4m3 -> f32, K-major
  const uint32_t nbuf = 1u << p.nshift, colw = 512u >> p.nshift;
  uint32_t gt = 0, n = 0, st = 0, ph = 0;  // n: Q loads consumed
  const IxRange r = cta_range(p);
  const int i0 = r.i0, i1 = r.i1;
  int len[4], cur_g = -1;
  uint64_t bdesc = 0;
  lens_load(p, head_of(p, i0), i0 < i1, len);
  for (int item = i0; item < i1; ++item) {
    const IxHead h = head_of(p, item);
    const int nx = item + 1;
    int len_n[4];
    lens_load(p, head_of(p, nx), nx < i1, len_n);
    const IxItem it = item_from(p, h, len, item, r);
#pragma unroll
    for (int q = 0; q < 4; ++q) len[q] = len_n[q];
    if (it.tile0 >= it.tile1) continue;
    if (h.g != cur_g) {
      // a new group: the previous Q is read by no later MMA (the commit covers every MMA
      // issued so far), and this group's Q is waited for
      if (n > 0) mma_commit(c.bar(IB_Q_FREE + ((n - 1) & 1)));
      const uint32_t qb = n & 1;
      if (!c.wait(IB_Q_FULL + qb, (n >> 1) & 1)) return;
      bdesc = umma_desc(c.sbase + p.off_q + qb * p.q_bytes, 16, 1024, 2);
      ++n;
      cur_g = h.g;
    }
    for (int tile = it.tile0; tile < it.tile1; ++tile, ++gt) {
      const uint32_t db = gt & (nbuf - 1);
      if (!c.wait(IB_K_FULL + st, ph)) return;
      if (gt >= nbuf && !c.wait(IB_D_EMPTY + db, ((gt >> p.nshift) - 1) & 1)) return;
      tc_fence_after();
      const uint64_t adesc = umma_desc(c.sbase + p.off_stages + st * IX_STAGE_BYTES, 16, 1024, 2);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)  // 32 codes = 32 bytes of each row per MMA
        mma_ss_f8(tbase + db * colw, adesc + (kk * 32 >> 4), bdesc + (kk * 32 >> 4), idesc, kk > 0);
      mma_commit(c.bar(IB_D_FULL + db));
      if (++st == static_cast<uint32_t>(p.stages)) {
        st = 0;
        ph ^= 1u;
      }
    }
  }
}

// Epilogue warpgroup `grp` of NG (warps 4 grp .. 4 grp + 3; thread i = TMEM lane = cached
// token) takes the units u = (tile - base) * gs + q of the item with u % NG == grp, so that
// every warpgroup works at every group size (tiles in turn for one query token).  Each warp
// stages the item's head weights in its own shared-memory slice (no barrier beyond the warp)
// and reads them four at a time; a token's 64 accumulator columns are loaded and weighed in
// two halves of 32.  The key scale comes from the stage (loaded with the codes); the warp
// releases the stage once it has read it.
template <int NG>
__device__ void ix_epilogue(const IndexerParams& p, const IxCtx& c, uint32_t tbase, int i,
                            int grp, float* wsm, const float* scales) {
  const uint32_t lane_base = static_cast<uint32_t>((i >> 5) * 32) << 16;
  const int lane = i & 31;
  const uint32_t nbuf = 1u << p.nshift, colw = 512u >> p.nshift;
  const int lim = p.ld < p.max_pages * 64 ? p.ld : p.max_pages * 64;
  // the item's head weights (lane k holds entries k, k + 32, ...) and lengths, one item ahead
  auto w_load = [&](const IxHead& h, bool live, float (&w)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = lane + 32 * j;
      w[j] = (live && k < h.gs * 64) ? __ldg(p.w + static_cast<size_t>(h.t0) * 64 + k) : 0.f;
    }
  };
  uint32_t gt = 0, st = 0, ph = 0;
  const IxRange r = cta_range(p);
  const int i0 = r.i0, i1 = r.i1;
  int len[4], cur_g = -1;
  float wr[8];
  {
    const IxHead h0 = head_of(p, i0);
    lens_load(p, h0, i0 < i1, len);
    w_load(h0, i0 < i1, wr);
  }
  for (int item = i0; item < i1; ++item) {
    const IxHead h = head_of(p, item);
    const int nx = item + 1;
    const IxHead hn = head_of(p, nx);
    int len_n[4];
    float wr_n[8];
    lens_load(p, hn, nx < i1, len_n);
    w_load(hn, nx < i1, wr_n);
    const IxItem it = item_from(p, h, len, item, r);
    // valid prefix of the group's query tokens
    const int nq0 = min(len[0], lim), nq1 = min(len[1], lim), nq2 = min(len[2], lim), nq3 = min(len[3], lim);
    if (it.tile0 < it.tile1 && h.g != cur_g) {
      cur_g = h.g;
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (lane + 32 * j < it.gs * 64) wsm[lane + 32 * j] = wr[j];
      __syncwarp();
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) len[q] = len_n[q];
#pragma unroll
    for (int j = 0; j < 8; ++j) wr[j] = wr_n[j];
    if (it.tile0 >= it.tile1) continue;
    for (int tile = it.tile0; tile < it.tile1; ++tile, ++gt) {
      const uint32_t db = gt & (nbuf - 1);
      if (!c.wait_warp(IB_D_FULL + db, (gt >> p.nshift) & 1)) return;
      // the tile's copies have landed (already complete: the MMAs that read them are done)
      if (!c.wait_warp(IB_K_FULL + st, ph)) return;
      tc_fence_after();
      const float scale = p.num_pages > 0 ? scales[st * IX_TILE + i] : 0.f;
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(IB_K_EMPTY + st));
      if (++st == static_cast<uint32_t>(p.stages)) {
        st = 0;
        ph ^= 1u;
      }
      const int s = tile * IX_TILE + i;  // this thread's cached token
      // this warpgroup's units of the tile: the query tokens q with ((tile - base) gs + q) %
      // NG == grp; a token's 64 columns are weighed in two halves of 32
      const int q_first = ((grp - ((tile - it.base) * it.gs) % NG) + NG) % NG;
#pragma unroll
      for (int k = 0; k < (4 + NG - 1) / NG; ++k) {
        const int q = q_first + NG * k;
        if (q >= it.gs) break;
        const int nq = q == 0 ? nq0 : (q == 1 ? nq1 : (q == 2 ? nq2 : nq3));
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t r[32];
          tmem_ld16(tbase + lane_base + db * colw + q * 64 + hf * 32, r);
          tmem_ld16(tbase + lane_base + db * colw + q * 64 + hf * 32 + 16, r + 16);
          tmem_wait_ld();
          const float4* wq = reinterpret_cast<const float4*>(wsm + q * 64) + hf * 8;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 wv = wq[e];
            acc[0] = fmaf(wv.x, fmaxf(__uint_as_float(r[4 * e]), 0.f), acc[0]);
            acc[1] = fmaf(wv.y, fmaxf(__uint_as_float(r[4 * e + 1]), 0.f), acc[1]);
            acc[2] = fmaf(wv.z, fmaxf(__uint_as_float(r[4 * e + 2]), 0.f), acc[2]);
            acc[3] = fmaf(wv.w, fmaxf(__uint_as_float(r[4 * e + 3]), 0.f), acc[3]);
          }
        }
        if (s < nq)
          p.out[static_cast<size_t>(it.t0 + q) * p.ld + s] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) * scale;
      }
      tc_fence_before();
      mbar_arrive(c.bar(IB_D_EMPTY + db));
    }
  }
}

template <int NG>
__global__ void __launch_bounds__(IxWarps<NG>::kThreads, 1)
    indexer_kernel(const __grid_constant__ IndexerParams p) {
  using W = IxWarps<NG>;
  constexpr int kOffMisc = IxLayout<NG>::kOffMisc;
  extern __shared__ uint8_t ix_smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ix_smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  IxCtx c;
  c.sbase = smem_u32(sm);
  c.abort_flag = reinterpret_cast<volatile uint32_t*>(sm + kOffMisc + 16);
  c.status = p.status;
  if (threadIdx.x == 0) {
    *c.abort_flag = 0u;
    for (int b = 0; b < p.stages; ++b) {
      mbar_init(c.bar(IB_K_FULL + b), 1);
      mbar_init(c.bar(IB_K_EMPTY + b), W::kEpi);
    }
    for (int b = 0; b < 8; ++b) {
      mbar_init(c.bar(IB_D_FULL + b), 1);
      mbar_init(c.bar(IB_D_EMPTY + b), 128 * NG);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.bar(IB_Q_FULL + b), 1);
      mbar_init(c.bar(IB_Q_FREE + b), 1);
    }
    mbar_init(c.bar(IB_DRAIN), 1);
    mbar_init(c.bar(IB_NEVER), 1);
    fence_mbar_init_cluster();
  }
  if (warp == W::kMma) {
    tmem_alloc(c.sbase + kOffMisc, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(sm + kOffMisc);
  if (warp < W::kEpi) {
    ix_epilogue<NG>(p, c, tbase, threadIdx.x & 127, warp >> 2,
                reinterpret_cast<float*>(sm + IX_OFF_W) + warp * 256,
                reinterpret_cast<const float*>(sm + p.off_sc));
  } else if (warp == W::kProducer) {
    ix_producer(p, c, lane);
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
  if (warp == W::kMma) tmem_dealloc(tbase, 512);
}

}  // namespace

cudaError_t launch_indexer(const IndexerLaunch& L, cudaStream_t stream) {
  IndexerParams p;
  p.k_map = L.k_map;
  p.q_map = L.q_map;
  p.s_map = L.s_map;
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
  p.test_stall = L.test_stall;
  p.G = L.s_q < 4 ? L.s_q : 4;
  p.groups_per_req = (L.s_q + p.G - 1) / p.G;
  p.n_groups = (L.n_tok / L.s_q) * p.groups_per_req;
  p.nshift = p.G == 1 ? 3 : (p.G == 2 ? 2 : 1);
  const int max_tiles = (L.ld + IX_TILE - 1) / IX_TILE;
  // 16 key tiles per item: the page ids, lengths and weights of the next item are loaded while
  // the current one runs, and 16 tiles hide a cold miss; the SMs are balanced per tile
  p.chunk = 16;
  p.max_tiles = max_tiles > 0 ? max_tiles : 1;
  p.chunks = (max_tiles + p.chunk - 1) / p.chunk;
  if (p.chunks < 1) p.chunks = 1;
  p.n_items = p.n_groups * p.chunks;
  // stages: as many as fit beside the two Q buffers (at least 116 KB in all, so that one CTA
  // holds an SM: each CTA allocates all 512 tensor-memory columns)
  p.q_bytes = static_cast<uint32_t>(p.G) * 64 * 128;
  const bool three = p.G > 1;  // three epilogue warpgroups when a group has several tokens
  p.off_stages = static_cast<uint32_t>(three ? IxLayout<3>::kOffStages : IxLayout<2>::kOffStages);
  uint32_t smem = 0;
  for (p.stages = IX_MAX_STAGES; p.stages > 2; --p.stages) {
    p.off_sc = p.off_stages + p.stages * IX_STAGE_BYTES;
    p.off_q = (p.off_sc + p.stages * IX_SC_BYTES + 1023u) & ~1023u;
    smem = p.off_q + 2 * p.q_bytes + 1024;  // + slack to align the base
    if (smem <= static_cast<uint32_t>(IX_SMEM_MAX)) break;
  }
  if (smem < 116u * 1024) smem = 116u * 1024;
  void (*kernel)(IndexerParams) = three ? indexer_kernel<3> : indexer_kernel<2>;
  const int threads = three ? IxWarps<3>::kThreads : IxWarps<2>::kThreads;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t total_tiles = static_cast<int64_t>(p.n_groups) * p.max_tiles;
  int grid = total_tiles < L.num_sms ? static_cast<int>(total_tiles) : L.num_sms;
  if (grid < 1) grid = 1;
  kernel<<<grid, threads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
