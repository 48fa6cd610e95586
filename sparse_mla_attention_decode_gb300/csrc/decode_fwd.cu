// Sparse MLA decode pass for sm_103a: gather + FP8 dequant + tcgen05 QK^T + online softmax +
// tcgen05 PV, split-KV aware ("FlashMLA Sparse Decode 完整计算过程详解", steps 5-15;
// "FlashMLA 与 DSA：内核、流水线和正确性边界", sections 3.1-3.5 and 4.3).
//
// One partition of the split-KV plan runs on a cluster of two CTAs (one per SM) that split the
// work by role, because the fp32 output accumulator of one query token (128 heads x 512 dims)
// fills the whole tensor memory of one SM:
//
//   S-CTA (cluster rank 0): gathers the selected 656-byte rows, dequantizes them to an fp16
//     key tile [64 slots x 576 dims], computes S = Q K^T with tcgen05 MMAs (M = 128 heads,
//     N = 64 slots, K = 576; Q resident in tensor memory), runs the masked base-2 online
//     softmax (one thread per head) and streams each block's P (fp16, the precision the PV
//     MMA consumes) plus per-head rescale factors to its peer with one bulk copy into the
//     peer's shared memory.  It writes the log-sum-exp.
//   O-CTA (cluster rank 1): gathers the NoPE bytes + scales of the same rows, dequantizes them
//     to an fp16 value tile [64 slots x 512 dims], rescales its O rows when the S-CTA moved a
//     row's running max, accumulates O += P V with tcgen05 MMAs (M = 128, N = 2 x 256, K = 64;
//     O in all 512 tensor-memory columns) and writes the normalised output.
//
// Data moves between the two SMs in one direction only (17 KB per 64-slot block), and P is
// exactly the fp16 matrix the MMA uses, so the split adds no rounding.  Gathers are warp loads
// (16 bytes per thread, one block of look-ahead in registers); a prefetch warp pulls every row
// of a request range into L2 when the range starts.
//
// Keys and values are dequantized as 256 * K (folded back into the score scale and into the
// final 1/L) so that small fp32 scales stay in the fp16 normal range.  Invalid slots become NaN
// key rows (their scores are NaN and are masked) and zero value rows.
//
// Every wait is bounded: when one runs out the CTA records SMLA_DEV_TIMEOUT (and where) in the
// status words, every role leaves its loop, issued MMAs are drained and tensor memory is freed.
#include <cmath>

#include "../../include/sparse_mla.h"
#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int BT = 64;                  // top-k slots per block
constexpr int CHUNK = BT * 128;         // one [64 rows x 64 dims] fp16 tile, 128-byte swizzle
constexpr int KT_STAGE = 9 * CHUNK;     // S-CTA key tile: 8 NoPE chunks + 1 RoPE chunk
constexpr int VT_STAGE = 8 * CHUNK;     // O-CTA value tile: 8 NoPE chunks
constexpr int P_BYTES = 128 * BT * 2;   // P tile [128 heads x 64 slots] fp16, 128-byte swizzle
constexpr int MSG_ALPHA = P_BYTES;      // 128 x fp32 rescale factors
constexpr int MSG_INVL = P_BYTES + 512; // 128 x fp32 1 / (256 L) (last block of a range)
constexpr int MSG_BYTES = P_BYTES + 1024;
constexpr int MSG_STRIDE = 18432;       // 1024-aligned message slots
constexpr int NSTAGE = 2;               // tile / message double buffering
constexpr int NSBUF = 3;                // score buffers in tensor memory (S-CTA)

constexpr int OFF_TILE = 0;                                  // KT[2] or VT[2]
constexpr int OFF_MSG = NSTAGE * KT_STAGE;                   // S: staging, O: receive
constexpr int OFF_MISC = OFF_MSG + NSTAGE * MSG_STRIDE;
static_assert(OFF_MSG % 1024 == 0 && OFF_MISC % 1024 == 0, "alignment");

enum Bar {
  // S-CTA
  B_KT_FULL = 0,                    // [2] 256 dequant threads
  B_KT_EMPTY = B_KT_FULL + 2,       // [2] commit after QK
  B_S_FULL = B_KT_EMPTY + 2,        // [3] commit after QK
  B_S_EMPTY = B_S_FULL + NSBUF,     // [3] 128 softmax threads
  B_Q_FULL = B_S_EMPTY + NSBUF,     // 128 softmax threads
  B_MSG_FREE = B_Q_FULL + 1,        // [2] remote arrival from the O-CTA after PV consumed it
  // O-CTA
  B_VT_FULL = B_MSG_FREE + 2,       // [2] 256 dequant threads
  B_VT_EMPTY = B_VT_FULL + 2,       // [2] commit after PV
  B_MSG_FULL = B_VT_EMPTY + 2,      // [2] 1 local expect-tx arrival + the bulk copy's bytes
  B_CORR = B_MSG_FULL + 2,          // [2] 128 correction threads
  B_PV_DONE = B_CORR + 2,           // [2] commit after PV
  B_O_FULL = B_PV_DONE + 2,         // commit after the last PV of a range
  B_O_EMPTY = B_O_FULL + 1,         // 128 epilogue threads
  B_DRAIN = B_O_EMPTY + 1,          // MMA drain on the way out
  B_STAGED = B_DRAIN + 1,           // [2] 128 softmax threads wrote a message slot (S-CTA)
  NUM_BARS
};
constexpr int OFF_BARS = OFF_MISC;
constexpr int OFF_TMEM_SLOT = OFF_BARS + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 16;
constexpr int OFF_STARTED = OFF_ABORT + 16;  // request ranges whose Q is staged (S-CTA)
constexpr int SMEM_BYTES = OFF_STARTED + 16 + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// warps: 0-3 softmax (S) / correction + epilogue (O); 4-11 gather + dequant; 12 MMA;
// 13 L2 prefetch (S) / message relay (O)
constexpr int NTHREADS = 448;
constexpr uint32_t TM_Q = 0, TM_S = 288;  // S-CTA columns; the O-CTA uses all 512 for O
constexpr uint32_t IDESC_QK = umma_idesc_f16(128, BT, 0);
constexpr uint32_t IDESC_PV = umma_idesc_f16(128, 256, 1);
constexpr uint64_t kWaitNs = 1000000000ull;  // a wait gives up after one second
constexpr uint32_t F16_NAN2 = 0x7E007E00u;

struct Ctx {
  uint32_t sbase;
  volatile uint32_t* abort_flag;
  uint32_t* status;  // [0] SMLA_DEV_* bits, [1] where the first timed-out wait was
  uint32_t role;
  __device__ uint32_t bar(int i) const { return sbase + OFF_BARS + 8u * i; }
  // Records the first wait that ran out: 0x80000000 | rank << 24 | role << 16 | barrier << 8 |
  // parity, so a stuck pipeline can be diagnosed from the status words.
  __device__ void fail(int b, uint32_t parity) const {
    *abort_flag = 1u;
    atomicOr(status, SMLA_DEV_TIMEOUT);
    atomicCAS(status + 1, 0u, 0x80000000u | (cluster_ctarank() << 24) | (role << 16) |
                                  (static_cast<uint32_t>(b) << 8) | parity);
  }
  // Bounded wait on an mbarrier phase of this CTA; false when the wait ran out or another
  // role already gave up.
  __device__ bool wait(int b, uint32_t parity, bool cluster_scope = false) const {
    const uint32_t a = bar(b);
    uint64_t deadline = 0;
    for (uint32_t i = 0;; ++i) {
      if (cluster_scope ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity)) return true;
      if ((i & 127u) == 127u) {
        if (*abort_flag) return false;
        const uint64_t now = globaltimer_ns();
        if (deadline == 0) {
          deadline = now + kWaitNs;
        } else if (now > deadline) {
          fail(b, parity);
          return false;
        }
      }
    }
  }
  // Same, with one outcome for the whole warp (for roles that issue warp-collective
  // tensor-memory instructions: no lane may leave while the others continue).
  __device__ bool wait_warp(int b, uint32_t parity, bool cluster_scope = false) const {
    const bool ok = wait(b, parity, cluster_scope);
    return __all_sync(0xffffffffu, ok);
  }
  // Bounded wait that ignores the abort flag (used to drain issued MMAs).
  __device__ void drain(int b, uint32_t parity) const {
    const uint32_t a = bar(b);
    const uint64_t deadline = globaltimer_ns() + kWaitNs;
    while (!mbar_try_wait(a, parity)) {
      if (globaltimer_ns() > deadline) {
        atomicOr(status, SMLA_DEV_TIMEOUT);
        return;
      }
    }
  }
};

// The work of one partition: requests [begin_req, end_req], each with a block range, walked
// block by block in the same order by every role of both CTAs.
struct Plan {
  int begin_req, end_req, begin_block, end_block, begin_split, nb;
  __device__ int first_block(int req) const { return req == begin_req ? begin_block : 0; }
  __device__ int last_block(int req) const { return req == end_req ? end_block : nb; }
};
struct Cursor {
  int req, blk;  // current block; req > end_req once past the end
  __device__ void start(const Plan& pl) {
    req = pl.begin_req;
    blk = pl.first_block(req);
  }
  __device__ bool done(const Plan& pl) const { return req > pl.end_req; }
  __device__ void next(const Plan& pl) {
    if (++blk >= pl.last_block(req)) {
      ++req;
      if (req <= pl.end_req) blk = pl.first_block(req);
    }
  }
};

// ---------------------------------------------------------------------------------------
// Gather + dequant (warps 4-11 of both CTAs).  Thread t owns row t % 64 of every block and
// the 128-dim scale group q = t / 64 of its NoPE part (plus RoPE dims [16 q, 16 q + 16) on the
// S-CTA).  The loads of block g + 1 are issued before block g is converted.
struct RowData {
  uint4 nope[8];
  uint4 rope[2];
  uint4 scales;
  bool valid;
};

__device__ __forceinline__ int32_t load_index(const DecodeParams& p, int s, int req, int blk,
                                              int row) {
  const int slot = blk * BT + row;
  if (slot >= p.topk) return -1;
  return __ldg(p.indices + (static_cast<size_t>(req) * p.s_q + s) * p.topk + slot);
}

template <bool kScores>
__device__ __forceinline__ void load_row(const DecodeParams& p, int32_t idx, int q, RowData& d) {
  d.valid = idx >= 0 && idx < p.num_rows;
  if (!d.valid) return;
  const uint4* row = reinterpret_cast<const uint4*>(p.kv + static_cast<size_t>(idx) * kRowBytes);
#pragma unroll
  for (int k = 0; k < 8; ++k) d.nope[k] = __ldg(row + q * 8 + k);
  d.scales = __ldg(row + 32);
  if (kScores) {
    d.rope[0] = __ldg(row + 33 + q * 2);
    d.rope[1] = __ldg(row + 34 + q * 2);
  }
}

template <bool kScores>
__device__ __forceinline__ void store_row(uint32_t tile, int row, int q, const RowData& d,
                                          uint32_t& bad) {
  const uint32_t c0 = tile + (2 * q) * CHUNK;  // chunks 2q, 2q + 1 hold dims [128 q, 128 q + 128)
  if (d.valid) {
    const uint32_t sel =
        q == 0 ? d.scales.x : q == 1 ? d.scales.y : q == 2 ? d.scales.z : d.scales.w;
    const float scale = __uint_as_float(sel) * 256.f;
    bad |= !(scale >= 6.103515625e-05f && scale <= 65504.f);
    const uint32_t s2 = pack_f16x2(scale, scale);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t w[4] = {d.nope[k].x, d.nope[k].y, d.nope[k].z, d.nope[k].w};
      uint32_t o[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[2 * e] = hmul2(cvt_e4m3x2_f16x2(static_cast<uint16_t>(w[e] & 0xFFFFu)), s2);
        o[2 * e + 1] = hmul2(cvt_e4m3x2_f16x2(static_cast<uint16_t>(w[e] >> 16)), s2);
      }
      // 16 codes = dims [128 q + 16 k, + 16): chunk 2q + k / 4, 8-dim chunks 2 (k % 4) and + 1
      const uint32_t ch = c0 + (k >> 2) * CHUNK;
      st_shared_v4(ch + sw128_chunk(row, 2 * (k & 3)), o[0], o[1], o[2], o[3]);
      st_shared_v4(ch + sw128_chunk(row, 2 * (k & 3) + 1), o[4], o[5], o[6], o[7]);
    }
    if (kScores) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint32_t w[4] = {d.rope[k].x, d.rope[k].y, d.rope[k].z, d.rope[k].w};
        uint32_t o[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          o[e] = pack_f16x2(__uint_as_float(w[e] << 16) * 256.f,
                            __uint_as_float(w[e] & 0xFFFF0000u) * 256.f);
        st_shared_v4(tile + 8 * CHUNK + sw128_chunk(row, 2 * q + k), o[0], o[1], o[2], o[3]);
      }
    }
  } else {
    // invalid slot: NaN key (its score becomes NaN and is masked) or zero value
    const uint32_t f = kScores ? F16_NAN2 : 0u;
#pragma unroll
    for (int k = 0; k < 16; ++k)
      st_shared_v4(c0 + (k >> 3) * CHUNK + sw128_chunk(row, k & 7), f, f, f, f);
    if (kScores) {
#pragma unroll
      for (int k = 0; k < 2; ++k)
        st_shared_v4(tile + 8 * CHUNK + sw128_chunk(row, 2 * q + k), f, f, f, f);
    }
  }
}

template <bool kScores>
__device__ void role_dequant(const DecodeParams& p, const Ctx& c, const Plan& pl, int s, int t) {
  const int row = t & 63, q = t >> 6;
  const int bfull = kScores ? B_KT_FULL : B_VT_FULL;
  const int bempty = kScores ? B_KT_EMPTY : B_VT_EMPTY;
  const int stage_bytes = kScores ? KT_STAGE : VT_STAGE;
  uint32_t bad = 0;
  Cursor cur, ahead;
  cur.start(pl);
  ahead = cur;
  RowData d[2];
  load_row<kScores>(p, load_index(p, s, cur.req, cur.blk, row), q, d[0]);
  ahead.next(pl);
  int32_t idx_next = ahead.done(pl) ? -1 : load_index(p, s, ahead.req, ahead.blk, row);
  uint32_t g = 0;
#pragma unroll 1
  while (!cur.done(pl)) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {  // unrolled by two so the row buffers stay in registers
      if (cur.done(pl)) break;
      // look-ahead: issue the loads of the next block before converting this one
      if (!ahead.done(pl)) {
        load_row<kScores>(p, idx_next, q, d[u ^ 1]);
        ahead.next(pl);
        idx_next = ahead.done(pl) ? -1 : load_index(p, s, ahead.req, ahead.blk, row);
      }
      const uint32_t st = g & 1;
      if (g >= NSTAGE && !c.wait(bempty + st, ((g >> 1) - 1) & 1)) goto out;
      store_row<kScores>(c.sbase + OFF_TILE + st * stage_bytes, row, q, d[u], bad);
      fence_proxy_async_smem();
      mbar_arrive(c.bar(bfull + st));
      cur.next(pl);
      ++g;
    }
  }
out:
  if (bad) atomicOr(c.status, SMLA_DEV_SCALE_RANGE);
}

// ---------------------------------------------------------------------------------------
// S-CTA MMA warp (one lane): S[buf] = Q K^T for every block (36 MMAs of K = 16).
__device__ void role_mma_scores(const Ctx& c, const Plan& pl, uint32_t tbase) {
  uint32_t g = 0, item = 0;
  for (int req = pl.begin_req; req <= pl.end_req; ++req, ++item) {
    if (!c.wait(B_Q_FULL, item & 1)) return;
    for (int blk = pl.first_block(req); blk < pl.last_block(req); ++blk, ++g) {
      const uint32_t st = g & 1, sb = g % NSBUF;
      if (!c.wait(B_KT_FULL + st, (g >> 1) & 1)) return;
      if (g >= NSBUF && !c.wait(B_S_EMPTY + sb, ((g / NSBUF) - 1) & 1)) return;
      tc_fence_after();
      const uint32_t kt = c.sbase + OFF_TILE + st * KT_STAGE;
      const uint32_t d = tbase + TM_S + sb * BT;
#pragma unroll
      for (int kk = 0; kk < 36; ++kk)
        mma_ts(d, tbase + TM_Q + kk * 8,
               umma_desc(kt + (kk >> 2) * CHUNK + (kk & 3) * 32, 16, 1024, 2), IDESC_QK, kk > 0);
      mma_commit(c.bar(B_S_FULL + sb));
      mma_commit(c.bar(B_KT_EMPTY + st));
    }
  }
}

// O-CTA MMA warp (one lane): O += P V for every block (4 K-steps x 2 N-halves).
__device__ void role_mma_values(const Ctx& c, const Plan& pl, uint32_t tbase) {
  uint32_t g = 0, item = 0;
  for (int req = pl.begin_req; req <= pl.end_req; ++req, ++item) {
    const int b0 = pl.first_block(req), b1 = pl.last_block(req);
    for (int blk = b0; blk < b1; ++blk, ++g) {
      const uint32_t st = g & 1, par = (g >> 1) & 1;
      const bool first = blk == b0;
      if (!c.wait(B_VT_FULL + st, par)) return;
      if (!c.wait(B_MSG_FULL + st, par, true)) return;
      if (!c.wait(B_CORR + st, par)) return;
      if (first && item >= 1 && !c.wait(B_O_EMPTY, (item - 1) & 1)) return;
      tc_fence_after();
      const uint32_t pm = c.sbase + OFF_MSG + st * MSG_STRIDE;
      const uint32_t vt = c.sbase + OFF_TILE + st * VT_STAGE;
#pragma unroll
      for (int kk = 0; kk < BT / 16; ++kk) {
        const uint64_t a = umma_desc(pm + kk * 32, 16, 1024, 2);
#pragma unroll
        for (int nh = 0; nh < 2; ++nh)
          mma_ss(tbase + nh * 256, a, umma_desc(vt + nh * 4 * CHUNK + kk * 2048, CHUNK, 1024, 2),
                 IDESC_PV, !(first && kk == 0));
      }
      mma_commit(c.bar(B_VT_EMPTY + st));
      mma_commit(c.bar(B_PV_DONE + st));
      if (blk == b1 - 1) mma_commit(c.bar(B_O_FULL));
    }
  }
}

// ---------------------------------------------------------------------------------------
// S-CTA: Q of one query token into tensor memory (fp16, two dims per column), thread i = head i.
__device__ void stage_q(const DecodeParams& p, const Ctx& c, uint32_t tq, int tok, int i,
                        uint32_t& bad) {
  const bool live = i < p.h_q;
  const uint4* src = reinterpret_cast<const uint4*>(
      p.q + (static_cast<size_t>(tok) * p.h_q + (live ? i : 0)) * kDQk);
#pragma unroll 1
  for (int cc = 0; cc < 18; ++cc) {  // 18 x 32 dims
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = live ? __ldg(src + cc * 4 + k) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t in[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t r = pack_f16x2(__uint_as_float(in[e] << 16),
                                      __uint_as_float(in[e] & 0xFFFF0000u));
        bad |= ((r & 0x7C00u) == 0x7C00u) | ((r & 0x7C000000u) == 0x7C000000u);
        w[4 * k + e] = r;
      }
    }
    tmem_st16(tq + cc * 16, w);
  }
  tmem_wait_st();
  tc_fence_before();
  mbar_arrive(c.bar(B_Q_FULL));
}

// S-CTA softmax warpgroup: thread i owns head row i (tensor-memory lane i).
__device__ void role_softmax(const DecodeParams& p, const Ctx& c, const Plan& pl, int s,
                             uint32_t tbase, int i) {
  const uint32_t lane_base = static_cast<uint32_t>((i >> 5) * 32) << 16;
  const uint32_t tq = tbase + lane_base + TM_Q;
  const uint32_t ts = tbase + lane_base + TM_S;
  const uint32_t peer_msg = mapa(c.sbase + OFF_MSG, 1);
  const uint32_t peer_full = mapa(c.bar(B_MSG_FULL), 1);
  const bool live = i < p.h_q;
  uint32_t qbad = 0;
  uint32_t g = 0;
  volatile uint32_t* started = reinterpret_cast<volatile uint32_t*>(
      __cvta_shared_to_generic(c.sbase + OFF_STARTED));
  stage_q(p, c, tq, pl.begin_req * p.s_q + s, i, qbad);
  for (int req = pl.begin_req; req <= pl.end_req; ++req) {
    if (i == 0) *started = static_cast<uint32_t>(req - pl.begin_req + 1);
    const int b0 = pl.first_block(req), b1 = pl.last_block(req);
    float m = -INFINITY;  // running max (base-2 units) used as the exponent reference
    float l = 0.f;        // running exp-sum against m
    for (int blk = b0; blk < b1; ++blk, ++g) {
      const uint32_t sb = g % NSBUF, st = g & 1;
      if (!c.wait_warp(B_S_FULL + sb, (g / NSBUF) & 1)) goto out;
      tc_fence_after();
      uint32_t sr[BT];
#pragma unroll
      for (int k = 0; k < BT / 16; ++k) tmem_ld16(ts + sb * BT + k * 16, sr + k * 16);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(c.bar(B_S_EMPTY + sb));
      // mask (NaN = invalid slot) and scale to base-2 units
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < BT; ++k) {
        const float x = __uint_as_float(sr[k]);
        const float t = x == x ? x * p.score_scale_log2 : -INFINITY;
        sr[k] = __float_as_uint(t);
        mx = fmaxf(mx, t);
      }
      // lazy rescale: the reference only moves when a block's max passes it by more than 8
      // (p then stays <= 256, which fp16 holds with full precision)
      float alpha = 1.f;
      if (m == -INFINITY) {
        m = mx;
      } else if (mx > m + 8.f) {
        alpha = ex2(m - mx);
        m = mx;
      }
      const float mref = m == -INFINITY ? 0.f : m;
      // the message slot is free again once the O-CTA's PV that read it has finished
      if (g >= NSTAGE && !c.wait_warp(B_MSG_FREE + st, ((g >> 1) - 1) & 1, true)) goto out;
      const uint32_t msg = c.sbase + OFF_MSG + st * MSG_STRIDE;
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ex2(__uint_as_float(sr[8 * k + 2 * e]) - mref);
          const float p1 = ex2(__uint_as_float(sr[8 * k + 2 * e + 1]) - mref);
          sum += p0 + p1;
          w[e] = pack_f16x2(p0, p1);
        }
        st_shared_v4(msg + sw128_chunk(i, k), w[0], w[1], w[2], w[3]);
      }
      l = l * alpha + sum;
      st_shared_f32(msg + MSG_ALPHA + 4 * i, alpha);
      if (blk == b1 - 1) {
        // last block of the range: the O-CTA's normalisation, and the lse from here
        st_shared_f32(msg + MSG_INVL + 4 * i, l == 0.f ? 0.f : 1.f / (l * 256.f));
        if (live) {
          const int first_slot = p.nsplits[req];
          const bool no_split = p.nsplits[req + 1] - first_slot == 1;
          if (no_split) {
            p.lse[(static_cast<size_t>(req) * p.h_q + i) * p.s_q + s] =
                l == 0.f ? INFINITY : (log2f(l) + m) * 0.69314718055994530942f;
          } else {
            const int split = req == pl.begin_req ? pl.begin_split : first_slot;
            p.lse_accum[(static_cast<size_t>(split) * p.s_q + s) * p.h_q + i] =
                l == 0.f ? -INFINITY : log2f(l) + m;
          }
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(c.bar(B_STAGED + st));
      if (i == 0) {  // all 128 rows are in the slot: ship it to the O-CTA
        if (!c.wait(B_STAGED + st, (g >> 1) & 1)) goto out;
        bulk_s2s_cluster(peer_msg + st * MSG_STRIDE, msg, MSG_BYTES, peer_full + st * 8);
      }
    }
    // every QK^T of this range has completed: stage the next query token's Q
    if (req < pl.end_req) stage_q(p, c, tq, (req + 1) * p.s_q + s, i, qbad);
  }
out:
  if (qbad) atomicOr(c.status, SMLA_DEV_Q_RANGE);
}

// S-CTA prefetch warp: when a request range starts, pull every selected row into L2.
__device__ void role_prefetch(const DecodeParams& p, const Ctx& c, const Plan& pl, int s,
                              int lane) {
  volatile uint32_t* started = reinterpret_cast<volatile uint32_t*>(
      __cvta_shared_to_generic(c.sbase + OFF_STARTED));
  uint32_t item = 0;
  for (int req = pl.begin_req; req <= pl.end_req; ++req, ++item) {
    // run one request range ahead of the softmax (prefetches are hints: give up quietly)
    const uint64_t deadline = globaltimer_ns() + kWaitNs;
    while (*started < item && !*c.abort_flag && globaltimer_ns() < deadline) {
    }
    if (*c.abort_flag) return;
    const int32_t* idx = p.indices + (static_cast<size_t>(req) * p.s_q + s) * p.topk;
    const int lo = pl.first_block(req) * BT;
    const int hi = min(pl.last_block(req) * BT, p.topk);
    for (int j = lo + lane; j < hi; j += 32) {
      const int32_t id = __ldg(idx + j);
      if (id < 0 || id >= p.num_rows) continue;
      const uint8_t* row = p.kv + static_cast<size_t>(id) * kRowBytes;
#pragma unroll
      for (int k = 0; k < 6; ++k) prefetch_l2(row + k * 128);
      prefetch_l2(row + kRowBytes - 1);
    }
  }
}

// ---------------------------------------------------------------------------------------
// O-CTA correction + epilogue warpgroup: thread i owns O row i.
__device__ void role_values_epilogue(const DecodeParams& p, const Ctx& c, const Plan& pl, int s,
                                     uint32_t tbase, int i) {
  const uint32_t to = tbase + (static_cast<uint32_t>((i >> 5) * 32) << 16);
  const bool live = i < p.h_q;
  uint32_t g = 0, item = 0;
  for (int req = pl.begin_req; req <= pl.end_req; ++req, ++item) {
    const int b0 = pl.first_block(req), b1 = pl.last_block(req);
    float invl = 0.f;
    for (int blk = b0; blk < b1; ++blk, ++g) {
      const uint32_t st = g & 1;
      if (i == 0) mbar_arrive_expect_tx(c.bar(B_MSG_FULL + st), MSG_BYTES);
      if (!c.wait_warp(B_MSG_FULL + st, (g >> 1) & 1, true)) return;
      const uint32_t msg = c.sbase + OFF_MSG + st * MSG_STRIDE;
      const float alpha = ld_shared_f32(msg + MSG_ALPHA + 4 * i);
      if (blk == b1 - 1) invl = ld_shared_f32(msg + MSG_INVL + 4 * i);
      if (blk > b0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // the S-CTA moved this row's reference: rescale O once the previous PV has landed
        if (!c.wait_warp(B_PV_DONE + ((g - 1) & 1), ((g - 1) >> 1) & 1)) return;
        tc_fence_after();
#pragma unroll 1
        for (int k = 0; k < 512; k += 16) {
          uint32_t o[16];
          tmem_ld16(to + k, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st16(to + k, o);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(c.bar(B_CORR + st));
    }
    // epilogue: O / L of this request range
    if (!c.wait_warp(B_O_FULL, item & 1)) return;
    tc_fence_after();
    const int first_slot = p.nsplits[req];
    const bool no_split = p.nsplits[req + 1] - first_slot == 1;
    const int split = req == pl.begin_req ? pl.begin_split : first_slot;
    const int tok = req * p.s_q + s;
    if (no_split) {
      __nv_bfloat16* dst = p.out + (static_cast<size_t>(tok) * p.h_q + (live ? i : 0)) * kDV;
#pragma unroll 1
      for (int k = 0; k < 512; k += 32) {
        uint32_t o[32];
        tmem_ld16(to + k, o);
        tmem_ld16(to + k + 16, o + 16);
        tmem_wait_ld();
        if (live) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + k);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * e + 0]) * invl, __uint_as_float(o[8 * e + 1]) * invl);
            v.y = pack_bf16x2(__uint_as_float(o[8 * e + 2]) * invl, __uint_as_float(o[8 * e + 3]) * invl);
            v.z = pack_bf16x2(__uint_as_float(o[8 * e + 4]) * invl, __uint_as_float(o[8 * e + 5]) * invl);
            v.w = pack_bf16x2(__uint_as_float(o[8 * e + 6]) * invl, __uint_as_float(o[8 * e + 7]) * invl);
            d4[e] = v;
          }
        }
      }
    } else {
      float* dst = p.o_accum + ((static_cast<size_t>(split) * p.s_q + s) * p.h_q + (live ? i : 0)) * kDV;
#pragma unroll 1
      for (int k = 0; k < 512; k += 32) {
        uint32_t o[32];
        tmem_ld16(to + k, o);
        tmem_ld16(to + k + 16, o + 16);
        tmem_wait_ld();
        if (live) {
          float4* d4 = reinterpret_cast<float4*>(dst + k);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            d4[e] = make_float4(__uint_as_float(o[4 * e]) * invl, __uint_as_float(o[4 * e + 1]) * invl,
                                __uint_as_float(o[4 * e + 2]) * invl, __uint_as_float(o[4 * e + 3]) * invl);
        }
      }
    }
    tc_fence_before();
    mbar_arrive(c.bar(B_O_EMPTY));
  }
}

// O-CTA relay lane: once a block's PV has finished reading its message slot, hand the slot
// back to the S-CTA.
__device__ void role_relay(const Ctx& c, const Plan& pl) {
  const uint32_t peer_free = mapa(c.bar(B_MSG_FREE), 0);
  uint32_t g = 0;
  for (int req = pl.begin_req; req <= pl.end_req; ++req)
    for (int blk = pl.first_block(req); blk < pl.last_block(req); ++blk, ++g) {
      const uint32_t st = g & 1;
      if (!c.wait(B_PV_DONE + st, (g >> 1) & 1)) return;
      mbar_arrive_remote(peer_free + st * 8);
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    decode_kernel(const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool scores = rank == 0;
  const int part = blockIdx.x >> 1, s = blockIdx.y;
  Ctx c;
  c.sbase = smem_u32(sm);
  c.abort_flag = reinterpret_cast<volatile uint32_t*>(sm + OFF_ABORT);
  c.status = p.status;
  c.role = 0;
  const int32_t* m = p.meta + part * kMetaInts;
  Plan pl;
  pl.begin_req = m[0];
  pl.end_req = m[1];
  pl.begin_block = m[2];
  pl.end_block = m[3];
  pl.begin_split = m[4];
  pl.nb = (p.topk + BT - 1) / BT;
  const bool active = pl.begin_req < p.b;

  if (threadIdx.x == 0) {
    *c.abort_flag = 0u;
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.bar(B_KT_FULL + b), 256);
      mbar_init(c.bar(B_KT_EMPTY + b), 1);
      mbar_init(c.bar(B_MSG_FREE + b), 1);
      mbar_init(c.bar(B_VT_FULL + b), 256);
      mbar_init(c.bar(B_VT_EMPTY + b), 1);
      mbar_init(c.bar(B_MSG_FULL + b), 1);
      mbar_init(c.bar(B_CORR + b), 128);
      mbar_init(c.bar(B_PV_DONE + b), 1);
      mbar_init(c.bar(B_STAGED + b), 128);
    }
    *reinterpret_cast<volatile uint32_t*>(sm + OFF_STARTED) = 0u;
    for (int b = 0; b < NSBUF; ++b) {
      mbar_init(c.bar(B_S_FULL + b), 1);
      mbar_init(c.bar(B_S_EMPTY + b), 128);
    }
    mbar_init(c.bar(B_Q_FULL), 128);
    mbar_init(c.bar(B_O_FULL), 1);
    mbar_init(c.bar(B_O_EMPTY), 128);
    mbar_init(c.bar(B_DRAIN), 1);
    fence_mbar_init_cluster();
  }
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_TMEM_SLOT);
  if (warp == 12 && active) {
    tmem_alloc(c.sbase + OFF_TMEM_SLOT, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote access
  const uint32_t tbase = active ? *tslot : 0u;

  if (active) {
    c.role = (scores ? 0u : 8u) + (warp < 4 ? 1u : warp < 12 ? 2u : warp == 12 ? 3u : 4u);
    if (warp < 4) {
      if (scores) role_softmax(p, c, pl, s, tbase, threadIdx.x);
      else role_values_epilogue(p, c, pl, s, tbase, threadIdx.x);
    } else if (warp < 12) {
      if (scores) role_dequant<true>(p, c, pl, s, threadIdx.x - 128);
      else role_dequant<false>(p, c, pl, s, threadIdx.x - 128);
    } else if (warp == 12) {
      if (lane == 0) {
        if (scores) role_mma_scores(c, pl, tbase);
        else role_mma_values(c, pl, tbase);
        mma_commit(c.bar(B_DRAIN));  // every issued MMA has finished before TMEM is freed
        c.drain(B_DRAIN, 0);
      }
    } else {
      if (scores) role_prefetch(p, c, pl, s, lane);
      else if (lane == 0) role_relay(c, pl);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 12 && active) tmem_dealloc(tbase, 512);
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int parts, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(2 * parts), static_cast<unsigned>(p.s_q), 1);
  decode_kernel<<<grid, NTHREADS, SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
