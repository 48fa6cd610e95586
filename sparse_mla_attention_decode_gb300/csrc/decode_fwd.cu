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
// exactly the fp16 matrix the MMA uses, so the split adds no rounding.  Rows are gathered with
// cp.async straight into shared memory, one block of rows ahead of the conversion.
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
constexpr int NSTAGE = 2;               // tile double buffering
constexpr int NMSG = 2;                 // message slots (S-CTA staging = O-CTA receive)
constexpr int NSBUF = 3;                // score buffers in tensor memory (S-CTA)
constexpr int RAW_BYTES = 8 * 8 * 656;  // gathered-row rings of the 8 dequant warps (S-CTA size)

constexpr int OFF_TILE = 0;                                  // KT[2] or VT[2]
constexpr int OFF_MSG = NSTAGE * KT_STAGE;                   // S: staging, O: receive
constexpr int OFF_RAW = OFF_MSG + NMSG * MSG_STRIDE;         // gathered rows
constexpr int OFF_MISC = OFF_RAW + RAW_BYTES;
static_assert(OFF_MSG % 1024 == 0 && OFF_RAW % 1024 == 0 && OFF_MISC % 16 == 0, "alignment");

enum Bar {
  // S-CTA
  B_KT_FULL = 0,                    // [2] 256 dequant threads
  B_KT_EMPTY = B_KT_FULL + 2,       // [2] commit after QK
  B_S_FULL = B_KT_EMPTY + 2,        // [3] commit after QK
  B_S_EMPTY = B_S_FULL + NSBUF,     // [3] 128 softmax threads
  B_Q_FULL = B_S_EMPTY + NSBUF,     // 128 softmax threads
  B_MSG_FREE = B_Q_FULL + 1,        // [3] remote arrival from the O-CTA after PV consumed it
  // O-CTA
  B_VT_FULL = B_MSG_FREE + NMSG,    // [2] 256 dequant threads
  B_VT_EMPTY = B_VT_FULL + 2,       // [2] commit after PV
  B_MSG_FULL = B_VT_EMPTY + 2,      // [3] 1 local expect-tx arrival + the bulk copy's bytes
  B_CORR = B_MSG_FULL + NMSG,       // [3] 128 correction threads
  B_PV_DONE = B_CORR + NMSG,        // [3] commit after PV
  B_O_FULL = B_PV_DONE + NMSG,      // commit after the last PV of a range
  B_O_EMPTY = B_O_FULL + 1,         // 128 epilogue threads
  B_DRAIN = B_O_EMPTY + 1,          // MMA drain on the way out
  B_STAGED = B_DRAIN + 1,           // [NMSG] 128 softmax threads wrote a message slot (S-CTA)
  B_QLOAD = B_STAGED + NMSG,        // [9] 1 expect-tx arrival + the bytes of one Q chunk
  B_QREAD = B_QLOAD + 9,            // [2] 128 softmax threads: Q read out of key-tile stage 0 / 1
  B_OSTAGE = B_QREAD + 2,           // [8] 128 epilogue threads staged one output box (O-CTA)
  B_OFREE = B_OSTAGE + 8,           // the stores have read the staging tiles (O-CTA)
  B_LAST = B_OFREE + 1,             // one-shot commit after the partition's final PV (O-CTA)
  B_NEVER = B_LAST + 1,             // nothing arrives here (the test_stall hook waits on it)
  NUM_BARS
};
constexpr int OFF_BARS = OFF_MISC;
constexpr int OFF_TMEM_SLOT = OFF_BARS + NUM_BARS * 8;
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 16;
// S-CTA slot validity of a key-tile stage, on its way to tensor memory: 32 identical rows of
// 16 bytes, of which bytes 0-7 hold the block's bits (byte w: dequant warp w's rows w + 8 r,
// bit r)
constexpr int OFF_VMASK = (OFF_ABORT + 16 + 127) & ~127;
constexpr int VMASK_STAGE = 32 * 16;
constexpr int SMEM_BYTES = OFF_VMASK + NSTAGE * VMASK_STAGE + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// warps: 0-3 softmax (S) / correction + epilogue (O); 5-7, 9-11, 13-14 gather + dequant;
// 12 MMA; 8 message relay (O; idle on the S-CTA); 4 output store issuer (O; idle on the
// S-CTA).  The SM sub-partition that issues the MMAs (warps 0, 4, 8, 12) runs no dequant warp,
// so the single issuing thread is not starved of issue slots while a tile is being converted.
constexpr int NTHREADS = 480;
__device__ __forceinline__ int dequant_index(int warp) {
  if ((warp & 3) == 0 || warp < 5 || warp > 14) return -1;
  return warp - 5 - ((warp - 4) >> 2);  // 5, 6, 7 -> 0, 1, 2; 9, 10, 11 -> 3, 4, 5; 13, 14 -> 6, 7
}
// S-CTA tensor-memory columns: Q (fp16, 288), three score buffers (3 x 64) and the slot
// validity of the last NVMASK blocks (4 columns each, every lane the same); the O-CTA uses
// all 512 for O
constexpr uint32_t TM_Q = 0, TM_S = 288, TM_M = 480;
constexpr int NVMASK = 8;
static_assert(TM_S + NSBUF * BT == TM_M && TM_M + 4 * NVMASK == 512, "tensor-memory columns");
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
  // role already gave up.  The first test is inline; the polling loop is out of line so that
  // the many call sites keep the hot code small.
  __device__ __forceinline__ bool wait(int b, uint32_t parity, bool cluster_scope = false) const {
    const uint32_t a = bar(b);
    if (cluster_scope ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity)) return true;
    return wait_slow(b, parity, cluster_scope);
  }
  __device__ __noinline__ bool wait_slow(int b, uint32_t parity, bool cluster_scope) const {
    const uint32_t a = bar(b);
    uint64_t deadline = 0;
    for (uint32_t i = 0;; ++i) {
      if (cluster_scope ? mbar_try_wait_cluster(a, parity) : mbar_try_wait(a, parity)) return true;
      if ((i & 7u) == 7u) {
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
// A cluster's work: the request range of its partition (blocks [begin_block, nb) of
// begin_req, whole requests, blocks [0, end_block) of end_req), for each query position
// s = s0, s0 + s_step, ... below s_q in turn.  One (s, request) pair is an item; a cluster's
// items follow one another through the same pipeline, their counters running on.
struct Plan {
  int begin_req, end_req, begin_block, end_block, begin_split, nb;
  int s0, s_step, s_q;
  __device__ int first_block(int req) const { return req == begin_req ? begin_block : 0; }
  __device__ int last_block(int req) const { return req == end_req ? end_block : nb; }
  __device__ int last_s() const { return s0 + ((s_q - 1 - s0) / s_step) * s_step; }
  __device__ bool last_item(int s, int req) const { return req == end_req && s + s_step >= s_q; }
  __device__ int blocks_per_s() const {
    int n = 0;
    for (int r = begin_req; r <= end_req; ++r) n += last_block(r) - first_block(r);
    return n;
  }
};
struct Cursor {
  int s, req, blk;  // current block; s >= s_q once past the end
  uint32_t item;    // items begun before the current one
  __device__ void start(const Plan& pl) {
    s = pl.s0;
    req = pl.begin_req;
    blk = pl.first_block(req);
    item = 0;
  }
  __device__ bool done(const Plan& pl) const { return s >= pl.s_q; }
  __device__ void next(const Plan& pl) {
    if (++blk >= pl.last_block(req)) {
      ++item;
      if (++req > pl.end_req) {
        req = pl.begin_req;
        s += pl.s_step;
      }
      blk = pl.first_block(req);
    }
  }
};

// ---------------------------------------------------------------------------------------
// Gather + dequant (the eight dequant warps of both CTAs).  Dequant warp w owns rows w, w + 8, ..., w + 56 of every
// block and handles them four at a time: the eight lanes 8 r .. 8 r + 7 share a row, and lane
// j of the eight copies and converts 16-byte code chunks j, j + 8, j + 16, j + 24 of it
// (dims [16 c, 16 c + 16) of chunk c) and, on the S-CTA, RoPE chunk j; lane 0 of the eight
// also copies the 4 scales.  Rows are copied global -> shared with cp.async into a per-warp
// ring of 8 row slots that runs one block ahead of the conversion, so a block of rows per
// warp is in flight and no row passes through registers before it has landed.  A slot whose
// index is masked is zero-filled without a read.
constexpr int RING = 8;  // row slots per dequant warp
// Ring slot of one gathered row: the 656-byte row (S-CTA) or its NoPE codes + scales (O-CTA);
// for the later formats (both CTAs: the value is the whole key) the data row, then its scale
// row padded to 16 bytes.
template <bool kScores, int kF>
struct RowCopy {
  static constexpr int kBytes = kF == FMT_V32 ? (kScores ? kRowBytes : kDNope + 16)
                                              : FmtBytes<kF>::kData + 16;
};
static_assert(8 * RING * RowCopy<true, FMT_V32>::kBytes <= RAW_BYTES &&
                  8 * RING * RowCopy<true, FMT_V4>::kBytes <= RAW_BYTES &&
                  8 * RING * RowCopy<true, FMT_V41>::kBytes <= RAW_BYTES,
              "row ring");

// Index of one slot, -1 for a slot past the list or (kLen: the kernel instance for per-token
// lengths) past the token's topk_length; both loads are issued before either is tested.  The
// length test lives in its own instance because even an untaken test here slows the hot loop.
template <bool kLen>
__device__ __forceinline__ int32_t load_index(const DecodeParams& p, int s, int req, int blk,
                                              int row) {
  const int slot = blk * BT + row;
  if (slot >= p.topk) return -1;
  const size_t tok = static_cast<size_t>(req) * p.s_q + s;
  const int32_t ix = ldg_s32(p.indices + tok * p.topk + slot);
  if (kLen && slot >= ldg_s32(p.topk_length + tok)) return -1;
  return ix;
}

// The same for the extra list (block `blk` of it; kernel instances with an extra cache only).
__device__ __forceinline__ int32_t load_extra_index(const DecodeParams& p, int s, int req,
                                                    int blk, int row) {
  const int slot = blk * BT + row;
  if (slot >= p.extra_topk) return -1;
  const size_t tok = static_cast<size_t>(req) * p.s_q + s;
  const int32_t ix = ldg_s32(p.extra_indices + tok * p.extra_topk + slot);
  if (p.extra_topk_length != nullptr && slot >= ldg_s32(p.extra_topk_length + tok)) return -1;
  return ix;
}

// Copies this lane's share of one row (j = lane % 8) into its ring slot; one commit group per
// call covers the four rows of the warp step.
template <bool kScores>
__device__ __forceinline__ void issue_rows(const DecodeParams& p, int32_t idx, uint32_t slot,
                                           int j, bool extra = false) {
  const uint8_t* base = extra ? p.extra_kv : p.kv;
  const bool ok = idx >= 0 && idx < (extra ? p.extra_rows : p.num_rows);
  const uint8_t* src = base + static_cast<size_t>(ok ? idx : 0) * kRowBytes;
  const uint32_t n = ok ? 16u : 0u;
#pragma unroll
  for (int k = 0; k < 4; ++k) cp_async16(slot + (j + 8 * k) * 16, src + (j + 8 * k) * 16, n);
  if (j == 0) cp_async16(slot + kDNope, src + kDNope, n);  // scales
  if (kScores) cp_async16(slot + kDNope + 16 + j * 16, src + kDNope + 16 + j * 16, n);  // RoPE
  cp_async_commit();
}

// Converts this lane's share of one landed row into the fp16 tile (row `row`).
template <bool kScores>
__device__ __forceinline__ void store_rows(uint32_t tile, int row, int j, bool valid,
                                           const uint4 (&nope)[4], const uint4& scales,
                                           const uint4& rope, uint32_t& bad) {
  // code chunk c = j + 8 k -> 64-dim tile chunk c / 4 = j / 4 + 2 k, 8-dim sub-chunks
  // 2 (j % 4) and + 1; lanes 4-7 of the eight store their odd sub-chunk first, so the eight
  // lanes of a row hit 8 distinct 16-byte bank groups with every store (no bank conflict)
  const uint32_t flip = (j >> 2) & 1;
  const uint32_t u0 = 2 * (j & 3) + flip, u1 = 2 * (j & 3) + (flip ^ 1u);
  const uint32_t ch0 = tile + (j >> 2) * CHUNK;
  if (valid) {
    const uint32_t sc[4] = {scales.x, scales.y, scales.z, scales.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // code chunk j + 8 k lies in scale group k
      const float scale = __uint_as_float(sc[k]) * 256.f;
      bad |= !(scale >= 6.103515625e-05f && scale <= 65504.f);
      const uint32_t sc2 = pack_f16x2(scale, scale);
      // the first store goes to sub-chunk u0: the flipped lanes convert their second 8 codes
      // first (the two 8-byte halves of the unit swapped once, instead of every output word)
      const uint32_t w[4] = {flip ? nope[k].z : nope[k].x, flip ? nope[k].w : nope[k].y,
                             flip ? nope[k].x : nope[k].z, flip ? nope[k].y : nope[k].w};
      uint32_t o[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[2 * e] = hmul2(cvt_e4m3x2_f16x2(static_cast<uint16_t>(w[e] & 0xFFFFu)), sc2);
        o[2 * e + 1] = hmul2(cvt_e4m3x2_f16x2(static_cast<uint16_t>(w[e] >> 16)), sc2);
      }
      const uint32_t ch = ch0 + 2 * k * CHUNK;
      st_shared_v4(ch + sw128_chunk(row, u0), o[0], o[1], o[2], o[3]);
      st_shared_v4(ch + sw128_chunk(row, u1), o[4], o[5], o[6], o[7]);
    }
    if (kScores) {
      const uint32_t r[4] = {rope.x, rope.y, rope.z, rope.w};
      uint32_t q[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        q[e] = pack_f16x2(__uint_as_float(r[e] << 16) * 256.f,
                          __uint_as_float(r[e] & 0xFFFF0000u) * 256.f);
      st_shared_v4(tile + 8 * CHUNK + sw128_chunk(row, j), q[0], q[1], q[2], q[3]);
    }
  } else {
    // invalid slot: NaN key (its score becomes NaN and is masked) or zero value
    const uint32_t f = kScores ? F16_NAN2 : 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      st_shared_v4(ch0 + 2 * k * CHUNK + sw128_chunk(row, u0), f, f, f, f);
      st_shared_v4(ch0 + 2 * k * CHUNK + sw128_chunk(row, u1), f, f, f, f);
    }
    if (kScores) st_shared_v4(tile + 8 * CHUNK + sw128_chunk(row, j), f, f, f, f);
  }
}

// ---- the later formats (d_qk = d_v = 512, structure-of-arrays pages; "FlashMLA 与 DSA",
// sections 3.1, 2.1 and 6.4).  A page of 64 tokens holds the 64 data rows, then the 64 scale
// rows.  V4: 448 e4m3 codes (e8m0 scale per 64 dims) + 64 bf16 RoPE values, 8 scale bytes
// (7 + 1 pad); V4.1: 512 e4m3 codes, 16 e8m0 scales (per 32 dims); FP4 (the extra cache of a
// V4.1 cache only): 512 e2m1 values, two per byte with the even element in the low nibble, and
// 32 e4m3 scales (per 16 dims).  The value is the whole key, so both CTAs convert the same
// eight 64-dim chunks.

// Copies this lane's share of one row of a later format into its ring slot: data unit
// (16 bytes) j + 8 k, and the scale row (lane 0; FP4: lanes 0 and 1).  An invalid id reads
// nothing and zero-fills.  One commit group per call.
template <int kF>
__device__ __forceinline__ void issue_row_soa(const DecodeParams& p, int32_t idx, uint32_t slot,
                                              int j, bool extra) {
  const bool fp4 = kF == FMT_V41 && extra;
  const int data = fp4 ? FP4_DATA : FmtBytes<kF>::kData;
  const int scale = fp4 ? FP4_SCALE : FmtBytes<kF>::kScale;
  const uint8_t* base = extra ? p.extra_kv : p.kv;
  const bool ok = idx >= 0 && idx < (extra ? p.extra_rows : p.num_rows);
  const uint32_t t = ok ? static_cast<uint32_t>(idx) : 0u;
  const uint8_t* page = base + static_cast<size_t>(t >> 6) * (kPage * (data + scale));
  const uint8_t* src = page + (t & 63u) * data;
  const uint8_t* ssrc = page + kPage * data + (t & 63u) * scale;
  const uint32_t n = ok ? 16u : 0u;
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    const int u = j + 8 * k;
    if (u < data / 16) cp_async16(slot + u * 16, src + u * 16, n);
  }
  if (kF == FMT_V4 && !fp4) {
    if (j == 0) cp_async8(slot + data, ssrc, ok ? 8u : 0u);
  } else if (fp4) {
    if (j < 2) cp_async16(slot + data + 16 * j, ssrc + 16 * j, n);
  } else if (j == 0) {
    cp_async16(slot + data, ssrc, n);
  }
  cp_async_commit();
}

// This lane's share of a landed row: a[k] = data unit j + 8 k (V4: units j + 24 only for
// j < 4, c = RoPE unit 28 + j; FP4: a[0], a[1] = units j, j + 8), b = the scale row (FP4: the
// scale pairs 2 j, 2 j + 1 and 2 j + 16, 2 j + 17 in b.x).
template <int kF>
__device__ __forceinline__ void load_row_soa(uint32_t slot, int j, bool extra, uint4 (&a)[4],
                                             uint4& b, uint4& c) {
  if (kF == FMT_V41 && extra) {
    ld_shared_v4(slot + j * 16, a[0].x, a[0].y, a[0].z, a[0].w);
    ld_shared_v4(slot + (j + 8) * 16, a[1].x, a[1].y, a[1].z, a[1].w);
    b.x = ld_shared_u16(slot + FP4_DATA + 2 * j) | (ld_shared_u16(slot + FP4_DATA + 16 + 2 * j) << 16);
    return;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    if (kF == FMT_V4 && k == 3 && j >= 4) {
      a[k] = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    ld_shared_v4(slot + (j + 8 * k) * 16, a[k].x, a[k].y, a[k].z, a[k].w);
  }
  if (kF == FMT_V4) {
    ld_shared_v4(slot + (28 + j) * 16, c.x, c.y, c.z, c.w);
    ld_shared_v2(slot + FmtBytes<kF>::kData, b.x, b.y);
  } else {
    ld_shared_v4(slot + FmtBytes<kF>::kData, b.x, b.y, b.z, b.w);
  }
}

// 256 x an e8m0 scale as an f16x2 pair: 2^(e - 127 + 8) is the fp16 with exponent field
// e - 104 (normal for e in [105, 134]; others are flagged and clamped); 0xFF is NaN.
__device__ __forceinline__ uint32_t e8m0_x256_f16x2(uint32_t e, uint32_t& bad) {
  if (e == 255u) return F16_NAN2;
  const int ex = static_cast<int>(e) - 104;
  bad |= ex < 1 || ex > 30;
  const uint32_t h = static_cast<uint32_t>(ex < 1 ? 1 : (ex > 30 ? 30 : ex)) << 10;
  return h | (h << 16);
}

// Converts this lane's share of a landed row of a later format into the fp16 tile (row `row`,
// eight 64-dim chunks); invalid: NaN key (S-CTA) or zero value (O-CTA).
template <bool kScores, int kF>
__device__ __forceinline__ void store_row_soa(uint32_t tile, int row, int j, bool valid, bool extra,
                                              const uint4 (&a)[4], const uint4& b, const uint4& c,
                                              uint32_t& bad) {
  const uint32_t flip = (j >> 2) & 1;
  const uint32_t u0 = 2 * (j & 3) + flip, u1 = 2 * (j & 3) + (flip ^ 1u);
  const uint32_t ch0 = tile + (j >> 2) * CHUNK;
  if (!valid) {
    const uint32_t f = kScores ? F16_NAN2 : 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      st_shared_v4(ch0 + 2 * k * CHUNK + sw128_chunk(row, u0), f, f, f, f);
      st_shared_v4(ch0 + 2 * k * CHUNK + sw128_chunk(row, u1), f, f, f, f);
    }
    return;
  }
  if (kF == FMT_V41 && extra) {  // FP4: units j and j + 8, 32 dims each (4 sub-chunks)
#pragma unroll
    for (int uu = 0; uu < 2; ++uu) {
      const int u = j + 8 * uu;
      // the unit's two e4m3 scales (16 dims each) x 256 as fp16; 256 x 448 would overflow
      const uint32_t s2 = hmul2(cvt_e4m3x2_f16x2(static_cast<uint16_t>(uu ? b.x >> 16 : b.x & 0xFFFFu)),
                                0x5C005C00u);
      bad |= ((s2 & 0x7FFFu) == 0x7C00u) | (((s2 >> 16) & 0x7FFFu) == 0x7C00u);
      const uint32_t slo = (s2 & 0xFFFFu) * 0x10001u, shi = (s2 >> 16) * 0x10001u;
      const uint32_t wd[4] = {a[uu].x, a[uu].y, a[uu].z, a[uu].w};
      const uint32_t ch = tile + (u >> 1) * CHUNK;
#pragma unroll
      for (int m = 0; m < 4; ++m) {  // word m: dims 32 u + 8 m .. + 8 (scale 2 u + m / 2)
        const uint32_t sc = m < 2 ? slo : shi;
        st_shared_v4(ch + sw128_chunk(row, (u & 1) * 4 + m),
                     hmul2(cvt_e2m1x2_f16x2(wd[m] & 0xFFu), sc),
                     hmul2(cvt_e2m1x2_f16x2((wd[m] >> 8) & 0xFFu), sc),
                     hmul2(cvt_e2m1x2_f16x2((wd[m] >> 16) & 0xFFu), sc),
                     hmul2(cvt_e2m1x2_f16x2(wd[m] >> 24), sc));
      }
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {  // code unit j + 8 k -> chunk j / 4 + 2 k, as the 656-byte NoPE
    if (kF == FMT_V4 && k == 3 && j >= 4) continue;  // units 28-31 are RoPE, converted below
    uint32_t e;
    if (kF == FMT_V41) {  // scale of dims 32 s..: s = (j + 8 k) / 2 = j / 2 + 4 k
      const uint32_t wk = k == 0 ? b.x : k == 1 ? b.y : k == 2 ? b.z : b.w;
      e = (wk >> (8 * ((j >> 1) & 3))) & 0xFFu;
    } else {  // V4: scale of dims 64 s..: s = j / 4 + 2 k
      const int si = (j >> 2) + 2 * k;
      e = ((si < 4 ? b.x : b.y) >> (8 * (si & 3))) & 0xFFu;
    }
    const uint32_t sc2 = e8m0_x256_f16x2(e, bad);
    const uint32_t w[4] = {flip ? a[k].z : a[k].x, flip ? a[k].w : a[k].y,
                           flip ? a[k].x : a[k].z, flip ? a[k].y : a[k].w};
    uint32_t o[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      o[2 * q] = hmul2(cvt_e4m3x2_f16x2(static_cast<uint16_t>(w[q] & 0xFFFFu)), sc2);
      o[2 * q + 1] = hmul2(cvt_e4m3x2_f16x2(static_cast<uint16_t>(w[q] >> 16)), sc2);
    }
    const uint32_t ch = ch0 + 2 * k * CHUNK;
    st_shared_v4(ch + sw128_chunk(row, u0), o[0], o[1], o[2], o[3]);
    st_shared_v4(ch + sw128_chunk(row, u1), o[4], o[5], o[6], o[7]);
  }
  if (kF == FMT_V4) {  // RoPE unit j: dims 448 + 8 j .. + 8 (bf16 -> 256 x fp16), chunk 7
    const uint32_t r[4] = {c.x, c.y, c.z, c.w};
    uint32_t q[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      q[e] = pack_f16x2(__uint_as_float(r[e] << 16) * 256.f,
                        __uint_as_float(r[e] & 0xFFFF0000u) * 256.f);
    st_shared_v4(tile + 7 * CHUNK + sw128_chunk(row, j), q[0], q[1], q[2], q[3]);
  }
}

// kExtra: the kernel instance with an extra cache, whose blocks follow the main list's in the
// plan (blocks nb_main and up read the extra indices and rows).  kF: the main cache's format
// (the extra cache of a V4.1 cache is FP4; of a 656-byte cache, 656-byte).
template <bool kScores, bool kLen, bool kExtra, int kF>
__device__ void role_dequant(const DecodeParams& p, const Ctx& c, const Plan& pl, int t) {
  using RC = RowCopy<kScores, kF>;
  const int w = t >> 5, lane = t & 31;  // warp w of the 8 dequant warps
  const int j = lane & 7, rsel = lane >> 3;
  const int bfull = kScores ? B_KT_FULL : B_VT_FULL;
  const int bempty = kScores ? B_KT_EMPTY : B_VT_EMPTY;
  const int stage_bytes = kScores ? KT_STAGE : VT_STAGE;
  const uint32_t ring = c.sbase + OFF_RAW + w * RING * RC::kBytes;
  uint32_t bad = 0;
  auto in_extra = [&](const Cursor& k) -> bool { return kExtra && k.blk >= p.nb_main; };
  // Lane r < 8 holds the index of row w + 8 r of a block.
  auto idx_of = [&](const Cursor& k) -> int32_t {
    if (lane >= 8 || k.done(pl)) return -1;
    if (in_extra(k)) return load_extra_index(p, k.s, k.req, k.blk - p.nb_main, w + 8 * lane);
    return load_index<kLen>(p, k.s, k.req, k.blk, w + 8 * lane);
  };
  auto valid_bits = [&](int32_t ix, bool extra) -> uint32_t {
    const int rows = extra ? p.extra_rows : p.num_rows;
    return __ballot_sync(0xffffffffu, lane < 8 && ix >= 0 && ix < rows) & 0xFFu;
  };
  Cursor cur, fetch;
  cur.start(pl);
  fetch = cur;
  // prologue: the first block's rows in flight, the second block's indices loaded
  const int32_t ix0 = idx_of(fetch);
  uint32_t vmask = valid_bits(ix0, in_extra(fetch));  // bits 8 k + r: row r of block cur + k is valid
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = 4 * h + rsel;
    if (kF == FMT_V32)
      issue_rows<kScores>(p, __shfl_sync(0xffffffffu, ix0, r), ring + r * RC::kBytes, j,
                          in_extra(fetch));
    else
      issue_row_soa<kF>(p, __shfl_sync(0xffffffffu, ix0, r), ring + r * RC::kBytes, j,
                        in_extra(fetch));
  }
  fetch.next(pl);
  int32_t ixA = idx_of(fetch);  // block cur + 1
  fetch.next(pl);
  uint32_t g = 0;
#pragma unroll 1
  while (!cur.done(pl)) {
    const uint32_t st = g & 1;
    Cursor ah = cur;
    ah.next(pl);
    const bool issue_more = !ah.done(pl);  // block cur + 1 exists
    const bool extra_next = in_extra(ah);
    const bool extra_cur = in_extra(cur);
    const int32_t ixB = idx_of(fetch);      // block cur + 2, loaded one block early
    vmask |= valid_bits(ixA, extra_next) << 8;
    if (g >= NSTAGE && !c.wait_warp(bempty + st, ((g >> 1) - 1) & 1)) goto out;
    // each token's Q passes through the key-tile region on its way to tensor memory: the
    // first two tiles of a request (one per stage) wait until their stage's part of it has
    // been read out
    if (kScores && cur.blk - pl.first_block(cur.req) < NSTAGE &&
        !c.wait_warp(B_QREAD + st, cur.item & 1u))
      goto out;
    {
      const uint32_t tile = c.sbase + OFF_TILE + st * stage_bytes;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        const int r = 4 * h + rsel;  // this lane's row of the block: w + 8 r
        cp_async_wait<1>();          // the copies of this step (the older group) have landed
        __syncwarp();
        const uint32_t slot = ring + r * RC::kBytes;
        uint4 nope[4], scales = make_uint4(0u, 0u, 0u, 0u), rope = make_uint4(0u, 0u, 0u, 0u);
        if (kF == FMT_V32) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            ld_shared_v4(slot + (j + 8 * k) * 16, nope[k].x, nope[k].y, nope[k].z, nope[k].w);
          ld_shared_v4(slot + kDNope, scales.x, scales.y, scales.z, scales.w);
          if (kScores) ld_shared_v4(slot + kDNope + 16 + j * 16, rope.x, rope.y, rope.z, rope.w);
        } else {
          load_row_soa<kF>(slot, j, extra_cur, nope, scales, rope);
        }
        __syncwarp();  // every lane has read the slot: it can take the next block's row
        const int32_t nx = __shfl_sync(0xffffffffu, ixA, r);
        if (issue_more) {
          if (kF == FMT_V32) issue_rows<kScores>(p, nx, slot, j, extra_next);
          else issue_row_soa<kF>(p, nx, slot, j, extra_next);
        } else {
          cp_async_commit();  // an empty group keeps the count per step uniform
        }
        if (kF == FMT_V32)
          store_rows<kScores>(tile, w + 8 * r, j, (vmask >> r) & 1u, nope, scales, rope, bad);
        else
          store_row_soa<kScores, kF>(tile, w + 8 * r, j, (vmask >> r) & 1u, extra_cur, nope,
                                     scales, rope, bad);
      }
    }
    // the block's validity bits for the softmax (this warp's byte of all 32 rows); the MMA
    // warp copies them into tensor memory with the tile's QK.  The stage is free: its last
    // copy was done with the QK of block g - 2.
    if (kScores) st_shared_u8(c.sbase + OFF_VMASK + st * VMASK_STAGE + lane * 16 + w, vmask & 0xFFu);
    fence_proxy_async_smem();
    mbar_arrive(c.bar(bfull + st));
    vmask >>= 8;
    ixA = ixB;
    fetch.next(pl);
    cur.next(pl);
    ++g;
  }
out:
  cp_async_wait<0>();  // no copy may land after the CTA has moved on
  if (bad) atomicOr(c.status, SMLA_DEV_SCALE_RANGE);
}

// ---------------------------------------------------------------------------------------
// S-CTA MMA warp: S[buf] = Q K^T for every block (4 MMAs of K = 16 per 64-dim chunk: 36 at
// d_qk = 576, 32 at 512).  The whole warp runs
// the loop (waits included) and one elected lane issues each MMA and commit.
template <int kChunks>
__device__ void role_mma_scores(const Ctx& c, const Plan& pl, uint32_t tbase, bool stall) {
  // test hook: a wait that nothing ends, so every role runs into its bounded wait
  if (stall) {
    c.wait_warp(B_NEVER, 0);
    return;
  }
  uint32_t g = 0, item = 0;
  for (int s = pl.s0; s < pl.s_q; s += pl.s_step)
  for (int req = pl.begin_req; req <= pl.end_req; ++req, ++item) {
    if (!c.wait_warp(B_Q_FULL, item & 1)) return;
    for (int blk = pl.first_block(req); blk < pl.last_block(req); ++blk, ++g) {
      const uint32_t st = g & 1, sb = g % NSBUF;
      if (!c.wait_warp(B_KT_FULL + st, (g >> 1) & 1)) return;
      if (g >= NSBUF && !c.wait_warp(B_S_EMPTY + sb, ((g / NSBUF) - 1) & 1)) return;
      tc_fence_after();
      // the block's validity bits into columns TM_M + 4 (g % NVMASK); the softmax of block
      // g - 8, which read them last, released its scores before the QK of block g - 5
      tmem_cp_32x128b_x4_warp(tbase + TM_M + 4 * (g % NVMASK),
                              umma_desc(c.sbase + OFF_VMASK + st * VMASK_STAGE, 16, 128, 0));
      const uint64_t bdesc = umma_desc(c.sbase + OFF_TILE + st * KT_STAGE, 16, 1024, 2);
      const uint32_t d = tbase + TM_S + sb * BT;
#pragma unroll 4  // kept rolled: the issuing warp shares its instruction cache with the others
      for (int kk = 0; kk < 4 * kChunks; ++kk)  // descriptor start addresses advance in 16 bytes
        mma_ts_warp(d, tbase + TM_Q + kk * 8,
                    bdesc + ((((kk >> 2) * CHUNK) + (kk & 3) * 32) >> 4), IDESC_QK, kk > 0);
      mma_commit_warp(c.bar(B_S_FULL + sb));
      mma_commit_warp(c.bar(B_KT_EMPTY + st));
    }
  }
}

// O-CTA MMA warp: O += P V for every block (4 K-steps x 2 N-halves); the whole warp runs the
// loop and one elected lane issues.
__device__ void role_mma_values(const Ctx& c, const Plan& pl, uint32_t tbase) {
  uint32_t g = 0, item = 0;
  for (int s = pl.s0; s < pl.s_q; s += pl.s_step)
  for (int req = pl.begin_req; req <= pl.end_req; ++req, ++item) {
    const int b0 = pl.first_block(req), b1 = pl.last_block(req);
    for (int blk = b0; blk < b1; ++blk, ++g) {
      const uint32_t st = g & 1, ms = g % NMSG, mpar = (g / NMSG) & 1;
      const bool first = blk == b0;
      if (!c.wait_warp(B_VT_FULL + st, (g >> 1) & 1)) return;
      if (!c.wait_warp(B_MSG_FULL + ms, mpar, true)) return;
      if (!c.wait_warp(B_CORR + ms, mpar)) return;
      if (first && item >= 1 && !c.wait_warp(B_O_EMPTY, (item - 1) & 1)) return;
      tc_fence_after();
      const uint64_t adesc = umma_desc(c.sbase + OFF_MSG + ms * MSG_STRIDE, 16, 1024, 2);
      const uint64_t bdesc = umma_desc(c.sbase + OFF_TILE + st * VT_STAGE, CHUNK, 1024, 2);
#pragma unroll
      for (int kk = 0; kk < BT / 16; ++kk) {
#pragma unroll
        for (int nh = 0; nh < 2; ++nh)  // descriptor start addresses advance in 16-byte units
          mma_ss_warp(tbase + nh * 256, adesc + (kk * 32 >> 4),
                      bdesc + ((nh * 4 * CHUNK + kk * 2048) >> 4), IDESC_PV, !(first && kk == 0));
      }
      mma_commit_warp(c.bar(B_VT_EMPTY + st));
      mma_commit_warp(c.bar(B_PV_DONE + ms));
      if (blk == b1 - 1) mma_commit_warp(c.bar(B_O_FULL));
      if (blk == b1 - 1 && pl.last_item(s, req)) mma_commit_warp(c.bar(B_LAST));
    }
  }
}

// ---------------------------------------------------------------------------------------
// Q of one query token (request number `item` of the partition): nine tiled tensor copies (one
// per 64-dim chunk, h_q rows of 128 bytes, 128-byte swizzle), each with its own barrier, into
// the key-tile region; thread i = head i converts its row to fp16 into tensor memory chunk by
// chunk as the copies land.  The region is free then: every QK of the previous request has
// completed and the dequant warps hold the request's first two tiles back until B_QREAD of
// their stage (stage 0's part of Q is read out first, so the first tile can be written while
// the rest converts).  The
// swizzle puts unit u of row r at position u ^ (r % 8), so eight consecutive heads read eight
// distinct bank groups.  The fp16 range is checked on the bf16 magnitudes (a packed 16-bit
// max), not per converted value: the conversion is issue-bound on the SM sub-partitions.
// False if a wait ran out.
static_assert(9 * 128 * 128 <= OFF_MSG, "Q fits in the key-tile region");
// The copies alone (one thread).  For a cluster's later items they are issued as soon as the
// QK of the current item's last block has completed (the region and Q's tensor-memory columns
// are free from then on), so that they land while that block's softmax runs.
__device__ void issue_q(const DecodeParams& p, const Ctx& c, int tok) {
  const uint32_t qs = c.sbase + OFF_TILE;
  const uint32_t chunk_bytes = static_cast<uint32_t>(p.h_q) * 128;
  for (int ch = 0; ch < p.q_chunks; ++ch) {
    mbar_arrive_expect_tx(c.bar(B_QLOAD + ch), chunk_bytes);
    tma_load_2d(qs + ch * chunk_bytes, &p.q_map, ch * 64, tok * p.h_q, c.bar(B_QLOAD + ch));
  }
}
__device__ bool stage_q_bulk(const DecodeParams& p, const Ctx& c, uint32_t tq, int tok, int i,
                             uint32_t& bad, uint32_t item, bool issued = false) {
  const uint32_t qs = c.sbase + OFF_TILE;
  const uint32_t chunk_bytes = static_cast<uint32_t>(p.h_q) * 128;
  const int nch = p.q_chunks;
  if (i == 0 && !issued) issue_q(p, c, tok);
  const bool live = i < p.h_q;
  const uint32_t row = qs + static_cast<uint32_t>(i) * 128;
  const uint32_t sw = static_cast<uint32_t>(i & 7);
  // the chunks overlapping each key-tile stage: stage 0 is free once chunk lo_last is read,
  // stage 1 once the last chunk is (or at once when Q does not reach it)
  const int lo_last = min(nch, static_cast<int>((KT_STAGE + chunk_bytes - 1) / chunk_bytes)) - 1;
  const bool reaches_hi = static_cast<uint32_t>(nch) * chunk_bytes > KT_STAGE;
  if (!reaches_hi) mbar_arrive(c.bar(B_QREAD + 1));
  uint32_t mag[4] = {0u, 0u, 0u, 0u};  // largest bf16 magnitude seen, per 16-bit half (4 chains)
#pragma unroll 1
  for (int ch = 0; ch < nch; ++ch) {
    if (!c.wait_warp(B_QLOAD + ch, item & 1)) return false;
    uint32_t w[32];
    if (live) {
      uint32_t in[32];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        ld_shared_v4(row + ch * chunk_bytes + ((static_cast<uint32_t>(u) ^ sw) << 4), in[4 * u],
                     in[4 * u + 1], in[4 * u + 2], in[4 * u + 3]);
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        mag[e & 3] = vmax_u16x2(mag[e & 3], in[e] & 0x7FFF7FFFu);
        w[e] = pack_f16x2(__uint_as_float(in[e] << 16), __uint_as_float(in[e] & 0xFFFF0000u));
      }
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e) w[e] = 0u;
    }
    tmem_st16(tq + ch * 32, w);
    tmem_st16(tq + ch * 32 + 16, w + 16);
    if (ch == lo_last) mbar_arrive(c.bar(B_QREAD));  // this thread is done with stage 0
  }
  // bf16 magnitude 0x4780 (2^16) and above rounds to inf in fp16 (0x477F = 65280 is finite)
  const uint32_t m = vmax_u16x2(vmax_u16x2(mag[0], mag[1]), vmax_u16x2(mag[2], mag[3]));
  bad |= ((m >> 16) >= 0x4780u) | ((m & 0xFFFFu) >= 0x4780u);
  tmem_wait_st();
  tc_fence_before();
  mbar_arrive(c.bar(B_Q_FULL));
  if (reaches_hi) mbar_arrive(c.bar(B_QREAD + 1));  // and with stage 1
  return true;
}

// p = 2^(s * c2 - mref) for the 64 scores of row i (tensor-memory columns [scol, scol + 64)),
// stored as fp16 into the row's message slot; returns their sum.  kMasked: slot k is valid
// when bit 8 (k % 8) + k / 8 of vmask is set (byte w: rows w + 8 r of the dequant warp w);
// invalid slots get p = 0 (their keys are NaN).  The scores are read from tensor memory 32 at
// a time and the loop stays rolled (a small hot loop next to the other roles' code).
template <bool kMasked>
__device__ __forceinline__ float exp_pass(uint32_t scol, uint32_t msg, int i, float c2, float mref,
                                          uint64_t vmask) {
  float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t r32[32];
    tmem_ld16(scol + hh * 32, r32);
    tmem_ld16(scol + hh * 32 + 16, r32 + 16);
    const uint64_t vh = vmask >> (4 * hh);  // slot 32 hh + j: bit 8 (j % 8) + j / 8
    tmem_wait_ld();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int k0 = 8 * k + 2 * e;
        float p0 = ex2(fmaf(__uint_as_float(r32[k0]), c2, -mref));
        float p1 = ex2(fmaf(__uint_as_float(r32[k0 + 1]), c2, -mref));
        if (kMasked) {
          p0 = (vh >> (8 * (k0 & 7) + (k0 >> 3))) & 1u ? p0 : 0.f;
          p1 = (vh >> (8 * ((k0 + 1) & 7) + ((k0 + 1) >> 3))) & 1u ? p1 : 0.f;
        }
        sq[e] += p0 + p1;
        w[e] = pack_f16x2(p0, p1);
      }
      st_shared_v4(msg + sw128_chunk(i, 4 * hh + k), w[0], w[1], w[2], w[3]);
    }
  }
  return (sq[0] + sq[1]) + (sq[2] + sq[3]);
}

// S-CTA softmax warpgroup: thread i owns head row i (tensor-memory lane i).  The exponentials
// of invalid slots are zeroed by the block's validity bits (from the dequant warps, through
// tensor memory), so a NaN
// or +inf score of a valid slot (a NaN code in its row) is not masked: it makes the row's sum
// NaN, hence O and lse, as the definition gives, and the status word gets SMLA_DEV_NAN_INPUT.
__device__ void role_softmax(const DecodeParams& p, const Ctx& c, const Plan& pl,
                             uint32_t tbase, int i) {
  const uint32_t lane_base = static_cast<uint32_t>((i >> 5) * 32) << 16;
  const uint32_t tq = tbase + lane_base + TM_Q;
  const uint32_t ts = tbase + lane_base + TM_S;
  const uint32_t peer_msg = mapa(c.sbase + OFF_MSG, 1);
  const uint32_t peer_full = mapa(c.bar(B_MSG_FULL), 1);
  const bool live = i < p.h_q;
  uint32_t qbad = 0, nan_row = 0;
  uint32_t g = 0, item = 0;
  if (!stage_q_bulk(p, c, tq, pl.begin_req * p.s_q + pl.s0, i, qbad, 0)) goto out;
  for (int s = pl.s0; s < p.s_q; s += pl.s_step)
  for (int req = pl.begin_req; req <= pl.end_req; ++req, ++item) {
    const int b0 = pl.first_block(req), b1 = pl.last_block(req);
    float m = -INFINITY;  // running max (base-2 units) used as the exponent reference
    float l = 0.f;        // running exp-sum against m
    for (int blk = b0; blk < b1; ++blk, ++g) {
      const uint32_t sb = g % NSBUF, st = g % NMSG;
      if (!c.wait_warp(B_S_FULL + sb, (g / NSBUF) & 1)) goto out;
      tc_fence_after();
      // the item's last QK has completed: the next item's Q copies can start now (every item
      // has a last block: the plan splits a request only where both sides keep a block)
      if (i == 0 && blk == b1 - 1 && !pl.last_item(s, req)) {
        const int nreq = req < pl.end_req ? req + 1 : pl.begin_req;
        const int ns = req < pl.end_req ? s : s + pl.s_step;
        issue_q(p, c, nreq * p.s_q + ns);
      }
      // the block's validity bits, copied into tensor memory with its QK (the same commit)
      uint32_t mk[2];
      tmem_ld2(tbase + lane_base + TM_M + 4 * (g % NVMASK), mk);
      // block max in base-2 units: fmaxf skips the NaN scores of invalid slots, and the scale
      // is positive, so it applies to the max of the raw scores (four chains for ILP; two
      // halves of 32 scores, so that few registers are live)
      const float c2 = p.score_scale_log2;
      float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t sr[32];
        tmem_ld16(ts + sb * BT + hh * 32, sr);
        tmem_ld16(ts + sb * BT + hh * 32 + 16, sr + 16);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) mq[k & 3] = fmaxf(mq[k & 3], __uint_as_float(sr[k]));
      }
      const float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * c2;
      const uint64_t vmask = (static_cast<uint64_t>(mk[1]) << 32) | mk[0];
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
      if (g >= NMSG && !c.wait_warp(B_MSG_FREE + st, ((g / NMSG) - 1) & 1, true)) goto out;
      const uint32_t msg = c.sbase + OFF_MSG + st * MSG_STRIDE;
      // p = 2^(s * c2 - mref), 0 for an invalid slot (whose key is NaN).
      // A block whose slots are all valid (the mask is the same for every row, so the branch
      // is uniform) takes the loop without the mask.
      const float sum = vmask == ~0ull
                            ? exp_pass<false>(ts + sb * BT, msg, i, c2, mref, 0ull)
                            : exp_pass<true>(ts + sb * BT, msg, i, c2, mref, vmask);
      tc_fence_before();
      mbar_arrive(c.bar(B_S_EMPTY + sb));  // every read of this score buffer is done
      l = l * alpha + sum;
      st_shared_f32(msg + MSG_ALPHA + 4 * i, alpha);
      if (blk == b1 - 1) {
        // last block of the range: the O-CTA's normalisation, and the lse from here.  An
        // unsplit row with an attention sink divides by L + 2^(sink log2(e) - m) instead of
        // L (the sink as one more key with a zero value; split rows get it in the combine).
        const int first_slot = p.nsplits[req];
        const bool no_split = p.nsplits[req + 1] - first_slot == 1;
        float denom = l;
        if (no_split && live && p.attn_sink != nullptr && l != 0.f)
          denom += ex2(fmaf(__ldg(p.attn_sink + i), 1.4426950408889634f, -m));
        st_shared_f32(msg + MSG_INVL + 4 * i, l == 0.f ? 0.f : 1.f / (denom * 256.f));
        nan_row |= live && l != l;
        if (live) {
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
        if (!c.wait(B_STAGED + st, (g / NMSG) & 1)) goto out;
        bulk_s2s_cluster(peer_msg + st * MSG_STRIDE, msg, MSG_BYTES, peer_full + st * 8);
      }
    }
    // every QK^T of this range has completed: convert the next item's Q (the next request at
    // this position, else the first request at the cluster's next position), whose copies
    // were issued when the range's last QK completed
    if (!pl.last_item(s, req)) {
      const int nreq = req < pl.end_req ? req + 1 : pl.begin_req;
      const int ns = req < pl.end_req ? s : s + pl.s_step;
      if (!stage_q_bulk(p, c, tq, nreq * p.s_q + ns, i, qbad, item + 1, true)) goto out;
    }
  }
out:
  if (qbad) atomicOr(c.status, SMLA_DEV_Q_RANGE);
  if (nan_row) atomicOr(c.status, SMLA_DEV_NAN_INPUT);
}

// ---------------------------------------------------------------------------------------
// O-CTA epilogue: writes O row `head` (a lane of this warp's tensor-memory quarter) for columns
// [32 c0, 32 c1), scaled by invl: bf16 into out (unsplit request) or into the split's partial
// (fp32, or bf16 with partials_bf16).  The tensor-memory loads of the next 32 columns are in
// flight while the current 32 are scaled, converted and stored (32-byte stores when the
// buffers are aligned for them).
__device__ void drain_o(const DecodeParams& p, uint32_t to, int head, bool no_split, int split,
                        int tok, int s, float invl, int c0, int c1) {
  const bool live = head < p.h_q;
  const bool bf16_row = no_split || p.partials_bf16;
  const size_t prow = (static_cast<size_t>(split) * p.s_q + s) * p.h_q + (live ? head : 0);
  uint8_t* dst_row =
      no_split ? reinterpret_cast<uint8_t*>(p.out + (static_cast<size_t>(tok) * p.h_q + (live ? head : 0)) * kDV)
               : reinterpret_cast<uint8_t*>(p.o_accum) + prow * kDV * (bf16_row ? 2 : 4);
  auto store_chunk = [&](const uint32_t (&o)[32], int k) {  // columns [32 k, 32 k + 32)
    if (!live) return;
    if (bf16_row) {
      uint32_t v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e)
        v[e] = pack_bf16x2(__uint_as_float(o[2 * e]) * invl, __uint_as_float(o[2 * e + 1]) * invl);
      uint8_t* d = dst_row + k * 64;
      if (p.store32) {
        st_global_v8(d, *reinterpret_cast<const uint32_t(*)[8]>(v));
        st_global_v8(d + 32, *reinterpret_cast<const uint32_t(*)[8]>(v + 8));
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) st_global_v4(d + 16 * e, v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
      }
    } else {
      uint32_t v[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(o[e]) * invl);
      uint8_t* d = dst_row + k * 128;
      if (p.store32) {
#pragma unroll
        for (int e = 0; e < 4; ++e) st_global_v8(d + 32 * e, *reinterpret_cast<const uint32_t(*)[8]>(v + 8 * e));
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) st_global_v4(d + 16 * e, v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
      }
    }
  };
  uint32_t oa[32], ob[32];
  tmem_ld16(to + c0 * 32, oa);
  tmem_ld16(to + c0 * 32 + 16, oa + 16);
#pragma unroll 1
  for (int k = c0; k < c1; k += 2) {
    tmem_wait_ld();  // columns of chunk k are in oa
    tmem_ld16(to + (k + 1) * 32, ob);
    tmem_ld16(to + (k + 1) * 32 + 16, ob + 16);
    store_chunk(oa, k);
    tmem_wait_ld();  // chunk k + 1 in ob
    if (k + 2 < c1) {
      tmem_ld16(to + (k + 2) * 32, oa);
      tmem_ld16(to + (k + 2) * 32 + 16, oa + 16);
    }
    store_chunk(ob, k + 1);
  }
}

// O-CTA epilogue of the partition's last range: the rows go through the (now unused) value-tile
// region in the 128-byte-swizzled box layout of the output's tensor map and leave by tiled TMA
// stores, so the store traffic is whole lines instead of one 32-byte piece per row and lane.
// bf16 rows (the output, or bf16 split partials): one pass of 8 boxes (64 columns x h_q rows),
// whose 32-column chunks [k0, k1) this thread converts (two warpgroups share the pass); fp32
// split partial: two passes of 8 boxes (32 columns each), all chunks.  Thread `head` converts its own row and arrives on the box's barrier
// once its part of a box is written; the store issuer (role_store_issuer) sends each box as
// soon as all rows are in, so the stores overlap the conversion.  False if a wait ran out.
constexpr uint32_t OBOX = 16384;  // 128 rows x 128 bytes
__device__ bool drain_o_tma(const DecodeParams& p, const Ctx& c, uint32_t to, int head,
                            bool bf16_rows, float invl, int k0 = 0, int k1 = 16) {
  const uint32_t stage = c.sbase + OFF_TILE;
  const bool live = head < p.h_q;
  const uint32_t row = stage + static_cast<uint32_t>(head) * 128;
  const uint32_t sw = static_cast<uint32_t>(head & 7);
  const int passes = bf16_rows ? 1 : 2;
  auto stage_chunk = [&](const uint32_t (&o)[32], int k) {  // columns [32 k, 32 k + 32)
    if (live) {
      if (bf16_rows) {  // 4 units of 8 bf16; box k / 2, units (k % 2) * 4 + e
        const uint32_t base = row + (k >> 1) * OBOX;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t u = static_cast<uint32_t>((k & 1) * 4 + e);
          st_shared_v4(base + ((u ^ sw) << 4),
                       pack_bf16x2(__uint_as_float(o[8 * e + 0]) * invl, __uint_as_float(o[8 * e + 1]) * invl),
                       pack_bf16x2(__uint_as_float(o[8 * e + 2]) * invl, __uint_as_float(o[8 * e + 3]) * invl),
                       pack_bf16x2(__uint_as_float(o[8 * e + 4]) * invl, __uint_as_float(o[8 * e + 5]) * invl),
                       pack_bf16x2(__uint_as_float(o[8 * e + 6]) * invl, __uint_as_float(o[8 * e + 7]) * invl));
        }
      } else {  // 8 units of 4 fp32; one box per chunk of the pass
        const uint32_t base = row + (k & 7) * OBOX;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          st_shared_v4(base + ((static_cast<uint32_t>(e) ^ sw) << 4),
                       __float_as_uint(__uint_as_float(o[4 * e + 0]) * invl),
                       __float_as_uint(__uint_as_float(o[4 * e + 1]) * invl),
                       __float_as_uint(__uint_as_float(o[4 * e + 2]) * invl),
                       __float_as_uint(__uint_as_float(o[4 * e + 3]) * invl));
      }
    }
    // the box is complete for this row: bf16 after its second chunk, fp32 after each chunk
    if (!bf16_rows || (k & 1) == 1) {
      fence_proxy_async_smem();
      mbar_arrive(c.bar(B_OSTAGE + (bf16_rows ? (k >> 1) : (k & 7))));
    }
  };
  for (int pass = 0; pass < passes; ++pass) {
    if (pass > 0 && !c.wait_warp(B_OFREE, 0)) return false;
    const int c0 = bf16_rows ? k0 : pass * 8, c1 = bf16_rows ? k1 : c0 + 8;
    uint32_t oa[32], ob[32];
    tmem_ld16(to + c0 * 32, oa);
    tmem_ld16(to + c0 * 32 + 16, oa + 16);
#pragma unroll 1
    for (int k = c0; k < c1; k += 2) {
      tmem_wait_ld();
      tmem_ld16(to + (k + 1) * 32, ob);
      tmem_ld16(to + (k + 1) * 32 + 16, ob + 16);
      stage_chunk(oa, k);
      tmem_wait_ld();
      if (k + 2 < c1) {
        tmem_ld16(to + (k + 2) * 32, oa);
        tmem_ld16(to + (k + 2) * 32 + 16, oa + 16);
      }
      stage_chunk(ob, k + 1);
    }
  }
  return true;
}

// O-CTA store issuer (one lane of an otherwise idle warp): for the partition's last range,
// sends each staged output box with a tiled TMA store as soon as all its rows are in, and
// waits for the stores before the CTA may leave.
__device__ void role_store_issuer(const DecodeParams& p, const Ctx& c, const Plan& pl) {
  const int req = pl.end_req, s = pl.last_s();
  const int first_slot = p.nsplits[req];
  const bool no_split = p.nsplits[req + 1] - first_slot == 1;
  const int split = req == pl.begin_req ? pl.begin_split : first_slot;
  const int row0 = no_split ? (req * p.s_q + s) * p.h_q : (split * p.s_q + s) * p.h_q;
  const uint32_t stage = c.sbase + OFF_TILE;
  const bool bf16_rows = no_split || p.partials_bf16;
  const void* map = no_split ? static_cast<const void*>(&p.out_map)
                    : bf16_rows ? static_cast<const void*>(&p.acc16_map)
                                : static_cast<const void*>(&p.acc_map);
  const int passes = bf16_rows ? 1 : 2;
  bool ok = true;
  for (int pass = 0; pass < passes && ok; ++pass) {
    for (int box = 0; box < 8; ++box) {
      if (!c.wait(B_OSTAGE + box, static_cast<uint32_t>(pass) & 1u)) {
        ok = false;
        break;
      }
      tma_store_2d(map, bf16_rows ? box * 64 : (pass * 8 + box) * 32, row0, stage + box * OBOX);
      bulk_commit_group();
    }
    if (ok && pass + 1 < passes) {
      bulk_wait_read_all();  // the staging tiles may be written again
      mbar_arrive(c.bar(B_OFREE));
    }
  }
  bulk_wait_all();  // every issued store is complete before this CTA can leave
}

// ---------------------------------------------------------------------------------------
// O-CTA correction + epilogue warpgroup: thread i owns O row i.
__device__ void role_values_epilogue(const DecodeParams& p, const Ctx& c, const Plan& pl,
                                     uint32_t tbase, int i) {
  const uint32_t to = tbase + (static_cast<uint32_t>((i >> 5) * 32) << 16);
  const bool live = i < p.h_q;
  uint32_t g = 0, item = 0;
  for (int s = pl.s0; s < p.s_q; s += pl.s_step)
  for (int req = pl.begin_req; req <= pl.end_req; ++req, ++item) {
    const int b0 = pl.first_block(req), b1 = pl.last_block(req);
    float invl = 0.f;
    for (int blk = b0; blk < b1; ++blk, ++g) {
      const uint32_t st = g % NMSG;
      if (i == 0) mbar_arrive_expect_tx(c.bar(B_MSG_FULL + st), MSG_BYTES);
      if (!c.wait_warp(B_MSG_FULL + st, (g / NMSG) & 1, true)) return;
      const uint32_t msg = c.sbase + OFF_MSG + st * MSG_STRIDE;
      const float alpha = ld_shared_f32(msg + MSG_ALPHA + 4 * i);
      if (blk == b1 - 1) invl = ld_shared_f32(msg + MSG_INVL + 4 * i);
      if (blk > b0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // the S-CTA moved this row's reference: rescale O once the previous PV has landed
        if (!c.wait_warp(B_PV_DONE + ((g - 1) % NMSG), ((g - 1) / NMSG) & 1)) return;
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
    if (pl.last_item(s, req)) {  // the value tiles are free now: stage O there for TMA stores
      // bf16 rows: this warpgroup takes columns 0-255, warps 8-11 take 256-511
      const bool bf16_rows = no_split || p.partials_bf16;
      if (!drain_o_tma(p, c, to, i, bf16_rows, invl, 0, bf16_rows ? 8 : 16)) return;
    } else {  // the dequant warps are already filling the tiles for the next range
      drain_o(p, to, i, no_split, split, tok, s, invl, 0, 16);
    }
    tc_fence_before();
    mbar_arrive(c.bar(B_O_EMPTY));
  }
}

// O-CTA warps 8-11 once their own roles are done: when the partition's last range leaves as
// bf16 rows, they convert and stage columns 256-511 of it (row = their tensor-memory lane),
// beside the epilogue warpgroup's columns 0-255.  The row's 1 / L is still in the message slot
// of the partition's last block (no message follows it).
__device__ void drain_o_second_half(const DecodeParams& p, const Ctx& c, const Plan& pl,
                                    uint32_t tbase, int row) {
  const int req = pl.end_req;
  if (!(p.nsplits[req + 1] - p.nsplits[req] == 1 || p.partials_bf16)) return;
  const uint32_t nblk = static_cast<uint32_t>(pl.blocks_per_s()) *
                        static_cast<uint32_t>((pl.s_q - 1 - pl.s0) / pl.s_step + 1);
  const uint32_t msg = c.sbase + OFF_MSG + ((nblk - 1) % NMSG) * MSG_STRIDE;
  if (!c.wait_warp(B_LAST, 0)) return;
  tc_fence_after();
  const float invl = ld_shared_f32(msg + MSG_INVL + 4 * row);
  const uint32_t to = tbase + (static_cast<uint32_t>((row >> 5) * 32) << 16);
  drain_o_tma(p, c, to, row, true, invl, 8, 16);
}

// O-CTA relay lane: once a block's PV has finished reading its message slot, hand the slot
// back to the S-CTA.
__device__ void role_relay(const Ctx& c, const Plan& pl) {
  const uint32_t peer_free = mapa(c.bar(B_MSG_FREE), 0);
  uint32_t g = 0;
  for (int s = pl.s0; s < pl.s_q; s += pl.s_step)
  for (int req = pl.begin_req; req <= pl.end_req; ++req)
    for (int blk = pl.first_block(req); blk < pl.last_block(req); ++blk, ++g) {
      const uint32_t st = g % NMSG;
      if (!c.wait(B_PV_DONE + st, (g / NMSG) & 1)) return;
      mbar_arrive_remote(peer_free + st * 8);
    }
}

// kLen: per-token top-k lengths are given (p.topk_length is read); otherwise it is not.
// kExtra: an extra cache and index list follow the main ones.  kF: the cache format.
template <bool kLen, bool kExtra, int kF>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    decode_kernel(const __grid_constant__ DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool scores = rank == 0;
  const int part = blockIdx.x >> 1;
  Ctx c;
  c.sbase = smem_u32(sm);
  c.abort_flag = reinterpret_cast<volatile uint32_t*>(sm + OFF_ABORT);
  c.status = p.status;
  c.role = 0;

  // Set-up that touches no input: it overlaps the tail of the preceding kernel (the planner)
  // when this launch is allowed to start early.
  if (threadIdx.x == 0) {
    *c.abort_flag = 0u;
    for (int b = 0; b < NSTAGE; ++b) {
      mbar_init(c.bar(B_KT_FULL + b), 256);
      mbar_init(c.bar(B_KT_EMPTY + b), 1);
      mbar_init(c.bar(B_VT_FULL + b), 256);
      mbar_init(c.bar(B_VT_EMPTY + b), 1);
    }
    for (int b = 0; b < NMSG; ++b) {
      mbar_init(c.bar(B_MSG_FREE + b), 1);
      mbar_init(c.bar(B_MSG_FULL + b), 1);
      mbar_init(c.bar(B_CORR + b), 128);
      mbar_init(c.bar(B_PV_DONE + b), 1);
      mbar_init(c.bar(B_STAGED + b), 128);
    }
    for (int b = 0; b < NSBUF; ++b) {
      mbar_init(c.bar(B_S_FULL + b), 1);
      mbar_init(c.bar(B_S_EMPTY + b), 128);
    }
    mbar_init(c.bar(B_Q_FULL), 128);
    for (int b = 0; b < 9; ++b) mbar_init(c.bar(B_QLOAD + b), 1);
    for (int b = 0; b < NSTAGE; ++b) mbar_init(c.bar(B_QREAD + b), 128);
    for (int b = 0; b < 8; ++b) mbar_init(c.bar(B_OSTAGE + b), 128);
    mbar_init(c.bar(B_OFREE), 1);
    mbar_init(c.bar(B_LAST), 1);
    mbar_init(c.bar(B_NEVER), 1);

    mbar_init(c.bar(B_O_FULL), 1);
    mbar_init(c.bar(B_O_EMPTY), 128);
    mbar_init(c.bar(B_DRAIN), 1);
    fence_mbar_init_cluster();
  }
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_TMEM_SLOT);
  if (warp == 12) {
    tmem_alloc(c.sbase + OFF_TMEM_SLOT, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote access
  const uint32_t tbase = *tslot;

  griddep_wait();  // the plan, q, kv and indices of earlier kernels are visible from here on
  const int32_t* m = p.meta + part * kMetaInts;
  Plan pl;
  pl.begin_req = m[0];
  pl.end_req = m[1];
  pl.begin_block = m[2];
  pl.end_block = m[3];
  pl.begin_split = m[4];
  pl.nb = p.nb_total;
  pl.s0 = static_cast<int>(blockIdx.y);
  pl.s_step = p.s_step;
  pl.s_q = p.s_q;
  const bool active = pl.begin_req < p.b;

  if (active) {
    const int dq = dequant_index(warp);
    c.role = (scores ? 0u : 8u) + (warp < 4 ? 1u : dq >= 0 ? 2u : warp == 12 ? 3u : 4u);
    if (warp < 4) {
      if (scores) role_softmax(p, c, pl, tbase, threadIdx.x);
      else role_values_epilogue(p, c, pl, tbase, threadIdx.x);
    } else if (dq >= 0) {
      if (scores) role_dequant<true, kLen, kExtra, kF>(p, c, pl, dq * 32 + lane);
      else role_dequant<false, kLen, kExtra, kF>(p, c, pl, dq * 32 + lane);
    } else if (warp == 12) {
      if (scores) role_mma_scores<kF == FMT_V32 ? 9 : 8>(c, pl, tbase, p.test_stall != 0);
      else role_mma_values(c, pl, tbase);
      mma_commit_warp(c.bar(B_DRAIN));  // every issued MMA has finished before TMEM is freed
      if (lane == 0) c.drain(B_DRAIN, 0);
    } else if (warp == 8) {
      if (!scores && lane == 0) role_relay(c, pl);
    } else if (warp == 4) {
      if (!scores && lane == 0) role_store_issuer(p, c, pl);
    }
    __syncwarp();
    if (!scores && warp >= 8 && warp < 12) drain_o_second_half(p, c, pl, tbase, (warp & 3) * 32 + lane);

  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 12) tmem_dealloc(tbase, 512);
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int parts, cudaStream_t stream) {
  const bool len = p.topk_length != nullptr, extra = p.extra_indices != nullptr;
  void (*kernel)(DecodeParams) = nullptr;
  if (p.kv_fmt == FMT_V32)
    kernel = extra ? (len ? decode_kernel<true, true, FMT_V32> : decode_kernel<false, true, FMT_V32>)
                   : (len ? decode_kernel<true, false, FMT_V32> : decode_kernel<false, false, FMT_V32>);
  else if (p.kv_fmt == FMT_V4 && !extra)
    kernel = len ? decode_kernel<true, false, FMT_V4> : decode_kernel<false, false, FMT_V4>;
  else if (p.kv_fmt == FMT_V41)
    kernel = extra ? (len ? decode_kernel<true, true, FMT_V41> : decode_kernel<false, true, FMT_V41>)
                   : (len ? decode_kernel<true, false, FMT_V41> : decode_kernel<false, false, FMT_V41>);
  if (kernel == nullptr) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // Programmatic stream serialisation: the kernel's set-up may overlap the preceding kernel;
  // griddepcontrol.wait inside holds every read of the plan and the inputs until it is done.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(2 * parts), static_cast<unsigned>(p.s_step), 1);
  cfg.blockDim = dim3(NTHREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace smla
