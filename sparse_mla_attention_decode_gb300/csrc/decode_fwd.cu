// Sparse MLA decode pass for sm_103a: gather + FP8 dequant + tcgen05 QK^T + online softmax +
// tcgen05 PV, split-KV aware ("FlashMLA Sparse Decode 完整计算过程详解", steps 5-15;
// "FlashMLA 与 DSA：内核、流水线和正确性边界", sections 3.1-3.5 and 4.3).
//
// One partition of the split-KV plan is run by a cluster of two CTAs (one per SM).  CTA r of
// the pair owns half of the head dimension: NoPE dims [256 r, 256 r + 256) and RoPE dims
// [32 r, 32 r + 32), i.e. 336 of the 656 bytes of every gathered row.  Per 64-slot block of
// the top-k list each CTA
//   1. gathers its byte half of every selected row with cp.async.bulk (producer warp),
//   2. dequantizes it to an fp16 tile in the UMMA 128-byte-swizzle K-major layout (one
//      warpgroup; invalid slots become zero rows),
//   3. computes its partial scores S_r = Q[:, dims_r] K[:, dims_r]^T with tcgen05 MMAs
//      (M = 128 heads, N = 64 slots; Q NoPE stays in tensor memory, Q RoPE in shared memory),
//   4. sends S_r to the peer CTA through distributed shared memory and adds the peer's
//      partial, so both CTAs hold the identical full scores S = S_0 + S_1,
//   5. runs the masked base-2 online softmax (one thread per head row) and writes P (fp16),
//   6. accumulates O[:, r-half] += P V_r with a tcgen05 MMA (M = 128, N = 256, K = 64) whose B
//      operand is the same dequantized tile read with its dim axis as the N axis.
// Tensor memory (512 columns): O half [0,256), two score buffers [256,384), Q NoPE [384,512).
//
// Keys and values are dequantized as 256 * K (the 256 is folded back into the score scale and
// into the final 1/L), so small fp32 scales stay in the fp16 normal range.
//
// Every wait is bounded: when a wait runs out the CTA records SMLA_DEV_TIMEOUT in the status
// word, every role leaves its loop, in-flight tensor-core work is drained and tensor memory
// is freed before the CTA exits.
#include <cmath>

#include "../../include/sparse_mla.h"
#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {
namespace {

constexpr int BT = 64;                 // top-k slots per block
constexpr int NRAW = 2;                // raw (gathered) stages
constexpr int NKT = 2;                 // dequantized tile stages
constexpr int RAW_ROW = 336;           // NoPE half 256 | 4 scales 16 | RoPE half 64
constexpr int RAW_STAGE = BT * RAW_ROW;
constexpr int KT_CHUNK = BT * 128;     // [64 rows x 64 dims] fp16, 128-byte swizzle
constexpr int KT_STAGE = 5 * KT_CHUNK; // 4 NoPE chunks + 1 RoPE chunk (32 of 64 dims used)
constexpr int P_STAGE = 128 * 128;     // [128 heads x 64 slots] fp16, 128-byte swizzle
constexpr int XB_BYTES = 128 * BT * 4; // peer's fp32 partial scores, one 256-byte row per head
constexpr int QR_BYTES = 128 * 128;    // [128 heads x 64] fp16, RoPE dims 0..31 used

constexpr int OFF_KT = 0;
constexpr int OFF_RAW = OFF_KT + NKT * KT_STAGE;
constexpr int OFF_P = OFF_RAW + NRAW * RAW_STAGE;
constexpr int OFF_XB = OFF_P + 2 * P_STAGE;
constexpr int OFF_QR = OFF_XB + XB_BYTES;
constexpr int OFF_MISC = OFF_QR + QR_BYTES;
static_assert(OFF_P % 1024 == 0 && OFF_XB % 1024 == 0 && OFF_QR % 1024 == 0, "alignment");

// misc region: barriers then flags
enum Bar {
  B_RAW_FULL = 0,                  // [NRAW] 32 producer lanes + tx bytes
  B_RAW_EMPTY = B_RAW_FULL + NRAW, // [NRAW] 128 dequant threads
  B_KT_FULL = B_RAW_EMPTY + NRAW,  // [NKT]  128 dequant threads
  B_KT_EMPTY = B_KT_FULL + NKT,    // [NKT]  commit after PV
  B_S_FULL = B_KT_EMPTY + NKT,     // [2]    commit after QK
  B_S_EMPTY = B_S_FULL + 2,        // [2]    128 softmax threads
  B_P_FULL = B_S_EMPTY + 2,        // [2]    128 softmax threads
  B_P_EMPTY = B_P_FULL + 2,        // [2]    commit after PV
  B_O_FULL = B_P_EMPTY + 2,        // commit after the last PV of an item
  B_O_EMPTY,                       // 128 softmax threads after the epilogue
  B_Q_FULL,                        // 128 softmax threads after Q is staged
  B_X_FULL,                        // 1 local arrive + 32 KB of st.async from the peer
  B_X_EMPTY,                       // 128 remote arrivals from the peer
  B_DRAIN,                         // commit used to drain MMAs on the way out
  NUM_BARS
};
constexpr int OFF_BARS = OFF_MISC;
constexpr int OFF_RAW_VALID = OFF_BARS + NUM_BARS * 8;         // u8 [NRAW][64]
constexpr int OFF_KT_VALID = OFF_RAW_VALID + NRAW * BT;        // u8 [NKT][64]
constexpr int OFF_TMEM_SLOT = OFF_KT_VALID + NKT * BT;         // u32
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 16;                  // u32
constexpr int MISC_BYTES = OFF_ABORT + 16 - OFF_MISC;
constexpr int SMEM_BYTES = OFF_MISC + MISC_BYTES + 1024;       // + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr int NTHREADS = 320;  // WG0 softmax | WG1 dequant | warp 8 producer | warp 9 MMA
constexpr uint32_t TM_O = 0, TM_S = 256, TM_Q = 384;
constexpr uint32_t IDESC_QK = umma_idesc_f16(128, BT, 0);
constexpr uint32_t IDESC_PV = umma_idesc_f16(128, 256, 1);
constexpr uint64_t kWaitNs = 1000000000ull;  // a wait gives up after one second

struct Ctx {
  uint32_t sbase;
  volatile uint32_t* abort_flag;
  uint32_t* status;  // [0] SMLA_DEV_* bits, [1] where the first timed-out wait was
  uint32_t role;
  __device__ uint32_t bar(int i) const { return sbase + OFF_BARS + 8u * i; }
  // Records the first wait that ran out: 0x80000000 | rank << 24 | role << 16 | barrier << 8 |
  // parity, so a stuck pipeline can be diagnosed from the status words.
  __device__ void fail(int b = 0xFF, uint32_t parity = 0) const {
    *abort_flag = 1u;
    atomicOr(status, SMLA_DEV_TIMEOUT);
    atomicCAS(status + 1, 0u, 0x80000000u | (cluster_ctarank() << 24) | (role << 16) |
                                  (static_cast<uint32_t>(b) << 8) | parity);
  }
  // Bounded wait on a local mbarrier phase; false when the wait ran out (after kWaitNs) or
  // another role already gave up.
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
  // Bounded wait that ignores the abort flag (used to drain in-flight copies and MMAs).
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

// The items of one partition: requests [begin_req, end_req], each with a block range.
struct Plan {
  int begin_req, end_req, begin_block, end_block, begin_split, nb;
  __device__ int first_block(int req) const { return req == begin_req ? begin_block : 0; }
  __device__ int last_block(int req) const { return req == end_req ? end_block : nb; }
};

__device__ __forceinline__ uint32_t f16x2_from_bf16x2(uint32_t w, uint32_t& bad) {
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xFFFF0000u);
  const uint32_t r = pack_f16x2(lo, hi);
  // fp16 infinity or NaN after conversion: the value is outside the fp16 range
  bad |= ((r & 0x7C00u) == 0x7C00u) | ((r & 0x7C000000u) == 0x7C000000u);
  return r;
}

// ---------------------------------------------------------------------------------------
// Producer warp: indices -> validity flags and bulk copies of this CTA's byte half of rows.
__device__ void producer_loop(const DecodeParams& p, const Ctx& c, const Plan& pl, int s,
                              uint32_t rank, int lane, uint32_t& g) {
  for (int req = pl.begin_req; req <= pl.end_req; ++req) {
    const int tok = req * p.s_q + s;
    const int32_t* idx_row = p.indices + static_cast<size_t>(tok) * p.topk;
    for (int blk = pl.first_block(req); blk < pl.last_block(req); ++blk) {
      const uint32_t st = g % NRAW;
      if (g >= NRAW && !c.wait(B_RAW_EMPTY + st, ((g / NRAW) - 1) & 1)) return;
      const int slot = blk * BT + lane * 2;
      const int32_t i0 = slot < p.topk ? __ldg(idx_row + slot) : -1;
      const int32_t i1 = slot + 1 < p.topk ? __ldg(idx_row + slot + 1) : -1;
      const bool v0 = i0 >= 0 && i0 < p.num_rows;
      const bool v1 = i1 >= 0 && i1 < p.num_rows;
      uint8_t* valid = reinterpret_cast<uint8_t*>(
          __cvta_shared_to_generic(c.sbase + OFF_RAW_VALID + st * BT + lane * 2));
      valid[0] = v0;
      valid[1] = v1;
      const uint32_t bar = c.bar(B_RAW_FULL + st);
      mbar_arrive_expect_tx(bar, (static_cast<uint32_t>(v0) + v1) * RAW_ROW);
      const uint32_t dst = c.sbase + OFF_RAW + st * RAW_STAGE + lane * 2 * RAW_ROW;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const bool v = k ? v1 : v0;
        if (!v) continue;
        const uint8_t* row = p.kv + static_cast<size_t>(k ? i1 : i0) * kRowBytes;
        const uint32_t d = dst + k * RAW_ROW;
        if (rank == 0) {
          bulk_g2s(d, row, 256, bar);              // NoPE dims 0..255
          bulk_g2s(d + 256, row + 512, 80, bar);   // 4 scales + RoPE dims 0..31
        } else {
          bulk_g2s(d, row + 256, 272, bar);        // NoPE dims 256..511 + 4 scales
          bulk_g2s(d + 272, row + 592, 64, bar);   // RoPE dims 32..63
        }
      }
      ++g;
    }
  }
}

__device__ void role_producer(const DecodeParams& p, const Ctx& c, const Plan& pl, int s,
                              uint32_t rank, int lane) {
  uint32_t g = 0;  // blocks whose copies were issued
  producer_loop(p, c, pl, s, rank, lane, g);
  // Whatever happened, the copies this warp issued land before the CTA may exit: wait for the
  // last issued phase of every raw stage (already complete on the normal path).
  for (uint32_t st = 0; st < NRAW; ++st) {
    if (g <= st) continue;
    const uint32_t last = st + ((g - 1 - st) / NRAW) * NRAW;
    c.drain(B_RAW_FULL + st, (last / NRAW) & 1);
  }
}

// ---------------------------------------------------------------------------------------
// Dequant warpgroup: raw stage -> fp16 tile (256 * K) in the 128-byte-swizzle K-major layout.
// Thread t handles row t / 2 and half t % 2 of this CTA's 256 NoPE dims (one 128-dim scale
// group) plus 16 of its 32 RoPE dims.
__device__ void role_dequant(const DecodeParams& p, const Ctx& c, const Plan& pl, uint32_t rank,
                             int t) {
  const int row = t >> 1, half = t & 1;
  uint32_t g = 0;
  uint32_t bad = 0;
  for (int req = pl.begin_req; req <= pl.end_req; ++req) {
    for (int blk = pl.first_block(req); blk < pl.last_block(req); ++blk, ++g) {
      const uint32_t rs = g % NRAW, ks = g % NKT;
      if (!c.wait(B_RAW_FULL + rs, (g / NRAW) & 1)) return;
      if (g >= NKT && !c.wait(B_KT_EMPTY + ks, ((g / NKT) - 1) & 1)) return;
      const uint8_t* rawv = reinterpret_cast<const uint8_t*>(
          __cvta_shared_to_generic(c.sbase + OFF_RAW_VALID + rs * BT));
      const bool valid = rawv[row] != 0;
      const uint32_t kt = c.sbase + OFF_KT + ks * KT_STAGE;
      const uint32_t raw = c.sbase + OFF_RAW + rs * RAW_STAGE + row * RAW_ROW;
      if (valid) {
        uint32_t s0, s1, s2w, s3;
        ld_shared_v4(raw + 256, s0, s1, s2w, s3);  // the 4 fp32 scales of the row
        const uint32_t sel = rank ? (half ? s3 : s2w) : (half ? s1 : s0);
        const float scale = __uint_as_float(sel) * 256.f;
        bad |= !(scale >= 6.103515625e-05f && scale <= 65504.f);
        const uint32_t s2 = pack_f16x2(scale, scale);
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {  // 16 codes per 16-byte load
          uint32_t w[4];
          ld_shared_v4(raw + half * 128 + cc * 16, w[0], w[1], w[2], w[3]);
          uint32_t o[8];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            o[2 * k] = hmul2(cvt_e4m3x2_f16x2(static_cast<uint16_t>(w[k] & 0xFFFFu)), s2);
            o[2 * k + 1] = hmul2(cvt_e4m3x2_f16x2(static_cast<uint16_t>(w[k] >> 16)), s2);
          }
          const uint32_t ld = half * 128 + cc * 16;  // local dim of the first code
          const uint32_t chunk = kt + (ld >> 6) * KT_CHUNK;
          const uint32_t c8 = (ld & 63) >> 3;
          st_shared_v4(chunk + sw128_chunk(row, c8), o[0], o[1], o[2], o[3]);
          st_shared_v4(chunk + sw128_chunk(row, c8 + 1), o[4], o[5], o[6], o[7]);
        }
        // RoPE: 16 bf16 -> 256 * value in fp16 (exact scaling by a power of two)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t w[4];
          ld_shared_v4(raw + 272 + half * 32 + cc * 16, w[0], w[1], w[2], w[3]);
          uint32_t o[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float lo = __uint_as_float(w[k] << 16) * 256.f;
            const float hi = __uint_as_float(w[k] & 0xFFFF0000u) * 256.f;
            o[k] = pack_f16x2(lo, hi);
          }
          st_shared_v4(kt + 4 * KT_CHUNK + sw128_chunk(row, half * 2 + cc), o[0], o[1], o[2], o[3]);
        }
      } else {
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const uint32_t ld = half * 128 + cc * 16;
          const uint32_t chunk = kt + (ld >> 6) * KT_CHUNK;
          const uint32_t c8 = (ld & 63) >> 3;
          st_shared_v4(chunk + sw128_chunk(row, c8), 0u, 0u, 0u, 0u);
          st_shared_v4(chunk + sw128_chunk(row, c8 + 1), 0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
          st_shared_v4(kt + 4 * KT_CHUNK + sw128_chunk(row, half * 2 + cc), 0u, 0u, 0u, 0u);
      }
      if (half == 0) {
        uint8_t* ktv = reinterpret_cast<uint8_t*>(
            __cvta_shared_to_generic(c.sbase + OFF_KT_VALID + ks * BT));
        ktv[row] = valid;
      }
      fence_proxy_async_smem();
      mbar_arrive(c.bar(B_KT_FULL + ks));
      mbar_arrive(c.bar(B_RAW_EMPTY + rs));
    }
  }
  if (bad) atomicOr(c.status, SMLA_DEV_SCALE_RANGE);
}

// ---------------------------------------------------------------------------------------
// MMA warp (one elected lane): QK^T per block into a score buffer, PV into the O half.
__device__ void role_mma(const DecodeParams& p, const Ctx& c, const Plan& pl, uint32_t tbase) {
  (void)p;
  const uint32_t qr = c.sbase + OFF_QR;
  uint32_t g = 0, item = 0;
  auto pv = [&](uint32_t gp, bool first) -> bool {
    const uint32_t sb = gp & 1, ks = gp % NKT;
    if (!c.wait(B_P_FULL + sb, (gp >> 1) & 1)) return false;
    if (first && item >= 1 && !c.wait(B_O_EMPTY, (item - 1) & 1)) return false;
    tc_fence_after();
    const uint32_t pbuf = c.sbase + OFF_P + sb * P_STAGE;
    const uint32_t kt = c.sbase + OFF_KT + ks * KT_STAGE;
#pragma unroll
    for (int kk = 0; kk < BT / 16; ++kk)
      mma_ss(tbase + TM_O, umma_desc(pbuf + kk * 32, 16, 1024, 2),
             umma_desc(kt + kk * 2048, KT_CHUNK, 1024, 2), IDESC_PV, !(first && kk == 0));
    mma_commit(c.bar(B_P_EMPTY + sb));
    mma_commit(c.bar(B_KT_EMPTY + ks));
    return true;
  };
  for (int req = pl.begin_req; req <= pl.end_req; ++req, ++item) {
    if (!c.wait(B_Q_FULL, item & 1)) return;
    const int b0 = pl.first_block(req), b1 = pl.last_block(req);
    for (int blk = b0; blk < b1; ++blk, ++g) {
      const uint32_t ks = g % NKT, sb = g & 1;
      if (!c.wait(B_KT_FULL + ks, (g / NKT) & 1)) return;
      if (g >= 2 && !c.wait(B_S_EMPTY + sb, ((g >> 1) - 1) & 1)) return;
      tc_fence_after();
      const uint32_t kt = c.sbase + OFF_KT + ks * KT_STAGE;
      const uint32_t d = tbase + TM_S + sb * BT;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk)  // NoPE: Q from tensor memory
        mma_ts(d, tbase + TM_Q + kk * 8,
               umma_desc(kt + (kk >> 2) * KT_CHUNK + (kk & 3) * 32, 16, 1024, 2), IDESC_QK, kk > 0);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)   // RoPE: Q from shared memory
        mma_ss(d, umma_desc(qr + kk * 32, 16, 1024, 2),
               umma_desc(kt + 4 * KT_CHUNK + kk * 32, 16, 1024, 2), IDESC_QK, 1);
      mma_commit(c.bar(B_S_FULL + sb));
      if (blk > b0 && !pv(g - 1, blk - 1 == b0)) return;
    }
    if (!pv(g - 1, b1 - 1 == b0)) return;
    mma_commit(c.bar(B_O_FULL));
  }
}

// ---------------------------------------------------------------------------------------
// Softmax warpgroup: thread i owns head row i (tensor-memory lane i).
struct SoftmaxState {
  float m;  // running max, base-2 units
  float l;  // running exp-sum
};

__device__ bool stage_q(const DecodeParams& p, const Ctx& c, uint32_t tq, int tok, int i,
                        uint32_t rank, uint32_t& bad) {
  const bool live = i < p.h_q;
  const uint4* src = reinterpret_cast<const uint4*>(
      p.q + (static_cast<size_t>(tok) * p.h_q + (live ? i : 0)) * kDQk);
  // NoPE dims [256 rank, 256 rank + 256) -> tensor memory columns, two fp16 per column
#pragma unroll
  for (int cc = 0; cc < 8; ++cc) {
    uint32_t w[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint4 v = live ? __ldg(src + rank * 32 + cc * 4 + k) : make_uint4(0u, 0u, 0u, 0u);
      w[4 * k + 0] = f16x2_from_bf16x2(v.x, bad);
      w[4 * k + 1] = f16x2_from_bf16x2(v.y, bad);
      w[4 * k + 2] = f16x2_from_bf16x2(v.z, bad);
      w[4 * k + 3] = f16x2_from_bf16x2(v.w, bad);
    }
    tmem_st16(tq + cc * 16, w);
  }
  // RoPE dims [32 rank, 32 rank + 32) -> shared memory, 128-byte swizzle row i
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint4 v = live ? __ldg(src + 64 + rank * 4 + k) : make_uint4(0u, 0u, 0u, 0u);
    st_shared_v4(c.sbase + OFF_QR + sw128_chunk(i, k), f16x2_from_bf16x2(v.x, bad),
                 f16x2_from_bf16x2(v.y, bad), f16x2_from_bf16x2(v.z, bad),
                 f16x2_from_bf16x2(v.w, bad));
  }
  tmem_wait_st();
  fence_proxy_async_smem();
  tc_fence_before();
  mbar_arrive(c.bar(B_Q_FULL));
  return true;
}

__device__ void role_softmax(const DecodeParams& p, const Ctx& c, const Plan& pl, int s,
                             uint32_t rank, uint32_t tbase, int i) {
  const int warp = i >> 5;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t tq = tbase + lane_base + TM_Q;
  const uint32_t ts = tbase + lane_base + TM_S;
  const uint32_t to = tbase + lane_base + TM_O;
  const uint32_t peer = rank ^ 1u;
  const uint32_t xb_local = c.sbase + OFF_XB + i * 256;
  const uint32_t xb_peer = mapa(xb_local, peer);
  const uint32_t xfull_peer = mapa(c.bar(B_X_FULL), peer);
  const uint32_t xempty_peer = mapa(c.bar(B_X_EMPTY), peer);
  uint32_t qbad = 0;
  uint32_t g = 0, item = 0;
  stage_q(p, c, tq, pl.begin_req * p.s_q + s, i, rank, qbad);
  for (int req = pl.begin_req; req <= pl.end_req; ++req, ++item) {
    const int tok = req * p.s_q + s;
    const int b0 = pl.first_block(req), b1 = pl.last_block(req);
    SoftmaxState st{-INFINITY, 0.f};
    for (int blk = b0; blk < b1; ++blk, ++g) {
      const uint32_t sb = g & 1;
      if (!c.wait(B_S_FULL + sb, (g >> 1) & 1)) goto out;
      tc_fence_after();
      uint32_t sr[BT];
#pragma unroll
      for (int k = 0; k < BT / 16; ++k) tmem_ld16(ts + sb * BT + k * 16, sr + k * 16);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(c.bar(B_S_EMPTY + sb));
      // ---- exchange partial scores with the peer CTA
      if (g >= 1 && !c.wait(B_X_EMPTY, (g - 1) & 1, true)) goto out;
      if (i == 0) mbar_arrive_expect_tx(c.bar(B_X_FULL), XB_BYTES);
#pragma unroll
      for (int k = 0; k < 16; ++k)
        st_async_v4(xb_peer + ((k ^ (i & 15)) << 4), sr[4 * k], sr[4 * k + 1], sr[4 * k + 2],
                    sr[4 * k + 3], xfull_peer);
      if (!c.wait(B_X_FULL, g & 1, true)) goto out;
      float sv[BT];
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        uint32_t a, b, cq, d;
        ld_shared_v4(xb_local + ((k ^ (i & 15)) << 4), a, b, cq, d);
        sv[4 * k + 0] = __uint_as_float(sr[4 * k + 0]) + __uint_as_float(a);
        sv[4 * k + 1] = __uint_as_float(sr[4 * k + 1]) + __uint_as_float(b);
        sv[4 * k + 2] = __uint_as_float(sr[4 * k + 2]) + __uint_as_float(cq);
        sv[4 * k + 3] = __uint_as_float(sr[4 * k + 3]) + __uint_as_float(d);
      }
      mbar_arrive_remote(xempty_peer);
      // ---- mask (validity flags of this block's slots) and scale to base-2 units
      const uint32_t ks = g % NKT;
      if (!c.wait(B_KT_FULL + ks, (g / NKT) & 1)) goto out;
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t v4[4];
        ld_shared_v4(c.sbase + OFF_KT_VALID + ks * BT + k * 16, v4[0], v4[1], v4[2], v4[3]);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const bool v = (v4[e >> 2] >> ((e & 3) * 8)) & 0xFFu;
          const int j = k * 16 + e;
          sv[j] = v ? sv[j] * p.score_scale_log2 : -INFINITY;
          mx = fmaxf(mx, sv[j]);
        }
      }
      // ---- online softmax, base 2, with a lazy rescale: the running max only moves when a
      // block's max exceeds it by more than 8 (p then stays <= 256, exact enough in fp16).
      float alpha = 1.f;
      bool rescale = false;
      if (st.m == -INFINITY) {
        st.m = mx;  // first valid block of this item (O holds only zero contributions)
      } else if (mx > st.m + 8.f) {
        alpha = ex2(st.m - mx);
        st.m = mx;
        rescale = true;
      }
      const float mref = st.m == -INFINITY ? 0.f : st.m;
      // ---- P row -> shared memory (A operand of PV), 8 slots per 16-byte chunk
      if (g >= 2 && !c.wait(B_P_EMPTY + sb, ((g >> 1) - 1) & 1)) goto out;
      const uint32_t pbuf = c.sbase + OFF_P + sb * P_STAGE;
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = ex2(sv[8 * k + 2 * e] - mref), p1 = ex2(sv[8 * k + 2 * e + 1] - mref);
          sum += p0 + p1;
          w[e] = pack_f16x2(p0, p1);
        }
        st_shared_v4(pbuf + sw128_chunk(i, k), w[0], w[1], w[2], w[3]);
      }
      st.l = st.l * alpha + sum;
      // ---- rescale the O half when this row's max moved (rare)
      if (__any_sync(0xffffffffu, rescale) && blk > b0) {
        if (!c.wait(B_P_EMPTY + ((g - 1) & 1), ((g - 1) >> 1) & 1)) goto out;
        tc_fence_after();
#pragma unroll 1
        for (int k = 0; k < 256; k += 16) {
          uint32_t o[16];
          tmem_ld16(to + k, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st16(to + k, o);
        }
        tmem_wait_st();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(c.bar(B_P_FULL + sb));
    }
    // Q of the next item can be staged now: every QK^T of this item has completed.
    if (req < pl.end_req) stage_q(p, c, tq, tok + p.s_q, i, rank, qbad);
    // ---- epilogue
    {
      if (!c.wait(B_O_FULL, item & 1)) goto out;
      tc_fence_after();
      const int first_slot = p.nsplits[req];
      const bool no_split = p.nsplits[req + 1] - first_slot == 1;
      const int split = req == pl.begin_req ? pl.begin_split : first_slot;
      const bool empty = st.l == 0.f;
      const float inv = empty ? 0.f : 1.f / (st.l * 256.f);
      const bool live = i < p.h_q;
      if (no_split) {
        __nv_bfloat16* dst = p.out + (static_cast<size_t>(tok) * p.h_q + (live ? i : 0)) * kDV + rank * 256;
#pragma unroll 1
        for (int k = 0; k < 256; k += 32) {
          uint32_t o[32];
          tmem_ld16(to + k, o);
          tmem_ld16(to + k + 16, o + 16);
          tmem_wait_ld();
          if (live) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + k);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(o[8 * e + 0]) * inv, __uint_as_float(o[8 * e + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(o[8 * e + 2]) * inv, __uint_as_float(o[8 * e + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(o[8 * e + 4]) * inv, __uint_as_float(o[8 * e + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(o[8 * e + 6]) * inv, __uint_as_float(o[8 * e + 7]) * inv);
              d4[e] = v;
            }
          }
        }
        if (rank == 0 && live)
          p.lse[(static_cast<size_t>(req) * p.h_q + i) * p.s_q + s] =
              empty ? INFINITY : (log2f(st.l) + st.m) * 0.69314718055994530942f;
      } else {
        float* dst = p.o_accum + ((static_cast<size_t>(split) * p.s_q + s) * p.h_q + (live ? i : 0)) * kDV + rank * 256;
#pragma unroll 1
        for (int k = 0; k < 256; k += 32) {
          uint32_t o[32];
          tmem_ld16(to + k, o);
          tmem_ld16(to + k + 16, o + 16);
          tmem_wait_ld();
          if (live) {
            float4* d4 = reinterpret_cast<float4*>(dst + k);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              d4[e] = make_float4(__uint_as_float(o[4 * e]) * inv, __uint_as_float(o[4 * e + 1]) * inv,
                                  __uint_as_float(o[4 * e + 2]) * inv, __uint_as_float(o[4 * e + 3]) * inv);
          }
        }
        if (rank == 0 && live)
          p.lse_accum[(static_cast<size_t>(split) * p.s_q + s) * p.h_q + i] =
              empty ? -INFINITY : log2f(st.l) + st.m;
      }
      tc_fence_before();
      mbar_arrive(c.bar(B_O_EMPTY));
    }
  }
out:
  if (qbad) atomicOr(c.status, SMLA_DEV_Q_RANGE);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NTHREADS, 1)
    decode_kernel(const DecodeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
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
    for (int b = B_RAW_FULL; b < B_RAW_FULL + NRAW; ++b) mbar_init(c.bar(b), 32);
    for (int b = B_RAW_EMPTY; b < B_RAW_EMPTY + NRAW; ++b) mbar_init(c.bar(b), 128);
    for (int b = B_KT_FULL; b < B_KT_FULL + NKT; ++b) mbar_init(c.bar(b), 128);
    for (int b = B_KT_EMPTY; b < B_KT_EMPTY + NKT; ++b) mbar_init(c.bar(b), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(c.bar(B_S_FULL + b), 1);
      mbar_init(c.bar(B_S_EMPTY + b), 128);
      mbar_init(c.bar(B_P_FULL + b), 128);
      mbar_init(c.bar(B_P_EMPTY + b), 1);
    }
    mbar_init(c.bar(B_O_FULL), 1);
    mbar_init(c.bar(B_O_EMPTY), 128);
    mbar_init(c.bar(B_Q_FULL), 128);
    mbar_init(c.bar(B_X_FULL), 1);
    mbar_init(c.bar(B_X_EMPTY), 128);
    mbar_init(c.bar(B_DRAIN), 1);
    fence_mbar_init_cluster();
  }
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + OFF_TMEM_SLOT);
  if (warp == 9 && active) {
    tmem_alloc(c.sbase + OFF_TMEM_SLOT, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before any remote access
  const uint32_t tbase = active ? *tslot : 0u;

  if (active) {
    c.role = warp < 4 ? 1u : warp < 8 ? 2u : warp == 8 ? 3u : 4u;
    if (warp < 4) {
      role_softmax(p, c, pl, s, rank, tbase, threadIdx.x);
    } else if (warp < 8) {
      role_dequant(p, c, pl, rank, threadIdx.x - 128);
    } else if (warp == 8) {
      role_producer(p, c, pl, s, rank, lane);
    } else if (lane == 0) {
      role_mma(p, c, pl, tbase);
      // drain: every MMA this thread issued has finished before tensor memory is freed
      mma_commit(c.bar(B_DRAIN));
      c.drain(B_DRAIN, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9 && active) tmem_dealloc(tbase, 512);
  cluster_sync();  // no CTA leaves while its peer may still touch its shared memory
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int parts, cudaStream_t stream) {
  static_assert(SMEM_BYTES > 0, "");
  cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(2 * parts), static_cast<unsigned>(p.s_q), 1);
  decode_kernel<<<grid, NTHREADS, SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace smla
