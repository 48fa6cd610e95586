// Split-KV partition planner, LSE-weighted combine and the empty-problem fill kernel.
#include <cmath>

#include "ptx.cuh"
#include "smla_internal.h"

namespace smla {

// ---------------------------------------------------------------------------------------
// Greedy split-KV planner ("FlashMLA Sparse Decode 完整计算过程详解", step 3; "FlashMLA 与
// DSA：内核、流水线和正确性边界", section 3.2).  The top-k list of a request is cut into
// 64-slot blocks; each request costs its blocks plus a fixed overhead of 5; every partition
// gets payload = ceil(total / parts) + 5.  Partitions are filled left to right: the rest of
// the current request goes in whole when it fits, otherwise the partition takes
// remain - 5 blocks of it and closes (the request is split there); a partition that has
// room for no further block closes as well.
//
// Output per partition: {begin_req, end_req, begin_block, end_block (exclusive),
// begin_split_idx, is_first_req_splitted, is_last_req_splitted, 0}, plus the prefix sum of
// splits per request.  Split slots are numbered in partition order, so the splits of one
// request are consecutive and prefix[req] is the slot of its first split.
//
// Every request has the same nb = ceil(topk / 64) blocks and every partition the same
// payload, so the walk of one partition depends only on the block it starts at (and on the
// number of requests left).  The warp tabulates that walk for every start block in parallel;
// lane 0 then steps through the partitions with one table lookup each (falling back to the
// exact walk where the last requests cap it), staging the table in shared memory; the warp
// copies it out with 16-byte stores and fills the split prefix: a request r has one split plus
// one more for every partition that starts inside it, so prefix[r] = r + (number of
// partitions that start inside a request before r).
struct __align__(16) PartWalk {
  int end_req, end_block;    // last request touched (relative to the first) and its end block
  int last_split, reach;     // split at the end; furthest request touched (relative)
  int next_req, next_block;  // where the next partition starts (relative request, block)
  int slots, pad;            // splits this partition contributes
};

// One partition starting at block blk of request 0, with `left_reqs` requests available
// (the greedy rule: finish the current request if it fits, then whole requests, then split).
__device__ __forceinline__ PartWalk walk_partition(int nb, long long payload, int blk,
                                                    long long left_reqs) {
  const long long cost = nb + kFixedOverhead;
  PartWalk w;
  long long remain = payload;
  const int left = nb - blk;
  if (left + kFixedOverhead <= remain) {  // the rest of the current request fits
    remain -= left + kFixedOverhead;
    long long req = 1;
    w.end_req = 0; w.end_block = nb; w.slots = 1; w.last_split = 0;
    w.next_req = 1; w.next_block = 0;
    if (remain > kFixedOverhead && req < left_reqs) {
      // Whole requests that fit: the greedy takes one while it fits and stops once at most
      // the overhead is left, which is floor(remain / cost) when a request costs more than the
      // overhead (nb >= 1) and floor((remain - 1) / cost) when it costs exactly that (nb = 0).
      const long long num = cost > kFixedOverhead ? remain : remain - 1;
      long long whole = (num < 0x7FFFFFFF && cost < 0x7FFFFFFF)
                            ? static_cast<long long>(static_cast<uint32_t>(num) /
                                                     static_cast<uint32_t>(cost))
                            : num / cost;
      if (whole > left_reqs - req) whole = left_reqs - req;
      if (whole > 0) {
        remain -= whole * cost;
        req += whole;
        w.slots += static_cast<int>(whole);
        w.end_req = static_cast<int>(req - 1); w.end_block = nb;
        w.next_req = static_cast<int>(req);
      }
      if (req < left_reqs && remain > kFixedOverhead) {  // split the next request here
        const int take = static_cast<int>(remain - kFixedOverhead);
        w.slots += 1;
        w.end_req = static_cast<int>(req); w.end_block = take; w.last_split = 1;
        w.next_req = static_cast<int>(req); w.next_block = take;
      }
    }
  } else {  // take what fits of the current request and split it here
    const int take = static_cast<int>(remain - kFixedOverhead);  // >= 1: payload > 5
    w.end_req = 0; w.end_block = blk + take; w.slots = 1; w.last_split = 1;
    w.next_req = 0; w.next_block = blk + take;
  }
  w.reach = w.next_block > 0 ? w.next_req : w.end_req;
  w.pad = 0;
  return w;
}

// levels >= 0: the jump tables of 2^k partitions (k < levels, 2^levels >= parts) fit in shared
// memory and every lane finds the start of its partitions by pointer jumping; levels < 0: lane
// 0 walks all partitions in order.
__global__ void __launch_bounds__(32) sched_kernel(int b, int s_q, int topk, int parts,
                                                   int levels, int32_t* __restrict__ meta,
                                                   int32_t* __restrict__ prefix,
                                                   uint32_t* __restrict__ status) {
  (void)s_q;
  extern __shared__ __align__(16) int32_t sched_smem[];
  const int nb = (topk + kTopkBlock - 1) / kTopkBlock;
  const int nlev = levels > 0 ? levels : 0;
  PartWalk* table = reinterpret_cast<PartWalk*>(sched_smem);                   // [nb]
  int4* jump = reinterpret_cast<int4*>(table + nb);  // [nlev][nb]: {next block, +requests, +splits}
  int4* states = jump + static_cast<size_t>(nlev) * nb;  // [parts] (levels >= 0): {req, block, slot}
  int32_t* smeta = reinterpret_cast<int32_t*>(states + (levels >= 0 ? parts : 0));  // [parts][8]
  int32_t* split_starts = smeta + static_cast<size_t>(parts) * kMetaInts;       // [parts]
  int4* m4 = reinterpret_cast<int4*>(smeta);
  __shared__ int n_starts;
  griddep_launch_dependents();  // the decode pass may start its set-up; it waits for the plan
  const int lane = threadIdx.x;
  const long long total = static_cast<long long>(b) * (nb + kFixedOverhead);
  const long long payload = (total + parts - 1) / parts + kFixedOverhead;
  constexpr long long kUncapped = 0x7FFFFFFFFFFFll;
  for (int blk = lane; blk < nb; blk += 32) {
    const PartWalk w = walk_partition(nb, payload, blk, kUncapped);
    table[blk] = w;
    if (nlev > 0) jump[blk] = make_int4(w.next_block, w.next_req, w.slots, 0);
  }
  __syncwarp();
  for (int k = 1; k < nlev; ++k) {  // jump[k] = two jumps of jump[k - 1]
    for (int blk = lane; blk < nb; blk += 32) {
      const int4 x = jump[(k - 1) * nb + blk];
      const int4 y = jump[(k - 1) * nb + x.x];
      jump[k * nb + blk] = make_int4(y.x, x.y + y.y, x.z + y.z, 0);
    }
    __syncwarp();
  }
  int first = 0;  // first partition taken by the exact walk below
  int ns = 0;
  if (levels >= 0) {
    // start of partition p = p applications of the (uncapped) one-partition walk to (0, 0, 0)
    for (int p = lane; p < parts; p += 32) {
      int req = 0, blk = 0, slot = 0;
      for (int k = 0; k < nlev; ++k)
        if ((p >> k) & 1) {
          const int4 e = jump[k * nb + blk];
          req += e.y;
          slot += e.z;
          blk = e.x;
        }
      states[p] = make_int4(req, blk, slot, 0);
    }
    __syncwarp();
    // the first partition that is empty or whose walk the last requests may cap
    first = parts;
    for (int base = 0; base < parts && first == parts; base += 32) {
      const int p = base + lane;
      bool need = false;
      if (p < parts) {
        const int4 st = states[p];
        need = st.x >= b || st.x + table[st.y].reach >= b - 1;
      }
      const unsigned m = __ballot_sync(0xffffffffu, need);
      if (m) first = base + __ffs(m) - 1;
    }
    // partitions before it, in parallel; the split starts are compacted in partition order
    for (int base = 0; base < first; base += 32) {
      const int p = base + lane;
      bool fs = false;
      int4 st = make_int4(0, 0, 0, 0);
      if (p < first) {
        st = states[p];
        const PartWalk& w = table[st.y];
        fs = st.y > 0;
        m4[2 * p] = make_int4(st.x, st.x + w.end_req, st.y, w.end_block);
        m4[2 * p + 1] = make_int4(st.z, fs ? 1 : 0, w.last_split, 0);
      }
      const unsigned m = __ballot_sync(0xffffffffu, fs);
      if (fs) split_starts[ns + __popc(m & ((1u << lane) - 1u))] = st.x;
      ns += __popc(m);
    }
  }
  __syncwarp();
  if (lane == 0) {
    int req = 0, blk = 0, slot = 0;
    if (first > 0 && first < parts) {
      const int4 st = states[first];
      req = st.x; blk = st.y; slot = st.z;
    }
    for (int part = first; part < parts; ++part) {
      if (req >= b) {
        m4[2 * part] = make_int4(b, b, 0, 0);
        m4[2 * part + 1] = make_int4(slot, 0, 0, 0);
        continue;
      }
      PartWalk w;
      if (nb > 0) w = table[blk];
      // near the end the number of requests left may cap the walk: take it exactly there
      if (nb == 0 || req + w.reach >= b - 1) w = walk_partition(nb, payload, blk, b - req);
      const int first_split = blk > 0;
      if (first_split) split_starts[ns++] = req;
      m4[2 * part] = make_int4(req, req + w.end_req, blk, w.end_block);
      m4[2 * part + 1] = make_int4(slot, first_split, w.last_split, 0);
      slot += w.slots;
      req += w.next_req;
      blk = w.next_block;
    }
    n_starts = ns;
  }
  __syncwarp();
  // The plan is computed in shared memory from the shapes alone; the plan buffer may still be
  // read by the kernels of the previous decode on this stream, so nothing is written to global
  // memory before they are done (this launch may start early).
  griddep_wait();
  if (lane == 0) {
    status[0] = 0u;
    status[1] = 0u;
  }
  const int4* src = reinterpret_cast<const int4*>(smeta);
  int4* dst = reinterpret_cast<int4*>(meta);
  for (int i = lane; i < parts * (kMetaInts / 4); i += 32) dst[i] = src[i];
  ns = n_starts;
  for (int r = lane; r <= b; r += 32) {
    int lo = 0, hi = ns;  // number of entries < r (split_starts is ascending)
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (split_starts[mid] < r) lo = mid + 1; else hi = mid;
    }
    prefix[r] = r + lo;
  }
}

cudaError_t launch_sched(int b, int s_q, int topk, int parts, int32_t* meta, int32_t* prefix,
                         uint32_t* status, cudaStream_t stream) {
  const size_t nb = static_cast<size_t>((topk + kTopkBlock - 1) / kTopkBlock);
  int levels = 0;
  while ((1 << levels) < parts) ++levels;
  const size_t base = nb * sizeof(PartWalk) + static_cast<size_t>(parts) * (kMetaInts + 1) * 4;
  const size_t fast = base + static_cast<size_t>(levels) * nb * 16 + static_cast<size_t>(parts) * 16;
  size_t smem = base;
  if (nb > 0 && fast <= 48 * 1024) {
    smem = fast;
  } else {
    levels = -1;
  }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(sched_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  // Programmatic stream serialisation: the launch overlaps the tail of the preceding kernel;
  // griddepcontrol.wait inside holds every write until that kernel is done.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, sched_kernel, b, s_q, topk, parts, levels, meta, prefix, status);
}

// ---------------------------------------------------------------------------------------
// Combine ("FlashMLA Sparse Decode 完整计算过程详解", step 16): for a (request, position,
// head) with n > 1 splits, M = max_j lse2_j, w_j = 2^(lse2_j - M),
// out = sum_j w_j o_j / sum_j w_j, lse = (M + log2 sum_j w_j) * ln 2.  One warp per head, each
// lane owns 16 of the 512 output dims (four float4 columns 128 apart, so each split row is
// read as four coalesced 512-byte segments).  Launched with programmatic stream
// serialisation: griddepcontrol.wait holds it until the decode pass has finished.
__global__ void __launch_bounds__(256) combine_kernel(const CombineParams p) {
  griddep_wait();
  const int req = blockIdx.x, s = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.z * 8 + warp;
  if (h >= p.h_q) return;
  const int first = p.nsplits[req];
  const int n = p.nsplits[req + 1] - first;
  if (n <= 1) return;  // unsplit rows were written by the decode pass
  const size_t row_stride = static_cast<size_t>(p.s_q) * p.h_q;
  const float* lse2 = p.lse_accum + (static_cast<size_t>(first) * p.s_q + s) * p.h_q + h;
  float mx = -INFINITY;
  bool nan = false;
  for (int j = lane; j < n; j += 32) {
    const float v = lse2[j * row_stride];
    mx = fmaxf(mx, v);
    nan |= v != v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __nv_bfloat16* out = p.out + ((static_cast<size_t>(req) * p.s_q + s) * p.h_q + h) * kDV;
  float* lse_out = p.lse + (static_cast<size_t>(req) * p.h_q + h) * p.s_q + s;
  if (__any_sync(0xffffffffu, nan)) {  // a split saw a NaN or +inf score: the row is NaN
    const uint32_t qnan = 0x7FC07FC0u;  // bf16 NaN pair
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint2*>(out + c * 128 + lane * 4) = make_uint2(qnan, qnan);
    if (lane == 0) *lse_out = __uint_as_float(0x7FC00000u);
    return;
  }
  if (mx == -INFINITY) {  // every split empty: the defined output of a row with no valid slot
#pragma unroll
    for (int c = 0; c < 4; ++c)
      *reinterpret_cast<uint2*>(out + c * 128 + lane * 4) = make_uint2(0u, 0u);
    if (lane == 0) *lse_out = INFINITY;
    return;
  }
  float4 acc[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  const size_t row0 = (static_cast<size_t>(first) * p.s_q + s) * p.h_q + h;
  for (int j = 0; j < n; ++j) {
    const float w = exp2f(lse2[j * row_stride] - mx);
    wsum += w;
    const size_t row = row0 + j * row_stride;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float4 v;
      if (p.partials_bf16) {  // 4 bf16 per lane: the high half of an fp32 is the bf16 value
        const uint2 u = *reinterpret_cast<const uint2*>(
            reinterpret_cast<const __nv_bfloat16*>(p.o_accum) + row * kDV + c * 128 + lane * 4);
        v = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                        __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
      } else {
        v = *reinterpret_cast<const float4*>(p.o_accum + row * kDV + c * 128 + lane * 4);
      }
      acc[c].x += w * v.x; acc[c].y += w * v.y; acc[c].z += w * v.z; acc[c].w += w * v.w;
    }
  }
  // an attention sink adds one zero-value key of score attn_sink[h] to the merged row
  const float sink = p.attn_sink != nullptr
                         ? exp2f(fmaf(__ldg(p.attn_sink + h), 1.4426950408889634f, -mx))
                         : 0.f;
  const float inv = 1.f / (wsum + sink);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint2 pk;
    pk.x = pack_bf16x2(acc[c].x * inv, acc[c].y * inv);
    pk.y = pack_bf16x2(acc[c].z * inv, acc[c].w * inv);
    *reinterpret_cast<uint2*>(out + c * 128 + lane * 4) = pk;
  }
  if (lane == 0) *lse_out = (mx + log2f(wsum)) * 0.69314718055994530942f;
}

cudaError_t launch_combine(const CombineParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.b), static_cast<unsigned>(p.s_q),
                     static_cast<unsigned>((p.h_q + 7) / 8));
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

// ---------------------------------------------------------------------------------------
// topk == 0: no slot at all, so every row takes the defined empty output (out = 0,
// lse = +inf).
__global__ void fill_empty_kernel(__nv_bfloat16* out, float* lse, int64_t n_out16,
                                  int64_t n_lse) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t k = i; k < n_out16; k += stride)
    reinterpret_cast<uint4*>(out)[k] = make_uint4(0u, 0u, 0u, 0u);
  for (int64_t k = i; k < n_lse; k += stride) lse[k] = INFINITY;
}

cudaError_t launch_fill_empty(__nv_bfloat16* out, float* lse, int64_t rows_o, int64_t n_lse,
                              cudaStream_t stream) {
  const int64_t n_out16 = rows_o * kDV * 2 / 16;
  int64_t work = n_out16 > n_lse ? n_out16 : n_lse;
  int blocks = static_cast<int>((work + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  fill_empty_kernel<<<blocks, 256, 0, stream>>>(out, lse, n_out16, n_lse);
  return cudaGetLastError();
}

}  // namespace smla
