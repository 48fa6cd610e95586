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
// Every request has the same ceil(topk / 64) blocks, so one partition's walk is a few lines of
// arithmetic: finish the current request if it fits, then as many whole requests as the
// remaining capacity holds, then split the next one.  Lane 0 walks the partitions in order
// into shared memory (one thread's global stores would issue one by one); the warp then copies
// the table out with 16-byte stores and fills the split prefix: a request r has one split
// plus one more for every partition that starts inside it, so prefix[r] = r + (number of
// partitions that start inside a request before r).
__global__ void __launch_bounds__(32) sched_kernel(int b, int s_q, int topk, int parts,
                                                   int32_t* __restrict__ meta,
                                                   int32_t* __restrict__ prefix,
                                                   uint32_t* __restrict__ status) {
  (void)s_q;
  extern __shared__ __align__(16) int32_t sched_smem[];
  int32_t* smeta = sched_smem;                                       // [parts][8]
  int32_t* split_starts = sched_smem + static_cast<size_t>(parts) * kMetaInts;  // [parts]
  __shared__ int n_starts;
  griddep_launch_dependents();  // the decode pass may start its set-up; it waits for the plan
  const int lane = threadIdx.x;
  if (lane == 0) {
    status[0] = 0u;
    status[1] = 0u;
    const int nb = (topk + kTopkBlock - 1) / kTopkBlock;
    const long long cost = nb + kFixedOverhead;  // one whole request
    const long long total = static_cast<long long>(b) * cost;
    const long long payload = (total + parts - 1) / parts + kFixedOverhead;
    int req = 0, blk = 0, slot = 0, ns = 0;
    for (int part = 0; part < parts; ++part) {
      int32_t* m = smeta + static_cast<size_t>(part) * kMetaInts;
      if (req >= b) {
        m[0] = b; m[1] = b; m[2] = 0; m[3] = 0; m[4] = slot; m[5] = 0; m[6] = 0; m[7] = 0;
        continue;
      }
      long long remain = payload;
      const int begin_req = req, begin_block = blk, begin_slot = slot;
      const int first_split = blk > 0;
      if (first_split) split_starts[ns++] = req;
      int end_req = req, end_block = blk, last_split = 0;
      const int left = nb - blk;
      if (left + kFixedOverhead <= remain) {  // the rest of the current request fits
        remain -= left + kFixedOverhead;
        ++slot;
        end_req = req; end_block = nb;
        ++req; blk = 0;
        if (remain > kFixedOverhead && req < b) {
          long long whole = (remain < 0x7FFFFFFF && cost < 0x7FFFFFFF)  // whole requests that fit
                                ? static_cast<long long>(static_cast<uint32_t>(remain) /
                                                         static_cast<uint32_t>(cost))
                                : remain / cost;
          if (whole > b - req) whole = b - req;
          if (whole > 0) {
            remain -= whole * cost;
            slot += static_cast<int>(whole);
            req += static_cast<int>(whole);
            end_req = req - 1; end_block = nb;
          }
          if (req < b && remain > kFixedOverhead) {  // split the next request here
            const int take = static_cast<int>(remain - kFixedOverhead);
            ++slot;
            blk = take;
            end_req = req; end_block = take; last_split = 1;
          }
        }
      } else {  // take what fits of the current request and split it here
        const long long take = remain - kFixedOverhead;
        if (take > 0) {
          ++slot;
          blk += static_cast<int>(take);
          end_req = req; end_block = blk; last_split = 1;
        }
      }
      m[0] = begin_req; m[1] = end_req; m[2] = begin_block; m[3] = end_block;
      m[4] = begin_slot; m[5] = first_split; m[6] = last_split; m[7] = 0;
    }
    n_starts = ns;
  }
  __syncwarp();
  const int4* src = reinterpret_cast<const int4*>(smeta);
  int4* dst = reinterpret_cast<int4*>(meta);
  for (int i = lane; i < parts * (kMetaInts / 4); i += 32) dst[i] = src[i];
  const int ns = n_starts;
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
  const size_t smem = static_cast<size_t>(parts) * (kMetaInts + 1) * sizeof(int32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(sched_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  sched_kernel<<<1, 32, smem, stream>>>(b, s_q, topk, parts, meta, prefix, status);
  return cudaGetLastError();
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
  for (int j = lane; j < n; j += 32) mx = fmaxf(mx, lse2[j * row_stride]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  __nv_bfloat16* out = p.out + ((static_cast<size_t>(req) * p.s_q + s) * p.h_q + h) * kDV;
  float* lse_out = p.lse + (static_cast<size_t>(req) * p.h_q + h) * p.s_q + s;
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
  const float* o = p.o_accum + ((static_cast<size_t>(first) * p.s_q + s) * p.h_q + h) * kDV;
  for (int j = 0; j < n; ++j) {
    const float w = exp2f(lse2[j * row_stride] - mx);
    wsum += w;
    const float* oj = o + j * row_stride * kDV;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 v = *reinterpret_cast<const float4*>(oj + c * 128 + lane * 4);
      acc[c].x += w * v.x; acc[c].y += w * v.y; acc[c].z += w * v.z; acc[c].w += w * v.w;
    }
  }
  const float inv = 1.f / wsum;
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
