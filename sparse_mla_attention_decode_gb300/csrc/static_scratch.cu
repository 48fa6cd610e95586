// sparse_mla_decode_static: the plan -> decode -> combine sequence run on scratch memory that
// the library owns, for callers that cannot hand out device memory of their own.
//
// The scratch is one file-scope __device__ array, so it comes into existence when the CUDA
// module of this file is loaded and is never allocated, resized or freed by a call.  The
// first call on a device (with that device current) looks up the array's device address
// with cudaGetSymbolAddress, which can load the module; later calls on that device reuse
// the cached address.  The three steps themselves are the library's public entry points,
// called with pointers into the array.
#include <cstdint>
#include <mutex>

#include "../../include/sparse_mla.h"
#include "smla_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[SMLA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void* g_scratch_addr[kMaxDevices] = {};  // device address of g_static_scratch, per device

// Device address of the scratch array on the current device (looked up once per device).
smla_status scratch_address(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SMLA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return SMLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> guard(g_lock);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return SMLA_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return SMLA_OK;
}

}  // namespace

extern "C" smla_status sparse_mla_decode_static(const smla_dims* dims, int num_sms,
                                                const void* q, const void* kv_cache,
                                                const int32_t* indices, float sm_scale,
                                                void* out, float* lse, void* stream) {
  size_t sched_bytes = 0, accum_bytes = 0;
  smla_status st = sparse_mla_workspace_size(dims, num_sms, &sched_bytes, &accum_bytes);
  if (st != SMLA_OK) return st;
  // [split partials | plan], each 256-byte aligned; checked before any CUDA call
  const size_t plan_off = (accum_bytes + 255) & ~static_cast<size_t>(255);
  if (plan_off > SMLA_STATIC_SCRATCH_BYTES ||
      sched_bytes > SMLA_STATIC_SCRATCH_BYTES - plan_off)
    return SMLA_ERR_WORKSPACE;
  void* base = nullptr;
  if ((st = scratch_address(&base)) != SMLA_OK) return st;
  unsigned char* scratch = static_cast<unsigned char*>(base);
  void* accum = scratch;
  void* plan = scratch + plan_off;
  // The planner rewrites the whole plan and zeroes its status words on every call; the split
  // partials need no initial value (each slot is written by the decode pass before the
  // combine reads it), so nothing left by an earlier call is ever read.
  if ((st = sparse_mla_sched_meta(dims, num_sms, plan, sched_bytes, stream)) != SMLA_OK)
    return st;
  if ((st = sparse_mla_decode_fwd(dims, num_sms, q, kv_cache, indices, sm_scale, plan, accum,
                                  accum_bytes, out, lse, stream)) != SMLA_OK)
    return st;
  return sparse_mla_combine(dims, num_sms, plan, accum, accum_bytes, out, lse, stream);
}
