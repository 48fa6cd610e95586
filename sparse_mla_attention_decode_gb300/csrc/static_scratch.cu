// sparse_mla_decode_static: the plan -> decode -> combine sequence run on scratch memory that
// the library owns, for callers that cannot hand out device memory of their own.
//
// The scratch is one file-scope __device__ array, so it comes into existence when the CUDA
// module of this file is loaded and is never allocated, resized or freed by a call.  The
// first call on a device (with that device current) looks up the array's device address
// with cudaGetSymbolAddress, which can load the module; later calls on that device reuse
// the cached address for as long as the same CUDA context is current.  A device reset (or a
// primary-context release and re-creation) makes a new context, whose module may place the
// array elsewhere, so the cache is keyed on the context's unique id and the address is
// looked up again when the id changes.  The three steps themselves are the library's public
// entry points, called with pointers into the array.
#include <cstdint>
#include <mutex>

#include "../../include/sparse_mla.h"
#include "smla_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[SMLA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct CachedAddress {
  unsigned long long ctx_id;  // unique id of the context the address belongs to (0: none)
  void* addr;
};
std::mutex g_lock;
CachedAddress g_scratch[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// cuCtxGetCurrent and cuCtxGetId from the driver, looked up once (no link-time dependency on
// libcuda).  Null if the driver does not provide them.
void driver_ctx_fns(CtxGetCurrentFn* get_current, CtxGetIdFn* get_id) {
  static std::once_flag once;
  static CtxGetCurrentFn cur = nullptr;
  static CtxGetIdFn id = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      cur = reinterpret_cast<CtxGetCurrentFn>(f);
    else
      cudaGetLastError();
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      id = reinterpret_cast<CtxGetIdFn>(f);
    else
      cudaGetLastError();
  });
  *get_current = cur;
  *get_id = id;
}

// Unique id of the current context, 0 if there is none yet or it cannot be queried.
unsigned long long current_ctx_id() {
  CtxGetCurrentFn get_current;
  CtxGetIdFn get_id;
  driver_ctx_fns(&get_current, &get_id);
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device, for the current context.
smla_status scratch_address(void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SMLA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return SMLA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> guard(g_lock);
  const unsigned long long id = current_ctx_id();
  CachedAddress& c = g_scratch[dev];
  if (id == 0 || c.ctx_id != id || c.addr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return SMLA_ERR_CUDA;
    }
    // the lookup made the runtime's context current if none was: key the cache on it (an id
    // of 0, when the driver cannot report one, caches nothing and looks up every call)
    c.ctx_id = current_ctx_id();
    c.addr = p;
  }
  *addr = c.addr;
  return SMLA_OK;
}

// Offsets of the plan and of the split partials inside the scratch; SMLA_ERR_WORKSPACE when the
// problem does not fit (checked before any CUDA call).
smla_status scratch_layout(const smla_dims* dims, int num_sms, size_t* sched_bytes,
                           size_t* accum_bytes, size_t* plan_off) {
  smla_status st = sparse_mla_workspace_size(dims, num_sms, sched_bytes, accum_bytes);
  if (st != SMLA_OK) return st;
  // [split partials | plan], each 256-byte aligned
  *plan_off = (*accum_bytes + 255) & ~static_cast<size_t>(255);
  if (*plan_off > SMLA_STATIC_SCRATCH_BYTES || *sched_bytes > SMLA_STATIC_SCRATCH_BYTES - *plan_off)
    return SMLA_ERR_WORKSPACE;
  return SMLA_OK;
}

}  // namespace

extern "C" smla_status sparse_mla_decode_static(const smla_dims* dims, int num_sms,
                                                const void* q, const void* kv_cache,
                                                const int32_t* indices, float sm_scale,
                                                void* out, float* lse, void* stream) {
  size_t sched_bytes = 0, accum_bytes = 0, plan_off = 0;
  smla_status st = scratch_layout(dims, num_sms, &sched_bytes, &accum_bytes, &plan_off);
  if (st != SMLA_OK) return st;
  void* base = nullptr;
  if ((st = scratch_address(&base)) != SMLA_OK) return st;
  unsigned char* scratch = static_cast<unsigned char*>(base);
  void* accum = accum_bytes > 0 ? scratch : nullptr;
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

extern "C" smla_status sparse_mla_static_read_status(const smla_dims* dims, int num_sms,
                                                     int* code, void* stream) {
  size_t sched_bytes = 0, accum_bytes = 0, plan_off = 0;
  smla_status st = scratch_layout(dims, num_sms, &sched_bytes, &accum_bytes, &plan_off);
  if (st != SMLA_OK) return st;
  if (!code) return SMLA_ERR_INVALID_ARG;
  void* base = nullptr;
  if ((st = scratch_address(&base)) != SMLA_OK) return st;
  return sparse_mla_read_device_status(dims, num_sms, static_cast<unsigned char*>(base) + plan_off,
                                       code, stream);
}
