// static_workspace.cu -- mla_decode_run_static_ws: the verify decode with its split-KV
// scratch taken from a fixed device array that the library owns, for callers that
// cannot allocate device memory themselves.
//
// The array is a file-scope __device__ variable: every GPU that loads this library
// holds MLA_STATIC_WORKSPACE_BYTES of it until the process exits. In host code the
// variable's name is only a host-side stand-in, so its device address is fetched with
// cudaGetSymbolAddress, once per device and context, with that device current, and
// cached together with the context it belongs to: after a device reset (a new primary
// context) the next call looks the address up again instead of using a stale one.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "mla_decode.h"
#include "plan_format.h"
#include "status.h"

namespace mla {

size_t workspace_bytes_for(int n_part_rows);
int check_plan(const void* plan_host, size_t plan_bytes, const PlanHeader** out);

// Partial O rows and partial LSE of split units (same layout as a caller's workspace).
// Nothing in it needs to start at zero: every partial row the merge kernel reads is
// written by the fold kernel of the same call.
static __device__ __align__(256) unsigned char g_static_workspace[MLA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
static void* g_static_ws_ptr[kMaxDevices];
static CUcontext g_static_ws_ctx[kMaxDevices];
static bool g_static_ws_ready[kMaxDevices];
static std::mutex g_static_ws_mu;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// The calling thread's current context (the device's primary context once the runtime
// has initialised it), or nullptr when the driver entry point is unavailable.
static CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (CtxGetCurrentFn)f;
  });
  CUcontext c = nullptr;
  if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

// Device address of the array on the current device (looked up on first use, and again
// whenever the current context is not the one the cached address was taken in).
static int static_workspace_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(MLA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return set_error(MLA_ERR_CUDA, "device ordinal %d out of range", dev);
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lk(g_static_ws_mu);
  if (!g_static_ws_ready[dev] || g_static_ws_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || p == nullptr)
      return set_error(MLA_ERR_CUDA, "cudaGetSymbolAddress of the static workspace failed on device %d: %s", dev,
                       cudaGetErrorString(e));
    g_static_ws_ptr[dev] = p;
    g_static_ws_ctx[dev] = current_context();  // the runtime call above made the context current
    g_static_ws_ready[dev] = true;
  }
  *out = g_static_ws_ptr[dev];
  return MLA_OK;
}

}  // namespace mla

using namespace mla;

extern "C" int mla_decode_run_static_ws(const void* plan_dev, const void* plan_host, size_t plan_bytes, const void* q,
                                        const void* kv_cache, const int32_t* page_table, int page_table_stride,
                                        int num_pages, const int32_t* seq_lens, const int32_t* q_lens, float sm_scale,
                                        float kv_scale, void* out, float* lse, int32_t* status_dev, void* stream) {
  clear_error();
  const PlanHeader* h = nullptr;
  int rc = check_plan(plan_host, plan_bytes, &h);
  if (rc != MLA_OK) return rc;
  const size_t need = workspace_bytes_for(h->n_part_rows);
  if (need > (size_t)MLA_STATIC_WORKSPACE_BYTES)
    return set_error(MLA_ERR_BUFFER,
                     "this plan needs %zu bytes of split-KV scratch but the static workspace holds %zu; plan with "
                     "fewer splits (mla_plan_options.force_splits) or pass a workspace to mla_decode_run",
                     need, (size_t)MLA_STATIC_WORKSPACE_BYTES);
  void* ws = nullptr;
  if (need > 0) {
    rc = static_workspace_address(&ws);
    if (rc != MLA_OK) return rc;
  }
  return mla_decode_run(plan_dev, plan_host, plan_bytes, q, kv_cache, page_table, page_table_stride, num_pages, seq_lens,
                        q_lens, sm_scale, kv_scale, out, lse, ws, need > 0 ? (size_t)MLA_STATIC_WORKSPACE_BYTES : 0,
                        status_dev, stream);
}
