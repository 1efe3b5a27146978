// coli_moe_forward_static: the expert layer (coli_moe_forward) for callers
// that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: a plain C or FFI
// host that links only this library and owns no device allocator, or a
// runtime that keeps the whole device-memory budget to itself and forbids
// stray cudaMalloc calls (cudaMalloc can synchronise the device and fails
// once a fixed budget is spent).  For them this entry point takes its scratch
// from one file-scope device array that the library carries in its module:
// every GPU that loads the library holds COLI_STATIC_WS_BYTES of device memory
// for it until the process exits.  Nothing here calls cudaMalloc, cudaFree or
// any allocating routine.
#include <mutex>
#include "colimoe_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;

// The scratch.  Zero-initialised at module load; in host code its name is
// only a host-side stand-in, so the kernels get the device address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) uint8_t g_static_ws[COLI_STATIC_WS_BYTES];

std::mutex g_mu;
void* g_ptr[kMaxDevices] = {};

// Device address of g_static_ws on the current device, looked up once per
// device (with that device current) and cached.
int static_ws_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return COLI_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return COLI_EUNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return COLI_ECUDA;
    g_ptr[dev] = p;
  }
  *out = g_ptr[dev];
  return COLI_OK;
}

}  // namespace

extern "C" int coli_moe_forward_static(const coli_moe_cfg* cfg, const coli_moe_weights* weights,
                                       const float* x, int32_t T, const int32_t* topk_idx,
                                       const float* topk_w, float* y, cudaStream_t stream) {
  if (T < 0) return COLI_EINVAL;
  const size_t need = coli_moe_workspace_size(cfg, T);
  if (need == 0) return COLI_EINVAL;                      // invalid config
  if (need > (size_t)COLI_STATIC_WS_BYTES) return COLI_EWORKSPACE;  // T beyond the static limit
  void* ws = nullptr;
  const int rc = static_ws_ptr(&ws);
  if (rc != COLI_OK) return rc;
  // The tables and intermediates that coli_moe_forward keeps in its
  // workspace are rewritten by every call, and the fused single-position
  // kernel's counters come in two sets that each call clears for the next
  // one, so the previous call's contents never leak into the next one (the
  // scratch starts zeroed, like a workspace after coli_moe_workspace_init).
  return coli_moe_forward(cfg, weights, x, T, topk_idx, topk_w, y, ws, (size_t)COLI_STATIC_WS_BYTES, stream);
}
