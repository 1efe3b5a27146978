// coli_moe_stack_forward: a decode step through a stack of MoE layers with
// the hidden state resident on the device between layers (JustVugg/colibri
// README, "Never wait for the disk twice": the residual stream stays on the
// GPU across layers).  Each layer is one coli_moe_layer call; between layers
// one small kernel forms the next layer's input.
#include "colimoe_internal.cuh"

namespace {

using namespace colimoe;

// xs_next = (xs + (add_output ? y : 0)) + residual, elementwise in fp32.
// Launched with programmatic dependent launch: it may start while the
// layer's last kernel finishes, and reads y, xs and residual only after
// that kernel has completed.  It lets the next layer's kernels launch at
// once; they read their input only after this kernel has completed.
__global__ void __launch_bounds__(256) residual_kernel(const float4* __restrict__ x, const float4* __restrict__ y,
                                                       const float4* __restrict__ r, float4* __restrict__ out,
                                                       long long n4, int add_output) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    float4 v = x[i];
    if (add_output) {
      const float4 a = y[i];
      v.x = __fadd_rn(v.x, a.x); v.y = __fadd_rn(v.y, a.y); v.z = __fadd_rn(v.z, a.z); v.w = __fadd_rn(v.w, a.w);
    }
    if (r) {
      const float4 d = r[i];
      v.x = __fadd_rn(v.x, d.x); v.y = __fadd_rn(v.y, d.y); v.z = __fadd_rn(v.z, d.z); v.w = __fadd_rn(v.w, d.w);
    }
    out[i] = v;
  }
}

cudaError_t launch_residual(const float* x, const float* y, const float* r, float* out, long long n, int add_output,
                            cudaStream_t st) {
  const long long n4 = n / 4;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (n4 + 255) / 256;
  const long long cap = 2LL * (sms > 0 ? sms : 132);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, residual_kernel, reinterpret_cast<const float4*>(x),
                            reinterpret_cast<const float4*>(y), reinterpret_cast<const float4*>(r),
                            reinterpret_cast<float4*>(out), n4, add_output);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int coli_moe_stack_forward(const coli_moe_stack_layer* layers, int32_t n_layers, int32_t T, float* xs,
                                      const float* residual, int32_t add_output, int32_t* topk_idx, float* topk_w,
                                      float* y, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!layers || n_layers < 0 || T < 0 || (add_output != 0 && add_output != 1)) return COLI_EINVAL;
  if (n_layers == 0 || T == 0) return COLI_OK;
  if (!xs || !topk_idx || !topk_w || !y || !ws) return COLI_EINVAL;
  if (!aligned16(xs) || !aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(y) || !aligned16(ws) ||
      (residual && !aligned16(residual)))
    return COLI_EALIGN;
  const int H = layers[0].cfg.hidden, k = layers[0].cfg.top_k;
  // every layer is checked before anything is enqueued
  for (int l = 0; l < n_layers; ++l) {
    const coli_moe_stack_layer& Ly = layers[l];
    if (Ly.cfg.hidden != H || Ly.cfg.top_k != k) return COLI_EINVAL;
    const size_t need = coli_moe_workspace_size(&Ly.cfg, T);
    if (need == 0) return COLI_EINVAL;
    if (ws_bytes < need) return COLI_EWORKSPACE;
    const coli_moe_weights& w = Ly.weights;
    const bool shared = Ly.cfg.n_shared > 0 && Ly.cfg.ep_rank == 0;
    if (!Ly.router_w || !Ly.corr_bias || !w.experts || !w.expert_scales) return COLI_EINVAL;
    if (shared && (!w.shared || !w.shared_scales)) return COLI_EINVAL;
    if (!aligned16(Ly.router_w) || !aligned16(Ly.corr_bias) || !aligned16(w.experts) || !aligned16(w.expert_scales))
      return COLI_EALIGN;
    if (shared && (!aligned16(w.shared) || !aligned16(w.shared_scales))) return COLI_EALIGN;
  }
  // H % 128 == 0 (checked with the config), so every [T][H] slice keeps the
  // 16-byte alignment of its base
  const size_t act = (size_t)T * H, sel = (size_t)T * k;
  for (int l = 0; l < n_layers; ++l) {
    const coli_moe_stack_layer& Ly = layers[l];
    float* x_l = xs + (size_t)l * act;
    float* y_l = y + (size_t)l * act;
    int rc = coli_moe_layer(&Ly.cfg, &Ly.weights, x_l, T, Ly.router_w, Ly.corr_bias, topk_idx + (size_t)l * sel,
                            topk_w + (size_t)l * sel, y_l, ws, ws_bytes, stream);
    if (rc != COLI_OK) return rc;
    if (launch_residual(x_l, y_l, residual ? residual + (size_t)l * act : nullptr, x_l + act, (long long)act,
                        add_output, stream) != cudaSuccess)
      return COLI_ECUDA;
  }
  return COLI_OK;
}
