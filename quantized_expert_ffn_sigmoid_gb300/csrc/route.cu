// Router kernels: fp32 logits x . Wr^T, then the sigmoid noaux_tc group
// top-k selection ("Colibri (colibrì): GLM-5.2 local inference on 25 GB of
// RAM", "How it works (validated core mechanics)"; DeepSeek-V3 group
// limiting as named on that page).
#include "colimoe_internal.cuh"
#include "select_cta.cuh"

namespace colimoe {

// Logits for larger T: 64x64 output tiles, K steps of 16, 4x4 per thread;
// blockIdx.z picks one of gridDim.z K ranges of `kper` elements, whose
// partial logits go to part[z][T][E].  The next step's operands are loaded
// into registers while the current step is multiplied.
__global__ void __launch_bounds__(256) route_logits_tiled(const float* __restrict__ x, int T, int H,
                                                          const float* __restrict__ wr, int E,
                                                          float* __restrict__ part, int kper) {
  __shared__ float xs[16][64 + 4];
  __shared__ float ws[16][64 + 4];
  const int t0 = blockIdx.y * 64, e0 = blockIdx.x * 64;
  const int kb = blockIdx.z * kper, ke = kb + kper;
  const int tid = threadIdx.x;
  const int ty = tid / 16, tx = tid % 16;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  // loader: row = tid / 4 (0..63), k4 = tid % 4 (float4 index within 16)
  const int lr = tid / 4, lk = (tid % 4) * 4;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  auto ldx = [&](int k0) {
    return t0 + lr < T ? __ldg(reinterpret_cast<const float4*>(x + (size_t)(t0 + lr) * H + k0 + lk)) : zero;
  };
  auto ldw = [&](int k0) {
    return e0 + lr < E ? __ldg(reinterpret_cast<const float4*>(wr + (size_t)(e0 + lr) * H + k0 + lk)) : zero;
  };
  float4 xv = ldx(kb), wv = ldw(kb);
  for (int k0 = kb; k0 < ke; k0 += 16) {
    xs[lk + 0][lr] = xv.x; xs[lk + 1][lr] = xv.y; xs[lk + 2][lr] = xv.z; xs[lk + 3][lr] = xv.w;
    ws[lk + 0][lr] = wv.x; ws[lk + 1][lr] = wv.y; ws[lk + 2][lr] = wv.z; ws[lk + 3][lr] = wv.w;
    __syncthreads();
    if (k0 + 16 < ke) {
      xv = ldx(k0 + 16);
      wv = ldw(k0 + 16);
    }
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* out = part + (size_t)blockIdx.z * T * E;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) out[(size_t)t * E + e] = acc[i][j];
    }
  }
}

// One CTA per position: the logits are the K ranges' partials summed in range
// order, then the CTA-wide selection.
__global__ void __launch_bounds__(256) route_select(const float* __restrict__ part, int splits, int T,
                                                   int E, int G, int topk_group, int k, float rsf,
                                                   const float* __restrict__ bias,
                                                   int32_t* __restrict__ topk_idx,
                                                   float* __restrict__ topk_w,
                                                   uint32_t* __restrict__ status) {
  extern __shared__ __align__(16) float sm_sel[];  // [3E + 32] selection scratch, then [E] logits
  __shared__ SelShared s_sel;
  const int t = blockIdx.x;
  const float bias_reg = (int)threadIdx.x < E ? __ldg(bias + threadIdx.x) : 0.f;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the partials come from the previous kernel
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  float* lg = sm_sel + 3 * E + 32;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float l = 0.f;
#pragma unroll 8
    for (int s = 0; s < splits; ++s) l += __ldcg(part + ((size_t)s * T + t) * E + e);
    lg[e] = l;
  }
  __syncthreads();
  select_position_cta(lg, t, E, G, topk_group, k, rsf, bias, bias_reg, topk_idx, topk_w, status, sm_sel, s_sel, true);
}

__device__ __forceinline__ void pdl_wait_r() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger_r() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Router logits for T <= 8: every CTA writes partial logits for 8 experts x
// one K split.  With one position (fuse_select) the last CTA to finish (a
// counter in the workspace header, reset by that CTA) sums the splits and
// runs the CTA-wide selection; with more, route_select (one CTA per
// position) follows.
constexpr int RF_PRE = 8;  // router weight float4 per lane loaded before the dependency wait

__global__ void __launch_bounds__(256) route_fused(const float* __restrict__ x, int T, int H,
                                                  const float* __restrict__ wr, int E, int splits,
                                                  float* __restrict__ part, int G, int topk_group, int k,
                                                  float rsf, const float* __restrict__ bias,
                                                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                                  uint32_t* __restrict__ status, uint32_t* __restrict__ counter,
                                                  int fuse_select) {
  extern __shared__ __align__(16) float sm_rf[];
  __shared__ uint32_t s_last;
  __shared__ SelShared s_sel;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  const int s = blockIdx.y;
  // Weights (router rows, bias) are never written by this library's kernels,
  // so they are loaded before the grid dependency wait; x may be the output
  // of the kernel this launch overlaps and is read only after it.
  const float bias_reg = (int)threadIdx.x < E ? __ldg(bias + threadIdx.x) : 0.f;
  const int n4 = H / 4 / splits;
  const float4* w4 = reinterpret_cast<const float4*>(wr + (size_t)(e < E ? e : 0) * H) + (size_t)s * n4;
  float4 wv[RF_PRE];
#pragma unroll
  for (int m = 0; m < RF_PRE; ++m)
    if (e < E && lane + 32 * m < n4) wv[m] = __ldg(w4 + lane + 32 * m);
  pdl_wait_r();
  pdl_trigger_r();
  if (e < E) {
    float acc[ROUTE_GEMV_MAX_T];
#pragma unroll
    for (int t = 0; t < ROUTE_GEMV_MAX_T; ++t) acc[t] = 0.f;
    auto fma4 = [&](const float4& w, int i) {
#pragma unroll
      for (int t = 0; t < ROUTE_GEMV_MAX_T; ++t) {
        if (t < T) {
          const float4 v = __ldg(reinterpret_cast<const float4*>(x + (size_t)t * H) + (size_t)s * n4 + i);
          acc[t] = fmaf(w.x, v.x, acc[t]);
          acc[t] = fmaf(w.y, v.y, acc[t]);
          acc[t] = fmaf(w.z, v.z, acc[t]);
          acc[t] = fmaf(w.w, v.w, acc[t]);
        }
      }
    };
#pragma unroll
    for (int m = 0; m < RF_PRE; ++m)
      if (lane + 32 * m < n4) fma4(wv[m], lane + 32 * m);
    for (int i = lane + 32 * RF_PRE; i < n4; i += 32) fma4(__ldg(w4 + i), i);
#pragma unroll
    for (int t = 0; t < ROUTE_GEMV_MAX_T; ++t) {
      if (t < T) {
        const float v = warp_sum(acc[t]);
        if (lane == 0) part[((size_t)s * T + t) * E + e] = v;
      }
    }
  }
  if (!fuse_select) return;  // route_select follows
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const uint32_t total = gridDim.x * gridDim.y;
    const uint32_t old = atomicAdd(counter, 1u);
    s_last = (old == total - 1) ? 1u : 0u;
    if (s_last) {
      __threadfence();
      *counter = 0u;  // ready for the next call
    }
  }
  __syncthreads();
  if (!s_last) return;
  // logits = sum of the K-split partials in split order, all loads in flight
  float* s_logit = sm_rf + (size_t)3 * E + 32;  // [T][E]
  for (int i = threadIdx.x; i < T * E; i += blockDim.x) {
    const int t = i / E, e = i % E;
    float v[GEMV_SPLITS];
#pragma unroll
    for (int s = 0; s < GEMV_SPLITS; ++s) v[s] = s < splits ? __ldcg(part + ((size_t)s * T + t) * E + e) : 0.f;
    float l = 0.f;
#pragma unroll
    for (int s = 0; s < GEMV_SPLITS; ++s) if (s < splits) l += v[s];
    s_logit[i] = l;
  }
  __syncthreads();
  for (int t = 0; t < T; ++t)
    select_position_cta(s_logit + (size_t)t * E, t, E, G, topk_group, k, rsf, bias, bias_reg, topk_idx, topk_w, status,
               sm_rf, s_sel, true);
}

// route_select over `splits` partial-logit ranges, one CTA per position
// (programmatic dependent launch: it waits for the kernel that wrote them)
static cudaError_t launch_select(const float* part, int splits, int T, int E, int G, int topk_group, int k,
                                 float rsf, const float* bias, int32_t* topk_idx, float* topk_w, uint32_t* status,
                                 cudaStream_t st) {
  const size_t smem_s = ((size_t)4 * E + 32) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(route_select, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_s);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem_s;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_select, part, splits, T, E, G, topk_group, k, rsf, bias, topk_idx, topk_w,
                            status);
}

cudaError_t launch_route(const float* x, int T, int H, const float* wr, int E, int G, int topk_group, int k,
                         float rsf, const float* bias, int32_t* topk_idx, float* topk_w, float* part,
                         uint32_t* status, uint32_t* counter, cudaStream_t st) {
  if (T <= ROUTE_GEMV_MAX_T) {
    const size_t smem_f = ((size_t)(3 + T) * E + 32) * sizeof(float);
    int splits = GEMV_SPLITS;
    while (splits > 1 && (H / 4) % (splits * 32)) splits /= 2;
    cudaError_t e = cudaFuncSetAttribute(route_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_f);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((E + 7) / 8, splits);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = smem_f;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // one position: the last CTA selects; more: one CTA per position after
    e = cudaLaunchKernelEx(&cfg, route_fused, x, T, H, wr, E, splits, part, G, topk_group, k, rsf, bias, topk_idx,
                           topk_w, status, counter, T == 1 ? 1 : 0);
    if (e != cudaSuccess || T == 1) return e;
    return launch_select(part, splits, T, E, G, topk_group, k, rsf, bias, topk_idx, topk_w, status, st);
  }
  const int ks = route_ksplits(T, H, E);
  dim3 grid((E + 63) / 64, (T + 63) / 64, ks);
  route_logits_tiled<<<grid, 256, 0, st>>>(x, T, H, wr, E, part, H / ks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_select(part, ks, T, E, G, topk_group, k, rsf, bias, topk_idx, topk_w, status, st);
}

}  // namespace colimoe
