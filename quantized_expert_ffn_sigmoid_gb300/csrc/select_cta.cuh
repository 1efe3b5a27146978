// CTA-wide sigmoid noaux_tc selection of one position ("Colibri (colibrì):
// GLM-5.2 local inference on 25 GB of RAM", "How it works (validated core
// mechanics)"; DeepSeek-V3 group limiting as named on that page).
//
// Every step is a rank computation instead of a chain of arg-max rounds, so
// the whole CTA works in parallel and the critical path is a handful of
// barriers:
//   1. affinity s = sigmoid(logit), ranking score c = s + bias      (thread/expert)
//   2. group score = sum of the two largest c of the group          (warp/group)
//   3. keep the topk_group groups of highest score, lower id first  (thread/group)
//   4. rank every expert of a kept group among all kept experts by
//      (c descending, id ascending); ranks < top_k are selected     (thread/expert)
//   5. weights: s of the selected renormalised over the selection,
//      times routed_scaling_factor                                  (thread/slot)
// Output slot r holds the expert of rank r, which is the order the repeated
// arg-max of the definition produces.
#pragma once
#include "colimoe_internal.cuh"

namespace colimoe {

struct SelShared {
  float gs[MAX_GROUPS];
  int kg[MAX_GROUPS];
  int sel[MAX_TOPK];  // selected expert of each output slot (-1: none)
  float w[MAX_TOPK];  // its routing weight
};

// All threads of the CTA call this (it contains barriers).  `logits` holds
// the position's E logits and `scratch` 2*E floats, both in shared memory,
// 16-byte aligned, E a multiple of 4 when E/G is.  `bias_reg` is bias[tid]
// preloaded by the caller when E <= blockDim.x (else unused).  The result is
// left in sh.sel / sh.w and, when `write_out`, stored to topk_idx / topk_w.
// Returns false (slots -1 / 0, status flag set) for a non-finite logit or
// bias.
__device__ __forceinline__ bool select_cta(const float* logits, int t, int E, int G, int topk_group, int k,
                                           float rsf, const float* __restrict__ bias, float bias_reg,
                                           int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                           uint32_t* __restrict__ status, float* scratch, SelShared& sh,
                                           bool write_out) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  float* s_s = scratch;
  float* s_c = scratch + E;
  int bad = 0;
  for (int e = tid; e < E; e += nt) {
    const float l = logits[e];
    const float b = E <= nt ? bias_reg : __ldg(bias + e);
    bad |= !isfinite(l) || !isfinite(b);
    const float s = __fdiv_rn(1.0f, 1.0f + expf(-l));
    s_s[e] = s;
    s_c[e] = s + b;
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicOr(status, COLI_STATUS_NONFINITE);
    if (tid < k) {
      sh.sel[tid] = -1;
      sh.w[tid] = 0.f;
      if (write_out) {
        topk_idx[(size_t)t * k + tid] = -1;
        topk_w[(size_t)t * k + tid] = 0.f;
      }
    }
    __syncthreads();
    return false;
  }
  const int gsz = E / G;
  // 2. group scores: (largest, second largest) per lane, merged across the warp
  for (int g = warp; g < G; g += nw) {
    float b1 = -INFINITY, b2 = -INFINITY;
    for (int i = lane; i < gsz; i += 32) {
      const float v = s_c[g * gsz + i];
      if (v > b1) { b2 = b1; b1 = v; } else if (v > b2) { b2 = v; }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float o1 = __shfl_xor_sync(0xffffffffu, b1, o);
      const float o2 = __shfl_xor_sync(0xffffffffu, b2, o);
      const float n2 = fmaxf(fminf(b1, o1), fmaxf(b2, o2));
      b1 = fmaxf(b1, o1);
      b2 = n2;
    }
    if (lane == 0) sh.gs[g] = gsz >= 2 ? b1 + b2 : b1;
  }
  __syncthreads();
  // 3. group ranks
  if (tid < G) {
    const float my = sh.gs[tid];
    int r = 0;
    for (int h = 0; h < G; ++h) {
      const float o = sh.gs[h];
      r += (o > my) || (o == my && h < tid);
    }
    if (r < topk_group) sh.kg[r] = tid;
  }
  __syncthreads();
  // 4. expert ranks among the kept groups' experts
  const int nc = topk_group * gsz;
  for (int i = tid; i < nc; i += nt) {
    const int e = sh.kg[i / gsz] * gsz + i % gsz;
    const float v = s_c[e];
    int r = 0;
    for (int q = 0; q < topk_group; ++q) {
      const int base = sh.kg[q] * gsz;
      if ((gsz & 3) == 0) {
        const float4* c4 = reinterpret_cast<const float4*>(s_c + base);
#pragma unroll 4
        for (int u = 0; u < gsz / 4; ++u) {
          const float4 w = c4[u];
          const int j = base + 4 * u;
          r += (w.x > v) || (w.x == v && j < e);
          r += (w.y > v) || (w.y == v && j + 1 < e);
          r += (w.z > v) || (w.z == v && j + 2 < e);
          r += (w.w > v) || (w.w == v && j + 3 < e);
        }
      } else {
        for (int u = 0; u < gsz; ++u) {
          const float w = s_c[base + u];
          r += (w > v) || (w == v && base + u < e);
        }
      }
    }
    if (r < k) sh.sel[r] = e;
  }
  __syncthreads();
  // 5. weights from the unbiased affinities, summed in rank order
  if (tid < k) {
    const int e = sh.sel[tid];
    float tot = 0.f;
    for (int r = 0; r < k; ++r) tot += s_s[sh.sel[r]];
    const float w = tot > 0.f ? __fmul_rn(__fdiv_rn(s_s[e], tot), rsf) : 0.f;
    if (write_out) {
      topk_idx[(size_t)t * k + tid] = e;
      topk_w[(size_t)t * k + tid] = w;
    }
    sh.w[tid] = w;
  }
  __syncthreads();  // scratch and sh are reused by the next position
  return true;
}

}  // namespace colimoe
