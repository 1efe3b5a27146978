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
//      (c descending, id ascending); ranks < top_k are selected
//      (warp per (32 candidates, kept group), counts summed in shared memory)
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
  int asc[MAX_TOPK];  // position of sel[] among the selected ids in ascending order
};

// All threads of the CTA call this (it contains barriers).  `logits` holds
// the position's E logits and `scratch` 3*E + 32 words, both in shared memory,
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
      sh.asc[tid] = -1;
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
      r += (o > my) | ((o == my) & (h < tid));
    }
    if (r < topk_group) sh.kg[r] = tid;
  }
  __syncthreads();
  // 4. expert ranks among the kept groups' experts: warp task = (chunk of 32
  // candidates, kept group q), counting the group's experts that precede each
  int* s_rank = reinterpret_cast<int*>(scratch + 2 * E);
  unsigned* s_bits = reinterpret_cast<unsigned*>(scratch + 3 * E);
  const int nc = topk_group * gsz;
  for (int i = tid; i < nc; i += nt) s_rank[i] = 0;
  for (int i = tid; i < (E + 31) / 32; i += nt) s_bits[i] = 0u;
  __syncthreads();
  const int nch = (nc + 31) / 32;
  for (int task = warp; task < nch * topk_group; task += nw) {
    const int i = (task / topk_group) * 32 + lane, q = task % topk_group;
    const bool act = i < nc;
    const int e = act ? sh.kg[i / gsz] * gsz + i % gsz : 0;
    const float v = s_c[e];
    const int base = sh.kg[q] * gsz;
    int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
    if ((gsz & 3) == 0) {
      const float4* c4 = reinterpret_cast<const float4*>(s_c + base);
#pragma unroll 4
      for (int u = 0; u < gsz / 4; ++u) {
        const float4 w = c4[u];
        const int j = base + 4 * u;
        r0 += (w.x > v) | ((w.x == v) & (j < e));
        r1 += (w.y > v) | ((w.y == v) & (j + 1 < e));
        r2 += (w.z > v) | ((w.z == v) & (j + 2 < e));
        r3 += (w.w > v) | ((w.w == v) & (j + 3 < e));
      }
    } else {
      for (int u = 0; u < gsz; ++u) {
        const float w = s_c[base + u];
        r0 += (w > v) | ((w == v) & (base + u < e));
      }
    }
    const int r = r0 + r1 + r2 + r3;
    if (act && r) atomicAdd(&s_rank[i], r);
  }
  __syncthreads();
  for (int i = tid; i < nc; i += nt) {
    const int r = s_rank[i];
    if (r < k) {
      const int e = sh.kg[i / gsz] * gsz + i % gsz;
      sh.sel[r] = e;
      atomicOr(&s_bits[e >> 5], 1u << (e & 31));
    }
  }
  __syncthreads();
  // 5. weights from the unbiased affinities, summed in rank order
  if (tid < k) {
    const int e = sh.sel[tid];
    int a = __popc(s_bits[e >> 5] & ((1u << (e & 31)) - 1u));
    for (int i = 0; i < (e >> 5); ++i) a += __popc(s_bits[i]);
    sh.asc[tid] = a;
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

// Fast path for groups of exactly 32 experts with at most one group per warp
// and topk_group * min(k, 32) <= 32 (the GLM / DeepSeek-V3 shape: 256
// experts in 8 groups, 4 kept, top 8).  The warp of group g computes its
// experts' scores; every lane then scans the group's 32 scores from shared
// memory (16-byte broadcast loads, no shuffles) for both the group score
// (sum of the two largest) and its own rank inside the group.  The global
// top k lies within the union of the kept groups' top min(k, 32), which one
// warp ranks the same way.  Same result, ties and weight summation order as
// select_cta.
__device__ __forceinline__ bool select_fast_ok(int E, int G, int topk_group, int k, int n_warps) {
  // (E >= 64 so that the E + 160 scratch words fit in the 3 E + 32 given)
  return E == 32 * G && E >= 64 && G <= n_warps && topk_group * (k < 32 ? k : 32) <= 32;
}

__device__ __forceinline__ bool select_fast(const float* logits, int t, int E, int G, int topk_group, int k,
                                            float rsf, const float* __restrict__ bias, float bias_reg,
                                            int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                            uint32_t* __restrict__ status, float* scratch, SelShared& sh,
                                            bool write_out) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int kc = k < 32 ? k : 32;
  float* s_c = scratch;                                     // [E] biased scores
  float* c_v = scratch + E;                                 // [32] candidates: biased score
  int* c_e = reinterpret_cast<int*>(scratch + E + 32);      //      expert id
  float* c_s = scratch + E + 64;                            //      affinity
  int* r_e = reinterpret_cast<int*>(scratch + E + 96);      // [32] selected id by output slot
  float* r_s = scratch + E + 128;                           // [32] its affinity
  const int e = warp * 32 + lane;
  float s = 0.f, cv = -INFINITY;
  int bad = 0, r_in = 32;
  if (warp < G) {
    const float l = logits[e];
    const float b = E <= nt ? bias_reg : __ldg(bias + e);
    bad = !isfinite(l) || !isfinite(b);
    s = __fdiv_rn(1.0f, 1.0f + expf(-l));
    cv = s + b;
    s_c[e] = cv;
    __syncwarp();
    // one pass over the group: its two largest scores and this expert's rank
    const float4* g4 = reinterpret_cast<const float4*>(s_c + warp * 32);
    float b1 = -INFINITY, b2 = -INFINITY;
    int ra = 0, rb = 0;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float4 q = g4[u];
      const float vv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float v = vv[i];
        const int j = 4 * u + i;
        b2 = fmaxf(b2, fminf(b1, v));
        b1 = fmaxf(b1, v);
        const int gt = (v > cv) | ((v == cv) & (j < lane));
        if (i & 1) rb += gt; else ra += gt;
      }
    }
    r_in = ra + rb;
    if (lane == 0) sh.gs[warp] = b1 + b2;
  }
  if (__syncthreads_or(bad)) {
    if (tid == 0) atomicOr(status, COLI_STATUS_NONFINITE);
    if (tid < k) {
      sh.sel[tid] = -1;
      sh.w[tid] = 0.f;
      sh.asc[tid] = -1;
      if (write_out) {
        topk_idx[(size_t)t * k + tid] = -1;
        topk_w[(size_t)t * k + tid] = 0.f;
      }
    }
    __syncthreads();
    return false;
  }
  if (warp < G && r_in < kc) {
    const float my = sh.gs[warp];
    int gr = 0;
    for (int h = 0; h < G; ++h) {
      const float o = sh.gs[h];
      gr += (o > my) | ((o == my) & (h < warp));
    }
    if (gr < topk_group) {
      c_v[gr * kc + r_in] = cv;
      c_e[gr * kc + r_in] = e;
      c_s[gr * kc + r_in] = s;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const int nc = topk_group * kc;
    const bool act = lane < nc;
    const float v = act ? c_v[lane] : -INFINITY;
    const int ce = act ? c_e[lane] : 0x7fffffff;
    int ra = 0, rb = 0;
    const float4* v4 = reinterpret_cast<const float4*>(c_v);
    const int4* e4 = reinterpret_cast<const int4*>(c_e);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (4 * u < nc) {
        const float4 q = v4[u];
        const int4 qe = e4[u];
        ra += (q.x > v) | ((q.x == v) & (qe.x < ce));
        rb += (4 * u + 1 < nc) & ((q.y > v) | ((q.y == v) & (qe.y < ce)));
        ra += (4 * u + 2 < nc) & ((q.z > v) | ((q.z == v) & (qe.z < ce)));
        rb += (4 * u + 3 < nc) & ((q.w > v) | ((q.w == v) & (qe.w < ce)));
      }
    }
    const int r = ra + rb;
    if (act && r < k) {
      r_e[r] = ce;
      r_s[r] = c_s[lane];
    }
    __syncwarp();
    if (lane < k) {
      const int my_e = r_e[lane];
      float tot = 0.f;
      int a = 0;
      for (int q = 0; q < k; ++q) {
        tot += r_s[q];
        a += r_e[q] < my_e;
      }
      const float w = tot > 0.f ? __fmul_rn(__fdiv_rn(r_s[lane], tot), rsf) : 0.f;
      sh.sel[lane] = my_e;
      sh.asc[lane] = a;
      sh.w[lane] = w;
      if (write_out) {
        topk_idx[(size_t)t * k + lane] = my_e;
        topk_w[(size_t)t * k + lane] = w;
      }
    }
  }
  __syncthreads();
  return true;
}

// The selection of one position by the fastest applicable path.
__device__ __forceinline__ bool select_position_cta(const float* logits, int t, int E, int G, int topk_group, int k,
                                                    float rsf, const float* __restrict__ bias, float bias_reg,
                                                    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                                                    uint32_t* __restrict__ status, float* scratch, SelShared& sh,
                                                    bool write_out) {
  if (select_fast_ok(E, G, topk_group, k, blockDim.x / 32))
    return select_fast(logits, t, E, G, topk_group, k, rsf, bias, bias_reg, topk_idx, topk_w, status, scratch, sh,
                       write_out);
  return select_cta(logits, t, E, G, topk_group, k, rsf, bias, bias_reg, topk_idx, topk_w, status, scratch, sh,
                    write_out);
}

}  // namespace colimoe
