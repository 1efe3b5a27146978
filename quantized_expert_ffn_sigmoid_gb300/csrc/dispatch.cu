// Q8_0 activation quantisation and the batch-union dispatch tables.
//
// Q8_0: colibrì v1.0 README, "What's implemented" (integer-dot kernels on
// Q8_0-style int8 activations, blocks of 32 with one fp32 scale).
// Batch-union: same section ("Batch-union MoE": each distinct expert of a
// batch is read once and applied to every position routed to it).
#include "colimoe_internal.cuh"

namespace colimoe {

// Public quantiser: one warp per 32-block, natural element order.
__global__ void __launch_bounds__(256) quantize_act_kernel(const float* __restrict__ x, long long nblk,
                                                           int8_t* __restrict__ q, float* __restrict__ d) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long b = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); b < nblk; b += warps) {
    float v = x[b * QB + lane];
    float dd;
    bool bad;
    int c = q8_0_lane(v, &dd, &bad);
    q[b * QB + lane] = (int8_t)c;
    if (lane == 0) d[b] = dd;
  }
}

// Exclusive scan of one int per thread over a 1024-thread block; returns the
// prefix and writes the block total to *total (all threads).
__device__ int block_scan_excl(int v, int* scratch /*32 ints*/, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) scratch[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = scratch[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    scratch[lane] = wi - w;       // exclusive warp offsets
    if (lane == 31) scratch[32] = wi;
  }
  __syncthreads();
  int res = scratch[warp] + inc - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}


// Block 0 builds the union tables (1024 threads); blocks >= 1 quantise x.
//
// Tables (canonical, checked bit-exactly against the reference):
//   entries = distinct valid routed ids ascending, then the shared experts;
//   pairs of a routed entry in ascending (t, j); pair slots consecutive in
//   entry order; per entry the number of gate/up and down work items.
template <int BITS>
__global__ void __launch_bounds__(PREP_THREADS) prep_kernel(PrepParams P) {
  const coli_moe_cfg& c = P.cfg;
  const Layout& L = P.L;
  uint8_t* ws = P.ws;
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status);
  const int H = c.hidden, E = c.n_experts, k = c.top_k, T = P.T, ns = c.n_shared;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (blockIdx.x > 0) {
    // ---- Q8_0 of x, one warp per 32-block; int4 layout permuted within 8s
    const int nb = H / QB;
    const long long nblk = (long long)T * nb;
    const long long warps = (long long)(gridDim.x - 1) * (PREP_THREADS / 32);
    int8_t* qx = reinterpret_cast<int8_t*>(ws + L.qx);
    float* dx = reinterpret_cast<float*>(ws + L.dx);
    int32_t* xs = reinterpret_cast<int32_t*>(ws + L.xs);
    bool anybad = false;
    for (long long b = (long long)(blockIdx.x - 1) * (PREP_THREADS / 32) + warp; b < nblk; b += warps) {
      float v = P.x[b * QB + lane];
      float dd;
      bool bad;
      int q = q8_0_lane(v, &dd, &bad);
      anybad |= bad;
      int pos = act_pos(lane, BITS);
      qx[b * QB + pos] = (int8_t)q;
      int sum = warp_sum_i(q);
      if (lane == 0) {
        dx[b] = dd;
        xs[b] = code_bias(BITS) * sum;
      }
    }
    if (anybad && lane == 0) atomicOr(status, COLI_STATUS_NONFINITE);
    return;
  }

  // ---- block 0: tables
  extern __shared__ int sm_prep[];
  int* cnt = sm_prep;                    // [E]
  int* run = cnt + E;                    // [E]
  int* eoff = run + E;                   // [E] first pair slot of expert e
  int* eent = eoff + E;                  // [E] entry index of expert e
  int* scratch = eent + E;               // [64]
  uint16_t* wcnt = reinterpret_cast<uint16_t*>(scratch + 64);  // [32][E]

  uint32_t* ctr = reinterpret_cast<uint32_t*>(ws + L.counters);
  int32_t* hdr = reinterpret_cast<int32_t*>(ws + L.hdr);
  int32_t* ent_expert = reinterpret_cast<int32_t*>(ws + L.ent_expert);
  int32_t* ent_count = reinterpret_cast<int32_t*>(ws + L.ent_count);
  int32_t* ent_offset = reinterpret_cast<int32_t*>(ws + L.ent_offset);
  int32_t* ent_item_a = reinterpret_cast<int32_t*>(ws + L.ent_item_a);
  int32_t* ent_item_b = reinterpret_cast<int32_t*>(ws + L.ent_item_b);
  int32_t* pair_token = reinterpret_cast<int32_t*>(ws + L.pair_token);
  int32_t* pair_j = reinterpret_cast<int32_t*>(ws + L.pair_j);
  int32_t* slot = reinterpret_cast<int32_t*>(ws + L.slot);

  for (int i = tid; i < 1 + L.n_ent_max + L.n_tiles; i += PREP_THREADS) ctr[i] = 0u;
  for (int e = tid; e < E; e += PREP_THREADS) { cnt[e] = 0; run[e] = 0; }
  __syncthreads();
  const int npair = T * k;
  bool badidx = false;
  for (int p = tid; p < npair; p += PREP_THREADS) {
    int e = P.idx[p];
    if (e >= 0 && e < E) {
      if (ep_owned(c, e)) atomicAdd(&cnt[e], 1);   // another shard's expert: skipped
    } else if (e != -1) {
      badidx = true;
    }
  }
  if (__any_sync(0xffffffffu, badidx) && lane == 0) atomicOr(status, COLI_STATUS_BADIDX);
  __syncthreads();
  // per-expert first slot and entry number (E <= 1024: one expert per thread)
  int total_pairs, n_uniq;
  {
    int v = tid < E ? cnt[tid] : 0;
    int off = block_scan_excl(v, scratch, &total_pairs);
    int ent = block_scan_excl(v > 0 ? 1 : 0, scratch, &n_uniq);
    if (tid < E) {
      eoff[tid] = off;
      eent[tid] = ent;
      if (v > 0) {
        ent_expert[ent] = tid;
        ent_count[ent] = v;
        ent_offset[ent] = off;
      }
    }
  }
  const int n_ent = n_uniq + ns;
  for (int s = tid; s < ns; s += PREP_THREADS) {
    ent_expert[n_uniq + s] = E + s;
    ent_count[n_uniq + s] = T;
    ent_offset[n_uniq + s] = total_pairs + s * T;
  }
  if (tid == 0) ent_offset[n_ent] = total_pairs + ns * T;
  for (int i = tid; i < ns * T; i += PREP_THREADS) {
    pair_token[total_pairs + i] = i % T;
    pair_j[total_pairs + i] = -1;
  }
  __syncthreads();

  // ranks inside each routed entry in (t, j) order, chunk by chunk
  for (int base = 0; base < npair; base += PREP_THREADS) {
    for (int e = lane; e < E; e += 32) wcnt[warp * E + e] = 0;
    __syncwarp();
    const int p = base + tid;
    const int e = p < npair ? P.idx[p] : -1;
    const bool valid = e >= 0 && e < E && ep_owned(c, e);
    const unsigned same = __match_any_sync(0xffffffffu, valid ? e : -1);
    const int lrank = __popc(same & ((1u << lane) - 1u));
    if (valid && lrank == 0) wcnt[warp * E + e] = (uint16_t)__popc(same);
    __syncthreads();
    if (p < npair) {
      if (valid) {
        int pre = 0;
        for (int w = 0; w < warp; ++w) pre += wcnt[w * E + e];
        const int sl = eoff[e] + run[e] + pre + lrank;
        pair_token[sl] = p / k;
        pair_j[sl] = p % k;
        slot[p] = sl;
      } else {
        slot[p] = -1;
      }
    }
    __syncthreads();
    for (int ee = tid; ee < E; ee += PREP_THREADS) {
      int add = 0;
      for (int w = 0; w < PREP_THREADS / 32; ++w) add += wcnt[w * E + ee];
      run[ee] += add;
    }
    __syncthreads();
  }

  // work items per entry: (rows / tile) x ceil(count / TG)
  int na_run = 0, nb_run = 0, bt_run = 0;
  for (int base = 0; base < n_ent; base += PREP_THREADS) {
    const int u = base + tid;
    int ia = 0, ib = 0, ntg = 0;
    if (u < n_ent) {
      const int cntu = u < n_uniq ? cnt[ent_expert[u]] : T;
      const int iu = u < n_uniq ? c.inter : c.shared_inter;
      ntg = (cntu + TG - 1) / TG;
      ia = (iu / RA) * ntg;
      ib = (H / RB) * ntg;
    }
    int ta, tb, tt;
    int pa = block_scan_excl(ia, scratch, &ta);
    int pb = block_scan_excl(ib, scratch, &tb);
    block_scan_excl(ntg, scratch, &tt);
    if (u < n_ent) {
      ent_item_a[u] = na_run + pa;
      ent_item_b[u] = nb_run + pb;
    }
    na_run += ta;
    nb_run += tb;
    bt_run += tt;
  }
  if (tid == 0) {
    ent_item_a[n_ent] = na_run;
    ent_item_b[n_ent] = nb_run;
    hdr[H_NENT] = n_ent;
    hdr[H_NUNIQ] = n_uniq;
    hdr[H_NA] = na_run;
    hdr[H_NB] = nb_run;
    hdr[H_BTARGET] = bt_run;
    hdr[H_NPAIRS] = total_pairs + ns * T;
  }
}

__device__ __forceinline__ void pdl_wait_d() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger_d() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Dispatch for calls of at most GEMV_MAX_T positions (<= 256 pairs): every
// warp quantises x blocks, then warp 0 of block 0 builds the same canonical
// tables as prep_kernel with warp-level counting (ranks by comparing the
// <= 256 keys (expert, pair) in shared memory).  Both x and the routing may
// come from the kernel this launch overlaps, so everything waits for it.
template <int BITS>
__global__ void __launch_bounds__(256) prep_small_kernel(PrepParams P) {
  const coli_moe_cfg& c = P.cfg;
  const Layout& L = P.L;
  uint8_t* ws = P.ws;
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status);
  const int H = c.hidden, E = c.n_experts, k = c.top_k, T = P.T, ns = c.n_shared;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait_d();
  pdl_trigger_d();
  {
    const int nb = H / QB;
    const int nblk = T * nb;
    const int warps = gridDim.x * 8;
    int8_t* qx = reinterpret_cast<int8_t*>(ws + L.qx);
    float* dx = reinterpret_cast<float*>(ws + L.dx);
    int32_t* xs = reinterpret_cast<int32_t*>(ws + L.xs);
    bool anybad = false;
    for (int b = blockIdx.x * 8 + warp; b < nblk; b += warps) {
      const float v = P.x[(size_t)b * QB + lane];
      float dd;
      bool bad;
      const int q = q8_0_lane(v, &dd, &bad);
      anybad |= bad;
      qx[(size_t)b * QB + act_pos(lane, BITS)] = (int8_t)q;
      const int sum = warp_sum_i(q);
      if (lane == 0) {
        dx[b] = dd;
        xs[b] = code_bias(BITS) * sum;
      }
    }
    if (anybad && lane == 0) atomicOr(status, COLI_STATUS_NONFINITE);
  }
  if (blockIdx.x != 0 || warp != 0) return;

  __shared__ int key[GEMV_MAX_T * MAX_TOPK];
  __shared__ unsigned char first[GEMV_MAX_T * MAX_TOPK];
  __shared__ int s_entcnt[GEMV_MAX_T * MAX_TOPK + MAX_SHARED];
  uint32_t* ctr = reinterpret_cast<uint32_t*>(ws + L.counters);
  int32_t* hdr = reinterpret_cast<int32_t*>(ws + L.hdr);
  int32_t* ent_expert = reinterpret_cast<int32_t*>(ws + L.ent_expert);
  int32_t* ent_count = reinterpret_cast<int32_t*>(ws + L.ent_count);
  int32_t* ent_offset = reinterpret_cast<int32_t*>(ws + L.ent_offset);
  int32_t* ent_item_a = reinterpret_cast<int32_t*>(ws + L.ent_item_a);
  int32_t* ent_item_b = reinterpret_cast<int32_t*>(ws + L.ent_item_b);
  int32_t* pair_token = reinterpret_cast<int32_t*>(ws + L.pair_token);
  int32_t* pair_j = reinterpret_cast<int32_t*>(ws + L.pair_j);
  int32_t* slot = reinterpret_cast<int32_t*>(ws + L.slot);
  for (int i = lane; i < 1 + L.n_ent_max + L.n_tiles; i += 32) ctr[i] = 0u;

  const int npair = T * k;  // <= 256
  bool badidx = false;
  for (int p = lane; p < npair; p += 32) {
    const int e = P.idx[p];
    const bool inrange = e >= 0 && e < E;
    if (!inrange && e != -1) badidx = true;
    const bool valid = inrange && ep_owned(c, e);   // another shard's expert: skipped
    key[p] = valid ? (e << 8) | p : 0x7fffffff;
  }
  if (__any_sync(0xffffffffu, badidx) && lane == 0) atomicOr(status, COLI_STATUS_BADIDX);
  __syncwarp();
  // rank = sorted position of (expert, pair); first = no earlier pair of that expert
  int nvalid = 0, nfirst = 0;
  for (int p = lane; p < npair; p += 32) {
    const int kp = key[p];
    int rank = 0, before = 0;
    for (int q = 0; q < npair; ++q) {
      const int kq = key[q];
      rank += kq < kp;
      before += (kq >> 8) == (kp >> 8) && kq < kp;
    }
    if (kp != 0x7fffffff) {
      slot[p] = rank;
      pair_token[rank] = p / k;
      pair_j[rank] = p % k;
    } else {
      slot[p] = -1;
    }
    first[p] = kp != 0x7fffffff && before == 0;
  }
  for (int p = lane; p < npair; p += 32) {
    nvalid += key[p] != 0x7fffffff;
  }
  __syncwarp();
  for (int p = lane; p < npair; p += 32) nfirst += first[p];
  nvalid = warp_sum_i(nvalid);
  const int n_uniq = warp_sum_i(nfirst);
  for (int p = lane; p < npair; p += 32) {
    if (!first[p]) continue;
    const int kp = key[p], e = kp >> 8;
    int ent = 0, cnt = 0, off = 0;
    for (int q = 0; q < npair; ++q) {
      const int kq = key[q];
      ent += first[q] && (kq >> 8) < e;
      cnt += (kq >> 8) == e;
      off += kq < kp;
    }
    ent_expert[ent] = e;
    ent_count[ent] = cnt;
    ent_offset[ent] = off;
    s_entcnt[ent] = cnt;
  }
  for (int s = lane; s < ns; s += 32) {
    ent_expert[n_uniq + s] = E + s;
    ent_count[n_uniq + s] = T;
    ent_offset[n_uniq + s] = nvalid + s * T;
    s_entcnt[n_uniq + s] = T;
  }
  for (int i = lane; i < ns * T; i += 32) {
    pair_token[nvalid + i] = i % T;
    pair_j[nvalid + i] = -1;
  }
  const int n_ent = n_uniq + ns;
  if (lane == 0) ent_offset[n_ent] = nvalid + ns * T;
  __syncwarp();
  // work items per entry, exclusive prefix over entries (warp scan in chunks)
  int na_run = 0, nb_run = 0, bt_run = 0;
  for (int base = 0; base < n_ent; base += 32) {
    const int u = base + lane;
    int ia = 0, ib = 0, ntg = 0;
    if (u < n_ent) {
      const int cu = s_entcnt[u];
      const int iu = u < n_uniq ? c.inter : c.shared_inter;
      ntg = (cu + TG - 1) / TG;
      ia = (iu / RA) * ntg;
      ib = (H / RB) * ntg;
    }
    int sa = ia, sb = ib, st = ntg;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int na = __shfl_up_sync(0xffffffffu, sa, o), nbv = __shfl_up_sync(0xffffffffu, sb, o),
                nt = __shfl_up_sync(0xffffffffu, st, o);
      if (lane >= o) { sa += na; sb += nbv; st += nt; }
    }
    if (u < n_ent) {
      ent_item_a[u] = na_run + sa - ia;
      ent_item_b[u] = nb_run + sb - ib;
    }
    na_run += __shfl_sync(0xffffffffu, sa, 31);
    nb_run += __shfl_sync(0xffffffffu, sb, 31);
    bt_run += __shfl_sync(0xffffffffu, st, 31);
  }
  if (lane == 0) {
    ent_item_a[n_ent] = na_run;
    ent_item_b[n_ent] = nb_run;
    hdr[H_NENT] = n_ent;
    hdr[H_NUNIQ] = n_uniq;
    hdr[H_NA] = na_run;
    hdr[H_NB] = nb_run;
    hdr[H_BTARGET] = bt_run;
    hdr[H_NPAIRS] = nvalid + ns * T;
  }
}

cudaError_t launch_prep(const PrepParams& P, unsigned grid, size_t smem, cudaStream_t st) {
  cudaError_t e;
  if (P.cfg.weight_bits == 4) {
    e = cudaFuncSetAttribute(prep_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prep_kernel<4><<<grid, PREP_THREADS, smem, st>>>(P);
  } else if (P.cfg.weight_bits == 2) {
    e = cudaFuncSetAttribute(prep_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prep_kernel<2><<<grid, PREP_THREADS, smem, st>>>(P);
  } else {
    e = cudaFuncSetAttribute(prep_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prep_kernel<8><<<grid, PREP_THREADS, smem, st>>>(P);
  }
  return cudaGetLastError();
}

cudaError_t launch_prep_small(const PrepParams& P, unsigned grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (P.cfg.weight_bits == 4) return cudaLaunchKernelEx(&cfg, prep_small_kernel<4>, P);
  if (P.cfg.weight_bits == 2) return cudaLaunchKernelEx(&cfg, prep_small_kernel<2>, P);
  return cudaLaunchKernelEx(&cfg, prep_small_kernel<8>, P);
}

cudaError_t launch_quantize_act(const float* x, long long nblk, int8_t* q, float* d, unsigned blocks,
                                cudaStream_t st) {
  quantize_act_kernel<<<blocks, 256, 0, st>>>(x, nblk, q, d);
  return cudaGetLastError();
}

}  // namespace colimoe
