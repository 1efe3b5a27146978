// Internal definitions shared by the libcolimoe translation units:
// workspace layout, kernel parameter blocks, tiling constants and thin
// inline-PTX wrappers (mbarrier, bulk async copy, dp4a, fences).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include "../../include/coli_moe.h"

namespace colimoe {

// ---------------------------------------------------------------- constants
constexpr int QB = 32;          // Q8_0 block (values per fp32 scale)
constexpr int TG = 4;           // positions per expert work item
constexpr int RA = 32;          // gate/up rows per work item (= one h block)
constexpr int RB = 64;          // down rows per work item (= one combine tile)
constexpr int NS = 4;           // weight ring stages per CTA
constexpr int SB = 32768;       // bytes per weight stage
constexpr int NCW = 8;          // consumer warps per expert CTA
constexpr int EXPERT_THREADS = 32 * (NCW + 1);  // + one producer warp
constexpr int RED_BYTES = 8192; // cross-warp partial sums of one item
constexpr int MAX_E = 1024;
constexpr int MAX_TOPK = 32;
constexpr int MAX_SHARED = 8;
constexpr int MAX_GROUPS = 32;
// bytes at the start of a workspace that coli_moe_workspace_init clears:
// status and counter words, then the router's tagged exchange words
constexpr size_t WS_STATUS_BYTES = 512;  // status word and device counters (128 words)
constexpr size_t WS_HEADER_BYTES = WS_STATUS_BYTES + 8 * (size_t)MAX_E;
constexpr int GEMV_SPLITS = 8;  // K splits of the router GEMV (T <= 8)
constexpr int ROUTE_GEMV_MAX_T = 8;
constexpr int PREP_THREADS = 1024;
constexpr int GEMV_MAX_T = 4;   // calls up to this many positions take the streaming GEMV path
constexpr int PF_MIN_T = 64;    // calls with at least this many positions use the tensor cores ...
constexpr int PF_MIN_PAIRS = 12;  // ... for the entries with at least this many pairs; the others
                                  // stream through the small-batch kernels in the same call

constexpr uint32_t SPIN_LIMIT = 1u << 22;  // bounded waits (about a second or more)

__host__ __device__ inline int row_bytes(int k, int bits) { return bits == 4 ? k / 2 : bits == 2 ? k / 4 : k; }

// Expert-parallel sharding: with ep_size > 1 a call computes the routed
// experts e with e mod ep_size == ep_rank, stored as local record e / ep_size.
__host__ __device__ inline bool ep_owned(const coli_moe_cfg& c, int e) {
  return c.ep_size <= 1 || e % c.ep_size == c.ep_rank;
}
// floor(e / ep_size) as one multiply-high by ep_mul(c) (kernels address
// records in their inner loops, where an integer division would cost ~20
// instructions): exact for e < 1024 and ep_size <= 1024.
__host__ __device__ inline uint64_t ep_mul(const coli_moe_cfg& c) {
  return c.ep_size <= 1 ? (1ull << 32) : (1ull << 32) / (uint64_t)c.ep_size + 1ull;
}
__host__ __device__ inline int ep_local_mul(uint64_t mul, int e) { return (int)(((uint64_t)e * mul) >> 32); }
__host__ __device__ inline int ep_local(const coli_moe_cfg& c, int e) { return c.ep_size <= 1 ? e : e / c.ep_size; }
// routed records held by this shard
__host__ __device__ inline int ep_records(const coli_moe_cfg& c) {
  return c.ep_size <= 1 ? c.n_experts : (c.n_experts - c.ep_rank + c.ep_size - 1) / c.ep_size;
}

// K ranges of the tiled router GEMM (calls of more than ROUTE_GEMV_MAX_T
// positions): about 1024 CTAs of 64 x 64 logits, at least 192 K elements
// each; the partial logits of every range are summed in range order.
__host__ __device__ inline int route_ksplits(int T, int H, int E) {
  const int tiles = ((E + 63) / 64) * ((T + 63) / 64);
  const int kmax = H / 192 > 0 ? H / 192 : 1;
  int ks = 1024 / tiles;
  ks = ks < 1 ? 1 : (ks > kmax ? kmax : ks);
  while (ks > 1 && H % (ks * 16)) --ks;
  return ks;
}
__host__ __device__ inline int pow2_floor(int v) { int p = 1; while (p * 2 <= v) p *= 2; return p; }
// gate+up rows per ring stage for reduction length H
__host__ __device__ inline int stage_rows_a(int H, int bits) {
  int rs = pow2_floor(SB / (2 * row_bytes(H, bits)));
  return rs > RA ? RA : rs;
}
// down rows per ring stage for reduction length I
__host__ __device__ inline int stage_rows_b(int I, int bits) {
  int rs = pow2_floor(SB / row_bytes(I, bits));
  return rs > RB ? RB : rs;
}
__host__ __device__ inline int splits_for(int tasks_per_split_unit, int nb) {
  int s = NCW / tasks_per_split_unit;
  if (s < 1) s = 1;
  while (s > 1 && nb % s) s /= 2;
  return s;
}
__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------------- layout
struct Layout {
  int T, P, n_ent_max, n_tiles, imax;
  size_t status, route_words, counters, hdr, ent_expert, ent_count, ent_offset, ent_item_a,
         ent_item_b, pair_token, pair_j, slot, route_part, qx, dx, xs, qh, dh, hs, o,
         pf_xs, pf_hb, pf_hs, total;
};
// Table header (ints at Layout::hdr)
enum HdrField { H_NENT = 0, H_NUNIQ, H_NA, H_NB, H_BTARGET, H_NPAIRS, H_FIELDS = 8 };
// Counters (uint32 at Layout::counters): [0] ticket, [1..n_ent_max] A done,
// then n_tiles combine counters.

__host__ __device__ inline Layout make_layout(const coli_moe_cfg& c, int T) {
  Layout L{};
  const int k = c.top_k, ns = c.n_shared, H = c.hidden, E = c.n_experts;
  L.T = T;
  L.P = T * k + ns * T;
  int routed_max = T * k < E ? T * k : E;
  L.n_ent_max = routed_max + ns;
  L.n_tiles = H / RB;
  L.imax = c.inter > c.shared_inter ? c.inter : c.shared_inter;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t r = off; off = align_up(off + bytes, 256); return r; };
  L.status = take(WS_STATUS_BYTES);
  L.route_words = take(8 * (size_t)MAX_E);  // zeroed by coli_moe_workspace_init with the status words
  L.counters = take(4 * (1 + L.n_ent_max + L.n_tiles));
  L.hdr = take(4 * H_FIELDS);
  L.ent_expert = take(4 * (size_t)L.n_ent_max);
  L.ent_count = take(4 * (size_t)L.n_ent_max);
  L.ent_offset = take(4 * ((size_t)L.n_ent_max + 1));
  L.ent_item_a = take(4 * ((size_t)L.n_ent_max + 1));
  L.ent_item_b = take(4 * ((size_t)L.n_ent_max + 1));
  L.pair_token = take(4 * (size_t)L.P);
  L.pair_j = take(4 * (size_t)L.P);
  L.slot = take(4 * (size_t)T * k);
  size_t gemv = (size_t)GEMV_SPLITS * (T < ROUTE_GEMV_MAX_T ? T : ROUTE_GEMV_MAX_T) * E;
  size_t tiled = (size_t)route_ksplits(T, H, E) * T * E;
  L.route_part = take(4 * (gemv > tiled ? gemv : tiled));
  L.qx = take((size_t)T * H);
  L.dx = take(4 * (size_t)T * (H / QB));
  L.xs = take(4 * (size_t)T * (H / QB));
  L.qh = take((size_t)L.P * L.imax);
  L.dh = take(4 * (size_t)L.P * (L.imax / QB));
  L.hs = take(4 * (size_t)L.P * (L.imax / QB));
  L.o = take(4 * (size_t)L.P * H);
  // tensor-core path only (calls of PF_MIN_T or more positions): activation
  // scales per pair, transposed [H/32][P]; h codes widened to fp16 [P][imax];
  // h scales transposed [imax/32][P]
  const bool pf = T >= PF_MIN_T;
  L.pf_xs = take(pf ? 4 * (size_t)(H / QB) * L.P : 0);
  L.pf_hb = take(pf ? 2 * (size_t)L.P * L.imax : 0);
  L.pf_hs = take(pf ? 4 * (size_t)(L.imax / QB) * L.P : 0);
  L.total = off;
  return L;
}

// Byte position, inside a 32-block, where natural element i is stored for
// packed-int4 weights: each group of 8 is stored 0,2,4,6,1,3,5,7 so that the
// low nibbles of 4 packed bytes meet the even elements in one 32-bit word and
// the high nibbles the odd ones.
__host__ __device__ inline int perm8(int i) {
  int r = i & 7;
  return (i & ~7) | ((r & 1) << 2) | (r >> 1);
}
// The same for packed-int2 weights: within each 16 elements (one 32-bit
// weight word) element 4j+m is stored at byte 4m+j, so that the m-th 2-bit
// field of 4 packed bytes meets elements m, 4+m, 8+m, 12+m in one 32-bit word.
__host__ __device__ inline int perm16(int i) { return (i & ~15) | ((i & 3) << 2) | ((i >> 2) & 3); }
// Position of natural element i of an activation block for weights of `bits`
// bits, and the offset-binary bias of those weight codes (the block sum of the
// activation codes times this bias is subtracted from each unsigned block dot).
__host__ __device__ inline int act_pos(int i, int bits) { return bits == 4 ? perm8(i) : bits == 2 ? perm16(i) : i; }
__host__ __device__ inline int code_bias(int bits) { return bits == 4 ? 8 : bits == 2 ? 2 : 0; }

// ---------------------------------------------------------------- params
struct ExpertParams {
  coli_moe_cfg cfg;
  const uint8_t* experts;
  const float* expert_scales;
  const uint8_t* shared;
  const float* shared_scales;
  const float* topk_w;
  float* y;
  uint8_t* ws;
  Layout L;
  int32_t* dump_gu;  // optional [P][2][imax][H/32]
  int32_t* dump_d;   // optional [P][H][imax/32]
  uint64_t ep_mul;   // ep_mul(cfg): local record of routed expert e = ep_local_mul(ep_mul, e)
};

struct PrepParams {
  coli_moe_cfg cfg;
  const float* x;
  const int32_t* idx;
  int T;
  uint8_t* ws;
  Layout L;
};

// ---------------------------------------------------------------- PTX
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase; on expiry sets COLI_STATUS_TIMEOUT and
// returns false (the caller carries on; results are then flagged invalid).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status) {
  for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i > 16) __nanosleep(64);
  }
  atomicOr(status, COLI_STATUS_TIMEOUT);
  return false;
}
// Bounded wait without sleeping between polls, for tight producer/consumer
// pipelines: try_wait itself suspends the thread in hardware until the phase
// completes or a short system time limit passes.
__device__ __forceinline__ bool mbar_wait_tight(uint64_t* bar, uint32_t parity, uint32_t* status) {
  for (uint32_t i = 0; i < SPIN_LIMIT; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  atomicOr(status, COLI_STATUS_TIMEOUT);
  return false;
}
// 1-D bulk async copy global -> shared, completion counted on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void red_relaxed_add(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_shared_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_shared_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
// 16 bytes global -> shared through L2 only (both 16-byte aligned)
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ uint32_t atom_acq_rel_add(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// unsigned bytes (a) times signed bytes (b), summed into c
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ void named_bar(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Q8_0 of one 32-block held one value per lane: returns this lane's code and
// writes the block scale to *d (all lanes).  IEEE fp32 throughout.
__device__ __forceinline__ int q8_0_lane(float v, float* d_out, bool* nonfinite) {
  bool bad = !isfinite(v);
  unsigned anybad = __ballot_sync(0xffffffffu, bad);
  float a = bad ? 0.f : fabsf(v);
  float amax = warp_max(a);
  float d = __fdiv_rn(amax, 127.0f);
  float inv = d > 0.f ? __fdiv_rn(1.0f, d) : 0.f;
  float r = roundf(__fmul_rn(bad ? 0.f : v, inv));
  r = fminf(fmaxf(r, -127.f), 127.f);
  *d_out = d;
  *nonfinite = anybad != 0;
  return (int)r;
}

}  // namespace colimoe
