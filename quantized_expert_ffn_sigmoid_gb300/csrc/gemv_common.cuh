// Device helpers shared by the streaming GEMV kernels (gemv.cu) and the
// fused single-position layer kernel (decode.cu): 128-bit streaming loads,
// register-held weight blocks with their integer block dots, expert record
// addressing and programmatic-dependent-launch controls.
#pragma once
#include "colimoe_internal.cuh"

namespace colimoe {

__device__ __forceinline__ uint4 ldg_stream(const void* p, uint64_t pol) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(pol));
  return v;
}

// One weight block (a Q8_0 block's worth of one row) in registers.
template <int BITS> struct WBlk;
template <> struct WBlk<4> {
  uint4 w;  // 32 nibbles
  __device__ __forceinline__ void load(const uint8_t* p, uint64_t pol) { w = ldg_stream(p, pol); }
  __device__ __forceinline__ void lds(const uint8_t* p) { w = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ int dot(const uint4& a0, const uint4& a1, int corr) const {
    // low nibbles masked in place; high nibbles masked without shifting, so
    // their products come out times 16 and one exact shift per block undoes it
    const uint32_t lo = 0x0F0F0F0Fu, hi = 0xF0F0F0F0u;
    int s = 0, r = 0;
    s = dp4a_us(w.x & lo, a0.x, s); r = dp4a_us(w.x & hi, a0.y, r);
    s = dp4a_us(w.y & lo, a0.z, s); r = dp4a_us(w.y & hi, a0.w, r);
    s = dp4a_us(w.z & lo, a1.x, s); r = dp4a_us(w.z & hi, a1.y, r);
    s = dp4a_us(w.w & lo, a1.z, s); r = dp4a_us(w.w & hi, a1.w, r);
    return (s + (r >> 4)) - corr;  // nibbles hold code + 8: remove 8 * sum(q_x)
  }
};
template <> struct WBlk<8> {
  uint4 a, b;  // 32 int8 codes
  __device__ __forceinline__ void load(const uint8_t* p, uint64_t pol) {
    a = ldg_stream(p, pol);
    b = ldg_stream(p + 16, pol);
  }
  __device__ __forceinline__ void lds(const uint8_t* p) {
    a = reinterpret_cast<const uint4*>(p)[0];
    b = reinterpret_cast<const uint4*>(p)[1];
  }
  __device__ __forceinline__ int dot(const uint4& a0, const uint4& a1, int) const {
    int s = 0, r = 0;
    s = dp4a_ss(a.x, a0.x, s); r = dp4a_ss(a.y, a0.y, r); s = dp4a_ss(a.z, a0.z, s); r = dp4a_ss(a.w, a0.w, r);
    s = dp4a_ss(b.x, a1.x, s); r = dp4a_ss(b.y, a1.y, r); s = dp4a_ss(b.z, a1.z, s); r = dp4a_ss(b.w, a1.w, r);
    return s + r;
  }
};

template <> struct WBlk<2> {
  uint2 w;  // 32 two-bit fields
  __device__ __forceinline__ void lds(const uint8_t* p) { w = *reinterpret_cast<const uint2*>(p); }
  __device__ __forceinline__ int dot(const uint4& a0, const uint4& a1, int corr) const {
    // field m of every byte masked in place: its products come out times 4^m,
    // and one exact shift per chain undoes it (activation word m of each half
    // block holds the elements that field m of the 4 weight bytes carries)
    int c0 = 0, c1 = 0, c2 = 0, c3 = 0;
    c0 = dp4a_us(w.x & 0x03030303u, a0.x, c0); c1 = dp4a_us(w.x & 0x0C0C0C0Cu, a0.y, c1);
    c2 = dp4a_us(w.x & 0x30303030u, a0.z, c2); c3 = dp4a_us(w.x & 0xC0C0C0C0u, a0.w, c3);
    c0 = dp4a_us(w.y & 0x03030303u, a1.x, c0); c1 = dp4a_us(w.y & 0x0C0C0C0Cu, a1.y, c1);
    c2 = dp4a_us(w.y & 0x30303030u, a1.z, c2); c3 = dp4a_us(w.y & 0xC0C0C0C0u, a1.w, c3);
    return (c0 + (c1 >> 2) + (c2 >> 4) + (c3 >> 6)) - corr;  // fields hold code + 2: remove 2 * sum(q_x)
  }
};

__device__ __forceinline__ const uint8_t* gemv_record(const ExpertParams& P, int expert, int* inter,
                                                      const float** sc) {
  const coli_moe_cfg& c = P.cfg;
  const int H = c.hidden, bits = c.weight_bits;
  const bool routed = expert < c.n_experts;
  const int I = routed ? c.inter : c.shared_inter;
  const int e = routed ? ep_local_mul(P.ep_mul, expert) : expert - c.n_experts;
  const size_t rec = (size_t)2 * I * row_bytes(H, bits) + (size_t)H * row_bytes(I, bits);
  *inter = I;
  // per-row scales (2 I + H per record) or one per 64 weights (3 I H / 64)
  const size_t nsc = c.group_size ? (size_t)3 * I * (H / c.group_size) : (size_t)2 * I + H;
  *sc = (routed ? P.expert_scales : P.shared_scales) + (size_t)e * nsc;
  return (routed ? P.experts : P.shared) + (size_t)e * rec;
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace colimoe
