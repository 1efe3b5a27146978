// The expert products of the routed-MoE layer as one persistent kernel.
//
// colibrì v1.0 README, "What's implemented": integer-dot kernels on Q8_0-style
// int8 activations against int8 / packed int4 / packed int2 weights with
// per-row scales;
// batch-union (each distinct expert read once for all positions routed to
// it); the always-on shared expert.  "Experimental Metal backend": the
// routed-expert SwiGLU.  The combine is the gate-weighted sum of the
// selected experts plus the shared expert.
//
// Work is a queue of items claimed with an atomic ticket:
//   A item (entry u, 32-row tile, <=4 positions): gate and up rows -> g, u,
//     h = silu(g)*u, Q8_0 of the 32 h values (one block) -> qh, dh;
//   B item (entry u, 64-row tile, <=4 positions): down rows on qh -> o;
//     the last B item of a 64-row tile combines y for that tile.
// All A tickets precede all B tickets, so a B item only waits for A items
// that running CTAs have already claimed: the wait always ends (it is still
// bounded).  Warp 0 (one lane) streams weight rows into a ring of shared
// memory stages with 1-D bulk async copies (TMA engine) and the activations
// of the next item into one of two slots; warps 1..8 compute.
#include "colimoe_internal.cuh"

namespace colimoe {

struct ItemDesc {
  int kind;   // 0 gate/up, 1 down, 2 end
  int ent;    // entry index
  int tile;   // row tile
  int ntok;   // positions in this item (<= TG)
  int pair0;  // first pair slot of the item
  int expert; // routed id, or E + s for shared expert s
  int inter;  // intermediate size of the entry
};

struct SmemPtrs {
  uint8_t* ring;
  uint8_t* act;
  float* red;
  int* t_item_a;
  int* t_item_b;
  int* t_count;
  int* t_offset;
  int* t_expert;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* afull;
  uint64_t* aempty;
  ItemDesc* desc;
  int* flag;
};

__host__ __device__ inline size_t act_slot_bytes(const coli_moe_cfg& c, int imax) {
  int kmax = c.hidden > imax ? c.hidden : imax;
  return align_up((size_t)TG * (kmax + kmax / 4), 128);
}

__host__ __device__ inline size_t expert_smem_bytes(const coli_moe_cfg& c, const Layout& L) {
  size_t b = (size_t)NS * SB + 2 * act_slot_bytes(c, L.imax) + RED_BYTES;
  b += align_up(sizeof(int) * 5 * ((size_t)L.n_ent_max + 1), 16);
  b += sizeof(uint64_t) * (2 * NS + 4) + sizeof(ItemDesc) * 2 + 16;
  return align_up(b, 128) + 128;
}

__device__ inline SmemPtrs carve(uint8_t* base, const coli_moe_cfg& c, const Layout& L) {
  SmemPtrs s;
  uint8_t* p = base;
  s.ring = p; p += (size_t)NS * SB;
  s.act = p; p += 2 * act_slot_bytes(c, L.imax);
  s.red = reinterpret_cast<float*>(p); p += RED_BYTES;
  int* ti = reinterpret_cast<int*>(p);
  const int n1 = L.n_ent_max + 1;
  s.t_item_a = ti; s.t_item_b = ti + n1; s.t_count = ti + 2 * n1; s.t_offset = ti + 3 * n1;
  s.t_expert = ti + 4 * n1;
  p += align_up(sizeof(int) * 5 * (size_t)n1, 16);
  uint64_t* bars = reinterpret_cast<uint64_t*>(p);
  s.full = bars; s.empty = bars + NS; s.afull = bars + 2 * NS; s.aempty = bars + 2 * NS + 2;
  p += sizeof(uint64_t) * (2 * NS + 4);
  s.desc = reinterpret_cast<ItemDesc*>(p); p += sizeof(ItemDesc) * 2;
  s.flag = reinterpret_cast<int*>(p);
  return s;
}

__device__ __forceinline__ void consumer_bar() { named_bar(1, 32 * NCW); }

__device__ __forceinline__ void unpack4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = w & 0x0F0F0F0Fu;
  hi = (w >> 4) & 0x0F0F0F0Fu;
}

// Integer dot of one 32-block: weights (16 bytes int4, 8 bytes int2 or 32
// bytes int8 in shared memory) against one activation block (32 bytes, layout
// matching).  For int4 / int2 the stored codes are unsigned (code + 8 / code
// + 2): the block sum of 8*q_x / 2*q_x is subtracted, giving the exact signed
// result.
template <int BITS>
struct BlockW {
  uint32_t v[8];
  __device__ __forceinline__ void load(const uint8_t* p) {
    if (BITS == 4) {
      uint4 w = *reinterpret_cast<const uint4*>(p);
      unpack4(w.x, v[0], v[1]); unpack4(w.y, v[2], v[3]);
      unpack4(w.z, v[4], v[5]); unpack4(w.w, v[6], v[7]);
    } else if (BITS == 2) {
      // word m of each half block: the m-th 2-bit field of its 4 bytes
      const uint2 w = *reinterpret_cast<const uint2*>(p);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        v[m] = (w.x >> (2 * m)) & 0x03030303u;
        v[4 + m] = (w.y >> (2 * m)) & 0x03030303u;
      }
    } else {
      uint4 a = reinterpret_cast<const uint4*>(p)[0], b = reinterpret_cast<const uint4*>(p)[1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
  }
  __device__ __forceinline__ int dot(const uint4& a0, const uint4& a1, int corr) const {
    // two independent dp4a chains (latency), joined at the end
    int s = 0, r = 0;
    if (BITS != 8) {
      s = dp4a_us(v[0], a0.x, s); r = dp4a_us(v[1], a0.y, r); s = dp4a_us(v[2], a0.z, s);
      r = dp4a_us(v[3], a0.w, r); s = dp4a_us(v[4], a1.x, s); r = dp4a_us(v[5], a1.y, r);
      s = dp4a_us(v[6], a1.z, s); r = dp4a_us(v[7], a1.w, r);
      return (s + r) - corr;
    } else {
      s = dp4a_ss(v[0], a0.x, s); r = dp4a_ss(v[1], a0.y, r); s = dp4a_ss(v[2], a0.z, s);
      r = dp4a_ss(v[3], a0.w, r); s = dp4a_ss(v[4], a1.x, s); r = dp4a_ss(v[5], a1.y, r);
      s = dp4a_ss(v[6], a1.z, s); r = dp4a_ss(v[7], a1.w, r);
      return s + r;
    }
  }
};

// fp32 scales of one expert record: per output row (2 I + H), or per 64
// weights of a row (gate [I][H/64] | up [I][H/64] | down [H][I/64])
__device__ __forceinline__ size_t scale_count(const coli_moe_cfg& c, int inter) {
  return c.group_size ? (size_t)3 * inter * (c.hidden / c.group_size) : (size_t)2 * inter + c.hidden;
}

__device__ __forceinline__ const uint8_t* entry_record(const ExpertParams& P, int expert, int* inter_out,
                                                       const float** scales_out) {
  const coli_moe_cfg& c = P.cfg;
  const int H = c.hidden, bits = c.weight_bits;
  if (expert < c.n_experts) {
    const size_t rec = (size_t)2 * c.inter * row_bytes(H, bits) + (size_t)H * row_bytes(c.inter, bits);
    *inter_out = c.inter;
    const int e = ep_local_mul(P.ep_mul, expert);
    *scales_out = P.expert_scales + (size_t)e * scale_count(c, c.inter);
    return P.experts + (size_t)e * rec;
  }
  const int s = expert - c.n_experts;
  const size_t rec = (size_t)2 * c.shared_inter * row_bytes(H, bits) + (size_t)H * row_bytes(c.shared_inter, bits);
  *inter_out = c.shared_inter;
  *scales_out = P.shared_scales + (size_t)s * scale_count(c, c.shared_inter);
  return P.shared + (size_t)s * rec;
}

// ---------------------------------------------------------------- producer
// A decoded work item plus the positions it needs (loaded one item ahead so
// that their latency hides behind the previous item's weight stream).
struct Pending {
  ItemDesc d;
  const uint8_t* rec;
  int tok[TG];
};

template <int BITS>
__device__ __forceinline__ Pending decode_ticket(const ExpertParams& P, const SmemPtrs& S, uint32_t ticket,
                                                 int nA, int nB, int n_ent) {
  Pending pd;
  ItemDesc& d = pd.d;
  d = ItemDesc{};
  pd.rec = nullptr;
  if (ticket >= (uint32_t)(nA + nB)) {
    d.kind = 2;
    return pd;
  }
  const bool isA = ticket < (uint32_t)nA;
  const int local = isA ? (int)ticket : (int)ticket - nA;
  const int* pref = isA ? S.t_item_a : S.t_item_b;
  int lo = 0, hi = n_ent - 1;  // largest u with pref[u] <= local
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= local) lo = mid; else hi = mid - 1;
  }
  const int u = lo;
  const int cnt = S.t_count[u];
  const int ntg = (cnt + TG - 1) / TG;
  const int li = local - pref[u];
  d.kind = isA ? 0 : 1;
  d.ent = u;
  d.tile = li / ntg;
  const int tg = li % ntg;
  d.ntok = min(TG, cnt - tg * TG);
  d.pair0 = S.t_offset[u] + tg * TG;
  d.expert = S.t_expert[u];
  const float* scales;
  pd.rec = entry_record(P, d.expert, &d.inter, &scales);
  if (isA) {
    const int32_t* pair_token = reinterpret_cast<const int32_t*>(P.ws + P.L.pair_token);
#pragma unroll
    for (int i = 0; i < TG; ++i) pd.tok[i] = i < d.ntok ? __ldcg(pair_token + d.pair0 + i) : 0;
  }
  return pd;
}

template <int BITS>
__device__ void producer_loop(const ExpertParams& P, const SmemPtrs& S, int nA, int nB, int n_ent) {
  const coli_moe_cfg& c = P.cfg;
  const Layout& L = P.L;
  uint8_t* ws = P.ws;
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status);
  uint32_t* ctr = reinterpret_cast<uint32_t*>(ws + L.counters);
  const int H = c.hidden;
  const int nbH = H / QB;
  const int rbA = row_bytes(H, BITS);
  const int rsA = stage_rows_a(H, BITS);
  const size_t slot_bytes = act_slot_bytes(c, L.imax);
  const uint64_t pol_w = policy_evict_first();
  const uint64_t pol_a = policy_evict_last();
  uint32_t stage = 0, item = 0;
  Pending cur = decode_ticket<BITS>(P, S, atomicAdd(&ctr[0], 1u), nA, nB, n_ent);
  uint32_t next_ticket = atomicAdd(&ctr[0], 1u);
  for (;; ++item) {
    const int as = item & 1;
    const ItemDesc& d = cur.d;
    mbar_wait(&S.aempty[as], ((item >> 1) & 1u) ^ 1u, status);
    S.desc[as] = d;
    if (d.kind == 2) {
      mbar_arrive(&S.afull[as]);
      break;
    }
    uint8_t* A = S.act + as * slot_bytes;
    if (d.kind == 0) {
      const uint32_t tokbytes = (uint32_t)(H + 2 * nbH * 4);
      mbar_arrive_expect_tx(&S.afull[as], (uint32_t)d.ntok * tokbytes);
#pragma unroll
      for (int i = 0; i < TG; ++i) {
        if (i < d.ntok) {
          const int t = cur.tok[i];
          bulk_g2s(A + i * H, ws + L.qx + (size_t)t * H, H, &S.afull[as], pol_a);
          bulk_g2s(A + TG * H + i * nbH * 4, ws + L.dx + (size_t)t * nbH * 4, nbH * 4, &S.afull[as], pol_a);
          bulk_g2s(A + TG * H + TG * nbH * 4 + i * nbH * 4, ws + L.xs + (size_t)t * nbH * 4, nbH * 4,
                   &S.afull[as], pol_a);
        }
      }
    } else {
      // down products need every h block of this entry
      const uint32_t target = (uint32_t)(S.t_item_a[d.ent + 1] - S.t_item_a[d.ent]);
      const uint32_t* done = &ctr[1 + d.ent];
      bool ok = false;
      for (uint32_t i = 0; i < SPIN_LIMIT; ++i) {
        if (ld_acquire_u32(done) >= target) { ok = true; break; }
        __nanosleep(64);
      }
      if (!ok) atomicOr(status, COLI_STATUS_TIMEOUT);
      fence_proxy_async_global();
      const int im = L.imax, nbI = im / QB;
      mbar_arrive_expect_tx(&S.afull[as], (uint32_t)d.ntok * (im + 2 * nbI * 4));
      bulk_g2s(A, ws + L.qh + (size_t)d.pair0 * im, d.ntok * im, &S.afull[as], pol_a);
      bulk_g2s(A + TG * im, ws + L.dh + (size_t)d.pair0 * nbI * 4, d.ntok * nbI * 4, &S.afull[as], pol_a);
      bulk_g2s(A + TG * im + TG * nbI * 4, ws + L.hs + (size_t)d.pair0 * nbI * 4, d.ntok * nbI * 4,
               &S.afull[as], pol_a);
    }
    // look one item ahead: its ticket and positions load while this item's
    // weight stages stream
    const Pending nxt = decode_ticket<BITS>(P, S, next_ticket, nA, nB, n_ent);
    if (nxt.d.kind != 2) next_ticket = atomicAdd(&ctr[0], 1u);

    if (d.kind == 0) {
      const int nst = RA / rsA;
      const uint32_t bytes = (uint32_t)rsA * rbA;
      for (int st = 0; st < nst; ++st, ++stage) {
        const int s = stage % NS;
        mbar_wait(&S.empty[s], ((stage / NS) & 1u) ^ 1u, status);
        const int row0 = d.tile * RA + st * rsA;
        uint8_t* dst = S.ring + (size_t)s * SB;
        mbar_arrive_expect_tx(&S.full[s], 2 * bytes);
        bulk_g2s(dst, cur.rec + (size_t)row0 * rbA, bytes, &S.full[s], pol_w);
        bulk_g2s(dst + bytes, cur.rec + (size_t)d.inter * rbA + (size_t)row0 * rbA, bytes, &S.full[s], pol_w);
      }
    } else {
      const int rbB = row_bytes(d.inter, BITS);
      const int rsB = stage_rows_b(d.inter, BITS);
      const int nst = RB / rsB;
      const uint32_t bytes = (uint32_t)rsB * rbB;
      const uint8_t* down = cur.rec + (size_t)2 * d.inter * rbA;
      for (int st = 0; st < nst; ++st, ++stage) {
        const int s = stage % NS;
        mbar_wait(&S.empty[s], ((stage / NS) & 1u) ^ 1u, status);
        const int row0 = d.tile * RB + st * rsB;
        mbar_arrive_expect_tx(&S.full[s], bytes);
        bulk_g2s(S.ring + (size_t)s * SB, down + (size_t)row0 * rbB, bytes, &S.full[s], pol_w);
      }
    }
    cur = nxt;
  }
}

// ---------------------------------------------------------------- consumers
template <int BITS, bool DUMP>
__device__ void consume_a(const ExpertParams& P, const SmemPtrs& S, const ItemDesc& d, const uint8_t* A,
                          uint32_t& stage, int cw, int lane) {
  const coli_moe_cfg& c = P.cfg;
  const int H = c.hidden, nb = H / QB;
  const int rb = row_bytes(H, BITS);
  const int rs = stage_rows_a(H, BITS);
  const int SA = splits_for(rs, nb);
  const int ntask = rs * SA;
  const int npc = nb / SA;
  const int8_t* qa = reinterpret_cast<const int8_t*>(A);
  const float* da = reinterpret_cast<const float*>(A + TG * H);
  const int* xa = reinterpret_cast<const int*>(A + TG * H + TG * nb * 4);
  const int cbytes = QB * BITS / 8;
  uint32_t* status = reinterpret_cast<uint32_t*>(P.ws + P.L.status);
  const int nst = RA / rs;
  // group-scaled weights: the scale of (row, block cc) is gsc[row * ngr + cc / 2]
  const int gsz = c.group_size, ngr = gsz ? H / gsz : 0;
  int e_inter;
  const float* esc;
  entry_record(P, d.expert, &e_inter, &esc);
  for (int st = 0; st < nst; ++st, ++stage) {
    const int s = stage % NS;
    mbar_wait(&S.full[s], (stage / NS) & 1u, status);
    const uint8_t* base = S.ring + (size_t)s * SB;
    for (int task = cw; task < ntask; task += NCW) {
      const int rp = task / SA, sp = task % SA;
      const int grow_i = d.tile * RA + st * rs + rp;
      const float* gsc_g = esc + (size_t)grow_i * ngr;
      const float* gsc_u = esc + (size_t)(e_inter + grow_i) * ngr;
      const uint8_t* grow = base + (size_t)rp * rb;
      const uint8_t* urow = base + (size_t)rs * rb + (size_t)rp * rb;
      float pg[TG], pu[TG];
#pragma unroll
      for (int t = 0; t < TG; ++t) { pg[t] = 0.f; pu[t] = 0.f; }
      const int cend = (sp + 1) * npc;
      for (int cc = sp * npc + lane; cc < cend; cc += 32) {
        BlockW<BITS> wg, wu;
        wg.load(grow + (size_t)cc * cbytes);
        wu.load(urow + (size_t)cc * cbytes);
        const float sgc = gsz ? __ldg(gsc_g + cc * QB / gsz) : 1.0f;
        const float suc = gsz ? __ldg(gsc_u + cc * QB / gsz) : 1.0f;
#pragma unroll
        for (int t = 0; t < TG; ++t) {
          if (t < d.ntok) {
            const uint4* a = reinterpret_cast<const uint4*>(qa + (size_t)t * H + (size_t)cc * QB);
            const uint4 a0 = a[0], a1 = a[1];
            const int corr = xa[t * nb + cc];
            const int ig = wg.dot(a0, a1, corr);
            const int iu = wu.dot(a0, a1, corr);
            const float dv = da[t * nb + cc];
            pg[t] = fmaf(__fmul_rn(dv, sgc), (float)ig, pg[t]);
            pu[t] = fmaf(__fmul_rn(dv, suc), (float)iu, pu[t]);
            if (DUMP && P.dump_gu) {
              const int row = d.tile * RA + st * rs + rp;
              const size_t pbase = (size_t)(d.pair0 + t) * 2 * P.L.imax;
              P.dump_gu[(pbase + row) * nb + cc] = ig;
              P.dump_gu[(pbase + P.L.imax + row) * nb + cc] = iu;
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < TG; ++t) {
        if (t < d.ntok) {
          const float g = warp_sum(pg[t]);
          const float u = warp_sum(pu[t]);
          if (lane == 0) {
            const int r = st * rs + rp;
            S.red[((r * SA + sp) * 2 + 0) * TG + t] = g;
            S.red[((r * SA + sp) * 2 + 1) * TG + t] = u;
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
  }
}

template <int BITS>
__device__ void finish_a(const ExpertParams& P, const SmemPtrs& S, const ItemDesc& d, int cw, int lane) {
  const coli_moe_cfg& c = P.cfg;
  const Layout& L = P.L;
  const int H = c.hidden, nb = H / QB;
  const int rs = stage_rows_a(H, BITS);
  const int SA = splits_for(rs, nb);
  uint8_t* ws = P.ws;
  uint32_t* status = reinterpret_cast<uint32_t*>(ws + L.status);
  consumer_bar();
  if (cw < d.ntok) {
    const int t = cw, r = lane;
    float gs = 0.f, us = 0.f;
    for (int sp = 0; sp < SA; ++sp) {
      gs += S.red[((r * SA + sp) * 2 + 0) * TG + t];
      us += S.red[((r * SA + sp) * 2 + 1) * TG + t];
    }
    int inter;
    const float* sc;
    entry_record(P, d.expert, &inter, &sc);
    const int row = d.tile * RA + r;
    // group-scaled sums already carry their weight scales
    const float g = c.group_size ? gs : __fmul_rn(sc[row], gs);
    const float u = c.group_size ? us : __fmul_rn(sc[inter + row], us);
    const float h = __fmul_rn(__fdiv_rn(g, 1.0f + expf(-g)), u);
    float dd;
    bool bad;
    const int q = q8_0_lane(h, &dd, &bad);
    const int qs = warp_sum_i(q);
    const int p = d.pair0 + t;
    const int pos = act_pos(r, BITS);
    int8_t* qh = reinterpret_cast<int8_t*>(ws + L.qh);
    qh[(size_t)p * L.imax + d.tile * RA + pos] = (int8_t)q;
    if (lane == 0) {
      const int nbI = L.imax / QB;
      reinterpret_cast<float*>(ws + L.dh)[(size_t)p * nbI + d.tile] = dd;
      reinterpret_cast<int32_t*>(ws + L.hs)[(size_t)p * nbI + d.tile] = code_bias(BITS) * qs;
      if (bad) atomicOr(status, COLI_STATUS_NONFINITE);
    }
  }
  // the CTA's qh/dh stores happen-before thread 0's release through the
  // barrier, and release is cumulative: one gpu-scope release publishes them
  consumer_bar();
  if (cw == 0 && lane == 0) {
    uint32_t* ctr = reinterpret_cast<uint32_t*>(ws + L.counters);
    red_release_add(&ctr[1 + d.ent], 1u);
  }
}

template <int BITS, bool DUMP>
__device__ void consume_b(const ExpertParams& P, const SmemPtrs& S, const ItemDesc& d, const uint8_t* A,
                          uint32_t& stage, int cw, int lane) {
  const Layout& L = P.L;
  const int I = d.inter, im = L.imax, nbI = im / QB, nb = I / QB;
  const int rb = row_bytes(I, BITS);
  const int rs = stage_rows_b(I, BITS);
  const int nrg = rs / 4;
  const int SBk = splits_for(nrg, nb);
  const int ntask = nrg * SBk;
  const int npc = nb / SBk;
  const int8_t* qa = reinterpret_cast<const int8_t*>(A);
  const float* da = reinterpret_cast<const float*>(A + TG * im);
  const int* xa = reinterpret_cast<const int*>(A + TG * im + TG * nbI * 4);
  const int cbytes = QB * BITS / 8;
  uint32_t* status = reinterpret_cast<uint32_t*>(P.ws + L.status);
  const int H = P.cfg.hidden;
  const int nst = RB / rs;
  // group-scaled weights: the scale of (down row, block cc) is
  // esc[2 * I * H / g + row * I / g + cc / (g / 32)]
  const int gsz = P.cfg.group_size;
  int e_inter;
  const float* esc;
  entry_record(P, d.expert, &e_inter, &esc);
  const float* gsc_d = gsz ? esc + (size_t)2 * I * (H / gsz) : esc;
  for (int st = 0; st < nst; ++st, ++stage) {
    const int s = stage % NS;
    mbar_wait(&S.full[s], (stage / NS) & 1u, status);
    const uint8_t* base = S.ring + (size_t)s * SB;
    for (int task = cw; task < ntask; task += NCW) {
      const int rg = task / SBk, sp = task % SBk;
      const uint8_t* row0 = base + (size_t)(rg * 4) * rb;
      float acc[4][TG];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < TG; ++t) acc[r][t] = 0.f;
      const int cend = (sp + 1) * npc;
      for (int cc = sp * npc + lane; cc < cend; cc += 32) {
        BlockW<BITS> w[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) w[r].load(row0 + (size_t)r * rb + (size_t)cc * cbytes);
        float sdc[4];
#pragma unroll
        for (int r = 0; r < 4; ++r)
          sdc[r] = gsz ? __ldg(gsc_d + (size_t)(d.tile * RB + st * rs + rg * 4 + r) * (I / gsz) + cc * QB / gsz)
                       : 1.0f;
#pragma unroll
        for (int t = 0; t < TG; ++t) {
          if (t < d.ntok) {
            const uint4* a = reinterpret_cast<const uint4*>(qa + (size_t)t * im + (size_t)cc * QB);
            const uint4 a0 = a[0], a1 = a[1];
            const int corr = xa[t * nbI + cc];
            const float dv = da[t * nbI + cc];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const int iv = w[r].dot(a0, a1, corr);
              acc[r][t] = fmaf(__fmul_rn(dv, sdc[r]), (float)iv, acc[r][t]);
              if (DUMP && P.dump_d) {
                const int row = d.tile * RB + st * rs + rg * 4 + r;
                P.dump_d[((size_t)(d.pair0 + t) * H + row) * nbI + cc] = iv;
              }
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < TG; ++t) {
          if (t < d.ntok) {
            const float v = warp_sum(acc[r][t]);
            if (lane == 0) S.red[((st * rs + rg * 4 + r) * SBk + sp) * TG + t] = v;
          }
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
  }
  (void)SBk;
}

template <int BITS>
__device__ void finish_b(const ExpertParams& P, const SmemPtrs& S, const ItemDesc& d, int ctid, int n_uniq) {
  const coli_moe_cfg& c = P.cfg;
  const Layout& L = P.L;
  uint8_t* ws = P.ws;
  const int H = c.hidden, k = c.top_k, T = L.T;
  const int I = d.inter, nb = I / QB;
  const int rs = stage_rows_b(I, BITS);
  const int SBk = splits_for(rs / 4, nb);
  float* o = reinterpret_cast<float*>(ws + L.o);
  consumer_bar();
  int inter;
  const float* sc;
  entry_record(P, d.expert, &inter, &sc);
  for (int i = ctid; i < RB * d.ntok; i += 32 * NCW) {
    const int r = i % RB, t = i / RB;
    float sum = 0.f;
    for (int sp = 0; sp < SBk; ++sp) sum += S.red[(r * SBk + sp) * TG + t];
    const int row = d.tile * RB + r;
    o[(size_t)(d.pair0 + t) * H + row] = c.group_size ? sum : __fmul_rn(sc[2 * inter + row], sum);
  }
  // one acq_rel atomic publishes this CTA's o rows (cumulative release after
  // the barrier) and, for the last arriver, acquires everyone else's
  consumer_bar();
  if (ctid == 0) {
    uint32_t* ctr = reinterpret_cast<uint32_t*>(ws + L.counters);
    const int32_t* hdr = reinterpret_cast<const int32_t*>(ws + L.hdr);
    const uint32_t old = atom_acq_rel_add(&ctr[1 + L.n_ent_max + d.tile], 1u);
    *S.flag = (old + 1u == (uint32_t)hdr[H_BTARGET]) ? 1 : 0;
  }
  consumer_bar();
  if (*S.flag) {
    // last down item of this tile: y[t][rows] = sum_j w_j o_j + shared
    const int32_t* slot = reinterpret_cast<const int32_t*>(ws + L.slot);
    for (int i = ctid; i < T * RB; i += 32 * NCW) {
      const int t = i / RB, r = i % RB;
      const int row = d.tile * RB + r;
      float acc = 0.f;
      for (int j = 0; j < k; ++j) {
        const int p = slot[(size_t)t * k + j];
        if (p >= 0) acc = fmaf(P.topk_w[(size_t)t * k + j], __ldcg(o + (size_t)p * H + row), acc);
      }
      for (int s = 0; s < c.n_shared; ++s) {
        const int p = S.t_offset[n_uniq + s] + t;
        acc = __fadd_rn(acc, __ldcg(o + (size_t)p * H + row));
      }
      P.y[(size_t)t * H + row] = acc;
    }
  }
}

template <int BITS, bool DUMP>
__global__ void __launch_bounds__(EXPERT_THREADS, 1) experts_kernel(ExpertParams P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>(align_up(reinterpret_cast<size_t>(smem_raw), 128));
  const SmemPtrs S = carve(base, P.cfg, P.L);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t* hdr = reinterpret_cast<const int32_t*>(P.ws + P.L.hdr);
  const int n_ent = hdr[H_NENT], n_uniq = hdr[H_NUNIQ], nA = hdr[H_NA], nB = hdr[H_NB];
  {
    const int32_t* ia = reinterpret_cast<const int32_t*>(P.ws + P.L.ent_item_a);
    const int32_t* ib = reinterpret_cast<const int32_t*>(P.ws + P.L.ent_item_b);
    const int32_t* ec = reinterpret_cast<const int32_t*>(P.ws + P.L.ent_count);
    const int32_t* eo = reinterpret_cast<const int32_t*>(P.ws + P.L.ent_offset);
    const int32_t* ee = reinterpret_cast<const int32_t*>(P.ws + P.L.ent_expert);
    for (int i = tid; i <= n_ent; i += EXPERT_THREADS) {
      S.t_item_a[i] = ia[i];
      S.t_item_b[i] = ib[i];
      S.t_offset[i] = eo[i];
      if (i < n_ent) { S.t_count[i] = ec[i]; S.t_expert[i] = ee[i]; }
    }
  }
  if (nB == 0) {
    // no entry at all (every slot skipped and no shared expert, e.g. a shard
    // of an expert-parallel layer that owns none of the call's experts): the
    // combine below never runs, so y = 0 is written here
    const size_t n = (size_t)P.L.T * P.cfg.hidden;
    for (size_t i = (size_t)blockIdx.x * EXPERT_THREADS + tid; i < n; i += (size_t)gridDim.x * EXPERT_THREADS)
      P.y[i] = 0.f;
    return;
  }
  if (tid == 0) {
    for (int i = 0; i < NS; ++i) { mbar_init(&S.full[i], 1); mbar_init(&S.empty[i], NCW); }
    for (int i = 0; i < 2; ++i) { mbar_init(&S.afull[i], 1); mbar_init(&S.aempty[i], NCW); }
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) producer_loop<BITS>(P, S, nA, nB, n_ent);
    return;
  }
  const int cw = warp - 1, ctid = tid - 32;
  uint32_t* status = reinterpret_cast<uint32_t*>(P.ws + P.L.status);
  uint32_t stage = 0, item = 0;
  const size_t slot_bytes = act_slot_bytes(P.cfg, P.L.imax);
  for (;; ++item) {
    const int as = item & 1;
    mbar_wait(&S.afull[as], (item >> 1) & 1u, status);
    const ItemDesc d = S.desc[as];
    if (d.kind == 2) break;
    const uint8_t* A = S.act + as * slot_bytes;
    if (d.kind == 0) {
      consume_a<BITS, DUMP>(P, S, d, A, stage, cw, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.aempty[as]);
      finish_a<BITS>(P, S, d, cw, lane);
    } else {
      consume_b<BITS, DUMP>(P, S, d, A, stage, cw, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.aempty[as]);
      finish_b<BITS>(P, S, d, ctid, n_uniq);
    }
  }
}

size_t experts_smem_bytes(const coli_moe_cfg& c, const Layout& L) { return expert_smem_bytes(c, L); }

template <int BITS, bool DUMP>
static cudaError_t launch_one(const ExpertParams& P, int grid, size_t smem, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(experts_kernel<BITS, DUMP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  experts_kernel<BITS, DUMP><<<grid, EXPERT_THREADS, smem, st>>>(P);
  return cudaGetLastError();
}

cudaError_t launch_experts(const ExpertParams& P, int grid, size_t smem, cudaStream_t st, bool dump) {
  if (P.cfg.weight_bits == 4)
    return dump ? launch_one<4, true>(P, grid, smem, st) : launch_one<4, false>(P, grid, smem, st);
  if (P.cfg.weight_bits == 2)
    return dump ? launch_one<2, true>(P, grid, smem, st) : launch_one<2, false>(P, grid, smem, st);
  return dump ? launch_one<8, true>(P, grid, smem, st) : launch_one<8, false>(P, grid, smem, st);
}

}  // namespace colimoe
