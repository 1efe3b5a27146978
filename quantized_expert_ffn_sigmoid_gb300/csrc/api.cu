// Host side of the C ABI: argument validation, workspace layout, launches on
// the caller's stream.  Allocates nothing and never synchronises (except
// coli_moe_status, whose job it is).
#include <cstring>
#include "colimoe_internal.cuh"

namespace colimoe {
cudaError_t launch_route(const float* x, int T, int H, const float* wr, int E, int G, int topk_group, int k,
                         float rsf, const float* bias, int32_t* topk_idx, float* topk_w, float* part,
                         uint32_t* status, uint32_t* counter, cudaStream_t st);
cudaError_t launch_quantize_act(const float* x, long long nblk, int8_t* q, float* d, unsigned blocks,
                                cudaStream_t st);
cudaError_t launch_prep(const PrepParams& P, unsigned grid, size_t smem, cudaStream_t st);
cudaError_t launch_prep_small(const PrepParams& P, unsigned grid, cudaStream_t st);
cudaError_t launch_experts(const ExpertParams& P, int grid, size_t smem, cudaStream_t st, bool dump);
cudaError_t launch_gemv(const ExpertParams& P, int n_sm, cudaStream_t st, bool dump);
bool decode_fits(const coli_moe_cfg& c);
cudaError_t launch_decode(const ExpertParams& P, const float* x, const int32_t* topk_idx, bool from_ws, int n_sm,
                          cudaStream_t st, bool dump);
bool decode_route_fits(const coli_moe_cfg& c);
cudaError_t launch_decode_routed(const ExpertParams& P, const float* x, const float* router_w, const float* bias,
                                 int32_t* topk_idx, float* topk_w, int n_sm, cudaStream_t st);
bool gemv_fits(const coli_moe_cfg& c, const Layout& L);
bool prefill_fits(const coli_moe_cfg& c, int T);
cudaError_t launch_prefill(const ExpertParams& P, int T, int n_sm, cudaStream_t st, bool dump, bool mixed);
bool sb_fits(const coli_moe_cfg& c, const Layout& L, bool large_T_ok);
cudaError_t launch_sb(const ExpertParams& P, int n_sm, cudaStream_t st, bool dump, int max_pairs);
size_t experts_smem_bytes(const coli_moe_cfg& c, const Layout& L);
}  // namespace colimoe

using namespace colimoe;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_cfg(const coli_moe_cfg* c) {
  if (!c) return COLI_EINVAL;
  if (c->hidden <= 0 || c->hidden % 128 || c->n_experts <= 0 || c->n_groups <= 0) return COLI_EINVAL;
  if (c->n_experts > MAX_E || c->n_groups > MAX_GROUPS) return COLI_EUNSUPPORTED;
  if (c->n_experts % c->n_groups) return COLI_EINVAL;
  if (c->topk_group < 1 || c->topk_group > c->n_groups) return COLI_EINVAL;
  if (c->top_k < 1 || c->top_k > c->topk_group * (c->n_experts / c->n_groups)) return COLI_EINVAL;
  if (c->top_k > MAX_TOPK) return COLI_EUNSUPPORTED;
  if (c->inter <= 0 || c->inter % 128) return COLI_EINVAL;
  if (c->n_shared < 0 || c->n_shared > MAX_SHARED) return COLI_EINVAL;
  if (c->n_shared > 0 && (c->shared_inter <= 0 || c->shared_inter % 128)) return COLI_EINVAL;
  if (c->weight_bits != 2 && c->weight_bits != 4 && c->weight_bits != 8) return COLI_EINVAL;
  if (c->group_size != 0 && c->group_size != 64) return COLI_EINVAL;
  if (c->group_size != 0 && c->weight_bits != 4) return COLI_EUNSUPPORTED;  // group scales: int4 only
  if (!(c->routed_scaling_factor == c->routed_scaling_factor)) return COLI_EINVAL;
  // a gate+up stage must hold at least one row pair, a down stage four rows
  if (2 * row_bytes(c->hidden, c->weight_bits) > SB) return COLI_EUNSUPPORTED;
  const int imax = c->inter > c->shared_inter ? c->inter : c->shared_inter;
  if (4 * row_bytes(imax, c->weight_bits) > SB) return COLI_EUNSUPPORTED;
  if (c->hidden % RB) return COLI_EUNSUPPORTED;
  // expert-parallel shard: 0 <= ep_rank < ep_size <= E, or no sharding
  if (c->ep_size < 0 || c->ep_size > c->n_experts || c->ep_rank < 0) return COLI_EINVAL;
  if (c->ep_rank >= (c->ep_size > 1 ? c->ep_size : 1)) return COLI_EINVAL;
  return COLI_OK;
}

// The few-position path takes per-row scales (int8, int4 or int2); the
// small-batch and prefill paths take int4 or int8 with per-row scales.
// Group-scaled int4 runs on the single-position kernel (which takes both
// scale layouts) or else on the general expert kernel, and packed int2
// beyond the few-position sizes on the general expert kernel.
bool per_row(const coli_moe_cfg& c) { return c.group_size == 0; }
// per-row scales: the few-position, small-batch and (int4 / int8) tensor-core kernels
bool fast_paths(const coli_moe_cfg& c) { return per_row(c); }

coli_moe_cfg normalized(const coli_moe_cfg* c) {
  coli_moe_cfg n = *c;
  if (n.ep_size <= 1) n.ep_size = 1;
  if (n.ep_rank != 0) n.n_shared = 0;   // the shared experts belong to shard 0
  if (n.n_shared == 0) n.shared_inter = n.inter;
  return n;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int rc_of(cudaError_t e) { return e == cudaSuccess ? COLI_OK : COLI_ECUDA; }

int check_ws(const coli_moe_cfg& c, int T, const void* ws, size_t ws_bytes, Layout* L) {
  if (!ws) return COLI_EINVAL;
  if (!aligned16(ws)) return COLI_EALIGN;
  *L = make_layout(c, T);
  if (ws_bytes < L->total) return COLI_EWORKSPACE;
  return COLI_OK;
}

size_t prep_smem(const coli_moe_cfg& c) {
  return (size_t)(4 * c.n_experts + 64) * 4 + (size_t)32 * c.n_experts * 2;
}

int do_dispatch(const coli_moe_cfg& c, const float* x, int T, const int32_t* idx, uint8_t* ws,
                const Layout& L, cudaStream_t st) {
  PrepParams P{c, x, idx, T, ws, L};
  if (T <= GEMV_MAX_T && T * c.top_k <= GEMV_MAX_T * MAX_TOPK) {
    const int nblk = T * (c.hidden / QB);
    const unsigned grid = (unsigned)((nblk + 7) / 8);  // one 32-block per warp
    return rc_of(launch_prep_small(P, grid > 0 ? grid : 1, st));
  }
  const long long nblk = (long long)T * (c.hidden / QB);
  long long nq = (nblk + PREP_THREADS / 32 - 1) / (PREP_THREADS / 32);
  const long long cap = 8LL * (sm_count() > 0 ? sm_count() : 132);
  if (nq > cap) nq = cap;
  return rc_of(launch_prep(P, (unsigned)(1 + nq), prep_smem(c), st));
}

// x / idx given: a single-position call runs the fused layer kernel, which
// builds its own tables; without them the kernels read what coli_moe_dispatch
// left in the workspace.
ExpertParams expert_params(const coli_moe_cfg& c, const coli_moe_weights* w, const float* topk_w, float* y,
                           uint8_t* ws, const Layout& L, int32_t* dump_gu, int32_t* dump_d) {
  ExpertParams P{};
  P.cfg = c;
  P.experts = static_cast<const uint8_t*>(w->experts);
  P.expert_scales = w->expert_scales;
  P.shared = static_cast<const uint8_t*>(w->shared);
  P.shared_scales = w->shared_scales;
  P.topk_w = topk_w;
  P.y = y;
  P.ws = ws;
  P.L = L;
  P.dump_gu = dump_gu;
  P.dump_d = dump_d;
  P.ep_mul = ep_mul(c);
  return P;
}

int do_experts(const coli_moe_cfg& c, const coli_moe_weights* w, int T, const float* topk_w, float* y,
               uint8_t* ws, const Layout& L, cudaStream_t st, int32_t* dump_gu, int32_t* dump_d,
               const float* x = nullptr, const int32_t* idx = nullptr) {
  const ExpertParams P = expert_params(c, w, topk_w, y, ws, L, dump_gu, dump_d);
  if (T == 1 && decode_fits(c)) {
    const int n_sm = sm_count();
    if (n_sm <= 0) return COLI_ECUDA;
    return rc_of(launch_decode(P, x, idx, x == nullptr, n_sm, st, dump_gu || dump_d));
  }
  if (fast_paths(c) && prefill_fits(c, T)) {
    // many positions: per entry, the experts with at least PF_MIN_PAIRS pairs
    // (and the shared experts) on the tensor cores, the others through the
    // small-batch kernels, then one combine of every pair's output
    const int n_sm = sm_count();
    if (n_sm <= 0) return COLI_ECUDA;
    const bool dump = dump_gu || dump_d;
    if (!sb_fits(c, L, true)) return rc_of(launch_prefill(P, T, n_sm, st, dump, false));
    const int rc = rc_of(launch_prefill(P, T, n_sm, st, dump, true));
    if (rc != COLI_OK) return rc;
    return rc_of(launch_sb(P, n_sm, st, dump, PF_MIN_PAIRS - 1));
  }
  if (T <= GEMV_MAX_T && per_row(c) && gemv_fits(c, L)) {
    // a few positions: stream the weights through the two GEMV kernels
    const int n_sm = sm_count();
    if (n_sm <= 0) return COLI_ECUDA;
    return rc_of(launch_gemv(P, n_sm, st, dump_gu || dump_d));
  }
  if (sb_fits(c, L, c.weight_bits == 2 || c.group_size != 0)) {
    // up to a few dozen positions (packed int2 and group-scaled int4: any
    // number, the tensor-core path takes per-row int4 and int8 only): weight
    // rows on lanes, K split over warps
    const int n_sm = sm_count();
    if (n_sm <= 0) return COLI_ECUDA;
    return rc_of(launch_sb(P, n_sm, st, dump_gu || dump_d, 0x7fffffff));
  }
  const size_t smem = experts_smem_bytes(c, L);
  int dev_smem = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&dev_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (smem > (size_t)dev_smem) return COLI_EUNSUPPORTED;
  const int grid = sm_count();
  if (grid <= 0) return COLI_ECUDA;
  return rc_of(launch_experts(P, grid, smem, st, dump_gu || dump_d));
}

int check_weights(const coli_moe_cfg& c, const coli_moe_weights* w) {
  if (!w || !w->experts || !w->expert_scales) return COLI_EINVAL;
  if (c.n_shared > 0 && (!w->shared || !w->shared_scales)) return COLI_EINVAL;
  if (!aligned16(w->experts) || !aligned16(w->expert_scales)) return COLI_EALIGN;
  if (c.n_shared > 0 && (!aligned16(w->shared) || !aligned16(w->shared_scales))) return COLI_EALIGN;
  return COLI_OK;
}

}  // namespace

extern "C" {

size_t coli_moe_workspace_size(const coli_moe_cfg* cfg, int32_t max_T) {
  if (check_cfg(cfg) != COLI_OK || max_T < 0) return 0;
  return make_layout(normalized(cfg), max_T).total;
}

int coli_moe_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!ws || ws_bytes < 256) return COLI_EINVAL;
  if (!aligned16(ws)) return COLI_EALIGN;
  const size_t n = ws_bytes < WS_HEADER_BYTES ? ws_bytes : WS_HEADER_BYTES;
  return cudaMemsetAsync(ws, 0, n, stream) == cudaSuccess ? COLI_OK : COLI_ECUDA;
}

int coli_moe_route(const coli_moe_cfg* cfg, const float* x, int32_t T, const float* router_w,
                   const float* corr_bias, int32_t* topk_idx, float* topk_w, void* ws, size_t ws_bytes,
                   cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (T < 0) return COLI_EINVAL;
  if (T == 0) return COLI_OK;
  if (!x || !router_w || !corr_bias || !topk_idx || !topk_w) return COLI_EINVAL;
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(corr_bias) || !aligned16(topk_idx) ||
      !aligned16(topk_w))
    return COLI_EALIGN;
  const coli_moe_cfg c = normalized(cfg);
  Layout L;
  if ((rc = check_ws(c, T, ws, ws_bytes, &L))) return rc;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  return rc_of(launch_route(x, T, c.hidden, router_w, c.n_experts, c.n_groups, c.topk_group, c.top_k,
                            c.routed_scaling_factor, corr_bias, topk_idx, topk_w,
                            reinterpret_cast<float*>(w8 + L.route_part),
                            reinterpret_cast<uint32_t*>(w8 + L.status),
                            reinterpret_cast<uint32_t*>(w8 + L.status) + 1, stream));
}

int coli_moe_quantize_act(const float* x, int32_t T, int32_t K, int8_t* q, float* d, cudaStream_t stream) {
  if (T < 0 || K <= 0 || K % QB) return COLI_EINVAL;
  if (T == 0) return COLI_OK;
  if (!x || !q || !d) return COLI_EINVAL;
  if (!aligned16(x) || !aligned16(q) || !aligned16(d)) return COLI_EALIGN;
  const long long nblk = (long long)T * (K / QB);
  long long blocks = (nblk + 7) / 8;
  const long long cap = 16LL * (sm_count() > 0 ? sm_count() : 132);
  if (blocks > cap) blocks = cap;
  return rc_of(launch_quantize_act(x, nblk, q, d, (unsigned)blocks, stream));
}

int coli_moe_dispatch(const coli_moe_cfg* cfg, const float* x, int32_t T, const int32_t* topk_idx, void* ws,
                      size_t ws_bytes, cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (T < 0) return COLI_EINVAL;
  if (T == 0) return COLI_OK;
  if (!x || !topk_idx) return COLI_EINVAL;
  if (!aligned16(x) || !aligned16(topk_idx)) return COLI_EALIGN;
  const coli_moe_cfg c = normalized(cfg);
  Layout L;
  if ((rc = check_ws(c, T, ws, ws_bytes, &L))) return rc;
  return do_dispatch(c, x, T, topk_idx, static_cast<uint8_t*>(ws), L, stream);
}

int coli_moe_experts(const coli_moe_cfg* cfg, const coli_moe_weights* weights, int32_t T, const float* topk_w,
                     float* y, void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (T < 0) return COLI_EINVAL;
  if (T == 0) return COLI_OK;
  const coli_moe_cfg c = normalized(cfg);
  if ((rc = check_weights(c, weights))) return rc;
  if (!topk_w || !y) return COLI_EINVAL;
  if (!aligned16(topk_w) || !aligned16(y)) return COLI_EALIGN;
  Layout L;
  if ((rc = check_ws(c, T, ws, ws_bytes, &L))) return rc;
  return do_experts(c, weights, T, topk_w, y, static_cast<uint8_t*>(ws), L, stream, nullptr, nullptr);
}

int coli_moe_forward(const coli_moe_cfg* cfg, const coli_moe_weights* weights, const float* x, int32_t T,
                     const int32_t* topk_idx, const float* topk_w, float* y, void* ws, size_t ws_bytes,
                     cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (T < 0) return COLI_EINVAL;
  if (T == 0) return COLI_OK;
  const coli_moe_cfg c = normalized(cfg);
  if ((rc = check_weights(c, weights))) return rc;
  if (!x || !topk_idx || !topk_w || !y) return COLI_EINVAL;
  if (!aligned16(x) || !aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(y)) return COLI_EALIGN;
  Layout L;
  if ((rc = check_ws(c, T, ws, ws_bytes, &L))) return rc;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  if (T == 1 && decode_fits(c)) return do_experts(c, weights, T, topk_w, y, w8, L, stream, nullptr, nullptr, x, topk_idx);
  if ((rc = do_dispatch(c, x, T, topk_idx, w8, L, stream))) return rc;
  return do_experts(c, weights, T, topk_w, y, w8, L, stream, nullptr, nullptr);
}

int coli_moe_layer(const coli_moe_cfg* cfg, const coli_moe_weights* weights, const float* x, int32_t T,
                   const float* router_w, const float* corr_bias, int32_t* topk_idx, float* topk_w, float* y,
                   void* ws, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (T < 0) return COLI_EINVAL;
  if (T == 0) return COLI_OK;
  const coli_moe_cfg c = normalized(cfg);
  if ((rc = check_weights(c, weights))) return rc;
  if (!x || !router_w || !corr_bias || !topk_idx || !topk_w || !y) return COLI_EINVAL;
  if (!aligned16(x) || !aligned16(router_w) || !aligned16(corr_bias) || !aligned16(topk_idx) ||
      !aligned16(topk_w) || !aligned16(y))
    return COLI_EALIGN;
  Layout L;
  if ((rc = check_ws(c, T, ws, ws_bytes, &L))) return rc;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  if (T == 1 && c.ep_size == 1 && decode_route_fits(c)) {
    // (a shard of an expert-parallel layer routes first: its experts are a
    // subset of the selection, which the fused kernel's schedule assumes whole)
    const int n_sm = sm_count();
    if (n_sm <= 0) return COLI_ECUDA;
    const ExpertParams P = expert_params(c, weights, topk_w, y, w8, L, nullptr, nullptr);
    return rc_of(launch_decode_routed(P, x, router_w, corr_bias, topk_idx, topk_w, n_sm, stream));
  }
  rc = rc_of(launch_route(x, T, c.hidden, router_w, c.n_experts, c.n_groups, c.topk_group, c.top_k,
                          c.routed_scaling_factor, corr_bias, topk_idx, topk_w,
                          reinterpret_cast<float*>(w8 + L.route_part), reinterpret_cast<uint32_t*>(w8 + L.status),
                          reinterpret_cast<uint32_t*>(w8 + L.status) + 1, stream));
  if (rc) return rc;
  if (T == 1 && decode_fits(c)) return do_experts(c, weights, T, topk_w, y, w8, L, stream, nullptr, nullptr, x, topk_idx);
  if ((rc = do_dispatch(c, x, T, topk_idx, w8, L, stream))) return rc;
  return do_experts(c, weights, T, topk_w, y, w8, L, stream, nullptr, nullptr);
}

int coli_moe_forward_dump(const coli_moe_cfg* cfg, const coli_moe_weights* weights, const float* x, int32_t T,
                          const int32_t* topk_idx, const float* topk_w, float* y, void* ws, size_t ws_bytes,
                          int32_t* acc_gu, int32_t* acc_d, cudaStream_t stream) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (T < 0) return COLI_EINVAL;
  if (T == 0) return COLI_OK;
  const coli_moe_cfg c = normalized(cfg);
  if ((rc = check_weights(c, weights))) return rc;
  if (!x || !topk_idx || !topk_w || !y) return COLI_EINVAL;
  if (!aligned16(x) || !aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(y)) return COLI_EALIGN;
  if ((acc_gu && !aligned16(acc_gu)) || (acc_d && !aligned16(acc_d))) return COLI_EALIGN;
  Layout L;
  if ((rc = check_ws(c, T, ws, ws_bytes, &L))) return rc;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  if (T == 1 && decode_fits(c)) return do_experts(c, weights, T, topk_w, y, w8, L, stream, acc_gu, acc_d, x, topk_idx);
  if ((rc = do_dispatch(c, x, T, topk_idx, w8, L, stream))) return rc;
  return do_experts(c, weights, T, topk_w, y, w8, L, stream, acc_gu, acc_d);
}

int coli_moe_status(void* ws, cudaStream_t stream, uint32_t* status) {
  if (!ws || !status) return COLI_EINVAL;
  uint32_t v = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return COLI_ECUDA;
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return COLI_ECUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(v), stream) != cudaSuccess) return COLI_ECUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return COLI_ECUDA;
  *status = v;
  return COLI_OK;
}

const char* coli_moe_strerror(int code) {
  switch (code) {
    case COLI_OK: return "ok";
    case COLI_EINVAL: return "invalid argument (shape, config or null pointer)";
    case COLI_EALIGN: return "pointer not 16-byte aligned";
    case COLI_EWORKSPACE: return "workspace too small";
    case COLI_ECUDA: return "CUDA launch or query failed";
    case COLI_EUNSUPPORTED: return "shape outside the kernels' limits";
    default: return "unknown error code";
  }
}

int coli_moe_workspace_layout(const coli_moe_cfg* cfg, int32_t max_T, coli_moe_ws_layout* out) {
  int rc = check_cfg(cfg);
  if (rc) return rc;
  if (!out || max_T < 0) return COLI_EINVAL;
  const Layout L = make_layout(normalized(cfg), max_T);
  out->status = L.status;
  out->n_entries = L.hdr + 4 * H_NENT;
  out->entry_expert = L.ent_expert;
  out->entry_count = L.ent_count;
  out->entry_offset = L.ent_offset;
  out->pair_token = L.pair_token;
  out->pair_slot_of = L.slot;
  out->qx = L.qx;
  out->dx = L.dx;
  out->qh = L.qh;
  out->dh = L.dh;
  out->o = L.o;
  out->total = L.total;
  return COLI_OK;
}

}  // extern "C"
