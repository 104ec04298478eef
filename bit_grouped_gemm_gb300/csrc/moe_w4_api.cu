// moe_w4_api.cu -- the C ABI of include/moe_w4.h: plan (scratch) management,
// host-side argument checks, tensor-map encoding and the launch sequence of
// one MoE layer (router+top-k, scan+block map, scatter, gather, gate/up GEMM,
// down GEMM, combine), all on the caller's stream with no host sync.
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <tuple>
#include <vector>

#include "moe_internal.h"

using namespace moe;

static constexpr float kRmsEps = 1e-6f;   // RMS-norm epsilon of the stack update

namespace {

struct TimedLaunch {
  int kind;
  cudaEvent_t a, b;
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {                 // byte offsets into the scratch allocation
  size_t topk_idx, topk_w, logits, blk_cnt, cnt8, cnt, off, tile_off, num_tiles, perm, inv, bmap,
      bmap2, num_tiles2, err, arrive, tlogits, sk_cnt, sk_ws, xs, act, d, dsh, total;
  int nblk_max, max_tiles, max_tiles2, rows_cap;
};

// The fused decode layer's router logits tagged with its launch count
// (at most 8 tokens).
size_t tlogits_bytes(const moe_plan_desc& d) {
  return (size_t)(d.max_tokens < 8 ? d.max_tokens : 8) * d.num_experts * 8;
}

Layout make_layout(const moe_plan_desc& d) {
  Layout L;
  const size_t Tm = (size_t)d.max_tokens, k = (size_t)d.top_k, E = (size_t)d.num_experts;
  L.nblk_max = (int)((Tm + kRouterTB - 1) / kRouterTB);
  L.max_tiles = (int)((Tm * k + kBM - 1) / kBM + E);
  L.rows_cap = (int)(Tm * k + (d.has_shared ? Tm : 0));
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t r = o;
    o = align_up(o + bytes, 256);
    return r;
  };
  L.topk_idx = take(Tm * k * 4);
  L.topk_w = take(Tm * k * 4);
  L.logits = take(Tm * E * 4);
  L.blk_cnt = take((size_t)L.nblk_max * E * 4);
  L.cnt8 = take(route_large_cnt8_bytes(L.nblk_max, (int)E));
  L.cnt = take(E * 4);
  L.off = take((E + 1) * 4);
  L.tile_off = take((E + 1) * 4);
  L.num_tiles = take(16);
  L.perm = take(Tm * k * 4);
  L.inv = take(Tm * k * 4);
  L.bmap = take((size_t)L.max_tiles * 3 * 4);
  L.max_tiles2 = (int)((Tm * k + 255) / 256 + E);
  L.bmap2 = take((size_t)L.max_tiles2 * 3 * 4);
  L.num_tiles2 = take(16);
  L.err = take(16);
  L.arrive = take(16);   // route_large arrivals and generation, fused-layer barrier, launch count
  L.tlogits = take(tlogits_bytes(d));
  L.sk_cnt = take(kSplitSlots * 4);
  L.sk_ws = take((size_t)kSplitSlots * kSplitSlotBytes);
  L.xs = take((size_t)L.rows_cap * d.hidden * 2);
  L.act = take((size_t)L.rows_cap * d.inter * 2);
  L.d = take(Tm * k * d.hidden * 2);
  L.dsh = take(d.has_shared ? Tm * d.hidden * 4 : 0);
  L.total = o;
  return L;
}

moe_status check_desc(const moe_plan_desc* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->hidden <= 0 || d->inter <= 0 || d->num_experts <= 0 || d->top_k <= 0 ||
      d->max_tokens <= 0)
    return MOE_ERR_INVALID_ARG;
  if (d->group_size != kGroup) return MOE_ERR_UNSUPPORTED;
  if (d->block_m != kBM) return MOE_ERR_UNSUPPORTED;
  if (d->hidden % d->group_size || d->inter % d->group_size) return MOE_ERR_INVALID_ARG;
  if (d->hidden % 256 || d->inter % 256) return MOE_ERR_UNSUPPORTED;
  if (d->num_experts % 8 || d->num_experts > 512) return MOE_ERR_UNSUPPORTED;
  if (d->top_k > d->num_experts) return MOE_ERR_INVALID_ARG;
  if (d->top_k > 32) return MOE_ERR_UNSUPPORTED;
  if (d->has_shared != 0 && d->has_shared != 1) return MOE_ERR_INVALID_ARG;
  if (d->gemm_path < 0 || d->gemm_path > 3) return MOE_ERR_INVALID_ARG;
  if (d->gemm_path == 2 && !smallm_fits(d->hidden, d->inter)) return MOE_ERR_UNSUPPORTED;
  if (d->small_m_max_tokens < 0 || d->wait_limit_ms < 0) return MOE_ERR_INVALID_ARG;
  // 32-bit row/element indices inside the kernels
  if ((long long)d->max_tokens * (d->top_k + 1) * d->hidden >= (1LL << 31))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

struct moe_plan {
  moe_plan_desc d;
  int device = 0;
  int num_sms = 0;
  Layout L;
  uint8_t* scratch = nullptr;
  CUtensorMap tm_xs[4], tm_act[4];   // box rows 128, 64, 32, 16
  bool timing = false;
  std::vector<TimedLaunch> timed;
  std::vector<cudaEvent_t> ev_pool;
  int last_path = 0;
  bool tail_split = false;   // tensor-core path: split the last round of units along K
  // encoded uint32 [rows][cols] maps of packed weights, by (base, rows, cols,
  // box rows): a layer's maps are encoded on its first call only
  std::map<std::tuple<const void*, uint64_t, uint64_t, uint32_t>, CUtensorMap> qmaps;
  // weight sets (scales, biases, count) whose fp16 operand range was checked
  std::set<std::tuple<const void*, const void*, size_t>> range_checked;

  // 3D slab map (encode_slab_3d) of a packed-word matrix [rows][K/8], cached
  // under the same table with the top bit of the box height set
  bool qmap3(CUtensorMap* out, const void* base, uint64_t rows, int K, uint32_t box_rows) {
    const auto key = std::make_tuple(base, rows, (uint64_t)K, box_rows | 0x80000000u);
    auto it = qmaps.find(key);
    if (it == qmaps.end()) {
      CUtensorMap m;
      if (!encode_slab_3d(&m, base, rows, K, box_rows)) return false;
      if (qmaps.size() >= 4096) qmaps.clear();
      it = qmaps.emplace(key, m).first;
    }
    *out = it->second;
    return true;
  }

  // router-weight map (encode_router_slices), cached under the same table
  bool rmap(CUtensorMap* out, const void* base, int H, int E) {
    const auto key = std::make_tuple(base, (uint64_t)H, (uint64_t)E, 0x40000000u);
    auto it = qmaps.find(key);
    if (it == qmaps.end()) {
      CUtensorMap m;
      if (!encode_router_slices(&m, base, H, E)) return false;
      if (qmaps.size() >= 4096) qmaps.clear();
      it = qmaps.emplace(key, m).first;
    }
    *out = it->second;
    return true;
  }

  bool qmap(CUtensorMap* out, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    const auto key = std::make_tuple(base, rows, cols, box_rows);
    auto it = qmaps.find(key);
    if (it == qmaps.end()) {
      CUtensorMap m;
      if (!encode_2d(&m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, base, rows, cols, 32, box_rows))
        return false;
      if (qmaps.size() >= 4096) qmaps.clear();
      it = qmaps.emplace(key, m).first;
    }
    *out = it->second;
    return true;
  }

  template <class T>
  T* at(size_t off) const {
    return reinterpret_cast<T*>(scratch + off);
  }
  DevErr err() const {
    DevErr e;
    e.word = at<int>(L.err);
    e.where = at<int>(L.err) + 1;
    e.limit_ns = (unsigned long long)(d.wait_limit_ms > 0 ? d.wait_limit_ms : 1000) * 1000000ull;
    return e;
  }
  cudaEvent_t event() {
    if (!ev_pool.empty()) {
      cudaEvent_t e = ev_pool.back();
      ev_pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};

namespace {

// Runs one launch; when timing is on, brackets it with events on `st`.
template <class F>
cudaError_t timed(moe_plan* p, int kind, cudaStream_t st, F&& launch) {
  if (!p->timing) return launch();
  TimedLaunch t{kind, p->event(), p->event()};
  cudaEventRecord(t.a, st);
  cudaError_t e = launch();
  cudaEventRecord(t.b, st);
  p->timed.push_back(t);
  return e;
}

moe_status st_of(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status check_w4(const moe_w4& m) {
  if (!m.qweight || !m.scales || !m.biases) return MOE_ERR_INVALID_ARG;
  if (!aligned16(m.qweight) || !aligned16(m.scales) || !aligned16(m.biases))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status check_experts(const moe_experts* x) {
  if (!x) return MOE_ERR_INVALID_ARG;
  moe_status s;
  if ((s = check_w4(x->gate)) != MOE_OK) return s;
  if ((s = check_w4(x->up)) != MOE_OK) return s;
  return check_w4(x->down);
}

W4Dev dev(const moe_w4& m) { return W4Dev{m.qweight, m.scales, m.biases}; }

// GEMM path the feed-forward part of a T-token call takes.
int ffn_path(const moe_plan* p, int T) {
  const moe_plan_desc& d = p->d;
  const int small_max = d.small_m_max_tokens > 0 ? d.small_m_max_tokens : 16;
  const int p0 = d.gemm_path == 3 ? 1 : d.gemm_path;
  return p0 != 0 ? p0 : (T <= small_max && smallm_fits(d.hidden, d.inter) ? 2 : 1);
}

// Whether the tensor-core path takes the SM-pair kernel (gemm_path 3, on a
// device that launches clusters).
bool use_pair_gemm(const moe_plan* p) { return p->d.gemm_path == 3 && tc2_supported(); }

// Routing. With `fuse_gather`, a routing launch that can also does the
// gather of the tensor-core path (x rows into the plan's xs) and sets
// *gathered; otherwise *gathered is false.
moe_status route_impl(moe_plan* p, const uint16_t* x, int T, const uint16_t* router_w,
                      const float* router_bias, moe_routing* out, bool want_logits,
                      cudaStream_t st, bool fuse_gather = false, bool* gathered = nullptr) {
  const moe_plan_desc& d = p->d;
  if (gathered) *gathered = false;
  const int nblk = (T + kRouterTB - 1) / kRouterTB;
  float* logits = p->at<float>(p->L.logits);   // the top-k kernel reads them back
  cudaError_t e;
  if (route_small_fits(T, d.hidden, d.num_experts, d.top_k)) {
    e = timed(p, 0, st, [&] {
      return launch_route_small(x, T, d.hidden, router_w, router_bias, d.num_experts, d.top_k,
                                logits, p->at<int32_t>(p->L.topk_idx), p->at<float>(p->L.topk_w),
                                p->at<int32_t>(p->L.cnt), p->at<int32_t>(p->L.off),
                                p->at<int32_t>(p->L.tile_off), p->at<int32_t>(p->L.bmap),
                                p->at<int32_t>(p->L.num_tiles), p->at<int32_t>(p->L.perm),
                                p->at<int32_t>(p->L.inv), p->at<unsigned>(p->L.arrive), st);
    });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  } else if (route_large_fits(T, d.num_experts, d.top_k, p->num_sms)) {
    e = timed(p, 0, st, [&] {
      return launch_router_logits(x, T, d.hidden, router_w, router_bias, d.num_experts, logits,
                                  p->err(), st);
    });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = timed(p, 8, st, [&] {
      unsigned* w = p->at<unsigned>(p->L.arrive);
      return launch_route_large(logits, T, d.num_experts, d.top_k, p->at<int32_t>(p->L.topk_idx),
                                p->at<float>(p->L.topk_w), p->at<uint8_t>(p->L.cnt8),
                                p->at<int32_t>(p->L.cnt), p->at<int32_t>(p->L.off),
                                p->at<int32_t>(p->L.tile_off), p->at<int32_t>(p->L.bmap),
                                p->at<int32_t>(p->L.num_tiles), p->at<int32_t>(p->L.perm),
                                p->at<int32_t>(p->L.inv), w, w + 1, p->err(), x,
                                fuse_gather ? p->at<uint16_t>(p->L.xs) : nullptr, d.hidden,
                                d.has_shared, st);
    });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (gathered) *gathered = fuse_gather;
  } else {
    e = timed(p, 0, st, [&] {
      return launch_router_logits(x, T, d.hidden, router_w, router_bias, d.num_experts, logits,
                                  p->err(), st);
    });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = timed(p, 8, st, [&] {
      return launch_router_select(logits, T, d.num_experts, d.top_k, p->at<int32_t>(p->L.topk_idx),
                                  p->at<float>(p->L.topk_w), p->at<int32_t>(p->L.blk_cnt), st);
    });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = timed(p, 1, st, [&] {
      return launch_route_scan(p->at<int32_t>(p->L.blk_cnt), nblk, T, d.top_k, d.num_experts,
                               p->at<int32_t>(p->L.cnt), p->at<int32_t>(p->L.off),
                               p->at<int32_t>(p->L.tile_off), p->at<int32_t>(p->L.bmap),
                               p->at<int32_t>(p->L.num_tiles), st);
    });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = timed(p, 2, st, [&] {
      return launch_route_scatter(p->at<int32_t>(p->L.topk_idx), p->at<int32_t>(p->L.blk_cnt), T,
                                  d.top_k, d.num_experts, p->at<int32_t>(p->L.perm),
                                  p->at<int32_t>(p->L.inv), st);
    });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (out) {
    out->topk_idx = p->at<int32_t>(p->L.topk_idx);
    out->topk_w = p->at<float>(p->L.topk_w);
    out->counts = p->at<int32_t>(p->L.cnt);
    out->offsets = p->at<int32_t>(p->L.off);
    out->tile_offsets = p->at<int32_t>(p->L.tile_off);
    out->perm = p->at<int32_t>(p->L.perm);
    out->inv = p->at<int32_t>(p->L.inv);
    out->block_map = p->at<int32_t>(p->L.bmap);
    out->num_tiles = p->at<int32_t>(p->L.num_tiles);
    out->logits = want_logits ? logits : nullptr;
  }
  return MOE_OK;
}

// The scales and biases of a weight set are checked against the fp16
// operand range once, on the first call that sees the set (by address), in a
// kernel on the stream; a value out of range latches DEVERR_RANGE.
cudaError_t check_weight_range(moe_plan* p, const moe_experts* routed, const moe_experts* shared,
                               cudaStream_t st) {
  const moe_plan_desc& d = p->d;
  const int H = d.hidden, I = d.inter, E = d.num_experts;
  auto range_check = [&](const moe_w4& m, size_t n) {
    if (p->range_checked.size() >= 4096) p->range_checked.clear();
    if (!p->range_checked.insert(std::make_tuple((const void*)m.scales, (const void*)m.biases, n)).second)
      return cudaSuccess;
    return launch_w4_range_check(m.scales, m.biases, n, p->err(), p->num_sms, st);
  };
  const size_t n_gu = (size_t)I * (H / kGroup), n_dn = (size_t)H * (I / kGroup);
  cudaError_t e = cudaSuccess;
  for (int i = 0; i < 3 && e == cudaSuccess; ++i) {
    const moe_w4& m = i == 0 ? routed->gate : i == 1 ? routed->up : routed->down;
    e = range_check(m, (i < 2 ? n_gu : n_dn) * E);
    if (e == cudaSuccess && d.has_shared && shared) {
      const moe_w4& ms = i == 0 ? shared->gate : i == 1 ? shared->up : shared->down;
      e = range_check(ms, i < 2 ? n_gu : n_dn);
    }
  }
  return e;
}

// Whether a T-token chunk of moe_forward_stack takes the fused decode layer.
bool use_decode_fused(const moe_plan* p, int T) {
  const moe_plan_desc& d = p->d;
  return ffn_path(p, T) == 2 &&
         decode_fused_fits(T, d.hidden, d.inter, d.num_experts, d.top_k, d.has_shared, p->num_sms);
}

// One layer of a decode-sized chunk in one launch: x = bf16(x + alpha *
// moe(rmsnorm(x))); the routing lands in the plan's routing arrays and y (FP32)
// in the shared-output buffer, for inspection.
moe_status decode_layer_impl(moe_plan* p, uint16_t* x, int T, const moe_layer& Ly, float alpha,
                             cudaStream_t st) {
  const moe_plan_desc& d = p->d;
  const int H = d.hidden, I = d.inter, E = d.num_experts;
  const moe_experts* shared = d.has_shared ? &Ly.shared : nullptr;
  if (check_weight_range(p, &Ly.routed, shared, st) != cudaSuccess) return MOE_ERR_CUDA;
  DecodeLayerArgs a;
  a.T = T;
  a.H = H;
  a.I = I;
  a.E = E;
  a.k = d.top_k;
  a.has_shared = d.has_shared;
  a.alpha = alpha;
  a.eps = kRmsEps;
  a.x = x;
  a.router_w = Ly.router_w;
  a.router_bias = Ly.router_bias;
  a.gate = dev(Ly.routed.gate);
  a.up = dev(Ly.routed.up);
  a.down = dev(Ly.routed.down);
  const moe_experts& sh = d.has_shared ? Ly.shared : Ly.routed;
  a.sgate = dev(sh.gate);
  a.sup = dev(sh.up);
  a.sdown = dev(sh.down);
  const uint64_t er = d.has_shared ? 1 : (uint64_t)E;
  // 3D slabs, all K: 8 rows for a gate/up warp's unit, 16 down rows per CTA
  bool ok = p->qmap3(&a.maps[0], Ly.routed.gate.qweight, (uint64_t)E * I, H, 8) &&
            p->qmap3(&a.maps[1], Ly.routed.up.qweight, (uint64_t)E * I, H, 8) &&
            p->qmap3(&a.maps[2], Ly.routed.down.qweight, (uint64_t)E * H, I, 16) &&
            p->qmap3(&a.maps[3], sh.gate.qweight, er * I, H, 8) &&
            p->qmap3(&a.maps[4], sh.up.qweight, er * I, H, 8) &&
            p->qmap3(&a.maps[5], sh.down.qweight, er * H, I, 16) &&
            p->rmap(&a.router_map, Ly.router_w, H, E);
  if (!ok) return MOE_ERR_CUDA;
  a.act = p->at<uint16_t>(p->L.act);
  a.topk_idx = p->at<int32_t>(p->L.topk_idx);
  a.topk_w = p->at<float>(p->L.topk_w);
  a.y_out = d.has_shared ? p->at<float>(p->L.dsh) : nullptr;
  a.bar = p->at<unsigned>(p->L.arrive) + 2;
  a.epoch = p->at<unsigned>(p->L.arrive) + 3;
  a.tlogits = p->at<unsigned long long>(p->L.tlogits);
  p->last_path = 3;
  return st_of(timed(p, 9, st, [&] { return launch_decode_layer(a, p->err(), p->num_sms, st); }));
}

// The stack update fused into the combine (moe_forward_layer_residual).
struct ResidualUpdate {
  float alpha;
  uint16_t* x;    // residual stream, updated in place
  uint16_t* xn;   // next layer's RMS-normalised input
};

// Exactly one of y (the block output) and res (the fused stack update) is set.
// `pre_gathered`: the routing launch already wrote the gathered rows.
moe_status ffn_impl(moe_plan* p, const uint16_t* x, int T, const moe_routing* r,
                    const moe_experts* routed, const moe_experts* shared, float* y,
                    const ResidualUpdate* res, cudaStream_t st, bool pre_gathered = false) {
  const moe_plan_desc& d = p->d;
  const int H = d.hidden, I = d.inter, E = d.num_experts, k = d.top_k;
  const int hs = d.has_shared;
  const int path = ffn_path(p, T);
  p->last_path = path == 1 && use_pair_gemm(p) ? 4 : path;

  cudaError_t e = check_weight_range(p, routed, shared, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;

  // the tensor-core path reads gathered rows with TMA; the small-M path reads
  // the token rows itself
  if (path == 1 && !pre_gathered) {
    e = timed(p, 3, st, [&] {
      return launch_gather_rows(x, r->perm, T, k, H, hs, p->at<uint16_t>(p->L.xs), p->err(), st);
    });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }

  long long bound = ((long long)T * k + kBM - 1) / kBM + E;
  if (bound > (long long)T * k) bound = (long long)T * k;

  GemmProblem g{};
  g.T = T;
  g.k = k;
  g.E = E;
  g.has_shared = hs;
  g.bmap = r->block_map;
  g.num_tiles = r->num_tiles;
  g.max_routed_tiles = (int)bound;
  g.topk_w = r->topk_w;
  g.perm = r->perm;
  if (p->tail_split) {
    g.sk_ws = p->at<float>(p->L.sk_ws);
    g.sk_cnt = p->at<unsigned>(p->L.sk_cnt);
    g.sk_slots = kSplitSlots;
  }

  // gate/up: B = xs [rows][H], out = act [rows][I]
  GemmProblem g0 = g;
  g0.K = H;
  g0.N = I;
  g0.act_in = p->at<uint16_t>(p->L.xs);
  g0.gather_x = path == 2 ? x : nullptr;
  g0.out = p->at<uint16_t>(p->L.act);
  g0.out_ld = I;
  g0.w0 = dev(routed->gate);
  g0.w1 = dev(routed->up);
  if (hs) {
    g0.sw0 = dev(shared->gate);
    g0.sw1 = dev(shared->up);
  }
  if (path == 2) {   // the small-M gate/up pass prefetches the down rows into L2
    g0.next = dev(routed->down);
    if (hs) g0.snext = dev(shared->down);
    g0.next_K = I;
  }
  // down: B = act [rows][I], out = d [rows][H]
  GemmProblem g1 = g;
  g1.K = I;
  g1.N = H;
  g1.act_in = p->at<uint16_t>(p->L.act);
  g1.out = p->at<uint16_t>(p->L.d);
  g1.out_sh = hs ? p->at<float>(p->L.dsh) : nullptr;
  g1.out_ld = H;
  g1.w0 = dev(routed->down);
  g1.w1 = dev(routed->down);
  if (hs) {
    g1.sw0 = dev(shared->down);
    g1.sw1 = dev(shared->down);
  }

  if (path == 1) {
    TcMaps m0{}, m1{};
    for (int i = 0; i < 4; ++i) {
      m0.b[i] = p->tm_xs[i];
      m1.b[i] = p->tm_act[i];
    }
    bool ok = p->qmap(&m0.q0, routed->gate.qweight, (uint64_t)E * I, H / 8, 128) &&
              p->qmap(&m0.q1, routed->up.qweight, (uint64_t)E * I, H / 8, 128) &&
              p->qmap(&m1.q0, routed->down.qweight, (uint64_t)E * H, I / 8, 128);
    m1.q1 = m1.q0;
    if (ok && hs) {
      ok = p->qmap(&m0.sq0, shared->gate.qweight, I, H / 8, 128) &&
           p->qmap(&m0.sq1, shared->up.qweight, I, H / 8, 128) &&
           p->qmap(&m1.sq0, shared->down.qweight, H, I / 8, 128);
      m1.sq1 = m1.sq0;
    } else if (ok) {
      m0.sq0 = m0.q0;
      m0.sq1 = m0.q1;
      m1.sq0 = m1.sq1 = m1.q0;
    }
    if (!ok) return MOE_ERR_CUDA;
    if (use_pair_gemm(p)) {
      // 256-row tiles from the routing offsets, then both passes on SM pairs
      // (gate/up weight boxes of 64 rows: each CTA takes 64 gate + 64 up rows)
      int32_t* bmap2 = p->at<int32_t>(p->L.bmap2);
      int32_t* nt2 = p->at<int32_t>(p->L.num_tiles2);
      e = timed(p, 1, st, [&] { return launch_build_tiles256(r->offsets, E, bmap2, nt2, st); });
      if (e != cudaSuccess) return MOE_ERR_CUDA;
      TcMaps p0 = m0;
      ok = p->qmap(&p0.q0, routed->gate.qweight, (uint64_t)E * I, H / 8, 64) &&
           p->qmap(&p0.q1, routed->up.qweight, (uint64_t)E * I, H / 8, 64);
      if (ok && hs)
        ok = p->qmap(&p0.sq0, shared->gate.qweight, I, H / 8, 64) &&
             p->qmap(&p0.sq1, shared->up.qweight, I, H / 8, 64);
      if (!ok) return MOE_ERR_CUDA;
      if (!hs) {
        p0.sq0 = p0.q0;
        p0.sq1 = p0.q1;
      }
      long long bound2 = ((long long)T * k + 255) / 256 + E;
      if (bound2 > (long long)T * k) bound2 = (long long)T * k;
      e = timed(p, 4, st, [&] {
        return launch_gemm_tc2(0, g0, p0, bmap2, nt2, (int)bound2, p->err(), p->num_sms, st);
      });
      if (e != cudaSuccess) return MOE_ERR_CUDA;
      e = timed(p, 5, st, [&] {
        return launch_gemm_tc2(1, g1, m1, bmap2, nt2, (int)bound2, p->err(), p->num_sms, st);
      });
      if (e != cudaSuccess) return MOE_ERR_CUDA;
    } else {
      e = timed(p, 4, st, [&] { return launch_gemm_tc(0, g0, m0, p->err(), p->num_sms, st); });
      if (e != cudaSuccess) return MOE_ERR_CUDA;
      e = timed(p, 5, st, [&] { return launch_gemm_tc(1, g1, m1, p->err(), p->num_sms, st); });
      if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
  } else {
    const uint32_t r0 = smallm_rows_per_unit(0), r1 = smallm_rows_per_unit(1);
    SmallMaps s0{}, s1{};
    bool ok = p->qmap(&s0.q0, routed->gate.qweight, (uint64_t)E * I, H / 8, r0) &&
              p->qmap(&s0.q1, routed->up.qweight, (uint64_t)E * I, H / 8, r0) &&
              p->qmap(&s1.q0, routed->down.qweight, (uint64_t)E * H, I / 8, r1);
    s1.q1 = s1.q0;
    if (ok && hs) {
      ok = p->qmap(&s0.sq0, shared->gate.qweight, I, H / 8, r0) &&
           p->qmap(&s0.sq1, shared->up.qweight, I, H / 8, r0) &&
           p->qmap(&s1.sq0, shared->down.qweight, H, I / 8, r1);
      s1.sq1 = s1.sq0;
    } else if (ok) {
      s0.sq0 = s0.q0;
      s0.sq1 = s0.q1;
      s1.sq0 = s1.sq1 = s1.q0;
    }
    if (!ok) return MOE_ERR_CUDA;
    e = timed(p, 4, st, [&] { return launch_gemm_smallm(0, g0, s0, p->err(), p->num_sms, st); });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = timed(p, 5, st, [&] { return launch_gemm_smallm(1, g1, s1, p->err(), p->num_sms, st); });
    if (e != cudaSuccess) return MOE_ERR_CUDA;
  }
  e = timed(p, 6, st, [&] {
    if (res)
      return launch_combine_residual_norm(p->at<uint16_t>(p->L.d),
                                          hs ? p->at<float>(p->L.dsh) : nullptr, r->inv, T, k, H,
                                          res->alpha, res->x, res->xn, kRmsEps, st);
    return launch_combine(p->at<uint16_t>(p->L.d), hs ? p->at<float>(p->L.dsh) : nullptr,
                          r->inv, T, k, H, y, st);
  });
  return st_of(e);
}

moe_status check_T(const moe_plan* p, int T) {
  if (T < 1) return MOE_ERR_INVALID_ARG;
  if (T > p->d.max_tokens) return MOE_ERR_CAPACITY;
  return MOE_OK;
}

moe_status check_route_args(const moe_plan* p, const uint16_t* x, int T, const uint16_t* rw,
                            const float* rb) {
  moe_status s = check_T(p, T);
  if (s != MOE_OK) return s;
  if (!x || !rw || !aligned16(x) || !aligned16(rw)) return MOE_ERR_INVALID_ARG;
  if (rb && (reinterpret_cast<uintptr_t>(rb) & 3u)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status check_ffn_args(const moe_plan* p, const uint16_t* x, int T, const moe_routing* r,
                          const moe_experts* routed, const moe_experts* shared,
                          const float* y) {
  moe_status s = check_T(p, T);
  if (s != MOE_OK) return s;
  if (!x || !y || !aligned16(x) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  const size_t xbytes = (size_t)T * p->d.hidden * 2, ybytes = (size_t)T * p->d.hidden * 4;
  const uint8_t* xb = reinterpret_cast<const uint8_t*>(x);
  const uint8_t* yb = reinterpret_cast<const uint8_t*>(y);
  if (xb < yb + ybytes && yb < xb + xbytes) return MOE_ERR_INVALID_ARG;   // y overlaps x
  if ((s = check_experts(routed)) != MOE_OK) return s;
  if (p->d.has_shared) {
    if ((s = check_experts(shared)) != MOE_OK) return s;
  } else if (shared) {
    return MOE_ERR_INVALID_ARG;
  }
  if (r && (!r->topk_w || !r->perm || !r->inv || !r->block_map || !r->num_tiles))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_plan_scratch_bytes(const moe_plan_desc* desc, size_t* bytes) {
  moe_status s = check_desc(desc);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = make_layout(*desc).total;
  return MOE_OK;
}

moe_status moe_plan_create(const moe_plan_desc* desc, int device, moe_plan_t* out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  moe_status s = check_desc(desc);
  if (s != MOE_OK) return s;
  if (device < 0) return MOE_ERR_INVALID_ARG;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device >= ndev) return MOE_ERR_CUDA;
  int prev = 0;
  cudaGetDevice(&prev);
  if (cudaSetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return MOE_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) {   // kernels are built for sm_103a only
    cudaSetDevice(prev);
    return MOE_ERR_UNSUPPORTED;
  }
  moe_plan* p = new moe_plan();
  p->d = *desc;
  p->device = device;
  p->num_sms = prop.multiProcessorCount;
  p->L = make_layout(*desc);
  if (cudaMalloc(&p->scratch, p->L.total) != cudaSuccess) {
    delete p;
    cudaSetDevice(prev);
    return MOE_ERR_CUDA;
  }
  cudaMemset(p->scratch + p->L.err, 0, 16);
  cudaMemset(p->scratch + p->L.arrive, 0, 16);
  cudaMemset(p->scratch + p->L.tlogits, 0, tlogits_bytes(*desc));
  cudaMemset(p->scratch + p->L.sk_cnt, 0, kSplitSlots * 4);
  bool ok = true;
  for (int i = 0; i < 4 && ok; ++i) {
    const uint32_t box_rows = 128u >> i;
    ok = encode_2d(&p->tm_xs[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p->at<uint16_t>(p->L.xs),
                   p->L.rows_cap, desc->hidden, 64, box_rows) &&
         encode_2d(&p->tm_act[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                   p->at<uint16_t>(p->L.act), p->L.rows_cap, desc->inter, 64, box_rows);
  }
  if (!ok || cudaDeviceSynchronize() != cudaSuccess) {
    cudaFree(p->scratch);
    delete p;
    cudaSetDevice(prev);
    return MOE_ERR_CUDA;
  }
  cudaSetDevice(prev);
  *out = p;
  return MOE_OK;
}

moe_status moe_plan_destroy(moe_plan_t p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(p->device);
  cudaDeviceSynchronize();
  for (auto& t : p->timed) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  for (auto e : p->ev_pool) cudaEventDestroy(e);
  cudaFree(p->scratch);
  cudaSetDevice(prev);
  delete p;
  return MOE_OK;
}

moe_status moe_route(moe_plan_t p, const uint16_t* x, int T, const uint16_t* router_w,
                     const float* router_bias, moe_routing* out, moe_stream_t stream) {
  if (!p || !out) return MOE_ERR_INVALID_ARG;
  moe_status s = check_route_args(p, x, T, router_w, router_bias);
  if (s != MOE_OK) return s;
  return route_impl(p, x, T, router_w, router_bias, out, true,
                    reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_grouped_w4_ffn(moe_plan_t p, const uint16_t* x, int T, const moe_routing* r,
                              const moe_experts* routed, const moe_experts* shared, float* y,
                              moe_stream_t stream) {
  if (!p || !r) return MOE_ERR_INVALID_ARG;
  moe_status s = check_ffn_args(p, x, T, r, routed, shared, y);
  if (s != MOE_OK) return s;
  return ffn_impl(p, x, T, r, routed, shared, y, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

moe_status moe_forward_layer(moe_plan_t p, const uint16_t* x, int T, const uint16_t* router_w,
                             const float* router_bias, const moe_experts* routed,
                             const moe_experts* shared, float* y, moe_stream_t stream) {
  if (!p) return MOE_ERR_INVALID_ARG;
  moe_status s = check_route_args(p, x, T, router_w, router_bias);
  if (s != MOE_OK) return s;
  s = check_ffn_args(p, x, T, nullptr, routed, shared, y);
  if (s != MOE_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  moe_routing r;
  bool gathered = false;
  s = route_impl(p, x, T, router_w, router_bias, &r, false, st, ffn_path(p, T) == 1, &gathered);
  if (s != MOE_OK) return s;
  return ffn_impl(p, x, T, &r, routed, shared, y, nullptr, st, gathered);
}

moe_status moe_forward_layer_residual(moe_plan_t p, const uint16_t* xn, int T,
                                      const uint16_t* router_w, const float* router_bias,
                                      const moe_experts* routed, const moe_experts* shared,
                                      float alpha, uint16_t* x, uint16_t* xn_out,
                                      moe_stream_t stream) {
  if (!p) return MOE_ERR_INVALID_ARG;
  moe_status s = check_route_args(p, xn, T, router_w, router_bias);
  if (s != MOE_OK) return s;
  if (!x || !xn_out || !aligned16(x) || !aligned16(xn_out) || x == xn || x == xn_out)
    return MOE_ERR_INVALID_ARG;
  if ((s = check_experts(routed)) != MOE_OK) return s;
  if (p->d.has_shared) {
    if ((s = check_experts(shared)) != MOE_OK) return s;
  } else if (shared) {
    return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  moe_routing r;
  bool gathered = false;
  s = route_impl(p, xn, T, router_w, router_bias, &r, false, st, ffn_path(p, T) == 1, &gathered);
  if (s != MOE_OK) return s;
  const ResidualUpdate res{alpha, x, xn_out};
  return ffn_impl(p, xn, T, &r, routed, shared, nullptr, &res, st, gathered);
}

moe_status moe_forward_stack(moe_plan_t p, uint16_t* x, uint16_t* xn, int T,
                             const moe_layer* layers, int num_layers, float alpha,
                             moe_stream_t stream) {
  if (!p || !x || !xn || !layers || num_layers < 1 || T < 1) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(xn) || x == xn) return MOE_ERR_INVALID_ARG;
  const int H = p->d.hidden, chunk = p->d.max_tokens;
  // the stream and xn must not overlap (xn holds one chunk)
  const uint8_t *xb = reinterpret_cast<const uint8_t*>(x), *nb = reinterpret_cast<const uint8_t*>(xn);
  const size_t xbytes = (size_t)T * H * 2, nbytes = (size_t)(T < chunk ? T : chunk) * H * 2;
  if (xb < nb + nbytes && nb < xb + xbytes) return MOE_ERR_INVALID_ARG;
  moe_status s;
  for (int l = 0; l < num_layers; ++l) {
    const moe_layer& L = layers[l];
    if (!L.router_w || !aligned16(L.router_w)) return MOE_ERR_INVALID_ARG;
    if (L.router_bias && (reinterpret_cast<uintptr_t>(L.router_bias) & 3u)) return MOE_ERR_INVALID_ARG;
    if ((s = check_experts(&L.routed)) != MOE_OK) return s;
    if (p->d.has_shared && (s = check_experts(&L.shared)) != MOE_OK) return s;
  }
  for (int c0 = 0; c0 < T; c0 += chunk) {
    const int Tc = T - c0 < chunk ? T - c0 : chunk;
    uint16_t* xc = x + (size_t)c0 * H;
    if (use_decode_fused(p, Tc)) {
      // decode-sized chunk: one launch per layer (the norm is taken inside),
      // then the chunk's normalised stream for the caller
      cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
      for (int l = 0; l < num_layers; ++l)
        if ((s = decode_layer_impl(p, xc, Tc, layers[l], alpha, st)) != MOE_OK)
          return s;
      if ((s = moe_residual_add(p, xc, nullptr, Tc, 0.f, xc, xn, stream)) != MOE_OK) return s;
      continue;
    }
    if ((s = moe_residual_add(p, xc, nullptr, Tc, 0.f, xc, xn, stream)) != MOE_OK) return s;
    for (int l = 0; l < num_layers; ++l) {
      const moe_layer& L = layers[l];
      s = moe_forward_layer_residual(p, xn, Tc, L.router_w, L.router_bias, &L.routed,
                                     p->d.has_shared ? &L.shared : nullptr, alpha, xc, xn, stream);
      if (s != MOE_OK) return s;
    }
  }
  return MOE_OK;
}

moe_status moe_residual_add(moe_plan_t p, const uint16_t* x, const float* y, int T,
                            float alpha, uint16_t* x_out, uint16_t* xn_out, moe_stream_t stream) {
  if (!p || !x) return MOE_ERR_INVALID_ARG;
  moe_status s = check_T(p, T);
  if (s != MOE_OK) return s;
  if (!x_out) x_out = const_cast<uint16_t*>(x);
  if (!aligned16(x) || !aligned16(x_out) || (y && !aligned16(y)) || (xn_out && !aligned16(xn_out)))
    return MOE_ERR_INVALID_ARG;
  if (!y && !xn_out && x_out == x) return MOE_OK;
  if (xn_out && (xn_out == x || xn_out == x_out)) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  return st_of(timed(p, 7, st, [&] {
    return launch_residual_norm(x, y, T, p->d.hidden, alpha, x_out, xn_out, kRmsEps, st);
  }));
}

moe_status moe_get_error(moe_plan_t p) {
  if (!p) return MOE_ERR_INVALID_ARG;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(p->device);
  int h[2] = {0, 0};
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(h, p->at<int>(p->L.err), 8, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(p->at<int>(p->L.err), 0, 8);
  // a launch that gave up at a barrier leaves its arrival counters set, and
  // the fused layer's launch count and tagged logits may disagree
  if (e == cudaSuccess && (h[0] & DEVERR_TIMEOUT_BIT)) e = cudaMemset(p->at<int>(p->L.arrive), 0, 16);
  if (e == cudaSuccess && (h[0] & DEVERR_TIMEOUT_BIT))
    e = cudaMemset(p->scratch + p->L.tlogits, 0, tlogits_bytes(p->d));
  // so may the split last round's counters of a GEMM that gave up
  if (e == cudaSuccess && (h[0] & DEVERR_TIMEOUT_BIT))
    e = cudaMemset(p->scratch + p->L.sk_cnt, 0, kSplitSlots * 4);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  cudaSetDevice(prev);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (h[0] & DEVERR_TIMEOUT_BIT) return MOE_ERR_DEVICE_TIMEOUT;
  if (h[0] & DEVERR_RANGE_BIT) return MOE_ERR_OPERAND_RANGE;
  return MOE_OK;
}

moe_status moe_debug_wait_timeout(moe_plan_t p, int limit_us, moe_stream_t stream) {
  if (!p || limit_us <= 0 || limit_us > 10000000) return MOE_ERR_INVALID_ARG;
  DevErr e = p->err();
  e.limit_ns = (unsigned long long)limit_us * 1000ull;
  return st_of(launch_debug_wait(e, reinterpret_cast<cudaStream_t>(stream)));
}

moe_status moe_set_tail_split(moe_plan_t p, int on) {
  if (!p) return MOE_ERR_INVALID_ARG;
  p->tail_split = on != 0;
  return MOE_OK;
}

moe_status moe_enable_timing(moe_plan_t p, int on) {
  if (!p) return MOE_ERR_INVALID_ARG;
  p->timing = on != 0;
  return MOE_OK;
}

moe_status moe_read_timing(moe_plan_t p, moe_timing* out) {
  if (!p || !out) return MOE_ERR_INVALID_ARG;
  memset(out, 0, sizeof(*out));
  moe_status s = MOE_OK;
  for (auto& t : p->timed) {
    if (cudaEventSynchronize(t.b) != cudaSuccess) s = MOE_ERR_CUDA;
    float ms = 0.f;
    if (s == MOE_OK && cudaEventElapsedTime(&ms, t.a, t.b) == cudaSuccess) {
      out->ms[t.kind] += ms;
      out->launches[t.kind] += 1;
    }
    p->ev_pool.push_back(t.a);
    p->ev_pool.push_back(t.b);
  }
  p->timed.clear();
  return s;
}

int moe_last_gemm_path(moe_plan_t p) { return p ? p->last_path : 0; }

void* moe_debug_buffer(moe_plan_t p, int which) {
  if (!p) return nullptr;
  switch (which) {
    case 0: return p->scratch + p->L.xs;
    case 1: return p->scratch + p->L.act;
    case 2: return p->scratch + p->L.d;
    case 3: return p->d.has_shared ? p->scratch + p->L.dsh : nullptr;
  }
  return nullptr;
}

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_CAPACITY: return "T above plan capacity";
    case MOE_ERR_DEVICE_TIMEOUT: return "device bounded wait timed out";
    case MOE_ERR_OPERAND_RANGE: return "operand outside the fp16 range of the MMAs";
  }
  return "unknown status";
}

int moe_version(void) { return 200; }

}  // extern "C"
