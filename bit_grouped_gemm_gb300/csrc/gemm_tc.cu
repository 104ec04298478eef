// gemm_tc.cu -- grouped W4A16 expert GEMM on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA) for sm_103a.
//
// The grouped GEMM with block-wise fused dequantisation of "Perplexity libera
// Lily, un motor de IA que supera a MLX-LM en Apple Silicon"
// (diariobitcoin.com), section "Las optimizaciones en el prefill": packed
// 4-bit weights are rebuilt block by block on chip, the rebuilt values never
// reach device memory, and products accumulate in FP32. The packed format is
// the one of section "Qwen3.6 combina tres cargas de trabajo" (groups of 64,
// one bf16 scale and one bf16 bias per group).
//
// GB300 design (not the pages' Metal design):
//   * the weights are the MMA's M side: a unit is a 128-token tile of one
//     expert (a block-map tile) times two 128-row weight blocks (gate and up
//     rows n0..n0+127 for the gate/up pass; rows n0..n0+255 of down for the
//     down pass), K swept in chunks of 64 (one quantisation group);
//   * packed weight tiles arrive by TMA (128-byte swizzle) into shared
//     memory; 8 dequant warps turn each thread's 64 nibbles of one weight row
//     into fp16 (one fused multiply-add, one rounding) and store them with
//     tcgen05.st straight into tensor memory, where the MMA reads them as its
//     A operand -- rebuilt weights never touch shared or global memory;
//   * token activations (the B operand, N = tile rows rounded up to 16) come
//     by TMA in the canonical 128-byte-swizzled K-major layout;
//   * MMA operands are fp16: the bf16 activations are converted exactly (the
//     block's input is RMS-normalised, far inside fp16's range) when they are
//     gathered, and fp16's 11-bit significand keeps the rounding of the
//     dequantised weights and SwiGLU activations 8x below bf16's;
//   * one thread issues tcgen05.mma (M=128, K=16, fp16 in, fp32 in TMEM) for
//     both weight blocks; 8 epilogue warps, two per TMEM lane quarter taking
//     alternate 32-token groups, read the accumulators back with tcgen05.ld
//     and apply SwiGLU (gate/up) or the top-k weight (down);
//   * persistent CTAs (one per SM, 512 TMEM columns each) walk the units;
//     the number of units is read from device memory, never from the host;
//   * optionally (the kSplit instantiation, which the plan selects), the
//     last, partial round of units is split along K when it would leave at
//     least half the SMs idle: each of its units goes to two CTAs, one K
//     half each, which write their fp32 partial sums to device memory; the
//     CTA that arrives second at the unit's counter copies the other half's
//     sums into shared memory, adds them to its own (the same bits whichever
//     CTA that is) and runs the epilogue.
// Every wait is bounded: on timeout the CTA latches an error, drains its own
// TMA copies and MMAs, frees TMEM and exits.
#include "moe_common.cuh"

namespace moe {
namespace tc {

constexpr int kThreads = 640;             // 20 warps
constexpr int kBStages = 6;               // activation chunks (64 K) in flight
constexpr int kQStages = 3;               // packed-weight chunks (256 K) in flight
constexpr int kAStages = 4;               // TMEM weight stages (64 K)
constexpr int kBTileBytes = 128 * 128;    // 128 token rows x 64 fp16
constexpr int kQTileBytes = 128 * 128;    // 128 weight rows x 32 words
constexpr int kQStageBytes = 2 * kQTileBytes;
constexpr int kOffB = 0;
constexpr int kOffQ = kOffB + kBStages * kBTileBytes;
constexpr int kOffW = kOffQ + kQStages * kQStageBytes;   // epilogue row weights [8][128]
constexpr int kOffX = kOffW + 8 * 128 * 4;               // epilogue transpose [8][32 x 32 fp16]
constexpr int kOffBar = kOffX + 8 * 2048;
constexpr int kSmemBytes = kOffBar + 512 + 1024;   // barriers + alignment slack
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol0 = 0, kAccCol1 = 128, kAStageCol = 256;

struct Params {
  TcMaps maps;
  int mode;             // 0: gate/up + SwiGLU, 1: down * top-k weight
  int T, k, E, K, N;
  int nblk;             // units per tile
  int has_shared;
  const int32_t* bmap;
  const int32_t* num_tiles;
  W4Dev w0, w1, sw0, sw1;
  uint16_t* out;
  float* out_sh;
  int out_ld;
  const float* topk_w;
  const int32_t* perm;
  float* sk_ws;         // split last round: fp32 partials, one slot per CTA
  unsigned* sk_cnt;     // split last round: arrivals per unit (zero between launches)
  int sk_slots;         // slots in sk_ws (0: no split)
  DevErr err;
};

// One slot of split partial sums: [weight block][token][row] fp32.
constexpr int kSlotFloats = 2 * kBM * 128;
static_assert(kSlotFloats * 4 == (int)kSplitSlotBytes, "split slot size");

// A CTA's k-th work item: unit u, 256-K weight stages [q0, q1), piece `piece`
// of `pieces`. The full rounds deal whole units (unit k * grid + CTA); in the
// last round r units are left for the grid's G CTAs, and when r <= G / 2 each
// is cut into 2 pieces (K halves), piece i of unit t on CTA 2 t + i. Two
// pieces make the sum order-free: fp32 addition is commutative, so the unit
// gets the same bits whichever piece's CTA adds them.
struct Item {
  int u, q0, q1, piece, pieces;
};

__device__ __forceinline__ int tail_pieces(const Params& p, int r, int nq) {
  const int G = gridDim.x;
  if (r == 0 || G > p.sk_slots) return 1;
  return G / r >= 2 && nq >= 2 ? 2 : 1;
}

__device__ __forceinline__ bool item_at(const Params& p, int k, int units, int nq, Item& it) {
  const int G = gridDim.x, b = blockIdx.x, R = units / G, r = units - R * G;
  if (k < R) {
    it = {k * G + b, 0, nq, 0, 1};
    return true;
  }
  if (k > R || r == 0) return false;
  const int s = tail_pieces(p, r, nq);
  if (b >= r * s) return false;
  const int t = b / s, i = b - t * s;
  it = {R * G + t, i * nq / s, (i + 1) * nq / s, i, s};
  return true;
}

// A CTA's walk over its work items, the same in every role. Without the
// split: units blockIdx.x, blockIdx.x + grid, ..., each over all K; with
// it: the items of item_at.
template <bool kSplit>
struct Deal;

template <>
struct Deal<false> {
  int u, units, nq;
  __device__ __forceinline__ Deal(const Params&, int units_, int nq_) : u(blockIdx.x), units(units_), nq(nq_) {}
  __device__ __forceinline__ bool valid() const { return u < units; }
  __device__ __forceinline__ int unit() const { return u; }
  __device__ __forceinline__ int q_begin() const { return 0; }
  __device__ __forceinline__ int q_end() const { return nq; }
  __device__ __forceinline__ int pieces() const { return 1; }
  __device__ __forceinline__ int next_unit() const { return u + (int)gridDim.x; }   // may be >= units
  __device__ __forceinline__ bool has_next() const { return u + (int)gridDim.x < units; }
  __device__ __forceinline__ int next_q_begin() const { return 0; }
  __device__ __forceinline__ void advance() { u += gridDim.x; }
};

template <>
struct Deal<true> {
  const Params& p;
  int units, nq, k;
  Item cur, nxt;
  bool has, hn;
  __device__ __forceinline__ Deal(const Params& p_, int units_, int nq_)
      : p(p_), units(units_), nq(nq_), k(0) {
    has = item_at(p, 0, units, nq, cur);
    hn = has && item_at(p, 1, units, nq, nxt);
  }
  __device__ __forceinline__ bool valid() const { return has; }
  __device__ __forceinline__ int unit() const { return has ? cur.u : units; }
  __device__ __forceinline__ int q_begin() const { return cur.q0; }
  __device__ __forceinline__ int q_end() const { return cur.q1; }
  __device__ __forceinline__ int pieces() const { return cur.pieces; }
  __device__ __forceinline__ int next_unit() const { return hn ? nxt.u : units; }
  __device__ __forceinline__ bool has_next() const { return hn; }
  __device__ __forceinline__ int next_q_begin() const { return hn ? nxt.q0 : 0; }
  __device__ __forceinline__ void advance() {
    cur = nxt;
    has = hn;
    ++k;
    hn = has && item_at(p, k + 1, units, nq, nxt);
  }
};

struct Unit {
  int e, m0, rows, j;
  bool shared;
};

// The block-map entry of unit u (zeros for a shared-expert unit), fetched a
// unit ahead so that its global-load latency hides behind the current unit.
struct UnitRaw {
  int e, m0, rows;
};

__device__ __forceinline__ UnitRaw fetch_unit(const Params& p, int u, int n_routed) {
  UnitRaw r = {0, 0, 0};
  const int tile = u / p.nblk;
  if (tile < n_routed) {
    const int32_t* m = p.bmap + 3 * (size_t)tile;
    r.e = __ldg(m);
    r.m0 = __ldg(m + 1);
    r.rows = __ldg(m + 2);
  }
  return r;
}

__device__ __forceinline__ Unit make_unit(const Params& p, int u, int n_routed, const UnitRaw& raw) {
  Unit r;
  const int tile = u / p.nblk;
  r.j = u - tile * p.nblk;
  if (tile < n_routed) {
    r.e = raw.e;
    r.m0 = raw.m0;
    r.rows = raw.rows;
    r.shared = false;
  } else {
    const int i = tile - n_routed;
    r.e = 0;
    r.m0 = p.T * p.k + kBM * i;
    r.rows = min(kBM, p.T - kBM * i);
    r.shared = true;
  }
  return r;
}

// first weight row of block `blk` of unit j
__device__ __forceinline__ int block_row0(const Params& p, int j, int blk) {
  return p.mode == 0 ? 128 * j : 256 * j + 128 * blk;
}

#ifdef MOE_TC_STATS
// Profiling build only: cycles each role spends in each wait site, and in
// total, summed over CTAs (read with moe_debug_tc_stats). Each CTA sums in
// shared memory and adds its totals to the global counters once, at exit.
__device__ unsigned long long g_tc_stats[64];   // [mode*32 + site], roles at +16
__shared__ unsigned long long s_tc_stats[32];
#define TC_STAT_BEGIN() const long long tc_t0 = clock64()
#define TC_STAT_END(site) atomicAdd(&s_tc_stats[(site)], (unsigned long long)(clock64() - tc_t0))
#else
#define TC_STAT_BEGIN()
#define TC_STAT_END(site)
#endif

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          const DevErr& err, int site, int = 0) {
  TC_STAT_BEGIN();
  bool ok = mbar_wait(bar, parity, abort_flag, err.limit_ns);
  ok = __all_sync(0xffffffffu, ok);
#ifdef MOE_TC_STATS
  if ((threadIdx.x & 31) == 0) TC_STAT_END(site);
#endif
  if (!ok) {
    if ((threadIdx.x & 31) == 0 && !*abort_flag) report_timeout(err, site);
    *abort_flag = 1;
  }
  return ok;
}

template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1) w4_grouped_gemm_tc(const __grid_constant__ Params p) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* smem_b = smem + kOffB;
  uint8_t* smem_q = smem + kOffQ;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* b_full = bars;
  uint64_t* b_empty = b_full + kBStages;
  uint64_t* q_full = b_empty + kBStages;
  uint64_t* q_empty = q_full + kQStages;
  uint64_t* a_full = q_empty + kQStages;
  uint64_t* acc_full = a_full + kAStages;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  uint64_t* sk_bar = drain + 1;   // split: the other piece's partials landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sk_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* sk_last = reinterpret_cast<volatile int*>(tmem_slot + 2);   // split: this CTA reduces

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 8);
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(&a_full[i], 9);   // 8 dequant warps + the activation forwarder
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 8);
    mbar_init(drain, 1);
    if constexpr (kSplit) mbar_init(sk_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    for (int i = 0; i < 4; ++i) tma_prefetch_desc(&p.maps.b[i]);
    tma_prefetch_desc(&p.maps.q0);
    tma_prefetch_desc(&p.maps.q1);
    if (p.has_shared) {
      tma_prefetch_desc(&p.maps.sq0);
      tma_prefetch_desc(&p.maps.sq1);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
    tc_fence_before();
  }
#ifdef MOE_TC_STATS
  if (threadIdx.x < 32) s_tc_stats[threadIdx.x] = 0;
#endif
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
#ifdef MOE_TC_STATS
  const long long role_t0 = clock64();
#endif

  const int n_routed = *p.num_tiles;
  const int n_shared = p.has_shared ? (p.T + kBM - 1) / kBM : 0;
  const int units = (n_routed + n_shared) * p.nblk;
  const int nchunk = p.K / 64;
  const int kgroups = p.K / 64;
  const int nq = nchunk / 4;   // 256-K weight stages per unit

  if (warp == 0) {
    // ------------------------------------------ TMA producer: activations
    uint32_t bcnt = 0;
    bool ok = true;
    Deal<kSplit> d(p, units, nq);
    UnitRaw nxt = fetch_unit(p, d.unit(), n_routed);
    for (; d.valid() && ok; d.advance()) {
      const Unit U = make_unit(p, d.unit(), n_routed, nxt);
      nxt = fetch_unit(p, d.next_unit(), n_routed);
      // smallest box covering the tile's rows: fewer bytes for small groups
      const int bi = U.rows > 64 ? 0 : U.rows > 32 ? 1 : U.rows > 16 ? 2 : 3;
      const uint32_t bytes = (uint32_t)kBTileBytes >> bi;
      for (int c = 4 * d.q_begin(); c < 4 * d.q_end() && ok; ++c) {
        const int s = bcnt % kBStages;
        if (!(ok = warp_wait(&b_empty[s], ((bcnt / kBStages) & 1) ^ 1, abort_flag, p.err, 2, 32 * p.mode)))
          break;
        if (elect_one_sync()) {
          mbar_arrive_expect_tx(&b_full[s], bytes);
          tma_load_2d(smem_b + s * kBTileBytes, &p.maps.b[bi], 64 * c, U.m0, &b_full[s]);
        }
        __syncwarp();
        ++bcnt;
      }
    }
    if (!ok) {
      // let this CTA's own copies land before shared memory is released
      for (int s = 0; s < kBStages; ++s) {
        const uint32_t uses = (bcnt + kBStages - 1 - s) / kBStages;
        if (uses) mbar_wait_drain(&b_full[s], (uses - 1) & 1, p.err.limit_ns);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------- TMA producer: packed weights
    // (its own warp, so weight tiles run ahead of the activation ring)
    uint32_t qcnt = 0;
    bool ok = true;
    Deal<kSplit> d(p, units, nq);
    UnitRaw nxt = fetch_unit(p, d.unit(), n_routed);
    for (; d.valid() && ok; d.advance()) {
      const Unit U = make_unit(p, d.unit(), n_routed, nxt);
      nxt = fetch_unit(p, d.next_unit(), n_routed);
      const int y0 = (U.shared ? 0 : U.e * p.N) + block_row0(p, U.j, 0);
      const int y1 = (U.shared ? 0 : U.e * p.N) + block_row0(p, U.j, 1);
      const CUtensorMap* m0 = U.shared ? &p.maps.sq0 : &p.maps.q0;
      const CUtensorMap* m1 = U.shared ? &p.maps.sq1 : &p.maps.q1;
      for (int qc = d.q_begin(); qc < d.q_end() && ok; ++qc) {
        const int s = qcnt % kQStages;
        if (!(ok = warp_wait(&q_empty[s], ((qcnt / kQStages) & 1) ^ 1, abort_flag, p.err, 1, 32 * p.mode)))
          break;
        if (elect_one_sync()) {
          mbar_arrive_expect_tx(&q_full[s], kQStageBytes);
          tma_load_2d(smem_q + s * kQStageBytes, m0, 32 * qc, y0, &q_full[s]);
          tma_load_2d(smem_q + s * kQStageBytes + kQTileBytes, m1, 32 * qc, y1, &q_full[s]);
        }
        __syncwarp();
        ++qcnt;
      }
    }
    if (!ok) {
      for (int s = 0; s < kQStages; ++s) {
        const uint32_t uses = (qcnt + kQStages - 1 - s) / kQStages;
        if (uses) mbar_wait_drain(&q_full[s], (uses - 1) & 1, p.err.limit_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and takes the waits; one elected lane
    // issues the MMAs and the commits that track them.
    uint32_t bcnt = 0, acnt = 0, itn = 0;
    bool ok = true;
    Deal<kSplit> d(p, units, nq);
    UnitRaw nxt = fetch_unit(p, d.unit(), n_routed);
    for (; d.valid() && ok; d.advance(), ++itn) {
      const Unit U = make_unit(p, d.unit(), n_routed, nxt);
      nxt = fetch_unit(p, d.next_unit(), n_routed);
      const int ntok = (U.rows + 15) & ~15;
      const uint32_t idesc = idesc_f16_f32(128, ntok);
      if (!(ok = warp_wait(acc_empty, (itn & 1) ^ 1, abort_flag, p.err, 3, 32 * p.mode))) break;
      tc_fence_after();
      const int c_first = 4 * d.q_begin();
      for (int c = c_first; c < 4 * d.q_end(); ++c) {
        const int bs = bcnt % kBStages, as = acnt % kAStages;
        // a_full also covers the activation chunk (the forwarder saw it land)
        if (!(ok = warp_wait(&a_full[as], (acnt / kAStages) & 1, abort_flag, p.err, 5, 32 * p.mode))) break;
        tc_fence_after();
        if (elect_one_sync()) {
          const uint32_t bbase = smem_u32(smem_b + bs * kBTileBytes);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bd = smem_desc_sw128(bbase + 32 * kk);
            const uint32_t a0 = tmem + kAStageCol + 64 * as + 8 * kk;
            const uint32_t acc = kSplit ? (uint32_t)((c != c_first) | (kk != 0)) : (uint32_t)((c | kk) != 0);
            mma_f16_ts(tmem + kAccCol0, a0, bd, idesc, acc);
            mma_f16_ts(tmem + kAccCol1, a0 + 32, bd, idesc, acc);
          }
          // one commit frees both the activation slot and the TMEM weight stage
          mma_commit(&b_empty[bs]);
        }
        __syncwarp();
        ++bcnt;
        ++acnt;
      }
      if (!ok) break;
      if (elect_one_sync()) mma_commit(acc_full);
      __syncwarp();
    }
    // all MMAs of this warp complete before TMEM is released
    if (elect_one_sync()) mma_commit(drain);
    __syncwarp();
    mbar_wait_drain(drain, 0, p.err.limit_ns);
  } else if (warp == 3) {
    // --------------------------------------------- activation forwarder
    // Waits for each activation chunk to land and adds the last arrival to
    // the chunk's TMEM weight stage, so the MMA warp takes one wait per
    // chunk and the dequant warps none for activations. It arrives for
    // chunk c only after the stage's phase for chunk c - kAStages is over,
    // so an early arrival can never count toward the previous phase.
    uint32_t cnt = 0;
    bool ok = true;
    for (Deal<kSplit> d(p, units, nq); d.valid() && ok; d.advance()) {
      for (int c = 4 * d.q_begin(); c < 4 * d.q_end(); ++c, ++cnt) {
        if (!(ok = warp_wait(&b_full[cnt % kBStages], (cnt / kBStages) & 1, abort_flag, p.err, 4,
                             32 * p.mode)))
          break;
        if (cnt >= (uint32_t)kAStages) {
          const uint32_t prev = cnt - kAStages;
          if (!(ok = warp_wait(&a_full[prev % kAStages], (prev / kAStages) & 1, abort_flag, p.err, 10,
                               32 * p.mode)))
            break;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[cnt % kAStages]);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------ dequant warps
    const int blk = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    uint32_t qcnt = 0, acnt = 0;
    bool ok = true;
    // scale/bias rows of this thread's weight row in unit u
    auto sb_rows = [&](const Unit& U, const uint16_t*& sr, const uint16_t*& br) {
      const W4Dev& w = U.shared ? (blk == 0 ? p.sw0 : p.sw1) : (blk == 0 ? p.w0 : p.w1);
      const size_t row = (U.shared ? 0 : (size_t)U.e * p.N) + block_row0(p, U.j, blk) + r;
      sr = w.s + row * kgroups;
      br = w.b + row * kgroups;
    };
    const uint16_t *srow = nullptr, *brow = nullptr;
    uint2 s4 = make_uint2(0u, 0u), b4 = make_uint2(0u, 0u);
    Deal<kSplit> d(p, units, nq);
    UnitRaw nxt = fetch_unit(p, d.unit(), n_routed);
    if (d.valid()) {
      sb_rows(make_unit(p, d.unit(), n_routed, nxt), srow, brow);
      s4 = __ldg(reinterpret_cast<const uint2*>(srow + 4 * d.q_begin()));
      b4 = __ldg(reinterpret_cast<const uint2*>(brow + 4 * d.q_begin()));
    }
    for (; d.valid() && ok; d.advance()) {
      nxt = fetch_unit(p, d.next_unit(), n_routed);
      const uint16_t *nsrow = nullptr, *nbrow = nullptr;
      for (int qc = d.q_begin(); qc < d.q_end() && ok; ++qc) {
        // scales/biases of the next 4 groups, one step ahead (also across units)
        uint2 s4n = s4, b4n = b4;
        if (qc + 1 < d.q_end()) {
          s4n = __ldg(reinterpret_cast<const uint2*>(srow + 4 * (qc + 1)));
          b4n = __ldg(reinterpret_cast<const uint2*>(brow + 4 * (qc + 1)));
        } else if (d.has_next()) {
          sb_rows(make_unit(p, d.next_unit(), n_routed, nxt), nsrow, nbrow);
          s4n = __ldg(reinterpret_cast<const uint2*>(nsrow + 4 * d.next_q_begin()));
          b4n = __ldg(reinterpret_cast<const uint2*>(nbrow + 4 * d.next_q_begin()));
        }
        const int qs = qcnt % kQStages;
        if (!(ok = warp_wait(&q_full[qs], (qcnt / kQStages) & 1, abort_flag, p.err, 6, 32 * p.mode))) break;
        const uint8_t* qrow = smem_q + qs * kQStageBytes + blk * kQTileBytes + r * 128;
        const uint32_t sw = r & 7;
        // this thread's 64 weights of chunk `sub` of the stage, as fp16
        auto dequant_chunk = [&](int sub, uint32_t (&out)[32]) {
          const uint4 wa = *reinterpret_cast<const uint4*>(qrow + (((2 * sub) ^ sw) << 4));
          const uint4 wb = *reinterpret_cast<const uint4*>(qrow + (((2 * sub + 1) ^ sw) << 4));
          const uint32_t sbits = (sub & 1) ? (((sub >> 1) ? s4.y : s4.x) >> 16)
                                           : (((sub >> 1) ? s4.y : s4.x) & 0xFFFFu);
          const uint32_t bbits = (sub & 1) ? (((sub >> 1) ? b4.y : b4.x) >> 16)
                                           : (((sub >> 1) ? b4.y : b4.x) & 0xFFFFu);
          // bf16 scale and bias as fp16 (exact inside fp16's normal range)
          const __half2 s2 = __half2half2(__float2half_rn(bf16_to_f32((uint16_t)sbits)));
          const __half2 b2 = __half2half2(__float2half_rn(bf16_to_f32((uint16_t)bbits)));
          const uint32_t words[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint32_t o4[4];
            dequant_word_f16_perm8(words[i], s2, b2, o4);
            out[4 * i + 0] = o4[0];
            out[4 * i + 1] = o4[1];
            out[4 * i + 2] = o4[2];
            out[4 * i + 3] = o4[3];
          }
        };
        // Chunks go in pairs: one wait for two free TMEM stages, one wait for
        // the stores, and the second chunk's arithmetic overlaps the first
        // chunk's store.
#pragma unroll 1
        for (int pair = 0; pair < 2; ++pair) {
          uint32_t out[32];
          dequant_chunk(2 * pair, out);
          // Stage (acnt + 1) % kAStages is free once the MMAs of chunk
          // acnt + 1 - kAStages are done (their commit is the one on that
          // chunk's activation slot); MMAs complete in order, so that also
          // frees the stage of chunk acnt.
          if (acnt + 1 >= (uint32_t)kAStages) {
            const uint32_t prev = acnt + 1 - kAStages;
            if (!(ok = warp_wait(&b_empty[prev % kBStages], (prev / kBStages) & 1, abort_flag, p.err, 7,
                                 32 * p.mode)))
              break;
          }
          tc_fence_after();
          tmem_st_32x32b_x32(tmem + lane_base + kAStageCol + 64 * (acnt % kAStages) + 32 * blk, out);
          dequant_chunk(2 * pair + 1, out);
          tmem_st_32x32b_x32(tmem + lane_base + kAStageCol + 64 * ((acnt + 1) % kAStages) + 32 * blk, out);
#ifdef MOE_TC_STATS
          const long long st_t0 = clock64();
#endif
          tmem_wait_st();
#ifdef MOE_TC_STATS
          if (lane == 0) atomicAdd(&s_tc_stats[9], (unsigned long long)(clock64() - st_t0));
#endif
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&a_full[acnt % kAStages]);
            mbar_arrive(&a_full[(acnt + 1) % kAStages]);
          }
          acnt += 2;
        }
        if (!ok) break;
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_empty[qs]);
        ++qcnt;
        s4 = s4n;
        b4 = b4n;
      }
      srow = nsrow;
      brow = nbrow;
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------ epilogue warps
    // Two warps per TMEM lane quarter take alternate 32-token groups, so the
    // accumulators are read out (and released to the next unit) twice as
    // fast as with one.
    const int quarter = warp & 3, part = (warp - 12) >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    float* s_w = reinterpret_cast<float*>(smem + kOffW) + 128 * (warp - 12);   // this warp's copy
    uint16_t* s_x = reinterpret_cast<uint16_t*>(smem + kOffX) + 1024 * (warp - 12);  // 32 x 32 fp16
    // Output of one 32-token group: v0/v1 hold the two weight blocks' sums
    // (fp32 bits) of this lane's row for tokens c0 .. c0 + nval - 1.
    auto emit = [&](const Unit& U, int c0, int nval, const uint32_t (&v0)[32], const uint32_t (&v1)[32]) {
      // Lane l holds output column 32 * quarter + l for 32 consecutive
      // tokens, so one register stored by the whole warp writes 32 adjacent
      // columns of one token row: 64 (or 128) contiguous bytes.
      if (p.mode == 0) {
        // act = silu(gate) * up in fp16, columns in perm8 order. The 32 x 32
        // block goes through shared memory so that each lane stores 16-byte
        // pieces of token rows (measured faster here than one 2-byte store
        // per element).
        uint16_t* t16 = s_x;
        const int col = perm8_pos(lane);
#pragma unroll
        for (int cc = 0; cc < 32; ++cc)
          t16[cc * 32 + col] = f32_to_f16_sat(silu_fast(__uint_as_float(v0[cc])) *
                                              __uint_as_float(v1[cc]));
        __syncwarp();
        uint16_t* o = p.out + (size_t)(U.m0 + c0) * p.out_ld + 128 * U.j + 32 * quarter;
#pragma unroll
        for (int it4 = 0; it4 < 4; ++it4) {
          const int cc = it4 * 8 + (lane >> 2), seg = lane & 3;
          if (cc < nval)
            *reinterpret_cast<uint4*>(o + (size_t)cc * p.out_ld + 8 * seg) =
                *reinterpret_cast<const uint4*>(t16 + cc * 32 + 8 * seg);
        }
        __syncwarp();
      } else if (U.shared) {
        // shared expert (weight 1): kept in fp32, it is as large as the output
        float* o = p.out_sh + (size_t)(U.m0 - p.T * p.k + c0) * p.out_ld + 256 * U.j + 32 * quarter + lane;
#pragma unroll
        for (int cc = 0; cc < 32; ++cc)
          if (cc < nval) {
            o[(size_t)cc * p.out_ld] = __uint_as_float(v0[cc]);
            o[(size_t)cc * p.out_ld + 128] = __uint_as_float(v1[cc]);
          }
      } else {
        // routed expert: weighted by its top-k weight, bf16
        uint16_t* o = p.out + (size_t)(U.m0 + c0) * p.out_ld + 256 * U.j + 32 * quarter + lane;
#pragma unroll
        for (int cc = 0; cc < 32; ++cc)
          if (cc < nval) {
            const float w = s_w[(c0 + cc) & 127];
            o[(size_t)cc * p.out_ld] = f32_to_bf16(__uint_as_float(v0[cc]) * w);
            o[(size_t)cc * p.out_ld + 128] = f32_to_bf16(__uint_as_float(v1[cc]) * w);
          }
      }
    };
    // this CTA's piece of the split last round, if it has one (always its
    // last item)
    Item tl;
    const bool split = kSplit && item_at(p, units / (int)gridDim.x, units, nq, tl) && tl.pieces > 1;
    uint32_t itn = 0;
    bool ok = true;
    Deal<kSplit> d(p, units, nq);
    UnitRaw nxt = fetch_unit(p, d.unit(), n_routed);
    for (; d.valid() && ok; d.advance(), ++itn) {
      const Unit U = make_unit(p, d.unit(), n_routed, nxt);
      nxt = fetch_unit(p, d.next_unit(), n_routed);
      if (p.mode == 1 && !U.shared) {
        // top-k weights of the tile's rows, fetched while the MMAs still run
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = lane + 32 * i;
          if (row < U.rows) s_w[row] = __ldg(p.topk_w + __ldg(p.perm + U.m0 + row));
        }
        __syncwarp();
      }
      if (!(ok = warp_wait(acc_full, itn & 1, abort_flag, p.err, 8, 32 * p.mode))) break;
      tc_fence_after();
      if (32 * part >= U.rows) {
        // no group for this warp in this unit
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_relaxed(acc_empty);
      }
      for (int c0 = 32 * part; c0 < U.rows; c0 += 64) {
        uint32_t v0[32], v1[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kAccCol0 + c0, v0);
        tmem_ld_32x32b_x32(tmem + lane_base + kAccCol1 + c0, v1);
        tmem_wait_ld();
        if (c0 + 64 >= U.rows) {
          // this warp's accumulators fully read: let the next unit's MMAs start
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_relaxed(acc_empty);
        }
        const int nval = min(32, U.rows - c0);
        if (kSplit && d.pieces() > 1) {
          // a piece of a split unit: its partial sums, [block][token][row]
          float* slot = p.sk_ws + (size_t)blockIdx.x * kSlotFloats + 32 * quarter + lane;
#pragma unroll
          for (int cc = 0; cc < 32; ++cc)
            if (cc < nval) {
              slot[(size_t)(c0 + cc) * 128] = __uint_as_float(v0[cc]);
              slot[(size_t)(kBM + c0 + cc) * 128] = __uint_as_float(v1[cc]);
            }
        } else {
          emit(U, c0, nval, v0, v1);
        }
      }
      __syncwarp();
    }
    if (kSplit && split) {
      // Every epilogue warp comes here, whatever its waits gave, so that
      // both named barriers complete. The CTA arrives at its unit's counter
      // (release: every thread's fence, then one atomic) unless it gave up;
      // the CTA that arrives second clears the counter for the next launch,
      // adds the other half's partial sums to its own and writes the unit's
      // output.
      // (the proxy fence: the partials are read back by a bulk copy, the
      // async proxy)
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __threadfence();
      asm volatile("bar.sync 1, 256;" ::: "memory");
      const int t = tl.u - (units / (int)gridDim.x) * (int)gridDim.x;
      if (warp == 12 && lane == 0) {
        int last = 0;
        if (!*abort_flag) {
          const unsigned old = atomicAdd(p.sk_cnt + t, 1u);
          if (old == (unsigned)tl.pieces - 1u) {
            last = 1;
            __threadfence();
            p.sk_cnt[t] = 0u;
          }
        }
        *sk_last = last;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (*sk_last) {
        // the other piece's partials (block 0 and block 1, [token][row]) into
        // the operand buffers, which the unit's finished MMAs no longer read;
        // this piece's own sums are still in the accumulators
        const Unit U = make_unit(p, tl.u, n_routed, fetch_unit(p, tl.u, n_routed));
        float* o0 = reinterpret_cast<float*>(smem + kOffB);
        float* o1 = reinterpret_cast<float*>(smem + kOffQ);
        const uint32_t bytes = (uint32_t)U.rows * 128u * 4u;
        if (warp == 12 && lane == 0) {
          const float* src = p.sk_ws + (size_t)(2 * t + (tl.piece ^ 1)) * kSlotFloats;
          // generic-proxy accesses before the bulk copy: the other CTA's
          // stores of the partials (global), this CTA's reads of the
          // buffers (shared)
          asm volatile("fence.proxy.async;" ::: "memory");
          mbar_arrive_expect_tx(sk_bar, 2 * bytes);
          bulk_load(o0, src, bytes, sk_bar);
          bulk_load(o1, src + kBM * 128, bytes, sk_bar);
        }
        bool got = mbar_wait(sk_bar, 0, abort_flag, p.err.limit_ns);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          if (lane == 0) report_timeout(p.err, 11);
          *abort_flag = 1;
          // the copies land before shared memory is released
          if (warp == 12 && lane == 0) mbar_wait_drain(sk_bar, 0, p.err.limit_ns);
        } else {
          for (int c0 = 32 * part; c0 < U.rows; c0 += 64) {
            const int nval = min(32, U.rows - c0);
            uint32_t v0[32], v1[32];
            tmem_ld_32x32b_x32(tmem + lane_base + kAccCol0 + c0, v0);
            tmem_ld_32x32b_x32(tmem + lane_base + kAccCol1 + c0, v1);
            tmem_wait_ld();
            const int row = 32 * quarter + lane;
#pragma unroll
            for (int cc = 0; cc < 32; ++cc)
              if (cc < nval) {
                v0[cc] = __float_as_uint(__uint_as_float(v0[cc]) + o0[(c0 + cc) * 128 + row]);
                v1[cc] = __float_as_uint(__uint_as_float(v1[cc]) + o1[(c0 + cc) * 128 + row]);
              }
            emit(U, c0, nval, v0, v1);
          }
        }
      }
    }
  }

#ifdef MOE_TC_STATS
  if (lane == 0) {
    const int role = warp == 0 ? 0 : warp == 1 ? 1 : warp == 2 ? 2 : warp < 4 ? 3
                   : warp < 12 ? 4 : 5;
    atomicAdd(&s_tc_stats[16 + role], (unsigned long long)(clock64() - role_t0));
  }
#endif
  __syncthreads();
#ifdef MOE_TC_STATS
  if (threadIdx.x < 32) atomicAdd(&g_tc_stats[32 * p.mode + threadIdx.x], s_tc_stats[threadIdx.x]);
#endif
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tc

cudaError_t launch_gemm_tc(int mode, const GemmProblem& g, const TcMaps& maps, DevErr err,
                           int num_sms, cudaStream_t st) {
  tc::Params p;
  p.maps = maps;
  p.mode = mode;
  p.T = g.T;
  p.k = g.k;
  p.E = g.E;
  p.K = g.K;
  p.N = g.N;
  p.nblk = mode == 0 ? g.N / 128 : g.N / 256;
  p.has_shared = g.has_shared;
  p.bmap = g.bmap;
  p.num_tiles = g.num_tiles;
  p.w0 = g.w0;
  p.w1 = g.w1;
  p.sw0 = g.sw0;
  p.sw1 = g.sw1;
  p.out = g.out;
  p.out_sh = g.out_sh;
  p.out_ld = g.out_ld;
  p.topk_w = g.topk_w;
  p.perm = g.perm;
  p.sk_ws = g.sk_ws;
  p.sk_cnt = g.sk_cnt;
  p.sk_slots = g.sk_ws && g.sk_cnt ? g.sk_slots : 0;
  p.err = err;
  const int max_units = (g.max_routed_tiles + (g.has_shared ? (g.T + kBM - 1) / kBM : 0)) * p.nblk;
  int grid = num_sms < max_units ? num_sms : max_units;
  if (grid < 1) grid = 1;
  // the split last round only when the plan asks for it and the grid has a
  // slot per CTA; otherwise the kernel without it
  auto kern = p.sk_slots >= grid ? tc::w4_grouped_gemm_tc<true> : tc::w4_grouped_gemm_tc<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::kSmemBytes);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(tc::kThreads), tc::kSmemBytes, st, p);
}

#ifdef MOE_TC_STATS
extern "C" int moe_debug_tc_stats(unsigned long long* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, tc::g_tc_stats, sizeof(tc::g_tc_stats));
  unsigned long long z[64] = {};
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(tc::g_tc_stats, z, sizeof(z));
  return (int)e;
}
#endif

}  // namespace moe
