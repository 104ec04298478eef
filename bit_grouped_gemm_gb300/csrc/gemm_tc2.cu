// gemm_tc2.cu -- grouped W4A16 expert GEMM on pairs of SMs (tcgen05
// cta_group::2): the same product as gemm_tc.cu, with half its dequantisation
// work per multiply-add.
//
// The grouped GEMM with block-wise fused dequantisation of "Perplexity libera
// Lily, un motor de IA que supera a MLX-LM en Apple Silicon"
// (diariobitcoin.com), section "Las optimizaciones en el prefill" (4-bit
// weights rebuilt block by block on chip, FP32 accumulation), on the packed
// format of section "Qwen3.6 combina tres cargas de trabajo" (groups of 64,
// bf16 scale and bias).
//
// On one SM the kernel is bound by instruction issue, two thirds of it the
// rebuilding of weights: every 128-token tile rebuilds its expert's rows.
// Here a cluster of two CTAs on two SMs runs each MMA as one M = 256 x N <=
// 256 x K = 16 operation (tcgen05.mma.cta_group::2): each SM rebuilds only its
// own 128 weight rows into its tensor memory (the A operand), and holds only
// its half of the token tile (N/2 rows, the B operand) in shared memory; the
// tensor cores of the pair exchange the halves. Each rebuilt weight thus
// serves up to 256 tokens while each SM's activation stream stays at 128
// tokens per chunk.
//
// Unit: up to 256 expert-contiguous positions (a 256-row tile of one expert)
// times 256 weight rows: for the gate/up pass 128 gate and the matching 128
// up rows (CTA r rebuilds the 64 gate and 64 up rows of features
// f0 + 64 r .. + 63, interleaved by TMEM lane quarter -- lanes 0-15 gate,
// 16-31 up -- so SwiGLU pairs meet in one warp); for the down pass 256 down
// rows (128 per CTA). K is swept in chunks of 64 (one quantisation group).
//
// Roles per CTA (20 warps): warp 0 TMA of this CTA's token half, warp 2 TMA
// of its packed weights, warps 4-11 rebuild weights into TMEM (two per lane
// quarter, 32 K each per chunk), warps 12-19 read the accumulators back.
// Only the even CTA (the leader) issues MMAs (warp 1) and forwards
// "activations landed" (warp 3); the odd CTA's warp 3 forwards its own
// half's arrival, and its dequant and epilogue warps arrive on the leader's
// barriers through cluster addresses (relaxed arrivals after tcgen05 fences;
// the forwarders' after a release fence restricted to shared memory). The
// leader's commits are multicast to both CTAs, which
// frees both CTAs' activation slots and weight stages, and announces the
// accumulators.
//
// Every wait is bounded: on timeout a CTA latches the error, lets its own
// copies land, stops, and both CTAs meet at the final cluster barrier
// before the tensor memory is released.
#include "moe_common.cuh"

namespace moe {
namespace tc2 {

constexpr int kThreads = 640;
// Token-half slots = TMEM weight stages: a wait for chunk c - 8's MMAs (by
// the forwarder and the dequant warps) then always finds that slot's next
// phase still pending, since it needs an arrival made after the wait.
constexpr int kBStages = 8;               // token-half chunks (64 K) in flight
constexpr int kQStages = 3;               // packed-weight chunks (256 K) in flight
constexpr int kAStages = 8;               // TMEM weight stages (64 K, 32 columns)
constexpr int kBTileBytes = 128 * 128;    // up to 128 token rows x 64 fp16
constexpr int kQStageBytes = 128 * 128;   // 128 weight rows x 32 words
constexpr int kOffB = 0;
constexpr int kOffQ = kOffB + kBStages * kBTileBytes;
constexpr int kOffW = kOffQ + kQStages * kQStageBytes;   // epilogue row weights [8][256]
constexpr int kOffX = kOffW + 8 * 256 * 4;               // epilogue transpose [8][32 x 16 fp16]
constexpr int kOffBar = kOffX + 8 * 1024;
constexpr int kSmemBytes = kOffBar + 512 + 1024;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0, kAStageCol = 256;

struct Params {
  TcMaps maps;          // b[]: token rows (boxes 128/64/32/16); q0/q1 routed, sq0/sq1 shared
  int mode;             // 0: gate/up + SwiGLU, 1: down * top-k weight
  int T, k, E, K, N;
  int nblk;             // units per 256-row tile (I / 128 or H / 256)
  int has_shared;
  const int32_t* bmap2; // 256-row tiles (expert, first position, rows)
  const int32_t* num_tiles2;
  W4Dev w0, w1, sw0, sw1;
  uint16_t* out;
  float* out_sh;
  int out_ld;
  const float* topk_w;
  const int32_t* perm;
  DevErr err;
};

struct Unit {
  int e, m0, rows, j;
  bool shared;
};

// The tile-map entry of unit u (zeros for a shared-expert unit), fetched a
// unit ahead so that its global-load latency hides behind the current unit.
struct UnitRaw {
  int e, m0, rows;
};

__device__ __forceinline__ UnitRaw fetch_unit(const Params& p, int u, int n_routed) {
  UnitRaw r = {0, 0, 0};
  const int tile = u / p.nblk;
  if (tile < n_routed) {
    const int32_t* m = p.bmap2 + 3 * (size_t)tile;
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
    r.m0 = p.T * p.k + 256 * i;
    r.rows = min(256, p.T - 256 * i);
    r.shared = true;
  }
  return r;
}

// N of the pair MMA: rows rounded up to 32 (each CTA's half a multiple of 16)
__device__ __forceinline__ int unit_n(int rows) { return (rows + 31) & ~31; }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address, in the leader CTA (rank 0), of this CTA's shared variable `p`.
__device__ __forceinline__ uint32_t leader_addr(const void* p) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(smem_u32(p)));
  return r;
}
// Arrival on a barrier given by its cluster address, after a release fence
// restricted to shared::cta memory: orders the shared-memory writes this
// thread has observed (a token tile landed by TMA) before the arrival. A full
// release at cluster scope would also wait for every global access in flight
// and cost about a microsecond per arrival.
__device__ __forceinline__ void arrive_cluster_shared(uint32_t cluster_addr) {
  asm volatile("fence.release.sync_restrict::shared::cta.cluster;" ::: "memory");
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Relaxed arrival on a barrier given by its cluster address: for a thread
// whose tensor-memory accesses completed (tcgen05.wait) and are ordered by
// tcgen05.fence::before_thread_sync, so the arrival does not wait for the
// thread's unrelated global loads and stores to drain.
__device__ __forceinline__ void arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ bool try_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Suspend-time hint of the waits: a thread whose phase is not complete
// sleeps at most this long before it looks again.
constexpr uint32_t kHintNs = 100000;

#ifdef MOE_TC2_STATS
// Profiling build only: cycles spent in each wait site (site - 50), summed
// over the lane-0 threads of each CTA rank (read with moe_debug_tc2_stats).
__device__ unsigned long long g_tc2_stats[2][16];
#endif

// Whole-warp bounded wait (acquire at cluster scope: some arrivals are remote).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          const DevErr& err, int site) {
#ifdef MOE_TC2_STATS
  const long long st0 = clock64();
#endif
  bool ok = try_wait_cluster(bar, parity, 0);
  if (!ok) {
    const unsigned long long t0 = globaltimer_ns();
    while (true) {
      if (try_wait_cluster(bar, parity, kHintNs)) {
        ok = true;
        break;
      }
      if (*abort_flag) break;
      if (globaltimer_ns() - t0 > err.limit_ns) break;
    }
  }
  ok = __all_sync(0xffffffffu, ok);
#ifdef MOE_TC2_STATS
  if ((threadIdx.x & 31) == 0) {
    uint32_t rk;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rk));
    atomicAdd(&g_tc2_stats[rk & 1][(site - 50) & 15], (unsigned long long)(clock64() - st0));
  }
#endif
  if (!ok) {
    if ((threadIdx.x & 31) == 0 && !*abort_flag) report_timeout(err, site);
    *abort_flag = 1;
  }
  return ok;
}

__device__ __forceinline__ bool wait_drain(uint64_t* bar, uint32_t parity, unsigned long long limit) {
  if (try_wait_cluster(bar, parity, 0)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (try_wait_cluster(bar, parity, kHintNs)) return true;
    if (globaltimer_ns() - t0 > limit) return false;
  }
}

__device__ __forceinline__ void tmem_alloc2(uint32_t* slot) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
               "r"(kTmemCols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(kTmemCols)
               : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc] over the pair; kind::f16.
__device__ __forceinline__ void mma2_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the barrier at `bar`'s offset in both CTAs once every MMA issued
// so far by this thread is done.
__device__ __forceinline__ void mma2_commit_both(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"((unsigned short)3)
      : "memory");
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__global__ void __launch_bounds__(kThreads, 1) w4_grouped_gemm_tc2(const __grid_constant__ Params p) {
  pdl_begin();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t* smem_b = smem + kOffB;
  uint8_t* smem_q = smem + kOffQ;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* b_full = bars;                     // this CTA's token half landed (local)
  uint64_t* b_empty = b_full + kBStages;       // chunk's MMAs done (multicast commit)
  uint64_t* q_full = b_empty + kBStages;
  uint64_t* q_empty = q_full + kQStages;
  uint64_t* a_full = q_empty + kQStages;       // leader: 16 dequant warps + 2 forwarders
  uint64_t* acc_full = a_full + kAStages;      // multicast commit
  uint64_t* acc_empty = acc_full + 1;          // leader: 16 epilogue warps
  uint64_t* drain = acc_empty + 1;             // multicast commit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kBStages; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 8);
    }
    for (int i = 0; i < kAStages; ++i) mbar_init(&a_full[i], 18);
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 16);
    mbar_init(drain, 1);
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
  if (warp == 1) tmem_alloc2(tmem_slot);
  tc_fence_before();
  // both CTAs' barriers initialised and TMEM allocated before any remote arrival
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_routed = *p.num_tiles2;
  const int n_shared = p.has_shared ? (p.T + 255) / 256 : 0;
  const int units = (n_routed + n_shared) * p.nblk;
  const int nchunk = p.K / 64;
  const int kgroups = p.K / 64;
  const uint32_t a_full_l = leader_addr(a_full);      // (rank 0's a_full[0])
  const uint32_t acc_empty_l = leader_addr(acc_empty);

  if (warp == 0) {
    // ------------------------------------------ TMA: this CTA's token half
    uint32_t bcnt = 0;
    bool ok = true;
    UnitRaw nxt = fetch_unit(p, pair, n_routed);
    for (int u = pair; u < units && ok; u += npairs) {
      const Unit U = make_unit(p, u, n_routed, nxt);
      nxt = fetch_unit(p, u + npairs, n_routed);
      const int nh = unit_n(U.rows) >> 1;                // rows of each half
      const int bi = nh > 64 ? 0 : nh > 32 ? 1 : nh > 16 ? 2 : 3;
      const uint32_t bytes = (uint32_t)kBTileBytes >> bi;
      const int y0 = U.m0 + (int)rank * nh;
      for (int c = 0; c < nchunk && ok; ++c) {
        const int s = bcnt % kBStages;
        if (!(ok = warp_wait(&b_empty[s], ((bcnt / kBStages) & 1) ^ 1, abort_flag, p.err, 52))) break;
        if (elect_one_sync()) {
          mbar_arrive_expect_tx(&b_full[s], bytes);
          tma_load_2d(smem_b + s * kBTileBytes, &p.maps.b[bi], 64 * c, y0, &b_full[s]);
        }
        __syncwarp();
        ++bcnt;
      }
    }
    if (!ok) {   // this CTA's own copies land before its shared memory is released
      for (int s = 0; s < kBStages; ++s) {
        const uint32_t uses = (bcnt + kBStages - 1 - s) / kBStages;
        if (uses) wait_drain(&b_full[s], (uses - 1) & 1, p.err.limit_ns);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------- TMA: this CTA's packed weight rows
    uint32_t qcnt = 0;
    bool ok = true;
    UnitRaw nxt = fetch_unit(p, pair, n_routed);
    for (int u = pair; u < units && ok; u += npairs) {
      const Unit U = make_unit(p, u, n_routed, nxt);
      nxt = fetch_unit(p, u + npairs, n_routed);
      const int base = U.shared ? 0 : U.e * p.N;
      const CUtensorMap* m0 = U.shared ? &p.maps.sq0 : &p.maps.q0;
      const CUtensorMap* m1 = U.shared ? &p.maps.sq1 : &p.maps.q1;
      for (int qc = 0; qc < nchunk / 4 && ok; ++qc) {
        const int s = qcnt % kQStages;
        if (!(ok = warp_wait(&q_empty[s], ((qcnt / kQStages) & 1) ^ 1, abort_flag, p.err, 51))) break;
        if (elect_one_sync()) {
          mbar_arrive_expect_tx(&q_full[s], kQStageBytes);
          uint8_t* dst = smem_q + s * kQStageBytes;
          if (p.mode == 0) {   // 64 gate rows, then the matching 64 up rows
            const int f = base + 128 * U.j + 64 * (int)rank;
            tma_load_2d(dst, m0, 32 * qc, f, &q_full[s]);
            tma_load_2d(dst + kQStageBytes / 2, m1, 32 * qc, f, &q_full[s]);
          } else {             // 128 down rows
            tma_load_2d(dst, m0, 32 * qc, base + 256 * U.j + 128 * (int)rank, &q_full[s]);
          }
        }
        __syncwarp();
        ++qcnt;
      }
    }
    if (!ok) {
      for (int s = 0; s < kQStages; ++s) {
        const uint32_t uses = (qcnt + kQStages - 1 - s) / kQStages;
        if (uses) wait_drain(&q_full[s], (uses - 1) & 1, p.err.limit_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------- MMA issuer (leader only)
    if (leader) {
      uint32_t cnt = 0, it = 0;
      bool ok = true;
      UnitRaw nxt = fetch_unit(p, pair, n_routed);
      for (int u = pair; u < units && ok; u += npairs, ++it) {
        const Unit U = make_unit(p, u, n_routed, nxt);
        nxt = fetch_unit(p, u + npairs, n_routed);
        const int n = unit_n(U.rows);
        const uint32_t idesc = idesc_f16_f32(256, n);
        if (!(ok = warp_wait(acc_empty, (it & 1) ^ 1, abort_flag, p.err, 53))) break;
        tc_fence_after();
        for (int c = 0; c < nchunk; ++c) {
          const int bs = cnt % kBStages, as = cnt % kAStages;
          // a_full covers both CTAs' weight stage and both token halves
          if (!(ok = warp_wait(&a_full[as], (cnt / kAStages) & 1, abort_flag, p.err, 55))) break;
          tc_fence_after();
          if (elect_one_sync()) {
            const uint32_t bbase = smem_u32(smem_b + bs * kBTileBytes);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma2_f16_ts(tmem + kAccCol, tmem + kAStageCol + 32 * as + 8 * kk,
                          smem_desc_sw128(bbase + 32 * kk), idesc, (c | kk) != 0);
            mma2_commit_both(&b_empty[bs]);   // frees both token halves and weight stages
          }
          __syncwarp();
          ++cnt;
        }
        if (!ok) break;
        if (elect_one_sync()) mma2_commit_both(acc_full);
        __syncwarp();
      }
      if (elect_one_sync()) mma2_commit_both(drain);
      __syncwarp();
    }
  } else if (warp == 3) {
    // ------------------------------ forwarder: "this CTA's token half landed"
    // onto the leader's a_full. Chunk c may arrive only once the MMAs of chunk
    // c - kAStages are done (b_empty of that chunk, local: the commit is
    // multicast), so that no arrival can count toward the previous phase.
    uint32_t cnt = 0;
    bool ok = true;
    for (int u = pair; u < units && ok; u += npairs) {
      for (int c = 0; c < nchunk; ++c, ++cnt) {
        if (!(ok = warp_wait(&b_full[cnt % kBStages], (cnt / kBStages) & 1, abort_flag, p.err, 54)))
          break;
        if (cnt >= (uint32_t)kAStages) {
          const uint32_t prev = cnt - kAStages;
          if (!(ok = warp_wait(&b_empty[prev % kBStages], (prev / kBStages) & 1, abort_flag, p.err, 60)))
            break;
        }
        __syncwarp();
        if (lane == 0) arrive_cluster_shared(a_full_l + 8 * (cnt % kAStages));
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------ dequant warps
    // Two warps per TMEM lane quarter; warp half h2 rebuilds K 32 h2 .. + 31
    // of every chunk for the quarter's 32 rows.
    const int h2 = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = 32 * quarter + lane;                 // TMEM lane = this CTA's A row
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    // shared-memory row of this lane's weights, and its row in the matrix
    const int srow = p.mode == 0 ? (lane < 16 ? 16 * quarter + lane : 64 + 16 * quarter + lane - 16) : r;
    uint32_t qcnt = 0, acnt = 0;
    bool ok = true;
    auto sb_rows = [&](const Unit& U, const uint16_t*& sr, const uint16_t*& br) {
      const W4Dev& w = p.mode == 0 ? (lane < 16 ? (U.shared ? p.sw0 : p.w0) : (U.shared ? p.sw1 : p.w1))
                                   : (U.shared ? p.sw0 : p.w0);
      const int feat = p.mode == 0 ? 128 * U.j + 64 * (int)rank + 16 * quarter + (lane & 15)
                                   : 256 * U.j + 128 * (int)rank + r;
      const size_t row = (U.shared ? 0 : (size_t)U.e * p.N) + feat;
      sr = w.s + row * kgroups;
      br = w.b + row * kgroups;
    };
    const uint16_t *srow_p = nullptr, *brow_p = nullptr;
    uint2 s4 = make_uint2(0u, 0u), b4 = make_uint2(0u, 0u);
    UnitRaw nxt = fetch_unit(p, pair, n_routed);
    if (pair < units) {
      sb_rows(make_unit(p, pair, n_routed, nxt), srow_p, brow_p);
      s4 = __ldg(reinterpret_cast<const uint2*>(srow_p));
      b4 = __ldg(reinterpret_cast<const uint2*>(brow_p));
    }
    const int nq = nchunk / 4;
    for (int u = pair; u < units && ok; u += npairs) {
      nxt = fetch_unit(p, u + npairs, n_routed);
      const uint16_t *nsrow = nullptr, *nbrow = nullptr;
      for (int qc = 0; qc < nq && ok; ++qc) {
        uint2 s4n = s4, b4n = b4;
        if (qc + 1 < nq) {
          s4n = __ldg(reinterpret_cast<const uint2*>(srow_p + 4 * (qc + 1)));
          b4n = __ldg(reinterpret_cast<const uint2*>(brow_p + 4 * (qc + 1)));
        } else if (u + npairs < units) {
          sb_rows(make_unit(p, u + npairs, n_routed, nxt), nsrow, nbrow);
          s4n = __ldg(reinterpret_cast<const uint2*>(nsrow));
          b4n = __ldg(reinterpret_cast<const uint2*>(nbrow));
        }
        const int qs = qcnt % kQStages;
        if (!(ok = warp_wait(&q_full[qs], (qcnt / kQStages) & 1, abort_flag, p.err, 56))) break;
        const uint8_t* qrow = smem_q + qs * kQStageBytes + srow * 128;
        const uint32_t sw = srow & 7;
        // this thread's 32 weights of chunk `sub` of the stage, as fp16 (perm8)
        auto dequant_chunk = [&](int sub, uint32_t (&out)[16]) {
          const uint4 wa = *reinterpret_cast<const uint4*>(qrow + (((2 * sub + h2) ^ sw) << 4));
          const uint32_t sv = (sub >> 1) ? s4.y : s4.x, bv = (sub >> 1) ? b4.y : b4.x;
          const uint32_t sbits = (sub & 1) ? (sv >> 16) : (sv & 0xFFFFu);
          const uint32_t bbits = (sub & 1) ? (bv >> 16) : (bv & 0xFFFFu);
          const __half2 s2 = __half2half2(__float2half_rn(bf16_to_f32((uint16_t)sbits)));
          const __half2 b2 = __half2half2(__float2half_rn(bf16_to_f32((uint16_t)bbits)));
          const uint32_t words[4] = {wa.x, wa.y, wa.z, wa.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t o4[4];
            dequant_word_f16_perm8(words[i], s2, b2, o4);
            out[4 * i + 0] = o4[0];
            out[4 * i + 1] = o4[1];
            out[4 * i + 2] = o4[2];
            out[4 * i + 3] = o4[3];
          }
        };
        // chunks in pairs: one wait for two free stages, one wait for the stores
#pragma unroll 1
        for (int pr = 0; pr < 2; ++pr) {
          uint32_t out[16];
          dequant_chunk(2 * pr, out);
          // stage (acnt + 1) % kAStages is free once the MMAs of chunk
          // acnt + 1 - kAStages are done (that chunk's b_empty; the MMAs
          // complete in order, so the stage of chunk acnt is free too)
          if (acnt + 1 >= (uint32_t)kAStages) {
            const uint32_t prev = acnt + 1 - kAStages;
            if (!(ok = warp_wait(&b_empty[prev % kBStages], (prev / kBStages) & 1, abort_flag, p.err, 57)))
              break;
          }
          tc_fence_after();
          tmem_st_32x32b_x16(tmem + lane_base + kAStageCol + 32 * (acnt % kAStages) + 16 * h2, out);
          dequant_chunk(2 * pr + 1, out);
          tmem_st_32x32b_x16(tmem + lane_base + kAStageCol + 32 * ((acnt + 1) % kAStages) + 16 * h2, out);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            arrive_cluster_relaxed(a_full_l + 8 * (acnt % kAStages));
            arrive_cluster_relaxed(a_full_l + 8 * ((acnt + 1) % kAStages));
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
      srow_p = nsrow;
      brow_p = nbrow;
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------ epilogue warps
    // Two warps per lane quarter, alternate 32-token groups.
    const int quarter = warp & 3, part = (warp - 12) >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    float* s_w = reinterpret_cast<float*>(smem + kOffW) + 256 * (warp - 12);
    uint16_t* s_x = reinterpret_cast<uint16_t*>(smem + kOffX) + 512 * (warp - 12);   // 32 x 16 fp16
    uint32_t it = 0;
    bool ok = true;
    UnitRaw nxt = fetch_unit(p, pair, n_routed);
    for (int u = pair; u < units && ok; u += npairs, ++it) {
      const Unit U = make_unit(p, u, n_routed, nxt);
      nxt = fetch_unit(p, u + npairs, n_routed);
      if (p.mode == 1 && !U.shared) {
        // top-k weights of the tile's rows, fetched while the MMAs still run
        for (int row = lane; row < U.rows; row += 32) s_w[row] = __ldg(p.topk_w + __ldg(p.perm + U.m0 + row));
        __syncwarp();
      }
      if (!(ok = warp_wait(acc_full, it & 1, abort_flag, p.err, 58))) break;
      tc_fence_after();
      if (32 * part >= U.rows) {   // no group for this warp in this unit
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_cluster_relaxed(acc_empty_l);
      }
      for (int c0 = 32 * part; c0 < U.rows; c0 += 64) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + lane_base + kAccCol + c0, v);
        tmem_wait_ld();
        if (c0 + 64 >= U.rows) {   // this warp's accumulators read: let the next unit's MMAs start
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_cluster_relaxed(acc_empty_l);
        }
        const int nval = min(32, U.rows - c0);
        if (p.mode == 0) {
          // lanes 0-15 hold gate features 16 q + i, lanes 16-31 the matching
          // up features: act = silu(gate) * up for 16 features x 32 tokens,
          // transposed through shared memory into 32-byte pieces of token rows
          const int fcol = perm8_pos(lane & 15);
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            const float other = __shfl_xor_sync(0xffffffffu, __uint_as_float(v[cc]), 16);
            if (lane < 16)
              s_x[cc * 16 + fcol] = f32_to_f16_sat(silu_fast(__uint_as_float(v[cc])) * other);
          }
          __syncwarp();
          if (lane < nval) {
            uint16_t* o = p.out + (size_t)(U.m0 + c0 + lane) * p.out_ld + 128 * U.j + 64 * rank + 16 * quarter;
            const uint4* src = reinterpret_cast<const uint4*>(s_x + lane * 16);
            reinterpret_cast<uint4*>(o)[0] = src[0];
            reinterpret_cast<uint4*>(o)[1] = src[1];
          }
          __syncwarp();
        } else if (U.shared) {
          // shared expert (weight 1): fp32
          float* o = p.out_sh + (size_t)(U.m0 - p.T * p.k + c0) * p.out_ld + 256 * U.j + 128 * rank + 32 * quarter + lane;
#pragma unroll
          for (int cc = 0; cc < 32; ++cc)
            if (cc < nval) o[(size_t)cc * p.out_ld] = __uint_as_float(v[cc]);
        } else {
          // routed expert: weighted by its top-k weight, bf16
          uint16_t* o = p.out + (size_t)(U.m0 + c0) * p.out_ld + 256 * U.j + 128 * rank + 32 * quarter + lane;
#pragma unroll
          for (int cc = 0; cc < 32; ++cc)
            if (cc < nval) o[(size_t)cc * p.out_ld] = f32_to_bf16(__uint_as_float(v[cc]) * s_w[c0 + cc]);
        }
      }
      __syncwarp();
    }
  }

#ifdef MOE_TC2_STATS
  if (lane == 0 && warp < 2) {
    // total cycles of the kernel per rank (warps 0/1), for scale
    atomicAdd(&g_tc2_stats[rank & 1][14 + warp], (unsigned long long)clock64());
  }
#endif
  // the leader's last commit tells both CTAs that every MMA is done
  __syncthreads();
  if (warp == 1) wait_drain(drain, 0, p.err.limit_ns);
  tc_fence_before();
  // neither CTA leaves (or frees TMEM) while the other may still touch it
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc2(tmem);
}

}  // namespace tc2

#ifdef MOE_TC2_STATS
extern "C" int moe_debug_tc2_stats(unsigned long long* out) {
  cudaError_t e = cudaMemcpyFromSymbol(out, tc2::g_tc2_stats, sizeof(tc2::g_tc2_stats));
  unsigned long long z[32] = {};
  if (e == cudaSuccess) e = cudaMemcpyToSymbol(tc2::g_tc2_stats, z, sizeof(z));
  return (int)e;
}
#endif

cudaError_t launch_gemm_tc2(int mode, const GemmProblem& g, const TcMaps& maps,
                            const int32_t* bmap2, const int32_t* num_tiles2, int max_tiles2,
                            DevErr err, int num_sms, cudaStream_t st) {
  tc2::Params p;
  p.maps = maps;
  p.mode = mode;
  p.T = g.T;
  p.k = g.k;
  p.E = g.E;
  p.K = g.K;
  p.N = g.N;
  p.nblk = mode == 0 ? g.N / 128 : g.N / 256;
  p.has_shared = g.has_shared;
  p.bmap2 = bmap2;
  p.num_tiles2 = num_tiles2;
  p.w0 = g.w0;
  p.w1 = g.w1;
  p.sw0 = g.sw0;
  p.sw1 = g.sw1;
  p.out = g.out;
  p.out_sh = g.out_sh;
  p.out_ld = g.out_ld;
  p.topk_w = g.topk_w;
  p.perm = g.perm;
  p.err = err;
  cudaError_t e = cudaFuncSetAttribute(tc2::w4_grouped_gemm_tc2,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, tc2::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int max_units = (max_tiles2 + (g.has_shared ? (g.T + 255) / 256 : 0)) * p.nblk;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(tc2::kThreads);
  cfg.dynamicSmemBytes = tc2::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // pairs: as many as can be resident at once (persistent), at most one per unit
  static int max_clusters = -1;
  if (max_clusters < 0) {
    cfg.gridDim = dim3(2 * (num_sms / 2));
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, tc2::w4_grouped_gemm_tc2, &cfg) != cudaSuccess || n < 1)
      n = num_sms / 2;
    max_clusters = n;
  }
  int pairs = max_clusters < max_units ? max_clusters : max_units;
  if (pairs < 1) pairs = 1;
  cfg.gridDim = dim3(2 * pairs);
  static int pdl_ok = -1;   // whether the runtime takes clusters with programmatic launch
  if (pdl_ok != 0) {
    e = cudaLaunchKernelEx(&cfg, tc2::w4_grouped_gemm_tc2, p);
    if (e == cudaSuccess) {
      pdl_ok = 1;
      return e;
    }
    cudaGetLastError();
    pdl_ok = 0;
  }
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc2::w4_grouped_gemm_tc2, p);
}

// ---------------------------------------------------------------------------
// 256-row tiles of the expert-contiguous positions (the pair kernel's units),
// from the routing offsets: tile (e, off[e] + 256 i, min(256, cnt[e] - 256 i)),
// expert-major. One CTA, one thread per expert.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(512) build_tiles256_kernel(const int32_t* __restrict__ off, int E,
                                                              int32_t* __restrict__ bmap2,
                                                              int32_t* __restrict__ num_tiles2) {
  pdl_begin();
  __shared__ int warp_sums[16];
  __shared__ int total_s;
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  const int o = e < E ? off[e] : 0;
  const int cnt = e < E ? off[e + 1] - o : 0;
  const int tiles = (cnt + 255) / 256;
  int inc = tiles;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += n;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int ws = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
    int wi = ws;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, d);
      if (lane >= d) wi += n;
    }
    if (lane < (int)(blockDim.x >> 5)) warp_sums[lane] = wi - ws;
    if (lane == 31) total_s = wi;
  }
  __syncthreads();
  const int t0 = inc - tiles + warp_sums[warp];
  for (int i = 0; i < tiles; ++i) {
    int32_t* m = bmap2 + 3 * (size_t)(t0 + i);
    m[0] = e;
    m[1] = o + 256 * i;
    m[2] = min(256, cnt - 256 * i);
  }
  if (e == 0) *num_tiles2 = total_s;
}

cudaError_t launch_build_tiles256(const int32_t* off, int E, int32_t* bmap2, int32_t* num_tiles2,
                                  cudaStream_t st) {
  if (E > 512) return cudaErrorInvalidValue;
  return launch_pdl(build_tiles256_kernel, dim3(1), dim3(512), 0, st, off, E, bmap2, num_tiles2);
}

bool tc2_supported() {
  static int ok = -1;
  if (ok < 0) {
    int dev = 0, cl = 0;
    ok = cudaGetDevice(&dev) == cudaSuccess &&
                 cudaDeviceGetAttribute(&cl, cudaDevAttrClusterLaunch, dev) == cudaSuccess && cl
             ? 1
             : 0;
  }
  return ok == 1;
}

}  // namespace moe
