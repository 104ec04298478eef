// decode_fused.cu -- one mixture-of-experts layer of a decode-sized batch
// (T <= 8 tokens) in one cooperative launch.
//
// The block of "Perplexity libera Lily, un motor de IA que supera a MLX-LM en
// Apple Silicon" (diariobitcoin.com): router and top-8 of section "Qwen3.6
// combina tres cargas de trabajo", the grouped 4-bit GEMM with on-chip
// dequantisation and FP32 accumulation of section "Las optimizaciones en el
// prefill", in the regime of section "El decode busca mover menos datos",
// where a layer moves its selected experts' packed bytes once and the time
// between dependent steps, not arithmetic, decides the speed.
//
// The general path runs a decode layer as four dependent launches (routing,
// gate/up, down, combine), each paying a launch boundary and one or two
// dependent round trips through L2. Here one persistent CTA per SM does the
// whole layer, with one grid barrier (arrival counter in device memory,
// bounded waits) and one hand-off through tagged values:
//   1. every CTA reads the residual rows x, computes their RMS norm and the
//      normalised rows xn = bf16(x / rms(x)) (kept in shared memory as the
//      fp16 MMA operand, in 16-byte pieces ordered for 128-bit fragment
//      loads), and router CTA c computes the logits of its experts on bf16
//      mma.sync (its router weight slice is copied from before the launch
//      waits on the previous one);
//   -- each logit is written with the launch's number in the high half of a
//      64-bit word; a top-k warp reads its token's row (one entry per lane
//      first, then all) until every entry carries this launch's number --
//   2. every CTA selects each token's top-k (the same warp top-k as the
//      routing kernels, so every CTA holds the same routing) and numbers the
//      active experts in ascending order: slot 0 the shared expert, then one
//      slot per selected routed expert with its list of tokens;
//   3. gate/up units (8 gate + the matching 8 up rows of one slot's expert,
//      one m16 tile) are dealt to warps over the whole grid; each warp takes
//      its unit's packed rows by TMA (3D boxes of 8 rows x all K, 128-byte
//      swizzle) into its own shared-memory buffer, rebuilds each group's
//      fp16 weights fp16(q s + b) in registers (one rounding, the same
//      weights the tensor-core GEMM rebuilds) and runs mma.sync with FP32
//      accumulation, SwiGLU in FP32 registers, activations stored as fp16
//      rows per (slot, token); no block barrier per unit;
//   -- grid barrier (all activations written) --
//   4. CTA c < H/16 owns 16 output columns: for every slot it multiplies
//      those 16 down rows (copied while it waits at the barrier) by the slot's
//      activation rows, then forms
//          y[t] = shared[t] + sum_j w[t][j] * expert_j[t]   (FP32, j in rank order)
//      and updates x[t] = bf16(x[t] + alpha * y[t]) in place.
// The next layer's launch (programmatic dependent launch) is the barrier
// between layers. Every wait is bounded: a CTA that gives up latches the
// error word, lets its own copies land and exits.
#include "moe_common.cuh"
#include "topk.cuh"

namespace moe {
namespace dec {

constexpr int kThreads = 256;
constexpr int kWarps = 8;
constexpr int kMaxT = 8;            // tokens
constexpr int kMaxSlots = 80;       // shared + distinct routed experts
constexpr int kGU = 8;              // gate rows (and the matching up rows) per unit: one m16 tile
// a gate/up warp's buffer: its unit's 8 gate and 8 up rows, all K (H / 2 bytes
// a row), then their scales and biases (gate s, gate b, up s, up b: 8 rows x
// H / 64 bf16 each)
__host__ __device__ constexpr uint32_t unit_words_bytes(int H) { return 2u * kGU * (uint32_t)H / 2; }
__host__ __device__ constexpr uint32_t unit_sb_bytes(int H) { return (uint32_t)kGU * (H / 64) * 2; }
__host__ __device__ constexpr uint32_t unit_bytes(int H) { return unit_words_bytes(H) + 4 * unit_sb_bytes(H); }
constexpr int kDn = 16;             // down rows (output columns) per CTA
constexpr int kSlotsPerChunk = 8;   // down slabs per ring buffer (one per warp)
constexpr int kRing = 4;            // shared-memory slab buffers
constexpr int kRBoxE = 8;           // router weight columns per TMA box (16-byte rows)
constexpr int kIssuer = 224;        // the thread that issues the ring's copies (warp 7, lane 0)
constexpr int kRBox = 256;          // router weight rows per TMA box

struct Params {
  int T, H, I, E, k, has_shared;
  float alpha, eps;
  int n_dn;                  // CTAs that own output columns (H / kDn)
  uint16_t* x;               // residual rows bf16 [T][H], updated in place
  const uint16_t* wr;        // router weight bf16 [H][E]
  const float* rbias;        // [E] or null
  W4Dev gate, up, down, sgate, sup, sdown;   // scales and biases (words via the maps)
  CUtensorMap mg, mu, msg, msu;   // gate/up packed words, 3D boxes (32 words, 8 rows, K/256)
  CUtensorMap md, msd;             // down packed words, 3D boxes (32 words, 16 rows, K/256)
  CUtensorMap mr;            // router weight bf16 [H][E], boxes of 8 experts x 256 rows
  unsigned* epoch;           // launches of this layer kernel so far on the plan
  unsigned long long* tlog;  // [T][E] router logits, tag epoch + 1 in the high word
  uint16_t* act;             // [rows][I] fp16, K order perm8 (row = slot offset + token)
  int32_t* topk_idx;         // [T][k] (written by CTA 0)
  float* topk_w;             // [T][k]
  float* y_out;              // [T][H] FP32 block output, or null
  unsigned* bar;             // grid-barrier arrival counter, 0 at launch
  DevErr err;
};

// Byte offsets of the dynamic shared memory (from a 1024-aligned base).
struct Smem {
  uint32_t slab, xw, xstride, wr, total, dsum_cap;
};

__host__ __device__ inline uint32_t align_u(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// The router slice (H x 8 bf16: the 16-byte box holding this CTA's columns)
// lives in the last ring buffer and the router's bf16 token rows in buffer 1,
// both before the routing is known; then the gate/up warps' unit buffers
// (kWarps x unit_bytes) take the whole ring, and after them the down slabs.
__host__ __device__ inline Smem smem_layout(int H, int I) {
  Smem L;
  const uint32_t dn = kSlotsPerChunk * (kDn * (I / 2) + 2u * kDn * (I / 64) * 2);
  const uint32_t gu = (kWarps * unit_bytes(H) + kRing - 1) / kRing;
  L.slab = align_u(dn > gu ? dn : gu, 1024);
  uint32_t o = kRing * L.slab;
  L.xw = o;
  // words per token row: 16-byte pieces, rows 4 pieces (mod 8) apart, so that
  // the two tokens of a 128-bit load phase hit disjoint banks when their row
  // numbers differ in parity
  L.xstride = H / 2 + 16;
  o += (kMaxT + 1) * L.xstride * 4;            // + one zero row
  L.dsum_cap = (kMaxT + 1) * L.xstride * 4;    // the down pass reuses the token rows
  o = align_u(o, 16);
  L.wr = (kRing - 1) * L.slab;
  L.total = o;
  return L;
}

// A relaxed load that the compiler must issue every time (polling loops).
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

#ifdef MOE_DEC_TRACE
// Profiling build only: %globaltimer inside the grid barriers of every CTA
// (after the first sync, the fence, the arrival, the wait, the last sync).
__device__ unsigned long long g_dec_btrace[256][2][5];
#define DEC_BTRACE(i) \
  if (blockIdx.x < 256) g_dec_btrace[blockIdx.x][site == 40 ? 0 : 1][(i)] = globaltimer_ns()
#else
#define DEC_BTRACE(i)
#endif

// Grid barrier: every CTA adds one arrival (after a fence that makes the
// CTA's writes visible), then waits (bounded, acquire loads) until the
// counter reaches `target`. Returns false on timeout (error latched).
// `during` runs on the other threads while thread 0 waits.
template <class F>
__device__ bool grid_barrier(unsigned* bar, unsigned target, const DevErr& err, int site,
                             int* flag_s, F&& during) {
  __syncthreads();
  if (threadIdx.x == 0) {
    DEC_BTRACE(0);
    __threadfence();
    DEC_BTRACE(1);
    atomicAdd(bar, 1u);
    DEC_BTRACE(2);
  }
  // `during` starts after the arrival: copies issued while the fence waits
  // for the CTA's stores delayed it (measured: 1.9% of a T = 8 decode step)
  __syncthreads();
  if (threadIdx.x != 0) {
    during();
  } else {
    int ok = 1;
    if (ld_acquire_u32(bar) < target) {
      const unsigned long long t0 = globaltimer_ns();
      while (ld_acquire_u32(bar) < target) {
        __nanosleep(32);
        if (globaltimer_ns() - t0 > err.limit_ns) {
          report_timeout(err, site);
          ok = 0;
          break;
        }
      }
    }
    DEC_BTRACE(3);
    // (no fence here: the acquire load that saw the count, then the CTA
    // barrier, order every thread's later reads after the other CTAs' writes;
    // a trailing fence measured ~0.5 us per barrier)
    *flag_s = ok;
  }
  __syncthreads();
  if (threadIdx.x == 0) { DEC_BTRACE(4); }
  return *flag_s != 0;
}

__device__ bool grid_barrier(unsigned* bar, unsigned target, const DevErr& err, int site,
                             int* flag_s) {
  return grid_barrier(bar, target, err, site, flag_s, [] {});
}

__device__ __forceinline__ uint2 lds_v2(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
// ldmatrix of four 8x8 b16 matrices (row addresses from lanes 8j .. 8j + 7 for
// matrix j), plain and transposed, and the bf16 m16n8k16 MMA (FP32 accumulation).
__device__ __forceinline__ void ldsm4(uint32_t a, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void ldsm4_t(uint32_t a, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(a));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// 128-bit load of shared memory that no copy rewrites while it is in use (the
// token rows): not volatile, so the compiler may schedule it freely.
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

// Byte offset, inside a 3D box of (32 words) x (rows) x (K/256 chunks) with
// the 128-byte swizzle, of the two packed words 8 j + 2 c and 8 j + 2 c + 1 of
// row y (group j of 64 K): chunk j / 4, 16-byte piece 2 (j % 4) + c / 2
// stored at piece ^ (y % 8), half c % 2 of it.
__device__ __forceinline__ uint32_t qoff(int y, int j, int c, int rows) {
  const int z = j >> 2, piece = 2 * (j & 3) + (c >> 1);
  return (uint32_t)((z * rows + y) * 128 + ((piece ^ (y & 7)) << 4) + ((c & 1) << 3));
}

#ifdef MOE_DEC_TRACE
// Profiling build only: %globaltimer at the phase boundaries of every CTA of
// the last launch (read with moe_debug_dec_trace).
__device__ unsigned long long g_dec_trace[256][16];
#define DEC_TRACE(i) \
  if (threadIdx.x == 0 && blockIdx.x < 256) g_dec_trace[blockIdx.x][(i)] = globaltimer_ns()
// finer marks inside phases 1 and 2
__device__ unsigned long long g_dec_trace2[256][8];
#define DEC_TRACE2(i) \
  if (threadIdx.x == 0 && blockIdx.x < 256) g_dec_trace2[blockIdx.x][(i)] = globaltimer_ns()
// per warp in step 3: copy issued, landed, MMAs done, stored (first unit),
// then landed and stored for a second unit
__device__ unsigned long long g_dec_wtrace[256][8][6];
#define DEC_WTRACE(i) \
  if ((threadIdx.x & 31) == 0 && blockIdx.x < 256) g_dec_wtrace[blockIdx.x][threadIdx.x >> 5][(i)] = globaltimer_ns()
#else
#define DEC_TRACE(i)
#define DEC_TRACE2(i)
#define DEC_WTRACE(i)
#endif

// Exclusive scan of one int per thread over the CTA; *total gets the sum.
__device__ __forceinline__ int block_excl_scan_i(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int ws = lane < nw ? warp_sums[lane] : 0;
    int wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < nw) warp_sums[lane] = wi - ws;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const int r = inc - v + warp_sums[warp];
  __syncthreads();
  return r;
}

template <int VPL, int EPC>   // top-k values per lane; router experts per CTA
__global__ void __launch_bounds__(kThreads, 1) moe_decode_layer_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full[kRing];
  __shared__ __align__(8) uint64_t wfull[kWarps];   // gate/up warps' unit buffers
  __shared__ __align__(8) uint64_t wbar;       // router slice landed
  __shared__ int idx_s[kMaxT][32];
  __shared__ float w_s[kMaxT][32];
  __shared__ int sc_s[kMaxT][32];              // slot * 16 + column of (token, rank)
  __shared__ unsigned tmask_s[512];            // per expert: tokens that selected it
  __shared__ int slot_of_s[512];
  __shared__ int slot_e[kMaxSlots], cnt_s[kMaxSlots], soff_s[kMaxSlots];
  __shared__ int tok_s[kMaxSlots][kMaxT];
  __shared__ float ss_w[kWarps][kMaxT];
  __shared__ float rpart_s[kWarps][kMaxT][kRBoxE];   // router partial sums per warp
  __shared__ float x_s[kMaxT][kDn];
  __shared__ int nslots_s, flag_s, abort_s;
  __shared__ int scan_a[kWarps], scan_c[kWarps];
  __shared__ unsigned ring_issued_s;           // first-round down chunks issued (bit per buffer)
  __shared__ float rinv_s[kMaxT];

  const int H = p.H, I = p.I, E = p.E, T = p.T, k = p.k;
  const int G = H / 64, GI = I / 64;
  const Smem L = smem_layout(H, I);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int cta = blockIdx.x, ncta = gridDim.x;
  const uint32_t sbase = smem_u32(smem);
  uint32_t* xw = reinterpret_cast<uint32_t*>(smem + L.xw);
  const uint16_t* wrs = reinterpret_cast<const uint16_t*>(smem + L.wr);
  uint16_t* xb = reinterpret_cast<uint16_t*>(smem + L.slab);   // xn bf16 [T][H + 8] (ring buffer 1)
  const int upe = I / kGU;                     // gate/up units per slot
  const uint32_t dn_q = (uint32_t)kDn * (I / 2), dn_s = (uint32_t)kDn * GI * 2;
  const int e0 = cta * EPC;                    // this CTA's router columns [e0, e0 + EPC)
  const bool router_cta = e0 < E;
  const int ebox = e0 & ~(kRBoxE - 1), ecol = e0 - ebox;   // the 16-byte box holding them

  DEC_TRACE(0);
  // ------------------------------------------------ prologue (weights only)
  if (tid == 0) {
    for (int b = 0; b < kRing; ++b) mbar_init(&full[b], 1);
    for (int w = 0; w < kWarps; ++w) mbar_init(&wfull[w], 1);
    mbar_init(&wbar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&p.mg);
    tma_prefetch_desc(&p.mu);
    tma_prefetch_desc(&p.md);
    if (p.has_shared) {
      tma_prefetch_desc(&p.msg);
      tma_prefetch_desc(&p.msu);
      tma_prefetch_desc(&p.msd);
    }
    abort_s = 0;
    ring_issued_s = 0u;
    if (router_cta) {   // the router slice [H][8] by TMA, H / 256 boxes
      mbar_arrive_expect_tx(&wbar, (uint32_t)H * kRBoxE * 2);
      for (int y = 0; y < H; y += kRBox)
        tma_load_2d(smem + L.wr + (size_t)y * kRBoxE * 2, &p.mr, ebox, y, &wbar);
    }
  }
  __syncthreads();

  // The ring of down slabs: chunk i (kSlotsPerChunk slots' 16 down rows) goes
  // to buffer i % kRing once the gate/up units are done with the ring: the
  // first kRing chunks from one thread each during the grid barrier, later
  // ones from kIssuer as buffers free up.
  int n_units = 0, n_dc = 0;             // set once the routing is known
  int issued = 0;                        // 1 + the last chunk this thread issued
  auto ring_buf = [](int i) { return i % kRing; };
  auto issue = [&](int i) {
    const int b = ring_buf(i);
    issued = i + 1;
    uint8_t* buf = smem + (size_t)b * L.slab;
    const int s0 = kSlotsPerChunk * i;
    const int ns = min(kSlotsPerChunk, nslots_s - s0);
    mbar_arrive_expect_tx(&full[b], (uint32_t)ns * (dn_q + 2 * dn_s));
    for (int q = 0; q < ns; ++q) {
      const int s = s0 + q;
      const bool sh = p.has_shared && s == 0;
      const int row0 = (sh ? 0 : slot_e[s] * H) + kDn * cta;
      const W4Dev& wd = sh ? p.sdown : p.down;
      tma_load_3d(buf + q * dn_q, sh ? &p.msd : &p.md, 0, row0, 0, &full[b]);
      bulk_load(buf + kSlotsPerChunk * dn_q + q * dn_s, wd.s + (size_t)row0 * GI, dn_s, &full[b]);
      bulk_load(buf + kSlotsPerChunk * (dn_q + dn_s) + q * dn_s, wd.b + (size_t)row0 * GI, dn_s,
                &full[b]);
    }
  };

  DEC_TRACE(1);
  pdl_begin();   // x and everything below come from the previous launch
  DEC_TRACE(2);
  const unsigned ep = __ldcg(p.epoch);   // set by the previous launch's last CTA
  bool ok = true;

  // ------------------------------------------- 1. norms, operand rows, router
  for (int e = tid; e < E; e += kThreads) tmask_s[e] = 0u;
  const int pieces = H / 8;                    // 8 hidden values per piece, <= 2 per thread
  // this CTA's output columns of x (only this CTA writes them), with the rows
  const bool own_x = cta < p.n_dn && tid < T * kDn;
  const float xo = own_x ? bf16_to_f32(p.x[(size_t)(tid / kDn) * H + kDn * cta + tid % kDn]) : 0.f;
  uint4 xv4[2][kMaxT];                         // this thread's pieces of every token row
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int pc = tid + it * kThreads;
#pragma unroll
    for (int t = 0; t < kMaxT; ++t)
      xv4[it][t] = (pc < pieces && t < T)
                       ? *reinterpret_cast<const uint4*>(p.x + (size_t)t * H + 8 * pc)
                       : make_uint4(0u, 0u, 0u, 0u);
  }
  float ss[kMaxT];
#pragma unroll
  for (int t = 0; t < kMaxT; ++t) {
    ss[t] = 0.f;
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const uint32_t wv[4] = {xv4[it][t].x, xv4[it][t].y, xv4[it][t].z, xv4[it][t].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        ss[t] = fmaf(bf16_lo(wv[i]), bf16_lo(wv[i]), ss[t]);
        ss[t] = fmaf(bf16_hi(wv[i]), bf16_hi(wv[i]), ss[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kMaxT; ++t)
    if (t < T) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss[t] += __shfl_xor_sync(0xffffffffu, ss[t], o);
      if (lane == 0) ss_w[warp][t] = ss[t];
    }
  DEC_TRACE2(0);
  if (own_x) x_s[tid / kDn][tid % kDn] = xo;
  __syncthreads();
  DEC_TRACE2(1);
  // each token's 1 / rms once (thread t), shared with the block
  if (tid < T) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += ss_w[w][tid];
    rinv_s[tid] = 1.0f / sqrtf(tot / (float)H + p.eps);
  }
  __syncthreads();
  float rinv[kMaxT];
#pragma unroll
  for (int t = 0; t < kMaxT; ++t) rinv[t] = t < T ? rinv_s[t] : 0.f;
  DEC_TRACE2(2);
  // xn = bf16(x * rinv): fp16 operand rows (perm8 K order), and bf16 rows for
  // the router (router CTAs)
  uint32_t over = 0u;
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int pc = tid + it * kThreads;
    if (pc >= pieces) continue;   // (uniform over each group of 8 lanes)
#pragma unroll
    for (int t = 0; t < kMaxT; ++t) {
      if (t >= T) continue;
      const uint32_t wv[4] = {xv4[it][t].x, xv4[it][t].y, xv4[it][t].z, xv4[it][t].w};
      uint32_t nb[4];   // xn as bf16 pairs
#pragma unroll
      for (int i = 0; i < 4; ++i) nb[i] = pack_bf16x2(bf16_lo(wv[i]) * rinv[t], bf16_hi(wv[i]) * rinv[t]);
      over |= bf16x2_f16_overflow(nb[0]) | bf16x2_f16_overflow(nb[1]) | bf16x2_f16_overflow(nb[2]) |
              bf16x2_f16_overflow(nb[3]);
      if (router_cta)   // xn rows as bf16 for the router (ring buffer 1, idle until routing)
        *reinterpret_cast<uint4*>(xb + (size_t)t * (H + 8) + 8 * pc) = make_uint4(nb[0], nb[1], nb[2], nb[3]);
      const uint4 o = f16x8_to_perm8(make_uint4(bf16x2_to_f16x2_sat(nb[0]), bf16x2_to_f16x2_sat(nb[1]),
                                                bf16x2_to_f16x2_sat(nb[2]), bf16x2_to_f16x2_sat(nb[3])));
      // piece u = pc % 8 of its group of 64 goes to position 4 (u % 2) + u / 2,
      // so that lane c of a B fragment finds its pieces 2c and 2c + 1 at
      // positions c and 4 + c (two 128-bit loads, adjacent lanes adjacent)
      const int u = pc & 7;
      *reinterpret_cast<uint4*>(xw + t * L.xstride + 32 * (pc >> 3) + 4 * (4 * (u & 1) + (u >> 1))) = o;
    }
  }
  report_range_warp(p.err, over != 0u);
  DEC_TRACE2(3);
  if (router_cta) {
    // router logits of the 8 experts of this CTA's weight box on mma.sync:
    // A = the bf16 token rows (rows 8 .. 15 of the tile hold no token), B = the
    // box's 16-byte weight rows by ldmatrix.trans; warp w takes K in
    // [w H/8, (w+1) H/8), FP32 accumulation. The slice's copy (thousands of
    // 16-byte rows) was issued at launch; the operand rows above were built
    // while it landed.
    if (!mbar_wait_drain(&wbar, 0, p.err.limit_ns)) {
      if (lane == 0) report_timeout(p.err, 44);
      abort_s = 1;
    }
    __syncthreads();
    const int kw = H / kWarps;
    // lane l gives the row address of matrix l / 8: token l % 8 at K offset
    // 8 (l / 8) (A), weight row 8 (l / 8) + l % 8 (B); token rows past T are
    // stale and only feed product rows that are never read
    const uint32_t xa = smem_u32(xb) + (uint32_t)(((lane & 7) * (H + 8) + 8 * (lane >> 3)) * 2);
    const uint32_t wa = smem_u32(wrs) + (uint32_t)((8 * (lane >> 3) + (lane & 7)) * kRBoxE * 2);
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = warp * kw; k0 < (warp + 1) * kw; k0 += 32) {
      uint32_t av[4], bv[4];
      ldsm4(xa + (uint32_t)k0 * 2, av);
      ldsm4_t(wa + (uint32_t)k0 * kRBoxE * 2, bv);
      mma_bf16_16816(d, av[0], 0u, av[1], 0u, bv[0], bv[1]);   // K k0 .. k0 + 15
      mma_bf16_16816(d, av[2], 0u, av[3], 0u, bv[2], bv[3]);   // K k0 + 16 .. k0 + 31
    }
    // D row g = token g, columns 2c and 2c + 1 = the box's experts
    rpart_s[warp][g][2 * c] = d[0];
    rpart_s[warp][g][2 * c + 1] = d[1];
  }
  DEC_TRACE2(4);
  // the zero token row (columns of a tile past its tokens)
  for (int i = tid; i < (int)L.xstride; i += kThreads) xw[kMaxT * L.xstride + i] = 0u;
  __syncthreads();
  DEC_TRACE2(5);
  if (router_cta && tid < T * EPC) {   // the warps' partial sums in warp order
    const int t = tid / EPC, q = tid % EPC;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) v += rpart_s[w][t][ecol + q];
    const int e = e0 + q;
    // one 64-bit store: the value and this launch's tag land together
    if (e < E)
      p.tlog[(size_t)t * E + e] = ((unsigned long long)(ep + 1u) << 32) |
                                  __float_as_uint(v + (p.rbias ? p.rbias[e] : 0.f));
  }

  DEC_TRACE(3);
  // (no grid barrier here: each top-k warp polls its token's logits until
  // every one carries this launch's tag)
  __syncthreads();
  DEC_TRACE(4);
  if (abort_s) goto drain;

  // ------------------------------------------------------- 2. top-k, slots
  if (warp < T) {
    // this token's logits, re-read (bounded) until all carry tag ep + 1
    float lv[VPL];
    const unsigned long long* lrow = p.tlog + (size_t)warp * E;
    const unsigned long long tw0 = globaltimer_ns();
    bool ready;
    {   // first one entry per lane (a 256-byte read per warp), until tagged
      const int e = lane + 32 * (VPL - 1) < E ? lane + 32 * (VPL - 1) : lane;
      while (!__all_sync(0xffffffffu, (unsigned)(ld_relaxed_u64(lrow + e) >> 32) == ep + 1u) &&
             globaltimer_ns() - tw0 <= p.err.limit_ns)
        __nanosleep(64);
    }
    for (;;) {
      bool mine = true;
#pragma unroll
      for (int i = 0; i < VPL; ++i) {
        const int e = lane + 32 * i;
        const unsigned long long v = e < E ? ld_relaxed_u64(lrow + e) : ((unsigned long long)(ep + 1u) << 32);
        mine &= (unsigned)(v >> 32) == ep + 1u;
        lv[i] = e < E ? __uint_as_float((unsigned)v) : -INFINITY;
      }
      if ((ready = __all_sync(0xffffffffu, mine))) break;
      if (globaltimer_ns() - tw0 > p.err.limit_ns) break;
      __nanosleep(32);
    }
    int idx = 0;
    float w = 0.f;
    if (ready) {
      topk_select<VPL>(lv, E, k, idx, w);
    } else {
      if (lane == 0) report_timeout(p.err, 40);
      abort_s = 1;
    }
    if (ready && lane < k) {
      idx_s[warp][lane] = idx;
      w_s[warp][lane] = w;
      atomicOr(&tmask_s[idx], 1u << warp);
      if (cta == 0) {
        if (p.topk_idx) p.topk_idx[warp * k + lane] = idx;
        if (p.topk_w) p.topk_w[warp * k + lane] = w;
      }
    }
  }
  __syncthreads();
  if (abort_s) goto drain;
  DEC_TRACE2(6);
  {
    // slots: 0 = shared (if any), then the selected experts in ascending
    // order, each with its tokens in ascending order; activation row offsets
    // likewise. One block-wide scan: thread i takes experts 2i and 2i + 1
    // and counts (selected experts, their tokens) up to itself.
    const int ea = 2 * tid, eb = 2 * tid + 1;
    const unsigned ma = ea < E ? tmask_s[ea] : 0u, mb = eb < E ? tmask_s[eb] : 0u;
    const int na = (ma != 0u) + (mb != 0u), nc = __popc(ma) + __popc(mb);
    int ia = na, ic = nc;   // inclusive scans over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int xa = __shfl_up_sync(0xffffffffu, ia, o), xc = __shfl_up_sync(0xffffffffu, ic, o);
      if (lane >= o) {
        ia += xa;
        ic += xc;
      }
    }
    if (lane == 31) {
      scan_a[warp] = ia;
      scan_c[warp] = ic;
    }
    __syncthreads();
    int pa = 0, pc = 0, ta = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int va = scan_a[w];
      if (w < warp) {
        pa += va;
        pc += scan_c[w];
      }
      ta += va;
    }
    int sl = p.has_shared + pa + ia - na;          // first slot of this thread's experts
    int so = p.has_shared * T + pc + ic - nc;       // their first activation row
    const unsigned mm[2] = {ma, mb};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const unsigned m = mm[q];
      if (m) {
        const int e = ea + q;
        slot_of_s[e] = sl;
        slot_e[sl] = e;
        cnt_s[sl] = __popc(m);
        soff_s[sl] = so;
        int col = 0;
        for (int t = 0; t < T; ++t)
          if (m & (1u << t)) tok_s[sl][col++] = t;
        ++sl;
        so += __popc(m);
      }
    }
    if (tid == 0) {
      nslots_s = p.has_shared + ta;
      if (p.has_shared) {
        slot_e[0] = -1;
        cnt_s[0] = T;
        soff_s[0] = 0;
      }
    }
    if (p.has_shared && tid < T) tok_s[0][tid] = tid;
  }
  __syncthreads();
  DEC_TRACE2(7);
  n_units = nslots_s * upe;
  n_dc = cta < p.n_dn ? (nslots_s + kSlotsPerChunk - 1) / kSlotsPerChunk : 0;
  DEC_TRACE(5);
  for (int i = tid; i < T * k; i += kThreads) {   // used by the combine, after later barriers
    const int t = i / k, j = i - t * k, e = idx_s[t][j];
    sc_s[t][j] = slot_of_s[e] * 16 + __popc(tmask_s[e] & ((1u << t) - 1u));
  }

  // ----------------------------------------------- 3. gate/up + SwiGLU units
  // One warp per unit: 8 gate rows and the matching 8 up rows of one slot's
  // expert (an m16 tile: row g is gate feature g, row g + 8 its up feature),
  // all K, its fp16 weights rebuilt in registers and SwiGLU in registers --
  // no reduction across warps, no block barrier per unit. Units
  // are dealt over the CTAs first (unit u: CTA u % ncta, warp u / ncta), so
  // every SM takes a share; a warp's unit arrives by TMA in two 3D boxes
  // (8 rows x all K, 128-byte swizzle) into its own buffer, and the scales
  // and biases by bulk copies behind them.
  {
    const int nw = ncta * kWarps, wrank = warp * ncta + cta;   // this warp's place in the deal
    const int nst = H / 256;                                   // 256-K stages per unit
    const int my_units = wrank < n_units ? (n_units - wrank + nw - 1) / nw : 0;
    const uint32_t ub = unit_bytes(H);
    uint8_t* wb = smem + (size_t)warp * ub;                    // in the ring's buffers
    const uint32_t wbase = smem_u32(wb);
    uint64_t* wf = &wfull[warp];
    const uint32_t uwb = unit_words_bytes(H), usb = unit_sb_bytes(H);
    auto wissue = [&](int ui) {   // lane 0: unit ui of this warp's deal
      const int uu = wrank + ui * nw, s = uu / upe, r = uu - s * upe;
      const bool sh = p.has_shared && s == 0;
      const int row0 = (sh ? 0 : slot_e[s] * I) + kGU * r;
      const W4Dev& wg = sh ? p.sgate : p.gate;
      const W4Dev& wu = sh ? p.sup : p.up;
      mbar_arrive_expect_tx(wf, ub);
      tma_load_3d(wb, sh ? &p.msg : &p.mg, 0, row0, 0, wf);
      tma_load_3d(wb + uwb / 2, sh ? &p.msu : &p.mu, 0, row0, 0, wf);
      bulk_load(wb + uwb, wg.s + (size_t)row0 * G, usb, wf);
      bulk_load(wb + uwb + usb, wg.b + (size_t)row0 * G, usb, wf);
      bulk_load(wb + uwb + 2 * usb, wu.s + (size_t)row0 * G, usb, wf);
      bulk_load(wb + uwb + 3 * usb, wu.b + (size_t)row0 * G, usb, wf);
    };
    // (no L2 prefetches anywhere in this kernel: bulk prefetches of the second
    // unit's rows, of the down slabs or of the next layer's router and shared
    // expert each measured slower, as they hold up the issuing SM's copies)
    if (lane == 0 && my_units > 0) wissue(0);
    DEC_WTRACE(0);
    bool wok = true;
    int ui = 0;
    for (; ui < my_units && wok; ++ui) {
      const int uu = wrank + ui * nw, s = uu / upe, r = uu - s * upe;
      const int cnt = cnt_s[s];
      // the token of this lane's B column (g)
      const int trow = g < cnt ? tok_s[s][g] : kMaxT;
      const uint32_t xrow = smem_u32(xw + trow * L.xstride);   // this lane's B column's token row
      // this lane's rows (gate and up row row0 + g): scales and biases of the
      // 4 groups of a stage, from the buffer
      const uint32_t sbrow = wbase + uwb + (uint32_t)(g * G * 2);
      const bool got = mbar_wait_drain(wf, (uint32_t)(ui & 1), p.err.limit_ns);
      if (!(wok = __all_sync(0xffffffffu, got))) {   // (warp-uniform: the MMAs below are warp-wide)
        if (lane == 0) report_timeout(p.err, 41);
        break;
      }
      if (ui == 0) { DEC_WTRACE(1); } else { DEC_WTRACE(4); }
      // rows g (gate) and g + 8 (up) of the m16 tile, fp16 weights fp16(q s + b)
      // rebuilt group by group (one rounding, as the tensor-core GEMM does);
      // one accumulator chain per group of a stage, summed at the end
      float acc[4][4];
#pragma unroll
      for (int gi = 0; gi < 4; ++gi)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[gi][v] = 0.f;
      for (int q = 0; q < nst; ++q) {
        uint2 sbq[4];   // gate s, gate b, up s, up b: groups 4q .. 4q + 3 of row g
#pragma unroll
        for (int a = 0; a < 4; ++a) sbq[a] = lds_v2(sbrow + a * usb + 8 * q);
        const uint32_t zb = wbase + (uint32_t)q * (kGU * 128);   // 256-K chunk q of the gate rows
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          const int grp = 4 * q + gi;
          const uint32_t col = (uint32_t)(((2 * gi + (c >> 1)) ^ g) << 4) + ((c & 1) << 3);
          const uint2 wg = lds_v2(zb + (uint32_t)(g * 128) + col);            // gate row g
          const uint2 wu = lds_v2(zb + uwb / 2 + (uint32_t)(g * 128) + col);   // up row g
          // the token row's pieces 2c (K steps 0, 1) and 2c + 1 (steps 2, 3)
          const uint4 xa = lds_v4(xrow + (uint32_t)(grp * 32 + 4 * c) * 4);
          const uint4 xb4 = lds_v4(xrow + (uint32_t)(grp * 32 + 16 + 4 * c) * 4);
          auto h2 = [&](const uint2& v) {   // this group's bf16 of a table as fp16 (x, x)
            const uint32_t wd = (gi >> 1) ? v.y : v.x;
            return __half2half2(__float2half_rn(bf16_to_f32((uint16_t)((gi & 1) ? wd >> 16 : wd & 0xFFFFu))));
          };
          const __half2 sg2 = h2(sbq[0]), bg2 = h2(sbq[1]), su2 = h2(sbq[2]), bu2 = h2(sbq[3]);
          uint32_t dg[2][4], du[2][4];
          dequant_word_f16_perm8(wg.x, sg2, bg2, dg[0]);
          dequant_word_f16_perm8(wg.y, sg2, bg2, dg[1]);
          dequant_word_f16_perm8(wu.x, su2, bu2, du[0]);
          dequant_word_f16_perm8(wu.y, su2, bu2, du[1]);
          mma_m16n8k16_f16(acc[gi], dg[0][0], du[0][0], dg[0][1], du[0][1], xa.x, xa.y);
          mma_m16n8k16_f16(acc[gi], dg[0][2], du[0][2], dg[0][3], du[0][3], xa.z, xa.w);
          mma_m16n8k16_f16(acc[gi], dg[1][0], du[1][0], dg[1][1], du[1][1], xb4.x, xb4.y);
          mma_m16n8k16_f16(acc[gi], dg[1][2], du[1][2], dg[1][3], du[1][3], xb4.z, xb4.w);
        }
      }
      // D rows g (gate) and g + 8 (up) at columns 2c and 2c + 1
      const float tg0 = (acc[0][0] + acc[1][0]) + (acc[2][0] + acc[3][0]);
      const float tg1 = (acc[0][1] + acc[1][1]) + (acc[2][1] + acc[3][1]);
      const float tu0 = (acc[0][2] + acc[1][2]) + (acc[2][2] + acc[3][2]);
      const float tu1 = (acc[0][3] + acc[1][3]) + (acc[2][3] + acc[3][3]);
      if (ui == 0) { DEC_WTRACE(2); }
      // every word of the unit has been read: the buffer takes the next unit
      __syncwarp();
      if (lane == 0 && ui + 1 < my_units) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        wissue(ui + 1);
      }
      // SwiGLU: feature kGU r + g of the slot's tokens 2c and 2c + 1 (fp16, perm8 order)
      const int fpos = perm8_pos(kGU * r + g);
      uint32_t big = 0u;
      if (2 * c < cnt) {
        const float a = silu_fast(tg0) * tu0;
        big |= fabsf(a) > kF16Max ? 1u : 0u;
        p.act[(size_t)(soff_s[s] + 2 * c) * I + fpos] = f32_to_f16_sat(a);
      }
      if (2 * c + 1 < cnt) {
        const float a = silu_fast(tg1) * tu1;
        big |= fabsf(a) > kF16Max ? 1u : 0u;
        p.act[(size_t)(soff_s[s] + 2 * c + 1) * I + fpos] = f32_to_f16_sat(a);
      }
      report_range_warp(p.err, big != 0u);
      if (ui == 0) { DEC_WTRACE(3); } else { DEC_WTRACE(5); }
    }
    if (!wok) {
      // this warp's own copy (unit ui, issued) lands before the CTA gives up
      mbar_wait_drain(wf, (uint32_t)(ui & 1), p.err.limit_ns);
      if (lane == 0) abort_s = 1;
    }
  }

  DEC_TRACE(6);
  // the first down chunks are issued while thread 0 waits in the grid
  // barrier (every warp's unit buffer, the whole ring, has been read at its
  // first sync), one chunk per issuing thread: lane 0 of warps 4 .. 7 takes
  // chunk warp - 4
  ok = grid_barrier(p.bar, (unsigned)ncta, p.err, 42, &flag_s, [&] {
    const int b = warp - (kWarps - kRing);
    if (lane == 0 && b >= 0 && b < n_dc && !abort_s) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(b);
      atomicOr(&ring_issued_s, 1u << b);
    }
  });
  DEC_TRACE(7);
  if (!ok || abort_s) goto drain;

  // ------------------------------------------ 4. down, combine, stack update
  if (n_dc > 0) {
    float* dsum = reinterpret_cast<float*>(smem + L.xw);   // [slot][kDn][kMaxT]
    // The activation row of this lane's column for slot s, all of its groups:
    // 16-byte pieces 8 grp + 2 c and the next (K blocks of 8), issued at once.
    auto load_act = [&](int s, uint4 (&v)[16]) {
      const bool have = s < nslots_s && g < cnt_s[s];
      const uint4* arow =
          reinterpret_cast<const uint4*>(p.act + (size_t)(have ? soff_s[s] + g : 0) * I);
#pragma unroll
      for (int grp = 0; grp < 8; ++grp) {
        v[2 * grp] = (have && grp < GI) ? __ldcg(arow + 8 * grp + 2 * c) : make_uint4(0u, 0u, 0u, 0u);
        v[2 * grp + 1] = (have && grp < GI) ? __ldcg(arow + 8 * grp + 2 * c + 1) : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    // One slot: its 16 down rows (ring buffer b, position q) times its
    // activation rows; the FP32 result goes to dsum. The rows' fp16 weights
    // fp16(q s + b) are rebuilt group by group, as in step 3.
    auto down_slot = [&](int s, int b, int q, const uint4 (&v)[16]) {
      const uint32_t bq = sbase + (uint32_t)b * L.slab + (uint32_t)q * dn_q;
      const uint16_t* ssc = reinterpret_cast<const uint16_t*>(
          smem + (size_t)b * L.slab + kSlotsPerChunk * dn_q + q * dn_s);
      const uint16_t* sbi = reinterpret_cast<const uint16_t*>(
          smem + (size_t)b * L.slab + kSlotsPerChunk * (dn_q + dn_s) + q * dn_s);
      float acc[4][4];
#pragma unroll
      for (int gi = 0; gi < 4; ++gi)
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) acc[gi][v4] = 0.f;
#pragma unroll
      for (int g0 = 0; g0 < 8; g0 += 4) {
        if (g0 >= GI) break;
        // four groups at a time, one accumulator chain each
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          const int grp = g0 + gi;
          // packed words of rows g (h = 0) and g + 8 (h = 1) of the tile
          const uint2 w0 = lds_v2(bq + qoff(g, grp, c, kDn));
          const uint2 w1 = lds_v2(bq + qoff(g + 8, grp, c, kDn));
          auto h2 = [](uint16_t v) { return __half2half2(__float2half_rn(bf16_to_f32(v))); };
          uint32_t d0[2][4], d1[2][4];
          {
            const __half2 s2 = h2(ssc[g * GI + grp]), b2 = h2(sbi[g * GI + grp]);
            dequant_word_f16_perm8(w0.x, s2, b2, d0[0]);
            dequant_word_f16_perm8(w0.y, s2, b2, d0[1]);
          }
          {
            const __half2 s2 = h2(ssc[(g + 8) * GI + grp]), b2 = h2(sbi[(g + 8) * GI + grp]);
            dequant_word_f16_perm8(w1.x, s2, b2, d1[0]);
            dequant_word_f16_perm8(w1.y, s2, b2, d1[1]);
          }
          const uint4 va = v[2 * grp], vb = v[2 * grp + 1];   // K steps 0, 1 and 2, 3
          mma_m16n8k16_f16(acc[gi], d0[0][0], d1[0][0], d0[0][1], d1[0][1], va.x, va.y);
          mma_m16n8k16_f16(acc[gi], d0[0][2], d1[0][2], d0[0][3], d1[0][3], va.z, va.w);
          mma_m16n8k16_f16(acc[gi], d0[1][0], d1[1][0], d0[1][1], d1[1][1], vb.x, vb.y);
          mma_m16n8k16_f16(acc[gi], d0[1][2], d1[1][2], d0[1][3], d1[1][3], vb.z, vb.w);
        }
      }
      // D rows g and g + 8 at columns 2c and 2c + 1
      float tot[4];
#pragma unroll
      for (int v4 = 0; v4 < 4; ++v4) tot[v4] = (acc[0][v4] + acc[1][v4]) + (acc[2][v4] + acc[3][v4]);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const int col = 2 * c + (qq & 1), row = g + 8 * (qq >> 1);
        dsum[(s * kDn + row) * kMaxT + col] = tot[qq];
      }
    };
#ifdef MOE_DEC_TRACE
    if (tid == 0 && blockIdx.x < 256) g_dec_trace[blockIdx.x][12] = globaltimer_ns();
#endif
    if (n_dc <= kRing) {
      // every down chunk's copy was issued during step 3: each warp walks its
      // slots (s = warp, warp + 8, ...), loading the next slot's activations
      // while it computes the current one
      uint4 cur[16], nxt[16];
      load_act(warp, cur);
      for (int s = warp; s < nslots_s; s += kSlotsPerChunk) {
        load_act(s + kSlotsPerChunk, nxt);
        const int i = s / kSlotsPerChunk, b = ring_buf(i);
        if (!mbar_wait_drain(&full[b], (uint32_t)((i / kRing) & 1), p.err.limit_ns)) {
          if (lane == 0) report_timeout(p.err, 43);
          abort_s = 1;
          break;
        }
        down_slot(s, b, s % kSlotsPerChunk, cur);
#pragma unroll
        for (int j = 0; j < 16; ++j) cur[j] = nxt[j];
      }
      __syncthreads();
      if (abort_s) goto drain;
    } else {
      // more chunks than buffers: chunk by chunk, reusing buffers
      for (int ch = 0; ch < n_dc; ++ch) {
        const int i = ch, b = ring_buf(i);
        uint4 cur[16];
        const int s = kSlotsPerChunk * ch + warp;
        load_act(s, cur);
        if (!mbar_wait_drain(&full[b], (uint32_t)((i / kRing) & 1), p.err.limit_ns)) {
          if (lane == 0) report_timeout(p.err, 43);
          abort_s = 1;
        }
        __syncthreads();
        if (abort_s) goto drain;
        if (s < nslots_s) down_slot(s, b, warp, cur);
        __syncthreads();
        if (tid == kIssuer && i + kRing < n_dc) issue(i + kRing);
      }
    }
#ifdef MOE_DEC_TRACE
    if (tid == 0 && blockIdx.x < 256) g_dec_trace[blockIdx.x][13] = globaltimer_ns();
#endif
    // y[t] = shared + sum_j w[t][j] * expert_j[t] (FP32, rank order); x update
    if (tid < T * kDn) {
      const int t = tid / kDn, hh = tid % kDn;
      float y = p.has_shared ? dsum[(0 * kDn + hh) * kMaxT + t] : 0.f;
      for (int j = 0; j < k; ++j) {
        const int scv = sc_s[t][j];
        y = fmaf(w_s[t][j], dsum[((scv >> 4) * kDn + hh) * kMaxT + (scv & 15)], y);
      }
      const int h = kDn * cta + hh;
      p.x[(size_t)t * H + h] = f32_to_bf16(fmaf(p.alpha, y, x_s[t][hh]));
      if (p.y_out) p.y_out[(size_t)t * H + h] = y;
    }
  }
  __syncthreads();
  DEC_TRACE(8);
  // the last CTA to leave sets the counter back to 0 and advances the launch
  // count (the next launch's logits tag)
  if (tid == 0 && atomicAdd(p.bar, 1u) == 2u * ncta - 1u) {
    *p.bar = 0u;
    *p.epoch = ep + 1u;
  }
  return;

drain:
  // a wait gave up: let this CTA's own copies land before it exits (the
  // counter stays set; moe_get_error clears it with the error word)
  __syncthreads();
  if (tid == 0 && router_cta) mbar_wait_drain(&wbar, 0, p.err.limit_ns);
  if (tid == kIssuer) {
    // buffer b holds first-round chunk b if its bit is set, then (step 4 with
    // more chunks than buffers, issued by kIssuer) chunks b + kRing, ... below
    // `issued`
    const int hi = issued > kRing ? issued : kRing;
    for (int b = 0; b < kRing; ++b) {
      if (!((ring_issued_s >> b) & 1u)) continue;
      const int last = b + ((hi - 1 - b) / kRing) * kRing;   // last chunk i = b (mod kRing)
      mbar_wait_drain(&full[ring_buf(b)], (uint32_t)((last / kRing) & 1), p.err.limit_ns);
    }
  }
  __syncthreads();
}

}  // namespace dec

#ifdef MOE_DEC_TRACE
extern "C" int moe_debug_dec_trace(unsigned long long* out) {
  return (int)cudaMemcpyFromSymbol(out, dec::g_dec_trace, sizeof(dec::g_dec_trace));
}
extern "C" int moe_debug_dec_trace2(unsigned long long* out) {
  return (int)cudaMemcpyFromSymbol(out, dec::g_dec_trace2, sizeof(dec::g_dec_trace2));
}
extern "C" int moe_debug_dec_btrace(unsigned long long* out) {
  return (int)cudaMemcpyFromSymbol(out, dec::g_dec_btrace, sizeof(dec::g_dec_btrace));
}
extern "C" int moe_debug_dec_wtrace(unsigned long long* out) {
  return (int)cudaMemcpyFromSymbol(out, dec::g_dec_wtrace, sizeof(dec::g_dec_wtrace));
}
#endif

bool decode_fused_fits(int T, int H, int I, int E, int k, int has_shared, int num_sms) {
  if (T < 1 || T > dec::kMaxT || k > 32 || E > 512 || E % 8) return false;
  if (H % 512 || I % 256 || I / 64 > 8 || H / 8 > 2 * dec::kThreads || H / dec::kDn > num_sms)
    return false;
  if (E % dec::kRBoxE || E / dec::kRBoxE > num_sms) return false;
  const dec::Smem L = dec::smem_layout(H, I);
  if ((uint32_t)H * dec::kRBoxE * 2 > L.slab) return false;   // router slice in one ring buffer
  if ((uint32_t)dec::kMaxT * (H + 8) * 2 > L.slab) return false;   // bf16 token rows in another
  const int slots = T * k + has_shared;
  if (slots > dec::kMaxSlots || (uint32_t)slots * dec::kDn * dec::kMaxT * 4 > L.dsum_cap) return false;
  if (L.total + 1024 > 227 * 1024) return false;
  int dev = 0, coop = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
    return false;
  auto kern = E <= 256 ? (E <= 2 * num_sms ? dec::moe_decode_layer_kernel<8, 2> : dec::moe_decode_layer_kernel<8, 8>)
                       : dec::moe_decode_layer_kernel<16, 8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.total + 1024) !=
      cudaSuccess)
    return false;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, dec::kThreads, L.total + 1024) !=
      cudaSuccess)
    return false;
  return per_sm >= 1;
}

cudaError_t launch_decode_layer(const DecodeLayerArgs& a, DevErr err, int num_sms, cudaStream_t st) {
  dec::Params p;
  p.T = a.T;
  p.H = a.H;
  p.I = a.I;
  p.E = a.E;
  p.k = a.k;
  p.has_shared = a.has_shared;
  p.alpha = a.alpha;
  p.eps = a.eps;
  p.n_dn = a.H / dec::kDn;
  p.x = a.x;
  p.wr = a.router_w;
  p.rbias = a.router_bias;
  p.gate = a.gate;
  p.up = a.up;
  p.down = a.down;
  p.sgate = a.sgate;
  p.sup = a.sup;
  p.sdown = a.sdown;
  p.mg = a.maps[0];
  p.mu = a.maps[1];
  p.md = a.maps[2];
  p.msg = a.maps[3];
  p.msu = a.maps[4];
  p.msd = a.maps[5];
  p.mr = a.router_map;
  p.epoch = a.epoch;
  p.tlog = a.tlogits;
  p.act = a.act;
  p.topk_idx = a.topk_idx;
  p.topk_w = a.topk_w;
  p.y_out = a.y_out;
  p.bar = a.bar;
  p.err = err;
  const dec::Smem L = dec::smem_layout(a.H, a.I);
  const size_t smem = L.total + 1024;
  auto kern = a.E <= 256 ? (a.E <= 2 * num_sms ? dec::moe_decode_layer_kernel<8, 2>
                                                : dec::moe_decode_layer_kernel<8, 8>)
                         : dec::moe_decode_layer_kernel<16, 8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(dec::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // cooperative (the CTAs wait on one another at the grid barriers), and,
  // where the runtime takes both, with programmatic dependent launch so the
  // prologue's weight copies overlap the previous launch
  static int pdl_ok = -1;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  if (pdl_ok != 0) {
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e == cudaSuccess) {
      pdl_ok = 1;
      return e;
    }
    cudaGetLastError();   // the combination was refused: cooperative only from now on
    pdl_ok = 0;
  }
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace moe
