// gemm_smallm.cu -- grouped W4A16 expert GEMM for decode-sized token groups.
//
// Same product as gemm_tc.cu (the grouped GEMM with block-wise dequant of
// "Perplexity libera Lily, un motor de IA que supera a MLX-LM en Apple
// Silicon", diariobitcoin.com, section "Las optimizaciones en el prefill"),
// for the regime of section "El decode busca mover menos datos": with a
// handful of tokens per expert the block is bound by streaming the packed
// weights once, so this kernel is written around HBM bandwidth and latency,
// not MMA rate.
//
// Design:
//   * a unit is (block-map tile, chunk of weight rows): 32 gate + 32 up rows
//     for the gate/up pass, 128 down rows for the down pass, so that a
//     decode-sized layer spreads over all SMs; 8 warps;
//   * the unit's weight slab is copied into shared memory by the TMA unit in
//     a few large requests (the copy engine takes a request every ~60 cycles
//     whatever its size, and per-thread 16-byte copies stall at a few tens
//     of GB/s per SM): 2D boxes of 32 packed words x the unit's rows with the
//     128-byte swizzle (fragment reads conflict-free without padding), and
//     one bulk copy each for the rows' scales and biases;
//   * warp w owns 16 output rows (row warp) and a slice of the K groups
//     (split K): each warp holds two 16-row m16n8k16 A tiles (gate and up
//     rows, or two down row slabs) and the tile's tokens are the n8 side, in
//     passes of 8*NT tokens; the split-K partial sums are added in a fixed
//     order through shared memory (deterministic);
//   * each thread reads 8 bytes of packed weights per row per group, and
//     converts nibbles to fp16 "1024 + q" with one LOP3 per pair (exact);
//     the MMA sums (1024+q)*x over one group of 64 in FP32, and the group's
//     affine map is applied to the 4 partial sums:
//         sum_k w_k x_k = s * sum_k (1024+q_k) x_k + (b - 1024 s) * sum_k x_k
//     which is exact algebra of w = q*s + b (the group sums of x are
//     precomputed in FP32 while the tokens are staged in shared memory);
//   * token rows are kept with each 8-element block in the order
//     (0,4,1,5,2,6,3,7), the order the nibble extraction yields, so A and B
//     fragments agree on which k each MMA slot holds without any shuffle;
//     the gate/up pass reads the layer's bf16 token rows through perm and
//     converts them itself (no gathered copy), the down pass reads the
//     SwiGLU rows the gate/up pass wrote in that order;
//   * the down pass follows the gate/up pass, which writes neither the block
//     map nor any weight, so it finds its unit and starts its slab copy
//     before waiting for that launch.
#include "moe_common.cuh"

namespace moe {
namespace sm {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kPF = 4;   // groups per batch (= one 8-byte scale/bias load)

struct Params {
  int mode;              // 0 gate/up + SwiGLU, 1 down * weight
  int T, k, E, K, N;
  int nchunk;            // units per tile
  int ru;                // weight rows per matrix in a unit (32 gate/up, 128 down)
  int has_shared;
  const int32_t* bmap;
  const int32_t* num_tiles;
  const uint16_t* act_in;
  const uint16_t* gather_x;   // gate/up: bf16 token rows read through perm
  uint16_t* out;
  float* out_sh;
  int out_ld;
  const float* topk_w;
  const int32_t* perm;
  W4Dev w0, w1, sw0, sw1;     // scales and biases (packed words come through the maps)
  W4Dev next, snext;          // gate/up: down matrices to prefetch into L2 (q null: none)
  int next_K, next_rows;      // their reduction size, and rows per gate/up unit
  SmallMaps maps;
  DevErr err;
};

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared memory of a CTA, in bytes from a 1024-aligned base:
//   slab  [nbuf] x { q [matrices][K/256 boxes][ru rows][128 B] (swizzled TMA
//         boxes), s, b [matrices][ru rows][K/64] bf16 each }
//   xw    [8*NT][K/2 + 1] words (token rows, perm8 fp16, padded)
//   xg    [8*NT][K/64] fp32 (token group sums)
//   red   [split-K - 1][row warps][32 lanes][2*NT*4] fp32
struct Layout {
  int nm, ru, rw, sk, nt, nbuf;
  size_t s, b, slab, xw, xg, red, total;
};

__host__ __device__ inline Layout layout(int mode, int K, int nt, int nbuf) {
  Layout L;
  L.nm = mode == 0 ? 2 : 1;
  L.ru = mode == 0 ? 32 : 128;
  L.rw = mode == 0 ? L.ru / 16 : L.ru / 32;   // row warps
  const int G = K / 64;
  int sk = kWarps / L.rw;                       // split K, whole batches of 4 groups each
  while (sk > 1 && (G % sk || (G / sk) % kPF)) --sk;
  L.sk = sk;
  L.nt = nt;
  L.nbuf = nbuf;
  const size_t qbytes = (size_t)L.nm * L.ru * K / 2;
  const size_t sbytes = (size_t)L.nm * L.ru * G * 2;
  L.s = qbytes;                                 // offsets inside one slab
  L.b = qbytes + sbytes;
  L.slab = (qbytes + 2 * sbytes + 1023) / 1024 * 1024;
  size_t o = L.slab * nbuf;
  L.xw = o;
  o += (size_t)8 * nt * (K / 2 + 1) * 4;
  L.xg = o;
  o += (size_t)8 * nt * G * 4;
  L.red = o;
  o += (size_t)(L.sk - 1) * L.rw * 32 * 8 * nt * 4;
  L.total = o;
  return L;
}

// A unit: the shared expert's tiles come first (their weights are known
// before the routing), then the routed tiles of the block map.
struct Unit {
  bool valid, shared;
  int ch, e, m0, rows;
};

template <int NT, int NBUF>
__global__ void __launch_bounds__(kThreads) w4_grouped_gemm_smallm(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t slab_bar[NBUF];
  __shared__ int src_row[8 * NT];   // source row of each token row of a pass (-1: none)
  const int K = p.K;
  const int G = K / 64;
  const Layout L = layout(p.mode, K, NT, NBUF);
  const int xstride = K / 2 + 1;
  uint32_t* xw = reinterpret_cast<uint32_t*>(smem + L.xw);
  float* xg = reinterpret_cast<float*>(smem + L.xg);
  float* red = reinterpret_cast<float*>(smem + L.red);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ru = L.ru;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int b = 0; b < NBUF; ++b) mbar_init(&slab_bar[b], 1);
    fence_mbar_init();
    tma_prefetch_desc(&p.maps.q0);
    tma_prefetch_desc(&p.maps.q1);
    tma_prefetch_desc(&p.maps.sq0);
    tma_prefetch_desc(&p.maps.sq1);
  }
  __syncthreads();

  // The down pass follows the gate/up pass, which writes neither the block
  // map nor any weight: it resolves units and copies slabs before waiting
  // for that launch. The gate/up pass follows the routing: only a shared
  // expert unit can start its copy before the wait.
  const bool early = p.mode == 1;
  bool waited = false;
  auto wait_prev = [&] {
    if (!waited) {
      pdl_begin();
      waited = true;
    }
  };
  const int n_shared_units = (p.has_shared ? (p.T + kBM - 1) / kBM : 0) * p.nchunk;
  int n_routed = -1;
  auto resolve = [&](int u) {
    Unit x;
    x.valid = true;
    if (u < n_shared_units) {
      const int i = u / p.nchunk;
      x.shared = true;
      x.ch = u - i * p.nchunk;
      x.e = 0;
      x.m0 = p.T * p.k + kBM * i;
      x.rows = min(kBM, p.T - kBM * i);
      return x;
    }
    if (n_routed < 0) {
      if (!early) wait_prev();
      n_routed = __ldcg(p.num_tiles);
    }
    const int v = u - n_shared_units, tile = v / p.nchunk;
    x.shared = false;
    x.valid = tile < n_routed;
    x.ch = v - tile * p.nchunk;
    x.e = x.m0 = x.rows = 0;
    if (x.valid) {
      x.e = __ldcg(p.bmap + 3 * tile);
      x.m0 = __ldcg(p.bmap + 3 * tile + 1);
      x.rows = __ldcg(p.bmap + 3 * tile + 2);
    }
    return x;
  };
  // slab copy of unit x into buffer b: TMA boxes of the packed words, bulk
  // copies of the scales and biases (one elected thread)
  auto issue = [&](const Unit& x, int b) {
    if (warp == 0 && elect_one_sync()) {
      uint8_t* slab = smem + (size_t)b * L.slab;
      const int nb = K / 256;
      const uint32_t sbytes = (uint32_t)ru * G * 2;
      const int grow0 = (x.shared ? 0 : x.e * p.N) + ru * x.ch;
      mbar_arrive_expect_tx(&slab_bar[b], (uint32_t)L.nm * (ru * K / 2 + 2 * sbytes));
      for (int m = 0; m < L.nm; ++m) {
        const CUtensorMap* map = x.shared ? (m ? &p.maps.sq1 : &p.maps.sq0)
                                          : (m ? &p.maps.q1 : &p.maps.q0);
        const W4Dev& w = x.shared ? (m ? p.sw1 : p.sw0) : (m ? p.w1 : p.w0);
        for (int bx = 0; bx < nb; ++bx)
          tma_load_2d(slab + ((size_t)m * nb + bx) * ru * 128, map, 32 * bx, grow0, &slab_bar[b]);
        bulk_load(slab + L.s + (size_t)m * sbytes, w.s + (size_t)grow0 * G, sbytes, &slab_bar[b]);
        bulk_load(slab + L.b + (size_t)m * sbytes, w.b + (size_t)grow0 * G, sbytes, &slab_bar[b]);
      }
      // gate/up: this unit's share of the expert's down rows goes to L2 now,
      // so that the down pass finds them there
      const W4Dev& nw = x.shared ? p.snext : p.next;
      if (nw.q) {
        const size_t r0 = (size_t)(x.shared ? 0 : x.e * p.K) + (size_t)p.next_rows * x.ch;
        const uint32_t rows = (uint32_t)p.next_rows;
        bulk_prefetch_l2(nw.q + r0 * (p.next_K / 8), rows * (uint32_t)(p.next_K / 2));
        bulk_prefetch_l2(nw.s + r0 * (p.next_K / 64), rows * (uint32_t)(p.next_K / 32));
        bulk_prefetch_l2(nw.b + r0 * (p.next_K / 64), rows * (uint32_t)(p.next_K / 32));
      }
    }
  };

  // ---- this warp's rows and K slice
  const int rw = warp % L.rw, ks = warp / L.rw;
  const bool computes = ks < L.sk;
  const int gw = G / L.sk, gbeg = ks * gw, gend = gbeg + gw;
  const int g = lane >> 2, c = lane & 3;
  // slab row of (A tile mt, half h) and its matrix
  int srow[2][2], smat[2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    smat[mt] = p.mode == 0 ? mt : 0;
#pragma unroll
    for (int h = 0; h < 2; ++h)
      srow[mt][h] = (p.mode == 0 ? 16 * rw : 32 * rw + 16 * mt) + g + 8 * h;
  }
  // byte offsets: row part of the q address (box 0) and the swizzled column
  // part of group i of a batch of 4 (words 8 i + 2 c, 8 i + 2 c + 1 sit in
  // 16-byte chunk 2 i + c/2, stored at chunk (2 i + c/2) ^ (row & 7), and
  // row & 7 = g for every row this thread reads)
  const int nb = K / 256;
  uint32_t qrow[2][2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h)
      qrow[mt][h] = smem_u32(smem) + (uint32_t)(((size_t)smat[mt] * nb * ru + srow[mt][h]) * 128);
  uint32_t qcol[kPF];
#pragma unroll
  for (int i = 0; i < kPF; ++i) qcol[i] = (uint32_t)((((2 * i + (c >> 1)) ^ g) << 4) + 8 * (c & 1));
  const uint32_t box_bytes = (uint32_t)ru * 128;

  int u = blockIdx.x;
  Unit cur = resolve(u);
  if (cur.valid) issue(cur, 0);
  for (int it = 0; cur.valid; ++it) {
    const int buf = NBUF == 2 ? (it & 1) : 0;
    const uint32_t parity = NBUF == 2 ? (uint32_t)((it >> 1) & 1) : (uint32_t)(it & 1);
    wait_prev();
    const uint32_t slab_u32 = (uint32_t)buf * (uint32_t)L.slab;
    const uint16_t* ss = reinterpret_cast<const uint16_t*>(smem + (size_t)buf * L.slab + L.s);
    const uint16_t* sb = reinterpret_cast<const uint16_t*>(smem + (size_t)buf * L.slab + L.b);
    auto ldq = [&](int mt, int h, int g0, int i) {
      uint2 v;
      asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                   : "=r"(v.x), "=r"(v.y)
                   : "r"(qrow[mt][h] + slab_u32 + (uint32_t)(g0 / 4) * box_bytes + qcol[i]));
      return v;
    };
    auto ldsb = [&](const uint16_t* base, int mt, int h, int g0) {
      return *reinterpret_cast<const uint2*>(base + ((size_t)smat[mt] * ru + srow[mt][h]) * G + g0);
    };
    const int un = u + gridDim.x;
    Unit next;
    next.valid = false;

    for (int pass0 = 0; pass0 < cur.rows; pass0 += 8 * NT) {
      const int prow = min(8 * NT, cur.rows - pass0);
      // stage tokens: source rows first (warp 1, one round trip for the perm
      // lookups, while warp 0 issues copies), then every thread issues all
      // its loads before using any of them
      if (threadIdx.x >= 32 && threadIdx.x < 32 + 8 * NT) {
        const int tr = threadIdx.x - 32, pos = cur.m0 + pass0 + tr;
        int sr = -1;
        if (tr < prow)
          sr = !p.gather_x ? pos : pos < p.T * p.k ? __ldg(p.perm + pos) / p.k : pos - p.T * p.k;
        src_row[tr] = sr;
      }
      __syncthreads();
      const uint16_t* rows_in = p.gather_x ? p.gather_x : p.act_in;
      uint32_t over = 0u;   // bf16 token values that saturate in fp16
      for (int base = 0; base < 8 * NT * G; base += 2 * kThreads) {
        uint4 v[2][8];
        int sr[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int idx = base + q * kThreads + threadIdx.x;
          const int tr = idx / G, grp = idx - tr * G;
          sr[q] = idx < 8 * NT * G ? src_row[tr] : -1;
          if (sr[q] >= 0) {
            const uint4* src =
                reinterpret_cast<const uint4*>(rows_in + (size_t)sr[q] * K + grp * 64);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[q][j] = __ldg(src + j);
          }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int idx = base + q * kThreads + threadIdx.x;
          if (idx >= 8 * NT * G) continue;
          const int tr = idx / G, grp = idx - tr * G;
          float sum = 0.f;
          uint32_t* dst = xw + tr * xstride + grp * 32;
          if (sr[q] >= 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint4 x8 = v[q][j];
              if (p.gather_x) {   // bf16 token values -> the fp16 perm8 operand of a gathered row
                over |= bf16x2_f16_overflow(x8.x) | bf16x2_f16_overflow(x8.y) |
                        bf16x2_f16_overflow(x8.z) | bf16x2_f16_overflow(x8.w);
                x8 = f16x8_to_perm8(make_uint4(bf16x2_to_f16x2_sat(x8.x), bf16x2_to_f16x2_sat(x8.y),
                                               bf16x2_to_f16x2_sat(x8.z), bf16x2_to_f16x2_sat(x8.w)));
              }
              dst[4 * j + 0] = x8.x;   // (x0, x4)
              dst[4 * j + 1] = x8.y;   // (x1, x5)
              dst[4 * j + 2] = x8.z;   // (x2, x6)
              dst[4 * j + 3] = x8.w;   // (x3, x7)
              sum += f16_lo(x8.x) + f16_hi(x8.x) + f16_lo(x8.y) + f16_hi(x8.y) +
                     f16_lo(x8.z) + f16_hi(x8.z) + f16_lo(x8.w) + f16_hi(x8.w);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) dst[j] = 0u;
          }
          xg[tr * G + grp] = sum;
        }
      }
      report_range_warp(p.err, over != 0u);
      if (pass0 == 0) {
        // bounded wait for the slab; on a timeout the error is latched and
        // the CTA stops (outputs of the unit left unwritten)
        bool ok = true;
        if (!mbar_wait_drain(&slab_bar[buf], parity, p.err.limit_ns)) {
          report_timeout(p.err, 20 + p.mode);
          ok = false;
        }
        if (__syncthreads_or(!ok)) return;
        // the next unit's copy goes into the other buffer while this one computes
        if (NBUF == 2) {
          next = resolve(un);
          if (next.valid) issue(next, buf ^ 1);
        }
      } else {
        __syncthreads();
      }

      float tot[2][NT][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int i = 0; i < 4; ++i) tot[mt][nt][i] = 0.f;

      if (computes) {
        uint2 qr[kPF][2][2];
#pragma unroll
        for (int i = 0; i < kPF; ++i)
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) qr[i][mt][h] = ldq(mt, h, gbeg, i);
        uint2 sr[2][2], br[2][2];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            sr[mt][h] = ldsb(ss, mt, h, gbeg);
            br[mt][h] = ldsb(sb, mt, h, gbeg);
          }

        for (int g0 = gbeg; g0 < gend; g0 += kPF) {
          uint2 srn[2][2], brn[2][2];
          const bool more = g0 + kPF < gend;
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              srn[mt][h] = more ? ldsb(ss, mt, h, g0 + kPF) : sr[mt][h];
              brn[mt][h] = more ? ldsb(sb, mt, h, g0 + kPF) : br[mt][h];
            }
#pragma unroll
          for (int i = 0; i < kPF; ++i) {
            const int grp = g0 + i;
            // A fragments: nibble pairs of this group's two words per row
            uint32_t pa[2][2][2][4];   // [mt][h][word][pair]
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                nibbles_to_f16x2_1024(qr[i][mt][h].x, pa[mt][h][0]);
                nibbles_to_f16x2_1024(qr[i][mt][h].y, pa[mt][h][1]);
              }
            if (more) {
#pragma unroll
              for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) qr[i][mt][h] = ldq(mt, h, g0 + kPF, i);
            }
            float acc[2][NT][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[mt][nt][q] = 0.f;
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              const int wsel = s >> 1, psel = 2 * (s & 1);
              const int wabs = grp * 8 + 2 * c + wsel;      // packed word index in the row
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const uint32_t* xr = xw + (nt * 8 + g) * xstride + 4 * wabs + psel;
                const uint32_t b0 = xr[0], b1 = xr[1];
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
                  mma_16816(acc[mt][nt], pa[mt][0][wsel][psel], pa[mt][1][wsel][psel],
                            pa[mt][0][wsel][psel + 1], pa[mt][1][wsel][psel + 1], b0, b1);
              }
            }
            // affine map of the group: s * acc + (b - 1024 s) * sum(x)
            const int half = (i & 1) ? 16 : 0;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              float sc[2], cb[2];
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint32_t sv = ((i >> 1) ? sr[mt][h].y : sr[mt][h].x) >> half;
                const uint32_t bv = ((i >> 1) ? br[mt][h].y : br[mt][h].x) >> half;
                sc[h] = bf16_to_f32(static_cast<uint16_t>(sv & 0xFFFFu));
                cb[h] = fmaf(-1024.0f, sc[h], bf16_to_f32(static_cast<uint16_t>(bv & 0xFFFFu)));
              }
#pragma unroll
              for (int nt = 0; nt < NT; ++nt) {
                const float x0 = xg[(nt * 8 + 2 * c) * G + grp];
                const float x1 = xg[(nt * 8 + 2 * c + 1) * G + grp];
                tot[mt][nt][0] += fmaf(sc[0], acc[mt][nt][0], cb[0] * x0);
                tot[mt][nt][1] += fmaf(sc[0], acc[mt][nt][1], cb[0] * x1);
                tot[mt][nt][2] += fmaf(sc[1], acc[mt][nt][2], cb[1] * x0);
                tot[mt][nt][3] += fmaf(sc[1], acc[mt][nt][3], cb[1] * x1);
              }
            }
          }
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              sr[mt][h] = srn[mt][h];
              br[mt][h] = brn[mt][h];
            }
        }
      }

      // split K: slices 1.. hand their sums to slice 0, which adds them in order
      if (L.sk > 1) {
        if (computes && ks > 0) {
          float* r = red + (((size_t)(ks - 1) * L.rw + rw) * 32 + lane) * 8 * NT;
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int q = 0; q < 4; ++q) r[(mt * NT + nt) * 4 + q] = tot[mt][nt][q];
        }
        __syncthreads();
        if (ks == 0) {
          for (int s2 = 1; s2 < L.sk; ++s2) {
            const float* r = red + (((size_t)(s2 - 1) * L.rw + rw) * 32 + lane) * 8 * NT;
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
              for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int q = 0; q < 4; ++q) tot[mt][nt][q] += r[(mt * NT + nt) * 4 + q];
          }
        }
      }
      if (ks == 0) {
        // epilogue (slice-0 warps); n0, n1: the rows' indices in the weight matrix
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int tok = nt * 8 + 2 * c + (q & 1);
            if (tok >= prow) continue;
            const int pos = cur.m0 + pass0 + tok;
            const int h = q >> 1;
            const int n0 = ru * cur.ch + srow[0][h], n1 = ru * cur.ch + srow[1][h];
            if (p.mode == 0) {
              const float a = silu_fast(tot[0][nt][q]) * tot[1][nt][q];
              p.out[(size_t)pos * p.out_ld + perm8_pos(n0)] = f32_to_f16_sat(a);
            } else if (cur.shared) {
              float* o = p.out_sh + (size_t)(pos - p.T * p.k) * p.out_ld;
              o[n0] = tot[0][nt][q];
              o[n1] = tot[1][nt][q];
            } else {
              const float wt = __ldg(p.topk_w + __ldg(p.perm + pos));
              p.out[(size_t)pos * p.out_ld + n0] = f32_to_bf16(tot[0][nt][q] * wt);
              p.out[(size_t)pos * p.out_ld + n1] = f32_to_bf16(tot[1][nt][q] * wt);
            }
          }
      }
      // token rows, group sums and split-K sums are rewritten by the next pass
      __syncthreads();
    }
    // the slab of this unit is free now: a single buffer takes the next copy
    if (NBUF == 1) {
      next = resolve(un);
      if (next.valid) issue(next, 0);
    }
    u = un;
    cur = next;
  }
}

size_t smem_bytes(int mode, int K, int nt, int nbuf) {
  return layout(mode, K, nt, nbuf).total + 1024;   // + alignment of the swizzled boxes
}

}  // namespace sm

int smallm_rows_per_unit(int mode) { return mode == 0 ? 32 : 128; }

bool smallm_fits(int H, int I) {
  // shapes the unit layout covers, and one pass of 8 token rows in shared memory
  return H % 256 == 0 && I % 256 == 0 && sm::smem_bytes(0, H, 1, 1) <= 227 * 1024 &&
         sm::smem_bytes(1, I, 1, 1) <= 227 * 1024;
}

cudaError_t launch_gemm_smallm(int mode, const GemmProblem& g, const SmallMaps& maps, DevErr err,
                               int num_sms, cudaStream_t st) {
  sm::Params p;
  p.mode = mode;
  p.T = g.T;
  p.k = g.k;
  p.E = g.E;
  p.K = g.K;
  p.N = g.N;
  p.ru = smallm_rows_per_unit(mode);
  p.nchunk = g.N / p.ru;
  p.has_shared = g.has_shared;
  p.bmap = g.bmap;
  p.num_tiles = g.num_tiles;
  p.act_in = g.act_in;
  p.gather_x = mode == 0 ? g.gather_x : nullptr;
  p.out = g.out;
  p.out_sh = g.out_sh;
  p.out_ld = g.out_ld;
  p.topk_w = g.topk_w;
  p.perm = g.perm;
  p.w0 = g.w0;
  p.w1 = g.w1;
  p.sw0 = g.sw0;
  p.sw1 = g.sw1;
  // prefetch shares: the down matrices have K (= H) rows per expert, split
  // evenly over the gate/up units of an expert (16-byte multiples only)
  p.next = p.snext = W4Dev{nullptr, nullptr, nullptr};
  p.next_K = g.next_K;
  p.next_rows = 0;
  if (mode == 0 && g.next.q && g.K % p.nchunk == 0) {
    const int rows = g.K / p.nchunk;
    if ((long long)rows * (g.next_K / 32) % 16 == 0) {
      p.next = g.next;
      p.snext = g.has_shared ? g.snext : W4Dev{nullptr, nullptr, nullptr};
      p.next_rows = rows;
    }
  }
  p.maps = maps;
  p.err = err;
  // persistent CTAs (one per SM: the kernel takes the whole register file)
  // walk the units; the host bound on the routed tiles only sizes the grid
  const int max_tiles = g.max_routed_tiles + (g.has_shared ? (g.T + kBM - 1) / kBM : 0);
  const long long units = (long long)max_tiles * p.nchunk;
  if (units < 1) return cudaSuccess;
  const int grid = (int)(units < num_sms ? units : num_sms);
  const int maxrows = g.T < kBM ? g.T : kBM;
  int nt = maxrows <= 8 ? 1 : maxrows <= 16 ? 2 : 4;
  while (nt > 1 && sm::smem_bytes(mode, p.K, nt, 1) > 227 * 1024) nt >>= 1;
  const int nbuf = sm::smem_bytes(mode, p.K, nt, 2) <= 227 * 1024 ? 2 : 1;
  const size_t smem = sm::smem_bytes(mode, p.K, nt, nbuf);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(sm::kThreads), smem, st, p);
  };
  cudaError_t e;
  if (nbuf == 2)
    e = nt == 1 ? launch(sm::w4_grouped_gemm_smallm<1, 2>)
        : nt == 2 ? launch(sm::w4_grouped_gemm_smallm<2, 2>) : launch(sm::w4_grouped_gemm_smallm<4, 2>);
  else
    e = nt == 1 ? launch(sm::w4_grouped_gemm_smallm<1, 1>)
        : nt == 2 ? launch(sm::w4_grouped_gemm_smallm<2, 1>) : launch(sm::w4_grouped_gemm_smallm<4, 1>);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
