// gemm_smallm.cu -- grouped W4A16 expert GEMM for decode-sized token groups.
//
// Same product as gemm_tc.cu (the grouped GEMM with block-wise dequant of
// "Perplexity libera Lily, un motor de IA que supera a MLX-LM en Apple
// Silicon", diariobitcoin.com, section "Las optimizaciones en el prefill"),
// for the regime of section "El decode busca mover menos datos": with a
// handful of tokens per expert the block is bound by streaming the packed
// weights once, so this kernel is written around HBM bandwidth, not MMA rate.
//
// Design:
//   * a unit is (block-map tile, chunk of weight rows); 4 warps; each warp
//     owns two 16-row m16n8k16 A tiles (gate and up rows for the gate/up
//     pass, two down row slabs for the down pass); the tile's tokens are the
//     n8 side, in passes of 8*NT tokens;
//   * the unit's whole weight slab (128 rows of packed words, scales and
//     biases) is copied into shared memory with cp.async at the start, all of
//     it in flight at once and overlapped with the token staging, so HBM sees
//     every CTA's bytes together (rows padded by 32 bytes so the fragment
//     reads are conflict-free); when the slab and the tokens do not fit in
//     shared memory, each thread streams its rows from global memory instead;
//   * each thread reads 8 bytes of packed weights per row per group, and
//     converts nibbles to fp16 "1024 + q" with
//     one LOP3 per pair (exact); the MMA sums (1024+q)*x over one group of 64
//     in FP32, and the group's affine map is applied to the 4 partial sums:
//         sum_k w_k x_k = s * sum_k (1024+q_k) x_k + (b - 1024 s) * sum_k x_k
//     which is exact algebra of w = q*s + b (the group sums of x are
//     precomputed in FP32 while the tokens are staged in shared memory);
//   * token rows (gathered activations, SwiGLU activations) are kept with
//     each 8-element block in the order (0,4,1,5,2,6,3,7), the order the
//     nibble extraction yields, so A and B fragments agree on which k each
//     MMA slot holds without any shuffle.
#include "moe_common.cuh"

namespace moe {
namespace sm {

constexpr int kWarps = 4;
constexpr int kPF = 4;   // groups prefetched (= one 8-byte scale/bias batch)

struct Params {
  int mode;              // 0 gate/up + SwiGLU, 1 down * weight
  int T, k, E, K, N;
  int nchunk;            // units per tile
  int rows_per_unit;     // 64 (gate/up: per matrix) or 128 (down)
  int has_shared;
  const int32_t* bmap;
  const int32_t* num_tiles;
  const uint16_t* act_in;
  const uint16_t* gather_x;   // gate/up: bf16 token rows read through perm (no gathered copy)
  uint16_t* out;
  float* out_sh;
  int out_ld;
  const float* topk_w;
  const int32_t* perm;
  W4Dev w0, w1, sw0, sw1;
};

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

// Shared-memory slab of a unit: 128 weight rows (gate rows then up rows, or
// 128 down rows) of K/8 words plus 8 words of padding, then the rows' scales
// and biases. Bytes for reduction size K.
__host__ __device__ __forceinline__ size_t slab_bytes(int K) {
  return (size_t)128 * (K / 8 + 8) * 4 + (size_t)2 * 128 * (K / 64) * 2;
}

template <int NT, bool STAGE>
__global__ void __launch_bounds__(kWarps * 32) w4_grouped_gemm_smallm(const Params p) {
  // The down pass follows the gate/up pass, which writes neither the block
  // map nor any weight: it finds its tile and starts its weight slab copy
  // before waiting for that launch. The gate/up pass follows the routing and
  // waits first.
  const bool early = p.mode == 1;
  if (!early) pdl_begin();
  extern __shared__ __align__(16) uint8_t smem[];
  const int K = p.K;
  const int G = K / 64;                           // groups
  const int xstride = K / 2 + 1;                  // words per staged token row
  uint32_t* xw = reinterpret_cast<uint32_t*>(smem);            // [8*NT][xstride]
  float* xg = reinterpret_cast<float*>(xw + 8 * NT * xstride);  // [8*NT][G]
  const int wstride = K / 8 + 8;                  // words per slab row
  uint32_t* slab = reinterpret_cast<uint32_t*>(xg + 8 * NT * G);  // [128][wstride]
  uint16_t* slab_s = reinterpret_cast<uint16_t*>(slab + 128 * wstride);  // [128][G]
  uint16_t* slab_b = slab_s + 128 * G;                                   // [128][G]

  const int n_routed = __ldcg(p.num_tiles);
  const int n_shared = p.has_shared ? (p.T + kBM - 1) / kBM : 0;
  const int u = blockIdx.x;
  if (u >= (n_routed + n_shared) * p.nchunk) return;
  const int tile = u / p.nchunk, ch = u - tile * p.nchunk;
  int e, m0, rows;
  bool shared;
  if (tile < n_routed) {
    e = __ldcg(p.bmap + 3 * tile);
    m0 = __ldcg(p.bmap + 3 * tile + 1);
    rows = __ldcg(p.bmap + 3 * tile + 2);
    shared = false;
  } else {
    const int i = tile - n_routed;
    e = 0;
    m0 = p.T * p.k + kBM * i;
    rows = min(kBM, p.T - kBM * i);
    shared = true;
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;

  // weight rows of this thread: A tile mt, half h (row g or g+8)
  const W4Dev wa = shared ? p.sw0 : p.w0;
  const W4Dev wb = shared ? p.sw1 : p.w1;
  const size_t ebase = shared ? 0 : (size_t)e * p.N;
  int nrow[2][2];
  const W4Dev* wm[2];
  if (p.mode == 0) {
    const int n0 = p.rows_per_unit * ch + 16 * warp;
    wm[0] = &wa;
    wm[1] = &wb;
    nrow[0][0] = n0 + g;
    nrow[0][1] = n0 + g + 8;
    nrow[1][0] = n0 + g;
    nrow[1][1] = n0 + g + 8;
  } else {
    const int n0 = p.rows_per_unit * ch + 32 * warp;
    wm[0] = &wa;
    wm[1] = &wa;
    nrow[0][0] = n0 + g;
    nrow[0][1] = n0 + g + 8;
    nrow[1][0] = n0 + 16 + g;
    nrow[1][1] = n0 + 16 + g + 8;
  }
  // slab row of (A tile mt, half h): gate rows 0..63 then up rows 64..127,
  // or the 128 down rows in order
  const int n0base = p.rows_per_unit * ch;
  auto slab_row = [&](int mt, int h) {
    return p.mode == 0 ? 64 * mt + (nrow[mt][h] - n0base) : nrow[mt][h] - n0base;
  };
  if (STAGE) {
    // the whole slab in flight at once (16-byte cp.async, L2 only)
    const int cpr = K / 32;                                 // 16-byte pieces per row
    for (int idx = threadIdx.x; idx < 128 * cpr; idx += blockDim.x) {
      const int r = idx / cpr, pc = idx - r * cpr;
      const W4Dev& w = (p.mode == 0 && r >= 64) ? wb : wa;
      const int grow = n0base + (p.mode == 0 ? (r & 63) : r);
      cp_async16(slab + r * wstride + 4 * pc, w.q + (ebase + grow) * (size_t)(K / 8) + 4 * pc);
    }
    const int cps = G / 8;                                  // pieces of one row's scales
    for (int idx = threadIdx.x; idx < 2 * 128 * cps; idx += blockDim.x) {
      const int which = idx / (128 * cps), rem = idx - which * 128 * cps;
      const int r = rem / cps, pc = rem - r * cps;
      const W4Dev& w = (p.mode == 0 && r >= 64) ? wb : wa;
      const int grow = n0base + (p.mode == 0 ? (r & 63) : r);
      const uint16_t* src = (which ? w.b : w.s) + (ebase + grow) * (size_t)G + 8 * pc;
      cp_async16((which ? slab_b : slab_s) + r * G + 8 * pc, src);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  }
  const uint2* qp[2][2];
  const uint2* sp[2][2];
  const uint2* bp[2][2];
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const size_t row = ebase + nrow[mt][h];
      if (STAGE) {
        const int r = slab_row(mt, h);
        qp[mt][h] = reinterpret_cast<const uint2*>(slab + r * wstride) + c;
        sp[mt][h] = reinterpret_cast<const uint2*>(slab_s + r * G);
        bp[mt][h] = reinterpret_cast<const uint2*>(slab_b + r * G);
      } else {
        qp[mt][h] = reinterpret_cast<const uint2*>(wm[mt]->q + row * (K / 8)) + c;
        sp[mt][h] = reinterpret_cast<const uint2*>(wm[mt]->s + row * G);
        bp[mt][h] = reinterpret_cast<const uint2*>(wm[mt]->b + row * G);
      }
    }
  if (early) pdl_begin();
  // global weights through the read-only path; the slab with plain loads
  auto ld = [](const uint2* ptr) { return STAGE ? *ptr : __ldg(ptr); };

  for (int pass0 = 0; pass0 < rows; pass0 += 8 * NT) {
    const int prow = min(8 * NT, rows - pass0);
    __syncthreads();
    // stage tokens: rows arrive in perm8 order, so word (4*w8 + i) of a row
    // already holds (x[8*w8 + i], x[8*w8 + i + 4])
    for (int idx = threadIdx.x; idx < 8 * NT * G; idx += blockDim.x) {
      const int tr = idx / G, grp = idx - tr * G;
      float sum = 0.f;
      uint32_t* dst = xw + tr * xstride + grp * 32;
      if (tr < prow) {
        const int pos = m0 + pass0 + tr;
        const uint16_t* row;
        if (p.gather_x) {
          const int src = pos < p.T * p.k ? __ldg(p.perm + pos) / p.k : pos - p.T * p.k;
          row = p.gather_x + (size_t)src * K;
        } else {
          row = p.act_in + (size_t)pos * K;
        }
        const uint4* src = reinterpret_cast<const uint4*>(row + grp * 64);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint4 x8 = __ldg(src + v);
          if (p.gather_x)   // bf16 token values -> the fp16 perm8 operand of a gathered row
            x8 = f16x8_to_perm8(make_uint4(bf16x2_to_f16x2_sat(x8.x), bf16x2_to_f16x2_sat(x8.y),
                                           bf16x2_to_f16x2_sat(x8.z), bf16x2_to_f16x2_sat(x8.w)));
          dst[4 * v + 0] = x8.x;   // (x0, x4)
          dst[4 * v + 1] = x8.y;   // (x1, x5)
          dst[4 * v + 2] = x8.z;   // (x2, x6)
          dst[4 * v + 3] = x8.w;   // (x3, x7)
          sum += f16_lo(x8.x) + f16_hi(x8.x) + f16_lo(x8.y) + f16_hi(x8.y) +
                 f16_lo(x8.z) + f16_hi(x8.z) + f16_lo(x8.w) + f16_hi(x8.w);
        }
      } else {
#pragma unroll
        for (int v = 0; v < 32; ++v) dst[v] = 0u;
      }
      xg[tr * G + grp] = sum;
    }
    if (STAGE && pass0 == 0) asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();

    float tot[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) tot[mt][nt][i] = 0.f;

    uint2 qr[kPF][2][2];
#pragma unroll
    for (int i = 0; i < kPF; ++i)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) qr[i][mt][h] = ld(qp[mt][h] + 4 * i);
    uint2 sr[2][2], br[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        sr[mt][h] = ld(sp[mt][h]);
        br[mt][h] = ld(bp[mt][h]);
      }

    for (int g0 = 0; g0 < G; g0 += kPF) {
      uint2 srn[2][2], brn[2][2];
      const bool more = g0 + kPF < G;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          srn[mt][h] = more ? ld(sp[mt][h] + (g0 + kPF) / 4) : sr[mt][h];
          brn[mt][h] = more ? ld(bp[mt][h] + (g0 + kPF) / 4) : br[mt][h];
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
            for (int h = 0; h < 2; ++h) qr[i][mt][h] = ld(qp[mt][h] + 4 * (grp + kPF));
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

    // epilogue
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int tok = nt * 8 + 2 * c + (q & 1);
        if (tok >= prow) continue;
        const int pos = m0 + pass0 + tok;
        const int h = q >> 1;
        if (p.mode == 0) {
          const float a = silu_fast(tot[0][nt][q]) * tot[1][nt][q];
          p.out[(size_t)pos * p.out_ld + perm8_pos(nrow[0][h])] = f32_to_f16_sat(a);
        } else if (shared) {
          float* o = p.out_sh + (size_t)(pos - p.T * p.k) * p.out_ld;
          o[nrow[0][h]] = tot[0][nt][q];
          o[nrow[1][h]] = tot[1][nt][q];
        } else {
          const float wt = __ldg(p.topk_w + __ldg(p.perm + pos));
          p.out[(size_t)pos * p.out_ld + nrow[0][h]] = f32_to_bf16(tot[0][nt][q] * wt);
          p.out[(size_t)pos * p.out_ld + nrow[1][h]] = f32_to_bf16(tot[1][nt][q] * wt);
        }
      }
  }
}

}  // namespace sm

cudaError_t launch_gemm_smallm(int mode, const GemmProblem& g, cudaStream_t st) {
  sm::Params p;
  p.mode = mode;
  p.T = g.T;
  p.k = g.k;
  p.E = g.E;
  p.K = g.K;
  p.N = g.N;
  p.rows_per_unit = mode == 0 ? 64 : 128;
  p.nchunk = g.N / p.rows_per_unit;
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
  const int max_tiles = g.max_routed_tiles + (g.has_shared ? (g.T + kBM - 1) / kBM : 0);
  const int grid = max_tiles * p.nchunk;
  if (grid < 1) return cudaSuccess;
  const int maxrows = g.T < kBM ? g.T : kBM;
  const int G = p.K / 64;
  const int nt = maxrows <= 8 ? 1 : maxrows <= 16 ? 2 : 4;
  const size_t base = (size_t)8 * nt * (p.K / 2 + 1) * 4 + (size_t)8 * nt * G * 4;
  const size_t staged = base + sm::slab_bytes(p.K);
  // staging copies scales in 16-byte pieces (8 groups): K a multiple of 512
  const bool stage = staged <= 227 * 1024 && p.K % 512 == 0;
  const size_t smem = stage ? staged : base;
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(sm::kWarps * 32), smem, st, p);
  };
  cudaError_t e;
  if (nt == 1)
    e = stage ? launch(sm::w4_grouped_gemm_smallm<1, true>) : launch(sm::w4_grouped_gemm_smallm<1, false>);
  else if (nt == 2)
    e = stage ? launch(sm::w4_grouped_gemm_smallm<2, true>) : launch(sm::w4_grouped_gemm_smallm<2, false>);
  else
    e = stage ? launch(sm::w4_grouped_gemm_smallm<4, true>) : launch(sm::w4_grouped_gemm_smallm<4, false>);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace moe
