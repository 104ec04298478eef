// route_kernels.cu -- GPU-resident routing of the MoE block and the small
// elementwise kernels around the grouped GEMMs.
//
// Routing follows "Perplexity libera Lily, un motor de IA que supera a MLX-LM
// en Apple Silicon" (diariobitcoin.com): section "Qwen3.6 combina tres cargas
// de trabajo" (router scores 256 experts, picks 8) and section "Las
// optimizaciones en el prefill" (histogram, prefix scan, scatter and block
// map kept on the GPU with no CPU synchronisation). Every step here is
// deterministic: counts are per token block, ranks inside an expert follow
// token order, and no result depends on atomic ordering.
#include <cuda_pipeline.h>

#include <mutex>

#include "moe_common.cuh"
#include "topk.cuh"

namespace moe {

// ------------------------------------------------------------ tensor maps ---
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

// 2D row-major tensor map: `rows` x `cols` elements, box `box_cols` x `box_rows`,
// 128-byte swizzle (box_cols * elem == 128).
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base,
               uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * (uint64_t)elem_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_router_slices(CUtensorMap* m, const void* base, int H, int E) {
  EncodeTiledFn enc = get_encode();
  if (!enc || H % 256 || E % 8) return false;
  cuuint64_t dims[2] = {(cuuint64_t)E, (cuuint64_t)H};
  cuuint64_t strides[1] = {(cuuint64_t)E * 2};
  cuuint32_t box[2] = {8, 256};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_slab_3d(CUtensorMap* m, const void* base, uint64_t rows, int K, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode();
  if (!enc || K % 256) return false;
  cuuint64_t dims[3] = {32, rows, (cuuint64_t)(K / 256)};
  cuuint64_t strides[2] = {(cuuint64_t)K / 2, 128};   // row, 128-byte chunk
  cuuint32_t box[3] = {32, box_rows, (cuuint32_t)(K / 256)};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box,
                   es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Router logits: logits[t][e] = sum_h x[t][h] * Wr[h][e] + bias[e], bf16
// inputs, FP32 accumulation on mma.sync m16n8k16. One CTA computes a 64-token
// x 128-expert tile: 8 warps of 32 tokens x 32 experts each (4 ldmatrix feed
// 8 MMAs per 16-wide K step), with a 4-stage cp.async pipeline over K in
// chunks of 64.
// ---------------------------------------------------------------------------
constexpr int kLgT = 64, kLgE = 128, kLgK = 64, kLgStages = 4;
constexpr int kLgXStride = kLgK + 8, kLgWStride = kLgE + 8;   // padded rows (bank spread)
constexpr int kLgXStage = kLgT * kLgXStride, kLgWStage = kLgK * kLgWStride;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(256) router_logits_kernel(
    const uint16_t* __restrict__ x, int T, int H, const uint16_t* __restrict__ wr,
    const float* __restrict__ bias, int E, float* __restrict__ logits) {
  pdl_begin();
  extern __shared__ __align__(128) uint8_t smem[];
  uint16_t* xs_s = reinterpret_cast<uint16_t*>(smem);              // [stage][64 t][72]
  uint16_t* wr_s = xs_s + kLgStages * kLgXStage;                    // [stage][64 k][136]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kLgT, e0 = blockIdx.y * kLgE;
  const int wm = warp & 1, wn = warp >> 1;   // 2 x 4 warps: 32 tokens x 32 experts each

  auto stage = [&](int buf, int kc) {
    const int k0 = kc * kLgK;
#pragma unroll
    for (int i = 0; i < 2; ++i) {   // x: 64 rows x 8 pieces of 16 B
      const int c = tid + 256 * i;
      const int r = c >> 3, col = (c & 7) * 8;
      const int t = t0 + r;
      cp_async16(xs_s + buf * kLgXStage + r * kLgXStride + col,
                 x + (size_t)(t < T ? t : 0) * H + k0 + col, t < T ? 16 : 0);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {   // Wr: 64 k-rows x 16 pieces of 16 B
      const int c = tid + 256 * i;
      const int r = c >> 4, col = (c & 15) * 8;
      const int e = e0 + col;
      cp_async16(wr_s + buf * kLgWStage + r * kLgWStride + col,
                 wr + (size_t)(k0 + r) * E + (e < E ? e : 0), e < E ? 16 : 0);
    }
    cp_async_commit();
  };

  float acc[2][4][4];
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][n][i] = 0.f;

  const int nk = H / kLgK;
#pragma unroll
  for (int s = 0; s < kLgStages - 1; ++s)
    if (s < nk) stage(s, s);
    else cp_async_commit();
  for (int kc = 0; kc < nk; ++kc) {
    cp_async_wait<kLgStages - 2>();
    __syncthreads();
    if (kc + kLgStages - 1 < nk) stage((kc + kLgStages - 1) % kLgStages, kc + kLgStages - 1);
    else cp_async_commit();
    const uint16_t* xb = xs_s + (kc % kLgStages) * kLgXStage;
    const uint16_t* wb = wr_s + (kc % kLgStages) * kLgWStage;
#pragma unroll
    for (int ks = 0; ks < kLgK / 16; ++ks) {
      uint32_t a[2][4], b[4][2];
#pragma unroll
      for (int m = 0; m < 2; ++m)
        ldsm_x4(smem_u32(xb + (wm * 32 + m * 16 + (lane & 15)) * kLgXStride + ks * 16 + (lane >> 4) * 8),
                a[m][0], a[m][1], a[m][2], a[m][3]);
#pragma unroll
      for (int np = 0; np < 2; ++np)
        ldsm_x4_t(smem_u32(wb + (ks * 16 + (lane & 15)) * kLgWStride + wn * 32 + np * 16 + (lane >> 4) * 8),
                  b[2 * np][0], b[2 * np][1], b[2 * np + 1][0], b[2 * np + 1][1]);
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int n = 0; n < 4; ++n)
          mma_16816(acc[m][n], a[m][0], a[m][1], a[m][2], a[m][3], b[n][0], b[n][1]);
    }
  }
  cp_async_wait<0>();
  const int g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    const int e = e0 + wn * 32 + n * 8 + 2 * c;
    if (e >= E) continue;
    const float b0 = bias ? bias[e] : 0.f, b1 = bias ? bias[e + 1] : 0.f;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int t = t0 + wm * 32 + m * 16 + g + 8 * h;
        if (t < T)
          *reinterpret_cast<float2*>(logits + (size_t)t * E + e) =
              make_float2(acc[m][n][2 * h] + b0, acc[m][n][2 * h + 1] + b1);
      }
  }
}

// ---------------------------------------------------------------------------
// Top-k + per-block histogram. One CTA = 32 tokens, one warp per token.
// Each of the k rounds takes the largest not-yet-selected logit (a lower
// expert index first on ties; a NaN logit ranks as -inf; -0 counts as +0),
// with the warp's choice made by two redux.sync reductions over an
// order-preserving integer key: the maximum key, then the lowest expert index
// holding it. Every round selects some expert not selected before, so the
// indices are always valid and distinct. Weights: softmax over the selected
// logits (equal to softmax over all E renormalised over the k). The block
// writes its per-expert counts to blk_cnt[block][E].
// ---------------------------------------------------------------------------
template <int VPL>
__global__ void __launch_bounds__(1024) router_topk_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, int32_t* __restrict__ blk_cnt) {
  pdl_begin();
  __shared__ int cnt_s[1024];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = blockIdx.x * kRouterTB;
  for (int i = tid; i < E; i += blockDim.x) cnt_s[i] = 0;
  __syncthreads();
  if (t0 + warp < T) {
    const int t = t0 + warp;
    int idx;
    float w;
    topk_warp<VPL>(logits + (size_t)t * E, E, k, idx, w);
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = idx;
      topk_w[(size_t)t * k + lane] = w;
      atomicAdd(&cnt_s[idx], 1);
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) blk_cnt[(size_t)blockIdx.x * E + e] = cnt_s[e];
}

// Router logits for decode-sized batches (T <= 16) on mma.sync: each of the
// E/16 CTAs multiplies the (padded) 16 x H token block by its 16 experts'
// H x 16 weight columns. The weight columns are copied into shared memory
// (two arrays of 8 experts, 16 bytes per k) before waiting for the previous
// launch, since no launch writes the weights; the tokens after it. Warp w
// takes the K steps [w H/8, (w+1) H/8): B fragments by ldmatrix.trans, FP32
// accumulation, and the 8 warps' partial sums are added in a fixed order:
// deterministic. Rows of the token block past T are never read back (a
// product row depends on its own token row only).
constexpr int kRsMaxT = 16;

__host__ __device__ constexpr size_t rs_smem_bytes(int H) {
  return (size_t)kRsMaxT * (H + 8) * 2 + (size_t)2 * H * 16 + (size_t)8 * 16 * 16 * 4;
}

__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}

// The CTA's weight columns: ws[a][k][0..7] = Wr[k][16 blockIdx + 8 a + 0..7].
__device__ __forceinline__ void rs_load_w(const uint16_t* __restrict__ wr, int H, int E,
                                          uint8_t* smem) {
  uint16_t* ws = reinterpret_cast<uint16_t*>(smem + (size_t)kRsMaxT * (H + 8) * 2);
  const int e0 = blockIdx.x * 16;
  for (int i = threadIdx.x; i < 2 * H; i += blockDim.x) {
    const int a = i & 1, k = i >> 1;
    uint16_t* dst = ws + ((size_t)a * H + k) * 8;
    if (e0 + 8 * a < E)
      cp_async_16(dst, wr + (size_t)k * E + e0 + 8 * a);
    else
      *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Logits of this CTA's 16 experts for all T tokens.
__device__ __forceinline__ void rs_logits(const uint16_t* __restrict__ x, int T, int H,
                                          const float* __restrict__ bias, int E,
                                          float* __restrict__ logits, uint8_t* smem) {
  const int xstr = H + 8;                                           // padded token row
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                 // [16][H + 8]
  const uint16_t* ws = xs + (size_t)kRsMaxT * xstr;                 // [2][H][8]
  float* red = reinterpret_cast<float*>(smem + (size_t)kRsMaxT * xstr * 2 + (size_t)2 * H * 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int vpr = H / 8;                                            // 16-byte pieces per row
  for (int i = tid; i < T * vpr; i += blockDim.x) {
    const int t = i / vpr, c = i - t * vpr;
    cp_async_16(xs + (size_t)t * xstr + 8 * c, x + (size_t)t * H + 8 * c);
  }
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
  __syncthreads();
  float d[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  const int steps = H / 128;                                        // K steps of 16 per warp
  const uint32_t a_base = smem_u32(xs + (size_t)(lane & 15) * xstr + 8 * (lane >> 4));
  const uint32_t b_base = smem_u32(ws + ((size_t)(lane >> 4) * H + (lane & 15)) * 8);
  for (int st = 0; st < steps; ++st) {
    const int k0 = (warp * steps + st) * 16;
    uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
    ldsm_x4(a_base + 2 * k0, a0, a1, a2, a3);
    ldsm_x4_t(b_base + 16 * k0, b0, b1, b2, b3);
    mma_16816(d[0], a0, a1, a2, a3, b0, b1);
    mma_16816(d[1], a0, a1, a2, a3, b2, b3);
  }
  // red[warp][token][expert]
  const int g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    float* r = red + (size_t)warp * 256 + nt * 8 + 2 * c;
    r[g * 16] = d[nt][0];
    r[g * 16 + 1] = d[nt][1];
    r[(g + 8) * 16] = d[nt][2];
    r[(g + 8) * 16 + 1] = d[nt][3];
  }
  __syncthreads();
  const int t = tid >> 4, el = tid & 15, ee = blockIdx.x * 16 + el;
  if (t < T && ee < E) {
    float sum = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < 8; ++w8) sum += red[w8 * 256 + t * 16 + el];
    logits[(size_t)t * E + ee] = sum + (bias ? bias[ee] : 0.f);
  }
}

// kEarlyW: copy the weight columns before waiting for the previous launch
// (the library's own launch sequences, where no launch writes the weights);
// otherwise after it (a caller's kernel just before may write them).
template <bool kEarlyW>
__global__ void __launch_bounds__(256) router_logits_small_kernel(
    const uint16_t* __restrict__ x, int T, int H, const uint16_t* __restrict__ wr,
    const float* __restrict__ bias, int E, float* __restrict__ logits) {
  extern __shared__ __align__(128) uint8_t smem[];
  if (kEarlyW) rs_load_w(wr, H, E, smem);
  pdl_begin();
  if (!kEarlyW) rs_load_w(wr, H, E, smem);
  rs_logits(x, T, H, bias, E, logits, smem);
}

// ---------------------------------------------------------------------------
// Router logits for prefill-sized batches on the tensor cores (tcgen05).
// logits = x Wr + bias is a plain GEMM whose K (the hidden size) is long next
// to both T and E, so it belongs on tcgen05 rather than mma.sync, whose rate
// it otherwise runs at. A CTA computes a 128-token x 64-expert tile: TMA
// brings 64-wide K chunks of x (K-major) and of the router weight in its own
// [H][E] layout (64 hidden rows x 64 experts, read by the MMA as an N-major
// operand), 128-byte swizzle, 6 stages; one thread issues M=128 N=64 K=16
// MMAs (bf16 in, FP32 accumulation in tensor memory), and four warps add the
// bias and store the rows. Every wait is bounded: on timeout the error is
// latched and the CTA stops issuing and exits once its own work is done.
// ---------------------------------------------------------------------------
constexpr int kRtM = 128, kRtN = 64, kRtStages = 6;
constexpr int kRtABytes = kRtM * 128, kRtBBytes = kRtN * 128;   // 64 bf16 of K per row
constexpr size_t kRtSmem = (size_t)kRtStages * (kRtABytes + kRtBBytes) + 1024;

struct RtParams {
  CUtensorMap ma;        // x, bf16 [T][H], box 64 x 128 rows
  CUtensorMap mb;        // router weight, bf16 [H][E], box 64 experts x 64 rows
  int T, H, E;
  const float* bias;
  float* logits;
  DevErr err;
};

// kind::f16 instruction descriptor: D fp32, A and B bf16, A K-major, B
// N-major (bit 16): B is read from the router weight's own [H][E] layout.
__host__ __device__ constexpr uint32_t idesc_bf16_f32_bn(int M, int N) {
  return (1u << 4)                                 // D format: f32
         | (1u << 7)                               // A format: bf16
         | (1u << 10)                              // B format: bf16
         | (1u << 16)                              // B N-major
         | (static_cast<uint32_t>(N >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);  // M / 16
}

// Shared-memory descriptor of an N-major tile with 128-byte swizzle: rows are
// K (64 N elements = 128 bytes each), 8-row groups 1024 bytes apart; one
// 64-wide N block per tile.
__device__ __forceinline__ uint64_t smem_desc_sw128_mn(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);        // start address
  d |= static_cast<uint64_t>(8192u >> 4) << 16;                   // LBO: next N block (none)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;                   // SBO: 8 K-rows * 128 B
  d |= static_cast<uint64_t>(1u) << 46;                           // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                           // 128-byte swizzle
  return d;
}

// D[tmem] (+)= A[smem desc] * B[smem desc]; kind::f16.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(128) router_logits_tc_kernel(const __grid_constant__ RtParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + kRtStages * kRtABytes;
  __shared__ __align__(8) uint64_t full[kRtStages], empty[kRtStages], acc_full;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 64);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    for (int i = 0; i < kRtStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(&acc_full, 1);
    fence_mbar_init();
    tma_prefetch_desc(&p.ma);
    tma_prefetch_desc(&p.mb);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  pdl_begin();   // x comes from the previous launch

  const int m0 = blockIdx.x * kRtM, n0 = blockIdx.y * kRtN;
  const int nk = p.H / 64;
  const unsigned long long lim = p.err.limit_ns;
  if (warp == 0) {
    // TMA producer
    for (int c = 0; c < nk; ++c) {
      const int s = c % kRtStages;
      if (c >= kRtStages && !mbar_wait_drain(&empty[s], ((c / kRtStages) & 1) ^ 1, lim)) {
        if (lane == 0) report_timeout(p.err, 40);
        break;
      }
      if (elect_one_sync()) {
        mbar_arrive_expect_tx(&full[s], kRtABytes + kRtBBytes);
        tma_load_2d(sa + s * kRtABytes, &p.ma, 64 * c, m0, &full[s]);
        tma_load_2d(sb + s * kRtBBytes, &p.mb, n0, 64 * c, &full[s]);
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // MMA issuer
    const uint32_t idesc = idesc_bf16_f32_bn(kRtM, kRtN);
    bool ok = true;
    for (int c = 0; c < nk; ++c) {
      const int s = c % kRtStages;
      if (!mbar_wait_drain(&full[s], (c / kRtStages) & 1, lim)) {
        if (lane == 0) report_timeout(p.err, 41);
        ok = false;
        break;
      }
      tc_fence_after();
      if (elect_one_sync()) {
        const uint32_t abase = smem_u32(sa + s * kRtABytes), bbase = smem_u32(sb + s * kRtBBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16_ss(tmem, smem_desc_sw128(abase + 32 * kk), smem_desc_sw128_mn(bbase + 2048 * kk),
                     idesc, (c | kk) != 0);
        mma_commit(&empty[s]);
      }
      __syncwarp();
    }
    if (ok && elect_one_sync()) mma_commit(&acc_full);
    __syncwarp();
  }
  // epilogue: thread = token row of the tile, 64 experts
  const bool have = mbar_wait_drain(&acc_full, 0, lim);
  if (!have && lane == 0) report_timeout(p.err, 42);
  tc_fence_after();
  uint32_t v0[32], v1[32];
  const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
  tmem_ld_32x32b_x32(taddr, v0);
  tmem_ld_32x32b_x32(taddr + 32, v1);
  tmem_wait_ld();
  const int t = m0 + 32 * warp + lane;
  if (have && t < p.T) {
    float4* o = reinterpret_cast<float4*>(p.logits + (size_t)t * p.E + n0);
    const float4* bb = reinterpret_cast<const float4*>(p.bias + n0);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint32_t* v = j < 8 ? v0 : v1;
      const int q = 4 * (j & 7);
      float4 r = make_float4(__uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                             __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
      if (p.bias) {
        const float4 b4 = __ldg(bb + j);
        r.x += b4.x;
        r.y += b4.y;
        r.z += b4.z;
        r.w += b4.w;
      }
      o[j] = r;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

bool router_tc_fits(int T, int H, int E) {
  return T > kRsMaxT && H % 64 == 0 && H <= 16384 && E % 64 == 0 && E <= 1024;
}

cudaError_t launch_router_logits_tc(const uint16_t* x, int T, int H, const uint16_t* wr,
                                    const float* bias, int E, float* logits, DevErr err,
                                    cudaStream_t st) {
  RtParams p;
  if (!encode_2d(&p.ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, x, T, H, 64, kRtM) ||
      !encode_2d(&p.mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, wr, H, E, 64, 64))
    return cudaErrorInvalidValue;
  p.T = T;
  p.H = H;
  p.E = E;
  p.bias = bias;
  p.logits = logits;
  p.err = err;
  cudaError_t e = cudaFuncSetAttribute(router_logits_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRtSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(router_logits_tc_kernel, dim3((T + kRtM - 1) / kRtM, E / kRtN), dim3(128),
                    kRtSmem, st, p);
}

cudaError_t launch_router_logits(const uint16_t* x, int T, int H, const uint16_t* wr,
                                 const float* bias, int E, float* logits, DevErr err,
                                 cudaStream_t st, bool weights_early) {
  if (!logits) return cudaErrorInvalidValue;
  // (the tensor-core epilogue moves logits and bias in 16-byte pieces)
  const bool al16 = ((reinterpret_cast<uintptr_t>(logits) | reinterpret_cast<uintptr_t>(bias)) & 15u) == 0;
  if (al16 && router_tc_fits(T, H, E))
    return launch_router_logits_tc(x, T, H, wr, bias, E, logits, err, st);
  if (T <= kRsMaxT && H % 128 == 0 && rs_smem_bytes(H) <= 227 * 1024) {
    const size_t smem = rs_smem_bytes(H);
    auto launch = [&](auto kern) -> cudaError_t {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      return launch_pdl(kern, dim3((E + 15) / 16), dim3(256), smem, st, x, T, H, wr, bias, E, logits);
    };
    return weights_early ? launch(router_logits_small_kernel<true>)
                         : launch(router_logits_small_kernel<false>);
  }
  const size_t smem = (size_t)kLgStages * (kLgXStage + kLgWStage) * 2;
  cudaError_t e = cudaFuncSetAttribute(router_logits_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((T + kLgT - 1) / kLgT, (E + kLgE - 1) / kLgE);
  return launch_pdl(router_logits_kernel, grid, dim3(256), smem, st, x, T, H, wr, bias, E, logits);
}

cudaError_t launch_router_select(const float* logits, int T, int E, int k, int32_t* topk_idx,
                                 float* topk_w, int32_t* blk_cnt, cudaStream_t st) {
  const int nblk = (T + kRouterTB - 1) / kRouterTB;
  if (E <= 256)
    return launch_pdl(router_topk_kernel<8>, dim3(nblk), dim3(32 * kRouterTB), 0, st, logits, T, E,
                      k, topk_idx, topk_w, blk_cnt);
  return launch_pdl(router_topk_kernel<16>, dim3(nblk), dim3(32 * kRouterTB), 0, st, logits, T, E,
                    k, topk_idx, topk_w, blk_cnt);
}

cudaError_t launch_router_topk(const uint16_t* x, int T, int H, const uint16_t* wr,
                               const float* bias, int E, int k, int32_t* topk_idx,
                               float* topk_w, float* logits, int32_t* blk_cnt, DevErr err,
                               cudaStream_t st, bool weights_early) {
  cudaError_t e = launch_router_logits(x, T, H, wr, bias, E, logits, err, st, weights_early);
  if (e != cudaSuccess) return e;
  return launch_router_select(logits, T, E, k, topk_idx, topk_w, blk_cnt, st);
}

// ---------------------------------------------------------------------------
// Prefix scans and block map (one CTA, one thread per expert).
//   blk_cnt[b][e] -> exclusive offset of block b inside expert e's segment
//   cnt[e], off[e] = sum_{e'<e} cnt[e'], tile_off[e] = sum_{e'<e} ceil(cnt/BM)
//   bmap[tile] = (e, off[e] + BM*i, min(BM, cnt[e] - BM*i))
// ---------------------------------------------------------------------------
__device__ __forceinline__ int block_excl_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += n;
  }
  if (lane == 31) warp_sums[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int ws = lane < nw ? warp_sums[lane] : 0;
    int wi = ws;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < nw) warp_sums[lane] = wi - ws;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  int r = inc - v + warp_sums[warp];
  __syncthreads();
  return r;
}

__global__ void route_scan_kernel(int32_t* __restrict__ blk_cnt, int nblk, int T, int k, int E,
                                  int32_t* __restrict__ cnt, int32_t* __restrict__ off,
                                  int32_t* __restrict__ tile_off, int32_t* __restrict__ bmap,
                                  int32_t* __restrict__ num_tiles) {
  pdl_begin();
  __shared__ int warp_sums[32];
  __shared__ int tot_rows, tot_tiles;
  const int e = threadIdx.x;
  const bool valid = e < E;
  // pass 1: expert totals (independent loads, 16 in flight)
  int total = 0;
  if (valid) {
    int b = 0;
    for (; b + 16 <= nblk; b += 16) {
      int c[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) c[i] = blk_cnt[(size_t)(b + i) * E + e];
#pragma unroll
      for (int i = 0; i < 16; ++i) total += c[i];
    }
    for (; b < nblk; ++b) total += blk_cnt[(size_t)b * E + e];
  }
  const int tiles = valid ? (total + kBM - 1) / kBM : 0;
  const int o = block_excl_scan(valid ? total : 0, warp_sums, &tot_rows);
  const int to = block_excl_scan(tiles, warp_sums, &tot_tiles);
  if (valid) {
    cnt[e] = total;
    off[e] = o;
    tile_off[e] = to;
    // pass 2: blk_cnt[b][e] <- offset of block b's first slot of expert e
    int run = o, b = 0;
    for (; b + 16 <= nblk; b += 16) {
      int c[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) c[i] = blk_cnt[(size_t)(b + i) * E + e];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        blk_cnt[(size_t)(b + i) * E + e] = run;
        run += c[i];
      }
    }
    for (; b < nblk; ++b) {
      const int c = blk_cnt[(size_t)b * E + e];
      blk_cnt[(size_t)b * E + e] = run;
      run += c;
    }
    for (int i = 0; i < tiles; ++i) {
      int rows = total - kBM * i;
      int32_t* m = bmap + 3 * (size_t)(to + i);
      m[0] = e;
      m[1] = o + kBM * i;
      m[2] = rows < kBM ? rows : kBM;
    }
  }
  if (threadIdx.x == 0) {
    off[E] = tot_rows;
    tile_off[E] = tot_tiles;
    num_tiles[0] = tot_tiles;
  }
}

cudaError_t launch_route_scan(int32_t* blk_cnt, int nblk, int T, int k, int E, int32_t* cnt,
                              int32_t* off, int32_t* tile_off, int32_t* bmap, int32_t* num_tiles,
                              cudaStream_t st) {
  int threads = ((E + 31) / 32) * 32;
  return launch_pdl(route_scan_kernel, dim3(1), dim3(threads), 0, st, blk_cnt, nblk, T, k, E, cnt, off, tile_off, bmap, num_tiles);
}

// ---------------------------------------------------------------------------
// Stable scatter: slot s = t*k + j of block b goes to
//   pos = blk_off[b][e] + #{t' < t in block b : token t' selected e}
// A token's k experts are distinct, so the count is the popcount of the
// block's per-expert token mask below bit t (blocks hold at most 32 tokens).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) route_scatter_kernel(
    const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ blk_off, int T, int k,
    int E, int32_t* __restrict__ perm, int32_t* __restrict__ inv) {
  pdl_begin();
  __shared__ int idx_s[kRouterTB * 32];
  __shared__ unsigned mask_s[1024];
  const int t0 = blockIdx.x * kRouterTB;
  const int nt = min(kRouterTB, T - t0);
  const int nslots = nt * k;
  for (int i = threadIdx.x; i < E; i += blockDim.x) mask_s[i] = 0u;
  for (int i = threadIdx.x; i < nslots; i += blockDim.x) idx_s[i] = topk_idx[(size_t)t0 * k + i];
  __syncthreads();
  for (int i = threadIdx.x; i < nslots; i += blockDim.x) atomicOr(&mask_s[idx_s[i]], 1u << (i / k));
  __syncthreads();
  for (int i = threadIdx.x; i < nslots; i += blockDim.x) {
    const int tl = i / k;
    const int e = idx_s[i];
    const int rank = __popc(mask_s[e] & ((1u << tl) - 1u));
    const int pos = blk_off[(size_t)blockIdx.x * E + e] + rank;
    const int slot = t0 * k + i;
    perm[pos] = slot;
    inv[slot] = pos;
  }
}

cudaError_t launch_route_scatter(const int32_t* topk_idx, const int32_t* blk_off, int T, int k,
                                 int E, int32_t* perm, int32_t* inv, cudaStream_t st) {
  const int nblk = (T + kRouterTB - 1) / kRouterTB;
  return launch_pdl(route_scatter_kernel, dim3(nblk), dim3(256), 0, st, topk_idx, blk_off, T, k, E, perm, inv);
}

// ---------------------------------------------------------------------------
// The whole routing of a decode-sized batch (T <= 16) in one launch. The E/16
// CTAs of the small-T logits GEMV each write their experts' logits; the CTA
// that finishes last (an arrival counter, which that CTA sets back to 0 for
// the next launch; no CTA ever waits) then does, in shared memory, each
// token's top-k, the expert counts, both prefix scans, the block map and the
// scatter. Same arithmetic in the same order as router_logits_small_kernel,
// router_topk_kernel, route_scan_kernel and route_scatter_kernel, so every
// output is bit-identical to theirs (one token block: its offsets are the
// expert offsets).
// ---------------------------------------------------------------------------
constexpr int kRsThreads = 256;

template <int VPL>
__global__ void __launch_bounds__(kRsThreads) route_small_kernel(
    const uint16_t* __restrict__ x, int T, int H, const uint16_t* __restrict__ wr,
    const float* __restrict__ bias, int E, int k, float* __restrict__ logits,
    int32_t* __restrict__ topk_idx, float* __restrict__ topk_w, int32_t* __restrict__ cnt,
    int32_t* __restrict__ off, int32_t* __restrict__ tile_off, int32_t* __restrict__ bmap,
    int32_t* __restrict__ num_tiles, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
    unsigned* __restrict__ arrive) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int idx_s[kRsMaxT * 32];
  __shared__ int cnt_s[512], off_s[512];
  __shared__ unsigned mask_s[512];   // per expert: the tokens that selected it
  __shared__ int warp_sums[32];
  __shared__ int tot_rows, tot_tiles, is_last;
  rs_load_w(wr, H, E, smem);   // weights: written by no launch of this library
  pdl_begin();
  rs_logits(x, T, H, bias, E, logits, smem);

  __threadfence();   // this CTA's logits, before its arrival
  __syncthreads();
  if (threadIdx.x == 0) is_last = atomicAdd(arrive, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!is_last) return;
  __threadfence();   // the other CTAs' logits, after their arrivals
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) *arrive = 0u;
  for (int e = tid; e < E; e += kRsThreads) {
    cnt_s[e] = 0;
    mask_s[e] = 0u;
  }
  __syncthreads();

  // top-k, one warp per token
  for (int t = warp; t < T; t += kRsThreads / 32) {
    int idx;
    float w;
    topk_warp<VPL>(logits + (size_t)t * E, E, k, idx, w);
    if (lane < k) {
      topk_idx[t * k + lane] = idx;
      topk_w[t * k + lane] = w;
      idx_s[t * k + lane] = idx;
      atomicAdd(&cnt_s[idx], 1);
      atomicOr(&mask_s[idx], 1u << t);
    }
  }
  __syncthreads();

  // scans and block map, one thread per expert (256 experts per pass)
  int carry_rows = 0, carry_tiles = 0;
  for (int e0 = 0; e0 < E; e0 += kRsThreads) {
    const int e = e0 + tid;
    const bool valid = e < E;
    const int total = valid ? cnt_s[e] : 0;
    const int tiles = (total + kBM - 1) / kBM;
    const int o = block_excl_scan(total, warp_sums, &tot_rows) + carry_rows;
    const int to = block_excl_scan(tiles, warp_sums, &tot_tiles) + carry_tiles;
    if (valid) {
      cnt[e] = total;
      off[e] = o;
      off_s[e] = o;
      tile_off[e] = to;
      for (int i = 0; i < tiles; ++i) {
        const int rows = total - kBM * i;
        int32_t* m = bmap + 3 * (size_t)(to + i);
        m[0] = e;
        m[1] = o + kBM * i;
        m[2] = rows < kBM ? rows : kBM;
      }
    }
    carry_rows += tot_rows;
    carry_tiles += tot_tiles;
  }
  if (tid == 0) {
    off[E] = carry_rows;
    tile_off[E] = carry_tiles;
    num_tiles[0] = carry_tiles;
  }
  __syncthreads();

  // stable scatter: rank = earlier tokens that selected the same expert (a
  // token's k experts are distinct, so the token mask's popcount below t)
  for (int i = tid; i < T * k; i += kRsThreads) {
    const int e = idx_s[i];
    const int tl = i / k;
    const int rank = __popc(mask_s[e] & ((1u << tl) - 1u));
    const int pos = off_s[e] + rank;
    perm[pos] = i;
    inv[i] = pos;
  }
}

bool route_small_fits(int T, int H, int E, int k) {
  return T <= kRsMaxT && H % 128 == 0 && rs_smem_bytes(H) <= 200 * 1024 && E <= 512 && k <= 32;
}

cudaError_t launch_route_small(const uint16_t* x, int T, int H, const uint16_t* wr,
                               const float* bias, int E, int k, float* logits,
                               int32_t* topk_idx, float* topk_w, int32_t* cnt, int32_t* off,
                               int32_t* tile_off, int32_t* bmap, int32_t* num_tiles,
                               int32_t* perm, int32_t* inv, unsigned* arrive, cudaStream_t st) {
  if (!route_small_fits(T, H, E, k) || !arrive) return cudaErrorInvalidValue;
  const size_t smem = rs_smem_bytes(H);
  auto launch = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3((E + 15) / 16), dim3(kRsThreads), smem, st, x, T, H, wr, bias, E,
                      k, logits, topk_idx, topk_w, cnt, off, tile_off, bmap, num_tiles, perm, inv,
                      arrive);
  };
  return E <= 256 ? launch(route_small_kernel<8>) : launch(route_small_kernel<16>);
}

// ---------------------------------------------------------------------------
// Selection, counts, scans, block map and scatter of a prefill-sized batch in
// one cooperative launch (all CTAs resident at once). CTA b takes tokens
// [32 b, 32 b + 32): one warp per token selects its top-k (the same
// topk_warp as router_topk_kernel) and the CTA writes its per-expert counts.
// A grid barrier follows (the last CTA to arrive sets the arrival counter
// back to 0 and advances a generation word; the others wait for it, bounded:
// on a timeout they latch the error and skip the scatter). Then every CTA
// reads the whole count table (one batch of loads from L2) and derives, in
// the same order as route_scan_kernel, the expert totals and offsets and its
// own block's offsets, and scatters its slots; CTA 0 also writes the totals,
// offsets, tile offsets and block map. Every output is bit-identical to
// router_topk_kernel + route_scan_kernel + route_scatter_kernel. Given `xs`,
// the CTA then also gathers its tokens' rows (gather_rows_kernel's output,
// bit-identical): each token row is read once and written to its k
// positions and its shared-expert row.
// ---------------------------------------------------------------------------
constexpr int kRlThreads = 32 * kRouterTB;   // one warp per token
constexpr int kRlMaxPer = 32;                // blocks per scanning thread (counts held in registers)

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Threads per expert in the scans (a power of two), each over a range of blocks.
__host__ __device__ inline int rl_tpe(int E) {
  int tpe = 1;
  while (tpe * 2 * E <= kRlThreads && tpe < 32) tpe *= 2;
  return tpe;
}

template <int VPL>
__global__ void __launch_bounds__(kRlThreads) route_large_kernel(
    const float* __restrict__ logits, int T, int E, int k, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, uint8_t* cnt8, int np, int32_t* __restrict__ cnt,
    int32_t* __restrict__ off, int32_t* __restrict__ tile_off, int32_t* __restrict__ bmap,
    int32_t* __restrict__ num_tiles, int32_t* __restrict__ perm, int32_t* __restrict__ inv,
    unsigned* arrive, unsigned* gen, DevErr err, const uint16_t* __restrict__ x,
    uint16_t* __restrict__ xs, int H, int with_shared) {
  pdl_begin();
  __shared__ int idx_s[kRouterTB * 32];
  __shared__ int pos_s[kRouterTB * 32];       // position of each of the block's slots
  __shared__ int cnt_s[512];
  __shared__ int part_s[1024], pre_s[1024];   // per-(range, expert): block sums, sums before b
  __shared__ int boff_s[512];                 // this block's first position per expert
  __shared__ unsigned mask_s[512];            // per expert: the block's tokens that selected it
  __shared__ int wrows_s[16], wtiles_s[16];
  __shared__ int go;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nblk = gridDim.x, b = blockIdx.x;
  const int t0 = b * kRouterTB;
  const int nt = min(kRouterTB, T - t0);
  for (int i = tid; i < E; i += kRlThreads) {
    cnt_s[i] = 0;
    mask_s[i] = 0u;
  }
  __syncthreads();

  // ---- top-k and this block's counts
  if (warp < nt) {
    const int t = t0 + warp;
    int idx;
    float w;
    topk_warp<VPL>(logits + (size_t)t * E, E, k, idx, w);
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = idx;
      topk_w[(size_t)t * k + lane] = w;
      idx_s[warp * k + lane] = idx;
      atomicAdd(&cnt_s[idx], 1);
      atomicOr(&mask_s[idx], 1u << warp);
    }
  }
  __syncthreads();
  // counts as bytes, expert-major (at most 32 per block and expert)
  for (int e = tid; e < E; e += kRlThreads) cnt8[(size_t)e * np + b] = (uint8_t)cnt_s[e];

  // ---- grid barrier (the block's counts are ordered before its arrival by
  // the CTA barrier and thread 0's fence, which is cumulative)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const unsigned g0 = ld_relaxed_u32(gen);   // moves only after every arrival
    int ok = 1;
    if (atomicAdd(arrive, 1u) == (unsigned)nblk - 1) {
      *arrive = 0u;
      st_release_u32(gen, g0 + 1u);
    } else if (ld_relaxed_u32(gen) == g0) {
      const unsigned long long start = globaltimer_ns();
      while (ld_relaxed_u32(gen) == g0) {
        __nanosleep(100);
        if (globaltimer_ns() - start > err.limit_ns) {
          report_timeout(err, 30);
          ok = 0;
          break;
        }
      }
    }
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    go = ok;
  }
  __syncthreads();
  if (!go) return;

  // ---- totals, offsets and this block's offsets, from the whole count table:
  // thread (e, q) takes blocks [q per, (q + 1) per) of expert e (per a
  // multiple of 16), its counts in one batch of 16-byte loads
  const int tpe = rl_tpe(E);
  const int e = tid % E, q = tid / E;
  const bool act = q < tpe;
  const int per = (nblk + tpe - 1) / tpe + 15 & ~15;
  const int b0 = min(nblk, q * per), b1 = min(nblk, b0 + per);
  uint4 cv[kRlMaxPer / 16];
#pragma unroll
  for (int i = 0; i < kRlMaxPer / 16; ++i)
    cv[i] = act && b0 + 16 * i < b1
                ? __ldcg(reinterpret_cast<const uint4*>(cnt8 + (size_t)e * np + b0) + i)
                : make_uint4(0u, 0u, 0u, 0u);
  int sum = 0, pre = 0;
#pragma unroll
  for (int i = 0; i < kRlMaxPer; ++i) {
    const uint4 v = cv[i >> 4];
    const uint32_t wd = (i & 15) < 4 ? v.x : (i & 15) < 8 ? v.y : (i & 15) < 12 ? v.z : v.w;
    const int c = b0 + i < b1 ? (int)((wd >> (8 * (i & 3))) & 0xFFu) : 0;
    sum += c;
    if (b0 + i < b) pre += c;
  }
  if (act) {
    part_s[q * E + e] = sum;
    pre_s[q * E + e] = pre;
  }
  __syncthreads();
  // expert totals (threads tid < E) and their exclusive scans over experts:
  // shuffles inside each warp, then the warps' sums
  int tot = 0, tiles = 0, before = 0;
  if (tid < E) {
#pragma unroll
    for (int qq = 0; qq < 32; ++qq)
      if (qq < tpe) {
        tot += part_s[qq * E + tid];
        before += pre_s[qq * E + tid];
      }
    tiles = (tot + kBM - 1) / kBM;
  }
  int ri = tot, ti = tiles;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int rn = __shfl_up_sync(0xffffffffu, ri, o);
    const int tn = __shfl_up_sync(0xffffffffu, ti, o);
    if (lane >= o) {
      ri += rn;
      ti += tn;
    }
  }
  if (lane == 31 && warp < 16) {
    wrows_s[warp] = ri;
    wtiles_s[warp] = ti;
  }
  __syncthreads();
  if (tid < E) {
    int ro = ri - tot, to = ti - tiles;
#pragma unroll
    for (int w2 = 0; w2 < 16; ++w2)
      if (w2 < warp) {
        ro += wrows_s[w2];
        to += wtiles_s[w2];
      }
    boff_s[tid] = ro + before;
    if (b == 0) {
      cnt[tid] = tot;
      off[tid] = ro;
      tile_off[tid] = to;
      for (int i = 0; i < tiles; ++i) {
        const int rows = tot - kBM * i;
        int32_t* m = bmap + 3 * (size_t)(to + i);
        m[0] = tid;
        m[1] = ro + kBM * i;
        m[2] = rows < kBM ? rows : kBM;
      }
    }
  }
  if (b == 0 && tid == 0) {
    int rows_all = 0, tiles_all = 0;
    for (int w2 = 0; w2 < (E + 31) / 32; ++w2) {
      rows_all += wrows_s[w2];
      tiles_all += wtiles_s[w2];
    }
    off[E] = rows_all;
    tile_off[E] = tiles_all;
    num_tiles[0] = tiles_all;
  }
  __syncthreads();

  // ---- stable scatter of this block's slots (rank: earlier tokens of the
  // block that selected the expert; a token's experts are distinct)
  const int nslots = nt * k;
  for (int i = tid; i < nslots; i += kRlThreads) {
    const int tl = i / k;
    const int ex = idx_s[i];
    const int rank = __popc(mask_s[ex] & ((1u << tl) - 1u));
    const int pos = boff_s[ex] + rank;
    const int slot = t0 * k + i;
    perm[pos] = slot;
    inv[slot] = pos;
    pos_s[i] = pos;
  }
  if (!xs) return;

  // ---- gather (the work of gather_rows_kernel, fused): one warp per token
  // of the block reads its row once and writes it, as fp16 in perm8 order, to
  // its k routed positions and its shared-expert row.
  __syncthreads();
  if (warp < nt) {
    const int t = t0 + warp;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H);
    uint32_t over = 0u;
    for (int v = lane; v < H / 8; v += 32) {
      const uint4 a = __ldg(src + v);
      over |= bf16x2_f16_overflow(a.x) | bf16x2_f16_overflow(a.y) | bf16x2_f16_overflow(a.z) |
              bf16x2_f16_overflow(a.w);
      const uint4 o = f16x8_to_perm8(make_uint4(bf16x2_to_f16x2_sat(a.x), bf16x2_to_f16x2_sat(a.y),
                                                bf16x2_to_f16x2_sat(a.z), bf16x2_to_f16x2_sat(a.w)));
      for (int j = 0; j < k; ++j)
        reinterpret_cast<uint4*>(xs + (size_t)pos_s[warp * k + j] * H)[v] = o;
      if (with_shared) reinterpret_cast<uint4*>(xs + ((size_t)T * k + t) * H)[v] = o;
    }
    report_range_warp(err, over != 0u);
  }
}

// Bytes of the expert-major count array for nblk blocks (with the slack the
// last block's vector loads may read past the end).
size_t route_large_cnt8_bytes(int nblk, int E) {
  const size_t np = (size_t)(nblk + 15) / 16 * 16;
  return np * E + (size_t)kRlMaxPer * 32;
}

// Blocks the cooperative launch needs resident at once, and whether they fit.
bool route_large_fits(int T, int E, int k, int num_sms) {
  if (E > 512 || k > 32 || T < 1) return false;
  const int nblk = (T + kRouterTB - 1) / kRouterTB;
  const int tpe = rl_tpe(E);
  if (((nblk + tpe - 1) / tpe + 15 & ~15) > kRlMaxPer) return false;
  int dev = 0, coop = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
    return false;
  auto occ = [&](auto kern) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kRlThreads, 0);
  };
  const cudaError_t e = E <= 256 ? occ(route_large_kernel<8>) : occ(route_large_kernel<16>);
  return e == cudaSuccess && nblk <= per_sm * num_sms;
}

cudaError_t launch_route_large(const float* logits, int T, int E, int k, int32_t* topk_idx,
                               float* topk_w, uint8_t* cnt8, int32_t* cnt, int32_t* off,
                               int32_t* tile_off, int32_t* bmap, int32_t* num_tiles,
                               int32_t* perm, int32_t* inv, unsigned* arrive, unsigned* gen,
                               DevErr err, const uint16_t* x, uint16_t* xs, int H,
                               int with_shared, cudaStream_t st) {
  const int nblk = (T + kRouterTB - 1) / kRouterTB;
  const int np = (nblk + 15) / 16 * 16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nblk);
  cfg.blockDim = dim3(kRlThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  // cooperative (the blocks wait on the last one), with ordinary stream
  // order: the launch starts once the previous kernel has completed
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (E <= 256)
    return cudaLaunchKernelEx(&cfg, route_large_kernel<8>, logits, T, E, k, topk_idx, topk_w, cnt8,
                              np, cnt, off, tile_off, bmap, num_tiles, perm, inv, arrive, gen, err,
                              x, xs, H, with_shared);
  return cudaLaunchKernelEx(&cfg, route_large_kernel<16>, logits, T, E, k, topk_idx, topk_w, cnt8,
                            np, cnt, off, tile_off, bmap, num_tiles, perm, inv, arrive, gen, err,
                            x, xs, H, with_shared);
}

// ---------------------------------------------------------------------------
// Gather: xs[pos] = x[perm[pos] / k] for routed positions, and
// xs[T*k + t] = x[t] for the shared expert's rows, converted from bf16 to the
// GEMMs' fp16 operand type (exact inside fp16's range, saturating outside),
// each block of 8 stored in perm8 order (the K order of the dequantised
// weights). One warp per row. A value of magnitude 2^16 or more (or inf, or
// NaN) saturates and latches DEVERR_RANGE.
// ---------------------------------------------------------------------------
__global__ void gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                                   int T, int k, int H, int with_shared,
                                   uint16_t* __restrict__ xs, DevErr err) {
  pdl_begin();
  const int rows = T * k + (with_shared ? T : 0);
  const int lane = threadIdx.x & 31;
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int nw = (gridDim.x * blockDim.x) >> 5;
  const int vec = H / 8;   // 16-byte vectors per row
  uint32_t over = 0u;
  for (int r = wid; r < rows; r += nw) {
    const int src = r < T * k ? perm[r] / k : r - T * k;
    const uint4* s = reinterpret_cast<const uint4*>(x + (size_t)src * H);
    uint4* d = reinterpret_cast<uint4*>(xs + (size_t)r * H);
    for (int i = lane; i < vec; i += 32) {
      const uint4 v = __ldg(s + i);
      over |= bf16x2_f16_overflow(v.x) | bf16x2_f16_overflow(v.y) | bf16x2_f16_overflow(v.z) |
              bf16x2_f16_overflow(v.w);
      d[i] = f16x8_to_perm8(make_uint4(bf16x2_to_f16x2_sat(v.x), bf16x2_to_f16x2_sat(v.y),
                                       bf16x2_to_f16x2_sat(v.z), bf16x2_to_f16x2_sat(v.w)));
    }
  }
  report_range_warp(err, over != 0u);
}

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* perm, int T, int k, int H,
                               int with_shared, uint16_t* xs, DevErr err, cudaStream_t st) {
  const int rows = T * k + (with_shared ? T : 0);
  int blocks = (rows + 7) / 8;
  if (blocks > 4096) blocks = 4096;
  return launch_pdl(gather_rows_kernel, dim3(blocks), dim3(256), 0, st, x, perm, T, k, H, with_shared,
                    xs, err);
}

// ---------------------------------------------------------------------------
// Operand range of a 4-bit weight set for the tensor-core path, which
// rebuilds each weight as fp16(q * scale + bias) from fp16 copies of the bf16
// scale and bias. Faithful when every scale is 0 or has magnitude in
// [2^-14, 2^12) (a normal fp16, and 15 * scale stays below 2^16) and every
// bias has magnitude below 2^11 (so |q * scale + bias| < 65504). Anything
// else (a subnormal or huge scale, a huge bias, inf, NaN) latches
// DEVERR_RANGE. Flags are computed on pairs of bf16 magnitudes m < 0x8000 by
// 32-bit adds that set bit 15 of a half when m reaches a bound (no carry
// crosses between the halves).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t w4_range_flags(uint32_t s2, uint32_t b2) {
  const uint32_t ms = s2 & 0x7FFF7FFFu, mb = b2 & 0x7FFF7FFFu;
  const uint32_t s_high = ms + 0x3A803A80u;    // m >= 0x4580 (2^12)
  const uint32_t s_nz = ms + 0x7FFF7FFFu;      // m >= 1
  const uint32_t s_norm = ms + 0x47804780u;    // m >= 0x3880 (2^-14)
  const uint32_t b_high = mb + 0x3B003B00u;    // m >= 0x4500 (2^11)
  return (s_high | (s_nz & ~s_norm) | b_high) & 0x80008000u;
}

__global__ void __launch_bounds__(256) w4_range_kernel(const uint16_t* __restrict__ s,
                                                       const uint16_t* __restrict__ b, size_t n,
                                                       DevErr err) {
  pdl_begin();
  uint32_t bad = 0u;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const size_t i0 = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint4* s4 = reinterpret_cast<const uint4*>(s);
  const uint4* b4 = reinterpret_cast<const uint4*>(b);
  for (size_t i = i0; i < n / 8; i += stride) {
    const uint4 sv = __ldg(s4 + i), bv = __ldg(b4 + i);
    bad |= w4_range_flags(sv.x, bv.x) | w4_range_flags(sv.y, bv.y) | w4_range_flags(sv.z, bv.z) |
           w4_range_flags(sv.w, bv.w);
  }
  for (size_t i = n / 8 * 8 + i0; i < n; i += stride)   // tail (n not a multiple of 8)
    bad |= w4_range_flags(s[i], b[i]) & 0x8000u;
  report_range_warp(err, bad != 0u);
}

cudaError_t launch_w4_range_check(const uint16_t* s, const uint16_t* b, size_t n, DevErr err,
                                  int num_sms, cudaStream_t st) {
  size_t blocks = (n / 8 + 255) / 256;
  if (blocks > (size_t)4 * num_sms) blocks = (size_t)4 * num_sms;
  if (blocks < 1) blocks = 1;
  return launch_pdl(w4_range_kernel, dim3((unsigned)blocks), dim3(256), 0, st, s, b, n, err);
}

// ---------------------------------------------------------------------------
// Combine: y[t] = d_sh[t] + sum_j d[inv[t*k + j]] in FP32, fixed order
// (shared, then j = 0..k-1). Routed rows of d are bf16 and already carry
// their top-k weight; the shared expert's rows are fp32 (weight 1). y is the
// block's FP32 output.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ d,
                                                      const float* __restrict__ d_sh,
                                                      const int32_t* __restrict__ inv, int T,
                                                      int k, int H, float* __restrict__ y) {
  pdl_begin();
  __shared__ int rows_s[33];
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < k) rows_s[threadIdx.x] = inv[(size_t)t * k + threadIdx.x];
    __syncthreads();
    for (int h0 = threadIdx.x * 8; h0 < H; h0 += blockDim.x * 8) {
      float acc[8];
      if (d_sh) {
        const float4* s = reinterpret_cast<const float4*>(d_sh + (size_t)t * H + h0);
        const float4 a = __ldg(s), b = __ldg(s + 1);
        acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
        acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      }
      for (int j = 0; j < k; ++j) {
        uint4 v = __ldg(reinterpret_cast<const uint4*>(d + (size_t)rows_s[j] * H + h0));
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] += bf16_lo(w[i]);
          acc[2 * i + 1] += bf16_hi(w[i]);
        }
      }
      float4* o = reinterpret_cast<float4*>(y + (size_t)t * H + h0);
      o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
  }
}

cudaError_t launch_combine(const uint16_t* d, const float* d_sh, const int32_t* inv, int T,
                           int k, int H, float* y, cudaStream_t st) {
  int blocks = T < 4096 ? T : 4096;
  return launch_pdl(combine_kernel, dim3(blocks), dim3(256), 0, st, d, d_sh, inv, T, k, H, y);
}

// ---------------------------------------------------------------------------
// Stack update between layers, one CTA per token row:
//   x_out = bf16(x + alpha * y)            (y fp32; skipped when y is NULL)
//   xn    = bf16(x_out / sqrt(mean(x_out^2) + eps))   (when xn is not NULL)
// The mean of squares is taken over the bf16-rounded x_out, in FP32.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) residual_norm_kernel(
    const uint16_t* __restrict__ x, const float* __restrict__ y, int T, int H, float alpha,
    uint16_t* __restrict__ x_out, uint16_t* __restrict__ xn, float eps) {
  pdl_begin();
  __shared__ float warp_ss[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    const uint16_t* xr = x + (size_t)t * H;
    float ss = 0.f;
    for (int h0 = threadIdx.x * 8; h0 < H; h0 += blockDim.x * 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(xr + h0);
      const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a);
      float v[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = bf16_lo(aw[j]);
        v[2 * j + 1] = bf16_hi(aw[j]);
      }
      if (y) {
        const float4* yr = reinterpret_cast<const float4*>(y + (size_t)t * H + h0);
        const float4 b0 = yr[0], b1 = yr[1];
        const float yb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = fmaf(alpha, yb[j], v[j]);
      }
      uint4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ow[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
        const float r0 = bf16_lo(ow[j]), r1 = bf16_hi(ow[j]);
        ss = fmaf(r0, r0, fmaf(r1, r1, ss));
      }
      if (y || x_out != x) *reinterpret_cast<uint4*>(x_out + (size_t)t * H + h0) = o;
    }
    if (!xn) continue;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    __syncthreads();
    if (lane == 0) warp_ss[warp] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += warp_ss[w];
    const float inv = 1.0f / sqrtf(tot / (float)H + eps);
    // second pass over the row this thread wrote (its own values)
    for (int h0 = threadIdx.x * 8; h0 < H; h0 += blockDim.x * 8) {
      const uint4 a = *reinterpret_cast<const uint4*>((y || x_out != x ? x_out : x) +
                                                      (size_t)t * H + h0);
      const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a);
      uint4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ow[j] = pack_bf16x2(bf16_lo(aw[j]) * inv, bf16_hi(aw[j]) * inv);
      *reinterpret_cast<uint4*>(xn + (size_t)t * H + h0) = o;
    }
  }
}

// Combine and stack update in one pass, one CTA per token row:
//   y     = d_sh[t] + sum_j d[inv[t*k + j]]      (FP32, shared first, j in order)
//   x     = bf16(x + alpha * y)                  (in place)
//   xn    = bf16(x / sqrt(mean(x^2) + eps))      (mean over the bf16-rounded x)
// Every FP32 operation is the one combine_kernel then residual_norm_kernel
// perform, in the same order, so the result is bit-identical to the two
// separate passes; y itself is never written.
__global__ void __launch_bounds__(256) combine_residual_norm_kernel(
    const uint16_t* __restrict__ d, const float* __restrict__ d_sh,
    const int32_t* __restrict__ inv, int T, int k, int H, float alpha, uint16_t* x,
    uint16_t* __restrict__ xn, float eps) {
  pdl_begin();
  __shared__ int rows_s[33];
  __shared__ float warp_ss[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    __syncthreads();
    if (threadIdx.x < k) rows_s[threadIdx.x] = inv[(size_t)t * k + threadIdx.x];
    __syncthreads();
    uint16_t* xr = x + (size_t)t * H;
    float ss = 0.f;
    for (int h0 = threadIdx.x * 8; h0 < H; h0 += blockDim.x * 8) {
      float acc[8];
      if (d_sh) {
        const float4* s4 = reinterpret_cast<const float4*>(d_sh + (size_t)t * H + h0);
        const float4 a = __ldg(s4), b = __ldg(s4 + 1);
        acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
        acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      }
      for (int j = 0; j < k; ++j) {
        uint4 v = __ldg(reinterpret_cast<const uint4*>(d + (size_t)rows_s[j] * H + h0));
        const uint32_t* w = reinterpret_cast<const uint32_t*>(&v);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc[2 * i] += bf16_lo(w[i]);
          acc[2 * i + 1] += bf16_hi(w[i]);
        }
      }
      const uint4 a = *reinterpret_cast<const uint4*>(xr + h0);
      const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a);
      float v[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = fmaf(alpha, acc[2 * j], bf16_lo(aw[j]));
        v[2 * j + 1] = fmaf(alpha, acc[2 * j + 1], bf16_hi(aw[j]));
      }
      uint4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        ow[j] = pack_bf16x2(v[2 * j], v[2 * j + 1]);
        const float r0 = bf16_lo(ow[j]), r1 = bf16_hi(ow[j]);
        ss = fmaf(r0, r0, fmaf(r1, r1, ss));
      }
      *reinterpret_cast<uint4*>(xr + h0) = o;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    __syncthreads();
    if (lane == 0) warp_ss[warp] = ss;
    __syncthreads();
    float tot = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += warp_ss[w];
    const float rinv = 1.0f / sqrtf(tot / (float)H + eps);
    // second pass over the row this thread wrote (its own values)
    for (int h0 = threadIdx.x * 8; h0 < H; h0 += blockDim.x * 8) {
      const uint4 a = *reinterpret_cast<const uint4*>(xr + h0);
      const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a);
      uint4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ow[j] = pack_bf16x2(bf16_lo(aw[j]) * rinv, bf16_hi(aw[j]) * rinv);
      *reinterpret_cast<uint4*>(xn + (size_t)t * H + h0) = o;
    }
  }
}

cudaError_t launch_combine_residual_norm(const uint16_t* d, const float* d_sh, const int32_t* inv,
                                         int T, int k, int H, float alpha, uint16_t* x,
                                         uint16_t* xn, float eps, cudaStream_t st) {
  int blocks = T < 4096 ? T : 4096;
  return launch_pdl(combine_residual_norm_kernel, dim3(blocks), dim3(256), 0, st, d, d_sh, inv, T, k, H, alpha, x, xn, eps);
}

cudaError_t launch_residual_norm(const uint16_t* x, const float* y, int T, int H, float alpha,
                                 uint16_t* x_out, uint16_t* xn, float eps, cudaStream_t st) {
  int blocks = T < 8192 ? T : 8192;
  return launch_pdl(residual_norm_kernel, dim3(blocks), dim3(256), 0, st, x, y, T, H, alpha, x_out, xn, eps);
}

// ---------------------------------------------------------------------------
// Failure-path check: wait on an mbarrier nobody arrives on; the bounded wait
// must give up, latch the timeout bit and return.
// ---------------------------------------------------------------------------
__global__ void debug_wait_kernel(DevErr err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait(&bar, 0, &abort_flag, err.limit_ns)) report_timeout(err, 99);
  }
}

cudaError_t launch_debug_wait(DevErr e, cudaStream_t st) {
  debug_wait_kernel<<<1, 32, 0, st>>>(e);
  return cudaGetLastError();
}

}  // namespace moe
