// moe_common.cuh -- device helpers shared by the kernels of the W4A16 MoE block
// (inline PTX wrappers for mbarrier, TMA, tcgen05 and the bounded waits).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {

// ------------------------------------------------ programmatic dependent launch ---
// Every kernel of this library is launched with launch_pdl and starts with
// pdl_begin(): it waits until the previous kernel on the stream has completed
// and its writes are visible, then lets the next kernel launch. The next
// kernel can thus be scheduled while this one runs instead of after it
// exits; it launches only once every CTA of this kernel has started, and
// waits for this kernel's completion before touching memory, so stream order
// is kept (and stays transitive along the stream).
//
// Because every kernel here lets its dependents launch only after its own
// wait, all launches before the previous one have completed by the time a
// kernel starts. A kernel may therefore read, before pdl_wait(), memory that
// the previous launch does not write: the weights (written by no launch of
// this library), and buffers the launch before the previous one wrote (read
// through L2 with ld.global.cg, never from L1).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_begin() {
  pdl_wait();
  pdl_trigger();
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ---------------------------------------------------------------- errors ---
// Device error word bits (latched with atomicOr, read by moe_get_error).
//   DEVERR_TIMEOUT: a bounded wait ran out;
//   DEVERR_RANGE:   an operand left the range in which its conversion to the
//                   MMAs' fp16 is faithful (see bf16x2_f16_overflow and
//                   w4_range_flags).
enum : int { DEVERR_TIMEOUT = DEVERR_TIMEOUT_BIT, DEVERR_RANGE = DEVERR_RANGE_BIT };

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void report_timeout(const DevErr& e, int site) {
  atomicOr(e.word, DEVERR_TIMEOUT);
  atomicCAS(e.where, 0, site);
}

// Latches DEVERR_RANGE once per warp that saw a flag (call with the whole
// warp converged).
__device__ __forceinline__ void report_range_warp(const DevErr& e, bool bad) {
  if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(e.word, DEVERR_RANGE);
}

// Nonzero when either bf16 of the pair has magnitude >= 2^16 (or is inf or
// NaN): its fp16 conversion saturates. The magnitudes m < 0x8000 of both
// halves get 0x8000 - 0x4780 added in one 32-bit add (no carry between the
// halves), which sets bit 15 of a half exactly when m >= 0x4780 (2^16).
__device__ __forceinline__ uint32_t bf16x2_f16_overflow(uint32_t v) {
  return ((v & 0x7FFF7FFFu) + 0x38803880u) & 0x80008000u;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// -------------------------------------------------------------- mbarrier ---
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// Arrival without release ordering: for a consumer whose reads have already
// completed (e.g. tcgen05.ld after tcgen05.wait::ld), so that the arrival does
// not wait for the thread's earlier global stores to drain.
__device__ __forceinline__ void mbar_arrive_relaxed(uint64_t* bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps until the phase completes or about `hint_ns` pass, instead of
// spinning and taking issue slots from the warps that do the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n"
      " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
constexpr uint32_t kWaitSleepNs = 100000;

// Bounded wait for the phase with the given parity. Returns false when the
// limit ran out or another role of the CTA raised `abort_flag`.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag,
                                          unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Bounded wait that ignores the abort flag: used to drain a CTA's own
// in-flight copies and MMAs before it releases shared and tensor memory.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity,
                                                unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepNs)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Elects one lane of the converged warp (the lowest active one): the lane that
// issues a role's single-thread operations while the whole warp runs the loop.
// Waits are taken by all 32 lanes; a wait by one lane whose siblings sit
// elsewhere costs hundreds of cycles per call on sm_103a.
__device__ __forceinline__ bool elect_one_sync() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .b32 r;\n .reg .pred p;\n elect.sync r|p, 0xffffffff;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(pred));
  return pred != 0;
}

// ------------------------------------------------------------------- TMA ---
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// Contiguous global -> shared copy by the TMA unit; both addresses 16-byte
// aligned, `bytes` a multiple of 16; completion counted on `bar` (bytes).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Prefetch of a contiguous global range into L2 (16-byte aligned address,
// size a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 2D tiled load global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 3D tiled load global -> shared, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, int x, int y, int z,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- mma.sync ---
// D (+)= A * B, m16n8k16, fp16 operands, fp32 accumulation. Not volatile:
// the compiler may interleave independent MMAs to hide their latency.
__device__ __forceinline__ void mma_m16n8k16_f16(float (&c)[4], uint32_t a0, uint32_t a1,
                                                 uint32_t a2, uint32_t a3, uint32_t b0,
                                                 uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- tcgen05 ---
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_result, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_result)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]; kind::f16 (16-bit inputs, fp32 accumulate).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 bit, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, "
      "%10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, "
      "%26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart (tile base 1024-byte aligned).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);        // start address
  d |= static_cast<uint64_t>(1u) << 16;                           // LBO (unused, swizzled K-major)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;                   // SBO: 8 rows * 128 B
  d |= static_cast<uint64_t>(1u) << 46;                           // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;                           // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B fp16, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                                 // D format: f32
         | (0u << 7)                               // A format: f16
         | (0u << 10)                              // B format: f16
         | (static_cast<uint32_t>(N >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);  // M / 16
}

// ------------------------------------------------------ bf16 / fp16 utils ---
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t v) {
  return __uint_as_float(static_cast<uint32_t>(v) << 16);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

// fp16 with saturation to the finite range (no inf from large inputs).
constexpr float kF16Max = 65504.0f;
__device__ __forceinline__ float sat_f16_range(float v) {
  return fminf(fmaxf(v, -kF16Max), kF16Max);
}
__device__ __forceinline__ uint16_t f32_to_f16_sat(float f) {
  __half h = __float2half_rn(sat_f16_range(f));
  return *reinterpret_cast<uint16_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16x2_sat(float lo, float hi) {
  __half2 v = __floats2half2_rn(sat_f16_range(lo), sat_f16_range(hi));
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ float f16_lo(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
}

// Bits of a LOP3: (a & b) | c.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Four f16x2 words holding 1024 + q for the eight nibbles of `w`, as pairs
// (q0,q4), (q1,q5), (q2,q6), (q3,q7): 0x6400 is fp16 1024.0, whose unit in
// the last place is 1, so a nibble in the low mantissa bits adds its value.
__device__ __forceinline__ void nibbles_to_f16x2_1024(uint32_t w, uint32_t (&p)[4]) {
  p[0] = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
  p[1] = lop3_and_or(w >> 4, 0x000F000Fu, 0x64006400u);
  p[2] = lop3_and_or(w >> 8, 0x000F000Fu, 0x64006400u);
  p[3] = lop3_and_or(w >> 12, 0x000F000Fu, 0x64006400u);
}

// Nibble pair j (j = 0..3: nibbles j and j + 4) of a packed word as the
// f16x2 word (1024 + q_j, 1024 + q_{j+4}) -- one element of
// nibbles_to_f16x2_1024, for callers that need only some of the four.
__device__ __forceinline__ uint32_t nibble_pair_1024(uint32_t w, int j) {
  return lop3_and_or(w >> (4 * j), 0x000F000Fu, 0x64006400u);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Dequantise one packed word (8 consecutive k) to 4 f16x2 words in k order:
// w_k = fp16(q_k * s + b), one rounding (f16x2 fused multiply-add of exact q).
__device__ __forceinline__ void dequant_word_f16(uint32_t w, __half2 s2, __half2 b2,
                                                 uint32_t (&out)[4]) {
  uint32_t p[4];
  nibbles_to_f16x2_1024(w, p);
  const __half2 c1024 = __floats2half2_rn(1024.0f, 1024.0f);
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 v = *reinterpret_cast<__half2*>(&p[i]);
    v = __hsub2(v, c1024);           // exact: q in 0..15
    v = __hfma2(v, s2, b2);          // round once to fp16
    r[i] = *reinterpret_cast<uint32_t*>(&v);
  }
  // (q0,q4) (q1,q5) (q2,q6) (q3,q7) -> (q0,q1) (q2,q3) (q4,q5) (q6,q7)
  out[0] = prmt(r[0], r[1], 0x5410);
  out[1] = prmt(r[2], r[3], 0x5410);
  out[2] = prmt(r[0], r[1], 0x7632);
  out[3] = prmt(r[2], r[3], 0x7632);
}

// The GEMM operands' K order inside every block of 8: position p holds
// element perm8[p] = (0,4,1,5,2,6,3,7)[p], the order in which the nibble
// extraction above yields the eight weights of a packed word. Activations
// stored in this order meet the dequantised weights without a shuffle.
// perm8_pos(i) is the position of element i.
__host__ __device__ __forceinline__ int perm8_pos(int i) {
  return (i & ~7) | ((i & 3) << 1) | ((i >> 2) & 1);
}

// Dequantise one packed word to 4 f16x2 words in perm8 order:
// (q0,q4) (q1,q5) (q2,q6) (q3,q7), each fp16(q * s + b) with one rounding.
__device__ __forceinline__ void dequant_word_f16_perm8(uint32_t w, __half2 s2, __half2 b2,
                                                       uint32_t (&out)[4]) {
  // Nibbles 0/4 and 2/6 land in the low mantissa bits of 1024.0 (value
  // 1024 + q); nibbles 1/5 and 3/7 are masked in place, four bits higher
  // (value 1024 + 16 q), which saves two shifts on the integer pipe. Both
  // forms are turned back into q exactly before the one rounding of q*s + b.
  const uint32_t w8 = w >> 8;
  const uint32_t p0 = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
  const uint32_t p1 = lop3_and_or(w, 0x00F000F0u, 0x64006400u);
  const uint32_t p2 = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);
  const uint32_t p3 = lop3_and_or(w8, 0x00F000F0u, 0x64006400u);
  const __half2 c1024 = __floats2half2_rn(1024.0f, 1024.0f);
  const __half2 c16th = __floats2half2_rn(0.0625f, 0.0625f);
  const __half2 cm64 = __floats2half2_rn(-64.0f, -64.0f);
  // (1024 + q) - 1024 = q and (1024 + 16 q) / 16 - 64 = q, both exact
  const __half2 q0 = __hsub2(*reinterpret_cast<const __half2*>(&p0), c1024);
  const __half2 q1 = __hfma2(*reinterpret_cast<const __half2*>(&p1), c16th, cm64);
  const __half2 q2 = __hsub2(*reinterpret_cast<const __half2*>(&p2), c1024);
  const __half2 q3 = __hfma2(*reinterpret_cast<const __half2*>(&p3), c16th, cm64);
  const __half2 r0 = __hfma2(q0, s2, b2), r1 = __hfma2(q1, s2, b2);
  const __half2 r2 = __hfma2(q2, s2, b2), r3 = __hfma2(q3, s2, b2);
  out[0] = *reinterpret_cast<const uint32_t*>(&r0);
  out[1] = *reinterpret_cast<const uint32_t*>(&r1);
  out[2] = *reinterpret_cast<const uint32_t*>(&r2);
  out[3] = *reinterpret_cast<const uint32_t*>(&r3);
}

// 8 fp16 in natural order (4 words) -> perm8 order
__device__ __forceinline__ uint4 f16x8_to_perm8(uint4 v) {
  return make_uint4(prmt(v.x, v.z, 0x5410), prmt(v.x, v.z, 0x7632), prmt(v.y, v.w, 0x5410),
                    prmt(v.y, v.w, 0x7632));
}

// bf16 bit pattern -> fp16 (saturating) bits, the pair packed as f16x2
__device__ __forceinline__ uint32_t bf16x2_to_f16x2_sat(uint32_t v) {
  return pack_f16x2_sat(bf16_lo(v), bf16_hi(v));
}

__device__ __forceinline__ float silu_f32(float g) { return g / (1.0f + expf(-g)); }
// silu with the fast exponential and division (relative error ~1e-6, far
// below the fp16 rounding of its result); for g below about -88 the
// denominator overflows and the result is -0.
__device__ __forceinline__ float silu_fast(float g) {
  return __fdividef(g, 1.0f + __expf(-g));
}

}  // namespace moe
