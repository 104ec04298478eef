// route_noalloc.cu -- routing for callers that cannot allocate device memory.
//
// moe_route needs a plan, and a plan allocates its scratch with cudaMalloc.
// Some callers cannot do that: a host framework that hands out all device
// memory from its own pool (a cudaMalloc behind its back can fail or
// fragment the memory it budgets), runtimes with no device allocator at
// all, and latency-bound callbacks that must not block (cudaMalloc can
// synchronise the device). moe_route_noalloc serves them: the caller passes
// inputs and every output buffer, and the only scratch the routing kernels
// need (the per-token-block expert counts) lives in a fixed array in this
// file, sized for at most kMaxTokens tokens and kMaxExperts experts.
#include <mutex>

#include "moe_internal.h"

namespace {

constexpr int kMaxTokens = 4096;
constexpr int kMaxExperts = 512;
constexpr int kMaxBlocks = (kMaxTokens + moe::kRouterTB - 1) / moe::kRouterTB;
constexpr int kMaxDevices = 64;

// Per-token-block expert counts, then the blocks' offsets into each
// expert's segment: 128 x 512 int32 = 256 KB on every GPU that loads the
// library, kept until the process exits. Every call overwrites all entries
// it reads, so nothing needs clearing between calls; calls that overlap on
// the GPU (different streams, no ordering) race on it.
static __device__ __align__(256) int32_t g_blk_cnt[kMaxBlocks * kMaxExperts];

// The error word of the tensor-core logits' bounded waits: bits as in the
// plan's error word, then the first failing site. Read and cleared by
// moe_route_noalloc_get_error.
static __device__ int g_err[2];

std::mutex g_mu;
struct Scratch {
  int32_t* blk;
  int* err;
};
Scratch g_addr[kMaxDevices] = {};

// Device addresses of the arrays above on the current device. In host code
// their names are only host-side stand-ins, so the addresses are looked up
// once per device, with that device current, and reused.
moe_status scratch_address(Scratch* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev].blk) {
    void *b = nullptr, *e = nullptr;
    if (cudaGetSymbolAddress(&b, g_blk_cnt) != cudaSuccess || !b ||
        cudaGetSymbolAddress(&e, g_err) != cudaSuccess || !e)
      return MOE_ERR_CUDA;
    g_addr[dev] = Scratch{static_cast<int32_t*>(b), static_cast<int*>(e)};
  }
  *out = g_addr[dev];
  return MOE_OK;
}

bool al(const void* p, unsigned a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // 1 s

}  // namespace

extern "C" moe_status moe_route_noalloc(const uint16_t* x, int T, int hidden,
                                        const uint16_t* router_w, const float* router_bias,
                                        int num_experts, int top_k, const moe_routing* out,
                                        moe_stream_t stream) {
  if (!x || !router_w || !out) return MOE_ERR_INVALID_ARG;
  if (T < 1 || hidden <= 0 || hidden % 64 || num_experts < 8 || num_experts % 8 ||
      top_k < 1 || top_k > num_experts)
    return MOE_ERR_INVALID_ARG;
  if (top_k > 32) return MOE_ERR_UNSUPPORTED;
  if (T > kMaxTokens || num_experts > kMaxExperts) return MOE_ERR_CAPACITY;
  if (!al(x, 16) || !al(router_w, 16) || (router_bias && !al(router_bias, 4)))
    return MOE_ERR_INVALID_ARG;
  const void* need[] = {out->topk_idx, out->topk_w, out->counts,    out->offsets,
                        out->tile_offsets, out->perm, out->inv, out->block_map,
                        out->num_tiles, out->logits};
  for (const void* q : need)
    if (!q || !al(q, 8)) return MOE_ERR_INVALID_ARG;

  Scratch sc;
  moe_status s = scratch_address(&sc);
  if (s != MOE_OK) return s;
  int32_t* blk = sc.blk;
  const moe::DevErr err{sc.err, sc.err + 1, kWaitLimitNs};
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int nblk = (T + moe::kRouterTB - 1) / moe::kRouterTB;
  // every input is read after the previous launch on the stream has
  // completed (weights_early = false): the caller's own kernel just before
  // may have written the router weight
  if (moe::launch_router_topk(x, T, hidden, router_w, router_bias, num_experts, top_k,
                              out->topk_idx, out->topk_w, out->logits, blk, err,
                              st, /*weights_early=*/false) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (moe::launch_route_scan(blk, nblk, T, top_k, num_experts, out->counts, out->offsets,
                             out->tile_offsets, out->block_map, out->num_tiles,
                             st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (moe::launch_route_scatter(out->topk_idx, blk, T, top_k, num_experts, out->perm, out->inv,
                                st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

extern "C" moe_status moe_route_noalloc_get_error(void) {
  Scratch sc;
  moe_status s = scratch_address(&sc);
  if (s != MOE_OK) return s;
  int h[2] = {0, 0};
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(h, sc.err, sizeof h, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(sc.err, 0, sizeof h);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return (h[0] & moe::DEVERR_TIMEOUT_BIT) ? MOE_ERR_DEVICE_TIMEOUT : MOE_OK;
}

extern "C" moe_status moe_route_noalloc_debug_wait_timeout(int limit_us, moe_stream_t stream) {
  if (limit_us <= 0 || limit_us > 10000000) return MOE_ERR_INVALID_ARG;
  Scratch sc;
  moe_status s = scratch_address(&sc);
  if (s != MOE_OK) return s;
  const moe::DevErr err{sc.err, sc.err + 1, (unsigned long long)limit_us * 1000ull};
  return moe::launch_debug_wait(err, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
