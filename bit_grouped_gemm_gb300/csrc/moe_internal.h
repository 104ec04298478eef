// moe_internal.h -- declarations shared by the library's .cu files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_w4.h"

namespace moe {

constexpr int kBM = 128;          // rows per block-map tile
constexpr int kRouterTB = 32;     // tokens per router / scatter block
constexpr int kGroup = 64;        // quantisation group

// Bits of the device error word.
constexpr int DEVERR_TIMEOUT_BIT = 1;   // a bounded wait ran out
constexpr int DEVERR_RANGE_BIT = 2;     // an operand outside the fp16 range

// Device error state: plain pointers, usable on host and device.
struct DevErr {
  int* word;                      // error bits (DEVERR_*)
  int* where;                     // first failing site code
  unsigned long long limit_ns;    // bounded-wait limit
};

struct W4Dev {                    // one matrix set (device pointers)
  const uint32_t* q;
  const uint16_t* s;
  const uint16_t* b;
};

// 2D row-major tensor map: `rows` x `cols` elements, box `box_cols` x
// `box_rows`, 128-byte swizzle (box_cols * elem == 128); false if the driver
// entry point is missing or rejects the map.
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base,
               uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows);

// -------------------------------------------------------------- routing ---
// Router logits: the tcgen05 path when router_tc_fits (and logits and bias
// are 16-byte aligned), else the mma.sync paths. weights_early: the small-T
// kernel may copy the router weight before waiting for the previous launch
// (true inside the library's own launch sequences, where no launch writes
// weights).
bool router_tc_fits(int T, int H, int E);
cudaError_t launch_router_logits(const uint16_t* x, int T, int H, const uint16_t* wr,
                                 const float* bias, int E, float* logits, DevErr err,
                                 cudaStream_t st, bool weights_early = true);
cudaError_t launch_router_select(const float* logits, int T, int E, int k, int32_t* topk_idx,
                                 float* topk_w, int32_t* blk_cnt, cudaStream_t st);
cudaError_t launch_router_topk(const uint16_t* x, int T, int H, const uint16_t* wr,
                               const float* bias, int E, int k, int32_t* topk_idx,
                               float* topk_w, float* logits, int32_t* blk_cnt, DevErr err,
                               cudaStream_t st, bool weights_early = true);
cudaError_t launch_route_scan(int32_t* blk_cnt, int nblk, int T, int k, int E,
                              int32_t* cnt, int32_t* off, int32_t* tile_off, int32_t* bmap,
                              int32_t* num_tiles, cudaStream_t st);
cudaError_t launch_route_scatter(const int32_t* topk_idx, const int32_t* blk_off, int T, int k,
                                 int E, int32_t* perm, int32_t* inv, cudaStream_t st);
// The whole routing of a decode-sized batch in one launch (logits, top-k,
// counts, scans, block map, scatter; bit-identical to the separate launches).
// `arrive` is a device word that is 0 between launches.
bool route_small_fits(int T, int H, int E, int k);
cudaError_t launch_route_small(const uint16_t* x, int T, int H, const uint16_t* wr,
                               const float* bias, int E, int k, float* logits,
                               int32_t* topk_idx, float* topk_w, int32_t* cnt, int32_t* off,
                               int32_t* tile_off, int32_t* bmap, int32_t* num_tiles,
                               int32_t* perm, int32_t* inv, unsigned* arrive, cudaStream_t st);
// Selection through scatter of a prefill-sized batch in one cooperative
// launch, from the logits (bit-identical to launch_router_select +
// launch_route_scan + launch_route_scatter). `arrive` is 0 between launches;
// `gen` is a generation word the launch advances. route_large_fits tells
// whether the blocks can all be resident.
// `cnt8` holds route_large_cnt8_bytes(blocks, E) bytes of scratch. When `xs`
// is set, the launch also does launch_gather_rows' work (x: bf16 [T][H]).
bool route_large_fits(int T, int E, int k, int num_sms);
size_t route_large_cnt8_bytes(int nblk, int E);
cudaError_t launch_route_large(const float* logits, int T, int E, int k, int32_t* topk_idx,
                               float* topk_w, uint8_t* cnt8, int32_t* cnt, int32_t* off,
                               int32_t* tile_off, int32_t* bmap, int32_t* num_tiles,
                               int32_t* perm, int32_t* inv, unsigned* arrive, unsigned* gen,
                               DevErr err, const uint16_t* x, uint16_t* xs, int H,
                               int with_shared, cudaStream_t st);
cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* perm, int T, int k, int H,
                               int with_shared, uint16_t* xs, DevErr err, cudaStream_t st);
// Checks the fp16 operand range of n scales and biases (bf16) of a 4-bit
// weight set; latches DEVERR_RANGE in err when one is out of range.
cudaError_t launch_w4_range_check(const uint16_t* s, const uint16_t* b, size_t n, DevErr err,
                                  int num_sms, cudaStream_t st);
cudaError_t launch_combine(const uint16_t* d, const float* d_sh, const int32_t* inv, int T,
                           int k, int H, float* y, cudaStream_t st);
// combine, then x = bf16(x + alpha * y) in place and xn = bf16(rmsnorm(x)),
// without writing y (bit-identical to launch_combine + launch_residual_norm)
cudaError_t launch_combine_residual_norm(const uint16_t* d, const float* d_sh, const int32_t* inv,
                                         int T, int k, int H, float alpha, uint16_t* x,
                                         uint16_t* xn, float eps, cudaStream_t st);
cudaError_t launch_residual_norm(const uint16_t* x, const float* y, int T, int H, float alpha,
                                 uint16_t* x_out, uint16_t* xn, float eps, cudaStream_t st);
cudaError_t launch_debug_wait(DevErr e, cudaStream_t st);

// ---------------------------------------------------------------- GEMMs ---
// Problem of one grouped GEMM launch (gate/up + SwiGLU, or down + weight).
struct GemmProblem {
  int T, k, E;
  int K;                    // reduction size (gate/up: H, down: I)
  int N;                    // weight rows per expert (gate/up: I, down: H)
  int has_shared;
  const int32_t* bmap;      // routed block map [tiles][3]
  const int32_t* num_tiles; // device count of routed tiles
  int max_routed_tiles;     // host upper bound (grid sizing)
  const uint16_t* act_in;   // B operand rows [rows][K] fp16 perm8 (xs or act)
  const uint16_t* gather_x; // small-M gate/up only: when set, B row `pos` is read from
                            // these bf16 token rows [T][K] (token perm[pos] / k, or
                            // pos - T*k for the shared expert) instead of act_in
  uint16_t* out;            // output rows [rows][out_ld] bf16 (down: routed rows only)
  float* out_sh;            // down: the shared expert's rows, fp32 [T][out_ld]
  int out_ld;
  const float* topk_w;      // down: per-slot weights (by slot)
  const int32_t* perm;      // down: position -> slot
  W4Dev w0, w1;             // routed: gate,up (mode 0) or down,down (mode 1)
  W4Dev sw0, sw1;           // shared expert, same roles
  W4Dev next, snext;        // small-M gate/up only: the down matrices (routed, shared),
                            // whose rows each unit prefetches into L2 (q null: none)
  int next_K;               // reduction size of the down matrices (I)
  float* sk_ws;             // tensor-core path: fp32 partials of the split last round,
                            // kSplitSlotBytes per slot (null: no split)
  unsigned* sk_cnt;         // one arrival counter per slot, zero between launches
  int sk_slots;             // slots of sk_ws and sk_cnt
};

// Split last round of the tensor-core GEMM: one slot per CTA of
// 2 weight blocks x 128 tokens x 128 rows fp32.
constexpr int kSplitSlots = 192;
constexpr size_t kSplitSlotBytes = 2u * 128u * 128u * 4u;

// tcgen05 tensor-core path. `maps` holds the encoded tensor maps the kernel
// needs (B operand, routed q for w0/w1, shared q for sw0/sw1).
struct TcMaps {
  CUtensorMap b[4];         // act_in, fp16 [rows][K], boxes 64 x {128,64,32,16} rows,
                            // swizzle 128B (the smallest box covering a tile is used)
  CUtensorMap q0, q1;       // routed q of w0/w1, uint32 [E*N][K/8], box 32 x 128
  CUtensorMap sq0, sq1;     // shared q
};
cudaError_t launch_gemm_tc(int mode, const GemmProblem& p, const TcMaps& maps, DevErr err,
                           int num_sms, cudaStream_t st);

// Pair kernel (cta_group::2, gemm_tc2.cu): units of 256-row tiles (bmap2,
// from launch_build_tiles256) x 256 weight rows. maps.q0/q1 (and sq0/sq1)
// use boxes of 64 rows for the gate/up pass (mode 0) and 128 rows for the
// down pass (mode 1).
cudaError_t launch_gemm_tc2(int mode, const GemmProblem& p, const TcMaps& maps,
                            const int32_t* bmap2, const int32_t* num_tiles2, int max_tiles2,
                            DevErr err, int num_sms, cudaStream_t st);
cudaError_t launch_build_tiles256(const int32_t* off, int E, int32_t* bmap2, int32_t* num_tiles2,
                                  cudaStream_t st);
bool tc2_supported();

// small-M mma.sync path (decode-sized token groups). `maps` holds the packed
// words of w0/w1 (routed) and sw0/sw1 (shared) as uint32 [rows][K/8] maps with
// 128-byte swizzle and boxes of 32 words x smallm_rows_per_unit(mode) rows.
struct SmallMaps {
  CUtensorMap q0, q1, sq0, sq1;
};
int smallm_rows_per_unit(int mode);
bool smallm_fits(int H, int I);
cudaError_t launch_gemm_smallm(int mode, const GemmProblem& p, const SmallMaps& maps, DevErr err,
                               int num_sms, cudaStream_t st);

// ------------------------------------------------------ fused decode layer ---
// One whole layer of a decode-sized batch (T <= 8) in one cooperative launch
// (decode_fused.cu): router, top-k, gate/up + SwiGLU, down, combine and the
// stack update x = bf16(x + alpha * y), with the RMS norm of x taken inside.
struct DecodeLayerArgs {
  int T, H, I, E, k, has_shared;
  float alpha, eps;
  uint16_t* x;                   // residual bf16 [T][H], updated in place
  const uint16_t* router_w;
  const float* router_bias;
  W4Dev gate, up, down, sgate, sup, sdown;
  CUtensorMap maps[6];           // gate, up, down, shared gate, up, down (encode_slab_3d:
                                 // 8-row boxes for gate/up, 16 for down)
  CUtensorMap router_map;        // router weight, encode_router_slices
  uint16_t* act;                 // [T*k + T][I] fp16 scratch
  int32_t* topk_idx;             // [T][k] routing of the layer (outputs)
  float* topk_w;
  float* y_out;                  // [T][H] FP32 block output, or null
  unsigned* bar;                 // grid-barrier counter, 0 between launches
  unsigned* epoch;               // launches of the fused layer so far (the logits' tag - 1)
  unsigned long long* tlogits;   // [T][E] logits with the launch's tag in the high word
};
bool decode_fused_fits(int T, int H, int I, int E, int k, int has_shared, int num_sms);
cudaError_t launch_decode_layer(const DecodeLayerArgs& a, DevErr err, int num_sms, cudaStream_t st);

// 2D map of the router weight bf16 [H][E] with boxes of 8 experts x 256 rows
// (16-byte rows, no swizzle).
bool encode_router_slices(CUtensorMap* m, const void* base, int H, int E);

// 3D map of a packed-word matrix uint32 [rows][K/8] as boxes of 32 words x
// box_rows rows x K/256 chunks (one box = box_rows whole rows), 128-byte swizzle.
bool encode_slab_3d(CUtensorMap* m, const void* base, uint64_t rows, int K, uint32_t box_rows);

}  // namespace moe
