// Internal launch interface between the plan/ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Sets the thread's moe_last_error() message and returns s (api.cu).
moe_status fail_message(moe_status s, const char* msg);

// A conversion x (bf16) -> x16 (fp16) of n8 * 8 elements that a kernel performs on the side with
// every thread of its grid (the 4-bit path's activation copy; convert_x16 in common.cuh);
// x16 == nullptr: none.
struct XConv {
  const uint16_t* x = nullptr;
  uint16_t* x16 = nullptr;
  size_t n8 = 0;
};

// Tokens per chunk of the grouping step: one 32-bit mask word per (chunk, expert).
constexpr int kChunk = 32;
// Row stride (32-bit words) of the per-chunk expert masks masks[e][c] for n_chunks chunks: a
// multiple of 4, so that rows are read as 16-byte vectors.
__host__ __device__ inline int group_mask_stride(int n_chunks) { return (n_chunks + 3) & ~3; }
// Largest number of rows one tensor-core unit handles (the MMA's N).
constexpr int kSegRowsMax = 128;

// One segment of the grouped problem: `rows` consecutive grouped rows of one expert starting
// at `row_start`.  An expert with more than kSegRowsMax rows has several parts; `first` is
// the index of its first part in the segment list and `nparts` their number.
struct Seg {
  int expert;
  int row_start;
  int rows;
  int first;
  int nparts;
  int pad0, pad1, pad2;
};

// ---- routing and grouping (route.cu) --------------------------------------------------------
// logits[t][e] = x[t] . w_router[e] + b[e] (fp32 accumulation).
cudaError_t launch_router_logits(const uint16_t* x, const float* w_router, const float* b_router, int T,
                                 int E, int d, float* logits, cudaStream_t st);
// Top-k + softmax gates per token.  The logits are sum_s parts[s][T][E] (+ bias[e]) and are
// written to logits_out if given.  If masks != nullptr also writes the per-chunk expert masks,
// expert-major: bit t of masks[e * n_chunks + c] <=> token c*32+t chose e.
// xc: an x -> fp16 conversion the launch performs on the side (none by default).
cudaError_t launch_topk(const float* parts, int nsplit, const float* bias, float* logits_out, int T, int E, int k,
                        int32_t* ids, float* gates, uint32_t* masks, uint32_t* err, cudaStream_t st,
                        const XConv& xc = XConv{});

// ---- tensor-core router (router_tc.cu) --------------------------------------------------------
// parts[s][T][E] = x[T][k-range s] . W_r[E][k-range s]^T with W_r split into three bf16 pieces
// (w3: 2-D map over [3E rows][d], box 64 x 128).  Requires E % 128 == 0 and d % 64 == 0.
int router_tc_splits(int T, int E, int d, int num_sms);
constexpr int kRouterTcMinT = 16;  // the tensor-core router serves T > 16

// Small-T router (d % 128 == 0): K-split partials parts[router_small_splits(d)][T][E], no bias.
int router_small_splits(int d);
cudaError_t launch_router_parts_small(const uint16_t* x, const float* w_router, int T, int E, int d, float* parts,
                                      cudaStream_t st);

// Top-k + counts + offsets + segments + stable permutation of a small step in one launch.
constexpr int kSmallRouteT = 64;
bool route_small_ok(int T, int E, int k, int nsplit);
// Router + top-k + grouping of a step of at most 8 tokens (d % 128 == 0) in one launch.
bool router_route_tiny_ok(int T, int E, int d, int k);
cudaError_t launch_router_route_tiny(const uint16_t* x, const float* w_router, const float* bias, int T, int E, int d,
                                     float* parts, int k, int32_t* ids, float* gates, int32_t* counts,
                                     int32_t* offsets, int32_t* perm, int32_t* inv, Seg* segs, int32_t* n_segs,
                                     int max_segs, uint32_t* done, uint32_t* err, cudaStream_t st,
                                     const XConv& xc = XConv{});

// `done`: a device counter that is 0 between launches (the last block resets it).
cudaError_t launch_route_small(const float* parts, int nsplit, const float* bias, int T, int E, int k, int32_t* ids,
                               float* gates, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv, Seg* segs,
                               int32_t* n_segs, int max_segs, uint32_t* done, uint32_t* err, cudaStream_t st,
                               const XConv& xc = XConv{});
// Persistent: min(items, num_sms) CTAs over the (expert tile, K split, token tile) items.
// xm: x [T][d] bf16, box {64, 128}, 128-byte swizzle.
cudaError_t launch_router_tc(const CUtensorMap* w3, const CUtensorMap* xm, int T, int E, int d, int nsplit,
                             float* parts, uint32_t* err, int num_sms, cudaStream_t st);
cudaError_t launch_split_router(const float* w, uint16_t* w3, size_t n, cudaStream_t st);
// Per-chunk expert masks from given ids (validates range / duplicates).
cudaError_t launch_masks_from_ids(const int32_t* ids, int T, int E, int k, uint32_t* masks,
                                  uint32_t* err, cudaStream_t st);
// Grouping in one launch from the chunk masks and the ids: counts, offsets (exclusive scan of
// counts, offsets[E] = total), perm / inv_perm (-1 for a dropped assignment) and, if segs is
// given, the segment list of the routed experts for the grouped GEMMs.
cudaError_t launch_group(const int32_t* ids, const uint32_t* masks, int T, int E, int k, int32_t* counts,
                         int32_t* offsets, int32_t* perm, int32_t* inv, Seg* segs, int32_t* n_segs, int max_segs,
                         uint32_t* err, cudaStream_t st);
// Segment list from offsets only (used by the separate experts entry point).
cudaError_t launch_segments_from_offsets(const int32_t* offsets, int E, Seg* segs, int32_t* n_segs,
                                         int max_segs, uint32_t* err, cudaStream_t st);

// ---- expert FFN, CUDA-core reference path (ffn_simt.cu) -------------------------------------
struct FfnWeights {
  // Routed experts.  bf16: w_gu [E][2f][d] with gate/up rows interleaved in groups of 8
  // (rows 16q..16q+7 = gate rows 8q..8q+7, rows 16q+8..16q+15 = up rows 8q..8q+7),
  // w_down [E][d][f] held as fp16.  MXFP4: the same row order for codes [.][.][K/2] and scales
  // [.][.][K/32]; w_down codes [E][d][f/2].
  const void* w_gu = nullptr;
  const uint8_t* s_gu = nullptr;
  const void* w_down = nullptr;
  const uint8_t* s_down = nullptr;
  int fp4 = 0;
  // Shared experts, n_shared concatenated: w_gu_s bf16 [n_s*2*f_s][d] interleaved the same
  // way per expert, w_down_s fp16 [n_s][d][f_s].
  const uint16_t* w_gu_s = nullptr;
  const uint16_t* w_down_s = nullptr;
  int n_shared = 0;
  int f_s = 0;
  int E = 0, k = 0, d = 0, f = 0;
  uint32_t* err = nullptr;
  // 1: bf16 routed / shared weights are in the tile-contiguous layouts of the tensor-core path;
  // fp4_tiled: 4-bit routed weights in the launch_tile_fp4 layout (scales inside the blocks)
  int tiled = 0, tiled_s = 0, fp4_tiled = 0;
};

// h, h_s, y, y_s are fp16.
cudaError_t launch_ffn_simt(const FfnWeights& w, const uint16_t* x, int T, const int32_t* offsets,
                            const int32_t* perm, uint16_t* h, uint16_t* h_s, uint16_t* y,
                            uint16_t* y_s, cudaStream_t st);

// ---- expert FFN, tcgen05 path (gemm_tc.cu) ---------------------------------------------------
struct TcMaps {
  CUtensorMap h;         // B for down: [R_max rows][f] fp16, box 64 x 32
  CUtensorMap h_s;       // B for shared down: [T_max rows][n_s*f_s] fp16, box 64 x 32
};

struct TcArgs {
  // tile-contiguous weights (launch_tile_gate_up / launch_tile_down layouts)
  const uint16_t* w_gu = nullptr;    // [E][f/64][d/64] blocks, bf16
  const uint16_t* w_gu_s = nullptr;  // [n_s*f_s/64][d/64] blocks, bf16
  const uint16_t* w_down = nullptr;  // [E][d/128][f/64] blocks, fp16
  const uint16_t* w_down_s = nullptr;  // [d/128][n_s][f_s/64] blocks, fp16
  // 4-bit routed weights (launch_tile_fp4 layout) for the fp4 kernels
  const uint8_t* q_gu = nullptr;     // [E][f/64][d/64] blocks of kFp4BlockBytes
  const uint8_t* q_down = nullptr;   // [E][d/128][f/64] blocks
  const uint16_t* x16 = nullptr;     // fp16 copy of x (4-bit path's B operand)
  const uint8_t* xq = nullptr;       // x as two e4m3 terms [T][2][d] (block-scaled gate/up's B operand)
  const uint8_t* xs = nullptr;       // their e8m0 scales [T][2][d / 32]
  uint32_t* sched = nullptr;         // persistent 4-bit kernels: the launch's unit hand-out words
  int routed = 1;                    // 0: the 16-bit kernels run the shared-expert units only
  const Seg* segs = nullptr;
  const int32_t* n_segs = nullptr;
  const int32_t* perm = nullptr;
  const uint16_t* x = nullptr;
  uint16_t* h = nullptr;
  uint16_t* h_s = nullptr;
  uint16_t* y = nullptr;
  uint16_t* y_s = nullptr;
  uint32_t* err = nullptr;
  int T = 0, E = 0, k = 0, d = 0, f = 0, n_shared = 0, f_s = 0;
  int n_shared_segs = 0;   // ceil(T / kSegRowsMax) when n_shared > 0 (shared tokens split evenly)
  int pair = 2;            // bf16 kernels: weight tiles per unit (2 shares each B stage; 1 for few units)
};

cudaError_t launch_tc_gateup(const TcMaps* maps, const TcArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_tc_down(const TcMaps* maps, const TcArgs& a, int num_sms, cudaStream_t st);

// ---- expert FFN with 4-bit routed weights, tcgen05 (gemm_fp4.cu) -----------------------------
// Routed units only (shared experts go through the 16-bit kernels with routed = 0).
cudaError_t launch_fp4_gateup(const TcMaps* maps, const TcArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_fp4_down(const TcMaps* maps, const TcArgs& a, int num_sms, cudaStream_t st);
// x16 = fp16(x), n elements (multiple of 8); out-of-range values clamp and flag MOE_DEVERR_RANGE.
cudaError_t launch_x_to_f16(const uint16_t* x, uint16_t* x16, size_t n, uint32_t* err, cudaStream_t st);
// ---- 4-bit gate/up on the block-scaled MMA (gemm_mx.cu) ------------------------------------------
// xq [T][2][d] e4m3 (hi, lo) and xs [T][2][d / 32] e8m0 from x (bf16); requires d % 128 == 0.
cudaError_t launch_x_to_mx(const uint16_t* x, uint8_t* xq, uint8_t* xs, int T, int d, cudaStream_t st);
// h = SwiGLU of the routed units (a.q_gu tiled 4-bit weights, a.xq / a.xs, a.sched: zeroed words
// [0] units handed out, [1] CTAs exited; the last CTA resets them).
cudaError_t launch_mx_gateup(const TcArgs& a, int num_sms, cudaStream_t st);
// y (fp16) of the routed units from W_down (a.q_down) and h in two e4m3 terms: a.xq = hq
// [R][2][f], a.xs = hs [R][2][mx_scale_bytes(f)] (launch_h_to_mx), a.sched as above.
cudaError_t launch_mx_down(const TcArgs& a, int num_sms, cudaStream_t st);
// hq / hs from h (fp16 [R][f]); f % 64 == 0.
cudaError_t launch_h_to_mx(const uint16_t* h, uint8_t* hq, uint8_t* hs, int R, int f, cudaStream_t st);
// scale bytes per quantised row of K elements (K / 32 rounded up to a multiple of 4)
int mx_scale_bytes(int K);

// ---- one-launch layer of a small step (layer_small.cu) ------------------------------------------
constexpr int kLsTMax = 8;                  // tokens per step
constexpr int kLsUnionBytes = 76 * 1024;    // x (bf16) and then h (fp16) of the step in shared memory
constexpr int kLsSyncWords = 8;            // launch-wide counters and flags
struct LsArgs {
  const uint16_t* x = nullptr;
  const float* w_router = nullptr;
  const float* b_router = nullptr;
  const uint16_t* w_gu = nullptr;      // tile-contiguous layouts of the tensor-core path
  const uint16_t* w_down = nullptr;
  const uint16_t* w_gu_s = nullptr;
  const uint16_t* w_down_s = nullptr;
  float* logits = nullptr;             // [T][E]
  int32_t* ids = nullptr;              // [T][k]
  float* gates = nullptr;              // [T][k]
  int32_t* counts = nullptr;           // [E]
  int32_t* offsets = nullptr;          // [E + 1]
  int32_t* perm = nullptr;             // [T k]
  int32_t* inv = nullptr;              // [T k]
  int32_t* touched = nullptr;          // [E]: touched experts, ascending
  int32_t* n_touched = nullptr;        // 1 word
  uint16_t* h = nullptr;               // fp16 [T k][f] grouped rows
  uint16_t* h_s = nullptr;             // fp16 [T][n_s f_s]
  float* y32 = nullptr;                // fp32 [T k][d] per assignment t k + j
  float* ys32 = nullptr;               // fp32 [T][d]
  uint16_t* out = nullptr;             // bf16 [T][d]
  uint32_t* sync = nullptr;            // kLsSyncWords plan-owned words, zero between launches
  uint32_t* err = nullptr;
  int T = 0, E = 0, k = 0, d = 0, f = 0, n_shared = 0, f_s = 0;
};
bool layer_small_ok(int T, int E, int k, int d, int f, int n_shared, int f_s);
cudaError_t launch_layer_small(const LsArgs& a, int num_sms, cudaStream_t st);

// ---- combine (combine.cu): out bf16; y and shared_y fp16 (the layer's intermediates) or fp32 ----
cudaError_t launch_combine(const uint16_t* y, const float* gates, const int32_t* inv,
                           const uint16_t* shared_y, int T, int k, int d, uint16_t* out,
                           cudaStream_t st);
cudaError_t launch_combine_f32(const float* y, const float* gates, const int32_t* inv, const float* shared_y, int T,
                               int k, int d, uint16_t* out, cudaStream_t st);

// ---- weight repacking at set-up (repack.cu) --------------------------------------------------
// dst [n][2f][K*elem] <- gate [n][f][K*elem], up [n][f][K*elem], rows interleaved by 8.
cudaError_t launch_interleave_gate_up(const uint8_t* gate, const uint8_t* up, uint8_t* dst, int n,
                                      int f, size_t row_bytes, cudaStream_t st);
// dst fp16 <- src bf16 (round to nearest even); *bad |= 1 if a value is outside the fp16 range.
cudaError_t launch_bf16_to_f16(const uint16_t* src, uint16_t* dst, size_t n, uint32_t* bad, cudaStream_t st);
// Tile-contiguous, pre-swizzled layouts of the tensor-core path (16 KB blocks of 128 rows x 64
// K elements).  A weight matrix of `tiles` 128-row tiles and nk K chunks stores its blocks at
// tile_chunk_offset: tiles are paired and the two tiles of a pair alternate along K, so both
// blocks of one K chunk are adjacent (one 32 KB copy); an odd last tile stands alone.
//   gate/up of n experts (rows interleaved by 8): one matrix per expert (f/64 tiles, d/64 chunks),
//     or with one_matrix the n experts as one matrix of n f/64 tiles (the shared experts);
//   down (bf16 -> fp16) of n matrices [rows][K]: by_matrix ? one matrix per expert (rows/128
//     tiles, K/64 chunks) : one matrix of rows/128 tiles whose K runs over all n (n K/64 chunks).
cudaError_t launch_tile_gate_up(const uint16_t* gate, const uint16_t* up, uint16_t* dst, int n, int f, int d,
                                int one_matrix, cudaStream_t st);
cudaError_t launch_tile_down(const uint16_t* src, uint16_t* dst, int n, int rows, int K, int by_matrix, uint32_t* bad,
                             cudaStream_t st);
constexpr int kTileElems = 128 * 64;
// 4-bit tile-contiguous blocks (launch_tile_fp4): 128 rows x 64 K elements, codes then scales.
constexpr int kFp4BlockBytes = 4096 + 256;
// e8m0 scale bytes for which e2m1 x 2^(s-127) is exact in fp16 (subnormals included): the
// tensor-core 4-bit path dequantises into fp16.
constexpr int kFp4ScaleMin = 104;
constexpr int kFp4ScaleMax = 140;
cudaError_t launch_tile_fp4(const uint8_t* codes_a, const uint8_t* scales_a, const uint8_t* codes_b,
                            const uint8_t* scales_b, uint8_t* dst, int n, int rows, int K, int gate_up,
                            uint32_t* scale_oor, cudaStream_t st);
// Element offset of block (tile t, K chunk kc) inside one tile-contiguous weight matrix.
__host__ __device__ inline size_t tile_chunk_offset(int t, int kc, int tiles, int nk) {
  const int pr = t >> 1, w = t & 1;
  const int np = tiles - 2 * pr < 2 ? tiles - 2 * pr : 2;
  return (static_cast<size_t>(pr) * 2 * nk + static_cast<size_t>(kc) * np + w) * kTileElems;
}
// Elements between consecutive K chunks of tile t (2 blocks inside a pair, 1 for a lone tile).
__host__ __device__ inline size_t tile_chunk_stride(int t, int tiles) {
  return static_cast<size_t>(tiles - 2 * (t >> 1) < 2 ? 1 : 2) * kTileElems;
}
// Element offset of (row r, K element kk) inside one 128 x 64 block (128-byte swizzle).
__host__ __device__ inline size_t tile_elem_offset(int r, int kk) {
  return static_cast<size_t>(r) * 64 + ((((kk >> 3) ^ (r & 7)) << 3) | (kk & 7));
}

}  // namespace moe
