// Internal interfaces between the C-ABI layer (api.cu) and the kernel files.
#pragma once
#include <atomic>
#include <utility>
#include <cuda.h>

#include <algorithm>
#include <cstddef>
#include <cstdint>

#include "common.cuh"

namespace moe {

// Raises a kernel's dynamic shared-memory limit once per device (the
// attribute is per device, and a process may drive several GPUs).
// `done` is the caller's per-kernel table, indexed by device; its flags are
// atomic so host threads launching on one device concurrently are safe (at
// worst both set the attribute).
constexpr int kMaxDevices = 64;
inline cudaError_t set_smem_once(const void* kern, int bytes, std::atomic<bool> (&done)[kMaxDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool slot = dev >= 0 && dev < kMaxDevices;
  if (slot && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && slot) done[dev].store(true, std::memory_order_release);
  return e;
}

// Number of SMs of the current device, queried once per device (atomic
// cache, same thread-safety rule as set_smem_once). Grid sizes and split
// counts follow it instead of assuming a particular part.
inline int device_sms() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  const bool slot = dev >= 0 && dev < kMaxDevices;
  if (slot) {
    const int n = cache[dev].load(std::memory_order_acquire);
    if (n > 0) return n;
  }
  int n = 0;
  if (dev < 0 || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (slot) cache[dev].store(n, std::memory_order_release);
  return n;
}

// Launch with programmatic stream serialization (the kernel must start with
// pdl_enter(), see common.cuh).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
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
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}


constexpr int kTokBlk = 32;   // tokens per dispatch block (histogram / scatter)

// launch accounting (host side, per calling thread)
void note_launch();
void reset_launch_count();
int launch_count();

struct RouteArgs {
  int T, H, E, k, S;
  float rs;
  bool route;                 // false: ids/wts are inputs
  const float* part;          // logits partials [KS][T][E] (or logits [T][E], KS = 1)
  int KS;
  float* logits;              // [T][E] summed logits out (may equal part when KS == 1)
  int32_t *ids;
  float* wts;
  int32_t *counts, *offsets, *touched, *n_touched, *poff;
  int32_t *hist, *base;       // [NB][G] each (multi-block path)
  int32_t *perm, *inv;
  float* w_row;
  const uint16_t* x;          // nullable: skip quantisation
  uint8_t *xq, *xs;
  int32_t* status;
};

int router_splits(int T, int H, int E);
// Router partials (KS * T * E floats) up to this many are summed inside the
// fused routing kernel, staged in its shared memory; larger sets are summed
// by a grid-wide pass first.
constexpr int64_t kRouteStage = 16 * 1024;
bool use_small_route(int T, int G, int kp);
cudaError_t launch_router(const uint16_t* x, const float* Wr, int T, int H, int E, int KS, float* part,
                          cudaStream_t st);
cudaError_t launch_route_dispatch(const RouteArgs& a, cudaStream_t st);
cudaError_t launch_topk_only(const float* logits, int T, int E, int k, float rs, int32_t* ids, float* w,
                             int32_t* status, cudaStream_t st);
cudaError_t launch_quant_rows(const uint16_t* src, int rows, int C, uint8_t* q, uint8_t* s, cudaStream_t st);

// ---- grouped GEMM on tcgen05 (gemm_tc.cu) -------------------------------------
// Same result layout as GemmArgs: out[s][r][n] = rowf(n) * 2^act_rowexp[r] *
// sum_k W_e[n][k] * a16[r][k], with rowf = gs[e] (NVFP4) or 2^wrowexp (MXFP8);
// the f16 activation rows a16 [R][K] come in through a TMA descriptor.
struct TcArgs {
  const uint8_t* w;
  const float* gs;            // [G] (NVFP4) or nullptr
  const int8_t* wrowexp;      // [G][tiles][128] (MXFP8) or nullptr
  int64_t tile_bytes;
  int tiles;
  int N, K, fmt;
  int interleave_I;
  const int32_t* offsets;
  const int32_t* touched;
  const int32_t* n_touched;
  const int32_t* act_rowexp;  // [R]
  float* out;
  int64_t split_stride;
  int S;
  int max_ctas;
  int32_t* status;
};
// Tensor maps of the f16 operand rows a16 [rows, cols], viewed as
// (64 columns, rows, cols / 64 chunks): m[i] loads a box of 8 << i rows of
// two consecutive 64-column chunks in one copy (128-byte swizzle), stored
// chunk after chunk.
struct TcMaps {
  CUtensorMap m[4];
};
bool make_tmaps_b(TcMaps* maps, const void* base, int64_t rows, int64_t cols);
// nt: tokens per MMA tile (16, 32 or 64); tc_token_tile picks it from the
// average rows per group.
int tc_token_tile(int T, int kp, int G);
cudaError_t launch_gemm_tc(const TcArgs& g, const TcMaps& maps, int nt, cudaStream_t st);
// a16[r] = f16 rows of the MXFP8 rows q/s [*, C] at row_map[r] / row_div
// (or r), rowexp[r] = the row's largest block exponent.
cudaError_t launch_act_f16(const uint8_t* q, const uint8_t* s, int C, const int32_t* row_map, int row_div, int R,
                           const int32_t* offsets, int G, uint16_t* a16, int32_t* rowexp, cudaStream_t st);

// W1 epilogue: sums the S partials, y = w_row * act(g, u), MXFP8 along I.
struct W1FinArgs {
  const float* P; int S; int64_t split_stride;
  int R; int I;
  const int32_t* offsets; int G;      // offsets[G] = rows present
  const float* w_row;
  ActParams act;
  uint8_t* y1q; uint8_t* y1s;
  uint16_t* h_save;                   // nullable [R][2I] bf16
  float* y_save;                      // nullable [R][I] fp32
  uint16_t* y16;                      // [R][I] f16 rows for the W2 B operand
  int32_t* y_rowexp;                  // [R] row exponent of y16
};
cudaError_t launch_w1_finalize(const W1FinArgs& a, cudaStream_t st);

// out[t][n] = bf16(sum_j bf16(sum_s P[s][inv[t*kp+j]][n])); z (nullable) gets
// the per-row bf16 values.
cudaError_t launch_finalize_combine(const float* P, int S, int64_t split_stride, int N, const int32_t* inv, int T,
                                    int kp, uint16_t* z, uint16_t* out, cudaStream_t st);
// z [R][N] = bf16(sum_s P[s][r][n]) for r < R.
cudaError_t launch_finalize_rows(const float* P, int S, int64_t split_stride, int N, int R, uint16_t* z,
                                 cudaStream_t st);
// out[t] = bf16(sum_j c_j z[inv[t*kp+j]]) with c_j from topk_w (nullable).
cudaError_t launch_combine(const uint16_t* z, const int32_t* inv, const float* topk_w, int T, int k, int kp, int H,
                           uint16_t* out, cudaStream_t st);

// Transposed MXFP8 copy: for each group e and padded row p < pad(count_e),
// dst[c][poff[e] + p] = MXFP8 along p (blocks of 32) of the value of row
// offsets[e] + p (zero past count_e). Source rows: bf16 rows of src16 at
// row_map[r] / row_div (gather), or fp32 rows src32[r].
struct ColQuantArgs {
  const uint16_t* src16; const int32_t* row_map; int row_div;
  const float* src32;
  int C;
  const int32_t* offsets; const int32_t* poff; int G;
  int64_t r_pad_max;                  // row length of dst
  uint8_t* q; uint8_t* s;             // [C][r_pad_max], [C][r_pad_max/32]
};
cudaError_t launch_quant_cols(const ColQuantArgs& a, cudaStream_t st);

// ---- backward pieces ----------------------------------------------------------
struct DswigluArgs {
  const float* P; int S; int64_t split_stride;   // dY1 partials [S][R][I]
  int R, I;
  const int32_t* offsets; int G;
  const uint16_t* h;                  // saved bf16 [R][2I]
  const float* w_row;
  ActParams act;
  float* dw_row;                      // [R]
  uint8_t* dhq; uint8_t* dhs;         // [R][2I], [R][2I/32]
  float* dh;                          // [R][2I] fp32 (for the transposed copy)
};
cudaError_t launch_dswiglu(const DswigluArgs& a, cudaStream_t st);

struct WgradArgs {
  const uint8_t* pq; const uint8_t* ps;   // [M][Rp], [M][Rp/32]
  const uint8_t* qq; const uint8_t* qs;   // [N][Rp], [N][Rp/32]
  int64_t Rp;
  int M, N, G;
  const int32_t* poff;
  uint16_t* out;                          // [G][M][N] bf16
};
cudaError_t launch_wgrad(const WgradArgs& a, cudaStream_t st);

cudaError_t launch_router_bwd(const float* topk_w, const int32_t* ids, const float* dw_row, const int32_t* inv,
                              int T, int E, int k, int kp, float rs, float* dlogits, cudaStream_t st);

// ---- prepack ----------------------------------------------------------------
cudaError_t launch_prepack(const uint8_t* q, const uint8_t* s, int G, int N, int K, int fmt, int interleave_I,
                           int tiles, int64_t tile_bytes, uint8_t* dst, cudaStream_t st);
// MXFP8: per packed row, the largest E8M0 scale exponent (unbiased) of the
// logical row, int8 [G][tiles][128] (0 for padding rows).
cudaError_t launch_prepack_rowexp(const uint8_t* s, int G, int N, int K, int interleave_I, int tiles, int8_t* dst,
                                  cudaStream_t st);

}  // namespace moe
