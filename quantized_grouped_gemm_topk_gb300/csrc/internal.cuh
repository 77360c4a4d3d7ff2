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
  int32_t* zero;              // nullable: [nzero] ints cleared by the routing kernel
  int64_t nzero;              // (the partitioned layer's hand-off counters)
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
// Sums the router's KS split-K partials [KS][T][E] into logits (ks order)
// and routes each token: one block per token.
cudaError_t launch_sum_topk(const float* part, int KS, int T, int E, int k, float rs, float* logits, int32_t* ids,
                            float* w, int32_t* status, cudaStream_t st);
cudaError_t launch_quant_rows(const uint16_t* src, int rows, int C, uint8_t* q, uint8_t* s, cudaStream_t st);

// ---- NVFP4 grouped GEMM on tcgen05 (gemm_tc.cu) ---------------------------------
// out[s][r][n] = gs[e] * 2^act_rowexp[r] * sum_k W_e[n][k] * a16[r][k] over
// K slice s; the f16 activation rows a16 [R][K] come in through a TMA
// descriptor.
// One matrix of the decoding GEMM.
struct TcMat {
  const uint8_t* w;
  const float* gs;            // [G]
  int64_t tile_bytes;
  int tiles;
  int N, K;
  int interleave_I;
  const int32_t* act_rowexp;  // [R]
  float* out;                 // fp32 K-slice partials [S][R][N]
  int64_t split_stride;
  int S;
};
// The fused layer's W1 epilogue and hand-off (nmat == 2, W1 unsplit along
// K): each W1 tile's unit applies act * w and the MXFP8 requant to the
// tile's features; the last W1 tile of a group to finish converts the
// group's y1 rows to the f16 W2 operand (y16, y_rowexp) and sets the
// group's ready flag, which the W2 units of that group wait for.
struct TcFused {
  const float* w_row;         // [R]
  ActParams act;
  int I;
  uint8_t* y1q; uint8_t* y1s; // [R][I], [R][I / 32]
  uint16_t* y16;              // [R][I]
  int32_t* y_rowexp;          // [R]
  int32_t* cnt;               // [G] W1 tiles done, [G] ready flags, [G] ring flags; zero on entry
  const float* b1;            // [G][2I] W1 bias (gate then up), nullable
  // Partitioned layer: CTAs [0, n_disp) fill the token ring (the f16 W1
  // operand rows a16 and their exponents, gathered from the dispatched MXFP8
  // rows xq / xs by row_map / row_div) group by group and raise the group's
  // ring flag; the other CTAs run W1 -> W2. n_disp = 0: a16 is filled before
  // the launch.
  int n_disp;
  const uint8_t* xq; const uint8_t* xs;
  const int32_t* row_map; int row_div;
  uint16_t* a16; int32_t* a_rowexp;
};
struct TcArgs {
  TcMat m[2];                 // m[0]: the (first) matrix; m[1]: W2 of the fused layer
  int nmat;                   // 1: one grouped GEMM over m[0]; 2: W1 -> W2 fused layer
  const PackHeader* hdr;      // the packed blob's header (checked on entry)
  int which;                  // MOE_PACK_FORWARD / MOE_PACK_DGRAD expected in hdr
  int G;
  const int32_t* offsets;
  const int32_t* touched;
  const int32_t* n_touched;
  int max_ctas;
  int32_t* status;
  int split_rows;             // > 0: the walk takes groups in blocks of this many rows (a multiple of the token tile)
  int bias;                   // the blob carries a W1 bias (checked against its header)
  TcFused f;
};
// Largest I the fused layer takes (a lane of the group conversion holds
// I / 256 code words of a row in registers).
constexpr int kFusedMaxI = 2048;
// Ints of the fused layer's counters for G groups.
inline int64_t tc_fused_counters(int G) { return 3LL * G; }
constexpr int kTcBoxes = 5;   // activation boxes of 8, 16, 32, 64, 128 rows
// Tensor maps of the f16 operand rows a16 [rows, cols], viewed as
// (64 columns, rows, cols / 64 chunks): m[i] loads a box of 8 << i rows of
// two consecutive 64-column chunks in one copy (128-byte swizzle), stored
// chunk after chunk.
struct TcMaps {
  CUtensorMap m[2][kTcBoxes]; // per matrix (the fused layer's W2 reads y16)
};
bool make_tmaps_b(CUtensorMap (&m)[kTcBoxes], const void* base, int64_t rows, int64_t cols);
// nt: tokens per MMA tile (16, 32, 64 or 128); tc_token_tile picks it from the
// average rows per group.
int tc_token_tile(int T, int kp, int G);
cudaError_t launch_gemm_tc(const TcArgs& g, const TcMaps& maps, int nt, cudaStream_t st);
// a16[r] = f16 rows of the MXFP8 rows q/s [*, C] at row_map[r] / row_div
// (or r), rowexp[r] = the row's largest block exponent.
cudaError_t launch_debug_flag_wait(const int32_t* flag, long long limit_cycles, int32_t* status, cudaStream_t st);
// zero / nzero (nullable): ints the kernel also sets to zero (the fused
// layer's counters, cleared by the launch just before it).
cudaError_t launch_act_f16(const uint8_t* q, const uint8_t* s, int C, const int32_t* row_map, int row_div, int R,
                           const int32_t* offsets, int G, uint16_t* a16, int32_t* rowexp, cudaStream_t st,
                           int32_t* zero = nullptr, int64_t nzero = 0);

// ---- block-scaled MXFP8 grouped GEMM (gemm_mx.cu) ----------------------------
// D_e[m][n] = sum_k A[m][k] * B[n][k], both operands MXFP8 (E4M3 bytes,
// K-major, one E8M0 scale byte per 32 K). Token-side modes (W1, Plain,
// Dswiglu): group e's A rows are offsets[e] .. offsets[e+1] of the A buffer,
// its B rows b_rows_per_group * e + n. Wgrad: A rows are the M gradient
// rows, B rows the N gradient columns, and group e's K range is
// poff[e] .. poff[e+1] (token axis, padded to kPadRows per group).
// Every scale array the kernel reads, or writes for another GEMM, is in the
// SF4 layout (common.cuh) with ld = the array's row count.
enum { kMxW1 = 0, kMxPlain = 1, kMxDswiglu = 2, kMxWgrad = 3 };
struct MxArgs {
  int mode;
  const PackHeader* hdr;        // token-side modes: the weight blob's header (checked on entry); Wgrad: nullptr
  int which;                    // MOE_PACK_FORWARD / MOE_PACK_DGRAD expected in hdr
  int G;
  int K;                        // token-side modes: reduction length
  int n_tiles;                  // 192-column tiles per group
  int N;                        // valid output columns (W1: unused, see I)
  int M, m_tiles;               // Wgrad: gradient rows and their 128-row tiles
  int64_t b_rows_per_group;
  const int32_t* offsets;       // [G + 1] token rows per group
  const int32_t* poff;          // [G + 1] padded token rows per group
  const uint8_t* a_sf; int64_t a_sf_ld; int64_t a_rows;   // A scales, SF4 with ld = a_sf_ld; rows < a_rows exist
  const uint8_t* b_sf; int64_t b_sf_ld; int64_t b_rows;   // B scales, SF4
  int b_fp4;                    // B elements are E2M1 (MXFP4 weights), else E4M3
  int bias;                     // the blob carries a W1 bias (checked against its header)
  const float* b1;              // W1 mode (nullable): [G][2I] bias, gate then up
  int gated;                    // 1 = gate / up halves (W1: in each tile; dSwiGLU: h and dh of 2I a row),
                                // 0 = sReLU (W1: 192 plain features a tile; dActivation: h and dh of I a row)
  int64_t R;                    // token rows (A rows of the token-side modes)
  const float* w_row;           // [R] routing weight per row
  ActParams act;
  int I;
  uint8_t* yq;                  // W1: y1 codes [R][I]; Dswiglu: dh codes [R][2I]
  uint8_t* ys;                  // W1: y1 scales [R][I/32] (row-major)
  uint8_t* yst;                 // W1 (nullable): y1 scales again, SF4, ld R; Dswiglu: dh scales, SF4, ld R
  uint16_t* hsave;              // W1: h bf16 [R][2I] out (nullable); Dswiglu: h in
  uint8_t* tq; uint8_t* ts; int64_t t_ld; int t_nf;   // transposed MXFP8 copy: codes [t_nf][t_ld], scales SF4
                                                       // (K = t_ld, ld = t_nf); W1: nullable
  uint16_t* out; int64_t out_ld;            // Plain: [R][out_ld]; Wgrad: [G][M][out_ld]
  float* dwpart;                // Dswiglu: [n_tiles][R]
  float* dbpart;                // Dswiglu (nullable): [R_pad / 32][db_ld] column sums of dh over each
  int db_ld;                    //   padded 32-row block (the W1 bias gradient's partials)
  float* amax;                  // W1 (nullable): [2] max |y|, max |H16/4 . block of y^T| (zeroed by the caller)
  int32_t* status;
};
struct MxMaps {
  CUtensorMap a[4];             // A boxes of 128 K-elements x 16 << i rows (the tile's rows pick one)
  CUtensorMap b;                // B box of 128 K-elements x mx_b_box_rows() rows
  CUtensorMap sfb;              // B's SF4 scale words: boxes of one word x 192 rows
};
// Matrix [rows][cols elements] as a 2-D tensor map, boxes of 128 elements x
// box_rows rows, 128-byte swizzle, zero fill past the edges. fp4: packed
// E2M1 (two per byte in memory) unpacked to one element per byte in shared
// memory, the layout the block-scaled MMA reads; else one byte per element.
bool make_tmap_mx(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows, bool fp4);
bool make_tmaps_mx_a(MxMaps* maps, const void* base, int64_t rows, int64_t cols);
// SF4 scale words [words][ld] (uint32) of `rows` rows as a 2-D tensor map,
// boxes of one word x 192 rows; ld must be a multiple of 4.
bool make_tmap_mx_sf(CUtensorMap* map, const void* sf, int64_t rows, int64_t words, int64_t ld);
int mx_tile_n();
int mx_b_box_rows();          // rows of B per tensor copy (each CTA of a pair copies this many)
int mx_tile_m();
cudaError_t launch_gemm_mx(const MxArgs& g, const MxMaps& maps, int grid, cudaStream_t st);
// dst rows r < min(R, offsets[G]) = MXFP8 rows src[row_map[r] / row_div];
// the source scales are row-major [*][C/32], the destination's SF4 (ld R).
cudaError_t launch_gather_mx(const uint8_t* q, const uint8_t* s, int C, const int32_t* row_map, int row_div, int R,
                             const int32_t* offsets, int G, uint8_t* dq, uint8_t* ds, cudaStream_t st);
// Row-major scales [R][C/32] -> SF4 (ld R).
cudaError_t launch_sf_to_sf4(const uint8_t* s, int C, int64_t R, uint8_t* d, cudaStream_t st);

// W1 epilogue of the NVFP4 path: sums the S partials, y = w_row * act(g, u),
// MXFP8 along I, and the f16 operand rows of W2.
struct W1FinArgs {
  const float* P; int S; int64_t split_stride;
  int R; int I;
  const int32_t* offsets; int G;      // offsets[G] = rows present
  const float* w_row;
  ActParams act;
  uint8_t* y1q; uint8_t* y1s;
  uint16_t* y16;                      // [R][I] f16 rows for the W2 B operand
  int32_t* y_rowexp;                  // [R] row exponent of y16
  const float* b1;                    // [G][2I] W1 bias (gate then up), nullable
  int gated;                          // 0: sReLU, P holds I columns a row (no up half)
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
// q[c][poff[e] + p] = MXFP8 along p (blocks of 32) of the value of row
// offsets[e] + p (zero past count_e), its scales in the SF4 layout (K =
// the padded row axis, ld = C). Source rows: bf16 rows of src16 at
// row_map[r] / row_div.
struct ColQuantArgs {
  const uint16_t* src16; const int32_t* row_map; int row_div;
  int C;
  const int32_t* offsets; const int32_t* poff; int G;
  int64_t r_pad_max;                  // row length of dst
  uint8_t* q; uint8_t* s;             // [C][r_pad_max], SF4 [r_pad_max/128][C] words
};
cudaError_t launch_quant_cols(const ColQuantArgs& a, cudaStream_t st);

// ---- backward pieces ----------------------------------------------------------
// dlogits from the routing-weight gradients dw_row[r] = sum over p < nparts of
// dwpart[p * R + r] (added in p order).
// W1 bias gradient: db[e][c] = sum over group e's padded 32-row blocks b (in
// block order) of part[b][c], c < N; groups without rows get zeros.
cudaError_t launch_bias_grad(const float* part, int N, const int32_t* poff, int G, float* db, cudaStream_t st);

cudaError_t launch_router_bwd(const float* topk_w, const int32_t* ids, const float* dwpart, int nparts, int64_t R,
                              const int32_t* inv, int T, int E, int k, int kp, float rs, float* dlogits,
                              cudaStream_t st);

// ---- prepack (prepack.cu) ------------------------------------------------------
cudaError_t launch_prepack_nv(const uint8_t* q, const uint8_t* s, int G, int N, int K, int interleave_I, int tiles,
                              int64_t tile_bytes, uint8_t* dst, cudaStream_t st);
cudaError_t launch_unpack_nv(const uint8_t* src, int G, int N, int K, int interleave_I, int tiles, int64_t tile_bytes,
                             uint8_t* q, uint8_t* s, cudaStream_t st);
// MXFP8 / MXFP4 rows: cb = code bytes per row (K, or K/2 for packed E2M1).
cudaError_t launch_prepack_mx(const uint8_t* q, const uint8_t* s, int G, int N, int K, int64_t cb, int interleave_I,
                              int NR, uint8_t* dq, uint8_t* ds, cudaStream_t st);
cudaError_t launch_unpack_mx(const uint8_t* dq, const uint8_t* ds, int G, int N, int K, int64_t cb, int interleave_I,
                             int NR, uint8_t* q, uint8_t* s, cudaStream_t st);

}  // namespace moe
