// C ABI of the routed-MoE layer: argument checks, workspace carving, and the
// launch sequence of each step. No allocation, no host sync (except
// moe_read_status): every call only enqueues kernels / async copies on the
// caller's stream.
#include <cstring>

#include "internal.cuh"

namespace moe {

static thread_local int g_launches = 0;
static thread_local cudaEvent_t g_phase[MOE_N_PHASE_EVENTS] = {};
static thread_local bool g_phase_on = false;
// Records phase event i on st. Under stream capture the record becomes an
// event-record node of the graph (a plain record there would only express a
// dependency), so each replay of the graph re-records the event.
static inline void phase(int i, cudaStream_t st) {
  if (!g_phase_on || !g_phase[i]) return;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(g_phase[i], st, cudaEventRecordExternal);
  else
    cudaEventRecord(g_phase[i], st);
}
void note_launch() { ++g_launches; }
void reset_launch_count() { g_launches = 0; }
int launch_count() { return g_launches; }

static inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Dims {
  int H, I, E, k, S, kp, G, Tmax;
  int64_t Rmax, RpMax;
};

static Dims dims_of(const moe_config_t& c) {
  Dims d;
  d.H = c.H; d.I = c.I; d.E = c.E; d.k = c.k; d.S = c.n_shared;
  d.kp = c.k + c.n_shared; d.G = c.E + c.n_shared; d.Tmax = c.T_max;
  d.Rmax = (int64_t)c.T_max * d.kp;
  d.RpMax = (int64_t)align_up((size_t)(d.Rmax + (kPadRows - 1LL) * d.G), kPadRows);
  return d;
}

static int64_t r_pad_for(const Dims& d, int T) {
  return (int64_t)align_up((size_t)((int64_t)T * d.kp + (kPadRows - 1LL) * d.G), kPadRows);
}

// W1 with gate and up halves (2I outputs); sReLU's W1 has I outputs.
static bool gated(const moe_config_t& c) { return c.act != MOE_ACT_SRELU; }

static bool backward_capable(const moe_config_t& c) {
  return c.weight_fmt == MOE_WFMT_MXFP8 && c.n_shared == 0;
}

// MXFP8 weights run on the block-scaled tensor-core GEMM (gemm_mx.cu); NVFP4
// weights on the decoding GEMM (gemm_tc.cu).
static bool mx_path(const moe_config_t& c) { return c.weight_fmt == MOE_WFMT_MXFP8 || c.weight_fmt == MOE_WFMT_MXFP4; }

// Code bytes of one packed row of K elements.
static int64_t row_bytes(int fmt, int K) { return fmt == MOE_WFMT_MXFP4 ? K / 2 : K; }

static int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ---- workspace layout -------------------------------------------------------
struct WsLayout {
  size_t status, logits, rpart, ids, wts, counts, offsets, touched, ntouch, poff, hist, base;
  size_t perm, inv, wrow, xq, xs, y1q, y1s, z;
  size_t P, a16, y16, rexp1, rexp2, P2, fcnt;            // NVFP4 path (P2, fcnt: the fused layer)
  size_t xg, xgs, y1st;                                   // MXFP8 path: gathered x rows, y1 scales (SF4)
  size_t dzq, dzs, dzg, dzgs, dztq, dzts, dhq, dhs, dhtq, dhts, dxp, dwpart;   // backward
  size_t dbpart;                                          // backward with a W1 bias
  size_t total;
};

static WsLayout ws_layout(const moe_config_t& c) {
  const Dims d = dims_of(c);
  WsLayout L;
  std::memset(&L, 0, sizeof(L));
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + std::max<size_t>(bytes, 1), 256); return at; };
  const int64_t T = d.Tmax, R = d.Rmax;
  const int NB = (int)((T + kTokBlk - 1) / kTokBlk);
  const int64_t rpart_rows = std::max<int64_t>(4096, T);     // KS * T <= max(4096, T)
  L.status = take(256);
  L.logits = take((size_t)T * d.E * 4);
  L.rpart = take((size_t)rpart_rows * d.E * 4);
  L.ids = take((size_t)T * d.k * 4);
  L.wts = take((size_t)T * d.k * 4);
  L.counts = take((size_t)d.G * 4);
  L.offsets = take((size_t)(d.G + 1) * 4);
  L.touched = take((size_t)d.G * 4);
  L.ntouch = take(4);
  L.poff = take((size_t)(d.G + 1) * 4);
  L.hist = take((size_t)NB * d.G * 4);
  L.base = take((size_t)NB * d.G * 4);
  L.perm = take((size_t)R * 4);
  L.inv = take((size_t)R * 4);
  L.wrow = take((size_t)R * 4);
  L.xq = take((size_t)T * d.H);
  L.xs = take((size_t)T * d.H / 32);
  L.y1q = take((size_t)R * d.I);
  L.y1s = take((size_t)R * d.I / 32);
  L.z = take((size_t)R * d.H * 2);
  if (!mx_path(c)) {
    L.P = take((size_t)R * std::max(2 * d.I, d.H) * 4);
    L.a16 = take((size_t)R * std::max(2 * d.I, d.H) * 2);
    L.y16 = take((size_t)R * d.I * 2);
    L.rexp1 = take((size_t)R * 4);
    L.rexp2 = take((size_t)R * 4);
    L.P2 = take((size_t)R * d.H * 4);
    L.fcnt = take((size_t)tc_fused_counters(d.G) * 4);
  } else {
    L.xg = take((size_t)R * d.H);
    L.xgs = take((size_t)sf4_bytes(d.H, R));
    L.y1st = take((size_t)sf4_bytes(d.I, R));
  }
  if (backward_capable(c)) {
    L.dzq = take((size_t)T * d.H);
    L.dzs = take((size_t)T * d.H / 32);
    L.dzg = take((size_t)R * d.H);
    L.dzgs = take((size_t)sf4_bytes(d.H, R));
    L.dztq = take((size_t)d.H * d.RpMax);
    L.dzts = take((size_t)sf4_bytes(d.RpMax, d.H));
    L.dhq = take((size_t)R * 2 * d.I);
    L.dhs = take((size_t)sf4_bytes(2 * d.I, R));
    L.dhtq = take((size_t)2 * d.I * d.RpMax);
    L.dhts = take((size_t)sf4_bytes(d.RpMax, 2 * d.I));
    L.dxp = take((size_t)R * d.H * 2);
    L.dwpart = take((size_t)ceil_div(d.I, kMxTileN) * R * 4);
    if (c.w1_bias) L.dbpart = take((size_t)(d.RpMax / 32) * 2 * d.I * 4);   // bias gradient partials
  }
  L.total = o;
  return L;
}

template <typename Tp>
static Tp* at(void* ws, size_t off) { return reinterpret_cast<Tp*>(reinterpret_cast<uint8_t*>(ws) + off); }

// ---- packed weights layout ------------------------------------------------------
struct PackLayout {
  int fmt, G;
  int N1, K1, N2, K2, il1;
  // NVFP4: 128-row tiles of 64-wide K chunks
  int tiles1, tiles2;
  int64_t tile_bytes1, tile_bytes2;
  size_t off_gs1, off_gs2;
  // MXFP8: plain rows
  int rows1, rows2;
  size_t off_s1, off_s2;
  size_t off_w1, off_w2, total;
  size_t off_b1;   // W1 bias [G][2I] fp32 (forward packs of configs with w1_bias), 0 for none
};

static PackLayout pack_layout(const moe_config_t& c, int which) {
  PackLayout P;
  std::memset(&P, 0, sizeof(P));
  P.fmt = c.weight_fmt;
  P.G = c.E + c.n_shared;
  if (which == MOE_PACK_FORWARD) {
    P.N1 = gated(c) ? 2 * c.I : c.I; P.K1 = c.H; P.il1 = gated(c) ? c.I : 0;
    P.N2 = c.H; P.K2 = c.I;
  } else {
    P.N1 = c.H; P.K1 = gated(c) ? 2 * c.I : c.I; P.il1 = 0;
    P.N2 = c.I; P.K2 = c.H;
  }
  size_t o = 256;
  if (P.fmt == MOE_WFMT_NVFP4) {
    const int CB = chunk_bytes(P.fmt);
    P.tiles1 = (P.N1 + kTileN - 1) / kTileN;
    P.tiles2 = (P.N2 + kTileN - 1) / kTileN;
    P.tile_bytes1 = (int64_t)(P.K1 / kChunkK) * CB;
    P.tile_bytes2 = (int64_t)(P.K2 / kChunkK) * CB;
    P.off_gs1 = o; o = align_up(o + (size_t)P.G * 4, 256);
    P.off_gs2 = o; o = align_up(o + (size_t)P.G * 4, 256);
    P.off_w1 = o; o = align_up(o + (size_t)P.G * P.tiles1 * P.tile_bytes1, 256);
    P.off_w2 = o; o = align_up(o + (size_t)P.G * P.tiles2 * P.tile_bytes2, 256);
  } else {
    P.rows1 = P.il1 > 0 ? ceil_div(P.il1, kMxTileN / 2) * kMxTileN : P.N1;
    P.rows2 = P.N2;
    P.off_w1 = o; o = align_up(o + (size_t)P.G * P.rows1 * row_bytes(P.fmt, P.K1), 256);
    P.off_s1 = o; o = align_up(o + (size_t)sf4_bytes(P.K1, (int64_t)P.G * P.rows1), 256);
    P.off_w2 = o; o = align_up(o + (size_t)P.G * P.rows2 * row_bytes(P.fmt, P.K2), 256);
    P.off_s2 = o; o = align_up(o + (size_t)sf4_bytes(P.K2, (int64_t)P.G * P.rows2), 256);
  }
  if (c.w1_bias && which == MOE_PACK_FORWARD) {
    P.off_b1 = o; o = align_up(o + (size_t)P.G * 2 * c.I * 4, 256);
  }
  P.total = o;
  return P;
}

__global__ void k_write_header(PackHeader h, uint8_t* dst) { *reinterpret_cast<PackHeader*>(dst) = h; }

// out[i] = sum over ks of part[ks * n + i], added in ks order; 16 loads in
// flight per thread.
__global__ void k_reduce_partials(const float* part, int KS, int64_t n, float* out) {
  pdl_enter();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    float v = part[i];
    int ks = 1;
    for (; ks + 16 <= KS; ks += 16) {
      float t[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) t[j] = part[(int64_t)(ks + j) * n + i];
#pragma unroll
      for (int j = 0; j < 16; ++j) v += t[j];
    }
    for (; ks < KS; ++ks) v += part[(int64_t)ks * n + i];
    out[i] = v;
  }
}


}  // namespace moe

using namespace moe;

#define MOE_CHECK_CUDA(x)                        \
  do {                                           \
    cudaError_t _e = (x);                        \
    if (_e != cudaSuccess) return MOE_ERR_CUDA;  \
  } while (0)

static inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
#define REQ(p) do { if (!(p) || !aligned16(p)) return MOE_ERR_INVALID_ARG; } while (0)
#define OPT(p) do { if ((p) && !aligned16(p)) return MOE_ERR_INVALID_ARG; } while (0)
// buffers whose size scales with T may be NULL when T == 0
#define REQ_T(p) do { if (T > 0) REQ(p); else OPT(p); } while (0)

extern "C" {

moe_status_t moe_config_validate(const moe_config_t* c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->H <= 0 || c->I <= 0 || c->H % 64 || c->I % 64) return MOE_ERR_INVALID_ARG;
  if (c->E <= 0 || c->k < 1 || c->k > c->E) return MOE_ERR_INVALID_ARG;
  if (c->n_shared < 0 || c->n_shared > 1) return MOE_ERR_INVALID_ARG;
  if (c->k + c->n_shared > 32 || c->E + c->n_shared > 2048) return MOE_ERR_INVALID_ARG;
  if (c->T_max < 0) return MOE_ERR_INVALID_ARG;
  if (c->act != MOE_ACT_SWIGLU && c->act != MOE_ACT_SWIGLU_CLAMP && c->act != MOE_ACT_GEGLU &&
      c->act != MOE_ACT_SRELU)
    return MOE_ERR_INVALID_ARG;
  if (c->act == MOE_ACT_SWIGLU_CLAMP && !(c->act_limit > 0.f)) return MOE_ERR_INVALID_ARG;
  if (c->weight_fmt != MOE_WFMT_NVFP4 && c->weight_fmt != MOE_WFMT_MXFP8 && c->weight_fmt != MOE_WFMT_MXFP4)
    return MOE_ERR_INVALID_ARG;
  // the unpacking tensor copy of E2M1 rows moves whole 128-element runs
  if (c->weight_fmt == MOE_WFMT_MXFP4 && (c->H % 128 || c->I % 128)) return MOE_ERR_INVALID_ARG;
  if (!(c->routed_scale > 0.f)) return MOE_ERR_INVALID_ARG;
  if (c->max_sms < 0) return MOE_ERR_INVALID_ARG;
  if (c->w1_bias != 0 && c->w1_bias != 1) return MOE_ERR_INVALID_ARG;
  if (c->dispatch_sms < 0 || c->dispatch_sms > 64) return MOE_ERR_INVALID_ARG;
  if (c->w1_bias && c->act == MOE_ACT_SRELU) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

moe_status_t moe_workspace_size(const moe_config_t* c, size_t* bytes) {
  moe_status_t s = moe_config_validate(c);
  if (s != MOE_OK) return s;
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(*c).total;
  return MOE_OK;
}

moe_status_t moe_workspace_view(const moe_config_t* c, void* ws, moe_ws_view_t* v) {
  moe_status_t s = moe_config_validate(c);
  if (s != MOE_OK) return s;
  if (!v) return MOE_ERR_INVALID_ARG;
  REQ(ws);
  const WsLayout L = ws_layout(*c);
  v->logits = at<float>(ws, L.logits);
  v->d.topk_ids = at<int32_t>(ws, L.ids);
  v->d.topk_w = at<float>(ws, L.wts);
  v->d.counts = at<int32_t>(ws, L.counts);
  v->d.offsets = at<int32_t>(ws, L.offsets);
  v->d.perm_src = at<int32_t>(ws, L.perm);
  v->d.inv = at<int32_t>(ws, L.inv);
  v->d.w_row = at<float>(ws, L.wrow);
  v->d.xq = at<uint8_t>(ws, L.xq);
  v->d.xs = at<uint8_t>(ws, L.xs);
  v->y1_q = at<uint8_t>(ws, L.y1q);
  v->y1_s = at<uint8_t>(ws, L.y1s);
  v->z = at<uint16_t>(ws, L.z);
  v->status = at<int32_t>(ws, L.status);
  return MOE_OK;
}

moe_status_t moe_packed_weights_size(const moe_config_t* c, int which, size_t* bytes) {
  moe_status_t s = moe_config_validate(c);
  if (s != MOE_OK) return s;
  if (!bytes || (which != MOE_PACK_FORWARD && which != MOE_PACK_DGRAD)) return MOE_ERR_INVALID_ARG;
  if (which == MOE_PACK_DGRAD && c->weight_fmt != MOE_WFMT_MXFP8) return MOE_ERR_UNSUPPORTED;
  *bytes = pack_layout(*c, which).total;
  return MOE_OK;
}

moe_status_t moe_train_sizes(const moe_config_t* c, int T, int64_t* r_pad_max) {
  moe_status_t s = moe_config_validate(c);
  if (s != MOE_OK) return s;
  if (!r_pad_max || T < 0 || T > c->T_max) return MOE_ERR_INVALID_ARG;
  *r_pad_max = r_pad_for(dims_of(*c), T);
  return MOE_OK;
}

moe_status_t moe_prepack_weights(const moe_config_t* c, const moe_weights_view_t* src, int which, void* dst,
                                 size_t dst_bytes, void* stream) {
  moe_status_t s = moe_config_validate(c);
  if (s != MOE_OK) return s;
  if (!src || (which != MOE_PACK_FORWARD && which != MOE_PACK_DGRAD)) return MOE_ERR_INVALID_ARG;
  if (which == MOE_PACK_DGRAD && c->weight_fmt != MOE_WFMT_MXFP8) return MOE_ERR_UNSUPPORTED;
  REQ(dst); REQ(src->w1_q); REQ(src->w1_s); REQ(src->w2_q); REQ(src->w2_s);
  if (c->weight_fmt == MOE_WFMT_NVFP4) { REQ(src->w1_gs); REQ(src->w2_gs); }
  if (c->w1_bias && which == MOE_PACK_FORWARD) REQ(src->b1);
  const PackLayout P = pack_layout(*c, which);
  if (dst_bytes < P.total) return MOE_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  reset_launch_count();
  uint8_t* d8 = reinterpret_cast<uint8_t*>(dst);
  PackHeader h;
  std::memset(&h, 0, sizeof(h));
  h.magic = kPackMagic; h.version = kPackVersion; h.fmt = P.fmt; h.which = which; h.G = P.G;
  h.N1 = P.N1; h.K1 = P.K1; h.N2 = P.N2; h.K2 = P.K2; h.interleave1 = P.il1;
  h.off_gs1 = P.off_gs1; h.off_gs2 = P.off_gs2; h.off_w1 = P.off_w1; h.off_w2 = P.off_w2;
  h.tile_bytes1 = P.tile_bytes1; h.tile_bytes2 = P.tile_bytes2; h.tiles1 = P.tiles1; h.tiles2 = P.tiles2;
  h.off_s1 = P.off_s1; h.off_s2 = P.off_s2; h.rows1 = P.rows1; h.rows2 = P.rows2;
  h.off_b1 = (int64_t)P.off_b1;
  k_write_header<<<1, 1, 0, st>>>(h, d8);
  note_launch();
  MOE_CHECK_CUDA(cudaGetLastError());
  if (c->weight_fmt == MOE_WFMT_NVFP4) {
    MOE_CHECK_CUDA(cudaMemcpyAsync(d8 + P.off_gs1, src->w1_gs, (size_t)P.G * 4, cudaMemcpyDeviceToDevice, st));
    MOE_CHECK_CUDA(cudaMemcpyAsync(d8 + P.off_gs2, src->w2_gs, (size_t)P.G * 4, cudaMemcpyDeviceToDevice, st));
    MOE_CHECK_CUDA(launch_prepack_nv(src->w1_q, src->w1_s, P.G, P.N1, P.K1, P.il1, P.tiles1, P.tile_bytes1,
                                     d8 + P.off_w1, st));
    MOE_CHECK_CUDA(launch_prepack_nv(src->w2_q, src->w2_s, P.G, P.N2, P.K2, 0, P.tiles2, P.tile_bytes2,
                                     d8 + P.off_w2, st));
  } else {
    MOE_CHECK_CUDA(launch_prepack_mx(src->w1_q, src->w1_s, P.G, P.N1, P.K1, row_bytes(P.fmt, P.K1), P.il1, P.rows1,
                                     d8 + P.off_w1, d8 + P.off_s1, st));
    MOE_CHECK_CUDA(launch_prepack_mx(src->w2_q, src->w2_s, P.G, P.N2, P.K2, row_bytes(P.fmt, P.K2), 0, P.rows2,
                                     d8 + P.off_w2, d8 + P.off_s2, st));
  }
  if (P.off_b1)
    MOE_CHECK_CUDA(cudaMemcpyAsync(d8 + P.off_b1, src->b1, (size_t)P.G * 2 * c->I * 4, cudaMemcpyDeviceToDevice,
                                   st));
  return MOE_OK;
}

moe_status_t moe_debug_unpack_weights(const moe_config_t* c, const void* packed, int which, int mat, uint8_t* q,
                                      uint8_t* sc, void* stream) {
  moe_status_t s = moe_config_validate(c);
  if (s != MOE_OK) return s;
  if ((which != MOE_PACK_FORWARD && which != MOE_PACK_DGRAD) || (mat != 1 && mat != 2)) return MOE_ERR_INVALID_ARG;
  if (which == MOE_PACK_DGRAD && c->weight_fmt != MOE_WFMT_MXFP8) return MOE_ERR_UNSUPPORTED;
  REQ(packed); REQ(q); REQ(sc);
  const PackLayout P = pack_layout(*c, which);
  cudaStream_t st = (cudaStream_t)stream;
  reset_launch_count();
  const uint8_t* b = reinterpret_cast<const uint8_t*>(packed);
  const int N = mat == 1 ? P.N1 : P.N2, K = mat == 1 ? P.K1 : P.K2, il = mat == 1 ? P.il1 : 0;
  if (c->weight_fmt == MOE_WFMT_NVFP4) {
    MOE_CHECK_CUDA(launch_unpack_nv(b + (mat == 1 ? P.off_w1 : P.off_w2), P.G, N, K, il,
                                    mat == 1 ? P.tiles1 : P.tiles2, mat == 1 ? P.tile_bytes1 : P.tile_bytes2, q, sc,
                                    st));
  } else {
    MOE_CHECK_CUDA(launch_unpack_mx(b + (mat == 1 ? P.off_w1 : P.off_w2), b + (mat == 1 ? P.off_s1 : P.off_s2), P.G,
                                    N, K, row_bytes(P.fmt, K), il, mat == 1 ? P.rows1 : P.rows2, q, sc, st));
  }
  return MOE_OK;
}

static moe_status_t check_T(const moe_config_t* c, int T) {
  moe_status_t s = moe_config_validate(c);
  if (s != MOE_OK) return s;
  if (T < 0 || T > c->T_max) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

moe_status_t moe_router_logits(const moe_config_t* c, const uint16_t* x, const float* W_r, int T, float* logits,
                               void* ws, void* stream) {
  moe_status_t s = check_T(c, T);
  if (s != MOE_OK) return s;
  REQ_T(x); REQ(W_r); REQ_T(logits); REQ(ws);
  cudaStream_t st = (cudaStream_t)stream;
  reset_launch_count();
  const WsLayout L = ws_layout(*c);
  const int KS = router_splits(T, c->H, c->E);
  if (KS == 1) {
    MOE_CHECK_CUDA(launch_router(x, W_r, T, c->H, c->E, 1, logits, st));
    return MOE_OK;
  }
  float* part = at<float>(ws, L.rpart);
  MOE_CHECK_CUDA(launch_router(x, W_r, T, c->H, c->E, KS, part, st));
  if (T > 0) {
    const int64_t n = (int64_t)T * c->E;
    k_reduce_partials<<<(int)std::min<int64_t>((n + 255) / 256, 4096), 256, 0, st>>>(part, KS, n, logits);
    note_launch();
    MOE_CHECK_CUDA(cudaGetLastError());
  }
  return MOE_OK;
}

static RouteArgs route_args(const moe_config_t* c, int T, const moe_dispatch_t* d, void* ws, const WsLayout& L) {
  RouteArgs a;
  a.T = T; a.H = c->H; a.E = c->E; a.k = c->k; a.S = c->n_shared; a.rs = c->routed_scale;
  a.route = true; a.part = nullptr; a.KS = 1; a.logits = nullptr;
  a.ids = d->topk_ids; a.wts = d->topk_w; a.counts = d->counts; a.offsets = d->offsets;
  a.touched = at<int32_t>(ws, L.touched); a.n_touched = at<int32_t>(ws, L.ntouch); a.poff = at<int32_t>(ws, L.poff);
  a.hist = at<int32_t>(ws, L.hist); a.base = at<int32_t>(ws, L.base);
  a.perm = d->perm_src; a.inv = d->inv; a.w_row = d->w_row;
  a.x = nullptr; a.xq = d->xq; a.xs = d->xs;
  a.status = at<int32_t>(ws, L.status);
  a.zero = nullptr; a.nzero = 0;
  return a;
}

static moe_status_t check_dispatch(const moe_dispatch_t* d, bool need_x, int T) {
  if (!d) return MOE_ERR_INVALID_ARG;
  REQ_T(d->topk_ids); REQ_T(d->topk_w); REQ(d->counts); REQ(d->offsets); REQ_T(d->perm_src); REQ_T(d->inv);
  REQ_T(d->w_row);
  if (need_x) { REQ_T(d->xq); REQ_T(d->xs); }
  return MOE_OK;
}

moe_status_t moe_route_topk(const moe_config_t* c, const float* logits, int T, int32_t* ids, float* w, void* ws,
                            void* stream) {
  moe_status_t s = check_T(c, T);
  if (s != MOE_OK) return s;
  REQ_T(logits); REQ_T(ids); REQ_T(w); REQ(ws);
  reset_launch_count();
  const WsLayout L = ws_layout(*c);
  MOE_CHECK_CUDA(launch_topk_only(logits, T, c->E, c->k, c->routed_scale, ids, w, at<int32_t>(ws, L.status),
                                  (cudaStream_t)stream));
  return MOE_OK;
}

moe_status_t moe_route_dispatch(const moe_config_t* c, const float* logits, const uint16_t* x, int T,
                                const moe_dispatch_t* d, void* ws, void* stream) {
  moe_status_t s = check_T(c, T);
  if (s != MOE_OK) return s;
  REQ_T(logits); REQ_T(x); REQ(ws);
  if ((s = check_dispatch(d, true, T)) != MOE_OK) return s;
  reset_launch_count();
  const WsLayout L = ws_layout(*c);
  RouteArgs a = route_args(c, T, d, ws, L);
  a.part = logits; a.KS = 1; a.logits = const_cast<float*>(logits); a.x = x;
  MOE_CHECK_CUDA(launch_route_dispatch(a, (cudaStream_t)stream));
  return MOE_OK;
}

moe_status_t moe_dispatch(const moe_config_t* c, const uint16_t* x, int T, const moe_dispatch_t* d, void* ws,
                          void* stream) {
  moe_status_t s = check_T(c, T);
  if (s != MOE_OK) return s;
  REQ_T(x); REQ(ws);
  if ((s = check_dispatch(d, true, T)) != MOE_OK) return s;
  reset_launch_count();
  const WsLayout L = ws_layout(*c);
  RouteArgs a = route_args(c, T, d, ws, L);
  a.route = false; a.x = x;
  MOE_CHECK_CUDA(launch_route_dispatch(a, (cudaStream_t)stream));
  return MOE_OK;
}

// K slices for the tcgen05 GEMM (one CTA per SM): about eight units per CTA
// for load balance, each unit at least eight 64-wide K chunks long, and
// S * R within the partial buffer.
static int tc_splits(const moe_config_t& c, int T, int tiles, int K, int grid) {
  const Dims d = dims_of(c);
  const double touched = c.E * (1.0 - std::pow(1.0 - (double)c.k / c.E, (double)T)) + c.n_shared;
  const double units = std::max(1.0, touched) * tiles;
  // about 8 units per CTA, each K slice at least 8 chunks (4 pairs)
  int S = (int)std::lround(8.0 * grid / units);
  S = std::min(S, std::max(1, K / kChunkK / 8));
  const int64_t R = std::max<int64_t>(1, (int64_t)T * d.kp);
  S = (int)std::min<int64_t>(S, std::max<int64_t>(1, d.Rmax / R));
  return std::max(1, std::min(S, 64));   // the GEMM stages at most 64 K-slice boundaries
}

struct TcRun {
  float* out;
  int64_t split_stride;
  int S;
};

// The fused layer (NVFP4 weights, small decode batches: at most 2 rows per
// group on average): W1, its epilogue and W2 in one persistent launch. It
// removes the W1 epilogue kernel and the W1 -> W2 launch boundary, which
// dominate at a few tokens; with more rows per group the per-tile epilogue
// work inside the kernel (each W1 tile's activation and requant, each
// group's conversion to the W2 operand) costs more than the boundary it
// saves (measured on the DeepSeek-V3 shape: -7 us at T = 1, even at T = 8
// and 32, +13 us at T = 128), and the separate kernels run instead.
static bool fused_layer(const moe_config_t& c, int T) {
  const int64_t R = (int64_t)T * (c.k + c.n_shared);
  return !mx_path(c) && gated(c) && T > 0 && R <= 2LL * (c.E + c.n_shared) && c.I <= kFusedMaxI;
}

// The decoding GEMM's fields shared by its matrices.
static void tc_common(TcArgs& g, const moe_config_t* c, const PackLayout& P, const void* packed, void* ws,
                      const WsLayout& L, const int32_t* offsets) {
  std::memset(&g, 0, sizeof(g));
  g.hdr = reinterpret_cast<const PackHeader*>(packed);
  g.which = MOE_PACK_FORWARD;
  g.G = P.G;
  g.offsets = offsets;
  g.touched = at<int32_t>(ws, L.touched);
  g.n_touched = at<int32_t>(ws, L.ntouch);
  int sms = device_sms();
  if (c->max_sms > 0) sms = std::min(sms, c->max_sms);
  g.max_ctas = sms;
  g.status = at<int32_t>(ws, L.status);
  g.bias = c->w1_bias;
}

// Packed matrix `mat` (1 or 2) of `packed` as one matrix of the decoding
// GEMM: B operand rows with exponents rexp, fp32 K-slice partials into out.
static TcMat tc_mat(const moe_config_t* c, const PackLayout& P, int mat, const void* packed, int T,
                    const int32_t* rexp, float* out, int sms) {
  TcMat m;
  std::memset(&m, 0, sizeof(m));
  const uint8_t* b = reinterpret_cast<const uint8_t*>(packed);
  if (mat == 1) {
    m.w = b + P.off_w1; m.gs = reinterpret_cast<const float*>(b + P.off_gs1);
    m.tile_bytes = P.tile_bytes1; m.tiles = P.tiles1; m.N = P.N1; m.K = P.K1; m.interleave_I = P.il1;
  } else {
    m.w = b + P.off_w2; m.gs = reinterpret_cast<const float*>(b + P.off_gs2);
    m.tile_bytes = P.tile_bytes2; m.tiles = P.tiles2; m.N = P.N2; m.K = P.K2; m.interleave_I = 0;
  }
  m.act_rowexp = rexp;
  m.out = out;
  const int64_t R = (int64_t)T * (c->k + c->n_shared);
  m.split_stride = R * m.N;
  // The fused layer runs both matrices unsplit: W1's tiles then need no
  // other CTA's partials, W2's units balance the load of W1's last round,
  // and W2's units stay long enough to hide the per-unit check of their
  // group's flag. The separate calls at those sizes split the same way, so
  // the layer and its steps give the same bits.
  m.S = fused_layer(*c, T) ? 1 : tc_splits(*c, T, m.tiles, m.K, sms);
  return m;
}

// One grouped GEMM over packed matrix `mat` (1 or 2) of `packed`, B operand
// the f16 rows a16 [T*k', K] with exponents rexp; fp32 K-slice partials into
// the workspace buffer P.
static moe_status_t tc_gemm(const moe_config_t* c, const PackLayout& P, int mat, const void* packed, void* ws,
                            const WsLayout& L, const int32_t* offsets, int T, const uint16_t* a16,
                            const int32_t* rexp, cudaStream_t st, TcRun* run) {
  TcArgs g;
  tc_common(g, c, P, packed, ws, L, offsets);
  g.nmat = 1;
  g.m[0] = tc_mat(c, P, mat, packed, T, rexp, at<float>(ws, L.P), g.max_ctas);
  const int64_t R = (int64_t)T * (c->k + c->n_shared);
  int nt = tc_token_tile(T, c->k + c->n_shared, c->E + c->n_shared);
  // 128-token tiles halve the weight decoding per FLOP, but with one MMA
  // issuer and two accumulators they pay off only on long K (measured on
  // the skewed prefill: W1, K = 4096, 1180 -> 1044 us; W2, K = 1536,
  // 668 -> 826 us)
  if (nt == 128 && g.m[0].K < 4096) nt = 64;
  // prefill-sized groups: units of at most 8 token tiles, so a hot group's
  // rows spread over many CTAs
  g.split_rows = nt >= 128 ? 4 * nt : nt >= 32 ? 8 * nt : 0;
  TcMaps maps;
  if (!make_tmaps_b(maps.m[0], a16, R, g.m[0].K)) return MOE_ERR_CUDA;
  std::memcpy(&maps.m[1], &maps.m[0], sizeof(maps.m[0]));
  MOE_CHECK_CUDA(launch_gemm_tc(g, maps, nt, st));
  run->out = g.m[0].out;
  run->split_stride = g.m[0].split_stride;
  run->S = g.m[0].S;
  return MOE_OK;
}

static int mx_grid(const moe_config_t& c) {
  int s = device_sms();
  if (c.max_sms > 0) s = std::min(s, c.max_sms);
  return s;
}

// Token-side block-scaled GEMM (modes kMxW1, kMxPlain, kMxDswiglu): A = the
// MXFP8 rows aq [R][K] in group order with scales as (SF4, ld R), B =
// matrix `mat` of the packed MXFP8 blob; g carries the epilogue fields.
static moe_status_t mx_token_gemm(const moe_config_t* c, MxArgs& g, int mode, const uint8_t* aq, const uint8_t* as,
                                  int64_t R, const void* packed, int which, int mat, const int32_t* offsets,
                                  const int32_t* poff, int32_t* status, cudaStream_t st) {
  const PackLayout P = pack_layout(*c, which);
  const uint8_t* b = reinterpret_cast<const uint8_t*>(packed);
  const int K = mat == 1 ? P.K1 : P.K2;
  const int rows = mat == 1 ? P.rows1 : P.rows2;
  g.mode = mode;
  g.hdr = reinterpret_cast<const PackHeader*>(b);
  g.which = which;
  g.G = P.G;
  g.K = K;
  g.b_rows_per_group = rows;
  g.offsets = offsets;
  g.poff = poff;
  g.a_sf = as; g.a_sf_ld = R; g.a_rows = R;
  g.b_sf = b + (mat == 1 ? P.off_s1 : P.off_s2); g.b_sf_ld = (int64_t)P.G * rows; g.b_rows = (int64_t)P.G * rows;
  g.b_fp4 = P.fmt == MOE_WFMT_MXFP4;
  g.bias = which == MOE_PACK_FORWARD && c->w1_bias;
  g.R = R;
  g.status = status;
  MxMaps maps;
  if (!make_tmaps_mx_a(&maps, aq, R, K) ||
      !make_tmap_mx(&maps.b, b + (mat == 1 ? P.off_w1 : P.off_w2), (int64_t)P.G * rows, K, mx_b_box_rows(),
                    g.b_fp4 != 0) ||
      !make_tmap_mx_sf(&maps.sfb, g.b_sf, g.b_rows, ceil_div(K, 128), g.b_sf_ld))
    return MOE_ERR_CUDA;
  MOE_CHECK_CUDA(launch_gemm_mx(g, maps, mx_grid(*c), st));
  return MOE_OK;
}

static MxArgs mx_args0() {
  MxArgs g;
  std::memset(&g, 0, sizeof(g));
  return g;
}

static ActParams act_params(const moe_config_t* c) {
  ActParams p;
  p.act = c->act;
  p.alpha = c->act == MOE_ACT_SWIGLU_CLAMP ? c->act_alpha : 1.f;
  p.limit = c->act_limit;
  return p;
}

// W1 -> W2 in one launch of the decoding GEMM (the counters in the workspace
// must be zero: the operand gather clears them). y1 (MXFP8) lands in y1q /
// y1s; W2's fp32 K-slice partials in run2.
static moe_status_t tc_fused(const moe_config_t* c, const moe_dispatch_t* d, int T, const void* packed, uint8_t* y1q,
                             uint8_t* y1s, void* ws, cudaStream_t st, TcRun* run2, int n_disp) {
  const WsLayout L = ws_layout(*c);
  const PackLayout P = pack_layout(*c, MOE_PACK_FORWARD);
  TcArgs g;
  tc_common(g, c, P, packed, ws, L, d->offsets);
  g.nmat = 2;
  g.m[0] = tc_mat(c, P, 1, packed, T, at<int32_t>(ws, L.rexp1), at<float>(ws, L.P), g.max_ctas);
  g.m[1] = tc_mat(c, P, 2, packed, T, at<int32_t>(ws, L.rexp2), at<float>(ws, L.P2), g.max_ctas);
  // the kernel's fused W1 epilogue reads one K slice, in 16-token tiles
  const int nt = tc_token_tile(T, c->k + c->n_shared, c->E + c->n_shared);
  if (g.m[0].S != 1 || nt != 16) return MOE_ERR_UNSUPPORTED;
  g.f.w_row = d->w_row;
  g.f.act = act_params(c);
  g.f.I = c->I;
  g.f.y1q = y1q;
  g.f.y1s = y1s;
  g.f.y16 = at<uint16_t>(ws, L.y16);
  g.f.y_rowexp = at<int32_t>(ws, L.rexp2);
  g.f.cnt = at<int32_t>(ws, L.fcnt);
  g.f.b1 = P.off_b1 ? reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(packed) + P.off_b1) : nullptr;
  // partitioned layer: the first n_disp CTAs gather the W1 operand rows
  if (n_disp >= g.max_ctas) return MOE_ERR_INVALID_ARG;
  g.f.n_disp = n_disp;
  g.f.xq = d->xq; g.f.xs = d->xs;
  g.f.row_map = d->perm_src; g.f.row_div = c->k + c->n_shared;
  g.f.a16 = at<uint16_t>(ws, L.a16); g.f.a_rowexp = at<int32_t>(ws, L.rexp1);
  const int64_t R = (int64_t)T * (c->k + c->n_shared);
  TcMaps maps;
  if (!make_tmaps_b(maps.m[0], at<uint16_t>(ws, L.a16), R, g.m[0].K) ||
      !make_tmaps_b(maps.m[1], g.f.y16, R, g.m[1].K))
    return MOE_ERR_CUDA;
  MOE_CHECK_CUDA(launch_gemm_tc(g, maps, nt, st));
  run2->out = g.m[1].out;
  run2->split_stride = g.m[1].split_stride;
  run2->S = g.m[1].S;
  return MOE_OK;
}

// W1 with its fused epilogue. NVFP4: f16 operand rows (unless a_ready),
// decoding tensor-core GEMM, then the SwiGLU / routing weight / MXFP8
// epilogue kernel. MXFP8: gathered MXFP8 rows (unless a_ready), then the
// block-scaled GEMM whose epilogue writes y1 (and, with save, h and the
// transposed copy of y).
static moe_status_t w1_impl(const moe_config_t* c, const moe_dispatch_t* d, int T, const void* packed, uint8_t* y1q,
                            uint8_t* y1s, const moe_train_save_t* save, void* ws, cudaStream_t st,
                            bool a_ready = false) {
  const WsLayout L = ws_layout(*c);
  const PackLayout P = pack_layout(*c, MOE_PACK_FORWARD);
  const int kp = c->k + c->n_shared, G = c->E + c->n_shared;
  const int R = T * kp;
  if (T == 0) return MOE_OK;
  int32_t* status = at<int32_t>(ws, L.status);
  if (mx_path(*c)) {
    uint8_t* xg = at<uint8_t>(ws, L.xg);
    uint8_t* xgs = at<uint8_t>(ws, L.xgs);
    if (!a_ready) MOE_CHECK_CUDA(launch_gather_mx(d->xq, d->xs, c->H, d->perm_src, kp, R, d->offsets, G, xg, xgs, st));
    MxArgs g = mx_args0();
    g.n_tiles = ceil_div(P.rows1, kMxTileN);
    g.I = c->I;
    g.gated = gated(*c);
    g.b1 = P.off_b1 ? reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(packed) + P.off_b1) : nullptr;
    g.w_row = d->w_row;
    g.act = act_params(c);
    g.yq = y1q; g.ys = y1s;
    g.yst = at<uint8_t>(ws, L.y1st);
    if (save) {
      g.hsave = save->h; g.tq = save->y1t_q; g.ts = save->y1t_s; g.t_ld = r_pad_for(dims_of(*c), T); g.t_nf = c->I;
      if (save->amax) {
        MOE_CHECK_CUDA(cudaMemsetAsync(save->amax, 0, 2 * sizeof(float), st));
        g.amax = save->amax;
      }
    }
    moe_status_t s = mx_token_gemm(c, g, kMxW1, xg, xgs, R, packed, MOE_PACK_FORWARD, 1, d->offsets,
                                   at<int32_t>(ws, L.poff), status, st);
    if (s != MOE_OK) return s;
    phase(2, st);
    phase(3, st);
    if (save)
      MOE_CHECK_CUDA(cudaMemcpyAsync(save->poff, at<int32_t>(ws, L.poff), (size_t)(G + 1) * 4,
                                     cudaMemcpyDeviceToDevice, st));
    return MOE_OK;
  }
  uint16_t* a16 = at<uint16_t>(ws, L.a16);
  int32_t* rexp1 = at<int32_t>(ws, L.rexp1);
  if (!a_ready)
    MOE_CHECK_CUDA(launch_act_f16(d->xq, d->xs, c->H, d->perm_src, kp, R, d->offsets, G, a16, rexp1, st));
  TcRun run;
  moe_status_t s = tc_gemm(c, P, 1, packed, ws, L, d->offsets, T, a16, rexp1, st, &run);
  if (s != MOE_OK) return s;
  phase(2, st);
  W1FinArgs f;
  f.P = run.out; f.S = run.S; f.split_stride = run.split_stride; f.R = R; f.I = c->I;
  f.offsets = d->offsets; f.G = G; f.w_row = d->w_row; f.act = act_params(c);
  f.y1q = y1q; f.y1s = y1s; f.gated = gated(*c);
  f.y16 = at<uint16_t>(ws, L.y16);
  f.y_rowexp = at<int32_t>(ws, L.rexp2);
  f.b1 = P.off_b1 ? reinterpret_cast<const float*>(reinterpret_cast<const uint8_t*>(packed) + P.off_b1) : nullptr;
  MOE_CHECK_CUDA(launch_w1_finalize(f, st));
  phase(3, st);
  return MOE_OK;
}

// W2 on the MXFP8 path: z [R][H] bf16 straight from the block-scaled GEMM.
// y1st: y1's scales in the SF4 layout (ld R); nullptr converts y1s (the
// row-major [R][I/32] layout) into the workspace first.
static moe_status_t w2_mx(const moe_config_t* c, const int32_t* offsets, int T, const uint8_t* y1q,
                          const uint8_t* y1s, const uint8_t* y1st, const void* packed, uint16_t* z, void* ws,
                          cudaStream_t st) {
  const WsLayout L = ws_layout(*c);
  const int64_t R = (int64_t)T * (c->k + c->n_shared);
  if (!y1st) {
    uint8_t* t = at<uint8_t>(ws, L.y1st);
    MOE_CHECK_CUDA(launch_sf_to_sf4(y1s, c->I, R, t, st));
    y1st = t;
  }
  MxArgs g = mx_args0();
  g.n_tiles = ceil_div(c->H, kMxTileN);
  g.N = c->H;
  g.out = z; g.out_ld = c->H;
  return mx_token_gemm(c, g, kMxPlain, y1q, y1st, R, packed, MOE_PACK_FORWARD, 2, offsets, at<int32_t>(ws, L.poff),
                       at<int32_t>(ws, L.status), st);
}

static moe_status_t check_save(const moe_config_t* c, const moe_train_save_t* save) {
  if (!save) return MOE_OK;
  if (!backward_capable(*c)) return MOE_ERR_UNSUPPORTED;
  REQ(save->h); REQ(save->y1t_q); REQ(save->y1t_s); REQ(save->at_q); REQ(save->at_s); REQ(save->poff);
  OPT(save->amax);
  return MOE_OK;
}

moe_status_t moe_grouped_gemm_w1_swiglu_quant(const moe_config_t* c, const moe_dispatch_t* d, int T,
                                              const void* packed_w, uint8_t* y1_q, uint8_t* y1_s,
                                              const moe_train_save_t* save, void* ws, void* stream) {
  moe_status_t s = check_T(c, T);
  if (s != MOE_OK) return s;
  if ((s = check_dispatch(d, true, T)) != MOE_OK) return s;
  REQ(packed_w); REQ_T(y1_q); REQ_T(y1_s); REQ(ws);
  if ((s = check_save(c, save)) != MOE_OK) return s;
  reset_launch_count();
  return w1_impl(c, d, T, packed_w, y1_q, y1_s, save, ws, (cudaStream_t)stream);
}

moe_status_t moe_grouped_gemm_w2(const moe_config_t* c, const moe_dispatch_t* d, int T, const uint8_t* y1_q,
                                 const uint8_t* y1_s, const void* packed_w, uint16_t* z, void* ws, void* stream) {
  moe_status_t s = check_T(c, T);
  if (s != MOE_OK) return s;
  if ((s = check_dispatch(d, false, T)) != MOE_OK) return s;
  REQ_T(y1_q); REQ_T(y1_s); REQ(packed_w); REQ_T(z); REQ(ws);
  reset_launch_count();
  if (T == 0) return MOE_OK;
  cudaStream_t st = (cudaStream_t)stream;
  if (mx_path(*c)) return w2_mx(c, d->offsets, T, y1_q, y1_s, nullptr, packed_w, z, ws, st);
  const WsLayout L = ws_layout(*c);
  const PackLayout P = pack_layout(*c, MOE_PACK_FORWARD);
  const int R = T * (c->k + c->n_shared);
  uint16_t* y16 = at<uint16_t>(ws, L.y16);
  int32_t* rexp2 = at<int32_t>(ws, L.rexp2);
  MOE_CHECK_CUDA(launch_act_f16(y1_q, y1_s, c->I, nullptr, 1, R, d->offsets, c->E + c->n_shared, y16, rexp2, st));
  TcRun run;
  s = tc_gemm(c, P, 2, packed_w, ws, L, d->offsets, T, y16, rexp2, st, &run);
  if (s != MOE_OK) return s;
  MOE_CHECK_CUDA(launch_finalize_rows(run.out, run.S, run.split_stride, c->H, R, z, st));
  return MOE_OK;
}

moe_status_t moe_combine(const moe_config_t* c, const uint16_t* z, const int32_t* inv, const float* topk_w, int T,
                         uint16_t* out, void* stream) {
  moe_status_t s = check_T(c, T);
  if (s != MOE_OK) return s;
  REQ_T(z); REQ_T(inv); OPT(topk_w); REQ_T(out);
  reset_launch_count();
  MOE_CHECK_CUDA(launch_combine(z, inv, topk_w, T, c->k, c->k + c->n_shared, c->H, out, (cudaStream_t)stream));
  return MOE_OK;
}

moe_status_t moe_layer_forward(const moe_config_t* c, const uint16_t* x, const float* W_r, const float* logits_in,
                               int T, const void* packed_w, uint16_t* out, const moe_train_save_t* save, void* ws,
                               void* stream) {
  moe_status_t s = check_T(c, T);
  if (s != MOE_OK) return s;
  if (W_r && logits_in) return MOE_ERR_INVALID_ARG;
  if (!W_r && !logits_in && T > 0) return MOE_ERR_INVALID_ARG;
  REQ_T(x); OPT(W_r); OPT(logits_in); REQ(packed_w); REQ_T(out); REQ(ws);
  if ((s = check_save(c, save)) != MOE_OK) return s;
  reset_launch_count();
  cudaStream_t st = (cudaStream_t)stream;
  const WsLayout L = ws_layout(*c);
  moe_ws_view_t v;
  moe_workspace_view(c, ws, &v);
  const int kp = c->k + c->n_shared, G = c->E + c->n_shared;
  RouteArgs a = route_args(c, T, &v.d, ws, L);
  a.x = x;
  a.logits = v.logits;
  // partitioned fused layer: the routing kernel clears the hand-off
  // counters and ring flags; the fused kernel gathers the W1 operand rows
  const int n_disp = T > 0 && fused_layer(*c, T) && !save ? c->dispatch_sms : 0;
  if (n_disp > 0 && n_disp >= mx_grid(*c)) return MOE_ERR_INVALID_ARG;   // no GEMM CTA would be left
  if (n_disp > 0) {
    a.zero = at<int32_t>(ws, L.fcnt);
    a.nzero = tc_fused_counters(G);
  }
  phase(0, st);
  if (W_r) {
    const int KS = router_splits(T, c->H, c->E);
    float* part = KS == 1 ? v.logits : at<float>(ws, L.rpart);
    MOE_CHECK_CUDA(launch_router(x, W_r, T, c->H, c->E, KS, part, st));
    a.part = part; a.KS = KS;
    const int64_t n = (int64_t)T * c->E;
    if (KS > 1 && n * KS > kRouteStage) {
      // too many partials for the routing kernel's single block to sum: a
      // block per token sums its partials (in ks order) into the logits and
      // routes it; the dispatch kernel takes the ids as given
      MOE_CHECK_CUDA(launch_sum_topk(part, KS, T, c->E, c->k, c->routed_scale, v.logits, v.d.topk_ids, v.d.topk_w,
                                     at<int32_t>(ws, L.status), st));
      a.part = v.logits; a.KS = 1; a.route = false;
    }
  } else {
    a.part = logits_in; a.KS = 1;
  }
  MOE_CHECK_CUDA(launch_route_dispatch(a, st));
  if (T > 0) {
    // gather the quantised rows into the W1 GEMM's operand (part of dispatch)
    if (mx_path(*c))
      MOE_CHECK_CUDA(launch_gather_mx(v.d.xq, v.d.xs, c->H, v.d.perm_src, kp, T * kp, v.d.offsets, G,
                                      at<uint8_t>(ws, L.xg), at<uint8_t>(ws, L.xgs), st));
    else if (n_disp > 0) {
      // the fused kernel's ring CTAs gather the rows
    } else if (fused_layer(*c, T) && !save)
      MOE_CHECK_CUDA(launch_act_f16(v.d.xq, v.d.xs, c->H, v.d.perm_src, kp, T * kp, v.d.offsets, G,
                                    at<uint16_t>(ws, L.a16), at<int32_t>(ws, L.rexp1), st, at<int32_t>(ws, L.fcnt),
                                    tc_fused_counters(G)));
    else
      MOE_CHECK_CUDA(launch_act_f16(v.d.xq, v.d.xs, c->H, v.d.perm_src, kp, T * kp, v.d.offsets, G,
                                    at<uint16_t>(ws, L.a16), at<int32_t>(ws, L.rexp1), st));
  }
  phase(1, st);
  if (T == 0) {
    for (int i = 2; i < MOE_N_PHASE_EVENTS; ++i) phase(i, st);
    return MOE_OK;
  }
  if (save) {
    // transposed MXFP8 copy of the gathered activations for the W1 wgrad
    ColQuantArgs q;
    q.src16 = x; q.row_map = v.d.perm_src; q.row_div = kp;
    q.C = c->H; q.offsets = v.d.offsets; q.poff = at<int32_t>(ws, L.poff); q.G = G;
    q.r_pad_max = r_pad_for(dims_of(*c), T); q.q = save->at_q; q.s = save->at_s;
    MOE_CHECK_CUDA(launch_quant_cols(q, st));
  }
  if (fused_layer(*c, T) && !save) {
    TcRun run;
    if ((s = tc_fused(c, &v.d, T, packed_w, v.y1_q, v.y1_s, ws, st, &run, n_disp)) != MOE_OK) return s;
    phase(2, st);
    phase(3, st);
    phase(4, st);
    MOE_CHECK_CUDA(launch_finalize_combine(run.out, run.S, run.split_stride, c->H, v.d.inv, T, kp, v.z, out, st));
    phase(5, st);
    return MOE_OK;
  }
  if ((s = w1_impl(c, &v.d, T, packed_w, v.y1_q, v.y1_s, save, ws, st, true)) != MOE_OK) return s;
  if (mx_path(*c)) {
    if ((s = w2_mx(c, v.d.offsets, T, v.y1_q, v.y1_s, at<uint8_t>(ws, L.y1st), packed_w, v.z, ws, st)) != MOE_OK)
      return s;
    phase(4, st);
    MOE_CHECK_CUDA(launch_combine(v.z, v.d.inv, nullptr, T, c->k, kp, c->H, out, st));
    phase(5, st);
    return MOE_OK;
  }
  const PackLayout P = pack_layout(*c, MOE_PACK_FORWARD);
  TcRun run;
  s = tc_gemm(c, P, 2, packed_w, ws, L, v.d.offsets, T, at<uint16_t>(ws, L.y16), at<int32_t>(ws, L.rexp2), st,
              &run);
  if (s != MOE_OK) return s;
  phase(4, st);
  MOE_CHECK_CUDA(launch_finalize_combine(run.out, run.S, run.split_stride, c->H, v.d.inv, T, kp, v.z, out, st));
  phase(5, st);
  return MOE_OK;
}

// Weight gradient of one matrix on the block-scaled GEMM: out[e][m][n] =
// sum over group e's padded token rows p of P[m][p] * Q[n][p] (both MXFP8
// along p).
static moe_status_t mx_wgrad(const moe_config_t* c, const uint8_t* pq, const uint8_t* ps, int M, const uint8_t* qq,
                             const uint8_t* qs, int N, int64_t Rp, const int32_t* poff, uint16_t* out,
                             int32_t* status, cudaStream_t st) {
  MxArgs g = mx_args0();
  g.mode = kMxWgrad;
  g.hdr = nullptr;
  g.G = c->E;
  g.M = M; g.m_tiles = ceil_div(M, mx_tile_m());
  g.N = N; g.n_tiles = ceil_div(N, mx_tile_n());
  g.poff = poff;
  g.a_sf = ps; g.a_sf_ld = M; g.a_rows = M;
  g.b_sf = qs; g.b_sf_ld = N; g.b_rows = N;
  g.out = out; g.out_ld = N;
  g.status = status;
  MxMaps maps;
  if (!make_tmaps_mx_a(&maps, pq, M, Rp) || !make_tmap_mx(&maps.b, qq, N, Rp, mx_b_box_rows(), false) ||
      !make_tmap_mx_sf(&maps.sfb, qs, N, Rp / 128, N))
    return MOE_ERR_CUDA;
  MOE_CHECK_CUDA(launch_gemm_mx(g, maps, mx_grid(*c), st));
  return MOE_OK;
}

moe_status_t moe_layer_backward(const moe_config_t* c, const uint16_t* dout, const uint16_t* x, int T,
                                const moe_train_save_t* save, const void* packed_w_dgrad, uint16_t* dx, uint16_t* dW1,
                                uint16_t* dW2, float* dlogits, float* db1, void* ws, void* stream) {
  moe_status_t s = check_T(c, T);
  if (s != MOE_OK) return s;
  if (!backward_capable(*c)) return MOE_ERR_UNSUPPORTED;
  if (!save) return MOE_ERR_INVALID_ARG;
  if ((s = check_save(c, save)) != MOE_OK) return s;
  REQ_T(dout); REQ_T(x); REQ(packed_w_dgrad); REQ_T(dx); REQ(dW1); REQ(dW2); REQ_T(dlogits); REQ(ws);
  if (c->w1_bias) { REQ(db1); } else if (db1) return MOE_ERR_INVALID_ARG;
  reset_launch_count();
  cudaStream_t st = (cudaStream_t)stream;
  const WsLayout L = ws_layout(*c);
  moe_ws_view_t v;
  moe_workspace_view(c, ws, &v);
  const Dims dm = dims_of(*c);
  const int kp = dm.kp, G = dm.G, I = c->I, H = c->H;
  const int N1 = gated(*c) ? 2 * I : I;   // W1 outputs: h and dh columns
  const int R = T * kp;
  const int64_t Rp = r_pad_for(dm, T);
  int32_t* status = at<int32_t>(ws, L.status);
  uint8_t* dzq = at<uint8_t>(ws, L.dzq);
  uint8_t* dzs = at<uint8_t>(ws, L.dzs);
  uint8_t* dzg = at<uint8_t>(ws, L.dzg);
  uint8_t* dzgs = at<uint8_t>(ws, L.dzgs);
  uint8_t* dztq = at<uint8_t>(ws, L.dztq);
  uint8_t* dzts = at<uint8_t>(ws, L.dzts);
  uint8_t* dhq = at<uint8_t>(ws, L.dhq);
  uint8_t* dhs = at<uint8_t>(ws, L.dhs);
  uint8_t* dhtq = at<uint8_t>(ws, L.dhtq);
  uint8_t* dhts = at<uint8_t>(ws, L.dhts);
  uint16_t* dxp = at<uint16_t>(ws, L.dxp);
  float* dwpart = at<float>(ws, L.dwpart);
  const int32_t* poff = at<int32_t>(ws, L.poff);
  const int nparts = ceil_div(I, mx_tile_n());
  if (T > 0) {
    // 1. dz rows: MXFP8 per token along H, gathered into group order, and the
    //    transposed copy along the padded row axis (W2 wgrad operand)
    MOE_CHECK_CUDA(launch_quant_rows(dout, T, H, dzq, dzs, st));
    ColQuantArgs q;
    q.src16 = dout; q.row_map = v.d.perm_src; q.row_div = kp;
    q.C = H; q.offsets = v.d.offsets; q.poff = poff; q.G = G; q.r_pad_max = Rp; q.q = dztq; q.s = dzts;
    MOE_CHECK_CUDA(launch_quant_cols(q, st));
    MOE_CHECK_CUDA(launch_gather_mx(dzq, dzs, H, v.d.perm_src, kp, R, v.d.offsets, G, dzg, dzgs, st));
    // 2. dY1 = dz . W2^T with the fused dSwiGLU + MXFP8 / transposed-copy
    //    epilogue and the routing-weight gradient partials
    MxArgs g = mx_args0();
    g.n_tiles = nparts;
    g.I = I;
    g.gated = gated(*c);
    g.w_row = v.d.w_row;
    g.act = act_params(c);
    g.hsave = save->h;
    g.yq = dhq; g.yst = dhs;
    g.tq = dhtq; g.ts = dhts; g.t_ld = Rp; g.t_nf = N1;
    g.dwpart = dwpart;
    if (c->w1_bias) { g.dbpart = at<float>(ws, L.dbpart); g.db_ld = N1; }
    if ((s = mx_token_gemm(c, g, kMxDswiglu, dzg, dzgs, R, packed_w_dgrad, MOE_PACK_DGRAD, 2, v.d.offsets, poff,
                           status, st)) != MOE_OK)
      return s;
    // 3. dXp = dh . W1^T (bf16 rows), then the slot-ordered combine backward
    MxArgs g2 = mx_args0();
    g2.n_tiles = ceil_div(H, mx_tile_n());
    g2.N = H;
    g2.out = dxp; g2.out_ld = H;
    if ((s = mx_token_gemm(c, g2, kMxPlain, dhq, dhs, R, packed_w_dgrad, MOE_PACK_DGRAD, 1, v.d.offsets, poff, status,
                           st)) != MOE_OK)
      return s;
    MOE_CHECK_CUDA(launch_combine(dxp, v.d.inv, nullptr, T, c->k, kp, H, dx, st));
  }
  // 4. wgrads over each group's padded rows (groups without rows: zeros)
  if ((s = mx_wgrad(c, save->at_q, save->at_s, H, dhtq, dhts, N1, Rp, poff, dW1, status, st)) != MOE_OK) return s;
  if ((s = mx_wgrad(c, save->y1t_q, save->y1t_s, I, dztq, dzts, H, Rp, poff, dW2, status, st)) != MOE_OK) return s;
  // 5. W1 bias: each group's padded 32-row block partials summed in order
  if (c->w1_bias) MOE_CHECK_CUDA(launch_bias_grad(at<float>(ws, L.dbpart), N1, poff, G, db1, st));
  // 6. router
  MOE_CHECK_CUDA(launch_router_bwd(v.d.topk_w, v.d.topk_ids, dwpart, nparts, R, v.d.inv, T, c->E, c->k, kp,
                                   c->routed_scale, dlogits, st));
  return MOE_OK;
}

moe_status_t moe_read_status(const moe_config_t* c, void* ws, int32_t* out, void* stream) {
  moe_status_t s = moe_config_validate(c);
  if (s != MOE_OK) return s;
  REQ(ws);
  if (!out) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(*c);
  cudaStream_t st = (cudaStream_t)stream;
  MOE_CHECK_CUDA(cudaStreamSynchronize(st));
  MOE_CHECK_CUDA(cudaMemcpy(out, at<int32_t>(ws, L.status), 4, cudaMemcpyDeviceToHost));
  MOE_CHECK_CUDA(cudaMemsetAsync(at<int32_t>(ws, L.status), 0, 4, st));
  MOE_CHECK_CUDA(cudaStreamSynchronize(st));
  return *out ? MOE_ERR_DEVICE : MOE_OK;
}

moe_status_t moe_clear_status(const moe_config_t* c, void* ws, void* stream) {
  moe_status_t s = moe_config_validate(c);
  if (s != MOE_OK) return s;
  REQ(ws);
  const WsLayout L = ws_layout(*c);
  MOE_CHECK_CUDA(cudaMemsetAsync(at<int32_t>(ws, L.status), 0, 4, (cudaStream_t)stream));
  return MOE_OK;
}

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null pointer, shape, alignment or T > T_max)";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE: return "workspace or output buffer too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE: return "device status word reports an error";
  }
  return "unknown status";
}

int moe_last_launch_count(void) { return launch_count(); }

moe_status_t moe_debug_flag_wait(const moe_config_t* c, const int32_t* flag, int64_t limit_cycles, void* ws,
                                 void* stream) {
  moe_status_t s = moe_config_validate(c);
  if (s != MOE_OK) return s;
  if (!flag || ((uintptr_t)flag & 3u) || limit_cycles <= 0) return MOE_ERR_INVALID_ARG;
  REQ(ws);
  reset_launch_count();
  const WsLayout L = ws_layout(*c);
  MOE_CHECK_CUDA(launch_debug_flag_wait(flag, (long long)limit_cycles, at<int32_t>(ws, L.status),
                                        (cudaStream_t)stream));
  return MOE_OK;
}

moe_status_t moe_layer_fused(const moe_config_t* c, int T, int32_t* fused) {
  moe_status_t s = check_T(c, T);
  if (s != MOE_OK) return s;
  if (!fused) return MOE_ERR_INVALID_ARG;
  *fused = fused_layer(*c, T) ? 1 : 0;
  return MOE_OK;
}

moe_status_t moe_set_phase_events(void* const* events) {
  if (!events) {
    g_phase_on = false;
    return MOE_OK;
  }
  for (int i = 0; i < MOE_N_PHASE_EVENTS; ++i) g_phase[i] = (cudaEvent_t)events[i];
  g_phase_on = true;
  return MOE_OK;
}

}  // extern "C"
