// S1 router logits, S2 top-k routing, S3 counts/offsets, S4 permutation and
// the MXFP8 quantisation of token rows.
//
// GC-MoE summary (arxiv-wiki "GC-MoE: Overlapping Expert-Parallel Token
// Dispatch with FP8/FP4 Grouped GEMM via CUDA Green Contexts"), Approach:
// role1 aggregates routing counts and places tokens into expert blocks.
// NVIDIA blog "Boosting MoE training throughput with advanced fusion
// kernels", section on removing host-device sync: per-group token counts stay
// in GPU memory so nothing waits on the host. On one GPU the cross-rank token
// pull becomes this local, deterministic permutation.
//
// Determinism: counts come from per-warp histograms built with warp match
// (no atomics: each count is a fixed sequence of integer additions); the row
// order inside a group is fixed by a stable, warp-sequential scatter in flat
// assignment order (t * k' + j).
#include "internal.cuh"

namespace moe {

// ---------------------------------------------------------------------------
// S1: logits partials, a register-tiled fp32 GEMM over one slice of H
// (the general kernel; the decode-size and mid-batch kernels below take
// every shape whose expert count is a multiple of 4).
// grid (ceil(T/TT), ceil(E/64), KS), block 256: thread (tx = tid % 16,
// ty = tid / 16) owns experts 4tx..4tx+3 and tokens ty*TT/16.. of the
// CTA's 64-expert x TT-token tile. The slice [h0, h1) (multiples of 8 rows)
// moves through shared memory in 128-row chunks by cp.async, two chunks in
// flight: a chunk's W rows (fp32) and x columns (bf16, as stored) are all
// requested at once, so a decode-sized slice of one chunk costs one memory
// round trip instead of one per load wave (W_r is streamed once; at decode
// the latency of the copies, not the FLOPs, sets the time). Every thread
// accumulates its h in increasing order: part[ks][t][e] = sum over the
// ks-th slice of H of x[t][h] * W_r[h][e].
// ---------------------------------------------------------------------------
constexpr int kRtKH = 128;                 // rows of H per chunk
constexpr int kRtXLd = kRtKH + 8;          // x row stride in shared memory (bf16; keeps 16-byte pieces aligned)

template <int TT>
constexpr int router_stage_bytes() { return kRtKH * 64 * 4 + TT * kRtXLd * 2; }
template <int TT>
constexpr int router_smem() { return 2 * router_stage_bytes<TT>(); }

// Slice ks of KS over H, in units of 8 rows (H is a multiple of 64).
__host__ __device__ __forceinline__ int router_slice_begin(int ks, int KS, int H) {
  return 8 * (int)((int64_t)ks * (H / 8) / KS);
}

// Requests chunk [hb, hb + hn) of the CTA's W columns e0..e0+63 and token
// rows t0..t0+TT-1 of x into stage buffers ws / xs (zero-filled outside the
// chunk, the experts and the tokens) and commits them as one group.
template <int TT>
__device__ __forceinline__ void router_issue(const uint16_t* __restrict__ x, const float* __restrict__ Wr, int T,
                                             int H, int E, int t0, int e0, int hb, int hn, float* ws,
                                             uint16_t* xs) {
  const uint32_t wsb = (uint32_t)__cvta_generic_to_shared(ws);
  const uint32_t xsb = (uint32_t)__cvta_generic_to_shared(xs);
  if ((E & 3) == 0) {
    for (int i = threadIdx.x; i < kRtKH * 16; i += 256) {       // 16 pieces of 4 experts a row
      const int r = i >> 4, c = (i & 15) * 4;
      const bool ok = r < hn && e0 + c < E;
      cp_async16_zfill(wsb + (uint32_t)(r * 64 + c) * 4u, ok ? Wr + (int64_t)(hb + r) * E + e0 + c : Wr, ok);
    }
  } else {
    for (int i = threadIdx.x; i < kRtKH * 64; i += 256) {       // rows not 16-byte aligned: one float at a time
      const int r = i >> 6, c = i & 63;
      const bool ok = r < hn && e0 + c < E;
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(wsb + (uint32_t)(r * 64 + c) * 4u),
                   "l"(ok ? Wr + (int64_t)(hb + r) * E + e0 + c : Wr), "r"(ok ? 4 : 0)
                   : "memory");
    }
  }
  for (int i = threadIdx.x; i < TT * (kRtKH / 8); i += 256) {  // 8 bf16 of one token a piece
    const int tt = i / (kRtKH / 8), c = (i % (kRtKH / 8)) * 8;
    const bool ok = t0 + tt < T && c < hn;
    cp_async16_zfill(xsb + (uint32_t)(tt * kRtXLd + c) * 2u, ok ? x + (int64_t)(t0 + tt) * H + hb + c : x, ok);
  }
  cp_async_commit();
}

template <int TT>
__global__ void __launch_bounds__(256) k_router_partial(const uint16_t* __restrict__ x,
                                                        const float* __restrict__ Wr, int T, int H, int E,
                                                        int KS, float* __restrict__ part) {
  extern __shared__ __align__(16) uint8_t rsm[];
  pdl_enter();
  constexpr int TPT = TT / 16;                     // tokens per thread
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int t0 = blockIdx.x * TT;
  const int e0 = blockIdx.y * 64;
  const int ks = blockIdx.z;
  const int h0 = router_slice_begin(ks, KS, H), h1 = router_slice_begin(ks + 1, KS, H);
  const int nch = (h1 - h0 + kRtKH - 1) / kRtKH;
  auto wbuf = [&](int b) { return reinterpret_cast<float*>(rsm + b * router_stage_bytes<TT>()); };
  auto xbuf = [&](int b) {
    return reinterpret_cast<uint16_t*>(rsm + b * router_stage_bytes<TT>() + kRtKH * 64 * 4);
  };
  float acc[TPT][4];
#pragma unroll
  for (int i = 0; i < TPT; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int c = 0; c < min(nch, 2); ++c)
    router_issue<TT>(x, Wr, T, H, E, t0, e0, h0 + c * kRtKH, min(kRtKH, h1 - h0 - c * kRtKH), wbuf(c), xbuf(c));
  for (int c = 0; c < nch; ++c) {
    if (c + 1 < nch) cp_async_wait<1>();
    else cp_async_wait<0>();
    __syncthreads();                               // chunk c has landed for every thread
    const float* ws = wbuf(c & 1);
    const uint16_t* xs = xbuf(c & 1);
#pragma unroll 8
    for (int hh = 0; hh < kRtKH; ++hh) {
      const float4 w = *reinterpret_cast<const float4*>(&ws[hh * 64 + tx * 4]);
      float a[TPT];
#pragma unroll
      for (int i = 0; i < TPT; ++i) a[i] = bf16_bits_to_f32(xs[(ty * TPT + i) * kRtXLd + hh]);
#pragma unroll
      for (int i = 0; i < TPT; ++i) {
        acc[i][0] = fmaf(a[i], w.x, acc[i][0]);
        acc[i][1] = fmaf(a[i], w.y, acc[i][1]);
        acc[i][2] = fmaf(a[i], w.z, acc[i][2]);
        acc[i][3] = fmaf(a[i], w.w, acc[i][3]);
      }
    }
    __syncthreads();                               // every thread is done with stage c & 1
    if (c + 2 < nch)
      router_issue<TT>(x, Wr, T, H, E, t0, e0, h0 + (c + 2) * kRtKH, min(kRtKH, h1 - h0 - (c + 2) * kRtKH),
                       wbuf(c & 1), xbuf(c & 1));
  }
#pragma unroll
  for (int i = 0; i < TPT; ++i) {
    const int t = t0 + ty * TPT + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) part[((int64_t)ks * T + t) * E + e] = acc[i][j];
    }
  }
}

// S1 at decode sizes (T <= 32, E a multiple of 4): one CTA per 64 experts x
// one slice of H, about one CTA per SM. The CTA's W rows go straight into
// registers, thread (tx = tid % 16, ty = tid / 16) holding experts
// 4tx..4tx+3 of rows ty, ty + 16, ..., ty + 176 of a 192-row chunk, every
// load of the chunk in flight at once; x comes in transposed to [h][token]
// through shared memory. Each W element is read from memory once and feeds
// all TT tokens from registers, so at T = 1 the kernel costs one memory
// round trip and at T = 32 it stays FMA-bound rather than bound by shared
// memory. Per logit: each thread's fmaf chain over its rows (increasing h),
// the two row groups of a warp added (lane l and l ^ 16), then the 8 warps'
// sums added in warp order; a fixed order, so the result is deterministic.
constexpr int kRrRPT = 12;                 // rows of a chunk per thread
constexpr int kRrRows = 16 * kRrRPT;       // 192 rows of H per chunk

static bool router_rows(int T, int E) { return T <= 32 && E % 4 == 0; }

template <int TT>
constexpr int router_rows_smem() { return kRrRows * TT * 2 + 8 * TT * 64 * 4; }

template <int TT>
__global__ void __launch_bounds__(256, 1) k_router_rows(const uint16_t* __restrict__ x, const float* __restrict__ Wr,
                                                        int T, int H, int E, int KS, float* __restrict__ part) {
  extern __shared__ __align__(16) uint8_t rsm[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(rsm);                     // [kRrRows][TT] bf16
  float* red = reinterpret_cast<float*>(rsm + kRrRows * TT * 2);       // [8][TT][64]
  pdl_enter();
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.x * 64, ks = blockIdx.y;
  const int h0 = router_slice_begin(ks, KS, H), h1 = router_slice_begin(ks + 1, KS, H);
  const bool ecol = e0 + tx * 4 < E;
  float acc[TT][4];
#pragma unroll
  for (int t = 0; t < TT; ++t)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[t][j] = 0.f;
  for (int hb = h0; hb < h1; hb += kRrRows) {
    const int hn = min(kRrRows, h1 - hb);
    float4 w[kRrRPT];
#pragma unroll
    for (int r = 0; r < kRrRPT; ++r) {
      const int row = ty + 16 * r;
      w[r] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (row < hn && ecol) w[r] = __ldg(reinterpret_cast<const float4*>(Wr + (int64_t)(hb + row) * E + e0 + tx * 4));
    }
    if (hb != h0) __syncthreads();                 // every thread is done with the previous chunk's x
    for (int i = threadIdx.x; i < TT * (kRrRows / 8); i += 256) {
      const int t = i / (kRrRows / 8), c = (i % (kRrRows / 8)) * 8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);        // tokens past T and rows past the slice read as zero
      if (t < T && c < hn) v = __ldg(reinterpret_cast<const uint4*>(x + (int64_t)t * H + hb + c));
      const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xs[(c + 2 * j) * TT + t] = (uint16_t)(wd[j] & 0xffffu);
        xs[(c + 2 * j + 1) * TT + t] = (uint16_t)(wd[j] >> 16);
      }
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRrRPT; ++r) {
      if constexpr (TT == 1) {                     // one token: one x value a row
        const float a0 = bf16_bits_to_f32(xs[ty + 16 * r]);
        acc[0][0] = fmaf(a0, w[r].x, acc[0][0]); acc[0][1] = fmaf(a0, w[r].y, acc[0][1]);
        acc[0][2] = fmaf(a0, w[r].z, acc[0][2]); acc[0][3] = fmaf(a0, w[r].w, acc[0][3]);
        continue;
      }
      const uint4* xr = reinterpret_cast<const uint4*>(xs + (ty + 16 * r) * TT);
#pragma unroll
      for (int q = 0; q < TT / 8; ++q) {
        const uint4 xv = xr[q];
        const uint32_t wd[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const float a0 = __uint_as_float(wd[p] << 16), a1 = __uint_as_float(wd[p] & 0xffff0000u);
          float* c0 = acc[q * 8 + 2 * p];
          float* c1 = acc[q * 8 + 2 * p + 1];
          c0[0] = fmaf(a0, w[r].x, c0[0]); c0[1] = fmaf(a0, w[r].y, c0[1]);
          c0[2] = fmaf(a0, w[r].z, c0[2]); c0[3] = fmaf(a0, w[r].w, c0[3]);
          c1[0] = fmaf(a1, w[r].x, c1[0]); c1[1] = fmaf(a1, w[r].y, c1[1]);
          c1[2] = fmaf(a1, w[r].z, c1[2]); c1[3] = fmaf(a1, w[r].w, c1[3]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < TT; ++t)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[t][j] += __shfl_xor_sync(kFull, acc[t][j], 16);
  if (lane < 16) {
#pragma unroll
    for (int t = 0; t < TT; ++t)
      if (t < T)
        *reinterpret_cast<float4*>(&red[(warp * TT + t) * 64 + tx * 4]) =
            make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
  }
  __syncthreads();
  for (int o = threadIdx.x; o < T * 64; o += 256) {
    const int t = o >> 6, e = o & 63;
    if (e0 + e >= E) continue;
    float v = red[t * 64 + e];
#pragma unroll
    for (int q = 1; q < 8; ++q) v += red[(q * TT + t) * 64 + e];
    part[((int64_t)ks * T + t) * E + e0 + e] = v;
  }
}

// S1 at large T (the tiles alone fill the SMs; no split of H): one CTA per
// 64 tokens x 128 experts, thread (tx = tid % 16, ty = tid / 16) owns tokens
// 4ty..4ty+3 and experts 4tx..4tx+3 and 64+4tx..64+4tx+3, so three 16-byte
// shared loads feed 32 FMAs. Both operands are staged per 16 rows of H in a
// double-buffered shared tile (x converted to fp32 and transposed to
// [h][token]); the next stage's global loads are in registers while the
// current one is multiplied. Each logit is the fmaf chain over h in
// increasing order, the same chain k_router_partial forms with one slice.
constexpr int kRbTT = 64, kRbTE = 128, kRbKH = 16;

static bool router_big(int T, int H, int E) {
  return H % kRbKH == 0 && E % 4 == 0 &&
         (int64_t)((T + kRbTT - 1) / kRbTT) * ((E + kRbTE - 1) / kRbTE) >= device_sms();
}

__global__ void __launch_bounds__(256) k_router_big(const uint16_t* __restrict__ x, const float* __restrict__ Wr,
                                                    int T, int H, int E, float* __restrict__ logits) {
  pdl_enter();
  __shared__ __align__(16) float xs[2][kRbKH][kRbTT];
  __shared__ __align__(16) float ws[2][kRbKH][kRbTE];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.x * kRbTT, e0 = blockIdx.y * kRbTE;
  // x stage: 64 tokens x 16 h, one 8-value chunk per thread < 128 (token
  // tid % 64, h half tid / 64); W stage: 16 h x 128 experts, two float4 per
  // thread (rows tid / 32 and 8 + tid / 32, experts 4 (tid % 32)..)
  const int xt = tid & 63, xh = (tid >> 6) & 1;
  const bool xok = tid < 128 && t0 + xt < T;
  const uint16_t* xp = x + (int64_t)(xok ? t0 + xt : 0) * H + xh * 8;
  const int we = e0 + (tid & 31) * 4;
  const bool wok = we < E;
  const float* wp = Wr + (int64_t)(tid >> 5) * E + (wok ? we : 0);
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  uint4 xr = make_uint4(0u, 0u, 0u, 0u);
  float4 wr0 = z4, wr1 = z4;
  auto gload = [&](int hb) {
    if (xok) xr = __ldg(reinterpret_cast<const uint4*>(xp + hb));
    if (wok) {
      wr0 = __ldg(reinterpret_cast<const float4*>(wp + (int64_t)hb * E));
      wr1 = __ldg(reinterpret_cast<const float4*>(wp + (int64_t)(hb + 8) * E));
    }
  };
  auto sstore = [&](int b) {
    if (tid < 128) {
      float* d = &xs[b][xh * 8][xt];
      const uint32_t v[4] = {xr.x, xr.y, xr.z, xr.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        d[(2 * q) * kRbTT] = __uint_as_float(v[q] << 16);
        d[(2 * q + 1) * kRbTT] = __uint_as_float(v[q] & 0xffff0000u);
      }
    }
    *reinterpret_cast<float4*>(&ws[b][tid >> 5][(tid & 31) * 4]) = wr0;
    *reinterpret_cast<float4*>(&ws[b][8 + (tid >> 5)][(tid & 31) * 4]) = wr1;
  };
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  gload(0);
  sstore(0);
  __syncthreads();
  const int nk = H / kRbKH;
  for (int kb = 0; kb < nk; ++kb) {
    const int b = kb & 1;
    if (kb + 1 < nk) gload((kb + 1) * kRbKH);
#pragma unroll
    for (int hh = 0; hh < kRbKH; ++hh) {
      const float4 a = *reinterpret_cast<const float4*>(&xs[b][hh][ty * 4]);
      const float4 w0 = *reinterpret_cast<const float4*>(&ws[b][hh][tx * 4]);
      const float4 w1 = *reinterpret_cast<const float4*>(&ws[b][hh][64 + tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], wv[j], acc[i][j]);
    }
    if (kb + 1 < nk) sstore(b ^ 1);          // the buffer read one stage ago
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
    float* row = logits + (int64_t)t * E;
    if (e0 + tx * 4 < E)
      *reinterpret_cast<float4*>(row + e0 + tx * 4) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    if (e0 + 64 + tx * 4 < E)
      *reinterpret_cast<float4*>(row + e0 + 64 + tx * 4) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
}

// S1 between the two (T > 32, E a multiple of 4, too few 64 x 128 tiles to
// fill the SMs): the same tile and thread layout as k_router_big, split
// along H into KS slices of whole 16-row stages (part[ks][t][e]), with both
// operands moving through a kRmStages-deep cp.async ring so that several
// stages of W are in flight while one is multiplied (one stage ahead, the
// tile waited on memory every stage). x stays bf16 in shared memory,
// [token][h] with a 48-byte row; a thread reads two h of each of its 4
// tokens in one 32-bit load. Each logit is its fmaf chain over the slice in
// increasing h.
constexpr int kRmStages = 6;
constexpr int kRmXLd = 24;                                   // bf16 per x row in shared memory
constexpr int kRmWBytes = kRbKH * kRbTE * 4;                 // 8 KB
constexpr int kRmStage = kRmWBytes + kRbTT * kRmXLd * 2;     // + 3 KB of x
constexpr int kRmSmem = kRmStages * kRmStage;

static bool router_mid(int T, int H, int E) { return T > 32 && E % 4 == 0 && H % kRbKH == 0 && !router_big(T, H, E); }

__global__ void __launch_bounds__(256) k_router_mid(const uint16_t* __restrict__ x, const float* __restrict__ Wr,
                                                    int T, int H, int E, int KS, float* __restrict__ part) {
  extern __shared__ __align__(16) uint8_t rsm[];
  pdl_enter();
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int t0 = blockIdx.x * kRbTT, e0 = blockIdx.y * kRbTE, ks = blockIdx.z;
  const int u0 = (int)((int64_t)ks * (H / kRbKH) / KS), u1 = (int)((int64_t)(ks + 1) * (H / kRbKH) / KS);
  const int nk = u1 - u0;                                    // 16-row stages of this slice
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(rsm);
  auto issue = [&](int kb) {
    if (kb < nk) {
      const int hb = (u0 + kb) * kRbKH;
      const uint32_t st = sbase + (uint32_t)((kb % kRmStages) * kRmStage);
#pragma unroll
      for (int j = 0; j < 2; ++j) {                          // W: 16 rows x 32 pieces of 4 experts
        const int i = tid + 256 * j, r = i >> 5, c = (i & 31) * 4;
        const bool ok = e0 + c < E;
        cp_async16_zfill(st + (uint32_t)(r * kRbTE + c) * 4u, ok ? Wr + (int64_t)(hb + r) * E + e0 + c : Wr, ok);
      }
      if (tid < 2 * kRbTT) {                                 // x: 64 tokens x 2 pieces of 8 h
        const int tt = tid >> 1, c = (tid & 1) * 8;
        const bool ok = t0 + tt < T;
        cp_async16_zfill(st + kRmWBytes + (uint32_t)(tt * kRmXLd + c) * 2u, ok ? x + (int64_t)(t0 + tt) * H + hb + c : x,
                         ok);
      }
    }
    cp_async_commit();                                       // an empty group past the end keeps the count uniform
  };
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
#pragma unroll
  for (int kb = 0; kb < kRmStages - 1; ++kb) issue(kb);
  for (int kb = 0; kb < nk; ++kb) {
    cp_async_wait<kRmStages - 2>();
    __syncthreads();                                         // stage kb landed; stage kb - 1 is free
    issue(kb + kRmStages - 1);
    const float* ws = reinterpret_cast<const float*>(rsm + (kb % kRmStages) * kRmStage);
    const uint16_t* xs = reinterpret_cast<const uint16_t*>(rsm + (kb % kRmStages) * kRmStage + kRmWBytes);
#pragma unroll
    for (int hh = 0; hh < kRbKH; hh += 2) {
      float a[2][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(&xs[(ty * 4 + i) * kRmXLd + hh]);
        a[0][i] = __uint_as_float(v << 16);
        a[1][i] = __uint_as_float(v & 0xffff0000u);
      }
#pragma unroll
      for (int d = 0; d < 2; ++d) {
        const float4 w0 = *reinterpret_cast<const float4*>(&ws[(hh + d) * kRbTE + tx * 4]);
        const float4 w1 = *reinterpret_cast<const float4*>(&ws[(hh + d) * kRbTE + 64 + tx * 4]);
        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[d][i], wv[j], acc[i][j]);
      }
    }
  }
  cp_async_wait<0>();
  float* out = part + (int64_t)ks * T * E;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
    float* row = out + (int64_t)t * E;
    if (e0 + tx * 4 < E)
      *reinterpret_cast<float4*>(row + e0 + tx * 4) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    if (e0 + 64 + tx * 4 < E)
      *reinterpret_cast<float4*>(row + e0 + 64 + tx * 4) = make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]);
  }
}

// ---------------------------------------------------------------------------
// S2: one warp routes one token. Logits are first summed over the KS
// partials in ks order and written out (or taken as given from row_src);
// then k rounds of a warp arg-max on (value desc, id asc). NaN logits rank
// below every number and raise MOE_DEV_NAN_LOGIT. Weights: softmax over the
// selected logits x scale.
//
// The arg-max runs on order-preserving integer keys: a larger logit has a
// larger key, -0 and +0 share one (they compare equal), and -inf (NaN) is
// above 0, the key of an expert that is taken or out of range. Each lane
// keeps its best untaken expert (the lowest id among equal keys: its ids
// grow with i), the warp's largest key comes from one redux.sync max, and
// the lowest id holding it from one redux.sync min, so a round costs two
// warp reductions instead of five shuffle-and-compare steps.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t logit_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Sum over ks of part[ks * n + i], in ks order, 16 loads in flight at a
// time (the tail's loads predicated, not serialised).
__device__ __forceinline__ float sum_partials(const float* __restrict__ part, int KS, int64_t n, int64_t i) {
  float v = 0.f;
  for (int ks = 0; ks < KS; ks += 16) {
    float t[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] = ks + j < KS ? part[(int64_t)(ks + j) * n + i] : 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (ks + j < KS) v += t[j];
  }
  return v;
}

// VPL: logits per lane kept in registers (E <= 32 * VPL). With row_src the
// token's E logits are read from there (any memory) and not written again.
template <int VPL>
__device__ void route_token(int t, int lane, const float* __restrict__ part, int KS, int T, int E, int k,
                            float rs, float* __restrict__ logits, int32_t* __restrict__ ids,
                            float* __restrict__ wts, int32_t* status, const float* row_src = nullptr) {
  bool nan_seen = false;
  const float* row_in = row_src ? row_src : part + (int64_t)t * E;
  float* row = logits + (int64_t)t * E;
  uint32_t keys[VPL];
#pragma unroll (VPL <= 8 ? VPL : 1)
  for (int i = 0; i < VPL; ++i) {
    const int e = lane + 32 * i;
    uint32_t key = 0;
    if (e < E) {
      float v = (KS == 1 || row_src) ? row_in[e] : sum_partials(part, KS, (int64_t)T * E, (int64_t)t * E + e);
      if (v != v) nan_seen = true;
      if (!row_src && row != row_in) row[e] = v;
      if (v != v) v = -INFINITY;
      key = logit_key(v);
    }
    keys[i] = key;
  }
  if (__any_sync(kFull, nan_seen) && lane == 0) set_status(status, MOE_DEV_NAN_LOGIT);
  uint64_t taken = 0;
  float sel_v = 0.f;    // lane j keeps the j-th selected logit
  int sel_i = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0;
    int bi = 0x7fffffff;
#pragma unroll (VPL <= 8 ? VPL : 1)
    for (int i = 0; i < VPL; ++i)
      if (!(taken >> i & 1ull) && keys[i] > bk) { bk = keys[i]; bi = lane + 32 * i; }
    const uint32_t mk = __reduce_max_sync(kFull, bk);
    const int win = (int)__reduce_min_sync(kFull, bk == mk ? (uint32_t)bi : 0xffffffffu);
    if (win >= 0 && (win & 31) == lane) taken |= 1ull << (win >> 5);
    if (lane == j) { sel_v = key_logit(mk); sel_i = win; }
  }
  // softmax over the selected logits (lane j holds selection j); the first
  // selection is the maximum.
  float m = __shfl_sync(kFull, sel_v, 0);
  float p = lane < k ? expf(sel_v - m) : 0.f;
  float sum = 0.f;
  for (int j = 0; j < k; ++j) sum += __shfl_sync(kFull, p, j);   // slot order
  if (lane < k) {
    ids[(int64_t)t * k + lane] = sel_i;
    wts[(int64_t)t * k + lane] = p / sum * rs;
  }
}

// grid: ceil(T / 8), block 256 (warp per token).
template <int VPL>
__global__ void __launch_bounds__(256) k_topk(const float* __restrict__ part, int KS, int T, int E, int k, float rs,
                                              float* __restrict__ logits, int32_t* __restrict__ ids,
                                              float* __restrict__ wts, int32_t* status) {
  pdl_enter();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t < T) route_token<VPL>(t, lane, part, KS, T, E, k, rs, logits, ids, wts, status);
}

static void launch_topk(const float* part, int KS, int T, int E, int k, float rs, float* logits, int32_t* ids,
                        float* wts, int32_t* status, cudaStream_t st) {
  if (E <= 256)
    launch_pdl(k_topk<8>, dim3((T + 7) / 8), dim3(256), 0, st, part, KS, T, E, k, rs, logits, ids, wts, status);
  else
    launch_pdl(k_topk<64>, dim3((T + 7) / 8), dim3(256), 0, st, part, KS, T, E, k, rs, logits, ids, wts, status);
}

// ---------------------------------------------------------------------------
// S3: per-block histograms of the assignments of kTokBlk tokens, without
// atomics. grid NB = ceil(T / kTokBlk), one warp per block. The warp walks
// the block's assignments 32 at a time; lanes holding the same expert are
// grouped with __match_any_sync and the group's lowest lane adds the group
// size. Within one step the adding lanes hold distinct experts, and the
// steps follow one another, so every count is a plain sequence of integer
// additions. Invalid ids are skipped (and flagged); shared slots count for
// every token.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int assignment_expert(const int32_t* ids, int t, int j, int k, int E) {
  if (j >= k) return E + (j - k);
  int e = ids[(int64_t)t * k + j];
  return (e >= 0 && e < E) ? e : -1;
}

// Adds the experts of assignments [a0, a1) to cnt (one warp; cnt is private
// to the warp). Returns true on any lane that met an invalid id.
__device__ __forceinline__ bool warp_count(int a0, int a1, const int32_t* ids, int k, int kp, int E, int32_t* cnt) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  bool bad = false;
  for (int c = a0; c < a1; c += kWarp) {
    const int a = c + lane;
    const int e = a < a1 ? assignment_expert(ids, a / kp, a % kp, k, E) : -2;
    if (e == -1) bad = true;
    const unsigned m = __match_any_sync(kFull, e);
    if (e >= 0 && (m & lt) == 0) cnt[e] += __popc(m);
    __syncwarp();
  }
  return bad;
}

__global__ void __launch_bounds__(32) k_hist(const int32_t* __restrict__ ids, int T, int k, int kp, int E, int G,
                                             int32_t* __restrict__ hist, int32_t* status) {
  extern __shared__ int32_t sh[];
  for (int e = threadIdx.x; e < G; e += kWarp) sh[e] = 0;
  __syncwarp();
  const int t0 = blockIdx.x * kTokBlk, t1 = min(T, t0 + kTokBlk);
  const bool bad = warp_count(t0 * kp, t1 * kp, ids, k, kp, E, sh);
  if (__any_sync(kFull, bad) && threadIdx.x == 0) set_status(status, MOE_DEV_BAD_EXPERT_ID);
  __syncwarp();
  for (int e = threadIdx.x; e < G; e += kWarp) hist[(int64_t)blockIdx.x * G + e] = sh[e];
}

// Three block-wide exclusive scans in one pass (one set of barriers):
// a, b, c each hold n ints in shared memory; totals returned in ta, tb, tc.
// scratch >= 3 * 33 ints.
__device__ void block_excl_scan3(int32_t* a, int32_t* b, int32_t* c, int n, int32_t* scratch, int& ta, int& tb,
                                 int& tc) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int per = (n + nt - 1) / nt;
  const int lo = tid * per, hi = min(n, lo + per);
  int sa = 0, sb = 0, sc = 0;
  for (int i = lo; i < hi; ++i) { sa += a[i]; sb += b[i]; sc += c[i]; }
  const int lane = tid & 31, warp = tid >> 5;
  int ia = sa, ib = sb, ic = sc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ya = __shfl_up_sync(kFull, ia, o), yb = __shfl_up_sync(kFull, ib, o),
              yc = __shfl_up_sync(kFull, ic, o);
    if (lane >= o) { ia += ya; ib += yb; ic += yc; }
  }
  if (lane == 31) { scratch[warp] = ia; scratch[33 + warp] = ib; scratch[66 + warp] = ic; }
  __syncthreads();
  if (warp == 0) {
    const int nw = nt / 32;
    const int xa = lane < nw ? scratch[lane] : 0, xb = lane < nw ? scratch[33 + lane] : 0,
              xc = lane < nw ? scratch[66 + lane] : 0;
    int pa = xa, pb = xb, pc = xc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ya = __shfl_up_sync(kFull, pa, o), yb = __shfl_up_sync(kFull, pb, o),
                yc = __shfl_up_sync(kFull, pc, o);
      if (lane >= o) { pa += ya; pb += yb; pc += yc; }
    }
    if (lane < nw) { scratch[lane] = pa - xa; scratch[33 + lane] = pb - xb; scratch[66 + lane] = pc - xc; }
    if (lane == 31) { scratch[32] = pa; scratch[65] = pb; scratch[98] = pc; }
  }
  __syncthreads();
  int ra = scratch[warp] + ia - sa, rb = scratch[33 + warp] + ib - sb, rc = scratch[66 + warp] + ic - sc;
  for (int i = lo; i < hi; ++i) {
    const int va = a[i], vb = b[i], vc = c[i];
    a[i] = ra; b[i] = rb; c[i] = rc;
    ra += va; rb += vb; rc += vc;
  }
  ta = scratch[32]; tb = scratch[65]; tc = scratch[98];
  __syncthreads();
}

// From per-block histograms: counts, offsets, per-block bases, the list of
// groups with rows (increasing id), and padded offsets (kPadRows rows).
// One block of 1024 threads; smem: 3 * (G + 1) + 99 ints.
__device__ void scan_groups(const int32_t* hist, int NB, int G, int32_t* counts, int32_t* offsets,
                            int32_t* base, int32_t* touched, int32_t* n_touched, int32_t* poff, int32_t* sm) {
  int32_t* off = sm;               // [G + 1]
  int32_t* flag = sm + (G + 1);    // [G + 1]
  int32_t* pad = flag + (G + 1);   // [G + 1]
  int32_t* scr = pad + (G + 1);    // [99]
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    int c = 0;
    for (int b = 0; b < NB; ++b) c += hist[(int64_t)b * G + e];
    counts[e] = c;
    off[e] = c;
    flag[e] = c > 0;
    pad[e] = (c + kPadRows - 1) / kPadRows * kPadRows;
  }
  __syncthreads();
  int tot, ntouch, ptot;
  block_excl_scan3(off, flag, pad, G, scr, tot, ntouch, ptot);
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    offsets[e] = off[e];
    if (poff) poff[e] = pad[e];
    int c = counts[e];
    if (c > 0) touched[flag[e]] = e;
    if (base) {
      int run = off[e];
      for (int b = 0; b < NB; ++b) {
        base[(int64_t)b * G + e] = run;
        run += hist[(int64_t)b * G + e];
      }
    }
  }
  if (threadIdx.x == 0) {
    offsets[G] = tot;
    if (poff) poff[G] = ptot;
    *n_touched = ntouch;
  }
}

__global__ void __launch_bounds__(1024) k_scan(const int32_t* __restrict__ hist, int NB, int G,
                                               int32_t* counts, int32_t* offsets, int32_t* base,
                                               int32_t* touched, int32_t* n_touched, int32_t* poff,
                                               int32_t* zero, int64_t nzero) {
  extern __shared__ int32_t sm[];
  for (int64_t i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
  scan_groups(hist, NB, G, counts, offsets, base, touched, n_touched, poff, sm);
}

// ---------------------------------------------------------------------------
// S4: stable scatter. One warp walks the assignments of a token block in
// flat order, 32 at a time; equal experts inside a step are ranked with
// __match_any_sync, and a per-group cursor (starting at the block's base)
// advances after each step. Invalid ids leave inv = -1.
// ---------------------------------------------------------------------------
__device__ void scatter_warp(int a0, int a1, const int32_t* ids, const float* wts, int k, int kp, int E,
                             int32_t* cursor, int32_t* perm, int32_t* inv, float* w_row) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int c = a0; c < a1; c += kWarp) {
    const int a = c + lane;
    int e = -1;
    float wt = 0.f;
    if (a < a1) {
      int t = a / kp, j = a % kp;
      e = assignment_expert(ids, t, j, k, E);
      wt = j < k ? wts[(int64_t)t * k + j] : 1.0f;
    }
    const unsigned m = __match_any_sync(kFull, e);
    const int rank = __popc(m & lt);
    int basev = e >= 0 ? cursor[e] : 0;
    __syncwarp();
    if (e >= 0) {
      int r = basev + rank;
      perm[r] = a;
      inv[a] = r;
      w_row[r] = wt;
      if (rank == 0) cursor[e] = basev + __popc(m);
    } else if (a < a1) {
      inv[a] = -1;
    }
    __syncwarp();
  }
}

// grid NB, block 32; smem G ints.
__global__ void __launch_bounds__(32) k_scatter(const int32_t* __restrict__ ids, const float* __restrict__ wts, int T,
                                                int k, int kp, int E, int G, const int32_t* __restrict__ base,
                                                int32_t* perm, int32_t* inv, float* w_row) {
  extern __shared__ int32_t cursor[];
  for (int e = threadIdx.x; e < G; e += kWarp) cursor[e] = base[(int64_t)blockIdx.x * G + e];
  __syncwarp();
  const int t0 = blockIdx.x * kTokBlk, t1 = min(T, t0 + kTokBlk);
  scatter_warp(t0 * kp, t1 * kp, ids, wts, k, kp, E, cursor, perm, inv, w_row);
}

// ---------------------------------------------------------------------------
// MXFP8 quantisation of bf16 rows [rows, C] (C % 32 == 0) into codes
// [rows, C] and scales [rows, C/32]. Each lane takes 8 elements, four lanes a
// 32-element block. Grid-stride over (row, 256-element group).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void quant_group_bf16(const uint16_t* __restrict__ src, int64_t row, int C, int grp,
                                                 uint8_t* __restrict__ q, uint8_t* __restrict__ s, int lane) {
  const int c0 = grp * 256 + lane * 8;
  const bool ok = c0 < C;
  float v[8];
  if (ok) {
    uint4 raw = *reinterpret_cast<const uint4*>(src + row * C + c0);
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(w[i] << 16);
      v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
  }
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(v[i]));
  am = fmaxf(am, __shfl_xor_sync(kFull, am, 1));
  am = fmaxf(am, __shfl_xor_sync(kFull, am, 2));
  const int e = mx_exponent(am);
  const float sc = pow2_neg(e);
  if (ok) {
    uint32_t lo = (uint32_t)f32x2_to_e4m3x2(v[0] * sc, v[1] * sc) | ((uint32_t)f32x2_to_e4m3x2(v[2] * sc, v[3] * sc) << 16);
    uint32_t hi = (uint32_t)f32x2_to_e4m3x2(v[4] * sc, v[5] * sc) | ((uint32_t)f32x2_to_e4m3x2(v[6] * sc, v[7] * sc) << 16);
    *reinterpret_cast<uint2*>(q + row * C + c0) = make_uint2(lo, hi);
    if ((lane & 3) == 0) s[row * (C / 32) + c0 / 32] = (uint8_t)(e + 127);
  }
}

__global__ void __launch_bounds__(256) k_quant_rows_bf16(const uint16_t* __restrict__ src, int rows, int C,
                                                         uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
  const int lane = threadIdx.x & 31;
  const int groups = (C + 255) / 256;
  const int64_t total = (int64_t)rows * groups;
  const int64_t wid = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t i = wid; i < total; i += nw) quant_group_bf16(src, i / groups, C, (int)(i % groups), q, s, lane);
}

// S3-S4 for at most 32 assignments (a one-token batch, or T * k' <= 32),
// without histograms or scans: warp 0 holds one assignment a lane (its
// group, weight, how many assignments share the group, whether it is the
// group's first), and every thread of the block derives its groups' count,
// offset, padded offset and place in the touched list by one pass over
// those <= 32 entries. The rank of an assignment in its group is the number
// of lower lanes holding the same group, so the row order is the stable
// flat order the general path produces; every output equals that path's.
__device__ void route_tiny(int n, const int32_t* ids, const float* wts, int k, int kp, int E, int G,
                           int32_t* counts, int32_t* offsets, int32_t* touched, int32_t* n_touched, int32_t* poff,
                           int32_t* perm, int32_t* inv, float* w_row, int32_t* status) {
  __shared__ int32_t te[kWarp], tcnt[kWarp], tfirst[kWarp];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int e = -2;
  float wt = 0.f;
  unsigned m = 0;
  if (warp == 0) {
    if (lane < n) {
      const int t = lane / kp, j = lane % kp;
      e = assignment_expert(ids, t, j, k, E);
      wt = j < k ? wts[(int64_t)t * k + j] : 1.0f;
    }
    if (__any_sync(kFull, e == -1) && lane == 0) set_status(status, MOE_DEV_BAD_EXPERT_ID);
    m = __match_any_sync(kFull, e);
    te[lane] = e;
    tcnt[lane] = __popc(m);
    tfirst[lane] = e >= 0 && (m & ((1u << lane) - 1u)) == 0;
  }
  __syncthreads();
  for (int g = threadIdx.x; g <= G; g += blockDim.x) {
    int cnt = 0, off = 0, pof = 0, tix = 0;
    for (int b = 0; b < n; ++b) {
      const int eb = te[b];
      if (eb < 0) continue;
      if (eb == g) ++cnt;
      if (eb < g) {
        ++off;
        if (tfirst[b]) { pof += (tcnt[b] + kPadRows - 1) / kPadRows * kPadRows; ++tix; }
      }
    }
    offsets[g] = off;
    if (poff) poff[g] = pof;
    if (g < G) {
      counts[g] = cnt;
      if (cnt > 0) touched[tix] = g;
    } else {
      *n_touched = tix;
    }
  }
  if (warp == 0 && lane < n) {
    if (e >= 0) {
      int r = __popc(m & ((1u << lane) - 1u));
      for (int b = 0; b < n; ++b) r += te[b] >= 0 && te[b] < e;
      perm[r] = lane;
      inv[lane] = r;
      w_row[r] = wt;
    } else {
      inv[lane] = -1;
    }
  }
}

// ---------------------------------------------------------------------------
// Small-T fused path: block 0 sums the router partials (all threads), routes
// every token (warp per token), histograms, scans and scatters; blocks 1..
// quantise x meanwhile. One launch for all of S2-S4.
// The scatter splits the flat assignment list into one contiguous segment per
// warp: each warp counts its segment per group, a per-group prefix over the
// warps (in warp order) gives every warp its cursors, then each warp places its
// segment exactly as a single sequential pass would (stable in flat order).
// smem: G (histogram) + 3 (G + 1) + 99 (scan) + 32 G (per-warp cursors) ints,
// then the staged router partials when KS > 1.
// ---------------------------------------------------------------------------
template <int VPL>
__global__ void __launch_bounds__(1024, 1) k_route_small(const float* __restrict__ part, int KS, int T, int E, int k,
                                                      int kp, int G, float rs, int route, float* __restrict__ logits,
                                                      int32_t* ids, float* wts, int32_t* counts, int32_t* offsets,
                                                      int32_t* touched, int32_t* n_touched, int32_t* poff,
                                                      int32_t* perm, int32_t* inv, float* w_row,
                                                      const uint16_t* __restrict__ x, int H, uint8_t* xq,
                                                      uint8_t* xs, int32_t* status, int32_t* zero,
                                                      int64_t nzero) {
  extern __shared__ int32_t sm[];
  pdl_enter();
  if (blockIdx.x == 0)
    for (int64_t i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0;
  if (blockIdx.x > 0) {
    const int lane = threadIdx.x & 31;
    const int groups = (H + 255) / 256;
    const int64_t total = (int64_t)T * groups;
    const int64_t wid = (int64_t)(blockIdx.x - 1) * 32 + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)(gridDim.x - 1) * 32;
    for (int64_t i = wid; i < total; i += nw) quant_group_bf16(x, i / groups, H, (int)(i % groups), xq, xs, lane);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t* hist = sm;                    // [G]
  int32_t* scan_sm = sm + G;             // 3 (G + 1) + 99
  int32_t* wc = scan_sm + 3 * (G + 1) + 99;   // [32][G]
  if (route) {
    const float* src = part;
    if (KS > 1) {
      // stage every partial in shared memory with all loads in flight at
      // once, then sum each logit in ks order (the launcher only sends
      // KS * T * E <= kRouteStage floats here)
      const int n = T * E;
      float* stg = reinterpret_cast<float*>(wc + 32 * G);
      const int tot = n * KS;
      for (int i0 = 0; i0 < tot; i0 += 16 * 1024) {     // 16 loads in flight per thread
        float t[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int i = i0 + j * 1024 + threadIdx.x;
          t[j] = i < tot ? part[i] : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int i = i0 + j * 1024 + threadIdx.x;
          if (i < tot) stg[i] = t[j];
        }
      }
      __syncthreads();
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        float v = stg[i];
        int ks = 1;
        for (; ks + 8 <= KS; ks += 8) {
          float t8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) t8[j] = stg[(ks + j) * n + i];
#pragma unroll
          for (int j = 0; j < 8; ++j) v += t8[j];
        }
        for (; ks < KS; ++ks) v += stg[ks * n + i];
        logits[i] = v;
        stg[i] = v;                     // the routing below reads the sums from here
      }
      __syncthreads();
      for (int t = warp; t < T; t += 32)
        route_token<VPL>(t, lane, nullptr, 1, T, E, k, rs, logits, ids, wts, status, stg + (int64_t)t * E);
    } else {
      for (int t = warp; t < T; t += 32) route_token<VPL>(t, lane, src, 1, T, E, k, rs, logits, ids, wts, status);
    }
  }
  __syncthreads();   // ids / wts written by this block are visible block-wide
  const int n = T * kp;
  if (n <= kWarp) {
    route_tiny(n, ids, wts, k, kp, E, G, counts, offsets, touched, n_touched, poff, perm, inv, w_row, status);
    return;
  }
  // per-warp segment counts (atomic-free, see warp_count); the histogram is
  // their sum in warp order
  const int seg = ((n + 31) / 32 + 31) / 32 * 32;
  const int a0 = min(n, warp * seg), a1 = min(n, a0 + seg);
  int32_t* wcw = wc + warp * G;
  for (int e = lane; e < G; e += 32) wcw[e] = 0;
  __syncwarp();
  const bool bad = warp_count(a0, a1, ids, k, kp, E, wcw);
  if (__syncthreads_or(bad) && threadIdx.x == 0) set_status(status, MOE_DEV_BAD_EXPERT_ID);
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    int c = 0;
    for (int w = 0; w < 32; ++w) c += wc[w * G + e];
    hist[e] = c;
  }
  __syncthreads();
  scan_groups(hist, 1, G, counts, offsets, nullptr, touched, n_touched, poff, scan_sm);
  __syncthreads();
  // cursors: group offset plus the counts of the earlier warps
  for (int e = threadIdx.x; e < G; e += blockDim.x) {
    int run = scan_sm[e];
    for (int w = 0; w < 32; ++w) {
      const int c = wc[w * G + e];
      wc[w * G + e] = run;
      run += c;
    }
  }
  __syncthreads();
  scatter_warp(a0, a1, ids, wts, k, kp, E, wcw, perm, inv, w_row);
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static int router_tile(int T) { return T <= 16 ? 16 : 32; }

// H slices: about two CTAs per SM, each slice >= 128 rows (two W tiles), and
// at most 4096 partial rows (KS * T) to sum afterwards.
int router_splits(int T, int H, int E) {
  if (router_big(T, H, E)) return 1;
  if (router_mid(T, H, E)) {
    // at most one CTA per SM, slices of at least 64 rows, KS * T <= 4096
    const int tiles = ((T + kRbTT - 1) / kRbTT) * ((E + kRbTE - 1) / kRbTE);
    int ks = std::max(1, std::min(device_sms() / tiles, H / 64));
    return std::max(1, std::min(ks, 4096 / std::max(T, 1)));
  }
  if (router_rows(T, E)) {
    // about one CTA per SM, slices of at least 64 rows, KS * T <= 4096
    const int et = (E + 63) / 64;
    int ks = std::max(1, std::min(device_sms() / et, H / 64));
    return std::max(1, std::min(ks, 4096 / std::max(T, 1)));
  }
  const int tiles = ((T + router_tile(T) - 1) / router_tile(T)) * ((E + 63) / 64);
  int ks = (2 * device_sms() + tiles - 1) / std::max(tiles, 1);
  ks = std::max(1, std::min(ks, std::max(1, H / 128)));
  if ((int64_t)ks * T > 4096) ks = std::max(1, 4096 / std::max(T, 1));
  return ks;
}

cudaError_t launch_router(const uint16_t* x, const float* Wr, int T, int H, int E, int KS, float* part,
                          cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (KS == 1 && router_big(T, H, E)) {
    cudaError_t e = launch_pdl(k_router_big, dim3((T + kRbTT - 1) / kRbTT, (E + kRbTE - 1) / kRbTE), dim3(256), 0,
                               st, x, Wr, T, H, E, part);
    note_launch();
    return e;
  }
  if (router_mid(T, H, E)) {
    static std::atomic<bool> dm[kMaxDevices] = {};
    cudaError_t e = set_smem_once((const void*)k_router_mid, kRmSmem, dm);
    if (e == cudaSuccess)
      e = launch_pdl(k_router_mid, dim3((T + kRbTT - 1) / kRbTT, (E + kRbTE - 1) / kRbTE, KS), dim3(256), kRmSmem, st,
                     x, Wr, T, H, E, KS, part);
    note_launch();
    return e;
  }
  if (router_rows(T, E)) {
    static std::atomic<bool> dr1[kMaxDevices] = {}, dr8[kMaxDevices] = {}, dr16[kMaxDevices] = {}, dr32[kMaxDevices] = {};
    dim3 grid((E + 63) / 64, KS);
    cudaError_t e;
    if (T == 1) {
      e = set_smem_once((const void*)k_router_rows<1>, router_rows_smem<1>(), dr1);
      if (e == cudaSuccess)
        e = launch_pdl(k_router_rows<1>, grid, dim3(256), router_rows_smem<1>(), st, x, Wr, T, H, E, KS, part);
    } else if (T <= 8) {
      e = set_smem_once((const void*)k_router_rows<8>, router_rows_smem<8>(), dr8);
      if (e == cudaSuccess)
        e = launch_pdl(k_router_rows<8>, grid, dim3(256), router_rows_smem<8>(), st, x, Wr, T, H, E, KS, part);
    } else if (T <= 16) {
      e = set_smem_once((const void*)k_router_rows<16>, router_rows_smem<16>(), dr16);
      if (e == cudaSuccess)
        e = launch_pdl(k_router_rows<16>, grid, dim3(256), router_rows_smem<16>(), st, x, Wr, T, H, E, KS, part);
    } else {
      e = set_smem_once((const void*)k_router_rows<32>, router_rows_smem<32>(), dr32);
      if (e == cudaSuccess)
        e = launch_pdl(k_router_rows<32>, grid, dim3(256), router_rows_smem<32>(), st, x, Wr, T, H, E, KS, part);
    }
    note_launch();
    return e;
  }
  const int tt = router_tile(T);
  dim3 grid((T + tt - 1) / tt, (E + 63) / 64, KS);
  static std::atomic<bool> done16[kMaxDevices] = {}, done32[kMaxDevices] = {};
  cudaError_t e;
  if (tt == 16) {
    e = set_smem_once((const void*)k_router_partial<16>, router_smem<16>(), done16);
    if (e == cudaSuccess)
      e = launch_pdl(k_router_partial<16>, grid, dim3(256), router_smem<16>(), st, x, Wr, T, H, E, KS, part);
  } else {
    e = set_smem_once((const void*)k_router_partial<32>, router_smem<32>(), done32);
    if (e == cudaSuccess)
      e = launch_pdl(k_router_partial<32>, grid, dim3(256), router_smem<32>(), st, x, Wr, T, H, E, KS, part);
  }
  note_launch();
  return e;
}

static size_t small_smem(int G) { return (size_t)(G + 3 * (G + 1) + 99 + 32 * G) * 4; }

bool use_small_route(int T, int G, int kp) { return T <= 256 && T * kp <= 4096 && small_smem(G) <= 200 * 1024; }

template <int VPL>
static void launch_small(const RouteArgs& a, int kp, int G, int nq, cudaStream_t st) {
  size_t smem = small_smem(G);
  if (a.route && a.KS > 1) smem += (size_t)a.KS * a.T * a.E * 4;   // staged partials
  static std::atomic<bool> done[kMaxDevices] = {};
  set_smem_once((const void*)k_route_small<VPL>, 200 * 1024, done);
  launch_pdl(k_route_small<VPL>, dim3(1 + nq), dim3(1024), smem, st, a.part, a.KS, a.T, a.E, a.k, kp, G, a.rs,
             a.route ? 1 : 0, a.logits, a.ids, a.wts, a.counts, a.offsets, a.touched, a.n_touched, a.poff, a.perm,
             a.inv, a.w_row, a.x, a.H, a.xq, a.xs, a.status, a.zero, a.zero ? a.nzero : 0);
}

cudaError_t launch_route_dispatch(const RouteArgs& a, cudaStream_t st) {
  const int kp = a.k + a.S, G = a.E + a.S;
  const int T = a.T;
  if (use_small_route(T, G, kp) && (!a.route || a.KS == 1 || (int64_t)a.KS * T * a.E <= kRouteStage)) {
    int nq = T == 0 ? 0 : std::min(64, std::max(1, (T * ((a.H + 255) / 256) + 31) / 32));
    if (!a.x) nq = 0;
    if (a.E <= 256) launch_small<8>(a, kp, G, nq, st);
    else launch_small<64>(a, kp, G, nq, st);
    note_launch();
    return cudaGetLastError();
  }
  const int NB = (T + kTokBlk - 1) / kTokBlk;
  if (a.route) {
    launch_topk(a.part, a.KS, T, a.E, a.k, a.rs, a.logits, a.ids, a.wts, a.status, st);
    note_launch();
  }
  k_hist<<<NB, 32, G * 4, st>>>(a.ids, T, a.k, kp, a.E, G, a.hist, a.status);
  note_launch();
  size_t smem = (size_t)(3 * (G + 1) + 99) * 4;
  if (smem > 48 * 1024) cudaFuncSetAttribute(k_scan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  k_scan<<<1, 1024, smem, st>>>(a.hist, NB, G, a.counts, a.offsets, a.base, a.touched, a.n_touched, a.poff,
                                a.zero, a.zero ? a.nzero : 0);
  note_launch();
  k_scatter<<<NB, 32, G * 4, st>>>(a.ids, a.wts, T, a.k, kp, a.E, G, a.base, a.perm, a.inv, a.w_row);
  note_launch();
  if (a.x) {
    int groups = (a.H + 255) / 256;
    int64_t warps = (int64_t)T * groups;
    int blocks = (int)std::min<int64_t>((warps + 7) / 8, device_sms() * 16);
    k_quant_rows_bf16<<<blocks, 256, 0, st>>>(a.x, T, a.H, a.xq, a.xs);
    note_launch();
  }
  return cudaGetLastError();
}

// Router split-K partials -> logits -> top-k, one block per token: its
// threads sum the partials of the token's experts in ks order (each a
// handful of independent loads), write the logits out and keep them in
// shared memory, where its first warp routes the token. (Staging the
// partials through shared memory with 1024-thread blocks measured slower:
// 7.7 against 5.4 us a launch for 38 partials x 256 experts.)
template <int VPL>
__global__ void __launch_bounds__(256) k_sum_topk(const float* __restrict__ part, int KS, int T, int E, int k,
                                                  float rs, float* __restrict__ logits, int32_t* __restrict__ ids,
                                                  float* __restrict__ wts, int32_t* status) {
  __shared__ float lg[32 * VPL];
  pdl_enter();
  const int t = blockIdx.x;
  const int64_t n = (int64_t)T * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const float v = sum_partials(part, KS, n, (int64_t)t * E + e);
    logits[(int64_t)t * E + e] = v;
    lg[e] = v;
  }
  __syncthreads();
  if (threadIdx.x < 32) route_token<VPL>(t, threadIdx.x, nullptr, 1, T, E, k, rs, logits, ids, wts, status, lg);
}

cudaError_t launch_sum_topk(const float* part, int KS, int T, int E, int k, float rs, float* logits, int32_t* ids,
                            float* w, int32_t* status, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  cudaError_t e = E <= 256 ? launch_pdl(k_sum_topk<8>, dim3(T), dim3(256), 0, st, part, KS, T, E, k, rs, logits,
                                        ids, w, status)
                           : launch_pdl(k_sum_topk<64>, dim3(T), dim3(256), 0, st, part, KS, T, E, k, rs, logits,
                                        ids, w, status);
  note_launch();
  return e;
}

cudaError_t launch_topk_only(const float* logits, int T, int E, int k, float rs, int32_t* ids, float* w,
                             int32_t* status, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  launch_topk(logits, 1, T, E, k, rs, const_cast<float*>(logits), ids, w, status, st);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_quant_rows(const uint16_t* src, int rows, int C, uint8_t* q, uint8_t* s, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  int groups = (C + 255) / 256;
  int64_t warps = (int64_t)rows * groups;
  int blocks = (int)std::min<int64_t>((warps + 7) / 8, device_sms() * 16);
  k_quant_rows_bf16<<<blocks, 256, 0, st>>>(src, rows, C, q, s);
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
