// Epilogues and the combine:
//  * W1 epilogue: y = w_row * SwiGLU(g, u), MXFP8 requantisation along I,
//    optional training saves (GC-MoE summary, Approach: SwiGLU, routing
//    weight and requantisation fused after W1; NVIDIA blog "Boosting MoE
//    training throughput with advanced fusion kernels", GLU epilogue fusion).
//  * W2 epilogue fused with the combine: z = bf16(W2 output), out[t] = sum
//    of the token's k' rows in slot order (GC-MoE summary, Approach: W2
//    emits BF16 fragments that role3 combines).
//  * transposed MXFP8 copies of gathered bf16 rows (same blog, MXFP8
//    quantisation with a transposed copy for the backward).
//  * the router backward.
#include "internal.cuh"

namespace moe {


// ---- W1 epilogue (NVFP4 path) --------------------------------------------------
// One CTA per row r: a warp per 32-block of I sums the K-slice partials,
// forms y = w_row * act(g, u) and quantises the block to MXFP8 (y1q, y1s).
// The CTA then writes the W2 GEMM's f16 operand row:
// y16[r][i] = E4M3 value * 2^(block exponent - row exponent), with
// y_rowexp[r] = the row's largest block exponent, exactly as the conversion
// pass k_act_f16 computes them from y1q / y1s. The row's codes and scales
// are staged in shared memory (I + I/32 bytes) until the row exponent is
// known, so y1 is not read back from memory.
__global__ void __launch_bounds__(1024) k_w1_finalize_rows(const W1FinArgs a) {
  extern __shared__ __align__(16) uint8_t fsm[];
  uint8_t* qs = fsm;            // [I] codes
  uint8_t* ss = fsm + a.I;      // [I / 32] scale codes
  __shared__ int wmax[32];
  pdl_enter();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int nb = a.I / 32;
  const int Rv = min(a.R, a.offsets[a.G]);
  const int64_t r = blockIdx.x;
  if (r >= Rv) return;
  const float* P = a.P + r * (a.gated ? 2 : 1) * a.I;   // W1's outputs of row r (sReLU: I, no up half)
  const float wr = a.w_row[r];
  const float* bg = nullptr;   // W1 bias of the row's group (the last e with offsets[e] <= r owns row r)
  if (a.b1) {
    int lo = 0, hi = a.G - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.offsets[mid] <= r) lo = mid; else hi = mid - 1;
    }
    bg = a.b1 + (int64_t)lo * 2 * a.I;
  }
  int mx = 0;
  for (int b = warp; b < nb; b += nwarps) {
    const int i = b * 32 + lane;
    float g = 0.f, u = 0.f;
    float y;
    if (a.gated) {
#pragma unroll 4
      for (int s = 0; s < a.S; ++s) {
        g += P[(int64_t)s * a.split_stride + i];
        u += P[(int64_t)s * a.split_stride + a.I + i];
      }
      if (bg) {
        g += bg[i];
        u += bg[a.I + i];
      }
      y = wr * act_fwd(g, u, a.act);
    } else {
#pragma unroll 4
      for (int s = 0; s < a.S; ++s) g += P[(int64_t)s * a.split_stride + i];
      y = wr * act_plain(g);
    }
    const int e = mx_exponent(warp_max(fabsf(y)));
    const uint8_t c = (uint8_t)(f32x2_to_e4m3x2(y * pow2_neg(e), 0.f) & 0xffu);
    a.y1q[r * a.I + i] = c;
    qs[i] = c;
    if (lane == 0) {
      a.y1s[r * nb + b] = (uint8_t)(e + 127);
      ss[b] = (uint8_t)(e + 127);
    }
    mx = max(mx, e + 127);
  }
  if (lane == 0) wmax[warp] = mx;
  __syncthreads();
  mx = wmax[0];
  for (int w = 1; w < nwarps; ++w) mx = max(mx, wmax[w]);
  if (threadIdx.x == 0) a.y_rowexp[r] = mx - 127;
  for (int c0 = threadIdx.x * 8; c0 < a.I; c0 += blockDim.x * 8) {
    const float f = ldexpf(1.0f, (int)ss[c0 / 32] - mx);
    const uint2 codes = *reinterpret_cast<const uint2*>(qs + c0);
    uint32_t outw[4];
    const uint32_t cw[2] = {codes.x, codes.y};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float2 lo = e4m3x2_to_f32x2((uint16_t)(cw[h] & 0xffffu));
      const float2 hi = e4m3x2_to_f32x2((uint16_t)(cw[h] >> 16));
      const __half2 h0 = __floats2half2_rn(lo.x * f, lo.y * f);
      const __half2 h1 = __floats2half2_rn(hi.x * f, hi.y * f);
      outw[2 * h] = *reinterpret_cast<const uint32_t*>(&h0);
      outw[2 * h + 1] = *reinterpret_cast<const uint32_t*>(&h1);
    }
    *reinterpret_cast<uint4*>(a.y16 + r * a.I + c0) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
  }
}

cudaError_t launch_w1_finalize(const W1FinArgs& a, cudaStream_t st) {
  if (a.R == 0) return cudaSuccess;
  if (!a.y16 || !a.y_rowexp) return cudaErrorInvalidValue;
  const size_t smem = (size_t)a.I + a.I / 32;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_w1_finalize_rows, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  // few rows (decode): a 1024-thread CTA per row spreads a row's blocks over
  // 32 warps; many rows: 256 threads per row
  cudaError_t e = launch_pdl(k_w1_finalize_rows, dim3(a.R), dim3(a.R < 4 * device_sms() ? 1024 : 256), smem, st, a);
  note_launch();
  return e;
}

// ---- W2 epilogue + combine --------------------------------------------------
__device__ __forceinline__ float4 sum_splits4(const float* P, int S, int64_t ss, int64_t off) {
  float4 v = *reinterpret_cast<const float4*>(P + off);
  for (int s = 1; s < S; ++s) {
    const float4 w = *reinterpret_cast<const float4*>(P + (int64_t)s * ss + off);
    v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
  }
  return v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  return (uint32_t)f32_to_bf16_bits(a) | ((uint32_t)f32_to_bf16_bits(b) << 16);
}

// One thread per (token, 4 columns): its slots' row indices, then every
// slot's row values, are requested eight slots at a time before any is used
// (two memory round trips a batch instead of two a slot); the sums are the
// ones below in the same order: each row's splits in s order, the slots'
// bf16-rounded rows in slot order.
__global__ void __launch_bounds__(256) k_finalize_combine(const float* __restrict__ P, int S, int64_t ss, int N,
                                                          const int32_t* __restrict__ inv, int T, int kp,
                                                          uint16_t* __restrict__ z, uint16_t* __restrict__ out) {
  pdl_enter();
  const int nq = N / 4;
  const int64_t total = (int64_t)T * nq;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = idx / nq;
    const int n = (int)(idx % nq) * 4;
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
    for (int j0 = 0; j0 < kp; j0 += 8) {
      int r[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) r[b] = j0 + b < kp ? inv[t * kp + j0 + b] : -1;
      float4 v[8];
#pragma unroll
      for (int b = 0; b < 8; ++b)
        v[b] = r[b] >= 0 ? *reinterpret_cast<const float4*>(P + (int64_t)r[b] * N + n) : make_float4(0.f, 0.f, 0.f, 0.f);
      for (int sp = 1; sp < S; ++sp) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if (r[b] < 0) continue;
          const float4 w = *reinterpret_cast<const float4*>(P + (int64_t)sp * ss + (int64_t)r[b] * N + n);
          v[b].x += w.x; v[b].y += w.y; v[b].z += w.z; v[b].w += w.w;
        }
      }
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        if (r[b] < 0) continue;
        const uint32_t lo = pack_bf16x2(v[b].x, v[b].y), hi = pack_bf16x2(v[b].z, v[b].w);
        if (z) *reinterpret_cast<uint2*>(z + (int64_t)r[b] * N + n) = make_uint2(lo, hi);
        o0 += __uint_as_float(lo << 16);
        o1 += __uint_as_float(lo & 0xffff0000u);
        o2 += __uint_as_float(hi << 16);
        o3 += __uint_as_float(hi & 0xffff0000u);
      }
    }
    *reinterpret_cast<uint2*>(out + t * N + n) = make_uint2(pack_bf16x2(o0, o1), pack_bf16x2(o2, o3));
  }
}

cudaError_t launch_finalize_combine(const float* P, int S, int64_t ss, int N, const int32_t* inv, int T, int kp,
                                    uint16_t* z, uint16_t* out, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  int64_t threads = (int64_t)T * (N / 4);
  int blocks = (int)std::min<int64_t>((threads + 255) / 256, device_sms() * 16);
  cudaError_t e = launch_pdl(k_finalize_combine, dim3(blocks), dim3(256), 0, st, P, S, ss, N, inv, T, kp, z, out);
  note_launch();
  return e;
}

__global__ void __launch_bounds__(256) k_finalize_rows(const float* __restrict__ P, int S, int64_t ss, int N, int R,
                                                       uint16_t* __restrict__ z) {
  const int nq = N / 4;
  const int64_t total = (int64_t)R * nq;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = idx / nq;
    const int n = (int)(idx % nq) * 4;
    const float4 v = sum_splits4(P, S, ss, r * N + n);
    *reinterpret_cast<uint2*>(z + r * N + n) = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

cudaError_t launch_finalize_rows(const float* P, int S, int64_t ss, int N, int R, uint16_t* z, cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  int64_t threads = (int64_t)R * (N / 4);
  int blocks = (int)std::min<int64_t>((threads + 255) / 256, device_sms() * 16);
  k_finalize_rows<<<blocks, 256, 0, st>>>(P, S, ss, N, R, z);
  note_launch();
  return cudaGetLastError();
}

__global__ void __launch_bounds__(256) k_combine(const uint16_t* __restrict__ z, const int32_t* __restrict__ inv,
                                                 const float* __restrict__ topk_w, int T, int k, int kp, int H,
                                                 uint16_t* __restrict__ out) {
  const int nq = H / 4;
  const int64_t total = (int64_t)T * nq;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = idx / nq;
    const int n = (int)(idx % nq) * 4;
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
    for (int j = 0; j < kp; ++j) {
      const int r = inv[t * kp + j];
      if (r < 0) continue;
      const float c = (topk_w && j < k) ? topk_w[t * k + j] : 1.0f;
      const uint2 v = *reinterpret_cast<const uint2*>(z + (int64_t)r * H + n);
      o0 = fmaf(c, __uint_as_float(v.x << 16), o0);
      o1 = fmaf(c, __uint_as_float(v.x & 0xffff0000u), o1);
      o2 = fmaf(c, __uint_as_float(v.y << 16), o2);
      o3 = fmaf(c, __uint_as_float(v.y & 0xffff0000u), o3);
    }
    *reinterpret_cast<uint2*>(out + t * H + n) = make_uint2(pack_bf16x2(o0, o1), pack_bf16x2(o2, o3));
  }
}

cudaError_t launch_combine(const uint16_t* z, const int32_t* inv, const float* topk_w, int T, int k, int kp, int H,
                           uint16_t* out, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  int64_t threads = (int64_t)T * (H / 4);
  int blocks = (int)std::min<int64_t>((threads + 255) / 256, device_sms() * 16);
  k_combine<<<blocks, 256, 0, st>>>(z, inv, topk_w, T, k, kp, H, out);
  note_launch();
  return cudaGetLastError();
}

// ---- transposed MXFP8 copies ---------------------------------------------------
// Work items are (128-row block, 128-column tile) pairs, row-block major.
// Groups are padded to multiples of 128 rows, so a row block lies in one
// group. A persistent CTA takes an even share of the items: it first finds,
// for each row block its share touches (at most kQcMaxRb; one warp per block),
// the block's group (the lanes count the groups whose padded start is <= the
// block's first row) and the source row of each of its 128 rows. It then
// streams its tiles through a three-stage cp.async ring in shared memory
// without a break at row-block boundaries (a warp copies two 256-byte row
// segments per request; pad rows and columns past C are zero-filled). In the
// ring, the 16-byte chunk k of row r sits at chunk k ^ 2(r / 32), so that the
// reads below are free of bank conflicts. Lane l of warp w owns the column
// pair 2(8w + l/4) and the 32-row block l % 4: it reads 32 words (both
// columns' values of its 32 rows), quantises each column along the row axis
// and writes its 2 x 32 code bytes; the four lanes of a pair fill whole
// 128-byte lines, and the first of them writes the pair's two scale words
// (one byte per 32-row block).
constexpr int kQcRows = 128, kQcCols = 128, kQcStages = 3, kQcMaxRb = 8;
constexpr int kQcRowBytes = kQcCols * 2;
constexpr int kQcTileBytes = kQcRows * kQcRowBytes;
constexpr int kQcSmem = kQcStages * kQcTileBytes + kQcMaxRb * kQcRows * 4;

// Elementwise max of |a| and |b| over the two bf16 halves; the result's sign
// bits are those of a xor b (callers mask them off). A NaN half yields the
// other input's half.
__device__ __forceinline__ uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// 32 bytes to a 32-byte aligned global address in one store.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

__device__ __forceinline__ void st_codes32(uint8_t* p, const uint32_t* v, bool a32) {
  if (a32) {
    st_global_v8(p, v);
  } else {
    uint4* d = reinterpret_cast<uint4*>(p);
    d[0] = make_uint4(v[0], v[1], v[2], v[3]);
    d[1] = make_uint4(v[4], v[5], v[6], v[7]);
  }
}

__global__ void __launch_bounds__(256, 2) k_quant_cols(const ColQuantArgs a) {
  extern __shared__ __align__(128) uint8_t qsm[];
  int* src_row = reinterpret_cast<int*>(qsm + kQcStages * kQcTileBytes);   // [kQcMaxRb][kQcRows]
  const int nct = (a.C + kQcCols - 1) / kQcCols;
  const int64_t nitem = (int64_t)(__ldg(&a.poff[a.G]) / kQcRows) * nct;
  const int64_t i0 = (int64_t)blockIdx.x * nitem / gridDim.x;
  const int njob = (int)((int64_t)(blockIdx.x + 1) * nitem / gridDim.x - i0);
  if (njob <= 0) return;
  const int rb0 = (int)(i0 / nct);
  const int ct_first = (int)(i0 - (int64_t)rb0 * nct);
  // row blocks of the share; the launch sizes the grid so that this is at
  // most kQcMaxRb (items beyond that are left out rather than misread)
  const int nrb = min((ct_first + njob - 1) / nct + 1, kQcMaxRb);
  const int njob_ok = min(njob, nrb * nct - ct_first);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (warp < nrb) {
    const int prow = (rb0 + warp) * kQcRows;
    int n = 0;                               // groups e < G with poff[e] <= prow
    for (int j = lane; j < a.G; j += 32) n += __ldg(&a.poff[j]) <= prow;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    const int e = n - 1;
    const int off = __ldg(&a.offsets[e]);
    const int cnt = __ldg(&a.offsets[e + 1]) - off;
    const int p0 = prow - __ldg(&a.poff[e]);
#pragma unroll
    for (int i = lane; i < kQcRows; i += 32)
      src_row[warp * kQcRows + i] = p0 + i < cnt ? __ldg(&a.row_map[off + p0 + i]) / a.row_div : -1;
  }
  __syncthreads();
  // Copies: thread t takes chunk t % 16 of rows t / 16 + 16k, k < 8; row r's
  // chunk lands at chunk ^ 2(r / 32) = chunk ^ (k & 6). The copy cursor
  // (row block, column tile, stage) runs two tiles ahead of the compute one.
  const int ch = threadIdx.x & 15;
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(qsm) + (uint32_t)((threadIdx.x >> 4) * kQcRowBytes);
  int cp_rb = 0, cp_ct = ct_first, cp_st = 0;
  auto issue_next = [&]() {
    const int c = cp_ct * kQcCols + ch * 8;
    const bool cok = c < a.C;
    const int* rows = src_row + cp_rb * kQcRows + (threadIdx.x >> 4);
    const uint32_t st = sbase + (uint32_t)(cp_st * kQcTileBytes);
#pragma unroll
    for (int k = 0; k < kQcRows / 16; ++k) {
      const int sr = rows[16 * k];
      const bool ok = cok && sr >= 0;
      cp_async16_zfill(st + (uint32_t)(16 * k * kQcRowBytes + ((ch ^ (k & 6)) << 4)),
                       ok ? a.src16 + (int64_t)sr * a.C + c : a.src16, ok);
    }
    if (++cp_ct == nct) { cp_ct = 0; ++cp_rb; }
    if (++cp_st == kQcStages) cp_st = 0;
  };
  const int rb = lane & 3;                   // 32-row block within the 128 rows
  const int cl = (warp * 8 + (lane >> 2)) * 2;  // even tile-local column
  const uint32_t roff = (uint32_t)(rb * 32 * kQcRowBytes + ((((cl >> 3) ^ (rb * 2))) << 4) + (cl & 7) * 2);
  const bool a32 = (reinterpret_cast<uintptr_t>(a.q) & 31) == 0;
  int q_rb = 0, q_ct = ct_first, q_st = 0;
  issue_next();
  cp_async_commit();
  if (njob_ok > 1) issue_next();
  cp_async_commit();
  for (int j = 0; j < njob_ok; ++j) {
    if (j + 2 < njob_ok) issue_next();       // into the stage read two tiles ago
    cp_async_commit();
    cp_async_wait<2>();                      // this thread's copies of tile j have landed
    __syncthreads();                         // ... and every other thread's
    const uint8_t* src = qsm + q_st * kQcTileBytes + roff;
    uint32_t w[32];                          // bf16 pairs: column cl (low half), cl + 1 (high half)
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = *reinterpret_cast<const uint32_t*>(src + i * kQcRowBytes);
    // |max| of each half over the 32 rows, four chains; signs of the result are dropped
    uint32_t m[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 32; ++i) m[i & 3] = bf16x2_absmax(m[i & 3], w[i]);
    const uint32_t mm = bf16x2_absmax(bf16x2_absmax(m[0], m[1]), bf16x2_absmax(m[2], m[3]));
    const int ex0 = mx_exponent(__uint_as_float((mm << 16) & 0x7fffffffu));
    const int ex1 = mx_exponent(__uint_as_float(mm & 0x7fff0000u));
    uint32_t s0 = 0, s1 = 0;                 // the pair's scale words, bytes in 32-row block order
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      s0 |= (uint32_t)(__shfl_sync(0xffffffffu, ex0, (lane & ~3) + r) + 127) << (8 * r);
      s1 |= (uint32_t)(__shfl_sync(0xffffffffu, ex1, (lane & ~3) + r) + 127) << (8 * r);
    }
    const int prow = (rb0 + q_rb) * kQcRows;
    const int c = q_ct * kQcCols + cl;
    if (c < a.C) {                           // C is a multiple of 8: c + 1 < C too
      const float2 sc = make_float2(pow2_neg(ex0), pow2_neg(ex1));
      uint32_t q0[8], q1[8];                 // codes of column cl, cl + 1: four rows per word
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 ya = __fmul2_rn(make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u)), sc);
        const float2 yb =
            __fmul2_rn(make_float2(__uint_as_float(w[i + 1] << 16), __uint_as_float(w[i + 1] & 0xffff0000u)), sc);
        const uint32_t p0 = f32x2_to_e4m3x2(ya.x, yb.x), p1 = f32x2_to_e4m3x2(ya.y, yb.y);
        if (i & 2) {
          q0[i >> 2] |= p0 << 16;
          q1[i >> 2] |= p1 << 16;
        } else {
          q0[i >> 2] = p0;
          q1[i >> 2] = p1;
        }
      }
      uint8_t* d0 = a.q + (int64_t)c * a.r_pad_max + prow + rb * 32;
      st_codes32(d0, q0, a32);
      st_codes32(d0 + a.r_pad_max, q1, a32);
      if (rb == 0)
        *reinterpret_cast<uint2*>(reinterpret_cast<uint32_t*>(a.s) + (int64_t)(prow / kQcRows) * a.C + c) =
            make_uint2(s0, s1);
    }
    if (++q_ct == nct) { q_ct = 0; ++q_rb; }
    if (++q_st == kQcStages) q_st = 0;
    __syncthreads();                         // the stage is refilled two iterations on
  }
}

cudaError_t launch_quant_cols(const ColQuantArgs& a, cudaStream_t st) {
  if (a.r_pad_max == 0) return cudaSuccess;
  if (a.C % 8 || a.r_pad_max % kQcRows) return cudaErrorInvalidValue;
  // Two CTAs per SM, or more when a share would span more than kQcMaxRb row
  // blocks: a share of ceil(nrb * nct / grid) <= (kQcMaxRb - 1) * nct items
  // touches at most kQcMaxRb row blocks.
  const int64_t nrb = a.r_pad_max / kQcRows;
  const int64_t grid = std::max<int64_t>(2 * device_sms(), (nrb + kQcMaxRb - 2) / (kQcMaxRb - 1));
  cudaError_t e = cudaFuncSetAttribute(k_quant_cols, cudaFuncAttributeMaxDynamicSharedMemorySize, kQcSmem);
  if (e != cudaSuccess) return e;
  k_quant_cols<<<(unsigned)grid, 256, kQcSmem, st>>>(a);
  note_launch();
  return cudaGetLastError();
}

// ---- W1 bias gradient ----------------------------------------------------------
// db[e][c] = sum over group e's padded 32-row blocks b, in block order, of
// part[b][c] (the dActivation epilogue's per-warp column sums of dh; pad
// rows hold zeros). Grid (column slices, G); a group without rows gets 0.
__global__ void __launch_bounds__(256) k_bias_grad(const float* __restrict__ part, int N,
                                                   const int32_t* __restrict__ poff, float* __restrict__ db) {
  pdl_enter();
  const int e = blockIdx.y;
  const int b0 = poff[e] / 32, b1 = poff[e + 1] / 32;
  for (int c = blockIdx.x * blockDim.x + threadIdx.x; c < N; c += gridDim.x * blockDim.x) {
    float acc = 0.f;
    for (int b = b0; b < b1; ++b) acc += part[(int64_t)b * N + c];
    db[(int64_t)e * N + c] = acc;
  }
}

cudaError_t launch_bias_grad(const float* part, int N, const int32_t* poff, int G, float* db, cudaStream_t st) {
  if (G == 0 || N == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(k_bias_grad, dim3((unsigned)((N + 255) / 256), (unsigned)G), dim3(256), 0, st, part, N,
                             poff, db);
  note_launch();
  return e;
}

// ---- router backward: softmax-over-selected Jacobian ---------------------------
__global__ void __launch_bounds__(256) k_router_bwd(const float* __restrict__ topk_w, const int32_t* __restrict__ ids,
                                                    const float* __restrict__ dwpart, int nparts, int64_t R,
                                                    const int32_t* __restrict__ inv, int T, int E, int k, int kp,
                                                    float rs, float* dlogits) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  for (int e = lane; e < E; e += 32) dlogits[(int64_t)t * E + e] = 0.f;
  float p = 0.f, dp = 0.f;
  if (lane < k) {
    p = topk_w[(int64_t)t * k + lane] / rs;
    const int r = inv[(int64_t)t * kp + lane];
    if (r >= 0) {
      float dw = 0.f;
      for (int i = 0; i < nparts; ++i) dw += dwpart[(int64_t)i * R + r];
      dp = rs * dw;
    }
  }
  float sdot = 0.f;
  for (int j = 0; j < k; ++j) sdot += __shfl_sync(kFull, p * dp, j);
  __syncwarp();
  if (lane < k) {
    const int e = ids[(int64_t)t * k + lane];
    if (e >= 0 && e < E) dlogits[(int64_t)t * E + e] = p * (dp - sdot);
  }
}

cudaError_t launch_router_bwd(const float* topk_w, const int32_t* ids, const float* dwpart, int nparts, int64_t R,
                              const int32_t* inv, int T, int E, int k, int kp, float rs, float* dlogits,
                              cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  k_router_bwd<<<(T + 7) / 8, 256, 0, st>>>(topk_w, ids, dwpart, nparts, R, inv, T, E, k, kp, rs, dlogits);
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
