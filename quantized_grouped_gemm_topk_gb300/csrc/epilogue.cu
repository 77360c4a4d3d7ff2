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
    for (int j = 0; j < kp; ++j) {
      const int r = inv[t * kp + j];
      if (r < 0) continue;
      const float4 v = sum_splits4(P, S, ss, (int64_t)r * N + n);
      const uint32_t lo = pack_bf16x2(v.x, v.y), hi = pack_bf16x2(v.z, v.w);
      if (z) *reinterpret_cast<uint2*>(z + (int64_t)r * N + n) = make_uint2(lo, hi);
      o0 += __uint_as_float(lo << 16);
      o1 += __uint_as_float(lo & 0xffff0000u);
      o2 += __uint_as_float(hi << 16);
      o3 += __uint_as_float(hi & 0xffff0000u);
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
// One CTA per padded 32-row block (grid-stride): the block's group is found
// once, the source row of each of its 32 rows is staged in shared memory,
// then the warps stride over 32-column chunks, lane = column: each lane
// gathers its column's 32 values (every row read is one coalesced 64-byte
// segment across the warp), quantises them along the row axis and writes
// 32 code bytes and its column's scale byte.
__global__ void __launch_bounds__(256) k_quant_cols(const ColQuantArgs a) {
  __shared__ int64_t src_row[32];
  __shared__ int blk_e;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int ncc = (a.C + 31) / 32;
  const int64_t npb = a.r_pad_max / 32;
  const int ptot = a.poff[a.G];
  for (int64_t pb = blockIdx.x; pb < npb; pb += gridDim.x) {
    const int prow = (int)(pb * 32);
    if (prow >= ptot) break;                 // blocks are visited in increasing order
    __syncthreads();                         // the previous block's staging is no longer read
    if (threadIdx.x == 0) {
      int lo = 0, hi = a.G - 1;              // group with poff[e] <= prow < poff[e+1]
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.poff[mid] <= prow) lo = mid; else hi = mid - 1;
      }
      blk_e = lo;
    }
    __syncthreads();
    const int e = blk_e;
    const int cnt = a.offsets[e + 1] - a.offsets[e];
    const int p0 = prow - a.poff[e];
    if (threadIdx.x < 32) {
      const int i = threadIdx.x;
      src_row[i] = p0 + i < cnt ? (int64_t)(a.row_map[a.offsets[e] + p0 + i] / a.row_div) : -1;
    }
    __syncthreads();
    for (int cc = warp; cc < ncc; cc += nwarps) {
      const int c = cc * 32 + lane;
      const bool cok = c < a.C;
      float v[32];
      float am = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int64_t sr = src_row[i];
        const float x = (cok && sr >= 0) ? bf16_bits_to_f32(a.src16[sr * a.C + c]) : 0.f;
        v[i] = x;
        am = fmaxf(am, fabsf(x));
      }
      if (!cok) continue;
      const int ex = mx_exponent(am);
      const float sc = pow2_neg(ex);
      uint32_t wds[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        wds[q] = (uint32_t)f32x2_to_e4m3x2(v[4 * q] * sc, v[4 * q + 1] * sc) |
                 ((uint32_t)f32x2_to_e4m3x2(v[4 * q + 2] * sc, v[4 * q + 3] * sc) << 16);
      }
      uint4* dst = reinterpret_cast<uint4*>(a.q + (int64_t)c * a.r_pad_max + prow);
      dst[0] = make_uint4(wds[0], wds[1], wds[2], wds[3]);
      dst[1] = make_uint4(wds[4], wds[5], wds[6], wds[7]);
      a.s[sf4_at(pb, c, a.C)] = (uint8_t)(ex + 127);
    }
  }
}

cudaError_t launch_quant_cols(const ColQuantArgs& a, cudaStream_t st) {
  if (a.r_pad_max == 0) return cudaSuccess;
  const int64_t npb = a.r_pad_max / 32;
  const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>(npb, (int64_t)device_sms() * 8));
  k_quant_cols<<<blocks, 256, 0, st>>>(a);
  note_launch();
  return cudaGetLastError();
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
