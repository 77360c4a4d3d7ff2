// Weight-gradient GEMMs and the one-time weight prepack.
//
// wgrad: out_e[m][n] = sum over the group's padded rows i of
//   P[m][poff_e + i] * Q[n][poff_e + i], both operands MXFP8-quantised along
//   the row axis (the transposed copies the forward and the backward
//   epilogues emit; NVIDIA blog "Boosting MoE training throughput with
//   advanced fusion kernels", MXFP8 quantisation with a transposed copy).
//   Groups without rows write zero gradients.
// prepack: GC-MoE summary, Developer notes: the caller converts the FP4
//   weights once into K-tiled prepacked form so the loader streams large
//   contiguous runs; NVIDIA blog, GLU epilogue fusion: gate and up columns
//   repacked so one tile holds half a tile of each.
#include "internal.cuh"

namespace moe {

constexpr int kWgT = 64;

__device__ __forceinline__ void load_mx_tile(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int64_t Rp,
                                             int rows, int r0, int64_t k0, float (*dst)[kWgT + 4], int tid) {
  // 64 rows x 32 codes: thread -> (row tid/4, 8 codes at (tid%4)*8)
  const int row = tid >> 2, kk = (tid & 3) * 8;
  float v[8];
  if (r0 + row < rows) {
    const uint2 c = *reinterpret_cast<const uint2*>(q + (int64_t)(r0 + row) * Rp + k0 + kk);
    const float sc = e8m0_to_f32(s[(int64_t)(r0 + row) * (Rp / 32) + k0 / 32]);
    float2 f;
    f = e4m3x2_to_f32x2((uint16_t)(c.x & 0xffffu)); v[0] = f.x * sc; v[1] = f.y * sc;
    f = e4m3x2_to_f32x2((uint16_t)(c.x >> 16));     v[2] = f.x * sc; v[3] = f.y * sc;
    f = e4m3x2_to_f32x2((uint16_t)(c.y & 0xffffu)); v[4] = f.x * sc; v[5] = f.y * sc;
    f = e4m3x2_to_f32x2((uint16_t)(c.y >> 16));     v[6] = f.x * sc; v[7] = f.y * sc;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) dst[kk + i][row] = v[i];
}

__global__ void __launch_bounds__(256) k_wgrad(const WgradArgs a) {
  __shared__ __align__(16) float As[32][kWgT + 4];
  __shared__ __align__(16) float Bs[32][kWgT + 4];
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  const int m0 = blockIdx.x * kWgT, n0 = blockIdx.y * kWgT, e = blockIdx.z;
  const int64_t p0 = a.poff[e], p1 = a.poff[e + 1];
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int64_t kb = p0; kb < p1; kb += 32) {
    __syncthreads();
    load_mx_tile(a.pq, a.ps, a.Rp, a.M, m0, kb, As, tid);
    load_mx_tile(a.qq, a.qs, a.Rp, a.N, n0, kb, Bs, tid);
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      const float4 av = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
      const float4 bv = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
      const float ar[4] = {av.x, av.y, av.z, av.w}, br[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
    }
  }
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < a.N) a.out[((int64_t)e * a.M + m) * a.N + n] = f32_to_bf16_bits(acc[i][j]);
    }
  }
}

cudaError_t launch_wgrad(const WgradArgs& a, cudaStream_t st) {
  dim3 grid((a.M + kWgT - 1) / kWgT, (a.N + kWgT - 1) / kWgT, a.G);
  k_wgrad<<<grid, 256, 0, st>>>(a);
  note_launch();
  return cudaGetLastError();
}

// ---- prepack ------------------------------------------------------------------
// One thread per (group, tile, chunk, packed row). Rows past N are zero.
__global__ void __launch_bounds__(256) k_prepack(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int G,
                                                 int N, int K, int fmt, int interleave_I, int tiles,
                                                 int64_t tile_bytes, uint8_t* __restrict__ dst) {
  const int nch = K / kChunkK;
  const int64_t total = (int64_t)G * tiles * nch * kTileN;
  const int CB = chunk_bytes(fmt);
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int p = (int)(idx % kTileN);
    int64_t rest = idx / kTileN;
    const int c = (int)(rest % nch);
    rest /= nch;
    const int j = (int)(rest % tiles);
    const int g = (int)(rest / tiles);
    int n;
    if (interleave_I > 0) n = p < 64 ? 64 * j + p : interleave_I + 64 * j + (p - 64);
    else n = kTileN * j + p;
    uint8_t* ch = dst + ((int64_t)g * tiles + j) * tile_bytes + (int64_t)c * CB;
    const bool ok = n < N;
    if (fmt == MOE_WFMT_NVFP4) {
      const uint8_t* row = q + ((int64_t)g * N + n) * (K / 2) + c * 32;
      const uint8_t* srow = s + ((int64_t)g * N + n) * (K / 16) + c * 4;
      for (int gi = 0; gi < 2; ++gi) {
        uint4 v = ok ? *reinterpret_cast<const uint4*>(row + gi * 16) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(ch + gi * 2048 + p * 16) = v;
      }
      uint32_t sc = 0;
      if (ok) sc = srow[0] | (srow[1] << 8) | (srow[2] << 16) | ((uint32_t)srow[3] << 24);
      *reinterpret_cast<uint32_t*>(ch + 4096 + p * 4) = sc;
    } else {
      const uint8_t* row = q + ((int64_t)g * N + n) * K + c * 64;
      const uint8_t* srow = s + ((int64_t)g * N + n) * (K / 32) + c * 2;
      for (int gi = 0; gi < 4; ++gi) {
        uint4 v = ok ? *reinterpret_cast<const uint4*>(row + gi * 16) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(ch + gi * 2048 + p * 16) = v;
      }
      uint16_t sc = ok ? (uint16_t)(srow[0] | (srow[1] << 8)) : (uint16_t)0;
      *reinterpret_cast<uint16_t*>(ch + 8192 + p * 2) = sc;
    }
  }
}

__global__ void __launch_bounds__(256) k_prepack_rowexp(const uint8_t* __restrict__ s, int G, int N, int K,
                                                        int interleave_I, int tiles, int8_t* __restrict__ dst) {
  const int64_t total = (int64_t)G * tiles * kTileN;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int p = (int)(idx % kTileN);
    const int j = (int)((idx / kTileN) % tiles);
    const int g = (int)(idx / ((int64_t)kTileN * tiles));
    int n;
    if (interleave_I > 0) n = p < 64 ? 64 * j + p : interleave_I + 64 * j + (p - 64);
    else n = kTileN * j + p;
    int mx = 127;
    if (n < N) {
      mx = 0;
      const uint8_t* row = s + ((int64_t)g * N + n) * (K / 32);
      for (int b = 0; b < K / 32; ++b) mx = max(mx, (int)row[b]);
    }
    dst[idx] = (int8_t)(mx - 127);
  }
}

cudaError_t launch_prepack_rowexp(const uint8_t* s, int G, int N, int K, int interleave_I, int tiles, int8_t* dst,
                                  cudaStream_t st) {
  const int64_t total = (int64_t)G * tiles * kTileN;
  if (total == 0) return cudaSuccess;
  int blocks = (int)std::min<int64_t>((total + 255) / 256, device_sms() * 32);
  k_prepack_rowexp<<<blocks, 256, 0, st>>>(s, G, N, K, interleave_I, tiles, dst);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_prepack(const uint8_t* q, const uint8_t* s, int G, int N, int K, int fmt, int interleave_I,
                           int tiles, int64_t tile_bytes, uint8_t* dst, cudaStream_t st) {
  const int64_t total = (int64_t)G * tiles * (K / kChunkK) * kTileN;
  if (total == 0) return cudaSuccess;
  int blocks = (int)std::min<int64_t>((total + 255) / 256, device_sms() * 32);
  k_prepack<<<blocks, 256, 0, st>>>(q, s, G, N, K, fmt, interleave_I, tiles, tile_bytes, dst);
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
