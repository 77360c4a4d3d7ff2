// The one-time weight prepack and its inverse (a debug export of the packed
// layout back to plain rows).
//
// GC-MoE summary, Developer notes: the caller converts the FP4 weights once
// into K-tiled prepacked form so the loader streams large contiguous runs.
// NVIDIA blog "Boosting MoE training throughput with advanced fusion
// kernels", GLU epilogue section: gate and up columns are repacked so one
// tile holds half a tile of each, done once at checkpoint load.
#include "internal.cuh"

namespace moe {

// NVFP4 packed row p of tile j -> logical row (W1 forward: 64 gate + 64 up
// features per 128-row tile).
__host__ __device__ inline int nv_pack_src_row(int j, int p, int il) {
  if (il > 0) return p < 64 ? 64 * j + p : il + 64 * j + (p - 64);
  return kTileN * j + p;
}

// ---- NVFP4 ------------------------------------------------------------------
// One thread per (group, tile, chunk, packed row). Rows past N are zero.
__global__ void __launch_bounds__(256) k_prepack_nv(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                                                    int G, int N, int K, int interleave_I, int tiles,
                                                    int64_t tile_bytes, uint8_t* __restrict__ dst) {
  const int nch = K / kChunkK;
  const int64_t total = (int64_t)G * tiles * nch * kTileN;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int p = (int)(idx % kTileN);
    int64_t rest = idx / kTileN;
    const int c = (int)(rest % nch);
    rest /= nch;
    const int j = (int)(rest % tiles);
    const int g = (int)(rest / tiles);
    const int n = nv_pack_src_row(j, p, interleave_I);
    uint8_t* ch = dst + ((int64_t)g * tiles + j) * tile_bytes + (int64_t)c * chunk_bytes(MOE_WFMT_NVFP4);
    const bool ok = n < N;
    const uint8_t* row = q + ((int64_t)g * N + n) * (K / 2) + c * 32;
    const uint8_t* srow = s + ((int64_t)g * N + n) * (K / 16) + c * 4;
    for (int gi = 0; gi < 2; ++gi) {
      uint4 v = ok ? *reinterpret_cast<const uint4*>(row + gi * 16) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(ch + gi * 2048 + p * 16) = v;
    }
    uint32_t sc = 0;
    if (ok) sc = srow[0] | (srow[1] << 8) | (srow[2] << 16) | ((uint32_t)srow[3] << 24);
    *reinterpret_cast<uint32_t*>(ch + 4096 + p * 4) = sc;
  }
}

// Inverse: logical row n of group g, chunk c, back to [G][N][K/2] and
// [G][N][K/16].
__global__ void __launch_bounds__(256) k_unpack_nv(const uint8_t* __restrict__ src, int G, int N, int K,
                                                   int interleave_I, int tiles, int64_t tile_bytes,
                                                   uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
  const int nch = K / kChunkK;
  const int64_t total = (int64_t)G * N * nch;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(idx % nch);
    const int n = (int)((idx / nch) % N);
    const int g = (int)(idx / ((int64_t)nch * N));
    int j, p;
    if (interleave_I > 0) {
      const int f = n < interleave_I ? n : n - interleave_I;
      j = f / 64;
      p = (n < interleave_I ? 0 : 64) + f % 64;
    } else {
      j = n / kTileN;
      p = n % kTileN;
    }
    const uint8_t* ch = src + ((int64_t)g * tiles + j) * tile_bytes + (int64_t)c * chunk_bytes(MOE_WFMT_NVFP4);
    uint8_t* row = q + ((int64_t)g * N + n) * (K / 2) + c * 32;
    for (int gi = 0; gi < 2; ++gi)
      *reinterpret_cast<uint4*>(row + gi * 16) = *reinterpret_cast<const uint4*>(ch + gi * 2048 + p * 16);
    const uint32_t sc = *reinterpret_cast<const uint32_t*>(ch + 4096 + p * 4);
    uint8_t* srow = s + ((int64_t)g * N + n) * (K / 16) + c * 4;
    for (int b = 0; b < 4; ++b) srow[b] = (uint8_t)(sc >> (8 * b));
  }
}

// ---- MXFP8 / MXFP4 ------------------------------------------------------------
// Codes: one thread per (group, packed row, 16-byte piece), [G][NR][cb]
// (cb = K bytes for E4M3, K/2 for packed E2M1);
// scales: one thread per (group, packed row, 4-block word), in the SF4
// layout over all groups' rows (ld G * NR), so the GEMM's scale loaders read
// one coalesced word per row and stage. Padding rows are zero.
__global__ void __launch_bounds__(256) k_prepack_mx(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s,
                                                    int G, int N, int K, int64_t cb, int interleave_I, int NR,
                                                    uint8_t* __restrict__ dq, uint8_t* __restrict__ ds) {
  const int cpr = (int)(cb / 16), spr = K / 32;
  const int64_t total_c = (int64_t)G * NR * cpr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total_c; idx += stride) {
    const int c = (int)(idx % cpr);
    const int p = (int)((idx / cpr) % NR);
    const int g = (int)(idx / ((int64_t)cpr * NR));
    const int n = mx_pack_src_row(p, N, interleave_I);
    const uint4 v = n >= 0 ? *reinterpret_cast<const uint4*>(q + ((int64_t)g * N + n) * cb + c * 16)
                           : make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(dq + ((int64_t)g * NR + p) * cb + c * 16) = v;
  }
  // scales: one thread per (group, packed row, 4-block word)
  const int wpr = (spr + 3) / 4;
  const int64_t total_w = (int64_t)G * NR * wpr;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total_w; idx += stride) {
    const int p = (int)(idx % NR);
    const int w = (int)((idx / NR) % wpr);
    const int g = (int)(idx / ((int64_t)NR * wpr));
    const int n = mx_pack_src_row(p, N, interleave_I);
    uint32_t v = 0;
    if (n >= 0)
      for (int j = 0; j < 4 && 4 * w + j < spr; ++j) v |= (uint32_t)s[((int64_t)g * N + n) * spr + 4 * w + j] << (8 * j);
    reinterpret_cast<uint32_t*>(ds)[(int64_t)w * G * NR + (int64_t)g * NR + p] = v;
  }
}

// Inverse of k_prepack_mx for the logical rows n < N.
__global__ void __launch_bounds__(256) k_unpack_mx(const uint8_t* __restrict__ dq, const uint8_t* __restrict__ ds,
                                                   int G, int N, int K, int64_t cb, int interleave_I, int NR,
                                                   uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
  const int cpr = (int)(cb / 16), spr = K / 32;
  const int64_t total_c = (int64_t)G * N * cpr, total_s = (int64_t)G * N * spr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int h = kMxTileN / 2;
  auto packed_row = [&](int n) {
    if (interleave_I <= 0) return n;
    const int f = n < interleave_I ? n : n - interleave_I;
    return (f / h) * kMxTileN + (n < interleave_I ? 0 : h) + f % h;
  };
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total_c; idx += stride) {
    const int c = (int)(idx % cpr);
    const int n = (int)((idx / cpr) % N);
    const int g = (int)(idx / ((int64_t)cpr * N));
    const int p = packed_row(n);
    *reinterpret_cast<uint4*>(q + ((int64_t)g * N + n) * cb + c * 16) =
        *reinterpret_cast<const uint4*>(dq + ((int64_t)g * NR + p) * cb + c * 16);
  }
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total_s; idx += stride) {
    const int b = (int)(idx % spr);
    const int n = (int)((idx / spr) % N);
    const int g = (int)(idx / ((int64_t)spr * N));
    s[((int64_t)g * N + n) * spr + b] = ds[sf4_at(b, (int64_t)g * NR + packed_row(n), (int64_t)G * NR)];
  }
}

static int grid_of(int64_t total) {
  return (int)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, (int64_t)device_sms() * 32));
}

cudaError_t launch_prepack_nv(const uint8_t* q, const uint8_t* s, int G, int N, int K, int interleave_I, int tiles,
                              int64_t tile_bytes, uint8_t* dst, cudaStream_t st) {
  const int64_t total = (int64_t)G * tiles * (K / kChunkK) * kTileN;
  if (total == 0) return cudaSuccess;
  k_prepack_nv<<<grid_of(total), 256, 0, st>>>(q, s, G, N, K, interleave_I, tiles, tile_bytes, dst);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_unpack_nv(const uint8_t* src, int G, int N, int K, int interleave_I, int tiles, int64_t tile_bytes,
                             uint8_t* q, uint8_t* s, cudaStream_t st) {
  const int64_t total = (int64_t)G * N * (K / kChunkK);
  if (total == 0) return cudaSuccess;
  k_unpack_nv<<<grid_of(total), 256, 0, st>>>(src, G, N, K, interleave_I, tiles, tile_bytes, q, s);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_prepack_mx(const uint8_t* q, const uint8_t* s, int G, int N, int K, int64_t cb, int interleave_I,
                              int NR, uint8_t* dq, uint8_t* ds, cudaStream_t st) {
  const int64_t total = (int64_t)G * NR * (cb / 16);
  if (total == 0) return cudaSuccess;
  k_prepack_mx<<<grid_of(total), 256, 0, st>>>(q, s, G, N, K, cb, interleave_I, NR, dq, ds);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_unpack_mx(const uint8_t* dq, const uint8_t* ds, int G, int N, int K, int64_t cb, int interleave_I,
                             int NR, uint8_t* q, uint8_t* s, cudaStream_t st) {
  const int64_t total = (int64_t)G * N * (cb / 16);
  if (total == 0) return cudaSuccess;
  k_unpack_mx<<<grid_of(total), 256, 0, st>>>(dq, ds, G, N, K, cb, interleave_I, NR, q, s);
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
