// Grouped GEMM over prepacked block-scaled weights on the CUDA cores.
//
// Work unit = (group with rows, 128-feature tile, K slice); units are read
// from the device-side list of groups with rows, so no host sync is needed
// (NVIDIA blog "Boosting MoE training throughput with advanced fusion
// kernels", section on removing host-device sync and CPU launch overhead).
// Thread p of a block owns packed row p of the tile and reads its 16-byte
// granules, so a warp reads 512 contiguous bytes per granule. Activation
// rows of the group are staged in shared memory as fp32 (E4M3 value times
// its E8M0 block scale, exact) in groups of 8 rows.
//
// Arithmetic per output: for each 16-element (NVFP4) or 32-element (MXFP8)
// weight block, sum q_w * a in fp32, multiply by the block scale and add
// into the fp32 accumulator; finally times the group's fp32 scale.
#include "internal.cuh"

namespace moe {

constexpr int kTG = 8;      // activation rows per pass
constexpr int kCSub = 4;    // 64-wide K chunks per staged activation slab

__device__ __forceinline__ void fma_pair(float (&part)[kTG], float wa, float wb, const float* act_k) {
  const float4 a0 = *reinterpret_cast<const float4*>(act_k);
  const float4 a1 = *reinterpret_cast<const float4*>(act_k + 4);
  const float4 b0 = *reinterpret_cast<const float4*>(act_k + kTG);
  const float4 b1 = *reinterpret_cast<const float4*>(act_k + kTG + 4);
  part[0] = fmaf(wa, a0.x, fmaf(wb, b0.x, part[0]));
  part[1] = fmaf(wa, a0.y, fmaf(wb, b0.y, part[1]));
  part[2] = fmaf(wa, a0.z, fmaf(wb, b0.z, part[2]));
  part[3] = fmaf(wa, a0.w, fmaf(wb, b0.w, part[3]));
  part[4] = fmaf(wa, a1.x, fmaf(wb, b1.x, part[4]));
  part[5] = fmaf(wa, a1.y, fmaf(wb, b1.y, part[5]));
  part[6] = fmaf(wa, a1.z, fmaf(wb, b1.z, part[6]));
  part[7] = fmaf(wa, a1.w, fmaf(wb, b1.w, part[7]));
}

template <int FMT>
__global__ void __launch_bounds__(128) k_gemm_cc(const GemmArgs g) {
  __shared__ __align__(16) float act[kCSub * kChunkK * kTG];   // [k][row]
  const int p = threadIdx.x;
  const int nt = *g.n_touched;
  const int per_group = g.tiles * g.S;
  const int64_t units = (int64_t)nt * per_group;
  const int nchunks = g.K / kChunkK;
  const int CB = chunk_bytes(FMT);
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int ti = (int)(u / per_group), rem = (int)(u % per_group);
    const int j = rem / g.S, s = rem % g.S;
    const int e = g.touched[ti];
    const int r0 = g.offsets[e], r1 = g.offsets[e + 1];
    const int c0 = (int)((int64_t)s * nchunks / g.S), c1 = (int)((int64_t)(s + 1) * nchunks / g.S);
    int n;
    if (g.interleave_I > 0) n = p < 64 ? 64 * j + p : g.interleave_I + 64 * j + (p - 64);
    else n = kTileN * j + p;
    const bool nvalid = n < g.N;
    const uint8_t* tile = g.w + ((int64_t)e * g.tiles + j) * g.tile_bytes;
    const float gsv = g.gs ? g.gs[e] : 1.0f;
    for (int rg = r0; rg < r1; rg += kTG) {
      const int nr = min(kTG, r1 - rg);
      float acc[kTG];
#pragma unroll
      for (int i = 0; i < kTG; ++i) acc[i] = 0.f;
      for (int cs = c0; cs < c1; cs += kCSub) {
        const int ce = min(c1, cs + kCSub);
        const int klen = (ce - cs) * kChunkK;
        const int kq = klen / 4;
        __syncthreads();
        for (int idx = p; idx < kTG * kq; idx += blockDim.x) {
          const int i = idx / kq, kk = (idx % kq) * 4;
          float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
          if (i < nr) {
            const int r = rg + i;
            const int64_t src = g.row_map ? (int64_t)(g.row_map[r] / g.row_div) : (int64_t)r;
            const int kg = cs * kChunkK + kk;
            const uint32_t c4 = *reinterpret_cast<const uint32_t*>(g.aq + src * g.K + kg);
            const float sc = e8m0_to_f32(g.as[src * (g.K / 32) + kg / 32]);
            const float2 a01 = e4m3x2_to_f32x2((uint16_t)(c4 & 0xffffu));
            const float2 a23 = e4m3x2_to_f32x2((uint16_t)(c4 >> 16));
            v0 = a01.x * sc; v1 = a01.y * sc; v2 = a23.x * sc; v3 = a23.y * sc;
          }
          act[(kk + 0) * kTG + i] = v0;
          act[(kk + 1) * kTG + i] = v1;
          act[(kk + 2) * kTG + i] = v2;
          act[(kk + 3) * kTG + i] = v3;
        }
        __syncthreads();
        for (int c = cs; c < ce; ++c) {
          const uint8_t* ch = tile + (int64_t)c * CB;
          const float* ak = act + (c - cs) * kChunkK * kTG;
          if (FMT == MOE_WFMT_NVFP4) {
            const uint4 g0 = __ldg(reinterpret_cast<const uint4*>(ch + p * 16));
            const uint4 g1 = __ldg(reinterpret_cast<const uint4*>(ch + 2048 + p * 16));
            const uint32_t sc4 = __ldg(reinterpret_cast<const uint32_t*>(ch + 4096 + p * 4));
            const uint32_t wd[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int b = 0; b < 4; ++b) {            // blocks of 16 along K
              float part[kTG];
#pragma unroll
              for (int i = 0; i < kTG; ++i) part[i] = 0.f;
#pragma unroll
              for (int wi = 0; wi < 2; ++wi) {
                const uint32_t w = wd[b * 2 + wi];
#pragma unroll
                for (int bi = 0; bi < 4; ++bi) {
                  const float2 f = h2_bits_to_f2(e2m1x2_to_f16x2((w >> (8 * bi)) & 0xffu));
                  const int k = b * 16 + wi * 8 + bi * 2;
                  fma_pair(part, f.x, f.y, ak + k * kTG);
                }
              }
              const float sv = e4m3_to_f32((uint8_t)(sc4 >> (8 * b)));
#pragma unroll
              for (int i = 0; i < kTG; ++i) acc[i] = fmaf(sv, part[i], acc[i]);
            }
          } else {
            const uint16_t sc2 = __ldg(reinterpret_cast<const uint16_t*>(ch + 8192 + p * 2));
#pragma unroll
            for (int b = 0; b < 2; ++b) {            // blocks of 32 along K
              float part[kTG];
#pragma unroll
              for (int i = 0; i < kTG; ++i) part[i] = 0.f;
#pragma unroll
              for (int gi = 0; gi < 2; ++gi) {
                const uint4 gr = __ldg(reinterpret_cast<const uint4*>(ch + (b * 2 + gi) * 2048 + p * 16));
                const uint32_t wd[4] = {gr.x, gr.y, gr.z, gr.w};
#pragma unroll
                for (int wi = 0; wi < 4; ++wi) {
                  const float2 f0 = e4m3x2_to_f32x2((uint16_t)(wd[wi] & 0xffffu));
                  const float2 f1 = e4m3x2_to_f32x2((uint16_t)(wd[wi] >> 16));
                  const int k = b * 32 + gi * 16 + wi * 4;
                  fma_pair(part, f0.x, f0.y, ak + k * kTG);
                  fma_pair(part, f1.x, f1.y, ak + (k + 2) * kTG);
                }
              }
              const float sv = e8m0_to_f32((sc2 >> (8 * b)) & 0xffu);
#pragma unroll
              for (int i = 0; i < kTG; ++i) acc[i] = fmaf(sv, part[i], acc[i]);
            }
          }
        }
      }
      if (nvalid) {
        for (int i = 0; i < nr; ++i) g.out[(int64_t)s * g.split_stride + (int64_t)(rg + i) * g.N + n] = acc[i] * gsv;
      }
    }
  }
}

cudaError_t launch_gemm_cc(const GemmArgs& g, cudaStream_t st) {
  const int grid = std::max(1, g.max_ctas);
  if (g.fmt == MOE_WFMT_NVFP4) k_gemm_cc<MOE_WFMT_NVFP4><<<grid, 128, 0, st>>>(g);
  else k_gemm_cc<MOE_WFMT_MXFP8><<<grid, 128, 0, st>>>(g);
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
