// Device helpers shared by the routed-MoE kernels (sm_103a).
#pragma once
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xffffffffu;

// ---- packed weight blob ---------------------------------------------------
// NVFP4: tiles of 128 output features; each tile is a run of 64-wide K
// chunks.
//   chunk: [granule g < 2][row p < 128][16 B of 32 E2M1 codes] (4096 B)
//          then [row p][4 E4M3 scale codes, one per 16 K] (512 B).
// MXFP8 / MXFP4: plain K-major rows, codes [G][rows][K] (MXFP4: packed
//   E2M1 nibbles, [G][rows][K/2]) and scales in the SF4 layout (below) over
//   all groups' rows;
//   W1's forward rows come in tiles of 192: 96 gate features then the same
//   96 up features (zero rows past I), every other matrix in its own row
//   order.
constexpr int kTileN = 128;
constexpr int kChunkK = 64;
constexpr int kMxTileN = 192;
constexpr uint32_t kPackMagic = 0x4d4f4557u;  // 'MOEW'
constexpr int kPackVersion = 3;

__host__ __device__ inline int chunk_bytes(int fmt) {
  return fmt == MOE_WFMT_NVFP4 ? (4096 + 512) : (8192 + 256);
}

// MXFP8 packed row p of a matrix -> its logical row (-1: zero padding row).
// il > 0: W1 forward (I = il), tiles of 96 gate + 96 up features.
__host__ __device__ inline int mx_pack_src_row(int p, int N, int il) {
  if (il <= 0) return p < N ? p : -1;
  const int j = p / kMxTileN, pp = p % kMxTileN, h = kMxTileN / 2;
  const int f = j * h + (pp < h ? pp : pp - h);
  if (f >= il) return -1;
  return pp < h ? f : il + f;
}

// Token rows of every expert group are padded to a multiple of this in the
// transposed (token-axis) MXFP8 copies of the training path.
constexpr int kPadRows = 128;

// Scale layout of everything the block-scaled GEMM reads ("SF4"): 32-bit
// words [ceil(K / 128)][ld rows]; byte j of the word of (w, row) is the E8M0
// scale of K block 4 w + j of that row, so one coalesced 32-bit load per row
// brings a whole 128-wide K stage of scales. sf4_at: byte offset of K block
// kb of row; sf4_bytes: the array's size.
__host__ __device__ inline int64_t sf4_at(int64_t kb, int64_t row, int64_t ld) {
  return (((kb >> 2) * ld + row) << 2) + (kb & 3);
}
__host__ __device__ inline int64_t sf4_bytes(int64_t K, int64_t rows) { return (K / 32 + 3) / 4 * rows * 4; }

struct PackHeader {            // first 256 bytes of a packed blob
  uint32_t magic;
  int32_t version, fmt, which, G;
  int32_t N1, K1, N2, K2;      // logical rows / K of the two matrices
  int32_t interleave1;         // W1 gate/up interleave (I), 0 for none
  int64_t off_gs1, off_gs2, off_w1, off_w2;   // byte offsets from the blob start
  int64_t tile_bytes1, tile_bytes2;           // NVFP4: bytes of one 128-row tile
  int32_t tiles1, tiles2;                     // NVFP4: tiles per group
  int64_t off_s1, off_s2;                     // MXFP8: scale arrays
  int32_t rows1, rows2;                       // MXFP8: packed rows per group
  int64_t off_b1;                             // W1 bias [G][2I] fp32, 0 for none
};
static_assert(sizeof(PackHeader) <= 256, "pack header fits its 256 bytes");

// True when the blob's header describes the packing a GEMM expects.
__device__ __forceinline__ bool pack_header_ok(const PackHeader* h, int fmt, int which, int G, bool bias = false) {
  return h->magic == kPackMagic && h->version == kPackVersion && h->fmt == fmt && h->which == which && h->G == G &&
         (h->off_b1 != 0) == bias;
}

// ---- conversions ------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// E4M3 decode of one code (exact).
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}

// Two E4M3 codes -> two floats (low byte first).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t c2) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)c2, __NV_E4M3);
  return __half22float2(__half2(h));
}

// Round-to-nearest-even E4M3 of two floats (saturating); a -> low byte.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float a, float b) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// One byte holding two E2M1 codes -> two halfs (element 2i in the low nibble
// lands in the low half).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{ .reg .b8 t; cvt.u8.u32 t, %1; cvt.rn.f16x2.e2m1x2 %0, t; }" : "=r"(r) : "r"(byte));
  return r;
}

__device__ __forceinline__ float2 h2_bits_to_f2(uint32_t h2) {
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// E8M0 code -> 2^(c - 127) for c in [1, 254] (exact, normal fp32).
__device__ __forceinline__ float e8m0_to_f32(uint32_t c) {
  if (c == 0) return __uint_as_float(0x00400000u);   // 2^-127 (subnormal)
  return __uint_as_float(c << 23);
}

// Smallest integer e with amax <= 448 * 2^e, clamped to [-127, 127];
// -127 for amax == 0 (or any value below the normal range). Exact: 448 is
// 1.75 * 2^8, so for amax = 1.m * 2^E the answer is E - 8, plus one when
// 1.m > 1.75.
__device__ __forceinline__ int mx_exponent(float amax) {
  uint32_t b = __float_as_uint(amax) & 0x7fffffffu;
  int ex = (int)(b >> 23);
  if (ex == 0) return -127;
  int e = ex - 127 - 8 + ((b & 0x7fffffu) > 0x600000u ? 1 : 0);
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as fp32 for e in [-127, 121] (all finite block maxima land there).
__device__ __forceinline__ float pow2_neg(int e) {
  return __uint_as_float((uint32_t)(127 - e) << 23);
}

// ---- warp helpers -----------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// ---- activation ---------------------------------------------------------------
struct ActParams {
  int act;
  float alpha, limit;
};

// The non-gated activation: sReLU, max(h, 0)^2 of W1's I outputs.
__device__ __forceinline__ float act_plain(float h) {
  const float r = fmaxf(h, 0.f);
  return r * r;
}
// Its gradient: d * 2 max(h, 0).
__device__ __forceinline__ float act_plain_bwd(float h, float d) { return d * (2.f * fmaxf(h, 0.f)); }

// Logistic sigmoid with the fast exponential and divide intrinsics: relative
// error ~1e-6, far inside the layer's tolerance, and several times cheaper
// than the IEEE forms in the epilogues that evaluate it per element.
__device__ __forceinline__ float sigmoidf_(float v) { return __fdividef(1.0f, 1.0f + __expf(-v)); }

// Phi(v), the standard normal CDF, and phi(v), its density (CUDA's erff /
// expf).
__device__ __forceinline__ float normal_cdf(float v) { return 0.5f * (1.0f + erff(v * 0.70710678118654752f)); }
__device__ __forceinline__ float normal_pdf(float v) { return 0.39894228040143268f * expf(-0.5f * v * v); }

__device__ __forceinline__ float act_fwd(float g, float u, const ActParams& p) {
  if (p.act == MOE_ACT_SWIGLU) return g * sigmoidf_(g) * u;
  if (p.act == MOE_ACT_GEGLU) return g * normal_cdf(g) * u;
  float gc = fminf(fmaxf(g, -p.limit), p.limit);
  float uc = fminf(fmaxf(u, -p.limit), p.limit);
  return gc * sigmoidf_(p.alpha * gc) * uc;
}

// Gradients of d * act(g, u): returns (dg, du).
__device__ __forceinline__ float2 act_bwd(float g, float u, float d, const ActParams& p) {
  if (p.act == MOE_ACT_SWIGLU) {
    float s = sigmoidf_(g);
    return make_float2(d * (s + g * s * (1.0f - s)) * u, d * g * s);
  }
  if (p.act == MOE_ACT_GEGLU) {
    const float c = normal_cdf(g);
    return make_float2(d * (c + g * normal_pdf(g)) * u, d * g * c);
  }
  float gc = fminf(fmaxf(g, -p.limit), p.limit);
  float uc = fminf(fmaxf(u, -p.limit), p.limit);
  float s = sigmoidf_(p.alpha * gc);
  float dg = (g >= -p.limit && g <= p.limit) ? d * (s + p.alpha * gc * s * (1.0f - s)) * uc : 0.0f;
  float du = (u >= -p.limit && u <= p.limit) ? d * gc * s : 0.0f;
  return make_float2(dg, du);
}

// act(g, u) and the gradients (dg, du) of d * act(g, u) in one evaluation
// (the backward epilogue needs both; the sigmoid / normal CDF is computed
// once). Same values as act_fwd / act_bwd.
__device__ __forceinline__ float3 act_fwd_bwd(float g, float u, float d, const ActParams& p) {
  if (p.act == MOE_ACT_SWIGLU) {
    const float s = sigmoidf_(g);
    const float gs = g * s;
    return make_float3(gs * u, d * (s + gs * (1.0f - s)) * u, d * gs);
  }
  if (p.act == MOE_ACT_GEGLU) {
    const float c = normal_cdf(g);
    const float gc = g * c;
    return make_float3(gc * u, d * (c + g * normal_pdf(g)) * u, d * gc);
  }
  const float gc = fminf(fmaxf(g, -p.limit), p.limit);
  const float uc = fminf(fmaxf(u, -p.limit), p.limit);
  const float s = sigmoidf_(p.alpha * gc);
  const float gs = gc * s;
  const float dg = (g >= -p.limit && g <= p.limit) ? d * (s + p.alpha * gs * (1.0f - s)) * uc : 0.0f;
  const float du = (u >= -p.limit && u <= p.limit) ? d * gs : 0.0f;
  return make_float3(gs * uc, dg, du);
}

// Programmatic dependent launch. Every kernel of the forward chain first
// waits until the kernel before it on the stream has completed and its
// memory is visible (a no-op when it was launched without the attribute),
// then lets the next kernel of the chain be launched, so the next kernel's
// launch and CTA setup overlap this kernel's run instead of following it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() {
  pdl_wait();
  pdl_trigger();
}

// gpu-scope acquire load / release store of a flag another CTA sets or reads.
__device__ __forceinline__ int ld_acquire_gpu(const int32_t* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int32_t* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// gpu-scope atomic add with acquire and release semantics; returns the old
// value. After a CTA barrier, one thread's release publishes the writes of
// every thread that reached the barrier; after its acquire and a barrier,
// every thread sees what the releasing CTAs published.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
// Orders this thread's generic-proxy global accesses with its async-proxy
// (tensor copy) ones.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// 16-byte cp.async into shared memory (L2 only); with ok false the
// destination is zero-filled and nothing is read.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, bool ok) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(ok ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// Waits until at most N of this thread's committed groups are in flight.
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ void set_status(int32_t* status, int bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace moe
