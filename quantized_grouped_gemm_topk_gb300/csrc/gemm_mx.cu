// Block-scaled grouped GEMM for MXFP8 operands on the 5th-generation tensor
// cores: tcgen05.mma kind::mxf8f6f4 with scale_vec::1X multiplies E4M3
// operands read straight from shared memory, each scaled by one UE8M0 factor
// per 32 elements of K held in tensor memory, and accumulates in fp32 in
// tensor memory. Nothing is decoded: the MXFP8 bytes the quantisers write
// are the MMA's operands.
//
// NVIDIA blog "Boosting MoE training throughput with advanced fusion
// kernels": the kernel families GroupGemm + Activation + Quantize/Transpose
// (forward) and GroupGemm + dActivation + Quantize/Transpose (backward); the
// GLU epilogue section (the gate and up columns of one tile meet in the
// epilogue, so SwiGLU never round-trips through global memory); the MXFP8
// section (the epilogue writes the row-quantised output and its transposed
// MXFP8 copy for the weight gradients). GC-MoE summary, Approach: W1's
// epilogue applies SwiGLU, the routing weight and the FP8 requantisation.
//
// One kernel, four epilogues (template MODE):
//   kMxW1       h = x_e . W1_e; y = w_row * act(gate, up) -> MXFP8 rows y1,
//               optionally h (bf16) and the transposed MXFP8 copy of y.
//   kMxPlain    D -> bf16 rows (W2 forward; W1 dgrad).
//   kMxDswiglu  dY1 = dz_e . W2_e^T; dh = dact(h; w_row * dY1) -> MXFP8 rows
//               and the transposed MXFP8 copy; per-tile routing-weight
//               gradient partials sum(dY1 * act(h)). Gated: h and dh hold
//               2I a row (gate then up); sReLU: I a row.
//   kMxWgrad    dW_e = P_e^T . Q_e over the group's padded token rows
//               (variable K per group) -> bf16; a group with no rows writes
//               zeros.
// Tiles: 128 rows (MMA M: tokens of one group, or weight-gradient rows) x
// 192 columns (MMA N) x 128 K per stage (4 MMAs of K = 32). W1's weight rows
// are prepacked so a 192-column tile holds 96 gate features and the same 96
// up features.
//
// With clusters (kMxCl > 1), the CTAs of a cluster take consecutive
// 128-row tiles of the same group and the same 192-column B tile; each CTA
// copies its part of the B tile and multicasts it into all of them, and a
// stage slot is refilled only after the MMAs of every CTA released it.
// Roles (one CTA per SM, persistent over the work units):
//   warp 0       TMA producer: per stage one 2-D tensor copy of the A tile
//                and one of the B tile (or its cluster part, multicast),
//                128-byte swizzle, into a 5-stage ring.
//   warp 1       MMA issuer: per stage 4 block-scaled MMAs (fewer at a K
//                tail); commits free the stage and the scale slot; a tile's
//                last commit hands its accumulator to the epilogue. Also
//                allocates / frees tensor memory.
//   warps 4-7    scale loaders: per stage, one 32-bit word per A and B row
//                (the four E8M0 scales of the stage's K blocks, SF4 layout)
//                written to an 8-slot scale ring in tensor memory. Four
//                stages of words are loaded ahead into registers.
//   warps 8-15   two epilogue warpgroups; tiles alternate between them and
//                between the two accumulator buffers, so a tile's epilogue
//                overlaps the next tile's MMAs.
// Tensor memory: accumulators at columns [0, 192) and [192, 384); scale
// slot j at 384 + 12 j: one 4-column group for A's 128 rows, two for B's
// rows 0-127 and 128-191. Within a group, lane 32 q + r, column c holds the
// word of row 32 c + r, identically in all four lane quarters q (the image
// a 32-row x 128-bit copy replicated to the four quarters leaves, which the
// block-scaled MMA reads).
// Every wait is bounded; on a timeout the CTA sets MOE_DEV_TIMEOUT, drains
// its copies and MMAs, frees tensor memory and returns.
#include "internal.cuh"
#include "tc.cuh"

namespace moe {

constexpr int kMxBM = 128;
constexpr int kMxBN = 192;
constexpr int kMxBK = 128;
constexpr int kMxStages = 5;
// CTAs per cluster. With 2, a pair takes two m-tiles sharing one B tile and
// multicasts it (28 KB per CTA-stage from L2 instead of 40 KB); measured on
// the training shapes it ran 5-10% slower than 1 (the mainloop is not
// bound by L2 read bandwidth), so 1 is the default.
constexpr int kMxCl = 1;
constexpr int kMxBHalf = kMxBN / kMxCl;           // B rows each CTA of the pair loads (multicast to both)
constexpr int kMxSfSlots = 8;
constexpr int kMxThreads = 512;
constexpr int kMxWProd = 0, kMxWMma = 1, kMxWSf = 4, kMxWEpi = 8;
constexpr int kMxAStage = kMxBM * kMxBK;          // 16 KB
constexpr int kMxBStage = kMxBN * kMxBK;          // 24 KB
constexpr int kMxStageBytes = kMxAStage + kMxBStage;
constexpr uint32_t kMxTmemCols = 512;
constexpr uint32_t kMxSfCol0 = 2 * kMxBN;         // 384
constexpr uint32_t kMxSfCols = 12;
constexpr int kMxMaxGroups = 2048;
constexpr int kMxBarBytes = 1024;
// B's scale words of a stage (one SF4 word per B row) come with the stage's
// tensor copies into shared memory: they are weight scales streamed from
// HBM, whose latency a register prefetch a few short stages deep (decode)
// does not cover.
constexpr int kMxSfbBytes = kMxBN * 4;
constexpr int kMxSmemBytes =
    1024 /*align*/ + kMxStages * (kMxStageBytes + kMxSfbBytes) + kMxBarBytes + 4 * (kMxMaxGroups + 1);
static_assert(kMxSfCol0 + kMxSfSlots * kMxSfCols <= kMxTmemCols, "tensor memory budget");
static_assert(kMxSmemBytes <= 227 * 1024, "shared memory budget");
static_assert(kMxSfSlots % 4 == 0, "scale prefetch depth divides the slot count");

struct MxUnit {
  int e, mi, ni;
  int a_row0, a_valid;    // first A row of the tile, rows of it that are real
  int b_row0;             // first B row of the tile
  int k0, klen;           // K range of the tile
  int cnt, pad;           // the group's rows and their padded count (token side)
};

// Unit u of the cluster -> (group, m-tile pair, n-tile) through the
// per-group prefix sums of m-tile pairs uoff (shared memory); the CTA of
// cluster rank `rank` takes m-tile 2 * pair + rank.
__device__ __forceinline__ void mx_unit(const MxArgs& g, const int32_t* uoff, int u, int rank, MxUnit& w) {
  const int ui = u / g.n_tiles;
  w.ni = u - ui * g.n_tiles;
  int lo = 0, hi = g.G - 1;   // last e with uoff[e] <= ui
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (uoff[mid] <= ui) lo = mid; else hi = mid - 1;
  }
  w.e = lo;
  w.mi = kMxCl * (ui - uoff[lo]) + rank;
  if (g.mode == kMxWgrad) {
    w.a_row0 = w.mi * kMxBM;
    w.a_valid = min(kMxBM, g.M - w.a_row0);
    w.b_row0 = w.ni * kMxBN;
    w.k0 = g.poff[w.e];
    w.klen = g.poff[w.e + 1] - w.k0;
    w.cnt = w.pad = 0;
  } else {
    const int r0 = g.offsets[w.e];
    w.cnt = g.offsets[w.e + 1] - r0;
    w.pad = (w.cnt + kPadRows - 1) / kPadRows * kPadRows;
    w.a_row0 = r0 + w.mi * kMxBM;
    w.a_valid = min(kMxBM, w.cnt - w.mi * kMxBM);
    w.b_row0 = (int)((int64_t)w.e * g.b_rows_per_group) + w.ni * kMxBN;
    w.k0 = 0;
    w.klen = g.K;
  }
}

__device__ __forceinline__ int mx_stages(int klen) { return (klen + kMxBK - 1) / kMxBK; }

// The A copy of a tile covers 16 << i rows, the fewest of 16 / 32 / 64 / 128
// that hold its real rows (a decode tile with a handful of tokens then moves
// 2 KB of activations a stage, not 16 KB). The MMA still reads all 128 rows:
// the rest hold an earlier stage's bytes, and the epilogue drops those
// accumulator rows (each output row depends on its own A row only).
__device__ __forceinline__ int mx_a_box(int a_valid) {
  return a_valid <= 16 ? 0 : a_valid <= 32 ? 1 : a_valid <= 64 ? 2 : 3;
}

// The SF4 word (the scales of one 128-wide K stage) of one row: one 32-bit
// load; lanes holding consecutive rows read consecutive words. Nothing
// consumes the value until the stage's tensor-memory store, four stages
// later, so the load's latency stays off the loader's path.
__device__ __forceinline__ uint32_t load_sf4_word(const uint32_t* col, int64_t ld, int kw) {
  return __ldg(col + (int64_t)kw * ld);
}

__device__ __forceinline__ uint32_t bf16x2_bits(float a, float b) {
  return (uint32_t)f32_to_bf16_bits(a) | ((uint32_t)f32_to_bf16_bits(b) << 16);
}

// 32 fp32 values of one row -> MXFP8 (one block): 32 code bytes to dst, the
// scale byte returned.
__device__ __forceinline__ uint8_t quant_block32_store(const float (&v)[32], uint8_t* dst) {
  float am = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) am = fmaxf(am, fabsf(v[i]));
  const int e = mx_exponent(am);
  const float sc = pow2_neg(e);
  uint32_t w[8];
#pragma unroll
  for (int q = 0; q < 8; ++q)
    w[q] = (uint32_t)f32x2_to_e4m3x2(v[4 * q] * sc, v[4 * q + 1] * sc) |
           ((uint32_t)f32x2_to_e4m3x2(v[4 * q + 2] * sc, v[4 * q + 3] * sc) << 16);
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return (uint8_t)(e + 127);
}

// Column quantiser of the transposed copies, 32 features at a time: the
// warp's 32 lanes are 32 consecutive padded rows (one MX block along the
// token axis), v[i] is the lane's value of feature f0 + i (0 where the row
// is padding). A reduce-scatter butterfly (16 + 8 + 4 + 2 + 1 shuffles)
// leaves in lane i the block maximum of feature f0 + i; its scale is
// broadcast back one feature at a time. Lane l writes the codes of its row,
// lane i the scale byte of feature f0 + i (SF4, K = the token axis, ld =
// nf features).
__device__ __forceinline__ void quant_cols32(const float (&v)[32], uint8_t* tq, uint8_t* ts, int64_t f0, int64_t ld,
                                             int nf, int64_t p, int lane) {
  float m[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) m[i] = fabsf(v[i]);
#pragma unroll
  for (int h = 16; h >= 1; h >>= 1) {
    const bool up = (lane & h) != 0;
#pragma unroll
    for (int j = 0; j < h; ++j) {
      const float send = up ? m[j] : m[j + h];
      const float keep = up ? m[j + h] : m[j];
      m[j] = fmaxf(keep, __shfl_xor_sync(kFull, send, h));
    }
  }
  const int e = mx_exponent(m[0]);
  const float sc_mine = pow2_neg(e);
  ts[sf4_at(p / 32, f0 + lane, nf)] = (uint8_t)(e + 127);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float sc = __shfl_sync(kFull, sc_mine, i);
    tq[(f0 + i) * ld + p] = (uint8_t)(f32x2_to_e4m3x2(v[i] * sc, 0.f) & 0xffu);
  }
}

// The NVFP4 training recipe's two amaxes over 32 features of the warp's 32
// rows (lane = row; rows that are not the group's count as zero): max |v|,
// and max |(H16 / 4) . block| of the transpose, the two 16-lane halves being
// two blocks of 16 consecutive rows of one expert (the warp's rows start at
// a multiple of 32 from the expert's first row). The Walsh-Hadamard
// butterfly over lanes gives lane l the sum over j of (-1)^popc(l & j) v_j.
// Both maxima go to amax[0..1] with an integer atomicMax on the float bits
// (valid for values >= 0; the result is independent of the order).
__device__ __forceinline__ void nvfp4_amax32(const float (&y)[32], bool live, float* amax, int lane) {
  float am = 0.f, amt = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float h = live ? y[i] : 0.f;
    am = fmaxf(am, fabsf(h));
#pragma unroll
    for (int s = 1; s < 16; s <<= 1) {
      const float o = __shfl_xor_sync(kFull, h, s);
      h = (lane & s) ? o - h : h + o;
    }
    amt = fmaxf(amt, fabsf(h));
  }
  am = warp_max(am);
  amt = warp_max(amt) * 0.25f;
  if (lane == 0) {
    atomicMax(reinterpret_cast<int*>(amax), __float_as_int(am));
    atomicMax(reinterpret_cast<int*>(amax) + 1, __float_as_int(amt));
  }
}

// Column sums over a warp's 32 rows: v[c] is the lane's row's value of
// column c; on return v[0] of lane l is the sum over the 32 lanes of column l
// (a butterfly that halves the columns a lane holds at each of 5 steps).
__device__ __forceinline__ float warp_colsum32(float (&v)[32], int lane) {
#pragma unroll
  for (int s = 16; s >= 1; s >>= 1) {
    const bool up = (lane & s) != 0;           // this lane keeps columns with bit s set
#pragma unroll
    for (int i = 0; i < s; ++i) {
      const float send = up ? v[i] : v[i + s];
      const float keep = up ? v[i + s] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
    }
  }
  return v[0];
}

template <int MODE>
__device__ __forceinline__ void mx_epilogue(const MxArgs& g, const MxUnit& w, uint32_t acc_tmem, int q, int lane,
                                            bool has_k) {
  const int m = q * 32 + lane;                 // accumulator lane = tile row
  const bool rvalid = m < w.a_valid;
  const int64_t row = (int64_t)w.a_row0 + m;   // token row (modes W1, Plain, Dswiglu) or gradient row (Wgrad)
  if (MODE == kMxPlain || MODE == kMxWgrad) {
    uint16_t* orow;
    if (MODE == kMxPlain) orow = g.out + row * g.out_ld;
    else orow = g.out + ((int64_t)w.e * g.M + row) * g.out_ld;
    for (int c0 = 0; c0 < kMxBN; c0 += 32) {
      const int n0 = w.ni * kMxBN + c0;
      uint32_t v[32];
      if (has_k) {
        tc::tmem_ld32(acc_tmem + c0, v);
        tc::tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0u;
      }
      if (!rvalid || n0 >= g.N) continue;
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) pk[i] = bf16x2_bits(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
      if (n0 + 32 <= g.N) {
        uint4* d = reinterpret_cast<uint4*>(orow + n0);
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      } else {
        for (int i = 0; i < 32 && n0 + i < g.N; ++i)
          orow[n0 + i] = (uint16_t)(i & 1 ? pk[i >> 1] >> 16 : pk[i >> 1] & 0xffffu);
      }
    }
  } else if (MODE == kMxW1 && !g.gated) {
    // sReLU: column c is feature ni * 192 + c of a W1 with I outputs; the
    // training saves are h (bf16, I a row) and the transposed copy of y
    const int f0 = w.ni * kMxBN;
    const float wr = rvalid ? g.w_row[row] : 0.f;
    const int rel = w.mi * kMxBM + m;
    const bool tblk = g.tq && (w.mi * kMxBM + q * 32) < w.pad;
    const int64_t p = g.tq ? (int64_t)g.poff[w.e] + rel : 0;
    for (int b = 0; b < kMxBN / 32; ++b) {
      const int f = f0 + 32 * b;
      if (f >= g.I) break;
      uint32_t v[32];
      tc::tmem_ld32(acc_tmem + 32 * b, v);
      tc::tmem_wait_ld();
      float y[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) y[i] = wr * act_plain(__uint_as_float(v[i]));
      if (rvalid) {
        const uint8_t sb = quant_block32_store(y, g.yq + row * g.I + f);
        g.ys[row * (g.I / 32) + f / 32] = sb;
        if (g.yst) g.yst[sf4_at(f / 32, row, g.R)] = sb;
        if (g.hsave) {
          uint32_t hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) hv[i] = bf16x2_bits(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          uint4* dh = reinterpret_cast<uint4*>(g.hsave + row * g.I + f);
#pragma unroll
          for (int i = 0; i < 4; ++i) dh[i] = make_uint4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
        }
      }
      if (g.amax) nvfp4_amax32(y, rel < w.cnt, g.amax, lane);
      if (tblk) {
        if (rel >= w.cnt) {
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] = 0.f;      // padding rows of the group
        }
        quant_cols32(y, g.tq, g.ts, f, g.t_ld, g.t_nf, p, lane);
      }
    }
  } else if (MODE == kMxW1) {
    // columns [0, 96): gate features f0 + c, [96, 192): the same up features
    const int f0 = w.ni * (kMxBN / 2);
    const float wr = rvalid ? g.w_row[row] : 0.f;
    const int rel = w.mi * kMxBM + m;                         // row index inside the group
    const bool tblk = g.tq && (w.mi * kMxBM + q * 32) < w.pad;  // this warp's 32-row block is in the padded range
    const int64_t p = g.tq ? (int64_t)g.poff[w.e] + rel : 0;
    for (int b = 0; b < kMxBN / 64; ++b) {
      const int f = f0 + 32 * b;
      if (f >= g.I) break;
      uint32_t gv[32], uv[32];
      tc::tmem_ld32(acc_tmem + 32 * b, gv);
      tc::tmem_ld32(acc_tmem + kMxBN / 2 + 32 * b, uv);
      tc::tmem_wait_ld();
      if (g.b1) {
        // W1 bias of the group: gate b, up c, before the activation (the
        // same value in every lane: one broadcast load each)
        const float* bb = g.b1 + (int64_t)w.e * 2 * g.I + f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          gv[i] = __float_as_uint(__uint_as_float(gv[i]) + __ldg(bb + i));
          uv[i] = __float_as_uint(__uint_as_float(uv[i]) + __ldg(bb + g.I + i));
        }
      }
      float y[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) y[i] = wr * act_fwd(__uint_as_float(gv[i]), __uint_as_float(uv[i]), g.act);
      if (rvalid) {
        const uint8_t sb = quant_block32_store(y, g.yq + row * g.I + f);
        g.ys[row * (g.I / 32) + f / 32] = sb;
        if (g.yst) g.yst[sf4_at(f / 32, row, g.R)] = sb;
        if (g.hsave) {
          uint32_t hg[16], hu[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            hg[i] = bf16x2_bits(__uint_as_float(gv[2 * i]), __uint_as_float(gv[2 * i + 1]));
            hu[i] = bf16x2_bits(__uint_as_float(uv[2 * i]), __uint_as_float(uv[2 * i + 1]));
          }
          uint4* dg = reinterpret_cast<uint4*>(g.hsave + row * 2 * g.I + f);
          uint4* du = reinterpret_cast<uint4*>(g.hsave + row * 2 * g.I + g.I + f);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            dg[i] = make_uint4(hg[4 * i], hg[4 * i + 1], hg[4 * i + 2], hg[4 * i + 3]);
            du[i] = make_uint4(hu[4 * i], hu[4 * i + 1], hu[4 * i + 2], hu[4 * i + 3]);
          }
        }
      }
      if (g.amax) nvfp4_amax32(y, rel < w.cnt, g.amax, lane);
      if (tblk) {
        if (rel >= w.cnt) {
#pragma unroll
          for (int i = 0; i < 32; ++i) y[i] = 0.f;      // padding rows of the group
        }
        quant_cols32(y, g.tq, g.ts, f, g.t_ld, g.t_nf, p, lane);
      }
    }
  } else if (!g.gated) {   // kMxDswiglu for sReLU: dh = w_row * dY1 * 2 max(h, 0), I features a row
    const int f0 = w.ni * kMxBN;
    const float wr = rvalid ? g.w_row[row] : 0.f;
    const int rel = w.mi * kMxBM + m;
    const bool tblk = (w.mi * kMxBM + q * 32) < w.pad;
    const bool live = rel < w.cnt;
    const int64_t p = (int64_t)g.poff[w.e] + rel;
    const int I = g.I;
    float dw = 0.f;
    for (int c0 = 0; c0 < kMxBN; c0 += 32) {
      const int f = f0 + c0;
      if (f >= I) break;
      uint32_t dv[32];
      tc::tmem_ld32(acc_tmem + c0, dv);
      tc::tmem_wait_ld();
      float dh[32];
      if (rvalid) {
        const uint4* h4 = reinterpret_cast<const uint4*>(g.hsave + row * I + f);
        uint32_t hw[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 a = h4[i];
          hw[4 * i] = a.x; hw[4 * i + 1] = a.y; hw[4 * i + 2] = a.z; hw[4 * i + 3] = a.w;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t x = hw[i >> 1];
          const float hh = __uint_as_float(i & 1 ? x & 0xffff0000u : x << 16);
          const float dy = __uint_as_float(dv[i]);
          dw = fmaf(dy, act_plain(hh), dw);
          dh[i] = act_plain_bwd(hh, wr * dy);
        }
        g.yst[sf4_at(f / 32, row, g.R)] = quant_block32_store(dh, g.yq + row * I + f);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) dh[i] = 0.f;
      }
      if (tblk) {
        if (!live) {
#pragma unroll
          for (int i = 0; i < 32; ++i) dh[i] = 0.f;   // padding rows of the group
        }
        quant_cols32(dh, g.tq, g.ts, f, g.t_ld, g.t_nf, p, lane);
      }
    }
    if (rvalid) g.dwpart[(int64_t)w.ni * g.R + row] = dw;
  } else {   // kMxDswiglu: columns = dY1 for features f0 + c
    const int f0 = w.ni * kMxBN;
    const float wr = rvalid ? g.w_row[row] : 0.f;
    const int rel = w.mi * kMxBM + m;
    const bool tblk = (w.mi * kMxBM + q * 32) < w.pad;
    const bool live = rel < w.cnt;
    const int64_t p = (int64_t)g.poff[w.e] + rel;
    const int I = g.I;
    float dw = 0.f;
    for (int c0 = 0; c0 < kMxBN; c0 += 32) {
      const int f = f0 + c0;
      if (f >= I) break;
      uint32_t dv[32];
      tc::tmem_ld32(acc_tmem + c0, dv);
      tc::tmem_wait_ld();
      float dg[32], du[32];
      if (rvalid) {
        const uint4* hg4 = reinterpret_cast<const uint4*>(g.hsave + row * 2 * I + f);
        const uint4* hu4 = reinterpret_cast<const uint4*>(g.hsave + row * 2 * I + I + f);
        uint32_t hg[16], hu[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 a = hg4[i], bb = hu4[i];
          hg[4 * i] = a.x; hg[4 * i + 1] = a.y; hg[4 * i + 2] = a.z; hg[4 * i + 3] = a.w;
          hu[4 * i] = bb.x; hu[4 * i + 1] = bb.y; hu[4 * i + 2] = bb.z; hu[4 * i + 3] = bb.w;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t gw = hg[i >> 1], uw = hu[i >> 1];
          const float gg = __uint_as_float(i & 1 ? gw & 0xffff0000u : gw << 16);
          const float uu = __uint_as_float(i & 1 ? uw & 0xffff0000u : uw << 16);
          const float dy = __uint_as_float(dv[i]);
          const float3 a = act_fwd_bwd(gg, uu, wr * dy, g.act);
          dw = fmaf(dy, a.x, dw);
          dg[i] = a.y;
          du[i] = a.z;
        }
        g.yst[sf4_at(f / 32, row, g.R)] = quant_block32_store(dg, g.yq + row * 2 * I + f);
        g.yst[sf4_at((I + f) / 32, row, g.R)] = quant_block32_store(du, g.yq + row * 2 * I + I + f);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) dg[i] = du[i] = 0.f;
      }
      if (tblk) {
        if (!live) {
#pragma unroll
          for (int i = 0; i < 32; ++i) dg[i] = du[i] = 0.f;   // padding rows of the group
        }
        quant_cols32(dg, g.tq, g.ts, f, g.t_ld, g.t_nf, p, lane);
        quant_cols32(du, g.tq, g.ts, (int64_t)I + f, g.t_ld, g.t_nf, p, lane);
      }
      if (g.dbpart && tblk) {
        // W1 bias gradient partials: this warp's 32 rows summed per column
        // (rows past the group's count hold zeros)
        float* dst = g.dbpart + (p - lane) / 32 * g.db_ld;
        const float sg = warp_colsum32(dg, lane);
        const float su = warp_colsum32(du, lane);
        dst[f + lane] = sg;
        dst[I + f + lane] = su;
      }
    }
    if (rvalid) g.dwpart[(int64_t)w.ni * g.R + row] = dw;
  }
}

// m-tile pairs of group e (the cluster's unit height).
template <int MODE>
__device__ __forceinline__ int mx_pairs(const MxArgs& g, int e) {
  const int mt = MODE == kMxWgrad ? g.m_tiles : (g.offsets[e + 1] - g.offsets[e] + kMxBM - 1) / kMxBM;
  return (mt + kMxCl - 1) / kMxCl;
}

template <int MODE>
__global__ void __launch_bounds__(kMxThreads, 1) k_gemm_mx(const __grid_constant__ MxArgs g,
                                                           const __grid_constant__ MxMaps maps) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* sa = smem;
  uint8_t* sb = smem + kMxStages * kMxAStage;
  uint8_t* sfb = smem + kMxStages * kMxStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sfb + kMxStages * kMxSfbBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + kMxStages;
  uint64_t* sffull = empty + kMxStages;
  uint64_t* sfempty = sffull + kMxSfSlots;
  uint64_t* accfull = sfempty + kMxSfSlots;
  uint64_t* accempty = accfull + 2;
  uint64_t* drain = accempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int32_t* uoff = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(bars) + kMxBarBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ int bad_pack;
  pdl_enter();
  if (threadIdx.x == 0) {
    bad_pack = g.hdr && !pack_header_ok(g.hdr, g.b_fp4 ? MOE_WFMT_MXFP4 : MOE_WFMT_MXFP8, g.which, g.G, g.bias != 0);
    if (bad_pack) set_status(g.status, MOE_DEV_BAD_PACK);
  }
  __syncthreads();
  if (bad_pack) return;   // the blob is not the packing this GEMM reads: write nothing
  // per-group prefix sums of m-tile pairs (a block-wide scan)
  {
    __shared__ int32_t wsum[kMxThreads / 32];
    const int G = g.G;
    const int per = (G + kMxThreads - 1) / kMxThreads;
    const int lo = threadIdx.x * per, hi = min(G, lo + per);
    int s = 0;
    for (int e = lo; e < hi; ++e)
      s += mx_pairs<MODE>(g, e);
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w2 = 0; w2 < warp; ++w2) base += wsum[w2];
    int run = base + incl - s;
    for (int e = lo; e < hi; ++e) {
      uoff[e] = run;
      run += mx_pairs<MODE>(g, e);
    }
    if (threadIdx.x == kMxThreads - 1) uoff[G] = base + incl;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < kMxStages; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], kMxCl);   // released by the MMAs of both CTAs of the pair
    }
    for (int i = 0; i < kMxSfSlots; ++i) {
      tc::mbar_init(&sffull[i], 4);    // one elected arrive per scale-loader warp
      tc::mbar_init(&sfempty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&accfull[i], 1);
      tc::mbar_init(&accempty[i], 4);  // one elected arrive per epilogue warp of the tile's warpgroup
    }
    tc::mbar_init(drain, 1);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == kMxWMma) tc::tmem_alloc(tmem_slot, kMxTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  // the peers' barriers are initialised before any copy or commit reaches them
  if constexpr (kMxCl > 1) tc::cluster_sync();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int U = uoff[g.G] * g.n_tiles;
  const int rank = kMxCl > 1 ? (int)tc::cluster_rank() : 0;
  const int cid = blockIdx.x / kMxCl, ncl = gridDim.x / kMxCl;

  if (warp == kMxWProd) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) tc::prefetch_tmap(&maps.a[i]);
      tc::prefetch_tmap(&maps.b);
      tc::prefetch_tmap(&maps.sfb);
      // bytes a stage's B copy reports to the barrier: packed E2M1 reports
      // its global bytes (two elements a byte) although it lands one element
      // a byte in shared memory (8 data bytes, then an 8-byte gap the copy
      // leaves untouched, per 16 elements)
      const uint32_t b_tx = g.b_fp4 ? kMxBStage / 2 : kMxBStage;
      uint32_t it = 0;
      bool ok = true;
      for (int u = cid; ok && u < U; u += ncl) {
        MxUnit w;
        mx_unit(g, uoff, u, rank, w);
        const int nk = mx_stages(w.klen);
        for (int s = 0; s < nk; ++s, ++it) {
          const int slot = it % kMxStages;
          if (!tc::mbar_wait(&empty[slot], ((it / kMxStages) & 1) ^ 1, abort)) { ok = false; break; }
          const int ai = mx_a_box(w.a_valid);
          tc::mbar_arrive_expect_tx(&full[slot], (uint32_t)(kMxBK * (16 << ai)) + b_tx + kMxSfbBytes);
          const int kx = w.k0 + s * kMxBK;
          tc::tma_load_2d_plain(sfb + slot * kMxSfbBytes, &maps.sfb, w.b_row0, kx / kMxBK, &full[slot]);
          tc::tma_load_2d_plain(sa + slot * kMxAStage, &maps.a[ai], kx, w.a_row0, &full[slot]);
          if constexpr (kMxCl > 1) {
            // this CTA's part of the shared B tile, into every CTA of the cluster
            tc::tma_load_2d_mc(sb + slot * kMxBStage + rank * (kMxBHalf * kMxBK), &maps.b, kx,
                               w.b_row0 + rank * kMxBHalf, &full[slot], (uint16_t)((1u << kMxCl) - 1));
          } else {
            tc::tma_load_2d_plain(sb + slot * kMxBStage, &maps.b, kx, w.b_row0, &full[slot]);
          }
        }
      }
      if (!ok || *abort) {
        // wind-down: wait (bounded, ignoring the abort flag) for the copies
        // still in flight into this CTA's shared memory
        volatile int never = 0;
        const uint32_t n = it < (uint32_t)kMxStages ? it : (uint32_t)kMxStages;
        for (uint32_t k = 0; k < n; ++k) {
          const uint32_t i2 = it - 1 - k;
          tc::mbar_wait(&full[i2 % kMxStages], (i2 / kMxStages) & 1, &never, 400000000ll);
        }
      }
    }
  } else if (warp == kMxWMma) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      uint32_t it = 0, tcount = 0;
      bool ok = true;
      const uint32_t btype = g.b_fp4 ? tc::kMxE2M1 : tc::kMxE4M3;
      for (int u = cid; ok && u < U; u += ncl, ++tcount) {
        MxUnit w;
        mx_unit(g, uoff, u, rank, w);
        const int nk = mx_stages(w.klen);
        const int d = tcount & 1;
        if (!tc::mbar_wait(&accempty[d], ((tcount >> 1) & 1) ^ 1, abort)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t dt = tmem + d * kMxBN;
        for (int s = 0; s < nk; ++s, ++it) {
          const int slot = it % kMxStages, fs = it % kMxSfSlots;
          if (!tc::mbar_wait(&full[slot], (it / kMxStages) & 1, abort)) { ok = false; break; }
          if (!tc::mbar_wait(&sffull[fs], (it / kMxSfSlots) & 1, abort)) { ok = false; break; }
          tc::fence_after_sync();
          const int kv = min(4, (w.klen - s * kMxBK) / 32);
          const uint64_t ad = tc::smem_desc_sw128(tc::smem_u32(sa + slot * kMxAStage));
          const uint64_t bd = tc::smem_desc_sw128(tc::smem_u32(sb + slot * kMxBStage));
          const uint32_t sfa = tmem + kMxSfCol0 + fs * kMxSfCols;
          const uint32_t sfb = sfa + 4;
          for (int j = 0; j < kv; ++j)
            tc::mma_mx_ss(dt, ad + 2 * j, bd + 2 * j, tc::idesc_mx(kMxBM, kMxBN, j, j, btype), sfa, sfb,
                          (s | j) != 0 ? 1u : 0u);
          if constexpr (kMxCl > 1) tc::mma_commit_mc(&empty[slot], (uint16_t)((1u << kMxCl) - 1));
          else tc::mma_commit(&empty[slot]);
          tc::mma_commit(&sfempty[fs]);
        }
        if (!ok) break;
        tc::mma_commit(&accfull[d]);
      }
      // every MMA of this thread has completed once `drain` fires
      tc::mma_commit(drain);
      volatile int never = 0;
      tc::mbar_wait(drain, 0, &never, 400000000ll);
    }
  } else if (warp >= kMxWSf && warp < kMxWSf + 4) {
    // ---------------- scale loaders ----------------
    // Every lane quarter gets the same image: lane (32 q + r), column c of a
    // 4-column group holds the scale word of row 32 c + r of that group's
    // 128 rows (A: one group; B: rows 0-127, then rows 128-191).
    const int q = warp - kMxWSf;                      // tensor-memory lane quarter
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    constexpr int kNB1 = (kMxBN - 128) / 32;          // valid words of B's second group
    static_assert(kNB1 == 2, "B's second group holds rows 128-191");
    uint32_t it = 0;
    bool ok = true;
    for (int u = cid; ok && u < U; u += ncl) {
      MxUnit w;
      mx_unit(g, uoff, u, rank, w);
      const int nk = mx_stages(w.klen);
      // each A row's SF4 column (nullptr: no such row); B's words come with
      // the stage into shared memory (sfb)
      const uint32_t* pa[4];
      const uint32_t* wa = reinterpret_cast<const uint32_t*>(g.a_sf);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int64_t ra = (int64_t)w.a_row0 + 32 * c + lane;
        pa[c] = ra < g.a_rows ? wa + ra : nullptr;
      }
      const int kw0 = w.k0 / kMxBK;
      // four stages of A's scale words in flight in registers
      uint32_t va[4][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bool live = j < nk;
#pragma unroll
        for (int c = 0; c < 4; ++c) va[j][c] = (pa[c] && live) ? load_sf4_word(pa[c], g.a_sf_ld, kw0 + j) : 0u;
      }
      for (int s0 = 0; s0 < nk; s0 += 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int s = s0 + j;
          if (s < nk && ok) {
            const int fs = it % kMxSfSlots, slot = it % kMxStages;
            // the warp's collective tensor-memory stores need one decision
            bool got = tc::mbar_wait(&sfempty[fs], ((it / kMxSfSlots) & 1) ^ 1, abort);
            got = got && tc::mbar_wait(&full[slot], (it / kMxStages) & 1, abort);
            if (!__all_sync(kFull, got)) {
              ok = false;
            } else {
              tc::fence_after_sync();
              const uint32_t* sw = reinterpret_cast<const uint32_t*>(sfb + slot * kMxSfbBytes);
              uint32_t vb[4 + kNB1];
#pragma unroll
              for (int c = 0; c < 4 + kNB1; ++c) vb[c] = sw[32 * c + lane];
              const uint32_t col = kMxSfCol0 + fs * kMxSfCols;
              tc::tmem_st4(lane_base + col, va[j][0], va[j][1], va[j][2], va[j][3]);
              tc::tmem_st4(lane_base + col + 4, vb[0], vb[1], vb[2], vb[3]);
              tc::tmem_st4(lane_base + col + 8, vb[4], vb[5], 0u, 0u);
              tc::tmem_wait_st();
              tc::fence_before_sync();
              __syncwarp();
              if (lane == 0) tc::mbar_arrive(&sffull[fs]);
              ++it;
              // refill this register slot with stage s + 4
              const int s4 = s + 4;
              const bool live = s4 < nk;
#pragma unroll
              for (int c = 0; c < 4; ++c)
                va[j][c] = (pa[c] && live) ? load_sf4_word(pa[c], g.a_sf_ld, kw0 + s4) : 0u;
            }
          }
        }
        if (!ok) break;
      }
    }
  } else if (warp >= kMxWEpi) {
    // ---------------- epilogue ----------------
    const int wg = (warp - kMxWEpi) >> 2;    // tiles with (index % 2) == wg, accumulator wg
    const int q = warp & 3;
    const uint32_t acc = tmem + ((uint32_t)(q * 32) << 16) + wg * kMxBN;
    uint32_t tcount = 0, mine = 0;
    for (int u = cid; u < U; u += ncl, ++tcount) {
      if ((int)(tcount & 1) != wg) continue;
      MxUnit w;
      mx_unit(g, uoff, u, rank, w);
      const bool got = tc::mbar_wait(&accfull[wg], mine & 1, abort);
      if (!__all_sync(kFull, got)) break;
      tc::fence_after_sync();
      mx_epilogue<MODE>(g, w, acc, q, lane, w.klen > 0);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&accempty[wg]);
      ++mine;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if constexpr (kMxCl > 1) {
    if (*abort) {
      // a CTA that gave up may have copies into its peers still in flight:
      // give them time to land (bounded) before the cluster can leave
      const long long t0 = clock64();
      while (clock64() - t0 < 100000) {
      }
    }
    // no CTA leaves while a peer may still multicast into it or arrive on it
    tc::cluster_sync();
  }
  if (threadIdx.x == 0 && *abort) set_status(g.status, MOE_DEV_TIMEOUT);
  if (warp == kMxWMma) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kMxTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFnMx)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFnMx encode_fn_mx() {
  static const EncodeTiledFnMx fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFnMx>(p);
    return (EncodeTiledFnMx) nullptr;
  }();
  return fn;
}

// Matrix [rows][cols] (cols = K elements, contiguous) as a 2-D tensor map
// with boxes of 128 K-elements x box_rows rows, 128-byte swizzle; reads past
// either edge return zero. fp4: packed E2M1 pairs (cols / 2 bytes a row;
// the unpacking copy wants cols % 128 == 0 and a 32-byte aligned base).
bool make_tmap_mx(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows, bool fp4) {
  EncodeTiledFnMx fn = encode_fn_mx();
  if (!fn || cols % (fp4 ? 128 : 16) != 0 || ((uintptr_t)base & (fp4 ? 31u : 15u))) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)std::max<int64_t>(rows, 1)};
  cuuint64_t strides[1] = {(cuuint64_t)(fp4 ? cols / 2 : cols)};
  cuuint32_t box[2] = {(cuuint32_t)kMxBK, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_mx_sf(CUtensorMap* map, const void* sf, int64_t rows, int64_t words, int64_t ld) {
  EncodeTiledFnMx fn = encode_fn_mx();
  if (!fn || ld % 4 != 0 || ((uintptr_t)sf & 15u) || rows > ld) return false;
  cuuint64_t dims[2] = {(cuuint64_t)std::max<int64_t>(rows, 1), (cuuint64_t)std::max<int64_t>(words, 1)};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
  cuuint32_t box[2] = {(cuuint32_t)kMxBN, 1u};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(sf), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The four A maps of one E4M3 matrix, boxes of 16 / 32 / 64 / 128 rows.
bool make_tmaps_mx_a(MxMaps* maps, const void* base, int64_t rows, int64_t cols) {
  for (int i = 0; i < 4; ++i)
    if (!make_tmap_mx(&maps->a[i], base, rows, cols, 16 << i, false)) return false;
  return true;
}

template <int MODE>
static cudaError_t launch_mx_t(const MxArgs& g, const MxMaps& maps, int grid_cap, cudaStream_t st) {
  static std::atomic<bool> done[kMaxDevices] = {};
  static std::atomic<int> max_clusters[kMaxDevices] = {};
  cudaError_t e = set_smem_once((const void*)k_gemm_mx<MODE>, kMxSmemBytes, done);
  if (e != cudaSuccess) return e;
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kMxThreads);
  cfg.dynamicSmemBytes = kMxSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kMxCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  // clusters that fit on the device at once (pairs of SMs of one GPC),
  // queried once per device
  const bool slot = dev >= 0 && dev < kMaxDevices;
  int nc = slot ? max_clusters[dev].load() : 0;
  if (nc <= 0) {
    cfg.gridDim = dim3(kMxCl * 64);
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&nc, k_gemm_mx<MODE>, &cfg) != cudaSuccess || nc <= 0)
      nc = std::max(1, device_sms() / kMxCl);
    if (slot) max_clusters[dev].store(nc);
  }
  const int ncl = std::max(1, std::min(nc, grid_cap / kMxCl));
  cfg.gridDim = dim3(ncl * kMxCl);
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_gemm_mx<MODE>, g, maps);
}

cudaError_t launch_gemm_mx(const MxArgs& g, const MxMaps& maps, int grid, cudaStream_t st) {
  if (g.G > kMxMaxGroups || g.n_tiles <= 0) return cudaErrorInvalidValue;
  grid = std::max(1, grid);
  cudaError_t e;
  switch (g.mode) {
    case kMxW1: e = launch_mx_t<kMxW1>(g, maps, grid, st); break;
    case kMxPlain: e = launch_mx_t<kMxPlain>(g, maps, grid, st); break;
    case kMxDswiglu: e = launch_mx_t<kMxDswiglu>(g, maps, grid, st); break;
    case kMxWgrad: e = launch_mx_t<kMxWgrad>(g, maps, grid, st); break;
    default: return cudaErrorInvalidValue;
  }
  note_launch();
  return e;
}

int mx_tile_n() { return kMxBN; }
int mx_b_box_rows() { return kMxBHalf; }
int mx_tile_m() { return kMxBM; }

// ---------------------------------------------------------------------------
// Row gather of MXFP8 rows: dst[r] = src[row_map[r] / row_div] (codes and
// scales), r < min(R, offsets[G]). One warp per row, 16-byte copies; the
// scales land in the SF4 layout (ld R) for the GEMM's scale loaders.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_gather_mx(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int C,
                                                   const int32_t* __restrict__ row_map, int row_div, int R,
                                                   const int32_t* __restrict__ offsets, int G,
                                                   uint8_t* __restrict__ dq, uint8_t* __restrict__ ds) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  const int Rv = min(R, offsets[G]);
  const int nw = gridDim.x * (blockDim.x / 32);
  for (int r = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < Rv; r += nw) {
    const int64_t src = row_map[r] / row_div;
    const uint4* sq = reinterpret_cast<const uint4*>(q + src * C);
    uint4* d = reinterpret_cast<uint4*>(dq + (int64_t)r * C);
    for (int i = lane; i < C / 16; i += 32) d[i] = sq[i];
    const int nb = C / 32;
    for (int wd = lane; wd < (nb + 3) / 4; wd += 32) {
      uint32_t v = 0;
      for (int j = 0; j < 4 && 4 * wd + j < nb; ++j) v |= (uint32_t)s[src * nb + 4 * wd + j] << (8 * j);
      reinterpret_cast<uint32_t*>(ds)[(int64_t)wd * R + r] = v;
    }
  }
}

cudaError_t launch_gather_mx(const uint8_t* q, const uint8_t* s, int C, const int32_t* row_map, int row_div, int R,
                             const int32_t* offsets, int G, uint8_t* dq, uint8_t* ds, cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  const int blocks = (int)std::min<int64_t>(((int64_t)R + 7) / 8, (int64_t)device_sms() * 16);
  cudaError_t e = launch_pdl(k_gather_mx, dim3(blocks), dim3(256), 0, st, q, s, C, row_map, row_div, R, offsets, G,
                             dq, ds);
  note_launch();
  return e;
}

// Row-major scales [R][C/32] -> SF4 (ld R): thread per (row, word), rows
// fastest so the word stores are coalesced.
__global__ void __launch_bounds__(256) k_sf_to_sf4(const uint8_t* __restrict__ s, int nb, int64_t R,
                                                   uint32_t* __restrict__ d) {
  const int nw = (nb + 3) / 4;
  const int64_t total = R * nw;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i % R;
    const int wd = (int)(i / R);
    uint32_t v = 0;
    for (int j = 0; j < 4 && 4 * wd + j < nb; ++j) v |= (uint32_t)s[r * nb + 4 * wd + j] << (8 * j);
    d[(int64_t)wd * R + r] = v;
  }
}

cudaError_t launch_sf_to_sf4(const uint8_t* s, int C, int64_t R, uint8_t* d, cudaStream_t st) {
  if (R == 0) return cudaSuccess;
  const int64_t total = R * ((C / 32 + 3) / 4);
  const int blocks = (int)std::min<int64_t>((total + 255) / 256, (int64_t)device_sms() * 16);
  k_sf_to_sf4<<<blocks, 256, 0, st>>>(s, C / 32, R, reinterpret_cast<uint32_t*>(d));
  note_launch();
  return cudaGetLastError();
}

}  // namespace moe
