// Grouped GEMM on the 5th-generation tensor cores (tcgen05), operand-swapped:
// the MMA's M side is 128 output features of one expert tile, its N side the
// expert's tokens (16..NT per MMA), so a decode step with a handful of tokens
// per expert still streams every weight byte exactly once.
//
// GC-MoE summary (arxiv-wiki "GC-MoE: Overlapping Expert-Parallel Token
// Dispatch with FP8/FP4 Grouped GEMM via CUDA Green Contexts"), key
// contributions: operand-swapped tcgen05 block-scaled MMA over K-prepacked FP4
// weights streamed in large bursts. That design pairs FP8 activations with
// per-32 power-of-two weight scales; NVFP4 weights carry E4M3 scales per 16
// elements, which no block-scaled tcgen05 kind accepts next to FP8
// activations. Here every weight element is decoded once, exactly, to f16
// (E2M1 value x E4M3 scale has at most 6 significant bits), written by a
// decoder warpgroup straight into tensor memory as the MMA's A operand, and
// multiplied with f16 activations (the E4M3 activation codes times
// 2^(block exponent - row exponent)) by tcgen05.mma kind::f16 with fp32
// accumulation in tensor memory.
//
// Roles (one CTA per SM, persistent over work units):
//   warps 0, 26 weight producers (even / odd stages): per stage one bulk
//               copy of a pair of consecutive 64-wide K chunks of the weight
//               tile (codes + scales) into the weight ring. A stage is
//               released as soon as its decoders have read it, so the ring's
//               bytes stay in flight instead of waiting for the MMAs. Each
//               bulk copy costs its issuing thread several hundred cycles,
//               more than one thread can afford at full bandwidth.
//   warp 25     activation producer: per pair of chunks one 3-D tensor copy
//               of the f16 activation rows (128-byte swizzle) into the
//               activation ring, released by the MMA commit. The row box is
//               the smallest of 8/16/32/64 rows holding the tile's valid
//               rows: at decode an expert often has 1-4 rows. A thread of
//               its own, because each copy instruction costs its issuing
//               thread a few hundred cycles.
//   warps 1-4   MMA issuers (P of them), taking pairs round-robin: 4 MMAs
//               (K = 16 each) per chunk, A from tensor memory, B from the
//               activation ring, each issuer into its own accumulator; the
//               commits free the A buffer and the activation slot.
//   warps 5-20  decoders, four groups of four warps, group g filling the A
//               buffer of every pair with index = g (mod 4): thread = weight
//               row = tensor-memory lane. Decoding is latency-bound (a chain
//               of loads, conversions and multiplies per row), so the SM
//               runs four independent groups.
//   warps 21-24 epilogue: tensor memory -> fp32 partials in global memory,
//               scaled by the per-row weight factor and the per-token
//               activation exponent
// Work unit = (expert with rows, 128-feature tile, K slice); within a unit
// the expert's rows are taken NT at a time.
// Every wait is bounded in time; on a timeout the CTA sets a status bit,
// drains its own copies and MMAs, frees tensor memory and returns.
#include "internal.cuh"
#include "tc.cuh"

namespace moe {

constexpr int kTcNA = 4;          // tensor-memory A buffers, two 64-K chunks (64 columns) each
constexpr int kTcNG = 4;          // decoder groups (group g fills A buffer g)
constexpr int kWIss = 1;          // first MMA-issuer warp
constexpr int kWDec = 5;          // first decoder warp
constexpr int kWEpi = kWDec + 4 * kTcNG;   // first epilogue warp
constexpr int kWBProd = kWEpi + 4;         // activation producer warp
constexpr int kWProd1 = kWBProd + 1;       // second weight producer warp
constexpr int kTcThreads = 32 * (kWProd1 + 1);   // 27 warps
static_assert(kTcNA % kTcNG == 0, "each A buffer belongs to one decoder group");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCol0 = kTcNA * 64;
constexpr int kSmemBudget = 212 * 1024;

template <int NT>
struct TcCfg {
  // Each MMA issuer accumulates into its own NT-column tile; a D buffer
  // holds all of them and the epilogue adds them.
  static constexpr int P = NT <= 32 ? 4 : NT <= 64 ? 2 : 1;          // MMA issuers
  static constexpr int DStride = P * NT;                             // TMEM columns per D buffer
  // D buffers: three where they fit next to the A buffers (16-token tiles),
  // so the epilogue may fall two units behind the MMAs when units are short
  static constexpr int ND = kDCol0 + 3 * DStride <= kTmemCols ? 3 : 2;
  static constexpr int CB = 4608;                                    // NVFP4 chunk bytes
  // A stage is one pair of chunks, so every stage feeds exactly one decoder
  // group and one MMA issuer: weight slot s always belongs to group
  // s % kTcNG and activation slot s to issuer s % P, and each waiter sees
  // every phase of its slots in order.
  static constexpr int WSlot = (2 * CB + 1023) / 1024 * 1024;
  static constexpr int BSlot = 2 * NT * 128;                         // two chunks x NT rows x 64 f16
  static constexpr int BS = NT == 16 ? 16 : NT == 128 ? 4 : 8;       // activation slots
  static constexpr int WSraw = (kSmemBudget - BS * BSlot) / WSlot / kTcNG * kTcNG;
  static constexpr int WS = WSraw > 24 ? 24 : WSraw;                 // weight stages
  static constexpr int SmemBytes = WS * WSlot + BS * BSlot + 1024 /*align*/ + 1024 /*barriers*/;
  static_assert(WS >= 2 * kTcNG && WS % kTcNG == 0, "weight slots must map to decoder groups");
  static_assert(BS % P == 0, "activation slots must map to MMA issuers");
};

struct TcUnit {
  int e, j, s, c0, c1, r0, r1;
};

// Groups with rows and the split boundaries, staged in shared memory once
// per CTA: every role decodes a unit at every unit boundary, and dependent
// global loads (touched list, then offsets) or divisions there would stall
// the pipeline each time (the role threads are single lanes whose dependent
// instructions issue slowly). Groups past the table's end are read from
// global memory.
constexpr int kUnitTab = 512;
constexpr int kMaxSplits = 64;
struct UnitTab {
  int e[kUnitTab], r0[kUnitTab], r1[kUnitTab];
  int cb[2][kMaxSplits + 1];   // matrix m's K slice s covers chunks [cb[m][s], cb[m][s + 1])
};

// Work unit u = (ti * tiles + j) * S + s of one matrix; the mixed-radix
// digits are advanced by the precomputed digits of gridDim.x, with no
// division per step.
struct UnitIt {
  uint32_t ti, j, s, mat;
};
struct UnitStep {
  uint32_t dti, dj, ds, tiles, S;
  __device__ void init(int tiles_, int S_, uint32_t step) {
    tiles = (uint32_t)tiles_;
    S = (uint32_t)S_;
    ds = step % S;
    dj = (step / S) % tiles;
    dti = step / (S * tiles);
  }
  __device__ UnitIt at(uint32_t u, uint32_t mat) const { return UnitIt{u / (S * tiles), (u / S) % tiles, u % S, mat}; }
  __device__ void next(UnitIt& it) const {
    it.s += ds;
    uint32_t cj = 0;
    if (it.s >= S) { it.s -= S; cj = 1; }
    it.j += dj + cj;
    uint32_t ct = 0;
    if (it.j >= tiles) { it.j -= tiles; ct = 1; }
    it.ti += dti + ct;
  }
};

// A CTA's walk over the units: u = cta, cta + ncta, ... (cta: the CTA's
// index among the ncta GEMM CTAs) through matrix 0's n_groups * tiles * S
// units and, in the fused layer, on through matrix 1's; every role visits
// the same sequence. Kept in shared memory (set once per CTA): the role loops
// then hold only their iterator in registers.
struct UnitWalk {
  UnitStep st0, st1;
  uint32_t n_groups, u0;   // u0: units of matrix 0
  uint32_t cta, ncta;
  int nmat;
  __device__ void init(const TcArgs& g, uint32_t ng, uint32_t cta_, uint32_t ncta_) {
    cta = cta_;
    ncta = ncta_;
    st0.init(g.m[0].tiles, g.m[0].S, ncta);
    st1.init(g.m[g.nmat - 1].tiles, g.m[g.nmat - 1].S, ncta);
    n_groups = ng;
    u0 = ng * (uint32_t)g.m[0].tiles * (uint32_t)g.m[0].S;
    nmat = g.nmat;
  }
  __device__ UnitIt first() const {
    UnitIt it = st0.at(cta, 0);
    if (it.ti >= n_groups) to_second(it);
    return it;
  }
  __device__ bool more(const UnitIt& it) const { return it.ti < n_groups; }
  __device__ void next(UnitIt& it) const {
    if (it.mat == 0) {
      st0.next(it);
      if (it.ti >= n_groups) to_second(it);
    } else {
      st1.next(it);
    }
  }
  // the first unit of matrix 1 on this CTA's stride: the smallest u >= u0
  // with u = cta (mod ncta), as an index into matrix 1's units
  __device__ void to_second(UnitIt& it) const {
    if (nmat < 2) return;
    it = st1.at((cta + ncta - u0 % ncta) % ncta, 1);
  }
};

__device__ __forceinline__ bool tc_unit(const TcArgs& g, const UnitTab& tab, const UnitIt& it, TcUnit& w) {
  w.j = (int)it.j;
  w.s = (int)it.s;
  if (it.ti < (uint32_t)kUnitTab) {
    w.e = tab.e[it.ti];
    w.r0 = tab.r0[it.ti];
    w.r1 = tab.r1[it.ti];
  } else {
    w.e = g.touched[it.ti];
    w.r0 = g.offsets[w.e];
    w.r1 = g.offsets[w.e + 1];
  }
  w.c0 = tab.cb[it.mat][it.s];
  w.c1 = tab.cb[it.mat][it.s + 1];
  return w.c1 > w.c0 && w.r1 > w.r0;
}

// Waits (bounded, as the mbarrier waits) for a flag another CTA sets with a
// release store; acquire on success.
__device__ __forceinline__ bool wait_flag(const int32_t* flag, volatile int* abort,
                                          long long limit_cycles = 4000000000ll) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    if (ld_acquire_gpu(flag) != 0) return true;
    if ((it & 15) == 15) {
      if (*abort) return false;
      if (clock64() - t0 > limit_cycles) {
        *abort = 1;
        return false;
      }
    }
    __nanosleep(128);
  }
}

// The four epilogue warps' own barrier, and the same barrier returning
// whether v held in every one of its threads.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, 128, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Fused layer, W1 tile (group w.e, features 64 j .. 64 j + 63 of gate and
// up), its partials just written by this CTA's epilogue: y = w_row *
// act(gate, up) and the MXFP8 requant per 32 features, the same arithmetic
// as the separate epilogue kernel (which sums K slices; here there is one).
// Warp q takes feature block q & 1 of the rows r0 + (q >> 1),
// r0 + (q >> 1) + 2, ...
__device__ __noinline__ void fused_w1_tile(const TcArgs& g, const TcUnit& w, int q, int lane) {
  const TcFused& f = g.f;
  const TcMat& M = g.m[0];
  const int I = f.I, nb = I / 32;
  const int b = q & 1;
  const int fi = 64 * w.j + 32 * b + lane;
  for (int r = w.r0 + (q >> 1); r < w.r1; r += 2) {
    const float* P = M.out + (int64_t)r * 2 * I;
    float gg = 0.f, uu = 0.f;
#pragma unroll 4
    for (int s = 0; s < M.S; ++s) {
      gg += __ldcg(P + (int64_t)s * M.split_stride + fi);
      uu += __ldcg(P + (int64_t)s * M.split_stride + I + fi);
    }
    if (f.b1) {   // W1 bias of the group: gate b, up c
      gg += f.b1[(int64_t)w.e * 2 * I + fi];
      uu += f.b1[(int64_t)w.e * 2 * I + I + fi];
    }
    const float y = f.w_row[r] * act_fwd(gg, uu, f.act);
    const int e = mx_exponent(warp_max(fabsf(y)));
    f.y1q[(int64_t)r * I + fi] = (uint8_t)(f32x2_to_e4m3x2(y * pow2_neg(e), 0.f) & 0xffu);
    if (lane == 0) f.y1s[(int64_t)r * nb + 2 * w.j + b] = (uint8_t)(e + 127);
  }
}

// Fused layer, after the group's last W1 tile: its rows as the W2 operand,
// y16[r][i] = E4M3 value * 2^(block exponent - row exponent) with
// y_rowexp[r] the row's largest block exponent (as the separate epilogue
// kernel and k_act_f16 compute them). Warp q takes rows r0 + q, r0 + q + 4,
// ...; a row's loads are issued four code words a lane at a time ahead of
// the conversions (each is an L2 round trip: the rows were written by other
// CTAs), the scale bytes shared across the warp by shuffles.
__device__ __noinline__ void fused_w2_rows(const TcArgs& g, const TcUnit& w, int q, int lane) {
  const TcFused& f = g.f;
  const int I = f.I, nb = I / 32, nw = (I + 255) / 256;   // column words of 8 a lane (the last one partial)
  constexpr int kB = 4;   // code words in flight per lane
  for (int r = w.r0 + q; r < w.r1; r += 4) {
    const uint8_t* ss = f.y1s + (int64_t)r * nb;
    const uint8_t* qs = f.y1q + (int64_t)r * I;
    uint2 codes[kB];
#pragma unroll
    for (int k = 0; k < kB; ++k)
      codes[k] = lane * 8 + 256 * k < I ? __ldcg(reinterpret_cast<const uint2*>(qs + lane * 8 + 256 * k))
                                        : make_uint2(0u, 0u);
    // scale bytes of blocks lane and lane + 32
    const int sb0 = lane < nb ? (int)__ldcg(ss + lane) : 0;
    const int sb1 = lane + 32 < nb ? (int)__ldcg(ss + lane + 32) : 0;
    int mx = max(sb0, sb1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(kFull, mx, o));
    if (lane == 0) f.y_rowexp[r] = mx - 127;
    for (int k0 = 0; k0 < nw; k0 += kB) {
      if (k0 > 0) {
#pragma unroll
        for (int k = 0; k < kB; ++k)
          codes[k] = lane * 8 + 256 * (k0 + k) < I
                         ? __ldcg(reinterpret_cast<const uint2*>(qs + lane * 8 + 256 * (k0 + k)))
                         : make_uint2(0u, 0u);
      }
#pragma unroll
      for (int k = 0; k < kB; ++k) {
        if (k0 + k >= nw) break;   // uniform across the warp
        const int b = lane / 4 + 8 * (k0 + k);                 // block of columns lane * 8 + 256 (k0 + k)
        const int v0 = __shfl_sync(kFull, sb0, b & 31), v1 = __shfl_sync(kFull, sb1, b & 31);
        const float fs = ldexpf(1.0f, (b < 32 ? v0 : v1) - mx);
        uint32_t outw[4];
        const uint32_t cw[2] = {codes[k].x, codes[k].y};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float2 lo = e4m3x2_to_f32x2((uint16_t)(cw[h] & 0xffffu));
          const float2 hi = e4m3x2_to_f32x2((uint16_t)(cw[h] >> 16));
          const __half2 h0 = __floats2half2_rn(lo.x * fs, lo.y * fs);
          const __half2 h1 = __floats2half2_rn(hi.x * fs, hi.y * fs);
          outw[2 * h] = *reinterpret_cast<const uint32_t*>(&h0);
          outw[2 * h + 1] = *reinterpret_cast<const uint32_t*>(&h1);
        }
        if (lane * 8 + 256 * (k0 + k) < I)
          *reinterpret_cast<uint4*>(f.y16 + (int64_t)r * I + lane * 8 + 256 * (k0 + k)) =
              make_uint4(outw[0], outw[1], outw[2], outw[3]);
      }
    }
  }
}

__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two) {
  uint32_t r;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(r) : "r"(two));
  return r;
}
__device__ __forceinline__ void e2m1x8_f16x2(uint32_t w, uint32_t& o0, uint32_t& o1, uint32_t& o2, uint32_t& o3) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(o0), "=r"(o1), "=r"(o2), "=r"(o3)
      : "r"(w));
}
// Decodes one 64-wide K chunk of packed NVFP4 weight row p into 32 f16x2
// words (element pairs in K order): E2M1 value x E4M3 block scale, exact in
// f16.
__device__ __forceinline__ void decode_chunk(const uint8_t* sa, int p, uint32_t (&v)[32]) {
  const uint4 g0 = *reinterpret_cast<const uint4*>(sa + p * 16);
  const uint4 g1 = *reinterpret_cast<const uint4*>(sa + 2048 + p * 16);
  const uint32_t sc = *reinterpret_cast<const uint32_t*>(sa + 4096 + p * 4);
  const uint32_t s01 = e4m3x2_f16x2(sc & 0xffffu), s23 = e4m3x2_f16x2(sc >> 16);
  const uint32_t ss[4] = {(s01 & 0xffffu) * 0x10001u, (s01 >> 16) * 0x10001u, (s23 & 0xffffu) * 0x10001u,
                          (s23 >> 16) * 0x10001u};
  const uint32_t wd[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t o0, o1, o2, o3;
    e2m1x8_f16x2(wd[i], o0, o1, o2, o3);
    const uint32_t s = ss[i >> 1];
    v[4 * i + 0] = hmul2_bits(o0, s);
    v[4 * i + 1] = hmul2_bits(o1, s);
    v[4 * i + 2] = hmul2_bits(o2, s);
    v[4 * i + 3] = hmul2_bits(o3, s);
  }
}

// First index >= base that is congruent to r modulo m. Each role steps over
// its own pairs directly: a single-thread loop that tested and skipped the
// other roles' pairs spent most of its time resolving branches.
__device__ __forceinline__ uint32_t first_own(uint32_t base, uint32_t r, uint32_t m) {
  return base + (r + m - base % m) % m;
}

// Index of the activation row box (8 << index rows) for a tile with nv valid
// rows; the MMA still spans round_up(nv, 16) rows, and rows past the box
// (other chunks' data or stale shared memory) only reach accumulator columns
// of tokens past nv, which the epilogue never reads.
__device__ __forceinline__ int box_index(int nv) {
  return nv <= 8 ? 0 : nv <= 16 ? 1 : nv <= 32 ? 2 : nv <= 64 ? 3 : 4;
}

// ---------------------------------------------------------------------------
// f16 activation rows for the B operand.
// a16[r][k] = E4M3 value * 2^(block exponent - row exponent), rowexp[r] =
// the largest block exponent of the row (unbiased), so the product of the
// two is the MXFP8 value exactly unless a block sits more than 15 binades
// below the row's largest block (then bits below 2^-24 of the row scale are
// rounded away). One warp per (row, kActSlice-column slice); every warp
// derives the row exponent from the row's scale bytes itself. After the
// row index, every load of an item (the slice's codes, their block scales
// and the row's scale bytes) is issued before any is used, so an item costs
// two memory round trips.
// ---------------------------------------------------------------------------
constexpr int kActSlice = 2048;            // 8 chunks of 8 columns per lane

__device__ __forceinline__ void act_f16_item(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int C,
                                             const int32_t* __restrict__ row_map, int row_div, int64_t r, int sl,
                                             uint16_t* __restrict__ a16, int32_t* __restrict__ rowexp, int lane) {
  const int nb = C / 32;
  const int64_t src = row_map ? (int64_t)(row_map[r] / row_div) : r;
  const uint8_t* sr = s + src * nb;
  const uint8_t* qr = q + src * C;
  uint2 codes[8];
  int bs[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int c0 = sl * kActSlice + j * 256 + lane * 8;
    codes[j] = make_uint2(0u, 0u);
    bs[j] = 0;
    if (c0 < C) {
      codes[j] = *reinterpret_cast<const uint2*>(qr + c0);
      bs[j] = sr[c0 / 32];
    }
  }
  int mx = 0;
  for (int b0 = 0; b0 < nb; b0 += 256) {
    int sv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int b = b0 + lane + 32 * i;
      sv[i] = b < nb ? (int)sr[b] : 0;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) mx = max(mx, sv[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(kFull, mx, o));
  if (sl == 0 && lane == 0) rowexp[r] = mx - 127;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int c0 = sl * kActSlice + j * 256 + lane * 8;
    if (c0 >= C) break;
    const float f = ldexpf(1.0f, bs[j] - mx);
    uint32_t outw[4];
    const uint32_t cw[2] = {codes[j].x, codes[j].y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float2 lo = e4m3x2_to_f32x2((uint16_t)(cw[i] & 0xffffu));
      const float2 hi = e4m3x2_to_f32x2((uint16_t)(cw[i] >> 16));
      const __half2 h0 = __floats2half2_rn(lo.x * f, lo.y * f);
      const __half2 h1 = __floats2half2_rn(hi.x * f, hi.y * f);
      outw[2 * i] = *reinterpret_cast<const uint32_t*>(&h0);
      outw[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&h1);
    }
    *reinterpret_cast<uint4*>(a16 + r * C + c0) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
  }
}

// The partitioned layer's ring CTAs (n_disp of them): CTA d fills the W1
// operand rows of the touched groups d, d + n_disp, ... (the order the GEMM
// CTAs' walk needs them), all its warps on one group at a time, then raises
// the group's ring flag with a release store behind the CTA barrier.
__device__ void fill_ring(const TcArgs& g) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int C = g.m[0].K;
  const int nsl = (C + kActSlice - 1) / kActSlice;
  const int ntouch = *g.n_touched;
  int32_t* ring = g.f.cnt + 2 * g.G;
  for (int ti = blockIdx.x; ti < ntouch; ti += g.f.n_disp) {
    const int e = g.touched[ti];
    const int r0 = g.offsets[e];
    const int64_t items = (int64_t)(g.offsets[e + 1] - r0) * nsl;
    for (int64_t wi = warp; wi < items; wi += nw)
      act_f16_item(g.f.xq, g.f.xs, C, g.f.row_map, g.f.row_div, r0 + wi / nsl, (int)(wi % nsl), g.f.a16,
                   g.f.a_rowexp, lane);
    __syncthreads();
    if (threadIdx.x == 0) st_release_gpu(ring + e, 1);
  }
}

template <int NT>
__global__ void __launch_bounds__(kTcThreads, 1) k_gemm_tc(const __grid_constant__ TcArgs g,
                                                           const __grid_constant__ TcMaps maps) {
  using C = TcCfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* wring = smem;
  uint8_t* bring = smem + C::WS * C::WSlot;
  uint64_t* bars = reinterpret_cast<uint64_t*>(bring + C::BS * C::BSlot);
  uint64_t* wfull = bars;
  uint64_t* wempty = wfull + C::WS;
  uint64_t* bfull = wempty + C::WS;
  uint64_t* bempty = bfull + C::BS;
  uint64_t* afull = bempty + C::BS;
  uint64_t* afree = afull + kTcNA;
  uint64_t* dfull = afree + kTcNA;
  uint64_t* dfree = dfull + C::ND;
  uint64_t* drain = dfree + C::ND;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  __shared__ UnitTab tab;
  __shared__ UnitWalk walk;
  __shared__ int bad_pack;
  __shared__ int epi_last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_enter();
  if (threadIdx.x == 0) {
    bad_pack = !pack_header_ok(g.hdr, MOE_WFMT_NVFP4, g.which, g.G, g.bias != 0);
    if (bad_pack) set_status(g.status, MOE_DEV_BAD_PACK);
  }
  __syncthreads();
  if (bad_pack) return;   // the blob is not the packing this GEMM reads: write nothing
  // partitioned layer: the first n_disp CTAs fill the token ring and leave
  int n_disp = 0;
  if constexpr (NT == 16) {
    if (g.nmat == 2) n_disp = g.f.n_disp;
    if ((int)blockIdx.x < n_disp) {
      fill_ring(g);
      return;
    }
  }
  __shared__ int vgroups;   // entries of the walk's group axis
  {
    // The walk's groups: each touched group or, with split_rows > 0, each
    // block of at most split_rows of its rows (a multiple of NT, so the
    // token tiles are the same). A unit then covers at most split_rows / NT
    // token tiles and the round-robin spreads a hot group over many CTAs;
    // the weights are streamed once per token tile either way. When the
    // blocks do not fit the table, whole groups.
    __shared__ int scan_w[kTcThreads / 32 + 1];
    const int ntouch = *g.n_touched;
    const int RB = g.split_rows;
    const bool split = RB > 0 && ntouch <= (int)blockDim.x;
    const int i = threadIdx.x;
    int nb = 0, e = 0, r0 = 0, r1 = 0;
    if (split && i < ntouch) {
      e = g.touched[i];
      r0 = g.offsets[e];
      r1 = g.offsets[e + 1];
      nb = (r1 - r0 + RB - 1) / RB;
    }
    int incl = nb;   // block-wide exclusive scan of nb
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) scan_w[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      constexpr int nw = kTcThreads / 32;
      const int v = lane < nw ? scan_w[lane] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
      }
      if (lane < nw) scan_w[lane] = x - v;
      if (lane == 31) scan_w[nw] = x;
    }
    __syncthreads();
    const int total = scan_w[kTcThreads / 32];
    if (split && total <= kUnitTab) {
      const int base = scan_w[warp] + incl - nb;
      for (int k = 0; k < nb; ++k) {
        tab.e[base + k] = e;
        tab.r0[base + k] = r0 + k * RB;
        tab.r1[base + k] = min(r1, r0 + (k + 1) * RB);
      }
      if (i == 0) vgroups = total;
    } else {
      const int nt = min(ntouch, kUnitTab);
      for (int j = i; j < nt; j += blockDim.x) {
        const int ej = g.touched[j];
        tab.e[j] = ej;
        tab.r0[j] = g.offsets[ej];
        tab.r1[j] = g.offsets[ej + 1];
      }
      if (i == 0) vgroups = ntouch;
    }
    for (int m = 0; m < g.nmat; ++m) {
      const int nchunks = g.m[m].K / kChunkK, S = g.m[m].S;
      for (int i = threadIdx.x; i <= S; i += blockDim.x) tab.cb[m][i] = (int)((int64_t)i * nchunks / S);
    }
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::WS; ++i) {
      tc::mbar_init(&wfull[i], 1);
      tc::mbar_init(&wempty[i], 4);   // the 4 warps of the slot's decoder group
    }
    for (int i = 0; i < C::BS; ++i) {
      tc::mbar_init(&bfull[i], 1);
      tc::mbar_init(&bempty[i], 1);
    }
    for (int i = 0; i < kTcNA; ++i) {
      tc::mbar_init(&afull[i], 4);     // one elected arrive per decoder warp
      tc::mbar_init(&afree[i], 1);
    }
    for (int i = 0; i < C::ND; ++i) {
      tc::mbar_init(&dfull[i], C::P);
      tc::mbar_init(&dfree[i], 4);     // one elected arrive per epilogue warp
    }
    tc::mbar_init(drain, C::P);     // one commit from each MMA issuer
    // groups with rows (or their row blocks), over the GEMM CTAs
    walk.init(g, (uint32_t)vgroups, blockIdx.x - (uint32_t)n_disp, gridDim.x - (uint32_t)n_disp);
    *abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == kWIss) tc::tmem_alloc(tmem_slot, kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;



  // Every role walks the same sequence: units -> token tiles -> chunk pairs;
  // `ait` counts pairs (= weight stages).
  if (warp == 0 || warp == kWProd1) {
    // ---------------- weight producers ----------------
    const uint32_t pid = warp == 0 ? 0u : 1u;   // stages with (index % 2) == pid; WS is even
    if (lane == 0) {
      const uint64_t pol_w = tc::policy_evict_first();
      uint32_t wit = 0, issued = 0;   // issued: one past the last stage this thread issued
      bool ok = true;
      for (UnitIt it = walk.first(); ok && walk.more(it); walk.next(it)) {
        TcUnit w;
        if (!tc_unit(g, tab, it, w)) continue;
        const TcMat& M = g.m[it.mat];
        const uint8_t* tile = M.w + ((int64_t)w.e * M.tiles + w.j) * M.tile_bytes;
        const uint32_t npt = (uint32_t)(w.c1 - w.c0 + 1) >> 1;   // chunk pairs per token tile
        for (int t0 = w.r0; ok && t0 < w.r1; t0 += NT, wit += npt) {
          for (uint32_t i = first_own(wit, pid, 2); i < wit + npt; i += 2) {
            const int c = w.c0 + 2 * (int)(i - wit);
            const int nc = min(2, w.c1 - c);
            const int ws = i % C::WS;
            if (!tc::mbar_wait(&wempty[ws], ((i / C::WS) & 1) ^ 1, abort)) { ok = false; break; }
            tc::mbar_arrive_expect_tx(&wfull[ws], nc * C::CB);
            tc::bulk_g2s(wring + ws * C::WSlot, tile + (int64_t)c * C::CB, nc * C::CB, &wfull[ws], pol_w);
            issued = i + 1;
          }
        }
      }
      if (!ok || *abort) {
        // wind-down: wait (bounded, ignoring the abort flag) until every copy
        // still in flight into this CTA's shared memory has landed
        volatile int never = 0;
        const uint32_t n = issued < (uint32_t)C::WS ? issued : (uint32_t)C::WS;
        for (uint32_t k = 0; k < n; ++k) {
          const uint32_t i2 = issued - 1 - k;
          if ((i2 & 1u) == pid) tc::mbar_wait(&wfull[i2 % C::WS], (i2 / C::WS) & 1, &never, 400000000ll);
        }
      }
    }
  } else if (warp == kWBProd) {
    // ---------------- activation producer ----------------
    if (lane == 0) {
      for (int m = 0; m < g.nmat; ++m)
        for (int i = 0; i < kTcBoxes; ++i) tc::prefetch_tmap(&maps.m[m][i]);
      const uint64_t pol_a = tc::policy_evict_last();
      const int32_t* ready = g.f.cnt + g.G;
      const int32_t* ring = g.f.cnt + 2 * g.G;
      uint32_t ait = 0;
      int ready_e = -1, ring_e = -1;
      bool ok = true;
      for (UnitIt it = walk.first(); ok && walk.more(it); walk.next(it)) {
        TcUnit w;
        if (!tc_unit(g, tab, it, w)) continue;
        if (it.mat == 0 && n_disp > 0 && w.e != ring_e) {
          // partitioned layer: the group's W1 operand rows come from a ring CTA
          if (!wait_flag(ring + w.e, abort)) { ok = false; break; }
          fence_proxy_async_global();
          ring_e = w.e;
        }
        if (it.mat == 1 && w.e != ready_e) {
          // fused layer: the group's W2 operand rows are written by the CTA
          // that finished its last W1 tile; the copies below read them
          if (!wait_flag(ready + w.e, abort)) { ok = false; break; }
          fence_proxy_async_global();
          ready_e = w.e;
        }
        for (int t0 = w.r0; ok && t0 < w.r1; t0 += NT) {
          const int bi = box_index(min(NT, w.r1 - t0));
          const uint32_t b_bytes = 2u * (8u << bi) * 128u;
          for (int c = w.c0; c < w.c1; c += 2, ++ait) {
            const int bs = ait % C::BS;
            if (!tc::mbar_wait(&bempty[bs], ((ait / C::BS) & 1) ^ 1, abort)) { ok = false; break; }
            tc::mbar_arrive_expect_tx(&bfull[bs], b_bytes);
            // 2 chunks x (8 << bi) rows; a chunk past K reads as zero
            tc::tma_load_3d(bring + bs * C::BSlot, &maps.m[it.mat][bi], 0, t0, c, &bfull[bs], pol_a);
          }
        }
      }
      if (!ok || *abort) {
        volatile int never = 0;
        const uint32_t n = ait < (uint32_t)C::BS ? ait : (uint32_t)C::BS;
        for (uint32_t k = 0; k < n; ++k) {
          const uint32_t i2 = ait - 1 - k;
          tc::mbar_wait(&bfull[i2 % C::BS], (i2 / C::BS) & 1, &never, 400000000ll);
        }
      }
    }
  } else if (warp < kWDec) {
    // ---------------- MMA issuers ----------------
    const uint32_t mine = (uint32_t)(warp - kWIss);   // pairs with (index % P) == mine
    if (lane == 0 && mine < (uint32_t)C::P) {
      uint32_t ait = 0, dit = 0;
      bool ok = true;
      for (UnitIt it = walk.first(); ok && walk.more(it); walk.next(it)) {
        TcUnit w;
        if (!tc_unit(g, tab, it, w)) continue;
        for (int t0 = w.r0; ok && t0 < w.r1; t0 += NT) {
          const int nv = min(NT, w.r1 - t0);
          const int nmma = ((nv + 15) >> 4) << 4;
          const uint32_t b_chunk = (8u << box_index(nv)) * 128u;   // bytes per chunk in an activation slot
          const uint32_t idesc = tc::idesc_f16_f32(128, nmma);
          const int d = dit % C::ND;
          if (!tc::mbar_wait(&dfree[d], ((dit / C::ND) & 1) ^ 1, abort)) { ok = false; break; }
          tc::fence_after_sync();
          const uint32_t dt = tmem + kDCol0 + d * C::DStride + mine * NT;
          const uint32_t npt = (uint32_t)(w.c1 - w.c0 + 1) >> 1;   // chunk pairs per token tile
          uint32_t acc = 0;                                       // first MMA of the tile overwrites
          for (uint32_t i = first_own(ait, mine, C::P); i < ait + npt; i += C::P) {
            const int a = i % kTcNA, bs = i % C::BS;
            if (!tc::mbar_wait(&bfull[bs], (i / C::BS) & 1, abort)) { ok = false; break; }
            if (!tc::mbar_wait(&afull[a], (i / kTcNA) & 1, abort)) { ok = false; break; }
            tc::fence_after_sync();
            const uint32_t ta = tmem + a * 64;
            const uint64_t bd0 = tc::smem_desc_sw128(tc::smem_u32(bring + bs * C::BSlot));
            tc::mma_f16_ts(dt, ta, bd0, idesc, acc);
            tc::mma_f16_ts(dt, ta + 8, bd0 + 2, idesc, 1u);
            tc::mma_f16_ts(dt, ta + 16, bd0 + 4, idesc, 1u);
            tc::mma_f16_ts(dt, ta + 24, bd0 + 6, idesc, 1u);
            if (w.c0 + 2 * (int)(i - ait) + 1 < w.c1) {   // second chunk of the pair
              const uint64_t bd1 = bd0 + (uint64_t)(b_chunk >> 4);
              tc::mma_f16_ts(dt, ta + 32, bd1, idesc, 1u);
              tc::mma_f16_ts(dt, ta + 40, bd1 + 2, idesc, 1u);
              tc::mma_f16_ts(dt, ta + 48, bd1 + 4, idesc, 1u);
              tc::mma_f16_ts(dt, ta + 56, bd1 + 6, idesc, 1u);
            }
            acc = 1u;
            tc::mma_commit(&afree[a]);
            tc::mma_commit(&bempty[bs]);
          }
          ait += npt;
          if (!ok) break;
          tc::mma_commit(&dfull[d]);
          ++dit;
        }
      }
      // every MMA of this thread has completed once `drain` fires
      tc::mma_commit(drain);
      volatile int never = 0;
      tc::mbar_wait(drain, 0, &never, 400000000ll);
    }
  } else if (warp < kWEpi) {
    // ---------------- decoders ----------------
    const uint32_t grp = (uint32_t)(warp - kWDec) >> 2;   // pairs with (index % kTcNG) == grp
    const int q = warp & 3;                               // tensor-memory lane quarter of this warp
    const int p = q * 32 + lane;                          // weight row = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    uint32_t ait = 0;
    bool ok = true;
    for (UnitIt it = walk.first(); ok && walk.more(it); walk.next(it)) {
      TcUnit w;
      if (!tc_unit(g, tab, it, w)) continue;
      const uint32_t npt = (uint32_t)(w.c1 - w.c0 + 1) >> 1;   // chunk pairs per token tile
      for (int t0 = w.r0; ok && t0 < w.r1; t0 += NT, ait += npt) {
        for (uint32_t i = first_own(ait, grp, kTcNG); i < ait + npt; i += kTcNG) {
          const int c = w.c0 + 2 * (int)(i - ait);
          const int nc = min(2, w.c1 - c);
          const int ws = i % C::WS;
          if (!tc::mbar_wait(&wfull[ws], (i / C::WS) & 1, abort)) { ok = false; break; }
          const uint8_t* sa = wring + ws * C::WSlot;
          uint32_t v[32];
          decode_chunk(sa, p, v);
          const int a = i % kTcNA;
          if (!tc::mbar_wait(&afree[a], ((i / kTcNA) & 1) ^ 1, abort)) { ok = false; break; }
          tc::fence_after_sync();
          tc::tmem_st32(lane_base + a * 64, v);
          if (nc > 1) {
            decode_chunk(sa + C::CB, p, v);
            tc::tmem_st32(lane_base + a * 64 + 32, v);
          }
          // this warp has read its rows of the pair: release them
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&wempty[ws]);
          tc::tmem_wait_st();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&afull[a]);
        }
      }
    }
  } else if (warp < kWBProd) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;
    const int p = q * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
    const int32_t* ready = g.f.cnt + g.G;
    const int32_t* ring = g.f.cnt + 2 * g.G;
    int ready_e = -1, ring_e = -1;
    uint32_t dit = 0, ait = 0;
    bool ok = true;
    for (UnitIt it = walk.first(); ok && walk.more(it); walk.next(it)) {
      TcUnit w;
      if (!tc_unit(g, tab, it, w)) continue;
      const TcMat& M = g.m[it.mat];
      if (it.mat == 0 && n_disp > 0 && w.e != ring_e) {
        // partitioned layer: the row exponents of the group's W1 operand
        // rows come from a ring CTA
        if (!wait_flag(ring + w.e, abort)) { ok = false; break; }
        ring_e = w.e;
      }
      if (it.mat == 1 && w.e != ready_e) {
        // fused layer: the row exponents of the group's W2 operand come from
        // another CTA (already published: the MMAs consumed those rows)
        if (!wait_flag(ready + w.e, abort)) { ok = false; break; }
        ready_e = w.e;
      }
      // chunk pairs per token tile (the sequence the issuers walk)
      const int pairs = (w.c1 - w.c0 + 1) >> 1;
      int n;
      if (M.interleave_I > 0) n = p < 64 ? 64 * w.j + p : M.interleave_I + 64 * w.j + (p - 64);
      else n = kTileN * w.j + p;
      const bool nvalid = n < M.N;
      const float rowf = M.gs[w.e];
      float* outp = M.out + (int64_t)w.s * M.split_stride + n;
      for (int t0 = w.r0; t0 < w.r1; t0 += NT) {
        const int nt = min(NT, w.r1 - t0);
        // the tile's token scales 2^exponent, one per lane, shuffled out per
        // token below (W2's exponents in the fused layer come from another
        // CTA: every lane did its own acquire of the group's flag first)
        const float px0 = ldexpf(1.0f, lane < nt ? M.act_rowexp[t0 + lane] : 0);
        const float px1 = ldexpf(1.0f, NT > 32 && lane + 32 < nt ? M.act_rowexp[t0 + 32 + lane] : 0);
        const float px2 = ldexpf(1.0f, NT > 64 && lane + 64 < nt ? M.act_rowexp[t0 + 64 + lane] : 0);
        const float px3 = ldexpf(1.0f, NT > 64 && lane + 96 < nt ? M.act_rowexp[t0 + 96 + lane] : 0);
        const uint32_t a_first = ait;
        ait += pairs;
        const int d = dit % C::ND;
        if (!tc::mbar_wait(&dfull[d], (dit / C::ND) & 1, abort)) { ok = false; break; }
        tc::fence_after_sync();
        for (int cb = 0; cb < nt; cb += 16) {
          float acc[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[i] = 0.f;
          // issuer tiles in the order of the tile's own pair residues (pair
          // k of the tile went to issuer (a_first + k) % P), so the sum does
          // not depend on how many pairs this CTA ran before
          if constexpr (C::P == 2) {
            // both issuers' tiles in flight behind one wait
            uint32_t v0[16], v1[16];
            const uint32_t base = lane_base + kDCol0 + d * C::DStride + cb;
            tc::tmem_ld16(base + (a_first % 2) * NT, v0);
            if (pairs > 1) tc::tmem_ld16(base + ((a_first + 1) % 2) * NT, v1);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] += __uint_as_float(v0[i]);
            if (pairs > 1) {
#pragma unroll
              for (int i = 0; i < 16; ++i) acc[i] += __uint_as_float(v1[i]);
            }
          } else {
#pragma unroll
            for (int k = 0; k < C::P; ++k) {
              if (k >= pairs) continue;
              const int ac = (int)((a_first + (uint32_t)k) % C::P);
              uint32_t v[16];
              tc::tmem_ld16(lane_base + kDCol0 + d * C::DStride + ac * NT + cb, v);
              tc::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) acc[i] += __uint_as_float(v[i]);
            }
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int kk = (cb + i) >> 5;
            const float px = __shfl_sync(kFull, kk == 0 ? px0 : kk == 1 ? px1 : kk == 2 ? px2 : px3,
                                         (cb + i) & 31);   // every lane
            if (nvalid && cb + i < nt) outp[(int64_t)(t0 + cb + i) * M.N] = acc[i] * rowf * px;
          }
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&dfree[d]);
        ++dit;
      }
      if constexpr (NT == 16) if (it.mat == 0 && g.nmat > 1) {
        // Fused layer (W1 unsplit along K; 16-token tiles only, the host
        // runs it at a few rows per group): this unit wrote its tile's whole
        // partials. The four warps agree first on whether all of them got
        // here (a warp whose wait gave up arrives with ok = false), so none
        // is left alone at the barriers below. Hand-offs between CTAs are
        // the barrier, then one thread's gpu-scope release / acquire atomic
        // (no full fence, which would wait out this SM's copies in flight).
        if (!epi_all(ok)) { ok = false; break; }
        int32_t* cnt = g.f.cnt;
        const int tiles1 = g.m[0].tiles;
        // act * w and the requant of the tile's features
        fused_w1_tile(g, w, q, lane);
        epi_sync();
        if (warp == kWEpi && lane == 0) epi_last = atom_add_acq_rel_gpu(cnt + w.e, 1) == tiles1 - 1;
        epi_sync();
        if (epi_last) {
          // the group's last tile: its rows as the W2 operand, then the
          // flag its W2 units wait for (the tensor copies of other CTAs
          // read y16: generic writes, the proxy fence, then the release)
          fused_w2_rows(g, w, q, lane);
          fence_proxy_async_global();
          epi_sync();
          if (warp == kWEpi && lane == 0) st_release_gpu(cnt + g.G + w.e, 1);
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x == 0 && *abort) set_status(g.status, MOE_DEV_TIMEOUT);
  if (warp == kWIss) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}


// f16 matrix [rows][cols] viewed as (64 columns, rows, cols / 64 chunks),
// strides (2 B, cols * 2 B, 128 B); boxes of 64 x (8 << i) x 2 chunks,
// 128-byte swizzle; rows past the end and chunks past the last read as zero.
bool make_tmaps_b(CUtensorMap (&m)[kTcBoxes], const void* base, int64_t rows, int64_t cols) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || cols % kChunkK != 0) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kChunkK, (cuuint64_t)std::max<int64_t>(rows, 1), (cuuint64_t)(cols / kChunkK)};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)kChunkK * 2};
  cuuint32_t estr[3] = {1, 1, 1};
  for (int i = 0; i < kTcBoxes; ++i) {
    cuuint32_t box[3] = {(cuuint32_t)kChunkK, 8u << i, 2u};
    if (fn(&m[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

template <int NT>
static cudaError_t launch_tc_t(const TcArgs& g, const TcMaps& maps, int grid, cudaStream_t st) {
  static std::atomic<bool> done[kMaxDevices] = {};
  cudaError_t e = set_smem_once((const void*)k_gemm_tc<NT>, TcCfg<NT>::SmemBytes, done);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_gemm_tc<NT>, dim3(grid), dim3(kTcThreads), (size_t)TcCfg<NT>::SmemBytes, st, g, maps);
}

int tc_token_tile(int T, int kp, int G) {
  const double avg = (double)T * kp / std::max(G, 1);
  if (avg <= 12.0) return 16;
  if (avg <= 24.0) return 32;
  if (avg <= 96.0) return 64;
  return 128;   // prefill-sized groups: each decoded weight pair feeds 128 tokens
}

cudaError_t launch_gemm_tc(const TcArgs& g, const TcMaps& maps, int nt, cudaStream_t st) {
  const int grid = std::max(1, g.max_ctas);
  const cudaError_t e = nt <= 16 ? launch_tc_t<16>(g, maps, grid, st)
                        : nt <= 32 ? launch_tc_t<32>(g, maps, grid, st)
                        : nt <= 64 ? launch_tc_t<64>(g, maps, grid, st)
                                   : launch_tc_t<128>(g, maps, grid, st);
  note_launch();
  return e;
}

__global__ void __launch_bounds__(256) k_act_f16(const uint8_t* __restrict__ q, const uint8_t* __restrict__ s, int C,
                                                 const int32_t* __restrict__ row_map, int row_div, int R,
                                                 const int32_t* __restrict__ offsets, int G, uint16_t* __restrict__ a16,
                                                 int32_t* __restrict__ rowexp, int32_t* __restrict__ zero,
                                                 int64_t nzero) {
  pdl_enter();
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nzero; i += (int64_t)gridDim.x * blockDim.x)
    zero[i] = 0;
  const int lane = threadIdx.x & 31;
  const int Rv = min(R, offsets[G]);
  const int nsl = (C + kActSlice - 1) / kActSlice;
  const int64_t total = (int64_t)Rv * nsl;
  const int64_t nw = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t wi = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); wi < total; wi += nw)
    act_f16_item(q, s, C, row_map, row_div, wi / nsl, (int)(wi % nsl), a16, rowexp, lane);
}

// The fused layer's flag wait on its own: one thread waits (bounded by
// limit_cycles) for *flag != 0 and sets MOE_DEV_TIMEOUT when it gives up.
__global__ void k_debug_flag_wait(const int32_t* flag, long long limit_cycles, int32_t* status) {
  __shared__ volatile int abort_;
  if (threadIdx.x != 0) return;
  abort_ = 0;
  if (!wait_flag(flag, &abort_, limit_cycles)) set_status(status, MOE_DEV_TIMEOUT);
}

cudaError_t launch_debug_flag_wait(const int32_t* flag, long long limit_cycles, int32_t* status, cudaStream_t st) {
  k_debug_flag_wait<<<1, 32, 0, st>>>(flag, limit_cycles, status);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_act_f16(const uint8_t* q, const uint8_t* s, int C, const int32_t* row_map, int row_div, int R,
                           const int32_t* offsets, int G, uint16_t* a16, int32_t* rowexp, cudaStream_t st,
                           int32_t* zero, int64_t nzero) {
  if (R == 0) return cudaSuccess;
  if (!zero) nzero = 0;
  const int64_t warps = (int64_t)R * ((C + kActSlice - 1) / kActSlice);
  const int64_t work = std::max<int64_t>((warps + 7) / 8, (nzero + 255) / 256);
  const int blocks = (int)std::min<int64_t>(work, (int64_t)device_sms() * 8);   // one wave
  cudaError_t e = launch_pdl(k_act_f16, dim3(blocks), dim3(256), 0, st, q, s, C, row_map, row_div, R, offsets, G,
                             a16, rowexp, zero, nzero);
  note_launch();
  return e;
}

}  // namespace moe
