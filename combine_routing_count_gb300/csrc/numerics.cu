// Kernels that compute on the payload: block-scaled fp8 quantisation of the dispatch rows,
// the fp8 identity expert (dequantisation to bf16), and the combine reduction.
//
// "Enabling trillion-parameter models on AWS EFA" (Perplexity), section "Evaluation":
// block-scaled fp8 dispatch and bf16 combine; section "Dispatch and combine": combine
// accumulates the tokens from the receive buffer into the output tensor, a weighted
// average over each token's experts, on the receiving side only.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Half a warp per 128-element block: each lane holds 8 bf16 values (one 16-byte load).
// amax over the block by xor-shuffles inside the half warp; scale = RN(amax / 448) (1 when
// amax is 0); codes = e4m3(RN(x / scale)), round to nearest even, saturating: bit for bit the
// fp32 division, computed without dividing (block_scale, quant_unit below).
// Output row: H codes, then H/128 fp32 scales. 4-byte stores (rows are 4-byte aligned).
// A warp takes kQuantUnroll pairs of blocks of one row per trip (one index division per
// trip) and issues all their loads first.
constexpr int kQuantUnroll = 4;

// Two fp32 values to two e4m3 codes, round to nearest even, saturating to +-448; lo goes to
// the low byte (the conversion puts its first source operand in the upper byte).
__device__ __forceinline__ uint32_t e4m3x2_rn_sat(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// Two e4m3 codes (low byte first) to two f16 values (exact: every e4m3 value is an f16 value).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t c) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(c));
  return d;
}

__device__ __forceinline__ float e4m3_value(uint32_t c) {
  return __half2float(__ushort_as_half((unsigned short)(e4m3x2_to_f16x2((uint16_t)c) & 0xffffu)));
}

// Four e4m3 codes (low byte first) of four fp32 values.
__device__ __forceinline__ uint32_t e4m3x4_rn_sat(float a, float b, float c, float d) {
  uint32_t w;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(w) : "f"(a), "f"(b), "f"(c), "f"(d));
  return w;
}

// The code of RN(x / scale) for a value whose bracket (below) gave the two adjacent codes cl and
// ch, values a and b, with the e4m3 rounding boundary m = (a + b) / 2 between them. m has at most
// five significant bits, so it is even in fp32 and RN(x / scale) == m (a tie, rounded to the even
// code) exactly when |x / scale - m| <= ulp(m) / 2, that is when |x - m * scale| <= t with
// t = ulp(m) / 2 * scale; otherwise the quotient lies on the side of m that x - m * scale has.
// d = fma(-m, scale, x) is that difference rounded once (exact for scale >= 2^-90): it has the
// exact sign and decides the comparison unless it lands on t itself, where the quotient is
// divided.
__device__ __forceinline__ uint32_t e4m3_resolve(float x, float scale, uint32_t cl, uint32_t ch) {
  const float a = e4m3_value(cl), b = e4m3_value(ch);
  const float m = __fmul_rn(__fadd_rn(a, b), 0.5f);
  const float d = __fmaf_rn(-m, scale, x);
  const float t = __fmul_rn(__fmul_rn(__uint_as_float(__float_as_uint(m) & 0x7f800000u), 0x1p-24f), scale);
  const float ad = fabsf(d);
  if (ad < t) return (cl & 1u) ? ch : cl;
  if (ad > t) return ((d > 0.0f) == (a > b)) ? cl : ch;
  return e4m3x2_rn_sat(__fdiv_rn(x, scale), 0.0f) & 0xffu;
}

// scale = RN(amax / 448) of a block's amax (a bf16 value), 1 for amax 0. Above 2^-100 without a
// division: q0 = RN(amax * c) with c = RN(1/448), the remainder amax - 448 * q0 (exact, one
// fma), and Markstein's correction RN(q0 + remainder * c). That this equals the correctly
// rounded quotient was checked, with exact rational arithmetic, for every bf16 value from
// 2^-100 up to the largest finite one.
__device__ __forceinline__ float block_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  if (amax < 0x1p-100f) return __fdiv_rn(amax, 448.0f);
  constexpr float c = 1.0f / 448.0f;
  const float q0 = __fmul_rn(amax, c);
  return __fmaf_rn(__fmaf_rn(-q0, 448.0f, amax), c, q0);
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Bit k of the result: byte k of d is nonzero.
__device__ __forceinline__ uint32_t nonzero_bytes(uint32_t d) {
  d |= d >> 4;
  d |= d >> 2;
  d |= d >> 1;
  return ((d & 0x01010101u) * 0x01020408u) >> 24;
}

// Codes of q = RN(x / scale) without a division per value. With r an approximate 1 / scale
// (relative error at most 2^-23), lo = RN(x * RN(r * (1 - 2^-19))) and hi = RN(x * RN(r * (1 +
// 2^-19))) bracket q strictly: r and the three roundings move a value by well under 2^-19
// together. Rounding to e4m3 is monotonic, so where lo and hi get the same code, q gets it too.
__device__ __forceinline__ void bracket_rcp(float scale, float& rlo, float& rhi) {
  const float r = rcp_approx(scale);
  rlo = __fmul_rn(r, 1.0f - 0x1p-19f);
  rhi = __fmul_rn(r, 1.0f + 0x1p-19f);
}

// The code of RN(x / scale) for one value, exactly: the bracket, and where its ends differ,
// e4m3_resolve; a tiny or subnormal scale divides.
__device__ __forceinline__ uint32_t e4m3_code_exact(float x, float scale) {
  if (scale < 0x1p-90f) return e4m3x2_rn_sat(__fdiv_rn(x, scale), 0.0f) & 0xffu;
  float rlo, rhi;
  bracket_rcp(scale, rlo, rhi);
  const uint32_t cl = e4m3x2_rn_sat(__fmul_rn(x, rlo), 0.0f) & 0xffu;
  const uint32_t ch = e4m3x2_rn_sat(__fmul_rn(x, rhi), 0.0f) & 0xffu;
  return cl == ch ? cl : e4m3_resolve(x, scale, cl, ch);
}

// One warp unit of a row: lane (half h, sub) loads blocks bbase + 2j (bbase already holds h)
// and quantises its 8 values of each; codes[j] are its codes, scale[j] its block's scale.
// Blocks at or past nb read as zeros. The codes come from the lower end of the quotient
// bracket; the values whose bracket ends disagree (about 1 in 200 for bf16 data, mostly exact
// ties) are flagged and settled afterwards, one by one, by e4m3_code_exact, which keeps that
// code out of the unrolled main path.
__device__ __forceinline__ void quant_unit(const uint16_t* xr, int bbase, int nb, uint32_t (&codes)[kQuantUnroll][2],
                                           float (&scale)[kQuantUnroll]) {
  uint4 v[kQuantUnroll];
#pragma unroll
  for (int j = 0; j < kQuantUnroll; ++j) {
    const int b = bbase + 2 * j;
    v[j] = b < nb ? ld_stream16(xr + b * 128) : make_uint4(0, 0, 0, 0);
  }
  uint32_t diff[kQuantUnroll][2];   // bytes where the bracket ends disagree
  uint32_t any = 0;
#pragma unroll
  for (int j = 0; j < kQuantUnroll; ++j) {
    const float f[8] = {bf16_lo(v[j].x), bf16_hi(v[j].x), bf16_lo(v[j].y), bf16_hi(v[j].y),
                        bf16_lo(v[j].z), bf16_hi(v[j].z), bf16_lo(v[j].w), bf16_hi(v[j].w)};
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o, 16));
    const float sc = block_scale(amax);
    scale[j] = sc;
    const bool tiny = sc < 0x1p-90f;
    float rlo, rhi;
    bracket_rcp(tiny ? 1.0f : sc, rlo, rhi);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float* fi = f + 4 * i;
      const uint32_t wl = e4m3x4_rn_sat(__fmul_rn(fi[0], rlo), __fmul_rn(fi[1], rlo), __fmul_rn(fi[2], rlo),
                                        __fmul_rn(fi[3], rlo));
      const uint32_t wh = e4m3x4_rn_sat(__fmul_rn(fi[0], rhi), __fmul_rn(fi[1], rhi), __fmul_rn(fi[2], rhi),
                                        __fmul_rn(fi[3], rhi));
      codes[j][i] = wl;
      diff[j][i] = tiny ? 0xffffffffu : (wl ^ wh);
      any |= diff[j][i];
    }
  }
  if (!any) return;
  uint32_t pend = 0;   // bit 8j + 4i + e: value e of word i of block j to settle
#pragma unroll
  for (int j = 0; j < kQuantUnroll; ++j)
#pragma unroll
    for (int i = 0; i < 2; ++i) pend |= nonzero_bytes(diff[j][i]) << (8 * j + 4 * i);
  while (pend) {
    const int bit = __ffs(pend) - 1;
    pend &= pend - 1;
    const int j = bit >> 3, w = bit >> 2, e = bit & 3;
    const int q = 2 * (w & 1) + (e >> 1);   // component of v[j] holding the value
    float sc = scale[0];
    uint32_t pair = v[0].x;
#pragma unroll
    for (int jj = 0; jj < kQuantUnroll; ++jj) {
      sc = j == jj ? scale[jj] : sc;
      pair = (j == jj && q == 0) ? v[jj].x : pair;
      pair = (j == jj && q == 1) ? v[jj].y : pair;
      pair = (j == jj && q == 2) ? v[jj].z : pair;
      pair = (j == jj && q == 3) ? v[jj].w : pair;
    }
    const uint32_t c = e4m3_code_exact((e & 1) ? bf16_hi(pair) : bf16_lo(pair), sc);
#pragma unroll
    for (int jj = 0; jj < kQuantUnroll; ++jj)
#pragma unroll
      for (int ii = 0; ii < 2; ++ii)
        if (w == 2 * jj + ii) codes[jj][ii] = (codes[jj][ii] & ~(0xffu << (8 * e))) | (c << (8 * e));
  }
}

__global__ void __launch_bounds__(256) k_quant_fp8(Geo g, const uint16_t* __restrict__ x, uint8_t* __restrict__ xq) {
  const int nb = g.H / 128;
  const int upr = (nb + 2 * kQuantUnroll - 1) / (2 * kQuantUnroll);   // warp units per row
  const int64_t units = (int64_t)g.N * g.T * upr;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 15;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  pdl_wait();
  for (int64_t u = warp; u < units; u += nwarps) {   // warp-uniform
    const int64_t row = units <= INT32_MAX ? (int64_t)((uint32_t)u / (uint32_t)upr) : u / upr;
    const int bbase = (int)(u - row * upr) * 2 * kQuantUnroll + (lane >> 4);   // block of j = 0
    uint32_t codes[kQuantUnroll][2];
    float scale[kQuantUnroll];
    quant_unit(x + row * g.H + sub * 8, bbase, nb, codes, scale);
    uint8_t* qr = xq + row * g.B;
#pragma unroll
    for (int j = 0; j < kQuantUnroll; ++j) {
      const int b = bbase + 2 * j;
      if (b < nb) {
        uint32_t* dst = reinterpret_cast<uint32_t*>(qr + b * 128 + sub * 8);
        dst[0] = codes[j][0];
        dst[1] = codes[j][1];
        if (sub == 0) *reinterpret_cast<float*>(qr + g.H + 4 * b) = scale[j];
      }
    }
  }
  pdl_trigger();
}

// Quantisation fused into the pack: a warp unit quantises its blocks of a token row once, in
// registers, and writes them into the R rows fan[token][k] of dst (send rows, or receive rows
// when pushing), so the fp8 rows are never staged in HBM. The bytes each row gets are those
// moe_quantize_fp8_b128 writes. W8: rows are 8-byte aligned (8-byte code stores).
// RANGED: only the token range [t0, t0 + nt) of every rank (else every token; t0, nt unused).
// ALL 1: the write and the shuffle as well (pack-all): every pair's codes and scales also go to
// its receive row (recv at grecv) and, when the pair is kept, to its grouped row (codes at
// ex + gslot * H, scales at exs + gslot * H / 128), the bytes moe_dispatch_recv writes.
// ALL 2: the same with direct push: no send rows (dst unused), and the receive rows, which no
// later kernel of the pass reads, go through L2 marked evict-first. A compile-time choice, as
// a run-time test of dst measured 20% more instructions in the default kernel.
struct FanAll {
  const int32_t* grecv;
  const int32_t* gslot;
  uint8_t* recv;
  uint8_t* ex;
  float* exs;
};

template <bool W8, bool RANGED, int ALL>
__global__ void __launch_bounds__(256) k_quant_pack(Geo g, const uint16_t* __restrict__ x,
                                                    const int32_t* __restrict__ fan, uint8_t* __restrict__ dst,
                                                    int t0, int nt, FanAll fa) {
  const int nb = g.H / 128;
  const int upr = (nb + 2 * kQuantUnroll - 1) / (2 * kQuantUnroll);
  const int64_t units = (int64_t)g.N * (RANGED ? nt : g.T) * upr;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 15;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  pdl_wait();
  for (int64_t u = warp; u < units; u += nwarps) {   // warp-uniform
    const int64_t rv = units <= INT32_MAX ? (int64_t)((uint32_t)u / (uint32_t)upr) : u / upr;
    const int bbase = (int)(u - rv * upr) * 2 * kQuantUnroll + (lane >> 4);
    const int64_t row = RANGED ? (rv / nt) * g.T + t0 + rv % nt : rv;   // token
    const int32_t* fr = fan + row * g.R;
    const int myp = lane < g.R ? __ldg(fr + lane) : -1;   // rows of pairs 0..31 (R > 32: loaded)
    const int myr = (ALL && lane < g.R) ? __ldg(fa.grecv + row * g.R + lane) : -1;
    const int myl = (ALL && lane < g.R) ? __ldg(fa.gslot + row * g.R + lane) : -1;
    uint32_t codes[kQuantUnroll][2];
    float scale[kQuantUnroll];
    quant_unit(x + row * g.H + sub * 8, bbase, nb, codes, scale);
#pragma unroll 1
    for (int k = 0; k < g.R; ++k) {
      const int p = k < 32 ? __shfl_sync(kFull, myp, k) : __ldg(fr + k);
      const int rr = ALL ? (k < 32 ? __shfl_sync(kFull, myr, k) : __ldg(fa.grecv + row * g.R + k)) : -1;
      const int rl = ALL ? (k < 32 ? __shfl_sync(kFull, myl, k) : __ldg(fa.gslot + row * g.R + k)) : -1;
      if (p < 0) continue;
#pragma unroll 1
      for (int dsel = ALL == 2 ? 1 : 0; dsel < (ALL ? 3 : 1); ++dsel) {   // send (none with direct push), receive, grouped
        if (dsel == 2 && rl < 0) break;
        uint8_t* dr = dsel == 0 ? dst + (int64_t)p * g.B
                                : dsel == 1 ? fa.recv + (int64_t)rr * g.B : fa.ex + (int64_t)rl * g.H;
#pragma unroll
        for (int j = 0; j < kQuantUnroll; ++j) {
          const int b = bbase + 2 * j;
          if (b < nb) {
            uint8_t* c = dr + b * 128 + sub * 8;
            if (W8 || dsel == 2) {   // grouped code rows (H bytes) are always 8-byte aligned
              *reinterpret_cast<uint2*>(c) = make_uint2(codes[j][0], codes[j][1]);
            } else {
              reinterpret_cast<uint32_t*>(c)[0] = codes[j][0];
              reinterpret_cast<uint32_t*>(c)[1] = codes[j][1];
            }
            if (sub == 0) {
              float* sp = dsel < 2 ? reinterpret_cast<float*>(dr + g.H + 4 * b) : fa.exs + (int64_t)rl * nb + b;
              *sp = scale[j];
            }
          }
        }
      }
    }
  }
  pdl_trigger();
}

// The fused quantise-and-pack for rows that are 16-byte multiples: 8 lanes per 128-value
// block and 16 consecutive values per lane (two 16-byte loads), so that each destination
// row gets one 16-byte code store per lane and block instead of two 8-byte ones. A warp
// unit covers blocks 8u .. 8u+7 of a row: lane (q, sub) takes block 8u + q + 4j, j < 2.
// Same products, conversions, bracket and settling as quant_unit, value for value.
constexpr int kQ16Blocks = 2;   // blocks per lane and unit

__device__ __forceinline__ void quant_unit16(const uint16_t* xr, int bbase, int nb, int sub,
                                             uint32_t (&codes)[kQ16Blocks][4], float (&scale)[kQ16Blocks]) {
  uint4 v[kQ16Blocks][2];
#pragma unroll
  for (int j = 0; j < kQ16Blocks; ++j) {
    const int b = bbase + 4 * j;
    const uint16_t* p = xr + b * 128 + sub * 16;
    v[j][0] = b < nb ? ld_stream16(p) : make_uint4(0, 0, 0, 0);
    v[j][1] = b < nb ? ld_stream16(p + 8) : make_uint4(0, 0, 0, 0);
  }
  uint32_t any = 0, pend = 0;   // pend bit 16j + 4i + e: value e of word i of block j to settle
#pragma unroll
  for (int j = 0; j < kQ16Blocks; ++j) {
    const uint32_t u[8] = {v[j][0].x, v[j][0].y, v[j][0].z, v[j][0].w, v[j][1].x, v[j][1].y, v[j][1].z, v[j][1].w};
    float f[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f[2 * i] = bf16_lo(u[i]);
      f[2 * i + 1] = bf16_hi(u[i]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
    for (int o = 4; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o, 8));
    const float sc = block_scale(amax);
    scale[j] = sc;
    const bool tiny = sc < 0x1p-90f;
    float rlo, rhi;
    bracket_rcp(tiny ? 1.0f : sc, rlo, rhi);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float* fi = f + 4 * i;
      const uint32_t wl = e4m3x4_rn_sat(__fmul_rn(fi[0], rlo), __fmul_rn(fi[1], rlo), __fmul_rn(fi[2], rlo),
                                        __fmul_rn(fi[3], rlo));
      const uint32_t wh = e4m3x4_rn_sat(__fmul_rn(fi[0], rhi), __fmul_rn(fi[1], rhi), __fmul_rn(fi[2], rhi),
                                        __fmul_rn(fi[3], rhi));
      codes[j][i] = wl;
      const uint32_t d = tiny ? 0xffffffffu : (wl ^ wh);
      any |= d;
      pend |= nonzero_bytes(d) << (16 * j + 4 * i);
    }
  }
  if (!any) return;
  while (pend) {
    const int bit = __ffs(pend) - 1;
    pend &= pend - 1;
    const int j = bit >> 4, i = (bit >> 2) & 3, e = bit & 3;
    const int k = 4 * i + e;            // value of the lane's 16
    const int h = k >> 3, q = (k & 7) >> 1;
    float sc = scale[0];
    uint32_t pair = v[0][0].x;
#pragma unroll
    for (int jj = 0; jj < kQ16Blocks; ++jj) {
      sc = j == jj ? scale[jj] : sc;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const bool at = j == jj && h == hh;
        pair = (at && q == 0) ? v[jj][hh].x : pair;
        pair = (at && q == 1) ? v[jj][hh].y : pair;
        pair = (at && q == 2) ? v[jj][hh].z : pair;
        pair = (at && q == 3) ? v[jj][hh].w : pair;
      }
    }
    const uint32_t c = e4m3_code_exact((k & 1) ? bf16_hi(pair) : bf16_lo(pair), sc);
#pragma unroll
    for (int jj = 0; jj < kQ16Blocks; ++jj)
#pragma unroll
      for (int ii = 0; ii < 4; ++ii)
        if (j == jj && i == ii) codes[jj][ii] = (codes[jj][ii] & ~(0xffu << (8 * e))) | (c << (8 * e));
  }
}

// moe_quantize_fp8_b128 for rows that are 16-byte multiples: quant_unit16's lane layout,
// one 16-byte code store per lane and block.
__global__ void __launch_bounds__(256) k_quant_fp8_16(Geo g, const uint16_t* __restrict__ x,
                                                      uint8_t* __restrict__ xq) {
  const int nb = g.H / 128;
  const int upr = (nb + 7) / 8;   // warp units per row
  const int64_t units = (int64_t)g.N * g.T * upr;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  pdl_wait();
  for (int64_t u = warp; u < units; u += nwarps) {   // warp-uniform
    const int64_t row = units <= INT32_MAX ? (int64_t)((uint32_t)u / (uint32_t)upr) : u / upr;
    const int bbase = (int)(u - row * upr) * 8 + (lane >> 3);   // block of j = 0
    uint32_t codes[kQ16Blocks][4];
    float scale[kQ16Blocks];
    quant_unit16(x + row * g.H, bbase, nb, sub, codes, scale);
    uint8_t* qr = xq + row * g.B;
#pragma unroll
    for (int j = 0; j < kQ16Blocks; ++j) {
      const int b = bbase + 4 * j;
      if (b < nb) {
        *reinterpret_cast<uint4*>(qr + b * 128 + sub * 16) = make_uint4(codes[j][0], codes[j][1], codes[j][2],
                                                                        codes[j][3]);
        if (sub == 0) *reinterpret_cast<float*>(qr + g.H + 4 * b) = scale[j];
      }
    }
  }
  pdl_trigger();
}

template <bool RANGED, int ALL>
__global__ void __launch_bounds__(256) k_quant_pack16(Geo g, const uint16_t* __restrict__ x,
                                                      const int32_t* __restrict__ fan, uint8_t* __restrict__ dst,
                                                      int t0, int nt, FanAll fa) {
  const int nb = g.H / 128;
  const int upr = (nb + 7) / 8;   // warp units per row
  const int64_t units = (int64_t)g.N * (RANGED ? nt : g.T) * upr;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 7;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  pdl_wait();
  for (int64_t u = warp; u < units; u += nwarps) {   // warp-uniform
    const int64_t rv = units <= INT32_MAX ? (int64_t)((uint32_t)u / (uint32_t)upr) : u / upr;
    const int bbase = (int)(u - rv * upr) * 8 + (lane >> 3);   // block of j = 0
    const int64_t row = RANGED ? (rv / nt) * g.T + t0 + rv % nt : rv;   // token
    const int32_t* fr = fan + row * g.R;
    const int myp = lane < g.R ? __ldg(fr + lane) : -1;   // rows of pairs 0..31 (R > 32: loaded)
    const int myr = (ALL && lane < g.R) ? __ldg(fa.grecv + row * g.R + lane) : -1;
    const int myl = (ALL && lane < g.R) ? __ldg(fa.gslot + row * g.R + lane) : -1;
    uint32_t codes[kQ16Blocks][4];
    float scale[kQ16Blocks];
    quant_unit16(x + row * g.H, bbase, nb, sub, codes, scale);
#pragma unroll 1
    for (int k = 0; k < g.R; ++k) {
      const int p = k < 32 ? __shfl_sync(kFull, myp, k) : __ldg(fr + k);
      const int rr = ALL ? (k < 32 ? __shfl_sync(kFull, myr, k) : __ldg(fa.grecv + row * g.R + k)) : -1;
      const int rl = ALL ? (k < 32 ? __shfl_sync(kFull, myl, k) : __ldg(fa.gslot + row * g.R + k)) : -1;
      if (p < 0) continue;
#pragma unroll 1
      for (int dsel = ALL == 2 ? 1 : 0; dsel < (ALL ? 3 : 1); ++dsel) {   // send (none with direct push), receive, grouped
        if (dsel == 2 && rl < 0) break;
        uint8_t* dr = dsel == 0 ? dst + (int64_t)p * g.B
                                : dsel == 1 ? fa.recv + (int64_t)rr * g.B : fa.ex + (int64_t)rl * g.H;
#pragma unroll
        for (int j = 0; j < kQ16Blocks; ++j) {
          const int b = bbase + 4 * j;
          if (b < nb) {
            const uint4 cw = make_uint4(codes[j][0], codes[j][1], codes[j][2], codes[j][3]);
            if (ALL == 2 && dsel == 1)   // direct push: no kernel of the pass reads the receive rows
              st16_hint(dr + b * 128 + sub * 16, cw, l2_evict_first_policy());
            else
              *reinterpret_cast<uint4*>(dr + b * 128 + sub * 16) = cw;
            if (sub == 0) {
              float* sp = dsel < 2 ? reinterpret_cast<float*>(dr + g.H + 4 * b) : fa.exs + (int64_t)rl * nb + b;
              *sp = scale[j];
            }
          }
        }
      }
    }
  }
  pdl_trigger();
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t a = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t b = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return a | (b << 16);
}

// y = bf16(float(code) * scale) for two codes (low byte first).
__device__ __forceinline__ uint32_t dequant2(uint16_t codes, float scale) {
  const uint32_t h = e4m3x2_to_f16x2(codes);
  const float lo = __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
  const float hi = __half2float(__ushort_as_half((unsigned short)(h >> 16)));
  return pack_bf16x2(__fmul_rn(lo, scale), __fmul_rn(hi, scale));
}

// Identity expert for the fp8 payload: one warp per used grouped row (found through the
// pairs' gslot), 16 codes per lane per load, kDequantUnroll loads in flight per lane.
// REV: pairs in descending order, for grouped rows that the unpack wrote in that order
// (direct push), so that the rows written last, still in L2, are read first. RANGED: only
// the pairs of tokens [t0, t0 + nt) of every rank (np = N * nt * R of them).
constexpr int kDequantUnroll = 4;

template <bool REV, bool RANGED>
__global__ void __launch_bounds__(256) k_dequant_fp8(Geo g, const int32_t* __restrict__ gslot,
                                                     const uint8_t* __restrict__ exq, const float* __restrict__ exs,
                                                     uint16_t* __restrict__ ey, int t0, int nt, int64_t np,
                                                     int64_t win_rows, int win_lo, int win_n) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nvec = g.H / 16;
  pdl_wait();
  for (int64_t q0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; q0 < np; q0 += nwarps) {
    int64_t q = REV ? np - 1 - q0 : q0;
    if (RANGED) {
      const int64_t span = (int64_t)nt * g.R, s = q / span;
      q = (s * g.T + t0) * g.R + (q - s * span);
    }
    const int gl = __ldg(gslot + q);
    if (gl < 0) continue;
    // a rank window: only the grouped rows of its ranks (win_rows = L * cap rows a rank)
    if (win_rows != 0 && (uint64_t)(gl / win_rows - win_lo) >= (uint64_t)win_n) continue;
    const uint8_t* qr = exq + (int64_t)gl * g.H;
    const float* sr = exs + (int64_t)gl * (g.H / 128);
    uint16_t* yr = ey + (int64_t)gl * g.H;
    for (int v0 = lane; v0 < nvec; v0 += 32 * kDequantUnroll) {
      uint4 c[kDequantUnroll];
      float sc[kDequantUnroll];
#pragma unroll
      for (int j = 0; j < kDequantUnroll; ++j) {
        const int v = v0 + 32 * j;
        if (v < nvec) {
          c[j] = ld_stream16(qr + v * 16);
          sc[j] = __ldg(sr + (v * 16) / 128);
        }
      }
#pragma unroll
      for (int j = 0; j < kDequantUnroll; ++j) {
        const int v = v0 + 32 * j;
        if (v >= nvec) continue;
        uint4 o0, o1;
        o0.x = dequant2((uint16_t)(c[j].x & 0xffffu), sc[j]);
        o0.y = dequant2((uint16_t)(c[j].x >> 16), sc[j]);
        o0.z = dequant2((uint16_t)(c[j].y & 0xffffu), sc[j]);
        o0.w = dequant2((uint16_t)(c[j].y >> 16), sc[j]);
        o1.x = dequant2((uint16_t)(c[j].z & 0xffffu), sc[j]);
        o1.y = dequant2((uint16_t)(c[j].z >> 16), sc[j]);
        o1.z = dequant2((uint16_t)(c[j].w & 0xffffu), sc[j]);
        o1.w = dequant2((uint16_t)(c[j].w >> 16), sc[j]);
        st16(yr + v * 16, o0);
        st16(yr + v * 16 + 8, o1);
      }
    }
  }
  pdl_trigger();
}

// acc (eight fp32 sums) += w * v, v a 16-byte vector of eight bf16: the product and the sum
// rounded separately (RN), as in the definition. Scalar __fmul_rn / __fadd_rn, which are
// never contracted into a fused multiply-add (the packed f32x2 multiply-then-add pair is:
// measured on sm_103a, it gave the fma result).
__device__ __forceinline__ void acc_pair(float (&acc)[8], const uint4& v, float w) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = __fadd_rn(acc[2 * i], __fmul_rn(w, bf16_lo(u[i])));
    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], __fmul_rn(w, bf16_hi(u[i])));
  }
}

// acc += v (no weight).
__device__ __forceinline__ void acc_add(float (&acc)[8], const uint4& v) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = __fadd_rn(acc[2 * i], bf16_lo(u[i]));
    acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], bf16_hi(u[i]));
  }
}

__device__ __forceinline__ void acc_zero(float (&acc)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
}

__device__ __forceinline__ void store_bf16x8(uint16_t* p, const float (&acc)[8]) {
  uint4 o;
  o.x = pack_bf16x2(acc[0], acc[1]);
  o.y = pack_bf16x2(acc[2], acc[3]);
  o.z = pack_bf16x2(acc[4], acc[5]);
  o.w = pack_bf16x2(acc[6], acc[7]);
  st16(p, o);
}

// Combine receive. Block (token u, column tile); a thread owns 8 bf16 columns (16 bytes).
// Lane j of each warp loads pair j's send row and weight and shares them by shuffle; the
// R rows are gathered with up to 8 loads in flight; fp32 products and sums are rounded
// separately with scalar __fmul_rn / __fadd_rn, in slot order; dropped or invalid pairs are
// skipped.
// RANGED: block x covers token x of the range [t0, t0 + nt) of every rank, rank-major (else
// token x; t0, nt unused).
constexpr int kReduceThreads = 128;

// FUSE 1: the combine pack and write in the same pass. The rows are read from the grouped
// expert outputs (src = ey, at gslot) instead of the combine rows, and each is also stored to
// its receive-order row csend[grecv] and its source's combine row crecv[gsend], the rows the
// combine send writes; the sum is the same, value for value. FUSE 2: the same with direct
// push, which has no receive-order rows (csend unused). A compile-time choice: a null check
// in the store loop cost the kernel registers and, next to the concurrent dispatch of the
// next micro-batch, 10% of the step (GB300). The fused kernels read the expert outputs and
// write the two copies for the last time in the pass, so both go through L2 marked evict-first:
// the next micro-batch's dispatch, running beside them, keeps its rows in L2 (measured on
// GB300: micro-batched steps 1.3-5.5% faster for bf16, 9% for fp8 with the expert).
template <bool RANGED, int FUSE>
__global__ void __launch_bounds__(kReduceThreads) k_combine_reduce(Geo g, const int32_t* __restrict__ gsend,
                                                                   const int32_t* __restrict__ gslot,
                                                                   const int32_t* __restrict__ grecv,
                                                                   const float* __restrict__ w,
                                                                   const uint16_t* __restrict__ src,
                                                                   uint16_t* __restrict__ csend,
                                                                   uint16_t* __restrict__ crecv,
                                                                   uint16_t* __restrict__ out, int t0, int nt) {
  const int64_t u = RANGED ? (int64_t)(blockIdx.x / nt) * g.T + t0 + blockIdx.x % nt : (int64_t)blockIdx.x;
  const int col = blockIdx.y * kReduceThreads + threadIdx.x;
  const int ncol = g.H / 8;
  const bool act = col < ncol;
  const int lane = threadIdx.x & 31;
  const int64_t q0 = u * g.R;
  float acc[8];
  acc_zero(acc);
  const uint64_t pol = FUSE ? l2_evict_first_policy() : 0;
  pdl_wait();
  for (int k0 = 0; k0 < g.R; k0 += 32) {
    int myrow = -1, mys = -1, myr = -1;
    float myw = 0.0f;
    if (k0 + lane < g.R) {
      const int gs = __ldg(gsend + q0 + k0 + lane);
      const int gl = __ldg(gslot + q0 + k0 + lane);
      if (gs >= 0 && gl >= 0) {
        myrow = FUSE ? gl : gs;
        myw = __ldg(w + q0 + k0 + lane);
        if (FUSE) {
          mys = gs;
          myr = __ldg(grecv + q0 + k0 + lane);
        }
      }
    }
    const int kn = min(32, g.R - k0);
    for (int j0 = 0; j0 < kn; j0 += 8) {
      int rk[8];
      float wk[8];
      uint4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        rk[j] = __shfl_sync(kFull, myrow, (j0 + j) & 31);
        wk[j] = __shfl_sync(kFull, myw, (j0 + j) & 31);
        if (j0 + j >= kn) rk[j] = -1;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[j] = make_uint4(0, 0, 0, 0);
        if (act && rk[j] >= 0) {
          const uint16_t* p = src + (int64_t)rk[j] * g.H + col * 8;
          v[j] = FUSE ? ld_stream16_hint(p, pol) : ld_stream16(p);
        }
      }
      if (FUSE) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int rs = __shfl_sync(kFull, mys, (j0 + j) & 31);
          const int rr = __shfl_sync(kFull, myr, (j0 + j) & 31);
          if (act && rk[j] >= 0) {
            if (FUSE == 1) st16_hint(csend + (int64_t)rr * g.H + col * 8, v[j], pol);
            st16_hint(crecv + (int64_t)rs * g.H + col * 8, v[j], pol);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (rk[j] >= 0) acc_pair(acc, v[j], wk[j]);
    }
  }
  if (act) store_bf16x8(out + u * g.H + col * 8, acc);
  pdl_trigger();
}

// ---- combine with expert-side partial sums --------------------------------------------
// A token's kept pairs are grouped by destination rank d = grecv / RB; groups are numbered
// in ascending d. Lane k of a warp describes pair k (k < R <= 32).
struct PairGroups {
  int row;      // global grouped row (gslot) of this lane's pair, or -1
  float w;      // its weight
  int j;        // its group number
  int ngroups;  // groups of the token (same in every lane)
};

__device__ __forceinline__ PairGroups token_groups(const Geo& g, const int32_t* gslot, const int32_t* grecv,
                                                   const float* w, int64_t q0, int lane) {
  PairGroups pg;
  int d = 0x7fffffff;
  pg.row = -1;
  pg.w = 0.0f;
  if (lane < g.R) {
    const int gl = __ldg(gslot + q0 + lane);
    if (gl >= 0) {
      pg.row = gl;
      pg.w = w ? __ldg(w + q0 + lane) : 0.0f;
      d = __ldg(grecv + q0 + lane) / (int)g.RB;   // grecv = d*RB + row, all below 2^31
    }
  }
  const bool kept = pg.row >= 0;
  const unsigned peers = __match_any_sync(kFull, d);
  const bool first = kept && (__ffs(peers) - 1 == lane);
  const unsigned firsts = __ballot_sync(kFull, first);
  pg.ngroups = __popc(firsts);
  int j = 0;
  for (unsigned f = firsts; f; f &= f - 1) {
    const int l = __ffs(f) - 1;
    const int dl = __shfl_sync(kFull, d, l);   // every lane runs the same trip count
    j += dl < d;
  }
  pg.j = j;
  return pg;
}

// Expert side: for each token and each group, cpart[s][t][j] = bf16(sum of w*y over the
// group's pairs, k ascending, fp32 with separate rounding). Block (token, 1024 columns).
// kSmall (R <= 8): a token's rows are gathered once into registers and summed group by
// group; a pair's row, weight and group are re-read by shuffle instead of being kept in
// arrays, which keeps the register count (and so the occupancy) close to the plain reduce.
// Otherwise each group's rows are gathered in batches of 8. The token's group count goes
// to tgroups[token] for the source side.
template <bool kSmall>
__global__ void __launch_bounds__(kReduceThreads) k_combine_partial(Geo g, const int32_t* __restrict__ gslot,
                                                                    const int32_t* __restrict__ grecv,
                                                                    const float* __restrict__ w,
                                                                    const uint16_t* __restrict__ ey,
                                                                    uint16_t* __restrict__ cpart,
                                                                    int32_t* __restrict__ tgroups) {
  const int64_t u = blockIdx.x;
  const int col = blockIdx.y * kReduceThreads + threadIdx.x;
  const int ncol = g.H / 8;
  const bool act = col < ncol;
  const int lane = threadIdx.x & 31;
  const int J = g.R < g.N ? g.R : g.N;
  pdl_wait();
  const PairGroups pg = token_groups(g, gslot, grecv, w, u * g.R, lane);
  if (blockIdx.y == 0 && threadIdx.x == 0) tgroups[u] = pg.ngroups;
  uint16_t* out0 = cpart + (u * J) * g.H + col * 8;
  const uint16_t* y0 = ey + col * 8;
  if (kSmall) {
    // Warp 0 lays the kept pairs out in group order (k ascending inside a group) in shared
    // memory; every thread then makes one pass over them, storing at each group's end.
    __shared__ int s_row[8], s_last[8], s_n;
    __shared__ float s_w[8];
    if (threadIdx.x < 32) {
      const int d = pg.row >= 0 ? pg.j : 0x7fffffff;   // group number orders like the rank
      const unsigned peers = __match_any_sync(kFull, d);
      const unsigned firsts = __ballot_sync(kFull, pg.row >= 0 && (__ffs(peers) - 1 == lane));
      int before = 0;   // kept pairs in groups before this lane's group
      for (unsigned f = firsts; f; f &= f - 1) {
        const int l = __ffs(f) - 1;
        const int jl = __shfl_sync(kFull, pg.j, l);
        const unsigned pl = __shfl_sync(kFull, peers, l);
        before += (jl < pg.j) ? __popc(pl) : 0;
      }
      if (pg.row >= 0) {
        const int p = before + __popc(peers & ((1u << lane) - 1u));
        s_row[p] = pg.row;
        s_w[p] = pg.w;
        s_last[p] = (32 - __clz(peers)) - 1 == lane;   // highest lane of the group
      }
      const unsigned kept = __ballot_sync(kFull, pg.row >= 0);
      if (lane == 0) s_n = __popc(kept);
    }
    __syncthreads();
    const int n = s_n;
    uint4 v[8];
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      v[p] = make_uint4(0, 0, 0, 0);
      if (act && p < n) v[p] = ld_stream16(y0 + (int64_t)s_row[p] * g.H);
    }
    float acc[8];
    acc_zero(acc);
    int j = 0;
#pragma unroll
    for (int p = 0; p < 8; ++p) {
      if (p >= n) break;
      acc_pair(acc, v[p], s_w[p]);
      if (s_last[p]) {
        if (act) store_bf16x8(out0 + (int64_t)j * g.H, acc);
        ++j;
        acc_zero(acc);
      }
    }
  } else {
    for (int j = 0; j < pg.ngroups; ++j) {
      float acc[8];
      acc_zero(acc);
      for (int k0 = 0; k0 < g.R; k0 += 8) {
        uint4 v[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int k = (k0 + m) & 31;
          const int row = __shfl_sync(kFull, pg.row, k);
          const int jm = __shfl_sync(kFull, pg.j, k);
          v[m] = make_uint4(0, 0, 0, 0);
          if (act && k0 + m < g.R && row >= 0 && jm == j) v[m] = ld_stream16(y0 + (int64_t)row * g.H);
        }
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const int k = (k0 + m) & 31;
          const int row = __shfl_sync(kFull, pg.row, k);
          const int jm = __shfl_sync(kFull, pg.j, k);
          const float wm = __shfl_sync(kFull, pg.w, k);
          if (k0 + m < g.R && row >= 0 && jm == j) acc_pair(acc, v[m], wm);
        }
      }
      if (act) store_bf16x8(out0 + (int64_t)j * g.H, acc);
    }
  }
  pdl_trigger();
}

// Source side: out[s][t] = bf16(sum over the token's groups j ascending of cpart[s][t][j]).
// Block (token, kSumVec * kReduceThreads * 8 columns): each thread sums kSumVec 16-byte
// column vectors, two groups' loads in flight at a time.
constexpr int kSumVec = 4;

__global__ void __launch_bounds__(kReduceThreads) k_combine_sum(Geo g, const int32_t* __restrict__ tgroups,
                                                                const uint16_t* __restrict__ cpart,
                                                                uint16_t* __restrict__ out) {
  const int64_t u = blockIdx.x;
  const int ncol = g.H / 8;
  const int J = g.R < g.N ? g.R : g.N;
  pdl_wait();
  const int ng = __ldg(tgroups + u);
  const uint16_t* in0 = cpart + (u * J) * g.H;
  int cols[kSumVec];
  float acc[kSumVec][8];
#pragma unroll
  for (int c = 0; c < kSumVec; ++c) {
    cols[c] = blockIdx.y * kSumVec * kReduceThreads + c * kReduceThreads + threadIdx.x;
    acc_zero(acc[c]);
  }
  for (int j0 = 0; j0 < ng; j0 += 2) {
    uint4 v[2][kSumVec];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int c = 0; c < kSumVec; ++c) {
        v[m][c] = make_uint4(0, 0, 0, 0);
        if (j0 + m < ng && cols[c] < ncol) v[m][c] = ld_stream16(in0 + (int64_t)(j0 + m) * g.H + cols[c] * 8);
      }
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      if (j0 + m >= ng) continue;
#pragma unroll
      for (int c = 0; c < kSumVec; ++c) acc_add(acc[c], v[m][c]);
    }
  }
#pragma unroll
  for (int c = 0; c < kSumVec; ++c)
    if (cols[c] < ncol) store_bf16x8(out + u * g.H + cols[c] * 8, acc[c]);
  pdl_trigger();
}

}  // namespace

cudaError_t launch_combine_partial(const Geo& g, const moe_layout_t* lay, const uint16_t* ey, const float* w,
                                   uint16_t* cpart, Ctx& c) {
  const int64_t tokens = (int64_t)g.N * g.T;
  if (tokens == 0) return cudaSuccess;
  const int ncol = g.H / 8;
  dim3 grid((unsigned)tokens, (unsigned)((ncol + kReduceThreads - 1) / kReduceThreads));
  LaunchScope ls(c, MOE_K_COMBINE_PARTIAL);
  int32_t* tg = lay->scratch + layout_scratch_tgroups_offset(g);
  if (g.R <= 8)
    return launch_kernel(k_combine_partial<true>, grid, dim3(kReduceThreads), 0, c, g, (const int32_t*)lay->gslot,
                         (const int32_t*)lay->grecv, w, ey, cpart, tg);
  return launch_kernel(k_combine_partial<false>, grid, dim3(kReduceThreads), 0, c, g, (const int32_t*)lay->gslot,
                       (const int32_t*)lay->grecv, w, ey, cpart, tg);
}

cudaError_t launch_combine_sum(const Geo& g, const moe_layout_t* lay, const uint16_t* cpart, uint16_t* out,
                               Ctx& c) {
  const int64_t tokens = (int64_t)g.N * g.T;
  if (tokens == 0) return cudaSuccess;
  const int ncol = g.H / 8;
  dim3 grid((unsigned)tokens, (unsigned)((ncol + kSumVec * kReduceThreads - 1) / (kSumVec * kReduceThreads)));
  LaunchScope ls(c, MOE_K_COMBINE_SUM);
  return launch_kernel(k_combine_sum, grid, dim3(kReduceThreads), 0, c, g,
                       (const int32_t*)(lay->scratch + layout_scratch_tgroups_offset(g)), cpart, out);
}

cudaError_t launch_quant_fp8(const Geo& g0, const uint16_t* x, uint8_t* xq, Ctx& c) {
  Geo g = g0;
  if (windowed(g0, c)) g.N = c.win_hi - c.win_lo;   // the window's token rows (window-local buffers)
  const int64_t upr = (g.H / 128 + 2 * kQuantUnroll - 1) / (2 * kQuantUnroll);
  const int64_t units = (int64_t)g.N * g.T * upr;   // one warp unit: 2 x kQuantUnroll blocks of a row
  if (units == 0) return cudaSuccess;
  int64_t blocks = (units + 7) / 8;                 // 8 warps per CTA
  const int64_t maxb = (int64_t)c.num_sms * 8;
  if (blocks > maxb) blocks = maxb;
  LaunchScope ls(c, MOE_K_QUANT_FP8);
  if (g.B % 16 == 0)   // 16-byte code stores (same unit count: 8 blocks of a row per warp)
    return launch_kernel(k_quant_fp8_16, dim3((unsigned)blocks), dim3(256), 0, c, g, x, xq);
  return launch_kernel(k_quant_fp8, dim3((unsigned)blocks), dim3(256), 0, c, g, x, xq);
}

template <int ALL>
cudaError_t run_quant_pack(const Geo& g, const uint16_t* x, const int32_t* fan, uint8_t* dst, Ctx& c, int t0, int nt,
                           const FanAll& fa, int64_t blocks) {
  const bool ranged = nt != g.T;
  if (g.B % 16 == 0) {   // 16-byte code stores (same unit count: 8 blocks of a row per warp)
    auto k16 = ranged ? k_quant_pack16<true, ALL> : k_quant_pack16<false, ALL>;
    return launch_kernel(k16, dim3((unsigned)blocks), dim3(256), 0, c, g, x, fan, dst, t0, nt, fa);
  }
  auto k = g.B % 8 == 0 ? (ranged ? k_quant_pack<true, true, ALL> : k_quant_pack<true, false, ALL>)
                        : (ranged ? k_quant_pack<false, true, ALL> : k_quant_pack<false, false, ALL>);
  return launch_kernel(k, dim3((unsigned)blocks), dim3(256), 0, c, g, x, fan, dst, t0, nt, fa);
}

cudaError_t launch_quant_pack(const Geo& g0, const int32_t* fan, const uint16_t* x, uint8_t* dst, Ctx& c, int t0,
                              int nt) {
  if (nt < 0) nt = g0.T;
  Geo g = g0;
  if (windowed(g0, c)) {   // the window's tokens into its window-local send rows
    if (nt != g0.T || (c.flags & MOE_FLAG_DIRECT_PUSH)) return cudaErrorInvalidValue;
    const int64_t q0 = (int64_t)c.win_lo * g0.TR;
    g.N = c.win_hi - c.win_lo;
    g.P = (int64_t)g.N * g0.TR;
    fan += q0;
    dst = rebase(dst, q0 * g0.B);
  }
  const int64_t upr = (g.H / 128 + 2 * kQuantUnroll - 1) / (2 * kQuantUnroll);
  const int64_t units = (int64_t)g.N * nt * upr;
  if (units == 0) return cudaSuccess;
  int64_t blocks = (units + 7) / 8;
  const int64_t maxb = (int64_t)c.num_sms * 8;
  if (blocks > maxb) blocks = maxb;
  LaunchScope ls(c, MOE_K_QUANT_PACK);
  return run_quant_pack<0>(g, x, fan, dst, c, t0, nt, FanAll{}, blocks);
}

cudaError_t launch_quant_dispatch_fused(const Geo& g, const moe_layout_t* lay, const uint16_t* x, uint8_t* send,
                                        uint8_t* recv, uint8_t* ex, float* exs, Ctx& c, int t0, int nt) {
  if (nt < 0) nt = g.T;
  if (windowed(g, c)) return cudaErrorInvalidValue;
  const int64_t upr = (g.H / 128 + 2 * kQuantUnroll - 1) / (2 * kQuantUnroll);
  const int64_t units = (int64_t)g.N * nt * upr;
  if (units == 0) return cudaSuccess;
  int64_t blocks = (units + 7) / 8;
  const int64_t maxb = (int64_t)c.num_sms * 8;
  if (blocks > maxb) blocks = maxb;
  LaunchScope ls(c, MOE_K_QUANT_DISPATCH_FUSED);
  const FanAll fa{lay->grecv, lay->gslot, recv, ex, exs};
  return send ? run_quant_pack<1>(g, x, lay->gsend, send, c, t0, nt, fa, blocks)
              : run_quant_pack<2>(g, x, lay->gsend, send, c, t0, nt, fa, blocks);
}

cudaError_t launch_dequant_fp8(const Geo& g, const moe_layout_t* lay, const uint8_t* exq, const float* exs,
                               uint16_t* ey, Ctx& c, int t0, int nt) {
  if (nt < 0) nt = g.T;
  const int64_t np = (int64_t)g.N * nt * g.R;
  if (np == 0) return cudaSuccess;
  int64_t blocks = (np + 7) / 8;
  const int64_t maxb = (int64_t)c.num_sms * 8;
  if (blocks > maxb) blocks = maxb;
  LaunchScope ls(c, MOE_K_EXPERT);
  const bool rev = (c.flags & MOE_FLAG_DIRECT_PUSH) != 0, ranged = nt != g.T;
  auto k = rev ? (ranged ? k_dequant_fp8<true, true> : k_dequant_fp8<true, false>)
               : (ranged ? k_dequant_fp8<false, true> : k_dequant_fp8<false, false>);
  int64_t win_rows = 0;
  int win_lo = 0, win_n = 0;
  if (windowed(g, c)) {   // the window's grouped rows, in window-local buffers
    if (ranged) return cudaErrorInvalidValue;
    win_rows = (int64_t)g.L * g.cap;
    win_lo = c.win_lo;
    win_n = c.win_hi - c.win_lo;
    exq = rebase(exq, win_lo * win_rows * g.H);
    exs = rebase(exs, win_lo * win_rows * (int64_t)(g.H / 128) * 4);
    ey = rebase(ey, win_lo * win_rows * 2 * (int64_t)g.H);
  }
  return launch_kernel(k, dim3((unsigned)blocks), dim3(256), 0, c, g, (const int32_t*)lay->gslot, exq, exs, ey, t0,
                       nt, np, win_rows, win_lo, win_n);
}

cudaError_t launch_combine_reduce(const Geo& g0, const moe_layout_t* lay, const uint16_t* crecv, const float* w,
                                  uint16_t* out, Ctx& c, int t0, int nt) {
  if (nt < 0) nt = g0.T;
  Geo g = g0;
  const int32_t* gsend = lay->gsend;
  const int32_t* gslot = lay->gslot;
  if (windowed(g0, c)) {   // the window's tokens: window-local weights, combine rows and output
    if (nt != g0.T) return cudaErrorInvalidValue;
    const int64_t q0 = (int64_t)c.win_lo * g0.TR;
    g.N = c.win_hi - c.win_lo;
    g.P = (int64_t)g.N * g0.TR;
    gsend += q0;
    gslot += q0;
    crecv = rebase(crecv, q0 * 2 * (int64_t)g0.H);
  }
  const int64_t tokens = (int64_t)g.N * nt;
  if (tokens == 0) return cudaSuccess;
  const int ncol = g.H / 8;
  dim3 grid((unsigned)tokens, (unsigned)((ncol + kReduceThreads - 1) / kReduceThreads));
  LaunchScope ls(c, MOE_K_COMBINE_REDUCE);
  return launch_kernel(nt != g.T ? k_combine_reduce<true, 0> : k_combine_reduce<false, 0>, grid,
                       dim3(kReduceThreads), 0, c, g, gsend, gslot, (const int32_t*)nullptr, w, crecv,
                       (uint16_t*)nullptr, (uint16_t*)nullptr, out, t0, nt);
}

cudaError_t launch_combine_fused(const Geo& g, const moe_layout_t* lay, const uint16_t* ey, uint16_t* csend,
                                 uint16_t* crecv, const float* w, uint16_t* out, Ctx& c, int t0, int nt) {
  if (nt < 0) nt = g.T;
  if (windowed(g, c)) return cudaErrorInvalidValue;
  const int64_t tokens = (int64_t)g.N * nt;
  if (tokens == 0) return cudaSuccess;
  const int ncol = g.H / 8;
  dim3 grid((unsigned)tokens, (unsigned)((ncol + kReduceThreads - 1) / kReduceThreads));
  LaunchScope ls(c, MOE_K_COMBINE_FUSED);
  auto k = csend ? (nt != g.T ? k_combine_reduce<true, 1> : k_combine_reduce<false, 1>)
                 : (nt != g.T ? k_combine_reduce<true, 2> : k_combine_reduce<false, 2>);
  return launch_kernel(k, grid, dim3(kReduceThreads), 0, c, g, (const int32_t*)lay->gsend, (const int32_t*)lay->gslot,
                       (const int32_t*)lay->grecv, w, ey, csend, crecv, out, t0, nt);
}

}  // namespace moe
