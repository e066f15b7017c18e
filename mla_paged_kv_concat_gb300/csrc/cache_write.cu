// Cache write: scatter new tokens' [kv_c | k_pe] rows into the paged latent
// cache through slot_mapping, optionally quantising to OCP E4M3.
//
// Restates "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
// csrc/cache_kernels.cu, concat_and_cache_mla_kernel.  That kernel runs one
// CTA per token with a strided scalar loop; here one warp moves one token at
// a time with 16-byte vector loads and stores (a 576-element bf16 row is 72
// such chunks), in a warp-stride loop over the tokens, and the E4M3 encoding
// avoids the division except next to a rounding boundary (see quant2).
//
// The fused variant also does the two steps the model runs just before that
// kernel ("frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
// vllm/model_executor/models/deepseek_v2.py and the MLA common forward):
// kv_a_layernorm (RMSNorm of kv_c, weight gamma) and rotary_emb (non-NeoX
// rotation of k_pe, and optionally of q_pe in place, by the token's
// position, with a caller-given fp32 cos | sin table).  The normalised and
// rotated rows are rounded to bf16 and then stored exactly as the plain
// write stores its inputs.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace mla {

namespace {

struct CacheWriteArgs {
  const uint16_t* kv_c;
  int64_t kv_c_stride;
  const uint16_t* k_pe;
  int64_t k_pe_stride;
  const int64_t* slot_mapping;
  int num_tokens;
  int R, P;
  void* cache;
  int64_t num_slots;  // num_blocks * block_size
  int block_size;
  int64_t block_stride;
  const float* scale;
  int* err_count;
  // fused RMSNorm + rotary (NR variant only)
  const uint16_t* gamma;  // bf16 [R]
  float eps;
  const int64_t* positions;  // [num_tokens]
  const float* table;        // fp32 [max_position][P]: cos | sin
  int64_t max_position;
  uint16_t* q_pe;            // bf16 [num_tokens][q_heads][P] at the strides below, or null
  int64_t q_pe_row_stride, q_pe_head_stride;
  int q_heads;
};

constexpr int kWarpsPerCta = 8;
// Rows per warp per pass.  Four (loaded together, then stored) made the
// whole-cache fp8 write slower (180 against 148 us for 248K tokens) at the
// occupancy their registers allow.
constexpr int kTokensPerWarp = 1;

// Cache element formats (template argument FMT of the kernel).
constexpr int kBf16 = 0, kE4M3 = 1, kE5M2 = 2;

// Two fp32 -> two fp8 codes of format FMT (round to nearest even,
// satfinite), low code first.
template <int FMT>
__device__ __forceinline__ uint32_t fp8x2(float lo, float hi) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(
      make_float2(lo, hi), __NV_SATFINITE, FMT == kE5M2 ? __NV_E5M2 : __NV_E4M3));
}

// fp8 codes of RN_f32(x0 / s), RN_f32(x1 / s) (IEEE division, then RNE to
// E4M3 or E5M2 with saturation), without a division in the common case.  With
// r = RN(1/s) (an IEEE division, once per thread), q = RN(x * r) is within
// 1.5 * 2^-23 |q| of RN_f32(x / s) (three roundings of relative size at most
// 2^-24).  fp8 rounding is monotone in the value, so when q - 2^-22 |q| and
// q + 2^-22 |q| get the same code, so does RN_f32(x / s); otherwise the
// quotient is within a few ulp of a boundary between two codes and the
// division is done.  Quotients too small for the relative bound (|q| below
// 2^-104) are all +-0 in both formats, with the sign that both sides agree
// on; |q| is clamped to 2^100 (every such value saturates to the largest
// finite code either way); NaN quotients take the division.  The bound needs
// r to be a normal number: for a scale below 2^-126 (r infinite) or at or
// above 2^126 (r subnormal, with a larger relative error) the caller passes
// r = 0 and every element takes the division.
template <int FMT>
__device__ __forceinline__ uint32_t quant2(float x0, float x1, float s, float r) {
  if (r == 0.f) return fp8x2<FMT>(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
  float q0 = x0 * r, q1 = x1 * r;
  if (q0 != q0 || q1 != q1) return fp8x2<FMT>(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
  q0 = fminf(fmaxf(q0, -0x1p100f), 0x1p100f);
  q1 = fminf(fmaxf(q1, -0x1p100f), 0x1p100f);
  const float d0 = fabsf(q0) * 0x1p-22f, d1 = fabsf(q1) * 0x1p-22f;
  const uint32_t lo = fp8x2<FMT>(q0 - d0, q1 - d1);
  const uint32_t hi = fp8x2<FMT>(q0 + d0, q1 + d1);
  if (lo == hi) return lo;
  return fp8x2<FMT>(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
}

// 8 bf16 values -> 8 fp8 bytes of x / scale (IEEE division, RNE, satfinite).
template <int FMT>
__device__ __forceinline__ uint2 quant8(uint4 v, float s, float r) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
  uint32_t w[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float2 a = __bfloat1622float2(h[2 * k]);
    const float2 b = __bfloat1622float2(h[2 * k + 1]);
    w[k] = quant2<FMT>(a.x, a.y, s, r) | (quant2<FMT>(b.x, b.y, s, r) << 16);
  }
  return make_uint2(w[0], w[1]);
}

template <int FMT>
__device__ __forceinline__ uint8_t quant1(uint16_t bits, float s) {
  float x = __bfloat162float(__ushort_as_bfloat16(bits));
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(x, s), __NV_SATFINITE,
                                                    FMT == kE5M2 ? __NV_E5M2 : __NV_E4M3));
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// Exact rounding of the fused write's results.
//
// The reference result of the RMSNorm and of the rotation is their fp64
// evaluation rounded once to bf16 (nearest, ties to even).  The kernel gets
// the same bits without evaluating fp64 on every element (fp64 is slow on
// this GPU).  bf16 rounding is monotone and changes only at the midpoints
// between consecutive bf16 values; whenever a computed value and a bound on
// its distance from the exact result show that no midpoint lies between
// them, the exact result, its fp64 evaluation (within 2^-44 relative of it
// for the RMSNorm, 2^-53 for the rotation) and the computed value round to
// the same bf16 value.  Three tiers:
//   1. fp32, as a plain evaluation would do it, with a bound of a few units
//      in the last place (ulp): decided unless the value lies within that
//      many ulps of a midpoint (about one element in 4000);
//   2. for those, double-float (an unevaluated sum h + lo of two fp32
//      values) with a bound near 2^-40 relative: decided unless the exact
//      result is practically on the midpoint (exact ties);
//   3. the rest in fp64, in the reference's operation order, every
//      operation correctly rounded, then rounded to bf16.
// Inputs outside the range where the bounds hold (NaN, infinities, results
// below 2^-100 or above 2^126, rows whose magnitudes span more than 2^100)
// go to the later tiers as well.  Tiers 2 and 3 are separate, non-inlined
// functions behind branches that are rarely taken, so that their
// instructions are not issued on the common path.

// s + e = a + b exactly (Knuth's two-sum; no ordering of |a|, |b| needed).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  const float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// fp64 -> bf16 bits, round to nearest, ties to even; any NaN -> 0x7FC0;
// results of 2^128 and above are infinities.
__device__ __forceinline__ uint32_t bf16_from_f64(double y) {
  const uint64_t u = static_cast<uint64_t>(__double_as_longlong(y));
  const uint32_t sign = static_cast<uint32_t>(u >> 48) & 0x8000u;
  const uint64_t a = u & 0x7FFFFFFFFFFFFFFFull;
  if (a > 0x7FF0000000000000ull) return 0x7FC0u;
  if (a >= 0x47F0000000000000ull) return sign | 0x7F80u;  // |y| >= 2^128
  if (a >= 0x3810000000000000ull) {                       // |y| >= 2^-126
    // keep 7 of the 52 fraction bits; the carry of the rounding increment
    // runs into the exponent field
    const uint64_t r = (a + 0x00000FFFFFFFFFFFull + ((a >> 45) & 1u)) >> 45;
    const uint64_t bits = r - (static_cast<uint64_t>(1023 - 127) << 7);
    return bits >= 0x7F80u ? (sign | 0x7F80u) : (sign | static_cast<uint32_t>(bits));
  }
  // below 2^-126: multiples of 2^-133 (|y| * 2^133 is exact and below 2^7;
  // rint rounds to nearest even; 128 is the smallest normal, 0x0080)
  const double n = rint(fabs(y) * 0x1p133);
  return sign | static_cast<uint32_t>(n);
}

// Tier 1 test on two values y0, y1, each known to lie within d0 (d1) of its
// exact result: both ends of each bracket [y - d, y + d] round to the same
// bf16 value (round to nearest even; rounding is monotone, so the exact
// result rounds there too), and that value is finite (an infinity or NaN
// here comes from an fp32 overflow or a non-finite input, which the fp64
// evaluation may treat differently).  On success *r holds the two bf16 values
// (y0 low).  Three conversions' worth of work per pair instead of a
// per-element distance test.
__device__ __forceinline__ bool bracket2(float y0, float d0, float y1, float d1, uint32_t& r) {
  const uint32_t lo = pack_bf16x2(y0 - d0, y1 - d1);
  const uint32_t hi = pack_bf16x2(y0 + d0, y1 + d1);
  r = lo;
  // a half whose exponent bits are all ones gets bit 15 set by the add
  const uint32_t nonfinite = ((lo & 0x7F807F80u) + 0x00800080u) & 0x80008000u;
  return lo == hi && nonfinite == 0u;
}

// Tier 2 rounding: y to bf16 from y ~= h + lo, |y - (h + lo)| <= B, when no
// bf16 midpoint lies within B of h + lo; false otherwise (and for h outside
// [2^-100, 2^126] in magnitude, where the callers' bounds stop).
__device__ __forceinline__ bool round_bf16_df(float h, float lo, float B, uint32_t& out) {
  const float ah = fabsf(h);
  if (!(ah >= 0x1p-100f && ah <= 0x1p126f)) return false;
  const uint32_t u = __float_as_uint(h);
  const uint32_t t = u & 0x7FFF0000u;  // |h| truncated to bf16
  // distance from the midpoint above t (same binade as |h|, so ah - mid is
  // exact), corrected by lo in the direction of |h|
  const float d = (ah - __uint_as_float(t | 0x8000u)) + ((u >> 31) ? -lo : lo);
  if (!(fabsf(d) > B)) return false;
  out = ((u >> 16) & 0x8000u) | ((t >> 16) + (d > 0.f ? 1u : 0u));
  return true;
}

__device__ __forceinline__ float bfv(uint32_t w, int hi) {
  return hi ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
}

// Per-token terms of the RMSNorm: x / sqrt(mean x^2 + eps) * gamma is
// computed as (x sc) gamma inv with sc = 2^-k (k the binade of the row's
// largest element, so that the scaled squares and their sum stay in range)
// and inv = 1 / sqrt(mean (x sc)^2 + eps sc^2) ~= inv32 + inv_lo.  Error
// budget: the scaled sum of squares is accumulated with two-sum (exact high
// part, low parts in fp32), within 2^-39 of the exact sum (the reference's
// sequential fp64 sum is within (R - 1) 2^-53 < 2^-44 of it); one Newton
// step on rsqrtf (error below 2^-21) leaves inv32 + inv_lo within 2^-39.5 of
// inv, and inv32, its rounding to fp32, within 2^-24 + 2^-39.5.  Since the
// largest scaled element is at least 1, the mean is at least 2^-9 and
// inv <= 2^4.5, so sc inv32 <= 2^24.5 for the tokens that take tier 1
// (k >= -20).
struct NormTerms {
  float sc, inv32, inv_lo;
  bool fast;  // false: every element takes the fp64 path
};

// Tier 1 of the RMSNorm for 8 elements: p = RN(xg inv_s), xg = x gamma
// (exact: two 8-bit significands; within 2^-150 if it underflows) and
// inv_s = sc inv32 (a power-of-two scaling of inv32, exact), is within
// 2^-23 |y| (1 + 2^-15) + 2^-125 of y (the absolute part covers a subnormal
// xg, inv_s being at most 2^24.5 on the tokens that take this tier); the
// bracket is 2^-20 |p| + 2^-120.  Bit 2i (pair i, both halves) of *need is
// set for each pair left to tier 2.
__device__ __forceinline__ uint4 norm8(uint4 x, uint4 g, float inv_s, uint32_t& need) {
  const uint32_t xv[4] = {x.x, x.y, x.z, x.w}, gv[4] = {g.x, g.y, g.z, g.w};
  uint32_t o[4];
  need = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float p0 = (bfv(xv[k], 0) * bfv(gv[k], 0)) * inv_s;
    const float p1 = (bfv(xv[k], 1) * bfv(gv[k], 1)) * inv_s;
    const float d0 = fmaf(fabsf(p0), 0x1p-20f, 0x1p-120f);
    const float d1 = fmaf(fabsf(p1), 0x1p-20f, 0x1p-120f);
    if (!bracket2(p0, d0, p1, d1, o[k])) need |= 3u << (2 * k);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Tier 2 of the RMSNorm for the elements flagged in `need`: p + lo with
// p = RN(xg inv32), its exact error (fma) and xg inv_lo, within 2^-38 |y| of
// y; the bound used is 2^-36 |p|.  Elements it cannot decide are flagged in
// *fb for tier 3.
__device__ __noinline__ uint4 norm8_df(uint4 x, uint4 g, float sc, float inv32, float inv_lo,
                                       uint4 cur, uint32_t need, uint32_t* fb) {
  const uint32_t xv[4] = {x.x, x.y, x.z, x.w}, gv[4] = {g.x, g.y, g.z, g.w};
  uint32_t o[4] = {cur.x, cur.y, cur.z, cur.w};
  uint32_t f = 0;
  for (int i = 0; i < 8; ++i) {
    if (!(need & (1u << i))) continue;
    const int k = i >> 1, j = i & 1;
    const float xs = bfv(xv[k], j) * sc;
    const float xg = xs * bfv(gv[k], j);
    const float p = xg * inv32;
    const float lo = fmaf(xg, inv_lo, fmaf(xg, inv32, -p));
    uint32_t r = 0;
    if (fabsf(xs) >= 0x1p-126f && round_bf16_df(p, lo, fabsf(p) * 0x1p-36f, r))
      o[k] = j ? ((o[k] & 0xFFFFu) | (r << 16)) : ((o[k] & 0xFFFF0000u) | r);
    else
      f |= 1u << i;
  }
  *fb = f;
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Tier 3 of the RMSNorm for the elements flagged in fb: (x * inv) * gamma in
// fp64, inv the reference's fp64 1 / sqrt(ss / R + eps).
__device__ __noinline__ uint4 norm8_f64(uint4 x, uint4 g, double inv, uint4 cur,
                                        uint32_t fb) {
  const uint32_t xv[4] = {x.x, x.y, x.z, x.w}, gv[4] = {g.x, g.y, g.z, g.w};
  uint32_t o[4] = {cur.x, cur.y, cur.z, cur.w};
  for (int i = 0; i < 8; ++i) {
    if (!(fb & (1u << i))) continue;
    const int k = i >> 1, j = i & 1;
    const double y = __dmul_rn(__dmul_rn(static_cast<double>(bfv(xv[k], j)), inv),
                               static_cast<double>(bfv(gv[k], j)));
    const uint32_t r = bf16_from_f64(y);
    o[k] = j ? ((o[k] & 0xFFFFu) | (r << 16)) : ((o[k] & 0xFFFF0000u) | r);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The reference's fp64 1 / sqrt(ss / R + eps), ss summed in element order
// from the row in memory (one thread).
__device__ __noinline__ double rms_inv_f64(const uint16_t* row, int R, float eps) {
  const uint4* src = reinterpret_cast<const uint4*>(row);
  double ss = 0.0;
  for (int c = 0; c < R / 8; ++c) {
    const uint4 w4 = __ldg(src + c);
    const uint32_t wv[4] = {w4.x, w4.y, w4.z, w4.w};
    for (int e = 0; e < 8; ++e) {
      const double xd = bfv(wv[e >> 1], e & 1);
      ss = __dadd_rn(ss, __dmul_rn(xd, xd));
    }
  }
  const double ms = __ddiv_rn(ss, static_cast<double>(R));
  return __ddiv_rn(1.0, __dsqrt_rn(__dadd_rn(ms, static_cast<double>(eps))));
}

// Tier 2 of one rotated value.  Double-float: both products split exactly
// into value + error (fma), their sum by two-sum, the errors added in fp32,
// the pair renormalised by a second two-sum (under cancellation the error
// terms can be as large as the result): within 2^-45 (|u c| + |v s|) of the
// exact result; the bound used is 2^-40 (|u c| + |v s|).  Products outside
// [2^-100, 2^126] (unless exactly zero from a zero factor) are left to
// tier 3, as are results next to a midpoint.
__device__ __forceinline__ bool rot1_df(float u, float c, float v, float s, float sgn,
                                        uint32_t& r) {
  const float p1 = u * c, p2 = sgn * (v * s);
  const float a1 = fabsf(p1), a2 = fabsf(p2);
  const bool in1 = (a1 >= 0x1p-100f && a1 <= 0x1p126f) || (p1 == 0.f && (u == 0.f || c == 0.f));
  const bool in2 = (a2 >= 0x1p-100f && a2 <= 0x1p126f) || (p2 == 0.f && (v == 0.f || s == 0.f));
  if (!(in1 && in2)) return false;
  const float e1 = fmaf(u, c, -p1);
  const float e2 = fmaf(sgn * v, s, -p2);
  float h, t, lo;
  two_sum(p1, p2, h, t);
  two_sum(h, t + (e1 + e2), h, lo);
  if (h == 0.f && lo == 0.f) {
    // exact zero (p1 = -p2 and no product error): the fp64 sum is +0
    // unless both terms are -0
    r = (__float_as_uint(p1) & __float_as_uint(p2)) == 0x80000000u ? 0x8000u : 0u;
    return true;
  }
  return round_bf16_df(h, lo, (a1 + a2) * 0x1p-40f, r);
}

// Non-NeoX rotation of 4 interleaved pairs (8 bf16) by angles with the given
// cos and sin: (a, b) -> (a c - b s, b c + a s), tier 1: y = fma(a, c, p2)
// with p2 = RN(-b s) (or fma(b, c, RN(a s))) is within 2^-24 (|p2| + |y|)
// + 2^-149 of the exact result (the product inside the fma is exact); the
// bracket is 2^-22 (|p2| + |y|) + 2^-120.  Bit i of *need is set for each
// element i left to tier 2 (both elements of a pair together).
__device__ __forceinline__ uint4 rope8(uint4 x, float4 c, float4 s, uint32_t& need) {
  const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
  const float cv[4] = {c.x, c.y, c.z, c.w}, sv[4] = {s.x, s.y, s.z, s.w};
  uint32_t o[4];
  need = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float a = bfv(xv[k], 0), b = bfv(xv[k], 1);
    const float q0 = -(b * sv[k]), q1 = a * sv[k];
    const float y0 = fmaf(a, cv[k], q0), y1 = fmaf(b, cv[k], q1);
    const float d0 = fmaf(fabsf(q0) + fabsf(y0), 0x1p-22f, 0x1p-120f);
    const float d1 = fmaf(fabsf(q1) + fabsf(y1), 0x1p-22f, 0x1p-120f);
    if (!bracket2(y0, d0, y1, d1, o[k])) need |= 3u << (2 * k);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Tiers 2 and 3 of the rotation for the elements flagged in `need`: the
// double-float value, and where it cannot decide, fp64 (products exact in
// fp64, one rounding for the sum, then one to bf16).
__device__ __noinline__ uint4 rope8_slow(uint4 x, float4 c, float4 s, uint4 cur,
                                         uint32_t need) {
  const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
  const float cv[4] = {c.x, c.y, c.z, c.w}, sv[4] = {s.x, s.y, s.z, s.w};
  uint32_t o[4] = {cur.x, cur.y, cur.z, cur.w};
  for (int i = 0; i < 8; ++i) {
    if (!(need & (1u << i))) continue;
    const int k = i >> 1, j = i & 1;
    // j = 0: a c - b s; j = 1: b c + a s
    const float u = bfv(xv[k], j), v = bfv(xv[k], j ^ 1);
    const float sgn = j ? 1.f : -1.f;
    uint32_t r;
    if (!rot1_df(u, cv[k], v, sv[k], sgn, r)) {
      const double pu = __dmul_rn(static_cast<double>(u), static_cast<double>(cv[k]));
      const double pv = __dmul_rn(static_cast<double>(v), static_cast<double>(sv[k]));
      r = bf16_from_f64(j ? __dadd_rn(pu, pv) : __dsub_rn(pu, pv));
    }
    o[k] = j ? ((o[k] & 0xFFFFu) | (r << 16)) : ((o[k] & 0xFFFF0000u) | r);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// VEC: every source row and destination row starts on a 16-byte boundary, so
// rows move as 16-byte chunks (8 elements); otherwise element by element.
// NR: the fused RMSNorm + rotary variant (VEC layout, P = 64 only).
template <int FMT, bool VEC, bool NR = false>
__global__ void __launch_bounds__(kWarpsPerCta * 32, NR ? 3 : 1)
    cache_write_kernel(const CacheWriteArgs a) {
  constexpr bool FP8 = FMT != kBf16;
  // The decode kernels that follow wait for this grid's completion before
  // they read anything; letting them launch now hides their launch latency.
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int D = a.R + a.P;
  const float s = FP8 ? __ldg(a.scale) : 1.0f;
  // RN(1/s), as quant2's bound assumes; 0 (always divide) unless it is a
  // normal number
  const float r_div = FP8 ? __fdiv_rn(1.0f, s) : 1.0f;
  const float r = fabsf(r_div) >= 0x1p-126f && fabsf(r_div) <= 0x1p126f ? r_div : 0.f;
  // Warp-stride loop over groups of kTokensPerWarp consecutive tokens (the
  // grid is sized to the GPU, not to the token count).  All loads of a group
  // (rows and slots) are issued before any of them is used, so that each
  // warp keeps several rows in flight: the write is bound by HBM, not by
  // load latency.
  const int nwarps = gridDim.x * kWarpsPerCta;
  const int warp_id = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  // fused variant: this lane's RMSNorm weights (latent chunks lane and
  // lane + 32), the same for every token
  uint4 gm[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
  if constexpr (NR) {
#pragma unroll
    for (int k = 0; k < 2; ++k)
      if (lane + 32 * k < a.R / 8)
        gm[k] = __ldg(reinterpret_cast<const uint4*>(a.gamma) + lane + 32 * k);
  }
  for (int t0 = warp_id * kTokensPerWarp; t0 < a.num_tokens; t0 += nwarps * kTokensPerWarp) {
    if constexpr (VEC) {
      // lane l holds 16-byte chunks l, l + 32, l + 64 of each D-element row
      // (D <= 576: at most 3)
      const int nc = a.R / 8, np = a.P / 8;
      // the position goes first: the table loads depend on it
      const int64_t pos = NR ? __ldg(a.positions + t0) : 0;
      uint4 v[kTokensPerWarp][3];
      int64_t slot[kTokensPerWarp];
#pragma unroll
      for (int j = 0; j < kTokensPerWarp; ++j) {
        const int t = t0 + j;
        const bool in = t < a.num_tokens;
        const uint4* src_c =
            reinterpret_cast<const uint4*>(a.kv_c + static_cast<int64_t>(t) * a.kv_c_stride);
        const uint4* src_p =
            reinterpret_cast<const uint4*>(a.k_pe + static_cast<int64_t>(t) * a.k_pe_stride);
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int c = lane + 32 * k;
          v[j][k] = !in ? make_uint4(0, 0, 0, 0)
                        : c < nc ? __ldg(src_c + c)
                                 : (c < nc + np ? __ldg(src_p + (c - nc)) : make_uint4(0, 0, 0, 0));
        }
        slot[j] = in ? __ldg(a.slot_mapping + t) : -1;
      }
      if constexpr (NR) {
        static_assert(kTokensPerWarp == 1, "the fused variant moves one token per warp");
        // every lane's 16-byte chunk of a P = 64 rotary row is pair group
        // lane & 7 (the rope chunks start at a multiple of 32 chunks)
        const int t = t0;
        const bool pos_ok = pos >= 0 && pos < a.max_position;
        const int sub = lane & 7;
        const float4* cs = reinterpret_cast<const float4*>(a.table + (pos_ok ? pos : 0) * 64);
        const float4 cv = __ldg(cs + sub), sv = __ldg(cs + 8 + sub);
        if (!pos_ok) {
          if (lane == 0 && a.err_count) atomicAdd(a.err_count, 1);
          continue;  // the whole token is skipped
        }
        // ---- RMSNorm terms (see NormTerms): the largest binade k of the
        // row, the scaled sum of squares as a two-sum pair, 1 / sqrt(t)
        NormTerms nt;
        {
          uint32_t ebits = 0;  // largest bf16 exponent field of this lane's elements
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (lane + 32 * k < nc) {
              const uint32_t xv[4] = {v[0][k].x, v[0][k].y, v[0][k].z, v[0][k].w};
#pragma unroll
              for (int e = 0; e < 4; ++e)
                ebits = max(ebits, max((xv[e] >> 7) & 0xFFu, (xv[e] >> 23) & 0xFFu));
            }
          }
          const int kexp = static_cast<int>(__reduce_max_sync(0xffffffffu, ebits)) - 127;
          // all-zero or subnormal-only rows, NaN or infinity (field 0xFF), or a
          // binade too far from 1 take the fp64 path
          nt.fast = kexp >= -20 && kexp <= 100;
          nt.sc = __uint_as_float(static_cast<uint32_t>(127 - (nt.fast ? kexp : 0)) << 23);
          float sh = 0.f, sl = 0.f;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            if (lane + 32 * k < nc) {
              const uint32_t xv[4] = {v[0][k].x, v[0][k].y, v[0][k].z, v[0][k].w};
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float xs = bfv(xv[e >> 1], e & 1) * nt.sc;
                float err;
                two_sum(sh, xs * xs, sh, err);  // xs^2 exact above 2^-126
                sl += err;
              }
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float oh = __shfl_xor_sync(0xffffffffu, sh, o);
            const float ol = __shfl_xor_sync(0xffffffffu, sl, o);
            float err;
            two_sum(sh, oh, sh, err);
            sl += ol + err;
          }
          // one value for the whole warp (lanes summed in different orders)
          sh = __shfl_sync(0xffffffffu, sh, 0);
          sl = __shfl_sync(0xffffffffu, sl, 0);
          const float rinv = 1.0f / static_cast<float>(a.R);  // a power of two: exact
          const float eps_s = a.eps * nt.sc * nt.sc;
          float th, tl;
          two_sum(sh * rinv, eps_s, th, tl);
          tl += sl * rinv;
          {
            const float h2 = th + tl;  // renormalise (|tl| << |th|)
            tl = tl - (h2 - th);
            th = h2;
          }
          nt.fast = nt.fast && eps_s <= 0x1p100f && th >= 0x1p-100f && th <= 0x1p100f;
          // Newton step on rsqrtf in double-float: e = 1 - t r0^2, inv =
          // r0 (1 + e/2 + 3e^2/8)
          const float r0 = rsqrtf(th);
          const float q2 = r0 * r0, q2l = fmaf(r0, r0, -q2);
          const float m = th * q2, ml = fmaf(th, q2, -m);
          const float e = ((1.0f - m) - ml) - fmaf(th, q2l, tl * q2);
          two_sum(r0, r0 * (e * fmaf(0.375f, e, 0.5f)), nt.inv32, nt.inv_lo);
        }
        // tier 1's scale: inv32 scaled back by sc (exact while normal)
        const float inv_s = nt.sc * nt.inv32;
        if (!(inv_s >= 0x1p-100f)) nt.fast = false;
        // Tier 1 for the latent chunks (0, 1) and the rope chunk (2); tier 2
        // for the elements it leaves; fbm: elements left to tier 3
        uint32_t fbm[3] = {0u, 0u, 0u};
        uint4 kpe_in = make_uint4(0, 0, 0, 0);
        const uint16_t* row = a.kv_c + static_cast<int64_t>(t) * a.kv_c_stride;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int c = lane + 32 * k;
          if (c < nc) {
            if (k < 2) {
              uint32_t need;
              const uint4 xin = v[0][k];
              v[0][k] = norm8(xin, gm[k], inv_s, need);
              if (!nt.fast)
                fbm[k] = 0xFFu;
              else if (need)
                v[0][k] = norm8_df(xin, gm[k], nt.sc, nt.inv32, nt.inv_lo, v[0][k], need,
                                   &fbm[k]);
            }
          } else if (c < nc + np) {
            uint32_t need;
            kpe_in = v[0][k];
            v[0][k] = rope8(kpe_in, cv, sv, need);
            if (need) v[0][k] = rope8_slow(kpe_in, cv, sv, v[0][k], need);
          }
        }
        if (__any_sync(0xffffffffu, (fbm[0] | fbm[1]) != 0u)) {
          // tier 3: the reference's fp64 1 / sqrt(ss / R + eps), from lane 0
          double inv64 = 0.0;
          if (lane == 0) inv64 = rms_inv_f64(row, a.R, a.eps);
          inv64 = __shfl_sync(0xffffffffu, inv64, 0);
#pragma unroll
          for (int k = 0; k < 2; ++k)
            if (fbm[k])
              v[0][k] = norm8_f64(__ldg(reinterpret_cast<const uint4*>(row) + lane + 32 * k),
                                  gm[k], inv64, v[0][k], fbm[k]);
        }
        if (a.q_pe != nullptr) {
          // q_pe of this token: q_heads x 8 chunks, chunk lane + 32 i is
          // pair group lane & 7 of head (lane + 32 i) / 8
          const int nq = a.q_heads * 8;
          uint16_t* qrow = a.q_pe + static_cast<int64_t>(t) * a.q_pe_row_stride;
          for (int c0 = 0; c0 < nq; c0 += 128) {
            uint4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int c = c0 + 32 * u + lane;
              if (c < nq)
                x[u] = *reinterpret_cast<const uint4*>(qrow + (c >> 3) * a.q_pe_head_stride +
                                                       (c & 7) * 8);
            }
            uint4 y[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (c0 + 32 * u + lane < nq) {
                uint32_t need;
                y[u] = rope8(x[u], cv, sv, need);
                if (need) y[u] = rope8_slow(x[u], cv, sv, y[u], need);
              }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int c = c0 + 32 * u + lane;
              if (c < nq)
                *reinterpret_cast<uint4*>(qrow + (c >> 3) * a.q_pe_head_stride + (c & 7) * 8) =
                    y[u];
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kTokensPerWarp; ++j) {
        if (slot[j] < 0) continue;  // padded token (or past the end)
        if (slot[j] >= a.num_slots) {
          if (lane == 0 && a.err_count) atomicAdd(a.err_count, 1);
          continue;
        }
        const int64_t blk = slot[j] / a.block_size;
        const int64_t off = slot[j] - blk * a.block_size;
        const int64_t dst_elem = blk * a.block_stride + off * D;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int c = lane + 32 * k;
          if (c >= nc + np) break;
          if constexpr (FP8) {
            uint8_t* dst = static_cast<uint8_t*>(a.cache) + dst_elem;
            reinterpret_cast<uint2*>(dst)[c] = quant8<FMT>(v[j][k], s, r);
          } else {
            uint16_t* dst = static_cast<uint16_t*>(a.cache) + dst_elem;
            reinterpret_cast<uint4*>(dst)[c] = v[j][k];
          }
        }
      }
    } else {
      for (int t = t0; t < t0 + kTokensPerWarp && t < a.num_tokens; ++t) {
        const uint16_t* src_c = a.kv_c + static_cast<int64_t>(t) * a.kv_c_stride;
        const uint16_t* src_p = a.k_pe + static_cast<int64_t>(t) * a.k_pe_stride;
        const int64_t slot = a.slot_mapping[t];
        if (slot < 0) continue;  // padded token
        if (slot >= a.num_slots) {
          if (lane == 0 && a.err_count) atomicAdd(a.err_count, 1);
          continue;
        }
        const int64_t blk = slot / a.block_size;
        const int64_t off = slot - blk * a.block_size;
        const int64_t dst_elem = blk * a.block_stride + off * D;
        for (int i = lane; i < D; i += 32) {
          const uint16_t x = (i < a.R) ? src_c[i] : src_p[i - a.R];
          if constexpr (FP8)
            static_cast<uint8_t*>(a.cache)[dst_elem + i] = quant1<FMT>(x, s);
          else
            static_cast<uint16_t*>(a.cache)[dst_elem + i] = x;
        }
      }
    }
  }
}

// Launches the fused variant KERNEL on min(need, one wave) CTAs, the wave
// being the CTAs resident at once (per SM x SMs of the current device, both
// queried once per device): with its one-row warps and three CTAs per SM, a
// grid past one wave left a partial last wave (whole-cache fp8 fused write
// 259 against 247 us).  The plain write keeps its larger grid, which
// measured faster than one wave (148 against 156 us).  A failed query is
// returned as the launch's error (nothing is launched).
template <auto KERNEL>
cudaError_t launch_one_wave(int64_t need, const CacheWriteArgs& a, cudaStream_t stream) {
  static std::atomic<int> per_sm_cache[kMaxDevices] = {};
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  e = device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  int per_sm = per_sm_cache[dev].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, KERNEL, kWarpsPerCta * 32, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    per_sm_cache[dev].store(per_sm, std::memory_order_relaxed);
  }
  const int64_t wave = static_cast<int64_t>(per_sm) * sms;
  const dim3 grid(static_cast<unsigned>(need < wave ? need : wave));
  KERNEL<<<grid, dim3(kWarpsPerCta * 32), 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cache_write(const void* kv_c, int64_t kv_c_stride,
                               const void* k_pe, int64_t k_pe_stride,
                               const int64_t* slot_mapping, int num_tokens,
                               int R, int P, void* cache, int num_blocks,
                               int block_size, int64_t block_stride, int fmt,
                               const float* scale, int* err_count,
                               cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const bool fp8 = fmt != kBf16;
  CacheWriteArgs a;
  a.kv_c = static_cast<const uint16_t*>(kv_c);
  a.kv_c_stride = kv_c_stride;
  a.k_pe = static_cast<const uint16_t*>(k_pe);
  a.k_pe_stride = k_pe_stride;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.R = R;
  a.P = P;
  a.cache = cache;
  a.num_slots = static_cast<int64_t>(num_blocks) * block_size;
  a.block_size = block_size;
  a.block_stride = block_stride;
  a.scale = scale;
  a.err_count = err_count;
  a.gamma = nullptr;
  a.eps = 0.f;
  a.positions = nullptr;
  a.table = nullptr;
  a.max_position = 0;
  a.q_pe = nullptr;
  a.q_pe_row_stride = a.q_pe_head_stride = 0;
  a.q_heads = 0;
  const size_t elt = fp8 ? 1 : 2;
  auto al16 = [](uintptr_t x) { return (x & 15u) == 0; };
  const bool vec = al16(reinterpret_cast<uintptr_t>(kv_c)) &&
                   al16(reinterpret_cast<uintptr_t>(k_pe)) &&
                   (kv_c_stride % 8 == 0) && (k_pe_stride % 8 == 0) &&
                   (R % 8 == 0) && (P % 8 == 0) &&
                   al16(reinterpret_cast<uintptr_t>(cache)) &&
                   ((block_stride * elt) % 16 == 0) &&
                   ((static_cast<size_t>(R + P) * elt) % 16 == 0) &&
                   ((static_cast<size_t>(R) * elt) % (fp8 ? 8 : 16) == 0);
  int sms = 0;
  cudaError_t e = device_sm_count(&sms);
  if (e != cudaSuccess) return e;
  const int64_t per_cta = static_cast<int64_t>(kWarpsPerCta) * kTokensPerWarp;
  const int64_t need = (static_cast<int64_t>(num_tokens) + per_cta - 1) / per_cta;
  const dim3 grid(static_cast<unsigned>(need < 8 * sms ? need : 8 * sms));
  const dim3 block(kWarpsPerCta * 32);
  if (fmt == kE4M3) {
    if (vec)
      cache_write_kernel<kE4M3, true><<<grid, block, 0, stream>>>(a);
    else
      cache_write_kernel<kE4M3, false><<<grid, block, 0, stream>>>(a);
  } else if (fmt == kE5M2) {
    if (vec)
      cache_write_kernel<kE5M2, true><<<grid, block, 0, stream>>>(a);
    else
      cache_write_kernel<kE5M2, false><<<grid, block, 0, stream>>>(a);
  } else {
    if (vec)
      cache_write_kernel<kBf16, true><<<grid, block, 0, stream>>>(a);
    else
      cache_write_kernel<kBf16, false><<<grid, block, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_norm_rope_cache_write(const void* kv_c, int64_t kv_c_stride, const void* k_pe,
                                         int64_t k_pe_stride, const int64_t* slot_mapping,
                                         int num_tokens, int R, void* cache, int num_blocks,
                                         int block_size, int64_t block_stride, int fmt,
                                         const float* scale, const void* gamma, float eps,
                                         const int64_t* positions, const float* table,
                                         int64_t max_position, void* q_pe,
                                         int64_t q_pe_row_stride, int64_t q_pe_head_stride,
                                         int q_heads, int* err_count, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  CacheWriteArgs a;
  a.kv_c = static_cast<const uint16_t*>(kv_c);
  a.kv_c_stride = kv_c_stride;
  a.k_pe = static_cast<const uint16_t*>(k_pe);
  a.k_pe_stride = k_pe_stride;
  a.slot_mapping = slot_mapping;
  a.num_tokens = num_tokens;
  a.R = R;
  a.P = 64;
  a.cache = cache;
  a.num_slots = static_cast<int64_t>(num_blocks) * block_size;
  a.block_size = block_size;
  a.block_stride = block_stride;
  a.scale = scale;
  a.err_count = err_count;
  a.gamma = static_cast<const uint16_t*>(gamma);
  a.eps = eps;
  a.positions = positions;
  a.table = table;
  a.max_position = max_position;
  a.q_pe = static_cast<uint16_t*>(q_pe);
  a.q_pe_row_stride = q_pe_row_stride;
  a.q_pe_head_stride = q_pe_head_stride;
  a.q_heads = q_heads;
  const int64_t need = (static_cast<int64_t>(num_tokens) + kWarpsPerCta - 1) / kWarpsPerCta;
  if (fmt == kE4M3) return launch_one_wave<cache_write_kernel<kE4M3, true, true>>(need, a, stream);
  if (fmt == kE5M2) return launch_one_wave<cache_write_kernel<kE5M2, true, true>>(need, a, stream);
  return launch_one_wave<cache_write_kernel<kBf16, true, true>>(need, a, stream);
}

}  // namespace mla
