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

// RMSNorm of 8 latent elements: bf16(x * inv * gamma).
__device__ __forceinline__ uint4 norm8(uint4 x, uint4 g, float inv) {
  const uint32_t xv[4] = {x.x, x.y, x.z, x.w}, gv[4] = {g.x, g.y, g.z, g.w};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k)
    o[k] = pack_bf16x2(bf_lo(xv[k]) * inv * bf_lo(gv[k]), bf_hi(xv[k]) * inv * bf_hi(gv[k]));
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// Non-NeoX rotation of 4 interleaved pairs (8 bf16) by angles with the given
// cos and sin: (a, b) -> (a c - b s, b c + a s), rounded to bf16.
__device__ __forceinline__ uint4 rope8(uint4 x, float4 c, float4 s) {
  const uint32_t xv[4] = {x.x, x.y, x.z, x.w};
  const float cv[4] = {c.x, c.y, c.z, c.w}, sv[4] = {s.x, s.y, s.z, s.w};
  uint32_t o[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float a = bf_lo(xv[k]), b = bf_hi(xv[k]);
    o[k] = pack_bf16x2(a * cv[k] - b * sv[k], b * cv[k] + a * sv[k]);
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
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int c = lane + 32 * k;
          if (c < nc) {
            const uint32_t xv[4] = {v[0][k].x, v[0][k].y, v[0][k].z, v[0][k].w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              ss += bf_lo(xv[e]) * bf_lo(xv[e]) + bf_hi(xv[e]) * bf_hi(xv[e]);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = __frsqrt_rn(ss * (1.0f / static_cast<float>(a.R)) + a.eps);
#pragma unroll
        for (int k = 0; k < 3; ++k) {
          const int c = lane + 32 * k;
          if (c < nc)
            v[0][k] = norm8(v[0][k], gm[k < 2 ? k : 0], inv);
          else if (c < nc + np)
            v[0][k] = rope8(v[0][k], cv, sv);
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
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int c = c0 + 32 * u + lane;
              if (c < nq)
                *reinterpret_cast<uint4*>(qrow + (c >> 3) * a.q_pe_head_stride + (c & 7) * 8) =
                    rope8(x[u], cv, sv);
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
