// Cache write: scatter new tokens' [kv_c | k_pe] rows into the paged latent
// cache through slot_mapping, optionally quantising to OCP E4M3.
//
// Restates "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
// csrc/cache_kernels.cu, concat_and_cache_mla_kernel.  That kernel runs one
// CTA per token with a strided scalar loop; here one warp moves one token at
// a time with 16-byte vector loads and stores (a 576-element bf16 row is 72
// such chunks), in a warp-stride loop over the tokens, and the E4M3 encoding
// avoids the division except next to a rounding boundary (see quant2).
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
};

constexpr int kWarpsPerCta = 8;
constexpr int kTokensPerWarp = 1;  // rows per warp per pass (more raised register use, not speed)

// Two fp32 -> two E4M3 codes (round to nearest even, satfinite), low code
// first.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// E4M3 codes of RN_f32(x0 / s), RN_f32(x1 / s) (IEEE division, then RNE to
// E4M3 with saturation), without a division in the common case.  With
// r = RN(1/s) (an IEEE division, once per thread), q = RN(x * r) is within
// 1.5 * 2^-23 |q| of RN_f32(x / s) (three roundings of relative size at most
// 2^-24).  E4M3 rounding is monotone in the value, so when q - 2^-22 |q| and
// q + 2^-22 |q| get the same code, so does RN_f32(x / s); otherwise the
// quotient is within a few ulp of a boundary between two codes and the
// division is done.  Quotients too small for the relative bound (|q| below
// 2^-104) are all +-0 in E4M3, with the sign that both sides agree on; |q|
// is clamped to 2^100 (every such value saturates to +-448 either way); NaN
// quotients take the division.
__device__ __forceinline__ uint32_t quant2(float x0, float x1, float s, float r) {
  float q0 = x0 * r, q1 = x1 * r;
  if (q0 != q0 || q1 != q1) return e4m3x2(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
  q0 = fminf(fmaxf(q0, -0x1p100f), 0x1p100f);
  q1 = fminf(fmaxf(q1, -0x1p100f), 0x1p100f);
  const float d0 = fabsf(q0) * 0x1p-22f, d1 = fabsf(q1) * 0x1p-22f;
  const uint32_t lo = e4m3x2(q0 - d0, q1 - d1);
  const uint32_t hi = e4m3x2(q0 + d0, q1 + d1);
  if (lo == hi) return lo;
  return e4m3x2(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
}

// 8 bf16 values -> 8 E4M3 bytes of x / scale (IEEE division, RNE, satfinite).
__device__ __forceinline__ uint2 quant8(uint4 v, float s, float r) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
  uint32_t w[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const float2 a = __bfloat1622float2(h[2 * k]);
    const float2 b = __bfloat1622float2(h[2 * k + 1]);
    w[k] = quant2(a.x, a.y, s, r) | (quant2(b.x, b.y, s, r) << 16);
  }
  return make_uint2(w[0], w[1]);
}

__device__ __forceinline__ uint8_t quant1(uint16_t bits, float s) {
  float x = __bfloat162float(__ushort_as_bfloat16(bits));
  return static_cast<uint8_t>(
      __nv_cvt_float_to_fp8(__fdiv_rn(x, s), __NV_SATFINITE, __NV_E4M3));
}

// VEC: every source row and destination row starts on a 16-byte boundary, so
// rows move as 16-byte chunks (8 elements); otherwise element by element.
template <bool FP8, bool VEC>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    cache_write_kernel(const CacheWriteArgs a) {
  // The decode kernels that follow wait for this grid's completion before
  // they read anything; letting them launch now hides their launch latency.
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int D = a.R + a.P;
  const float s = FP8 ? __ldg(a.scale) : 1.0f;
  const float r = FP8 ? __fdiv_rn(1.0f, s) : 1.0f;  // RN(1/s), as quant2's bound assumes
  // Warp-stride loop over groups of kTokensPerWarp consecutive tokens (the
  // grid is sized to the GPU, not to the token count).  All loads of a group
  // (rows and slots) are issued before any of them is used, so that each
  // warp keeps several rows in flight: the write is bound by HBM, not by
  // load latency.
  const int nwarps = gridDim.x * kWarpsPerCta;
  const int warp_id = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  for (int t0 = warp_id * kTokensPerWarp; t0 < a.num_tokens; t0 += nwarps * kTokensPerWarp) {
    if constexpr (VEC) {
      // lane l holds 16-byte chunks l, l + 32, l + 64 of each D-element row
      // (D <= 576: at most 3)
      const int nc = a.R / 8, np = a.P / 8;
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
            reinterpret_cast<uint2*>(dst)[c] = quant8(v[j][k], s, r);
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
            static_cast<uint8_t*>(a.cache)[dst_elem + i] = quant1(x, s);
          else
            static_cast<uint16_t*>(a.cache)[dst_elem + i] = x;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_cache_write(const void* kv_c, int64_t kv_c_stride,
                               const void* k_pe, int64_t k_pe_stride,
                               const int64_t* slot_mapping, int num_tokens,
                               int R, int P, void* cache, int num_blocks,
                               int block_size, int64_t block_stride, bool fp8,
                               const float* scale, int* err_count,
                               cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
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
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t per_cta = static_cast<int64_t>(kWarpsPerCta) * kTokensPerWarp;
  const int64_t need = (static_cast<int64_t>(num_tokens) + per_cta - 1) / per_cta;
  const dim3 grid(static_cast<unsigned>(need < 8 * sms ? need : 8 * sms));
  const dim3 block(kWarpsPerCta * 32);
  if (fp8) {
    if (vec)
      cache_write_kernel<true, true><<<grid, block, 0, stream>>>(a);
    else
      cache_write_kernel<true, false><<<grid, block, 0, stream>>>(a);
  } else {
    if (vec)
      cache_write_kernel<false, true><<<grid, block, 0, stream>>>(a);
    else
      cache_write_kernel<false, false><<<grid, block, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace mla
