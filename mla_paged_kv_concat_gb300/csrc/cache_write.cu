// Cache write: scatter new tokens' [kv_c | k_pe] rows into the paged latent
// cache through slot_mapping, optionally quantising to OCP E4M3.
//
// Restates "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
// csrc/cache_kernels.cu, concat_and_cache_mla_kernel.  That kernel runs one
// CTA per token with a strided scalar loop; here one warp moves one token
// with 16-byte vector loads and stores (a 576-element bf16 row is 72 such
// chunks), eight tokens per 256-thread CTA.
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

// 8 bf16 values -> 8 E4M3 bytes of x / scale (IEEE division, RNE, satfinite).
__device__ __forceinline__ uint2 quant8(uint4 v, float s) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
  uint32_t w[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    float2 a = __bfloat1622float2(h[2 * k]);
    float2 b = __bfloat1622float2(h[2 * k + 1]);
    __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(a.x, s), __fdiv_rn(a.y, s)), __NV_SATFINITE,
        __NV_E4M3);
    __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(b.x, s), __fdiv_rn(b.y, s)), __NV_SATFINITE,
        __NV_E4M3);
    w[k] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
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
  const int t = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (t >= a.num_tokens) return;
  const int64_t slot = a.slot_mapping[t];
  if (slot < 0) return;  // padded token
  if (slot >= a.num_slots) {
    if (lane == 0 && a.err_count) atomicAdd(a.err_count, 1);
    return;
  }
  const int D = a.R + a.P;
  const int64_t blk = slot / a.block_size;
  const int64_t off = slot - blk * a.block_size;
  const int64_t dst_elem = blk * a.block_stride + off * D;
  const uint16_t* src_c = a.kv_c + static_cast<int64_t>(t) * a.kv_c_stride;
  const uint16_t* src_p = a.k_pe + static_cast<int64_t>(t) * a.k_pe_stride;
  const float s = FP8 ? __ldg(a.scale) : 1.0f;

  if constexpr (VEC) {
    const int nc = a.R / 8, np = a.P / 8;
    for (int c = lane; c < nc + np; c += 32) {
      const uint4 v = (c < nc) ? __ldg(reinterpret_cast<const uint4*>(src_c) + c)
                               : __ldg(reinterpret_cast<const uint4*>(src_p) +
                                       (c - nc));
      if constexpr (FP8) {
        uint8_t* dst = static_cast<uint8_t*>(a.cache) + dst_elem;
        reinterpret_cast<uint2*>(dst)[c] = quant8(v, s);
      } else {
        uint16_t* dst = static_cast<uint16_t*>(a.cache) + dst_elem;
        reinterpret_cast<uint4*>(dst)[c] = v;
      }
    }
  } else {
    for (int i = lane; i < D; i += 32) {
      const uint16_t x = (i < a.R) ? src_c[i] : src_p[i - a.R];
      if constexpr (FP8)
        static_cast<uint8_t*>(a.cache)[dst_elem + i] = quant1(x, s);
      else
        static_cast<uint16_t*>(a.cache)[dst_elem + i] = x;
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
  const dim3 grid((num_tokens + kWarpsPerCta - 1) / kWarpsPerCta);
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
