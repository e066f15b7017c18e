// Cross-shard LSE merge: G disjoint shards of the KV tokens of the same rows
// (decode context parallelism) combined into the result over all of them.
//
// Restates "Triton and MLA: portable attention and multi-head latent
// attention", Design motivation (decode returns lse because decode context
// parallelism merges the per-shard (o, lse) pairs with cp_lse_ag_out_rs),
// with the LSE algebra of
// "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
// vllm/attention/ops/triton_decode_attention.py, _fwd_kernel_stage2: M = max
// lse_g over the non-empty shards, o = sum e^{lse_g - M} o_g / sum
// e^{lse_g - M}, lse = M + ln sum e^{lse_g - M}, shards added in index order;
// no non-empty shard gives o = 0, lse = -inf.
//
// One warp per (row, head); each lane owns R/32 latent columns as 16-byte
// groups of bf16; the rows of up to four non-empty shards are in flight at
// once.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kLseMergeWarps = 8;

struct LseMergeArgs {
  const uint16_t* o_parts;  // bf16 [G][rows][H][R], part stride in elements
  int64_t o_part_stride;
  const float* lse_parts;   // [G][rows][H], part stride in elements
  int64_t lse_part_stride;
  int num_parts;
  int64_t records;          // rows * H
  uint16_t* o;
  float* lse;
};

__device__ __forceinline__ void bf16x8_fma(float (&acc)[8], float w, uint4 x) {
  const uint32_t v[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    acc[2 * k] += w * __uint_as_float(v[k] << 16);
    acc[2 * k + 1] += w * __uint_as_float(v[k] & 0xFFFF0000u);
  }
}

template <int R>
__global__ void __launch_bounds__(kLseMergeWarps * 32) lse_merge_kernel(const LseMergeArgs a) {
  constexpr int NV = R / 256;  // 16-byte groups per lane
  const int lane = threadIdx.x & 31;
  const int64_t rec = static_cast<int64_t>(blockIdx.x) * kLseMergeWarps + (threadIdx.x >> 5);
  if (rec >= a.records) return;
  const int G = a.num_parts;
  float M = -INFINITY;
  for (int g = lane; g < G; g += 32) M = fmaxf(M, a.lse_parts[g * a.lse_part_stride + rec]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  uint4* orow = reinterpret_cast<uint4*>(a.o + rec * R);
  if (M == -INFINITY) {
#pragma unroll
    for (int k = 0; k < NV; ++k) orow[k * 32 + lane] = make_uint4(0, 0, 0, 0);
    if (lane == 0) a.lse[rec] = -INFINITY;
    return;
  }
  float acc[NV][8];
#pragma unroll
  for (int k = 0; k < NV; ++k)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[k][e] = 0.f;
  float den = 0.f;  // this lane's shards; summed over the warp at the end
  for (int c = 0; c < G; c += 32) {
    // lane j holds the weight of shard c + j
    const int g = c + lane;
    const float lg = g < G ? a.lse_parts[g * a.lse_part_stride + rec] : -INFINITY;
    const float w = lg == -INFINITY ? 0.f : __expf(lg - M);
    den += w;
    uint32_t mask = __ballot_sync(0xffffffffu, w != 0.f);
    while (mask) {
      int js[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        js[u] = mask ? __ffs(mask) - 1 : -1;
        mask &= mask ? mask - 1 : 0u;
      }
      uint4 x[4][NV];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (js[u] < 0) continue;
        const uint4* src = reinterpret_cast<const uint4*>(
            a.o_parts + static_cast<int64_t>(c + js[u]) * a.o_part_stride + rec * R);
#pragma unroll
        for (int k = 0; k < NV; ++k) x[u][k] = src[k * 32 + lane];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (js[u] < 0) continue;
        const float wj = __shfl_sync(0xffffffffu, w, js[u]);
#pragma unroll
        for (int k = 0; k < NV; ++k) bf16x8_fma(acc[k], wj, x[u][k]);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  const float inv = 1.f / den;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    orow[k * 32 + lane] = make_uint4(pack_bf16x2(acc[k][0] * inv, acc[k][1] * inv),
                                     pack_bf16x2(acc[k][2] * inv, acc[k][3] * inv),
                                     pack_bf16x2(acc[k][4] * inv, acc[k][5] * inv),
                                     pack_bf16x2(acc[k][6] * inv, acc[k][7] * inv));
  if (lane == 0) a.lse[rec] = M + __logf(den);
}

}  // namespace

cudaError_t launch_lse_merge(const void* o_parts, int64_t o_part_stride, const float* lse_parts,
                             int64_t lse_part_stride, int num_parts, int64_t records, int R,
                             void* o, float* lse, cudaStream_t stream) {
  if (records == 0) return cudaSuccess;
  LseMergeArgs a;
  a.o_parts = static_cast<const uint16_t*>(o_parts);
  a.o_part_stride = o_part_stride;
  a.lse_parts = lse_parts;
  a.lse_part_stride = lse_part_stride;
  a.num_parts = num_parts;
  a.records = records;
  a.o = static_cast<uint16_t*>(o);
  a.lse = lse;
  const dim3 grid(static_cast<unsigned>((records + kLseMergeWarps - 1) / kLseMergeWarps));
  if (R == 512)
    lse_merge_kernel<512><<<grid, kLseMergeWarps * 32, 0, stream>>>(a);
  else
    lse_merge_kernel<256><<<grid, kLseMergeWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
