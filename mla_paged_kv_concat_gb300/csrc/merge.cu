// Stage 2: merge split-KV partial outputs by their log-sum-exp.
//
// Restates "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
// vllm/attention/ops/triton_decode_attention.py, _fwd_kernel_stage2: for one
// (row, head), visit the non-empty splits in index order, weight each split's
// normalised output by exp(lse_s - M) with M the largest split lse, and
// divide by the sum of the weights.  The lse of the whole row is
// M + ln(sum of weights) ("Triton and MLA: portable attention and multi-head
// latent attention", Data flow: forward_mqa returns (o, lse)).
//
// One warp per (row, head); each lane owns R/32 latent columns in 16-byte
// groups, so every partial row is read with coalesced 512-byte warp loads.
// Stage 1 leaves every split slot of a non-empty sequence either holding a
// partial or marked with lse = -inf (a slot its partition did not use); the
// merge visits the slots in index order and skips the marked ones, so it
// needs no knowledge of how stage 1 partitioned the sequence.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kMergeWarps = 8;

template <int R>
__global__ void __launch_bounds__(kMergeWarps * 32)
    merge_kernel(const DecodeParams p) {
  constexpr int NV = R / 128;  // float4 groups per lane
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  const int H = p.num_heads;
  if (gw >= p.num_rows * H) return;
  const int row = gw / H, h = gw % H;
  const int S = p.num_splits;
  int L = __ldg(p.seq_lens + row / p.rows_per_seq);
  const int Lmax = p.max_blocks * p.block_size;
  L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
  uint16_t* orow = p.o + static_cast<int64_t>(gw) * R;
  if (L == 0) {
#pragma unroll
    for (int k = 0; k < NV; ++k)
      reinterpret_cast<uint2*>(orow)[k * 32 + lane] = make_uint2(0, 0);
    if (lane == 0) p.lse[gw] = -INFINITY;
    return;
  }
  const int64_t rec0 = static_cast<int64_t>(row) * S * H + h;  // split 0
  float M = -INFINITY;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, p.ws_lse[rec0 + static_cast<int64_t>(s) * H]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float4 acc[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int s = 0; s < S; ++s) {
    const int64_t rec = rec0 + static_cast<int64_t>(s) * H;
    const float ls = p.ws_lse[rec];
    if (ls == -INFINITY) continue;  // a slot stage 1 left without a partial
    const float w = __expf(ls - M);
    const float4* src = reinterpret_cast<const float4*>(p.ws_o + rec * R);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const float4 v = src[k * 32 + lane];
      acc[k].x += w * v.x;
      acc[k].y += w * v.y;
      acc[k].z += w * v.z;
      acc[k].w += w * v.w;
    }
    den += w;
  }
  const float inv = 1.f / den;
#pragma unroll
  for (int k = 0; k < NV; ++k)
    reinterpret_cast<uint2*>(orow)[k * 32 + lane] =
        make_uint2(pack_bf16x2(acc[k].x * inv, acc[k].y * inv),
                   pack_bf16x2(acc[k].z * inv, acc[k].w * inv));
  if (lane == 0) p.lse[gw] = M + __logf(den);
}

}  // namespace

cudaError_t launch_merge(const DecodeParams& p, int R, cudaStream_t stream) {
  const int64_t pairs = static_cast<int64_t>(p.num_rows) * p.num_heads;
  if (pairs == 0) return cudaSuccess;
  const dim3 grid(static_cast<unsigned>((pairs + kMergeWarps - 1) / kMergeWarps));
  if (R == 512)
    merge_kernel<512><<<grid, kMergeWarps * 32, 0, stream>>>(p);
  else
    merge_kernel<256><<<grid, kMergeWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mla
