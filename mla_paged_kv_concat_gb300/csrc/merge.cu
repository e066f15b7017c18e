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
// The split weights are computed from all lse values first, so the partial
// rows of several splits are in flight at once instead of one round trip per
// split.
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
constexpr int kInFlight = 2;  // partial rows loaded together per warp

template <int R>
__global__ void __launch_bounds__(kMergeWarps * 32, 3)
    merge_kernel(const DecodeParams p) {
  constexpr int NV = R / 128;  // float4 groups per lane
  griddep_wait();              // stage 1's partials are complete and visible
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  const int H = p.num_heads;
  if (gw >= p.num_rows * H) return;
  const int row = gw / H, h = gw % H;
  const int S = p.num_splits;
  const int64_t rec0 = static_cast<int64_t>(row) * S * H + h;  // split 0
  // The sequence length and the lse of the first 32 slots are loaded
  // together (one round trip); the slots of an empty sequence hold stale
  // values that are never used.
  int L = __ldg(p.seq_lens + row / p.rows_per_seq);
  const float ls0 = lane < S ? p.ws_lse[rec0 + static_cast<int64_t>(lane) * H] : -INFINITY;
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
  float M = ls0;
  for (int s = lane + 32; s < S; s += 32) M = fmaxf(M, p.ws_lse[rec0 + static_cast<int64_t>(s) * H]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));

  float4 acc[NV];
#pragma unroll
  for (int k = 0; k < NV; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;  // this lane's slots; summed over the warp at the end
  for (int c = 0; c < S; c += 32) {
    // Lane j holds the weight of slot c + j; the partial rows of up to
    // kInFlight non-empty slots are loaded together, then added in slot
    // order (few rows per warp, many warps per SM).
    const int s = c + lane;
    const float ls =
        c == 0 ? ls0 : (s < S ? p.ws_lse[rec0 + static_cast<int64_t>(s) * H] : -INFINITY);
    const float w = ls == -INFINITY ? 0.f : __expf(ls - M);
    den += w;
    uint32_t mask = __ballot_sync(0xffffffffu, w != 0.f);
    while (mask) {
      int js[kInFlight];
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) {
        js[u] = mask ? __ffs(mask) - 1 : -1;
        mask &= mask ? mask - 1 : 0u;
      }
      float4 v[kInFlight][NV];
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) {
        if (js[u] < 0) continue;
        const float4* src = reinterpret_cast<const float4*>(
            p.ws_o + (rec0 + static_cast<int64_t>(c + js[u]) * H) * R);
#pragma unroll
        for (int k = 0; k < NV; ++k) v[u][k] = src[k * 32 + lane];
      }
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) {
        if (js[u] < 0) continue;
        const float wj = __shfl_sync(0xffffffffu, w, js[u]);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          acc[k].x += wj * v[u][k].x;
          acc[k].y += wj * v[u][k].y;
          acc[k].z += wj * v[u][k].z;
          acc[k].w += wj * v[u][k].w;
        }
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
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
  // Overlaps its launch with the tail of stage 1 (which lets it start early).
  return R == 512 ? launch_overlapped(merge_kernel<512>, grid, dim3(kMergeWarps * 32), 0,
                                      stream, p)
                  : launch_overlapped(merge_kernel<256>, grid, dim3(kMergeWarps * 32), 0,
                                      stream, p);
}

}  // namespace mla
