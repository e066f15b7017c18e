// Launch entry points of the device kernels (host side, C++ linkage).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace mla {

// Largest number of (sequence, 16-vector block) units the persistent
// warp-MMA schedule handles; larger batches use one CTA per (unit, split).
constexpr int kMaxPersistUnits = 512;

// Device ordinals the per-device caches below cover.
constexpr int kMaxDevices = 64;

// SM count of the current device, queried once per device and cached (calls
// from several host threads may race to fill an entry; they store the same
// value).  Returns the query's error instead of guessing a count.
cudaError_t device_sm_count(int* sms);

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device, once per device: the attribute belongs to the device, so a process
// that drives several GPUs sets it on each.  `done` is one bit per device
// ordinal, owned by the caller (one per kernel instantiation).  Threads that
// race here set the same value; the bit is published only after success.
template <typename K>
inline cudaError_t set_smem_attr_once(K kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const uint64_t bit = uint64_t{1} << dev;
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  done.fetch_or(bit, std::memory_order_release);
  return cudaSuccess;
}

// Arguments of one decode call after host validation.  Pointers are device
// memory.  rows = num_seqs * rows_per_seq.
struct DecodeParams {
  const uint16_t* q;     // bf16 [rows, H, >= R]: dims [0, R) of each query vector
  int64_t q_row_stride, q_head_stride;
  const uint16_t* q_pe;  // bf16 [rows, H, >= P]: dims [R, R+P) (q + R for a concatenated q)
  int64_t q_pe_row_stride, q_pe_head_stride;
  int num_rows, num_heads, rows_per_seq, num_seqs;
  const int32_t* block_table;
  int64_t bt_stride;
  int max_blocks;
  const int32_t* seq_lens;
  int block_size, num_blocks;
  float sm_scale;
  const float* kv_scale;  // device; fp8 cache only (else nullptr)
  int kv_e5m2;            // fp8 cache holds E5M2 codes (else E4M3)
  int num_splits;
  float* ws_o;    // [rows][S][H][R] fp32 partial outputs (S > 1)
  float* ws_lse;  // [rows][S][H] fp32 partial lse (S > 1)
  uint16_t* o;    // bf16 [rows, H, R]
  float* lse;     // fp32 [rows, H]
  int* err_count;
  int q_tma;      // the warp-MMA kernel loads Q through its q tensor map
};

// Launches `kernel` so that it may start while the previous kernel of the
// stream is still running (programmatic stream serialization).  Every kernel
// launched this way calls griddep_wait() before touching global memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                     size_t smem, cudaStream_t stream, const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// fmt: cache element format, the mla_kv_dtype value (0 bf16, 1 E4M3, 2 E5M2).
cudaError_t launch_cache_write(const void* kv_c, int64_t kv_c_stride,
                               const void* k_pe, int64_t k_pe_stride,
                               const int64_t* slot_mapping, int num_tokens,
                               int R, int P, void* cache, int num_blocks,
                               int block_size, int64_t block_stride, int fmt,
                               const float* scale, int* err_count,
                               cudaStream_t stream);

// The cache write fused with RMSNorm of kv_c (weight gamma) and the non-NeoX
// rotation of k_pe (and of q_pe in place when q_pe is non-null) by position,
// table fp32 [max_position][64] = cos | sin.  Rows 16-byte aligned, P = 64.
cudaError_t launch_norm_rope_cache_write(const void* kv_c, int64_t kv_c_stride, const void* k_pe,
                                         int64_t k_pe_stride, const int64_t* slot_mapping,
                                         int num_tokens, int R, void* cache, int num_blocks,
                                         int block_size, int64_t block_stride, int fmt,
                                         const float* scale, const void* gamma, float eps,
                                         const int64_t* positions, const float* table,
                                         int64_t max_position, void* q_pe,
                                         int64_t q_pe_row_stride, int64_t q_pe_head_stride,
                                         int q_heads, int* err_count, cudaStream_t stream);

// Tensor maps of the two parts of q for the warp-MMA kernel: q_nope
// {R, H, rows} and q_pe {P, H, rows}, each with a {64, 16, 1} box and
// 128-byte swizzle.
struct QMaps {
  CUtensorMap nope;
  CUtensorMap pe;
};

// Stage 1 on warp-level MMA (mma.sync m16n8k16), any head count.  `tmap` is
// a 3-D tiled tensor map over the cache {R+P, block_size, num_blocks} with a
// {64, min(block_size, 64), 1} box: 128-byte swizzle for bf16, none for fp8.
// With p.q_tma, `qmap` holds the maps of q's two parts (heads a multiple of
// 16); otherwise it is unused and Q is gathered with cp.async.  With num_kv_splits > 1 it runs
// persistent, one CTA per SM (`sm_count`).  Launched overlapped with the
// previous kernel of the stream.
cudaError_t launch_decode_mma(const DecodeParams& p, const CUtensorMap& tmap,
                              const QMaps& qmap, int R, bool fp8, int sm_count,
                              cudaStream_t stream);

// Stage 1 on tcgen05/TMEM for bf16 caches with R = 512, 2-CTA clusters of 128
// query vectors.  With num_kv_splits > 1 (and at most kMaxPersistUnits
// (sequence, 128-vector block) units) it runs persistent, sm_count / 2 pairs
// with the tiles balanced over them; otherwise one pair per 128 vectors and
// group of `split_group` consecutive splits.  `tmap` as above ({64,
// min(block_size, 64), 1} box, 128-byte swizzle); `rope_map` the same tensor
// with a {32, min(block_size, 64), 1} box and 64-byte swizzle (each CTA of a
// pair takes half of the 64 rope dims).  Launched overlapped with the previous
// kernel of the stream.
cudaError_t launch_decode_tc(const DecodeParams& p, const CUtensorMap& tmap,
                             const CUtensorMap& rope_map, int split_group, int sm_count,
                             cudaStream_t stream);
// Consecutive splits a tcgen05 kernel processes per unit of `ctas_per_unit`
// CTAs (2: the 512-wide kernel's pairs; 1: the 256-wide kernel) in grid mode.
int tc_split_group(const DecodeParams& p, int sm_count, int ctas_per_unit);

// Stage 1 on tcgen05/TMEM for the 256-wide latent (R = 256), bf16 or fp8
// cache, one CTA per 128 query vectors (no cluster).  With num_kv_splits > 1
// (and at most kMaxPersistUnits (sequence, 128-vector block) units) it runs
// persistent, one CTA per SM (`sm_count`); otherwise one CTA per 128 vectors
// and group of `split_group` consecutive splits.  `tmap` as for the warp-MMA kernel.  Launched
// overlapped with the previous kernel of the stream.
cudaError_t launch_decode_tc1(const DecodeParams& p, const CUtensorMap& tmap, bool fp8,
                              int split_group, int sm_count, cudaStream_t stream);

// Stage 2: LSE merge of the split partials into o (bf16) and lse (fp32).
// Every stage-1 kernel leaves, for each (row, head) of a non-empty sequence,
// every split slot either holding a partial or with lse = -inf.
cudaError_t launch_merge(const DecodeParams& p, int R, cudaStream_t stream);

// Cross-shard LSE merge of num_parts bf16 (o, lse) results over disjoint KV
// token shards: records = rows * H, parts at the given element strides.
cudaError_t launch_lse_merge(const void* o_parts, int64_t o_part_stride, const float* lse_parts,
                             int64_t lse_part_stride, int num_parts, int64_t records, int R,
                             void* o, float* lse, cudaStream_t stream);

}  // namespace mla
