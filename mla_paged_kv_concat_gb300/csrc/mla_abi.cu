// C ABI of libmla (declared in include/mla.h): host-side validation, the
// split-count rule, workspace sizing, tensor-map encoding and dispatch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <new>

#include "../../include/mla.h"
#include "kernels.cuh"

namespace {

thread_local char g_last_cuda_error[256] = "";

mla_status cuda_fail(cudaError_t e) {
  snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s",
           cudaGetErrorName(e), cudaGetErrorString(e));
  return MLA_ERR_CUDA;
}

bool valid_kv_dtype(mla_kv_dtype t) {
  return t == MLA_KV_BF16 || t == MLA_KV_FP8_E4M3 || t == MLA_KV_FP8_E5M2;
}

bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// Tensor map over the cache viewed as {R+P (dims), block_size (rows),
// num_blocks}: one box is 64 dims x min(block_size, max_box_rows) rows of one
// block.
// bf16 boxes land 128-byte swizzled (the layout the MMA operand loads read);
// fp8 boxes land unswizzled, 64 bytes per row.
mla_status make_cache_tmap(CUtensorMap* map, const void* cache, bool fp8,
                           int D, int block_size, int num_blocks,
                           int64_t block_stride, int max_box_rows, int box_dims = 64) {
  auto fn = encode_fn();
  if (!fn) {
    snprintf(g_last_cuda_error, sizeof g_last_cuda_error,
             "cuTensorMapEncodeTiled unavailable");
    return MLA_ERR_CUDA;
  }
  const size_t elt = fp8 ? 1 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D),
                        static_cast<cuuint64_t>(block_size),
                        static_cast<cuuint64_t>(num_blocks)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * elt,
                           static_cast<cuuint64_t>(block_stride) * elt};
  cuuint32_t box[3] = {
      static_cast<cuuint32_t>(box_dims),
      static_cast<cuuint32_t>(block_size < max_box_rows ? block_size : max_box_rows), 1};
  // a bf16 box 32 dims wide (64-byte rows) lands with the 64-byte swizzle
  const CUtensorMapSwizzle swz = fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE
                                 : box_dims == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                  : CU_TENSOR_MAP_SWIZZLE_128B;
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map,
                  fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  3, const_cast<void*>(cache), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_cuda_error, sizeof g_last_cuda_error,
             "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

// Tensor map over q viewed as {R+P (dims), H, rows}: one box is 64 dims of
// 16 consecutive heads of one row, 128-byte swizzled (the layout of the
// warp-MMA kernel's Q buffer).  Needs 16-byte strides (validated) and heads a
// multiple of 16; returns false when q does not qualify.
bool make_q_tmap(CUtensorMap* map, const void* q, int D, int H, int rows,
                 int64_t q_head_stride, int64_t q_row_stride) {
  auto fn = encode_fn();
  if (!fn || H % 16 != 0) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(q_head_stride) * 2,
                           static_cast<cuuint64_t>(q_row_stride) * 2};
  cuuint32_t box[3] = {64, 16, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool supported_latent(int R, int P) {
  return (R == 512 || R == 256) && P == 64;
}

bool pow2_block(int bs) {
  return bs == 16 || bs == 32 || bs == 64 || bs == 128 || bs == 256;
}

// The tcgen05 kernels cover bf16 caches with a 512-wide latent (CTA pairs)
// and bf16 or fp8 caches with a 256-wide latent (one CTA per 128 vectors).
bool tc_supported(bool fp8, int R) { return R == 256 || (!fp8 && R == 512); }

}  // namespace

namespace mla {

cudaError_t device_sm_count(int* sms) {
  static std::atomic<int> cache[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidDevice;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  *sms = n;
  return cudaSuccess;
}

}  // namespace mla

extern "C" {

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
  }
  return "MLA_ERR_UNKNOWN";
}

const char* mla_last_cuda_error(void) { return g_last_cuda_error; }

int mla_num_kv_splits(int64_t max_seq_len, int sm_count) {
  int64_t s = (max_seq_len + 511) / 512;
  const int64_t cap = 2 * static_cast<int64_t>(sm_count);
  if (s > cap) s = cap;
  if (s < 1) s = 1;
  return static_cast<int>(s);
}

size_t mla_decode_workspace_bytes(int num_rows, int num_heads,
                                  int num_kv_splits, int kv_lora_rank) {
  if (num_rows <= 0 || num_heads <= 0 || num_kv_splits <= 1 ||
      kv_lora_rank <= 0)
    return 0;
  // rows * heads * splits * (R + 1) * 4, or SIZE_MAX when that does not fit
  // a size_t (no workspace can be that large, so every caller refuses it)
  size_t n = static_cast<size_t>(num_rows);
  const size_t f[4] = {static_cast<size_t>(num_heads), static_cast<size_t>(num_kv_splits),
                       static_cast<size_t>(kv_lora_rank) + 1, sizeof(float)};
  for (size_t x : f)
    if (__builtin_mul_overflow(n, x, &n)) return SIZE_MAX;
  return n;
}

}  // extern "C"

namespace {

// Validation (and, with do_launch, the launch) of the plain cache write.
mla_status cache_write_impl(const void* kv_c, int64_t kv_c_row_stride, const void* k_pe,
                            int64_t k_pe_row_stride, const int64_t* slot_mapping,
                            int num_tokens, int kv_lora_rank, int rope_dim, void* kv_cache,
                            int num_blocks, int block_size, int64_t block_stride,
                            mla_kv_dtype kv_dtype, const float* scale, int* err_count,
                            void* stream, bool do_launch) {
  if (num_tokens < 0 || kv_lora_rank <= 0 || rope_dim <= 0 ||
      num_blocks <= 0 || block_size <= 0 || block_size > 1024)
    return MLA_ERR_INVALID_ARG;
  if (!valid_kv_dtype(kv_dtype)) return MLA_ERR_INVALID_ARG;
  if (!supported_latent(kv_lora_rank, rope_dim)) return MLA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return MLA_OK;
  if (!kv_c || !k_pe || !slot_mapping || !kv_cache) return MLA_ERR_INVALID_ARG;
  const bool fp8 = kv_dtype != MLA_KV_BF16;
  if (fp8 && !scale) return MLA_ERR_INVALID_ARG;
  if (kv_c_row_stride < kv_lora_rank || k_pe_row_stride < rope_dim)
    return MLA_ERR_INVALID_ARG;
  const int D = kv_lora_rank + rope_dim;
  const size_t elt = fp8 ? 1 : 2;
  if (block_stride < static_cast<int64_t>(block_size) * D ||
      (block_stride * elt) % 16 != 0 || !aligned16(kv_cache))
    return MLA_ERR_INVALID_ARG;
  if (!do_launch) return MLA_OK;
  cudaError_t e = mla::launch_cache_write(
      kv_c, kv_c_row_stride, k_pe, k_pe_row_stride, slot_mapping, num_tokens,
      kv_lora_rank, rope_dim, kv_cache, num_blocks, block_size, block_stride,
      static_cast<int>(kv_dtype), scale, err_count, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : cuda_fail(e);
}

// Validation (and, with do_launch, the launch) of the fused write.
mla_status nr_write_impl(const void* kv_c, int64_t kv_c_row_stride, const void* k_pe,
                         int64_t k_pe_row_stride, const int64_t* slot_mapping, int num_tokens,
                         int kv_lora_rank, int rope_dim, void* kv_cache, int num_blocks,
                         int block_size, int64_t block_stride, mla_kv_dtype kv_dtype,
                         const float* scale, const void* gamma, float eps,
                         const int64_t* positions, const float* cos_sin_table,
                         int64_t max_position, void* q_pe, int64_t q_pe_row_stride,
                         int64_t q_pe_head_stride, int q_pe_heads, int* err_count, void* stream,
                         bool do_launch) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || block_size > 1024 ||
      max_position <= 0 || !(eps >= 0.f))
    return MLA_ERR_INVALID_ARG;
  if (!valid_kv_dtype(kv_dtype)) return MLA_ERR_INVALID_ARG;
  if (rope_dim != 64 || (kv_lora_rank != 512 && kv_lora_rank != 256))
    return MLA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return MLA_OK;
  if (!kv_c || !k_pe || !slot_mapping || !kv_cache || !gamma || !positions || !cos_sin_table)
    return MLA_ERR_INVALID_ARG;
  const bool fp8 = kv_dtype != MLA_KV_BF16;
  if (fp8 && !scale) return MLA_ERR_INVALID_ARG;
  if (kv_c_row_stride < kv_lora_rank || k_pe_row_stride < rope_dim ||
      kv_c_row_stride % 8 != 0 || k_pe_row_stride % 8 != 0 || !aligned16(kv_c) ||
      !aligned16(k_pe) || !aligned16(gamma) || !aligned16(cos_sin_table))
    return MLA_ERR_INVALID_ARG;
  const int D = kv_lora_rank + rope_dim;
  const size_t elt = fp8 ? 1 : 2;
  if (block_stride < static_cast<int64_t>(block_size) * D ||
      (block_stride * elt) % 16 != 0 || !aligned16(kv_cache))
    return MLA_ERR_INVALID_ARG;
  if (q_pe != nullptr &&
      (q_pe_heads < 1 || q_pe_heads > 1024 || !aligned16(q_pe) || q_pe_row_stride % 8 != 0 ||
       q_pe_head_stride % 8 != 0 || q_pe_head_stride < rope_dim ||
       q_pe_row_stride < static_cast<int64_t>(q_pe_heads) * rope_dim))
    return MLA_ERR_INVALID_ARG;
  if (!do_launch) return MLA_OK;
  cudaError_t e = mla::launch_norm_rope_cache_write(
      kv_c, kv_c_row_stride, k_pe, k_pe_row_stride, slot_mapping, num_tokens, kv_lora_rank,
      kv_cache, num_blocks, block_size, block_stride, static_cast<int>(kv_dtype), scale, gamma,
      eps, positions,
      cos_sin_table, max_position, q_pe, q_pe_row_stride, q_pe_head_stride,
      q_pe != nullptr ? q_pe_heads : 0, err_count, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : cuda_fail(e);
}

}  // namespace

extern "C" {

mla_status mla_cache_write(const void* kv_c, int64_t kv_c_row_stride,
                           const void* k_pe, int64_t k_pe_row_stride,
                           const int64_t* slot_mapping, int num_tokens,
                           int kv_lora_rank, int rope_dim, void* kv_cache,
                           int num_blocks, int block_size, int64_t block_stride,
                           mla_kv_dtype kv_dtype, const float* scale,
                           int* err_count, void* stream) {
  return cache_write_impl(kv_c, kv_c_row_stride, k_pe, k_pe_row_stride, slot_mapping,
                          num_tokens, kv_lora_rank, rope_dim, kv_cache, num_blocks, block_size,
                          block_stride, kv_dtype, scale, err_count, stream, true);
}

mla_status mla_norm_rope_cache_write(const void* kv_c, int64_t kv_c_row_stride,
                                     const void* k_pe, int64_t k_pe_row_stride,
                                     const int64_t* slot_mapping, int num_tokens,
                                     int kv_lora_rank, int rope_dim, void* kv_cache,
                                     int num_blocks, int block_size,
                                     int64_t block_stride, mla_kv_dtype kv_dtype,
                                     const float* scale, const void* gamma,
                                     float eps, const int64_t* positions,
                                     const float* cos_sin_table,
                                     int64_t max_position, void* q_pe,
                                     int64_t q_pe_row_stride,
                                     int64_t q_pe_head_stride, int q_pe_heads,
                                     int* err_count, void* stream) {
  return nr_write_impl(kv_c, kv_c_row_stride, k_pe, k_pe_row_stride, slot_mapping, num_tokens,
                       kv_lora_rank, rope_dim, kv_cache, num_blocks, block_size, block_stride,
                       kv_dtype, scale, gamma, eps, positions, cos_sin_table, max_position,
                       q_pe, q_pe_row_stride, q_pe_head_stride, q_pe_heads, err_count, stream,
                       true);
}

}  // extern "C"

namespace {

// Validates a decode call and fills `p`; returns MLA_OK or the error.
mla_status prepare_decode(const void* q, int64_t q_row_stride,
                          int64_t q_head_stride, const void* q_pe,
                          int64_t q_pe_row_stride, int64_t q_pe_head_stride,
                          int num_rows, int num_heads,
                          const void* kv_cache, mla_kv_dtype kv_dtype,
                          int num_blocks, int block_size, int64_t block_stride,
                          int kv_lora_rank, int rope_dim,
                          const int32_t* block_table,
                          int64_t block_table_stride, int max_blocks_per_seq,
                          const int32_t* seq_lens, int num_seqs, float sm_scale,
                          const float* kv_scale, int num_kv_splits,
                          void* workspace, size_t workspace_bytes, void* o,
                          float* lse, int* err_count, mla_decode_path path,
                          mla::DecodeParams* p) {
  // ---- shapes
  if (num_rows < 0 || num_seqs < 0 || num_heads < 1 || num_heads > 128 ||
      num_blocks <= 0 || block_size <= 0 || max_blocks_per_seq < 1 ||
      num_kv_splits < 1 || num_kv_splits > 65535)
    return MLA_ERR_INVALID_ARG;
  if (!valid_kv_dtype(kv_dtype)) return MLA_ERR_INVALID_ARG;
  if (path != MLA_PATH_AUTO && path != MLA_PATH_MMA_SYNC &&
      path != MLA_PATH_TCGEN05)
    return MLA_ERR_INVALID_ARG;
  if (!supported_latent(kv_lora_rank, rope_dim) || !pow2_block(block_size))
    return MLA_ERR_UNSUPPORTED;
  if (num_rows == 0) return MLA_OK;
  if (num_seqs == 0 || num_rows % num_seqs != 0 || num_seqs > 65535)
    return MLA_ERR_INVALID_ARG;
  const int D = kv_lora_rank + rope_dim;
  const bool fp8 = kv_dtype != MLA_KV_BF16;
  const size_t elt = fp8 ? 1 : 2;
  // ---- pointers, strides, alignment
  if (!q || !kv_cache || !block_table || !seq_lens || !o || !lse)
    return MLA_ERR_INVALID_ARG;
  if (fp8 && !kv_scale) return MLA_ERR_INVALID_ARG;
  // q alone holds all R+P dims, or q holds [0, R) and q_pe [R, R+P)
  if (!aligned16(q) || q_row_stride % 8 != 0 || q_head_stride % 8 != 0 ||
      q_head_stride < (q_pe ? kv_lora_rank : D) ||
      q_row_stride < static_cast<int64_t>(num_heads) * q_head_stride)
    return MLA_ERR_INVALID_ARG;
  if (q_pe && (!aligned16(q_pe) || q_pe_row_stride % 8 != 0 || q_pe_head_stride % 8 != 0 ||
               q_pe_head_stride < rope_dim ||
               q_pe_row_stride < static_cast<int64_t>(num_heads) * q_pe_head_stride))
    return MLA_ERR_INVALID_ARG;
  if (block_stride < static_cast<int64_t>(block_size) * D ||
      (block_stride * elt) % 16 != 0 || !aligned16(kv_cache))
    return MLA_ERR_INVALID_ARG;
  if (block_table_stride < max_blocks_per_seq) return MLA_ERR_INVALID_ARG;
  if (!aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return MLA_ERR_INVALID_ARG;
  const size_t need = mla_decode_workspace_bytes(num_rows, num_heads,
                                                 num_kv_splits, kv_lora_rank);
  if (need > 0) {
    if (!workspace) return MLA_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return MLA_ERR_INVALID_ARG;
    if (workspace_bytes < need) return MLA_ERR_WORKSPACE_TOO_SMALL;
  }
  // rows_per_seq * heads query vectors per sequence must fit the grid
  if (static_cast<int64_t>(num_rows / num_seqs) * num_heads > (1 << 24))
    return MLA_ERR_UNSUPPORTED;
  if (path == MLA_PATH_TCGEN05 && !tc_supported(fp8, kv_lora_rank))
    return MLA_ERR_UNSUPPORTED;

  p->q = static_cast<const uint16_t*>(q);
  p->q_row_stride = q_row_stride;
  p->q_head_stride = q_head_stride;
  if (q_pe) {
    p->q_pe = static_cast<const uint16_t*>(q_pe);
    p->q_pe_row_stride = q_pe_row_stride;
    p->q_pe_head_stride = q_pe_head_stride;
  } else {
    p->q_pe = p->q + kv_lora_rank;
    p->q_pe_row_stride = q_row_stride;
    p->q_pe_head_stride = q_head_stride;
  }
  p->num_rows = num_rows;
  p->num_heads = num_heads;
  p->rows_per_seq = num_rows / num_seqs;
  p->num_seqs = num_seqs;
  p->block_table = block_table;
  p->bt_stride = block_table_stride;
  p->max_blocks = max_blocks_per_seq;
  p->seq_lens = seq_lens;
  p->block_size = block_size;
  p->num_blocks = num_blocks;
  p->sm_scale = sm_scale;
  p->kv_scale = fp8 ? kv_scale : nullptr;
  p->kv_e5m2 = kv_dtype == MLA_KV_FP8_E5M2 ? 1 : 0;
  p->num_splits = num_kv_splits;
  const size_t n_o = static_cast<size_t>(num_rows) * num_heads * num_kv_splits *
                     kv_lora_rank;
  p->ws_o = need ? static_cast<float*>(workspace) : nullptr;
  p->ws_lse = need ? static_cast<float*>(workspace) + n_o : nullptr;
  p->o = static_cast<uint16_t*>(o);
  p->lse = lse;
  p->err_count = err_count;
  p->q_tma = 0;
  return MLA_OK;
}

// Stage-1 kernel choice: a tcgen05 kernel when forced, or (AUTO) when one
// supports the cache and the sequences have more than 32 query vectors for
// its M = 128 tile; the warp-MMA kernel otherwise.  Measured on GB300
// (32 sequences of 8192 tokens, stage 1 alone): the warp-MMA kernel's time
// steps up with its 16- or 32-vector units (its fragment loads from shared
// memory bound it), the tcgen05 kernels' hardly moves; at 32 vectors the
// warp-MMA kernel is ahead by 3-20 % (R = 512: 80 against 101 us; R = 256:
// 53 against 55 us bf16, 67 against 70 us E4M3), from 40 vectors on the
// tcgen05 kernels lead by 1.4-2.4 x (R = 512 at 48: 102 against 142 us;
// R = 256 at 40: 55 against 110 us bf16, 69 against 139 us E4M3).
bool use_tc(const mla::DecodeParams& p, bool fp8, int R, mla_decode_path path) {
  if (path == MLA_PATH_TCGEN05) return true;
  if (path == MLA_PATH_MMA_SYNC) return false;
  const int64_t nvec = static_cast<int64_t>(p.rows_per_seq) * p.num_heads;
  return tc_supported(fp8, R) && nvec > 32;
}

// Everything stage 1 needs at launch time, computed once per call (or once
// per plan).
struct Stage1 {
  mla::DecodeParams p;
  CUtensorMap tmap;
  CUtensorMap rope_map;  // the 512-wide tcgen05 kernel's 32-dim rope boxes
  mla::QMaps qmaps;
  bool tc, fp8;
  int R, split_group, sm_count;
};

mla_status build_stage1(const mla::DecodeParams& p_in, const void* kv_cache, bool fp8, int R,
                        int block_size, int num_blocks, int64_t block_stride,
                        mla_decode_path path, Stage1* s1) {
  s1->p = p_in;
  s1->fp8 = fp8;
  s1->R = R;
  cudaError_t e = mla::device_sm_count(&s1->sm_count);
  if (e != cudaSuccess) return cuda_fail(e);
  s1->tc = use_tc(s1->p, fp8, R, path);
  mla_status st = make_cache_tmap(&s1->tmap, kv_cache, fp8, R + 64, block_size, num_blocks,
                                  block_stride, 64);
  if (st != MLA_OK) return st;
  memset(&s1->rope_map, 0, sizeof s1->rope_map);
  if (s1->tc && R == 512) {
    st = make_cache_tmap(&s1->rope_map, kv_cache, fp8, R + 64, block_size, num_blocks,
                         block_stride, 64, 32);
    if (st != MLA_OK) return st;
  }
  memset(&s1->qmaps, 0, sizeof s1->qmaps);
  s1->p.q_tma = 0;
  if (!s1->tc) {
    const mla::DecodeParams& p = s1->p;
    s1->p.q_tma = make_q_tmap(&s1->qmaps.nope, p.q, R, p.num_heads, p.num_rows,
                              p.q_head_stride, p.q_row_stride) &&
                          make_q_tmap(&s1->qmaps.pe, p.q_pe, 64, p.num_heads, p.num_rows,
                                      p.q_pe_head_stride, p.q_pe_row_stride)
                      ? 1
                      : 0;
  }
  s1->split_group =
      s1->tc ? mla::tc_split_group(s1->p, s1->sm_count, R == 256 ? 1 : 2) : 1;
  return MLA_OK;
}

mla_status launch_stage1(const Stage1& s1, cudaStream_t s) {
  cudaError_t e;
  if (!s1.tc)
    e = mla::launch_decode_mma(s1.p, s1.tmap, s1.qmaps, s1.R, s1.fp8, s1.sm_count, s);
  else if (s1.R == 256)
    e = mla::launch_decode_tc1(s1.p, s1.tmap, s1.fp8, s1.split_group, s1.sm_count, s);
  else
    e = mla::launch_decode_tc(s1.p, s1.tmap, s1.rope_map, s1.split_group, s1.sm_count, s);
  return e == cudaSuccess ? MLA_OK : cuda_fail(e);
}

mla_status run_stage1(const mla::DecodeParams& p_in, const void* kv_cache,
                      bool fp8, int R, int block_size, int num_blocks,
                      int64_t block_stride, mla_decode_path path,
                      cudaStream_t s) {
  Stage1 s1;
  mla_status st =
      build_stage1(p_in, kv_cache, fp8, R, block_size, num_blocks, block_stride, path, &s1);
  if (st != MLA_OK) return st;
  return launch_stage1(s1, s);
}

}  // namespace

extern "C" {

mla_status mla_decode_splitkv(const void* q, int64_t q_row_stride,
                              int64_t q_head_stride, int num_rows,
                              int num_heads, const void* kv_cache,
                              mla_kv_dtype kv_dtype, int num_blocks,
                              int block_size, int64_t block_stride,
                              int kv_lora_rank, int rope_dim,
                              const int32_t* block_table,
                              int64_t block_table_stride,
                              int max_blocks_per_seq, const int32_t* seq_lens,
                              int num_seqs, float sm_scale,
                              const float* kv_scale, int num_kv_splits,
                              void* workspace, size_t workspace_bytes, void* o,
                              float* lse, int* err_count, void* stream,
                              mla_decode_path path) {
  mla::DecodeParams p;
  mla_status st = prepare_decode(
      q, q_row_stride, q_head_stride, nullptr, 0, 0, num_rows, num_heads, kv_cache, kv_dtype,
      num_blocks, block_size, block_stride, kv_lora_rank, rope_dim,
      block_table, block_table_stride, max_blocks_per_seq, seq_lens, num_seqs,
      sm_scale, kv_scale, num_kv_splits, workspace, workspace_bytes, o, lse,
      err_count, path, &p);
  if (st != MLA_OK || num_rows == 0) return st;
  return run_stage1(p, kv_cache, kv_dtype != MLA_KV_BF16, kv_lora_rank,
                    block_size, num_blocks, block_stride, path,
                    static_cast<cudaStream_t>(stream));
}

mla_status mla_decode_merge(int num_rows, int num_heads, int kv_lora_rank,
                            const int32_t* seq_lens, int num_seqs,
                            int block_size, int max_blocks_per_seq,
                            int num_kv_splits, const void* workspace,
                            size_t workspace_bytes, void* o, float* lse,
                            void* stream) {
  if (num_rows < 0 || num_heads < 1 || num_heads > 128 || num_seqs < 0 ||
      block_size <= 0 || max_blocks_per_seq < 1 || num_kv_splits < 1 ||
      num_kv_splits > 65535)
    return MLA_ERR_INVALID_ARG;
  if (kv_lora_rank != 512 && kv_lora_rank != 256) return MLA_ERR_UNSUPPORTED;
  if (num_rows == 0 || num_kv_splits == 1) return MLA_OK;
  if (num_seqs == 0 || num_rows % num_seqs != 0) return MLA_ERR_INVALID_ARG;
  if (!seq_lens || !workspace || !o || !lse || !aligned16(workspace) ||
      !aligned16(o) || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return MLA_ERR_INVALID_ARG;
  const size_t need = mla_decode_workspace_bytes(num_rows, num_heads,
                                                 num_kv_splits, kv_lora_rank);
  if (workspace_bytes < need) return MLA_ERR_WORKSPACE_TOO_SMALL;
  mla::DecodeParams p = {};
  p.num_rows = num_rows;
  p.num_heads = num_heads;
  p.rows_per_seq = num_rows / num_seqs;
  p.num_seqs = num_seqs;
  p.seq_lens = seq_lens;
  p.block_size = block_size;
  p.max_blocks = max_blocks_per_seq;
  p.num_splits = num_kv_splits;
  const size_t n_o = static_cast<size_t>(num_rows) * num_heads * num_kv_splits *
                     kv_lora_rank;
  p.ws_o = static_cast<float*>(const_cast<void*>(workspace));
  p.ws_lse = p.ws_o + n_o;
  p.o = static_cast<uint16_t*>(o);
  p.lse = lse;
  cudaError_t e = mla::launch_merge(p, kv_lora_rank, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : cuda_fail(e);
}

mla_status mla_lse_merge(const void* o_parts, int64_t o_part_stride,
                         const float* lse_parts, int64_t lse_part_stride,
                         int num_parts, int num_rows, int num_heads,
                         int kv_lora_rank, void* o, float* lse, void* stream) {
  if (num_parts < 1 || num_parts > 1024 || num_rows < 0 || num_heads < 1 || num_heads > 128)
    return MLA_ERR_INVALID_ARG;
  if (kv_lora_rank != 512 && kv_lora_rank != 256) return MLA_ERR_UNSUPPORTED;
  if (num_rows == 0) return MLA_OK;
  const int64_t records = static_cast<int64_t>(num_rows) * num_heads;
  if (!o_parts || !lse_parts || !o || !lse || !aligned16(o_parts) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse_parts) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return MLA_ERR_INVALID_ARG;
  if (o_part_stride % 8 != 0 || o_part_stride < records * kv_lora_rank ||
      lse_part_stride < records)
    return MLA_ERR_INVALID_ARG;
  cudaError_t e = mla::launch_lse_merge(o_parts, o_part_stride, lse_parts, lse_part_stride,
                                        num_parts, records, kv_lora_rank, o, lse,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MLA_OK : cuda_fail(e);
}

mla_status mla_decode_ex(const void* q, int64_t q_row_stride,
                         int64_t q_head_stride, int num_rows, int num_heads,
                         const void* kv_cache, mla_kv_dtype kv_dtype,
                         int num_blocks, int block_size, int64_t block_stride,
                         int kv_lora_rank, int rope_dim,
                         const int32_t* block_table,
                         int64_t block_table_stride, int max_blocks_per_seq,
                         const int32_t* seq_lens, int num_seqs, float sm_scale,
                         const float* kv_scale, int num_kv_splits,
                         void* workspace, size_t workspace_bytes, void* o,
                         float* lse, int* err_count, void* stream,
                         mla_decode_path path) {
  mla::DecodeParams p;
  mla_status st = prepare_decode(
      q, q_row_stride, q_head_stride, nullptr, 0, 0, num_rows, num_heads, kv_cache, kv_dtype,
      num_blocks, block_size, block_stride, kv_lora_rank, rope_dim,
      block_table, block_table_stride, max_blocks_per_seq, seq_lens, num_seqs,
      sm_scale, kv_scale, num_kv_splits, workspace, workspace_bytes, o, lse,
      err_count, path, &p);
  if (st != MLA_OK || num_rows == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = run_stage1(p, kv_cache, kv_dtype != MLA_KV_BF16, kv_lora_rank,
                  block_size, num_blocks, block_stride, path, s);
  if (st != MLA_OK) return st;
  if (num_kv_splits > 1) {
    cudaError_t e = mla::launch_merge(p, kv_lora_rank, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return MLA_OK;
}

mla_status mla_decode(const void* q, int64_t q_row_stride,
                      int64_t q_head_stride, int num_rows, int num_heads,
                      const void* kv_cache, mla_kv_dtype kv_dtype,
                      int num_blocks, int block_size, int64_t block_stride,
                      int kv_lora_rank, int rope_dim,
                      const int32_t* block_table, int64_t block_table_stride,
                      int max_blocks_per_seq, const int32_t* seq_lens,
                      int num_seqs, float sm_scale, const float* kv_scale,
                      int num_kv_splits, void* workspace,
                      size_t workspace_bytes, void* o, float* lse,
                      int* err_count, void* stream) {
  return mla_decode_ex(q, q_row_stride, q_head_stride, num_rows, num_heads,
                       kv_cache, kv_dtype, num_blocks, block_size, block_stride,
                       kv_lora_rank, rope_dim, block_table, block_table_stride,
                       max_blocks_per_seq, seq_lens, num_seqs, sm_scale,
                       kv_scale, num_kv_splits, workspace, workspace_bytes, o,
                       lse, err_count, stream, MLA_PATH_AUTO);
}

}  // extern "C"

// ------------------------------------------------------------------ plans

struct mla_decode_plan {
  mla_decode_desc d;
  bool has_stage1;
  Stage1 s1;
};

namespace {

// The plan's write: plain or fused, validated only (do_launch false) or run.
mla_status plan_write(const mla_decode_desc& d, void* stream, bool do_launch) {
  if (d.num_tokens == 0) return MLA_OK;
  if (!d.gamma)
    return cache_write_impl(d.kv_c, d.kv_c_row_stride, d.k_pe, d.k_pe_row_stride,
                            d.slot_mapping, d.num_tokens, d.kv_lora_rank, d.rope_dim,
                            d.kv_cache, d.num_blocks, d.block_size, d.block_stride, d.kv_dtype,
                            d.kv_scale, d.err_count, stream, do_launch);
  void* qr = nullptr;
  int64_t qr_rs = 0, qr_hs = 0;
  if (d.rotate_q) {
    if (d.q_pe) {
      qr = const_cast<void*>(d.q_pe);
      qr_rs = d.q_pe_row_stride;
      qr_hs = d.q_pe_head_stride;
    } else {
      qr = static_cast<uint16_t*>(const_cast<void*>(d.q)) + d.kv_lora_rank;
      qr_rs = d.q_row_stride;
      qr_hs = d.q_head_stride;
    }
  }
  return nr_write_impl(d.kv_c, d.kv_c_row_stride, d.k_pe, d.k_pe_row_stride, d.slot_mapping,
                       d.num_tokens, d.kv_lora_rank, d.rope_dim, d.kv_cache, d.num_blocks,
                       d.block_size, d.block_stride, d.kv_dtype, d.kv_scale, d.gamma, d.eps,
                       d.positions, d.cos_sin_table, d.max_position, qr, qr_rs, qr_hs,
                       d.num_heads, d.err_count, stream, do_launch);
}

}  // namespace

extern "C" {

mla_status mla_plan_create(const mla_decode_desc* desc, mla_decode_plan** plan) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  *plan = nullptr;
  if (!desc) return MLA_ERR_INVALID_ARG;
  const mla_decode_desc& d = *desc;
  if (d.num_tokens < 0) return MLA_ERR_INVALID_ARG;
  if (d.num_tokens > 0 && d.gamma && d.rotate_q &&
      (d.num_tokens != d.num_rows || d.q == nullptr))
    return MLA_ERR_INVALID_ARG;
  mla_status st = plan_write(d, nullptr, false);
  if (st != MLA_OK) return st;
  mla::DecodeParams p;
  st = prepare_decode(d.q, d.q_row_stride, d.q_head_stride, d.q_pe, d.q_pe_row_stride,
                      d.q_pe_head_stride, d.num_rows, d.num_heads, d.kv_cache, d.kv_dtype,
                      d.num_blocks, d.block_size, d.block_stride, d.kv_lora_rank, d.rope_dim,
                      d.block_table, d.block_table_stride, d.max_blocks_per_seq, d.seq_lens,
                      d.num_seqs, d.sm_scale, d.kv_scale, d.num_kv_splits, d.workspace,
                      d.workspace_bytes, d.o, d.lse, d.err_count, d.path, &p);
  if (st != MLA_OK) return st;
  mla_decode_plan* pl = new (std::nothrow) mla_decode_plan;
  if (!pl) return MLA_ERR_INVALID_ARG;
  pl->d = d;
  pl->has_stage1 = d.num_rows > 0;
  if (pl->has_stage1) {
    st = build_stage1(p, d.kv_cache, d.kv_dtype != MLA_KV_BF16, d.kv_lora_rank,
                      d.block_size, d.num_blocks, d.block_stride, d.path, &pl->s1);
    if (st != MLA_OK) {
      delete pl;
      return st;
    }
  }
  *plan = pl;
  return MLA_OK;
}

mla_status mla_plan_run(const mla_decode_plan* plan, void* stream) {
  if (!plan) return MLA_ERR_INVALID_ARG;
  mla_status st = plan_write(plan->d, stream, true);
  if (st != MLA_OK || !plan->has_stage1) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = launch_stage1(plan->s1, s);
  if (st != MLA_OK) return st;
  if (plan->d.num_kv_splits > 1) {
    cudaError_t e = mla::launch_merge(plan->s1.p, plan->d.kv_lora_rank, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return MLA_OK;
}

void mla_plan_destroy(mla_decode_plan* plan) { delete plan; }

}  // extern "C"
