// mla_decode_noalloc: mla_decode for callers that cannot allocate device
// memory.
//
// mla_decode needs a split-partials workspace that the caller allocates.  Some
// callers cannot do that: a plugin running inside a host application that
// owns all device memory through its own pool and forbids direct cudaMalloc,
// or a latency-critical serving loop where cudaMalloc / cudaFree are not
// allowed because they can block or implicitly synchronise the device.  This
// entry point gives them the same decode with the workspace taken from a
// fixed-size array that lives in this library's device image.
//
// The array is a file-scope __device__ variable, so every GPU that loads this
// module holds kNoAllocBytes of it until the process exits.  In host code its
// name is only a host-side stand-in, not a device address, so the device
// address is looked up with cudaGetSymbolAddress, once per device and
// context, with that device current, the first time this entry point runs
// there.  The address is cached together with the context's unique id: after
// cudaDeviceReset (or any other end of the primary context) the module is
// loaded again, perhaps at another address, and the next call looks the
// address up again.  Every call shares the array: nothing in it has to start
// at zero (stage 1 writes every partial the merge reads), but two calls whose
// kernels overlap on the GPU (different streams, or different host threads
// on one device) race on it.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "../../include/mla.h"

constexpr size_t kNoAllocBytes = MLA_NOALLOC_WORKSPACE_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoAllocBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
unsigned long long g_ctx_id[kMaxDevices] = {};

// Unique id of the current context (0 when the CUDA driver cannot say; then
// the address is looked up on every call).
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the array on the current device and context.
cudaError_t workspace_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  // (with no context current yet the id is 0; cudaGetSymbolAddress then
  // makes the device's primary context current and loads the module)
  void* p = g_addr[dev];
  const unsigned long long id = current_context_id();
  if (!p || id == 0 || id != g_ctx_id[dev]) {
    e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
    g_ctx_id[dev] = current_context_id();
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" {

mla_status mla_decode_noalloc(const void* q, int64_t q_row_stride,
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
                              void* o, float* lse, int* err_count,
                              void* stream) {
  const size_t need = mla_decode_workspace_bytes(num_rows, num_heads,
                                                 num_kv_splits, kv_lora_rank);
  // Larger requests are refused before anything runs.
  if (need > kNoAllocBytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = nullptr;
  if (need > 0 && workspace_address(&ws) != cudaSuccess) return MLA_ERR_CUDA;
  return mla_decode(q, q_row_stride, q_head_stride, num_rows, num_heads,
                    kv_cache, kv_dtype, num_blocks, block_size, block_stride,
                    kv_lora_rank, rope_dim, block_table, block_table_stride,
                    max_blocks_per_seq, seq_lens, num_seqs, sm_scale, kv_scale,
                    num_kv_splits, ws, ws ? kNoAllocBytes : 0, o, lse,
                    err_count, stream);
}

}  // extern "C"
