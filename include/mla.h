/*
 * mla.h - C ABI of libmla: MLA decode over a paged latent KV cache on GB300
 * (sm_103a).
 *
 * The library implements the decode hot path of multi-head latent attention
 * (MLA) as described on the vLLM pages it restates -- the cache write of a
 * step's new tokens (plain, or fused with the RMSNorm of the latent and the
 * rotary embedding), the split-KV attention pass over the paged latent cache
 * and the log-sum-exp merge -- plus the cross-shard merge of decode context
 * parallelism and prepared, CUDA-graph-safe plans of a whole step:
 *
 *   [diff] "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs" ("fix TP"),
 *          a unified diff of vLLM, cited by file section;
 *   [note] "Triton and MLA: portable attention and multi-head latent
 *          attention" (vLLM v0.25.1 architecture note), cited by section;
 *   [api]  "vllm.v1.attention.backends.mla.triton_mla" (API reference),
 *          TritonMLAMetadataBuilder.
 *
 * Conventions shared by every entry point:
 *   - Every data pointer is DEVICE memory owned by the caller.  The library
 *     keeps no pointer after a call returns and allocates no device memory.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL is the legacy default stream).  No call reads device memory on
 *     the host or synchronises the stream.
 *   - Arguments are validated on the host before any launch.  A failed check
 *     returns a non-zero mla_status and launches nothing.  A launch failure
 *     returns MLA_ERR_CUDA.  Device code never traps: an out-of-range slot or
 *     block id is skipped (slot) or read as zeros (block id) and counted in
 *     the optional device counter `err_count`.
 *   - Strides are in ELEMENTS of the tensor they describe.
 */
#ifndef MLA_GB300_MLA_H_
#define MLA_GB300_MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,         /* null pointer, bad shape/stride/alignment */
  MLA_ERR_UNSUPPORTED = 2,         /* valid but not implemented combination   */
  MLA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes below the required size */
  MLA_ERR_CUDA = 4                 /* a CUDA runtime call or launch failed     */
} mla_status;

/* Element type of the cache, the pages' kv_cache_dtype strings ([diff]
 * csrc/cache_kernels.cu, concat_and_cache_mla: DISPATCH_BY_KV_CACHE_DTYPE):
 * "auto" is MLA_KV_BF16 (the model's bf16 values unchanged), "fp8" /
 * "fp8_e4m3" MLA_KV_FP8_E4M3 and "fp8_e5m2" MLA_KV_FP8_E5M2 (OCP formats,
 * x / scale rounded to nearest even, finite overflow saturated). */
typedef enum {
  MLA_KV_BF16 = 0,
  MLA_KV_FP8_E4M3 = 1,
  MLA_KV_FP8_E5M2 = 2
} mla_kv_dtype;

/* Which stage-1 kernel mla_decode_ex runs.  AUTO picks the fastest kernel
 * that supports the shape; the others force one (for tests and benchmarks);
 * a forced kernel that does not support the shape returns
 * MLA_ERR_UNSUPPORTED. */
typedef enum {
  MLA_PATH_AUTO = 0,
  MLA_PATH_MMA_SYNC = 1, /* warp-level bf16 MMA: every cache type and shape   */
  MLA_PATH_TCGEN05 = 2   /* tcgen05/TMEM, 128 query vectors per 2-CTA cluster
                            (bf16 cache, kv_lora_rank 512) or per CTA
                            (kv_lora_rank 256, bf16 or fp8 cache); AUTO takes
                            it above 32 query vectors (rows x heads) per
                            sequence */
} mla_decode_path;

/*
 * mla_cache_write - write new tokens' latent rows into the paged cache.
 *
 * Restates [diff] csrc/cache_kernels.cu, concat_and_cache_mla_kernel and its
 * host wrapper concat_and_cache_mla (declared in csrc/cache.h).
 *
 * For each token t < num_tokens with s = slot_mapping[t]:
 *   s < 0               padded token (PAD_SLOT_ID = -1): nothing is written;
 *   s >= num_blocks*bs  skipped and counted in *err_count;
 *   otherwise           row (s % bs) of block (s / bs) receives
 *                       [kv_c[t, 0:R] | k_pe[t, 0:P]].
 * bf16 cache: the bf16 bits are stored unchanged.  fp8 cache: each element
 * is E4M3(x / *scale) (MLA_KV_FP8_E4M3) or E5M2(x / *scale)
 * (MLA_KV_FP8_E5M2), x / *scale an IEEE fp32 division, rounded to nearest
 * even with finite overflow saturated to +-448 (OCP E4M3, "e4m3fn") or
 * +-57344 (OCP E5M2).
 *
 *   kv_c            bf16 [>= num_tokens, kv_lora_rank], row stride
 *                   kv_c_row_stride (elements), unit column stride.
 *   k_pe            bf16 [>= num_tokens, rope_dim], row stride
 *                   k_pe_row_stride; may be a column slice of a wider tensor.
 *   slot_mapping    int64 [num_tokens].  num_tokens may be smaller than the
 *                   rows of kv_c/k_pe (CUDA-graph padding, as in the pages).
 *   kv_lora_rank R  512 or 256.  rope_dim P: 64.
 *   kv_cache        [num_blocks, block_size, R+P] of bf16 or fp8 bytes, the
 *                   start of block b at element b * block_stride
 *                   (block_stride >= block_size*(R+P); block_stride*elt a
 *                   multiple of 16 bytes; kv_cache 16-byte aligned).
 *   block_size      1 .. 1024.
 *   scale           device float; read only for the fp8 formats.
 *   err_count       device int, may be NULL; incremented per skipped slot.
 * Duplicate slots in one call race (unspecified winner), as in the pages.
 */
mla_status mla_cache_write(const void* kv_c, int64_t kv_c_row_stride,
                           const void* k_pe, int64_t k_pe_row_stride,
                           const int64_t* slot_mapping, int num_tokens,
                           int kv_lora_rank, int rope_dim, void* kv_cache,
                           int num_blocks, int block_size, int64_t block_stride,
                           mla_kv_dtype kv_dtype, const float* scale,
                           int* err_count, void* stream);

/*
 * mla_norm_rope_cache_write - the cache write fused with the two steps the
 * model runs just before it: RMSNorm of the latent and the rotary embedding
 * of k_pe (and, optionally, of q_pe).
 *
 * Restates [diff] vllm/model_executor/models/deepseek_v2.py
 * (kv_a_layernorm = RMSNorm(kv_lora_rank, eps=rms_norm_eps) on kv_c;
 * rotary_emb = get_rope(qk_rope_head_dim, ..., rope_type 'deepseek_yarn',
 * is_neox_style=False)) and the MLA common forward (q_pe, k_pe rotated by
 * input position, then concat_and_cache_mla).  The pages print neither body;
 * the readings taken: for each token t < num_tokens with p = positions[t],
 *   kv_n[d]   = bf16( kv_c[t, d] / sqrt(mean_d kv_c[t, d]^2 + eps) * gamma[d] )
 *   k_r[2i]   = bf16( k_pe[t, 2i] c_i - k_pe[t, 2i+1] s_i )
 *   k_r[2i+1] = bf16( k_pe[t, 2i+1] c_i + k_pe[t, 2i] s_i ),  i < P/2,
 * with c_i = table[p][i], s_i = table[p][P/2 + i] (any YaRN frequencies and
 * magnitude scale live in the table), computed in fp32 and rounded once to
 * bf16; then [kv_n | k_r] is stored at slot_mapping[t] exactly as
 * mla_cache_write stores [kv_c | k_pe] (bf16 copy or fp8(x / *scale)).
 * With q_pe != NULL every head of q_pe[t] is rotated the same way, in place.
 * kv_c and k_pe are not modified.
 *
 * Arguments as mla_cache_write, plus:
 *   gamma          device bf16 [kv_lora_rank], the RMSNorm weight; 16-byte
 *                  aligned.
 *   eps            RMSNorm epsilon (>= 0).
 *   positions      device int64 [num_tokens].
 *   cos_sin_table  device fp32 [max_position][rope_dim]: cos | sin; 16-byte
 *                  aligned.
 *   q_pe           device bf16 [num_tokens][q_pe_heads][rope_dim] at row /
 *                  head strides q_pe_row_stride / q_pe_head_stride (elements,
 *                  multiples of 8; may be the rope columns of q), or NULL.
 *                  16-byte aligned.
 * Restrictions: rope_dim == 64; kv_lora_rank 512 or 256; kv_c, k_pe 16-byte
 * aligned with row strides multiples of 8 (else MLA_ERR_INVALID_ARG).
 * A token with a position outside [0, max_position) is skipped entirely
 * (nothing written, q_pe untouched) and counted in *err_count, as is a slot
 * >= num_blocks * block_size.  A padded token (slot -1) writes nothing but
 * its q_pe is still rotated.
 */
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
                                     int* err_count, void* stream);

/*
 * mla_num_kv_splits - the split-count rule.
 *
 * [note] Key files, _compute_num_kv_splits: the KV split count is taken from
 * max_seq_len / 512 and capped at sm_count * 2.  Returns
 * min(ceil(max_seq_len / 512), 2 * sm_count), at least 1.  Batch-invariant
 * (deterministic) callers pass num_kv_splits = 1 to mla_decode instead
 * ([note] Data flow, VLLM_BATCH_INVARIANT).
 */
int mla_num_kv_splits(int64_t max_seq_len, int sm_count);

/*
 * mla_decode_workspace_bytes - bytes of fp32 split partials mla_decode needs:
 * num_rows * num_heads * num_kv_splits * (kv_lora_rank + 1) * 4, or 0 when
 * num_kv_splits == 1 (the single pass writes o and lse directly).  Same size
 * as the pages' attn_logits [B, H, S, R+1] fp32 buffer ([note] Data flow;
 * [api] _reserve_attn_logits_workspace), laid out as o partials
 * [rows][S][H][R] followed by lse partials [rows][S][H].  Returns SIZE_MAX
 * when the product does not fit a size_t; every decode entry point then
 * refuses the call with MLA_ERR_WORKSPACE_TOO_SMALL.
 */
size_t mla_decode_workspace_bytes(int num_rows, int num_heads,
                                  int num_kv_splits, int kv_lora_rank);

/*
 * mla_decode - split-KV MLA decode (stage 1) plus the LSE merge (stage 2).
 *
 * Restates [diff] vllm/attention/ops/triton_decode_attention.py
 * (decode_attention_fwd -> _fwd_grouped_kernel_stage1 -> _fwd_kernel_stage2)
 * and [note] Data flow (TritonMLAImpl.forward_mqa): MLA decode is MQA over
 * the latent cache; every head attends to the same cached rows.
 *
 * For row r (sequence b = r / (num_rows / num_seqs)), head h, L = seq_lens[b]:
 *   K_j = cache row of token j (page block_table[b][j / bs], row j % bs),
 *         dequantised as fp8 value * *kv_scale for an fp8 cache;
 *   s_j = sm_scale * sum_{d < R+P} q[r,h,d] K_j[d];
 *   o[r,h,:] = sum_j softmax(s)_j K_j[0:R]   (V = the kv_c part);
 *   lse[r,h] = ln sum_j exp(s_j)              (natural log, fp32).
 * L = 0 gives o = 0 and lse = -inf.  Rows of one sequence are its flattened
 * non-causal query rows ([api] TritonMLAMetadataBuilder): no causal mask.
 *
 *   q               bf16 [num_rows, num_heads, R+P]: row stride q_row_stride,
 *                   head stride q_head_stride, unit last stride; q and both
 *                   strides 16-byte aligned.  ([diff] _forward_decode builds
 *                   it as cat(q_nope, q_pe).)
 *   num_heads       1 .. 128.
 *   kv_cache        as in mla_cache_write; block_size one of 16, 32, 64,
 *                   128, 256.
 *   kv_lora_rank R  512 or 256; rope_dim P = 64 (head sizes 576 and 320,
 *                   [note] Boundaries: get_supported_head_sizes).
 *   block_table     int32 [num_seqs, >= max_blocks_per_seq], row stride
 *                   block_table_stride.  Entries past a sequence's last
 *                   page are never read.
 *   seq_lens        int32 [num_seqs].  Values are clamped to
 *                   [0, max_blocks_per_seq * block_size]; a clamp counts
 *                   one error.
 *   num_seqs        divides num_rows.
 *   sm_scale        softmax scale applied to q.k.
 *   kv_scale        device float, read only for an fp8 cache (the same scale
 *                   for K and V, [note] Data flow: k_scale = v_scale).
 *                   An fp8 cache needs a bf16 q ([note] Boundaries).
 *   num_kv_splits   >= 1.  The pages' partition (split s of
 *                   ceil(L / S) tokens) is an upper bound: the kernel rounds
 *                   each split up to whole 64-token tiles, so it may use
 *                   fewer, longer splits.  1 = one sequential pass per row in
 *                   a fixed order, bitwise deterministic and batch-invariant.
 *   workspace       device buffer of >= mla_decode_workspace_bytes(...)
 *                   bytes, 16-byte aligned; may be NULL when
 *                   num_kv_splits == 1.
 *   o               bf16 [num_rows, num_heads, R], contiguous.
 *   lse             fp32 [num_rows, num_heads], contiguous.
 *   err_count       device int, may be NULL: counts out-of-range block ids
 *                   and clamped seq_lens; +(1 << 20) if a pipeline wait
 *                   timed out (the kernel then returns early).
 * Every mode is run-to-run deterministic (no floating-point atomics).
 */
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
                      int* err_count, void* stream);

/* mla_decode with an explicit choice of stage-1 kernel (see mla_decode_path).
 * All arguments otherwise as mla_decode. */
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
                         mla_decode_path path);

/*
 * mla_decode_splitkv - stage 1 alone: the split-KV pass of mla_decode
 * ([diff] triton_decode_attention.py, _decode_grouped_att_m_fwd launching
 * _fwd_grouped_kernel_stage1).  With num_kv_splits == 1 it writes o and lse
 * directly; otherwise it writes the split partials into `workspace` and
 * mla_decode_merge must follow on the same stream.  Arguments as
 * mla_decode_ex.
 */
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
                              mla_decode_path path);

/*
 * mla_decode_merge - stage 2 alone: merge the split partials that
 * mla_decode_splitkv left in `workspace` into o (bf16) and lse (fp32)
 * ([diff] triton_decode_attention.py, _decode_softmax_reducev_fwd launching
 * _fwd_kernel_stage2).  seq_lens, block_size, max_blocks_per_seq and
 * num_kv_splits must be the values stage 1 was given: the split partition is
 * recomputed from them.  A no-op returning MLA_OK when num_kv_splits == 1.
 */
mla_status mla_decode_merge(int num_rows, int num_heads, int kv_lora_rank,
                            const int32_t* seq_lens, int num_seqs,
                            int block_size, int max_blocks_per_seq,
                            int num_kv_splits, const void* workspace,
                            size_t workspace_bytes, void* o, float* lse,
                            void* stream);

/* Size of the built-in workspace array of mla_decode_noalloc: 32 MiB. */
#define MLA_NOALLOC_WORKSPACE_BYTES ((size_t)32 << 20)

/*
 * mla_decode_noalloc - mla_decode without a caller-supplied workspace.
 *
 * The pages have no counterpart of this entry point; it exists for callers
 * that cannot allocate device memory themselves: a plugin inside a host
 * application that owns every device allocation through its own pool and
 * forbids direct cudaMalloc, or a latency-critical loop that may not call
 * cudaMalloc / cudaFree because they can block or synchronise the device.
 *
 * Same arguments and results as mla_decode, minus workspace and
 * workspace_bytes.  The split partials go to a fixed array of
 * MLA_NOALLOC_WORKSPACE_BYTES bytes inside the library's device image, which
 * every GPU that loads the library holds until the process exits.  The call
 * itself allocates nothing.  A call whose partials would not fit
 * (mla_decode_workspace_bytes(...) > MLA_NOALLOC_WORKSPACE_BYTES) returns
 * MLA_ERR_WORKSPACE_TOO_SMALL and launches nothing; use fewer splits or
 * mla_decode with your own workspace.
 *
 * The first call on a device (with that device current) looks up the
 * array's device address; make that first call before any stream capture.
 * The address is kept with the context's id: after cudaDeviceReset the next
 * call looks it up again (again, before any capture).
 * All calls share the one array: calls whose kernels overlap on the GPU
 * (other streams, other host threads on the same device) race on it and
 * must be serialised by the caller.
 */
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
                              void* stream);

/*
 * mla_lse_merge - cross-shard LSE merge (decode context parallelism).
 *
 * With decode context parallelism each rank holds a disjoint shard of every
 * sequence's KV tokens, decodes the same query vectors over its shard, and
 * the per-shard (o, lse) pairs are combined through their log-sum-exp
 * ([note] Design motivation: decode returns lse for the cross-shard merge,
 * cp_lse_ag_out_rs; [api] decode with DCP all-gathers the q heads).  The
 * arithmetic is the split merge's ([diff] triton_decode_attention.py,
 * _fwd_kernel_stage2): for each (row, head) record, M = max over the parts
 * of lse_g, o = sum e^{lse_g - M} o_g / sum e^{lse_g - M},
 * lse = M + ln sum e^{lse_g - M}.  Parts with lse_g = -inf hold no tokens
 * and are skipped; a record whose parts are all empty gets o = 0 and
 * lse = -inf.  This call is the combine step alone, after the (o, lse) of
 * every shard has been gathered onto this GPU; the exchange between ranks is
 * the caller's.
 *
 * o_parts    device, bf16 [num_parts][num_rows][num_heads][kv_lora_rank]:
 *            part g starts at element g * o_part_stride (a multiple of 8,
 *            >= num_rows * num_heads * kv_lora_rank); rows and heads dense.
 *            16-byte aligned.  Read only.
 * lse_parts  device, fp32 [num_parts][num_rows][num_heads], natural log:
 *            part g starts at element g * lse_part_stride
 *            (>= num_rows * num_heads).  Read only.
 * num_parts  1 .. 1024.  num_rows >= 0, num_heads 1 .. 128.
 * kv_lora_rank  512 or 256 (else MLA_ERR_UNSUPPORTED).
 * o          device, bf16 [num_rows][num_heads][kv_lora_rank], 16-byte
 *            aligned; lse  device, fp32 [num_rows][num_heads].  Written; they
 *            must not overlap the inputs.
 * stream     cudaStream_t (NULL: the legacy default stream).
 *
 * Errors: MLA_ERR_INVALID_ARG for null pointers, misalignment or bad sizes
 * (nothing launched); MLA_ERR_CUDA if the launch fails.  num_rows == 0 is a
 * no-op returning MLA_OK.  Asynchronous: results are ready when the stream
 * reaches the kernel.
 */
mla_status mla_lse_merge(const void* o_parts, int64_t o_part_stride,
                         const float* lse_parts, int64_t lse_part_stride,
                         int num_parts, int num_rows, int num_heads,
                         int kv_lora_rank, void* o, float* lse, void* stream);

/*
 * Decode plans: the validation, kernel choice and tensor-map encoding of a
 * decode step done once, for steps that repeat with the same buffers.
 *
 * The pages run decode under CUDA graphs: the graph is captured once over
 * fixed device buffers (slot_mapping, seq_lens, block_tables) and replayed
 * after new values are copied into them ([diff] triton_mla.py,
 * TritonMLAState: graph_capture, get_graph_input_buffers,
 * prepare_graph_input_buffers).  A plan is that contract for this library:
 * mla_plan_create checks every argument and prepares the launches;
 * mla_plan_run only launches kernels (no allocation, no synchronisation, no
 * host-side validation), so it may be captured into a CUDA graph and
 * replayed.  Between runs the CONTENTS of every buffer may change (seq_lens
 * up to max_blocks_per_seq * block_size, block ids, q, the new tokens), the
 * pointers, shapes and num_kv_splits may not.  The stage-1 schedule is
 * computed on the device from seq_lens at every run.
 *
 * The query may be given as one tensor holding all R+P dims (q_pe == NULL)
 * or as the pair (q_nope, q_pe) without a concatenation: the pages' decode
 * accepts q as a tensor or as a (q_nope, q_pe) tuple, which it concatenates
 * ([note] Data flow, forward_mqa; this library reads both parts in
 * place).
 *
 * A plan may include the cache write of the step's new tokens, plain
 * (mla_cache_write) or fused with RMSNorm and the rotary embedding
 * (gamma != NULL: mla_norm_rope_cache_write); with rotate_q != 0 the fused
 * write also rotates the rope dims of the query in place (q_pe, or dims
 * [R, R+P) of q), which needs num_tokens == num_rows (one new token per
 * query row, in the same order).
 *
 * Every field has the meaning, layout and constraints of the argument of
 * the same name in mla_decode_ex, mla_cache_write and
 * mla_norm_rope_cache_write.  num_tokens == 0 means no write.  The plan
 * copies the description; the caller keeps the buffers alive for as long as
 * the plan runs.
 */
typedef struct {
  /* query: dims [0, R) (all R+P when q_pe is NULL) */
  const void* q;
  int64_t q_row_stride, q_head_stride;
  const void* q_pe; /* dims [R, R+P), or NULL */
  int64_t q_pe_row_stride, q_pe_head_stride;
  int num_rows, num_heads;
  /* cache */
  void* kv_cache;
  mla_kv_dtype kv_dtype;
  int num_blocks, block_size;
  int64_t block_stride;
  int kv_lora_rank, rope_dim;
  const float* kv_scale;
  /* batch */
  const int32_t* block_table;
  int64_t block_table_stride;
  int max_blocks_per_seq;
  const int32_t* seq_lens;
  int num_seqs;
  float sm_scale;
  int num_kv_splits;
  void* workspace;
  size_t workspace_bytes;
  void* o;
  float* lse;
  int* err_count;
  mla_decode_path path;
  /* cache write before stage 1 (num_tokens == 0: none) */
  const void* kv_c;
  int64_t kv_c_row_stride;
  const void* k_pe;
  int64_t k_pe_row_stride;
  const int64_t* slot_mapping;
  int num_tokens;
  /* fused RMSNorm + rotary write when gamma != NULL */
  const void* gamma;
  float eps;
  const int64_t* positions;
  const float* cos_sin_table;
  int64_t max_position;
  int rotate_q;
} mla_decode_desc;

typedef struct mla_decode_plan mla_decode_plan; /* opaque, host memory */

/* Validates *desc and prepares its launches.  On MLA_OK *plan is a new plan
 * (release it with mla_plan_destroy); on error *plan is NULL and nothing was
 * launched.  Call it with the plan's device current and outside any stream
 * capture (it queries the device and encodes tensor maps). */
mla_status mla_plan_create(const mla_decode_desc* desc, mla_decode_plan** plan);

/* Launches the plan's step on `stream` (cudaStream_t; NULL: the legacy
 * default stream): the write (if any), stage 1 and, with num_kv_splits > 1,
 * the merge.  Asynchronous.  MLA_ERR_INVALID_ARG for a NULL plan,
 * MLA_ERR_CUDA if a launch fails. */
mla_status mla_plan_run(const mla_decode_plan* plan, void* stream);

/* Frees a plan (NULL is ignored).  Launches already made are unaffected. */
void mla_plan_destroy(mla_decode_plan* plan);

/* Human-readable name of a status code (static string, never NULL). */
const char* mla_status_string(mla_status status);

/* Text of the last CUDA error seen by a call on this host thread that
 * returned MLA_ERR_CUDA, or "" (static per-thread buffer). */
const char* mla_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_MLA_H_ */
