// Split-KV MLA decode, stage 1, on the 5th-generation tensor cores
// (tcgen05.mma with TMEM accumulators), for 128 query vectors per CTA pair.
//
// Restates the same operation as the warp-MMA kernel ("frozenleaves/vllm
// compare v0.11.0...mla_cuda_graphs", vllm/attention/ops/
// triton_decode_attention.py, _fwd_grouped_kernel_stage1): per split, the
// paged rows' scores s = sm_scale * q.k over all R+P dims, an online softmax,
// and O += P.V with V the latent part of the same rows.
//
// GB300 design.  128 query vectors (one row's 128 heads, or several rows of
// one sequence) share every KV row, so the work is a dense contraction:
// S = Q K^T (M=128 vectors, N=64 tokens, K=576) and O = P V (M=128, N=512,
// K=64).  An fp32 O of 128 x 512 fills all of a CTA's TMEM (512 columns), so
// the latent dimension is split over a 2-CTA cluster:
//   rank 0 holds dims [0, 256)   : S partial over them, O[:, 0:256)
//   rank 1 holds dims [256, 576) : S partial over them, O[:, 256:512)
// Each CTA loads only its own dims of every KV tile (no byte is read twice),
// computes its partial S into TMEM, and the two partials are exchanged
// through distributed shared memory (st.async completing on the peer's
// mbarrier); both CTAs then run the same softmax on S = S_lo + S_hi
// (identical bits on both sides) and each accumulates its half of O.
//
// TMEM (512 columns): O [0, 256), S [256, 320), P [320, 352) as packed
// bf16, Q [352, 512) as packed bf16 (rank 1 needs 160 columns for its 320
// dims).  Q and P are A operands read straight from TMEM by the MMAs; only K
// and V tiles live in shared memory, which leaves room for a 4-stage ring of
// 64-token tiles (enough bytes in flight to cover the HBM latency).  Tiles
// are 64 tokens so that each S MMA has N = 64 (an MMA instruction costs
// about the same to issue up to N = 64).
//
// Roles per CTA (192 threads):
//   warps 0-3  softmax: thread i owns TMEM lane i = query vector i; the
//              row max / row sum are thread-local; lazy rescaling of O
//              (only when the running max grows by more than 2^8);
//   warp 4     TMA producer: 64-token tiles of the paged cache into a
//              4-stage mbarrier ring (128-byte swizzled boxes);
//   warp 5     MMA issuer (one thread) and TMEM owner.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.cuh"
#include "ptx.cuh"
#include "tc.cuh"

namespace mla {

namespace {

constexpr int TBN = 64;                   // tokens per tile
constexpr int TSTAGES = 4;                // KV ring depth
constexpr int TMAXCH = 5;                 // max 64-dim chunks per CTA
constexpr int CHUNK_BYTES = TBN * 128;    // one 64-dim box of a tile (8 KiB)
constexpr int STAGE_BYTES = TMAXCH * CHUNK_BYTES;
constexpr int XS_ROW = TBN * 4;           // bytes of one exchanged S row
constexpr int XS_BYTES = 128 * XS_ROW;
constexpr int OFF_STAGE = 0;
constexpr int OFF_XS = OFF_STAGE + TSTAGES * STAGE_BYTES;
constexpr int OFF_BAR = OFF_XS + 2 * XS_BYTES;
constexpr int NBARS = 2 * TSTAGES + 2 + 4 + 1;
constexpr int OFF_TMEMSLOT = OFF_BAR + NBARS * 8;
constexpr int TC_SMEM = OFF_TMEMSLOT + 16 + 1024;  // + alignment slack
constexpr int TC_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 256;  // S, 64 fp32 columns
constexpr uint32_t P_COL = 320;  // P, 64 bf16 in 32 columns
constexpr uint32_t Q_COL = 352;  // Q, up to 320 bf16 in 160 columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

static_assert(OFF_XS % 1024 == 0, "alignment");
static_assert(TC_SMEM <= 227 * 1024, "shared memory");

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// All lanes wait; the result is made warp-uniform.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// Byte offset of 16-byte chunk `c` (0..15) of exchanged S row `r`: the chunk
// index is XORed with r mod 8 so that 8 consecutive rows hit all 32 banks.
__device__ __forceinline__ uint32_t xs_off(uint32_t r, uint32_t c) {
  return r * XS_ROW + ((c ^ (r & 7u)) << 4);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TC_THREADS, 1)
    decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap,
                     const int split_group) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + TSTAGES;
  uint64_t* xs_full = bars + 2 * TSTAGES;  // two exchange buffers
  uint64_t* s_full = xs_full + 2;
  uint64_t* s_free = xs_full + 3;
  uint64_t* p_full = xs_full + 4;
  uint64_t* pv_done = xs_full + 5;
  uint64_t* mma_done = xs_full + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEMSLOT);

  const uint32_t rank = tc::cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int nch = rank == 0 ? 4 : 5;       // local 64-dim chunks
  const int c0 = rank == 0 ? 0 : 4;        // first global chunk
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g_blk = blockIdx.x >> 1, ysplit = blockIdx.y, b = blockIdx.z;
  const int H = p.num_heads;
  const int nvec = p.rows_per_seq * H;
  const int v0 = g_blk * 128;
  const int S = p.num_splits;
  if (threadIdx.x == 128) tma_prefetch_desc(&tmap);
  // Launched overlapped with the previous kernel of the stream: nothing in
  // global memory is read before it has completed.
  griddep_wait();
  griddep_launch_dependents();

  int L = __ldg(p.seq_lens + b);
  const int Lmax = p.max_blocks * p.block_size;
  if (L < 0) L = 0;
  if (L > Lmax) {
    if (threadIdx.x == 0 && rank == 0 && ysplit == 0 && g_blk == 0 && p.err_count)
      atomicAdd(p.err_count, 1);
    L = Lmax;
  }
  const int per = L > 0 ? cdiv(cdiv(L, S), 64) * 64 : 64;
  const int s0 = ysplit * split_group;
  const int s1 = min(S, s0 + split_group);
  const int start = s0 * per;
  const int end = min(L, s1 * per);
  const int ntiles = start < end ? cdiv(end - start, TBN) : 0;

  if (ntiles == 0) {
    // Both CTAs of the pair take this branch together.
    if (threadIdx.x < 128) {
      const int v = v0 + threadIdx.x;
      if (v < nvec) {
        const int row = b * p.rows_per_seq + v / H, h = v % H;
        if (S == 1) {
          // Empty sequence in single-pass mode: o = 0, lse = -inf.
          uint16_t* orow = p.o + (static_cast<int64_t>(row) * H + h) * 512 + rank * 256;
          for (int c = 0; c < 256; c += 8)
            *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
          if (rank == 0) p.lse[static_cast<int64_t>(row) * H + h] = -INFINITY;
        } else if (L > 0 && rank == 0) {
          // Splits past the end of a non-empty sequence: no partial.
          for (int s = s0; s < s1; ++s)
            p.ws_lse[(static_cast<int64_t>(row) * S + s) * H + h] = -INFINITY;
        }
      }
    }
    return;
  }

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    for (int i = 0; i < TSTAGES; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&xs_full[i], 1);  // expect_tx by one thread
    mbar_init(s_full, 1);
    mbar_init(s_free, 128);
    mbar_init(p_full, 128);
    mbar_init(pv_done, 1);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();  // the peer's barriers exist before any remote traffic
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  if (warp < 4) {
    // Q: thread i puts its vector's dims [64*c0, 64*(c0+nch)) into TMEM lane
    // i as packed bf16 pairs (padding vectors are zeros).
    const int v = v0 + threadIdx.x;
    const uint16_t* src = nullptr;
    if (v < nvec) {
      const int row = b * p.rows_per_seq + v / H, h = v % H;
      src = p.q + row * p.q_row_stride + h * p.q_head_stride + c0 * 64;
    }
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    for (int c = 0; c < nch; ++c) {
      uint32_t r[32];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 x = src ? __ldg(reinterpret_cast<const uint4*>(src + c * 64) + j)
                            : make_uint4(0, 0, 0, 0);
        r[4 * j] = x.x;
        r[4 * j + 1] = x.y;
        r[4 * j + 2] = x.z;
        r[4 * j + 3] = x.w;
      }
      tc::st_32x32b_x32(tmem + lane_base + Q_COL + c * 32, r);
    }
    tc::wait_st();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t stage_base = smem_u32(smem + OFF_STAGE);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int bs = p.block_size;
      const int rows_box = bs < TBN ? bs : TBN;
      const int npg = TBN / rows_box;
      const int32_t* bt = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
      for (int n = 0; n < ntiles; ++n) {
        const int st = n % TSTAGES;
        const uint32_t ph = (n / TSTAGES) & 1;
        if (!mbar_wait(&kv_empty[st], ph ^ 1)) {
          if (p.err_count) atomicAdd(p.err_count, kTimeoutErr);
          break;
        }
        const int tok0 = start + n * TBN;
        int npages = 0;
        for (int pg = 0; pg < npg; ++pg)
          if (tok0 + pg * rows_box < end) ++npages;
        mbar_arrive_expect_tx(&kv_full[st],
                              static_cast<uint32_t>(npages * nch * rows_box * 128));
        uint8_t* dst = smem + OFF_STAGE + st * STAGE_BYTES;
        for (int pg = 0; pg < npages; ++pg) {
          const int t = tok0 + pg * rows_box;
          const int blk = __ldg(bt + t / bs);
          const int row0 = t % bs;
          if ((blk < 0 || blk >= p.num_blocks) && p.err_count && rank == 0)
            atomicAdd(p.err_count, 1);
          for (int cl = 0; cl < nch; ++cl)
            tma_load_3d(dst + cl * CHUNK_BYTES + pg * rows_box * 128, &tmap,
                        &kv_full[st], (c0 + cl) * 64, row0, blk);
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idS = tc::idesc_bf16(128, TBN, 0, 0);
    constexpr uint32_t idPV = tc::idesc_bf16(128, 256, 0, 1);
    const int nks = nch * 4;
    bool ok = true;
    auto issue_pv = [&](int k) -> bool {
      if (!warp_wait(p_full, k & 1)) return false;
      tc::fence_after_sync();
      if (lane == 0) {
        const uint32_t stb = stage_base + (k % TSTAGES) * STAGE_BYTES;
#pragma unroll
        for (int kk = 0; kk < TBN / 16; ++kk) {
          // A = P (TMEM, 16 tokens = 8 packed columns per step); B = V:
          // MN-major, 128-byte swizzle (N step = next 64-dim box, K step =
          // 8 tokens = 1024 B).
          const uint64_t bd = tc::smem_desc(stb + kk * 2048, CHUNK_BYTES, 1024,
                                            tc::kLayoutSw128);
          tc::mma_ts(tmem, tmem + P_COL + kk * 8, bd, idPV, (k > 0 || kk > 0) ? 1u : 0u);
        }
        tc::commit(pv_done);
        tc::commit(&kv_empty[k % TSTAGES]);
      }
      __syncwarp();
      return true;
    };
    for (int n = 0; n < ntiles && ok; ++n) {
      const int st = n % TSTAGES;
      if (!warp_wait(&kv_full[st], (n / TSTAGES) & 1)) {
        ok = false;
        break;
      }
      const int valid = min(TBN, end - (start + n * TBN));
      if (valid < TBN) {
        // Rows past the split end hold other tokens or NaN: zero them so the
        // P.V product sees 0 * 0 there (their scores are masked to -inf).
        uint8_t* stp = smem + OFF_STAGE + st * STAGE_BYTES;
        const int nz = (TBN - valid) * nch * 8;
        for (int i = lane; i < nz; i += 32) {
          const int r = valid + i / (nch * 8), rem = i % (nch * 8);
          *reinterpret_cast<uint4*>(stp + (rem >> 3) * CHUNK_BYTES + r * 128 +
                                    (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (n >= 1 && !warp_wait(s_free, (n - 1) & 1)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      if (lane == 0) {
        // S = Q K^T: A = Q from TMEM (16 dims = 8 packed columns per step),
        // B = K tile, K-major with 128-byte swizzle.
        const uint32_t stb = stage_base + st * STAGE_BYTES;
        for (int ks = 0; ks < nks; ++ks) {
          const uint64_t bd = tc::smem_desc(stb + (ks >> 2) * CHUNK_BYTES + (ks & 3) * 32, 16,
                                            1024, tc::kLayoutSw128);
          tc::mma_ts(tmem + S_COL, tmem + Q_COL + ks * 8, bd, idS, ks > 0 ? 1u : 0u);
        }
        tc::commit(s_full);
      }
      __syncwarp();
      if (n >= 1 && !issue_pv(n - 1)) {
        ok = false;
        break;
      }
    }
    if (ok) ok = issue_pv(ntiles - 1);
    if (!ok && lane == 0 && p.err_count) atomicAdd(p.err_count, kTimeoutErr);
    if (lane == 0) tc::commit(mma_done);
    __syncwarp();
    warp_wait(mma_done, 0);  // nothing of ours still runs on the tensor core
  } else {
    // ------------------------------------------------------------ softmax
    const int row_i = threadIdx.x;  // TMEM lane / query vector
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float scale_log2 = p.sm_scale * kLog2e;
    const uint32_t xs_local = smem_u32(smem + OFF_XS);
    const uint32_t xs_peer = tc::map_peer(xs_local, peer);
    const uint32_t xsbar_peer0 = tc::map_peer(smem_u32(&xs_full[0]), peer);
    const uint32_t xsbar_peer1 = tc::map_peer(smem_u32(&xs_full[1]), peer);
    float m_used = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int n = 0; n < ntiles; ++n) {
      const int bb = n & 1;             // exchange buffer
      const uint32_t u = (n >> 1) & 1;  // its phase parity
      if (!warp_wait(s_full, n & 1)) { ok = false; break; }
      tc::fence_after_sync();
      uint32_t sr[64];
      tc::ld_32x32b_x32(tmem + lane_base + S_COL,
                        *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tc::ld_32x32b_x32(tmem + lane_base + S_COL + 32,
                        *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tc::wait_ld();
      tc::fence_before_sync();
      mbar_arrive(s_free);
      // partial S -> the peer's exchange buffer with st.async: each store
      // completes its bytes on the peer's xs_full[bb]; one local thread
      // announces the 128 x 64 x 4 bytes this CTA expects from the peer.
      if (row_i == 0) mbar_arrive_expect_tx(&xs_full[bb], 128 * TBN * 4);
      {
        const uint32_t dst = xs_peer + bb * XS_BYTES;
        const uint32_t pbar = bb ? xsbar_peer1 : xsbar_peer0;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          tc::st_async_v4(dst + xs_off(row_i, j), __uint_as_float(sr[4 * j]),
                          __uint_as_float(sr[4 * j + 1]), __uint_as_float(sr[4 * j + 2]),
                          __uint_as_float(sr[4 * j + 3]), pbar);
      }
      const bool got = tc::mbar_wait_cluster(&xs_full[bb], u);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      const uint8_t* xs = smem + OFF_XS + bb * XS_BYTES;
      const int valid = min(TBN, end - (start + n * TBN));
      float mt = -INFINITY;
#pragma unroll
      for (int j4 = 0; j4 < 16; ++j4) {
        const float4 t = *reinterpret_cast<const float4*>(xs + xs_off(row_i, j4));
        const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = 4 * j4 + e;
          const float own = __uint_as_float(sr[j]);
          // S = S_lo + S_hi on both CTAs (same operands, same bits)
          const float s = rank == 0 ? own + tv[e] : tv[e] + own;
          const float x = j < valid ? s * scale_log2 : -INFINITY;
          sr[j] = __float_as_uint(x);
          mt = fmaxf(mt, x);
        }
      }
      const float m_new = fmaxf(m_used, mt);
      const bool need = m_new > m_used + kRescaleThreshold;
      if (__any_sync(0xffffffffu, need)) {
        const float alpha = ex2(m_used - m_new);
        if (n > 0) {
          if (!warp_wait(pv_done, (n - 1) & 1)) { ok = false; break; }
          tc::fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < 256; c += 32) {
            uint32_t o[32];
            tc::ld_32x32b_x32(tmem + lane_base + c, o);
            tc::wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tc::st_32x32b_x32(tmem + lane_base + c, o);
          }
          tc::wait_st();
        }
        l_run *= alpha;
        m_used = m_new;
      }
      uint32_t pk[32];
      float psum = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float a0 = ex2(__uint_as_float(sr[2 * j]) - m_used);
        const float a1 = ex2(__uint_as_float(sr[2 * j + 1]) - m_used);
        psum += a0 + a1;
        pk[j] = pack_bf16x2(a0, a1);
      }
      l_run += psum;
      // P's TMEM columns are free once the previous P.V has completed
      if (n >= 1 && !warp_wait(pv_done, (n - 1) & 1)) { ok = false; break; }
      tc::fence_after_sync();
      tc::st_32x32b_x32(tmem + lane_base + P_COL, pk);
      tc::wait_st();
      tc::fence_before_sync();
      mbar_arrive(p_full);
    }
    if (!ok) {
      if (lane == 0 && p.err_count) atomicAdd(p.err_count, kTimeoutErr);
    } else if (warp_wait(pv_done, (ntiles - 1) & 1)) {
      tc::fence_after_sync();
      const int v = v0 + row_i;
      const bool valid_v = v < nvec;
      const int row = valid_v ? b * p.rows_per_seq + v / H : 0;
      const int h = valid_v ? v % H : 0;
      const float inv = 1.f / l_run;
      float lg;
      asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(l_run));
      const float lse = (m_used + lg) * kLn2;
      const int64_t rec = (static_cast<int64_t>(row) * S + s0) * H + h;
#pragma unroll 1
      for (int c = 0; c < 256; c += 32) {
        uint32_t o[32];
        tc::ld_32x32b_x32(tmem + lane_base + c, o);
        tc::wait_ld();
        if (!valid_v) continue;
        const int col = rank * 256 + c;
        if (S == 1) {
          uint16_t* dst = p.o + (static_cast<int64_t>(row) * H + h) * 512 + col;
#pragma unroll
          for (int j = 0; j < 32; j += 8)
            *reinterpret_cast<uint4*>(dst + j) = make_uint4(
                pack_bf16x2(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv),
                pack_bf16x2(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv),
                pack_bf16x2(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv),
                pack_bf16x2(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv));
        } else {
          float* dst = p.ws_o + rec * 512 + col;
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + j) =
                make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                            __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
        }
      }
      if (valid_v && rank == 0) {
        if (S == 1) {
          p.lse[static_cast<int64_t>(row) * H + h] = lse;
        } else {
          p.ws_lse[rec] = lse;
          // splits fused into this CTA pair hold no partial of their own
          for (int s = s0 + 1; s < s1; ++s)
            p.ws_lse[(static_cast<int64_t>(row) * S + s) * H + h] = -INFINITY;
        }
      }
    } else if (lane == 0 && p.err_count) {
      atomicAdd(p.err_count, kTimeoutErr);
    }
  }

  // ---------------------------------------------------------------- teardown
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();  // no CTA leaves while its peer may still write to it
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

int tc_split_group(const DecodeParams& p, int sm_count) {
  // Fuse consecutive splits into CTA pairs.  With f splits per pair the
  // launch has units * ceil(S / f) pairs; the estimated cost (in units of one
  // split's KV stream) is the number of waves times the work of one pair, plus
  // the partial outputs each pair writes and the merge reads back (about 0.85
  // of a split's bytes per 128-vector unit).  Pick f with the lowest cost.
  const int qblocks = (p.rows_per_seq * p.num_heads + 127) / 128;
  const int64_t units = static_cast<int64_t>(qblocks) * p.num_seqs;
  const int64_t pairs = sm_count >= 2 ? sm_count / 2 : 1;
  const int S = p.num_splits;
  int best_f = S;
  double best_cost = 1e300;
  for (int f = S; f >= 1; --f) {
    const int64_t groups = (S + f - 1) / f;
    if (f < S && (S + f) / (f + 1) == groups) continue;  // same grid as f + 1
    const int64_t ctas = units * groups;
    const int64_t waves = (ctas + pairs - 1) / pairs;
    const double cost = static_cast<double>(waves) * f * pairs + 0.85 * ctas;
    if (cost < best_cost) {
      best_cost = cost;
      best_f = f;
    }
  }
  return best_f;
}

cudaError_t launch_decode_tc(const DecodeParams& p, const CUtensorMap& tmap,
                             int split_group, cudaStream_t stream) {
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(
        decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, TC_SMEM);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const int qblocks = (p.rows_per_seq * p.num_heads + 127) / 128;
  const int groups = (p.num_splits + split_group - 1) / split_group;
  const dim3 grid(2 * qblocks, groups, p.num_seqs);
  return launch_overlapped(decode_tc_kernel, grid, dim3(TC_THREADS), TC_SMEM, stream, p, tmap,
                           split_group);
}

}  // namespace mla
