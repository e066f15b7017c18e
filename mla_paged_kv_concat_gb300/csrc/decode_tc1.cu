// Split-KV MLA decode, stage 1, on the 5th-generation tensor cores for the
// 256-wide latent (kv_lora_rank 256, head 320), one CTA per 128 query
// vectors, bf16 or fp8 (E4M3 / E5M2) cache.
//
// The same operation as the other stage-1 kernels ("frozenleaves/vllm compare
// v0.11.0...mla_cuda_graphs", vllm/attention/ops/triton_decode_attention.py,
// _fwd_grouped_kernel_stage1; "Triton and MLA", Data flow, with k_scale =
// v_scale dequantising an fp8 cache): per split, s = sm_scale * q.k over all
// 320 dims, an online softmax, O += P.V with V the 256 latent dims.
//
// GB300 design.  With a 256-wide latent the fp32 O of 128 query vectors is
// 128 x 256 = 256 TMEM columns, so one CTA holds everything and the softmax
// of a row is local (no cluster exchange, unlike the 512-wide kernel):
//   TMEM (512 columns): O [0, 256), S [256, 384) as two 64-token buffers,
//     Q dims [0, 256) [384, 512) as packed bf16 (the A operand of S);
//   shared memory: Q dims [256, 320) (the rope part of the A operand of S,
//     128 rows x 128 B, 128-byte swizzled K-major), two P buffers (the A
//     operand of P.V, same layout), the bf16 tile ring (the B operand of S,
//     K-major, and of P.V, MN-major), and for an fp8 cache a ring of raw fp8
//     tiles that converter warps turn into bf16 tiles (exactly: every E4M3
//     and E5M2 value is a bf16 value; the scale folds into the score scale
//     and the output).
// S = Q K^T is M=128, N=64, K=16 per instruction (20 per tile), P.V is
// M=128, N=256, K=16 (4 per tile).  Query vectors past the sequence's count
// fill the M tile with zero rows, whose results are never stored.
//
// Roles: warps 0-3 softmax (thread = TMEM lane = query vector), warp 4 TMA
// producer, warp 5 MMA issuer and TMEM owner, warps 6-9 fp8 converters (fp8
// caches only).  With several splits the kernel is persistent: one CTA per
// SM takes an equal share of all tiles of all (sequence, 128-vector block)
// units, cut into segments at unit boundaries, each segment yielding one
// partial (o, lse) in the unit's next split slot (the same schedule as the
// 512-wide tcgen05 kernel, per CTA instead of per CTA pair).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "kernels.cuh"
#include "ptx.cuh"
#include "tc.cuh"

namespace mla {

namespace {

constexpr int TBN = 64;                      // tokens per tile
constexpr int NCH = 5;                       // 64-dim chunks of a 320-dim row
constexpr int CHUNK_BYTES = TBN * 128;       // one bf16 64-dim box (8 KiB)
constexpr int TILE_BYTES = NCH * CHUNK_BYTES;
constexpr int RAW_CHUNK = TBN * 64;          // one fp8 64-dim box (4 KiB)
constexpr int RAW_BYTES = NCH * RAW_CHUNK;
constexpr int RSTAGES = 3;                   // raw fp8 ring
constexpr int PSTAGES = 2;                   // fp8: rope-dim chunk ring (S only)
constexpr int P_BYTES = 128 * 128;           // 128 rows x 64 bf16
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 256;   // two 64-column S buffers
constexpr uint32_t QN_COL = 384;  // Q dims [0, 256): 128 columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kClampedBit = 1 << 30;

// bf16 cache: the TMA fills whole bf16 tiles (five boxes) in a 4-stage ring,
// each held until its P.V has run.  fp8 cache: the converters fill the four
// latent boxes of a tile into a 3-stage ring (held until P.V) and the rope
// box into a 2-stage ring of its own (free as soon as S has read it), which
// is what lets a raw ring of three stages fit beside them.
template <bool FP8>
struct Tc1Cfg {
  static constexpr int TSTAGES = FP8 ? 3 : 4;  // bf16 tile (or latent-box) ring
  static constexpr int STAGE_B = FP8 ? 4 * CHUNK_BYTES : TILE_BYTES;
  static constexpr int NWARPS = FP8 ? 10 : 6;
  static constexpr int NTHREADS = NWARPS * 32;
  static constexpr int OFF_TILE = 0;
  static constexpr int OFF_ROPE = OFF_TILE + TSTAGES * STAGE_B;
  static constexpr int OFF_RAW = OFF_ROPE + (FP8 ? PSTAGES * CHUNK_BYTES : 0);
  static constexpr int OFF_P = OFF_RAW + (FP8 ? RSTAGES * RAW_BYTES : 0);
  static constexpr int OFF_QPE = OFF_P + 2 * P_BYTES;
  static constexpr int OFF_PRE = OFF_QPE + P_BYTES;
  static constexpr int OFF_LEN = OFF_PRE + (kMaxPersistUnits + 1) * 4;
  static constexpr int OFF_BAR = (OFF_LEN + kMaxPersistUnits * 4 + 7) & ~7;
  static constexpr int NBARS = 2 * TSTAGES + 2 * RSTAGES + PSTAGES + 11;
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBARS * 8;
  static constexpr int SMEM = OFF_TMEMSLOT + 16 + 1024;  // + alignment slack
  static_assert(OFF_P % 1024 == 0 && OFF_QPE % 1024 == 0 && OFF_RAW % 1024 == 0 &&
                    OFF_ROPE % 1024 == 0,
                "swizzle alignment");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-row buffer with the
// 128-byte swizzle (the canonical K-major layout of an MMA operand).
__device__ __forceinline__ uint32_t sw_off(uint32_t r, uint32_t c) {
  return r * 128u + ((c ^ (r & 7u)) << 4);
}

// 16 fp8 bytes -> 16 bf16 values (exact: every E4M3 and E5M2 value is a
// bf16 value).
__device__ __forceinline__ void fp8x16_bf16(uint4 raw, bool e5m2, uint4& lo, uint4& hi) {
  const uint16_t* b = reinterpret_cast<const uint16_t*>(&raw);
  uint32_t out[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(b[k]),
                                               e5m2 ? __NV_E5M2 : __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
    out[k] = pack_bf16x2(f.x, f.y);
  }
  lo = make_uint4(out[0], out[1], out[2], out[3]);
  hi = make_uint4(out[4], out[5], out[6], out[7]);
}

// One unit of work: tokens [start, end) of sequence b for 128-vector block
// g, result to split slot `slot` (or o / lse when `direct`); mark_* are the
// slots this segment marks unused (lse = -inf).
struct Seg1 {
  int b, g, start, end, slot, mark_lo, mark_hi, mark2_lo, mark2_hi;
  bool direct;
};

template <bool FP8>
__global__ void __launch_bounds__(Tc1Cfg<FP8>::NTHREADS, 1)
    decode_tc1_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap,
                      const int split_group, const int persistent) {
  using C = Tc1Cfg<FP8>;
  constexpr int TS = C::TSTAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* tile_full = bars;              // [TS] bf16 tile ready (TMA or converters)
  uint64_t* tile_empty = bars + TS;        // [TS] P.V of the tile done
  uint64_t* raw_full = bars + 2 * TS;      // [RSTAGES] fp8 tile landed
  uint64_t* raw_empty = raw_full + RSTAGES;  // [RSTAGES] fp8 tile converted
  uint64_t* rope_empty = raw_empty + RSTAGES;  // [PSTAGES] fp8: S has read the rope box
  uint64_t* s_full = rope_empty + PSTAGES;  // [2]
  uint64_t* s_free = s_full + 2;           // [2] every softmax thread read it
  uint64_t* p_full = s_full + 4;           // [2] P in smem, O rescaled
  uint64_t* pv_done = s_full + 6;          // [2]
  uint64_t* q_ready = s_full + 8;
  uint64_t* o_free = s_full + 9;
  uint64_t* mma_done = s_full + 10;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMSLOT);
  int* pre = reinterpret_cast<int*>(smem + C::OFF_PRE);
  int* lens = reinterpret_cast<int*>(smem + C::OFF_LEN);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The MMA warp polls two barriers without sleeping; it sits on SM
  // sub-partition 1, away from softmax warp 0 (the only live one when a unit
  // has at most 32 query vectors); the producer, which sleeps in its waits,
  // takes sub-partition 0.
  constexpr int kMmaWarp = 5, kProdWarp = 4;
  const int H = p.num_heads;
  const int nvec = p.rows_per_seq * H;
  const int qblocks = cdiv(nvec, 128);
  const int S = p.num_splits;
  const int Lmax = p.max_blocks * p.block_size;
  if (threadIdx.x == kProdWarp * 32) tma_prefetch_desc(&tmap);
  // Launched overlapped with the previous kernel of the stream: nothing in
  // global memory is read before it has completed.
  griddep_wait();
  griddep_launch_dependents();

  // ---------------------------------------------------------- schedule
  // Persistent: the tiles of all units (sequence, 128-vector block) form one
  // list; CTA c takes tiles [c * C, (c + 1) * C), cut into segments at unit
  // boundaries.  A sequence with several 128-vector blocks is listed in
  // chunks of CH tiles, all blocks of a chunk side by side (the CTAs holding
  // them then stream the same KV tiles at about the same time and L2 serves
  // the later readers); a chunk of one block spans at most SPC CTAs and
  // owns SPC split slots.  Grid: one segment per CTA, split_group
  // consecutive splits of one unit.
  int Cn = 1, lo = 0, hi = 0, cidx = 0;
  int CH = 1 << 30, SPC = 1;
  Seg1 gseg{};
  int nseg = 0;
  if (persistent) {
    cidx = blockIdx.x;
    const int units = p.num_seqs * qblocks;
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
      const int b = u / qblocks;
      const int raw = __ldg(p.seq_lens + b);
      const int L = raw < 0 ? 0 : (raw > Lmax ? Lmax : raw);
      pre[u + 1] = cdiv(L, TBN);
      if (u == b * qblocks) lens[b] = L | (raw > Lmax ? kClampedBit : 0);
    }
    if (threadIdx.x == 0) pre[0] = 0;
    __syncthreads();
    __shared__ int s_max;
    if (warp == 0) {
      int carry = 0, mx = 0;
      for (int base = 1; base <= units; base += 32) {
        const int i = base + lane;
        int v = i <= units ? pre[i] : 0;
        mx = max(mx, v);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += t;
        }
        if (i <= units) pre[i] = v + carry;
        carry += __shfl_sync(0xffffffffu, v, 31);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      if (lane == 0) s_max = mx;
    }
    __syncthreads();
    const int total = pre[units];
    Cn = max(max(cdiv(total, static_cast<int>(gridDim.x)), cdiv(s_max, max(S - 1, 1))), 1);
    lo = cidx * Cn;
    hi = min(total, lo + Cn);
    SPC = S;
    if (qblocks > 1) {
      // smallest m with (chunks) x (slots per chunk) <= S; m = cdiv(s_max, C)
      // (one chunk) always qualifies because C >= cdiv(s_max, S - 1)
      for (int m = 1;; ++m) {
        const int J = cdiv(s_max, Cn * m);
        if (J * (m + 1) <= S || J == 1) {
          CH = Cn * m;
          SPC = m + 1;
          break;
        }
      }
    }
    if (lo >= hi) return;
  } else {
    const int b = blockIdx.z, ysplit = blockIdx.y;
    int L = __ldg(p.seq_lens + b);
    if (L < 0) L = 0;
    if (L > Lmax) {
      if (threadIdx.x == 0 && ysplit == 0 && blockIdx.x == 0 && p.err_count)
        atomicAdd(p.err_count, 1);
      L = Lmax;
    }
    const int per = L > 0 ? cdiv(cdiv(L, S), TBN) * TBN : TBN;
    const int s0 = ysplit * split_group;
    const int s1 = min(S, s0 + split_group);
    gseg.b = b;
    gseg.g = blockIdx.x;
    gseg.start = s0 * per;
    gseg.end = min(L, s1 * per);
    gseg.slot = s0;
    gseg.mark_lo = s0 + 1;
    gseg.mark_hi = s1;
    gseg.mark2_lo = gseg.mark2_hi = 0;
    gseg.direct = S == 1;
    if (gseg.start >= gseg.end) {
      if (threadIdx.x < 128) {
        const int v = gseg.g * 128 + threadIdx.x;
        if (v < nvec) {
          const int row = b * p.rows_per_seq + v / H, h = v % H;
          if (S == 1) {
            // Empty sequence in single-pass mode: o = 0, lse = -inf.
            uint16_t* orow = p.o + (static_cast<int64_t>(row) * H + h) * 256;
            for (int c = 0; c < 256; c += 8)
              *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
            p.lse[static_cast<int64_t>(row) * H + h] = -INFINITY;
          } else if (L > 0) {
            // Splits past the end of a non-empty sequence: no partial.
            for (int s = s0; s < s1; ++s)
              p.ws_lse[(static_cast<int64_t>(row) * S + s) * H + h] = -INFINITY;
          }
        }
      }
      return;
    }
    nseg = 1;
  }
  // The segment that starts at list tile t (lo <= t < hi); returns the list
  // position where the next segment starts.
  auto seg_at = [&](int t, Seg1& s) -> int {
    int a = 0, z = p.num_seqs - 1;  // sequence: the last with pre[b * qblocks] <= t
    while (a < z) {
      const int m = (a + z + 1) >> 1;
      if (pre[m * qblocks] <= t) a = m; else z = m - 1;
    }
    const int b = a;
    const int Ob = pre[b * qblocks];
    const int Tb = pre[b * qblocks + 1] - Ob;  // tiles of the sequence
    const int Jb = cdiv(Tb, CH);
    const int span = qblocks * CH;
    const int x = t - Ob;
    const int j = min(x / span, Jb - 1);
    const int len = j == Jb - 1 ? Tb - (Jb - 1) * CH : CH;
    const int y = x - j * span;
    const int g = y / len;
    const int in = y - g * len;
    const int vstart = Ob + j * span + g * len;
    const int vend = vstart + len;
    const int seg_end = min(hi, vend);
    const int L = lens[b] & ~kClampedBit;
    s.b = b;
    s.g = g;
    s.start = (j * CH + in) * TBN;
    s.end = min(L, (j * CH + in + (seg_end - t)) * TBN);
    const int cf = vstart / Cn;  // the CTA where chunk j of block g begins
    s.slot = j * SPC + (cidx - cf);
    const bool first = cidx == cf;
    s.mark_lo = first ? j * SPC + ((vend - 1) / Cn - cf + 1) : 0;
    s.mark_hi = first ? (j + 1) * SPC : 0;
    s.mark2_lo = first && j == 0 ? Jb * SPC : 0;  // slots past the last chunk
    s.mark2_hi = first && j == 0 ? S : 0;
    s.direct = false;
    return seg_end;
  };
  // Walks this CTA's segments in order: f(seg, index, first tile (a running
  // count over the CTA's segments), next segment or nullptr).
  auto for_each_seg = [&](auto&& f) {
    if (!persistent) {
      if (nseg) f(gseg, 0, 0, static_cast<const Seg1*>(nullptr));
      return;
    }
    if (lo >= hi) return;
    Seg1 cur, nxt;
    int t_next = seg_at(lo, cur);
    for (int k = 0, n0 = 0;; ++k) {
      const bool more = t_next < hi;
      int t_after = hi;
      if (more) t_after = seg_at(t_next, nxt);
      if (cur.slot == 0 && cur.g == 0 && (lens[cur.b] & kClampedBit) && threadIdx.x == 0 &&
          p.err_count)
        atomicAdd(p.err_count, 1);  // seq_len beyond the block table, once per sequence
      if (!f(cur, k, n0, more ? &nxt : static_cast<const Seg1*>(nullptr))) return;
      if (!more) return;
      n0 += cdiv(cur.end - cur.start, TBN);
      cur = nxt;
      t_next = t_after;
    }
  };

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    for (int i = 0; i < TS; ++i) {
      mbar_init(&tile_full[i], FP8 ? 128 : 1);  // converter threads, or TMA bytes
      mbar_init(&tile_empty[i], 1);
    }
    for (int i = 0; i < RSTAGES; ++i) {
      mbar_init(&raw_full[i], 1);
      mbar_init(&raw_empty[i], 4);  // the four converter warps
    }
    for (int i = 0; i < PSTAGES; ++i) mbar_init(&rope_empty[i], 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 128);
      mbar_init(&p_full[i], 128);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(q_ready, 128);
    mbar_init(o_free, 128);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tile_base = smem_u32(smem + C::OFF_TILE);
  const uint32_t rope_base = smem_u32(smem + C::OFF_ROPE);
  const uint32_t p_base = smem_u32(smem + C::OFF_P);
  const uint32_t qpe_base = smem_u32(smem + C::OFF_QPE);

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    // 64-token tiles of the paged cache: into the bf16 tile ring (128-byte
    // swizzled boxes) or, for an fp8 cache, the raw ring (unswizzled 64-byte
    // rows).
    if (lane == 0) {
      const int bs = p.block_size;
      const int rows_box = bs < TBN ? bs : TBN;
      const int npg = TBN / rows_box;
      constexpr int ROWB = FP8 ? 64 : 128;
      constexpr int NST = FP8 ? RSTAGES : TS;
      constexpr int STB = FP8 ? RAW_BYTES : C::STAGE_B;
      uint64_t* full = FP8 ? raw_full : tile_full;
      uint64_t* empty = FP8 ? raw_empty : tile_empty;
      uint8_t* ring = smem + (FP8 ? C::OFF_RAW : C::OFF_TILE);
      int n = 0;
      for_each_seg([&](const Seg1& sg, int, int, const Seg1*) -> bool {
        const int32_t* bt = p.block_table + static_cast<int64_t>(sg.b) * p.bt_stride;
        const int ntiles = cdiv(sg.end - sg.start, TBN);
        auto ids_of = [&](int t, int (&ids)[4]) {
#pragma unroll
          for (int pg = 0; pg < 4; ++pg) {
            const int tk = sg.start + t * TBN + pg * rows_box;
            ids[pg] = (pg < npg && t < ntiles && tk < sg.end) ? __ldg(bt + tk / bs) : 0;
          }
        };
        int cur[4], nxt[4];
        ids_of(0, cur);
        for (int t = 0; t < ntiles; ++t, ++n) {
          ids_of(t + 1, nxt);
          const int st = n % NST;
          if (!mbar_wait(&empty[st], ((n / NST) & 1) ^ 1)) {
            if (p.err_count) atomicAdd(p.err_count, kTimeoutErr);
            return false;
          }
          int npages = 0;
          for (int pg = 0; pg < npg; ++pg)
            if (sg.start + t * TBN + pg * rows_box < sg.end) ++npages;
          mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(npages * NCH * rows_box * ROWB));
          uint8_t* dst = ring + st * STB;
#pragma unroll
          for (int pg = 0; pg < 4; ++pg) {
            if (pg >= npages) break;
            const int tk = sg.start + t * TBN + pg * rows_box;
            const int blk = cur[pg];
            if ((blk < 0 || blk >= p.num_blocks) && p.err_count) atomicAdd(p.err_count, 1);
            for (int c = 0; c < NCH; ++c)
              tma_load_3d(dst + c * (TBN * ROWB) + pg * rows_box * ROWB, &tmap, &full[st],
                          c * 64, tk % bs, blk);
          }
#pragma unroll
          for (int pg = 0; pg < 4; ++pg) cur[pg] = nxt[pg];
        }
        return true;
      });
    }
  } else if (FP8 && warp >= 6) {
    // ------------------------------------------------------------ converters
    // Raw fp8 tile -> bf16 tile (128-byte swizzled, K-major rows of 64
    // dims); rows past the segment end become zeros, so that the P.V
    // product sees 0 * 0 there (their scores are masked).
    const int ctid = threadIdx.x - 6 * 32;  // 0 .. 127
    const bool e5m2 = p.kv_e5m2 != 0;
    int n = 0;
    bool ok = true;
    for_each_seg([&](const Seg1& sg, int, int, const Seg1*) -> bool {
      const int ntiles = cdiv(sg.end - sg.start, TBN);
      for (int t = 0; t < ntiles; ++t, ++n) {
        const int rs = n % RSTAGES, ts = n % TS, ps = n % PSTAGES;
        if (!warp_wait(&raw_full[rs], (n / RSTAGES) & 1) ||
            !warp_wait(&tile_empty[ts], ((n / TS) & 1) ^ 1) ||
            !warp_wait(&rope_empty[ps], ((n / PSTAGES) & 1) ^ 1)) {
          ok = false;
          return false;
        }
        const int valid = min(TBN, sg.end - (sg.start + t * TBN));
        const uint8_t* raw = smem + C::OFF_RAW + rs * RAW_BYTES;
        uint8_t* dst = smem + C::OFF_TILE + ts * C::STAGE_B;
        uint8_t* dst_rope = smem + C::OFF_ROPE + ps * CHUNK_BYTES;
        // 1280 16-byte pieces, 10 per thread, in two batches of five whose
        // loads are all issued before any is converted
        constexpr int kPer = NCH * TBN * 4 / 128, kBatch = 5;
        static_assert(kPer % kBatch == 0, "batches");
#pragma unroll
        for (int j0 = 0; j0 < kPer; j0 += kBatch) {
          uint4 x[kBatch];
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const int i = ctid + (j0 + j) * 128;
            const int c = i / (TBN * 4), r = (i >> 2) % TBN, kq = i & 3;
            x[j] = *reinterpret_cast<const uint4*>(raw + c * RAW_CHUNK + r * 64 + kq * 16);
          }
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const int i = ctid + (j0 + j) * 128;
            const int c = i / (TBN * 4), r = (i >> 2) % TBN, kq = i & 3;
            uint4 lo4 = make_uint4(0, 0, 0, 0), hi4 = lo4;
            if (r < valid) fp8x16_bf16(x[j], e5m2, lo4, hi4);
            uint8_t* d = c < 4 ? dst + c * CHUNK_BYTES : dst_rope;
            *reinterpret_cast<uint4*>(d + sw_off(r, 2 * kq)) = lo4;
            *reinterpret_cast<uint4*>(d + sw_off(r, 2 * kq + 1)) = hi4;
          }
        }
        fence_proxy_async_smem();  // the MMA reads the tile through the async proxy
        mbar_arrive(&tile_full[ts]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&raw_empty[rs]);
      }
      return true;
    });
    if (!ok && lane == 0 && p.err_count) atomicAdd(p.err_count, kTimeoutErr);
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idS = tc::idesc_bf16(128, TBN, 0, 0);
    constexpr uint32_t idPV = tc::idesc_bf16(128, 256, 0, 1);
    // S of tile n needs its bf16 tile, its S buffer (n & 1) read by every
    // softmax thread (tile n - 2) and, first in a segment, the segment's Q;
    // P.V of tile n needs P of tile n and, first in a segment, the previous
    // segment's O read out.  The two streams are issued as soon as each is
    // ready (P.V first), so S runs up to two tiles ahead of the softmax.
    bool ok = true;
    int ns = 0, npv = 0;  // global tile counters
    for_each_seg([&](const Seg1& sg, int k, int n0, const Seg1*) -> bool {
      const int n1 = n0 + cdiv(sg.end - sg.start, TBN);
      uint64_t t_idle = 0;
      uint32_t spins = 0;
      bool have_q = false, have_o = k == 0;
      while (npv < n1) {
        bool progress = false;
        if (!have_o) have_o = __shfl_sync(0xffffffffu, mbar_test(o_free, (k - 1) & 1), 0);
        const bool pv_ready =
            have_o && __shfl_sync(0xffffffffu,
                                  npv < ns && mbar_test(&p_full[npv & 1], (npv >> 1) & 1), 0);
        if (pv_ready) {
          tc::fence_after_sync();
          fence_proxy_async_smem();
          if (tc::elect_one()) {
            // A = P (smem, K-major, 128-byte swizzle: 16 tokens = 32 B = 2
            // in the descriptor's address field per step); B = V: the tile's
            // first four 64-dim boxes, MN-major (N step = next box, K step =
            // 8 tokens = 1024 B; 16 tokens = 128 in the address field).
            const uint64_t a0 =
                tc::smem_desc(p_base + (npv & 1) * P_BYTES, 16, 1024, tc::kLayoutSw128);
            const uint64_t d0 = tc::smem_desc(tile_base + (npv % TS) * C::STAGE_B, CHUNK_BYTES,
                                              1024, tc::kLayoutSw128);
#pragma unroll
            for (int kk = 0; kk < TBN / 16; ++kk)
              tc::mma_ss(tmem, a0 + static_cast<uint64_t>(kk * 2),
                         d0 + static_cast<uint64_t>(kk * 128), idPV,
                         (npv > n0 || kk > 0) ? 1u : 0u);
            tc::commit(&pv_done[npv & 1]);
            tc::commit(&tile_empty[npv % TS]);
          }
          __syncwarp();
          ++npv;
          progress = true;
        }
        if (!have_q) have_q = __shfl_sync(0xffffffffu, mbar_test(q_ready, k & 1), 0);
        const bool s_ready =
            have_q &&
            __shfl_sync(0xffffffffu,
                        ns < n1 && mbar_test(&tile_full[ns % TS], (ns / TS) & 1) &&
                            (ns < 2 || mbar_test(&s_free[ns & 1], ((ns - 2) >> 1) & 1)),
                        0);
        if (s_ready) {
          const int ts = ns % TS;
          if constexpr (!FP8) {
            const int valid = min(TBN, sg.end - (sg.start + (ns - n0) * TBN));
            if (valid < TBN) {
              // Rows past the segment end hold other tokens or NaN: zero the
              // latent boxes' rows so the P.V product sees 0 * 0 there.
              uint8_t* stp = smem + C::OFF_TILE + ts * C::STAGE_B;
              const int nz = (TBN - valid) * 4 * 8;
              for (int i = lane; i < nz; i += 32) {
                const int r = valid + i / 32, rem = i % 32;
                *reinterpret_cast<uint4*>(stp + (rem >> 3) * CHUNK_BYTES + r * 128 +
                                          (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
          }
          tc::fence_after_sync();
          if (tc::elect_one()) {
            // S = Q K^T: A = Q dims [0, 256) from TMEM (16 dims = 8 packed
            // columns per step) then dims [256, 320) from shared memory; B =
            // the tile's five boxes, K-major, 128-byte swizzle (one box =
            // CHUNK_BYTES / 16 in the address field, a 16-dim step 2).
            // Issued from the converged warp by one elected lane, unrolled.
            const uint64_t d0 =
                tc::smem_desc(tile_base + ts * C::STAGE_B, 16, 1024, tc::kLayoutSw128);
            // the rope box: the tile's fifth box (bf16) or the rope ring (fp8)
            const uint64_t dr =
                FP8 ? tc::smem_desc(rope_base + (ns % PSTAGES) * CHUNK_BYTES, 16, 1024,
                                    tc::kLayoutSw128)
                    : d0 + static_cast<uint64_t>(4 * (CHUNK_BYTES >> 4));
            const uint64_t aq = tc::smem_desc(qpe_base, 16, 1024, tc::kLayoutSw128);
            const uint32_t sd = tmem + S_COL + (ns & 1) * TBN;
#pragma unroll
            for (int ks = 0; ks < 16; ++ks)
              tc::mma_ts(sd, tmem + QN_COL + ks * 8,
                         d0 + static_cast<uint64_t>((ks >> 2) * (CHUNK_BYTES >> 4) + (ks & 3) * 2),
                         idS, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              tc::mma_ss(sd, aq + static_cast<uint64_t>(kk * 2), dr + static_cast<uint64_t>(kk * 2),
                         idS, 1u);
            tc::commit(&s_full[ns & 1]);
            if (FP8) tc::commit(&rope_empty[ns % PSTAGES]);
          }
          __syncwarp();
          ++ns;
          progress = true;
        }
        if (progress) {
          t_idle = 0;
          spins = 0;
        } else if ((++spins & 1023u) == 0) {
          const uint64_t now = globaltimer();
          if (t_idle == 0) {
            t_idle = now;
          } else if (now - t_idle > kWaitTimeoutNs) {
            ok = false;
            return false;
          }
        }
      }
      return true;
    });
    if (!ok && lane == 0 && p.err_count) atomicAdd(p.err_count, kTimeoutErr);
    if (lane == 0) tc::commit(mma_done);
    __syncwarp();
    warp_wait(mma_done, 0);  // nothing of ours still runs on the tensor core
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax
    // Thread = TMEM lane = query vector row_i of the unit's 128.
    const int row_i = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float kv_s = FP8 ? __ldg(p.kv_scale) : 1.0f;
    uint8_t* pbuf = smem + C::OFF_P;
    uint8_t* qpe_s = smem + C::OFF_QPE;
    bool ok = true;
    const float scale_log2 = p.sm_scale * kv_s * kLog2e;

    // Q of a segment: dims [0, 256) into TMEM lane row_i as packed bf16
    // pairs, dims [256, 320) into the shared-memory rope part (padding
    // vectors are zeros).  Called once the previous segment's S products,
    // which read Q, are complete.
    auto load_q = [&](const Seg1& sg) {
      const int v = sg.g * 128 + row_i;
      const bool valid_v = v < nvec;
      const int row = valid_v ? sg.b * p.rows_per_seq + v / H : 0;
      const int hd = valid_v ? v % H : 0;
      const uint16_t* qn = valid_v ? p.q + row * p.q_row_stride + hd * p.q_head_stride : p.q;
      const uint16_t* qp =
          valid_v ? p.q_pe + row * p.q_pe_row_stride + hd * p.q_pe_head_stride : p.q_pe;
      uint32_t r[32];
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        const uint4* src = reinterpret_cast<const uint4*>(qn + c * 64);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 x = valid_v ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
          r[4 * j] = x.x;
          r[4 * j + 1] = x.y;
          r[4 * j + 2] = x.z;
          r[4 * j + 3] = x.w;
        }
        tc::st_32x32b_x32(tmem + lane_base + QN_COL + c * 32, r);
      }
      const uint4* srcp = reinterpret_cast<const uint4*>(qp);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4*>(qpe_s + sw_off(row_i, j)) =
            valid_v ? __ldg(srcp + j) : make_uint4(0, 0, 0, 0);
      tc::wait_st();
      tc::fence_before_sync();
      fence_proxy_async_smem();
      mbar_arrive(q_ready);
    };

    for_each_seg([&](const Seg1& sg, int k, int n0, const Seg1* next) -> bool {
      const int n1 = n0 + cdiv(sg.end - sg.start, TBN);
      const int v = sg.g * 128 + row_i;
      const bool valid_v = v < nvec;
      const int row = valid_v ? sg.b * p.rows_per_seq + v / H : 0;
      const int hd = valid_v ? v % H : 0;
      if (k == 0) load_q(sg);  // later segments' Q is loaded at the end of the previous one
      // A warp whose 32 rows are all padding (fewer than 128 query vectors
      // in the unit) does no softmax work: its rows of S, P and O are never
      // used (an MMA row depends only on the same row of A).  It keeps the
      // hand-off protocol: each arrival waits for the event that opens its
      // phase, so it never runs a phase ahead of the other warps.
      const bool live = __any_sync(0xffffffffu, valid_v);
      if (!live) {
        for (int n = n0; n < n1; ++n) {
          const int b = n & 1;
          if (!warp_wait(&s_full[b], (n >> 1) & 1)) { ok = false; break; }
          mbar_arrive(&s_free[b]);
          if (n >= 2 && !warp_wait(&pv_done[b], ((n - 2) >> 1) & 1)) { ok = false; break; }
          mbar_arrive(&p_full[b]);
        }
        if (!ok) return false;
        if (next) load_q(*next);
        if (!warp_wait(&pv_done[(n1 - 1) & 1], ((n1 - 1) >> 1) & 1)) { ok = false; return false; }
        mbar_arrive(o_free);
        return true;
      }
      float m_used = -INFINITY, l_run = 0.f;
      for (int n = n0; n < n1; ++n) {
        const int b = n & 1;
        if (!warp_wait(&s_full[b], (n >> 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        uint32_t sr[64];
        tc::ld_32x32b_x32(tmem + lane_base + S_COL + b * TBN,
                          *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tc::ld_32x32b_x32(tmem + lane_base + S_COL + b * TBN + 32,
                          *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tc::wait_ld();
        tc::fence_before_sync();
        mbar_arrive(&s_free[b]);
        tc::reg_fence(sr);
        // ---- online softmax with lazy rescaling (O is rescaled only when
        // the running max grows by more than 2^8)
        const int valid = min(TBN, sg.end - (sg.start + (n - n0) * TBN));
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float x = j < valid ? __uint_as_float(sr[j]) * scale_log2 : -INFINITY;
          sr[j] = __float_as_uint(x);
          mt = fmaxf(mt, x);
        }
        const float m_new = fmaxf(m_used, mt);
        float alpha = 1.f;
        if (m_new > m_used + kRescaleThreshold) {
          alpha = n > n0 ? ex2(m_used - m_new) : 1.f;
          l_run *= alpha;
          m_used = m_new;
        }
        uint32_t pk[32];
        float psum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float a0 = ex2(__uint_as_float(sr[2 * j]) - m_used);
          const float a1 = ex2(__uint_as_float(sr[2 * j + 1]) - m_used);
          psum[j & 3] += a0 + a1;
          pk[j] = pack_bf16x2(a0, a1);
        }
        l_run += (psum[0] + psum[1]) + (psum[2] + psum[3]);
        // ---- rescale this row of O once the previous P.V has completed
        if (n > n0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!warp_wait(&pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1)) { ok = false; break; }
          tc::fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < 256; c += 32) {
            uint32_t o[32];
            tc::ld_32x32b_x32(tmem + lane_base + c, o);
            tc::wait_ld();
            tc::reg_fence(o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tc::st_32x32b_x32(tmem + lane_base + c, o);
          }
          tc::wait_st();
        }
        // ---- P into buffer b, free once the P.V of tile n - 2 has run
        if (n >= 2 && !warp_wait(&pv_done[b], ((n - 2) >> 1) & 1)) { ok = false; break; }
        {
          uint8_t* dst = pbuf + b * P_BYTES;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(dst + sw_off(row_i, j)) =
                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
        tc::fence_before_sync();
        fence_proxy_async_smem();
        mbar_arrive(&p_full[b]);
      }
      if (!ok) return false;
      // ---- the next segment's Q first, so that its S products start while
      // this segment's O is read out
      if (next) load_q(*next);
      // ---- epilogue: this row of O (normalised) and lse
      if (!warp_wait(&pv_done[(n1 - 1) & 1], ((n1 - 1) >> 1) & 1)) { ok = false; return false; }
      tc::fence_after_sync();
      const float inv = kv_s / l_run;
      const int64_t rec = (static_cast<int64_t>(row) * S + sg.slot) * H + hd;
      auto store_cols = [&](int c, const uint32_t (&o)[32]) {
        if (!valid_v) return;
        if (sg.direct) {
          uint16_t* dst = p.o + (static_cast<int64_t>(row) * H + hd) * 256 + c;
#pragma unroll
          for (int j = 0; j < 32; j += 8)
            *reinterpret_cast<uint4*>(dst + j) = make_uint4(
                pack_bf16x2(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv),
                pack_bf16x2(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv),
                pack_bf16x2(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv),
                pack_bf16x2(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv));
        } else {
          float* dst = p.ws_o + rec * 256 + c;
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + j) =
                make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                            __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
        }
      };
      // two TMEM loads in flight: columns c + 32 come in while c is stored
      uint32_t oa[32], ob[32];
      tc::ld_32x32b_x32(tmem + lane_base, oa);
#pragma unroll 1
      for (int c = 0; c < 256; c += 64) {
        tc::wait_ld();
        tc::reg_fence(oa);
        tc::ld_32x32b_x32(tmem + lane_base + c + 32, ob);
        store_cols(c, oa);
        tc::wait_ld();
        tc::reg_fence(ob);
        if (c + 64 < 256) tc::ld_32x32b_x32(tmem + lane_base + c + 64, oa);
        store_cols(c + 32, ob);
      }
      tc::fence_before_sync();
      mbar_arrive(o_free);
      if (valid_v) {
        float lg;
        asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(l_run));
        const float lse = (m_used + lg) * kLn2;
        if (sg.direct) {
          p.lse[static_cast<int64_t>(row) * H + hd] = lse;
        } else {
          p.ws_lse[rec] = lse;
          for (int s = sg.mark_lo; s < sg.mark_hi; ++s)
            p.ws_lse[(static_cast<int64_t>(row) * S + s) * H + hd] = -INFINITY;
          for (int s = sg.mark2_lo; s < sg.mark2_hi; ++s)
            p.ws_lse[(static_cast<int64_t>(row) * S + s) * H + hd] = -INFINITY;
        }
      }
      return true;
    });
    if (!ok && lane == 0 && p.err_count) atomicAdd(p.err_count, kTimeoutErr);
  }

  // ---------------------------------------------------------------- teardown
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <bool FP8>
cudaError_t launch_tc1(const DecodeParams& p, const CUtensorMap& tmap, int split_group,
                       int sm_count, cudaStream_t stream) {
  using C = Tc1Cfg<FP8>;
  static std::atomic<uint64_t> attr_done{0};  // one bit per device
  cudaError_t e = set_smem_attr_once(decode_tc1_kernel<FP8>, C::SMEM, attr_done);
  if (e != cudaSuccess) return e;
  const int qblocks = (p.rows_per_seq * p.num_heads + 127) / 128;
  const int64_t units = static_cast<int64_t>(qblocks) * p.num_seqs;
  if (p.num_splits > 1 && units <= kMaxPersistUnits)
    return launch_overlapped(decode_tc1_kernel<FP8>, dim3(sm_count), dim3(C::NTHREADS), C::SMEM,
                             stream, p, tmap, split_group, 1);
  const int groups = (p.num_splits + split_group - 1) / split_group;
  const dim3 grid(qblocks, groups, p.num_seqs);
  return launch_overlapped(decode_tc1_kernel<FP8>, grid, dim3(C::NTHREADS), C::SMEM, stream, p,
                           tmap, split_group, 0);
}

}  // namespace

cudaError_t launch_decode_tc1(const DecodeParams& p, const CUtensorMap& tmap, bool fp8,
                              int split_group, int sm_count, cudaStream_t stream) {
  return fp8 ? launch_tc1<true>(p, tmap, split_group, sm_count, stream)
             : launch_tc1<false>(p, tmap, split_group, sm_count, stream);
}

}  // namespace mla
