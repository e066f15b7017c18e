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
// the work is split over a 2-CTA cluster by dims:
//   rank r holds latent dims [256 r, 256 r + 256) and rope dims
//   [32 r, 32 r + 32): its S partial over them, and O[:, 256 r : 256 r + 256)
// Each CTA loads only its own dims of every KV tile (no byte is read twice)
// and computes its partial S into TMEM.  The softmax of vector v is owned by
// one CTA (rank v / 64): the other CTA sends it its partial S row for v
// (fp32, bulk shared-memory copies per 32-token half), the owner adds the
// two partials, runs the online softmax and writes its P rows (bf16) into
// the P buffer of both CTAs (its own, and the peer's by a bulk copy, with
// the rows' rescale factors); both CTAs then accumulate their half of O with
// that buffer as the A operand.  Per tile and direction that is 16 KiB of
// scores plus 8 KiB of P, and each CTA evaluates only 64 x 64 exponentials.
//
// TMEM (512 columns): O [0, 256); S [256, 352) as a ring of three 32-token
// slots (S is computed per 32-token half, so the next tile's first half can
// be computed before this tile's S has been read); Q [352, 496) as packed
// bf16.  Q is an A operand read from TMEM; K and V tiles (a 4-stage ring of
// 64 tokens), the P buffers (two, by tile parity) and the exchange buffers
// live in shared memory.
//
// Roles per CTA (256 threads):
//   softmax: thread = TMEM lane = query vector.  The 64 vectors the peer
//              owns are forwarded by the two warps of their lane quarters
//              (partial scores out, the rescale factors of returned P in,
//              whichever is ready); the 64 this CTA owns get four warps,
//              two per lane quarter, each taking one half of the 64 tokens;
//              the two of a quarter share the row maximum and sum through
//              shared memory and send the quarter's P rows to the peer
//              (lazy rescaling of O only when the running max grows by more
//              than 2^8);
//   one warp   MMA issuer (one elected thread) and TMEM owner;
//   one warp   TMA producer: 64-token tiles of the paged cache into a
//              4-stage mbarrier ring (swizzled boxes).
//   The MMA and producer warps sit on the lane quarters (sub-partitions) of
//   the forwarding warps, the lighter softmax work.
//
// With several splits the kernel is persistent: one CTA pair per two SMs
// takes an equal share of all tiles of all (sequence, 128-vector block)
// units, cut into segments at unit boundaries, each segment yielding one
// partial (o, lse) in the unit's next split slot.
#include <cuda_bf16.h>
#include <stdint.h>

#include <type_traits>


#include "kernels.cuh"
#include "ptx.cuh"
#include "tc.cuh"

namespace mla {

namespace {

constexpr int TBN = 64;                   // tokens per tile
constexpr int TSTAGES = 4;                // KV ring depth
constexpr int TLAT = 4;                   // 64-dim latent chunks per CTA
constexpr int CHUNK_BYTES = TBN * 128;    // one 64-dim box of a tile (8 KiB)
constexpr int ROPE_BYTES = TBN * 64;      // the CTA's 32 rope dims of a tile
constexpr int STAGE_BYTES = TLAT * CHUNK_BYTES + ROPE_BYTES;
// Partial scores travel as two planes, one per 32-token half, each 64 rows
// of 128 bytes (the plane an own-row warp reads).
constexpr int XS_PLANE = 64 * 128;
constexpr int XS_BYTES = 2 * XS_PLANE;    // 64 vectors' partial scores of a tile
// P of a tile, the A operand of P.V: 128 rows (vectors) of 64 bf16 tokens,
// 128 bytes each, 128-byte swizzle; rows [64 r, 64 r + 64) are rank r's.
constexpr int P_BYTES = 128 * 128;
constexpr int P_HALF = 64 * 128;
constexpr int OFF_STAGE = 0;
constexpr int OFF_XIN = OFF_STAGE + TSTAGES * STAGE_BYTES;  // peer partials, x2
constexpr int OFF_P = OFF_XIN + 2 * XS_BYTES;               // P, x2 (own half + peer's)
constexpr int OFF_XOUT = OFF_P + 2 * P_BYTES;               // one plane per forwarding warp
constexpr int OFF_AIN = OFF_XOUT + 2 * (XS_PLANE / 2);      // peer's rescale factors, x2
constexpr int OFF_AOUT = OFF_AIN + 2 * 256;                 // own rescale factors
constexpr int OFF_FIN = OFF_AOUT + 256;                     // 1 / l from the peer
constexpr int OFF_RED = OFF_FIN + 256;                      // own rows: max / sum exchange
constexpr int OFF_PRE = OFF_RED + 6 * 64 * 4;               // schedule: unit tile prefix
constexpr int OFF_LEN = OFF_PRE + (kMaxPersistUnits + 1) * 4;  // schedule: sequence lengths
constexpr int OFF_BAR = (OFF_LEN + kMaxPersistUnits * 4 + 7) & ~7;
constexpr int NBARS = 2 * TSTAGES + 20;
constexpr int OFF_TMEMSLOT = OFF_BAR + NBARS * 8;
constexpr int TC_SMEM = OFF_TMEMSLOT + 16 + 1024;  // + alignment slack
constexpr int TC_THREADS = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 256;  // S, a ring of three 32-token fp32 slots (96 columns)
constexpr uint32_t Q_COL = 352;  // Q, 288 bf16 in 144 columns
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

static_assert(OFF_XIN % 1024 == 0 && OFF_P % 1024 == 0 && OFF_XOUT % 16 == 0 &&
                  OFF_AIN % 16 == 0 && OFF_AOUT % 16 == 0,
              "alignment");
static_assert(TC_SMEM <= 227 * 1024, "shared memory");

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// All lanes wait; the result is made warp-uniform.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity) {
  const bool ok = tc::mbar_wait_cluster(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// Byte offset of 16-byte chunk `c` of row `r` in an exchange buffer whose
// rows are `row_bytes` long: the chunk index is XORed with r mod 8 so that
// eight consecutive rows hit all 32 banks.
__device__ __forceinline__ uint32_t xoff(uint32_t r, uint32_t c, uint32_t row_bytes) {
  return r * row_bytes + ((c ^ (r & 7u)) << 4);
}

// One unit of work of a CTA pair: tokens [start, end) of sequence b for the
// 128-vector block g, whose result goes to split slot `slot` (or straight to
// o / lse when `direct`).  `mark_lo..mark_hi` and `mark2_lo..mark2_hi` are
// slots this segment marks unused (lse = -inf): fused splits in grid mode,
// or the slots the persistent partition leaves free (written by the first
// segment of a chunk).
struct TcSeg {
  int b, g, start, end, slot, mark_lo, mark_hi, mark2_lo, mark2_hi;
  bool direct;
};

constexpr int kClampedBit = 1 << 30;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(TC_THREADS, 1)
    decode_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmap,
                     const __grid_constant__ CUtensorMap rope_map, const int split_group,
                     const int persistent) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + TSTAGES;
  // S is computed in halves of 32 tokens; half e of tile t is ring position
  // q = 2 t + e, in TMEM slot q % 3, the (q / 3)-th use of that slot.
  uint64_t* s_slot_full = bars + 2 * TSTAGES;  // [3] S half landed in the slot
  uint64_t* s_slot_free = s_slot_full + 3;     // [3] the slot has been read
  uint64_t* p_full = s_slot_free + 3;   // [2] P.V inputs of tiles with this parity ready
  uint64_t* pv_done = p_full + 2;       // [2] P.V of tiles with this parity completed
  uint64_t* mma_done = pv_done + 2;
  uint64_t* xin_full = mma_done + 1;    // [2] peer partial scores landed
  uint64_t* pin_full = xin_full + 2;    // [2] peer P landed
  uint64_t* fin_full = pin_full + 2;    // peer's 1 / l landed (one per segment)
  uint64_t* q_ready = fin_full + 1;     // Q of the segment is in TMEM
  uint64_t* o_free = q_ready + 1;       // the segment's O has been read out
  uint64_t* peer_pv = o_free + 1;       // [2] the peer's P.V of tiles with this parity completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEMSLOT);
  int* pre = reinterpret_cast<int*>(smem + OFF_PRE);
  int* lens = reinterpret_cast<int*>(smem + OFF_LEN);

  const uint32_t rank = tc::cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  // This CTA's dims of the 576: latent [256 rank, 256 rank + 256) as four
  // 64-dim chunks and rope [32 rank, 32 rank + 32) (dims 512 + 32 rank on).
  const int c0 = TLAT * rank;  // first latent chunk
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The MMA issuer and the producer share the SM sub-partitions (warp % 4)
  // of the two softmax warps that only forward rows, not of the two that run
  // the softmax: warps 2, 3 forward on rank 0, warps 0, 1 on rank 1.
  const int mma_warp = rank == 0 ? 6 : 4;
  const int prod_warp = mma_warp + 1;
  const int H = p.num_heads;
  const int nvec = p.rows_per_seq * H;
  const int qblocks = cdiv(nvec, 128);
  const int S = p.num_splits;
  const int Lmax = p.max_blocks * p.block_size;
  if (threadIdx.x == 128) {
    tma_prefetch_desc(&tmap);
    tma_prefetch_desc(&rope_map);
  }
  // Launched overlapped with the previous kernel of the stream: nothing in
  // global memory is read before it has completed.
  griddep_wait();
  griddep_launch_dependents();

  // ---------------------------------------------------------- schedule
  // Persistent: the tiles of all units (sequence, 128-vector block) form one
  // list; pair c takes tiles [c * C, (c + 1) * C), cut into segments at unit
  // boundaries (the same walk as the warp-MMA kernel's).  Grid: one segment
  // per pair, split_group consecutive splits of one unit.
  int units = 0, C = 1, lo = 0, hi = 0, cidx = 0;
  // Sequences with several 128-vector blocks are cut into chunks of CH
  // tiles and listed chunk by chunk, all blocks of a chunk side by side, so
  // that the pairs holding the blocks of one chunk stream the same KV tiles
  // at about the same time and L2 serves all but the first reader.  A chunk
  // of one block spans at most SPC pairs and owns SPC split slots.
  int CH = 1 << 30, SPC = 1;
  TcSeg gseg{};
  int nseg = 0;
  if (persistent) {
    cidx = blockIdx.x >> 1;
    units = p.num_seqs * qblocks;
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
    const int npairs = gridDim.x >> 1;
    C = max(max(cdiv(total, npairs), cdiv(s_max, max(S - 1, 1))), 1);
    lo = cidx * C;
    hi = min(total, lo + C);
    SPC = S;  // one block per sequence: one chunk, slot = pair - first pair
    if (qblocks > 1) {
      // smallest m with (chunks) x (slots per chunk) <= S; m = cdiv(s_max, C)
      // (one chunk) always qualifies because C >= cdiv(s_max, S - 1)
      for (int m = 1;; ++m) {
        const int J = cdiv(s_max, C * m);
        if (J * (m + 1) <= S || J == 1) {
          CH = C * m;
          SPC = m + 1;
          break;
        }
      }
    }
    if (lo >= hi) return;  // both CTAs of the pair leave together
  } else {
    const int b = blockIdx.z, ysplit = blockIdx.y;
    int L = __ldg(p.seq_lens + b);
    if (L < 0) L = 0;
    if (L > Lmax) {
      if (threadIdx.x == 0 && rank == 0 && ysplit == 0 && (blockIdx.x >> 1) == 0 && p.err_count)
        atomicAdd(p.err_count, 1);
      L = Lmax;
    }
    const int per = L > 0 ? cdiv(cdiv(L, S), 64) * 64 : 64;
    const int s0 = ysplit * split_group;
    const int s1 = min(S, s0 + split_group);
    gseg.b = b;
    gseg.g = blockIdx.x >> 1;
    gseg.start = s0 * per;
    gseg.end = min(L, s1 * per);
    gseg.slot = s0;
    gseg.mark_lo = s0 + 1;
    gseg.mark_hi = s1;
    gseg.mark2_lo = gseg.mark2_hi = 0;
    gseg.direct = S == 1;
    if (gseg.start >= gseg.end) {
      // Both CTAs of the pair take this branch together.
      if (threadIdx.x < 128) {
        const int v = gseg.g * 128 + threadIdx.x;
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
    nseg = 1;
  }
  // Walks this pair's segments in order, calling f(seg, index, first tile
  // (a running count over the pair's segments), next segment or nullptr).
  // The pair's segment that starts at tile t of the list (lo <= t < hi);
  // returns the list position where the next segment starts.
  auto seg_at = [&](int t, TcSeg& s) -> int {
    int a = 0, z = p.num_seqs - 1;  // sequence b: the last with pre[b * qblocks] <= t
    while (a < z) {
      const int m = (a + z + 1) >> 1;
      if (pre[m * qblocks] <= t) a = m; else z = m - 1;
    }
    const int b = a;
    const int Ob = pre[b * qblocks];
    const int Tb = pre[b * qblocks + 1] - Ob;  // tiles of the sequence
    const int Jb = cdiv(Tb, CH);
    // list tiles of a full chunk (CH is 2^30 only with one block per sequence)
    const int span = qblocks * CH;
    const int x = t - Ob;
    const int j = min(x / span, Jb - 1);
    const int len = j == Jb - 1 ? Tb - (Jb - 1) * CH : CH;  // tiles of chunk j
    const int y = x - j * span;
    const int g = y / len;
    const int in = y - g * len;  // tile of the chunk where this segment starts
    const int vstart = Ob + j * span + g * len;
    const int vend = vstart + len;
    const int seg_end = min(hi, vend);
    const int L = lens[b] & ~kClampedBit;
    s.b = b;
    s.g = g;
    s.start = (j * CH + in) * TBN;
    s.end = min(L, (j * CH + in + (seg_end - t)) * TBN);
    const int cf = vstart / C;  // the pair where chunk j of block g begins
    s.slot = j * SPC + (cidx - cf);
    const bool first = cidx == cf;
    s.mark_lo = first ? j * SPC + ((vend - 1) / C - cf + 1) : 0;
    s.mark_hi = first ? (j + 1) * SPC : 0;
    s.mark2_lo = first && j == 0 ? Jb * SPC : 0;  // slots past the last chunk
    s.mark2_hi = first && j == 0 ? S : 0;
    s.direct = false;
    return seg_end;
  };
  auto for_each_seg = [&](auto&& f) {
    if (!persistent) {
      if (nseg) f(gseg, 0, 0, static_cast<const TcSeg*>(nullptr));
      return;
    }
    if (lo >= hi) return;
    TcSeg cur, nxt;
    int t_next = seg_at(lo, cur);
    for (int k = 0, n0 = 0;; ++k) {
      const bool more = t_next < hi;
      int t_after = hi;
      if (more) t_after = seg_at(t_next, nxt);
      if (cur.slot == 0 && cur.g == 0 && (lens[cur.b] & kClampedBit) && threadIdx.x == 0 &&
          rank == 0 && p.err_count)
        atomicAdd(p.err_count, 1);  // seq_len beyond the block table, once per sequence
      if (!f(cur, k, n0, more ? &nxt : static_cast<const TcSeg*>(nullptr))) return;
      if (!more) return;
      n0 += cdiv(cur.end - cur.start, TBN);
      cur = nxt;
      t_next = t_after;
    }
  };

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    for (int i = 0; i < TSTAGES; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(&s_slot_full[i], 1);
      // an S half is read by the 64 forwarding threads and the 64 own-row
      // threads of its token half
      mbar_init(&s_slot_free[i], 128);
    }
    // Q / O hand-offs: 64 forwarding + 128 own-row threads; P: the six
    // softmax warps
    mbar_init(&p_full[0], 6);
    mbar_init(&p_full[1], 6);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&pv_done[i], 1);
      mbar_init(&peer_pv[i], 1);  // arrived by the peer's tensor-core commit
    }
    mbar_init(mma_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&xin_full[i], 1);  // local expect-tx arrival + the peer's bytes
      mbar_init(&pin_full[i], 1);
    }
    mbar_init(fin_full, 1);
    mbar_init(q_ready, 192);
    mbar_init(o_free, 192);
    fence_mbar_init();
  }
  if (warp == mma_warp) {
    tc::tmem_alloc(tmem_slot, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::cluster_sync();  // the peer's barriers exist before any remote traffic
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t stage_base = smem_u32(smem + OFF_STAGE);
  const uint32_t p_base = smem_u32(smem + OFF_P);

  if (warp == prod_warp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const int bs = p.block_size;
      const int rows_box = bs < TBN ? bs : TBN;
      const int npg = TBN / rows_box;
      int n = 0;  // tiles issued (ring position)
      for_each_seg([&](const TcSeg& sg, int, int, const TcSeg*) -> bool {
        const int32_t* bt = p.block_table + static_cast<int64_t>(sg.b) * p.bt_stride;
        const int ntiles = cdiv(sg.end - sg.start, TBN);
        // Block ids of tile t of the segment (pages past its end read as 0
        // and are not loaded).
        auto ids_of = [&](int t, int (&ids)[4]) {
#pragma unroll
          for (int pg = 0; pg < 4; ++pg) {
            const int tk = sg.start + t * TBN + pg * rows_box;
            ids[pg] = (pg < npg && t < ntiles && tk < sg.end) ? __ldg(bt + tk / bs) : 0;
          }
        };
        auto pages_of = [&](int t) {
          int np = 0;
          for (int pg = 0; pg < npg; ++pg)
            if (sg.start + t * TBN + pg * rows_box < sg.end) ++np;
          return t < ntiles ? np : 0;
        };
        // Ids are read one tile before they are used, so the block-table
        // latency hides behind a tile's worth of waiting.
        int cur[4], nxt[4];
        ids_of(0, cur);
        for (int t = 0; t < ntiles; ++t, ++n) {
          ids_of(t + 1, nxt);
          const int st = n % TSTAGES;
          const uint32_t ph = (n / TSTAGES) & 1;
          if (!mbar_wait(&kv_empty[st], ph ^ 1)) {
            if (p.err_count) atomicAdd(p.err_count, kTimeoutErr);
            return false;
          }
          const int npages = pages_of(t);
          mbar_arrive_expect_tx(&kv_full[st],
                                static_cast<uint32_t>(npages * rows_box * (TLAT * 128 + 64)));
          uint8_t* dst = smem + OFF_STAGE + st * STAGE_BYTES;
#pragma unroll
          for (int pg = 0; pg < 4; ++pg) {
            if (pg >= npages) break;
            const int tk = sg.start + t * TBN + pg * rows_box;
            const int blk = cur[pg];
            const int row0 = tk % bs;
            if ((blk < 0 || blk >= p.num_blocks) && p.err_count && rank == 0)
              atomicAdd(p.err_count, 1);
            for (int cl = 0; cl < TLAT; ++cl)
              tma_load_3d(dst + cl * CHUNK_BYTES + pg * rows_box * 128, &tmap,
                          &kv_full[st], (c0 + cl) * 64, row0, blk);
            tma_load_3d(dst + TLAT * CHUNK_BYTES + pg * rows_box * 64, &rope_map, &kv_full[st],
                        512 + 32 * static_cast<int>(rank), row0, blk);
          }
#pragma unroll
          for (int pg = 0; pg < 4; ++pg) cur[pg] = nxt[pg];
        }
        return true;
      });
    }
  } else if (warp == mma_warp) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idS = tc::idesc_bf16(128, TBN / 2, 0, 0);
    constexpr uint32_t idPV = tc::idesc_bf16(128, 256, 0, 1);
    // Half e of S of tile n (ring position q = 2n + e) needs its KV stage,
    // its TMEM slot (the readers of position q - 3 are done) and, first in
    // a segment, the segment's Q; P.V of tile n needs P of tile n and, first
    // in a segment, the previous segment's O read out.  Within a segment the
    // two streams are issued as soon as each is ready (P.V first), so S
    // runs ahead of the P round trip between the CTAs.
    bool ok = true;
    int qs = 0, npv = 0;  // global S ring position, global P.V tile counter
    for_each_seg([&](const TcSeg& sg, int k, int n0, const TcSeg*) -> bool {
      const int n1 = n0 + cdiv(sg.end - sg.start, TBN);
      uint64_t t_idle = 0;
      uint32_t spins = 0;
      bool have_q = false, have_o = k == 0;
      while (npv < n1) {
        bool progress = false;
        // (lane 0 decides, so the warp stays converged)
        if (!have_o) have_o = __shfl_sync(0xffffffffu, mbar_test(o_free, (k - 1) & 1), 0);
        const bool pv_ready =
            have_o && __shfl_sync(0xffffffffu,
                                  npv < (qs >> 1) && mbar_test(&p_full[npv & 1], (npv >> 1) & 1),
                                  0);
        if (pv_ready) {
          tc::fence_after_sync();
          if (tc::elect_one()) {
            // A = P (shared memory, K-major with 128-byte swizzle, 8-row
            // groups 1024 B apart; 16 tokens = 32 B = 2 in the address
            // field per step); B = V: MN-major, 128-byte swizzle (N step =
            // next 64-dim box, K step = 8 tokens = 1024 B; 16 tokens per MMA
            // = 2048 B = 128 in the address field).
            const uint64_t d0 = tc::smem_desc(stage_base + (npv % TSTAGES) * STAGE_BYTES,
                                              CHUNK_BYTES, 1024, tc::kLayoutSw128);
            const uint64_t da =
                tc::smem_desc(p_base + (npv & 1) * P_BYTES, 16, 1024, tc::kLayoutSw128);
#pragma unroll
            for (int kk = 0; kk < TBN / 16; ++kk)
              tc::mma_ss(tmem, da + static_cast<uint64_t>(kk * 2),
                         d0 + static_cast<uint64_t>(kk * 128), idPV,
                         (npv > n0 || kk > 0) ? 1u : 0u);
            tc::commit(&pv_done[npv & 1]);
            // (the peer may then write the P of tile npv + 2 into this
            // CTA's buffer npv & 1)
            tc::commit_multicast(&peer_pv[npv & 1], static_cast<uint16_t>(1u << peer));
            tc::commit(&kv_empty[npv % TSTAGES]);
          }
          __syncwarp();
          ++npv;
          progress = true;
        }
        if (!have_q) have_q = __shfl_sync(0xffffffffu, mbar_test(q_ready, k & 1), 0);
        const int ns = qs >> 1, e = qs & 1;  // tile and token half of position qs
        const bool s_ready =
            have_q &&
            __shfl_sync(0xffffffffu,
                        ns < n1 && mbar_test(&kv_full[ns % TSTAGES], (ns / TSTAGES) & 1) &&
                            (qs < 3 || mbar_test(&s_slot_free[qs % 3], ((qs - 3) / 3) & 1)),
                        0);
        if (s_ready) {
          const int st = ns % TSTAGES;
          const int valid = min(TBN, sg.end - (sg.start + (ns - n0) * TBN));
          if (e == 0 && valid < TBN) {
            // Rows past the segment end hold other tokens or NaN: zero their
            // latent part so the P.V product sees 0 * 0 there (their scores
            // are masked; the rope part only enters those scores).
            uint8_t* stp = smem + OFF_STAGE + st * STAGE_BYTES;
            const int nz = (TBN - valid) * TLAT * 8;
            for (int i = lane; i < nz; i += 32) {
              const int r = valid + i / (TLAT * 8), rem = i % (TLAT * 8);
              *reinterpret_cast<uint4*>(stp + (rem >> 3) * CHUNK_BYTES + r * 128 +
                                        (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          tc::fence_after_sync();
          if (tc::elect_one()) {
            // S half e = Q K^T over tokens [32 e, 32 e + 32): A = Q from
            // TMEM (16 dims = 8 packed columns per step), B = those 32 K
            // rows, K-major: the latent chunks with 128-byte swizzle (8-row
            // groups 1024 B apart, 32 rows = 4096 B), then the rope part with
            // 64-byte swizzle (groups 512 B apart, 32 rows = 2048 B).  The
            // descriptor's start-address field (bytes / 16) is advanced by
            // addition: one 64-dim box is CHUNK_BYTES / 16, one 16-dim step 2.
            const uint32_t sa = stage_base + st * STAGE_BYTES;
            const uint32_t dS = tmem + S_COL + (qs % 3) * 32;
            const uint64_t d0 = tc::smem_desc(sa + e * 4096, 16, 1024, tc::kLayoutSw128);
            const uint64_t dr =
                tc::smem_desc(sa + TLAT * CHUNK_BYTES + e * 2048, 16, 512, tc::kLayoutSw64);
#pragma unroll
            for (int ks = 0; ks < TLAT * 4; ++ks)
              tc::mma_ts(dS, tmem + Q_COL + ks * 8,
                         d0 + static_cast<uint64_t>((ks >> 2) * (CHUNK_BYTES >> 4) + (ks & 3) * 2),
                         idS, ks > 0 ? 1u : 0u);
#pragma unroll
            for (int kr = 0; kr < 2; ++kr)
              tc::mma_ts(dS, tmem + Q_COL + TLAT * 32 + kr * 8,
                         dr + static_cast<uint64_t>(kr * 2), idS, 1u);
            tc::commit(&s_slot_full[qs % 3]);
          }
          __syncwarp();
          ++qs;
          progress = true;
        }
        if (progress) {
          t_idle = 0;
          spins = 0;
        } else if ((++spins & 1023u) == 0) {
          // bounded: give up when nothing became ready for the wait limit
          // (the timer is read every 1024 idle polls; it is slow to read)
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
  } else if (warp != mma_warp && warp != prod_warp) {
    // ------------------------------------------------------------ softmax
    // Thread = TMEM lane = query vector row_i.  The vectors the peer owns are
    // forwarded by the two warps of their lane quarters; the vectors this CTA
    // owns get two warps per lane quarter, one per half of the 64 tokens
    // (h), which share the row maximum and sum through shared memory.
    const int quad = warp & 3;
    const int row_i = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const bool own = static_cast<uint32_t>(row_i >> 6) == rank;
    const int h = warp >> 2;        // token half (own rows); 0 on forwarding warps
    const int xi = row_i & 63;      // row within the 64-vector exchange blocks
    const bool lead = xi == 0 && h == 0;  // registers the expected bytes of each message
    // (own rows) the lane quarter among the CTA's two, and the thread that
    // sends that quarter's P rows and rescale factors to the peer
    const int oq = xi >> 5;
    const bool qlead = own && h == 0 && (xi & 31) == 0;
    const float scale_log2 = p.sm_scale * kLog2e;
    const uint8_t* xin = smem + OFF_XIN;
    uint8_t* pbuf = smem + OFF_P;
    const float* ain = reinterpret_cast<const float*>(smem + OFF_AIN);
    float* aout = reinterpret_cast<float*>(smem + OFF_AOUT);
    float* red = reinterpret_cast<float*>(smem + OFF_RED);  // [2 tiles][2 halves][64]
    float* lred = red + 2 * 2 * 64;                          // [2 halves][64]
    // The peer's buffers and barriers (bulk copies and st.async stores
    // complete their bytes on the receiving CTA's barrier).
    const uint32_t xin_peer = tc::map_peer(smem_u32(smem + OFF_XIN), peer);
    const uint32_t p_peer = tc::map_peer(p_base, peer);
    const uint32_t ain_peer = tc::map_peer(smem_u32(smem + OFF_AIN), peer);
    const uint32_t fin_peer = tc::map_peer(smem_u32(smem + OFF_FIN), peer);
    const uint32_t xin_bar_peer0 = tc::map_peer(smem_u32(&xin_full[0]), peer);
    const uint32_t pin_bar_peer0 = tc::map_peer(smem_u32(&pin_full[0]), peer);
    const uint32_t fin_bar_peer = tc::map_peer(smem_u32(fin_full), peer);
    bool ok = true;
    // Meeting of the two warps (one per token half) of a lane quarter of
    // this CTA's own rows (named barrier 1 or 2), which also ANDs their
    // flags.  Every wait of theirs is bounded, so each reaches every
    // meeting; one that gave up on a wait passes false, and both take the
    // same exit after the meeting.  The two quarters share no data and move
    // on independently.
    auto own_sync = [&](bool good) -> bool { return named_bar_and(1 + oq, 64, good); };
    // This thread's O columns: all 256 on forwarding rows, half on own rows.
    const int o_c0 = own ? 128 * h : 0, o_c1 = own ? 128 * h + 128 : 256;
    // P.V of tile m has completed.  pv_done[m & 1] completes once per two
    // tiles; every caller waits for m before P.V of m + 2 can have been
    // issued, so the parity is never two phases behind.
    auto pv_wait = [&](int m) -> bool { return warp_wait(&pv_done[m & 1], (m >> 1) & 1); };

    // Rescales this thread's O columns by alpha once the previous P.V has
    // completed; warp-uniform (lanes with alpha = 1 keep their values).  Not
    // needed on a segment's first tile (O is empty).
    auto rescale_o = [&](int n, int n0, float alpha) -> bool {
      if (n == n0 || !__any_sync(0xffffffffu, alpha != 1.f)) return true;
      if (!pv_wait(n - 1)) return false;
      tc::fence_after_sync();
#pragma unroll 1
      for (int c = o_c0; c < o_c1; c += 32) {
        uint32_t o[32];
        tc::ld_32x32b_x32(tmem + lane_base + c, o);
        tc::wait_ld();
        tc::reg_fence(o);
#pragma unroll
        for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
        tc::st_32x32b_x32(tmem + lane_base + c, o);
      }
      tc::wait_st();
      return true;
    };
    // This warp's part of tile n's P.V inputs is in place (its O rows
    // rescaled, its P rows written and made visible to the async proxy).
    // One barrier per tile parity: a warp's arrival for tile n + 2 comes
    // after P.V of tile n has completed (owners wait for it before writing
    // P; forwarders arrive once the peer's P of tile n + 2 has landed, which
    // the peer sends only after this CTA's tensor core signalled that P.V),
    // so the phases of one barrier never mix two tiles.
    auto p_ready = [&](int n) {
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[n & 1]);
    };
    // S ring position q: its slot's columns, wait and release.
    auto s_col = [&](int q) -> uint32_t { return tmem + lane_base + S_COL + (q % 3) * 32; };
    auto s_test = [&](int q) -> bool { return mbar_test(&s_slot_full[q % 3], (q / 3) & 1); };
    auto s_done = [&](int q) {
      tc::wait_ld();
      tc::fence_before_sync();
      mbar_arrive(&s_slot_free[q % 3]);
    };

    // ---- Q of a segment: this thread's vector, the CTA's latent dims (four
    // 64-dim chunks) and then its 32 rope dims, into TMEM lane row_i as
    // packed bf16 pairs (padding vectors are zeros); on own rows one warp
    // takes chunks 0-1, the other chunks 2-3 and the rope part.  Called once
    // the previous segment's S products, which read Q, are complete.
    auto load_q = [&](const TcSeg& sg) {
      const int v = sg.g * 128 + row_i;
      const bool valid_v = v < nvec;
      const int row = valid_v ? sg.b * p.rows_per_seq + v / H : 0;
      const int hd = valid_v ? v % H : 0;
      const int q_lo = own ? 2 * h : 0, q_hi = own ? 2 * h + 2 : TLAT;
      const bool q_rope = !own || h == 1;
      // dims [0, 512) come from q_nope, [512, 576) from q_pe
      const uint16_t* qn = valid_v ? p.q + row * p.q_row_stride + hd * p.q_head_stride : p.q;
      const uint16_t* qp =
          valid_v ? p.q_pe + row * p.q_pe_row_stride + hd * p.q_pe_head_stride : p.q_pe;
      uint32_t r[2][32];
      auto load_chunk = [&](int c, uint32_t (&d)[32]) {
        const uint4* src = reinterpret_cast<const uint4*>(qn + (c0 + c) * 64);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 x = valid_v ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
          d[4 * j] = x.x;
          d[4 * j + 1] = x.y;
          d[4 * j + 2] = x.z;
          d[4 * j + 3] = x.w;
        }
      };
      // the loads of chunk c + 1 are issued before chunk c goes to TMEM
      load_chunk(q_lo, r[0]);
#pragma unroll 1
      for (int c = q_lo; c < q_hi; c += 2) {
        if (c + 1 < q_hi) load_chunk(c + 1, r[1]);
        tc::st_32x32b_x32(tmem + lane_base + Q_COL + c * 32, r[0]);
        if (c + 1 < q_hi) {
          if (c + 2 < q_hi) load_chunk(c + 2, r[0]);
          tc::st_32x32b_x32(tmem + lane_base + Q_COL + (c + 1) * 32, r[1]);
        }
      }
      if (q_rope) {
        const uint4* src = reinterpret_cast<const uint4*>(qp + 32 * rank);
        uint32_t d[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 x = valid_v ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
          d[4 * j] = x.x;
          d[4 * j + 1] = x.y;
          d[4 * j + 2] = x.z;
          d[4 * j + 3] = x.w;
        }
        tc::st_32x32b_x16(tmem + lane_base + Q_COL + TLAT * 32, d);
      }
      tc::wait_st();
      tc::fence_before_sync();
      mbar_arrive(q_ready);
    };
    // L2 prefetch of a segment's Q lines for this thread (used at its start)
    auto prefetch_q = [&](const TcSeg& sg) {
      const int v = sg.g * 128 + row_i;
      if (v >= nvec) return;
      const int row = sg.b * p.rows_per_seq + v / H, hd = v % H;
      const uint16_t* qn = p.q + row * p.q_row_stride + hd * p.q_head_stride;
      const uint16_t* qp = p.q_pe + row * p.q_pe_row_stride + hd * p.q_pe_head_stride;
      for (int c = 0; c < TLAT; ++c)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qn + (c0 + c) * 64));
      asm volatile("prefetch.global.L2 [%0];" ::"l"(qp + 32 * rank));
    };

    for_each_seg([&](const TcSeg& sg, int k, int n0, const TcSeg* next) -> bool {
      const int n1 = n0 + cdiv(sg.end - sg.start, TBN);
      const int v = sg.g * 128 + row_i;
      const bool valid_v = v < nvec;
      const int row = valid_v ? sg.b * p.rows_per_seq + v / H : 0;
      const int hd = valid_v ? v % H : 0;
      if (k == 0) load_q(sg);  // later segments' Q is loaded at the end of the previous one
      if (next) prefetch_q(*next);
      float m_used = -INFINITY, l_run = 0.f;

      if (!own) {
        // Forwarding rows.  Each warp handles the P of tile np as soon as
        // it has come back (first: it gates the P.V that frees a KV stage;
        // only the rescale factors are read, P itself is the MMA's operand
        // in place) and sends its rows' partial scores of tile ns as soon as
        // S is there.  ns <= np + 1 keeps the answer barrier of tile ns - 2
        // observed before it is armed again, and the rescale factors of
        // tile ns - 2 read before the peer can send those of tile ns.
        const int fw = xi >> 5;  // which of the two forwarding warps
        uint8_t* xo = smem + OFF_XOUT + fw * (XS_PLANE / 2);
        int fq = 2 * n0, np = n0;  // next S ring position to forward, next P tile
        uint64_t t_idle = 0;
        uint32_t spins = 0;
        while (np < n1) {
          bool did = false;
          if (np < (fq >> 1) &&
              __shfl_sync(0xffffffffu, tc::mbar_test_cluster(&pin_full[np & 1], (np >> 1) & 1),
                          0)) {
            const float alpha = ain[(np & 1) * 64 + xi];
            if (!rescale_o(np, n0, alpha)) { ok = false; break; }
            p_ready(np);
            ++np;
            did = true;
          }
          const int ns = fq >> 1, e = fq & 1;  // tile and token half of position fq
          if (ns < n1 && ns <= np + 1 && __shfl_sync(0xffffffffu, s_test(fq), 0)) {
            tc::fence_after_sync();
            uint32_t sr[32];
            tc::ld_32x32b_x32(s_col(fq), sr);
            s_done(fq);
            tc::reg_fence(sr);
            const int bb = ns & 1;
            if (e == 0 && lead) mbar_arrive_expect_tx(&pin_full[bb], P_HALF + 256);  // P of ns
            // The warp's 32 rows of this token half (plane e) are staged in
            // its 4 KiB buffer (once the previous plane's copy has read it)
            // and handed to the peer as one bulk copy; scaled by sm_scale *
            // log2(e), so that the owner's sum is one fused multiply-add.
            if (lane == 0) tc::bulk_wait_read();
            __syncwarp();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(xo + xoff(xi & 31, j, 128)) = make_uint4(
                  __float_as_uint(__uint_as_float(sr[4 * j]) * scale_log2),
                  __float_as_uint(__uint_as_float(sr[4 * j + 1]) * scale_log2),
                  __float_as_uint(__uint_as_float(sr[4 * j + 2]) * scale_log2),
                  __float_as_uint(__uint_as_float(sr[4 * j + 3]) * scale_log2));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0)
              tc::bulk_copy_to_peer(xin_peer + bb * XS_BYTES + e * XS_PLANE + fw * 32 * 128, xo,
                                    32 * 128, xin_bar_peer0 + bb * 8);
            ++fq;
            did = true;
          }
          if (did) {
            t_idle = 0;
            spins = 0;
          } else if ((++spins & 1023u) == 0) {
            const uint64_t now = globaltimer();
            if (t_idle == 0) {
              t_idle = now;
            } else if (now - t_idle > kWaitTimeoutNs) {
              ok = false;
              break;
            }
          }
        }
        if (lane == 0) tc::bulk_wait_read();  // the local copy is read before leaving
      } else {
        bool bad = false;  // this warp gave up on a wait since the last meeting
        for (int n = n0; n < n1; ++n) {
          const int bb = n & 1;              // exchange buffer
          const uint32_t u = (n >> 1) & 1;   // its phase parity
          uint32_t sr[32];
          float mt = -INFINITY;
          // ---- this half's 32 partial scores
          const int q = 2 * n + h;  // S ring position of this half
          if (!bad && warp_wait(&s_slot_full[q % 3], (q / 3) & 1)) {
            tc::fence_after_sync();
            tc::ld_32x32b_x32(s_col(q), sr);
            s_done(q);
            tc::reg_fence(sr);
            // The P buffer of parity bb: P.V of tile n - 2 has read this
            // CTA's half of it, and the peer's P.V of tile n - 2 its half in
            // the peer, where this tile's copy goes (checked before the wait
            // for the peer's partial scores, which it overlaps).
            if (n >= 2 && !pv_wait(n - 2)) bad = true;
            if (!bad && h == 0 && n >= 2 &&
                !warp_wait_cluster(&peer_pv[bb], ((n - 2) >> 1) & 1))
              bad = true;
            // ---- add the peer's partial scores for them (xin[bb] is not
            // rewritten before the peer has received this tile's P)
            if (lead) mbar_arrive_expect_tx(&xin_full[bb], XS_BYTES);
            if (!bad && warp_wait_cluster(&xin_full[bb], u)) {
              const uint8_t* src = xin + bb * XS_BYTES + h * XS_PLANE;  // this half's plane
              const int valid = min(TBN, sg.end - (sg.start + (n - n0) * TBN)) - 32 * h;
              // x = (own partial + peer partial) * sm_scale * log2(e), the
              // peer's part arriving scaled; tokens past the segment end
              // (only in its last tile) get -inf
              auto add_partials = [&](auto masked) {
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                  const float4 t = *reinterpret_cast<const float4*>(src + xoff(xi, j4, 128));
                  const float tv[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const int j = 4 * j4 + e;
                    float x = fmaf(__uint_as_float(sr[j]), scale_log2, tv[e]);
                    if (decltype(masked)::value) x = j < valid ? x : -INFINITY;
                    sr[j] = __float_as_uint(x);
                    mt = fmaxf(mt, x);
                  }
                }
              };
              if (valid >= 32)
                add_partials(std::false_type());
              else
                add_partials(std::true_type());
            } else {
              bad = true;
            }
          } else {
            bad = true;
          }
          // ---- row maximum over both halves (buffer by tile parity: the
          // other half reads this tile's value before either writes the
          // tile after next's)
          red[(bb * 2 + h) * 64 + xi] = mt;
          // (the previous tile's bulk copies have read this quarter's P rows
          // and factors)
          if (qlead) tc::bulk_wait_read();
          if (!own_sync(!bad)) { ok = false; break; }
          mt = fmaxf(red[(bb * 2) * 64 + xi], red[(bb * 2 + 1) * 64 + xi]);
          // ---- online softmax with lazy rescaling (both halves take the
          // same decision from the same values)
          const float m_new = fmaxf(m_used, mt);
          float alpha = 1.f;
          if (m_new > m_used + kRescaleThreshold) {
            alpha = n > n0 ? ex2(m_used - m_new) : 1.f;
            l_run *= alpha;
            m_used = m_new;
          }
          uint32_t pk[16];
          float psum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float a0 = ex2(__uint_as_float(sr[2 * j]) - m_used);
            const float a1 = ex2(__uint_as_float(sr[2 * j + 1]) - m_used);
            psum[j & 3] += a0 + a1;
            pk[j] = pack_bf16x2(a0, a1);
          }
          l_run += (psum[0] + psum[1]) + (psum[2] + psum[3]);
          // ---- this half of P into the P buffer of tile parity bb (its
          // rows of this CTA); then the quarter's 32 rows and rescale
          // factors go to the same place in the peer's buffer as one bulk
          // copy each, which run in the background.
          uint8_t* pdst = pbuf + bb * P_BYTES + rank * P_HALF;
          {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(pdst + xoff(xi, 4 * h + j, 128)) =
                  make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
            if (h == 0) aout[xi] = alpha;
            fence_proxy_async_smem();  // read by the MMA and the bulk copies
          }
          own_sync(true);  // (no wait since the last meeting)
          if (qlead) {
            tc::bulk_copy_to_peer(p_peer + bb * P_BYTES + rank * P_HALF + oq * (P_HALF / 2),
                                  pdst + oq * (P_HALF / 2), P_HALF / 2, pin_bar_peer0 + bb * 8);
            tc::bulk_copy_to_peer(ain_peer + bb * 256 + oq * 128, aout + oq * 32, 128,
                                  pin_bar_peer0 + bb * 8);
          }
          if (!rescale_o(n, n0, alpha)) {
            bad = true;  // the next meeting ends the loop
            continue;
          }
          p_ready(n);
        }
        // ---- row sum over both halves (both warps of a quarter leave the
        // loop together, so both come here; a failure in the last tile's
        // second half shows at this meeting)
        if (ok) {
          lred[h * 64 + xi] = l_run;
          if (!own_sync(!bad)) ok = false;
          l_run = lred[xi] + lred[64 + xi];
        }
        // the last copy has read the outbound buffer before this CTA can
        // leave (the next segment's first tile waits for it anyway)
        if (qlead) tc::bulk_wait_read();
      }

      // ---- the owner's 1 / l reaches the other CTA as the segment's last
      // message (the peer read the previous segment's before it sent any
      // partial scores of this one)
      float inv = 0.f;
      if (ok) {
        if (own) {
          inv = 1.f / l_run;
          if (h == 0) tc::st_async_b32(fin_peer + 4 * xi, __float_as_uint(inv), fin_bar_peer);
        } else {
          if (lead) mbar_arrive_expect_tx(fin_full, 64 * 4);
          if (warp_wait_cluster(fin_full, k & 1))
            inv = reinterpret_cast<const float*>(smem + OFF_FIN)[xi];
          else
            ok = false;
        }
      }
      if (!ok) return false;
      // ---- the next segment's Q first, so that its S products start while
      // this segment's O is read out.  Every S half reads all of Q: the
      // own-row warps of the first token half, which read no second half,
      // first wait for the last tile's second half to complete.
      bool q_ok = true;
      if (next) {
        if (own && h == 0) {
          const int ql = 2 * (n1 - 1) + 1;
          q_ok = warp_wait(&s_slot_full[ql % 3], (ql / 3) & 1);
        }
        if (q_ok) load_q(*next);
      }
      // ---- epilogue: this thread's O columns (normalised) and, from the
      // owner, lse
      const bool pv_ok = pv_wait(n1 - 1) && q_ok;
      if ((own && !own_sync(pv_ok)) || !pv_ok) {  // a quarter's owners leave together
        ok = false;
        return false;
      }
      tc::fence_after_sync();
      const int64_t rec = (static_cast<int64_t>(row) * S + sg.slot) * H + hd;
      // two TMEM loads in flight: columns c + 32 come in while c is stored
      auto store_cols = [&](int c, const uint32_t (&o)[32]) {
        if (!valid_v) return;
        const int col = rank * 256 + c;
        if (sg.direct) {
          uint16_t* dst = p.o + (static_cast<int64_t>(row) * H + hd) * 512 + col;
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
      };
      uint32_t oa[32], ob[32];
      tc::ld_32x32b_x32(tmem + lane_base + o_c0, oa);
#pragma unroll 1
      for (int c = o_c0; c < o_c1; c += 64) {
        tc::wait_ld();
        tc::reg_fence(oa);
        tc::ld_32x32b_x32(tmem + lane_base + c + 32, ob);  // o_c1 - o_c0 is a multiple of 64
        store_cols(c, oa);
        tc::wait_ld();
        tc::reg_fence(ob);
        if (c + 64 < o_c1) tc::ld_32x32b_x32(tmem + lane_base + c + 64, oa);
        store_cols(c + 32, ob);
      }
      tc::fence_before_sync();
      mbar_arrive(o_free);
      if (valid_v && own && h == 0) {
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
  tc::cluster_sync();  // no CTA leaves while its peer may still write to it
  if (warp == mma_warp) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

int tc_split_group(const DecodeParams& p, int sm_count, int ctas_per_unit) {
  // Fuse consecutive splits into one CTA pair (ctas_per_unit 2) or CTA (1).
  // With f splits per pair the launch has units * ceil(S / f) pairs; the
  // estimated cost (in units of one split's KV stream) is the number of
  // waves times the work of one pair, plus the partial outputs each pair
  // writes and the merge reads back (about 0.85 of a split's bytes per
  // 128-vector unit).  Pick f with the lowest cost.
  const int qblocks = (p.rows_per_seq * p.num_heads + 127) / 128;
  const int64_t units = static_cast<int64_t>(qblocks) * p.num_seqs;
  const int64_t pairs = sm_count >= ctas_per_unit ? sm_count / ctas_per_unit : 1;
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
                             const CUtensorMap& rope_map, int split_group, int sm_count,
                             cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};  // one bit per device
  cudaError_t e = set_smem_attr_once(decode_tc_kernel, TC_SMEM, attr_done);
  if (e != cudaSuccess) return e;
  const int qblocks = (p.rows_per_seq * p.num_heads + 127) / 128;
  const int64_t units = static_cast<int64_t>(qblocks) * p.num_seqs;
  if (p.num_splits > 1 && units <= kMaxPersistUnits) {
    // persistent: one CTA pair per two SMs, tiles balanced over the pairs
    const int pairs = sm_count >= 2 ? sm_count / 2 : 1;
    return launch_overlapped(decode_tc_kernel, dim3(2 * pairs), dim3(TC_THREADS), TC_SMEM,
                             stream, p, tmap, rope_map, split_group, 1);
  }
  const int groups = (p.num_splits + split_group - 1) / split_group;
  const dim3 grid(2 * qblocks, groups, p.num_seqs);
  return launch_overlapped(decode_tc_kernel, grid, dim3(TC_THREADS), TC_SMEM, stream, p, tmap,
                           rope_map, split_group, 0);
}

}  // namespace mla
