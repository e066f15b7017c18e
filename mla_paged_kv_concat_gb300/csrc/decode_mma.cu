// Split-KV MLA decode, stage 1, on warp-level tensor-core MMA.
//
// Restates "frozenleaves/vllm compare v0.11.0...mla_cuda_graphs",
// vllm/attention/ops/triton_decode_attention.py, _fwd_grouped_kernel_stage1:
// a program streams its split's tokens through the block table, computes q.k
// over the latent and rope parts, scales, runs an online softmax and
// accumulates P.V with V the latent part of the same row; it emits the
// normalised split output and its lse.
//
// GB300 design (not the page's):
//   * A "unit" is 16*MT query vectors of one sequence (heads of one row, or
//     several rows of one sequence); all of them share every KV tile, so a
//     tile is read from HBM once per unit.
//   * Persistent mode (num_kv_splits > 1): one CTA per SM.  The tiles of all
//     units form one list; each CTA takes an equal contiguous share of it, so
//     every SM streams the same number of bytes whatever the length mix.  A
//     CTA's share is cut into segments at unit boundaries; each segment
//     yields one partial (o, lse) in the unit's next free split slot, and the
//     first segment of a unit marks the slots it does not use with
//     lse = -inf.  The producer runs ahead across segment boundaries (Q of
//     the next segment goes into a second buffer), so the load pipeline never
//     drains inside a CTA.
//   * Grid mode (num_kv_splits == 1, and very large batches): one CTA per
//     (unit, split) as in the pages; with one split the CTA writes o and lse
//     itself, one sequential pass in a fixed order (batch-invariant).
//   * A producer warp streams 64-token tiles with TMA (one 3-D box per 64
//     dims per page, 128-byte swizzle) into an mbarrier ring; the box
//     coordinate is the page's block id from the block table.  Block ids
//     outside the cache read as zeros (TMA out-of-bounds fill).
//   * 4*MT consumer warps: S = Q.K^T with each warp owning 16 tokens of the
//     tile (mma.sync m16n8k16, bf16 in, fp32 accumulate, four independent
//     accumulator chains over the 576-long reduction); softmax maxima and
//     sums are exchanged through shared memory; P (bf16) goes to shared
//     memory; O += P.V with each warp owning a quarter of the latent columns,
//     accumulators in registers.
//   * fp8 (E4M3 or E5M2) tiles are converted exactly to bf16 in shared memory by the
//     consumers; the dequantisation scale is folded into the score scale and
//     the final output scale.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "kernels.cuh"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kBN = 64;  // tokens per tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int R, bool FP8, int MT>
struct MmaCfg {
  static constexpr int D = R + 64;
  static constexpr int NCH = D / 64;   // 64-dim chunks per row
  static constexpr int NCW = 4 * MT;   // consumer warps
  static constexpr int NTHREADS = 32 * (NCW + 1);
  static constexpr int TILE = NCH * kBN * 128;  // bf16 tile, bytes
  static constexpr int RAW = NCH * kBN * 64;    // raw fp8 tile, bytes
  static constexpr int STAGE_BYTES = FP8 ? RAW : TILE;
  static constexpr int STAGES = FP8 ? (R == 512 ? 2 : 4) : (R == 512 ? 2 : 4);
  static constexpr int QBOX = 16 * MT * 128;    // one 64-dim chunk of Q
  static constexpr int QBYTES = NCH * QBOX;
  static constexpr int PPITCH = kBN + 8;        // P row pitch (elements)
  static constexpr int PBYTES = 16 * MT * PPITCH * 2;
  // fp8 with R = 256: two converted tiles, so that the conversion of tile
  // n + 1 runs between the S products of tile n (software pipelining); the
  // 576-wide fp8 tiles leave room for one
  static constexpr bool PIPE = FP8 && R == 256;
  static constexpr int NCONV = FP8 ? (PIPE ? 2 : 1) : 0;
  static constexpr int OFF_STAGES = 0;
  static constexpr int OFF_CONV = STAGES * STAGE_BYTES;
  static constexpr int OFF_Q = OFF_CONV + NCONV * TILE;  // two Q buffers
  static constexpr int OFF_P = OFF_Q + 2 * QBYTES;
  static constexpr int OFF_RED = OFF_P + PBYTES;
  static constexpr int RED_BYTES = 2 * MT * 4 * 16 * 4;
  static constexpr int OFF_BAR = OFF_RED + RED_BYTES;
  static constexpr int NBARS = 2 * STAGES + 4;
  static constexpr int OFF_PRE = OFF_BAR + NBARS * 8;
  static constexpr int OFF_LEN = OFF_PRE + (kMaxPersistUnits + 1) * 4;
  static constexpr int SMEM = OFF_LEN + kMaxPersistUnits * 4 + 1024;
  static_assert(OFF_Q % 1024 == 0 && QBOX % 1024 == 0, "swizzle alignment");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// 16 fp8 bytes (E4M3, or E5M2 when e5m2) -> 16 bf16 values (exact: every
// E4M3 and every E5M2 value is a bf16 value).
__device__ __forceinline__ void fp8x16_to_bf16(uint4 raw, bool e5m2, uint4& lo,
                                               uint4& hi) {
  const uint16_t* b = reinterpret_cast<const uint16_t*>(&raw);
  uint32_t out[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(b[k]),
                                               e5m2 ? __NV_E5M2 : __NV_E4M3);
    float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
    out[k] = pack_bf16x2(f.x, f.y);
  }
  lo = make_uint4(out[0], out[1], out[2], out[3]);
  hi = make_uint4(out[4], out[5], out[6], out[7]);
}

// Converts 64-dim chunks [c_lo, c_hi) of a raw fp8 tile (64 rows of 64
// bytes per chunk) into a bf16 tile (64 rows of 128 bytes per chunk,
// 128-byte swizzled); rows at or past `valid` become zeros.  Thread `ctid`
// of `nthreads` takes every nthreads-th 16-byte piece.
__device__ __forceinline__ void convert_chunks(const uint8_t* raw, uint8_t* conv, int c_lo,
                                               int c_hi, int valid, bool e5m2, int ctid,
                                               int nthreads) {
  const int n = (c_hi - c_lo) * kBN * 4;
  for (int i = ctid; i < n; i += nthreads) {
    const int c = c_lo + i / (kBN * 4), r = (i >> 2) % kBN, kq = i & 3;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
    if (r < valid)
      fp8x16_to_bf16(*reinterpret_cast<const uint4*>(raw + c * (kBN * 64) + r * 64 + kq * 16),
                     e5m2, lo, hi);
    uint8_t* dst = conv + c * (kBN * 128);
    *reinterpret_cast<uint4*>(dst + sw128(r, 2 * kq)) = lo;
    *reinterpret_cast<uint4*>(dst + sw128(r, 2 * kq + 1)) = hi;
  }
}

__device__ __forceinline__ int clamp_len(const DecodeParams& p, int b) {
  int L = __ldg(p.seq_lens + b);
  const int Lmax = p.max_blocks * p.block_size;
  return L < 0 ? 0 : (L > Lmax ? Lmax : L);
}

constexpr int kClampedBit = 1 << 30;

// One segment of work: tiles [t_lo, t_hi) of unit (b, g) whose sequence has
// L tokens; its result goes to split slot `slot` (or straight to o/lse when
// `direct`).  Block-major schedule: `first` segments (slot 0) also mark
// slots [nslots, S) unused.  Chunked schedule: the first segment of a chunk
// marks [mark_lo, mark_hi) and [mark2_lo, mark2_hi) unused; `first` is
// slot 0 (once per sequence and vector block).
struct Seg {
  int b, g, L;
  int t_lo, t_hi;
  int slot, nslots;                              // block-major schedule
  int mark_lo, mark_hi, mark2_lo, mark2_hi;      // chunked schedule
  bool first, direct, clamped;
};

// Persistent schedule, identical in every warp that walks it.  The list is
// the tiles of all (sequence, vector block) units; a sequence with several
// vector blocks is listed in chunks of CH tiles, all its blocks of a chunk
// side by side, so that the CTAs holding the blocks of one chunk stream the
// same KV tiles at about the same time and L2 serves the later readers.  A
// chunk of one block spans at most SPC CTAs and owns SPC split slots.  CTA c
// takes list tiles [lo, hi) = [c C, (c + 1) C).
struct Sched {
  const int* pre;  // [units + 1] first list tile of each unit (block-major)
  const int* len;  // [sequences] clamped length, | kClampedBit if clamped
  int units, qblocks, num_seqs, C, CH, SPC, S, lo, hi, c;
  // Block-major schedule (one vector block per sequence): units in order.
  __device__ int first_unit() const {
    int a = 0, z = units;  // smallest u with pre[u + 1] > lo
    while (a < z) {
      const int m = (a + z) >> 1;
      if (pre[m + 1] > lo) z = m; else a = m + 1;
    }
    return a;
  }
  // Fills `s` with the segment of unit `u` (must intersect [lo, hi)).
  __device__ void seg(const DecodeParams& p, int u, Seg& s) const {
    s.b = u / qblocks;
    s.g = u - s.b * qblocks;
    s.L = len[s.b] & ~kClampedBit;
    s.clamped = (len[s.b] & kClampedBit) != 0;
    const int a = max(lo, pre[u]), z = min(hi, pre[u + 1]);
    s.t_lo = a - pre[u];
    s.t_hi = z - pre[u];
    const int cf = pre[u] / C;
    s.slot = c - cf;
    s.nslots = (pre[u + 1] - 1) / C - cf + 1;
    s.first = s.slot == 0;
    s.direct = false;
  }
  // Chunked schedule: fills `s` with the segment that starts at list tile t
  // (lo <= t < hi);
  // returns the list tile where the next segment starts.
  __device__ int seg_at(int t, Seg& s) const {
    int a = 0, z = num_seqs - 1;  // the last sequence b with pre[b * qblocks] <= t
    while (a < z) {
      const int m = (a + z + 1) >> 1;
      if (pre[m * qblocks] <= t) a = m; else z = m - 1;
    }
    const int b = a;
    const int Ob = pre[b * qblocks];
    const int Tb = pre[b * qblocks + 1] - Ob;  // tiles of the sequence
    const int Jb = ceil_div(Tb, CH);
    // list tiles of a full chunk (CH is 2^30 only with one block per sequence)
    const int span = qblocks * CH;
    const int x = t - Ob;
    const int j = min(x / span, Jb - 1);
    const int clen = j == Jb - 1 ? Tb - (Jb - 1) * CH : CH;  // tiles of chunk j
    const int y = x - j * span;
    const int g = y / clen;
    const int in = y - g * clen;
    const int vstart = Ob + j * span + g * clen;
    const int vend = vstart + clen;
    const int seg_end = min(hi, vend);
    s.b = b;
    s.g = g;
    s.L = len[b] & ~kClampedBit;
    s.clamped = (len[b] & kClampedBit) != 0;
    s.t_lo = j * CH + in;
    s.t_hi = s.t_lo + (seg_end - t);
    const int cf = vstart / C;  // the CTA where chunk j of block g begins
    s.slot = j * SPC + (c - cf);
    const bool first = c == cf;
    s.mark_lo = first ? j * SPC + ((vend - 1) / C - cf + 1) : 0;
    s.mark_hi = first ? (j + 1) * SPC : 0;
    s.mark2_lo = first && j == 0 ? Jb * SPC : 0;  // slots past the last chunk
    s.mark2_hi = first && j == 0 ? S : 0;
    s.first = s.slot == 0;
    s.direct = false;
    return seg_end;
  }
};
// PM: 0 = one CTA per (vector block, split); 1 = persistent, block-major
// list (one vector block per sequence); 2 = persistent, chunked list.
template <int R, bool FP8, int MT, int PM>
__global__ void __launch_bounds__(MmaCfg<R, FP8, MT>::NTHREADS, 1)
    decode_mma_kernel(const DecodeParams p,
                      const __grid_constant__ CUtensorMap tmap,
                      const __grid_constant__ QMaps qmap) {
  using C = MmaCfg<R, FP8, MT>;
  constexpr int D = C::D, NCH = C::NCH, NCW = C::NCW, STAGES = C::STAGES;
  constexpr int NT = R / 32;  // 8-column MMA tiles per warp in P.V
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_stage = smem + C::OFF_STAGES;
  uint8_t* s_conv = smem + C::OFF_CONV;
  uint16_t* s_p = reinterpret_cast<uint16_t*>(smem + C::OFF_P);
  float* red_max = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* red_sum = red_max + MT * 4 * 16;
  uint64_t* bar_full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* bar_empty = bar_full + STAGES;
  uint64_t* q_full = bar_empty + STAGES;
  uint64_t* q_empty = q_full + 2;
  int* pre = reinterpret_cast<int*>(smem + C::OFF_PRE);
  int* lens = reinterpret_cast<int*>(smem + C::OFF_LEN);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.num_heads;
  const int nvec = p.rows_per_seq * H;
  const int qblocks = ceil_div(nvec, 16 * MT);
  const int S = p.num_splits;
  if (threadIdx.x == NCW * 32) {
    tma_prefetch_desc(&tmap);
    if (p.q_tma) {
      tma_prefetch_desc(&qmap.nope);
      tma_prefetch_desc(&qmap.pe);
    }
  }
  // Launched overlapped with the previous kernel of the stream: nothing in
  // global memory is read before it has completed.
  griddep_wait();
  griddep_launch_dependents();

  // ---------------------------------------------------------- schedule
  Sched sch;
  int nseg = 0;    // grid mode: 0 or 1 segment
  Seg gseg;        // grid mode segment
  if constexpr (PM != 0) {
    const int units = p.num_seqs * qblocks;
    // pre[u + 1] = tiles of unit u, then an inclusive scan by warp 0
    for (int u = threadIdx.x; u < units; u += blockDim.x) {
      const int b = u / qblocks;
      const int raw = __ldg(p.seq_lens + b);
      const int L = clamp_len(p, b);
      pre[u + 1] = ceil_div(L, kBN);
      if (u == b * qblocks) lens[b] = L | (raw > L ? kClampedBit : 0);
    }
    if (threadIdx.x == 0) pre[0] = 0;
    __syncthreads();
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
      if (lane == 0) red_max[0] = __int_as_float(mx);
    }
    __syncthreads();
    const int total = pre[units];
    const int max_n = __float_as_int(red_max[0]);
    int Cc = ceil_div(total, gridDim.x);
    Cc = max(Cc, ceil_div(max_n, S - 1));  // at most S slots per unit
    Cc = max(Cc, 1);
    sch.pre = pre;
    sch.len = lens;
    sch.units = units;
    sch.qblocks = qblocks;
    sch.num_seqs = p.num_seqs;
    sch.C = Cc;
    sch.S = S;
    sch.CH = 1 << 30;
    sch.SPC = S;
    if constexpr (PM == 2) {
      // smallest m with (chunks) x (slots per chunk) <= S; m = ceil(max_n / C)
      // (one chunk) always qualifies because C >= ceil(max_n / (S - 1))
      for (int m = 1;; ++m) {
        const int J = ceil_div(max_n, Cc * m);
        if (J * (m + 1) <= S || J == 1) {
          sch.CH = Cc * m;
          sch.SPC = m + 1;
          break;
        }
      }
    }
    sch.c = blockIdx.x;
    sch.lo = blockIdx.x * Cc;
    sch.hi = min(total, sch.lo + Cc);
    __syncthreads();  // red_max reused below
    if (sch.lo >= sch.hi) return;
  } else {
    gseg.g = blockIdx.x;
    gseg.b = blockIdx.z;
    const int split = blockIdx.y;
    int L = __ldg(p.seq_lens + gseg.b);
    const int Lmax = p.max_blocks * p.block_size;
    if (L < 0) L = 0;
    if (L > Lmax) {
      if (threadIdx.x == 0 && split == 0 && gseg.g == 0 && p.err_count)
        atomicAdd(p.err_count, 1);
      L = Lmax;
    }
    gseg.L = L;
    const int per = L > 0 ? ceil_div(ceil_div(L, S), kBN) * kBN : kBN;
    const int start = split * per;
    const int end = min(L, start + per);
    gseg.t_lo = start / kBN;
    gseg.t_hi = start < end ? ceil_div(end, kBN) : gseg.t_lo;
    gseg.slot = split;
    gseg.nslots = S;
    gseg.mark_lo = gseg.mark_hi = gseg.mark2_lo = gseg.mark2_hi = 0;
    gseg.first = false;
    gseg.direct = S == 1;
    gseg.clamped = false;  // counted above
    nseg = gseg.t_hi > gseg.t_lo ? 1 : 0;
    if (nseg == 0) {
      if (warp < NCW) {
        const int v0 = gseg.g * 16 * MT;
        for (int i = threadIdx.x; i < 16 * MT * R; i += NCW * 32) {
          const int qv = i / R, col = i % R, v = v0 + qv;
          if (v >= nvec) continue;
          const int row = gseg.b * p.rows_per_seq + v / H, h = v % H;
          if (S == 1) {
            // Empty sequence in single-pass mode: o = 0, lse = -inf.
            p.o[(static_cast<int64_t>(row) * H + h) * R + col] = 0;
            if (col == 0) p.lse[static_cast<int64_t>(row) * H + h] = -INFINITY;
          } else if (col == 0 && L > 0) {
            // A split past the end of a non-empty sequence: no partial.
            p.ws_lse[(static_cast<int64_t>(row) * S + split) * H + h] = -INFINITY;
          }
        }
      }
      return;
    }
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&bar_full[i], 1);
      mbar_init(&bar_empty[i], NCW);
    }
    for (int i = 0; i < 2; ++i) {
      // TMA: one expect-tx arrival; cp.async: one arrival per producer lane
      mbar_init(&q_full[i], p.q_tma ? 1 : 32);
      mbar_init(&q_empty[i], NCW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // Walks the CTA's segments in order, calling f(seg, index).
  auto for_each_seg = [&](auto&& f) {
    if constexpr (PM == 1) {
      int k = 0;
      for (int u = sch.first_unit(); u < sch.units && sch.pre[u] < sch.hi; ++u) {
        if (sch.pre[u + 1] <= max(sch.lo, sch.pre[u])) continue;  // empty unit
        Seg s;
        sch.seg(p, u, s);
        if (!f(s, k++)) return;
      }
    } else if constexpr (PM == 2) {
      int k = 0;
      for (int t = sch.lo; t < sch.hi;) {
        Seg s;
        t = sch.seg_at(t, s);
        if (!f(s, k++)) return;
      }
    } else {
      if (nseg) f(gseg, 0);
    }
  };

  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    const int bs = p.block_size;
    const int rows_box = bs < kBN ? bs : kBN;
    const int npg = kBN / rows_box;
    constexpr int ROWB = FP8 ? 64 : 128;
    int it = 0;  // tiles issued so far (ring position)
    for_each_seg([&](const Seg& sg, int k) -> bool {
      // Q of this segment -> buffer k & 1 (all lanes), once the consumers are
      // done with the segment that used it two segments ago.
      if (!__all_sync(0xffffffffu, mbar_wait(&q_empty[k & 1], ((k >> 1) & 1) ^ 1))) {
        if (lane == 0 && p.err_count) atomicAdd(p.err_count, kTimeoutErr);
        return false;
      }
      const int v0 = sg.g * 16 * MT;
      uint8_t* q_dst = smem + C::OFF_Q + (k & 1) * C::QBYTES;
      if (p.q_tma) {
        // Heads come in multiples of 16, so each 16-vector M tile is 16
        // consecutive heads of one row: one {64, 16, 1} box per 64 dims.
        // M tiles past the last vector are not loaded (their rows stay
        // unused).
        if (lane == 0) {
          int ntile = 0;
          for (int i = 0; i < MT; ++i) ntile += v0 + 16 * i < nvec ? 1 : 0;
          mbar_arrive_expect_tx(&q_full[k & 1], static_cast<uint32_t>(ntile * NCH * 2048));
          for (int i = 0; i < ntile; ++i) {
            const int v = v0 + 16 * i;
            const int row = sg.b * p.rows_per_seq + v / H, h0 = v % H;
            // dims [0, R) from q_nope, [R, R+P) from q_pe
            for (int c = 0; c < NCH; ++c) {
              const bool pe = c >= R / 64;
              tma_load_3d(q_dst + c * C::QBOX + i * 2048, pe ? &qmap.pe : &qmap.nope,
                          &q_full[k & 1], (pe ? c - R / 64 : c) * 64, h0, row);
            }
          }
        }
      } else {
        // cp.async: the copies proceed while this warp goes on issuing
        // tiles; q_full completes when every lane's copies have landed.
        const uint32_t s_q = smem_u32(q_dst);
        for (int i = lane; i < 16 * MT * (D / 8); i += 32) {
          const int qr = i / (D / 8), ch = i % (D / 8);
          const int v = v0 + qr;
          const uint16_t* src = p.q;
          if (v < nvec) {
            const int row = sg.b * p.rows_per_seq + v / H, h = v % H;
            src = ch < R / 8 ? p.q + row * p.q_row_stride + h * p.q_head_stride + ch * 8
                             : p.q_pe + row * p.q_pe_row_stride + h * p.q_pe_head_stride +
                                   (ch - R / 8) * 8;
          }
          cp_async16(s_q + (ch >> 3) * C::QBOX + sw128(qr, ch & 7), src, v < nvec ? 16u : 0u);
        }
        cp_async_arrive(&q_full[k & 1]);
      }
      if (lane == 0) {
        const int32_t* bt = p.block_table + static_cast<int64_t>(sg.b) * p.bt_stride;
        // block ids of the next tile are loaded one tile ahead
        auto fetch = [&](int t, int (&ids)[4]) {
#pragma unroll
          for (int pg = 0; pg < 4; ++pg) {
            const int tk = t * kBN + pg * rows_box;
            ids[pg] = (pg < npg && t < sg.t_hi && tk < sg.L) ? __ldg(bt + tk / bs) : 0;
          }
        };
        int cur[4], nxt[4];
        fetch(sg.t_lo, cur);
        for (int t = sg.t_lo; t < sg.t_hi; ++t, ++it) {
          fetch(t + 1, nxt);
          const int st = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!mbar_wait(&bar_empty[st], ph ^ 1)) {
            if (p.err_count) atomicAdd(p.err_count, kTimeoutErr);
            it = -1;
            break;
          }
          const int tok0 = t * kBN;
          int npages = 0;
          for (int pg = 0; pg < npg; ++pg)
            if (tok0 + pg * rows_box < sg.L) ++npages;
          mbar_arrive_expect_tx(&bar_full[st],
                                static_cast<uint32_t>(npages * NCH * rows_box * ROWB));
          uint8_t* dst = s_stage + st * C::STAGE_BYTES;
#pragma unroll
          for (int pg = 0; pg < 4; ++pg) {
            if (pg >= npages) break;
            const int tk = tok0 + pg * rows_box;
            const int blk = cur[pg];
            const int row0 = tk % bs;
            if ((blk < 0 || blk >= p.num_blocks) && p.err_count)
              atomicAdd(p.err_count, 1);
#pragma unroll 1
            for (int c = 0; c < NCH; ++c)
              tma_load_3d(dst + c * (kBN * ROWB) + pg * rows_box * ROWB, &tmap,
                          &bar_full[st], c * 64, row0, blk);
          }
#pragma unroll
          for (int pg = 0; pg < 4; ++pg) cur[pg] = nxt[pg];
        }
      }
      it = __shfl_sync(0xffffffffu, it, 0);
      return it >= 0;
    });
    return;
  }

  // -------------------------------------------------------------- consumers
  const int mt = warp >> 2;   // which 16-vector M tile
  const int q4 = warp & 3;    // token quarter (S) / latent quarter (P.V)
  const int ctid = threadIdx.x;  // 0 .. NCW*32-1
  const float kv_s = FP8 ? __ldg(p.kv_scale) : 1.0f;
  const float scale_log2 = p.sm_scale * kv_s * kLog2e;
  const int g = lane >> 2, tq = lane & 3;
  const int prow0 = mt * 16 + g;  // this thread's rows in P / the M tile
  const uint32_t p_base = smem_u32(s_p);
  int it = 0;  // tiles consumed so far (ring position)

  for_each_seg([&](const Seg& sg, int k) -> bool {
    if (!mbar_wait(&q_full[k & 1], (k >> 1) & 1)) {
      if (lane == 0 && p.err_count) atomicAdd(p.err_count, kTimeoutErr);
      return false;
    }
    const uint32_t q_base = smem_u32(smem + C::OFF_Q + (k & 1) * C::QBYTES);
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n)
      acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

    if constexpr (C::PIPE) {
      // the segment's first tile is converted here; every later one during
      // the S products of the tile before it
      if (sg.t_lo < sg.t_hi) {
        const int st = it % STAGES;
        if (!mbar_wait(&bar_full[st], (it / STAGES) & 1)) {
          if (lane == 0 && p.err_count) atomicAdd(p.err_count, kTimeoutErr);
          return false;
        }
        named_bar_sync(1, NCW * 32);  // the buffer's previous tile has been read
        convert_chunks(s_stage + st * C::STAGE_BYTES, s_conv + (it & 1) * C::TILE, 0, NCH,
                       min(kBN, sg.L - sg.t_lo * kBN), p.kv_e5m2 != 0, ctid, NCW * 32);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_empty[st]);
        named_bar_sync(1, NCW * 32);
      }
    }
    for (int t = sg.t_lo; t < sg.t_hi; ++t, ++it) {
      const int st = it % STAGES;
      const uint32_t ph = (it / STAGES) & 1;
      const int valid = min(kBN, sg.L - t * kBN);
      // pipelined fp8: the next tile of the segment is converted during this
      // tile's S products (its raw stage must have landed first)
      const bool pf = C::PIPE && t + 1 < sg.t_hi;
      const int st_n = (it + 1) % STAGES;
      const int valid_n = min(kBN, sg.L - (t + 1) * kBN);
      uint8_t* conv_n = s_conv + ((it + 1) & 1) * C::TILE;
      if (!C::PIPE || pf) {
        const int wst = C::PIPE ? st_n : st;
        const uint32_t wph = C::PIPE ? ((it + 1) / STAGES) & 1 : ph;
        if (!mbar_wait(&bar_full[wst], wph)) {
          if (lane == 0 && p.err_count) atomicAdd(p.err_count, kTimeoutErr);
          return false;
        }
      }
      uint8_t* tile;
      if constexpr (C::PIPE) {
        tile = s_conv + (it & 1) * C::TILE;
      } else if constexpr (FP8) {
        // All warps are done reading the previous converted tile.
        named_bar_sync(1, NCW * 32);
        convert_chunks(s_stage + st * C::STAGE_BYTES, s_conv, 0, NCH, valid, p.kv_e5m2 != 0,
                       ctid, NCW * 32);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_empty[st]);
        named_bar_sync(1, NCW * 32);
        tile = s_conv;
      } else {
        tile = s_stage + st * C::STAGE_BYTES;
        if (valid < kBN) {
          // Rows past the sequence end may hold anything (other tokens'
          // data, NaN); zero them so that 0 * row stays 0 in P.V.
          const int nz = (kBN - valid) * NCH * 8;
          for (int idx = ctid; idx < nz; idx += NCW * 32) {
            const int r = valid + idx / (NCH * 8), rem = idx % (NCH * 8);
            *reinterpret_cast<uint4*>(tile + (rem >> 3) * (kBN * 128) + r * 128 +
                                      (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          named_bar_sync(1, NCW * 32);
        }
      }
      const uint32_t t_base = smem_u32(tile);

      // ---- S = Q K^T for this warp's 16 tokens (two 8-token MMA tiles),
      // four independent accumulator chains over the reduction
      float sc[2][4];
      {
        float ch[4][2][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int jn = 0; jn < 2; ++jn)
            ch[a][jn][0] = ch[a][jn][1] = ch[a][jn][2] = ch[a][jn][3] = 0.f;
        const int j = lane >> 3, r8 = lane & 7;
        const uint32_t a_row = mt * 16 + (j & 1) * 8 + r8;  // Q row for ldmatrix
        const uint32_t a_kc = j >> 1;
        const uint32_t b_row = q4 * 16 + (j >> 1) * 8 + r8;  // K row (token)
        const uint32_t b_kc = j & 1;
#pragma unroll
        for (int c64 = 0; c64 < NCH; ++c64) {
          // pipelined fp8: chunk c64 of the next tile, between the products
          if (pf)
            convert_chunks(s_stage + st_n * C::STAGE_BYTES, conv_n, c64, c64 + 1, valid_n,
                           p.kv_e5m2 != 0, ctid, NCW * 32);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t kc = kk * 2;
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            ldsm_x4(q_base + c64 * C::QBOX + sw128(a_row, kc + a_kc), a0, a1, a2, a3);
            ldsm_x4(t_base + c64 * (kBN * 128) + sw128(b_row, kc + b_kc), b0, b1, b2, b3);
            mma_bf16_16816(ch[kk][0], a0, a1, a2, a3, b0, b1);
            mma_bf16_16816(ch[kk][1], a0, a1, a2, a3, b2, b3);
          }
        }
        if (pf) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_empty[st_n]);  // the raw stage is converted
        }
#pragma unroll
        for (int jn = 0; jn < 2; ++jn)
#pragma unroll
          for (int e = 0; e < 4; ++e)
            sc[jn][e] = (ch[0][jn][e] + ch[1][jn][e]) + (ch[2][jn][e] + ch[3][jn][e]);
      }

      // ---- online softmax (log2 domain), rows prow0 and prow0 + 8
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int jn = 0; jn < 2; ++jn)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int tok = q4 * 16 + jn * 8 + 2 * tq + (e & 1);
          const float tv = tok < valid ? sc[jn][e] * scale_log2 : -INFINITY;
          sc[jn][e] = tv;
          mx[e >> 1] = fmaxf(mx[e >> 1], tv);
        }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      }
      if (tq == 0) {
        red_max[(mt * 4 + q4) * 16 + g] = mx[0];
        red_max[(mt * 4 + q4) * 16 + g + 8] = mx[1];
      }
      named_bar_sync(1, NCW * 32);
      float m_new[2], alpha[2], ps[2] = {0.f, 0.f};
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float tm = red_max[(mt * 4 + 0) * 16 + g + 8 * r];
#pragma unroll
        for (int w = 1; w < 4; ++w)
          tm = fmaxf(tm, red_max[(mt * 4 + w) * 16 + g + 8 * r]);
        m_new[r] = fmaxf(m_run[r], tm);
        alpha[r] = ex2(m_run[r] - m_new[r]);
      }
#pragma unroll
      for (int jn = 0; jn < 2; ++jn) {
        float pe[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          pe[e] = ex2(sc[jn][e] - m_new[e >> 1]);
          ps[e >> 1] += pe[e];
        }
        const int col = q4 * 16 + jn * 8 + 2 * tq;
        *reinterpret_cast<uint32_t*>(s_p + prow0 * C::PPITCH + col) =
            pack_bf16x2(pe[0], pe[1]);
        *reinterpret_cast<uint32_t*>(s_p + (prow0 + 8) * C::PPITCH + col) =
            pack_bf16x2(pe[2], pe[3]);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        ps[r] += __shfl_xor_sync(0xffffffffu, ps[r], 1);
        ps[r] += __shfl_xor_sync(0xffffffffu, ps[r], 2);
      }
      if (tq == 0) {
        red_sum[(mt * 4 + q4) * 16 + g] = ps[0];
        red_sum[(mt * 4 + q4) * 16 + g + 8] = ps[1];
      }
      named_bar_sync(1, NCW * 32);
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        float s_tile = red_sum[(mt * 4 + 0) * 16 + g + 8 * r];
#pragma unroll
        for (int w = 1; w < 4; ++w) s_tile += red_sum[(mt * 4 + w) * 16 + g + 8 * r];
        l_run[r] = l_run[r] * alpha[r] + s_tile;
        m_run[r] = m_new[r];
      }
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        acc[n][0] *= alpha[0];
        acc[n][1] *= alpha[0];
        acc[n][2] *= alpha[1];
        acc[n][3] *= alpha[1];
      }

      // ---- O += P V over this warp's R/4 latent columns
      {
        const int j = lane >> 3, r8 = lane & 7;
        const uint32_t pa_row = mt * 16 + (j & 1) * 8 + r8;
        const uint32_t pa_col = (j >> 1) * 8;
        const uint32_t v_tok = (j & 1) * 8 + r8;
        const uint32_t v_nc = j >> 1;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(p_base + (pa_row * C::PPITCH + kk * 16 + pa_col) * 2, a0, a1, a2, a3);
          const uint32_t tok = kk * 16 + v_tok;
#pragma unroll
          for (int n = 0; n < NT; n += 2) {
            const uint32_t d8 = (q4 * (R / 4) + n * 8) / 8 + v_nc;  // 8-dim chunk
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(t_base + (d8 >> 3) * (kBN * 128) + sw128(tok, d8 & 7), b0, b1, b2, b3);
            mma_bf16_16816(acc[n], a0, a1, a2, a3, b0, b1);
            mma_bf16_16816(acc[n + 1], a0, a1, a2, a3, b2, b3);
          }
        }
      }
      if constexpr (!FP8) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_empty[st]);
      }
      // pipelined fp8: every warp has read this tile's buffer and written
      // its part of the next tile's before the next tile starts
      if constexpr (C::PIPE) named_bar_sync(1, NCW * 32);
    }

    // ---- segment epilogue: normalise and write (final o/lse, or a partial)
    const int v0 = sg.g * 16 * MT;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int v = v0 + prow0 + 8 * r;
      if (v >= nvec) continue;
      const int row = sg.b * p.rows_per_seq + v / H, h = v % H;
      const float inv = kv_s / l_run[r];
      float lse2;
      asm("lg2.approx.f32 %0, %1;" : "=f"(lse2) : "f"(l_run[r]));
      const float lse = (m_run[r] + lse2) * kLn2;
      if (sg.direct) {
        uint16_t* orow = p.o + (static_cast<int64_t>(row) * H + h) * R;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const int col = q4 * (R / 4) + n * 8 + 2 * tq;
          *reinterpret_cast<uint32_t*>(orow + col) =
              pack_bf16x2(acc[n][2 * r] * inv, acc[n][2 * r + 1] * inv);
        }
        if (q4 == 0 && tq == 0) p.lse[static_cast<int64_t>(row) * H + h] = lse;
      } else {
        const int64_t rec = (static_cast<int64_t>(row) * S + sg.slot) * H + h;
        float* orow = p.ws_o + rec * R;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const int col = q4 * (R / 4) + n * 8 + 2 * tq;
          *reinterpret_cast<float2*>(orow + col) =
              make_float2(acc[n][2 * r] * inv, acc[n][2 * r + 1] * inv);
        }
        if (q4 == 0 && tq == 0) {
          p.ws_lse[rec] = lse;
          // slots the partition leaves unused
          if constexpr (PM == 2) {
            for (int s = sg.mark_lo; s < sg.mark_hi; ++s)
              p.ws_lse[(static_cast<int64_t>(row) * S + s) * H + h] = -INFINITY;
            for (int s = sg.mark2_lo; s < sg.mark2_hi; ++s)
              p.ws_lse[(static_cast<int64_t>(row) * S + s) * H + h] = -INFINITY;
          } else if (sg.first) {
            for (int s = sg.nslots; s < S; ++s)
              p.ws_lse[(static_cast<int64_t>(row) * S + s) * H + h] = -INFINITY;
          }
        }
      }
    }
    if (sg.first && sg.clamped && sg.g == 0 && warp == 0 && lane == 0 && p.err_count)
      atomicAdd(p.err_count, 1);  // seq_len beyond the block table, once per sequence
    __syncwarp();
    if (lane == 0) mbar_arrive(&q_empty[k & 1]);
    return true;
  });
}

template <int R, bool FP8, int MT, int PM>
cudaError_t launch_mt(const DecodeParams& p, const CUtensorMap& tmap, const QMaps& qmap,
                      int sm_count, cudaStream_t stream) {
  using C = MmaCfg<R, FP8, MT>;
  static std::atomic<uint64_t> attr_done{0};  // per instantiation, one bit per device
  cudaError_t e = set_smem_attr_once(decode_mma_kernel<R, FP8, MT, PM>, C::SMEM, attr_done);
  if (e != cudaSuccess) return e;
  const int nvec = p.rows_per_seq * p.num_heads;
  const int qblocks = (nvec + 16 * MT - 1) / (16 * MT);
  const dim3 grid = PM != 0 ? dim3(sm_count) : dim3(qblocks, p.num_splits, p.num_seqs);
  return launch_overlapped(decode_mma_kernel<R, FP8, MT, PM>, grid, dim3(C::NTHREADS),
                           C::SMEM, stream, p, tmap, qmap);
}

template <int R, bool FP8, int MT>
cudaError_t launch_r2(const DecodeParams& p, const CUtensorMap& tmap, const QMaps& qmap,
                      int sm_count, cudaStream_t stream) {
  const int qblocks = (p.rows_per_seq * p.num_heads + 16 * MT - 1) / (16 * MT);
  const int64_t units = static_cast<int64_t>(qblocks) * p.num_seqs;
  if (p.num_splits > 1 && units <= kMaxPersistUnits) {
    // (a single 16-vector block per CTA, MT = 1, means one block per sequence)
    if constexpr (MT > 1)
      if (qblocks > 1) return launch_mt<R, FP8, MT, 2>(p, tmap, qmap, sm_count, stream);
    return launch_mt<R, FP8, MT, 1>(p, tmap, qmap, sm_count, stream);
  }
  return launch_mt<R, FP8, MT, 0>(p, tmap, qmap, sm_count, stream);
}

template <int R, bool FP8>
cudaError_t launch_r(const DecodeParams& p, const CUtensorMap& tmap, const QMaps& qmap,
                     int sm_count, cudaStream_t stream) {
  const int nvec = p.rows_per_seq * p.num_heads;
  if (nvec <= 16) return launch_r2<R, FP8, 1>(p, tmap, qmap, sm_count, stream);
  return launch_r2<R, FP8, 2>(p, tmap, qmap, sm_count, stream);
}

}  // namespace

cudaError_t launch_decode_mma(const DecodeParams& p, const CUtensorMap& tmap,
                              const QMaps& qmap, int R, bool fp8, int sm_count,
                              cudaStream_t stream) {
  if (R == 512) return fp8 ? launch_r<512, true>(p, tmap, qmap, sm_count, stream)
                           : launch_r<512, false>(p, tmap, qmap, sm_count, stream);
  return fp8 ? launch_r<256, true>(p, tmap, qmap, sm_count, stream)
             : launch_r<256, false>(p, tmap, qmap, sm_count, stream);
}

}  // namespace mla
