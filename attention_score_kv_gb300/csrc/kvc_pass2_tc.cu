// Pass 2 of the two-pass scorer plus pooling (TideKV, Fig. 3): per key, the
// normalised attention weights summed over the window queries and the GQA
// group, average-pooled, then written as scores or appended to the key
// range's candidate list.
//
// A = 128-key tile (M = 128), B = window queries (N = G*W rounded to 16), so
// tensor-memory lane i holds key i of the tile and the query axis runs along
// the columns.  The per-query normaliser enters the MMA itself: one extra
// K-step multiplies a constant (1, 1, 1, 0, ...) block on the key side with
// the query's bias -lse2_q / (log2(e)/sqrt(D)), split into three bf16 terms
// (hi, mid, lo) on the query side, so the accumulator already holds
// q.k - lse_q in raw units and a weight is 2^(acc * log2(e)/sqrt(D)).
//
// Sixteen softmax warps, four per tensor-memory lane quarter, share every
// tile: warp k of a quarter reads column slice k of the accumulator once
// (up to 64 columns), hands the buffer back to the MMA warp at once, then
// exponentiates and sums its columns in registers.  So the MMA of the next
// tiles never waits on the exponentials, only on the loads.  Each thread
// owns one key; the four slice sums of a key go to a shared-memory ring.  A
// pooling warp consumes the ring in key order: it adds the four slices, keeps
// the last pool_k-1 masses of the previous tile, forms the centred average
// for keys t0 - h .. t0 + 127 - h, and appends the non-mandatory keys that
// beat the range's running threshold.
#include "kvc_scan_common.cuh"

namespace kvc {
namespace {

using namespace scan;

constexpr int kStages2 = 4;
// The bias K-step's operands (16 K elements a row) in the unswizzled
// core-matrix layout: row r of a block at (r/8)*256 + (r%8)*16 for K
// elements 0-7, +128 for 8-15, so a row takes 32 bytes instead of a
// 128-byte swizzled row.
constexpr uint32_t kOnesBytes = kTile * 32;
constexpr uint32_t kBiasBytes = kMaxGWP * 32;
constexpr uint32_t kBiasLbo = 128, kBiasSbo = 256;
constexpr int kSmxWarps = 16;                    // four per TMEM lane quarter
constexpr int kSlices = kSmxWarps / 4;           // column slices of a tile
constexpr int kPoolWarp = 2 + kSmxWarps;         // warps 18 and 19 pool alternate tiles
constexpr int kThreads = 32 * (kPoolWarp + 2);
constexpr int kRing = 4;
constexpr int kRingPad = 16;                     // room for the previous tile's last 2h masses
static_assert(kMaxPool - 1 <= kRingPad, "the pooling halo must fit the ring pad");
constexpr float kNoWeight = -1.0e30f;            // bias of padding rows: weight 0

struct RingBars {
  uint64_t rfull[kRing], rempty[kRing], mass[kRing], hand[2], bias_free;
};

// State of a segment's candidate list, handed from the pooling warp of one
// tile to the pooling warp of the next.
struct ListHand {
  int cnt;
  long long tau;
};

struct WarpCompact {
  int hist[256];
};
constexpr int kCompactBatch = 4;   // list entries per lane in flight while compacting

__device__ __forceinline__ uint64_t rank_key(uint64_t e) {
  // (score bits, ~index): larger is better, the lower index wins a score tie
  return (e & 0xFFFFFFFF00000000ull) | (uint64_t)(~(uint32_t)e);
}

__device__ __forceinline__ uint32_t bf16_bits(float x) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// One warp keeps the n_keep best entries of buf[0..cnt) in place (order
// kept) by an 8-bit radix select on rank_key, and returns the new count;
// *tau becomes the score bits a later (higher-index) key must beat.  Out of
// line: it runs only when a list fills, and the pooling warps' hot code
// stays short (the pass ran about 1 us faster per layer).
__device__ __noinline__ int warp_compact(uint64_t* buf, int cnt, int n_keep, WarpCompact* wc, long long* tau, int* status) {
  const int lane = threadIdx.x & 31;
  if (n_keep <= 0) {
    *tau = LLONG_MAX;
    return 0;
  }
  unsigned long long prefix = 0;
  int need = n_keep;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = lane; i < 256; i += 32) wc->hist[i] = 0;
    __syncwarp();
    // kCompactBatch independent loads in flight per lane
    for (int i0 = 0; i0 < cnt; i0 += 32 * kCompactBatch) {
      uint64_t e[kCompactBatch];
#pragma unroll
      for (int q = 0; q < kCompactBatch; ++q) {
        const int i = i0 + 32 * q + lane;
        e[q] = i < cnt ? buf[i] : 0ull;
      }
#pragma unroll
      for (int q = 0; q < kCompactBatch; ++q) {
        const uint64_t key = rank_key(e[q]);
        if (i0 + 32 * q + lane < cnt && (shift == 56 || (key >> (shift + 8)) == (prefix >> (shift + 8))))
          atomicAdd(&wc->hist[(key >> shift) & 255], 1);
      }
    }
    __syncwarp();
    int local = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) local += wc->hist[255 - 8 * lane - i];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int before = incl - local;
    int d = -1, nd = 0, full = 0;
    if (before < need && need <= incl) {
      int cum = before;
      for (int i = 0; i < 8; ++i) {
        const int c = wc->hist[255 - 8 * lane - i];
        if (cum + c >= need) {
          d = 255 - 8 * lane - i;
          nd = need - cum;
          full = (nd == c);
          break;
        }
        cum += c;
      }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, d >= 0);
    __syncwarp();
    if (bal == 0) {  // inconsistent counts: keep everything
      if (lane == 0) record_status(status, kStatusCandOverflow);
      *tau = -1;
      return cnt;
    }
    const int src = __ffs(bal) - 1;
    d = __shfl_sync(0xffffffffu, d, src);
    nd = __shfl_sync(0xffffffffu, nd, src);
    full = __shfl_sync(0xffffffffu, full, src);
    prefix |= (unsigned long long)d << shift;
    need = nd;
    if (full) break;
  }
  const uint64_t T = prefix;
  int out = 0;
  // In place: a batch reads all of [b0, b0 + 32 * kCompactBatch) before it
  // writes, and every write lands below b0 + 32 * kCompactBatch (out never
  // passes the entries read), so no entry is overwritten before it is read.
  for (int b0 = 0; b0 < cnt; b0 += 32 * kCompactBatch) {
    uint64_t e[kCompactBatch];
#pragma unroll
    for (int q = 0; q < kCompactBatch; ++q) {
      const int i = b0 + 32 * q + lane;
      e[q] = i < cnt ? buf[i] : 0ull;
    }
#pragma unroll
    for (int q = 0; q < kCompactBatch; ++q) {
      const bool f = b0 + 32 * q + lane < cnt && rank_key(e[q]) >= T;
      const unsigned bal = __ballot_sync(0xffffffffu, f);
      if (f) buf[out + __popc(bal & ((1u << lane) - 1u))] = e[q];
      out += __popc(bal);
    }
    __syncwarp();
  }
  if (out != n_keep && lane == 0) record_status(status, kStatusCandOverflow);
  *tau = (long long)(T >> 32);
  return out;
}

// Whole warp: writes the bias operand of each segment (after the previous
// segment's MMAs are done with it); lane 0 issues the MMAs.
template <int D, int NL>
__device__ void mma_warp(const ScanArgs& A, PipeBars* bars, RingBars* rb, const Seg* segs, int nseg, uint32_t sQ,
                         uint32_t sK, uint32_t sOnes, uint32_t sBias, uint32_t tmem, volatile int* abort_flag) {
  constexpr int NKH = D / 64;
  constexpr int KSTEPS = D / 16;
  constexpr uint32_t kTileBytes = kTile * 128 * NKH;
  const int lane = threadIdx.x & 31;
  const uint32_t q_half = (uint32_t)A.nq * 128;
  const int hw = (A.pool_k - 1) / 2;
  const uint32_t idesc = tc::idesc_bf16(128, A.gwp16);
  // key side of the bias K-step: row r, K elements 0..2 = 1.0, the rest 0;
  // 16-byte unit i holds row 8*(i/16) + i%8, K elements 8*((i/8)%2) .. +7
  for (int i = lane; i < (int)(kOnesBytes / 16); i += 32) {
    const bool first = ((i >> 3) & 1) == 0;
    const uint4 val = first ? make_uint4(0x3F803F80u, 0x00003F80u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(sOnes + i * 16), "r"(val.x), "r"(val.y),
                 "r"(val.z), "r"(val.w)
                 : "memory");
  }
  // query side: only K elements 0..2 of each row ever hold data
  for (int i = lane; i < A.nq * 2; i += 32)
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};\n" ::"r"(sBias + i * 16), "r"(0u) : "memory");
  uint32_t stage = 0, phase = 0, qphase = 0, buf = 0, tphase = 0, bphase = 0;
  // query side of the bias K-step: row q, K elements 0..2 = the row's bias
  // split into three bf16 terms; lane l handles rows l, l+32, ....  The
  // next segment's biases are loaded as soon as the current segment's
  // operand is written, so they are in registers by the time its MMAs drain
  // (fetched at the switch, they held the switch up by about 3 us).
  float bv[kMaxGWP / 32];
  auto load_bias = [&](int si) {
#pragma unroll
    for (int i = 0; i < kMaxGWP / 32; ++i) {
      const int row = lane + 32 * i;
      bv[i] = (row < A.gwp16) ? A.bias[(size_t)segs[si].bh * A.gwp16 + row] : kNoWeight;
    }
  };
  load_bias(0);
  for (int s = 0; s < nseg; ++s) {
    const Seg sg = segs[s];
    int okl = 1;
    if (s > 0) {
      if (lane == 0) okl = wait_bar(smem_u32(&rb->bias_free), bphase, abort_flag, A.status, A.wait_limit);
      bphase ^= 1;
    }
    if (!__shfl_sync(0xffffffffu, okl, 0)) return;
#pragma unroll
    for (int i = 0; i < kMaxGWP / 32; ++i) {
      const int row = lane + 32 * i;
      if (row < A.nq) {
        const float b = bv[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(b);
        const float r1 = b - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);
        const uint32_t x = bf16_bits(__bfloat162float(hi)) | (bf16_bits(__bfloat162float(mid)) << 16);
        const uint32_t y = bf16_bits(r2);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %3};\n" ::"r"(sBias + (row >> 3) * kBiasSbo + (row & 7) * 16),
                     "r"(x), "r"(y), "r"(0u)
                     : "memory");
      }
    }
    tc::fence_proxy_async();
    __syncwarp();
    if (s + 1 < nseg) load_bias(s + 1);
    if (lane == 0) {
      if (!wait_bar(smem_u32(&bars->qfull), qphase, abort_flag, A.status, A.wait_limit)) okl = 0;
      qphase ^= 1;
      const int ntiles = (sg.b - sg.a + 2 * hw + kTile - 1) / kTile;
      for (int t = 0; t < ntiles && okl; ++t) {
        if (!wait_bar(smem_u32(&bars->full[stage]), phase, abort_flag, A.status, A.wait_limit) ||
            !wait_bar(smem_u32(&bars->tempty[buf]), tphase ^ 1, abort_flag, A.status, A.wait_limit)) {
          okl = 0;
          break;
        }
        tc::fence_after_sync();
        const uint32_t kb = sK + stage * kTileBytes;
        const uint32_t dacc = tmem + buf * (NL == 4 ? 256u : 128u);
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
          const uint32_t koff = (ks >> 2) * (kTile * 128) + (ks & 3) * 32;
          const uint32_t qoff = (ks >> 2) * q_half + (ks & 3) * 32;
          tc::mma_bf16(dacc, tc::desc_sw128(kb + koff), tc::desc_sw128(sQ + qoff), idesc, ks > 0);
        }
        tc::mma_bf16(dacc, tc::desc_nosw(sOnes, kBiasLbo, kBiasSbo), tc::desc_nosw(sBias, kBiasLbo, kBiasSbo), idesc, 1);
        tc::mma_commit(smem_u32(&bars->empty[stage]));
        tc::mma_commit(smem_u32(&bars->tfull[buf]));
        if (++stage == kStages2) { stage = 0; phase ^= 1; }
        if (++buf == (NL == 4 ? 2u : 4u)) { buf = 0; tphase ^= 1; }
      }
      if (okl) {
        tc::mma_commit(smem_u32(&bars->qempty));
        tc::mma_commit(smem_u32(&rb->bias_free));
      }
    }
    if (!__shfl_sync(0xffffffffu, okl, 0)) return;
  }
}

// The pooled scores of four keys for a pool width other than 7 (the
// long-context workloads use 7), out of line: the window's masses summed
// in ascending key order, as the inline 7-wide path does.
__device__ __noinline__ float4 pool_generic(const float* rr, int hw, int pool_k, float inv_pool) {
  const int lane = threadIdx.x & 31;
  const float* win = rr + kRingPad - 2 * hw + 4 * lane;
  float sc[4];
  for (int k = 0; k < 4; ++k) {
    float acc = 0.f;
    for (int d = 0; d <= 2 * hw; ++d) acc += win[k + d];
    sc[k] = pool_k == 1 ? acc : acc * inv_pool;
  }
  return make_float4(sc[0], sc[1], sc[2], sc[3]);
}

// NL: 16-column accumulator chunks each softmax warp loads.  Windows of up
// to 128 rows (G*W <= 128: at most two chunks a warp) run with NL = 2 and
// four 128-column accumulators in tensor memory, so the MMA runs up to four
// tiles ahead of the exponentials; wider windows with NL = 4 and two
// 256-column accumulators.
template <int D, bool CAND, int NL>
__global__ void __launch_bounds__(kThreads, 1)
kvc_tc_pass2_kernel(const __grid_constant__ ScanArgs A, const __grid_constant__ SelParams sel,
                    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap) {
  constexpr int NKH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  __shared__ PipeBars bars;
  __shared__ RingBars rbars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ __align__(16) float s_ring[kRing][kRingPad + kTile];   // key masses, pooled in key order
  __shared__ __align__(16) float s_part[kRing][kSlices][kTile];     // per-slice sums of each key
  __shared__ WarpCompact s_wc;
  __shared__ ListHand s_hand[2];

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sOnes = base;                       // the small blocks first: 12 KB, keeps sQ 1024-aligned
  const uint32_t sBias = sOnes + kOnesBytes;
  const uint32_t sQ = sBias + kBiasBytes;
  const uint32_t sK = sQ + (uint32_t)A.nq * 128 * NKH;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    init_pipe_bars(&bars, kSmxWarps, kStages2);
    for (int i = 0; i < kRing; ++i) {
      tc::mbar_init(smem_u32(&rbars.rfull[i]), kSmxWarps);
      // a slot is free once its own pooling warp and the next tile's (which
      // reads the last masses as its halo) are done with it
      tc::mbar_init(smem_u32(&rbars.rempty[i]), 2);
      tc::mbar_init(smem_u32(&rbars.mass[i]), 1);
    }
    tc::mbar_init(smem_u32(&rbars.hand[0]), 1);
    tc::mbar_init(smem_u32(&rbars.hand[1]), 1);
    tc::mbar_init(smem_u32(&rbars.bias_free), 1);
    s_abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(&s_tmem), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  // Everything above overlaps the previous grid.  Its outputs (the row
  // biases) are read below; when the keys and queries are known to be ready,
  // the TMA warp starts loading them at once.
  if (!(A.inputs_ready && warp == 0)) grid_dep_wait();
  grid_dep_launch();

  const int hw = (A.pool_k - 1) / 2;
  Seg segs[kMaxSegs];
  const int nseg = cta_segments(A, blockIdx.x, segs);

  if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&qmap);
      tc::tma_prefetch_desc(&kmap);
      producer<D, 2, kStages2>(A, &qmap, &kmap, &bars, sQ, sK, &s_abort);
    }
  } else if (warp == 1) {
    mma_warp<D, NL>(A, &bars, &rbars, segs, nseg, sQ, sK, sOnes, sBias, tmem, &s_abort);
    if (lane == 0) drain_mma(smem_u32(&bars.drain[0]), A.status);   // its MMAs are done before TMEM is freed
  } else if (warp < kPoolWarp) {
    // ---------------------------------------------------- softmax warps
    // Warp k of a lane quarter owns column chunks [k*cw, k*cw + cw) of the
    // G*W (rounded to 16) window columns, cw = ceil(chunks / 4) <= NL.  It
    // always loads NL 16-column chunks (they stay inside its accumulator:
    // columns c0*16 .. c0*16 + 16*NL - 1 with c0 <= 3*cw, at most 127 of 128
    // with NL = 2 and 255 of 256 with NL = 4); chunks past its slice or past
    // the last one weigh nothing.
    const int k = (warp - 2) >> 2;
    const int quarter = warp & 3;
    const int krow = quarter * 32 + lane;
    const int nch = A.gwp16 / 16;
    const int cw = (nch + kSlices - 1) / kSlices;
    const int c0 = k * cw;
    const int c_end = min(c0 + cw, nch);     // chunks c0 .. c_end-1 are this warp's
    const float c2 = A.c2;
    const float2 cc = make_float2(c2, c2);
    const uint32_t tlane = (uint32_t)(quarter * 32) << 16;
    int tcount = 0;
    bool ok = true;
    for (int s = 0; s < nseg && ok; ++s) {
      const Seg sg = segs[s];
      const int n_iter = (sg.b - sg.a + 2 * hw + kTile - 1) / kTile;
      for (int it = 0; it < n_iter; ++it, ++tcount) {
        const int t0 = sg.a - hw + it * kTile;
        constexpr uint32_t kBufs = NL == 4 ? 2u : 4u, kCols = NL == 4 ? 256u : 128u;
        const uint32_t buf = (uint32_t)tcount % kBufs;
        if (!wait_bar_warp(smem_u32(&bars.tfull[buf]), ((uint32_t)tcount / kBufs) & 1u, &s_abort, A.status,
                           A.wait_limit)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        float v[16 * NL];
        const uint32_t taddr = tmem + buf * kCols + tlane + (uint32_t)c0 * 16;
#pragma unroll
        for (int i = 0; i < NL; ++i) tc::tmem_ld16(taddr + i * 16, v + 16 * i);
        tc::tmem_wait_ld();
        tc::reg_fence(v, 16 * NL);
        // the accumulator is free for the MMA warp as soon as it is in registers
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(smem_u32(&bars.tempty[buf]));
        // Chunks past this warp's slice carry no weight and are skipped (a
        // warp-uniform test per chunk: G*W = 128 fills only half of the 16
        // chunks, G*W = 160 ten); in tiles near the window, the window
        // queries a key comes after (query i of column g*W + i sees key j
        // only when j <= S - W + i) become -inf (2^-inf = 0).  Every key
        // then runs the same arithmetic in the same order, so keys with equal
        // inputs get bit-identical masses wherever they sit.
        const int nv = c_end - c0;   // chunks of this warp that carry weight
        if (t0 + kTile - 1 > A.S - A.W) {
          const int dj = t0 + krow - (A.S - A.W);
          if (dj > 0) {
            int wi = (c0 * 16) % A.W;
#pragma unroll
            for (int c = 0; c < 16 * NL; ++c) {
              if (wi < dj) v[c] = -INFINITY;
              if (++wi == A.W) wi = 0;
            }
          }
        }
        float2 a0 = make_float2(0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
#pragma unroll
        for (int ch = 0; ch < NL; ++ch) {
          if (ch < nv) {
#pragma unroll
            for (int c = 16 * ch; c < 16 * ch + 16; c += 8) {
              const float2 x0 = __fmul2_rn(make_float2(v[c], v[c + 1]), cc);
              const float2 x1 = __fmul2_rn(make_float2(v[c + 2], v[c + 3]), cc);
              const float2 x2 = __fmul2_rn(make_float2(v[c + 4], v[c + 5]), cc);
              const float2 x3 = __fmul2_rn(make_float2(v[c + 6], v[c + 7]), cc);
              a0 = __fadd2_rn(a0, make_float2(ex2(x0.x), ex2(x0.y)));
              a1 = __fadd2_rn(a1, make_float2(ex2(x1.x), ex2(x1.y)));
              a2 = __fadd2_rn(a2, make_float2(ex2(x2.x), ex2(x2.y)));
              a3 = __fadd2_rn(a3, make_float2(ex2(x3.x), ex2(x3.y)));
            }
          }
        }
        const float r = (a0.x + a0.y) + (a1.x + a1.y) + ((a2.x + a2.y) + (a3.x + a3.y));
        const int slot = tcount % kRing;
        if (!wait_bar_warp(smem_u32(&rbars.rempty[slot]), ((tcount / kRing) & 1) ^ 1, &s_abort, A.status,
                           A.wait_limit)) {
          ok = false;
          break;
        }
        s_part[slot][k][krow] = r;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(smem_u32(&rbars.rfull[slot]));
      }
    }
  } else {
    // ------------------------------------------------------ pooling warps
    // Warp `who` pools the tiles with tcount % 2 == who.  A tile's pad (the
    // previous tile's last 2h masses) is read from the previous slot once
    // its pooling warp has written them; the list state (count, threshold)
    // comes from the previous tile's warp after its appends, so the list is
    // written in key order.
    const int who = warp - kPoolWarp;
    const float inv_pool = 1.0f / (float)A.pool_k;
    int tcount = 0;
    bool ok = true;
    for (int s = 0; s < nseg && ok; ++s) {
      const Seg sg = segs[s];
      const int hk = sg.bh % A.H_kv;
      const size_t slot_id = (size_t)blockIdx.x * A.maxseg + (size_t)(sg.bh - segs[0].bh);
      uint64_t* my_cand = CAND ? A.cand + slot_id * A.cap : nullptr;
      const int n_keep = CAND ? sel.n_sel[hk] : 0;
      const int n_iter = (sg.b - sg.a + 2 * hw + kTile - 1) / kTile;
      for (int it = 0; it < n_iter; ++it, ++tcount) {
        if ((tcount & 1) != who) continue;
        const int t0 = sg.a - hw + it * kTile;
        const int slot = tcount % kRing;
        const int prev = (tcount + kRing - 1) % kRing;
        float* rr = s_ring[slot];   // [kRingPad - 2h, kRingPad): previous tile's last masses
        if (!wait_bar_warp(smem_u32(&rbars.rfull[slot]), (tcount / kRing) & 1, &s_abort, A.status, A.wait_limit)) {
          ok = false;
          break;
        }
        {
          // key mass = the sum of its four slice sums; keys outside [0, S) weigh nothing
          const int jb = t0 + 4 * lane;
          float4 m4 = *reinterpret_cast<const float4*>(&s_part[slot][0][4 * lane]);
#pragma unroll
          for (int q = 1; q < kSlices; ++q) {
            const float4 p4 = *reinterpret_cast<const float4*>(&s_part[slot][q][4 * lane]);
            m4.x += p4.x;
            m4.y += p4.y;
            m4.z += p4.z;
            m4.w += p4.w;
          }
          if (jb < 0 || jb + 3 >= A.S) {
            if (jb + 0 < 0 || jb + 0 >= A.S) m4.x = 0.f;
            if (jb + 1 < 0 || jb + 1 >= A.S) m4.y = 0.f;
            if (jb + 2 < 0 || jb + 2 >= A.S) m4.z = 0.f;
            if (jb + 3 < 0 || jb + 3 >= A.S) m4.w = 0.f;
          }
          *reinterpret_cast<float4*>(&rr[kRingPad + 4 * lane]) = m4;
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(smem_u32(&rbars.mass[slot]));
        }
        // the pad: the previous tile's last 2h masses, or none at a segment start
        if (it > 0) {
          const int tp = tcount - 1;
          if (!wait_bar_warp(smem_u32(&rbars.mass[prev]), (tp / kRing) & 1, &s_abort, A.status, A.wait_limit)) {
            ok = false;
            break;
          }
          if (lane < 2 * hw) rr[kRingPad - 2 * hw + lane] = s_ring[prev][kRingPad + kTile - 2 * hw + lane];
        } else if (lane < kRingPad) {
          rr[lane] = 0.f;
        }
        __syncwarp();
        if (tcount > 0 && lane == 0) tc::mbar_arrive(smem_u32(&rbars.rempty[prev]));
        // lane l pools keys t0 - h + 4l + k, k = 0..3, over the masses of keys
        // t0 - 2h + 4l + k .. t0 + 4l + k, summed in ascending key order
        float sc[4];
        if (hw == 3) {
          // the 7-wide pool of the long-context workloads: three aligned
          // 16-byte loads cover the ten masses a lane needs
          const float* b4 = rr + kRingPad - 8 + 4 * lane;
          const float4 x0 = *reinterpret_cast<const float4*>(b4);
          const float4 x1 = *reinterpret_cast<const float4*>(b4 + 4);
          const float4 x2 = *reinterpret_cast<const float4*>(b4 + 8);
          const float w[12] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w, x2.x, x2.y, x2.z, x2.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            float acc = w[2 + k];
#pragma unroll
            for (int d = 1; d <= 6; ++d) acc += w[2 + k + d];
            sc[k] = acc * inv_pool;
          }
        } else {
          const float4 g4 = pool_generic(rr, hw, A.pool_k, inv_pool);
          sc[0] = g4.x;
          sc[1] = g4.y;
          sc[2] = g4.z;
          sc[3] = g4.w;
        }
        const int j0 = t0 - hw + 4 * lane;
        if (!CAND) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            if (j0 + k >= sg.a && j0 + k < sg.b) A.scores[(size_t)sg.bh * A.S + j0 + k] = sc[k];
        } else {
          uint32_t u[4];
          bool is_cand[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            u[k] = __float_as_uint(sc[k]);
            if (u[k] == 0x80000000u) u[k] = 0u;
            const int jo = j0 + k;
            is_cand[k] = jo >= sg.a && jo < sg.b && jo >= sel.r_lo && jo < sel.r_hi;
          }
          // the list as the previous tile of this segment left it (a new
          // segment starts an empty list); the previous tile's hand-off is
          // awaited even then, so its reader is done with the slot this
          // tile's state overwrites
          int cnt = 0;
          long long tau = -1;
          if (tcount > 0) {
            const int tp = tcount - 1;
            if (!wait_bar_warp(smem_u32(&rbars.hand[tp & 1]), (tp >> 1) & 1, &s_abort, A.status, A.wait_limit)) {
              ok = false;
              break;
            }
            if (it > 0) {
              cnt = s_hand[tp & 1].cnt;
              tau = s_hand[tp & 1].tau;
            }
          }
          // a key's place in the list: the candidates of lower lanes first,
          // then this lane's lower keys (four ballots, no scan)
          const unsigned lt = (1u << lane) - 1u;
          for (int tries = 0;; ++tries) {
            bool take[4];
            unsigned bal[4];
            int before = 0, n_new = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              take[k] = is_cand[k] && (long long)u[k] > tau;
              bal[k] = __ballot_sync(0xffffffffu, take[k]);
              before += __popc(bal[k] & lt);
              n_new += __popc(bal[k]);
            }
            if (cnt + n_new > A.cap) {
              if (cnt <= n_keep || tries >= 2) {
                if (lane == 0) record_status(A.status, kStatusCandOverflow);
                break;
              }
              cnt = warp_compact(my_cand, cnt, n_keep, &s_wc, &tau, A.status);
              continue;
            }
            int pos = cnt + before;
            if (take[0] && take[1] && take[2] && take[3] && ((reinterpret_cast<uintptr_t>(my_cand + pos) & 15u) == 0)) {
              // all four keys of the lane (the common case while the list has
              // room): two 16-byte stores, so a warp writes 1 KB contiguously
              ulonglong2 e01, e23;
              e01.x = ((uint64_t)u[0] << 32) | (uint32_t)(j0 + 0);
              e01.y = ((uint64_t)u[1] << 32) | (uint32_t)(j0 + 1);
              e23.x = ((uint64_t)u[2] << 32) | (uint32_t)(j0 + 2);
              e23.y = ((uint64_t)u[3] << 32) | (uint32_t)(j0 + 3);
              *reinterpret_cast<ulonglong2*>(my_cand + pos) = e01;
              *reinterpret_cast<ulonglong2*>(my_cand + pos + 2) = e23;
            } else {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                if (take[k]) my_cand[pos++] = ((uint64_t)u[k] << 32) | (uint32_t)(j0 + k);
              }
            }
            cnt += n_new;
            break;
          }
          if (lane == 0) {
            s_hand[tcount & 1].cnt = cnt;
            s_hand[tcount & 1].tau = tau;
            if (it + 1 == n_iter) A.cand_cnt[slot_id] = cnt;
          }
        }
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(smem_u32(&rbars.hand[tcount & 1]));
          tc::mbar_arrive(smem_u32(&rbars.rempty[slot]));
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// Bias of every window row: -lse2 / (log2(e)/sqrt(D)), from (m, Z) in
// natural units or from the pass-1 slots; padding rows get no weight.
// One warp per window row: the lanes merge the row's pass-1 slots in
// parallel, then a butterfly merges the lanes.
__global__ void kvc_lse_bias_kernel(const __grid_constant__ ScanArgs A, float* __restrict__ bias) {
  grid_dep_wait();
  grid_dep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int r = blockIdx.x * (blockDim.x >> 5) + warp;
  if (r >= A.gwp16) return;
  const int b = bh / A.H_kv, h = bh % A.H_kv, G = A.H_q / A.H_kv;
  float out = kNoWeight;
  if (r < A.gw) {
    float lse2;
    if (A.m_in != nullptr) {
      const size_t src = (size_t)(b * A.H_q + h * G) * A.W + r;
      lse2 = A.m_in[src] * kLog2e + log2f(A.z_in[src]);
    } else {
      const int64_t S = A.S, total = (int64_t)A.B * A.H_kv * A.S;
      const int c_first = (int)range_of((int64_t)bh * S, A.L, S, total);
      const int c_last = (int)range_of(((int64_t)bh + 1) * S - 1, A.L, S, total);
      float2 st = make_float2(-INFINITY, 0.f);
      for (int c = c_first + lane; c <= c_last; c += 32) {
        const int seg = bh - (int)(range_begin(c, A.L, S, total) / S);
        const size_t o = ((size_t)c * A.maxseg + seg) * A.gwp16 + r;
        st = merge_mz(st, make_float2(A.pm_in[o], A.pz_in[o]));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, st.x, o), __shfl_xor_sync(0xffffffffu, st.y, o));
        st = merge_mz(st, other);
      }
      lse2 = st.x + log2f(st.y);
    }
    out = -lse2 / A.c2;
  }
  if (lane == 0) bias[(size_t)bh * A.gwp16 + r] = out;
}

template <typename Kern>
cudaError_t launch(Kern kernel, int grid, size_t smem, cudaStream_t st, const ScanArgs& A, const SelParams& sp,
                   const CUtensorMap& qm, const CUtensorMap& km) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if ((e = launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, st, A, sp, qm, km)) != cudaSuccess) return e;
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pass2(const __nv_bfloat16* q, const __nv_bfloat16* k, const float* m, const float* Z,
                         const float* part_m, const float* part_z, float* bias_ws, int B, int H_q, int H_kv, int S,
                         int D, int W, int pool_k, const ScanPlan& pl, int gwp, const SelParams* sel, Pass2Out out,
                         bool inputs_ready, cudaStream_t st) {
  (void)gwp;
  ScanArgs A = base_args(pl, B, H_q, H_kv, S, D, W);
  A.nq = A.gwp16;
  A.pool_k = pool_k;
  A.inputs_ready = inputs_ready ? 1 : 0;
  A.m_in = m;
  A.z_in = Z;
  A.pm_in = part_m;
  A.pz_in = part_z;
  A.bias = bias_ws;
  A.scores = out.scores;
  A.cand = out.cand;
  A.cand_cnt = out.cand_cnt;
  A.cap = out.cap;
  cudaError_t e = launch_pdl(kvc_lse_bias_kernel, dim3((A.gwp16 + 7) / 8, B * H_kv), dim3(256), 0, st, A, bias_ws);
  note_launches(1);
  if (e != cudaSuccess) return e;
  CUtensorMap qm, km;
  if (!make_map(&qm, q, D, (uint64_t)B * H_q * W, 1, A.nq) || !make_map(&km, k, D, S, (uint64_t)B * H_kv, kTile))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + kOnesBytes + kBiasBytes + (size_t)A.nq * 128 * (D / 64) +
                      (size_t)kStages2 * kTile * 128 * (D / 64);
  const bool cand = out.cand != nullptr;
  const bool narrow = A.gwp16 <= 128;   // two chunks a softmax warp, four accumulators
  if (D == 64) {
    if (narrow)
      return cand ? launch(kvc_tc_pass2_kernel<64, true, 2>, pl.P, smem, st, A, *sel, qm, km)
                  : launch(kvc_tc_pass2_kernel<64, false, 2>, pl.P, smem, st, A, *sel, qm, km);
    return cand ? launch(kvc_tc_pass2_kernel<64, true, 4>, pl.P, smem, st, A, *sel, qm, km)
                : launch(kvc_tc_pass2_kernel<64, false, 4>, pl.P, smem, st, A, *sel, qm, km);
  }
  if (narrow)
    return cand ? launch(kvc_tc_pass2_kernel<128, true, 2>, pl.P, smem, st, A, *sel, qm, km)
                : launch(kvc_tc_pass2_kernel<128, false, 2>, pl.P, smem, st, A, *sel, qm, km);
  return cand ? launch(kvc_tc_pass2_kernel<128, true, 4>, pl.P, smem, st, A, *sel, qm, km)
              : launch(kvc_tc_pass2_kernel<128, false, 4>, pl.P, smem, st, A, *sel, qm, km);
}

}  // namespace kvc
