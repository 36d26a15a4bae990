// Pass 1 of the two-pass scorer (TideKV, Fig. 3): per window query, the
// log-sum-exp normalisers over the prefix keys, kept as W-length state.
//
// A = window queries (one or two 128-row MMA blocks), B = 128-key tile, both
// read by the tensor core from shared memory; the accumulators rotate
// through four 128-column tensor-memory buffers, one per (tile, query block)
// "sub-tile".  Two threads on different warps issue the MMAs, taking
// alternate sub-tiles: a thread that waits on an mbarrier stops feeding the
// tensor core for a few hundred cycles, which a lone issuer of 64-cycle
// MMAs cannot hide, while two issuers cover each other's waits.  Sixteen
// softmax warps, four per tensor-memory lane quarter: with two query blocks,
// warp k of a quarter reads block k/2, columns 64*(k%2) .. +63 of each tile;
// with one block, columns 32*k .. +31.  A warp hands its buffer back as soon
// as its columns are in registers, so the MMAs run ahead of the
// exponentials by up to four sub-tiles.  Each thread owns one query row and
// keeps a reference maximum m (raw dot-product units) and the sum Z of
// 2^(x - m * c), x = q.k * c, c = log2(e)/sqrt(D), over its columns of the
// segment; at the end of a segment the warps that share a row merge their
// (m, Z) and write the row's (m * c, Z) partial to the segment's slot.
#include "kvc_scan_common.cuh"

namespace kvc {
namespace {

using namespace scan;

constexpr int kSmxWarps = 16;
constexpr int kSmxThreads = kSmxWarps * 32;
constexpr int kFirstSmx = 3;                  // warp 0 TMA, warps 1-2 MMA issuers
constexpr int kThreads = 32 * kFirstSmx + kSmxThreads;
constexpr uint32_t kP1Bufs = 4;               // 128-column accumulator buffers
constexpr float kBatchSumLimit = 1.152921504606846976e18f;   // 2^60

__device__ __forceinline__ void smx_sync() { asm volatile("bar.sync 1, %0;\n" ::"n"(kSmxThreads) : "memory"); }

// Largest of N values (two chains).
template <int N>
__device__ __forceinline__ float batch_max(const float* v) {
  float mx0 = fmaxf(v[0], v[1]), mx1 = fmaxf(v[2], v[3]);
#pragma unroll
  for (int c = 4; c < N; c += 4) {
    mx0 = fmaxf(mx0, fmaxf(v[c], v[c + 1]));
    mx1 = fmaxf(mx1, fmaxf(v[c + 2], v[c + 3]));
  }
  return fmaxf(mx0, mx1);
}

// Sum of 2^(v * c2 + nm) over N values, as two partial sums.
template <int N>
__device__ __forceinline__ float2 batch_sum(const float* v, float c2, float nm) {
  const float2 cc = make_float2(c2, c2), nn = make_float2(nm, nm);
  float2 a0 = make_float2(0.f, 0.f), a1 = a0, a2 = a0, a3 = a0;
#pragma unroll
  for (int c = 0; c < N; c += 8) {
    const float2 x0 = __ffma2_rn(make_float2(v[c], v[c + 1]), cc, nn);
    const float2 x1 = __ffma2_rn(make_float2(v[c + 2], v[c + 3]), cc, nn);
    const float2 x2 = __ffma2_rn(make_float2(v[c + 4], v[c + 5]), cc, nn);
    const float2 x3 = __ffma2_rn(make_float2(v[c + 6], v[c + 7]), cc, nn);
    a0 = __fadd2_rn(a0, make_float2(ex2(x0.x), ex2(x0.y)));
    a1 = __fadd2_rn(a1, make_float2(ex2(x1.x), ex2(x1.y)));
    a2 = __fadd2_rn(a2, make_float2(ex2(x2.x), ex2(x2.y)));
    a3 = __fadd2_rn(a3, make_float2(ex2(x3.x), ex2(x3.y)));
  }
  return __fadd2_rn(__fadd2_rn(a0, a1), __fadd2_rn(a2, a3));
}

// A batch whose sum would pass 2^60 (a score far above the reference),
// redone against a raised reference.  Rare, and out of line so that the
// unrolled hot loop stays short: the values come in a local copy, and the
// arithmetic is the hot path's, in the same order.
template <int N>
__device__ __noinline__ float2 redo_batch(const float* v, float c2, float2 z2, float* mref) {
  const float mnew = fmaxf(*mref, batch_max<N>(v));
  const float sc = ex2((*mref - mnew) * c2);
  z2.x *= sc;
  z2.y *= sc;
  *mref = mnew;
  return __fadd2_rn(z2, batch_sum<N>(v, c2, -mnew * c2));
}

// MMA issuer `who` (0 or 1) of pass 1: sub-tiles u = NMB * tile + block with
// u % 2 == who, in order.  A tile's ring stage is released by a commit of
// each issuer that used it; the queries of a segment, by a commit of both.
template <int D, int NMB>
__device__ void mma_pass1(const ScanArgs& A, PipeBars* bars, const Seg* segs, int nseg, uint32_t sQ, uint32_t sK,
                          uint32_t tmem, int who, volatile int* abort_flag) {
  constexpr int NKH = D / 64;
  constexpr int KSTEPS = D / 16;
  constexpr uint32_t kTileBytes = kTile * 128 * NKH;
  const uint32_t q_half = (uint32_t)A.nq * 128;
  const uint32_t idesc = tc::idesc_bf16(128, 128);
  uint32_t qphase = 0, u = 0, tcount = 0;
  for (int si = 0; si < nseg; ++si) {
    const Seg sg = segs[si];
    if (!wait_bar(smem_u32(&bars->qfull), qphase, abort_flag, A.status, A.wait_limit)) return;
    qphase ^= 1;
    const int ntiles = (sg.b - sg.a + kTile - 1) / kTile;
    for (int t = 0; t < ntiles; ++t, ++tcount) {
      const uint32_t stage = tcount % kStages, phase = (tcount / kStages) & 1u;
      bool mine = false;
      for (int mb = 0; mb < NMB; ++mb, ++u) {
        if ((int)(u & 1u) != who) continue;
        if (!mine) {
          if (!wait_bar(smem_u32(&bars->full[stage]), phase, abort_flag, A.status, A.wait_limit)) return;
          mine = true;
        }
        const uint32_t b = u % kP1Bufs;
        if (!wait_bar(smem_u32(&bars->tempty[b]), ((u / kP1Bufs) & 1u) ^ 1u, abort_flag, A.status, A.wait_limit))
          return;
        tc::fence_after_sync();
        const uint32_t kb = sK + stage * kTileBytes;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
          const uint32_t koff = (ks >> 2) * (kTile * 128) + (ks & 3) * 32;
          const uint32_t qoff = (ks >> 2) * q_half + mb * (128 * 128) + (ks & 3) * 32;
          tc::mma_bf16(tmem + b * 128, tc::desc_sw128(sQ + qoff), tc::desc_sw128(kb + koff), idesc, ks > 0);
        }
        tc::mma_commit(smem_u32(&bars->tfull[b]));
      }
      if (mine) tc::mma_commit(smem_u32(&bars->empty[stage]));
    }
    // the queries in shared memory are free once this segment's MMAs are done
    tc::mma_commit(smem_u32(&bars->qempty));
  }
}

template <int D, int NMB, bool EXACT_MAX>
__global__ void __launch_bounds__(kThreads, 1)
kvc_tc_pass1_kernel(const __grid_constant__ ScanArgs A, const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap) {
  constexpr int NCW = NMB == 2 ? 64 : 32;       // accumulator columns per softmax warp per tile
  constexpr int NPART = NMB == 2 ? 2 : 4;       // warps sharing a query row
  extern __shared__ uint8_t smem_raw[];
  __shared__ PipeBars bars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ float2 s_part[4][128];

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sK = base + (uint32_t)A.nq * 128 * (D / 64);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    // a stage is used by both issuers with two query blocks, by one otherwise
    init_pipe_bars(&bars, kSmxWarps / NMB, kStages, NMB, 2);
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
  // everything above overlaps the previous grid; its outputs are read below
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&qmap);
      tc::tma_prefetch_desc(&kmap);
      producer<D, 1>(A, &qmap, &kmap, &bars, sQ, sK, &s_abort);
    }
  } else if (warp < kFirstSmx) {
    if (lane == 0) {
      Seg segs[kMaxSegs];
      const int nseg = cta_segments(A, blockIdx.x, segs);
      mma_pass1<D, NMB>(A, &bars, segs, nseg, sQ, sK, tmem, warp - 1, &s_abort);
      drain_mma(smem_u32(&bars.drain[warp - 1]), A.status);   // its MMAs are done before TMEM is freed
    }
  } else {
    const int k = (warp - kFirstSmx) >> 2;     // 0..3
    const int quarter = warp & 3;              // TMEM lanes this warp may read
    const int mb = NMB == 2 ? (k >> 1) : 0;
    const int part = NMB == 2 ? (k & 1) : k;   // column slice of the tile
    const int col0 = part * NCW;
    const int row = mb * 128 + quarter * 32 + lane;
    const bool active = (mb * 128 + quarter * 32) < A.gw;
    const float c2 = A.c2;
    const int t_row = A.S - A.W + (row % A.W);
    Seg segs[kMaxSegs];
    const int nseg = cta_segments(A, blockIdx.x, segs);
    uint32_t tcount = 0;
    bool ok = true;
    // every warp passes the two named barriers of each segment even after a
    // wait gave up, so none is left waiting there
    for (int si = 0; si < nseg; ++si) {
      const Seg sg = segs[si];
      float mref = -INFINITY;
      float2 z2 = make_float2(0.f, 0.f);
      const int ntiles = (sg.b - sg.a + kTile - 1) / kTile;
      for (int ti = 0; ti < ntiles && ok; ++ti, ++tcount) {
        const int t = p1_tile_order(ti, ntiles);
        const uint32_t u = (uint32_t)NMB * tcount + (uint32_t)mb;   // this warp's sub-tile
        const uint32_t buf = u % kP1Bufs;
        if (!wait_bar_warp(smem_u32(&bars.tfull[buf]), (u / kP1Bufs) & 1u, &s_abort, A.status, A.wait_limit)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t taddr = tmem + buf * 128 + col0 + ((uint32_t)(quarter * 32) << 16);
        // Every warp loads, active or not (a load under a runtime condition
        // costs far more than the rows an idle warp never uses); the buffer
        // goes back to the MMA warp right after.
        float v[NCW];
#pragma unroll
        for (int c = 0; c < NCW; c += 16) tc::tmem_ld16(taddr + c, v + c);
        tc::tmem_wait_ld();
        tc::reg_fence(v, NCW);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(smem_u32(&bars.tempty[buf]));
        if (!active) continue;
        const int t0 = sg.a + t * kTile + col0;
        if (t0 + NCW - 1 >= sg.b || t0 + NCW - 1 > A.S - A.W) {
#pragma unroll
          for (int c = 0; c < NCW; ++c) {
            const int j = t0 + c;
            if (j >= sg.b || j > t_row) v[c] = -INFINITY;
          }
        }
        if (EXACT_MAX) {
          // running maximum: the sum so far is rescaled when it grows
          const float mx = batch_max<NCW>(v);
          if (mx > mref) {
            const float sc = (mref == -INFINITY) ? 0.f : ex2((mref - mx) * c2);
            z2.x *= sc;
            z2.y *= sc;
            mref = mx;
          }
          if (mref > -INFINITY) z2 = __fadd2_rn(z2, batch_sum<NCW>(v, c2, -mref * c2));
          continue;
        }
        // The sum is kept relative to a reference mref (raw units): the
        // first finite batch maximum of the segment.  A batch whose sum
        // passes 2^60 (a score far above mref) is redone against a raised
        // reference, so the fp32 state never overflows; any reference gives
        // the same log-sum-exp.
        if (mref == -INFINITY) mref = batch_max<NCW>(v);
        if (mref > -INFINITY) {
          const float2 bs = batch_sum<NCW>(v, c2, -mref * c2);
          if (!(bs.x + bs.y <= kBatchSumLimit)) {
            float vv[NCW];
#pragma unroll
            for (int c = 0; c < NCW; ++c) vv[c] = v[c];
            z2 = redo_batch<NCW>(vv, c2, z2, &mref);
          } else {
            z2 = __fadd2_rn(z2, bs);
          }
        }
      }
      // segment done: the NPART column slices of a row are merged in slice order
      const float2 mine = make_float2(mref == -INFINITY ? -INFINITY : mref * c2, z2.x + z2.y);
      const size_t slot = (size_t)blockIdx.x * A.maxseg + (size_t)(sg.bh - segs[0].bh);
      s_part[k][quarter * 32 + lane] = mine;
      smx_sync();
      if (part == 0 && ok && row < A.gwp16) {
        float2 st = mine;
#pragma unroll
        for (int q = 1; q < NPART; ++q) st = merge_mz(st, s_part[k + q][quarter * 32 + lane]);
        A.part_m[slot * A.gwp16 + row] = st.x;
        A.part_z[slot * A.gwp16 + row] = st.y;
      }
      smx_sync();
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// m, Z (natural-log units) of every window row from the pass-1 slots.
__global__ void kvc_pass1_combine_kernel(const __grid_constant__ ScanArgs A, float* __restrict__ m,
                                         float* __restrict__ Z) {
  grid_dep_wait();
  grid_dep_launch();
  const int bh = blockIdx.x;
  const int b = bh / A.H_kv, h = bh % A.H_kv, G = A.H_q / A.H_kv;
  for (int r = threadIdx.x; r < A.gw; r += blockDim.x) {
    const float2 st = combine_partials(A, bh, r);
    const size_t dst = (size_t)(b * A.H_q + h * G) * A.W + r;
    m[dst] = st.x / kLog2e;
    Z[dst] = st.y;
  }
}

template <typename Kern>
cudaError_t launch(Kern kernel, int grid, size_t smem, cudaStream_t st, const ScanArgs& A, const CUtensorMap& qm,
                   const CUtensorMap& km) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if ((e = launch_pdl(kernel, dim3(grid), dim3(kThreads), smem, st, A, qm, km)) != cudaSuccess) return e;
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pass1(const __nv_bfloat16* q, const __nv_bfloat16* k, int B, int H_q, int H_kv, int S, int D,
                         int W, const ScanPlan& pl, int gwp, float* part_m, float* part_z, bool exact_max,
                         cudaStream_t st) {
  (void)gwp;
  ScanArgs A = base_args(pl, B, H_q, H_kv, S, D, W);
  A.nq = 128 * A.n_mb;
  A.part_m = part_m;
  A.part_z = part_z;
  CUtensorMap qm, km;
  if (!make_map(&qm, q, D, (uint64_t)B * H_q * W, 1, A.nq) || !make_map(&km, k, D, S, (uint64_t)B * H_kv, kTile))
    return cudaErrorInvalidValue;
  const size_t smem = pipe_smem(D, A.nq);
  const bool two = A.n_mb == 2;
  if (D == 64) {
    if (exact_max)
      return two ? launch(kvc_tc_pass1_kernel<64, 2, true>, pl.P, smem, st, A, qm, km)
                 : launch(kvc_tc_pass1_kernel<64, 1, true>, pl.P, smem, st, A, qm, km);
    return two ? launch(kvc_tc_pass1_kernel<64, 2, false>, pl.P, smem, st, A, qm, km)
               : launch(kvc_tc_pass1_kernel<64, 1, false>, pl.P, smem, st, A, qm, km);
  }
  if (exact_max)
    return two ? launch(kvc_tc_pass1_kernel<128, 2, true>, pl.P, smem, st, A, qm, km)
               : launch(kvc_tc_pass1_kernel<128, 1, true>, pl.P, smem, st, A, qm, km);
  return two ? launch(kvc_tc_pass1_kernel<128, 2, false>, pl.P, smem, st, A, qm, km)
             : launch(kvc_tc_pass1_kernel<128, 1, false>, pl.P, smem, st, A, qm, km);
}

cudaError_t launch_pass1_combine(const float* part_m, const float* part_z, int B, int H_q, int H_kv, int S, int W,
                                 const ScanPlan& pl, int gwp, float* m, float* Z, cudaStream_t st) {
  (void)gwp;
  ScanArgs A = base_args(pl, B, H_q, H_kv, S, 64, W);
  A.pm_in = part_m;
  A.pz_in = part_z;
  const cudaError_t e = launch_pdl(kvc_pass1_combine_kernel, dim3(B * H_kv), dim3(256), 0, st, A, m, Z);
  if (e != cudaSuccess) return e;
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace kvc
