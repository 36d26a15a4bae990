// Two-pass blockwise scorer (TideKV, Fig. 3) on the 5th-generation tensor
// cores: TMA-staged key tiles, tcgen05 MMA into tensor memory, softmax warps
// reading the accumulators with tcgen05.ld.
//
// Work split.  The flattened key space [B*H_kv][S] is cut into P contiguous
// ranges of L keys, one CTA each (P ~ number of SMs), so every SM gets the
// same number of keys whatever B, H_kv and S are.  A range can cross KV-head
// boundaries; each piece (one head, keys [a, b)) is a "segment".  Pass-1
// partial normalisers and pass-2 candidate lists live in per-(CTA, segment)
// slots whose number depends on P and B*H_kv only, never on S.
//
// Roles (320 threads): warp 0 issues TMA loads (the group's window queries
// once per segment, then 128-key tiles through a 4-stage ring), warp 1 owns
// tensor memory and issues the MMAs from one thread, warps 2..9 are the
// softmax warps.  Tensor memory holds two accumulator buffers of 256 columns,
// so the MMA of tile t+1 runs while tile t is being reduced.
//
// Pass 1 (A = window queries, M = 128 rows per block, B = key tile, N = 128):
//   each softmax thread owns one query row and keeps its running max and
//   sum of 2^(x - max), x = q.k * log2(e)/sqrt(D), over the segment.
// Pass 2 (A = key tile, M = 128 keys, B = window queries, N = G*W rounded to
//   16): each softmax thread owns one key and sums 2^(x - lse2) over its half
//   of the window rows; the halves are added in shared memory, average-pooled
//   with a (pool_k-1)/2 halo recomputed at segment edges, then written as
//   scores or appended to the segment's candidate list.
//
// Every mbarrier wait is bounded; a wait that gives up records a timeout in
// the status word and the CTA drains and returns.
#include <cudaTypedefs.h>

#include <cfloat>
#include <climits>

#include "kvc_device.cuh"
#include "kvc_internal.cuh"
#include "kvc_tc.cuh"

namespace kvc {
namespace {

constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kScanThreads = 64 + kEpiThreads;
constexpr int kStages = 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccStride = 256;          // TMEM columns per accumulator buffer
constexpr uint32_t kWaitLimit = 1u << 22;     // polls before a wait gives up
constexpr float kLog2e = 1.4426950408889634f;

struct ScanArgs {
  int B, H_q, H_kv, S, W, gw, gwp16, n_mb, nq, P, maxseg, pool_k, cap;
  int64_t L;
  float c2;
  float* part_m;             // pass 1 out: [P*maxseg][gwp16] (log2 units)
  float* part_z;
  const float* m_in;         // pass 2: natural-unit m, Z [B][H_q][W] ...
  const float* z_in;
  const float* pm_in;        // ... or pass-1 partials
  const float* pz_in;
  float* scores;             // pass 2 out: dense [BH][S] or nullptr
  uint64_t* cand;            // pass 2 out: [P*maxseg][cap]
  int* cand_cnt;             // [P*maxseg]
  int* status;
};

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;\n" ::"n"(kEpiThreads) : "memory"); }

// Bounded wait; on giving up, flags the CTA and the status word.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status) {
  for (uint32_t i = 0; i < kWaitLimit; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 4095u) == 4095u && *abort_flag) return false;
  }
  *abort_flag = 1;
  record_status(status, kStatusTimeout);
  return false;
}

struct Seg {
  int bh, a, b;
};

// Segments of CTA c in order: returns the count and fills up to `max` of them.
__device__ __forceinline__ int cta_segments(const ScanArgs& A, int c, Seg* out, int max_out) {
  const int64_t total = (int64_t)A.B * A.H_kv * A.S;
  const int64_t f0 = (int64_t)c * A.L;
  const int64_t f1 = min(f0 + A.L, total);
  if (f0 >= f1) return 0;
  const int h0 = (int)(f0 / A.S), h1 = (int)((f1 - 1) / A.S);
  int n = 0;
  for (int h = h0; h <= h1 && n < max_out; ++h, ++n) {
    out[n].bh = h;
    out[n].a = (int)max((int64_t)0, f0 - (int64_t)h * A.S);
    out[n].b = (int)min((int64_t)A.S, f1 - (int64_t)h * A.S);
  }
  return n;
}

__device__ __forceinline__ float2 merge_mz(float2 a, float2 b) {
  if (b.y == 0.f) return a;
  if (a.y == 0.f) return b;
  const float m = fmaxf(a.x, b.x);
  return make_float2(m, a.y * ex2(a.x - m) + b.y * ex2(b.x - m));
}

// lse2 of window row `row` of head bh from the pass-1 partial slots.
__device__ float lse2_from_partials(const ScanArgs& A, int bh, int row) {
  const int64_t S = A.S;
  const int c_first = (int)(((int64_t)bh * S) / A.L);
  const int c_last = (int)((((int64_t)bh + 1) * S - 1) / A.L);
  float2 st = make_float2(-INFINITY, 0.f);
  for (int c = c_first; c <= c_last; ++c) {
    const int seg = bh - (int)(((int64_t)c * A.L) / S);
    const size_t o = ((size_t)c * A.maxseg + seg) * A.gwp16 + row;
    st = merge_mz(st, make_float2(A.pm_in[o], A.pz_in[o]));
  }
  return st.x + log2f(st.y);
}

struct Bars {
  uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], qfull, qempty;
};

// ------------------------------------------------------------- producer
template <int D, int PASS>
__device__ void producer(const ScanArgs& A, const CUtensorMap* qmap, const CUtensorMap* kmap, Bars* bars,
                         uint32_t sQ, uint32_t sK, volatile int* abort_flag) {
  constexpr int NKH = D / 64;
  constexpr uint32_t kTileBytes = kTile * 128 * NKH;
  const uint32_t q_half = (uint32_t)A.nq * 128;
  const uint32_t q_bytes = q_half * NKH;
  const int hw = PASS == 2 ? (A.pool_k - 1) / 2 : 0;
  Seg segs[8];
  const int nseg = cta_segments(A, blockIdx.x, segs, 8);
  const int G = A.H_q / A.H_kv;
  uint32_t stage = 0, phase = 0, qphase = 0;
  int issued = 0;
  for (int s = 0; s < nseg; ++s) {
    const Seg sg = segs[s];
    if (s > 0) {
      if (!wait_bar(smem_u32(&bars->qempty), qphase, abort_flag, A.status)) return;
      qphase ^= 1;
    }
    const int b_idx = sg.bh / A.H_kv, hk = sg.bh % A.H_kv;
    const int qrow = (b_idx * A.H_q + hk * G) * A.W;
    tc::mbar_arrive_expect_tx(smem_u32(&bars->qfull), q_bytes);
    for (int kh = 0; kh < NKH; ++kh)
      tc::tma_load_3d(sQ + kh * q_half, qmap, smem_u32(&bars->qfull), kh * 64, qrow, 0);
    const int start = sg.a - hw;
    const int ntiles = (sg.b - sg.a + 2 * hw + kTile - 1) / kTile;
    for (int t = 0; t < ntiles; ++t) {
      if (!wait_bar(smem_u32(&bars->empty[stage]), phase ^ 1, abort_flag, A.status)) return;
      const uint32_t dst = sK + stage * kTileBytes;
      tc::mbar_arrive_expect_tx(smem_u32(&bars->full[stage]), kTileBytes);
      for (int kh = 0; kh < NKH; ++kh)
        tc::tma_load_3d(dst + kh * (kTile * 128), kmap, smem_u32(&bars->full[stage]), kh * 64, start + t * kTile,
                        sg.bh);
      ++issued;
      if (++stage == kStages) { stage = 0; phase ^= 1; }
    }
  }
  (void)issued;
}

// ------------------------------------------------------------ MMA issuer
template <int D, int PASS>
__device__ void mma_issuer(const ScanArgs& A, Bars* bars, uint32_t sQ, uint32_t sK, uint32_t tmem,
                           volatile int* abort_flag) {
  constexpr int NKH = D / 64;
  constexpr int KSTEPS = D / 16;
  constexpr uint32_t kTileBytes = kTile * 128 * NKH;
  const uint32_t q_half = (uint32_t)A.nq * 128;
  const int hw = PASS == 2 ? (A.pool_k - 1) / 2 : 0;
  Seg segs[8];
  const int nseg = cta_segments(A, blockIdx.x, segs, 8);
  uint32_t stage = 0, phase = 0, qphase = 0, buf = 0, tphase = 0;
  const uint32_t idesc = PASS == 1 ? tc::idesc_bf16(128, 128) : tc::idesc_bf16(128, A.gwp16);
  for (int s = 0; s < nseg; ++s) {
    const Seg sg = segs[s];
    if (!wait_bar(smem_u32(&bars->qfull), qphase, abort_flag, A.status)) return;
    qphase ^= 1;
    const int ntiles = (sg.b - sg.a + 2 * hw + kTile - 1) / kTile;
    for (int t = 0; t < ntiles; ++t) {
      if (!wait_bar(smem_u32(&bars->full[stage]), phase, abort_flag, A.status)) return;
      if (!wait_bar(smem_u32(&bars->tempty[buf]), tphase ^ 1, abort_flag, A.status)) return;
      tc::fence_after_sync();
      const uint32_t kb = sK + stage * kTileBytes;
      const uint32_t dacc = tmem + buf * kAccStride;
      if (PASS == 1) {
        for (int mb = 0; mb < A.n_mb; ++mb) {
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            const uint32_t koff = (ks >> 2) * (kTile * 128) + (ks & 3) * 32;
            const uint32_t qoff = (ks >> 2) * q_half + mb * (128 * 128) + (ks & 3) * 32;
            tc::mma_bf16(dacc + mb * 128, tc::desc_sw128(sQ + qoff), tc::desc_sw128(kb + koff), idesc, ks > 0);
          }
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
          const uint32_t koff = (ks >> 2) * (kTile * 128) + (ks & 3) * 32;
          const uint32_t qoff = (ks >> 2) * q_half + (ks & 3) * 32;
          tc::mma_bf16(dacc, tc::desc_sw128(kb + koff), tc::desc_sw128(sQ + qoff), idesc, ks > 0);
        }
      }
      tc::mma_commit(smem_u32(&bars->empty[stage]));
      tc::mma_commit(smem_u32(&bars->tfull[buf]));
      if (++stage == kStages) { stage = 0; phase ^= 1; }
      if (++buf == 2) { buf = 0; tphase ^= 1; }
    }
    tc::mma_commit(smem_u32(&bars->qempty));
  }
}

// --------------------------------------------------------------- pass 1
template <int D, int NMB>
__global__ void __launch_bounds__(kScanThreads, 1)
kvc_tc_pass1_kernel(const __grid_constant__ ScanArgs A, const __grid_constant__ CUtensorMap qmap,
                    const __grid_constant__ CUtensorMap kmap) {
  constexpr int NKH = D / 64;
  constexpr int NC = NMB == 2 ? 128 : 64;       // accumulator columns per softmax thread
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ float2 s_half[128];

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sK = base + (uint32_t)A.nq * 128 * NKH;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(smem_u32(&bars.full[i]), 1);
      tc::mbar_init(smem_u32(&bars.empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(smem_u32(&bars.tfull[i]), 1);
      tc::mbar_init(smem_u32(&bars.tempty[i]), kEpiWarps);
    }
    tc::mbar_init(smem_u32(&bars.qfull), 1);
    tc::mbar_init(smem_u32(&bars.qempty), 1);
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

  if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&qmap);
      tc::tma_prefetch_desc(&kmap);
      producer<D, 1>(A, &qmap, &kmap, &bars, sQ, sK, &s_abort);
    }
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<D, 1>(A, &bars, sQ, sK, tmem, &s_abort);
  } else {
    // softmax warps
    const int e = warp - 2;
    const int quarter = warp & 3;              // TMEM lanes this warp may read
    const int k = e >> 2;                      // 0 or 1
    const int mb = NMB == 2 ? k : 0;
    const int col0 = NMB == 2 ? 0 : 64 * k;
    const int row = mb * 128 + quarter * 32 + lane;
    const bool active = (mb * 128 + quarter * 32) < A.gw;
    const float c2 = A.c2;
    const int t_row = A.S - A.W + (row % A.W);
    Seg segs[8];
    const int nseg = cta_segments(A, blockIdx.x, segs, 8);
    uint32_t buf = 0, tphase = 0;
    bool ok = true;
    for (int s = 0; s < nseg && ok; ++s) {
      const Seg sg = segs[s];
      float mrun = -INFINITY;
      float2 z2 = make_float2(0.f, 0.f);
      const int ntiles = (sg.b - sg.a + kTile - 1) / kTile;
      for (int t = 0; t < ntiles; ++t) {
        if (!wait_bar(smem_u32(&bars.tfull[buf]), tphase, &s_abort, A.status)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t taddr = tmem + buf * kAccStride + mb * 128 + col0 + ((uint32_t)(quarter * 32) << 16);
        // 64 accumulator columns at a time; the buffer is handed back to the
        // MMA warp right after the last batch has been read
#pragma unroll 1
        for (int bt = 0; bt < NC / 64; ++bt) {
          float v[64];
          if (active) {
#pragma unroll
            for (int c = 0; c < 64; c += 16) tc::tmem_ld16(taddr + bt * 64 + c, v + c);
            tc::tmem_wait_ld();
            tc::reg_fence(v, 64);
          }
          if (bt == NC / 64 - 1) {
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(smem_u32(&bars.tempty[buf]));
          }
          if (!active) continue;
          const int t0 = sg.a + t * kTile + col0 + bt * 64;
          if (t0 + 63 >= sg.b || t0 + 63 > A.S - A.W) {
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const int j = t0 + c;
              if (j >= sg.b || j > t_row) v[c] = -INFINITY;
            }
          }
          float mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < 64; c += 2) mx = fmaxf(mx, fmaxf(v[c], v[c + 1]));
          if (mx > mrun) {
            const float sc = (mrun == -INFINITY) ? 0.f : ex2((mrun - mx) * c2);
            z2.x *= sc;
            z2.y *= sc;
            mrun = mx;
          }
          if (mrun > -INFINITY) {
            const float nm = -mrun * c2;
            const float2 cc = make_float2(c2, c2), nn = make_float2(nm, nm);
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
              const float2 x = __ffma2_rn(make_float2(v[c], v[c + 1]), cc, nn);
              acc = __fadd2_rn(acc, make_float2(ex2(x.x), ex2(x.y)));
            }
            z2 = __fadd2_rn(z2, acc);
          }
        }
        if (++buf == 2) { buf = 0; tphase ^= 1; }
      }
      if (!ok) break;
      // segment done: the two column halves of a row (NMB == 1) are merged
      const float2 mine = make_float2(mrun == -INFINITY ? -INFINITY : mrun * c2, z2.x + z2.y);
      const size_t slot = (size_t)blockIdx.x * A.maxseg + (size_t)(sg.bh - segs[0].bh);
      if (NMB == 2) {
        if (row < A.gwp16) {
          A.part_m[slot * A.gwp16 + row] = mine.x;
          A.part_z[slot * A.gwp16 + row] = mine.y;
        }
      } else {
        if (k == 1) s_half[quarter * 32 + lane] = mine;
        epi_sync();
        if (k == 0 && row < A.gwp16) {
          const float2 st = merge_mz(mine, s_half[quarter * 32 + lane]);
          A.part_m[slot * A.gwp16 + row] = st.x;
          A.part_z[slot * A.gwp16 + row] = st.y;
        }
        epi_sync();
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

// ----------------------------------------------------- candidate lists
__device__ __forceinline__ uint64_t rank_key(uint64_t e) {
  return (e & 0xFFFFFFFF00000000ull) | (uint64_t)(~(uint32_t)e);
}

struct CompactSmem {
  int hist[256];
  int scan[32];
  int need, full;
  unsigned long long prefix;
};

// Inclusive scan over the softmax threads (etid in [0, kEpiThreads)).
__device__ __forceinline__ int epi_scan(int v, int etid, int* scratch, int* total) {
  const int lane = etid & 31, w = etid >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) scratch[w] = v;
  epi_sync();
  int before = 0, tot = 0;
#pragma unroll
  for (int i = 0; i < kEpiWarps; ++i) {
    before += i < w ? scratch[i] : 0;
    tot += scratch[i];
  }
  epi_sync();
  *total = tot;
  return v + before;
}

// Keep the n_keep best entries of buf[0..cnt) in place (order kept) and
// return, through s_tau, the score bits a later (higher-index) key must beat.
__device__ void epi_compact(uint64_t* buf, int cnt, int n_keep, int etid, CompactSmem* cs, int* s_cnt,
                            long long* s_tau, int* status) {
  if (n_keep <= 0) {
    if (etid == 0) { *s_cnt = 0; *s_tau = LLONG_MAX; }
    epi_sync();
    return;
  }
  unsigned long long prefix = 0;
  int need = n_keep;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = etid; i < 256; i += kEpiThreads) cs->hist[i] = 0;
    epi_sync();
    for (int i = etid; i < cnt; i += kEpiThreads) {
      const uint64_t key = rank_key(buf[i]);
      if (shift == 56 || (key >> (shift + 8)) == (prefix >> (shift + 8))) atomicAdd(&cs->hist[(key >> shift) & 255], 1);
    }
    epi_sync();
    if (etid == 0) {
      int cum = 0, d = 255;
      for (; d > 0; --d) {
        if (cum + cs->hist[d] >= need) break;
        cum += cs->hist[d];
      }
      cs->need = need - cum;
      cs->full = (need - cum == cs->hist[d]);
      cs->prefix = prefix | ((unsigned long long)d << shift);
    }
    epi_sync();
    need = cs->need;
    prefix = cs->prefix;
    const int full = cs->full;
    epi_sync();
    if (full) break;
  }
  const uint64_t T = prefix;
  int out = 0;
  for (int b0 = 0; b0 < cnt; b0 += kEpiThreads) {
    const int i = b0 + etid;
    const uint64_t e = i < cnt ? buf[i] : 0ull;
    const int f = (i < cnt && rank_key(e) >= T) ? 1 : 0;
    int tot;
    const int incl = epi_scan(f, etid, cs->scan, &tot);
    if (f) buf[out + incl - 1] = e;
    out += tot;
    epi_sync();
  }
  if (etid == 0) {
    if (out != n_keep) record_status(status, kStatusCandOverflow);
    *s_cnt = out;
    *s_tau = (long long)(T >> 32);
  }
  epi_sync();
}

// --------------------------------------------------------------- pass 2
template <int D, bool CAND>
__global__ void __launch_bounds__(kScanThreads, 1)
kvc_tc_pass2_kernel(const __grid_constant__ ScanArgs A, const __grid_constant__ SelParams sel,
                    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap) {
  constexpr int NKH = D / 64;
  extern __shared__ uint8_t smem_raw[];
  __shared__ Bars bars;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ __align__(16) float s_nlse[kMaxGWP];
  __shared__ float s_rhalf[2][kTile];
  __shared__ float s_rbuf[2 * 7 + kTile];
  __shared__ int s_wtot[kEpiWarps];
  __shared__ int s_cnt;
  __shared__ long long s_tau;
  __shared__ CompactSmem cs;

  const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t sQ = base;
  const uint32_t sK = base + (uint32_t)A.nq * 128 * NKH;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      tc::mbar_init(smem_u32(&bars.full[i]), 1);
      tc::mbar_init(smem_u32(&bars.empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(smem_u32(&bars.tfull[i]), 1);
      tc::mbar_init(smem_u32(&bars.tempty[i]), kEpiWarps);
    }
    tc::mbar_init(smem_u32(&bars.qfull), 1);
    tc::mbar_init(smem_u32(&bars.qempty), 1);
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

  if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&qmap);
      tc::tma_prefetch_desc(&kmap);
      producer<D, 2>(A, &qmap, &kmap, &bars, sQ, sK, &s_abort);
    }
  } else if (warp == 1) {
    if (lane == 0) mma_issuer<D, 2>(A, &bars, sQ, sK, tmem, &s_abort);
  } else {
    const int etid = threadIdx.x - 64;
    const int e = warp - 2;
    const int quarter = warp & 3;
    const int k = e >> 2;
    const int krow = quarter * 32 + lane;          // key row of the tile this thread reduces
    const int nch = A.gwp16 / 16;                  // 16-column chunks
    const int ch_lo = k == 0 ? 0 : (nch + 1) / 2;
    const int ch_hi = k == 0 ? (nch + 1) / 2 : nch;
    const int hw = (A.pool_k - 1) / 2;
    const float c2 = A.c2;
    const float inv_pool = 1.0f / (float)A.pool_k;
    float* rtile = s_rbuf + 2 * hw;
    Seg segs[8];
    const int nseg = cta_segments(A, blockIdx.x, segs, 8);
    uint32_t buf = 0, tphase = 0;
    bool ok = true;
    for (int s = 0; s < nseg && ok; ++s) {
      const Seg sg = segs[s];
      const int b_idx = sg.bh / A.H_kv, hk = sg.bh % A.H_kv;
      const int G = A.H_q / A.H_kv;
      // negated lse2 of every window row of this head (padding rows: -inf weight)
      for (int r = etid; r < A.gwp16; r += kEpiThreads) {
        float l = INFINITY;
        if (r < A.gw) {
          if (A.m_in != nullptr) {
            const size_t src = (size_t)(b_idx * A.H_q + hk * G) * A.W + r;
            l = A.m_in[src] * kLog2e + log2f(A.z_in[src]);
          } else {
            l = lse2_from_partials(A, sg.bh, r);
          }
        }
        s_nlse[r] = -l;
      }
      for (int i = etid; i < 2 * hw; i += kEpiThreads) s_rbuf[i] = 0.f;
      if (etid == 0) { s_cnt = 0; s_tau = -1; }
      epi_sync();
      const size_t slot = (size_t)blockIdx.x * A.maxseg + (size_t)(sg.bh - segs[0].bh);
      uint64_t* my_cand = CAND ? A.cand + slot * A.cap : nullptr;
      const int n_keep = CAND ? sel.n_sel[hk] : 0;
      const int n_iter = (sg.b - sg.a + 2 * hw + kTile - 1) / kTile;
      for (int it = 0; it < n_iter; ++it) {
        const int t0 = sg.a - hw + it * kTile;
        if (!wait_bar(smem_u32(&bars.tfull[buf]), tphase, &s_abort, A.status)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t taddr = tmem + buf * kAccStride + ((uint32_t)(quarter * 32) << 16);
        const int j = t0 + krow;
        const bool need_mask = (t0 + kTile - 1 > A.S - A.W);
        float2 acc = make_float2(0.f, 0.f);
        const float2 cc = make_float2(c2, c2);
        // four 16-column chunks (64 columns) at a time; the buffer goes back to
        // the MMA warp once this warp's last chunk is in registers
        const int nbt = (ch_hi - ch_lo + 3) / 4;
#pragma unroll 1
        for (int bt = 0; bt < max(nbt, 1); ++bt) {
          float v[64];
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (ch_lo + 4 * bt + i < ch_hi) tc::tmem_ld16(taddr + (ch_lo + 4 * bt + i) * 16, v + 16 * i);
          tc::tmem_wait_ld();
          tc::reg_fence(v, 64);
          if (bt == max(nbt, 1) - 1) {
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(smem_u32(&bars.tempty[buf]));
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (ch_lo + 4 * bt + i < ch_hi) {
              const int cb = (ch_lo + 4 * bt + i) * 16;
#pragma unroll
              for (int q4 = 0; q4 < 16; q4 += 4) {
                const float4 nl = *reinterpret_cast<const float4*>(&s_nlse[cb + q4]);
                float2 x0 = __ffma2_rn(make_float2(v[16 * i + q4], v[16 * i + q4 + 1]), cc, make_float2(nl.x, nl.y));
                float2 x1 =
                    __ffma2_rn(make_float2(v[16 * i + q4 + 2], v[16 * i + q4 + 3]), cc, make_float2(nl.z, nl.w));
                if (need_mask) {
                  const int tb = A.S - A.W;
                  if (j > tb + ((cb + q4) % A.W)) x0.x = -INFINITY;
                  if (j > tb + ((cb + q4 + 1) % A.W)) x0.y = -INFINITY;
                  if (j > tb + ((cb + q4 + 2) % A.W)) x1.x = -INFINITY;
                  if (j > tb + ((cb + q4 + 3) % A.W)) x1.y = -INFINITY;
                }
                acc = __fadd2_rn(acc, make_float2(ex2(x0.x), ex2(x0.y)));
                acc = __fadd2_rn(acc, make_float2(ex2(x1.x), ex2(x1.y)));
              }
            }
          }
        }
        if (++buf == 2) { buf = 0; tphase ^= 1; }
        s_rhalf[k][krow] = acc.x + acc.y;
        epi_sync();
        if (k == 0) rtile[krow] = (j >= 0 && j < A.S) ? s_rhalf[0][krow] + s_rhalf[1][krow] : 0.f;
        epi_sync();

        // pooled scores of keys t0 - hw + etid (etid < 128)
        const int jo = t0 - hw + etid;
        const bool valid = etid < kTile && jo >= sg.a && jo < sg.b;
        float sc = 0.f;
        if (etid < kTile) {
          for (int d = 0; d <= 2 * hw; ++d) sc += s_rbuf[etid + d];
          sc = (A.pool_k == 1) ? sc : sc * inv_pool;
        }
        if (!CAND) {
          if (valid) A.scores[(size_t)sg.bh * A.S + jo] = sc;
        } else {
          uint32_t u = __float_as_uint(sc);
          if (u == 0x80000000u) u = 0u;
          const bool is_cand = valid && jo >= sel.r_lo && jo < sel.r_hi;
          for (int tries = 0;; ++tries) {
            const bool flag = is_cand && (long long)u > s_tau;
            const unsigned bal = __ballot_sync(0xffffffffu, flag);
            if (lane == 0) s_wtot[e] = __popc(bal);
            epi_sync();
            int tot = 0, before = 0;
#pragma unroll
            for (int w = 0; w < kEpiWarps; ++w) {
              before += (w < e) ? s_wtot[w] : 0;
              tot += s_wtot[w];
            }
            const int cnt0 = s_cnt;
            if (cnt0 + tot > A.cap) {
              if (cnt0 <= n_keep || tries >= 2) {
                if (etid == 0) record_status(A.status, kStatusCandOverflow);
                epi_sync();
                break;
              }
              epi_sync();
              epi_compact(my_cand, cnt0, n_keep, etid, &cs, &s_cnt, &s_tau, A.status);
              continue;
            }
            if (flag) my_cand[cnt0 + before + __popc(bal & ((1u << lane) - 1u))] = ((uint64_t)u << 32) | (uint32_t)jo;
            epi_sync();
            if (etid == 0) s_cnt = cnt0 + tot;
            break;
          }
        }
        epi_sync();
        if (etid < 2 * hw) s_rbuf[etid] = rtile[kTile - 2 * hw + etid];
        epi_sync();
      }
      if (CAND && ok && etid == 0) A.cand_cnt[slot] = s_cnt;
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
  const int bh = blockIdx.x;
  const int b = bh / A.H_kv, h = bh % A.H_kv, G = A.H_q / A.H_kv;
  const int64_t S = A.S;
  const int c_first = (int)(((int64_t)bh * S) / A.L);
  const int c_last = (int)((((int64_t)bh + 1) * S - 1) / A.L);
  for (int r = threadIdx.x; r < A.gw; r += blockDim.x) {
    float2 st = make_float2(-INFINITY, 0.f);
    for (int c = c_first; c <= c_last; ++c) {
      const int seg = bh - (int)(((int64_t)c * A.L) / S);
      const size_t o = ((size_t)c * A.maxseg + seg) * A.gwp16 + r;
      st = merge_mz(st, make_float2(A.pm_in[o], A.pz_in[o]));
    }
    const size_t dst = (size_t)(b * A.H_q + h * G) * A.W + r;
    m[dst] = st.x / kLog2e;
    Z[dst] = st.y;
  }
}

// ------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D map over a [d2][d1][d0] bf16 tensor with 128-byte swizzled 64 x box1 boxes.
bool make_map(CUtensorMap* map, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box1) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {64, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

size_t scan_smem(int D, int nq) { return 1024 + (size_t)nq * 128 * (D / 64) + (size_t)kStages * kTile * 128 * (D / 64); }

template <typename K>
cudaError_t launch(K kernel, int grid, size_t smem, cudaStream_t st, const ScanArgs& A, const CUtensorMap& qm,
                   const CUtensorMap& km) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kScanThreads, smem, st>>>(A, qm, km);
  note_launches(1);
  return cudaGetLastError();
}

template <typename K>
cudaError_t launch2(K kernel, int grid, size_t smem, cudaStream_t st, const ScanArgs& A, const SelParams& sp,
                    const CUtensorMap& qm, const CUtensorMap& km) {
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kScanThreads, smem, st>>>(A, sp, qm, km);
  note_launches(1);
  return cudaGetLastError();
}

ScanArgs base_args(const ScanPlan& pl, int B, int H_q, int H_kv, int S, int D, int W) {
  ScanArgs A{};
  A.B = B;
  A.H_q = H_q;
  A.H_kv = H_kv;
  A.S = S;
  A.W = W;
  A.gw = (H_q / H_kv) * W;
  A.gwp16 = (A.gw + 15) / 16 * 16;
  A.n_mb = A.gw > 128 ? 2 : 1;
  A.P = pl.P;
  A.L = pl.L;
  A.maxseg = pl.maxseg;
  A.c2 = 1.4426950408889634f / sqrtf((float)D);
  A.status = status_word_ptr();
  A.pool_k = 1;
  return A;
}

}  // namespace

cudaError_t launch_pass1(const __nv_bfloat16* q, const __nv_bfloat16* k, int B, int H_q, int H_kv, int S, int D,
                         int W, const ScanPlan& pl, int gwp, float* part_m, float* part_z, cudaStream_t st) {
  (void)gwp;
  ScanArgs A = base_args(pl, B, H_q, H_kv, S, D, W);
  A.nq = 128 * A.n_mb;
  A.part_m = part_m;
  A.part_z = part_z;
  CUtensorMap qm, km;
  if (!make_map(&qm, q, D, (uint64_t)B * H_q * W, 1, A.nq) || !make_map(&km, k, D, S, (uint64_t)B * H_kv, kTile))
    return cudaErrorInvalidValue;
  const size_t smem = scan_smem(D, A.nq);
  if (D == 64)
    return A.n_mb == 2 ? launch(kvc_tc_pass1_kernel<64, 2>, pl.P, smem, st, A, qm, km)
                       : launch(kvc_tc_pass1_kernel<64, 1>, pl.P, smem, st, A, qm, km);
  return A.n_mb == 2 ? launch(kvc_tc_pass1_kernel<128, 2>, pl.P, smem, st, A, qm, km)
                     : launch(kvc_tc_pass1_kernel<128, 1>, pl.P, smem, st, A, qm, km);
}

cudaError_t launch_pass1_combine(const float* part_m, const float* part_z, int B, int H_q, int H_kv, int S,
                                 int W, const ScanPlan& pl, int gwp, float* m, float* Z, cudaStream_t st) {
  (void)gwp;
  ScanArgs A = base_args(pl, B, H_q, H_kv, S, 64, W);
  A.pm_in = part_m;
  A.pz_in = part_z;
  kvc_pass1_combine_kernel<<<B * H_kv, 256, 0, st>>>(A, m, Z);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_pass2(const __nv_bfloat16* q, const __nv_bfloat16* k, const float* m, const float* Z,
                         const float* part_m, const float* part_z, int B, int H_q, int H_kv, int S, int D, int W,
                         int pool_k, const ScanPlan& pl, int gwp, const SelParams* sel, Pass2Out out,
                         cudaStream_t st) {
  (void)gwp;
  ScanArgs A = base_args(pl, B, H_q, H_kv, S, D, W);
  A.nq = A.gwp16;
  A.pool_k = pool_k;
  A.m_in = m;
  A.z_in = Z;
  A.pm_in = part_m;
  A.pz_in = part_z;
  A.scores = out.scores;
  A.cand = out.cand;
  A.cand_cnt = out.cand_cnt;
  A.cap = out.cap;
  CUtensorMap qm, km;
  if (!make_map(&qm, q, D, (uint64_t)B * H_q * W, 1, A.nq) || !make_map(&km, k, D, S, (uint64_t)B * H_kv, kTile))
    return cudaErrorInvalidValue;
  const size_t smem = scan_smem(D, A.nq);
  const bool cand = out.cand != nullptr;
  if (D == 64)
    return cand ? launch2(kvc_tc_pass2_kernel<64, true>, pl.P, smem, st, A, *sel, qm, km)
                : launch2(kvc_tc_pass2_kernel<64, false>, pl.P, smem, st, A, *sel, qm, km);
  return cand ? launch2(kvc_tc_pass2_kernel<128, true>, pl.P, smem, st, A, *sel, qm, km)
              : launch2(kvc_tc_pass2_kernel<128, false>, pl.P, smem, st, A, *sel, qm, km);
}

}  // namespace kvc
