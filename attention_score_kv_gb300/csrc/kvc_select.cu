// Per-head top-k selection and gather (TideKV, Fig. 2 and Fig. 3).
//
// Selection keeps, per (b, KV head), the mandatory set R_mand = [0, sink) u
// [S - recent, S) and the n_sel best other keys by (score desc, index asc),
// listed in ascending position.  Scores become 32-bit keys that order like
// the values (the fused scorer's scores are >= 0 and keep their fp32 bits;
// dense scores of either sign are mapped by flipping the sign bit of
// positive values and all bits of negative ones); a three-round radix select
// over those bits (11, 11 and 10 bits, each round a histogram of the keys
// that share the digits found so far) finds the n_sel-th score T and how many
// keys scoring exactly T are still needed.  Ties at T are taken in ascending
// index order, resolved with per-warp counts and an ordered ballot write.
// All of it runs in one launch with one thread-block cluster per head.
//
// The keys come either from a dense score array (mode 0) or from the
// per-range candidate lists of the fused scorer (mode 1, entries
// (score bits << 32 | index), ascending index within each range, ranges in
// ascending key order).
#include <algorithm>

#include "kvc_device.cuh"
#include "kvc_internal.cuh"

namespace kvc {
namespace {

struct SegView {
  int mode;
  const float* scores;     // mode 0: [BH][S]
  const uint64_t* cand;    // mode 1: [slots][cap]
  const int* cand_cnt;     // mode 1: [slots]
  int cap;
};

// Candidate slot of range `part` of head `seg` (mode 1), or -1 past the last
// scan CTA that touches the head.  Scan CTA c_first holds the head's first
// key (and may start in an earlier head); every later CTA that touches the
// head starts inside it, so its slot is that CTA's first one.
__device__ __forceinline__ int64_t cand_slot(const SelParams& sp, int seg, int part) {
  const int64_t S = sp.S;
  const int64_t c_first = range_of((int64_t)seg * S, sp.L, S, sp.total);
  const int64_t c_last = range_of(((int64_t)seg + 1) * S - 1, sp.L, S, sp.total);
  const int64_t c = c_first + part;
  if (c > c_last) return -1;
  if (part > 0) return c * sp.maxseg;
  return c * sp.maxseg + (seg - range_begin(c, sp.L, S, sp.total) / S);
}

// One thread-block cluster per (b, KV head).  The head's entries are cut
// into kCl contiguous shares, one per CTA, and each share is copied once
// into that CTA's shared memory (up to stage_cap entries; the rest, if any, is
// re-read from global memory in every round).  The radix rounds, the counts
// and the ordered write then run on chip: per-CTA histograms (plain
// shared-memory atomics) are summed by reading the other CTAs' shared
// memory, and hardware cluster barriers separate the phases, so no CTA waits
// on anything outside its cluster.  After the first round each CTA keeps
// only the keys that share its digit (when they fit), so the later rounds
// histogram those alone.
constexpr int kMaxCl = 16;              // CTAs per head at most (a non-portable cluster size)
constexpr int kClThreads = 1024;
constexpr int kClWarps = kClThreads / 32;
static_assert(kClWarps <= 32, "one warp holds the per-warp counts");
constexpr int kStageC = 16384;          // entries per CTA kept in shared memory (clusters of <= 8)
constexpr int kStageC16 = 8192;         // ... in clusters of 16, two CTAs per SM
constexpr int kCopyBatch = 8;

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ uint4 ld_dsmem_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];\n" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

struct __align__(16) ClSmem {
  uint32_t hist[kHist1 + kHist2 + kHist3];   // this CTA's histogram of each round
  uint32_t red[kHist1 + kHist2 + kHist3];    // cluster sums of the bins this CTA owns
  int scan[32];
  int digit, need;
  int wgt[kClWarps], weq[kClWarps], wout[kClWarps], weqb[kClWarps];
  int nsurv, surv_fill;                      // keys that share the round-0 digit; survivors placed
  int cta_gt, cta_eq;                        // this CTA's keys above / at the threshold
};

// The head's entries in key order: mode 0 the dense scores of the
// non-mandatory keys, mode 1 the concatenated candidate lists of its key
// ranges (pref = exclusive prefix of the list lengths).
struct HeadView {
  const SegView* v;
  const SelParams* sp;
  int seg;
  const int* pref;
  const int64_t* slot_of;   // mode 1: candidate slot of each part (-1: none)
  int nparts;
  int stage_cap;   // entries of the share held in shared memory
};

__device__ __forceinline__ uint64_t head_entry(const HeadView& hv, int f) {
  if (hv.v->mode == 0) {
    const int j = hv.sp->r_lo + f;
    uint32_t bits = __float_as_uint(hv.v->scores[(size_t)hv.seg * hv.sp->S + j]);
    bits = (bits == 0x80000000u) ? 0u : bits;                      // -0 ranks as +0
    bits = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);    // order-preserving for either sign
    return ((uint64_t)bits << 32) | (uint32_t)j;
  }
  int lo = 0, hi = hv.nparts - 1;   // last part whose list starts at or before f
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (hv.pref[mid] <= f) lo = mid; else hi = mid - 1;
  }
  return hv.v->cand[(size_t)hv.slot_of[lo] * hv.v->cap + (f - hv.pref[lo])];
}

// Entry f0 + i of this CTA's share (n entries).
__device__ __forceinline__ uint64_t share_entry(const HeadView& hv, const uint64_t* stage, int f0, int n, int i) {
  return (n <= hv.stage_cap || i < hv.stage_cap) ? stage[i] : head_entry(hv, f0 + i);
}

__device__ __forceinline__ int radix_bin(uint32_t u, int round, uint32_t prefix) {
  if (round == 0) return (int)(u >> 21);
  if (round == 1) return (u >> 21) == prefix ? (int)((u >> 10) & 2047u) : -1;
  return (u >> 10) == prefix ? (int)(u & 1023u) : -1;
}

// This CTA's histogram of round `round` over its share.
__device__ void cl_hist(const HeadView& hv, const uint64_t* stage, int f0, int n, int round, uint32_t prefix,
                        uint32_t* h) {
  for (int i0 = 0; i0 < n; i0 += kClThreads) {
    const int i = i0 + threadIdx.x;
    int bin = -1;
    if (i < n) bin = radix_bin((uint32_t)(share_entry(hv, stage, f0, n, i) >> 32), round, prefix);
    if (bin >= 0) atomicAdd(&h[bin], 1u);
  }
}

// This CTA's histogram of round `round` over the survivors of round 0 (their
// score bits, in any order).
__device__ void cl_hist_surv(const uint32_t* surv, int ns, int round, uint32_t prefix, uint32_t* h) {
  for (int i0 = 0; i0 < ns; i0 += kClThreads) {
    const int i = i0 + threadIdx.x;
    const int bin = i < ns ? radix_bin(surv[i], round, prefix) : -1;
    if (bin >= 0) atomicAdd(&h[bin], 1u);
  }
}

// After round 0: the score bits of this CTA's keys whose top 11 bits equal
// d0 are copied, in no particular order, into surv (the round-0 histogram,
// which no CTA reads any more), when they fit; returns their number (this
// CTA's round-0 count of d0), or -1 when they do not fit and the later rounds
// scan the whole share.  Each warp claims room for its survivors with one
// shared-memory atomic per 32 entries.
__device__ int cl_survivors(const HeadView& hv, const uint64_t* stage, int f0, int n, uint32_t d0, ClSmem* cs,
                            uint32_t* surv, int cap) {
  if (threadIdx.x == 0) {
    cs->nsurv = (int)surv[d0];
    cs->surv_fill = 0;
  }
  __syncthreads();
  const int total = cs->nsurv;
  if (total > cap) return -1;
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int i0 = 0; i0 < n; i0 += kClThreads) {
    const int i = i0 + threadIdx.x;
    const uint32_t u = i < n ? (uint32_t)(share_entry(hv, stage, f0, n, i) >> 32) : 0u;
    const bool keep = i < n && (u >> 21) == d0;
    const unsigned b = __ballot_sync(0xffffffffu, keep);
    int base = 0;
    if (lane == 0 && b != 0u) base = atomicAdd(&cs->surv_fill, __popc(b));
    base = __shfl_sync(0xffffffffu, base, 0);
    const int at = base + __popc(b & lt);
    if (keep && at < cap) surv[at] = u;
  }
  __syncthreads();
  return total;
}

// Sum round `round`'s histograms over the cluster and find the digit that
// holds the need-th largest key and how many keys of that digit are needed.
// CTA r owns bin slice r: it adds that slice over the cluster (16-byte
// remote loads) into its `red` array; after a cluster barrier every CTA
// reads the summed histogram from the owners and scans it.
template <int kCl>
__device__ void cl_resolve(ClSmem* cs, int round, int need, int* digit, int* need_out) {
  const int nbins = round == 2 ? kHist3 : kHist1;
  const int base = round == 0 ? 0 : round == 1 ? kHist1 : kHist1 + kHist2;
  const int slice = nbins / kCl;                // a multiple of 4
  const uint32_t rank = cluster_rank();
  for (int q = threadIdx.x; q < slice / 4; q += kClThreads) {
    const int bin = base + (int)rank * slice + 4 * q;
    uint4 t[kCl];
#pragma unroll
    for (int r = 0; r < kCl; ++r) t[r] = ld_dsmem_v4(dsmem_addr(&cs->hist[bin], (uint32_t)r));
    uint4 acc = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int r = 0; r < kCl; ++r) {
      acc.x += t[r].x;
      acc.y += t[r].y;
      acc.z += t[r].z;
      acc.w += t[r].w;
    }
    *reinterpret_cast<uint4*>(&cs->red[bin]) = acc;
  }
  cluster_sync_all();
  // thread t holds bins b0 .. b0+3, b0 = nbins - 4(t+1): highest digits first
  const int b0 = nbins - 4 * ((int)threadIdx.x + 1);
  uint32_t c[4] = {0u, 0u, 0u, 0u};
  if (b0 >= 0) {
    const uint4 t = ld_dsmem_v4(dsmem_addr(&cs->red[base + b0], (uint32_t)(b0 / slice)));
    c[0] = t.w;
    c[1] = t.z;
    c[2] = t.y;
    c[3] = t.x;
  }
  const int hi = b0 + 3;
  const int local = (int)(c[0] + c[1] + c[2] + c[3]);
  if (threadIdx.x == 0) { cs->digit = 0; cs->need = 0; }
  int tot;
  const int incl = block_inclusive_scan(local, cs->scan, &tot);
  const int before = incl - local;
  if (b0 >= 0 && before < need && need <= incl) {
    int cum = before;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (cum < need && cum + (int)c[i] >= need) {
        cs->digit = hi - i;
        cs->need = need - cum;
      }
      cum += (int)c[i];
    }
  }
  __syncthreads();
  *digit = cs->digit;
  *need_out = cs->need;
  __syncthreads();
}

template <int kCl>
__global__ void __launch_bounds__(kClThreads, 1)
kvc_select_kernel(SegView v, const __grid_constant__ SelParams sp, int stage_cap, int32_t* __restrict__ idx,
                  int* status) {
  extern __shared__ __align__(16) uint8_t cl_dyn[];
  uint64_t* stage = reinterpret_cast<uint64_t*>(cl_dyn);
  int64_t* slot_of = reinterpret_cast<int64_t*>(cl_dyn + (size_t)stage_cap * sizeof(uint64_t));
  int* pref = reinterpret_cast<int*>(slot_of + (v.mode == 0 ? 0 : sp.nparts));
  __shared__ ClSmem cs;
  const int seg = blockIdx.x / kCl;
  const int rank = (int)cluster_rank();
  const int b = seg / sp.H_kv, h = seg % sp.H_kv;
  const int n_sel = sp.n_sel[h];
  const int nparts = v.mode == 0 ? 1 : sp.nparts;

  for (int i = threadIdx.x; i < kHist1 + kHist2 + kHist3; i += kClThreads) cs.hist[i] = 0u;
  // each part's candidate slot (64-bit divisions) needs nothing the previous
  // grid writes: worked out while it finishes; thread p reads it back below
  if (v.mode != 0)
    for (int p = threadIdx.x; p < nparts; p += kClThreads) slot_of[p] = cand_slot(sp, seg, p);
  grid_dep_wait();   // the scores or candidate lists come from the previous grid
  grid_dep_launch();
  // list lengths and their exclusive prefix (mode 1), else the dense range
  int E;
  if (v.mode == 0) {
    E = sp.r_hi - sp.r_lo;
    if (threadIdx.x == 0) pref[0] = 0;
  } else {
    int carry = 0;
    for (int p0 = 0; p0 < nparts; p0 += kClThreads) {
      const int p = p0 + threadIdx.x;
      int len = 0;
      if (p < nparts) {
        const int64_t slot = slot_of[p];
        len = slot < 0 ? 0 : min(max(v.cand_cnt[slot], 0), v.cap);
      }
      int tot;
      const int incl = block_inclusive_scan(len, cs.scan, &tot);
      if (p < nparts) pref[p] = carry + incl - len;
      carry += tot;
    }
    E = carry;
  }
  __syncthreads();
  HeadView hv{&v, &sp, seg, pref, slot_of, nparts, stage_cap};
  const int f0 = (int)((int64_t)E * rank / kCl), f1 = (int)((int64_t)E * (rank + 1) / kCl);
  const int n = f1 - f0;
  const int mode = n_sel <= 0 ? 0 : n_sel >= E ? 2 : 1;
  // when the whole share fits in shared memory, the first radix round's
  // histogram is taken as the entries arrive, not in a pass of its own
  const bool hist0_in_copy = mode == 1 && n <= stage_cap;

  // copy this CTA's share into shared memory, list by list
  if (mode != 0) {
    const int ns = min(n, stage_cap);
    if (v.mode == 0) {
      for (int i0 = 0; i0 < ns; i0 += kCopyBatch * kClThreads) {
        uint64_t t[kCopyBatch];
#pragma unroll
        for (int q = 0; q < kCopyBatch; ++q) {
          const int i = i0 + q * kClThreads + threadIdx.x;
          t[q] = i < ns ? head_entry(hv, f0 + i) : 0ull;
        }
#pragma unroll
        for (int q = 0; q < kCopyBatch; ++q) {
          const int i = i0 + q * kClThreads + threadIdx.x;
          if (i < ns) {
            stage[i] = t[q];
            if (hist0_in_copy) atomicAdd(&cs.hist[(uint32_t)(t[q] >> 53)], 1u);
          }
        }
      }
    } else {
      for (int p = 0; p < nparts; ++p) {
        const int a = max(f0, pref[p]);
        const int e = min(f0 + ns, p + 1 < nparts ? pref[p + 1] : E);
        if (a >= e) continue;
        const uint64_t* src = v.cand + (size_t)slot_of[p] * v.cap - pref[p];
        // kCopyBatch independent loads in flight per thread
        for (int f = a + threadIdx.x; f < e; f += kCopyBatch * kClThreads) {
          uint64_t t[kCopyBatch];
#pragma unroll
          for (int q = 0; q < kCopyBatch; ++q) {
            const int ff = f + q * kClThreads;
            // written by the previous grid: a load through L2, not the
            // read-only path
            t[q] = ff < e ? __ldcg(reinterpret_cast<const unsigned long long*>(src + ff)) : 0ull;
          }
#pragma unroll
          for (int q = 0; q < kCopyBatch; ++q) {
            const int ff = f + q * kClThreads;
            if (ff < e) {
              stage[ff - f0] = t[q];
              if (hist0_in_copy) atomicAdd(&cs.hist[(uint32_t)(t[q] >> 53)], 1u);
            }
          }
        }
      }
    }
  }
  __syncthreads();

  // radix rounds: T = the n_sel-th largest score bits, need_eq = ties at T to take
  uint32_t T = 0u;
  int need_eq = 0;
  if (mode == 1) {
    uint32_t prefix = 0u;
    int need = n_sel;
    int ns = -1;   // survivors of round 0 held in cs.hist[0 .. kHist1), or -1: scan the share
    for (int round = 0; round < 3; ++round) {
      uint32_t* hr = cs.hist + (round == 0 ? 0 : round == 1 ? kHist1 : kHist1 + kHist2);
      if (round == 1) ns = cl_survivors(hv, stage, f0, n, prefix, &cs, cs.hist, kHist1);
      if (round > 0 && ns >= 0)
        cl_hist_surv(cs.hist, ns, round, prefix, hr);
      else if (round > 0 || !hist0_in_copy)
        cl_hist(hv, stage, f0, n, round, prefix, hr);
      cluster_sync_all();
      int d, nd;
      cl_resolve<kCl>(&cs, round, need, &d, &nd);
      prefix = round == 0 ? (uint32_t)d : (prefix << (round == 1 ? 11 : 10)) | (uint32_t)d;
      need = nd;
    }
    T = prefix;
    need_eq = need;
  }

  // per-warp counts over contiguous stretches of the share, then the CTA's
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int chunk = (n + kClWarps - 1) / kClWarps;
  const int lo = min(n, w * chunk), hi = min(n, lo + chunk);
  int gtw = 0, eqw = 0;
  if (mode == 2) {
    gtw = lane == 0 ? hi - lo : 0;
  } else if (mode == 1) {
    for (int i = lo + lane; i < hi; i += 32) {
      const uint32_t u = (uint32_t)(share_entry(hv, stage, f0, n, i) >> 32);
      gtw += u > T;
      eqw += u == T;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gtw += __shfl_xor_sync(0xffffffffu, gtw, o);
    eqw += __shfl_xor_sync(0xffffffffu, eqw, o);
  }
  if (lane == 0) { cs.wgt[w] = gtw; cs.weq[w] = eqw; }
  __syncthreads();
  if (w == 0) {   // lane q holds warp q's counts
    int g = lane < kClWarps ? cs.wgt[lane] : 0, e = lane < kClWarps ? cs.weq[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, o);
      e += __shfl_xor_sync(0xffffffffu, e, o);
    }
    if (lane == 0) {
      cs.cta_gt = g;
      cs.cta_eq = e;
    }
  }
  cluster_sync_all();

  // keys taken by the lower-ranked CTAs of the head: all above T and, of
  // the ties, as many as were still needed in key order.  Lane r of warp 0
  // reads CTA r's counts (all remote loads in flight together); the ties
  // seen before r come from a prefix sum.
  if (threadIdx.x < 32) {
    const int r = (int)threadIdx.x;
    int g = 0, e = 0;
    if (r < rank) {
      g = (int)ld_dsmem_u32(dsmem_addr(&cs.cta_gt, (uint32_t)r));
      e = (int)ld_dsmem_u32(dsmem_addr(&cs.cta_eq, (uint32_t)r));
    }
    int e_incl = e;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, e_incl, o);
      if (r >= o) e_incl += t;
    }
    const int e_before = e_incl - e;
    int took = r < rank ? g + (mode == 2 ? 0 : max(0, min(e, need_eq - e_before))) : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) took += __shfl_xor_sync(0xffffffffu, took, o);
    const int eb_all = __shfl_sync(0xffffffffu, e_incl, 31);
    // lane q: where warp q's stretch starts writing (after the lower CTAs'
    // keys and the keys warps 0 .. q-1 take) and how many ties come before it
    const int qg = r < kClWarps ? cs.wgt[r] : 0, qe = r < kClWarps ? cs.weq[r] : 0;
    int qe_incl = qe;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, qe_incl, o);
      if (r >= o) qe_incl += t;
    }
    const int eb = eb_all + qe_incl - qe;
    const int qtake = qg + (mode == 2 ? 0 : max(0, min(qe, need_eq - eb)));
    int qt_incl = qtake;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, qt_incl, o);
      if (r >= o) qt_incl += t;
    }
    if (r < kClWarps) {
      cs.wout[r] = took + qt_incl - qtake;
      cs.weqb[r] = eb;
    }
  }
  __syncthreads();
  // no CTA reads another's shared memory after this point; a CTA may leave
  // once every CTA of the cluster has arrived here (the wait is at the end)
  cluster_arrive();

  const int n_take = mode == 0 ? 0 : mode == 2 ? E : n_sel;
  int32_t* out = idx + (size_t)b * sp.T + sp.off[h];
  if (rank == 0) {
    for (int jj = threadIdx.x; jj < sp.r_lo; jj += kClThreads) out[jj] = jj;
    for (int jj = sp.r_hi + threadIdx.x; jj < sp.S; jj += kClThreads) out[sp.r_lo + n_take + (jj - sp.r_hi)] = jj;
  }
  if (mode != 0) {
    int written = cs.wout[w], eq_seen = cs.weqb[w];
    const unsigned lt = (1u << lane) - 1u;
    for (int i0 = lo; i0 < hi; i0 += 32) {
      const int i = i0 + lane;
      const bool in = i < hi;
      const uint64_t e = in ? share_entry(hv, stage, f0, n, i) : 0ull;
      const uint32_t u = (uint32_t)(e >> 32);
      const bool is_gt = in && (mode == 2 || u > T);
      const bool is_eq = in && mode != 2 && u == T;
      const unsigned eqb = __ballot_sync(0xffffffffu, is_eq);
      const bool f = is_gt || (is_eq && eq_seen + __popc(eqb & lt) < need_eq);
      const unsigned fb = __ballot_sync(0xffffffffu, f);
      if (f) {
        const int r = written + __popc(fb & lt);
        if (r < n_take) out[sp.r_lo + r] = (int32_t)(uint32_t)e;
        else record_status(status, kStatusSelectMismatch);
      }
      written += __popc(fb);
      eq_seen += __popc(eqb);
    }
  }
  cluster_wait();
}

// Gather retained rows: one 16-byte vector per lane, D/8 lanes per row.
template <int D>
__global__ void __launch_bounds__(256)
kvc_gather_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
              const int32_t* idx, const __grid_constant__ SelParams sp, int B,
              __nv_bfloat16* __restrict__ k_out, __nv_bfloat16* __restrict__ v_out, int32_t* pos_out,
              int* status) {
  grid_dep_wait();   // the positions come from the previous grid
  grid_dep_launch();
  constexpr int LPR = D / 8;             // lanes per row
  constexpr int RPW = 32 / LPR;          // rows per warp step
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, cl = lane % LPR;
  const int64_t rows = (int64_t)B * sp.T;
  const int64_t warp_g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t r = warp_g * RPW + sub; r < rows; r += nwarps * RPW) {
    const int b = (int)(r / sp.T);
    const int64_t within = r - (int64_t)b * sp.T;
    int lo = 0, hi = sp.H_kv - 1;
    while (lo < hi) {  // last head whose offset is <= within
      const int mid = (lo + hi + 1) >> 1;
      if (sp.off[mid] <= within) lo = mid; else hi = mid - 1;
    }
    if (within < sp.off[lo] || within - sp.off[lo] >= sp.kept[lo]) continue;   // a row the layout leaves free
    const int j = idx[r];
    if (j < 0 || j >= sp.S) {
      if (cl == 0) record_status(status, kStatusSelectMismatch);
      continue;
    }
    const size_t src = (((size_t)b * sp.H_kv + lo) * sp.S + j) * D + cl * 8;
    const uint4 kv = *reinterpret_cast<const uint4*>(k + src);
    const uint4 vv = *reinterpret_cast<const uint4*>(v + src);
    *reinterpret_cast<uint4*>(k_out + (size_t)r * D + cl * 8) = kv;
    *reinterpret_cast<uint4*>(v_out + (size_t)r * D + cl * 8) = vv;
    if (cl == 0 && pos_out != idx) pos_out[r] = j;
  }
}

}  // namespace

cudaError_t launch_select(int mode, const float* scores, const uint64_t* cand, const int* cand_cnt,
                          int cap, int B, const SelParams& sel, int32_t* idx, cudaStream_t st) {
  SegView v{mode, scores, cand, cand_cnt, cap};
  const int BH = B * sel.H_kv;
  cudaError_t e = cudaSuccess;
  const int np = mode == 0 ? 1 : sel.nparts;
  auto smem_for = [np, mode](int cap) {
    return (size_t)cap * sizeof(uint64_t) + (mode == 0 ? 0 : (size_t)np * sizeof(int64_t)) +
           (size_t)(np + 1) * sizeof(int);
  };
  if (smem_for(kStageC) > 200 * 1024) return cudaErrorInvalidConfiguration;
  // the widest cluster that still gives every head its own CTAs in one wave;
  // 16 (smaller shared-memory shares) only where the device co-schedules a
  // cluster of 16 for every head at once.  Short heads keep clusters of 8:
  // narrower clusters were slower there (Llama 8K: 18.6 us at 8, 21.6 at 2,
  // 24.8 at 1), the cluster's parallel sweeps outweigh its barriers.
  int cl = sel.S >= 65536 ? kMaxCl : 8;
  while (cl > 1 && (int64_t)BH * cl > num_sms()) cl >>= 1;
  auto pick = [](int c) {
    return c == 16 ? kvc_select_kernel<16> : c == 8 ? kvc_select_kernel<8> : c == 4 ? kvc_select_kernel<4>
           : c == 2 ? kvc_select_kernel<2> : kvc_select_kernel<1>;
  };
  static int s_ncl16[64] = {0};   // per device: clusters of 16 resident at once + 1 (0: not asked yet)
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (cl == 16 && s_ncl16[dev] > 0) cl = s_ncl16[dev] - 1 >= BH ? 16 : 8;
  if (cl == 16 && s_ncl16[dev] == 0) {
    auto k16 = pick(16);
    int nclusters = 0;
    bool ok16 = cudaFuncSetAttribute(k16, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess &&
                cudaFuncSetAttribute(k16, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_for(kStageC16)) ==
                    cudaSuccess;
    if (ok16) {
      cudaLaunchConfig_t q{};
      q.gridDim = dim3((unsigned)(BH * 16));
      q.blockDim = dim3(kClThreads);
      q.dynamicSmemBytes = smem_for(kStageC16);
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = 16;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      q.attrs = qa;
      q.numAttrs = 1;
      ok16 = cudaOccupancyMaxActiveClusters(&nclusters, k16, &q) == cudaSuccess;
    }
    if (!ok16) {
      (void)cudaGetLastError();
      nclusters = 0;
    }
    s_ncl16[dev] = nclusters + 1;
    if (nclusters < BH) cl = 8;
  }
  const int stage_cap = cl == 16 ? kStageC16 : kStageC;
  const size_t smem = smem_for(stage_cap);
  auto kern = pick(cl);
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
    return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)(BH * cl));
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  int* status = status_word_ptr();
  if ((e = cudaLaunchKernelEx(&cfg, kern, v, sel, stage_cap, idx, status)) != cudaSuccess) return e;
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_gather(const __nv_bfloat16* k, const __nv_bfloat16* v, const int32_t* idx, int B,
                          const SelParams& sp, int D, __nv_bfloat16* k_out, __nv_bfloat16* v_out,
                          int32_t* pos_out, cudaStream_t st) {
  const int64_t T = sp.T;
  const int64_t rows = (int64_t)B * T;
  if (rows == 0) return cudaSuccess;
  const int rows_per_block = (256 / 32) * (32 / (D / 8));
  int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
  if (blocks > 4 * 1024) blocks = 4 * 1024;
  cudaError_t e;
  if (D == 64)
    e = launch_pdl(kvc_gather_kernel<64>, dim3((unsigned)blocks), dim3(256), 0, st, k, v, idx, sp, B, k_out, v_out,
                   pos_out, status_word_ptr());
  else
    e = launch_pdl(kvc_gather_kernel<128>, dim3((unsigned)blocks), dim3(256), 0, st, k, v, idx, sp, B, k_out, v_out,
                   pos_out, status_word_ptr());
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvc
