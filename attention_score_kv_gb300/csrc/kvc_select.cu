// Per-head top-k selection and gather (TideKV, Fig. 2 and Fig. 3).
//
// Selection keeps, per (b, KV head), the mandatory set R_mand = [0, sink) u
// [S - recent, S) and the n_sel best other keys by (score desc, index asc),
// listed in ascending position.  Scores are >= 0, so their fp32 bit patterns
// order like the values; a three-round radix select over those bits (11, 11
// and 10 bits, each round a histogram of the keys that share the digits found
// so far) finds the n_sel-th score T and how many keys scoring exactly T are
// still needed.  Ties at T are taken in ascending index order, resolved with
// per-unit counts and an ordered block scan.  All of it runs in one
// cooperative launch whose phases are separated by bounded grid barriers.
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

constexpr int kSelThreads = 256;
constexpr int kBatch = 4;   // independent entry loads in flight per thread
constexpr int kSplit = kSelectSplit;   // CTAs sharing one key range

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
  const int64_t c_first = ((int64_t)seg * S) / sp.L;
  const int64_t c_last = (((int64_t)seg + 1) * S - 1) / sp.L;
  const int64_t c = c_first + part;
  if (c > c_last) return -1;
  if (part > 0) return c * sp.maxseg;
  return c * sp.maxseg + (seg - (c * sp.L) / S);
}

// Number of entries of range `part` of head `seg`; for mode 0 also the first
// key index of the range, for mode 1 the slot.
__device__ __forceinline__ int range_len(const SegView& v, const SelParams& sp, int seg, int part,
                                         int64_t* first) {
  if (v.mode == 0) {
    const int ncand = sp.r_hi - sp.r_lo;
    const int per = (ncand + sp.nparts - 1) / sp.nparts;
    const int lo = part * per;
    const int hi = min(ncand, lo + per);
    *first = sp.r_lo + lo;
    return max(0, hi - lo);
  }
  const int64_t slot = cand_slot(sp, seg, part);
  *first = slot;
  return slot < 0 ? 0 : min(max(v.cand_cnt[slot], 0), v.cap);
}

__device__ __forceinline__ void entry_at(const SegView& v, const SelParams& sp, int seg, int part,
                                         int64_t first, int i, uint32_t* u, int* j) {
  (void)part;
  if (v.mode == 0) {
    *j = (int)first + i;
    uint32_t bits = __float_as_uint(v.scores[(size_t)seg * sp.S + first + i]);
    *u = (bits == 0x80000000u) ? 0u : bits;
  } else {
    const uint64_t e = v.cand[(size_t)first * v.cap + i];
    *u = (uint32_t)(e >> 32);
    *j = (int)(uint32_t)e;
  }
}

// Shared-memory copy of a CTA's first unit: up to kStage entries stay on
// chip for every round, so only the first round reads them from L2.
constexpr int kStage = 4096;
constexpr int kMaxUnits = 8;                  // units one CTA may own
constexpr uint32_t kBarLimit = 1u << 22;      // polls before a grid barrier gives up

struct FindSmem {
  int scan[32];
  int digit, need, total;
};

// Given a histogram in global memory (nbins, digit d counts keys whose next
// digit is d) and the number `need` of keys still to take among them, find
// the digit holding the need-th largest key, how many keys of that digit are
// still needed, and the histogram's total.
__device__ void find_digit(const uint32_t* hist, int nbins, int need, FindSmem* fs, int* digit_out, int* need_out,
                           int* total_out) {
  const int tid = threadIdx.x;
  const int per = nbins / kSelThreads;   // 8 or 4 bins per thread, highest digits first
  const int hi = nbins - 1 - tid * per;  // this thread covers digits hi, hi-1, ..., hi-per+1
  if (tid == 0) { fs->digit = 0; fs->need = 0; }
  uint32_t c[8];
  int local = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) c[i] = i < per ? __ldcg(&hist[hi - i]) : 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) local += (int)c[i];
  int tot;
  const int incl = block_inclusive_scan(local, fs->scan, &tot);
  const int before = incl - local;
  if (before < need && need <= incl) {
    int cum = before;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < per && cum < need && cum + (int)c[i] >= need) {
        fs->digit = hi - i;
        fs->need = need - cum;
      }
      cum += (int)c[i];
    }
  }
  __syncthreads();
  *digit_out = fs->digit;
  *need_out = fs->need;
  *total_out = tot;
  __syncthreads();
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of a cooperative launch over a monotonic counter that
// starts at zero: the k-th barrier waits for k * gridDim.x arrivals.  The
// wait is bounded; giving up records a timeout and makes the CTA return.
__device__ bool grid_barrier(uint32_t* ctr, uint32_t k, volatile int* s_abort, int* status) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ctr, 1u);
    const uint32_t target = k * gridDim.x;
    uint32_t i = 0;
    while (ld_acquire_u32(ctr) < target) {
      if (++i == kBarLimit) {
        record_status(status, kStatusTimeout);
        *s_abort = 1;
        break;
      }
      __nanosleep(64);
    }
    __threadfence();
  }
  __syncthreads();
  return *s_abort == 0;
}

// One unit of selection work: sub-range `sub` of key range `part` of head
// `seg`, entries [lo, hi) of the range.
struct UnitSmem {
  int seg[kMaxUnits], blk[kMaxUnits], lo[kMaxUnits], hi[kMaxUnits];
  int mode[kMaxUnits], need[kMaxUnits], total[kMaxUnits];
  int64_t first[kMaxUnits];
  uint32_t prefix[kMaxUnits];
  int n, staged;   // units of this CTA; entries of unit 0 held in shared memory
};

__device__ __forceinline__ void unit_entry(const SegView& v, const SelParams& sp, const UnitSmem& us, int ui,
                                           const uint64_t* stage, int i, uint32_t* u, int* j) {
  if (ui == 0 && i - us.lo[0] < us.staged) {
    const uint64_t e = stage[i - us.lo[0]];
    *u = (uint32_t)(e >> 32);
    *j = (int)(uint32_t)e;
  } else {
    entry_at(v, sp, us.seg[ui], 0, us.first[ui], i, u, j);
  }
}

// Histogram of round `round` over unit ui into sh, then added to the head's
// global histogram.  Round 0 also fills the shared-memory copy of unit 0.
__device__ void unit_hist(const SegView& v, const SelParams& sp, const UnitSmem& us, int ui, int round,
                          uint64_t* stage, uint32_t* sh, uint32_t* hist) {
  const int nb = round == 2 ? kHist3 : kHist1;
  const uint32_t prefix = us.prefix[ui];
  for (int i = threadIdx.x; i < nb; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  const int lo = us.lo[ui], hi = us.hi[ui];
  for (int i0 = lo; i0 < hi; i0 += kBatch * kSelThreads) {
    uint32_t u[kBatch];
    int jj[kBatch];
    bool in[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int i = i0 + q * kSelThreads + threadIdx.x;
      in[q] = i < hi;
      u[q] = 0u;
      jj[q] = 0;
      if (in[q]) {
        if (round == 0) entry_at(v, sp, us.seg[ui], 0, us.first[ui], i, &u[q], &jj[q]);
        else unit_entry(v, sp, us, ui, stage, i, &u[q], &jj[q]);
      }
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int i = i0 + q * kSelThreads + threadIdx.x;
      if (round == 0 && ui == 0 && in[q] && i - lo < kStage) stage[i - lo] = ((uint64_t)u[q] << 32) | (uint32_t)jj[q];
      int bin = -1;
      if (in[q]) {
        if (round == 0) bin = (int)(u[q] >> 21);
        else if (round == 1) bin = (u[q] >> 21) == prefix ? (int)((u[q] >> 10) & 2047u) : -1;
        else bin = (u[q] >> 10) == prefix ? (int)(u[q] & 1023u) : -1;
      }
      // scores of one head share their leading bits, so many lanes hit the
      // same digit: equal digits are merged into one shared-memory atomic
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (bin >= 0 && (int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&sh[bin], (uint32_t)__popc(peers));
    }
  }
  __syncthreads();
  uint32_t* dst = hist + (size_t)us.seg[ui] * kHistPerSeg + (round == 0 ? 0 : round == 1 ? kHist1 : kHist1 + kHist2);
  for (int i = threadIdx.x; i < nb; i += blockDim.x)
    if (sh[i]) atomicAdd(&dst[i], sh[i]);
  __syncthreads();
}

// Resolve round `round`'s digit of unit ui's head from the global histogram.
__device__ void unit_resolve(const SelParams& sp, UnitSmem& us, int ui, int round, const uint32_t* hist,
                             FindSmem* fs) {
  const uint32_t* hseg = hist + (size_t)us.seg[ui] * kHistPerSeg;
  int d, nd, tot;
  if (round == 0) {
    const int n_sel = sp.n_sel[us.seg[ui] % sp.H_kv];
    find_digit(hseg, kHist1, n_sel, fs, &d, &nd, &tot);
    if (threadIdx.x == 0) {
      us.total[ui] = tot;
      us.mode[ui] = n_sel <= 0 ? 0 : n_sel >= tot ? 2 : 1;
      us.prefix[ui] = (uint32_t)d;
      us.need[ui] = nd;
    }
  } else {
    if (us.mode[ui] != 1) return;
    const int nb = round == 1 ? kHist2 : kHist3;
    find_digit(hseg + (round == 1 ? kHist1 : kHist1 + kHist2), nb, us.need[ui], fs, &d, &nd, &tot);
    if (threadIdx.x == 0) {
      us.prefix[ui] = (us.prefix[ui] << (round == 1 ? 11 : 10)) | (uint32_t)d;
      us.need[ui] = nd;
    }
  }
  __syncthreads();
}

// Keys of unit ui above T and exactly T.
__device__ int2 unit_count(const SegView& v, const SelParams& sp, const UnitSmem& us, int ui, const uint64_t* stage,
                           int* scan) {
  const int mode = us.mode[ui];
  const uint32_t T = us.prefix[ui];
  int gt = 0, eq = 0;
  if (mode == 1) {
    for (int i0 = us.lo[ui]; i0 < us.hi[ui]; i0 += kBatch * kSelThreads) {
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int i = i0 + q * kSelThreads + threadIdx.x;
        if (i < us.hi[ui]) {
          uint32_t u;
          int j;
          unit_entry(v, sp, us, ui, stage, i, &u, &j);
          gt += u > T;
          eq += u == T;
        }
      }
    }
  } else if (mode == 2) {
    gt = threadIdx.x == 0 ? us.hi[ui] - us.lo[ui] : 0;
  }
  int tg, te;
  block_inclusive_scan(gt, scan, &tg);
  block_inclusive_scan(eq, scan, &te);
  return make_int2(tg, te);
}

// Ordered write of the retained positions of unit ui; the head's first unit
// also writes the mandatory positions.
__device__ void unit_write(const SegView& v, const SelParams& sp, const UnitSmem& us, int ui, const uint64_t* stage,
                           const int2* pcnt, int32_t* idx, int* scan, int* status) {
  const int seg = us.seg[ui], blk = us.blk[ui];
  const int b = seg / sp.H_kv, h = seg % sp.H_kv;
  const int mode = us.mode[ui], need_eq = us.need[ui], total = us.total[ui];
  const uint32_t T = us.prefix[ui];
  const int n_sel = sp.n_sel[h];
  const int n_take = mode == 0 ? 0 : mode == 2 ? total : n_sel;
  int32_t* out = idx + (size_t)b * sp.T + sp.off[h];
  if (blk == 0) {
    for (int jj = threadIdx.x; jj < sp.r_lo; jj += blockDim.x) out[jj] = jj;
    for (int jj = sp.r_hi + threadIdx.x; jj < sp.S; jj += blockDim.x) out[sp.r_lo + n_take + (jj - sp.r_hi)] = jj;
  }
  if (mode == 0) return;
  // exclusive prefix over the earlier units of this head (in key order): a
  // unit takes all its keys above T and, of its ties, as many as are still
  // needed after the ties of the units before it
  const int2* pc = pcnt + (size_t)seg * sp.nparts * kSplit;
  int out_before = 0, eq_before = 0;
  for (int q0 = 0; q0 < blk; q0 += kSelThreads) {
    const int q = q0 + threadIdx.x;
    int2 c = make_int2(0, 0);
    if (q < blk) {
      const long long raw = __ldcg(reinterpret_cast<const long long*>(pc + q));
      c = make_int2((int)(uint32_t)raw, (int)(raw >> 32));
    }
    int tot_eq;
    const int eq_incl = block_inclusive_scan(c.y, scan, &tot_eq);
    const int eqb_q = eq_before + eq_incl - c.y;
    const int contrib = c.x + (mode == 2 ? 0 : max(0, min(c.y, need_eq - eqb_q)));
    int tot_c;
    block_inclusive_scan(contrib, scan, &tot_c);
    out_before += tot_c;
    eq_before += tot_eq;
  }
  // each warp owns a contiguous stretch of the unit: count it, then write it
  // in order with ballots; one block-wide exchange places the warps
  constexpr int kWarps = kSelThreads / 32;
  __shared__ int s_wgt[kWarps], s_weq[kWarps], s_wout[kWarps], s_weqb[kWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int chunk = (us.hi[ui] - us.lo[ui] + kWarps - 1) / kWarps;
  const int lo = min(us.hi[ui], us.lo[ui] + w * chunk), hi = min(us.hi[ui], lo + chunk);
  int gtw = 0, eqw = 0;
  if (mode == 2) {
    gtw = lane == 0 ? hi - lo : 0;
  } else {
    for (int i = lo + lane; i < hi; i += 32) {
      uint32_t u;
      int j;
      unit_entry(v, sp, us, ui, stage, i, &u, &j);
      gtw += u > T;
      eqw += u == T;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    gtw += __shfl_xor_sync(0xffffffffu, gtw, o);
    eqw += __shfl_xor_sync(0xffffffffu, eqw, o);
  }
  if (lane == 0) { s_wgt[w] = gtw; s_weq[w] = eqw; }
  __syncthreads();
  if (threadIdx.x == 0) {
    int ob = out_before, eb = eq_before;
    for (int q = 0; q < kWarps; ++q) {
      s_wout[q] = ob;
      s_weqb[q] = eb;
      ob += s_wgt[q] + (mode == 2 ? 0 : max(0, min(s_weq[q], need_eq - eb)));
      eb += s_weq[q];
    }
  }
  __syncthreads();
  int written = s_wout[w], eq_seen = s_weqb[w];
  const unsigned lt = (1u << lane) - 1u;
  for (int i0 = lo; i0 < hi; i0 += 32) {
    const int i = i0 + lane;
    uint32_t u = 0u;
    int j = 0;
    const bool in = i < hi;
    if (in) unit_entry(v, sp, us, ui, stage, i, &u, &j);
    const bool is_gt = in && (mode == 2 || u > T);
    const bool is_eq = in && mode != 2 && u == T;
    const unsigned eqb = __ballot_sync(0xffffffffu, is_eq);
    const bool f = is_gt || (is_eq && eq_seen + __popc(eqb & lt) < need_eq);
    const unsigned fb = __ballot_sync(0xffffffffu, f);
    if (f) {
      const int r = written + __popc(fb & lt);
      if (r < n_take) out[sp.r_lo + r] = j;
      else record_status(status, kStatusSelectMismatch);
    }
    written += __popc(fb);
    eq_seen += __popc(eqb);
  }
  __syncthreads();
}

// The whole selection in one cooperative launch.  Each CTA owns up to
// kMaxUnits units (sub-ranges of one head's key ranges).  Phases, separated
// by grid barriers: three radix histogram rounds (each CTA resolves the
// previous round's digit of its own heads from the global histogram), the
// per-unit counts above and at the threshold, and the ordered write.
__global__ void __launch_bounds__(kSelThreads)
kvc_select_kernel(SegView v, const __grid_constant__ SelParams sp, int n_units, uint32_t* __restrict__ hist,
                  int2* __restrict__ pcnt, int32_t* __restrict__ idx, int* status) {
  __shared__ uint32_t sh[kHist1];
  __shared__ uint64_t stage[kStage];
  __shared__ FindSmem fs;
  __shared__ UnitSmem us;
  __shared__ volatile int s_abort;
  uint32_t* bar = hist + kHistBins;   // head 0's state word: the barrier counter
  const int per_head = sp.nparts * kSplit;
  if (threadIdx.x == 0) {
    s_abort = 0;
    int n = 0;
    for (int u = blockIdx.x; u < n_units && n < kMaxUnits; u += gridDim.x, ++n) {
      const int seg = u / per_head, blk = u % per_head;
      const int part = blk / kSplit, sub = blk % kSplit;
      int64_t first;
      const int plen = range_len(v, sp, seg, part, &first);
      us.seg[n] = seg;
      us.blk[n] = blk;
      us.first[n] = first;
      us.lo[n] = (int)((int64_t)plen * sub / kSplit);
      us.hi[n] = (int)((int64_t)plen * (sub + 1) / kSplit);
      us.prefix[n] = 0;
    }
    us.n = n;
    us.staged = 0;
  }
  __syncthreads();
  const int nu = us.n;
  for (int ui = 0; ui < nu; ++ui) unit_hist(v, sp, us, ui, 0, stage, sh, hist);
  if (threadIdx.x == 0 && nu > 0) us.staged = min(us.hi[0] - us.lo[0], kStage);
  for (int round = 1; round <= 3; ++round) {
    if (!grid_barrier(bar, (uint32_t)round, &s_abort, status)) return;
    for (int ui = 0; ui < nu; ++ui) {
      unit_resolve(sp, us, ui, round - 1, hist, &fs);
      if (round < 3 && us.mode[ui] == 1) unit_hist(v, sp, us, ui, round, stage, sh, hist);
    }
  }
  // us.prefix is now the threshold T and us.need the ties at T still needed
  for (int ui = 0; ui < nu; ++ui) {
    const int2 c = unit_count(v, sp, us, ui, stage, fs.scan);
    if (threadIdx.x == 0) pcnt[(size_t)us.seg[ui] * per_head + us.blk[ui]] = c;
  }
  if (!grid_barrier(bar, 4u, &s_abort, status)) return;
  for (int ui = 0; ui < nu; ++ui) unit_write(v, sp, us, ui, stage, pcnt, idx, fs.scan, status);
}

// Gather retained rows: one 16-byte vector per lane, D/8 lanes per row.
template <int D>
__global__ void __launch_bounds__(256)
kvc_gather_kernel(const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
              const int32_t* idx, const __grid_constant__ SelParams sp, int B,
              __nv_bfloat16* __restrict__ k_out, __nv_bfloat16* __restrict__ v_out, int32_t* pos_out,
              int* status) {
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
                          int cap, int B, const SelParams& sel, uint32_t* hist, int2* pcnt,
                          int32_t* idx, cudaStream_t st) {
  SegView v{mode, scores, cand, cand_cnt, cap};
  const int BH = B * sel.H_kv;
  cudaError_t e = cudaMemsetAsync(hist, 0, (size_t)BH * kHistPerSeg * sizeof(uint32_t), st);
  if (e != cudaSuccess) return e;
  int n_units = sel.nparts * kSplit * BH;
  static int occ[64] = {0};
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (occ[dev] == 0 &&
      (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[dev], kvc_select_kernel, kSelThreads, 0)) != cudaSuccess)
    return e;
  const int grid = std::min(n_units, std::max(occ[dev], 1) * num_sms());
  if ((int64_t)grid * kMaxUnits < n_units) return cudaErrorInvalidConfiguration;
  int* status = status_word_ptr();
  void* args[] = {&v, const_cast<SelParams*>(&sel), &n_units, &hist, &pcnt, &idx, &status};
  e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kvc_select_kernel), dim3(grid), dim3(kSelThreads), args,
                                  0, st);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gather(const __nv_bfloat16* k, const __nv_bfloat16* v, const int32_t* idx, int B,
                          int H_kv, int S, int D, int64_t T, const int64_t* off_host,
                          __nv_bfloat16* k_out, __nv_bfloat16* v_out, int32_t* pos_out, cudaStream_t st) {
  SelParams sp{};
  sp.S = S;
  sp.H_kv = H_kv;
  sp.T = T;
  for (int h = 0; h < H_kv; ++h) sp.off[h] = off_host[h];
  const int64_t rows = (int64_t)B * T;
  if (rows == 0) return cudaSuccess;
  const int rows_per_block = (256 / 32) * (32 / (D / 8));
  int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
  if (blocks > 4 * 1024) blocks = 4 * 1024;
  if (D == 64)
    kvc_gather_kernel<64><<<(unsigned)blocks, 256, 0, st>>>(k, v, idx, sp, B, k_out, v_out, pos_out, status_word_ptr());
  else
    kvc_gather_kernel<128><<<(unsigned)blocks, 256, 0, st>>>(k, v, idx, sp, B, k_out, v_out, pos_out, status_word_ptr());
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace kvc
