// Per-head top-k selection and gather (TideKV, Fig. 2 and Fig. 3).
//
// Selection keeps, per (b, KV head), the mandatory set R_mand = [0, sink) u
// [S - recent, S) and the n_sel best other keys by (score desc, index asc),
// listed in ascending position.  Scores are >= 0, so their fp32 bit patterns
// order like the values; a three-round radix select over those bits (11, 11
// and 10 bits, each round a histogram of the keys that share the digits found
// so far) finds the n_sel-th score T and how many keys scoring exactly T are
// still needed.  Ties at T are taken in ascending index order, which the last
// two kernels resolve with per-range counts and an ordered block scan.
//
// The keys come either from a dense score array (mode 0) or from the
// per-range candidate lists of the fused scorer (mode 1, entries
// (score bits << 32 | index), ascending index within each range, ranges in
// ascending key order).
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

struct FindSmem {
  int scan[32];
  int digit, need;
};

// Given a histogram (nbins, digit d counts keys whose next digit is d) and the
// number `need` of keys still to take among them, find the digit holding the
// need-th largest key and how many keys of that digit are still needed.
__device__ void find_digit(const uint32_t* hist, int nbins, int need, FindSmem* fs, int* digit_out,
                           int* need_out) {
  const int tid = threadIdx.x;
  const int per = nbins / kSelThreads;   // 8 or 4 bins per thread, highest digits first
  const int hi = nbins - 1 - tid * per;  // this thread covers digits hi, hi-1, ..., hi-per+1
  if (tid == 0) { fs->digit = 0; fs->need = 0; }
  int local = 0;
  for (int i = 0; i < per; ++i) local += (int)__ldcg(&hist[hi - i]);
  int tot;
  const int incl = block_inclusive_scan(local, fs->scan, &tot);
  const int before = incl - local;
  if (before < need && need <= incl) {
    int cum = before;
    for (int i = 0; i < per; ++i) {
      const int c = (int)__ldcg(&hist[hi - i]);
      if (cum + c >= need) {
        fs->digit = hi - i;
        fs->need = need - cum;
        break;
      }
      cum += c;
    }
  }
  __syncthreads();
  *digit_out = fs->digit;
  *need_out = fs->need;
  __syncthreads();
}


// Histogram round `round` (0, 1, 2) over one key range.
__global__ void __launch_bounds__(kSelThreads)
kvc_hist_kernel(SegView v, const __grid_constant__ SelParams sp, int round, uint32_t* __restrict__ hist) {
  const int part = blockIdx.x / kSplit, sub = blockIdx.x % kSplit, seg = blockIdx.y, h = seg % sp.H_kv;
  __shared__ uint32_t sh[kHist1];
  __shared__ FindSmem fs;
  const int n_sel = sp.n_sel[h];
  uint32_t* hseg = hist + (size_t)seg * kHistPerSeg;
  SelState* st = reinterpret_cast<SelState*>(hseg + kHistBins);
  uint32_t prefix = 0;
  int need = 0;
  if (round > 0) {
    if (st->mode != 1) return;  // nothing to rank: every CTA of the head leaves
    prefix = st->prefix;
    need = st->need;
  }
  const int nb = round == 2 ? kHist3 : kHist1;
  for (int i = threadIdx.x; i < nb; i += blockDim.x) sh[i] = 0;
  __syncthreads();
  int64_t first;
  const int plen = range_len(v, sp, seg, part, &first);
  const int lo = (int)((int64_t)plen * sub / kSplit), len = (int)((int64_t)plen * (sub + 1) / kSplit);
  // Scores of one head share their leading bits, so many keys hit the same
  // digit: lanes with equal digits are merged into one shared-memory atomic.
  // kBatch independent loads per thread are in flight before any is used.
  for (int i0 = lo; i0 < len; i0 += kBatch * kSelThreads) {
    uint32_t u[kBatch];
    bool in[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int i = i0 + q * kSelThreads + threadIdx.x;
      in[q] = i < len;
      int j;
      u[q] = 0u;
      if (in[q]) entry_at(v, sp, seg, part, first, i, &u[q], &j);
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      int bin = -1;
      if (in[q]) {
        if (round == 0) bin = (int)(u[q] >> 21);
        else if (round == 1) bin = (u[q] >> 21) == prefix ? (int)((u[q] >> 10) & 2047u) : -1;
        else bin = (u[q] >> 10) == prefix ? (int)(u[q] & 1023u) : -1;
      }
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      if (bin >= 0 && (int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&sh[bin], (uint32_t)__popc(peers));
    }
  }
  __syncthreads();
  uint32_t* dst = hseg + (round == 0 ? 0 : round == 1 ? kHist1 : kHist1 + kHist2);
  for (int i = threadIdx.x; i < nb; i += blockDim.x)
    if (sh[i]) atomicAdd(&dst[i], sh[i]);
  // the last CTA of this head to finish resolves the round's digit once
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&st->done[round], 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (round == 0) {
    int c = 0;
    for (int i = threadIdx.x; i < kHist1; i += blockDim.x) c += (int)__ldcg(&dst[i]);
    int total;
    block_inclusive_scan(c, fs.scan, &total);
    if (threadIdx.x == 0) {
      st->total = total;
      st->mode = n_sel <= 0 ? 0 : n_sel >= total ? 2 : 1;
    }
    if (n_sel <= 0 || n_sel >= total) return;
  }
  int d, nd;
  find_digit(dst, nb, round == 0 ? n_sel : need, &fs, &d, &nd);
  if (threadIdx.x == 0) {
    st->prefix = round == 0 ? (uint32_t)d : round == 1 ? (prefix << 11) | (uint32_t)d : (prefix << 10) | (uint32_t)d;
    st->need = nd;
  }
}

// Exact threshold T and the count of keys equal to T still needed, as left
// by the histogram rounds.  mode 0: take none, 2: take every candidate.
__device__ __forceinline__ void threshold(const SelState* st, uint32_t* T, int* need_eq, int* mode, int* total) {
  *mode = st->mode;
  *T = st->prefix;
  *need_eq = st->need;
  *total = st->total;
}

// Per range: number of keys scoring above T and exactly T.
__global__ void __launch_bounds__(kSelThreads)
kvc_count_kernel(SegView v, const __grid_constant__ SelParams sp, const uint32_t* __restrict__ hist,
             int2* __restrict__ pcnt) {
  const int part = blockIdx.x / kSplit, sub = blockIdx.x % kSplit, seg = blockIdx.y;
  __shared__ int scan[32];
  uint32_t T;
  int need_eq, mode, total;
  threshold(reinterpret_cast<const SelState*>(hist + (size_t)seg * kHistPerSeg + kHistBins), &T, &need_eq, &mode,
            &total);
  int64_t first;
  const int plen = range_len(v, sp, seg, part, &first);
  const int lo = (int)((int64_t)plen * sub / kSplit), len = (int)((int64_t)plen * (sub + 1) / kSplit);
  int gt = 0, eq = 0;
  if (mode == 1) {
    for (int i0 = lo; i0 < len; i0 += kBatch * kSelThreads) {
      uint32_t u[kBatch];
      bool in[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int i = i0 + q * kSelThreads + threadIdx.x;
        int j;
        u[q] = 0u;
        in[q] = i < len;
        if (in[q]) entry_at(v, sp, seg, part, first, i, &u[q], &j);
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        gt += (in[q] && u[q] > T);
        eq += (in[q] && u[q] == T);
      }
    }
  } else if (mode == 2) {
    gt = threadIdx.x == 0 ? len - lo : 0;
  }
  int tg, te;
  block_inclusive_scan(gt, scan, &tg);
  block_inclusive_scan(eq, scan, &te);
  if (threadIdx.x == 0) pcnt[(size_t)seg * sp.nparts * kSplit + blockIdx.x] = make_int2(tg, te);
}

// Ordered write of the retained positions of one range; range 0 also writes
// the mandatory positions.
__global__ void __launch_bounds__(kSelThreads)
kvc_write_kernel(SegView v, const __grid_constant__ SelParams sp, const uint32_t* __restrict__ hist,
             const int2* __restrict__ pcnt, int32_t* __restrict__ idx, int* status) {
  const int part = blockIdx.x / kSplit, seg = blockIdx.y;
  const int b = seg / sp.H_kv, h = seg % sp.H_kv;
  __shared__ int scan[32];
  uint32_t T;
  int need_eq, mode, total;
  threshold(reinterpret_cast<const SelState*>(hist + (size_t)seg * kHistPerSeg + kHistBins), &T, &need_eq, &mode,
            &total);
  const int n_sel = sp.n_sel[h];
  const int n_take = mode == 0 ? 0 : mode == 2 ? total : n_sel;
  int32_t* out = idx + (size_t)b * sp.T + sp.off[h];
  if (blockIdx.x == 0) {
    for (int jj = threadIdx.x; jj < sp.r_lo; jj += blockDim.x) out[jj] = jj;
    for (int jj = sp.r_hi + threadIdx.x; jj < sp.S; jj += blockDim.x) out[sp.r_lo + n_take + (jj - sp.r_hi)] = jj;
  }
  if (mode == 0) return;
  // exclusive prefix over the earlier sub-ranges of this head (in key order):
  // a sub-range q takes all its keys above T and, of its ties, as many as
  // are still needed after the ties of the sub-ranges before it
  const int nb = blockIdx.x;
  const int2* pc = pcnt + (size_t)seg * sp.nparts * kSplit;
  int out_before = 0, eq_before = 0;
  for (int q0 = 0; q0 < nb; q0 += kSelThreads) {
    const int q = q0 + threadIdx.x;
    const int2 c = q < nb ? pc[q] : make_int2(0, 0);
    int tot_eq;
    const int eq_incl = block_inclusive_scan(c.y, scan, &tot_eq);
    const int eqb_q = eq_before + eq_incl - c.y;
    int contrib = c.x + (mode == 2 ? 0 : max(0, min(c.y, need_eq - eqb_q)));
    int tot_c;
    block_inclusive_scan(contrib, scan, &tot_c);
    out_before += tot_c;
    eq_before += tot_eq;
  }
  int64_t first;
  const int plen = range_len(v, sp, seg, part, &first);
  const int sub = blockIdx.x % kSplit;
  const int slo = (int)((int64_t)plen * sub / kSplit), shi = (int)((int64_t)plen * (sub + 1) / kSplit);
  // each warp owns a contiguous stretch of the sub-range: count it, then
  // write it in order with ballots; one block-wide exchange places the warps
  constexpr int kWarps = kSelThreads / 32;
  __shared__ int s_wgt[kWarps], s_weq[kWarps], s_wout[kWarps], s_weqb[kWarps];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int chunk = (shi - slo + kWarps - 1) / kWarps;
  const int lo = min(shi, slo + w * chunk), hi = min(shi, lo + chunk);
  int gtw = 0, eqw = 0;
  if (mode == 2) {
    gtw = lane == 0 ? hi - lo : 0;
  } else {
    for (int i0 = lo; i0 < hi; i0 += 32 * kBatch) {
      uint32_t u[kBatch];
      bool in[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const int i = i0 + 32 * q + lane;
        int j;
        u[q] = 0u;
        in[q] = i < hi;
        if (in[q]) entry_at(v, sp, seg, part, first, i, &u[q], &j);
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        gtw += (in[q] && u[q] > T);
        eqw += (in[q] && u[q] == T);
      }
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
  for (int b0 = lo; b0 < hi; b0 += 32 * kBatch) {
    uint32_t u[kBatch];
    int jj[kBatch];
    bool in[kBatch];
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int i = b0 + 32 * q + lane;
      u[q] = 0u;
      jj[q] = 0;
      in[q] = i < hi;
      if (in[q]) entry_at(v, sp, seg, part, first, i, &u[q], &jj[q]);
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const bool is_gt = in[q] && (mode == 2 || u[q] > T);
      const bool is_eq = in[q] && mode != 2 && u[q] == T;
      const unsigned eqb = __ballot_sync(0xffffffffu, is_eq);
      const bool f = is_gt || (is_eq && eq_seen + __popc(eqb & lt) < need_eq);
      const unsigned fb = __ballot_sync(0xffffffffu, f);
      if (f) {
        const int r = written + __popc(fb & lt);
        if (r < n_take) out[sp.r_lo + r] = jj[q];
        else record_status(status, kStatusSelectMismatch);
      }
      written += __popc(fb);
      eq_seen += __popc(eqb);
    }
  }
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
  dim3 grid(sel.nparts * kSplit, BH);
  for (int round = 0; round < 3; ++round) {
    kvc_hist_kernel<<<grid, kSelThreads, 0, st>>>(v, sel, round, hist);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  kvc_count_kernel<<<grid, kSelThreads, 0, st>>>(v, sel, hist, pcnt);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  kvc_write_kernel<<<grid, kSelThreads, 0, st>>>(v, sel, hist, pcnt, idx, status_word_ptr());
  note_launches(5);
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
