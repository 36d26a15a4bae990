// HeteroCache's measurement and allocation steps on the device (HeteroCache,
// "Key Contributions" 1-2 and "Methodology": Phases 1-2).
//
// Overlap coefficient of two top-k index sets, |A n B| / min(|A|, |B|): the
// measure behind the stability score (a head's top-k during decoding against
// its prefill set) and the similarity score (the largest overlap between a
// head and any other head of its layer).  Sets are ascending, duplicate-free
// int32 position lists, as kvc_select_topk writes them; each thread looks up
// elements of the shorter list in the longer one by binary search, and the
// CTA adds the hits.  An empty set gives 0.
//
// Inverse-stability budgets: per layer, the HeteroCache weights w_h = 1/s_h,
// shares total * w_h / sum(w) rounded by largest remainder (ties to the lower
// head) and clamped to [lo, hi] -- the same float64 operations, in the same
// order, as the host kvc_budget_inverse_stability, so both give identical
// budgets.
#include "kvc_device.cuh"
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kOvThreads = 256;
constexpr int kMaxSteps = kMaxDecodeSteps;

// Hits of the shorter list in the longer one, summed over the CTA.
__device__ int intersect_count(const int32_t* a, int na, const int32_t* b, int nb, int* scratch) {
  const int32_t* s = na <= nb ? a : b;
  const int32_t* l = na <= nb ? b : a;
  const int ns = min(na, nb), nl = max(na, nb);
  int hits = 0;
  for (int i = threadIdx.x; i < ns; i += blockDim.x) {
    const int32_t x = s[i];
    int lo = 0, hi = nl;   // first element >= x
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (l[mid] < x) lo = mid + 1; else hi = mid;
    }
    hits += (lo < nl && l[lo] == x) ? 1 : 0;
  }
  int total;
  block_inclusive_scan(hits, scratch, &total);
  return total;
}

__device__ __forceinline__ float overlap_of(int inter, int na, int nb) {
  const int mn = min(na, nb);
  return mn > 0 ? __fdiv_rn((float)inter, (float)mn) : 0.f;
}

// One CTA per pair (A_i, B_i).
__global__ void __launch_bounds__(kOvThreads)
kvc_overlap_kernel(const int32_t* __restrict__ a, const int64_t* __restrict__ a_off, const int32_t* __restrict__ b,
                   const int64_t* __restrict__ b_off, float* __restrict__ out) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int scratch[32];
  const int p = blockIdx.x;
  const int64_t a0 = a_off[p], b0 = b_off[p];
  const int na = (int)(a_off[p + 1] - a0), nb = (int)(b_off[p + 1] - b0);
  const int inter = intersect_count(a + a0, na, b + b0, nb, scratch);
  if (threadIdx.x == 0) out[p] = overlap_of(inter, na, nb);
}

// One CTA per head i of a group of H sets: max over j != i of overlap(i, j).
__global__ void __launch_bounds__(kOvThreads)
kvc_similarity_kernel(const int32_t* __restrict__ idx, const int64_t* __restrict__ off, int H, float* __restrict__ sim) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int scratch[32];
  const int g = blockIdx.y, i = blockIdx.x;   // group (e.g. batch element x layer), head
  const int64_t* o = off + (size_t)g * (H + 1);
  const int ni = (int)(o[i + 1] - o[i]);
  float best = 0.f;
  for (int j = 0; j < H; ++j) {
    if (j == i) continue;
    const int nj = (int)(o[j + 1] - o[j]);
    const int inter = intersect_count(idx + o[i], ni, idx + o[j], nj, scratch);
    best = fmaxf(best, overlap_of(inter, ni, nj));
  }
  if (threadIdx.x == 0) sim[(size_t)g * H + i] = H > 1 ? best : 0.f;
}

// Phase 1 over decoding steps.  One CTA per (head h, step t): the overlap of
// the head's top-k at step t with its prefill set, into per_step[t][h].
__global__ void __launch_bounds__(kOvThreads)
kvc_stability_step_kernel(const int32_t* __restrict__ dec_idx, const int64_t* __restrict__ dec_off,
                          const int32_t* __restrict__ pre_idx, const int64_t* __restrict__ pre_off, int H,
                          float* __restrict__ per_step) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ int scratch[32];
  const int h = blockIdx.x, t = blockIdx.y;
  const size_t d = (size_t)t * H + h;
  const int nd = (int)(dec_off[d + 1] - dec_off[d]), np_ = (int)(pre_off[h + 1] - pre_off[h]);
  const int inter = intersect_count(dec_idx + dec_off[d], nd, pre_idx + pre_off[h], np_, scratch);
  if (threadIdx.x == 0) per_step[d] = overlap_of(inter, nd, np_);
}

// One CTA per head: the median over T steps of x[t][h].  Order statistics by
// rank counting (value v holds ranks #{x < v} .. #{x <= v} - 1); for odd T
// the middle one, for even T the two middle ones averaged exactly in fp64
// and rounded once to fp32.  -0 counts as +0; NaN inputs give NaN.
__global__ void __launch_bounds__(kOvThreads)
kvc_median_kernel(const float* __restrict__ x, int T, int H, float* __restrict__ out) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float v[kMaxSteps];
  __shared__ float s_lo, s_hi;
  const int h = blockIdx.x;
  if (threadIdx.x == 0) {
    s_lo = __int_as_float(0x7fc00000);
    s_hi = s_lo;
  }
  for (int t = threadIdx.x; t < T; t += blockDim.x) v[t] = x[(size_t)t * H + h] + 0.0f;
  __syncthreads();
  const int k_lo = (T - 1) / 2, k_hi = T / 2;
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    const float a = v[t];
    int lt = 0, le = 0;
    for (int u = 0; u < T; ++u) {
      lt += v[u] < a ? 1 : 0;
      le += v[u] <= a ? 1 : 0;
    }
    // threads holding equal values write the same value
    if (lt <= k_lo && k_lo < le) s_lo = a;
    if (lt <= k_hi && k_hi < le) s_hi = a;
  }
  __syncthreads();
  if (threadIdx.x == 0)
    out[h] = (T & 1) ? s_lo : __double2float_rn(((double)s_lo + (double)s_hi) * 0.5);
}

// One CTA per layer, one thread per head.
__global__ void kvc_budget_kernel(const double* __restrict__ s_stable, int H, int64_t total, int lo, int hi,
                                  int32_t* __restrict__ K_l, int* status) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ double s_w[kMaxHkv], s_rem[kMaxHkv];
  __shared__ int64_t s_base[kMaxHkv];
  __shared__ double s_wsum;
  __shared__ int64_t s_short;
  __shared__ int s_bad;
  const int layer = blockIdx.x, h = threadIdx.x;
  const double* s = s_stable + (size_t)layer * H;
  if (h == 0) s_bad = 0;
  __syncthreads();
  if (h < H) {
    const double x = s[h];
    if (!(x > 0.0) || !(x < INFINITY)) s_bad = 1;
    s_w[h] = __ddiv_rn(1.0, x);
  }
  __syncthreads();
  if (h == 0) {
    double wsum = 0.0;   // left to right, in head order
    for (int j = 0; j < H; ++j) wsum = __dadd_rn(wsum, s_w[j]);
    s_wsum = wsum;
  }
  __syncthreads();
  if (h < H) {
    const double exact = __ddiv_rn(__dmul_rn((double)total, s_w[h]), s_wsum);
    const double fl = floor(exact);
    s_base[h] = (int64_t)fl;
    s_rem[h] = __dsub_rn(exact, fl);
  }
  __syncthreads();
  if (h == 0) {
    int64_t assigned = 0;
    for (int j = 0; j < H; ++j) assigned += s_base[j];
    s_short = total - assigned;
  }
  __syncthreads();
  if (h < H) {
    int rank = 0;   // heads before h in (remainder descending, index ascending) order
    for (int j = 0; j < H; ++j) rank += (s_rem[j] > s_rem[h] || (s_rem[j] == s_rem[h] && j < h)) ? 1 : 0;
    int64_t v = s_base[h] + (rank < s_short ? 1 : 0);
    v = v < lo ? lo : v > hi ? hi : v;
    if (s_bad) {
      v = lo;
      if (h == 0) record_status(status, kStatusBadInput);
    }
    K_l[(size_t)layer * H + h] = (int32_t)v;
  }
}

}  // namespace

cudaError_t launch_overlap(const int32_t* a, const int64_t* a_off, const int32_t* b, const int64_t* b_off,
                           int n_pairs, float* out, cudaStream_t st) {
  cudaError_t e = launch_pdl(kvc_overlap_kernel, dim3(n_pairs), dim3(kOvThreads), 0, st, a, a_off, b, b_off, out);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_similarity(const int32_t* idx, const int64_t* off, int n_groups, int H, float* sim,
                              cudaStream_t st) {
  cudaError_t e = launch_pdl(kvc_similarity_kernel, dim3(H, n_groups), dim3(kOvThreads), 0, st, idx, off, H, sim);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_stability_steps(const int32_t* dec_idx, const int64_t* dec_off, const int32_t* pre_idx,
                                   const int64_t* pre_off, int T, int H, float* per_step, cudaStream_t st) {
  cudaError_t e = launch_pdl(kvc_stability_step_kernel, dim3(H, T), dim3(kOvThreads), 0, st, dec_idx, dec_off, pre_idx,
                             pre_off, H, per_step);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_median(const float* x, int T, int H, float* out, cudaStream_t st) {
  cudaError_t e = launch_pdl(kvc_median_kernel, dim3(H), dim3(kOvThreads), 0, st, x, T, H, out);
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_budget(const double* s_stable, int n_layers, int H, int64_t total, int lo, int hi,
                          int32_t* K_l, cudaStream_t st) {
  const int threads = (H + 31) / 32 * 32;
  cudaError_t e = launch_pdl(kvc_budget_kernel, dim3(n_layers), dim3(threads), 0, st, s_stable, H, total, lo, hi, K_l,
                             status_word_ptr());
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace kvc
