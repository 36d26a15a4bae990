// Two-pass blockwise scorer (TideKV, Fig. 3) on warp-level bf16 MMA.
//
// Pass 1: each CTA owns one key range of one (b, KV head), streams its keys
// in 128-key tiles through shared memory (double-buffered async copies) and
// keeps per window-query running (max, sum-of-exp) in the log2 domain.  Only
// G*W values of state survive the range: m2 = max_j x_j and
// Z = sum_j 2^(x_j - m2), with x_j = (q . k_j) * log2(e) / sqrt(D).
//
// Pass 2: each CTA rescans its key range (plus (pool_k-1)/2 halo keys on each
// side), forms the normalised weights 2^(x - lse2) with
// lse2 = m2 + log2(Z), sums them over all G*W window rows of the group in
// registers (each thread owns keys, the query axis runs along the MMA N
// dimension), average-pools the per-key masses and either writes the scores
// or appends the non-mandatory keys to the range's candidate list.
#include <cfloat>
#include <climits>

#include "kvc_device.cuh"
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
__device__ __forceinline__ void load_q(uint32_t sQ, const __nv_bfloat16* qsrc, int gw, int gwp) {
  constexpr int CPR = D / 8;
  for (int c = threadIdx.x; c < gwp * CPR; c += blockDim.x) {
    const int row = c / CPR, ch = c % CPR;
    const __nv_bfloat16* src = qsrc + (size_t)min(row, gw - 1) * D + ch * 8;
    cp_async16(sQ + swz<D>(row, ch), src, row < gw ? 16 : 0);
  }
}

template <int D>
__device__ __forceinline__ void load_k(uint32_t sK, const __nv_bfloat16* kbase, int S, int t0) {
  constexpr int CPR = D / 8;
  for (int c = threadIdx.x; c < kTile * CPR; c += blockDim.x) {
    const int row = c / CPR, ch = c % CPR;
    const int j = t0 + row;
    const bool ok = (j >= 0) && (j < S);
    const __nv_bfloat16* src = kbase + (size_t)(ok ? j : 0) * D + ch * 8;
    cp_async16(sK + swz<D>(row, ch), src, ok ? 16 : 0);
  }
}

// Merge (m, z) pairs of the log2-domain online normaliser.
__device__ __forceinline__ float2 merge_mz(float2 a, float2 b) {
  if (b.y == 0.f) return a;
  if (a.y == 0.f) return b;
  const float m = fmaxf(a.x, b.x);
  return make_float2(m, a.y * ex2(a.x - m) + b.y * ex2(b.x - m));
}

// ------------------------------------------------------------------ pass 1
template <int D, int KS>
__global__ void __launch_bounds__(kThreads)
kvc_pass1_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
             int H_q, int H_kv, int S, int W, int nparts, int gwp, float c2,
             float* __restrict__ part_m, float* __restrict__ part_z) {
  constexpr int NT = 16 / KS;      // 8-key MMA tiles per work unit
  constexpr int KEYS = kTile / KS; // keys per work unit
  const int p = blockIdx.x, bh = blockIdx.y;
  const int b = bh / H_kv, h = bh % H_kv;
  const int G = H_q / H_kv, gw = G * W, n_rb = gwp / 16;
  const int R = ((S + nparts - 1) / nparts + kTile - 1) / kTile * kTile;
  const int a = p * R, e = min(S, a + R);
  float* pm = part_m + ((size_t)bh * nparts + p) * gwp;
  float* pz = part_z + ((size_t)bh * nparts + p) * gwp;
  if (a >= e) {
    for (int i = threadIdx.x; i < gwp; i += blockDim.x) { pm[i] = -INFINITY; pz[i] = 0.f; }
    return;
  }
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sK = smem + (size_t)gwp * D * 2;
  float2* stage = reinterpret_cast<float2*>(sK + 2 * kTile * D * 2);  // [n_rb*KS][16]
  float2* run = stage + n_rb * KS * 16;                               // [gwp]

  const __nv_bfloat16* qsrc = q + (size_t)(b * H_q + h * G) * W * D;
  const __nv_bfloat16* kbase = k + (size_t)bh * S * D;
  load_q<D>(smem_u32(sQ), qsrc, gw, gwp);
  load_k<D>(smem_u32(sK), kbase, S, a);
  cp_async_commit();
  for (int i = threadIdx.x; i < gwp; i += blockDim.x) run[i] = make_float2(-INFINITY, 0.f);

  const int ntiles = (e - a + kTile - 1) / kTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int units = n_rb * KS;
  const uint32_t qb = smem_u32(sQ);
  for (int t = 0; t < ntiles; ++t) {
    const int t0 = a + t * kTile;
    cp_async_wait_all();
    __syncthreads();
    if (t + 1 < ntiles) {
      load_k<D>(smem_u32(sK + ((t + 1) & 1) * kTile * D * 2), kbase, S, t0 + kTile);
      cp_async_commit();
    }
    const uint32_t kb = smem_u32(sK + (t & 1) * kTile * D * 2);
    const bool need_mask = (t0 + kTile - 1 > S - W);
    for (int u = warp; u < units; u += kThreads / 32) {
      const int rb = u / KS, ks = u % KS;
      float acc[NT][4];
#pragma unroll
      for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t af[4];
        ldsm_x4(qb + swz<D>(rb * 16 + (lane & 15), 2 * kk + (lane >> 4)), af[0], af[1], af[2], af[3]);
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          const int n0 = ks * KEYS + np * 16;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + swz<D>(n0 + ((lane >> 4) << 3) + (lane & 7), 2 * kk + ((lane >> 3) & 1)), b0, b1, b2, b3);
          mma_bf16(acc[2 * np], af, b0, b1);
          mma_bf16(acc[2 * np + 1], af, b2, b3);
        }
      }
      const int r0 = rb * 16 + (lane >> 2), r1 = r0 + 8;
      const int tq0 = S - W + (r0 % W), tq1 = S - W + (r1 % W);
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e2 = 0; e2 < 2; ++e2) {
          const int j = t0 + ks * KEYS + nt * 8 + 2 * (lane & 3) + e2;
          float x0 = acc[nt][e2] * c2, x1 = acc[nt][2 + e2] * c2;
          if (need_mask) {
            if (j > tq0) x0 = -INFINITY;
            if (j > tq1) x1 = -INFINITY;
          }
          acc[nt][e2] = x0;
          acc[nt][2 + e2] = x1;
          mx0 = fmaxf(mx0, x0);
          mx1 = fmaxf(mx1, x1);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      float z0 = 0.f, z1 = 0.f;
      if (mx0 > -INFINITY) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) z0 += ex2(acc[nt][0] - mx0) + ex2(acc[nt][1] - mx0);
      }
      if (mx1 > -INFINITY) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) z1 += ex2(acc[nt][2] - mx1) + ex2(acc[nt][3] - mx1);
      }
      z0 += __shfl_xor_sync(0xffffffffu, z0, 1);
      z0 += __shfl_xor_sync(0xffffffffu, z0, 2);
      z1 += __shfl_xor_sync(0xffffffffu, z1, 1);
      z1 += __shfl_xor_sync(0xffffffffu, z1, 2);
      if ((lane & 3) == 0) {
        stage[(rb * KS + ks) * 16 + (lane >> 2)] = make_float2(mx0, z0);
        stage[(rb * KS + ks) * 16 + (lane >> 2) + 8] = make_float2(mx1, z1);
      }
    }
    __syncthreads();
    for (int qq = threadIdx.x; qq < gwp; qq += blockDim.x) {
      const int rb = qq >> 4, rr = qq & 15;
      float2 st = run[qq];
      for (int ks = 0; ks < KS; ++ks) st = merge_mz(st, stage[(rb * KS + ks) * 16 + rr]);
      run[qq] = st;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < gwp; i += blockDim.x) {
    pm[i] = run[i].x;
    pz[i] = run[i].y;
  }
}

// Combine the per-range partials of pass 1 into m, Z (natural-log units).
__global__ void kvc_pass1_combine_kernel(const float* __restrict__ part_m, const float* __restrict__ part_z,
                                     int H_q, int H_kv, int W, int nparts, int gwp,
                                     float* __restrict__ m, float* __restrict__ Z) {
  const int bh = blockIdx.x;
  const int b = bh / H_kv, h = bh % H_kv, G = H_q / H_kv;
  for (int qq = threadIdx.x; qq < G * W; qq += blockDim.x) {
    float2 st = make_float2(-INFINITY, 0.f);
    for (int p = 0; p < nparts; ++p) {
      const size_t o = ((size_t)bh * nparts + p) * gwp + qq;
      st = merge_mz(st, make_float2(part_m[o], part_z[o]));
    }
    const size_t dst = (size_t)(b * H_q + h * G) * W + qq;
    m[dst] = st.x / kLog2e;
    Z[dst] = st.y;
  }
}

// --------------------------------------------------------- candidate lists
__device__ __forceinline__ uint64_t rank_key(uint64_t e) {
  // (score bits, ~index): larger is better, the lower index wins a score tie
  return (e & 0xFFFFFFFF00000000ull) | (uint64_t)(~(uint32_t)e);
}

struct CompactSmem {
  int hist[256];
  int scan[32];
  int need, full;
  unsigned long long prefix;
};

// Keep the n_keep best entries of buf[0..cnt) (in place, order preserved) and
// return the filter threshold for later, higher-index entries: an entry with
// score bits u is worth appending only if u > tau.
__device__ void cta_compact(uint64_t* buf, int cnt, int n_keep, CompactSmem* cs,
                            int* s_cnt, long long* s_tau, int* status) {
  const int tid = threadIdx.x;
  if (n_keep <= 0) {
    if (tid == 0) { *s_cnt = 0; *s_tau = LLONG_MAX; }
    __syncthreads();
    return;
  }
  unsigned long long prefix = 0;
  int need = n_keep;
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += blockDim.x) cs->hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < cnt; i += blockDim.x) {
      const uint64_t key = rank_key(buf[i]);
      if (shift == 56 || (key >> (shift + 8)) == (prefix >> (shift + 8)))
        atomicAdd(&cs->hist[(key >> shift) & 255], 1);
    }
    __syncthreads();
    if (tid == 0) {
      int cum = 0, d = 255;
      for (; d > 0; --d) {
        if (cum + cs->hist[d] >= need) break;
        cum += cs->hist[d];
      }
      cs->need = need - cum;
      cs->full = (need - cum == cs->hist[d]);
      cs->prefix = prefix | ((unsigned long long)d << shift);
    }
    __syncthreads();
    need = cs->need;
    prefix = cs->prefix;
    const int full = cs->full;
    __syncthreads();
    if (full) break;
  }
  const uint64_t T = prefix;
  int out = 0;
  for (int base = 0; base < cnt; base += blockDim.x) {
    const int i = base + tid;
    const uint64_t e = i < cnt ? buf[i] : 0ull;
    const int f = (i < cnt && rank_key(e) >= T) ? 1 : 0;
    int tot;
    const int incl = block_inclusive_scan(f, cs->scan, &tot);
    if (f) buf[out + incl - 1] = e;
    out += tot;
    __syncthreads();
  }
  if (tid == 0) {
    if (out != n_keep) record_status(status, kStatusCandOverflow);
    *s_cnt = out;
    *s_tau = (long long)(T >> 32);
  }
  __syncthreads();
}

// ------------------------------------------------------------------ pass 2
template <int D, bool CAND>
__global__ void __launch_bounds__(kThreads)
kvc_pass2_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
             const float* __restrict__ m, const float* __restrict__ Z,
             const float* __restrict__ part_m, const float* __restrict__ part_z,
             int H_q, int H_kv, int S, int W, int pool_k, int nparts, int gwp, float c2,
             float* __restrict__ scores, uint64_t* __restrict__ cand, int* __restrict__ cand_cnt,
             int cap, const __grid_constant__ SelParams sel, int* status) {
  const int p = blockIdx.x, bh = blockIdx.y;
  const int b = bh / H_kv, h = bh % H_kv;
  const int G = H_q / H_kv, gw = G * W;
  const int hw = (pool_k - 1) / 2;
  const int R = (S + nparts - 1) / nparts;
  const int a = p * R, e = min(S, a + R);
  if (a >= e) {
    if (CAND && threadIdx.x == 0) cand_cnt[(size_t)bh * nparts + p] = 0;
    return;
  }
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sQ = smem;
  uint8_t* sK = smem + (size_t)gwp * D * 2;
  float* lse2 = reinterpret_cast<float*>(sK + 2 * kTile * D * 2);   // [gwp]
  float* rbuf = lse2 + gwp;                                         // [2*hw + kTile]
  __shared__ CompactSmem cs;
  __shared__ int s_wtot[kThreads / 32];
  __shared__ int s_cnt;
  __shared__ long long s_tau;

  const __nv_bfloat16* qsrc = q + (size_t)(b * H_q + h * G) * W * D;
  const __nv_bfloat16* kbase = k + (size_t)bh * S * D;
  load_q<D>(smem_u32(sQ), qsrc, gw, gwp);
  load_k<D>(smem_u32(sK), kbase, S, a - hw);
  cp_async_commit();

  for (int qq = threadIdx.x; qq < gwp; qq += blockDim.x) {
    float l = INFINITY;
    if (qq < gw) {
      if (m != nullptr) {
        const size_t src = (size_t)(b * H_q + h * G) * W + qq;
        l = m[src] * kLog2e + log2f(Z[src]);
      } else {
        float2 st = make_float2(-INFINITY, 0.f);
        for (int pp = 0; pp < nparts; ++pp) {
          const size_t o = ((size_t)bh * nparts + pp) * gwp + qq;
          st = merge_mz(st, make_float2(part_m[o], part_z[o]));
        }
        l = st.x + log2f(st.y);
      }
    }
    lse2[qq] = l;
  }
  for (int i = threadIdx.x; i < 2 * hw; i += blockDim.x) rbuf[i] = 0.f;
  if (threadIdx.x == 0) { s_cnt = 0; s_tau = -1; }

  uint64_t* my_cand = CAND ? cand + ((size_t)bh * nparts + p) * cap : nullptr;
  const int n_keep = CAND ? sel.n_sel[h] : 0;
  const float inv_pool = 1.0f / (float)pool_k;
  const int n_iter = (e - a + 2 * hw + kTile - 1) / kTile;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_nt = gwp / 8;
  const uint32_t qb = smem_u32(sQ);
  float* rtile = rbuf + 2 * hw;

  for (int it = 0; it < n_iter; ++it) {
    const int t0 = a - hw + it * kTile;
    cp_async_wait_all();
    __syncthreads();
    if (it + 1 < n_iter) {
      load_k<D>(smem_u32(sK + ((it + 1) & 1) * kTile * D * 2), kbase, S, t0 + kTile);
      cp_async_commit();
    }
    const uint32_t kb = smem_u32(sK + (it & 1) * kTile * D * 2);
    uint32_t af[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      ldsm_x4(kb + swz<D>(warp * 16 + (lane & 15), 2 * kk + (lane >> 4)), af[kk][0], af[kk][1], af[kk][2], af[kk][3]);
    const int j0 = t0 + warp * 16 + (lane >> 2), j1 = j0 + 8;
    const bool need_mask = (t0 + kTile - 1 > S - W);
    float r0 = 0.f, r1 = 0.f;
    for (int c0 = 0; c0 < n_nt; c0 += 8) {
      float acc[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int nt = c0 + 2 * np;
          if (nt < n_nt) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(qb + swz<D>(nt * 8 + ((lane >> 4) << 3) + (lane & 7), 2 * kk + ((lane >> 3) & 1)), b0, b1, b2, b3);
            mma_bf16(acc[2 * np], af[kk], b0, b1);
            mma_bf16(acc[2 * np + 1], af[kk], b2, b3);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int nt = c0 + t;
        if (nt < n_nt) {
          const int col = nt * 8 + 2 * (lane & 3);
          const float la = lse2[col], lb = lse2[col + 1];
          const float e00 = ex2(fmaf(acc[t][0], c2, -la));
          const float e01 = ex2(fmaf(acc[t][1], c2, -lb));
          const float e10 = ex2(fmaf(acc[t][2], c2, -la));
          const float e11 = ex2(fmaf(acc[t][3], c2, -lb));
          if (!need_mask) {
            r0 += e00 + e01;
            r1 += e10 + e11;
          } else {
            const int ta = S - W + (col % W), tb = S - W + ((col + 1) % W);
            r0 += (j0 <= ta ? e00 : 0.f) + (j0 <= tb ? e01 : 0.f);
            r1 += (j1 <= ta ? e10 : 0.f) + (j1 <= tb ? e11 : 0.f);
          }
        }
      }
    }
    r0 += __shfl_xor_sync(0xffffffffu, r0, 1);
    r0 += __shfl_xor_sync(0xffffffffu, r0, 2);
    r1 += __shfl_xor_sync(0xffffffffu, r1, 1);
    r1 += __shfl_xor_sync(0xffffffffu, r1, 2);
    if ((lane & 3) == 0) {
      rtile[warp * 16 + (lane >> 2)] = (j0 >= 0 && j0 < S) ? r0 : 0.f;
      rtile[warp * 16 + (lane >> 2) + 8] = (j1 >= 0 && j1 < S) ? r1 : 0.f;
    }
    __syncthreads();

    // pooled scores of keys t0 - hw + tid
    const int j = t0 - hw + (int)threadIdx.x;
    const bool valid = threadIdx.x < kTile && j >= a && j < e;
    float s = 0.f;
    if (threadIdx.x < kTile) {
      for (int d = 0; d <= 2 * hw; ++d) s += rbuf[threadIdx.x + d];
      s = (pool_k == 1) ? s : s * inv_pool;
    }
    if (!CAND) {
      if (valid) scores[(size_t)bh * S + j] = s;
    } else {
      uint32_t u = __float_as_uint(s);
      if (u == 0x80000000u) u = 0u;
      const bool is_cand = valid && j >= sel.r_lo && j < sel.r_hi;
      for (int tries = 0;; ++tries) {
        const bool flag = is_cand && (long long)u > s_tau;
        const unsigned bal = __ballot_sync(0xffffffffu, flag);
        if (lane == 0) s_wtot[warp] = __popc(bal);
        __syncthreads();
        int tot = 0, before = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) {
          before += (w < warp) ? s_wtot[w] : 0;
          tot += s_wtot[w];
        }
        const int base = s_cnt;
        if (base + tot > cap) {
          if (base <= n_keep || tries >= 2) {  // cannot happen when cap >= n_keep + kTile
            record_status(status, kStatusCandOverflow);
            break;
          }
          __syncthreads();
          cta_compact(my_cand, base, n_keep, &cs, &s_cnt, &s_tau, status);
          continue;
        }
        if (flag) {
          const int pos = base + before + __popc(bal & ((1u << lane) - 1u));
          my_cand[pos] = ((uint64_t)u << 32) | (uint32_t)j;
        }
        __syncthreads();
        if (threadIdx.x == 0) s_cnt = base + tot;
        break;
      }
    }
    __syncthreads();
    if (threadIdx.x < 2 * hw) rbuf[threadIdx.x] = rtile[kTile - 2 * hw + threadIdx.x];
  }
  if (CAND) {
    __syncthreads();
    if (threadIdx.x == 0) cand_cnt[(size_t)bh * nparts + p] = s_cnt;
  }
}

template <int D, int KS>
cudaError_t run_pass1(dim3 grid, size_t smem, cudaStream_t st, const __nv_bfloat16* q,
                      const __nv_bfloat16* k, int H_q, int H_kv, int S, int W, int nparts,
                      int gwp, float c2, float* pm, float* pz) {
  cudaError_t e = cudaFuncSetAttribute(kvc_pass1_kernel<D, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kvc_pass1_kernel<D, KS><<<grid, kThreads, smem, st>>>(q, k, H_q, H_kv, S, W, nparts, gwp, c2, pm, pz);
  note_launches(1);
  return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_pass1(int KS, dim3 grid, size_t smem, cudaStream_t st, const __nv_bfloat16* q,
                           const __nv_bfloat16* k, int H_q, int H_kv, int S, int W, int nparts,
                           int gwp, float c2, float* pm, float* pz) {
  switch (KS) {
    case 1: return run_pass1<D, 1>(grid, smem, st, q, k, H_q, H_kv, S, W, nparts, gwp, c2, pm, pz);
    case 2: return run_pass1<D, 2>(grid, smem, st, q, k, H_q, H_kv, S, W, nparts, gwp, c2, pm, pz);
    case 4: return run_pass1<D, 4>(grid, smem, st, q, k, H_q, H_kv, S, W, nparts, gwp, c2, pm, pz);
    default: return run_pass1<D, 8>(grid, smem, st, q, k, H_q, H_kv, S, W, nparts, gwp, c2, pm, pz);
  }
}

template <int D, bool CAND>
cudaError_t run_pass2(dim3 grid, size_t smem, cudaStream_t st, const __nv_bfloat16* q,
                      const __nv_bfloat16* k, const float* m, const float* Z, const float* pm,
                      const float* pz, int H_q, int H_kv, int S, int W, int pool_k, int nparts,
                      int gwp, float c2, const SelParams* sel, Pass2Out out) {
  cudaError_t e = cudaFuncSetAttribute(kvc_pass2_kernel<D, CAND>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kvc_pass2_kernel<D, CAND><<<grid, kThreads, smem, st>>>(q, k, m, Z, pm, pz, H_q, H_kv, S, W, pool_k, nparts, gwp,
                                                       c2, out.scores, out.cand, out.cand_cnt, out.cap, *sel,
                                                       status_word_ptr());
  note_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pass1(const __nv_bfloat16* q, const __nv_bfloat16* k, int B, int H_q, int H_kv,
                         int S, int D, int W, int nparts, int gwp, float* part_m, float* part_z,
                         cudaStream_t st) {
  const int n_rb = gwp / 16;
  int g = 8;
  while (g > 1 && (n_rb % g) != 0) g >>= 1;
  const int KS = 8 / g;
  const size_t smem = (size_t)gwp * D * 2 + 2 * (size_t)kTile * D * 2 + (size_t)n_rb * KS * 16 * 8 + (size_t)gwp * 8;
  const float c2 = 1.4426950408889634f / sqrtf((float)D);
  dim3 grid(nparts, B * H_kv);
  if (D == 64) return dispatch_pass1<64>(KS, grid, smem, st, q, k, H_q, H_kv, S, W, nparts, gwp, c2, part_m, part_z);
  return dispatch_pass1<128>(KS, grid, smem, st, q, k, H_q, H_kv, S, W, nparts, gwp, c2, part_m, part_z);
}

cudaError_t launch_pass1_combine(const float* part_m, const float* part_z, int B, int H_q, int H_kv,
                                 int W, int D, int nparts, int gwp, int S, float* m, float* Z,
                                 cudaStream_t st) {
  (void)D;
  (void)S;
  kvc_pass1_combine_kernel<<<B * H_kv, 256, 0, st>>>(part_m, part_z, H_q, H_kv, W, nparts, gwp, m, Z);
  note_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_pass2(const __nv_bfloat16* q, const __nv_bfloat16* k, const float* m, const float* Z,
                         const float* part_m, const float* part_z, int B, int H_q, int H_kv, int S,
                         int D, int W, int pool_k, int nparts, int gwp, const SelParams* sel,
                         Pass2Out out, cudaStream_t st) {
  const int hw = (pool_k - 1) / 2;
  const size_t smem = (size_t)gwp * D * 2 + 2 * (size_t)kTile * D * 2 + (size_t)gwp * 4 +
                      (size_t)(2 * hw + kTile) * 4;
  const float c2 = 1.4426950408889634f / sqrtf((float)D);
  dim3 grid(nparts, B * H_kv);
  const bool cand = out.cand != nullptr;
  if (D == 64) {
    return cand ? run_pass2<64, true>(grid, smem, st, q, k, m, Z, part_m, part_z, H_q, H_kv, S, W, pool_k, nparts, gwp, c2, sel, out)
                : run_pass2<64, false>(grid, smem, st, q, k, m, Z, part_m, part_z, H_q, H_kv, S, W, pool_k, nparts, gwp, c2, sel, out);
  }
  return cand ? run_pass2<128, true>(grid, smem, st, q, k, m, Z, part_m, part_z, H_q, H_kv, S, W, pool_k, nparts, gwp, c2, sel, out)
              : run_pass2<128, false>(grid, smem, st, q, k, m, Z, part_m, part_z, H_q, H_kv, S, W, pool_k, nparts, gwp, c2, sel, out);
}

}  // namespace kvc
