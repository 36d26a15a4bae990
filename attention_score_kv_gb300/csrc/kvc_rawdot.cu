// Single-pass raw inner-product scorer with INT8 keys (HillInfer,
// "Algorithmic Simplification" and "Streaming Execution and Asymmetric
// Precision"): rank keys by the raw product with one scoring query per KV
// head, computed in INT8 on keys cast on the fly from bf16.
//
// The scoring query of head h is the float32 sum of its group's G*W window
// queries, row by row in (g, i) order.  Every row -- that query and each key
// -- is cast to symmetric INT8: amax = max |x|, code = rint(x * (127/amax))
// clamped to [-127, 127], scale = amax / 127 (all float32, an all-zero row
// has codes 0 and scale 0).  score_j = float32(float32(dot_j) * scale_q) *
// scale_k, dot_j the exact integer product of the codes.  Each arithmetic
// step is one correctly rounded float32 operation, so the scores are
// reproducible bit for bit.
//
// Kernel 1 builds the query codes of every head; kernel 2 streams the keys
// once: D/32 lanes per key row, the row maximum by shuffles, the dot product
// by dp4a.
#include <algorithm>

#include "kvc_scan_common.cuh"

namespace kvc {
namespace {

__device__ __forceinline__ int code8(float x, float inv) {
  const int c = __float2int_rn(__fmul_rn(x, inv));
  return max(-127, min(127, c));
}

// One block per (b, KV head).  The group's G*W contiguous window rows are
// staged through shared memory in 32 KB chunks, 16-byte vectors with several
// loads in flight per thread (a per-row global load chain would leave the
// block waiting on one memory latency per row); then thread d < D sums
// column d over the chunk's rows in (g, i) order.
constexpr int kQueryThreads = 512;
constexpr int kQueryChunkVecs = 2048;      // 32 KB of rows per chunk

__global__ void __launch_bounds__(kQueryThreads)
kvc_rawdot_query_kernel(const __nv_bfloat16* __restrict__ q, int H_q, int H_kv, int W, int D,
                        int8_t* __restrict__ qcode, float* __restrict__ qscale) {
  __shared__ uint4 s_rows[kQueryChunkVecs];
  __shared__ float s_max[kQueryThreads / 32];
  grid_dep_wait();
  grid_dep_launch();
  const int bh = blockIdx.x;
  const int b = bh / H_kv, h = bh % H_kv, G = H_q / H_kv;
  const int d = threadIdx.x;
  const int vec_per_row = D / 8;
  const int chunk_rows = kQueryChunkVecs / vec_per_row;
  const int rows = G * W;
  const uint4* src = reinterpret_cast<const uint4*>(q + ((size_t)(b * H_q + h * G) * W) * D);
  const __nv_bfloat16* srow = reinterpret_cast<const __nv_bfloat16*>(s_rows);
  float acc = 0.f;
  for (int r0 = 0; r0 < rows; r0 += chunk_rows) {
    const int nvec = min(chunk_rows, rows - r0) * vec_per_row;
    const uint4* csrc = src + (size_t)r0 * vec_per_row;
#pragma unroll 4
    for (int v = threadIdx.x; v < nvec; v += kQueryThreads) s_rows[v] = __ldg(csrc + v);
    __syncthreads();
    if (d < D) {
      const int nr = nvec / vec_per_row;
      for (int r = 0; r < nr; ++r) acc = __fadd_rn(acc, __bfloat162float(srow[r * D + d]));
    }
    __syncthreads();
  }
  float a = d < D ? fabsf(acc) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((d & 31) == 0) s_max[d >> 5] = a;
  __syncthreads();
  float amax = 0.f;
  for (int w = 0; w < (D + 31) / 32; ++w) amax = fmaxf(amax, s_max[w]);
  if (d >= D) return;
  const float inv = amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f;
  qcode[(size_t)bh * D + d] = (int8_t)(amax > 0.f ? code8(acc, inv) : 0);
  if (d == 0) qscale[bh] = amax > 0.f ? __fdiv_rn(amax, 127.f) : 0.f;
}

// Key rows stream through a shared-memory ring filled by bulk copies (one
// producer thread), so the bytes in flight do not depend on the consumers'
// registers.  Each CTA owns a contiguous range of rows; a stage holds
// 32 KB of rows.  Eight consumer warps take their rows in two passes, four
// lanes per row (two at D = 64), 32 elements per lane.  Lane (row sub, c)
// reads 16-byte chunk (4i + c + sub) mod (D/8) of its row at step i: the
// eight rows of a warp then fall on distinct shared-memory bank groups.
constexpr int kRingStages = 3;          // 3 x 32 KB: two CTAs per SM
constexpr int kRingPasses = 2;          // row passes of each consumer warp per stage
constexpr int kConsumerWarps = 8;
constexpr int kRawThreads = 32 * (1 + kConsumerWarps);
template <int D>
__host__ __device__ constexpr int ring_rows() { return kConsumerWarps * (32 / (D / 32)) * kRingPasses; }   // 32 KB of rows

template <int D>
__global__ void __launch_bounds__(kRawThreads)
kvc_rawdot_score_kernel(const __nv_bfloat16* __restrict__ k, int64_t rows, int64_t per_cta, int S,
                        const int8_t* __restrict__ qcode, const float* __restrict__ qscale, float* __restrict__ scores,
                        int* status) {
  constexpr int ROWB = D * 2;              // bytes per key row
  constexpr int NCH = ROWB / 16;           // 16-byte chunks per row
  constexpr int LPR = D / 32;              // lanes per row
  constexpr int NLD = NCH / LPR;           // chunks per lane
  constexpr int kRingRows = ring_rows<D>();
  constexpr uint32_t kStageBytes = kRingRows * ROWB;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kRingStages], empty[kRingStages];
  __shared__ volatile int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRingStages; ++i) {
      tc::mbar_init(smem_u32(&full[i]), 1);
      tc::mbar_init(smem_u32(&empty[i]), kConsumerWarps);
    }
    s_abort = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  grid_dep_wait();   // the query codes come from the previous grid
  grid_dep_launch();
  const int64_t r_a = (int64_t)blockIdx.x * per_cta;
  const int64_t r_b = min(rows, r_a + per_cta);
  const int nchunks = r_a < r_b ? (int)((r_b - r_a + kRingRows - 1) / kRingRows) : 0;
  const uint32_t base = smem_u32(ring);
  if (warp == 0) {
    if (lane == 0) {
      uint32_t st = 0, ph = 0, loaded = 0, last_par = 0;
      for (int t = 0; t < nchunks; ++t) {
        if (!scan::wait_bar(smem_u32(&empty[st]), ph ^ 1u, &s_abort, status)) break;
        const int64_t r = r_a + (int64_t)t * kRingRows;
        const uint32_t bytes = (uint32_t)(min((int64_t)kRingRows, r_b - r) * ROWB);
        tc::mbar_arrive_expect_tx(smem_u32(&full[st]), bytes);
        tc::bulk_g2s(base + st * kStageBytes, k + (size_t)r * D, bytes, smem_u32(&full[st]));
        loaded |= 1u << st;
        last_par = (last_par & ~(1u << st)) | (ph << st);
        if (++st == kRingStages) { st = 0; ph ^= 1u; }
      }
      // every copy issued has landed before this thread may leave the CTA
      for (int s = 0; s < kRingStages; ++s)
        if (loaded & (1u << s)) scan::drain_wait(smem_u32(&full[s]), (last_par >> s) & 1u, status);
    }
    return;
  }
  const int w = warp - 1;
  const int sub = lane / LPR, cl = lane % LPR;
  const unsigned group_mask = ((1u << LPR) - 1u) << (sub * LPR);
  constexpr int RPW = 32 / LPR;            // rows per warp per pass
  uint32_t st = 0, ph = 0;
  for (int t = 0; t < nchunks; ++t) {
    if (!scan::wait_bar_warp(smem_u32(&full[st]), ph, &s_abort, status)) break;
    const int64_t r0 = r_a + (int64_t)t * kRingRows;
    // head of the stage's first row; a stage of kRingRows rows crosses at
    // most one head boundary when S >= kRingRows
    const int64_t h0 = r0 / S;
    const int off0 = (int)(r0 - h0 * S);
#pragma unroll
    for (int pass = 0; pass < kRingPasses; ++pass) {
      const int rr = (pass * kConsumerWarps + w) * RPW + sub;   // row within the stage
      const int64_t r = r0 + rr;
      const bool valid = r < r_b;
      const uint32_t rowaddr = base + st * kStageBytes + rr * ROWB;
      uint4 raw[NLD];
      int chs[NLD];
#pragma unroll
      for (int i = 0; i < NLD; ++i) {
        chs[i] = (i * LPR + cl + sub) % NCH;
        raw[i] = make_uint4(0u, 0u, 0u, 0u);
        if (valid)
          asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                       : "=r"(raw[i].x), "=r"(raw[i].y), "=r"(raw[i].z), "=r"(raw[i].w)
                       : "r"(rowaddr + chs[i] * 16));
      }
      const int within = off0 + (valid ? rr : 0);
      const int bh = (int)h0 + (S >= kRingRows ? (within >= S ? 1 : 0) : within / S);
      // max |x| on bf16 pairs: exact, and the same value as in float32
      __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
#pragma unroll
      for (int i = 0; i < NLD; ++i) {
        const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw[i]);
#pragma unroll
        for (int e = 0; e < 4; ++e) m2 = __hmax2(m2, __habs2(p2[e]));
      }
      float a = fmaxf(__low2float(m2), __high2float(m2));
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(group_mask, a, o));
      // |x| <= a and inv = fl(127/a), so y = fl(x * inv) has |y| < 127.5 and
      // rint stays in [-127, 127] without a clamp.  rint(y) is taken by
      // adding 1.5 * 2^23 in float32: the sum lies in [2^23, 2^24), where the
      // spacing is 1, so round-to-nearest-even leaves y + 1.5 * 2^23 rounded
      // to an integer with ties to even (1.5 * 2^23 is even), and the low
      // byte of the sum's bit pattern is rint(y) mod 256, the code's
      // two's-complement byte.
      // The product and the sum are separate round-to-nearest intrinsics,
      // which are never merged into a fused multiply-add.  (The packed
      // f32x2 forms gave the codes of a single rounding on the GPU, so they
      // are not used here.)
      const float inv = a > 0.f ? __fdiv_rn(127.f, a) : 0.f;
      int dot = 0;
#pragma unroll
      for (int i = 0; i < NLD; ++i) {
        const uint32_t* wd = reinterpret_cast<const uint32_t*>(&raw[i]);
        uint32_t c[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          c[2 * e] = __float_as_uint(__fadd_rn(__fmul_rn(__uint_as_float(wd[e] << 16), inv), 12582912.f));
          c[2 * e + 1] = __float_as_uint(__fadd_rn(__fmul_rn(__uint_as_float(wd[e] & 0xffff0000u), inv), 12582912.f));
        }
        const int kp0 = (int)__byte_perm(__byte_perm(c[0], c[1], 0x0040), __byte_perm(c[2], c[3], 0x0040), 0x5410);
        const int kp1 = (int)__byte_perm(__byte_perm(c[4], c[5], 0x0040), __byte_perm(c[6], c[7], 0x0040), 0x5410);
        const int2 qp = *reinterpret_cast<const int2*>(qcode + (size_t)bh * D + chs[i] * 8);
        dot = __dp4a(kp0, qp.x, dot);
        dot = __dp4a(kp1, qp.y, dot);
      }
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(group_mask, dot, o);
      if (cl == 0 && valid) {
        const float sk = a > 0.f ? __fdiv_rn(a, 127.f) : 0.f;
        scores[r] = __fmul_rn(__fmul_rn((float)dot, qscale[bh]), sk);
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(smem_u32(&empty[st]));
    if (++st == kRingStages) { st = 0; ph ^= 1u; }
  }
}

}  // namespace

cudaError_t launch_rawdot_int8(const __nv_bfloat16* q, const __nv_bfloat16* k, int B, int H_q, int H_kv, int S,
                               int D, int W, int8_t* qcode, float* qscale, float* scores, cudaStream_t st) {
  const int BH = B * H_kv;
  cudaError_t e = launch_pdl(kvc_rawdot_query_kernel, dim3(BH), dim3(kQueryThreads), 0, st, q, H_q, H_kv, W, D,
                             qcode, qscale);
  note_launches(1);
  if (e != cudaSuccess) return e;
  const int64_t rows = (int64_t)BH * S;
  const int ctas = std::max(1, num_sms() * 2);
  const int64_t per_cta = (rows + ctas - 1) / ctas;
  const size_t smem = (size_t)kRingStages * (D == 64 ? ring_rows<64>() : ring_rows<128>()) * D * 2;
  const int grid = (int)((rows + per_cta - 1) / per_cta);
  if (D == 64) {
    if ((e = cudaFuncSetAttribute(kvc_rawdot_score_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
      return e;
    e = launch_pdl(kvc_rawdot_score_kernel<64>, dim3(grid), dim3(kRawThreads), smem, st, k, rows, per_cta, S, qcode,
                   qscale, scores, status_word_ptr());
  } else {
    if ((e = cudaFuncSetAttribute(kvc_rawdot_score_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
      return e;
    e = launch_pdl(kvc_rawdot_score_kernel<128>, dim3(grid), dim3(kRawThreads), smem, st, k, rows, per_cta, S, qcode,
                   qscale, scores, status_word_ptr());
  }
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvc
