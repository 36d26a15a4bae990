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
// Kernel 1 sums every head's window rows; kernel 2 streams the keys once
// (one lane per key row, the dot product by dp4a), after forming the query
// codes of the heads its range touches.
#include <algorithm>

#include "kvc_scan_common.cuh"

namespace kvc {
namespace {

__device__ __forceinline__ int code8(float x, float inv) {
  const int c = __float2int_rn(__fmul_rn(x, inv));
  return max(-127, min(127, c));
}

// The scoring query's float32 column sums.  Block (b*H_kv + h, cg) sums
// columns 8*cg .. 8*cg + 7 of the group's G*W contiguous window rows: each
// thread stages one row's 16-byte slice in shared memory (one load latency
// for the whole block), then thread c < 8 adds column 8*cg + c over the rows
// in (g, i) order.  The codes are formed by the scorer, per CTA, from these
// sums.
constexpr int kQsumThreads = 256;

__global__ void __launch_bounds__(kQsumThreads)
kvc_rawdot_qsum_kernel(const __nv_bfloat16* __restrict__ q, int H_q, int H_kv, int W, int D,
                       float* __restrict__ qsum) {
  __shared__ uint4 s_rows[kQsumThreads];
  grid_dep_wait();
  grid_dep_launch();
  const int bh = blockIdx.x, cg = blockIdx.y;
  const int b = bh / H_kv, h = bh % H_kv, G = H_q / H_kv;
  const int rows = G * W;
  const __nv_bfloat16* src = q + ((size_t)(b * H_q + h * G) * W) * D + cg * 8;
  const int c = threadIdx.x;
  float acc = 0.f;
  for (int r0 = 0; r0 < rows; r0 += kQsumThreads) {
    const int nr = min(kQsumThreads, rows - r0);
    if (c < nr) s_rows[c] = __ldg(reinterpret_cast<const uint4*>(src + (size_t)(r0 + c) * D));
    __syncthreads();
    if (c < 8) {
      // 16 loads in flight, then the ordered adds
      const __nv_bfloat16* sv = reinterpret_cast<const __nv_bfloat16*>(s_rows);
      int r = 0;
      for (; r + 16 <= nr; r += 16) {
        float v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) v[u] = __bfloat162float(sv[(r + u) * 8 + c]);
#pragma unroll
        for (int u = 0; u < 16; ++u) acc = __fadd_rn(acc, v[u]);
      }
      for (; r < nr; ++r) acc = __fadd_rn(acc, __bfloat162float(sv[r * 8 + c]));
    }
    __syncthreads();
  }
  if (c < 8) qsum[(size_t)bh * D + cg * 8 + c] = acc;
}

// Key rows stream through a shared-memory ring filled by bulk copies (one
// producer thread), so the bytes in flight do not depend on the consumers'
// registers.  Each CTA (one per SM) owns a contiguous range of rows; a stage
// holds 128 rows, cut into blocks of 32.  Consumer warp w takes blocks w,
// w + 12, w + 24, ... of the CTA's range, one lane per row: the per-row work
// (maximum, the two divisions, the store) then costs one instruction per 32
// rows.  A lane loads its whole row into registers and hands the block back
// at once, so a stage is held only for the loads and the ring's bytes stay
// in flight while the rows are quantised.  At step j a lane reads 16-byte
// chunk (j + lane) mod (D/8) of its row, so the 32 rows of a block spread
// evenly over the bank groups.
//
// Measured at Mistral 128K: four lanes per row took 43 warp-instructions
// per row; one lane per row reading the row twice from shared memory, 32;
// and with a stage held until its rows were scored, the consumers held
// nearly the whole ring, so the stream ran near 5 TB/s.
//
// A warp waits on the full barrier of each stage it takes with the stage's
// phase parity.  Warp w's next block lies W blocks on, W = kConsumerWarps;
// when W is at most the number of block slots in the ring (kRingStages *
// kBlocks), the slot's previous stage is one this warp has already seen
// loaded, so the parity cannot name an earlier phase of the same parity.
constexpr int kRingStages = 6;          // 6 x 32 KB at D = 128: one CTA per SM
constexpr int kBlocks = 4;              // 32-row blocks per stage
constexpr int kRingRows = 32 * kBlocks;
constexpr int kRawCtasPerSm = 1;
constexpr int kConsumerWarps = 12;
static_assert(kConsumerWarps <= kRingStages * kBlocks, "a consumer warp could run two phases ahead of a slot");
constexpr int kRawThreads = 32 * (1 + kConsumerWarps);
// The query codes and scales of the heads a CTA's range touches are staged
// in shared memory; the launcher sizes the grid so that a range spans at
// most 15*S rows, hence at most 16 heads.
constexpr int kMaxQHeads = 16;
constexpr int kMaxRangeHeads = kMaxQHeads - 1;

template <int D>
__global__ void __launch_bounds__(kRawThreads, kRawCtasPerSm)
kvc_rawdot_score_kernel(const __nv_bfloat16* __restrict__ k, int64_t rows, int64_t per_cta, int S,
                        const float* __restrict__ qsum, float* __restrict__ scores, int* status) {
  constexpr int ROWB = D * 2;                      // bytes per key row
  constexpr int NCH = ROWB / 16;                   // 16-byte chunks per row
  constexpr uint32_t kStageBytes = kRingRows * ROWB;
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kRingStages], empty[kRingStages];
  __shared__ __align__(16) int8_t s_qc[kMaxQHeads * D];
  __shared__ float s_qs[kMaxQHeads];
  __shared__ float s_red[kConsumerWarps];
  __shared__ volatile int s_abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRingStages; ++i) {
      tc::mbar_init(smem_u32(&full[i]), 1);
      tc::mbar_init(smem_u32(&empty[i]), kBlocks);
    }
    s_abort = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  // The producer streams keys at once: the column-sum kernel this one
  // depends on waits for its own predecessor before it lets this grid start,
  // so every earlier write to k has landed.  Only the consumers wait for the
  // column sums.
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
  grid_dep_wait();   // the column sums come from the previous grid
  const int w = warp - 1;
  const int nblk = r_a < r_b ? (int)((r_b - r_a + 31) / 32) : 0;
  const int h_first = (int)(r_a / S);
  // at most kMaxQHeads by the launcher's grid; the clamps only keep every
  // shared-memory access in bounds
  const int nh = min(kMaxQHeads, r_a < r_b ? (int)((r_b - 1) / S) - h_first + 1 : 0);
  {
    // query codes and scales of heads h_first .. h_first + nh - 1, from
    // their column sums: D threads per head, kConsumerWarps * 32 / D heads
    // at a time; the maximum over a head's D columns goes through s_red
    constexpr int kHeadsPar = kConsumerWarps * 32 / D;
    constexpr int kWarpsPerHead = D / 32;
    const int tid = threadIdx.x - 32;
    const int slot = tid / D, d = tid % D;
    for (int hb = 0; hb < nh; hb += kHeadsPar) {
      const int hh = hb + slot;
      const bool act = hh < nh;
      // written by the previous grid while this one ran: a load through L2,
      // not the read-only path
      const float acc = act ? __ldcg(qsum + (size_t)(h_first + hh) * D + d) : 0.f;
      float am = fabsf(acc);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
      if (lane == 0) s_red[w] = am;
      asm volatile("bar.sync 1, %0;\n" ::"n"(kConsumerWarps * 32) : "memory");
      if (act) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < kWarpsPerHead; ++i) amax = fmaxf(amax, s_red[slot * kWarpsPerHead + i]);
        const float inv = amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f;
        s_qc[hh * D + d] = (int8_t)(amax > 0.f ? code8(acc, inv) : 0);
        if (d == 0) s_qs[hh] = amax > 0.f ? __fdiv_rn(amax, 127.f) : 0.f;
      }
      asm volatile("bar.sync 1, %0;\n" ::"n"(kConsumerWarps * 32) : "memory");   // consumer warps only
    }
  }
  const uint32_t qbase = smem_u32(s_qc);
  // (h0, off0): head and in-head offset of the warp's current block start,
  // advanced by 32 * kConsumerWarps rows per block
  int64_t rb0 = r_a + (int64_t)w * 32;
  int h0 = (int)(rb0 / S);
  int off0 = (int)(rb0 - (int64_t)h0 * S);
  for (int g = w; g < nblk; g += kConsumerWarps) {
    const int t = g / kBlocks;
    const uint32_t st = (uint32_t)(t % kRingStages), ph = (uint32_t)((t / kRingStages) & 1);
    if (!scan::wait_bar_warp(smem_u32(&full[st]), ph, &s_abort, status)) break;
    const int64_t r = r_a + (int64_t)g * 32 + lane;
    const bool valid = r < r_b;
    // rows past the range end read stale stage bytes; their result is dropped
    const uint32_t rowaddr = base + st * kStageBytes + ((g % kBlocks) * 32 + lane) * ROWB;
    // lanes past the range end take the head of the block's last row, so
    // every query-code load stays inside the codes of existing heads
    const int lane_r = valid ? lane : (int)(r_b - 1 - (r_a + (int64_t)g * 32));
    const int within = off0 + lane_r;
    const int bh = h0 + (S >= 32 ? (within >= S ? 1 : 0) : within / S);
    const int hq = min(bh - h_first, kMaxQHeads - 1);   // slot of the head's staged codes
    // the whole row into registers, then the block goes back to the producer
    uint4 raw[NCH];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int c = (j + lane) % NCH;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];\n"
                   : "=r"(raw[j].x), "=r"(raw[j].y), "=r"(raw[j].z), "=r"(raw[j].w) : "r"(rowaddr + c * 16));
    }
    // max |x| on bf16 pairs (exact, the same value as in float32); using
    // every loaded value here also completes the loads before the hand-back
    __nv_bfloat162 m2[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) m2[e] = __habs2(reinterpret_cast<const __nv_bfloat162*>(&raw[0])[e]);
#pragma unroll
    for (int j = 1; j < NCH; ++j) {
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
#pragma unroll
      for (int e = 0; e < 4; ++e) m2[e] = __hmax2(m2[e], __habs2(p2[e]));
    }
    const __nv_bfloat162 mm = __hmax2(__hmax2(m2[0], m2[1]), __hmax2(m2[2], m2[3]));
    const float a = fmaxf(__low2float(mm), __high2float(mm));
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(smem_u32(&empty[st]));
    // |x| <= a and inv = fl(127/a), so y = fl(x * inv) has |y| < 127.5 and
    // rint stays in [-127, 127] without a clamp.  rint(y) is taken by
    // adding 1.5 * 2^23 in float32: the sum lies in [2^23, 2^24), where the
    // spacing is 1, so round-to-nearest-even leaves y + 1.5 * 2^23 rounded to
    // an integer with ties to even (1.5 * 2^23 is even), and the low byte of
    // the sum's bit pattern is rint(y) mod 256, the code's two's-complement
    // byte.  The product and the sum are separate round-to-nearest
    // intrinsics, which are never merged into a fused multiply-add.  (The
    // packed f32x2 forms gave the codes of a single rounding on the GPU, so
    // they are not used here.)
    const float inv = a > 0.f ? __fdiv_rn(127.f, a) : 0.f;
    const float sk = a > 0.f ? __fdiv_rn(a, 127.f) : 0.f;
    const uint32_t qrow = qbase + hq * D;
    int dot0 = 0, dot1 = 0;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int c = (j + lane) % NCH;
      int2 qp;
      asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];\n" : "=r"(qp.x), "=r"(qp.y) : "r"(qrow + c * 8));
      const uint32_t* wd = reinterpret_cast<const uint32_t*>(&raw[j]);
      uint32_t cc[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        cc[2 * e] = __float_as_uint(__fadd_rn(__fmul_rn(__uint_as_float(wd[e] << 16), inv), 12582912.f));
        cc[2 * e + 1] = __float_as_uint(__fadd_rn(__fmul_rn(__uint_as_float(wd[e] & 0xffff0000u), inv), 12582912.f));
      }
      const int kp0 = (int)__byte_perm(__byte_perm(cc[0], cc[1], 0x0040), __byte_perm(cc[2], cc[3], 0x0040), 0x5410);
      const int kp1 = (int)__byte_perm(__byte_perm(cc[4], cc[5], 0x0040), __byte_perm(cc[6], cc[7], 0x0040), 0x5410);
      dot0 = __dp4a(kp0, qp.x, dot0);
      dot1 = __dp4a(kp1, qp.y, dot1);
    }
    if (valid) scores[r] = __fmul_rn(__fmul_rn((float)(dot0 + dot1), s_qs[hq]), sk);
    for (off0 += 32 * kConsumerWarps; off0 >= S; off0 -= S) ++h0;
  }
}

}  // namespace

cudaError_t launch_rawdot_int8(const __nv_bfloat16* q, const __nv_bfloat16* k, int B, int H_q, int H_kv, int S,
                               int D, int W, float* qsum, float* scores, cudaStream_t st) {
  const int BH = B * H_kv;
  cudaError_t e = launch_pdl(kvc_rawdot_qsum_kernel, dim3(BH, D / 8), dim3(kQsumThreads), 0, st, q, H_q, H_kv, W, D,
                             qsum);
  note_launches(1);
  if (e != cudaSuccess) return e;
  const int64_t rows = (int64_t)BH * S;
  // at least ceil(BH / 15) CTAs, so a range holds at most 15*S rows and
  // touches at most 16 heads
  const int64_t ctas = std::max<int64_t>(std::max(1, num_sms() * kRawCtasPerSm),
                                         (BH + kMaxRangeHeads - 1) / kMaxRangeHeads);
  const int64_t per_cta = (rows + ctas - 1) / ctas;
  const size_t smem = (size_t)kRingStages * kRingRows * D * 2;
  const int grid = (int)((rows + per_cta - 1) / per_cta);
  if (D == 64) {
    if ((e = cudaFuncSetAttribute(kvc_rawdot_score_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
      return e;
    e = launch_pdl(kvc_rawdot_score_kernel<64>, dim3(grid), dim3(kRawThreads), smem, st, k, rows, per_cta, S, qsum,
                   scores, status_word_ptr());
  } else {
    if ((e = cudaFuncSetAttribute(kvc_rawdot_score_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
      return e;
    e = launch_pdl(kvc_rawdot_score_kernel<128>, dim3(grid), dim3(kRawThreads), smem, st, k, rows, per_cta, S, qsum,
                   scores, status_word_ptr());
  }
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvc
