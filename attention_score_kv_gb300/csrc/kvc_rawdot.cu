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
// once: D/8 lanes per key row, one 16-byte load per lane, the row maximum
// by shuffles, the dot product by dp4a.
#include <algorithm>

#include "kvc_device.cuh"
#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr int kRowsPerThreadStep = 2;   // independent rows in flight per lane

__device__ __forceinline__ int code8(float x, float inv) {
  const int c = __float2int_rn(__fmul_rn(x, inv));
  return max(-127, min(127, c));
}

// One block per (b, KV head), one thread per dimension.
__global__ void kvc_rawdot_query_kernel(const __nv_bfloat16* __restrict__ q, int H_q, int H_kv, int W, int D,
                                        int8_t* __restrict__ qcode, float* __restrict__ qscale) {
  grid_dep_wait();
  grid_dep_launch();
  const int bh = blockIdx.x;
  const int b = bh / H_kv, h = bh % H_kv, G = H_q / H_kv;
  const int d = threadIdx.x;
  const __nv_bfloat16* src = q + ((size_t)(b * H_q + h * G) * W) * D;
  float acc = 0.f;
  for (int r = 0; r < G * W; ++r) acc = __fadd_rn(acc, __bfloat162float(src[(size_t)r * D + d]));
  __shared__ float s_max[32];
  float a = fabsf(acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  if ((d & 31) == 0) s_max[d >> 5] = a;
  __syncthreads();
  float amax = 0.f;
  for (int w = 0; w < (D + 31) / 32; ++w) amax = fmaxf(amax, s_max[w]);
  const float inv = amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f;
  qcode[(size_t)bh * D + d] = (int8_t)(amax > 0.f ? code8(acc, inv) : 0);
  if (d == 0) qscale[bh] = amax > 0.f ? __fdiv_rn(amax, 127.f) : 0.f;
}

template <int D>
__global__ void __launch_bounds__(256)
kvc_rawdot_score_kernel(const __nv_bfloat16* __restrict__ k, int64_t rows, int S, const int8_t* __restrict__ qcode,
                        const float* __restrict__ qscale, float* __restrict__ scores) {
  grid_dep_wait();   // the query codes come from the previous grid
  grid_dep_launch();
  constexpr int LPR = D / 8;             // lanes per key row
  constexpr int RPW = 32 / LPR;          // rows per warp step
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR, cl = lane % LPR;
  const unsigned group_mask = (LPR == 32) ? 0xffffffffu : (((1u << LPR) - 1u) << (sub * LPR));
  const int64_t warp_g = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t stride = nwarps * RPW;
  for (int64_t r0 = warp_g * RPW + sub; r0 - sub < rows; r0 += kRowsPerThreadStep * stride) {
    uint4 raw[kRowsPerThreadStep];
#pragma unroll
    for (int u = 0; u < kRowsPerThreadStep; ++u) {
      const int64_t r = r0 + u * stride;
      raw[u] = r < rows ? __ldg(reinterpret_cast<const uint4*>(k + (size_t)r * D) + cl) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kRowsPerThreadStep; ++u) {
      const int64_t r = r0 + u * stride;
      const int bh = (int)((r < rows ? r : 0) / S);
      const __nv_bfloat162* p2 = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
      float x[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(p2[i]);
        x[2 * i] = f.x;
        x[2 * i + 1] = f.y;
      }
      float a = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(x[i]));
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(group_mask, a, o));
      const float inv = a > 0.f ? __fdiv_rn(127.f, a) : 0.f;
      int c[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = a > 0.f ? code8(x[i], inv) : 0;
      const int kp0 = (c[0] & 0xff) | ((c[1] & 0xff) << 8) | ((c[2] & 0xff) << 16) | ((c[3] & 0xff) << 24);
      const int kp1 = (c[4] & 0xff) | ((c[5] & 0xff) << 8) | ((c[6] & 0xff) << 16) | ((c[7] & 0xff) << 24);
      const int2 qp = *reinterpret_cast<const int2*>(qcode + (size_t)bh * D + cl * 8);
      int dot = __dp4a(kp0, qp.x, 0);
      dot = __dp4a(kp1, qp.y, dot);
#pragma unroll
      for (int o = LPR / 2; o > 0; o >>= 1) dot += __shfl_xor_sync(group_mask, dot, o);
      if (cl == 0 && r < rows) {
        const float sk = a > 0.f ? __fdiv_rn(a, 127.f) : 0.f;
        scores[r] = __fmul_rn(__fmul_rn((float)dot, qscale[bh]), sk);
      }
    }
  }
}

}  // namespace

cudaError_t launch_rawdot_int8(const __nv_bfloat16* q, const __nv_bfloat16* k, int B, int H_q, int H_kv, int S,
                               int D, int W, int8_t* qcode, float* qscale, float* scores, cudaStream_t st) {
  const int BH = B * H_kv;
  cudaError_t e = launch_pdl(kvc_rawdot_query_kernel, dim3(BH), dim3(D), 0, st, q, H_q, H_kv, W, D, qcode, qscale);
  note_launches(1);
  if (e != cudaSuccess) return e;
  const int64_t rows = (int64_t)BH * S;
  const int rows_per_block = (256 / 32) * (32 / (D / 8)) * kRowsPerThreadStep;
  int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
  blocks = std::min<int64_t>(std::max<int64_t>(blocks, 1), (int64_t)num_sms() * 16);
  if (D == 64)
    e = launch_pdl(kvc_rawdot_score_kernel<64>, dim3((unsigned)blocks), dim3(256), 0, st, k, rows, S, qcode, qscale,
                   scores);
  else
    e = launch_pdl(kvc_rawdot_score_kernel<128>, dim3((unsigned)blocks), dim3(256), 0, st, k, rows, S, qcode, qscale,
                   scores);
  note_launches(1);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvc
