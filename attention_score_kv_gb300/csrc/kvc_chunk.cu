// Layer-major chunked prefill around the layer-end compress (TideKV, Fig. 1(d)
// and Fig. 2): the keys and values of each prompt chunk j (C positions, the
// last one ragged) are written into the active layer's full-prompt buffer at
// positions j*C .. ; after the last chunk the layer is compressed and its
// retained rows are committed into the cross-layer cache, at the layer's own
// row offset (kvc_cache_layout), after which the full buffer can be reused
// for the next layer.
//
// The append is a strided copy: one 16-byte vector per thread, rows of D
// values, every (b, head) moving one contiguous block of the chunk.
#include <algorithm>

#include "kvc_device.cuh"
#include "kvc_internal.cuh"

namespace kvc {
namespace {

__global__ void __launch_bounds__(256)
kvc_append_chunk_kernel(const uint4* __restrict__ kc, const uint4* __restrict__ vc, int64_t n_vec, int c_len,
                        int S, int64_t pos0, int vec_per_row, uint4* __restrict__ ka, uint4* __restrict__ va) {
  grid_dep_wait();   // the chunk may come from the previous grid
  grid_dep_launch();
  const int64_t per_head = (int64_t)c_len * vec_per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t bh = i / per_head;
    const int64_t within = i - bh * per_head;   // row t of the chunk, vector e of the row
    const int64_t dst = (bh * S + pos0) * vec_per_row + within;
    ka[dst] = kc[i];
    va[dst] = vc[i];
  }
}

}  // namespace

cudaError_t launch_append_chunk(const __nv_bfloat16* k_chunk, const __nv_bfloat16* v_chunk, int B, int H_kv, int S,
                                int C, int D, int j, __nv_bfloat16* k_act, __nv_bfloat16* v_act, cudaStream_t st) {
  const int64_t pos0 = (int64_t)j * C;
  const int c_len = (int)std::min<int64_t>(C, S - pos0);
  const int vec_per_row = D / 8;
  const int64_t n_vec = (int64_t)B * H_kv * c_len * vec_per_row;
  if (n_vec == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n_vec + 255) / 256, (int64_t)num_sms() * 16);
  cudaError_t e = launch_pdl(kvc_append_chunk_kernel, dim3((unsigned)blocks), dim3(256), 0, st,
                             reinterpret_cast<const uint4*>(k_chunk), reinterpret_cast<const uint4*>(v_chunk), n_vec,
                             c_len, S, pos0, vec_per_row, reinterpret_cast<uint4*>(k_act),
                             reinterpret_cast<uint4*>(v_act));
  note_launches(1);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace kvc
