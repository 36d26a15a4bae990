// Device helpers shared by the kvc kernels: shared-memory addresses,
// programmatic dependent launch, exp2, a block scan and the status word.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace kvc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch.  grid_dep_wait: block until the grid this
// one was launched behind has completed and its writes are visible (returns
// at once when there is none).  grid_dep_launch: let the next grid on the
// stream be scheduled as SMs free up; it still waits for this grid's
// completion before it reads anything this grid writes.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }

// 2^x with the hardware approximation (relative error about 2^-22); 2^-inf = 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

// Inclusive sum over a block of blockDim.x (multiple of 32, <= 1024) threads.
// `scratch` holds 32 ints.  Returns the inclusive prefix; *total gets the sum.
__device__ __forceinline__ int block_inclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    scratch[lane] = w;
  }
  __syncthreads();
  int res = v + (warp > 0 ? scratch[warp - 1] : 0);
  *total = scratch[nw - 1];
  __syncthreads();
  return res;
}

__device__ __forceinline__ void record_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

}  // namespace kvc
