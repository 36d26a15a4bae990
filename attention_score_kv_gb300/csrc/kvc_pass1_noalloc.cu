// Pass 1 of the scorer for callers that cannot allocate device memory.
//
// kvc_score_pass1 takes its scratch (the per-key-range partial normalisers)
// from a caller-provided workspace.  Some callers cannot provide one: code
// running inside a host framework that owns all device memory through its
// own pool (a cudaMalloc there fails or breaks the pool's accounting), and
// plugin or real-time paths that are not allowed to call the CUDA allocator
// at all, since cudaMalloc/cudaFree may synchronise the whole device.  For
// them this entry point keeps the scratch in a fixed array in the library's
// own device memory and allocates nothing.
//
// The array lives for as long as the library is loaded, on every GPU that
// loads it (1 MiB each).  All calls share it: two calls whose kernels overlap
// on the GPU (on different streams, or from different host threads) race on
// it and must be serialised by the caller.  Nothing in it needs to start at
// zero: pass 1 writes every partial it later reads.
#include <algorithm>
#include <mutex>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;   // 1 MiB per device
constexpr size_t kNoAllocScratchFloats = kNoAllocScratchBytes / sizeof(float);

static __device__ __align__(256) float g_pass1_noalloc_scratch[kNoAllocScratchFloats];

std::mutex g_na_mu;
float* g_na_ptr[64] = {nullptr};

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device, with that device current, and cached.
int scratch_on_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return set_error(KVC_ERR_UNSUPPORTED, "device ordinal %d above 63", dev);
  std::lock_guard<std::mutex> lk(g_na_mu);
  if (!g_na_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pass1_noalloc_scratch);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress of the pass-1 scratch array");
    g_na_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_na_ptr[dev];
  return KVC_OK;
}

}  // namespace
}  // namespace kvc

using namespace kvc;

extern "C" int kvc_score_pass1_noalloc(const kvc_bf16* q_win, const kvc_bf16* k, int B, int H_q, int H_kv,
                                       int S, int D, int W, int b_s, float* m, float* Z,
                                       kvc_stream_t stream) {
  int rc;
  if ((rc = check_shapes(B, H_q, H_kv, S, D, W)) || (rc = check_bs(b_s))) return rc;
  if ((rc = check_ptr(q_win, 16, "q_win")) || (rc = check_ptr(k, 16, "k")) || (rc = check_ptr(m, 4, "m")) ||
      (rc = check_ptr(Z, 4, "Z")))
    return rc;

  // Partials need 2 * gwp floats per (scan CTA, KV head it touches).  Use the
  // default scan plan when its partials fit the fixed array, else one CTA per
  // head (one slot per head); refuse shapes where even that does not fit.
  const int BH = B * H_kv;
  const int gwp = ((H_q / H_kv) * W + 15) / 16 * 16;
  const int64_t per_slot = (int64_t)gwp * 2;
  if ((int64_t)BH * per_slot > (int64_t)kNoAllocScratchFloats)
    return set_error(KVC_ERR_UNSUPPORTED,
                     "B*H_kv*G*W too large for the allocation-free pass 1: needs %lld bytes of scratch, "
                     "the fixed array holds %zu",
                     (long long)((int64_t)BH * per_slot * (int64_t)sizeof(float)), kNoAllocScratchBytes);
  if (num_sms() <= 0) return set_error(KVC_ERR_CUDA, "no CUDA device");
  ScanPlan pl = make_plan(BH, S);
  if ((int64_t)pl.P * pl.maxseg * per_slot > (int64_t)kNoAllocScratchFloats) pl = plan_for(BH, S, BH);
  const int64_t slots = (int64_t)pl.P * pl.maxseg;

  float* scratch = nullptr;
  rc = scratch_on_current_device(&scratch);
  if (rc != KVC_OK) return rc;
  float* pm = scratch;
  float* pz = scratch + slots * gwp;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  auto q = reinterpret_cast<const __nv_bfloat16*>(q_win);
  auto kk = reinterpret_cast<const __nv_bfloat16*>(k);
  cudaError_t e = launch_pass1(q, kk, B, H_q, H_kv, S, D, W, pl, gwp, pm, pz, true, st);
  if (e != cudaSuccess) return cuda_error(e, "allocation-free pass 1 launch");
  e = launch_pass1_combine(pm, pz, B, H_q, H_kv, S, W, pl, gwp, m, Z, st);
  if (e != cudaSuccess) return cuda_error(e, "allocation-free pass 1 combine launch");
  return KVC_OK;
}
