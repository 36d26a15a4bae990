// Internal declarations shared by the kvc CUDA translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

// ---------------------------------------------------------------- limits
constexpr int kTile = 128;          // keys per scan tile (MMA M or N extent)
constexpr int kMaxHkv = 128;        // KV heads per call (selection params live in the kernel argument block)
constexpr int kMaxGWP = 256;        // G*W rounded up to 16
constexpr int kMaxPool = 15;        // widest average pool
constexpr int kMaxSeg = 8;          // KV heads one scan CTA may touch
constexpr int kMinKeysPerCta = 1024;
constexpr int kMaxDecodeSteps = 4096;  // decoding steps a Phase-1 median runs over
constexpr int kHist1 = 2048;        // radix digits: bits 31..21, 20..10, 9..0 of the score
constexpr int kHist2 = 2048;
constexpr int kHist3 = 1024;

// device status word codes
constexpr int kStatusOk = 0;
constexpr int kStatusCandOverflow = 1;
constexpr int kStatusSelectMismatch = 2;
constexpr int kStatusTimeout = 3;
constexpr int kStatusBadInput = 4;      // a device-resident input broke the contract

// How the flattened key space [B*H_kv][S] is cut into scan CTAs: CTA c owns
// keys [range_begin(c), range_begin(c + 1)) and touches at most `maxseg` KV
// heads; one head is touched by at most `nparts` CTAs.  Per-(CTA, head)
// "slots" hold pass-1 partials and pass-2 candidate lists:
// slot = c * maxseg + (head - first head of c).
struct ScanPlan {
  int P;
  int64_t L;
  int maxseg;
  int nparts;
};

// Scratch layout inside the caller's workspace (all offsets 256-aligned).
struct WsLayout {
  ScanPlan plan;
  int slots;       // partial / candidate slots reserved
  int gwp;         // G*W rounded up to 16
  int cap;         // candidate capacity per slot (K_l_max + b_s)
  size_t off_bias;                 // float  [BH][gwp]    pass-2 per-row bias
  size_t off_part_m, off_part_z;   // float  [slots][gwp]
  size_t off_cand_cnt;             // int    [slots]
  size_t off_cand;                 // uint64 [slots][cap]
  size_t total;
};

// Per-head selection parameters, passed by value in the kernel argument block.
// Start of scan CTA c's key range: c*L, moved onto the nearest head
// boundary when it lies within min(L/4, kSnapKeys) keys of one.  A CTA that
// would end with a sliver of the next head (or start with the tail of the
// previous one) pays a whole segment switch for it (the queries reloaded,
// the pipeline drained and refilled), several times the cost of a few more
// tiles.  The ranges stay ordered and at least L/2 long.
constexpr int64_t kSnapKeys = 4 * kTile;
__host__ __device__ inline int64_t range_begin(int64_t c, int64_t L, int64_t S, int64_t total) {
  const int64_t f = c * L;
  if (f <= 0) return 0;
  if (f >= total) return total;
  const int64_t snap = L / 4 < kSnapKeys ? L / 4 : kSnapKeys;
  const int64_t r = f % S;
  if (r != 0 && r <= snap) return f - r;
  if (r != 0 && S - r <= snap) return f + (S - r) < total ? f + (S - r) : total;
  return f;
}
// The scan CTA whose range holds key f, 0 <= f < total.
__host__ __device__ inline int64_t range_of(int64_t f, int64_t L, int64_t S, int64_t total) {
  int64_t c = f / L;
  if (f < range_begin(c, L, S, total)) --c;
  else if (f >= range_begin(c + 1, L, S, total)) ++c;
  return c;
}

struct SelParams {
  int S, sink, recent, H_kv, nparts;
  int64_t total;        // B * H_kv * S: the flattened key space of the scan plan
  int r_lo;             // min(sink, S): mandatory keys at the front
  int r_hi;             // max(S - recent, r_lo): first mandatory key at the back
  int64_t T;            // retained rows per batch element
  int64_t L;            // scan plan (candidate-list mode)
  int maxseg;
  int n_sel[kMaxHkv];   // non-mandatory keys kept per head (or all candidates)
  int kept[kMaxHkv];    // rows head h fills: min(K_l[h], S)
  int64_t off[kMaxHkv]; // row offset of head h inside a batch element
};

// ------------------------------------------------------------ host helpers
int set_error(int code, const char* fmt, ...);
// Argument checks shared by the entry points (KVC_OK or an error code with
// the message set).
int check_shapes(int B, int H_q, int H_kv, int S, int D, int W);
int check_bs(int b_s);
int check_pool(int pool_k);
int check_ptr(const void* p, size_t align, const char* name);
int check_ws(void* ws, size_t ws_bytes, size_t need);
int cuda_error(cudaError_t e, const char* what);
int num_sms();
int scan_ctas_target();                             // SM count or the tuning override
uint32_t wait_limit_polls();                        // polls before a pipeline wait gives up
ScanPlan plan_for(int BH, int S, int P);            // exact plan for P CTAs
ScanPlan make_plan(int BH, int S);                  // default plan
int max_slots(int BH);                              // S-independent bound on plan slots
int max_parts(int BH);                              // S-independent bound on plan.nparts
bool layout_ws(int B, int H_q, int H_kv, int D, int W, int b_s, int K_l_max, int pool_k, int S,
               WsLayout* L);                        // S < 0: the S-independent upper bound

// Launch `kernel` so that it may start while the previous grid on the stream
// finishes (programmatic stream serialization); the kernel calls
// grid_dep_wait() before it touches anything that grid produces.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// --------------------------------------------------------- kernel launchers
// pass 1: per-slot partial normalisers (log2-domain reference m, Z relative
// to it).  exact_max: m is the slot's maximum score (the pass-1 results the
// API returns); otherwise m is any reference with the same m + log2 Z, which
// is all the bias of pass 2 needs and skips a max per score.
cudaError_t launch_pass1(const __nv_bfloat16* q, const __nv_bfloat16* k, int B, int H_q, int H_kv, int S, int D,
                         int W, const ScanPlan& pl, int gwp, float* part_m, float* part_z, bool exact_max,
                         cudaStream_t st);
cudaError_t launch_pass1_combine(const float* part_m, const float* part_z, int B, int H_q, int H_kv, int S,
                                 int W, const ScanPlan& pl, int gwp, float* m, float* Z, cudaStream_t st);
// pass 2: lse from (m, Z) (natural units) or from pass-1 partials; output
// either dense scores or per-slot candidate lists
struct Pass2Out {
  float* scores;          // dense [BH][S] or nullptr
  uint64_t* cand;         // [slots][cap] or nullptr
  int* cand_cnt;          // [slots]
  int cap;
};
cudaError_t launch_pass2(const __nv_bfloat16* q, const __nv_bfloat16* k, const float* m, const float* Z,
                         const float* part_m, const float* part_z, float* bias_ws, int B, int H_q, int H_kv, int S,
                         int D, int W, int pool_k, const ScanPlan& pl, int gwp, const SelParams* sel, Pass2Out out,
                         bool inputs_ready, cudaStream_t st);
// single-pass raw inner-product scores with INT8 keys: the scoring queries'
// float32 column sums into qsum [BH][D], then dense scores
cudaError_t launch_rawdot_int8(const __nv_bfloat16* q, const __nv_bfloat16* k, int B, int H_q, int H_kv, int S,
                               int D, int W, float* qsum, float* scores, cudaStream_t st);
// chunk j of the active layer's keys and values into its full-prompt buffer
cudaError_t launch_append_chunk(const __nv_bfloat16* k_chunk, const __nv_bfloat16* v_chunk, int B, int H_kv, int S,
                                int C, int D, int j, __nv_bfloat16* k_act, __nv_bfloat16* v_act, cudaStream_t st);
// HeteroCache measurement and allocation (overlap coefficient, head
// similarity, inverse-stability budgets on the device)
cudaError_t launch_overlap(const int32_t* a, const int64_t* a_off, const int32_t* b, const int64_t* b_off,
                           int n_pairs, float* out, cudaStream_t st);
cudaError_t launch_similarity(const int32_t* idx, const int64_t* off, int n_groups, int H, float* sim,
                              cudaStream_t st);
// Phase 1 over decoding steps: per-step stability overlaps, medians over steps
cudaError_t launch_stability_steps(const int32_t* dec_idx, const int64_t* dec_off, const int32_t* pre_idx,
                                   const int64_t* pre_off, int T, int H, float* per_step, cudaStream_t st);
cudaError_t launch_median(const float* x, int T, int H, float* out, cudaStream_t st);
cudaError_t launch_budget(const double* s_stable, int n_layers, int H, int64_t total, int lo, int hi,
                          int32_t* K_l, cudaStream_t st);
// selection over dense scores (mode 0) or candidate lists (mode 1)
cudaError_t launch_select(int mode, const float* scores, const uint64_t* cand, const int* cand_cnt, int cap, int B,
                          const SelParams& sel, int32_t* idx, cudaStream_t st);
// rows of head h inside a batch element: off[h] .. off[h] + kept[h] - 1 of a
// T-row block; other rows of the block are left untouched
cudaError_t launch_gather(const __nv_bfloat16* k, const __nv_bfloat16* v, const int32_t* idx, int B,
                          const SelParams& sel, int D, __nv_bfloat16* k_out, __nv_bfloat16* v_out,
                          int32_t* pos_out, cudaStream_t st);

int* status_word_ptr();     // device address of the status word
void note_launches(int n);  // count kernels issued (measurement)

}  // namespace kvc
