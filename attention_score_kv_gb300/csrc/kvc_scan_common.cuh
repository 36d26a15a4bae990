// Pieces shared by the two scans of the two-pass scorer (TideKV, Fig. 3):
// the work split, the TMA producer, the tcgen05 MMA issuer and host-side
// tensor-map set-up.
//
// Work split.  The flattened key space [B*H_kv][S] is cut into P contiguous
// ranges of about L keys, one CTA each (P ~ number of SMs), so every SM gets
// nearly the same number of keys whatever B, H_kv and S are; a range
// boundary near a head boundary is moved onto it (range_begin).  A range can
// cross KV-head boundaries; each piece (one head, keys [a, b)) is a
// "segment".  Pass-1
// partial normalisers and pass-2 candidate lists live in per-(CTA, segment)
// slots whose number depends on P and B*H_kv only, never on S.
//
// Warp 0 issues TMA loads (the group's window queries once per segment, then
// 128-key tiles through a shared-memory ring); the MMA warps and the softmax
// warps of each scan are described in its own file.  Every mbarrier wait is
// bounded; a wait that gives up records a timeout in the status word and the
// CTA drains and returns.
#pragma once

#include <cudaTypedefs.h>

#include <cfloat>
#include <climits>

#include "kvc_device.cuh"
#include "kvc_internal.cuh"
#include "kvc_tc.cuh"

namespace kvc {
namespace scan {

#ifndef KVC_P1_STAGES
#define KVC_P1_STAGES 4
#endif
constexpr int kStages = KVC_P1_STAGES;        // key-tile ring depth of pass 1
constexpr int kMaxStages = 8;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccStride = 256;          // TMEM columns per accumulator buffer
constexpr uint32_t kWaitLimit = 1u << 22;     // polls before a wait gives up (default)
constexpr uint32_t kDrainLimit = 1u << 26;    // polls while draining copies / MMAs already issued
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSegs = 8;

struct ScanArgs {
  int B, H_q, H_kv, S, W, gw, gwp16, n_mb, nq, P, maxseg, pool_k, cap;
  uint32_t wait_limit;       // polls before a pipeline wait gives up
  int inputs_ready;          // pass 2: keys and queries were complete before the previous grid ran
  int64_t L;
  float c2;                  // log2(e) / sqrt(D)
  float* part_m;             // pass 1 out: [P*maxseg][gwp16] (log2 units)
  float* part_z;
  const float* m_in;         // pass 2: natural-unit m, Z [B][H_q][W] ...
  const float* z_in;
  const float* pm_in;        // ... or pass-1 partials
  const float* pz_in;
  const float* bias;         // pass 2: per-row -lse2 / c2 [BH][gwp16]
  float* scores;             // pass 2 out: dense [BH][S] or nullptr
  uint64_t* cand;            // pass 2 out: [P*maxseg][cap]
  int* cand_cnt;             // [P*maxseg]
  int* status;
};

struct Seg {
  int bh, a, b;
};

// Bounded wait; on giving up, flags the CTA and the status word.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                         uint32_t limit = kWaitLimit) {
  for (uint32_t i = 0; i < limit; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 4095u) == 4095u && *abort_flag) return false;
  }
  *abort_flag = 1;
  record_status(status, kStatusTimeout);
  return false;
}

// Bounded wait by a whole warp.  Every lane reads the barrier in the same
// instruction, so the warp never diverges: a barrier that is already
// complete costs one read (about 20 cycles), where one polling lane plus a
// broadcast costs over 300 (the warp splits and reconverges around the poll).
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag, int* status,
                                              uint32_t limit = kWaitLimit) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  for (uint32_t i = 0; i < limit; ++i) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    if ((i & 4095u) == 4095u && *abort_flag) return false;
  }
  *abort_flag = 1;
  if ((threadIdx.x & 31) == 0) record_status(status, kStatusTimeout);
  return false;
}

// Draining before a CTA leaves.  Copies and MMAs a CTA has issued always
// complete, whether or not a wait gave up meanwhile; shared and tensor memory
// must not be released before they have.  So every thread that issued them
// waits for their completion barriers first, with a limit far above any
// completion time (the pipeline waits above may have been given a short
// one).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int* status) {
  for (uint32_t i = 0; i < kDrainLimit; ++i)
    if (tc::mbar_try_wait(bar, parity)) return;
  record_status(status, kStatusTimeout);
}
// All MMAs (and tensor-memory copies) issued so far by this thread.
__device__ __forceinline__ void drain_mma(uint32_t bar, int* status) {
  tc::mma_commit(bar);
  drain_wait(bar, 0, status);
}

// Pass-1 tile order within a segment: the leading third of the keys comes
// last, so pass 2, which starts there, finds those keys still in L2.  Each
// stretch is read in ascending order.
__device__ __forceinline__ int p1_tile_order(int i, int ntiles) {
  const int lead = ntiles / 3;
  return i < ntiles - lead ? lead + i : i - (ntiles - lead);
}

// Segments of CTA c, in key order.
__device__ __forceinline__ int cta_segments(const ScanArgs& A, int c, Seg* out) {
  const int64_t total = (int64_t)A.B * A.H_kv * A.S;
  const int64_t f0 = range_begin(c, A.L, A.S, total);
  const int64_t f1 = range_begin(c + 1, A.L, A.S, total);
  if (f0 >= f1) return 0;
  const int h0 = (int)(f0 / A.S), h1 = (int)((f1 - 1) / A.S);
  int n = 0;
  for (int h = h0; h <= h1 && n < kMaxSegs; ++h, ++n) {
    out[n].bh = h;
    out[n].a = (int)max((int64_t)0, f0 - (int64_t)h * A.S);
    out[n].b = (int)min((int64_t)A.S, f1 - (int64_t)h * A.S);
  }
  return n;
}

__device__ __forceinline__ float2 merge_mz(float2 a, float2 b) {
  if (b.y == 0.f) return a;
  if (a.y == 0.f) return b;
  const float m = fmaxf(a.x, b.x);
  return make_float2(m, a.y * ex2(a.x - m) + b.y * ex2(b.x - m));
}

// (max, Z) of window row `row` of head bh over all pass-1 slots of the head.
__device__ __forceinline__ float2 combine_partials(const ScanArgs& A, int bh, int row) {
  const int64_t S = A.S, total = (int64_t)A.B * A.H_kv * A.S;
  const int c_first = (int)range_of((int64_t)bh * S, A.L, S, total);
  const int c_last = (int)range_of(((int64_t)bh + 1) * S - 1, A.L, S, total);
  float2 st = make_float2(-INFINITY, 0.f);
  for (int c = c_first; c <= c_last; ++c) {
    const int seg = bh - (int)(range_begin(c, A.L, S, total) / S);
    const size_t o = ((size_t)c * A.maxseg + seg) * A.gwp16 + row;
    st = merge_mz(st, make_float2(A.pm_in[o], A.pz_in[o]));
  }
  return st;
}

struct PipeBars {
  uint64_t full[kMaxStages], empty[kMaxStages], tfull[4], tempty[4], qfull, qempty, drain[2];
};

// empty_count / qempty_count: commits that free a ring stage / the queries
// (one per MMA-issuing thread that used them).
__device__ __forceinline__ void init_pipe_bars(PipeBars* b, int tempty_count, int nst = kStages, int empty_count = 1,
                                               int qempty_count = 1) {
  for (int i = 0; i < nst; ++i) {
    tc::mbar_init(smem_u32(&b->full[i]), 1);
    tc::mbar_init(smem_u32(&b->empty[i]), empty_count);
  }
  for (int i = 0; i < 4; ++i) {
    tc::mbar_init(smem_u32(&b->tfull[i]), 1);
    tc::mbar_init(smem_u32(&b->tempty[i]), tempty_count);
  }
  tc::mbar_init(smem_u32(&b->qfull), 1);
  tc::mbar_init(smem_u32(&b->qempty), qempty_count);
  tc::mbar_init(smem_u32(&b->drain[0]), 1);
  tc::mbar_init(smem_u32(&b->drain[1]), 1);
}

// TMA producer (one thread): per segment the window queries, then the key
// tiles through a ring of NST stages.
template <int D, int PASS, int NST = kStages>
__device__ void producer(const ScanArgs& A, const CUtensorMap* qmap, const CUtensorMap* kmap, PipeBars* bars,
                         uint32_t sQ, uint32_t sK, volatile int* abort_flag) {
  constexpr int NKH = D / 64;
  constexpr uint32_t kTileBytes = kTile * 128 * NKH;
  const uint32_t q_half = (uint32_t)A.nq * 128;
  const uint32_t q_bytes = q_half * NKH;
  const int hw = PASS == 2 ? (A.pool_k - 1) / 2 : 0;
  Seg segs[kMaxSegs];
  const int nseg = cta_segments(A, blockIdx.x, segs);
  const int G = A.H_q / A.H_kv;
  const uint64_t k_policy = PASS == 2 ? tc::l2_evict_first_policy() : 0ull;
  uint32_t stage = 0, phase = 0, qphase = 0;
  uint32_t loaded = 0, last_par = 0;   // per stage: ever loaded / parity of its last load (bit masks)
  bool q_loaded = false, ok = true;
  for (int si = 0; si < nseg && ok; ++si) {
    const Seg sg = segs[si];
    if (si > 0) {
      if (!wait_bar(smem_u32(&bars->qempty), qphase, abort_flag, A.status, A.wait_limit)) break;
      qphase ^= 1;
    }
    const int b_idx = sg.bh / A.H_kv, hk = sg.bh % A.H_kv;
    const int qrow = (b_idx * A.H_q + hk * G) * A.W;
    tc::mbar_arrive_expect_tx(smem_u32(&bars->qfull), q_bytes);
    for (int kh = 0; kh < NKH; ++kh)
      tc::tma_load_3d(sQ + kh * q_half, qmap, smem_u32(&bars->qfull), kh * 64, qrow, 0);
    q_loaded = true;
    const int start = sg.a - hw;
    const int ntiles = (sg.b - sg.a + 2 * hw + kTile - 1) / kTile;
    for (int ti = 0; ti < ntiles; ++ti) {
      const int t = PASS == 1 ? p1_tile_order(ti, ntiles) : ti;
      if (!wait_bar(smem_u32(&bars->empty[stage]), phase ^ 1, abort_flag, A.status, A.wait_limit)) {
        ok = false;
        break;
      }
      const uint32_t dst = sK + stage * kTileBytes;
      tc::mbar_arrive_expect_tx(smem_u32(&bars->full[stage]), kTileBytes);
      for (int kh = 0; kh < NKH; ++kh) {
        if (PASS == 2)   // the last full read of the keys: evict them first, keep the candidate lists in L2
          tc::tma_load_3d_hint(dst + kh * (kTile * 128), kmap, smem_u32(&bars->full[stage]), kh * 64,
                               start + t * kTile, sg.bh, k_policy);
        else
          tc::tma_load_3d(dst + kh * (kTile * 128), kmap, smem_u32(&bars->full[stage]), kh * 64, start + t * kTile,
                          sg.bh);
      }
      loaded |= 1u << stage;
      last_par = (last_par & ~(1u << stage)) | (phase << stage);
      if (++stage == NST) { stage = 0; phase ^= 1; }
    }
  }
  // every copy issued has landed before the CTA may leave
  for (int st = 0; st < NST; ++st)
    if (loaded & (1u << st)) drain_wait(smem_u32(&bars->full[st]), (last_par >> st) & 1u, A.status);
  if (q_loaded) drain_wait(smem_u32(&bars->qfull), qphase, A.status);
}

// ------------------------------------------------------------- host side
inline PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 3-D map over a [d2][d1][d0] bf16 tensor with 128-byte swizzled 64 x box1 boxes.
inline bool make_map(CUtensorMap* map, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box1) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
  cuuint32_t box[3] = {64, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

inline size_t pipe_smem(int D, int nq) {
  return 1024 + (size_t)nq * 128 * (D / 64) + (size_t)kStages * kTile * 128 * (D / 64);
}

inline ScanArgs base_args(const ScanPlan& pl, int B, int H_q, int H_kv, int S, int D, int W) {
  ScanArgs A{};
  A.B = B;
  A.H_q = H_q;
  A.H_kv = H_kv;
  A.S = S;
  A.W = W;
  A.gw = (H_q / H_kv) * W;
  A.gwp16 = (A.gw + 15) / 16 * 16;
  A.n_mb = A.gw > 128 ? 2 : 1;
  A.P = pl.P;
  A.L = pl.L;
  A.maxseg = pl.maxseg;
  A.c2 = kLog2e / sqrtf((float)D);
  A.status = status_word_ptr();
  A.wait_limit = wait_limit_polls();
  A.pool_k = 1;
  return A;
}

}  // namespace scan
}  // namespace kvc
