// C ABI of the layer-end compressor: argument validation, scan plan, scratch
// layout and kernel launches.  Every check runs on the host before the first
// launch.
#include <algorithm>
#include <array>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "kvc_internal.cuh"

namespace kvc {

__device__ int g_status_word;

namespace {
thread_local char t_err[512] = "";
int64_t g_opt_scan_ctas = 0;
int64_t g_opt_wait_limit = 0;
std::mutex g_mu;
int g_sms[64] = {0};
int* g_status_ptr[64] = {nullptr};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// stage timing (kvc_profile_begin / kvc_profile_end)
std::atomic<int64_t> g_launch_count{0};
bool g_prof = false;
int64_t g_prof_launch_base = 0;
std::vector<std::array<cudaEvent_t, KVC_N_STAGES + 1>> g_prof_ev;
size_t g_prof_used = 0;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
}  // namespace

void note_launches(int n) { g_launch_count += n; }

// Next event set for a profiled call, or nullptr when not profiling.
cudaEvent_t* prof_slot() {
  if (!g_prof) return nullptr;
  if (g_prof_used == g_prof_ev.size()) {
    std::array<cudaEvent_t, KVC_N_STAGES + 1> ev{};
    for (auto& e : ev)
      if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_prof_ev.push_back(ev);
  }
  return g_prof_ev[g_prof_used++].data();
}

int set_error(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_err, sizeof(t_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_error(cudaError_t e, const char* what) {
  return set_error(KVC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

int* status_word_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

uint32_t wait_limit_polls() {
  return g_opt_wait_limit > 0 ? (uint32_t)std::min<int64_t>(g_opt_wait_limit, 1LL << 30) : (1u << 22);
}

int scan_ctas_target() {
  if (g_opt_scan_ctas > 0) return (int)std::min<int64_t>(g_opt_scan_ctas, 1 << 16);
  return num_sms();
}

ScanPlan plan_for(int BH, int S, int P) {
  const int64_t total = (int64_t)BH * S;
  int64_t p = std::max<int64_t>(1, std::min<int64_t>(P, total));
  const int64_t L = ceil_div(total, p);
  p = ceil_div(total, L);
  ScanPlan pl;
  pl.P = (int)p;
  pl.L = L;
  int maxseg = 1;
  for (int64_t c = 0; c < p; ++c) {
    const int64_t f0 = range_begin(c, L, S, total), f1 = range_begin(c + 1, L, S, total);
    if (f1 > f0) maxseg = std::max<int>(maxseg, (int)((f1 - 1) / S - f0 / S + 1));
  }
  int nparts = 1;
  for (int64_t h = 0; h < BH; ++h)
    nparts = std::max<int>(nparts, (int)(range_of((h + 1) * S - 1, L, S, total) - range_of(h * S, L, S, total) + 1));
  pl.maxseg = maxseg;
  pl.nparts = nparts;
  return pl;
}

ScanPlan make_plan(int BH, int S) {
  const int64_t total = (int64_t)BH * S;
  int64_t P = scan_ctas_target();
  if (g_opt_scan_ctas <= 0) P = std::min<int64_t>(P, ceil_div(total, kMinKeysPerCta));
  P = std::max<int64_t>(P, ceil_div(BH, kMaxSeg - 2));
  return plan_for(BH, S, (int)std::max<int64_t>(P, 1));
}

static int max_ctas(int BH) {
  return std::max<int>(std::max(scan_ctas_target(), 1), (int)ceil_div(BH, kMaxSeg - 2));
}
int max_slots(int BH) { return BH + 3 * max_ctas(BH); }
int max_parts(int BH) { return max_ctas(BH); }

bool layout_ws(int B, int H_q, int H_kv, int D, int W, int b_s, int K_l_max, int pool_k, int S, WsLayout* L) {
  (void)D;
  (void)pool_k;
  if (num_sms() <= 0) return false;
  const int BH = B * H_kv;
  const int gw = (H_q / H_kv) * W;
  if (S > 0) {
    L->plan = make_plan(BH, S);
    L->slots = L->plan.P * L->plan.maxseg;
  } else {
    L->plan = ScanPlan{0, 0, 0, 0};
    L->slots = max_slots(BH);
  }
  L->gwp = (gw + 15) / 16 * 16;
  L->cap = std::max(K_l_max, 0) + b_s;
  size_t o = 0;
  L->off_bias = o;     o = align256(o + (size_t)BH * L->gwp * sizeof(float));
  L->off_part_m = o;   o = align256(o + (size_t)L->slots * L->gwp * sizeof(float));
  L->off_part_z = o;   o = align256(o + (size_t)L->slots * L->gwp * sizeof(float));
  L->off_cand_cnt = o; o = align256(o + (size_t)L->slots * sizeof(int));
  L->off_cand = o;     o = align256(o + (size_t)L->slots * (size_t)L->cap * sizeof(uint64_t));
  L->total = o;
  return true;
}

}  // namespace kvc

using namespace kvc;

namespace kvc {

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_shapes(int B, int H_q, int H_kv, int S, int D, int W) {
  if (B < 1 || H_q < 1 || H_kv < 1 || S < 1 || W < 1)
    return set_error(KVC_ERR_INVALID_ARG, "B, H_q, H_kv, S and W must be >= 1 (got B=%d H_q=%d H_kv=%d S=%d W=%d)", B,
                     H_q, H_kv, S, W);
  if (H_q % H_kv != 0) return set_error(KVC_ERR_INVALID_ARG, "H_q (%d) must be a multiple of H_kv (%d)", H_q, H_kv);
  if (W > S) return set_error(KVC_ERR_INVALID_ARG, "W (%d) must be <= S (%d)", W, S);
  if (S > (1 << 30)) return set_error(KVC_ERR_UNSUPPORTED, "S (%d) above 2^30", S);
  if (D != 64 && D != 128) return set_error(KVC_ERR_UNSUPPORTED, "head dim D=%d: only 64 and 128 are supported", D);
  if (H_kv > kMaxHkv) return set_error(KVC_ERR_UNSUPPORTED, "H_kv=%d above %d", H_kv, kMaxHkv);
  if ((H_q / H_kv) * W > kMaxGWP)
    return set_error(KVC_ERR_UNSUPPORTED, "G*W=%d above %d window rows per KV head", (H_q / H_kv) * W, kMaxGWP);
  if ((int64_t)B * H_q * W > (1LL << 31) || (int64_t)B * H_kv > (1LL << 24))
    return set_error(KVC_ERR_UNSUPPORTED, "batch too large");
  return KVC_OK;
}

int check_bs(int b_s) {
  if (b_s < kTile) return set_error(KVC_ERR_INVALID_ARG, "b_s=%d must be >= %d", b_s, kTile);
  // the candidate capacity K_l_max + b_s (K_l_max <= S <= 2^30) stays an int
  if (b_s > (1 << 29)) return set_error(KVC_ERR_UNSUPPORTED, "b_s=%d above 2^29", b_s);
  return KVC_OK;
}

int check_pool(int pool_k) {
  if (pool_k < 1 || pool_k % 2 == 0) return set_error(KVC_ERR_INVALID_ARG, "pool_k=%d must be odd and >= 1", pool_k);
  if (pool_k > kMaxPool) return set_error(KVC_ERR_UNSUPPORTED, "pool_k=%d above %d", pool_k, kMaxPool);
  return KVC_OK;
}

int check_ptr(const void* p, size_t align, const char* name) {
  if (!p) return set_error(KVC_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned(p, align)) return set_error(KVC_ERR_INVALID_ARG, "%s is not %zu-byte aligned", name, align);
  return KVC_OK;
}

int check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (need == 0) return KVC_OK;
  if (!ws) return set_error(KVC_ERR_WORKSPACE, "workspace is NULL (need %zu bytes)", need);
  if (!aligned(ws, 256)) return set_error(KVC_ERR_WORKSPACE, "workspace is not 256-byte aligned");
  if (ws_bytes < need) return set_error(KVC_ERR_WORKSPACE, "workspace of %zu bytes, need %zu", ws_bytes, need);
  return KVC_OK;
}

}  // namespace kvc

namespace {

// Rows of each head inside a batch element's block of the retained cache:
// head h fills min(K_l[h], S) rows from out_off[h]; the block is
// out_off[H_kv] rows long.  out_off NULL: the packed layout of
// kvc_retained_layout.  K_l[h] >= lo_rows is required.
int make_layout(int S, int H_kv, const int32_t* K_l, const int64_t* out_off, int lo_rows, SelParams* sp) {
  if (!K_l) return set_error(KVC_ERR_INVALID_ARG, "K_l is NULL");
  int64_t off = 0;
  for (int h = 0; h < H_kv; ++h) {
    if (K_l[h] < 0) return set_error(KVC_ERR_INVALID_ARG, "K_l[%d]=%d is negative", h, K_l[h]);
    if (K_l[h] < lo_rows)
      return set_error(KVC_ERR_INVALID_ARG, "K_l[%d]=%d is smaller than the mandatory set (%d keys)", h, K_l[h],
                       lo_rows);
    const int kept = std::min(K_l[h], S);
    if (out_off) {
      if (out_off[h] < off)
        return set_error(KVC_ERR_INVALID_ARG, "out_off[%d]=%lld overlaps the rows before it (need >= %lld)", h,
                         (long long)out_off[h], (long long)off);
      off = out_off[h];
    }
    sp->kept[h] = kept;
    sp->off[h] = off;
    off += kept;
  }
  if (out_off) {
    if (out_off[H_kv] < off)
      return set_error(KVC_ERR_INVALID_ARG, "out_off[%d]=%lld is shorter than the rows of the last head (need >= %lld)",
                       H_kv, (long long)out_off[H_kv], (long long)off);
    off = out_off[H_kv];
  }
  sp->T = off;
  return KVC_OK;
}

// Selection parameters from the host budget array and the output layout.
int make_sel(int S, int H_kv, const int32_t* K_l, const int64_t* out_off, int sink, int recent, SelParams* sp,
             int* K_l_eff_max) {
  if (!K_l) return set_error(KVC_ERR_INVALID_ARG, "K_l is NULL");
  if (sink < 0 || recent < 0) return set_error(KVC_ERR_INVALID_ARG, "sink/recent must be >= 0");
  std::memset(sp, 0, sizeof(*sp));
  sp->S = S;
  sp->sink = sink;
  sp->recent = recent;
  sp->H_kv = H_kv;
  sp->nparts = 1;
  sp->r_lo = std::min(sink, S);
  sp->r_hi = std::max(S - std::min(recent, S), sp->r_lo);
  const int rsz = sp->r_lo + (S - sp->r_hi);
  int rc = make_layout(S, H_kv, K_l, out_off, rsz, sp);
  if (rc) return rc;
  int mx = 0;
  for (int h = 0; h < H_kv; ++h) {
    sp->n_sel[h] = sp->kept[h] - rsz;
    mx = std::max(mx, sp->kept[h]);
  }
  if (K_l_eff_max) *K_l_eff_max = mx;
  return KVC_OK;
}

int launch_status(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return cuda_error(e, what);
  return KVC_OK;
}

}  // namespace

namespace {

// kvc_compress_layer with an optional event the gather waits on (the values
// are read by the gather only).
int compress_layer(int N, int layer, int B, int S, int C, int H_q, int H_kv, int D, int W, const int32_t* K_l,
                   int sink, int recent, int pool_k, int b_s, const kvc_bf16* q_win, const kvc_bf16* k,
                   const kvc_bf16* v, kvc_bf16* k_out, kvc_bf16* v_out, int32_t* pos_out,
                   const int64_t* out_off, void* ws, size_t ws_bytes, cudaEvent_t v_ready, kvc_stream_t stream) {
  int rc;
  if (N < 1 || layer < 0 || layer >= N) return set_error(KVC_ERR_INVALID_ARG, "layer %d outside [0, N=%d)", layer, N);
  if ((rc = check_shapes(B, H_q, H_kv, S, D, W)) || (rc = check_bs(b_s)) || (rc = check_pool(pool_k))) return rc;
  if (C < W || C > S) return set_error(KVC_ERR_INVALID_ARG, "chunk C=%d must satisfy W=%d <= C <= S=%d", C, W, S);
  if ((rc = check_ptr(q_win, 16, "q_win")) || (rc = check_ptr(k, 16, "k")) || (rc = check_ptr(v, 16, "v")) ||
      (rc = check_ptr(k_out, 16, "k_out")) || (rc = check_ptr(v_out, 16, "v_out")) ||
      (rc = check_ptr(pos_out, 4, "pos_out")))
    return rc;
  SelParams sp;
  int kmax = 0;
  if ((rc = make_sel(S, H_kv, K_l, out_off, sink, recent, &sp, &kmax))) return rc;
  WsLayout L;
  if (!layout_ws(B, H_q, H_kv, D, W, b_s, kmax, pool_k, S, &L)) return set_error(KVC_ERR_CUDA, "no CUDA device");
  if ((rc = check_ws(ws, ws_bytes, L.total))) return rc;
  sp.nparts = L.plan.nparts;
  sp.L = L.plan.L;
  sp.maxseg = L.plan.maxseg;
  sp.total = (int64_t)B * H_kv * S;
  char* w = static_cast<char*>(ws);
  float* pm = reinterpret_cast<float*>(w + L.off_part_m);
  float* pz = reinterpret_cast<float*>(w + L.off_part_z);
  uint64_t* cand = reinterpret_cast<uint64_t*>(w + L.off_cand);
  int* cnt = reinterpret_cast<int*>(w + L.off_cand_cnt);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  auto q = reinterpret_cast<const __nv_bfloat16*>(q_win);
  auto kk = reinterpret_cast<const __nv_bfloat16*>(k);
  auto vv = reinterpret_cast<const __nv_bfloat16*>(v);
  cudaEvent_t* ev = prof_slot();
  if (ev) cudaEventRecord(ev[0], st);
  if ((rc = launch_status(launch_pass1(q, kk, B, H_q, H_kv, S, D, W, L.plan, L.gwp, pm, pz, false, st), "pass 1 launch")))
    return rc;
  if (ev) cudaEventRecord(ev[1], st);
  Pass2Out out{nullptr, cand, cnt, L.cap};
  float* bias = reinterpret_cast<float*>(w + L.off_bias);
  if ((rc = launch_status(launch_pass2(q, kk, nullptr, nullptr, pm, pz, bias, B, H_q, H_kv, S, D, W, pool_k, L.plan,
                                       L.gwp, &sp, out, true, st),
                          "pass 2 launch")))
    return rc;
  if (ev) cudaEventRecord(ev[2], st);
  if ((rc = launch_status(launch_select(1, nullptr, cand, cnt, L.cap, B, sp, pos_out, st),
                          "selection launch")))
    return rc;
  if (ev) cudaEventRecord(ev[3], st);
  if (v_ready && (rc = launch_status(cudaStreamWaitEvent(st, v_ready, 0), "wait for v_ready")))
    return rc;
  rc = launch_status(launch_gather(kk, vv, pos_out, B, sp, D, reinterpret_cast<__nv_bfloat16*>(k_out),
                                   reinterpret_cast<__nv_bfloat16*>(v_out), pos_out, st),
                     "gather launch");
  if (ev) cudaEventRecord(ev[4], st);
  return rc;
}

}  // namespace

extern "C" {

const char* kvc_last_error(void) { return t_err; }

int kvc_version(void) { return 300; }

int kvc_set_option(int option, int64_t value) {
  if (option == KVC_OPT_SCAN_CTAS) {
    if (value < 0) return set_error(KVC_ERR_INVALID_ARG, "scan CTA count must be >= 0");
    g_opt_scan_ctas = value;
    return KVC_OK;
  }
  if (option == KVC_OPT_WAIT_LIMIT) {
    if (value < 0) return set_error(KVC_ERR_INVALID_ARG, "wait limit must be >= 0");
    g_opt_wait_limit = value;
    return KVC_OK;
  }
  return set_error(KVC_ERR_INVALID_ARG, "unknown option %d", option);
}

size_t kvc_workspace_size(int B, int H_q, int H_kv, int D, int W, int b_s, int K_l_max, int pool_k) {
  // S is not an argument: use W as the smallest legal S for the shape checks.
  if (check_shapes(B, H_q, H_kv, W, D, W) != KVC_OK) return 0;
  if (check_bs(b_s) != KVC_OK || check_pool(pool_k) != KVC_OK) return 0;
  if (K_l_max < 0) {
    set_error(KVC_ERR_INVALID_ARG, "K_l_max must be >= 0");
    return 0;
  }
  // a budget above S keeps min(K_l, S) rows, and S <= 2^30
  K_l_max = std::min(K_l_max, 1 << 30);
  WsLayout L;
  if (!layout_ws(B, H_q, H_kv, D, W, b_s, K_l_max, pool_k, -1, &L)) {
    set_error(KVC_ERR_CUDA, "no CUDA device to size the workspace for");
    return 0;
  }
  return L.total;
}

int kvc_score_pass1(const kvc_bf16* q_win, const kvc_bf16* k, int B, int H_q, int H_kv, int S, int D, int W,
                    int b_s, float* m, float* Z, void* ws, size_t ws_bytes, kvc_stream_t stream) {
  int rc;
  if ((rc = check_shapes(B, H_q, H_kv, S, D, W)) || (rc = check_bs(b_s))) return rc;
  if ((rc = check_ptr(q_win, 16, "q_win")) || (rc = check_ptr(k, 16, "k")) || (rc = check_ptr(m, 4, "m")) ||
      (rc = check_ptr(Z, 4, "Z")))
    return rc;
  WsLayout L;
  if (!layout_ws(B, H_q, H_kv, D, W, b_s, 0, 1, S, &L)) return set_error(KVC_ERR_CUDA, "no CUDA device");
  if ((rc = check_ws(ws, ws_bytes, L.off_part_z + (size_t)L.slots * L.gwp * sizeof(float)))) return rc;
  char* w = static_cast<char*>(ws);
  float* pm = reinterpret_cast<float*>(w + L.off_part_m);
  float* pz = reinterpret_cast<float*>(w + L.off_part_z);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  auto q = reinterpret_cast<const __nv_bfloat16*>(q_win);
  auto kk = reinterpret_cast<const __nv_bfloat16*>(k);
  if ((rc = launch_status(launch_pass1(q, kk, B, H_q, H_kv, S, D, W, L.plan, L.gwp, pm, pz, true, st), "pass 1 launch")))
    return rc;
  return launch_status(launch_pass1_combine(pm, pz, B, H_q, H_kv, S, W, L.plan, L.gwp, m, Z, st),
                       "pass 1 combine launch");
}

int kvc_score_pass2_pool(const kvc_bf16* q_win, const kvc_bf16* k, const float* m, const float* Z, int B, int H_q,
                         int H_kv, int S, int D, int W, int b_s, int pool_k, float* scores, void* ws,
                         size_t ws_bytes, kvc_stream_t stream) {
  int rc;
  if ((rc = check_shapes(B, H_q, H_kv, S, D, W)) || (rc = check_bs(b_s)) || (rc = check_pool(pool_k))) return rc;
  if ((rc = check_ptr(q_win, 16, "q_win")) || (rc = check_ptr(k, 16, "k")) || (rc = check_ptr(m, 4, "m")) ||
      (rc = check_ptr(Z, 4, "Z")) || (rc = check_ptr(scores, 4, "scores")))
    return rc;
  WsLayout L;
  if (!layout_ws(B, H_q, H_kv, D, W, b_s, 0, pool_k, S, &L)) return set_error(KVC_ERR_CUDA, "no CUDA device");
  SelParams sp{};
  sp.S = S;
  sp.H_kv = H_kv;
  if ((rc = check_ws(ws, ws_bytes, L.off_bias + (size_t)B * H_kv * L.gwp * sizeof(float)))) return rc;
  Pass2Out out{scores, nullptr, nullptr, 0};
  float* bias = reinterpret_cast<float*>(static_cast<char*>(ws) + L.off_bias);
  return launch_status(launch_pass2(reinterpret_cast<const __nv_bfloat16*>(q_win),
                                    reinterpret_cast<const __nv_bfloat16*>(k), m, Z, nullptr, nullptr, bias, B, H_q,
                                    H_kv, S, D, W, pool_k, L.plan, L.gwp, &sp, out, false,
                                    reinterpret_cast<cudaStream_t>(stream)),
                       "pass 2 launch");
}

int kvc_score_rawdot_int8(const kvc_bf16* q_win, const kvc_bf16* k, int B, int H_q, int H_kv, int S, int D,
                          int W, float* scores, void* ws, size_t ws_bytes, kvc_stream_t stream) {
  int rc;
  if ((rc = check_shapes(B, H_q, H_kv, S, D, W))) return rc;
  if ((rc = check_ptr(q_win, 16, "q_win")) || (rc = check_ptr(k, 16, "k")) || (rc = check_ptr(scores, 4, "scores")))
    return rc;
  const size_t BH = (size_t)B * H_kv;
  if ((rc = check_ws(ws, ws_bytes, BH * (size_t)D * sizeof(float)))) return rc;
  return launch_status(launch_rawdot_int8(reinterpret_cast<const __nv_bfloat16*>(q_win),
                                          reinterpret_cast<const __nv_bfloat16*>(k), B, H_q, H_kv, S, D, W,
                                          static_cast<float*>(ws), scores, reinterpret_cast<cudaStream_t>(stream)),
                       "INT8 raw-product scorer launch");
}

int kvc_select_topk(const float* scores, int B, int H_kv, int S, const int32_t* K_l, const int64_t* out_off,
                    int sink, int recent, int32_t* idx, void* ws, size_t ws_bytes, kvc_stream_t stream) {
  int rc;
  if (B < 1 || H_kv < 1 || S < 1) return set_error(KVC_ERR_INVALID_ARG, "B, H_kv and S must be >= 1");
  if (H_kv > kMaxHkv) return set_error(KVC_ERR_UNSUPPORTED, "H_kv=%d above %d", H_kv, kMaxHkv);
  if ((rc = check_ptr(scores, 4, "scores")) || (rc = check_ptr(idx, 4, "idx"))) return rc;
  SelParams sp;
  if ((rc = make_sel(S, H_kv, K_l, out_off, sink, recent, &sp, nullptr))) return rc;
  (void)ws;
  (void)ws_bytes;
  sp.nparts = 1;
  return launch_status(launch_select(0, scores, nullptr, nullptr, 0, B, sp, idx, reinterpret_cast<cudaStream_t>(stream)),
                       "selection launch");
}

int kvc_gather(const kvc_bf16* k, const kvc_bf16* v, const int32_t* idx, const int64_t* out_off, int B, int H_kv,
               int S, int D, const int32_t* K_l, kvc_bf16* k_out, kvc_bf16* v_out, int32_t* pos_out,
               kvc_stream_t stream) {
  int rc;
  if (B < 1 || H_kv < 1 || S < 1) return set_error(KVC_ERR_INVALID_ARG, "B, H_kv and S must be >= 1");
  if (D != 64 && D != 128) return set_error(KVC_ERR_UNSUPPORTED, "head dim D=%d: only 64 and 128 are supported", D);
  if (H_kv > kMaxHkv) return set_error(KVC_ERR_UNSUPPORTED, "H_kv=%d above %d", H_kv, kMaxHkv);
  if ((rc = check_ptr(k, 16, "k")) || (rc = check_ptr(v, 16, "v")) || (rc = check_ptr(idx, 4, "idx")) ||
      (rc = check_ptr(k_out, 16, "k_out")) || (rc = check_ptr(v_out, 16, "v_out")) ||
      (rc = check_ptr(pos_out, 4, "pos_out")))
    return rc;
  SelParams sp{};
  sp.S = S;
  sp.H_kv = H_kv;
  if ((rc = make_layout(S, H_kv, K_l, out_off, 0, &sp))) return rc;
  return launch_status(
      launch_gather(reinterpret_cast<const __nv_bfloat16*>(k), reinterpret_cast<const __nv_bfloat16*>(v), idx, B, sp,
                    D, reinterpret_cast<__nv_bfloat16*>(k_out), reinterpret_cast<__nv_bfloat16*>(v_out), pos_out,
                    reinterpret_cast<cudaStream_t>(stream)),
      "gather launch");
}

int kvc_compress_layer(int N, int layer, int B, int S, int C, int H_q, int H_kv, int D, int W, const int32_t* K_l,
                       int sink, int recent, int pool_k, int b_s, const kvc_bf16* q_win, const kvc_bf16* k,
                       const kvc_bf16* v, kvc_bf16* k_out, kvc_bf16* v_out, int32_t* pos_out,
                       const int64_t* out_off, void* ws, size_t ws_bytes, kvc_stream_t stream) {
  return compress_layer(N, layer, B, S, C, H_q, H_kv, D, W, K_l, sink, recent, pool_k, b_s, q_win, k, v, k_out,
                        v_out, pos_out, out_off, ws, ws_bytes, nullptr, stream);
}

int kvc_compress_layer_deferred_v(int N, int layer, int B, int S, int C, int H_q, int H_kv, int D, int W,
                                  const int32_t* K_l, int sink, int recent, int pool_k, int b_s,
                                  const kvc_bf16* q_win, const kvc_bf16* k, const kvc_bf16* v, kvc_bf16* k_out,
                                  kvc_bf16* v_out, int32_t* pos_out, const int64_t* out_off, void* ws,
                                  size_t ws_bytes, kvc_event_t v_ready, kvc_stream_t stream) {
  return compress_layer(N, layer, B, S, C, H_q, H_kv, D, W, K_l, sink, recent, pool_k, b_s, q_win, k, v, k_out,
                        v_out, pos_out, out_off, ws, ws_bytes, reinterpret_cast<cudaEvent_t>(v_ready), stream);
}

int kvc_scan_ranges(int BH, int S, int P, int64_t* starts) {
  if (BH < 1 || S < 1 || P < 1) return set_error(KVC_ERR_INVALID_ARG, "BH, S and P must be >= 1");
  if (!starts) return set_error(KVC_ERR_INVALID_ARG, "starts must be non-NULL");
  const ScanPlan pl = plan_for(BH, S, P);
  const int64_t total = (int64_t)BH * S;
  for (int c = 0; c <= pl.P; ++c) starts[c] = range_begin(c, pl.L, S, total);
  return pl.P;
}

int kvc_retained_layout(int H_kv, int S, const int32_t* K_l, int64_t* out_off) {
  if (H_kv < 1 || S < 1) return set_error(KVC_ERR_INVALID_ARG, "H_kv and S must be >= 1");
  if (!K_l || !out_off) return set_error(KVC_ERR_INVALID_ARG, "K_l and out_off must be non-NULL");
  out_off[0] = 0;
  for (int h = 0; h < H_kv; ++h) {
    if (K_l[h] < 0) return set_error(KVC_ERR_INVALID_ARG, "K_l[%d] is negative", h);
    out_off[h + 1] = out_off[h] + std::min(K_l[h], S);
  }
  return KVC_OK;
}

int kvc_append_chunk(const kvc_bf16* k_chunk, const kvc_bf16* v_chunk, int B, int H_kv, int S, int C, int D, int j,
                     kvc_bf16* k_act, kvc_bf16* v_act, kvc_stream_t stream) {
  int rc;
  if (B < 1 || H_kv < 1 || S < 1 || C < 1) return set_error(KVC_ERR_INVALID_ARG, "B, H_kv, S and C must be >= 1");
  if (D != 64 && D != 128) return set_error(KVC_ERR_UNSUPPORTED, "head dim D=%d: only 64 and 128 are supported", D);
  if (j < 0 || (int64_t)j * C >= S)
    return set_error(KVC_ERR_INVALID_ARG, "chunk %d of size %d starts beyond S=%d", j, C, S);
  if ((rc = check_ptr(k_chunk, 16, "k_chunk")) || (rc = check_ptr(v_chunk, 16, "v_chunk")) ||
      (rc = check_ptr(k_act, 16, "k_act")) || (rc = check_ptr(v_act, 16, "v_act")))
    return rc;
  return launch_status(launch_append_chunk(reinterpret_cast<const __nv_bfloat16*>(k_chunk),
                                           reinterpret_cast<const __nv_bfloat16*>(v_chunk), B, H_kv, S, C, D, j,
                                           reinterpret_cast<__nv_bfloat16*>(k_act),
                                           reinterpret_cast<__nv_bfloat16*>(v_act),
                                           reinterpret_cast<cudaStream_t>(stream)),
                       "chunk append launch");
}

int kvc_cache_layout(int N, int B, int H_kv, int S, const int32_t* K_l, int64_t* layer_row_off) {
  if (N < 1 || B < 1 || H_kv < 1 || S < 1) return set_error(KVC_ERR_INVALID_ARG, "N, B, H_kv and S must be >= 1");
  if (!K_l || !layer_row_off) return set_error(KVC_ERR_INVALID_ARG, "K_l and layer_row_off must be non-NULL");
  layer_row_off[0] = 0;
  for (int l = 0; l < N; ++l) {
    int64_t T = 0;
    for (int h = 0; h < H_kv; ++h) {
      const int32_t k = K_l[(size_t)l * H_kv + h];
      if (k < 0) return set_error(KVC_ERR_INVALID_ARG, "K_l[%d][%d] is negative", l, h);
      T += std::min(k, S);
    }
    layer_row_off[l + 1] = layer_row_off[l] + (int64_t)B * T;
  }
  return KVC_OK;
}

int kvc_budget_pyramid(int N, int budget, int k_min, int32_t* K_l_out) {
  if (N < 1 || !K_l_out) return set_error(KVC_ERR_INVALID_ARG, "need N >= 1 and an output array");
  if (k_min < 0 || k_min > budget) return set_error(KVC_ERR_INVALID_ARG, "need 0 <= k_min <= budget");
  if (2 * (int64_t)budget - k_min > INT32_MAX)
    return set_error(KVC_ERR_INVALID_ARG, "first-layer budget 2*budget - k_min = %lld does not fit int32",
                     (long long)(2 * (int64_t)budget - k_min));
  if (N == 1) {
    K_l_out[0] = budget;
    return KVC_OK;
  }
  const double k_max = 2.0 * (double)budget - (double)k_min;
  std::vector<double> rem(N);
  std::vector<int64_t> base(N);
  int64_t assigned = 0;
  for (int l = 0; l < N; ++l) {
    const double exact = k_max - (k_max - (double)k_min) * (double)l / (double)(N - 1);
    base[l] = (int64_t)std::floor(exact);
    rem[l] = exact - (double)base[l];
    assigned += base[l];
  }
  std::vector<int> order(N);
  for (int l = 0; l < N; ++l) order[l] = l;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return rem[a] > rem[b]; });
  const int64_t total = (int64_t)N * budget;
  for (int64_t i = 0; i < total - assigned && i < N; ++i) base[order[i]] += 1;
  for (int l = 0; l < N; ++l) K_l_out[l] = (int32_t)base[l];
  return KVC_OK;
}

int kvc_budget_inverse_stability(int H_kv, const double* s_stable, int64_t total, int lo, int hi, int32_t* K_l_out) {
  if (H_kv < 1 || !s_stable || !K_l_out) return set_error(KVC_ERR_INVALID_ARG, "bad budget arguments");
  if (total < 0 || lo < 0 || hi < lo) return set_error(KVC_ERR_INVALID_ARG, "need total >= 0 and 0 <= lo <= hi");
  std::vector<double> w(H_kv), exact(H_kv), rem(H_kv);
  double wsum = 0.0;
  for (int h = 0; h < H_kv; ++h) {
    if (!(s_stable[h] > 0.0)) return set_error(KVC_ERR_INVALID_ARG, "stability score %d must be > 0", h);
    w[h] = 1.0 / s_stable[h];
    wsum += w[h];
    if (!std::isfinite(w[h]) || !std::isfinite(wsum))
      return set_error(KVC_ERR_INVALID_ARG, "stability score %d = %g: the inverse weights overflow fp64", h,
                       s_stable[h]);
  }
  std::vector<int64_t> base(H_kv);
  int64_t assigned = 0;
  for (int h = 0; h < H_kv; ++h) {
    exact[h] = (double)total * w[h] / wsum;
    if (!std::isfinite(exact[h]))
      return set_error(KVC_ERR_INVALID_ARG, "share of head %d overflows fp64 (total %lld, s = %g)", h,
                       (long long)total, s_stable[h]);
    base[h] = (int64_t)std::floor(exact[h]);
    rem[h] = exact[h] - (double)base[h];
    assigned += base[h];
  }
  std::vector<int> order(H_kv);
  for (int h = 0; h < H_kv; ++h) order[h] = h;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return rem[a] > rem[b]; });
  for (int64_t i = 0; i < total - assigned && i < H_kv; ++i) base[order[i]] += 1;
  for (int h = 0; h < H_kv; ++h) K_l_out[h] = (int32_t)std::min<int64_t>(std::max<int64_t>(base[h], lo), hi);
  return KVC_OK;
}

int kvc_overlap_coefficient(const int32_t* a, const int64_t* a_off, const int32_t* b, const int64_t* b_off,
                            int n_pairs, float* out, kvc_stream_t stream) {
  int rc;
  if (n_pairs < 0) return set_error(KVC_ERR_INVALID_ARG, "n_pairs must be >= 0");
  if (n_pairs == 0) return KVC_OK;
  if ((rc = check_ptr(a, 4, "a")) || (rc = check_ptr(b, 4, "b")) || (rc = check_ptr(a_off, 8, "a_off")) ||
      (rc = check_ptr(b_off, 8, "b_off")) || (rc = check_ptr(out, 4, "out")))
    return rc;
  if (n_pairs > (1 << 30)) return set_error(KVC_ERR_UNSUPPORTED, "n_pairs above 2^30");
  return launch_status(launch_overlap(a, a_off, b, b_off, n_pairs, out, reinterpret_cast<cudaStream_t>(stream)),
                       "overlap launch");
}

int kvc_head_similarity(const int32_t* idx, const int64_t* off, int n_groups, int H, float* sim,
                        kvc_stream_t stream) {
  int rc;
  if (n_groups < 1 || H < 1) return set_error(KVC_ERR_INVALID_ARG, "n_groups and H must be >= 1");
  if (H > 65535 || n_groups > 65535) return set_error(KVC_ERR_UNSUPPORTED, "n_groups and H must be <= 65535");
  if ((rc = check_ptr(idx, 4, "idx")) || (rc = check_ptr(off, 8, "off")) || (rc = check_ptr(sim, 4, "sim")))
    return rc;
  return launch_status(launch_similarity(idx, off, n_groups, H, sim, reinterpret_cast<cudaStream_t>(stream)),
                       "similarity launch");
}

static int check_steps(int T, int H) {
  if (T < 1 || H < 1) return set_error(KVC_ERR_INVALID_ARG, "T and H must be >= 1");
  if (T > kMaxDecodeSteps) return set_error(KVC_ERR_UNSUPPORTED, "T=%d above %d steps", T, kMaxDecodeSteps);
  if (H > 65535) return set_error(KVC_ERR_UNSUPPORTED, "H=%d above 65535", H);
  return KVC_OK;
}

int kvc_median_over_steps(const float* x, int T, int H, float* med, kvc_stream_t stream) {
  int rc;
  if ((rc = check_steps(T, H)) || (rc = check_ptr(x, 4, "x")) || (rc = check_ptr(med, 4, "med"))) return rc;
  return launch_status(launch_median(x, T, H, med, reinterpret_cast<cudaStream_t>(stream)), "median launch");
}

int kvc_head_stability_over_steps(const int32_t* dec_idx, const int64_t* dec_off, const int32_t* pre_idx,
                                  const int64_t* pre_off, int T, int H, float* per_step, float* stability,
                                  kvc_stream_t stream) {
  int rc;
  if ((rc = check_steps(T, H)) || (rc = check_ptr(dec_idx, 4, "dec_idx")) || (rc = check_ptr(dec_off, 8, "dec_off")) ||
      (rc = check_ptr(pre_idx, 4, "pre_idx")) || (rc = check_ptr(pre_off, 8, "pre_off")) ||
      (rc = check_ptr(per_step, 4, "per_step")) || (rc = check_ptr(stability, 4, "stability")))
    return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = launch_status(launch_stability_steps(dec_idx, dec_off, pre_idx, pre_off, T, H, per_step, st),
                          "stability overlap launch")))
    return rc;
  return launch_status(launch_median(per_step, T, H, stability, st), "median launch");
}

int kvc_head_similarity_over_steps(const int32_t* idx, const int64_t* off, int T, int H, float* per_step,
                                   float* similarity, kvc_stream_t stream) {
  int rc;
  if ((rc = check_steps(T, H)) || (rc = check_ptr(idx, 4, "idx")) || (rc = check_ptr(off, 8, "off")) ||
      (rc = check_ptr(per_step, 4, "per_step")) || (rc = check_ptr(similarity, 4, "similarity")))
    return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if ((rc = launch_status(launch_similarity(idx, off, T, H, per_step, st), "similarity launch"))) return rc;
  return launch_status(launch_median(per_step, T, H, similarity, st), "median launch");
}

int kvc_budget_inverse_stability_device(int n_layers, int H_kv, const double* s_stable, int64_t total, int lo,
                                        int hi, int32_t* K_l_out, kvc_stream_t stream) {
  int rc;
  if (n_layers < 1 || H_kv < 1) return set_error(KVC_ERR_INVALID_ARG, "n_layers and H_kv must be >= 1");
  if (H_kv > kMaxHkv) return set_error(KVC_ERR_UNSUPPORTED, "H_kv=%d above %d", H_kv, kMaxHkv);
  if (total < 0 || lo < 0 || hi < lo) return set_error(KVC_ERR_INVALID_ARG, "need total >= 0 and 0 <= lo <= hi");
  if ((rc = check_ptr(s_stable, 8, "s_stable")) || (rc = check_ptr(K_l_out, 4, "K_l_out"))) return rc;
  return launch_status(launch_budget(s_stable, n_layers, H_kv, total, lo, hi, K_l_out,
                                     reinterpret_cast<cudaStream_t>(stream)),
                       "budget launch");
}

int kvc_profile_begin(void) {
  g_prof = true;
  g_prof_used = 0;
  g_prof_launch_base = g_launch_count.load();
  return KVC_OK;
}

int kvc_profile_end(double* stage_ms, int64_t* calls, int64_t* launches) {
  g_prof = false;
  if (stage_ms)
    for (int i = 0; i < KVC_N_STAGES; ++i) stage_ms[i] = 0.0;
  if (calls) *calls = (int64_t)g_prof_used;
  if (launches) *launches = g_launch_count.load() - g_prof_launch_base;
  if (g_prof_used == 0) return KVC_OK;
  cudaError_t e = cudaEventSynchronize(g_prof_ev[g_prof_used - 1][KVC_N_STAGES]);
  if (e != cudaSuccess) return cuda_error(e, "profile event synchronize");
  for (size_t c = 0; c < g_prof_used; ++c) {
    for (int i = 0; i < KVC_N_STAGES; ++i) {
      float ms = 0.f;
      if ((e = cudaEventElapsedTime(&ms, g_prof_ev[c][i], g_prof_ev[c][i + 1])) != cudaSuccess)
        return cuda_error(e, "profile elapsed time");
      if (stage_ms) stage_ms[i] += ms;
    }
  }
  return KVC_OK;
}

int kvc_check_status(kvc_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "stream synchronize");
  int v = 0;
  if ((e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int))) != cudaSuccess) return cuda_error(e, "status read");
  const int zero = 0;
  if ((e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int))) != cudaSuccess) return cuda_error(e, "status clear");
  if (v == kStatusOk) return KVC_OK;
  if (v == kStatusTimeout) return set_error(KVC_ERR_TIMEOUT, "a device wait gave up");
  return set_error(KVC_ERR_DEVICE, "kernel status %d (%s)", v,
                   v == kStatusCandOverflow   ? "candidate list overflow"
                   : v == kStatusBadInput     ? "a device-resident input broke the contract"
                                              : "selection count mismatch");
}

}  // extern "C"
