/*
 * kvc.h -- C ABI of the layer-end KV-cache compressor (GB300, sm_103a).
 *
 * The library scores every prefix key of a layer by how much attention the
 * last W prompt positions (the observation window) pay to it, and keeps, per
 * KV head, a fixed number of keys: the sink and recent keys plus the best
 * scoring others.  It is TideKV's memory-controlled two-pass blockwise scorer
 * ("TideKV: Delayed KV Eviction via Layer-Wise Chunked Prefill", Fig. 3),
 * with unequal per-head budgets as in HeteroCache's inverse-stability
 * allocation (HeteroCache summary, Phase 2).
 *
 * Notation (TideKV, Table 1): N layers, B batch, S prompt length, C prefill
 * chunk, H_q query heads, H_kv KV heads, D head dim.  G = H_q / H_kv query
 * heads share one KV head; query head g reads KV head g / G.  W is the
 * observation window (window query i sits at absolute position
 * t_i = S - W + i and attends to keys j <= t_i), b_s the key block of the
 * scan, K_l the per-head budget, sink/recent the mandatory set
 * R_mand = [0, sink) u [S - recent, S), pool_k the average-pool width.
 *
 * Conventions for every call
 *  - Tensor pointers are DEVICE pointers owned by the caller, contiguous
 *    row-major in the shapes given; bf16 tensors are 16-byte aligned, fp32
 *    and int32 tensors 4-byte aligned.  Budget arrays (K_l) and stability
 *    scores are HOST arrays.
 *  - The library allocates no device memory.  Scratch comes from the
 *    caller's `ws` buffer of at least kvc_workspace_size(...) bytes (256-byte
 *    aligned).  Its size does not depend on S.
 *  - Calls are asynchronous on `stream` (NULL = legacy default stream) and
 *    return KVC_OK once the work is enqueued.  All arguments are validated on
 *    the host before anything is launched; on error nothing is launched and
 *    kvc_last_error() describes the problem.
 *  - Kernels never trap.  A kernel that detects an inconsistency records a
 *    code in a device status word; kvc_check_status() reads and clears it.
 *  - Calls on one stream may run back to back; two calls that share a `ws`
 *    buffer must not overlap on the GPU.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t kvc_bf16;                 /* raw bfloat16 bits */
typedef struct CUstream_st* kvc_stream_t;  /* the same type as cudaStream_t */
typedef struct CUevent_st* kvc_event_t;    /* the same type as cudaEvent_t */

enum kvc_status_code {
  KVC_OK = 0,
  KVC_ERR_INVALID_ARG = -1,  /* a size, pointer or budget breaks the contract */
  KVC_ERR_UNSUPPORTED = -2,  /* valid, but outside what the kernels handle
                                (D not 64/128, G*W > 256, pool_k > 15, H_kv > 128) */
  KVC_ERR_WORKSPACE = -3,    /* ws missing, misaligned or too small */
  KVC_ERR_CUDA = -4,         /* a CUDA runtime call failed (message has details) */
  KVC_ERR_TIMEOUT = -5,      /* a bounded device wait gave up */
  KVC_ERR_DEVICE = -6        /* a kernel recorded an inconsistency */
};

/* Message of the last failed call on this host thread ("" if none). */
const char* kvc_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int kvc_version(void);

/*
 * Bytes of scratch every entry point below needs for these sizes on the
 * current device.  There is no S argument: the scan keeps only W-length
 * normaliser state per key range and, per key range, at most K_l_max + b_s
 * candidate keys (TideKV Fig. 3: Temp = O(W b_s + K_l), independent of S).
 * 128 <= b_s <= 2^29; K_l_max above 2^30 (the largest S) sizes as 2^30.
 * Returns 0 and sets kvc_last_error() on invalid sizes or without a device.
 */
size_t kvc_workspace_size(int B, int H_q, int H_kv, int D, int W, int b_s,
                          int K_l_max, int pool_k);

/*
 * Pass 1 of the two-pass scorer (TideKV Fig. 3): scan the prefix keys block
 * by block against the window queries and keep only the log-sum-exp
 * normalisers of each window query.
 *   q_win [B, H_q, W, D] bf16   the window queries (last W prompt positions)
 *   k     [B, H_kv, S, D] bf16  the layer's prefix keys
 *   m     [B, H_q, W] fp32 out  m = max_{j <= t_i} q.k_j / sqrt(D)
 *   Z     [B, H_q, W] fp32 out  Z = sum_{j <= t_i} exp(q.k_j / sqrt(D) - m)
 * b_s must be >= 128 and <= 2^29 (KVC_ERR_UNSUPPORTED above).
 */
int kvc_score_pass1(const kvc_bf16* q_win, const kvc_bf16* k, int B, int H_q,
                    int H_kv, int S, int D, int W, int b_s, float* m, float* Z,
                    void* ws, size_t ws_bytes, kvc_stream_t stream);

/*
 * kvc_score_pass1 without a workspace, for callers that cannot allocate
 * device memory: code inside a framework that owns all device memory through
 * its own pool (a cudaMalloc there fails or breaks the pool's accounting),
 * and plugin or real-time paths that may not call the CUDA allocator, whose
 * cudaMalloc/cudaFree can synchronise the whole device.  The pages have no
 * counterpart of this call; it only changes where the scratch lives.
 *
 * Same arguments and results as kvc_score_pass1, minus ws.  The scratch is a
 * fixed 1 MiB array in the library's device memory, present on every GPU
 * that loads the library until the process exits; nothing is allocated.
 * Shapes with B * H_kv * roundup16(G*W) * 8 bytes above 1 MiB are rejected
 * with KVC_ERR_UNSUPPORTED before any launch.  The first call on each device
 * looks up the array's device address (cudaGetSymbolAddress) with that
 * device current; make that first call before any stream capture.  Every
 * call shares the array: calls whose kernels could overlap on the GPU race
 * and must be serialised by the caller.
 */
int kvc_score_pass1_noalloc(const kvc_bf16* q_win, const kvc_bf16* k, int B,
                            int H_q, int H_kv, int S, int D, int W, int b_s,
                            float* m, float* Z, kvc_stream_t stream);

/*
 * Pass 2 plus pooling (TideKV Fig. 3): rescan the keys, form the normalised
 * weights exp(q.k/sqrt(D) - m) / Z, sum them over the window queries and the
 * GQA group of each KV head (r_j), and average-pool r into per-key scores
 *   s_j = (1/pool_k) * sum_{|d| <= (pool_k-1)/2} r_{j+d}   (r = 0 outside [0,S)).
 *   m, Z    [B, H_q, W] fp32 from kvc_score_pass1
 *   scores  [B, H_kv, S] fp32 out
 * pool_k is odd, 1 <= pool_k <= 15 (1 = no pooling).
 */
int kvc_score_pass2_pool(const kvc_bf16* q_win, const kvc_bf16* k,
                         const float* m, const float* Z, int B, int H_q,
                         int H_kv, int S, int D, int W, int b_s, int pool_k,
                         float* scores, void* ws, size_t ws_bytes,
                         kvc_stream_t stream);

/*
 * Single-pass raw inner-product scores with INT8 keys (HillInfer,
 * "Algorithmic Simplification" and "Streaming Execution and Asymmetric
 * Precision"): no exponentials and no 1/sqrt(D), one read of K.
 *   q_win  [B, H_q, W, D] bf16; the scoring query of KV head h is the
 *          float32 sum of its group's G*W window rows, in row order
 *   k      [B, H_kv, S, D] bf16
 *   scores [B, H_kv, S] fp32 out (any sign):
 *          float32(float32(dot_j) * scale_q) * scale_k, where each row (the
 *          scoring query, each key) is cast to symmetric INT8 with
 *          code = rint(x * (127 / max|x|)) in [-127, 127], scale = max|x| /
 *          127, and dot_j is the exact integer product of the codes.
 *   ws     >= B*H_kv*D*4 bytes, 256-byte aligned (the scoring queries'
 *          float32 column sums); kvc_workspace_size(...) bytes always
 *          suffice.
 * Rank the scores with kvc_select_topk and fetch the full-precision rows
 * with kvc_gather.  Errors as for the other calls.
 */
int kvc_score_rawdot_int8(const kvc_bf16* q_win, const kvc_bf16* k, int B,
                          int H_q, int H_kv, int S, int D, int W,
                          float* scores, void* ws, size_t ws_bytes,
                          kvc_stream_t stream);

/*
 * Output layout shared by kvc_select_topk, kvc_gather and kvc_compress_layer
 * (TideKV Fig. 2: the layer's retained cache, one block of rows per batch
 * element).  out_off is a HOST int64 array [H_kv + 1], or NULL:
 *  - NULL: the packed layout of kvc_retained_layout -- head h owns rows
 *    off[h] .. off[h] + min(K_l[h], S) - 1, heads back to back, and a batch
 *    element's block is T = sum_h min(K_l[h], S) rows long.
 *  - given: head h fills min(K_l[h], S) rows starting at row out_off[h] of
 *    its batch element's block, and the block is out_off[H_kv] rows long
 *    (batch element b starts at row b * out_off[H_kv]).  A caller can so
 *    keep fixed-size per-head slots (e.g. out_off[h] = h * K_max) or
 *    leading room; rows a head does not fill are left untouched.  Required:
 *    out_off[0] >= 0, out_off[h] + min(K_l[h], S) <= out_off[h+1];
 *    otherwise KVC_ERR_INVALID_ARG before any launch.
 */

/*
 * Per-head selection (TideKV Fig. 3): keep R_mand and the top
 * (K_l[h] - |R_mand|) other keys by (score descending, index ascending).
 *   scores  [B, H_kv, S] fp32, finite, any sign (-0 ranks as +0)
 *   K_l     HOST [H_kv]; K_l[h] >= |R_mand|.  A head with K_l[h] >= S keeps
 *           every key.
 *   out_off HOST [H_kv + 1] or NULL: the output layout (above)
 *   idx     out, int32 positions, ascending within each head, in the
 *           layout out_off describes.
 */
int kvc_select_topk(const float* scores, int B, int H_kv, int S,
                    const int32_t* K_l, const int64_t* out_off, int sink,
                    int recent, int32_t* idx, void* ws, size_t ws_bytes,
                    kvc_stream_t stream);

/*
 * Gather of the retained cache (TideKV Fig. 2): copy K and V rows at the
 * selected positions and record the positions.
 *   k, v    [B, H_kv, S, D] bf16
 *   idx     int32 positions in the layout out_off and K_l describe (the
 *           first min(K_l[h], S) rows of each head's slot, values in [0,S))
 *   out_off HOST [H_kv + 1] or NULL: the output layout (above)
 *   k_out, v_out [B * T, D] bf16 out, pos_out [B * T] int32 out (T the
 *           block length of the layout); only the rows the heads fill are
 *           written
 * idx and pos_out may be the same buffer.
 */
int kvc_gather(const kvc_bf16* k, const kvc_bf16* v, const int32_t* idx,
               const int64_t* out_off, int B, int H_kv, int S, int D,
               const int32_t* K_l, kvc_bf16* k_out, kvc_bf16* v_out,
               int32_t* pos_out, kvc_stream_t stream);

/*
 * The whole layer-end compress of layer `layer` (TideKV Fig. 2 and 3):
 * pass 1, pass 2 with pooling, selection, gather -- the step that runs once
 * per layer after all of its prompt chunks, before the next layer starts.
 * N, layer and C are the pages' symbols and are only validated:
 * 0 <= layer < N and 1 <= W <= C <= S (the window is the tail of the last
 * chunk); C does not change the result.  Outputs as kvc_gather, in the
 * layout out_off describes (NULL: packed).
 * The per-head score vector is never materialised: each key range keeps a
 * candidate list of at most K_l_max + b_s keys in `ws`.
 */
int kvc_compress_layer(int N, int layer, int B, int S, int C, int H_q,
                       int H_kv, int D, int W, const int32_t* K_l, int sink,
                       int recent, int pool_k, int b_s,
                       const kvc_bf16* q_win, const kvc_bf16* k,
                       const kvc_bf16* v, kvc_bf16* k_out, kvc_bf16* v_out,
                       int32_t* pos_out, const int64_t* out_off, void* ws,
                       size_t ws_bytes, kvc_stream_t stream);

/*
 * kvc_compress_layer for callers that upload the values while the scans
 * run.  In the compress only the final gather reads v (pass 1, pass 2 and
 * the selection read q_win and k).  Here the gather first waits on v_ready:
 * an event the caller records after v is complete, typically on the stream
 * that copies v from the host, so that the copy overlaps the scans.
 *   v_ready  caller-owned CUDA event, or NULL for no wait (then this call
 *            is kvc_compress_layer itself).  The library only waits on it
 *            (cudaStreamWaitEvent on `stream`) and does not keep it.
 * Arguments, results and errors otherwise as kvc_compress_layer; q_win and
 * k must be complete in stream order, as there.
 */
int kvc_compress_layer_deferred_v(int N, int layer, int B, int S, int C,
                                  int H_q, int H_kv, int D, int W,
                                  const int32_t* K_l, int sink, int recent,
                                  int pool_k, int b_s, const kvc_bf16* q_win,
                                  const kvc_bf16* k, const kvc_bf16* v,
                                  kvc_bf16* k_out, kvc_bf16* v_out,
                                  int32_t* pos_out, const int64_t* out_off,
                                  void* ws, size_t ws_bytes,
                                  kvc_event_t v_ready, kvc_stream_t stream);

/*
 * Overlap coefficient of index sets (HeteroCache, "Key Contributions" 1 and
 * "Methodology", Phase 1): out[i] = |A_i n B_i| / min(|A_i|, |B_i|), fp32
 * (|A n B| and the minimum are exact integers, divided once in float32),
 * 0 when either set is empty.  The measure behind HeteroCache's stability
 * score (a head's decoding top-k against its prefill set).
 *   a, b          int32 positions; set i is a[a_off[i] .. a_off[i+1]-1], each
 *                 set ascending and without duplicates (as kvc_select_topk
 *                 writes them)
 *   a_off, b_off  int64 [n_pairs + 1], device
 *   out           fp32 [n_pairs], device
 */
int kvc_overlap_coefficient(const int32_t* a, const int64_t* a_off,
                            const int32_t* b, const int64_t* b_off,
                            int n_pairs, float* out, kvc_stream_t stream);

/*
 * HeteroCache's similarity score of every head (Phase 1): for each group g
 * (say a batch element of one layer) of H index sets and each head i,
 * sim[g*H + i] = max over j != i of the overlap coefficient of sets i and j
 * (0 when H = 1).
 *   idx  int32 positions, sets as in kvc_overlap_coefficient
 *   off  int64 [n_groups][H + 1], device: set (g, i) is
 *        idx[off[g][i] .. off[g][i+1]-1]
 *   sim  fp32 [n_groups * H], device
 */
int kvc_head_similarity(const int32_t* idx, const int64_t* off, int n_groups,
                        int H, float* sim, kvc_stream_t stream);

/*
 * HeteroCache's Phase-1 scores over decoding steps (HeteroCache summary,
 * "Methodology", Phase 1): the stability score of a head is the median over
 * T decoding steps of the overlap coefficient between its top-k at that
 * step and its prefill set; the similarity score is the median over the
 * same steps of the largest overlap with another head of its layer.  Median
 * of T fp32 values: the middle one for odd T; for even T the two middle
 * ones averaged exactly (fp64) and rounded once to fp32; -0 counts as +0,
 * NaN gives NaN.  1 <= T <= 4096 (else KVC_ERR_UNSUPPORTED), 1 <= H <= 65535.
 *
 * kvc_median_over_steps: x fp32 [T][H], device -> med fp32 [H], device.
 */
int kvc_median_over_steps(const float* x, int T, int H, float* med,
                          kvc_stream_t stream);

/*
 *   dec_idx, dec_off  the decoding-step sets: set (t, h) is
 *                     dec_idx[dec_off[t*H + h] .. dec_off[t*H + h + 1] - 1]
 *                     (dec_off int64 [T*H + 1]); sets ascending, no
 *                     duplicates, as kvc_select_topk writes them
 *   pre_idx, pre_off  the prefill sets of the H heads (pre_off [H + 1])
 *   per_step          fp32 [T][H] out: the per-step overlaps (also the
 *                     scratch of the median; the caller owns it)
 *   stability         fp32 [H] out
 * All device pointers.
 */
int kvc_head_stability_over_steps(const int32_t* dec_idx,
                                  const int64_t* dec_off,
                                  const int32_t* pre_idx,
                                  const int64_t* pre_off, int T, int H,
                                  float* per_step, float* stability,
                                  kvc_stream_t stream);

/*
 *   idx, off    step t's H sets, as kvc_head_similarity's groups: set (t, h)
 *               is idx[off[t][h] .. off[t][h+1] - 1], off int64 [T][H + 1]
 *   per_step    fp32 [T][H] out: each step's largest overlap per head
 *   similarity  fp32 [H] out
 * All device pointers.
 */
int kvc_head_similarity_over_steps(const int32_t* idx, const int64_t* off,
                                   int T, int H, float* per_step,
                                   float* similarity, kvc_stream_t stream);

/*
 * kvc_budget_inverse_stability on the device, for n_layers layers at once
 * (HeteroCache, Phase 2): the same float64 operations in the same order, so
 * the budgets equal the host function's.
 *   s_stable  fp64 [n_layers][H_kv], device, each > 0 and finite; a layer
 *             with a bad score gets lo everywhere and the status word records
 *             KVC_ERR_DEVICE (see kvc_check_status)
 *   K_l_out   int32 [n_layers][H_kv], device
 */
int kvc_budget_inverse_stability_device(int n_layers, int H_kv,
                                        const double* s_stable, int64_t total,
                                        int lo, int hi, int32_t* K_l_out,
                                        kvc_stream_t stream);

/*
 * Layer-major chunked prefill (TideKV, Fig. 1(d) and Fig. 2): write the keys
 * and values of prompt chunk j into the active layer's full-prompt buffer.
 *   k_chunk, v_chunk  [B, H_kv, c, D] bf16, c = min(C, S - j*C) positions
 *   k_act, v_act      [B, H_kv, S, D] bf16; positions j*C .. j*C + c - 1 of
 *                     every (b, head) are overwritten, the rest untouched
 * 0 <= j*C < S.  After the last chunk, kvc_compress_layer reads k_act/v_act
 * and may write straight into the cross-layer cache (kvc_cache_layout); the
 * active buffers are then free for the next layer.
 */
int kvc_append_chunk(const kvc_bf16* k_chunk, const kvc_bf16* v_chunk, int B,
                     int H_kv, int S, int C, int D, int j, kvc_bf16* k_act,
                     kvc_bf16* v_act, kvc_stream_t stream);

/*
 * Host helper: rows of the cross-layer retained cache C^[0..N-1] (TideKV,
 * Fig. 2 and Fig. 4).  Layer l occupies rows layer_row_off[l] ..
 * layer_row_off[l+1] - 1 of K^ / V^ ([rows, D]) and of the positions, laid out
 * inside as kvc_retained_layout describes (batch element b at b*T_l).
 *   K_l            HOST [N][H_kv] budgets (>= 0)
 *   layer_row_off  HOST [N + 1] out; layer_row_off[N] is the total row count
 */
int kvc_cache_layout(int N, int B, int H_kv, int S, const int32_t* K_l,
                     int64_t* layer_row_off);

/*
 * Host helper: per-layer budgets that shrink from the first layer to the
 * last, PyramidKV-style (TideKV's Tables 3-4 run TideKV-PyramidKV at
 * average budgets 256, 1024 and 4096; the pages give no schedule).  Reading:
 * a linear ramp from k_max = 2*budget - k_min at layer 0 down to k_min at
 * layer N-1 (mean = budget), rounded by largest remainder (ties to the
 * lower layer) so that the layers sum to exactly N * budget.
 *   K_l_out HOST [N]; 0 <= k_min <= budget, and the first layer's
 *   2*budget - k_min must fit int32 (else KVC_ERR_INVALID_ARG).  N = 1 gives
 *   budget.
 */
int kvc_budget_pyramid(int N, int budget, int k_min, int32_t* K_l_out);

/*
 * Host helper: CSR layout of one batch element's retained rows.
 * out_off HOST [H_kv + 1]: head h owns rows out_off[h] .. out_off[h+1]-1,
 * with min(K_l[h], S) rows; out_off[H_kv] is the per-batch-element stride T.
 */
int kvc_retained_layout(int H_kv, int S, const int32_t* K_l, int64_t* out_off);

/*
 * Host helper: the key ranges the two scans give their CTAs when P CTAs are
 * asked for (the library asks for the SM count).  The flattened key space
 * [BH][S] (BH = B * H_kv) is cut at c * L, L = ceil(BH*S / P), and a cut that
 * lies within min(L/4, 512) keys of a head boundary is moved onto it, so no
 * CTA spends a segment switch on a sliver of a head.
 *   starts HOST [P + 1] out: range c is keys starts[c] .. starts[c+1]-1 of
 *          the flattened space; starts[n] = BH * S.
 * Returns n, the number of ranges (1 <= n <= P), or a negative code on
 * invalid sizes (BH, S, P < 1) or a NULL pointer.  No device is touched.
 */
int kvc_scan_ranges(int BH, int S, int P, int64_t* starts);

/*
 * Host helper (HeteroCache summary, Phase 2): per-KV-head budgets
 * proportional to w_h = 1 / s_h.  The exact shares total * w_h / sum(w) are
 * rounded by largest remainder (ties to the lower head index) so that they
 * sum to `total`, then clamped to [lo, hi].  s_stable HOST [H_kv], > 0.
 * Scores so small that 1/s, the sum of the weights or a share overflows
 * fp64 are rejected with KVC_ERR_INVALID_ARG (the device variant does not
 * check this and leaves such budgets unspecified).
 */
int kvc_budget_inverse_stability(int H_kv, const double* s_stable,
                                 int64_t total, int lo, int hi,
                                 int32_t* K_l_out);

/*
 * Waits for `stream`, then reads and clears the device status word.
 * Returns KVC_OK, or KVC_ERR_DEVICE / KVC_ERR_TIMEOUT with a message.
 */
int kvc_check_status(kvc_stream_t stream);

/* Tuning knobs (process-wide, not thread-safe; 0 restores the default). */
enum kvc_option {
  KVC_OPT_SCAN_CTAS = 1,  /* CTAs (key ranges) of the two scans; default: the SM count */
  KVC_OPT_WAIT_LIMIT = 2  /* polls before a wait inside a scan pipeline gives up and the
                             call ends with KVC_ERR_TIMEOUT (kvc_check_status); default
                             2^22.  A wait that gives up stops the CTA's pipeline; the
                             copies and MMAs it already issued are waited for before the
                             CTA leaves.  Results of such a call are undefined. */
};
int kvc_set_option(int option, int64_t value);

/*
 * Stage timing of kvc_compress_layer, for measurement.  Between
 * kvc_profile_begin() and kvc_profile_end() every kvc_compress_layer call
 * records CUDA events on its own stream around its stages (0 pass 1,
 * 1 pass 2 + pooling + candidate lists, 2 selection, 3 gather).
 * kvc_profile_end waits for the last recorded event and returns, per stage,
 * the device time summed over the recorded calls (stage_ms[KVC_N_STAGES]),
 * the number of calls and the number of kernels (and memsets) the library
 * launched meanwhile.  Events are created once and reused; process-wide,
 * not thread-safe.
 */
#define KVC_N_STAGES 4
int kvc_profile_begin(void);
int kvc_profile_end(double* stage_ms, int64_t* calls, int64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
