/*
 * focus.h -- C ABI of the Focus attention inference path on GB300 (sm_103a).
 *
 * Focus (arXiv 2604.03260, "Why Attend to Everything? Focus is the Key")
 * restricts causal attention to the token pairs (i, j), j <= i, that lie in a
 * local window (i - j < window) or share at least one of their top-k learned
 * centroid groups.  Sources, web summaries of the paper:
 *   gist.science/zh, technical summary 2.1.1 (token grouping), 2.1.2 (gated
 *   attention: local window or shared group), 2.1.3 (inference: hard top-k
 *   groups, within-group causal attention plus cross-group local attention);
 *   gist.science/nl, Technische samenvatting, Kerncomponenten 1, 3, 4.
 *
 * Conventions shared by every entry point
 *   - Data pointers are DEVICE pointers to caller-owned memory unless a
 *     function says otherwise; all must be 16-byte aligned.  The library never
 *     allocates, frees or synchronises; it only enqueues work on `stream`
 *     (a cudaStream_t; NULL = the legacy default stream).
 *   - bf16 tensors are passed as `const void *` (IEEE bfloat16, row-major).
 *   - Arguments are validated on the host before anything is launched.  A
 *     non-zero status means nothing was enqueued, except FOCUS_ERR_CUDA, which
 *     reports a launch error (work enqueued before it may still run).
 *   - Device-side waits inside the kernels are bounded.  A wait that runs out
 *     makes the kernel finish early and records FOCUS_ERR_TIMEOUT in a device
 *     status word, read with focus_get_device_status().
 *   - Index types are int32: B * n * topk must stay below 2^31.
 */
#ifndef FOCUS_GB300_H
#define FOCUS_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int focus_status_t;
#define FOCUS_OK                 0
#define FOCUS_ERR_INVALID_ARG    1   /* null/misaligned pointer, bad size   */
#define FOCUS_ERR_UNSUPPORTED    2   /* valid but outside supported shapes  */
#define FOCUS_ERR_WORKSPACE      3   /* workspace smaller than required     */
#define FOCUS_ERR_CUDA           4   /* a CUDA runtime/launch error         */
#define FOCUS_ERR_TIMEOUT        5   /* a bounded device wait ran out       */
#define FOCUS_ERR_CAPACITY       6   /* a decode group list was full        */

/* Human-readable name of a status code (static storage). */
const char *focus_status_string(focus_status_t status);

/* Library version string, e.g. "focus-gb300 0.1.0 sm_103a". */
const char *focus_version(void);

/*
 * focus_assign -- centroid scoring and hard top-k group membership.
 * gist.science/zh 2.1.1: hidden states are projected into centroid space and
 * scored against every centroid; 2.1.3 and gist.science/nl Kerncomponent 4:
 * at inference a token belongs to its k highest-scoring groups.
 *
 *   z_i = x_i W_g (d_g values), s_{i,c} = z_i . C_c, ids_i = the topk
 *   largest s_{i,.} in descending order, equal scores -> lower id first.
 *
 *   X      [B, n, hidden]  bf16        hidden states
 *   Wg     [hidden, d_g]   fp32        projection into centroid space
 *   C      [K, d_g]        fp32        centroids of this layer
 *   ids    [B, n, topk]    int32 out   group ids by descending score
 *   margin [B, n]          fp32 out    nullable: smallest gap between
 *                          consecutive scores among the top min(topk+1, K)
 *                          (+inf when K == 1); a small margin flags a
 *                          near-tie whose order depends on rounding.
 *   ws, ws_bytes: device workspace of at least
 *          focus_assign_workspace_size(B, n, hidden, d_g, K, topk) bytes (may
 *          be NULL when that size is 0).
 * Arithmetic: fp32-accurate scores on the tensor cores where hidden % 64 == 0
 * and K <= 256 (X is exact in bf16; fp32 factors are split into two bf16 or
 * fp16 parts; fp32 accumulation), in one of two orders:
 *   - more centroids than centroid dimensions (K > d_g rounded up to 64,
 *     d_g <= 128): the pages' order, Z = X W_g, then Z C^T, with each row of
 *     Z scaled by a power of two and split into two fp16 parts;
 *   - otherwise X (W_g C^T), with W_g C^T formed once per call.
 * Other shapes use an fp32 FMA kernel for (X W_g) C^T.  Rounding differs
 * from an exact evaluation only below the margin, so ids can differ only
 * where the margin is tiny.
 * Supported: hidden % 8 == 0, 1 <= d_g <= 256, 1 <= K <= 1024,
 *            1 <= topk <= min(K, 8).
 */
size_t focus_assign_workspace_size(int B, int n, int hidden, int d_g, int K, int topk);
focus_status_t focus_assign(const void *X, const float *Wg, const float *C,
                            int B, int n, int hidden, int d_g, int K, int topk,
                            int32_t *ids, float *margin,
                            void *ws, size_t ws_bytes, void *stream);

/*
 * focus_bucket -- per-group member lists (histogram, exclusive scan, stable
 * scatter).  Implied by running "within-group causal attention"
 * (gist.science/zh 2.1.3) over each group's members as one dense problem.
 *
 *   ids     [B, n, topk]  int32 in   (values in [0, K); the topk ids of a
 *                                     token must be distinct)
 *   offsets [B, K+1]      int32 out  offsets[b][g] = number of memberships
 *                                     of groups < g in batch b
 *   pos     [B, n*topk]   int32 out  pos[b][offsets[b][g] + r] = r-th
 *                                     smallest token of group g
 *   inv     [B, n, topk]  int32 out  index in pos[b] of (i, ids[b][i][s])
 *   ws, ws_bytes: device workspace of at least
 *                 focus_bucket_workspace_size(B, n, K, topk) bytes.
 * Result is exact integer data (deterministic).
 * Supported: 1 <= K <= 1024, 1 <= topk <= 8.
 */
size_t focus_bucket_workspace_size(int B, int n, int K, int topk);
focus_status_t focus_bucket(const int32_t *ids, int B, int n, int K, int topk,
                            int32_t *offsets, int32_t *pos, int32_t *inv,
                            void *ws, size_t ws_bytes, void *stream);

/*
 * focus_bucket_static -- focus_bucket without a workspace argument, for
 * callers that cannot allocate device memory themselves: code that runs
 * where cudaMalloc is not allowed, such as inside another allocator's
 * callback, or in an engine that reserves the device's memory up front and
 * forbids further allocations while it executes.  (The paper has no
 * counterpart; this is an interface convenience.)
 *
 * Same arguments, results and validation as focus_bucket, minus ws/ws_bytes.
 * The scratch it needs lives in one fixed array of 16 MiB of device memory
 * inside the library, which every GPU that loads the library keeps until the
 * process exits.  Problems whose scratch, focus_bucket_workspace_size(B, n,
 * K, topk), exceeds 16 MiB are rejected with FOCUS_ERR_UNSUPPORTED (that
 * limit is far above the sizes this library targets: n = 1M, K = 256 needs
 * about 0.5 MiB).  The call allocates and frees nothing.
 *
 * The first call on a device looks up the array's device address (a runtime
 * query, once per device); make that first call before any stream capture.
 * All calls share the one array and each call overwrites the parts it uses
 * before reading them, so calls that overlap on the GPU (on different
 * streams, or from different host threads at once) race: serialise them.
 */
focus_status_t focus_bucket_static(const int32_t *ids, int B, int n, int K, int topk,
                                   int32_t *offsets, int32_t *pos, int32_t *inv,
                                   void *stream);

/*
 * focus_attention_fwd -- exact softmax attention over the allowed pairs
 * (gist.science/nl Kerncomponent 3: exact softmax within the allowed pairs;
 * gist.science/zh 2.1.2-2.1.3: local window or shared group, causal).
 *
 *   A_i = { j <= i : i - j < window  or  ids_i and ids_j share a group }
 *   O_i = sum_{j in A_i} softmax_j(scale * q_i . k_j) v_j
 *   lse_i = ln sum_{j in A_i} exp(scale * q_i . k_j)
 *
 * Executed as three tcgen05/TMEM kernels: a sliding-window attention over
 * every pair with i - j < window, a causal attention over every group's
 * gathered members that takes the pairs with i - j >= window (a pair shared
 * through several groups is counted only in the lowest shared group), and a
 * log-sum-exp merge of the partial results.
 *
 *   Q      [B, n, Hq, d]   bf16      K, V [B, n, Hkv, d] bf16
 *          query head h reads kv head h / (Hq / Hkv)
 *   window w >= 0 (0: group pairs only; the token itself is always allowed)
 *   scale  softmax scale; <= 0 selects 1/sqrt(d)
 *   ids, offsets, pos, inv: as produced by focus_assign / focus_bucket
 *   O      [B, n, Hq, d]   bf16 out
 *   lse    [B, Hq, n]      fp32 out, nullable (natural log)
 *   ws, ws_bytes: device workspace of at least
 *          focus_attention_workspace_size(B, n, Hq, Hkv, d, K, topk) bytes.
 * Arithmetic: bf16 operands, fp32 accumulation and softmax, probabilities
 * rounded to bf16 for the P.V product, partial outputs kept in fp16 with a
 * power-of-two scale per row (11-bit significand at any magnitude).
 * Supported: d in {64, 128}, Hq % Hkv == 0, 1 <= topk <= 8,
 *            1 <= K <= 1024 (the group kernel's shared memory holds the
 *            group bitmaps of two key tiles, 16 K bytes each, next to the
 *            Q/K/V tiles), B * K <= 4096 (the work list is sorted by one
 *            block with every group of every batch in shared memory).
 *            Otherwise FOCUS_ERR_UNSUPPORTED.
 */
size_t focus_attention_workspace_size(int B, int n, int Hq, int Hkv, int d,
                                      int K, int topk);
focus_status_t focus_attention_fwd(const void *Q, const void *K, const void *V,
                                   int B, int n, int Hq, int Hkv, int d,
                                   int window, float scale,
                                   const int32_t *ids, const int32_t *offsets,
                                   const int32_t *pos, const int32_t *inv,
                                   int num_groups, int topk,
                                   void *O, float *lse,
                                   void *ws, size_t ws_bytes, void *stream);

/*
 * focus_prefill -- the whole path in one call: focus_assign, focus_bucket and
 * focus_attention_fwd on one stream.  With io_on_host != 0, X, Wg, C, Q, K, V
 * are HOST pointers (page-locked for asynchronous copies), O and lse are host
 * pointers, and the copies in and out are enqueued around the kernels (the
 * caller synchronises `stream` before reading O).  The copies of K, V and Q
 * run on a second stream that the library creates once per device, after the
 * copy of X and beside the assignment; `stream` waits for K and V before the
 * gather and for Q before the group kernel, and the copies start only after
 * the work already on `stream`.  With
 * io_on_host == 0 every pointer is a device pointer.  ids_out (nullable, device) receives the
 * group ids.  Workspace: focus_prefill_workspace_size(...) device bytes.
 */
size_t focus_prefill_workspace_size(int B, int n, int hidden, int Hq, int Hkv,
                                    int d, int d_g, int K, int topk,
                                    int io_on_host);
focus_status_t focus_prefill(const void *X, const float *Wg, const float *C,
                             const void *Q, const void *K, const void *V,
                             int B, int n, int hidden, int Hq, int Hkv, int d,
                             int d_g, int num_groups, int topk, int window,
                             float scale, void *O, float *lse, int32_t *ids_out,
                             void *ws, size_t ws_bytes, int io_on_host,
                             void *stream);

/*
 * Decode: one new token per sequence against a key/value cache.  At inference
 * a token belongs to its k highest-scoring groups (gist.science/nl
 * Kerncomponent 4; gist.science/zh 2.1.3) and attends with an exact softmax
 * to the keys in its local window or sharing one of its groups (nl
 * Kerncomponent 3; zh 2.1.2).  The cache's group memberships are kept as
 * per-group position lists that only grow:
 *   glen [B, K]        int32   entries in each group's list
 *   gpos [B, K, cap]   int32   token positions of group g in ascending order,
 *                              gpos[b][g][0 .. glen[b][g])
 *
 * focus_decode_lists_init -- the lists of the first n tokens, from their
 * bucketing (offsets [B, K+1], pos [B, n*topk] of focus_bucket).  cap is the
 * room of every list; a group larger than cap keeps its first cap members
 * and records FOCUS_ERR_CAPACITY in the device status word.
 */
focus_status_t focus_decode_lists_init(const int32_t *offsets, const int32_t *pos, int B, int n,
                                       int num_groups, int topk, int cap, int32_t *glen,
                                       int32_t *gpos, void *stream);

/*
 * focus_decode_fwd -- the new token i = L - 1 of every sequence: appends i to
 * the lists of its k groups, then computes its attention over
 *   A_i = { j <= i : i - j < window  or  ids_i and ids_j share a group }
 * as a split over the keys (window keys, and each shared key once, from the
 * list of the lowest shared group) with a log-sum-exp merge.
 *
 *   q      [B, Hq, d]        bf16   the new token's query
 *   Kc, Vc [B, Lmax, Hkv, d] bf16   the cache; row L - 1 holds the new token
 *   ids    [B, Lmax, topk]   int32  group ids of the cached tokens (row
 *                                   L - 1: the new token's, e.g. from
 *                                   focus_assign on its hidden state)
 *   glen, gpos, cap                 the group lists (updated in place); call
 *                                   once per new token
 *   O      [B, Hq, d]        bf16 out;  lse [B, Hq] fp32 out, nullable
 *   ws, ws_bytes: at least focus_decode_workspace_size(B, Hq, Hkv, d) bytes.
 * Arithmetic: fp32 scores, softmax and accumulation from bf16 inputs, O
 * rounded to bf16.  A list already holding cap entries is not appended to
 * and FOCUS_ERR_CAPACITY is recorded in the device status word.
 * Supported: d in {64, 128}, Hq % Hkv == 0 with Hq / Hkv <= 8,
 *            1 <= topk <= min(K, 8), K <= 1024, 1 <= L <= Lmax.
 */
size_t focus_decode_workspace_size(int B, int Hq, int Hkv, int d);
focus_status_t focus_decode_fwd(const void *q, const void *Kc, const void *Vc, const int32_t *ids,
                                int B, int L, int Lmax, int Hq, int Hkv, int d, int window,
                                float scale, int num_groups, int topk, int32_t *glen,
                                int32_t *gpos, int cap, void *O, float *lse, void *ws,
                                size_t ws_bytes, void *stream);

/*
 * focus_gated_attention_fwd / _bwd -- the soft-gated attention of training
 * over every causal pair (gist.science/zh technical summary 2.1.2 "gated
 * attention"; gist.science/nl Kerncomponent 4: soft gates over all pairs in
 * training), and its backward.  The page prints the score as
 *     s_ij = q_i . k_j * (1_local + (1 - 1_local) * sigma(lambda * a_ij));
 * readings: 1_local = [i - j < window], a_ij = g_i . g_j (the tokens' soft
 * group assignments, rows of G, e.g. P of focus_sinkhorn), q . k scaled by
 * `scale` (0 selects 1/sqrt(d)) before the gate, softmax over j <= i.
 *   Q [B, n, Hq, d], K and V [B, n, Hkv, d] bf16; G [B, n, Kg] fp32
 *   fwd: O [B, n, Hq, d] bf16 out; lse [B, Hq, n] fp32 out (natural log),
 *        needed by the backward
 *   bwd: O, lse from the forward; dO [B, n, Hq, d] bf16 (the gradient of the
 *        loss by O) -> dQ [B, n, Hq, d], dK and dV [B, n, Hkv, d],
 *        dG [B, n, Kg] fp32, *dlambda fp32 (one value, device), all overwritten
 *   ws, ws_bytes: at least focus_gated_workspace_size(B, n, Hq, Hkv, Kg) bytes.
 * Arithmetic: tensor-core tiles with fp32 accumulation: Q K^T, P V and the
 * gradient products in bf16, G G^T and the dG products in fp16; the gate,
 * softmax and dS in fp32.  The backward recomputes P from lse; every sum has
 * a fixed order (no atomics), so results repeat bit for bit.
 * Supported: d in {64, 128}, Hq % Hkv == 0, 1 <= Kg <= 128, window >= 0,
 * n >= 1.  Errors: FOCUS_ERR_INVALID_ARG (null or unaligned pointers, values
 * out of range), FOCUS_ERR_UNSUPPORTED, FOCUS_ERR_WORKSPACE; nothing is
 * launched then.
 */
size_t focus_gated_workspace_size(int B, int n, int Hq, int Hkv, int Kg);
focus_status_t focus_gated_attention_fwd(const void *Q, const void *K, const void *V,
                                         const float *G, int B, int n, int Hq, int Hkv, int d,
                                         int Kg, int window, float lambda, float scale, void *O,
                                         float *lse, void *ws, size_t ws_bytes, void *stream);
focus_status_t focus_gated_attention_bwd(const void *Q, const void *K, const void *V,
                                         const float *G, const void *O, const float *lse,
                                         const void *dO, int B, int n, int Hq, int Hkv, int d,
                                         int Kg, int window, float lambda, float scale,
                                         float *dQ, float *dK, float *dV, float *dG,
                                         float *dlambda, void *ws, size_t ws_bytes,
                                         void *stream);

/*
 * focus_sinkhorn -- Sinkhorn normalisation of the training-time token-group
 * affinities (gist.science/nl Kerncomponenten 2: group balance forced as a
 * hard structural constraint; gist.science/zh technical summary 2.1.1:
 * Sinkhorn instead of softmax, every group receiving an equal mass of
 * tokens).  For each sequence b, the kernel A = exp(S_b / tau) is scaled to
 * P = diag(u) A diag(v) by `iters` Sinkhorn-Knopp rounds from v = 1, each a
 * row update u_i = 1 / sum_c A_ic v_c then a column update
 * v_c = (n / K) / sum_i A_ic u_i: after every round each group's mass is
 * n / K, and each token's mass tends to 1 as rounds are added.
 *   S      [B, n, K] fp32 affinities (e.g. z_i . C_c), device
 *   tau    temperature > 0 (0 selects 1)
 *   iters  rounds, 1 <= iters <= 100000
 *   P      [B, n, K] fp32 out, nullable (then only the potentials)
 *   log_u  [B, n] fp32 out (natural log of u), nullable
 *   log_v  [B, K] fp32 out (natural log of v), nullable
 *   ws, ws_bytes: at least focus_sinkhorn_workspace_size(B, n, K) bytes.
 * Arithmetic: fp32, base-2 log-sum-exp per row; a group mass that
 * underflows float is taken as the smallest subnormal.  One read of S per
 * round, plus one read of S and one write of P at the end.
 * Supported: 1 <= K <= 1024, n >= 1, B >= 1.  Errors: FOCUS_ERR_INVALID_ARG
 * for null or unaligned (16-byte) pointers or values out of range,
 * FOCUS_ERR_WORKSPACE for a short workspace; nothing is launched then.
 */
size_t focus_sinkhorn_workspace_size(int B, int n, int K);
focus_status_t focus_sinkhorn(const float *S, int B, int n, int K, float tau, int iters,
                              float *P, float *log_u, float *log_v, void *ws, size_t ws_bytes,
                              void *stream);

/*
 * focus_dense_causal_fwd -- plain causal attention (every j <= i) with the
 * same tcgen05 mainloop; the baseline the sparse path is compared with.
 *   Q [B, n, Hq, d], K/V [B, n, Hkv, d] bf16; O [B, n, Hq, d] bf16;
 *   lse [B, Hq, n] fp32 nullable.  Supported: d in {64, 128}.
 */
focus_status_t focus_dense_causal_fwd(const void *Q, const void *K, const void *V,
                                      int B, int n, int Hq, int Hkv, int d,
                                      float scale, void *O, float *lse,
                                      void *stream);

/*
 * focus_count_pairs -- |A_i| for every query (the work the method does), for
 * effective-FLOP accounting and the "every pair counted once" check.
 *   per_query [B, n] int64 out, nullable
 *   totals    [2]    int64 out (device): totals[0] = sum_i |A_i|,
 *                    totals[1] = number of pairs that share a group.
 */
focus_status_t focus_count_pairs(const int32_t *ids, const int32_t *offsets,
                                 const int32_t *pos, const int32_t *inv,
                                 int B, int n, int num_groups, int topk,
                                 int window, int64_t *per_query,
                                 int64_t *totals, void *stream);

/*
 * Debug variant of focus_attention_fwd: identical result, and each scored
 * pair adds 1 to pair_count[b*n + i] (int32, device, caller-zeroed) for query
 * head 0, so the caller can check that every allowed pair was scored exactly
 * once (pair_count == |A_i|).
 */
focus_status_t focus_attention_fwd_counted(const void *Q, const void *K, const void *V,
                                           int B, int n, int Hq, int Hkv, int d,
                                           int window, float scale,
                                           const int32_t *ids, const int32_t *offsets,
                                           const int32_t *pos, const int32_t *inv,
                                           int num_groups, int topk,
                                           void *O, float *lse,
                                           void *ws, size_t ws_bytes,
                                           int32_t *pair_count, void *stream);

/*
 * Reads (and with reset != 0 clears) the device status word of the current
 * device: FOCUS_OK, FOCUS_ERR_TIMEOUT or FOCUS_ERR_CAPACITY.  Synchronises
 * the device.
 */
focus_status_t focus_get_device_status(int reset);

/*
 * Sets the limit of the bounded device-side waits of the assignment and merge
 * kernels for the launches this library enqueues after the call (any host
 * thread, any device), in nanoseconds of the GPU's global timer; 0 restores
 * the default, 2 s.  (The attention kernels keep the fixed 2 s limit: a run-
 * time limit in their waits measured 1.6 % slower.)  A testing aid: a tiny
 * limit makes the waits of the next launches run out, so
 * that their error path (the kernel finishes early, lets the copies and
 * tensor-core operations it issued land, and records FOCUS_ERR_TIMEOUT in the
 * device status word) can be exercised without faulting or hanging the GPU.
 * Outputs of launches whose waits ran out are undefined.
 */
focus_status_t focus_set_wait_limit(unsigned long long ns);

/* Number of kernels the last successful call on this host thread enqueued. */
int focus_last_launch_count(void);

/*
 * Per-kernel timing for measurement.  While enabled (per host thread), each
 * kernel the library launches is bracketed by two CUDA events recorded on
 * its stream.  focus_profile_read() waits for those events, writes up to
 * max_entries rows (kernel name into names[i * name_stride], NUL-terminated;
 * summed milliseconds into total_ms[i]; launch count into launches[i]; any
 * output pointer may be NULL), clears the record and returns the number of
 * rows, or -1 on a CUDA error.  All pointers are host pointers.
 */
void focus_profile_enable(int enable);
int focus_profile_read(char *names, int name_stride, double *total_ms, int *launches,
                       int max_entries);

/*
 * Pipeline wait tracing of the attention kernels (a debugging aid).  For
 * launches from this host thread, the group / window / dense kernels write,
 * per persistent CTA, 32 int64 counters of SM cycles into the given DEVICE
 * buffers (each at least 32 x the number of SMs entries; NULL disables):
 * time each role spent waiting on each pipeline barrier, the producer's
 * work-item preparation, the softmax epilogue, and item and tile counts.
 * Slot meanings are listed with the kernels' trace enum.
 */
void focus_trace_attention(long long *group_buf, long long *window_buf, long long *dense_buf);

/*
 * Pipeline wait tracing of the gated backward (a debugging aid).  For
 * launches from this host thread, the query-side and key-side kernels write,
 * for each CTA whose linear index (x fastest, then y, then z) is below
 * max_ctas, 32 int64 counters of SM cycles into the given DEVICE buffers
 * (each at least 32 x max_ctas entries; NULL or max_ctas <= 0 disables):
 * the producer's, the MMA thread's and the first elementwise thread's time
 * waiting on each pipeline barrier and in each phase, and the tile count.
 * Slot meanings are listed with the kernel's trace enum.
 */
void focus_trace_gated(long long *query_buf, long long *key_buf, int max_ctas);

#ifdef __cplusplus
}
#endif

#endif /* FOCUS_GB300_H */
