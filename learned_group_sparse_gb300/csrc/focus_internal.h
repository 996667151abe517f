// Internal launch interface between the C-ABI layer (focus_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace focus {

// Kernel launch with programmatic stream serialization: the grid may be
// scheduled while the previous kernel on the stream drains.  Every kernel
// launched this way calls grid_dep_sync() before its first global memory
// access, so it sees all of that kernel's writes and completes after it,
// which keeps the stream's order transitive.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

#ifdef __CUDACC__
// Device side of launch_pdl: let the next grid be scheduled once every CTA of
// this one has started, then wait until the previous grid has completed and
// its memory operations are visible.
__device__ __forceinline__ void grid_dep_sync()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
#endif

// Control of the kernels' bounded mbarrier waits, passed by value in every
// launch that waits: the device status word (a wait that runs out writes
// FOCUS_ERR_TIMEOUT there) and the limit, in ns of %globaltimer (a kernel
// argument, so reading it costs no memory access).
struct WaitCtl {
    int *status;
    unsigned long long limit_ns;
};

// Per-kernel timing hooks (no-ops unless focus_profile_enable(1) was called
// on this host thread).
void prof_begin(const char *name, cudaStream_t s);
void prof_end(cudaStream_t s);

// Records the kernel count that focus_last_launch_count() reports.
void set_last_launches(int launches);

// Wait-time trace buffer of an attention mode (0 group, 1 window, 2 dense)
// for launches from this host thread, or nullptr (see focus_trace_attention).
long long *trace_buffer(int mode);
// Trace buffer of the gated backward's query side (0) or key side (1) for
// launches from this host thread: nullptr, or the buffer and its CTA count.
void gated_trace_buffer(int side, long long **buf, int *ctas);

struct AssignLaunch {
    const __nv_bfloat16 *X;
    const float *Wg;
    const float *C;
    int64_t ntok;
    int hidden, dg, K, topk;
    int32_t *ids;
    float *margin;
};
// SIMT fp32 path (any K <= 1024).
cudaError_t launch_assign(const AssignLaunch &p, cudaStream_t s, int *launches);
// 2-D bf16 (or fp16) tensor map [outer, inner] (inner contiguous), box
// {box_inner, box_outer}, 128-byte swizzle.
bool make_map_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                 uint32_t box_inner, uint32_t box_outer, bool f16);
// 4-D bf16 (or fp16) tensor map of a [B, rows, H, d] tensor (d contiguous),
// boxes of 64 x 1 x box_rows x 1, 128-byte swizzle; reads past an edge give 0.
bool make_map_4d(CUtensorMap *m, const void *base, bool f16, int B, int64_t rows, int H, int d,
                 uint32_t box_rows);

// A prepared assignment: the path, its TMA maps and launch sizes.
// assign_prepare validates nothing that focus_assign's host checks cover, and
// enqueues nothing; assign_launch enqueues the kernels.
//   path 0: SIMT fp32 kernel, (X W_g) C^T;
//   path 1: tensor cores, X (W_g C^T) with W_g C^T split into bf16 hi + lo;
//   path 2: tensor cores in the order (X W_g) C^T, for more centroids than
//           centroid dimensions (focus_assign_z.cu).
struct AssignPlan {
    CUtensorMap map[4];
    AssignLaunch p;
    int path;
    WaitCtl wc;
    int Kp, dgp, stages, stages2;
    size_t smem, smem2;
    int64_t grid, grid2;
    void *mhi;                 // path 1: [M_hi; M_lo]
    void *wt, *ch, *z;         // path 2: W_g^T hi/lo, C hi/lo, Z hi/lo
    float *zscale;             // path 2: per-token scale of Z
};
int assign_path(int hidden, int dg, int K, int topk);
size_t assign_ws_bytes(int64_t ntok, int hidden, int dg, int K, int topk);
cudaError_t assign_prepare(const AssignLaunch &p, void *ws, const WaitCtl &wc, AssignPlan *plan);
cudaError_t assign_launch(const AssignPlan &plan, cudaStream_t s, int *launches);
// the paths' own halves of the above
bool assign_tc_supported(int hidden, int K, int topk);
cudaError_t assign_tc_prepare(const AssignLaunch &p, void *ws, const WaitCtl &wc, AssignPlan *plan);
cudaError_t assign_tc_launch(const AssignPlan &plan, cudaStream_t s, int *launches);
size_t assign_tc_ws_bytes(int hidden, int K);
int assign_z_dgp(int dg);
bool assign_z_supported(int hidden, int dg, int K, int topk);
size_t assign_z_ws_bytes(int64_t ntok, int hidden, int dg, int K);
cudaError_t assign_z_prepare(const AssignLaunch &p, void *ws, const WaitCtl &wc, AssignPlan *plan);
cudaError_t assign_z_launch(const AssignPlan &plan, cudaStream_t s, int *launches);

// ---- bucket: histogram per chunk, scan, offsets, stable scatter
// Host-side validation of a bucketing call (a focus.h status code; nothing
// is enqueued) and the status of a CUDA runtime result.
int check_bucket(const int32_t *ids, int B, int n, int K, int topk, const int32_t *offsets,
                 const int32_t *pos, const int32_t *inv);
int cuda_status(cudaError_t e);
constexpr int kBucketChunk = 4096;   // (token, slot) entries per chunk
size_t bucket_ws_bytes(int B, int n, int K, int topk);
cudaError_t launch_bucket(const int32_t *ids, int B, int n, int K, int topk, int32_t *offsets,
                          int32_t *pos, int32_t *inv, void *ws, cudaStream_t s, int *launches);

// ---- attention helpers
// Work list of the group kernel ordered by decreasing cost: entries (b*K + g, t)
// for the 128-row query tiles t of every group, or, with pair_tiles, for the
// pairs of consecutive tiles (2t, 2t+1).  ntiles[0] = the list's length;
// ntiles[1] and ntiles[2] are set to 0: the work counters from which the group
// and window kernels' CTAs take their items.
cudaError_t launch_plan(const int32_t *offsets, int B, int K, int pair_tiles, int2 *tiles,
                        int *ntiles, cudaStream_t s, int *launches);
// Kp[b][r] = K[b][pos[b][r]] and Vp likewise: rows of Hkv*d bf16;
// gidp[b][r] = the group ids of token pos[b][r].
cudaError_t launch_gather(const __nv_bfloat16 *K, const __nv_bfloat16 *V, const int32_t *pos,
                          const int32_t *ids, int B, int n, int topk, int Hkv, int d,
                          __nv_bfloat16 *Kp, __nv_bfloat16 *Vp, int32_t *gidp, cudaStream_t s,
                          int *launches);
// Group bitmaps of every key tile of the group kernel (tab_g, mask_tiles_group
// slots per batch): [slot][K] uint4, word j bit c = key row 32 j + c of the
// tile is in the group; group tile u of group g is slot floor(off[g] / 128) +
// g + u.  And the window bound of every group-order row (wlo [B, n*topk]): the
// first row of its group whose token lies inside the row's window (its own row
// + 1 at window 0); the group kernel scores the keys before it.
int64_t mask_tiles_group(int n, int K, int topk);
cudaError_t launch_mask_tables(const int32_t *offsets, const int32_t *gidp, const int32_t *ids,
                               const int32_t *pos, const int32_t *inv, int B, int n, int K,
                               int topk, int window, uint4 *tab_g, int32_t *wlo, cudaStream_t s,
                               int *launches);
cudaError_t launch_count_pairs(const int32_t *ids, const int32_t *offsets, const int32_t *pos,
                               const int32_t *inv, int B, int n, int K, int topk, int window,
                               int64_t *per_query, int64_t *totals, cudaStream_t s,
                               int *launches);

// ---- decode: one new token per sequence against per-group position lists
struct DecodeLaunch {
    const __nv_bfloat16 *q, *k, *v;
    const int32_t *ids;
    int32_t *glen, *gpos;
    int B, L, Lmax, Hq, Hkv, d, K, topk, cap, window;
    float scale_log2;
    __nv_bfloat16 *O;
    float *lse;
    void *ws;
    int *status;   // device status word (a list that would overflow)
    WaitCtl wc;    // limit of the attention kernel's waits
};
int decode_splits(int B, int Hkv);
size_t decode_ws_bytes(int B, int Hq, int Hkv, int d);
size_t decode_smem_bytes(int d);
cudaError_t decode_preflight(int d);
cudaError_t launch_decode_lists_init(const int32_t *offsets, const int32_t *pos, int B, int n,
                                     int K, int topk, int cap, int32_t *glen, int32_t *gpos,
                                     int *status, cudaStream_t s, int *launches);
cudaError_t launch_decode(const DecodeLaunch &p, cudaStream_t s, int *launches);

// ---- soft-gated attention of training and its backward
struct GatedLaunch {
    const __nv_bfloat16 *q, *k, *v, *o, *dO;
    const float *G, *lse;
    __nv_bfloat16 *out;
    float *lse_out, *dq, *dk, *dv, *dg, *dlam;
    int B, n, Hq, Hkv, d, Kg, window;
    float scale, lambda;
    WaitCtl wc;   // the forward kernel's bounded waits
};
size_t gated_ws_bytes(int B, int n, int Hq, int Hkv, int Kg);
// Query heads per query-side CTA of the gated backward: one partial of the
// row side of dG per chunk, in the workspace that gated_ws_bytes sizes.
constexpr int kGatedHeadChunk = 4;
// The tensor-core forward (focus_gated_tc.cu): its launch attributes and TMA
// maps (gated_tc_prepare enqueues nothing), then the launch.  g16 is the
// fp16 copy of G, [B, n, kp] with kp = K_g rounded up to 16.
struct GatedTcPlan {
    CUtensorMap map[5];   // Q, K, V, Gq (128-row boxes), Gk (64-row boxes)
    GatedLaunch p;
    int kp, pair_heads, grid;
};
cudaError_t gated_tc_preflight(int d, int Kg);
// The tensor-core backward (focus_gated_bwd_tc.cu): the query-side and
// key-side kernels' attributes and TMA maps (enqueues nothing), then their
// launches, given -lse log2(e) and -dO . O in rows padded to npad (rowv,
// [2][B, Hq, npad]) and the partial buffers of d lambda and dG.
struct GatedBwTcPlan {
    CUtensorMap map[12];   // query side: Q, dO, G_q, K, V, G_k; key side: K, V, G_k, Q, dO, G_q
    GatedLaunch p;
    int kp;
};
cudaError_t gated_bwd_tc_preflight(int d, int Kg);
cudaError_t gated_bwd_tc_prepare(const GatedLaunch &p, const __half *g16, int kp,
                                 GatedBwTcPlan *plan);
cudaError_t gated_bwd_tc_launch(const GatedBwTcPlan &plan, const float *rowv, int npad,
                                float *dlam_part, float *dg_part, cudaStream_t s, int *launches);
int gated_bwd_tc_dlam_count(int B, int n, int Hq);
cudaError_t gated_tc_prepare(const GatedLaunch &p, const __half *g16, int kp, GatedTcPlan *plan);
cudaError_t gated_tc_launch(const GatedTcPlan &plan, cudaStream_t s, int *launches);
cudaError_t launch_gated_fwd(const GatedLaunch &p, void *ws, cudaStream_t s, int *launches);
cudaError_t launch_gated_bwd(const GatedLaunch &p, void *ws, cudaStream_t s, int *launches);

// ---- Sinkhorn normalisation of token-group affinities
int sinkhorn_ctas(int B, int n, int K);
size_t sinkhorn_ws_bytes(int B, int n, int K);
cudaError_t launch_sinkhorn(const float *S, int B, int n, int K, float tau, int iters, float *P,
                            float *log_u, float *log_v, void *ws, const WaitCtl &wc,
                            cudaStream_t s, int *launches);

// ---- tcgen05 attention kernels
struct AttnLaunch {
    const CUtensorMap *tmQ, *tmK, *tmV;
    int B, n, Hq, Hkv, d;
    int rows;
    int window;
    float scale_log2;
    int K, topk;
    int pair_heads;   // the attention kernels pair heads (1) or query tiles (0)
    const int32_t *gids, *offsets, *pos;
    const int2 *tiles;
    const int *ntiles;
    const __nv_bfloat16 *q;  // kGroup: the original Q, whose rows the kernel gathers
    const uint4 *masks;      // kGroup: key-tile group bitmaps
    int64_t mask_tiles;      // mask slots per batch
    const int32_t *wlo;      // kGroup: window bound of each group-order row
    int *work;               // nullable: work-item counter, zero before the launch
    int64_t grid;
    __nv_bfloat16 *out;
    float *lse;
    __half *part_out16, *win_out16;
    float2 *part_meta_out, *win_meta_out;
    WaitCtl wc;
    int32_t *pair_count;
};
// O = log-sum-exp merge of the window partial and the topk group partials.
// wc: the bounded waits of the bulk-copy path.
cudaError_t launch_merge(const __half *win16, const float2 *win_meta, const __half *part16,
                         const float2 *part_meta, const int32_t *inv, int B, int n, int topk,
                         int Hq, int d, __nv_bfloat16 *O, float *lse, const WaitCtl &wc,
                         cudaStream_t s, int *launches);
cudaError_t launch_attn_group(const AttnLaunch &p, cudaStream_t s, int *launches);
// Sets the launch attributes of the group and window kernels for (d, K) and
// checks their register split; enqueues nothing.
cudaError_t attn_preflight(int d, int K);
cudaError_t attn_window_preflight(int d, int K);
// Shared memory the group and window kernels need for (d, K).
size_t attn_smem_needed(int d, int K);
constexpr size_t kMaxSmemPerBlock = 232448;   // 227 KB opt-in limit of sm_103a
cudaError_t launch_attn_window(const AttnLaunch &p, cudaStream_t s, int *launches);
cudaError_t launch_attn_dense(const AttnLaunch &p, cudaStream_t s, int *launches);

}  // namespace focus
