// C ABI of the Focus attention inference path (declared in include/focus.h):
// host-side validation, workspace layout, TMA descriptors, and the order of
// the kernel launches on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/focus.h"
#include "focus_internal.h"

namespace focus {

namespace {

thread_local int g_last_launches = 0;

// Device status word: set by a kernel whose bounded wait ran out.
__device__ int g_device_status = 0;

// Limit of the kernels' bounded waits for the launches that follow
// (focus_set_wait_limit); it travels in each launch's arguments.
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};

constexpr int kMaxDevices = 64;
int *g_status_addr[kMaxDevices] = {nullptr};
std::mutex g_status_mu;

cudaError_t status_ptr(int **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_status_mu);
    if (!g_status_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_device_status);
        if (e != cudaSuccess) return e;
        g_status_addr[dev] = static_cast<int *>(p);
    }
    *out = g_status_addr[dev];
    return cudaSuccess;
}

// The bounded-wait control of a launch on the current device.
cudaError_t wait_ctl(WaitCtl *out)
{
    cudaError_t e = status_ptr(&out->status);
    out->limit_ns = g_wait_limit_ns.load();
    return e;
}

// The second stream of focus_prefill's host path (input copies that overlap
// the assignment), created once per device; never destroyed.
cudaStream_t g_copy_stream[kMaxDevices] = {nullptr};
std::mutex g_copy_mu;

cudaError_t copy_stream(cudaStream_t *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_copy_mu);
    if (!g_copy_stream[dev]) {
        e = cudaStreamCreateWithFlags(&g_copy_stream[dev], cudaStreamNonBlocking);
        if (e != cudaSuccess) return e;
    }
    *out = g_copy_stream[dev];
    return cudaSuccess;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [B, rows, H, d] bf16 -> a 4-D map with 64 x 1 x 128 x 1 boxes, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, int B, int64_t rows, int H, int d)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2,
                                   (cuuint64_t)rows * H * d * 2};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

}  // namespace

bool make_map_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                 uint32_t box_inner, uint32_t box_outer, bool f16)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    const cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_4d(CUtensorMap *m, const void *base, bool f16, int B, int64_t rows, int H, int d,
                 uint32_t box_rows)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2,
                                   (cuuint64_t)rows * H * d * 2};
    const cuuint32_t box[4] = {64, 1, box_rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
              const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct AttnWs {
    size_t kp, vp, gidp, opart, lpart, owin, lwin, tiles, ntiles, mtab_g, wlo, total;
};

int64_t max_tiles(int B, int n, int K, int topk)
{
    const int64_t nk = (int64_t)n * topk;
    return (int64_t)B * ((nk + 127) / 128 + K);
}

AttnWs attn_ws(int B, int n, int Hq, int Hkv, int d, int K, int topk)
{
    const size_t nk = (size_t)n * topk;
    AttnWs w;
    size_t off = 0;
    w.kp = off;    off += align256((size_t)B * nk * Hkv * d * 2);
    w.vp = off;    off += align256((size_t)B * nk * Hkv * d * 2);
    w.gidp = off;  off += align256((size_t)B * nk * topk * 4);
    w.opart = off; off += align256((size_t)B * nk * Hq * d * 2);   // fp16 group partials
    w.lpart = off; off += align256((size_t)B * nk * Hq * 8);       // {lse, scale}
    w.owin = off;  off += align256((size_t)B * n * Hq * d * 2);    // fp16 window partials
    w.lwin = off;  off += align256((size_t)B * n * Hq * 8);
    w.tiles = off; off += align256((size_t)max_tiles(B, n, K, topk) * 8);
    w.ntiles = off; off += 256;
    w.mtab_g = off; off += align256((size_t)B * mask_tiles_group(n, K, topk) * K * 16);
    w.wlo = off;   off += align256((size_t)B * nk * 4);
    w.total = off;
    return w;
}

struct PrefillWs {
    size_t ids, offsets, pos, inv, assign, bucket, attn, x, wg, c, q, k, v, o, lse, total;
};

PrefillWs prefill_ws(int B, int n, int hidden, int Hq, int Hkv, int d, int dg, int K, int topk,
                     bool host)
{
    const size_t nk = (size_t)n * topk;
    PrefillWs w;
    size_t off = 0;
    w.ids = off;     off += align256((size_t)B * nk * 4);
    w.offsets = off; off += align256((size_t)B * (K + 1) * 4);
    w.pos = off;     off += align256((size_t)B * nk * 4);
    w.inv = off;     off += align256((size_t)B * nk * 4);
    w.assign = off;  off += align256(assign_ws_bytes((int64_t)B * n, hidden, dg, K, topk));
    w.bucket = off;  off += align256(bucket_ws_bytes(B, n, K, topk));
    w.attn = off;    off += align256(attn_ws(B, n, Hq, Hkv, d, K, topk).total);
    w.x = w.wg = w.c = w.q = w.k = w.v = w.o = w.lse = 0;
    if (host) {
        w.x = off;   off += align256((size_t)B * n * hidden * 2);
        w.wg = off;  off += align256((size_t)hidden * dg * 4);
        w.c = off;   off += align256((size_t)K * dg * 4);
        w.q = off;   off += align256((size_t)B * n * Hq * d * 2);
        w.k = off;   off += align256((size_t)B * n * Hkv * d * 2);
        w.v = off;   off += align256((size_t)B * n * Hkv * d * 2);
        w.o = off;   off += align256((size_t)B * n * Hq * d * 2);
        w.lse = off; off += align256((size_t)B * Hq * n * 4);
    }
    w.total = off;
    return w;
}


// ------------------------------------------------------------ validation
focus_status_t check_assign(const void *X, const float *Wg, const float *C, int B, int n,
                            int hidden, int dg, int K, int topk, const int32_t *ids,
                            const float *margin)
{
    if (!X || !Wg || !C || !ids) return FOCUS_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(Wg) || !aligned16(C) || !aligned16(ids) ||
        (margin && !aligned16(margin)))
        return FOCUS_ERR_INVALID_ARG;
    if (B < 1 || n < 0 || hidden < 1 || dg < 1 || K < 1 || topk < 1 || topk > K)
        return FOCUS_ERR_INVALID_ARG;
    if ((int64_t)B * n * topk >= ((int64_t)1 << 31)) return FOCUS_ERR_UNSUPPORTED;
    if (hidden % 8 != 0 || dg > 256 || K > 1024 || topk > 8) return FOCUS_ERR_UNSUPPORTED;
    return FOCUS_OK;
}

focus_status_t check_attn_shapes(int B, int n, int Hq, int Hkv, int d, int window)
{
    if (B < 1 || n < 1 || Hq < 1 || Hkv < 1 || window < 0) return FOCUS_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return FOCUS_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return FOCUS_ERR_UNSUPPORTED;
    if (B > 65535 || Hq > 65535) return FOCUS_ERR_UNSUPPORTED;
    return FOCUS_OK;
}

// Everything focus_attention_fwd needs before its first launch: validated
// arguments, the workspace carve-up, the TMA maps and the kernels' launch
// attributes.  attention_prepare enqueues nothing, so an entry point that
// calls it before its own first copy or launch keeps the "non-zero status
// means nothing was enqueued" rule; attention_enqueue then only launches.
struct AttnPrep {
    const void *Q, *Kt, *V;
    const int32_t *ids, *offsets, *pos, *inv;
    void *O;
    float *lse;
    int B, n, Hq, Hkv, d, K, topk;
    int64_t grid_group, grid_win;
    __nv_bfloat16 *Kp, *Vp;
    int32_t *gidp;
    __half *Opart, *Owin;
    float2 *Mpart, *Mwin;
    int2 *tiles;
    int *ntiles;
    uint4 *mtab_g;
    int32_t *wlo;
    CUtensorMap mk, mv, wq, wk, wv;
    AttnLaunch p;     // fields shared by the group and window launches
};

focus_status_t attention_prepare(const void *Q, const void *Kt, const void *V, int B, int n,
                                 int Hq, int Hkv, int d, int window, float scale,
                                 const int32_t *ids, const int32_t *offsets, const int32_t *pos,
                                 const int32_t *inv, int K, int topk, void *O, float *lse,
                                 void *ws, size_t ws_bytes, int32_t *pair_count, AttnPrep *ap)
{
    if (!Q || !Kt || !V || !ids || !offsets || !pos || !inv || !O || !ws)
        return FOCUS_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(Kt) || !aligned16(V) || !aligned16(O) || !aligned16(ws) ||
        !aligned16(ids) || !aligned16(offsets) || !aligned16(pos) || !aligned16(inv) ||
        (lse && !aligned16(lse)) || (pair_count && !aligned16(pair_count)))
        return FOCUS_ERR_INVALID_ARG;
    focus_status_t st = check_attn_shapes(B, n, Hq, Hkv, d, window);
    if (st) return st;
    if (K < 1 || topk < 1 || topk > K) return FOCUS_ERR_INVALID_ARG;
    if (K > 1024 || topk > 8 || (int64_t)B * K > 4096) return FOCUS_ERR_UNSUPPORTED;
    if (attn_smem_needed(d, K) > kMaxSmemPerBlock) return FOCUS_ERR_UNSUPPORTED;
    if ((int64_t)B * n * topk >= ((int64_t)1 << 31)) return FOCUS_ERR_UNSUPPORTED;
    const AttnWs w = attn_ws(B, n, Hq, Hkv, d, K, topk);
    if (ws_bytes < w.total) return FOCUS_ERR_WORKSPACE;
    ap->grid_group = max_tiles(B, n, K, topk) * Hq;
    const int64_t nqt = (n + 127) / 128;
    ap->grid_win = (int64_t)B * nqt * Hq;
    if (ap->grid_group >= ((int64_t)1 << 31) || ap->grid_win >= ((int64_t)1 << 31))
        return FOCUS_ERR_UNSUPPORTED;

    WaitCtl wc;
    if (wait_ctl(&wc) != cudaSuccess) return FOCUS_ERR_CUDA;
    // the kernels' shared-memory and register limits, checked before any launch
    if (attn_preflight(d, K) != cudaSuccess) return FOCUS_ERR_CUDA;
    uint8_t *base = static_cast<uint8_t *>(ws);
    ap->Q = Q;
    ap->Kt = Kt;
    ap->V = V;
    ap->ids = ids;
    ap->offsets = offsets;
    ap->pos = pos;
    ap->inv = inv;
    ap->O = O;
    ap->lse = lse;
    ap->B = B;
    ap->n = n;
    ap->Hq = Hq;
    ap->Hkv = Hkv;
    ap->d = d;
    ap->K = K;
    ap->topk = topk;
    ap->Kp = reinterpret_cast<__nv_bfloat16 *>(base + w.kp);
    ap->Vp = reinterpret_cast<__nv_bfloat16 *>(base + w.vp);
    ap->gidp = reinterpret_cast<int32_t *>(base + w.gidp);
    ap->Opart = reinterpret_cast<__half *>(base + w.opart);
    ap->Mpart = reinterpret_cast<float2 *>(base + w.lpart);
    ap->Owin = reinterpret_cast<__half *>(base + w.owin);
    ap->Mwin = reinterpret_cast<float2 *>(base + w.lwin);
    ap->tiles = reinterpret_cast<int2 *>(base + w.tiles);
    ap->ntiles = reinterpret_cast<int *>(base + w.ntiles);
    ap->mtab_g = reinterpret_cast<uint4 *>(base + w.mtab_g);
    ap->wlo = reinterpret_cast<int32_t *>(base + w.wlo);
    const int64_t nk = (int64_t)n * topk;
    if (!make_map(&ap->mk, ap->Kp, B, nk, Hkv, d) || !make_map(&ap->mv, ap->Vp, B, nk, Hkv, d) ||
        !make_map(&ap->wq, Q, B, n, Hq, d) || !make_map(&ap->wk, Kt, B, n, Hkv, d) ||
        !make_map(&ap->wv, V, B, n, Hkv, d))
        return FOCUS_ERR_CUDA;

    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)d);
    AttnLaunch &p = ap->p;
    memset(&p, 0, sizeof p);
    p.B = B;
    p.n = n;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.d = d;
    p.window = window;
    p.scale_log2 = sc * 1.4426950408889634f;
    p.K = K;
    p.topk = topk;
    p.offsets = offsets;
    p.pos = pos;
    p.tiles = ap->tiles;
    p.ntiles = ap->ntiles;
    p.wc = wc;
    p.pair_count = pair_count;
    // Two query tiles per CTA share the key/value stream: heads 2s, 2s+1 when
    // they share a key/value head, else consecutive query tiles of one head.
    p.pair_heads = (Hq / Hkv) % 2 == 0 ? 1 : 0;
    return FOCUS_OK;
}

// Launches the prepared attention: plan, gather, mask tables, group kernel,
// window kernel, merge.  q_ready (nullable): an event the group kernel waits
// for (Q may still be arriving from the host while the gather runs).
focus_status_t attention_enqueue(AttnPrep &ap, cudaStream_t s, int *launches,
                                 cudaEvent_t q_ready = nullptr)
{
    AttnLaunch &p = ap.p;
    const int B = ap.B, n = ap.n, K = ap.K, topk = ap.topk;
    if (launch_plan(ap.offsets, B, K, !p.pair_heads, ap.tiles, ap.ntiles, s, launches) !=
        cudaSuccess)
        return FOCUS_ERR_CUDA;
    if (launch_gather(static_cast<const __nv_bfloat16 *>(ap.Kt),
                      static_cast<const __nv_bfloat16 *>(ap.V), ap.pos, ap.ids, B, n, topk,
                      ap.Hkv, ap.d, ap.Kp, ap.Vp, ap.gidp, s, launches) != cudaSuccess)
        return FOCUS_ERR_CUDA;
    if (launch_mask_tables(ap.offsets, ap.gidp, ap.ids, ap.pos, ap.inv, B, n, K, topk, p.window,
                           ap.mtab_g, ap.wlo, s, launches) != cudaSuccess)
        return FOCUS_ERR_CUDA;

    // the group kernel copies its query rows from Q itself (tmQ unused)
    p.tmQ = &ap.wq;
    p.q = static_cast<const __nv_bfloat16 *>(ap.Q);
    p.tmK = &ap.mk;
    p.tmV = &ap.mv;
    p.rows = (int)((int64_t)n * topk);
    p.gids = ap.gidp;
    p.masks = ap.mtab_g;
    p.mask_tiles = mask_tiles_group(n, K, topk);
    p.wlo = ap.wlo;
    p.work = ap.ntiles + 1;    // zeroed by the plan kernel
    p.grid = ap.grid_group;
    p.part_out16 = ap.Opart;
    p.part_meta_out = ap.Mpart;
    if (q_ready && cudaStreamWaitEvent(s, q_ready, 0) != cudaSuccess) return FOCUS_ERR_CUDA;
    if (launch_attn_group(p, s, launches) != cudaSuccess) return FOCUS_ERR_CUDA;

    p.tmQ = &ap.wq;
    p.tmK = &ap.wk;
    p.tmV = &ap.wv;
    p.rows = n;
    p.gids = nullptr;      // every pair of the window: no group masks
    p.masks = nullptr;
    p.mask_tiles = 0;
    p.wlo = nullptr;
    p.work = ap.ntiles + 2;    // zeroed by the plan kernel
    p.grid = ap.grid_win;
    p.win_out16 = ap.Owin;
    p.win_meta_out = ap.Mwin;
    if (launch_attn_window(p, s, launches) != cudaSuccess) return FOCUS_ERR_CUDA;

    if (launch_merge(ap.Owin, ap.Mwin, ap.Opart, ap.Mpart, ap.inv, B, n, topk, ap.Hq, ap.d,
                     static_cast<__nv_bfloat16 *>(ap.O), ap.lse, p.wc, s, launches) != cudaSuccess)
        return FOCUS_ERR_CUDA;
    return FOCUS_OK;
}

focus_status_t attention_impl(const void *Q, const void *Kt, const void *V, int B, int n, int Hq,
                              int Hkv, int d, int window, float scale, const int32_t *ids,
                              const int32_t *offsets, const int32_t *pos, const int32_t *inv,
                              int K, int topk, void *O, float *lse, void *ws, size_t ws_bytes,
                              int32_t *pair_count, cudaStream_t s, int *launches)
{
    AttnPrep ap;
    focus_status_t st = attention_prepare(Q, Kt, V, B, n, Hq, Hkv, d, window, scale, ids, offsets,
                                          pos, inv, K, topk, O, lse, ws, ws_bytes, pair_count, &ap);
    if (st) return st;
    return attention_enqueue(ap, s, launches);
}

}  // namespace

void set_last_launches(int launches) { g_last_launches = launches; }

// Shared with focus_bucket_static (focus_bucket.cu): one validation and one
// status mapping for both bucketing entry points.
int cuda_status(cudaError_t e) { return e == cudaSuccess ? FOCUS_OK : FOCUS_ERR_CUDA; }

int check_bucket(const int32_t *ids, int B, int n, int K, int topk,
                            const int32_t *offsets, const int32_t *pos, const int32_t *inv)
{
    if (!ids || !offsets || !pos || !inv) return FOCUS_ERR_INVALID_ARG;
    if (!aligned16(ids) || !aligned16(offsets) || !aligned16(pos) || !aligned16(inv))
        return FOCUS_ERR_INVALID_ARG;
    if (B < 1 || n < 0 || K < 1 || topk < 1 || topk > K) return FOCUS_ERR_INVALID_ARG;
    if ((int64_t)B * n * topk >= ((int64_t)1 << 31)) return FOCUS_ERR_UNSUPPORTED;
    if (K > 1024 || topk > 8 || B > 65535) return FOCUS_ERR_UNSUPPORTED;
    return FOCUS_OK;
}


}  // namespace focus

using namespace focus;

extern "C" {

const char *focus_status_string(focus_status_t status)
{
    switch (status) {
    case FOCUS_OK: return "FOCUS_OK";
    case FOCUS_ERR_INVALID_ARG: return "FOCUS_ERR_INVALID_ARG";
    case FOCUS_ERR_UNSUPPORTED: return "FOCUS_ERR_UNSUPPORTED";
    case FOCUS_ERR_WORKSPACE: return "FOCUS_ERR_WORKSPACE";
    case FOCUS_ERR_CUDA: return "FOCUS_ERR_CUDA";
    case FOCUS_ERR_TIMEOUT: return "FOCUS_ERR_TIMEOUT";
    case FOCUS_ERR_CAPACITY: return "FOCUS_ERR_CAPACITY";
    default: return "FOCUS_ERR_UNKNOWN";
    }
}

const char *focus_version(void) { return "focus-gb300 0.1.0 sm_103a"; }

int focus_last_launch_count(void) { return g_last_launches; }

size_t focus_assign_workspace_size(int B, int n, int hidden, int d_g, int K, int topk)
{
    if (B < 1 || n < 0 || hidden < 1 || d_g < 1 || K < 1 || topk < 1) return 0;
    return assign_ws_bytes((int64_t)B * n, hidden, d_g, K, topk);
}

focus_status_t focus_assign(const void *X, const float *Wg, const float *C, int B, int n,
                            int hidden, int d_g, int K, int topk, int32_t *ids, float *margin,
                            void *ws, size_t ws_bytes, void *stream)
{
    focus_status_t st = check_assign(X, Wg, C, B, n, hidden, d_g, K, topk, ids, margin);
    if (st) return st;
    const size_t need = assign_ws_bytes((int64_t)B * n, hidden, d_g, K, topk);
    if (need && (!ws || ws_bytes < need)) return FOCUS_ERR_WORKSPACE;
    if (need && !aligned16(ws)) return FOCUS_ERR_INVALID_ARG;
    WaitCtl wc;
    if (wait_ctl(&wc) != cudaSuccess) return FOCUS_ERR_CUDA;
    AssignLaunch p{static_cast<const __nv_bfloat16 *>(X), Wg, C, (int64_t)B * n, hidden, d_g, K,
                   topk, ids, margin};
    AssignPlan plan;
    if (assign_prepare(p, ws, wc, &plan) != cudaSuccess) return FOCUS_ERR_CUDA;
    int launches = 0;
    cudaError_t e = assign_launch(plan, static_cast<cudaStream_t>(stream), &launches);
    if (e == cudaSuccess) g_last_launches = launches;
    return cuda_status(e);
}

size_t focus_bucket_workspace_size(int B, int n, int K, int topk)
{
    if (B < 1 || n < 0 || K < 1 || topk < 1) return 0;
    return bucket_ws_bytes(B, n, K, topk);
}

focus_status_t focus_bucket(const int32_t *ids, int B, int n, int K, int topk, int32_t *offsets,
                            int32_t *pos, int32_t *inv, void *ws, size_t ws_bytes, void *stream)
{
    focus_status_t st = check_bucket(ids, B, n, K, topk, offsets, pos, inv);
    if (st) return st;
    if (!ws || !aligned16(ws)) return FOCUS_ERR_INVALID_ARG;
    if (ws_bytes < bucket_ws_bytes(B, n, K, topk)) return FOCUS_ERR_WORKSPACE;
    int launches = 0;
    cudaError_t e = launch_bucket(ids, B, n, K, topk, offsets, pos, inv, ws,
                                  static_cast<cudaStream_t>(stream), &launches);
    if (e == cudaSuccess) g_last_launches = launches;
    return cuda_status(e);
}

size_t focus_attention_workspace_size(int B, int n, int Hq, int Hkv, int d, int K, int topk)
{
    if (B < 1 || n < 1 || Hq < 1 || Hkv < 1 || d < 1 || K < 1 || topk < 1) return 0;
    return attn_ws(B, n, Hq, Hkv, d, K, topk).total;
}

focus_status_t focus_attention_fwd(const void *Q, const void *K, const void *V, int B, int n,
                                   int Hq, int Hkv, int d, int window, float scale,
                                   const int32_t *ids, const int32_t *offsets, const int32_t *pos,
                                   const int32_t *inv, int num_groups, int topk, void *O,
                                   float *lse, void *ws, size_t ws_bytes, void *stream)
{
    int launches = 0;
    focus_status_t st = attention_impl(Q, K, V, B, n, Hq, Hkv, d, window, scale, ids, offsets,
                                       pos, inv, num_groups, topk, O, lse, ws, ws_bytes, nullptr,
                                       static_cast<cudaStream_t>(stream), &launches);
    if (st == FOCUS_OK) g_last_launches = launches;
    return st;
}

focus_status_t focus_attention_fwd_counted(const void *Q, const void *K, const void *V, int B,
                                           int n, int Hq, int Hkv, int d, int window, float scale,
                                           const int32_t *ids, const int32_t *offsets,
                                           const int32_t *pos, const int32_t *inv,
                                           int num_groups, int topk, void *O, float *lse,
                                           void *ws, size_t ws_bytes, int32_t *pair_count,
                                           void *stream)
{
    if (!pair_count) return FOCUS_ERR_INVALID_ARG;
    int launches = 0;
    focus_status_t st = attention_impl(Q, K, V, B, n, Hq, Hkv, d, window, scale, ids, offsets,
                                       pos, inv, num_groups, topk, O, lse, ws, ws_bytes,
                                       pair_count, static_cast<cudaStream_t>(stream), &launches);
    if (st == FOCUS_OK) g_last_launches = launches;
    return st;
}

size_t focus_prefill_workspace_size(int B, int n, int hidden, int Hq, int Hkv, int d, int d_g,
                                    int K, int topk, int io_on_host)
{
    if (B < 1 || n < 1 || hidden < 1 || Hq < 1 || Hkv < 1 || d < 1 || d_g < 1 || K < 1 ||
        topk < 1)
        return 0;
    return prefill_ws(B, n, hidden, Hq, Hkv, d, d_g, K, topk, io_on_host != 0).total;
}

focus_status_t focus_prefill(const void *X, const float *Wg, const float *C, const void *Q,
                             const void *K, const void *V, int B, int n, int hidden, int Hq,
                             int Hkv, int d, int d_g, int num_groups, int topk, int window,
                             float scale, void *O, float *lse, int32_t *ids_out, void *ws,
                             size_t ws_bytes, int io_on_host, void *stream)
{
    if (!X || !Wg || !C || !Q || !K || !V || !O || !ws) return FOCUS_ERR_INVALID_ARG;
    focus_status_t st = check_attn_shapes(B, n, Hq, Hkv, d, window);
    if (st) return st;
    const bool host = io_on_host != 0;
    const PrefillWs w = prefill_ws(B, n, hidden, Hq, Hkv, d, d_g, num_groups, topk, host);
    if (!aligned16(ws)) return FOCUS_ERR_INVALID_ARG;
    if (ws_bytes < w.total) return FOCUS_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *base = static_cast<uint8_t *>(ws);
    int32_t *ids = ids_out ? ids_out : reinterpret_cast<int32_t *>(base + w.ids);
    int32_t *offsets = reinterpret_cast<int32_t *>(base + w.offsets);
    int32_t *pos = reinterpret_cast<int32_t *>(base + w.pos);
    int32_t *inv = reinterpret_cast<int32_t *>(base + w.inv);
    const void *dX = X, *dQ = Q, *dK = K, *dV = V;
    const float *dWg = Wg, *dC = C;
    void *dO = O;
    float *dL = lse;
    if (host) {
        dX = base + w.x;
        dWg = reinterpret_cast<const float *>(base + w.wg);
        dC = reinterpret_cast<const float *>(base + w.c);
        dQ = base + w.q;
        dK = base + w.k;
        dV = base + w.v;
        dO = base + w.o;
        dL = lse ? reinterpret_cast<float *>(base + w.lse) : nullptr;
    } else if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
               (lse && !aligned16(lse))) {
        return FOCUS_ERR_INVALID_ARG;
    }
    // Every check of every step, before anything is enqueued: the assignment,
    // the bucketing, and the attention (shapes, shared memory, grid bounds,
    // TMA maps, kernel attributes).
    st = check_assign(dX, dWg, dC, B, n, hidden, d_g, num_groups, topk, ids, nullptr);
    if (st) return st;
    st = check_bucket(ids, B, n, num_groups, topk, offsets, pos, inv);
    if (st) return st;
    AssignLaunch asg{static_cast<const __nv_bfloat16 *>(dX), dWg, dC, (int64_t)B * n, hidden,
                     d_g, num_groups, topk, ids, nullptr};
    AssignPlan aplan;
    WaitCtl wc;
    if (wait_ctl(&wc) != cudaSuccess) return FOCUS_ERR_CUDA;
    if (assign_prepare(asg, base + w.assign, wc, &aplan) != cudaSuccess) return FOCUS_ERR_CUDA;
    const AttnWs aw = attn_ws(B, n, Hq, Hkv, d, num_groups, topk);
    AttnPrep attn;
    st = attention_prepare(dQ, dK, dV, B, n, Hq, Hkv, d, window, scale, ids, offsets, pos, inv,
                           num_groups, topk, dO, dL, base + w.attn, aw.total, nullptr, &attn);
    if (st) return st;

    int launches = 0;
    cudaError_t e = cudaSuccess;
    cudaEvent_t ev_x = nullptr, ev_kv = nullptr, ev_q = nullptr;   // host path only
    // (the events are released when the call returns; waits enqueued on them
    // stay valid)
    struct EventGuard {
        cudaEvent_t *ev[3];
        ~EventGuard()
        {
            for (cudaEvent_t *e : ev)
                if (*e) cudaEventDestroy(*e);
        }
    } guard{{&ev_x, &ev_kv, &ev_q}};
    if (host) {
        const size_t xb = (size_t)B * n * hidden * 2, qb = (size_t)B * n * Hq * d * 2,
                     kb = (size_t)B * n * Hkv * d * 2;
        // X, W_g and C on `stream`; then K, V and Q on the copy stream while
        // the assignment and bucketing run (the link carries one copy at its
        // full rate, so they follow X rather than share the link with it).
        // `stream` waits for K and V before the gather and for Q before the
        // group kernel.
        cudaStream_t cs = nullptr;
        if ((e = copy_stream(&cs)) != cudaSuccess) return FOCUS_ERR_CUDA;
        if ((e = cudaEventCreateWithFlags(&ev_x, cudaEventDisableTiming)) ||
            (e = cudaEventCreateWithFlags(&ev_kv, cudaEventDisableTiming)) ||
            (e = cudaEventCreateWithFlags(&ev_q, cudaEventDisableTiming)))
            return FOCUS_ERR_CUDA;
        if ((e = cudaMemcpyAsync(base + w.x, X, xb, cudaMemcpyHostToDevice, s)) ||
            (e = cudaMemcpyAsync(base + w.wg, Wg, (size_t)hidden * d_g * 4, cudaMemcpyHostToDevice, s)) ||
            (e = cudaMemcpyAsync(base + w.c, C, (size_t)num_groups * d_g * 4, cudaMemcpyHostToDevice, s)) ||
            (e = cudaEventRecord(ev_x, s)) || (e = cudaStreamWaitEvent(cs, ev_x, 0)) ||
            (e = cudaMemcpyAsync(base + w.k, K, kb, cudaMemcpyHostToDevice, cs)) ||
            (e = cudaMemcpyAsync(base + w.v, V, kb, cudaMemcpyHostToDevice, cs)) ||
            (e = cudaEventRecord(ev_kv, cs)) ||
            (e = cudaMemcpyAsync(base + w.q, Q, qb, cudaMemcpyHostToDevice, cs)) ||
            (e = cudaEventRecord(ev_q, cs)))
            return FOCUS_ERR_CUDA;
    }
    if ((e = assign_launch(aplan, s, &launches)) != cudaSuccess) return FOCUS_ERR_CUDA;
    if ((e = launch_bucket(ids, B, n, num_groups, topk, offsets, pos, inv, base + w.bucket, s,
                           &launches)) != cudaSuccess)
        return FOCUS_ERR_CUDA;
    if (host && (e = cudaStreamWaitEvent(s, ev_kv, 0)) != cudaSuccess) return FOCUS_ERR_CUDA;
    st = attention_enqueue(attn, s, &launches, host ? ev_q : nullptr);
    if (st) return st;
    if (host) {
        if ((e = cudaMemcpyAsync(O, dO, (size_t)B * n * Hq * d * 2, cudaMemcpyDeviceToHost, s)))
            return FOCUS_ERR_CUDA;
        if (lse && (e = cudaMemcpyAsync(lse, dL, (size_t)B * Hq * n * 4, cudaMemcpyDeviceToHost, s)))
            return FOCUS_ERR_CUDA;
    }
    g_last_launches = launches;
    return FOCUS_OK;
}

focus_status_t focus_dense_causal_fwd(const void *Q, const void *K, const void *V, int B, int n,
                                      int Hq, int Hkv, int d, float scale, void *O, float *lse,
                                      void *stream)
{
    if (!Q || !K || !V || !O) return FOCUS_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) ||
        (lse && !aligned16(lse)))
        return FOCUS_ERR_INVALID_ARG;
    focus_status_t st = check_attn_shapes(B, n, Hq, Hkv, d, 0);
    if (st) return st;
    const int64_t grid = (int64_t)B * ((n + 127) / 128) * Hq;
    if (grid >= ((int64_t)1 << 31)) return FOCUS_ERR_UNSUPPORTED;
    WaitCtl wc;
    if (wait_ctl(&wc) != cudaSuccess) return FOCUS_ERR_CUDA;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, Q, B, n, Hq, d) || !make_map(&mk, K, B, n, Hkv, d) ||
        !make_map(&mv, V, B, n, Hkv, d))
        return FOCUS_ERR_CUDA;
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)d);
    AttnLaunch p;
    memset(&p, 0, sizeof p);
    p.tmQ = &mq;
    p.tmK = &mk;
    p.tmV = &mv;
    p.B = B;
    p.n = n;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.d = d;
    p.rows = n;
    p.window = n;
    p.scale_log2 = sc * 1.4426950408889634f;
    p.K = 1;
    p.topk = 1;
    p.pair_heads = (Hq / Hkv) % 2 == 0 ? 1 : 0;
    p.grid = grid;
    p.out = static_cast<__nv_bfloat16 *>(O);
    p.lse = lse;
    p.wc = wc;
    int launches = 0;
    cudaError_t e = launch_attn_dense(p, static_cast<cudaStream_t>(stream), &launches);
    if (e == cudaSuccess) g_last_launches = launches;
    return cuda_status(e);
}

focus_status_t focus_count_pairs(const int32_t *ids, const int32_t *offsets, const int32_t *pos,
                                 const int32_t *inv, int B, int n, int num_groups, int topk,
                                 int window, int64_t *per_query, int64_t *totals, void *stream)
{
    focus_status_t st = check_bucket(ids, B, n, num_groups, topk, offsets, pos, inv);
    if (st) return st;
    if (!totals || window < 0) return FOCUS_ERR_INVALID_ARG;
    if (!aligned16(totals) || (per_query && !aligned16(per_query))) return FOCUS_ERR_INVALID_ARG;
    int launches = 0;
    cudaError_t e = launch_count_pairs(ids, offsets, pos, inv, B, n, num_groups, topk, window,
                                       per_query, totals, static_cast<cudaStream_t>(stream),
                                       &launches);
    if (e == cudaSuccess) g_last_launches = launches;
    return cuda_status(e);
}

size_t focus_gated_workspace_size(int B, int n, int Hq, int Hkv, int Kg)
{
    if (B < 1 || n < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Kg < 1 || Kg > 128) return 0;
    return gated_ws_bytes(B, n, Hq, Hkv, Kg);
}

static focus_status_t check_gated(const void *Q, const void *K, const void *V, const float *G,
                                  int B, int n, int Hq, int Hkv, int d, int Kg, int window,
                                  float lambda, float scale, const void *ws, size_t ws_bytes)
{
    if (!Q || !K || !V || !G || !ws) return FOCUS_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(G) || !aligned16(ws))
        return FOCUS_ERR_INVALID_ARG;
    if (B < 1 || n < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Kg < 1 || window < 0 ||
        !(fabsf(lambda) < INFINITY) || !(scale >= 0.f) || !(scale < INFINITY))
        return FOCUS_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || Kg > 128 || (int64_t)B * n * Hq * d >= ((int64_t)1 << 40) ||
        (n + 63) / 64 > 65535 || Hq > 65535 || B > 65535)
        return FOCUS_ERR_UNSUPPORTED;
    if (ws_bytes < gated_ws_bytes(B, n, Hq, Hkv, Kg)) return FOCUS_ERR_WORKSPACE;
    return FOCUS_OK;
}

focus_status_t focus_gated_attention_fwd(const void *Q, const void *K, const void *V,
                                         const float *G, int B, int n, int Hq, int Hkv, int d,
                                         int Kg, int window, float lambda, float scale, void *O,
                                         float *lse, void *ws, size_t ws_bytes, void *stream)
{
    focus_status_t st = check_gated(Q, K, V, G, B, n, Hq, Hkv, d, Kg, window, lambda, scale, ws,
                                    ws_bytes);
    if (st) return st;
    if (!O || !lse || !aligned16(O) || !aligned16(lse)) return FOCUS_ERR_INVALID_ARG;
    GatedLaunch p{};
    if (wait_ctl(&p.wc) != cudaSuccess) return FOCUS_ERR_CUDA;
    p.q = static_cast<const __nv_bfloat16 *>(Q);
    p.k = static_cast<const __nv_bfloat16 *>(K);
    p.v = static_cast<const __nv_bfloat16 *>(V);
    p.G = G;
    p.out = static_cast<__nv_bfloat16 *>(O);
    p.lse_out = lse;
    p.B = B;
    p.n = n;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.d = d;
    p.Kg = Kg;
    p.window = window;
    p.lambda = lambda;
    p.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)d);
    int launches = 0;
    cudaError_t e = launch_gated_fwd(p, ws, static_cast<cudaStream_t>(stream), &launches);
    if (e == cudaSuccess) g_last_launches = launches;
    return cuda_status(e);
}

focus_status_t focus_gated_attention_bwd(const void *Q, const void *K, const void *V,
                                         const float *G, const void *O, const float *lse,
                                         const void *dO, int B, int n, int Hq, int Hkv, int d,
                                         int Kg, int window, float lambda, float scale,
                                         float *dQ, float *dK, float *dV, float *dG,
                                         float *dlambda, void *ws, size_t ws_bytes, void *stream)
{
    focus_status_t st = check_gated(Q, K, V, G, B, n, Hq, Hkv, d, Kg, window, lambda, scale, ws,
                                    ws_bytes);
    if (st) return st;
    if (!O || !lse || !dO || !dQ || !dK || !dV || !dG || !dlambda) return FOCUS_ERR_INVALID_ARG;
    if (!aligned16(O) || !aligned16(lse) || !aligned16(dO) || !aligned16(dQ) || !aligned16(dK) ||
        !aligned16(dV) || !aligned16(dG) || ((uintptr_t)dlambda & 3u))
        return FOCUS_ERR_INVALID_ARG;
    GatedLaunch p{};
    if (wait_ctl(&p.wc) != cudaSuccess) return FOCUS_ERR_CUDA;
    p.q = static_cast<const __nv_bfloat16 *>(Q);
    p.k = static_cast<const __nv_bfloat16 *>(K);
    p.v = static_cast<const __nv_bfloat16 *>(V);
    p.o = static_cast<const __nv_bfloat16 *>(O);
    p.dO = static_cast<const __nv_bfloat16 *>(dO);
    p.G = G;
    p.lse = lse;
    p.dq = dQ;
    p.dk = dK;
    p.dv = dV;
    p.dg = dG;
    p.dlam = dlambda;
    p.B = B;
    p.n = n;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.d = d;
    p.Kg = Kg;
    p.window = window;
    p.lambda = lambda;
    p.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)d);
    int launches = 0;
    cudaError_t e = launch_gated_bwd(p, ws, static_cast<cudaStream_t>(stream), &launches);
    if (e == cudaSuccess) g_last_launches = launches;
    return cuda_status(e);
}

size_t focus_sinkhorn_workspace_size(int B, int n, int K)
{
    if (B < 1 || n < 1 || K < 1 || K > 1024) return 0;
    return sinkhorn_ws_bytes(B, n, K);
}

focus_status_t focus_sinkhorn(const float *S, int B, int n, int K, float tau, int iters,
                              float *P, float *log_u, float *log_v, void *ws, size_t ws_bytes,
                              void *stream)
{
    if (!S || !ws) return FOCUS_ERR_INVALID_ARG;
    if (!aligned16(S) || !aligned16(ws) || (P && !aligned16(P)) || (log_u && !aligned16(log_u)) ||
        (log_v && !aligned16(log_v)))
        return FOCUS_ERR_INVALID_ARG;
    if (B < 1 || n < 1 || K < 1 || K > 1024 || !(tau >= 0.f) || !(tau < INFINITY) || iters < 1 ||
        iters > 100000 || (int64_t)B * n > ((int64_t)1 << 40))
        return FOCUS_ERR_INVALID_ARG;
    if (ws_bytes < sinkhorn_ws_bytes(B, n, K)) return FOCUS_ERR_WORKSPACE;
    WaitCtl wc;
    if (wait_ctl(&wc) != cudaSuccess) return FOCUS_ERR_CUDA;
    int launches = 0;
    cudaError_t e = launch_sinkhorn(S, B, n, K, tau > 0.f ? tau : 1.f, iters, P, log_u, log_v,
                                    ws, wc, static_cast<cudaStream_t>(stream), &launches);
    if (e == cudaSuccess) g_last_launches = launches;
    return cuda_status(e);
}

size_t focus_decode_workspace_size(int B, int Hq, int Hkv, int d)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || d < 1 || Hq % Hkv != 0) return 0;
    return decode_ws_bytes(B, Hq, Hkv, d);
}

focus_status_t focus_decode_lists_init(const int32_t *offsets, const int32_t *pos, int B, int n,
                                       int num_groups, int topk, int cap, int32_t *glen,
                                       int32_t *gpos, void *stream)
{
    if (!offsets || !pos || !glen || !gpos) return FOCUS_ERR_INVALID_ARG;
    if (!aligned16(offsets) || !aligned16(pos) || !aligned16(glen) || !aligned16(gpos))
        return FOCUS_ERR_INVALID_ARG;
    if (B < 1 || n < 0 || num_groups < 1 || topk < 1 || topk > num_groups || cap < 1)
        return FOCUS_ERR_INVALID_ARG;
    if (num_groups > 1024 || topk > 8 || (int64_t)B * n * topk >= ((int64_t)1 << 31) ||
        (int64_t)B * num_groups > 65535)
        return FOCUS_ERR_UNSUPPORTED;
    int *status = nullptr;
    if (status_ptr(&status) != cudaSuccess) return FOCUS_ERR_CUDA;
    int launches = 0;
    cudaError_t e = launch_decode_lists_init(offsets, pos, B, n, num_groups, topk, cap, glen,
                                             gpos, status, static_cast<cudaStream_t>(stream),
                                             &launches);
    if (e == cudaSuccess) g_last_launches = launches;
    return cuda_status(e);
}

focus_status_t focus_decode_fwd(const void *q, const void *Kc, const void *Vc, const int32_t *ids,
                                int B, int L, int Lmax, int Hq, int Hkv, int d, int window,
                                float scale, int num_groups, int topk, int32_t *glen,
                                int32_t *gpos, int cap, void *O, float *lse, void *ws,
                                size_t ws_bytes, void *stream)
{
    if (!q || !Kc || !Vc || !ids || !glen || !gpos || !O || !ws) return FOCUS_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(Kc) || !aligned16(Vc) || !aligned16(ids) ||
        !aligned16(glen) || !aligned16(gpos) || !aligned16(O) || !aligned16(ws) ||
        (lse && !aligned16(lse)))
        return FOCUS_ERR_INVALID_ARG;
    if (B < 1 || L < 1 || L > Lmax || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || window < 0 ||
        num_groups < 1 || topk < 1 || topk > num_groups || cap < 1)
        return FOCUS_ERR_INVALID_ARG;
    if ((d != 64 && d != 128) || Hq / Hkv > 8 || num_groups > 1024 || topk > 8 ||
        B > 65535 || Hkv > 65535 || (int64_t)B * Hq > ((int64_t)1 << 31) - 1)
        return FOCUS_ERR_UNSUPPORTED;
    if (ws_bytes < decode_ws_bytes(B, Hq, Hkv, d)) return FOCUS_ERR_WORKSPACE;
    int *status = nullptr;
    if (status_ptr(&status) != cudaSuccess) return FOCUS_ERR_CUDA;
    if (decode_preflight(d) != cudaSuccess) return FOCUS_ERR_CUDA;
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf((float)d);
    DecodeLaunch p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k = static_cast<const __nv_bfloat16 *>(Kc);
    p.v = static_cast<const __nv_bfloat16 *>(Vc);
    p.ids = ids;
    p.glen = glen;
    p.gpos = gpos;
    p.B = B;
    p.L = L;
    p.Lmax = Lmax;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.d = d;
    p.K = num_groups;
    p.topk = topk;
    p.cap = cap;
    p.window = window;
    p.scale_log2 = sc * 1.4426950408889634f;
    p.O = static_cast<__nv_bfloat16 *>(O);
    p.lse = lse;
    p.ws = ws;
    p.status = status;
    if (wait_ctl(&p.wc) != cudaSuccess) return FOCUS_ERR_CUDA;
    int launches = 0;
    cudaError_t e = launch_decode(p, static_cast<cudaStream_t>(stream), &launches);
    if (e == cudaSuccess) g_last_launches = launches;
    return cuda_status(e);
}

focus_status_t focus_set_wait_limit(unsigned long long ns)
{
    g_wait_limit_ns.store(ns ? ns : 2000000000ull);
    return FOCUS_OK;
}

focus_status_t focus_get_device_status(int reset)
{
    int *p = nullptr;
    if (status_ptr(&p) != cudaSuccess) return FOCUS_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return FOCUS_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return FOCUS_ERR_CUDA;
    if (reset) {
        const int z = 0;
        if (cudaMemcpy(p, &z, sizeof z, cudaMemcpyHostToDevice) != cudaSuccess)
            return FOCUS_ERR_CUDA;
    }
    return v;
}

}  // extern "C"
