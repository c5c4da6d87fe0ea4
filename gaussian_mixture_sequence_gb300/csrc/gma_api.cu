// C ABI of libgma: host-side validation, workspace layout and launch order.
// The operations are those of the GMA explainer "Gaussian Mixture Attention:
// Linear-Time Sequence Mixing via Probabilistic Latent Routing" (technical
// summary, "핵심 메커니즘" and "변형 및 학습"); see include/gma.h.
#include "gma_internal.cuh"

#include <math.h>

#include <atomic>
#include <mutex>

using namespace gma;

namespace {

struct WsPlan {
    size_t zq = 0;        // the routing of Q's zero-lo-plane flags (bounded routing, split layout)
    size_t prm = 0, cst = 0, gq = 0, gk = 0, partial = 0, total = 0, mem = 0, wimg = 0, wimg3 = 0, pimg = 0,
           cimg = 0, pimg2 = 0, dctl = 0, dlist = 0, dlist2 = 0, bytes = 0;
    long long dcap = 0;   // dense-list entries per head
    bool pruned = false;  // the bounded routing (K = 128, d = 64)
    bool gtc = false;     // the tensor-core routing for 17 <= K <= 256 (not 128), d = 64
};

bool valid_width(int w) { return w == 16 || w == 32 || w == 64 || w == 128; }

gma_status make_dims_raw(const gma_shape *s, Dims *dm);
#define GMA_TRY_DIMS(expr)                                                                                 \
    do {                                                                                                   \
        const gma_status _d = (expr);                                                                      \
        if (_d != GMA_OK) return _d;                                                                       \
    } while (0)

// Dims of one operation: only the causal form uses the tensor-core chunking.
gma_status make_dims(const gma_shape *s, Dims *dm, gma_op op = GMA_OP_CAUSAL)
{
    const gma_status st = make_dims_raw(s, dm);
    if (st == GMA_OK && op != GMA_OP_CAUSAL && op != GMA_OP_BIDIR && dm->C == 128) {
        dm->C = 64;
        dm->blk = kBlockRows;
        dm->KG = dm->KP;
    }
    return st;
}

// Dims of the gradient pass: the CUDA-core chunking (C = 64, blocks of kBlockRows rows) and
// fp32 responsibilities whatever the shape's chunk and product type.
gma_status make_dims_bwd(const gma_shape *s, Dims *dm)
{
    if (!s) return GMA_ERR_INVALID_ARG;
    gma_shape t = *s;
    t.chunk = 64;
    t.gemm_dtype = GMA_F32;
    GMA_TRY_DIMS(make_dims_raw(&t, dm));
    return GMA_OK;
}

gma_status make_dims_raw(const gma_shape *s, Dims *dm)
{
    if (!s) return GMA_ERR_INVALID_ARG;
    if (s->B < 1 || s->H < 1 || s->N < 0 || s->K < 1 || s->d_route < 1 || s->d_v < 1 || s->chunk < 0)
        return GMA_ERR_INVALID_ARG;
    if (!(s->eps >= 0.f) || !isfinite(s->eps)) return GMA_ERR_INVALID_ARG;
    if ((unsigned)s->x_dtype > 1u || (unsigned)s->v_dtype > 1u || (unsigned)s->gemm_dtype > 1u)
        return GMA_ERR_INVALID_ARG;
    if (!valid_width(s->d_route) || !valid_width(s->d_v) || s->K > 512) return GMA_ERR_UNSUPPORTED;
    const bool tc = tc_path_eligible(s->K, s->d_v, s->gemm_dtype == GMA_BF16);
    const int C = s->chunk == 0 ? (tc ? 128 : 64) : s->chunk;
    if (C != 16 && C != 32 && C != 64 && !(C == 128 && tc)) return GMA_ERR_UNSUPPORTED;
    const long long BH = (long long)s->B * s->H;
    if (BH > 65535) return GMA_ERR_UNSUPPORTED;
    const long long w = s->K > s->d_v ? (s->K > s->d_route ? s->K : s->d_route)
                                      : (s->d_v > s->d_route ? s->d_v : s->d_route);
    if (BH * (long long)s->N * w >= (1LL << 40)) return GMA_ERR_UNSUPPORTED;
    dm->B = s->B; dm->H = s->H; dm->N = s->N; dm->D = s->d_route; dm->DV = s->d_v; dm->K = s->K;
    dm->KP = (int)round_up(s->K, 8);
    dm->KG = C == 128 ? tc_kpad(s->K) : dm->KP;
    dm->C = C;
    dm->blk = C == 128 ? 128 : kBlockRows;
    dm->eps = s->eps;
    dm->x_bf16 = s->x_dtype == GMA_BF16;
    dm->v_bf16 = s->v_dtype == GMA_BF16;
    dm->g_bf16 = s->gemm_dtype == GMA_BF16;
    return GMA_OK;
}

// The bounded routing's per-head images and its two tile lists (dcap entries per head each), and
// (zq_words > 0) the routing of Q's flags of tiles whose lo plane it leaves unwritten.
template <class Take>
void plan_pruned(WsPlan &p, int H, long long dcap, Take &&take, long long zq_words = 0)
{
    p.pruned = true;
    if (zq_words > 0) p.zq = take((size_t)zq_words * 4);
    p.wimg = take((size_t)H * kPrunedWBytes);
    p.wimg3 = take((size_t)H * kPrunedW3Bytes);
    p.pimg = take((size_t)H * kPrunedPBytes);
    p.cimg = take((size_t)H * kPrunedCBytes);
    p.pimg2 = take((size_t)H * kPrunedP2Bytes);
    p.dcap = dcap;
    p.dctl = take((size_t)H * 2 * 4);
    p.dlist = take((size_t)H * dcap * 8);
    p.dlist2 = take((size_t)H * dcap * 8);
}

int gamma_layout(const Dims &dm);

WsPlan plan(const Dims &dm, gma_op op)
{
    WsPlan p;
    size_t off = 0;
    auto take = [&](size_t n) {
        const size_t o = off;
        off = (size_t)round_up((long long)(off + n), 256);
        return o;
    };
    p.prm = take((size_t)dm.H * dm.K * (dm.D / 2) * 16);
    p.cst = take((size_t)dm.H * dm.K * 4);
    if (op != GMA_OP_DECODE && resp_pruned_applies(dm))   // both routings of a head; the flags where
        plan_pruned(p, dm.H, 2 * routing_tiles(dm.B, dm.N), take,   // the chunk kernels read split planes
                    (op == GMA_OP_BIDIR || op == GMA_OP_CAUSAL) && gamma_layout(dm) == GL_SPLIT
                        ? dm.BH() * ((dm.N + 127) / 128) : 0);
    if (op != GMA_OP_DECODE && resp_gtc_applies(dm)) {
        p.gtc = true;
        p.wimg3 = take(gtc_image_bytes(dm));
    }
    if (op == GMA_OP_USAGE) {   // Gamma in fp32, then the per-block partial sums and counts
        p.gq = take((size_t)dm.BH() * dm.N * dm.K * 4);
        p.partial = take((size_t)dm.BH() * usage_blocks(dm) * dm.K * 4);
        p.total = take((size_t)dm.BH() * usage_blocks(dm) * dm.K * 4);
    }
    if (op == GMA_OP_BIDIR || op == GMA_OP_CAUSAL) {
        const size_t gb = dm.g_bf16 ? 2 : 4;
        p.gq = take((size_t)dm.BH() * dm.N * dm.KG * gb);
        p.gk = take((size_t)dm.BH() * dm.N * dm.KG * gb);
        p.partial = take((size_t)dm.BH() * dm.nblk() * dm.state_size() * 4);
        const bool tc = tc_path_applies(dm);
        if (op == GMA_OP_BIDIR)   // the total memory: fp32, or in operand form on the tensor-core path
            p.total = take((size_t)dm.BH() * (tc ? tc_mem_words(dm) : dm.state_size()) * 4);
        if (op == GMA_OP_CAUSAL && tc)   // the carried memory of every chunk in operand form
            p.mem = take((size_t)dm.BH() * dm.nblk() * tc_mem_words(dm) * 4);
    }
    p.bytes = off;
    return p;
}

// Workspace form of the responsibilities: the fp32 tensor-core path takes split bf16 planes.
int gamma_layout(const Dims &dm) { return dm.g_bf16 ? GL_BF16 : (tc_path_applies(dm) ? GL_SPLIT : GL_F32); }

bool aligned(const void *p) { return ((uintptr_t)p & 15u) == 0; }

gma_status check_ptr(const void *p, bool required = true)
{
    if (!p) return required ? GMA_ERR_INVALID_ARG : GMA_OK;
    return aligned(p) ? GMA_OK : GMA_ERR_ALIGNMENT;
}

gma_status check_params(const gma_params &p)
{
    gma_status s;
    if ((s = check_ptr(p.mu)) != GMA_OK) return s;
    if ((s = check_ptr(p.var_raw)) != GMA_OK) return s;
    return check_ptr(p.logit_pi);
}

gma_status check_ws(void *ws, size_t ws_bytes, const WsPlan &wp)
{
    if (!ws || ws_bytes < wp.bytes) return GMA_ERR_WORKSPACE;
    return aligned(ws) ? GMA_OK : GMA_ERR_ALIGNMENT;
}

#define GMA_TRY(expr)                                                                                      \
    do {                                                                                                   \
        gma_status _s = (expr);                                                                            \
        if (_s != GMA_OK) return _s;                                                                       \
    } while (0)
// The CUDA error behind the last GMA_ERR_CUDA returned on this thread.
thread_local cudaError_t g_last_cuda = cudaSuccess;
#define GMA_CUDA(expr)                                                                                     \
    do {                                                                                                   \
        const cudaError_t _e = (expr);                                                                     \
        if (_e != cudaSuccess) {                                                                           \
            g_last_cuda = _e;                                                                              \
            return GMA_ERR_CUDA;                                                                           \
        }                                                                                                  \
    } while (0)

// A bounded device wait that expired since the last report on the current device:
// GMA_ERR_TIMEOUT once (the flag is cleared), else GMA_OK.  Never allocates and
// never synchronises: a timeout becomes visible once the kernel that hit it has
// written the flag.
gma_status take_timeout()
{
    volatile unsigned int *f = timeout_flag_host();
    if (f && *f) {
        *f = 0u;
        return GMA_ERR_TIMEOUT;
    }
    return GMA_OK;
}

template <typename T>
T *at(void *ws, size_t off) { return reinterpret_cast<T *>(static_cast<char *>(ws) + off); }

// Device copies of the inputs and the output for gma_forward_causal_host.
struct HostStaging {
    size_t q = 0, k = 0, v = 0, out = 0, bytes = 0;
};
HostStaging host_staging(const Dims &dm)
{
    HostStaging h;
    const size_t rows = (size_t)dm.BH() * dm.N;
    auto take = [&](size_t n) {
        const size_t o = h.bytes;
        h.bytes = (size_t)round_up((long long)(h.bytes + n), 256);
        return o;
    };
    h.q = take(rows * dm.D * (dm.x_bf16 ? 2 : 4));
    h.k = take(rows * dm.D * (dm.x_bf16 ? 2 : 4));
    h.v = take(rows * dm.DV * (dm.v_bf16 ? 2 : 4));
    h.out = take(rows * dm.DV * 4);
    return h;
}

// Workspace of the gradient pass.
struct BwdPlan {
    WsPlan w;   // parameters, routing images, gq / gk (fp32), forward memory (partial, total)
    size_t dgq = 0, dgk = 0, u = 0, mem = 0, rtot = 0, pmu = 0, pvar = 0, plp = 0, bytes = 0;
};
BwdPlan plan_bwd_full(const Dims &dm)
{
    BwdPlan b;
    size_t off = 0;
    auto take = [&](size_t n) {
        const size_t o = off;
        off = (size_t)round_up((long long)(off + n), 256);
        return o;
    };
    WsPlan &p = b.w;
    p.prm = take((size_t)dm.H * dm.K * (dm.D / 2) * 16);
    p.cst = take((size_t)dm.H * dm.K * 4);
    if (resp_pruned_applies(dm)) plan_pruned(p, dm.H, 2 * routing_tiles(dm.B, dm.N), take);
    if (resp_gtc_applies(dm)) {
        p.gtc = true;
        p.wimg3 = take(gtc_image_bytes(dm));
    }
    const size_t rows = (size_t)dm.BH() * dm.N, nb = (size_t)dm.BH() * dm.nblk();
    p.gq = take(rows * dm.KP * 4);
    p.gk = take(rows * dm.KP * 4);
    p.partial = take(nb * dm.state_size() * 4);
    p.total = take((size_t)dm.BH() * dm.state_size() * 4);
    b.dgq = take(rows * dm.KP * 4);
    b.dgk = take(rows * dm.KP * 4);
    b.u = take(rows * bwd_u_pitch(dm) * 4);
    b.mem = take(nb * dm.K * bwd_u_pitch(dm) * 4);
    b.rtot = take((size_t)dm.BH() * dm.K * bwd_u_pitch(dm) * 4);
    b.pmu = take(2 * nb * dm.K * dm.D * 4);
    b.pvar = take(2 * nb * dm.K * dm.D * 4);
    b.plp = take(2 * nb * dm.K * 4);
    b.bytes = p.bytes = off;
    return b;
}
WsPlan plan_bwd(const Dims &dm) { return plan_bwd_full(dm).w; }

PrunedImages images(void *ws, const WsPlan &wp)
{
    return PrunedImages{at<unsigned char>(ws, wp.wimg), at<unsigned char>(ws, wp.wimg3), at<float4>(ws, wp.pimg),
                        at<float>(ws, wp.cimg), at<float4>(ws, wp.pimg2), at<unsigned int>(ws, wp.dctl),
                        at<int2>(ws, wp.dlist), at<int2>(ws, wp.dlist2), wp.dcap,
                        wp.zq ? at<unsigned int>(ws, wp.zq) : nullptr};
}

// The routing images a call passes to launch_resp (null for the generic CUDA-core routing).
const PrunedImages *routing_images(const WsPlan &wp, const PrunedImages &img)
{
    return wp.pruned || wp.gtc ? &img : nullptr;
}

// The per-head parameters and the images of the routing kernel the shape takes.
cudaError_t prep_routing(const Dims &dm, const gma_params &params, float4 *prm, float *cst, const WsPlan &wp,
                         const PrunedImages &img, cudaStream_t st)
{
    if (wp.pruned) return launch_prep_all(dm, params, prm, cst, img, st);
    cudaError_t e = launch_prep(dm, params, prm, cst, st);
    if (e == cudaSuccess && wp.gtc) e = launch_prep_gtc(dm, prm, cst, img.w3, st);
    return e;
}

} // namespace

extern "C" {

size_t gma_workspace_size(const gma_shape *shape, gma_op op)
{
    Dims dm;
    if (op == GMA_OP_CAUSAL_HOST) {
        if (make_dims(shape, &dm, GMA_OP_CAUSAL) != GMA_OK) return 0;
        return host_staging(dm).bytes + plan(dm, GMA_OP_CAUSAL).bytes;
    }
    if (op == GMA_OP_BACKWARD) return make_dims_bwd(shape, &dm) == GMA_OK ? plan_bwd(dm).bytes : 0;
    if (((unsigned)op > 3u && op != GMA_OP_USAGE) || make_dims(shape, &dm, op) != GMA_OK) return 0;
    return plan(dm, op).bytes;
}

const char *gma_last_cuda_error(void) { return cudaGetErrorName(g_last_cuda); }

const char *gma_status_string(gma_status status)
{
    switch (status) {
    case GMA_OK: return "ok";
    case GMA_ERR_INVALID_ARG: return "invalid argument";
    case GMA_ERR_UNSUPPORTED: return "unsupported size";
    case GMA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case GMA_ERR_WORKSPACE: return "workspace missing or too small";
    case GMA_ERR_CUDA: return "CUDA error";
    case GMA_ERR_TIMEOUT: return "a bounded device wait expired";
    default: return "unknown status";
    }
}

gma_status gma_responsibilities(const gma_shape *shape, gma_params params, const void *x, float *gamma,
                                void *ws, size_t ws_bytes, gma_stream_t stream)
{
    GMA_TRY(take_timeout());
    Dims dm;
    GMA_TRY(make_dims(shape, &dm, GMA_OP_RESPONSIBILITIES));
    GMA_TRY(check_params(params));
    GMA_TRY(check_ptr(x, dm.N > 0));
    GMA_TRY(check_ptr(gamma, dm.N > 0));
    const WsPlan wp = plan(dm, GMA_OP_RESPONSIBILITIES);
    GMA_TRY(check_ws(ws, ws_bytes, wp));
    if (dm.N == 0) return GMA_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float4 *prm = at<float4>(ws, wp.prm);
    float *cst = at<float>(ws, wp.cst);
    const PrunedImages img = images(ws, wp);
    GMA_CUDA(prep_routing(dm, params, prm, cst, wp, img, st));
    GMA_CUDA(launch_resp(dm, prm, cst, routing_images(wp, img), x, gamma, dm.K, GL_F32, st, 0));
    if (wp.pruned) GMA_CUDA(launch_resp_dense(dm, x, gamma, dm, nullptr, nullptr, img, GL_F32, st));
    return GMA_OK;
}

gma_status gma_responsibility_stats(const gma_shape *shape, gma_params params, const void *x, float *usage,
                                    long long *counts, float *entropy, int *assign, void *ws, size_t ws_bytes,
                                    gma_stream_t stream)
{
    GMA_TRY(take_timeout());
    Dims dm;
    GMA_TRY(make_dims(shape, &dm, GMA_OP_USAGE));
    GMA_TRY(check_params(params));
    GMA_TRY(check_ptr(x, dm.N > 0));
    GMA_TRY(check_ptr(usage));
    GMA_TRY(check_ptr(counts));
    GMA_TRY(check_ptr(entropy));
    GMA_TRY(check_ptr(assign, false));
    const WsPlan wp = plan(dm, GMA_OP_USAGE);
    GMA_TRY(check_ws(ws, ws_bytes, wp));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float *gamma = at<float>(ws, wp.gq);
    if (dm.N > 0) {
        float4 *prm = at<float4>(ws, wp.prm);
        float *cst = at<float>(ws, wp.cst);
        const PrunedImages img = images(ws, wp);
        GMA_CUDA(prep_routing(dm, params, prm, cst, wp, img, st));
        GMA_CUDA(launch_resp(dm, prm, cst, routing_images(wp, img), x, gamma, dm.K, GL_F32, st, 0));
        if (wp.pruned) GMA_CUDA(launch_resp_dense(dm, x, gamma, dm, nullptr, nullptr, img, GL_F32, st));
    }
    GMA_CUDA(launch_usage(dm, gamma, dm.K, at<float>(ws, wp.partial), at<int>(ws, wp.total), assign, usage, counts,
                          entropy, st));
    return GMA_OK;
}


} // extern "C"

namespace {

// Records the profiling event of the next launch (no-op without a profile).
struct Marks {
    gma_profile *prof;
    int n = 0;
    cudaStream_t st;
    cudaError_t mark(const char *name)
    {
        if (!prof) return cudaSuccess;
        if (n >= GMA_PROFILE_MAX_STAGES) return cudaErrorInvalidValue;
        prof->stage_name[n] = name;
        return cudaEventRecord(static_cast<cudaEvent_t>(prof->events[n++]), st);
    }
    cudaError_t finish()
    {
        if (!prof) return cudaSuccess;
        prof->n_stages = n;
        return cudaEventRecord(static_cast<cudaEvent_t>(prof->events[n]), st);
    }
};

gma_status check_prof(gma_profile *prof)
{
    if (!prof) return GMA_OK;
    for (int i = 0; i <= GMA_PROFILE_MAX_STAGES; ++i)
        if (!prof->events[i]) return GMA_ERR_INVALID_ARG;
    prof->n_stages = 0;
    return GMA_OK;
}

gma_status run_bidir(const gma_shape *shape, gma_params params, const void *qx, const void *kx, const void *v,
                     float *out, void *ws, size_t ws_bytes, gma_stream_t stream, gma_profile *prof)
{
    Dims dm;
    GMA_TRY(make_dims(shape, &dm, GMA_OP_BIDIR));
    GMA_TRY(check_params(params));
    GMA_TRY(check_ptr(qx, dm.N > 0));
    GMA_TRY(check_ptr(kx, dm.N > 0));
    GMA_TRY(check_ptr(v, dm.N > 0));
    GMA_TRY(check_ptr(out, dm.N > 0));
    const WsPlan wp = plan(dm, GMA_OP_BIDIR);
    GMA_TRY(check_ws(ws, ws_bytes, wp));
    GMA_TRY(check_prof(prof));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Marks mk{prof, 0, st};
    if (dm.N == 0) {
        GMA_CUDA(mk.finish());
        return GMA_OK;
    }
    float4 *prm = at<float4>(ws, wp.prm);
    float *cst = at<float>(ws, wp.cst);
    void *gq = at<char>(ws, wp.gq), *gk = at<char>(ws, wp.gk);
    float *partial = at<float>(ws, wp.partial), *total = at<float>(ws, wp.total);
    const PrunedImages img = images(ws, wp);
    const PrunedImages *imgp = routing_images(wp, img);
    GMA_CUDA(mk.mark(wp.pruned ? "prep" : "prep_params"));
    GMA_CUDA(prep_routing(dm, params, prm, cst, wp, img, st));
    GMA_CUDA(mk.mark("resp_q"));
    GMA_CUDA(launch_resp(dm, prm, cst, imgp, qx, gq, dm.KG, gamma_layout(dm), st, 0));
    GMA_CUDA(mk.mark("resp_k"));
    GMA_CUDA(launch_resp(dm, prm, cst, imgp, kx, gk, dm.KG, gamma_layout(dm), st, 1));
    if (wp.pruned) {
        GMA_CUDA(mk.mark("resp_dense"));
        GMA_CUDA(launch_resp_dense(dm, qx, gq, dm, kx, gk, img, gamma_layout(dm), st));
    }
    if (tc_path_applies(dm)) {
        GMA_CUDA(mk.mark("chunk_state_tc"));
        GMA_CUDA(launch_chunk_state_tc(dm, gk, v, partial, st));
        GMA_CUDA(mk.mark("state_reduce"));
        unsigned char *tot = at<unsigned char>(ws, wp.total);
        GMA_CUDA(launch_scan_split(dm, partial, nullptr, nullptr, tot, nullptr, st));
        GMA_CUDA(mk.mark("bidir_read_tc"));
        GMA_CUDA(launch_chunk_out_tc(dm, false, gq, gk, v, tot, out, st, img.zq));
    } else {
        GMA_CUDA(mk.mark("block_state"));
        GMA_CUDA(launch_block_state(dm, gk, v, partial, st));
        GMA_CUDA(mk.mark("state_reduce"));
        GMA_CUDA(launch_scan(dm, partial, nullptr, total, false, st));
        GMA_CUDA(mk.mark("bidir_read"));
        GMA_CUDA(launch_chunk_out(dm, false, gq, gk, v, total, out, st));
    }
    GMA_CUDA(mk.finish());
    return GMA_OK;
}

// Workspace of the cross form: queries of dm_q, keys and values of dm_kv (same B, H, d, K).
WsPlan plan_cross(const Dims &dq, const Dims &dk)
{
    WsPlan p;
    size_t off = 0;
    auto take = [&](size_t n) {
        const size_t o = off;
        off = (size_t)round_up((long long)(off + n), 256);
        return o;
    };
    p.prm = take((size_t)dq.H * dq.K * (dq.D / 2) * 16);
    p.cst = take((size_t)dq.H * dq.K * 4);
    if (resp_pruned_applies(dq))
        plan_pruned(p, dq.H, routing_tiles(dq.B, dq.N) + routing_tiles(dk.B, dk.N), take,
                    gamma_layout(dq) == GL_SPLIT ? dq.BH() * ((dq.N + 127) / 128) : 0);
    if (resp_gtc_applies(dq)) {
        p.gtc = true;
        p.wimg3 = take(gtc_image_bytes(dq));
    }
    const size_t gb = dq.g_bf16 ? 2 : 4;
    p.gq = take((size_t)dq.BH() * dq.N * dq.KG * gb);
    p.gk = take((size_t)dk.BH() * dk.N * dk.KG * gb);
    p.partial = take((size_t)dk.BH() * dk.nblk() * dk.state_size() * 4);
    p.total = take((size_t)dk.BH() * (tc_path_applies(dq) ? tc_mem_words(dq) : dk.state_size()) * 4);
    p.bytes = off;
    return p;
}

gma_status cross_dims(const gma_shape *shape, int n_kv, Dims *dq, Dims *dk)
{
    GMA_TRY(make_dims(shape, dq, GMA_OP_BIDIR));
    if (n_kv < 0) return GMA_ERR_INVALID_ARG;
    gma_shape sk = *shape;
    sk.N = n_kv;
    return make_dims(&sk, dk, GMA_OP_BIDIR);
}

// Queries of dq read the memory written by all keys of dk: the bidirectional write over
// dk's rows, then the bidirectional read over dq's rows.
gma_status run_cross(const gma_shape *shape, int n_kv, gma_params params, const void *qx, const void *kx,
                     const void *v, float *out, void *ws, size_t ws_bytes, gma_stream_t stream)
{
    Dims dq, dk;
    GMA_TRY(cross_dims(shape, n_kv, &dq, &dk));
    GMA_TRY(check_params(params));
    GMA_TRY(check_ptr(qx, dq.N > 0));
    GMA_TRY(check_ptr(out, dq.N > 0));
    GMA_TRY(check_ptr(kx, dk.N > 0 && dq.N > 0));
    GMA_TRY(check_ptr(v, dk.N > 0 && dq.N > 0));
    const WsPlan wp = plan_cross(dq, dk);
    GMA_TRY(check_ws(ws, ws_bytes, wp));
    if (dq.N == 0) return GMA_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float4 *prm = at<float4>(ws, wp.prm);
    float *cst = at<float>(ws, wp.cst);
    void *gq = at<char>(ws, wp.gq), *gk = at<char>(ws, wp.gk);
    float *partial = at<float>(ws, wp.partial), *total = at<float>(ws, wp.total);
    const PrunedImages img = images(ws, wp);
    const PrunedImages *imgp = routing_images(wp, img);
    GMA_CUDA(prep_routing(dq, params, prm, cst, wp, img, st));
    GMA_CUDA(launch_resp(dq, prm, cst, imgp, qx, gq, dq.KG, gamma_layout(dq), st, 0));
    if (dk.N > 0) GMA_CUDA(launch_resp(dk, prm, cst, imgp, kx, gk, dk.KG, gamma_layout(dk), st, 1));
    if (wp.pruned)
        GMA_CUDA(launch_resp_dense(dq, qx, gq, dk, dk.N > 0 ? kx : nullptr, gk, img, gamma_layout(dq), st));
    const bool tc = tc_path_applies(dq);
    if (dk.N == 0) {   // no keys: an empty memory (zeros in either layout)
        GMA_CUDA(cudaMemsetAsync(total, 0, (size_t)dk.BH() * (tc ? tc_mem_words(dk) : dk.state_size()) * 4, st));
    } else {
        if (tc) {
            GMA_CUDA(launch_chunk_state_tc(dk, gk, v, partial, st));
            GMA_CUDA(launch_scan_split(dk, partial, nullptr, nullptr, reinterpret_cast<unsigned char *>(total),
                                       nullptr, st));
        } else {
            GMA_CUDA(launch_block_state(dk, gk, v, partial, st));
            GMA_CUDA(launch_scan(dk, partial, nullptr, total, false, st));
        }
    }
    if (tc)
        GMA_CUDA(launch_chunk_out_tc(dq, false, gq, gq, nullptr, reinterpret_cast<unsigned char *>(total), out, st,
                                     img.zq));
    else
        GMA_CUDA(launch_chunk_out(dq, false, gq, gq, nullptr, total, out, st));
    return GMA_OK;
}

gma_status run_decode(const gma_shape *shape, gma_params params, const void *qx, const void *kx, const void *v,
                      float *state, float *out, void *ws, size_t ws_bytes, gma_stream_t stream, gma_profile *prof)
{
    Dims dm;
    GMA_TRY(make_dims(shape, &dm, GMA_OP_DECODE));
    GMA_TRY(check_params(params));
    GMA_TRY(check_ptr(qx));
    GMA_TRY(check_ptr(kx));
    GMA_TRY(check_ptr(v));
    GMA_TRY(check_ptr(state));
    GMA_TRY(check_ptr(out));
    const WsPlan wp = plan(dm, GMA_OP_DECODE);
    GMA_TRY(check_ws(ws, ws_bytes, wp));
    GMA_TRY(check_prof(prof));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Marks mk{prof, 0, st};
    float4 *prm = at<float4>(ws, wp.prm);
    float *cst = at<float>(ws, wp.cst);
    // one stage: the decode kernel is a programmatic dependent of the parameter preparation and
    // overlaps it (an event recorded between the two would serialise them)
    GMA_CUDA(mk.mark("decode"));
    GMA_CUDA(launch_prep(dm, params, prm, cst, st));
    GMA_CUDA(launch_decode(dm, prm, cst, qx, kx, v, state, out, st));
    GMA_CUDA(mk.finish());
    return GMA_OK;
}

gma_status run_causal(const gma_shape *shape, gma_params params, const void *qx, const void *kx,
                      const void *v, const float *state_in, float *state_out, float *out, void *ws,
                      size_t ws_bytes, gma_stream_t stream, gma_profile *prof)
{
    Dims dm;
    GMA_TRY(make_dims(shape, &dm));
    GMA_TRY(check_params(params));
    GMA_TRY(check_ptr(qx, dm.N > 0));
    GMA_TRY(check_ptr(kx, dm.N > 0));
    GMA_TRY(check_ptr(v, dm.N > 0));
    GMA_TRY(check_ptr(out, dm.N > 0));
    GMA_TRY(check_ptr(state_in, false));
    GMA_TRY(check_ptr(state_out, false));
    const WsPlan wp = plan(dm, GMA_OP_CAUSAL);
    GMA_TRY(check_ws(ws, ws_bytes, wp));
    GMA_TRY(check_prof(prof));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    Marks mk{prof, 0, st};
    if (dm.N == 0) {
        if (state_out && state_out != state_in) {
            const size_t bytes = (size_t)dm.BH() * dm.state_size() * 4;
            if (state_in)
                GMA_CUDA(cudaMemcpyAsync(state_out, state_in, bytes, cudaMemcpyDeviceToDevice, st));
            else
                GMA_CUDA(cudaMemsetAsync(state_out, 0, bytes, st));
        }
        GMA_CUDA(mk.finish());
        return GMA_OK;
    }
    float4 *prm = at<float4>(ws, wp.prm);
    float *cst = at<float>(ws, wp.cst);
    void *gq = at<char>(ws, wp.gq), *gk = at<char>(ws, wp.gk);
    float *partial = at<float>(ws, wp.partial);
    const PrunedImages img = images(ws, wp);
    const PrunedImages *imgp = routing_images(wp, img);
    GMA_CUDA(mk.mark(wp.pruned ? "prep" : "prep_params"));
    GMA_CUDA(prep_routing(dm, params, prm, cst, wp, img, st));
    GMA_CUDA(mk.mark("resp_q"));
    GMA_CUDA(launch_resp(dm, prm, cst, imgp, qx, gq, dm.KG, gamma_layout(dm), st, 0));
    GMA_CUDA(mk.mark("resp_k"));
    GMA_CUDA(launch_resp(dm, prm, cst, imgp, kx, gk, dm.KG, gamma_layout(dm), st, 1));
    if (wp.pruned) {
        GMA_CUDA(mk.mark("resp_dense"));
        GMA_CUDA(launch_resp_dense(dm, qx, gq, dm, kx, gk, img, gamma_layout(dm), st));
    }
    if (tc_path_applies(dm)) {
        GMA_CUDA(mk.mark("chunk_state_tc"));
        GMA_CUDA(launch_chunk_state_tc(dm, gk, v, partial, st));
        GMA_CUDA(mk.mark("state_scan"));
        unsigned char *mem = at<unsigned char>(ws, wp.mem);
        GMA_CUDA(launch_scan_split(dm, partial, state_in, mem, nullptr, state_out, st));
        GMA_CUDA(mk.mark("chunk_out_tc"));
        GMA_CUDA(launch_chunk_out_tc(dm, true, gq, gk, v, mem, out, st, img.zq));
    } else {
        GMA_CUDA(mk.mark("block_state"));
        GMA_CUDA(launch_block_state(dm, gk, v, partial, st));
        GMA_CUDA(mk.mark("state_scan"));
        GMA_CUDA(launch_scan(dm, partial, state_in, state_out, true, st));
        GMA_CUDA(mk.mark("chunk_out"));
        GMA_CUDA(launch_chunk_out(dm, true, gq, gk, v, partial, out, st));
    }
    GMA_CUDA(mk.finish());
    return GMA_OK;
}

} // namespace

extern "C" {

gma_status gma_forward_causal(const gma_shape *shape, gma_params params, const void *qx, const void *kx,
                              const void *v, const float *state_in, float *state_out, float *out, void *ws,
                              size_t ws_bytes, gma_stream_t stream)
{
    GMA_TRY(take_timeout());
    return run_causal(shape, params, qx, kx, v, state_in, state_out, out, ws, ws_bytes, stream, nullptr);
}

gma_status gma_forward_bidir(const gma_shape *shape, gma_params params, const void *qx, const void *kx,
                             const void *v, float *out, void *ws, size_t ws_bytes, gma_stream_t stream)
{
    GMA_TRY(take_timeout());
    return run_bidir(shape, params, qx, kx, v, out, ws, ws_bytes, stream, nullptr);
}

gma_status gma_forward_bidir_profiled(const gma_shape *shape, gma_params params, const void *qx,
                                      const void *kx, const void *v, float *out, void *ws, size_t ws_bytes,
                                      gma_stream_t stream, gma_profile *prof)
{
    GMA_TRY(take_timeout());
    if (!prof) return GMA_ERR_INVALID_ARG;
    return run_bidir(shape, params, qx, kx, v, out, ws, ws_bytes, stream, prof);
}

gma_status gma_decode_step(const gma_shape *shape, gma_params params, const void *qx, const void *kx,
                           const void *v, float *state, float *out, void *ws, size_t ws_bytes,
                           gma_stream_t stream)
{
    GMA_TRY(take_timeout());
    return run_decode(shape, params, qx, kx, v, state, out, ws, ws_bytes, stream, nullptr);
}

gma_status gma_decode_step_profiled(const gma_shape *shape, gma_params params, const void *qx, const void *kx,
                                    const void *v, float *state, float *out, void *ws, size_t ws_bytes,
                                    gma_stream_t stream, gma_profile *prof)
{
    GMA_TRY(take_timeout());
    if (!prof) return GMA_ERR_INVALID_ARG;
    return run_decode(shape, params, qx, kx, v, state, out, ws, ws_bytes, stream, prof);
}

gma_status gma_forward_causal_profiled(const gma_shape *shape, gma_params params, const void *qx,
                                       const void *kx, const void *v, const float *state_in,
                                       float *state_out, float *out, void *ws, size_t ws_bytes,
                                       gma_stream_t stream, gma_profile *prof)
{
    GMA_TRY(take_timeout());
    if (!prof) return GMA_ERR_INVALID_ARG;
    return run_causal(shape, params, qx, kx, v, state_in, state_out, out, ws, ws_bytes, stream, prof);
}


} // extern "C"

// ---- causal forward on host buffers ----------------------------------------
namespace {

constexpr int kMaxCopyDevices = 64;
std::once_flag g_copy_once[kMaxCopyDevices];
cudaStream_t g_copy_in[kMaxCopyDevices], g_copy_out[kMaxCopyDevices];
cudaError_t g_copy_err[kMaxCopyDevices];

// The two copy streams of the current device (created once, never destroyed).
gma_status copy_streams(cudaStream_t *in, cudaStream_t *out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GMA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxCopyDevices) return GMA_ERR_UNSUPPORTED;
    std::call_once(g_copy_once[dev], [dev] {
        g_copy_err[dev] = cudaStreamCreateWithFlags(&g_copy_in[dev], cudaStreamNonBlocking);
        if (g_copy_err[dev] == cudaSuccess)
            g_copy_err[dev] = cudaStreamCreateWithFlags(&g_copy_out[dev], cudaStreamNonBlocking);
    });
    if (g_copy_err[dev] != cudaSuccess) return GMA_ERR_CUDA;
    *in = g_copy_in[dev];
    *out = g_copy_out[dev];
    return GMA_OK;
}

// Records an event on `from` and makes `to` wait for it.
cudaError_t join(cudaStream_t to, cudaStream_t from)
{
    cudaEvent_t e;
    cudaError_t err = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (err != cudaSuccess) return err;
    err = cudaEventRecord(e, from);
    if (err == cudaSuccess) err = cudaStreamWaitEvent(to, e, 0);
    cudaEventDestroy(e);   // released once the recorded work completes
    return err;
}

} // namespace

extern "C" gma_status gma_forward_causal_host(const gma_shape *shape, gma_params params, const void *qx,
                                              const void *kx, const void *v, const float *state_in,
                                              float *state_out, float *out, void *ws, size_t ws_bytes,
                                              gma_stream_t stream)
{
    GMA_TRY(take_timeout());
    Dims dm;
    GMA_TRY(make_dims(shape, &dm));
    GMA_TRY(check_params(params));
    if (dm.N > 0 && (!qx || !kx || !v || !out)) return GMA_ERR_INVALID_ARG;
    GMA_TRY(check_ptr(state_in, false));
    GMA_TRY(check_ptr(state_out, false));
    const HostStaging hs = host_staging(dm);
    const WsPlan wp = plan(dm, GMA_OP_CAUSAL);
    if (!ws || ws_bytes < hs.bytes + wp.bytes) return GMA_ERR_WORKSPACE;
    if (!aligned(ws)) return GMA_ERR_ALIGNMENT;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char *w = static_cast<char *>(ws);
    char *cws = w + hs.bytes;
    const size_t cws_bytes = ws_bytes - hs.bytes;
    if (dm.N == 0)
        return run_causal(shape, params, nullptr, nullptr, nullptr, state_in, state_out, nullptr, cws, cws_bytes,
                          stream, nullptr);
    cudaStream_t cin, cout_;
    GMA_TRY(copy_streams(&cin, &cout_));
    // groups of slices: one batch entry and a range of heads, about eight groups in all
    const int split = dm.B >= 8 ? 1 : (8 + dm.B - 1) / dm.B;
    const int hg = (dm.H + split - 1) / split;
    const size_t xe = dm.x_bf16 ? 2 : 4, ve = dm.v_bf16 ? 2 : 4;
    const size_t xrow = (size_t)dm.N * dm.D * xe, vrow = (size_t)dm.N * dm.DV * ve, orow = (size_t)dm.N * dm.DV * 4;
    const long long SZ = dm.state_size();
    // the staging buffers may still be read by earlier work on `stream`
    GMA_CUDA(join(cin, st));
    for (int b = 0; b < dm.B; ++b)
        for (int h0 = 0; h0 < dm.H; h0 += hg) {
            const int hn = dm.H - h0 < hg ? dm.H - h0 : hg;
            const size_t s0 = (size_t)b * dm.H + h0;   // first slice of the group
            GMA_CUDA(cudaMemcpyAsync(w + hs.q + s0 * xrow, static_cast<const char *>(qx) + s0 * xrow, hn * xrow,
                                     cudaMemcpyHostToDevice, cin));
            GMA_CUDA(cudaMemcpyAsync(w + hs.k + s0 * xrow, static_cast<const char *>(kx) + s0 * xrow, hn * xrow,
                                     cudaMemcpyHostToDevice, cin));
            GMA_CUDA(cudaMemcpyAsync(w + hs.v + s0 * vrow, static_cast<const char *>(v) + s0 * vrow, hn * vrow,
                                     cudaMemcpyHostToDevice, cin));
            GMA_CUDA(join(st, cin));
            gma_shape sg = *shape;
            sg.B = 1;
            sg.H = hn;
            const gma_params pg{params.mu + (size_t)h0 * dm.K * dm.D, params.var_raw + (size_t)h0 * dm.K * dm.D,
                                params.logit_pi + (size_t)h0 * dm.K};
            GMA_TRY(run_causal(&sg, pg, w + hs.q + s0 * xrow, w + hs.k + s0 * xrow, w + hs.v + s0 * vrow,
                               state_in ? state_in + s0 * SZ : nullptr, state_out ? state_out + s0 * SZ : nullptr,
                               reinterpret_cast<float *>(w + hs.out + s0 * orow), cws, cws_bytes, stream, nullptr));
            GMA_CUDA(join(cout_, st));
            GMA_CUDA(cudaMemcpyAsync(reinterpret_cast<char *>(out) + s0 * orow, w + hs.out + s0 * orow, hn * orow,
                                     cudaMemcpyDeviceToHost, cout_));
        }
    GMA_CUDA(join(st, cout_));   // `stream` completes after the last output copy
    return GMA_OK;
}

// ---- decode step whose scratch is a file-scope device array ----------------
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[GMA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_noalloc_addr[kMaxDevices];

// Device address of the array on the current device.  In host code the
// array's name only stands in for it, so the address is looked up with that
// device current, and kept once a lookup has succeeded (a failed lookup, for
// example one made during a stream capture, is retried by the next call).
gma_status noalloc_scratch(void **addr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GMA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GMA_ERR_UNSUPPORTED;
    void *p = g_noalloc_addr[dev].load(std::memory_order_acquire);
    if (!p) {
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            g_last_cuda = e != cudaSuccess ? e : cudaErrorInvalidSymbol;
            return GMA_ERR_CUDA;
        }
        g_noalloc_addr[dev].store(p, std::memory_order_release);
    }
    *addr = p;
    return GMA_OK;
}

} // namespace

extern "C" gma_status gma_decode_step_noalloc(const gma_shape *shape, gma_params params, const void *qx,
                                              const void *kx, const void *v, float *state, float *out,
                                              gma_stream_t stream)
{
    GMA_TRY(take_timeout());
    Dims dm;
    GMA_TRY(make_dims(shape, &dm, GMA_OP_DECODE));
    GMA_TRY(check_params(params));
    GMA_TRY(check_ptr(qx));
    GMA_TRY(check_ptr(kx));
    GMA_TRY(check_ptr(v));
    GMA_TRY(check_ptr(state));
    GMA_TRY(check_ptr(out));
    const WsPlan wp = plan(dm, GMA_OP_DECODE);
    if (wp.bytes > GMA_NOALLOC_SCRATCH_BYTES) return GMA_ERR_WORKSPACE;
    void *ws = nullptr;
    GMA_TRY(noalloc_scratch(&ws));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float4 *prm = at<float4>(ws, wp.prm);
    float *cst = at<float>(ws, wp.cst);
    GMA_CUDA(launch_prep(dm, params, prm, cst, st));
    GMA_CUDA(launch_decode(dm, prm, cst, qx, kx, v, state, out, st));
    return GMA_OK;
}

extern "C" gma_status gma_sync_status(gma_stream_t stream)
{
    const cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        g_last_cuda = e;
        return GMA_ERR_CUDA;
    }
    return take_timeout();
}

extern "C" gma_status gma_test_wait_timeout(long long limit_cycles, gma_stream_t stream)
{
    if (limit_cycles < 1 || limit_cycles > 4000000000LL) return GMA_ERR_INVALID_ARG;
    GMA_CUDA(launch_expire_wait(limit_cycles, reinterpret_cast<cudaStream_t>(stream)));
    return GMA_OK;
}

extern "C" size_t gma_cross_workspace_size(const gma_shape *shape, int n_kv)
{
    Dims dq, dk;
    if (cross_dims(shape, n_kv, &dq, &dk) != GMA_OK) return 0;
    return plan_cross(dq, dk).bytes;
}

extern "C" gma_status gma_forward_cross(const gma_shape *shape, int n_kv, gma_params params, const void *qx,
                                        const void *kx, const void *v, float *out, void *ws, size_t ws_bytes,
                                        gma_stream_t stream)
{
    GMA_TRY(take_timeout());
    return run_cross(shape, n_kv, params, qx, kx, v, out, ws, ws_bytes, stream);
}

extern "C" gma_status gma_backward(const gma_shape *shape, int causal, gma_params params, const void *qx,
                                   const void *kx, const void *v, const float *dout, float *dqx, float *dkx,
                                   float *dv, float *dmu, float *dvar_raw, float *dlogit_pi, void *ws,
                                   size_t ws_bytes, gma_stream_t stream)
{
    GMA_TRY(take_timeout());
    Dims dm;
    GMA_TRY(make_dims_bwd(shape, &dm));
    if (causal != 0 && causal != 1) return GMA_ERR_INVALID_ARG;
    GMA_TRY(check_params(params));
    const bool any = dm.N > 0;
    GMA_TRY(check_ptr(qx, any));
    GMA_TRY(check_ptr(kx, any));
    GMA_TRY(check_ptr(v, any));
    GMA_TRY(check_ptr(dout, any));
    GMA_TRY(check_ptr(dqx, any));
    GMA_TRY(check_ptr(dkx, any));
    GMA_TRY(check_ptr(dv, any));
    GMA_TRY(check_ptr(dmu));
    GMA_TRY(check_ptr(dvar_raw));
    GMA_TRY(check_ptr(dlogit_pi));
    const BwdPlan bp = plan_bwd_full(dm);
    const WsPlan &wp = bp.w;
    GMA_TRY(check_ws(ws, ws_bytes, wp));
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!any) {
        GMA_CUDA(cudaMemsetAsync(dmu, 0, (size_t)dm.H * dm.K * dm.D * 4, st));
        GMA_CUDA(cudaMemsetAsync(dvar_raw, 0, (size_t)dm.H * dm.K * dm.D * 4, st));
        GMA_CUDA(cudaMemsetAsync(dlogit_pi, 0, (size_t)dm.H * dm.K * 4, st));
        return GMA_OK;
    }
    float4 *prm = at<float4>(ws, wp.prm);
    float *cst = at<float>(ws, wp.cst);
    float *gq = at<float>(ws, wp.gq), *gk = at<float>(ws, wp.gk);
    float *partial = at<float>(ws, wp.partial), *total = at<float>(ws, wp.total);
    const PrunedImages img = images(ws, wp);
    const PrunedImages *imgp = routing_images(wp, img);
    // the forward's responsibilities (fp32) and memory
    GMA_CUDA(prep_routing(dm, params, prm, cst, wp, img, st));
    GMA_CUDA(launch_resp(dm, prm, cst, imgp, qx, gq, dm.KP, GL_F32, st, 0));
    GMA_CUDA(launch_resp(dm, prm, cst, imgp, kx, gk, dm.KP, GL_F32, st, 1));
    if (wp.pruned) GMA_CUDA(launch_resp_dense(dm, qx, gq, dm, kx, gk, img, GL_F32, st));
    GMA_CUDA(launch_block_state(dm, gk, v, partial, st));
    GMA_CUDA(launch_scan(dm, partial, nullptr, causal ? nullptr : total, causal != 0, st));
    // query side, key / value side, then the routings and the parameters
    float *dgq = at<float>(ws, bp.dgq), *dgk = at<float>(ws, bp.dgk), *u = at<float>(ws, bp.u);
    GMA_CUDA(launch_bwd_q(dm, causal != 0, gq, gk, v, dout, causal ? partial : total, u, dgq, st));
    GMA_CUDA(launch_bwd_kv(dm, causal != 0, gq, gk, v, u, at<float>(ws, bp.mem), at<float>(ws, bp.rtot), dgk, dv, st));
    const size_t pass = (size_t)dm.BH() * dm.nblk() * dm.K;
    float *pmu = at<float>(ws, bp.pmu), *pvar = at<float>(ws, bp.pvar), *plp = at<float>(ws, bp.plp);
    GMA_CUDA(launch_bwd_route(dm, qx, prm, gq, dgq, dqx, pmu, pvar, plp, st));
    GMA_CUDA(launch_bwd_route(dm, kx, prm, gk, dgk, dkx, pmu + pass * dm.D, pvar + pass * dm.D, plp + pass, st));
    GMA_CUDA(launch_bwd_final(dm, params, pmu, pvar, plp, dmu, dvar_raw, dlogit_pi, st));
    return GMA_OK;
}
