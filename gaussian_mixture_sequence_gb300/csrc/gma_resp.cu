// Parameter preparation (S0) and the responsibility kernel (S1).
//
// S0 follows the reparameterisation of the GMA explainer ("변형 및 학습"):
// sigma^2 = softplus(var_raw), pi = softmax(logit_pi).  S1 evaluates the
// diagonal-GMM posterior of "핵심 메커니즘":
//   l_ik  = log pi_k - 1/2 sum_d [ (x_id - mu_kd)^2 / sigma_kd^2 + log sigma_kd^2 ]
//   gamma = softmax_k(l)              (the -d/2 log 2pi term cancels)
// The quadratic form is evaluated directly as ((x - mu) / sigma)^2 — never by
// expanding it into x^2 and x terms, which cancel catastrophically — using one
// packed fp32x2 FMA for (x * s - mu * s) and one for the square-accumulate.
#include "gma_internal.cuh"

#include <float.h>

namespace gma {
namespace {

__device__ __forceinline__ float softplus(float r) { return fmaxf(r, 0.f) + log1pf(expf(-fabsf(r))); }

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Grid (H, ceil(K / 32)): each CTA recomputes its head's log-sum-exp of the
// mixture logits (K <= 512 values, one per thread) and prepares 32 components,
// 16 threads per component over groups of four features (all of a thread's
// loads are issued before their results are used).
constexpr int kPrepComps = 32, kPrepThreads = 512;

__global__ void __launch_bounds__(kPrepThreads) k_prep(int K, int D, const float *__restrict__ mu,
                                                       const float *__restrict__ var_raw,
                                                       const float *__restrict__ logit_pi,
                                                       float4 *__restrict__ prm, float *__restrict__ cst)
{
    constexpr int NW = kPrepThreads / 32;
    __shared__ float red[NW];
    __shared__ float bcast[2];
    // a kernel launched as a programmatic dependent of this one (the decode step) may start
    // now; it waits for this grid's results before it reads them
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int h = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = blockIdx.y * kPrepComps + (tid >> 4), part = tid & 15;
    const float *l = logit_pi + (long long)h * K;

    // this thread's features 4 part + 64 j of component k (D / 4 groups of four, up to 2 per thread)
    const int G = D / 4;
    float4 r4[2], u4[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int g = part + 16 * j;
        const bool on = k < K && g < G;
        const long long e = ((long long)h * K + k) * D + 4 * g;
        r4[j] = on ? *reinterpret_cast<const float4 *>(var_raw + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        u4[j] = on ? *reinterpret_cast<const float4 *>(mu + e) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float lv = tid < K ? l[tid] : -FLT_MAX;

    float t = warp_max(lv);
    if (lane == 0) red[warp] = t;
    __syncthreads();
    if (warp == 0) {
        t = warp_max(lane < NW ? red[lane] : -FLT_MAX);
        if (lane == 0) bcast[0] = t;
    }
    __syncthreads();
    const float lmax = bcast[0];
    t = warp_sum(tid < K ? expf(lv - lmax) : 0.f);
    __syncthreads();   // red is reused
    if (lane == 0) red[warp] = t;
    __syncthreads();
    if (warp == 0) {
        t = warp_sum(lane < NW ? red[lane] : 0.f);
        if (lane == 0) bcast[1] = lmax + logf(t);
    }

    float lsum = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int g = part + 16 * j;
        if (k < K && g < G) {
            const float rv[4] = {r4[j].x, r4[j].y, r4[j].z, r4[j].w}, uv[4] = {u4[j].x, u4[j].y, u4[j].z, u4[j].w};
            float4 *pr = prm + ((long long)h * K + k) * (D / 2) + 2 * g;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const float v0 = softplus(rv[2 * q]), v1 = softplus(rv[2 * q + 1]);
                const float s0 = 1.0f / sqrtf(v0), s1 = 1.0f / sqrtf(v1);
                pr[q] = make_float4(s0, s1, -uv[2 * q] * s0, -uv[2 * q + 1] * s1);
                lsum += logf(v0) + logf(v1);
            }
        }
    }
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);   // the component's 16 threads
    __syncthreads();   // bcast[1]
    if (part == 0 && k < K) cst[(long long)h * K + k] = (l[k] - bcast[1]) - 0.5f * lsum;
}

// Responsibilities of a range of rows of one (b, h) slice.
//   Lanes: HALVES lanes share a routing row, each holding DH = D / HALVES of
//   its features (interleaved in pairs, so that the lanes of a row read
//   neighbouring 16-byte parameter words: no bank conflicts); a thread holds
//   RPT = 2 rows.  The partial quadratic forms of a row are combined with
//   shuffles.  Each warp owns a set of components of the current parameter
//   tile (parameters broadcast from shared memory); the log-joint l_ik goes to
//   a shared [ROWS][K|1] tile and a warp per row then normalises it.
template <int D>
struct RespCfg {
    static constexpr int HALVES = D >= 64 ? D / 32 : 1;        // lanes per row
    static constexpr int DH = D / HALVES;                      // features per lane
    static constexpr int RPT = 2;                              // rows per thread
    static constexpr int WROWS = 32 / HALVES * RPT;            // rows per warp
    static constexpr int ROWS = 64;                            // rows per tile
    static constexpr int GROUPS = ROWS / WROWS;                // warp groups per tile
    static constexpr int WPG = (kThreads / 32) / GROUPS;       // warps per group
    static constexpr int KT = D == 128 ? 64 : 128;             // components per parameter tile
    static constexpr int ROWS_PER_CTA = 256;
    static size_t smem(int K) { return (size_t)KT * (D / 2) * 16 + KT * 4 + (size_t)ROWS * (K | 1) * 4; }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    k_resp(int N, int K, int H, const void *__restrict__ x, bool x_bf16, const float4 *__restrict__ prm,
           const float *__restrict__ cst, void *__restrict__ gamma, int ldg, int layout)
{
    using Cfg = RespCfg<D>;
    constexpr int DP = D / 2, HALVES = Cfg::HALVES, DH = Cfg::DH, RPT = Cfg::RPT, ROWS = Cfg::ROWS,
                  KT = Cfg::KT, WPG = Cfg::WPG;
    extern __shared__ __align__(16) unsigned char smem[];
    float4 *prm_s = reinterpret_cast<float4 *>(smem);
    float *cst_s = reinterpret_cast<float *>(prm_s + KT * DP);
    float *ell = cst_s + KT;
    const int LDE = K | 1;

    const long long bh = blockIdx.y;
    const int h = (int)(bh % H);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int half = lane % HALVES, slot = lane / HALVES;
    const int group = warp / WPG, wig = warp % WPG;
    const int row_begin = blockIdx.x * Cfg::ROWS_PER_CTA;
    const int row_end = min(N, row_begin + Cfg::ROWS_PER_CTA);
    const int ntiles = (K + KT - 1) / KT;
    const float4 *prm_h = prm + (long long)h * K * DP;
    const float *cst_h = cst + (long long)h * K;

    auto load_tile = [&](int t) {
        const int k0 = t * KT, kn = min(KT, K - k0);
        for (int i = tid; i < kn * DP; i += kThreads) prm_s[i] = prm_h[(long long)k0 * DP + i];
        for (int i = tid; i < kn; i += kThreads) cst_s[i] = cst_h[k0 + i];
    };
    if (ntiles == 1) load_tile(0);

    for (int r0 = row_begin; r0 < row_end; r0 += ROWS) {
        // this thread's rows (tile-local) and its feature pairs 2 * (dp * HALVES + half) + {0, 1}
        int lrow[RPT];
        float2 xr[RPT][DH / 2];
#pragma unroll
        for (int j = 0; j < RPT; ++j) {
            lrow[j] = group * Cfg::WROWS + slot + j * (32 / HALVES);
            const int row = r0 + lrow[j];
            const long long off = (bh * N + row) * D;
#pragma unroll
            for (int dp = 0; dp < DH / 2; ++dp) {
                const int f = 2 * (dp * HALVES + half);
                if (row < row_end) {
                    if (x_bf16) {
                        const uint32_t u =
                            *reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(x) + off + f);
                        xr[j][dp] = make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
                    } else {
                        xr[j][dp] = *reinterpret_cast<const float2 *>(static_cast<const float *>(x) + off + f);
                    }
                } else {
                    xr[j][dp] = make_float2(0.f, 0.f);
                }
            }
        }
        for (int t = 0; t < ntiles; ++t) {
            if (ntiles > 1) {
                __syncthreads();
                load_tile(t);
            }
            __syncthreads();
            const int k0 = t * KT, kn = min(KT, K - k0);
            // two components per pass: four independent accumulation chains per row pair
            for (int kk = wig; kk < kn; kk += 2 * WPG) {
                const bool two = kk + WPG < kn;
                const float4 *pa = prm_s + kk * DP + half;
                const float4 *pb = prm_s + (two ? kk + WPG : kk) * DP + half;
                float2 acc[2][RPT][2];
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int j = 0; j < RPT; ++j) acc[c][j][0] = acc[c][j][1] = make_float2(0.f, 0.f);
#pragma unroll
                for (int dp = 0; dp < DH / 2; ++dp) {
                    const float4 p = pa[dp * HALVES], q = pb[dp * HALVES];
                    const float2 sa = make_float2(p.x, p.y), na = make_float2(p.z, p.w);
                    const float2 sb = make_float2(q.x, q.y), nb = make_float2(q.z, q.w);
#pragma unroll
                    for (int j = 0; j < RPT; ++j) {
                        const float2 ya = __ffma2_rn(xr[j][dp], sa, na); // (x - mu) / sigma
                        acc[0][j][dp & 1] = __ffma2_rn(ya, ya, acc[0][j][dp & 1]);
                        const float2 yb = __ffma2_rn(xr[j][dp], sb, nb);
                        acc[1][j][dp & 1] = __ffma2_rn(yb, yb, acc[1][j][dp & 1]);
                    }
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int kc = kk + c * WPG;
                    const float cc = cst_s[two ? kc : kk];
#pragma unroll
                    for (int j = 0; j < RPT; ++j) {
                        float q = (acc[c][j][0].x + acc[c][j][0].y) + (acc[c][j][1].x + acc[c][j][1].y);
#pragma unroll
                        for (int o = 1; o < HALVES; o <<= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
                        if (half == 0 && (c == 0 || two)) ell[lrow[j] * LDE + k0 + kc] = fmaf(-0.5f, q, cc);
                    }
                }
            }
        }
        __syncthreads();
        for (int r = warp; r < ROWS; r += kThreads / 32) {
            const int row = r0 + r;
            if (row >= row_end) break;
            float *er = ell + r * LDE;
            float m = -FLT_MAX;
            for (int k = lane; k < K; k += 32) m = fmaxf(m, er[k]);
            m = warp_max(m);
            float s = 0.f;
            for (int k = lane; k < K; k += 32) {
                const float e = expf(er[k] - m);
                er[k] = e;
                s += e;
            }
            const float inv = 1.0f / warp_sum(s);
            const long long go = (bh * N + row) * (long long)ldg, plane = (long long)gridDim.y * N * ldg;
            for (int k = lane; k < ldg; k += 32) store_g(gamma, go + k, plane, k < K ? er[k] * inv : 0.f, layout);
        }
        __syncthreads();
    }
}

template <int D>
cudaError_t launch_resp_d(const Dims &dm, const float4 *prm, const float *cst, const void *x, void *gamma,
                          int ldg, int layout, cudaStream_t st)
{
    using Cfg = RespCfg<D>;
    const size_t smem = Cfg::smem(dm.K);
    static std::atomic<unsigned long long> smem_set{0};
    const cudaError_t attr = allow_smem(k_resp<D>, Cfg::smem(512), smem_set);
    if (attr != cudaSuccess) return attr;
    dim3 grid((dm.N + Cfg::ROWS_PER_CTA - 1) / Cfg::ROWS_PER_CTA, (unsigned)dm.BH());
    k_resp<D><<<grid, kThreads, smem, st>>>(dm.N, dm.K, dm.H, x, dm.x_bf16, prm, cst, gamma, ldg, layout);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_prep(const Dims &dm, const gma_params &p, float4 *prm, float *cst, cudaStream_t st)
{
    dim3 grid(dm.H, (dm.K + kPrepComps - 1) / kPrepComps);
    k_prep<<<grid, kPrepThreads, 0, st>>>(dm.K, dm.D, p.mu, p.var_raw, p.logit_pi, prm, cst);
    return cudaGetLastError();
}

cudaError_t launch_resp(const Dims &dm, const float4 *prm, const float *cst, const PrunedImages *img,
                        const void *x, void *gamma, int ldg, int layout, cudaStream_t st, int src)
{
    if (img && resp_pruned_applies(dm)) return launch_resp_pruned(dm, *img, x, gamma, ldg, layout, st, src);
    switch (dm.D) {
    case 16: return launch_resp_d<16>(dm, prm, cst, x, gamma, ldg, layout, st);
    case 32: return launch_resp_d<32>(dm, prm, cst, x, gamma, ldg, layout, st);
    case 64: return launch_resp_d<64>(dm, prm, cst, x, gamma, ldg, layout, st);
    case 128: return launch_resp_d<128>(dm, prm, cst, x, gamma, ldg, layout, st);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace gma
