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

// Responsibilities of any K <= 512 and d_route in {16, 32, 64, 128}.
//   One persistent CTA of kGThreads per SM walks a contiguous range of the
//   (slice, tile) items; a tile is R rows by all K components.  LPR lanes
//   share a group of eight rows: lane q holds feature pairs q + LPR j (j <
//   PPL) of those eight rows in registers, so one parameter word read from
//   shared memory feeds sixteen packed FMAs.  Warps split WR x CS: WR warps
//   cover the tile's rows, CS slices of the components.  A pass takes two
//   components; the eight rows' partial quadratic forms of the LPR lanes are
//   combined by recursive halving, after which each lane holds NV = 16 / LPR
//   log-joints of one component.  The parameters of a chunk of KC components
//   are staged in shared memory (all K when they fit, then they stay for every
//   tile of the head); the log-joints of the tile go to a shared [R][LDE]
//   array (LDE = K rounded up to 32, plus the softmax's threads per row, so
//   that its reads hit distinct banks), whose rows are normalised and stored.
constexpr int kGThreads = 512, kGWarps = kGThreads / 32;
constexpr size_t kGSmemMax = 232448 - 1024;   // opt-in limit of a CTA, less the reserved kilobyte

template <int D>
struct GenCfg {
    static constexpr int DP = D / 2;                  // feature pairs
    static constexpr int LPR = D <= 32 ? 4 : D / 8;   // lanes per row group
    static constexpr int PPL = DP / LPR;              // feature pairs per lane
    static constexpr int RPW = 32 / LPR * 8;          // rows per warp
    static constexpr int NV = 16 / LPR;               // log-joints per lane per pass
    static_assert(DP % LPR == 0 && PPL <= 4, "feature split");
};

struct GenPlan {
    int R, LDE, KC;
    size_t smem;
};

// Rows per tile, log-joint pitch, components per parameter chunk and shared memory.
GenPlan gen_plan(int K, int D)
{
    GenPlan g;
    g.R = K <= 256 ? 128 : 64;
    g.LDE = (int)round_up(K, 32) + kGThreads / g.R;
    const size_t fixed = (size_t)g.R * g.LDE * 4 + (size_t)round_up(K, 4) * 4 + (size_t)g.R * 4;
    const size_t per = (size_t)D * 8;   // one component's packed parameters
    long long kc = (long long)((kGSmemMax - fixed) / per) / 16 * 16;
    if (kc >= K) kc = K;
    g.KC = (int)kc;
    g.smem = fixed + per * (size_t)kc;
    return g;
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kGThreads, 1)
    k_resp(int N, int K, int H, long long items, int tiles, int R, int LDE, int KC, const void *__restrict__ x,
           bool x_bf16, const float4 *__restrict__ prm, const float *__restrict__ cst, void *__restrict__ gamma,
           int ldg, long long plane, int layout, bool vec)
{
    using Cfg = GenCfg<D>;
    constexpr int DP = Cfg::DP, LPR = Cfg::LPR, PPL = Cfg::PPL, RPW = Cfg::RPW, NV = Cfg::NV;
    extern __shared__ __align__(16) unsigned char smem[];
    float4 *prm_s = reinterpret_cast<float4 *>(smem);
    float *ell = reinterpret_cast<float *>(prm_s + (size_t)KC * DP);
    float *cst_s = ell + (size_t)R * LDE;
    float *rinv = cst_s + round_up(K, 4);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int WR = R / RPW, CS = kGWarps / WR;
    const int wr = warp % WR, cs = warp / WR;
    const int q = lane % LPR, trow = wr * RPW + (lane / LPR) * 8;   // this thread's rows trow .. trow + 7
    // the rows whose log-joints a lane holds after the halving: rbase .. rbase + NV - 1
    int rbase = 4 * ((q >> 1) & 1);
    if (LPR >= 8) rbase += 2 * ((q >> 2) & 1);
    if (LPR >= 16) rbase += (q >> 3) & 1;
    const int nch = (K + KC - 1) / KC;
    const long long per = (items + gridDim.x - 1) / gridDim.x;
    const long long i0 = blockIdx.x * per, i1 = min(items, i0 + per);
    int cur_h = -1, cur_c = -1;
    for (long long it = i0; it < i1; ++it) {
        const long long bh = it / tiles;
        const int h = (int)(bh % H), row0 = (int)(it % tiles) * R;
        float2 xr[8][PPL];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int row = row0 + trow + r;
            const long long off = (bh * N + row) * D + 2 * q;
#pragma unroll
            for (int j = 0; j < PPL; ++j) {
                if (row < N) {
                    if (x_bf16) {
                        const uint32_t u =
                            __ldcg(reinterpret_cast<const unsigned int *>(static_cast<const uint16_t *>(x) + off + 2 * LPR * j));
                        xr[r][j] = make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
                    } else {
                        xr[r][j] = __ldcg(reinterpret_cast<const float2 *>(static_cast<const float *>(x) + off + 2 * LPR * j));
                    }
                } else {
                    xr[r][j] = make_float2(0.f, 0.f);
                }
            }
        }
        for (int c = 0; c < nch; ++c) {
            const int k_lo = c * KC, kn = min(KC, K - k_lo);
            if (h != cur_h || c != cur_c) {
                __syncthreads();   // every warp is done with the previous parameters (and the tile's c_k)
                const float4 *src = prm + ((long long)h * K + k_lo) * DP;
                for (int i = tid; i < kn * DP; i += kGThreads) cp_async16(prm_s + i, src + i);
                asm volatile("cp.async.commit_group;" ::: "memory");
                if (h != cur_h)
                    for (int k = tid; k < K; k += kGThreads) cst_s[k] = cst[(long long)h * K + k];
                asm volatile("cp.async.wait_group 0;" ::: "memory");
                __syncthreads();
                cur_h = h;
                cur_c = c;
            }
            // this warp's slice of the chunk, in pairs of components
            const int KS = ((kn + CS - 1) / CS + 1) & ~1;
            const int kb0 = cs * KS, kb1 = min(kn, kb0 + KS);
#pragma unroll 1
            for (int kb = kb0; kb < kb1; kb += 2) {
                const bool two = kb + 1 < kb1;
                const float4 *pa = prm_s + kb * DP + q, *pb = prm_s + (two ? kb + 1 : kb) * DP + q;
                float2 acc[2][8];
#pragma unroll
                for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                    for (int r = 0; r < 8; ++r) acc[cc][r] = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < PPL; ++j) {
                    const float4 a = pa[LPR * j], b = pb[LPR * j];
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const float2 ya = __ffma2_rn(xr[r][j], make_float2(a.x, a.y), make_float2(a.z, a.w));
                        acc[0][r] = __ffma2_rn(ya, ya, acc[0][r]);   // ((x - mu) / sigma)^2, two features
                        const float2 yb = __ffma2_rn(xr[r][j], make_float2(b.x, b.y), make_float2(b.z, b.w));
                        acc[1][r] = __ffma2_rn(yb, yb, acc[1][r]);
                    }
                }
                // v[8 c + r]: partial sum of component kb + c, row trow + r; the halving over the
                // row group's lanes: xor 1 keeps one component, xor 2, 4, 8 halve the rows
                float v[16];
#pragma unroll
                for (int cc = 0; cc < 2; ++cc)
#pragma unroll
                    for (int r = 0; r < 8; ++r) v[8 * cc + r] = acc[cc][r].x + acc[cc][r].y;
#pragma unroll
                for (int o = 1, n = 8; o < LPR; o <<= 1, n >>= 1) {
                    const bool up = (q & o) != 0;
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (e < n) {
                            const float send = up ? v[e] : v[e + n], keep = up ? v[e + n] : v[e];
                            v[e] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                        }
                }
                const int k = kb + (q & 1);
                if ((q & 1) == 0 || two) {
                    const float ck = cst_s[k_lo + k];
#pragma unroll
                    for (int i = 0; i < NV; ++i) ell[(trow + rbase + i) * LDE + k_lo + k] = fmaf(-0.5f, v[i], ck);
                }
            }
        }
        __syncthreads();
        // softmax over the components: TR threads per row, components strided by TR
        {
            const int TR = kGThreads / R, r = tid / TR, j0 = tid % TR;
            float *er = ell + r * LDE;
            float m = -FLT_MAX;
            for (int k = j0; k < K; k += TR) m = fmaxf(m, er[k]);
            for (int o = 1; o < TR; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float sum = 0.f;
            for (int k = j0; k < K; k += TR) {
                const float e = expf(er[k] - m);
                er[k] = e;
                sum += e;
            }
            for (int o = 1; o < TR; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (j0 == 0) rinv[r] = 1.0f / sum;
        }
        __syncthreads();
        // rows out, a warp per row; columns K .. ldg - 1 are zero
        for (int r = warp; r < R; r += kGWarps) {
            const int row = row0 + r;
            if (row >= N) break;
            const float inv = rinv[r];
            const float *er = ell + r * LDE;
            const long long go = (bh * N + row) * (long long)ldg;
            if (vec) {   // ldg % 4 == 0, rows 16-byte (fp32) or 8-byte (16-bit) aligned
                for (int k = 4 * lane; k < ldg; k += 128) {
                    float w[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) w[u] = k + u < K ? er[k + u] * inv : 0.f;
                    if (layout == GL_F32) {
                        *reinterpret_cast<float4 *>(static_cast<float *>(gamma) + go + k) = make_float4(w[0], w[1], w[2], w[3]);
                    } else {
                        uint32_t hw[2], lw[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            __nv_bfloat16 h0, l0, h1, l1;
                            split_bf16(w[2 * u], h0, l0);
                            split_bf16(w[2 * u + 1], h1, l1);
                            hw[u] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                            lw[u] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
                        }
                        __nv_bfloat16 *g = static_cast<__nv_bfloat16 *>(gamma);
                        *reinterpret_cast<uint2 *>(g + go + k) = make_uint2(hw[0], hw[1]);
                        if (layout == GL_SPLIT) *reinterpret_cast<uint2 *>(g + plane + go + k) = make_uint2(lw[0], lw[1]);
                    }
                }
            } else {
                for (int k = lane; k < ldg; k += 32) store_g(gamma, go + k, plane, k < K ? er[k] * inv : 0.f, layout);
            }
        }
        __syncthreads();   // the log-joint array is reused by the next tile
    }
}

template <int D>
cudaError_t launch_resp_d(const Dims &dm, const float4 *prm, const float *cst, const void *x, void *gamma,
                          int ldg, int layout, cudaStream_t st)
{
    if (dm.K < 1 || dm.K > 512 || ldg < dm.K) return cudaErrorInvalidValue;
    const GenPlan g = gen_plan(dm.K, D);
    static std::atomic<unsigned long long> smem_set{0};
    const cudaError_t attr = allow_smem(k_resp<D>, kGSmemMax, smem_set);
    if (attr != cudaSuccess) return attr;
    const int tiles = (dm.N + g.R - 1) / g.R;
    const long long items = dm.BH() * tiles;
    if (items == 0) return cudaSuccess;
    const long long plane = dm.BH() * dm.N * (long long)ldg;
    const size_t align = layout == GL_F32 ? 16 : 8;
    const bool vec = ldg % 4 == 0 && reinterpret_cast<uintptr_t>(gamma) % align == 0 &&
                     (layout != GL_SPLIT || (plane * 2) % (long long)align == 0);
    const int grid = (int)(items < sm_count() ? items : sm_count());
    k_resp<D><<<grid, kGThreads, g.smem, st>>>(dm.N, dm.K, dm.H, items, tiles, g.R, g.LDE, g.KC, x, dm.x_bf16, prm,
                                               cst, gamma, ldg, plane, layout, vec);
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
    if (img && img->w3 && resp_gtc_applies(dm) && resp_gtc_output_ok(dm, ldg, layout))
        return launch_resp_gtc(dm, img->w3, prm, cst, x, gamma, ldg, layout, st);
    switch (dm.D) {
    case 16: return launch_resp_d<16>(dm, prm, cst, x, gamma, ldg, layout, st);
    case 32: return launch_resp_d<32>(dm, prm, cst, x, gamma, ldg, layout, st);
    case 64: return launch_resp_d<64>(dm, prm, cst, x, gamma, ldg, layout, st);
    case 128: return launch_resp_d<128>(dm, prm, cst, x, gamma, ldg, layout, st);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace gma
