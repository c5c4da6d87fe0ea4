// Responsibilities (S1) for K = 128 components and d_route = 64, with a
// tensor-core bound that decides which components need the exact logit.
//
// The posterior of the GMA explainer ("핵심 메커니즘": gamma_ik = p(z = k | x_i)
// under the diagonal GMM) is a softmax over the log-joints
//   l_ik = c_k - 1/2 sum_d ((x_id - mu_kd) / sigma_kd)^2 .
// Components whose log-joint lies more than T = 30 below the row's best get a
// posterior below e^-30 ~ 1e-13, far below fp32 resolution of the sum; their
// gamma is written as 0 and the softmax is taken over the others.  Finding
// them is cheap on the tensor cores: expanding the square,
//   l_ik = c'_k + sum_d ( -1/2 a_kd x_id^2 + a_kd mu_kd x_id ),   a = 1/sigma^2,
// is one bf16 GEMM [x^2 | x] (128 x 128) times W (128 x 128 components) per
// tile of 128 rows.  That form cancels badly, so it is used only as a bound:
// with bf16 operands (unit roundoff 2^-9) and fp32 accumulation,
//   |l~_ik - l_ik| <= delta_ik = U (1/2 A_k sum_d x_d^2 + M_k sum_d |x_d|) + 1e-3,
// U = 4e-3, A_k = max_d a_kd, M_k = max_d |a_kd mu_kd|.  Component k is kept
// when l~_ik + delta_ik >= max_j (l~_ij - delta_ij) - T, which keeps every
// component within T of the true maximum.  The kept components get the same
// exact fp32 evaluation as the dense kernel (one packed FMA for (x - mu)/sigma,
// one for the square-accumulate, per feature pair).
//
// One CTA = 16 warps over tiles of 128 rows: the four warps 4q + w' share the
// TMEM lanes 32 w' .. +31 (one row each) and take component quarter q.  The
// per-head bound matrix, padded parameters and constants are built once per
// call by k_prep_pruned and bulk-copied into shared memory; routing rows
// arrive by double-buffered TMA.
#include "gma_internal.cuh"
#include "gma_tc.cuh"

#include <float.h>

namespace gma {
namespace {

using namespace tc;

constexpr int kPK = 128, kPD = 64, kPDP = kPD / 2;
constexpr int kPThreads = 512, kPRows = 128, kPRowsPerCta = 1024;
constexpr int kPStride = kPDP + 1;            // padded float4 row of exact parameters
constexpr float kPT = 30.f;                   // log-joint window kept exactly
constexpr float kPU = 4.0e-3f;                // bf16 product + fp32 accumulation bound

struct PrunedSmem {
    static constexpr uint32_t W = kPrunedWBytes;                        // bf16 [128][128], SW128
    static constexpr uint32_t X = kPRows * kPD * 4;                     // one routing tile (fp32 worst case)
    static constexpr uint32_t P = kPrunedPBytes;                        // float4 [128][33]
    static constexpr uint32_t F = (4 + 12) * kPK * 4;                   // constants + exchange slots
    static constexpr size_t bytes = 1024 + W + 2 * X + P + F + 64;
};

__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}

// One CTA per head: the bound matrix W (bf16, in the swizzled B-operand
// layout), the exact parameters with padded rows, and c, c', A, M.
__global__ void __launch_bounds__(256) k_prep_pruned(const float4 *__restrict__ prm, const float *__restrict__ cst,
                                                     unsigned char *__restrict__ wimg, float4 *__restrict__ pimg,
                                                     float *__restrict__ cimg)
{
    const int h = blockIdx.x, tid = threadIdx.x;
    const float4 *ph = prm + (long long)h * kPK * kPDP;
    unsigned char *wh = wimg + (long long)h * kPrunedWBytes;
    float4 *pp = pimg + (long long)h * kPK * kPStride;
    for (int e = tid; e < kPK * kPStride; e += 256) {
        const int k = e / kPStride, dp = e % kPStride;
        pp[e] = dp < kPDP ? ph[k * kPDP + dp] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int e = tid; e < kPK * kPDP; e += 256) {
        const int k = e / kPDP, dp = e % kPDP;
        const float4 p = ph[e];
        const float s[2] = {p.x, p.y}, nm[2] = {p.z, p.w};   // 1/sigma, -mu/sigma
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int f = 2 * dp + j;
            *reinterpret_cast<__nv_bfloat16 *>(wh + sw128_offset(k, f, kPK, 2)) =
                __float2bfloat16_rn(-0.5f * s[j] * s[j]);
            *reinterpret_cast<__nv_bfloat16 *>(wh + sw128_offset(k, kPD + f, kPK, 2)) =
                __float2bfloat16_rn(-s[j] * nm[j]);
        }
    }
    if (tid < kPK) {
        float amu2 = 0.f, amax = 0.f, mmax = 0.f;
        for (int dp = 0; dp < kPDP; ++dp) {
            const float4 p = ph[tid * kPDP + dp];
            amu2 = fmaf(p.z, p.z, fmaf(p.w, p.w, amu2));
            amax = fmaxf(amax, fmaxf(p.x * p.x, p.y * p.y));
            mmax = fmaxf(mmax, fmaxf(fabsf(p.x * p.z), fabsf(p.y * p.w)));
        }
        const float c = cst[(long long)h * kPK + tid];
        float *ch = cimg + (long long)h * 4 * kPK;
        ch[tid] = c;
        ch[kPK + tid] = c - 0.5f * amu2;
        ch[2 * kPK + tid] = amax;
        ch[3 * kPK + tid] = mmax;
    }
}

__global__ void __launch_bounds__(kPThreads, 1)
    k_resp_pruned(const __grid_constant__ CUtensorMap xmap, int N, int H, bool x_bf16,
                  const unsigned char *__restrict__ wimg, const float4 *__restrict__ pimg,
                  const float *__restrict__ cimg, void *__restrict__ gamma, int ldg, bool g_bf16)
{
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *w_s = sm;                                                  // B operand W
    unsigned char *xb = sm + PrunedSmem::W;                                   // [2] routing tiles
    float4 *p_s = reinterpret_cast<float4 *>(xb + 2 * PrunedSmem::X);        // exact parameters
    float *f_s = reinterpret_cast<float *>(reinterpret_cast<unsigned char *>(p_s) + PrunedSmem::P);
    const float *c_s = f_s, *cp_s = f_s + kPK, *a_s = f_s + 2 * kPK, *m_s = f_s + 3 * kPK;
    float *ex0 = f_s + 4 * kPK;    // [4][128] exchange slots between the quarters of a row
    float *ex1 = f_s + 8 * kPK;
    float *ex2 = f_s + 12 * kPK;
    uint64_t *bar = reinterpret_cast<uint64_t *>(f_s + 16 * kPK);   // setup, mma, x[2]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp >> 2;                      // component quarter
    const uint32_t lane0 = 32 * (warp & 3);
    const int i = lane0 + lane;                   // row of the tile (TMEM lane)
    const long long bh = blockIdx.y;
    const int head = (int)(bh % H);
    const int row_begin = blockIdx.x * kPRowsPerCta;
    const int row_end = min(N, row_begin + kPRowsPerCta);
    const int ntiles = (row_end - row_begin + kPRows - 1) / kPRows;
    const uint32_t xbytes = kPRows * kPD * (x_bf16 ? 2 : 4);
    constexpr uint32_t A_COL = 0, D_COL = 128;

    auto load_x = [&](int t) {   // one thread: TMA of tile t into buffer t & 1
        const uint32_t b = smem_addr(bar + 2 + (t & 1));
        unsigned char *dst = xb + (t & 1) * PrunedSmem::X;
        const int y = (int)(bh * N + row_begin + t * kPRows);
        mbar_expect_tx(b, xbytes);
        if (x_bf16) {
            tma_load_2d(smem_addr(dst), &xmap, 0, y, b);
        } else {
            tma_load_2d(smem_addr(dst), &xmap, 0, y, b);
            tma_load_2d(smem_addr(dst + kPRows * 128), &xmap, 32, y, b);
        }
    };
    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 4; ++b) mbar_init(smem_addr(bar + b), 1);
        mbar_init_fence();
        mbar_expect_tx(smem_addr(bar), kPrunedWBytes + kPrunedPBytes + kPrunedCBytes);
        bulk_g2s(smem_addr(w_s), wimg + (long long)head * kPrunedWBytes, kPrunedWBytes, smem_addr(bar));
        bulk_g2s(smem_addr(p_s), pimg + (long long)head * kPK * kPStride, kPrunedPBytes, smem_addr(bar));
        bulk_g2s(smem_addr(f_s), cimg + (long long)head * 4 * kPK, kPrunedCBytes, smem_addr(bar));
        if (ntiles > 0) load_x(0);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *tslot;
    const uint32_t id = idesc(128, kPK, kFmtBF16);
    bool ok = mbar_wait(smem_addr(bar), 0);

    for (int t = 0; t < ntiles; ++t) {
        if (tid == 0 && t + 1 < ntiles) {
            fence_proxy_async();
            load_x(t + 1);
        }
        const int row = row_begin + t * kPRows + i;
        const bool valid = row < row_end;
        ok = mbar_wait(smem_addr(bar + 2 + (t & 1)), (uint32_t)((t >> 1) & 1)) && ok;
        // the row (every quarter holds all 64 features) and its sums for the bound
        const unsigned char *xt = xb + (t & 1) * PrunedSmem::X;
        float2 xr[kPDP];
        if (x_bf16) {
#pragma unroll
            for (int g = 0; g < kPD / 8; ++g) {
                const uint4 u = *reinterpret_cast<const uint4 *>(xt + sw128_offset(i, 8 * g, kPRows, 2));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    xr[4 * g + e] = make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
            }
        } else {
#pragma unroll
            for (int g = 0; g < kPD / 4; ++g) {
                const float4 u = *reinterpret_cast<const float4 *>(xt + sw128_offset(i, 4 * g, kPRows, 4));
                xr[2 * g] = make_float2(u.x, u.y);
                xr[2 * g + 1] = make_float2(u.z, u.w);
            }
        }
        float s2 = 0.f, s1 = 0.f;
#pragma unroll
        for (int g = 0; g < kPDP; ++g) {
            s2 = fmaf(xr[g].x, xr[g].x, fmaf(xr[g].y, xr[g].y, s2));
            s1 += fabsf(xr[g].x) + fabsf(xr[g].y);
        }
        // A = [x^2 | x] in bf16: quarter q writes operand columns [16q, 16q + 16)
        {
            uint32_t p[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float2 v = (q & 1) ? xr[16 + j] : xr[j];   // static indices keep xr in registers
                p[j] = q < 2 ? pack2(v.x * v.x, v.y * v.y) : pack2(v.x, v.y);
            }
            tmem_st16(tmem_at(tbase, lane0, A_COL + 16 * q), p);
        }
        tmem_wait_st();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (tid == 0) {
#pragma unroll 1
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t kb = kk * 32;
                const uint32_t boff = (kb >> 7) * (kPK * 128) + (kb & 127);
                mma_ts(0u, tbase + D_COL, tbase + A_COL + kk * 8, sdesc_sw128(smem_addr(w_s + boff)), id,
                       kk > 0 ? 1u : 0u);
            }
            mma_commit(smem_addr(bar + 1));
        }
        __syncwarp();
        ok = mbar_wait(smem_addr(bar + 1), (uint32_t)(t & 1)) && ok;
        fence_after_sync();

        // bound: best lower bound of this quarter, then of the row; then the kept set
        auto bound = [&](int b, float (&lt)[16], float (&dk)[16]) {
            uint32_t r[16];
            tmem_ld16(tmem_at(tbase, lane0, D_COL + 32 * q + 16 * b), r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int k = 32 * q + 16 * b + j;
                lt[j] = __uint_as_float(r[j]) + cp_s[k];
                dk[j] = fmaf(kPU, fmaf(0.5f * a_s[k], s2, m_s[k] * s1), 1e-3f);
            }
        };
        float lo_max = -FLT_MAX;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            float lt[16], dk[16];
            bound(b, lt, dk);
#pragma unroll
            for (int j = 0; j < 16; ++j) lo_max = fmaxf(lo_max, lt[j] - dk[j]);
        }
        ex0[q * kPK + i] = lo_max;
        __syncthreads();
        const float keep_from =
            fmaxf(fmaxf(ex0[i], ex0[kPK + i]), fmaxf(ex0[2 * kPK + i], ex0[3 * kPK + i])) - kPT;
        uint32_t mask = 0;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            float lt[16], dk[16];
            bound(b, lt, dk);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (!ok || lt[j] + dk[j] >= keep_from) mask |= 1u << (16 * b + j);
        }

        // exact log-joint of a kept component
        auto exact = [&](int k) {
            const float4 *pk = p_s + k * kPStride;
            float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int dp = 0; dp < kPDP; dp += 2) {
                const float4 p = pk[dp], r = pk[dp + 1];
                const float2 y0 = __ffma2_rn(xr[dp], make_float2(p.x, p.y), make_float2(p.z, p.w));
                acc0 = __ffma2_rn(y0, y0, acc0);
                const float2 y1 = __ffma2_rn(xr[dp + 1], make_float2(r.x, r.y), make_float2(r.z, r.w));
                acc1 = __ffma2_rn(y1, y1, acc1);
            }
            return fmaf(-0.5f, (acc0.x + acc0.y) + (acc1.x + acc1.y), c_s[k]);
        };
        // exact pass 1: online maximum and sum over the kept components of this quarter
        float mt = -FLT_MAX, st = 0.f;
        for (uint32_t mm = mask; mm; mm &= mm - 1) {
            const float l = exact(32 * q + __ffs(mm) - 1);
            if (l > mt) {
                st = st * expf(mt - l) + 1.f;
                mt = l;
            } else {
                st += expf(l - mt);
            }
        }
        ex1[q * kPK + i] = mt;
        ex2[q * kPK + i] = st;
        __syncthreads();
        float m = ex1[i];
#pragma unroll
        for (int g = 1; g < 4; ++g) m = fmaxf(m, ex1[g * kPK + i]);
        float ssum = 0.f;
#pragma unroll
        for (int g = 0; g < 4; ++g) ssum += ex2[g * kPK + i] * expf(ex1[g * kPK + i] - m);
        const float inv = 1.0f / ssum;
        // exact pass 2: zero this quarter of the output row, then write the kept posteriors
        if (valid) {
            const long long go = (bh * N + row) * (long long)ldg + 32 * q;
            if (g_bf16) {
                uint4 *z = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(gamma) + go);
#pragma unroll
                for (int g = 0; g < 4; ++g) z[g] = make_uint4(0, 0, 0, 0);
            } else {
                float4 *z = reinterpret_cast<float4 *>(static_cast<float *>(gamma) + go);
#pragma unroll
                for (int g = 0; g < 8; ++g) z[g] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            for (uint32_t mm = mask; mm; mm &= mm - 1) {
                const int b = __ffs(mm) - 1;
                store_elem(gamma, go + b, expf(exact(32 * q + b) - m) * inv, g_bf16);
            }
        }
        fence_before_sync();
        __syncthreads();   // exchange slots, the accumulator and this x buffer are reused
        fence_after_sync();
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

} // namespace

bool resp_pruned_applies(const Dims &dm) { return dm.K == kPK && dm.D == kPD; }

cudaError_t launch_prep_pruned(const Dims &dm, const float4 *prm, const float *cst, const PrunedImages &img,
                               cudaStream_t st)
{
    k_prep_pruned<<<dm.H, 256, 0, st>>>(prm, cst, img.w, img.p, img.c);
    return cudaGetLastError();
}

cudaError_t launch_resp_pruned(const Dims &dm, const PrunedImages &img, const void *x, void *gamma, int ldg,
                               bool gamma_bf16, cudaStream_t st)
{
    constexpr size_t smem = PrunedSmem::bytes;
    static cudaError_t attr = allow_smem(k_resp_pruned, smem);
    if (attr != cudaSuccess) return attr;
    CUtensorMap xmap;
    if (!make_tma_2d(&xmap, x, dm.x_bf16, (unsigned long long)dm.BH() * dm.N, kPD, kPRows))
        return cudaErrorInvalidValue;
    dim3 grid((dm.N + kPRowsPerCta - 1) / kPRowsPerCta, (unsigned)dm.BH());
    k_resp_pruned<<<grid, kPThreads, smem, st>>>(xmap, dm.N, dm.H, dm.x_bf16, img.w, img.p, img.c, gamma, ldg,
                                                 gamma_bf16);
    return cudaGetLastError();
}

} // namespace gma
