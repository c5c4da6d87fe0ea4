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
// One CTA = 8 warps, tiles of 128 rows; warps w and w + 4 share TMEM lanes
// 32 (w % 4) .. +31 (one row each) and split the components in halves.
#include "gma_internal.cuh"
#include "gma_tc.cuh"

#include <float.h>

namespace gma {
namespace {

using namespace tc;

constexpr int kPK = 128, kPD = 64, kPDP = kPD / 2;
constexpr int kPThreads = 256, kPRows = 128, kPRowsPerCta = 512;
constexpr int kPStride = kPDP + 1;            // padded float4 row of exact parameters
constexpr float kPT = 30.f;                   // log-joint window kept exactly
constexpr float kPU = 4.0e-3f;                // bf16 product + fp32 accumulation bound

struct PrunedSmem {
    static constexpr uint32_t W = kPK * 2 * kPD * 2;                    // bf16 [128][128], SW128
    static constexpr uint32_t P = kPK * kPStride * 16;                  // float4 [128][33]
    static constexpr size_t bytes = 1024 + W + P + 10 * kPK * 4 + 64;
};

__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}

__global__ void __launch_bounds__(kPThreads, 2)
    k_resp_pruned(int N, int H, const void *__restrict__ x, bool x_bf16, const float4 *__restrict__ prm,
                  const float *__restrict__ cst, void *__restrict__ gamma, int ldg, bool g_bf16)
{
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *w_s = sm;                                          // B operand W
    float4 *p_s = reinterpret_cast<float4 *>(sm + PrunedSmem::W);    // exact parameters
    float *f_s = reinterpret_cast<float *>(sm + PrunedSmem::W + PrunedSmem::P);
    float *c_s = f_s;              // c_k
    float *cp_s = f_s + kPK;       // c'_k = c_k - 1/2 sum_d a mu^2
    float *a_s = f_s + 2 * kPK;    // A_k
    float *m_s = f_s + 3 * kPK;    // M_k
    float *x0 = f_s + 4 * kPK;     // [2][128] exchange between the two halves of a row
    float *x1 = f_s + 6 * kPK;     // [2][128]
    float *x2 = f_s + 8 * kPK;     // [2][128]
    uint64_t *bar = reinterpret_cast<uint64_t *>(f_s + 10 * kPK);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = warp >> 2;                      // component half
    const uint32_t lane0 = 32 * (warp & 3);
    const int i = lane0 + lane;                   // row of the tile (TMEM lane)
    const long long bh = blockIdx.y;
    const int head = (int)(bh % H);
    const int row_begin = blockIdx.x * kPRowsPerCta;
    const int row_end = min(N, row_begin + kPRowsPerCta);
    constexpr uint32_t A_COL = 0, D_COL = 128;

    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(smem_addr(bar), 1);
        mbar_init_fence();
    }
    // exact parameters of this head, and W / per-component constants built from them
    const float4 *prm_h = prm + (long long)head * kPK * kPDP;
    for (int e = tid; e < kPK * kPDP; e += kPThreads) p_s[(e / kPDP) * kPStride + e % kPDP] = prm_h[e];
    {
        const int k = tid % kPK, part = tid / kPK;   // two threads per component, 16 feature pairs each
        float amu2 = 0.f, amax = 0.f, mmax = 0.f;
        for (int dp = 16 * part; dp < 16 * part + 16; ++dp) {
            const float4 p = prm_h[k * kPDP + dp];
            const float s[2] = {p.x, p.y}, nm[2] = {p.z, p.w};   // 1/sigma, -mu/sigma
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int f = 2 * dp + e;
                const float a = s[e] * s[e], amu = -s[e] * nm[e];
                *reinterpret_cast<__nv_bfloat16 *>(w_s + sw128_offset(k, f, kPK, 2)) = __float2bfloat16_rn(-0.5f * a);
                *reinterpret_cast<__nv_bfloat16 *>(w_s + sw128_offset(k, kPD + f, kPK, 2)) = __float2bfloat16_rn(amu);
                amu2 = fmaf(nm[e], nm[e], amu2);
                amax = fmaxf(amax, a);
                mmax = fmaxf(mmax, fabsf(amu));
            }
        }
        x0[part * kPK + k] = amu2;
        x1[part * kPK + k] = amax;
        x2[part * kPK + k] = mmax;
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid < kPK) {
        const float c = cst[(long long)head * kPK + tid];
        c_s[tid] = c;
        cp_s[tid] = c - 0.5f * (x0[tid] + x0[kPK + tid]);
        a_s[tid] = fmaxf(x1[tid], x1[kPK + tid]);
        m_s[tid] = fmaxf(x2[tid], x2[kPK + tid]);
    }
    fence_proxy_async();   // W written by threads, read by the tensor core
    __syncthreads();
    const uint32_t tbase = *tslot;
    const uint32_t id = idesc(128, kPK, kFmtBF16);

    int tile = 0;
    for (int r0 = row_begin; r0 < row_end; r0 += kPRows, ++tile) {
        const int row = r0 + i;
        const bool valid = row < row_end;
        // the row (both halves hold all 64 features), its sums for the bound
        float2 xr[kPDP];
        {
            const long long off = (bh * N + row) * (long long)kPD;
#pragma unroll
            for (int q = 0; q < kPD / 4; ++q) {
                const float4 t = valid ? load4(x, off + 4 * q, x_bf16) : make_float4(0.f, 0.f, 0.f, 0.f);
                xr[2 * q] = make_float2(t.x, t.y);
                xr[2 * q + 1] = make_float2(t.z, t.w);
            }
        }
        float s2 = 0.f, s1 = 0.f;
#pragma unroll
        for (int q = 0; q < kPDP; ++q) {
            s2 = fmaf(xr[q].x, xr[q].x, fmaf(xr[q].y, xr[q].y, s2));
            s1 += fabsf(xr[q].x) + fabsf(xr[q].y);
        }
        // A = [x^2 | x] in bf16 (features 0..63 squared, 64..127 plain); half h writes its part
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            uint32_t p[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float2 v = xr[16 * b + j];
                p[j] = h == 0 ? pack2(v.x * v.x, v.y * v.y) : pack2(v.x, v.y);
            }
            tmem_st16(tmem_at(tbase, lane0, A_COL + 32 * h + 16 * b), p);
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
            mma_commit(smem_addr(bar));
        }
        __syncwarp();
        const bool ok = mbar_wait(smem_addr(bar), (uint32_t)(tile & 1));
        fence_after_sync();

        // bound pass 1: the best lower bound of this half; then of the row
        float lo_max = -FLT_MAX;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            uint32_t r[16];
            tmem_ld16(tmem_at(tbase, lane0, D_COL + 64 * h + 16 * b), r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int k = 64 * h + 16 * b + j;
                const float lt = __uint_as_float(r[j]) + cp_s[k];
                const float dk = fmaf(kPU, fmaf(0.5f * a_s[k], s2, m_s[k] * s1), 1e-3f);
                lo_max = fmaxf(lo_max, lt - dk);
            }
        }
        x0[h * kPK + i] = lo_max;
        __syncthreads();
        const float keep_from = fmaxf(x0[i], x0[kPK + i]) - kPT;
        // bound pass 2: candidate mask of this half (all components if the MMA wait failed)
        uint64_t mask = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            uint32_t r[16];
            tmem_ld16(tmem_at(tbase, lane0, D_COL + 64 * h + 16 * b), r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int k = 64 * h + 16 * b + j;
                const float lt = __uint_as_float(r[j]) + cp_s[k];
                const float dk = fmaf(kPU, fmaf(0.5f * a_s[k], s2, m_s[k] * s1), 1e-3f);
                if (!ok || lt + dk >= keep_from) mask |= 1ull << (16 * b + j);
            }
        }
        // exact log-joint of a kept component
        auto exact = [&](int k) {
            const float4 *pk = p_s + k * kPStride;
            float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int dp = 0; dp < kPDP; dp += 2) {
                const float4 p = pk[dp], q = pk[dp + 1];
                const float2 y0 = __ffma2_rn(xr[dp], make_float2(p.x, p.y), make_float2(p.z, p.w));
                acc0 = __ffma2_rn(y0, y0, acc0);
                const float2 y1 = __ffma2_rn(xr[dp + 1], make_float2(q.x, q.y), make_float2(q.z, q.w));
                acc1 = __ffma2_rn(y1, y1, acc1);
            }
            return fmaf(-0.5f, (acc0.x + acc0.y) + (acc1.x + acc1.y), c_s[k]);
        };
        // exact pass 1: online maximum and sum over the kept components of this half
        float mt = -FLT_MAX, st = 0.f;
        for (uint64_t mm = mask; mm; mm &= mm - 1) {
            const float l = exact(64 * h + __ffsll((long long)mm) - 1);
            if (l > mt) {
                st = st * expf(mt - l) + 1.f;
                mt = l;
            } else {
                st += expf(l - mt);
            }
        }
        x1[h * kPK + i] = mt;
        x2[h * kPK + i] = st;
        __syncthreads();
        const float ma = x1[i], mb = x1[kPK + i];
        const float m = fmaxf(ma, mb);
        const float inv = 1.0f / (x2[i] * expf(ma - m) + x2[kPK + i] * expf(mb - m));
        // exact pass 2: zero this half of the output row, then write the kept posteriors
        if (valid) {
            const long long go = (bh * N + row) * (long long)ldg + 64 * h;
            if (g_bf16) {
                uint4 *z = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(gamma) + go);
#pragma unroll
                for (int q = 0; q < 8; ++q) z[q] = make_uint4(0, 0, 0, 0);
            } else {
                float4 *z = reinterpret_cast<float4 *>(static_cast<float *>(gamma) + go);
#pragma unroll
                for (int q = 0; q < 16; ++q) z[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            for (uint64_t mm = mask; mm; mm &= mm - 1) {
                const int b = __ffsll((long long)mm) - 1;
                store_elem(gamma, go + b, expf(exact(64 * h + b) - m) * inv, g_bf16);
            }
        }
        fence_before_sync();
        __syncthreads();   // exchange slots and the accumulator are reused by the next tile
        fence_after_sync();
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

} // namespace

bool resp_pruned_applies(const Dims &dm) { return dm.K == kPK && dm.D == kPD; }

cudaError_t launch_resp_pruned(const Dims &dm, const float4 *prm, const float *cst, const void *x, void *gamma,
                               int ldg, bool gamma_bf16, cudaStream_t st)
{
    constexpr size_t smem = PrunedSmem::bytes;
    static cudaError_t attr = allow_smem(k_resp_pruned, smem);
    if (attr != cudaSuccess) return attr;
    dim3 grid((dm.N + kPRowsPerCta - 1) / kPRowsPerCta, (unsigned)dm.BH());
    k_resp_pruned<<<grid, kPThreads, smem, st>>>(dm.N, dm.H, x, dm.x_bf16, prm, cst, gamma, ldg, gamma_bf16);
    return cudaGetLastError();
}

} // namespace gma
