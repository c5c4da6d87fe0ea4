// Gradients of the GMA forward (causal and bidirectional), CUDA-core path.
//
// The GMA explainer ("Gaussian Mixture Attention: Linear-Time Sequence Mixing
// via Probabilistic Latent Routing", "변형 및 학습") trains mu, sigma^2 and pi
// end to end by backpropagation through the softplus and softmax
// reparameterisations; its gradient analysis ("주요 기여", gradient structure)
// notes that every gradient passes through the responsibilities.  With
// U_i = Gamma_Q,i S_i = [numerator | denominator - eps] and g_i = dL/dO_i:
//   u_i      = dL/dU_i = [g_i / den_i | -(g_i . O_i) / den_i]
//   dGamma_Q,i = S_i u_i                    (S_i: the memory row i reads)
//   R_j      = sum over the rows i that read key j of Gamma_Q,i^T u_i
//   dGamma_K,j = R_j [v_j | 1],   dV_j = (Gamma_K,j R_j)[:, :d_v]
// (causal: S_i over j <= i, R_j over i >= j; bidirectional: the totals), then
// through the softmax over components delta = Gamma (dGamma - rowsum(Gamma dGamma)),
// and through the log-joint with y = (x - mu) / sigma, a = 1 / sigma^2:
//   dx_d = -sum_k delta_k a_kd (x_d - mu_kd) = -sum_k delta_k y_kd s_kd
//   dmu_kd += delta_k y_kd s_kd,   dsigma^2_kd += delta_k a_kd (y_kd^2 - 1) / 2,
//   dlog pi_k += delta_k,
// and the reparameterisation: dvar_raw = dsigma^2 sigmoid(var_raw),
// dlogit_k = G_k - pi_k sum_k' G_k'.
//
// Layout and order follow the forward's CUDA-core path: blocks of kBlockRows
// rows per (b, h) slice, chunks of C = 64 rows inside a block (dense
// intra-chunk products, carried memory), every reduction in a fixed order.
//   k_bwd_q      per block, chunks in order, carrying S: u and dGamma_Q
//   k_bwd_mem    per block: M = Gamma_Q^T u   (then k_scan_rev: the suffix R)
//   k_bwd_k      per block, chunks in reverse order, carrying R: dGamma_K, dV
//   k_bwd_delta  delta in place of dGamma (both routings)
//   k_bwd_dx     dx per routing row
//   k_bwd_param  per block of rows: the parameter partial sums
//   k_bwd_final  per head: the sums over slices and blocks, the reparameterisation
#include "gma_internal.cuh"

#include <float.h>

namespace gma {
namespace {

constexpr int kBC = 64;    // chunk rows
constexpr int kBKC = 32;   // components per tile (two CTAs of the chunk kernels fit on an SM)

template <int DV>
struct BwdCfg {
    static constexpr int UW = DV + 16;        // row pitch of u: d_v values, the denominator part, zeros
    static constexpr int LG = kBKC + 1, LP = kBC + 1;
};

// rows [0, nr) of a [rows][KP] fp32 responsibility array into a [kBC][LG] tile (components k0 ..)
__device__ __forceinline__ void stage_rows(float *dst, int LG, const float *src, long long row0, int nr, int KP,
                                           int k0)
{
    for (int i = threadIdx.x; i < kBC * kBKC / 4; i += kThreads) {
        const int r = i / (kBKC / 4), c = (i % (kBKC / 4)) * 4, k = k0 + c;
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < nr && k < KP) val = *reinterpret_cast<const float4 *>(src + (row0 + r) * KP + k);
        float *d = dst + r * LG + c;
        d[0] = val.x; d[1] = val.y; d[2] = val.z; d[3] = val.w;
    }
}

// ---------------------------------------------------------------------------
// Query side.  Per chunk: [numerator | den] as in the forward (P = Gq Gk^T
// masked, the carried memory S), then u, then
//   dGq = u[:, :dv] S[:, :dv]^T + u[:, dv] Z^T + (Q' masked) Gk,
//   Q'_ij = u_i . [v_j | 1]  (j <= i),
// then S advances by Gk^T [V | 1] (causal).  Bidirectional: S is the total, no P, no Q'.
template <int DV>
struct BwdQSmem {
    static constexpr int UW = BwdCfg<DV>::UW, LG = BwdCfg<DV>::LG, LP = BwdCfg<DV>::LP;
    static constexpr int VP = DV + 1;   // row pitch of the V rows and the memory rows (odd: no bank conflicts)
    static constexpr size_t floats = (size_t)kBC * LG * 2 + (size_t)kBC * VP + (size_t)kBC * DV + (size_t)kBC * LP +
                                     (size_t)kBKC * VP + kBKC + (size_t)kBC * UW + kBC + (size_t)kBC * 16 + kThreads;
    static constexpr size_t bytes = floats * 4;
};

template <int DV>
__global__ void __launch_bounds__(kThreads, 2)
    k_bwd_q(int N, int K, int KP, bool causal, float eps, const float *__restrict__ gq, const float *__restrict__ gk,
            const void *__restrict__ v, bool v_bf16, const float *__restrict__ dout, float *states,
            long long st_bh_stride, long long st_blk_stride, float *__restrict__ u, float *__restrict__ dgq)
{
    using Cfg = BwdCfg<DV>;
    constexpr int C = kBC, KC = kBKC, UW = Cfg::UW, LG = Cfg::LG, LP = Cfg::LP, VP = BwdQSmem<DV>::VP;
    constexpr int TM = C / 16, TN = DV / 16, TP = C / 16, TK = KC / 16, PARTS = kThreads / C;
    extern __shared__ __align__(16) float sm[];
    float *gq_s = sm;                  // [C][LG]
    float *gk_s = gq_s + C * LG;       // [C][LG]
    float *v_s = gk_s + C * LG;        // [C][VP]
    float *g_s = v_s + C * VP;         // [C][DV]  dL/dO rows
    float *p_s = g_s + C * DV;         // [C][LP]
    float *s_s = p_s + C * LP;         // [KC][VP]
    float *z_s = s_s + KC * VP;        // [KC]
    float *u_s = z_s + KC;             // [C][UW]
    float *den_s = u_s + C * UW;       // [C]
    float *dot_s = den_s + C;          // [C][16]
    float *dpart = dot_s + C * 16;     // [kThreads]

    const long long bh = blockIdx.y;
    const int blk = blockIdx.x;
    const int r_begin = blk * kBlockRows, r_end = min(N, r_begin + kBlockRows);
    const int tid = threadIdx.x, tm = tid / 16, tn = tid % 16;
    const int drow = tid % C, dpartn = tid / C;
    float *st = states + bh * st_bh_stride + blk * st_blk_stride;
    const int ktiles = (K + KC - 1) / KC;

    auto stage_s = [&](int k0) {
        for (int i = tid; i < KC * DV; i += kThreads) {
            const int k = i / DV, c = i % DV;
            s_s[k * VP + c] = (k0 + k < K) ? st[(long long)(k0 + k) * DV + c] : 0.f;
        }
        for (int i = tid; i < KC; i += kThreads) z_s[i] = (k0 + i < K) ? st[(long long)K * DV + k0 + i] : 0.f;
    };

    for (int c0 = r_begin; c0 < r_end; c0 += C) {
        const int nr = min(C, r_end - c0);
        const long long row0 = bh * N + c0;
        for (int i = tid; i < C * DV / 4; i += kThreads) {
            const int r = i / (DV / 4), c = (i % (DV / 4)) * 4;
            float4 vv = make_float4(0.f, 0.f, 0.f, 0.f), gg = vv;
            if (r < nr) {
                vv = load4(v, (row0 + r) * DV + c, v_bf16);
                gg = *reinterpret_cast<const float4 *>(dout + (row0 + r) * DV + c);
            }
            float *vd = v_s + r * VP + c;
            vd[0] = vv.x; vd[1] = vv.y; vd[2] = vv.z; vd[3] = vv.w;
            *reinterpret_cast<float4 *>(g_s + r * DV + c) = gg;
        }
        // the forward read: numerator (acc), P, Gq . Z
        float acc[TM][TN], pacc[TP][TP];
        float dacc = 0.f;
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
#pragma unroll
        for (int i = 0; i < TP; ++i)
#pragma unroll
            for (int j = 0; j < TP; ++j) pacc[i][j] = 0.f;
        for (int kt = 0; kt < ktiles; ++kt) {
            const int k0 = kt * KC;
            stage_rows(gq_s, LG, gq, row0, nr, KP, k0);
            if (causal) stage_rows(gk_s, LG, gk, row0, nr, KP, k0);
            stage_s(k0);
            __syncthreads();
            if (causal) {
                for (int kk = 0; kk < KC; ++kk) {
                    float a[TP], b[TP];
#pragma unroll
                    for (int i = 0; i < TP; ++i) a[i] = gq_s[(tm * TP + i) * LG + kk];
#pragma unroll
                    for (int j = 0; j < TP; ++j) b[j] = gk_s[(tn * TP + j) * LG + kk];
#pragma unroll
                    for (int i = 0; i < TP; ++i)
#pragma unroll
                        for (int j = 0; j < TP; ++j) pacc[i][j] = fmaf(a[i], b[j], pacc[i][j]);
                }
            }
            for (int kk = 0; kk < KC; ++kk) {
                float a[TM], b[TN];
#pragma unroll
                for (int i = 0; i < TM; ++i) a[i] = gq_s[(tm * TM + i) * LG + kk];
#pragma unroll
                for (int j = 0; j < TN; ++j) b[j] = s_s[kk * VP + tn * TN + j];
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            for (int kk = dpartn; kk < KC; kk += PARTS) dacc = fmaf(gq_s[drow * LG + kk], z_s[kk], dacc);
            __syncthreads();
        }
        if (causal) {
#pragma unroll
            for (int i = 0; i < TP; ++i)
#pragma unroll
                for (int j = 0; j < TP; ++j) {
                    const int r = tm * TP + i, c = tn * TP + j;
                    p_s[r * LP + c] = (c <= r) ? pacc[i][j] : 0.f;
                }
            __syncthreads();
            for (int jj = 0; jj < C; ++jj) {
                float a[TM], b[TN];
#pragma unroll
                for (int i = 0; i < TM; ++i) a[i] = p_s[(tm * TM + i) * LP + jj];
#pragma unroll
                for (int j = 0; j < TN; ++j) b[j] = v_s[jj * VP + tn * TN + j];
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            for (int jj = dpartn; jj < C; jj += PARTS) dacc += p_s[drow * LP + jj];
        }
        dpart[tid] = dacc;
        __syncthreads();
        if (tid < C) {
            float d = 0.f;
            for (int p = 0; p < PARTS; ++p) d += dpart[tid + p * C];
            den_s[tid] = d + eps;
        }
        __syncthreads();
        // u = [g / den | -(g . O) / den]
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int r = tm * TM + i;
            const float inv = 1.0f / den_s[r];
            float dp = 0.f;
#pragma unroll
            for (int j = 0; j < TN; ++j) {
                const int c = tn * TN + j;
                const float g = g_s[r * DV + c];
                u_s[r * UW + c] = g * inv;
                dp = fmaf(g, acc[i][j] * inv, dp);
            }
            dot_s[r * 16 + tn] = dp;
        }
        __syncthreads();
        if (tid < C) {
            float d = 0.f;
#pragma unroll
            for (int p = 0; p < 16; ++p) d += dot_s[tid * 16 + p];
            u_s[tid * UW + DV] = -d / den_s[tid];
#pragma unroll
            for (int c = DV + 1; c < UW; ++c) u_s[tid * UW + c] = 0.f;
        }
        __syncthreads();
        for (int i = tid; i < nr * (UW / 4); i += kThreads) {
            const int r = i / (UW / 4), c = (i % (UW / 4)) * 4;
            *reinterpret_cast<float4 *>(u + (row0 + r) * UW + c) = *reinterpret_cast<const float4 *>(u_s + r * UW + c);
        }
        // Q'_ij = u_i . [v_j | 1] for j <= i (causal), into p_s
        if (causal) {
            float qacc[TP][TP];
#pragma unroll
            for (int i = 0; i < TP; ++i)
#pragma unroll
                for (int j = 0; j < TP; ++j) qacc[i][j] = u_s[(tm * TP + i) * UW + DV];
            for (int c = 0; c < DV; ++c) {
                float a[TP], b[TP];
#pragma unroll
                for (int i = 0; i < TP; ++i) a[i] = u_s[(tm * TP + i) * UW + c];
#pragma unroll
                for (int j = 0; j < TP; ++j) b[j] = v_s[(tn * TP + j) * VP + c];
#pragma unroll
                for (int i = 0; i < TP; ++i)
#pragma unroll
                    for (int j = 0; j < TP; ++j) qacc[i][j] = fmaf(a[i], b[j], qacc[i][j]);
            }
            __syncthreads();   // p_s (P) has been read by every thread
#pragma unroll
            for (int i = 0; i < TP; ++i)
#pragma unroll
                for (int j = 0; j < TP; ++j) {
                    const int r = tm * TP + i, c = tn * TP + j;
                    p_s[r * LP + c] = (c <= r && c < nr) ? qacc[i][j] : 0.f;
                }
        }
        // dGq, one tile of components at a time
        for (int kt = 0; kt < ktiles; ++kt) {
            const int k0 = kt * KC;
            __syncthreads();   // Q' in place; the previous tile's operands have been read
            if (causal) stage_rows(gk_s, LG, gk, row0, nr, KP, k0);
            stage_s(k0);
            __syncthreads();
            float d2[TM][TK];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TK; ++j) d2[i][j] = u_s[(tm * TM + i) * UW + DV] * z_s[tn * TK + j];
            for (int c = 0; c < DV; ++c) {
                float a[TM], b[TK];
#pragma unroll
                for (int i = 0; i < TM; ++i) a[i] = u_s[(tm * TM + i) * UW + c];
#pragma unroll
                for (int j = 0; j < TK; ++j) b[j] = s_s[(tn * TK + j) * VP + c];
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TK; ++j) d2[i][j] = fmaf(a[i], b[j], d2[i][j]);
            }
            if (causal) {
                for (int jj = 0; jj < C; ++jj) {
                    float a[TM], b[TK];
#pragma unroll
                    for (int i = 0; i < TM; ++i) a[i] = p_s[(tm * TM + i) * LP + jj];
#pragma unroll
                    for (int j = 0; j < TK; ++j) b[j] = gk_s[jj * LG + tn * TK + j];
#pragma unroll
                    for (int i = 0; i < TM; ++i)
#pragma unroll
                        for (int j = 0; j < TK; ++j) d2[i][j] = fmaf(a[i], b[j], d2[i][j]);
                }
            }
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const int r = tm * TM + i;
                if (r < nr)
#pragma unroll
                    for (int j = 0; j < TK; ++j) {
                        const int k = k0 + tn * TK + j;
                        if (k < KP) dgq[(row0 + r) * KP + k] = k < K ? d2[i][j] : 0.f;
                    }
            }
        }
        __syncthreads();
        // the carried memory advances by Gk^T [V | 1] (causal)
        if (causal) {
            constexpr int TU = KC / 16;
            for (int kt = 0; kt < ktiles; ++kt) {
                const int k0 = kt * KC;
                stage_rows(gk_s, LG, gk, row0, nr, KP, k0);
                stage_s(k0);
                __syncthreads();
                float a2[TU][TN];
#pragma unroll
                for (int i = 0; i < TU; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) a2[i][j] = s_s[(tm * TU + i) * VP + tn * TN + j];
                for (int jj = 0; jj < C; ++jj) {
                    float a[TU], b[TN];
#pragma unroll
                    for (int i = 0; i < TU; ++i) a[i] = gk_s[jj * LG + tm * TU + i];
#pragma unroll
                    for (int j = 0; j < TN; ++j) b[j] = v_s[jj * VP + tn * TN + j];
#pragma unroll
                    for (int i = 0; i < TU; ++i)
#pragma unroll
                        for (int j = 0; j < TN; ++j) a2[i][j] = fmaf(a[i], b[j], a2[i][j]);
                }
#pragma unroll
                for (int i = 0; i < TU; ++i) {
                    const int k = k0 + tm * TU + i;
                    if (k < K)
#pragma unroll
                        for (int j = 0; j < TN; ++j) st[(long long)k * DV + tn * TN + j] = a2[i][j];
                }
                if (tid < KC && k0 + tid < K) {
                    float z = z_s[tid];
                    for (int jj = 0; jj < C; ++jj) z += gk_s[jj * LG + tid];
                    st[(long long)K * DV + k0 + tid] = z;
                }
                __syncthreads();
            }
        }
    }
}

// ---------------------------------------------------------------------------
// M[bh][blk] = Gq[rows of blk]^T u[rows of blk]   ([K][UW] per block; KC components per CTA).
template <int UW>
__global__ void __launch_bounds__(kThreads)
    k_bwd_mem(int N, int K, int KP, const float *__restrict__ gq, const float *__restrict__ u,
              float *__restrict__ mem, int nblk)
{
    constexpr int KC = 128, RS = 32, TM = KC / 16, TN = UW / 16;
    __shared__ __align__(16) float g_s[RS][KC];
    __shared__ __align__(16) float u_s[RS][UW];
    const long long bh = blockIdx.y;
    const int blk = blockIdx.x, k0 = blockIdx.z * KC;
    const int r_begin = blk * kBlockRows, r_end = min(N, r_begin + kBlockRows);
    const int tid = threadIdx.x, tm = tid / 16, tn = tid % 16;
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
    for (int r0 = r_begin; r0 < r_end; r0 += RS) {
        for (int i = tid; i < RS * KC / 4; i += kThreads) {
            const int r = i / (KC / 4), c = (i % (KC / 4)) * 4, row = r0 + r, k = k0 + c;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row < r_end && k < KP) val = *reinterpret_cast<const float4 *>(gq + (bh * N + row) * KP + k);
            *reinterpret_cast<float4 *>(&g_s[r][c]) = val;
        }
        for (int i = tid; i < RS * UW / 4; i += kThreads) {
            const int r = i / (UW / 4), c = (i % (UW / 4)) * 4, row = r0 + r;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row < r_end) val = *reinterpret_cast<const float4 *>(u + (bh * N + row) * UW + c);
            *reinterpret_cast<float4 *>(&u_s[r][c]) = val;
        }
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < RS; ++r) {
            float a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = g_s[r][tm * TM + i];
#pragma unroll
            for (int j = 0; j < TN; ++j) b[j] = u_s[r][tn * TN + j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    float *o = mem + (bh * nblk + blk) * (long long)K * UW;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int k = k0 + tm * TM + i;
        if (k < K)
#pragma unroll
            for (int j = 0; j < TN; ++j) o[(long long)k * UW + tn * TN + j] = acc[i][j];
    }
}

// Suffix over blocks for every element (fixed order): mem[bh][blk] <- sum_{b > blk} mem[bh][b]
// (exclusive), and total[bh] <- the sum over all blocks (nullable).
__global__ void __launch_bounds__(kThreads) k_scan_rev(long long SZ, int nblk, float *__restrict__ mem,
                                                       float *__restrict__ total, bool exclusive)
{
    const long long e = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (e >= SZ) return;
    const long long bh = blockIdx.y;
    float *p = mem + bh * nblk * SZ + e;
    float run = 0.f;
    for (int b = nblk - 1; b >= 0; --b) {
        const float t = p[(long long)b * SZ];
        if (exclusive) p[(long long)b * SZ] = run;
        run += t;
    }
    if (total) total[bh * SZ + e] = run;
}

// ---------------------------------------------------------------------------
// Key / value side.  Per chunk, last to first, with R the memory of the rows
// after the chunk (causal) or the total (bidirectional):
//   dGk_j = [v_j | 1] R^T + sum_{i >= j in chunk} (u_i . [v_j | 1]) Gq_i
//   dV_j  = Gk_j R[:, :dv] + sum_{i >= j in chunk} (Gk_j . Gq_i) u_i[:dv]
// then R advances by Gq^T u (causal).
template <int DV>
struct BwdKSmem {
    static constexpr int UW = BwdCfg<DV>::UW, LG = BwdCfg<DV>::LG, LP = BwdCfg<DV>::LP;
    static constexpr int UP = UW + 1;   // row pitch of the u rows and the memory rows (odd: no bank conflicts)
    static constexpr size_t floats = (size_t)kBC * LG * 2 + (size_t)kBC * DV + (size_t)kBC * UP + (size_t)kBC * LP * 2 +
                                     (size_t)kBKC * UP;
    static constexpr size_t bytes = floats * 4;
};

template <int DV>
__global__ void __launch_bounds__(kThreads, 2)
    k_bwd_k(int N, int K, int KP, bool causal, const float *__restrict__ gq, const float *__restrict__ gk,
            const void *__restrict__ v, bool v_bf16, const float *__restrict__ u, float *rmem,
            long long r_bh_stride, long long r_blk_stride, float *__restrict__ dgk, float *__restrict__ dv)
{
    using Cfg = BwdCfg<DV>;
    constexpr int C = kBC, KC = kBKC, UW = Cfg::UW, LG = Cfg::LG, LP = Cfg::LP, UP = BwdKSmem<DV>::UP;
    constexpr int TM = C / 16, TN = DV / 16, TP = C / 16, TK = KC / 16;
    extern __shared__ __align__(16) float sm[];
    float *gq_s = sm;                  // [C][LG]
    float *gk_s = gq_s + C * LG;       // [C][LG]
    float *v_s = gk_s + C * LG;        // [C][DV]
    float *u_s = v_s + C * DV;         // [C][UP]
    float *q_s = u_s + C * UP;         // [C][LP]  Q''_ji = u_i . [v_j | 1], i >= j
    float *p_s = q_s + C * LP;         // [C][LP]  P_ji = Gk_j . Gq_i, i >= j
    float *r_s = p_s + C * LP;         // [KC][UP]

    const long long bh = blockIdx.y;
    const int blk = blockIdx.x;
    const int r_begin = blk * kBlockRows, r_end = min(N, r_begin + kBlockRows);
    const int tid = threadIdx.x, tm = tid / 16, tn = tid % 16;
    float *rm = rmem + bh * r_bh_stride + blk * r_blk_stride;
    const int ktiles = (K + KC - 1) / KC;

    auto stage_r = [&](int k0) {
        for (int i = tid; i < KC * UW / 4; i += kThreads) {
            const int k = i / (UW / 4), c = (i % (UW / 4)) * 4;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k0 + k < K) val = *reinterpret_cast<const float4 *>(rm + (long long)(k0 + k) * UW + c);
            float *rd = r_s + k * UP + c;
            rd[0] = val.x; rd[1] = val.y; rd[2] = val.z; rd[3] = val.w;
        }
    };

    const int nchunks = (r_end - r_begin + C - 1) / C;
    for (int ci = nchunks - 1; ci >= 0; --ci) {
        const int c0 = r_begin + ci * C;
        const int nr = min(C, r_end - c0);
        const long long row0 = bh * N + c0;
        for (int i = tid; i < C * DV / 4; i += kThreads) {
            const int r = i / (DV / 4), c = (i % (DV / 4)) * 4;
            float4 vv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < nr) vv = load4(v, (row0 + r) * DV + c, v_bf16);
            *reinterpret_cast<float4 *>(v_s + r * DV + c) = vv;
        }
        for (int i = tid; i < C * UW / 4; i += kThreads) {
            const int r = i / (UW / 4), c = (i % (UW / 4)) * 4;
            float4 uu = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < nr) uu = *reinterpret_cast<const float4 *>(u + (row0 + r) * UW + c);
            float *ud = u_s + r * UP + c;
            ud[0] = uu.x; ud[1] = uu.y; ud[2] = uu.z; ud[3] = uu.w;
        }
        __syncthreads();
        if (causal) {   // Q''_ji (rows j, columns i) for i >= j
            float qacc[TP][TP];
#pragma unroll
            for (int j = 0; j < TP; ++j)
#pragma unroll
                for (int i = 0; i < TP; ++i) qacc[j][i] = u_s[(tn * TP + i) * UP + DV];
            for (int c = 0; c < DV; ++c) {
                float a[TP], b[TP];
#pragma unroll
                for (int j = 0; j < TP; ++j) a[j] = v_s[(tm * TP + j) * DV + c];
#pragma unroll
                for (int i = 0; i < TP; ++i) b[i] = u_s[(tn * TP + i) * UP + c];
#pragma unroll
                for (int j = 0; j < TP; ++j)
#pragma unroll
                    for (int i = 0; i < TP; ++i) qacc[j][i] = fmaf(a[j], b[i], qacc[j][i]);
            }
#pragma unroll
            for (int j = 0; j < TP; ++j)
#pragma unroll
                for (int i = 0; i < TP; ++i) {
                    const int rj = tm * TP + j, ci2 = tn * TP + i;
                    q_s[rj * LP + ci2] = (ci2 >= rj && ci2 < nr) ? qacc[j][i] : 0.f;
                }
        }
        float dvacc[TM][TN], pacc[TP][TP];
#pragma unroll
        for (int i = 0; i < TM; ++i)
#pragma unroll
            for (int j = 0; j < TN; ++j) dvacc[i][j] = 0.f;
#pragma unroll
        for (int i = 0; i < TP; ++i)
#pragma unroll
            for (int j = 0; j < TP; ++j) pacc[i][j] = 0.f;
        for (int kt = 0; kt < ktiles; ++kt) {
            const int k0 = kt * KC;
            __syncthreads();   // Q'' in place; the previous tile's operands have been read
            stage_rows(gk_s, LG, gk, row0, nr, KP, k0);
            if (causal) stage_rows(gq_s, LG, gq, row0, nr, KP, k0);
            stage_r(k0);
            __syncthreads();
            // dGk tile: rows j (tm), components k (tn)
            float d2[TM][TK];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TK; ++j) d2[i][j] = r_s[(tn * TK + j) * UP + DV];
            for (int c = 0; c < DV; ++c) {
                float a[TM], b[TK];
#pragma unroll
                for (int i = 0; i < TM; ++i) a[i] = v_s[(tm * TM + i) * DV + c];
#pragma unroll
                for (int j = 0; j < TK; ++j) b[j] = r_s[(tn * TK + j) * UP + c];
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TK; ++j) d2[i][j] = fmaf(a[i], b[j], d2[i][j]);
            }
            if (causal) {
                for (int ii = 0; ii < C; ++ii) {
                    float a[TM], b[TK];
#pragma unroll
                    for (int i = 0; i < TM; ++i) a[i] = q_s[(tm * TM + i) * LP + ii];
#pragma unroll
                    for (int j = 0; j < TK; ++j) b[j] = gq_s[ii * LG + tn * TK + j];
#pragma unroll
                    for (int i = 0; i < TM; ++i)
#pragma unroll
                        for (int j = 0; j < TK; ++j) d2[i][j] = fmaf(a[i], b[j], d2[i][j]);
                }
            }
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const int r = tm * TM + i;
                if (r < nr)
#pragma unroll
                    for (int j = 0; j < TK; ++j) {
                        const int k = k0 + tn * TK + j;
                        if (k < KP) dgk[(row0 + r) * KP + k] = k < K ? d2[i][j] : 0.f;
                    }
            }
            // dV += Gk R[:, :dv] over this tile; P_ji += Gk_j . Gq_i
            for (int kk = 0; kk < KC; ++kk) {
                float a[TM], b[TN];
#pragma unroll
                for (int i = 0; i < TM; ++i) a[i] = gk_s[(tm * TM + i) * LG + kk];
#pragma unroll
                for (int j = 0; j < TN; ++j) b[j] = r_s[kk * UP + tn * TN + j];
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) dvacc[i][j] = fmaf(a[i], b[j], dvacc[i][j]);
            }
            if (causal) {
                for (int kk = 0; kk < KC; ++kk) {
                    float a[TP], b[TP];
#pragma unroll
                    for (int j = 0; j < TP; ++j) a[j] = gk_s[(tm * TP + j) * LG + kk];
#pragma unroll
                    for (int i = 0; i < TP; ++i) b[i] = gq_s[(tn * TP + i) * LG + kk];
#pragma unroll
                    for (int j = 0; j < TP; ++j)
#pragma unroll
                        for (int i = 0; i < TP; ++i) pacc[j][i] = fmaf(a[j], b[i], pacc[j][i]);
                }
            }
        }
        if (causal) {
#pragma unroll
            for (int j = 0; j < TP; ++j)
#pragma unroll
                for (int i = 0; i < TP; ++i) {
                    const int rj = tm * TP + j, ci2 = tn * TP + i;
                    p_s[rj * LP + ci2] = (ci2 >= rj && ci2 < nr) ? pacc[j][i] : 0.f;
                }
            __syncthreads();
            for (int ii = 0; ii < C; ++ii) {
                float a[TM], b[TN];
#pragma unroll
                for (int i = 0; i < TM; ++i) a[i] = p_s[(tm * TM + i) * LP + ii];
#pragma unroll
                for (int j = 0; j < TN; ++j) b[j] = u_s[ii * UP + tn * TN + j];
#pragma unroll
                for (int i = 0; i < TM; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) dvacc[i][j] = fmaf(a[i], b[j], dvacc[i][j]);
            }
        }
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int r = tm * TM + i;
            if (r < nr)
#pragma unroll
                for (int j = 0; j < TN; ++j) dv[(row0 + r) * DV + tn * TN + j] = dvacc[i][j];
        }
        // R advances by Gq^T u (causal): rows of R (components, tm), columns of u (tn)
        if (causal) {
            constexpr int TU = KC / 16, TW = UW / 16;
            for (int kt = 0; kt < ktiles; ++kt) {
                const int k0 = kt * KC;
                __syncthreads();
                stage_rows(gq_s, LG, gq, row0, nr, KP, k0);
                stage_r(k0);
                __syncthreads();
                float a2[TU][TW];
#pragma unroll
                for (int i = 0; i < TU; ++i)
#pragma unroll
                    for (int j = 0; j < TW; ++j) a2[i][j] = r_s[(tm * TU + i) * UP + tn * TW + j];
                for (int ii = 0; ii < C; ++ii) {
                    float a[TU], b[TW];
#pragma unroll
                    for (int i = 0; i < TU; ++i) a[i] = gq_s[ii * LG + tm * TU + i];
#pragma unroll
                    for (int j = 0; j < TW; ++j) b[j] = u_s[ii * UP + tn * TW + j];
#pragma unroll
                    for (int i = 0; i < TU; ++i)
#pragma unroll
                        for (int j = 0; j < TW; ++j) a2[i][j] = fmaf(a[i], b[j], a2[i][j]);
                }
#pragma unroll
                for (int i = 0; i < TU; ++i) {
                    const int k = k0 + tm * TU + i;
                    if (k < K)
#pragma unroll
                        for (int j = 0; j < TW; ++j) rm[(long long)k * UW + tn * TW + j] = a2[i][j];
                }
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// delta = Gamma (dGamma - rowsum(Gamma dGamma)), in place of dGamma; a warp per row.
__global__ void __launch_bounds__(kThreads) k_bwd_delta(long long rows, int K, int KP, const float *__restrict__ g,
                                                        float *__restrict__ dg)
{
    const long long row = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float *gr = g + row * KP;
    float *dr = dg + row * KP;
    float dot = 0.f;
    for (int k = lane; k < K; k += 32) dot = fmaf(gr[k], dr[k], dot);
#pragma unroll
    for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    for (int k = lane; k < K; k += 32) dr[k] = gr[k] * (dr[k] - dot);
}

// dx_d = -sum_k delta_k y_kd s_kd with y = x s - mu s: rows of one slice, a thread per
// (four consecutive rows, feature pair), the parameters of KT components at a time in
// shared memory.  One 16-byte parameter word and one 16-byte word of delta (the tile is
// held transposed, [component][row]) serve the thread's four rows.
constexpr int kDxRows = 4;   // rows per thread
template <int D>
struct DxCfg {
    static constexpr int DP = D / 2, RG = kThreads / DP, RT = RG * kDxRows;   // row groups, rows per CTA
    static constexpr int KT = D == 128 ? 32 : 64;                                // components per tile
    static constexpr int DPITCH = RT + 4;   // delta tile pitch: 16-byte rows, 4-way conflicts when staged
};

template <int D>
__global__ void __launch_bounds__(kThreads) k_bwd_dx(int N, int K, int KP, int H, const void *__restrict__ x,
                                                     bool x_bf16, const float4 *__restrict__ prm,
                                                     const float *__restrict__ delta, float *__restrict__ dx)
{
    using Cfg = DxCfg<D>;
    constexpr int DP = Cfg::DP, RT = Cfg::RT, KT = Cfg::KT, DPITCH = Cfg::DPITCH;
    __shared__ float4 p_s[KT * DP];
    __shared__ __align__(16) float d_s[KT * DPITCH];
    const long long bh = blockIdx.y;
    const int h = (int)(bh % H), tid = threadIdx.x, dp = tid % DP, rg = tid / DP;
    const int row0 = blockIdx.x * RT + rg * kDxRows;   // this thread's rows row0 .. row0 + 3
    float2 xv[kDxRows], acc[kDxRows];
#pragma unroll
    for (int i = 0; i < kDxRows; ++i) {
        const int row = row0 + i;
        const long long xo = (bh * N + row) * D + 2 * dp;
        xv[i] = make_float2(0.f, 0.f);
        acc[i] = make_float2(0.f, 0.f);
        if (row < N) {
            if (x_bf16) {
                const uint32_t w = *reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(x) + xo);
                xv[i] = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
            } else {
                xv[i] = *reinterpret_cast<const float2 *>(static_cast<const float *>(x) + xo);
            }
        }
    }
    for (int k0 = 0; k0 < K; k0 += KT) {
        const int kn = min(KT, K - k0);
        __syncthreads();
        for (int i = tid; i < kn * DP; i += kThreads) p_s[i] = prm[((long long)h * K + k0) * DP + i];
        for (int i = tid; i < RT * KT; i += kThreads) {   // coalesced along the components
            const int r = i / KT, k = i % KT, rw = blockIdx.x * RT + r;
            d_s[k * DPITCH + r] = (rw < N && k < kn) ? delta[(bh * N + rw) * KP + k0 + k] : 0.f;
        }
        __syncthreads();
        for (int k = 0; k < kn; ++k) {
            const float4 p = p_s[k * DP + dp];
            const float4 d4 = *reinterpret_cast<const float4 *>(d_s + k * DPITCH + rg * kDxRows);
            const float dk[kDxRows] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
            for (int i = 0; i < kDxRows; ++i) {
                const float y0 = fmaf(xv[i].x, p.x, p.z), y1 = fmaf(xv[i].y, p.y, p.w);
                acc[i].x = fmaf(dk[i] * p.x, y0, acc[i].x);
                acc[i].y = fmaf(dk[i] * p.y, y1, acc[i].y);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kDxRows; ++i) {
        const int row = row0 + i;
        if (row < N)
            *reinterpret_cast<float2 *>(dx + (bh * N + row) * D + 2 * dp) = make_float2(-acc[i].x, -acc[i].y);
    }
}

// Parameter partial sums of one block of kBlockRows rows of one slice: a thread per
// (component, feature pair) of a tile of KT components, rows RS at a time.
//   pmu[bh][blk][k][d] = sum_rows delta_k y s,  pvar[..] = sum_rows delta_k s^2 (y^2 - 1) / 2,
//   plp[bh][blk][k]    = sum_rows delta_k
// s is constant over the rows, so the row loop sums delta y and delta y^2 (four packed
// operations per feature pair and row) and the factors s and s^2 / 2 are applied once.
template <int D>
__global__ void __launch_bounds__(kThreads) k_bwd_param(int N, int K, int KP, int H, const void *__restrict__ x,
                                                        bool x_bf16, const float4 *__restrict__ prm,
                                                        const float *__restrict__ delta, float *__restrict__ pmu,
                                                        float *__restrict__ pvar, float *__restrict__ plp, int nblk)
{
    constexpr int DP = D / 2, KT = kThreads / DP * 4 > 128 ? 128 : kThreads / DP * 4;   // components per CTA
    constexpr int PER = KT * DP / kThreads;                                               // (k, pair) per thread
    constexpr int RS = 32;
    __shared__ float2 x_s[RS][DP];
    __shared__ float d_s[RS][KT + 1];
    const long long bh = blockIdx.y;
    const int h = (int)(bh % H), blk = blockIdx.x, k0 = blockIdx.z * KT, tid = threadIdx.x;
    const int r_begin = blk * kBlockRows, r_end = min(N, r_begin + kBlockRows);
    float4 p[PER];
    float2 ga[PER], gb[PER];   // sums over the rows of delta y and delta y^2
    float sd[PER];             // sum over the rows of delta
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        const int f = tid + e * kThreads, k = f / DP, dp = f % DP;
        p[e] = k0 + k < K ? prm[((long long)h * K + k0 + k) * DP + dp] : make_float4(0.f, 0.f, 0.f, 0.f);
        ga[e] = gb[e] = make_float2(0.f, 0.f);
        sd[e] = 0.f;
    }
    float lp = 0.f;
    for (int r0 = r_begin; r0 < r_end; r0 += RS) {
        __syncthreads();
        for (int i = tid; i < RS * DP; i += kThreads) {
            const int r = i / DP, dp = i % DP, row = r0 + r;
            float2 v2 = make_float2(0.f, 0.f);
            if (row < r_end) {
                const long long xo = (bh * N + row) * D + 2 * dp;
                if (x_bf16) {
                    const uint32_t w = *reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(x) + xo);
                    v2 = make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
                } else {
                    v2 = *reinterpret_cast<const float2 *>(static_cast<const float *>(x) + xo);
                }
            }
            x_s[r][dp] = v2;
        }
        for (int i = tid; i < RS * KT; i += kThreads) {
            const int r = i / KT, k = i % KT, row = r0 + r;
            d_s[r][k] = (row < r_end && k0 + k < K) ? delta[(bh * N + row) * KP + k0 + k] : 0.f;
        }
        __syncthreads();
        const int nr = min(RS, r_end - r0);
        for (int r = 0; r < nr; ++r) {
#pragma unroll
            for (int e = 0; e < PER; ++e) {
                const int f = tid + e * kThreads, k = f / DP, dp = f % DP;
                const float dk = d_s[r][k];
                const float2 y = __ffma2_rn(x_s[r][dp], make_float2(p[e].x, p[e].y), make_float2(p[e].z, p[e].w));
                const float2 dy = __fmul2_rn(make_float2(dk, dk), y);
                ga[e] = __fadd2_rn(ga[e], dy);
                gb[e] = __ffma2_rn(dy, y, gb[e]);
                sd[e] += dk;
            }
            if (tid < KT) lp += d_s[r][tid];
        }
    }
    const long long base = (bh * nblk + blk) * (long long)K;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        const int f = tid + e * kThreads, k = f / DP, dp = f % DP;
        if (k0 + k < K) {
            const float2 gm = make_float2(p[e].x * ga[e].x, p[e].y * ga[e].y);
            const float2 gv = make_float2(0.5f * p[e].x * p[e].x * (gb[e].x - sd[e]),
                                          0.5f * p[e].y * p[e].y * (gb[e].y - sd[e]));
            reinterpret_cast<float2 *>(pmu + (base + k0 + k) * D)[dp] = gm;
            reinterpret_cast<float2 *>(pvar + (base + k0 + k) * D)[dp] = gv;
        }
    }
    if (tid < KT && k0 + tid < K) plp[base + k0 + tid] = lp;
}

// Per head: the partial sums over both routings, the slices of the head (b in order) and
// the blocks, then the reparameterisation.  A thread per (component, feature) element.
__global__ void __launch_bounds__(kThreads) k_bwd_final(int B, int H, int K, int D, int nblk,
                                                        const float *__restrict__ pmu, const float *__restrict__ pvar,
                                                        const float *__restrict__ plp, long long pass_stride,
                                                        long long pass_stride_lp, const float *__restrict__ var_raw,
                                                        const float *__restrict__ logit_pi, float *__restrict__ dmu,
                                                        float *__restrict__ dvar, float *__restrict__ dlogit)
{
    const int h = blockIdx.y, tid = threadIdx.x;
    const long long e = (long long)blockIdx.x * kThreads + tid;
    const long long KD = (long long)K * D;
    if (e < KD) {
        float m = 0.f, s = 0.f;
        for (int pass = 0; pass < 2; ++pass)
            for (int b = 0; b < B; ++b) {
                const long long bh = (long long)b * H + h;
                for (int blk = 0; blk < nblk; ++blk) {
                    const long long o = pass * pass_stride + (bh * nblk + blk) * KD + e;
                    m += pmu[o];
                    s += pvar[o];
                }
            }
        const float r = var_raw[(long long)h * KD + e];
        dmu[(long long)h * KD + e] = m;
        dvar[(long long)h * KD + e] = s / (1.f + expf(-r));   // softplus' = sigmoid
    }
    if (blockIdx.x == 0) {   // the logits of the head: G_k - pi_k sum G
        __shared__ float red[kThreads];
        __shared__ float bc[2];
        float g[2] = {0.f, 0.f}, l[2] = {-FLT_MAX, -FLT_MAX};
        for (int j = 0; j < 2; ++j) {
            const int k = tid + j * kThreads;
            if (k >= K) continue;
            for (int pass = 0; pass < 2; ++pass)
                for (int b = 0; b < B; ++b) {
                    const long long bh = (long long)b * H + h;
                    for (int blk = 0; blk < nblk; ++blk) g[j] += plp[pass * pass_stride_lp + (bh * nblk + blk) * K + k];
                }
            l[j] = logit_pi[(long long)h * K + k];
        }
        // max of the logits, then sum of exp, then sum of G (fixed tree order)
        red[tid] = fmaxf(l[0], l[1]);
        __syncthreads();
        for (int st = kThreads / 2; st > 0; st >>= 1) {
            if (tid < st) red[tid] = fmaxf(red[tid], red[tid + st]);
            __syncthreads();
        }
        const float lmax = red[0];
        __syncthreads();
        float ex = 0.f;
        for (int j = 0; j < 2; ++j)
            if (tid + j * kThreads < K) ex += expf(l[j] - lmax);
        red[tid] = ex;
        __syncthreads();
        for (int st = kThreads / 2; st > 0; st >>= 1) {
            if (tid < st) red[tid] += red[tid + st];
            __syncthreads();
        }
        if (tid == 0) bc[0] = red[0];
        __syncthreads();
        red[tid] = g[0] + g[1];
        __syncthreads();
        for (int st = kThreads / 2; st > 0; st >>= 1) {
            if (tid < st) red[tid] += red[tid + st];
            __syncthreads();
        }
        if (tid == 0) bc[1] = red[0];
        __syncthreads();
        for (int j = 0; j < 2; ++j) {
            const int k = tid + j * kThreads;
            if (k < K) dlogit[(long long)h * K + k] = g[j] - expf(l[j] - lmax) / bc[0] * bc[1];
        }
    }
}

template <int DV>
cudaError_t launch_bwd_q_dv(const Dims &dm, bool causal, const float *gq, const float *gk, const void *v,
                            const float *dout, float *states, float *u, float *dgq, cudaStream_t st)
{
    constexpr size_t smem = BwdQSmem<DV>::bytes;
    static std::atomic<unsigned long long> smem_set{0};
    const cudaError_t attr = allow_smem(k_bwd_q<DV>, smem, smem_set);
    if (attr != cudaSuccess) return attr;
    const long long SZ = dm.state_size();
    k_bwd_q<DV><<<dim3(dm.nblk(), (unsigned)dm.BH()), kThreads, smem, st>>>(
        dm.N, dm.K, dm.KP, causal, dm.eps, gq, gk, v, dm.v_bf16, dout, states, causal ? (long long)dm.nblk() * SZ : SZ,
        causal ? SZ : 0, u, dgq);
    return cudaGetLastError();
}

template <int DV>
cudaError_t launch_bwd_kv_dv(const Dims &dm, bool causal, const float *gq, const float *gk, const void *v,
                             const float *u, float *mem, float *rtot, float *dgk, float *dv, cudaStream_t st)
{
    constexpr int UW = BwdCfg<DV>::UW;
    const long long RSZ = (long long)dm.K * UW;
    k_bwd_mem<UW><<<dim3(dm.nblk(), (unsigned)dm.BH(), (dm.K + 127) / 128), kThreads, 0, st>>>(dm.N, dm.K, dm.KP, gq, u,
                                                                                            mem, dm.nblk());
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_scan_rev<<<dim3((unsigned)((RSZ + kThreads - 1) / kThreads), (unsigned)dm.BH()), kThreads, 0, st>>>(
        RSZ, dm.nblk(), mem, causal ? nullptr : rtot, causal);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    constexpr size_t smem = BwdKSmem<DV>::bytes;
    static std::atomic<unsigned long long> smem_set{0};
    e = allow_smem(k_bwd_k<DV>, smem, smem_set);
    if (e != cudaSuccess) return e;
    float *r = causal ? mem : rtot;
    k_bwd_k<DV><<<dim3(dm.nblk(), (unsigned)dm.BH()), kThreads, smem, st>>>(
        dm.N, dm.K, dm.KP, causal, gq, gk, v, dm.v_bf16, u, r, causal ? (long long)dm.nblk() * RSZ : RSZ,
        causal ? RSZ : 0, dgk, dv);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_route_d(const Dims &dm, const void *x, const float4 *prm, const float *delta, float *dx,
                               float *pmu, float *pvar, float *plp, cudaStream_t st)
{
    constexpr int DP = D / 2, RT = DxCfg<D>::RT;
    k_bwd_dx<D><<<dim3((dm.N + RT - 1) / RT, (unsigned)dm.BH()), kThreads, 0, st>>>(dm.N, dm.K, dm.KP, dm.H, x,
                                                                                  dm.x_bf16, prm, delta, dx);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    constexpr int KT = kThreads / DP * 4 > 128 ? 128 : kThreads / DP * 4;
    k_bwd_param<D><<<dim3(dm.nblk(), (unsigned)dm.BH(), (dm.K + KT - 1) / KT), kThreads, 0, st>>>(
        dm.N, dm.K, dm.KP, dm.H, x, dm.x_bf16, prm, delta, pmu, pvar, plp, dm.nblk());
    return cudaGetLastError();
}

} // namespace

size_t bwd_u_pitch(const Dims &dm) { return (size_t)dm.DV + 16; }

cudaError_t launch_bwd_q(const Dims &dm, bool causal, const float *gq, const float *gk, const void *v,
                         const float *dout, float *states, float *u, float *dgq, cudaStream_t st)
{
    switch (dm.DV) {
    case 16: return launch_bwd_q_dv<16>(dm, causal, gq, gk, v, dout, states, u, dgq, st);
    case 32: return launch_bwd_q_dv<32>(dm, causal, gq, gk, v, dout, states, u, dgq, st);
    case 64: return launch_bwd_q_dv<64>(dm, causal, gq, gk, v, dout, states, u, dgq, st);
    case 128: return launch_bwd_q_dv<128>(dm, causal, gq, gk, v, dout, states, u, dgq, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_kv(const Dims &dm, bool causal, const float *gq, const float *gk, const void *v,
                          const float *u, float *mem, float *rtot, float *dgk, float *dv, cudaStream_t st)
{
    switch (dm.DV) {
    case 16: return launch_bwd_kv_dv<16>(dm, causal, gq, gk, v, u, mem, rtot, dgk, dv, st);
    case 32: return launch_bwd_kv_dv<32>(dm, causal, gq, gk, v, u, mem, rtot, dgk, dv, st);
    case 64: return launch_bwd_kv_dv<64>(dm, causal, gq, gk, v, u, mem, rtot, dgk, dv, st);
    case 128: return launch_bwd_kv_dv<128>(dm, causal, gq, gk, v, u, mem, rtot, dgk, dv, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_route(const Dims &dm, const void *x, const float4 *prm, const float *gamma, float *dgamma,
                             float *dx, float *pmu, float *pvar, float *plp, cudaStream_t st)
{
    const long long rows = dm.BH() * dm.N;
    k_bwd_delta<<<(unsigned)((rows + kThreads / 32 - 1) / (kThreads / 32)), kThreads, 0, st>>>(rows, dm.K, dm.KP,
                                                                                             gamma, dgamma);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    switch (dm.D) {
    case 16: return launch_bwd_route_d<16>(dm, x, prm, dgamma, dx, pmu, pvar, plp, st);
    case 32: return launch_bwd_route_d<32>(dm, x, prm, dgamma, dx, pmu, pvar, plp, st);
    case 64: return launch_bwd_route_d<64>(dm, x, prm, dgamma, dx, pmu, pvar, plp, st);
    case 128: return launch_bwd_route_d<128>(dm, x, prm, dgamma, dx, pmu, pvar, plp, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_final(const Dims &dm, const gma_params &p, const float *pmu, const float *pvar,
                             const float *plp, float *dmu, float *dvar, float *dlogit, cudaStream_t st)
{
    const long long KD = (long long)dm.K * dm.D;
    const long long pass = dm.BH() * dm.nblk() * KD, pass_lp = dm.BH() * dm.nblk() * (long long)dm.K;
    k_bwd_final<<<dim3((unsigned)((KD + kThreads - 1) / kThreads), (unsigned)dm.H), kThreads, 0, st>>>(
        dm.B, dm.H, dm.K, dm.D, dm.nblk(), pmu, pvar, plp, pass, pass_lp, p.var_raw, p.logit_pi, dmu, dvar, dlogit);
    return cudaGetLastError();
}

} // namespace gma
