// Latent-memory write / read kernels (S2, S3, S4), generic CUDA-core path.
//
// The write phase of the GMA explainer ("핵심 메커니즘") aggregates values into
// K slots, Vt = Gamma_K^T V and Z = Gamma_K^T 1; the read phase returns
// O = Gamma_Q Vt / (Gamma_Q Z + eps).  The causal variant ("변형 및 학습") uses
// prefix sums, evaluated here in the chunkwise-parallel form described by the
// linear-attention page ("선형 어텐션 원리 정리", "쉽게 이해하기"): the sequence
// is cut into blocks of kBlockRows rows, each block's memory contribution is
// computed independently (k_block_state), an exclusive scan over blocks gives
// each block its incoming memory (k_scan), and inside a block chunks of C rows
// use a dense masked intra-chunk product plus a read of the carried memory,
// which is then advanced by the chunk (k_chunk_out).  Every reduction runs in
// a fixed order (no atomics), so repeated calls give identical bits.
#include "gma_internal.cuh"

namespace gma {
namespace {

// partial[bh][blk] = Gamma_K[rows of blk]^T [V | 1]   (KC components per CTA).
template <int DV>
__global__ void __launch_bounds__(kThreads)
    k_block_state(int N, int K, int KP, const void *__restrict__ gk, bool g_bf16, const void *__restrict__ v,
                  bool v_bf16, float *__restrict__ partial, int nblk)
{
    constexpr int KC = 128, RS = 32, TM = KC / 16, TN = DV / 16;
    __shared__ __align__(16) float g_s[RS][KC];
    __shared__ __align__(16) float v_s[RS][DV];
    const long long bh = blockIdx.y;
    const int blk = blockIdx.x, k0 = blockIdx.z * KC;
    const int r_begin = blk * kBlockRows, r_end = min(N, r_begin + kBlockRows);
    const int tid = threadIdx.x, tm = tid / 16, tn = tid % 16;
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
    float z = 0.f;

    for (int r0 = r_begin; r0 < r_end; r0 += RS) {
        for (int i = tid; i < RS * KC / 4; i += kThreads) {
            const int r = i / (KC / 4), c = (i % (KC / 4)) * 4, row = r0 + r, k = k0 + c;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row < r_end && k < KP) val = load4(gk, (bh * N + row) * KP + k, g_bf16);
            *reinterpret_cast<float4 *>(&g_s[r][c]) = val;
        }
        for (int i = tid; i < RS * DV / 4; i += kThreads) {
            const int r = i / (DV / 4), c = (i % (DV / 4)) * 4, row = r0 + r;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row < r_end) val = load4(v, (bh * N + row) * DV + c, v_bf16);
            *reinterpret_cast<float4 *>(&v_s[r][c]) = val;
        }
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < RS; ++r) {
            float a[TM], b[TN];
#pragma unroll
            for (int i = 0; i < TM; ++i) a[i] = g_s[r][tm * TM + i];
#pragma unroll
            for (int j = 0; j < TN; ++j) b[j] = v_s[r][tn * TN + j];
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            if (tid < KC) z += g_s[r][tid];
        }
        __syncthreads();
    }
    const long long SZ = (long long)K * DV + K;
    float *o = partial + (bh * nblk + blk) * SZ;
#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int k = k0 + tm * TM + i;
        if (k < K)
#pragma unroll
            for (int j = 0; j < TN; ++j) o[(long long)k * DV + tn * TN + j] = acc[i][j];
    }
    if (tid < KC && k0 + tid < K) o[(long long)K * DV + k0 + tid] = z;
}

// Serial scan over blocks for every state element (fixed order, deterministic).
//   exclusive: partial[bh][blk] <- state_in + sum_{b < blk} partial[bh][b]
//   total (nullable) <- state_in + sum_b partial[bh][b]
//   tr_k > 0: blocks hold Vt transposed (tr_dv rows of tr_k, then Z); state_in / total
//   keep the caller layout (Vt as tr_k rows of tr_dv, then Z).
__global__ void __launch_bounds__(kThreads) k_scan(long long SZ, int nblk, float *__restrict__ partial,
                                                   const float *state_in, float *total, bool exclusive, int tr_k,
                                                   int tr_dv)
{
    const long long e = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (e >= SZ) return;
    const long long bh = blockIdx.y;
    long long eu = e;   // the same element in the caller's layout
    if (tr_k > 0 && e < (long long)tr_k * tr_dv) eu = (e % tr_k) * tr_dv + e / tr_k;
    float run = state_in ? state_in[bh * SZ + eu] : 0.f;
    float *__restrict__ p = partial + bh * nblk * SZ + e;
    constexpr int U = 32; // loads in flight per thread
    int b = 0;
    for (; b + U <= nblk; b += U) {
        float t[U];
#pragma unroll
        for (int u = 0; u < U; ++u) t[u] = p[(long long)(b + u) * SZ];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (exclusive) p[(long long)(b + u) * SZ] = run;
            run += t[u];
        }
    }
    for (; b < nblk; ++b) {
        const float t = p[(long long)b * SZ];
        if (exclusive) p[(long long)b * SZ] = run;
        run += t;
    }
    if (total) total[bh * SZ + eu] = run;
}

// Output of one block of kBlockRows rows, chunk by chunk (C rows each).
//   causal: O_c = [(Gq_c Gk_c^T) .* tril] [V_c | 1] + Gq_c [Vt | Z]   then divide,
//           and the block's memory (initialised by k_scan) advances by Gk_c^T [V_c | 1].
//   bidir : O_c = Gq_c [Vt | Z] with the fixed total memory, then divide.
template <int DV, int C>
struct ChunkSmem {
    static constexpr int KC = 64;
    static constexpr size_t floats = (size_t)C * (KC + 1) * 2 + (size_t)C * DV + (size_t)C * (C + 1) +
                                     (size_t)KC * DV + KC + C + kThreads;
    static constexpr size_t bytes = floats * 4;
};

template <int DV, int C>
__global__ void __launch_bounds__(kThreads, 1)
    k_chunk_out(int N, int K, int KP, bool causal, float eps, const void *__restrict__ gq,
                const void *__restrict__ gk, bool g_bf16, const void *__restrict__ v, bool v_bf16,
                float *states, long long st_bh_stride, long long st_blk_stride, float *__restrict__ out)
{
    constexpr int KC = ChunkSmem<DV, C>::KC;
    constexpr int TM = C / 16, TN = DV / 16, TP = C / 16, TU = KC / 16, PARTS = kThreads / C;
    constexpr int LG = KC + 1, LP = C + 1;
    extern __shared__ __align__(16) float sm[];
    float *gq_s = sm;                  // [C][LG]
    float *gk_s = gq_s + C * LG;       // [C][LG]
    float *v_s = gk_s + C * LG;        // [C][DV]
    float *p_s = v_s + C * DV;         // [C][LP]
    float *s_s = p_s + C * LP;         // [KC][DV]
    float *z_s = s_s + KC * DV;        // [KC]
    float *den_s = z_s + KC;           // [C]
    float *dpart = den_s + C;          // [kThreads]

    const long long bh = blockIdx.y;
    const int blk = blockIdx.x;
    const int r_begin = blk * kBlockRows, r_end = min(N, r_begin + kBlockRows);
    const int tid = threadIdx.x, tm = tid / 16, tn = tid % 16;
    const int drow = tid % C, dpartn = tid / C;
    const long long SZ = (long long)K * DV + K;
    float *st = states + bh * st_bh_stride + blk * st_blk_stride;
    const int ktiles = (K + KC - 1) / KC;

    auto stage_g = [&](float *dst, const void *src, int c0, int nr, int k0) {
        for (int i = tid; i < C * KC / 4; i += kThreads) {
            const int r = i / (KC / 4), c = (i % (KC / 4)) * 4, k = k0 + c;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < nr && k < KP) val = load4(src, (bh * N + c0 + r) * KP + k, g_bf16);
            float *d = dst + r * LG + c;
            d[0] = val.x; d[1] = val.y; d[2] = val.z; d[3] = val.w;
        }
    };
    auto stage_s = [&](int k0) {
        for (int i = tid; i < KC * DV; i += kThreads) {
            const int k = i / DV, c = i % DV;
            s_s[i] = (k0 + k < K) ? st[(long long)(k0 + k) * DV + c] : 0.f;
        }
        for (int i = tid; i < KC; i += kThreads) z_s[i] = (k0 + i < K) ? st[(long long)K * DV + k0 + i] : 0.f;
    };

    for (int c0 = r_begin; c0 < r_end; c0 += C) {
        const int nr = min(C, r_end - c0);
        if (causal) {
            for (int i = tid; i < C * DV / 4; i += kThreads) {
                const int r = i / (DV / 4), c = (i % (DV / 4)) * 4;
                float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < nr) val = load4(v, (bh * N + c0 + r) * DV + c, v_bf16);
                *reinterpret_cast<float4 *>(v_s + r * DV + c) = val;
            }
        }
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
            stage_g(gq_s, gq, c0, nr, k0);
            if (causal) stage_g(gk_s, gk, c0, nr, k0);
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
                for (int j = 0; j < TN; ++j) b[j] = s_s[kk * DV + tn * TN + j];
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
                for (int j = 0; j < TN; ++j) b[j] = v_s[jj * DV + tn * TN + j];
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
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            const int r = tm * TM + i;
            if (r < nr) {
                const float dn = den_s[r];
#pragma unroll
                for (int j = 0; j < TN; ++j) out[(bh * N + c0 + r) * DV + tn * TN + j] = acc[i][j] / dn;
            }
        }
        if (causal) {
            for (int kt = 0; kt < ktiles; ++kt) {
                const int k0 = kt * KC;
                stage_g(gk_s, gk, c0, nr, k0);
                stage_s(k0);
                __syncthreads();
                float u[TU][TN];
#pragma unroll
                for (int i = 0; i < TU; ++i)
#pragma unroll
                    for (int j = 0; j < TN; ++j) u[i][j] = s_s[(tm * TU + i) * DV + tn * TN + j];
                for (int jj = 0; jj < C; ++jj) {
                    float a[TU], b[TN];
#pragma unroll
                    for (int i = 0; i < TU; ++i) a[i] = gk_s[jj * LG + tm * TU + i];
#pragma unroll
                    for (int j = 0; j < TN; ++j) b[j] = v_s[jj * DV + tn * TN + j];
#pragma unroll
                    for (int i = 0; i < TU; ++i)
#pragma unroll
                        for (int j = 0; j < TN; ++j) u[i][j] = fmaf(a[i], b[j], u[i][j]);
                }
#pragma unroll
                for (int i = 0; i < TU; ++i) {
                    const int k = k0 + tm * TU + i;
                    if (k < K)
#pragma unroll
                        for (int j = 0; j < TN; ++j) st[(long long)k * DV + tn * TN + j] = u[i][j];
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
    (void)SZ;
}

template <int DV>
cudaError_t launch_block_state_dv(const Dims &dm, const void *gk, const void *v, float *partial, cudaStream_t st)
{
    dim3 grid(dm.nblk(), (unsigned)dm.BH(), (dm.K + 127) / 128);
    k_block_state<DV><<<grid, kThreads, 0, st>>>(dm.N, dm.K, dm.KP, gk, dm.g_bf16, v, dm.v_bf16, partial,
                                                 dm.nblk());
    return cudaGetLastError();
}

template <int DV, int C>
cudaError_t launch_chunk_out_c(const Dims &dm, bool causal, const void *gq, const void *gk, const void *v,
                               float *states, float *out, cudaStream_t st)
{
    constexpr size_t smem = ChunkSmem<DV, C>::bytes;
    static std::atomic<unsigned long long> smem_set{0};
    const cudaError_t attr = allow_smem(k_chunk_out<DV, C>, smem, smem_set);
    if (attr != cudaSuccess) return attr;
    const long long SZ = dm.state_size();
    const long long bh_stride = causal ? (long long)dm.nblk() * SZ : SZ;
    const long long blk_stride = causal ? SZ : 0;
    dim3 grid(dm.nblk(), (unsigned)dm.BH());
    k_chunk_out<DV, C><<<grid, kThreads, smem, st>>>(dm.N, dm.K, dm.KP, causal, dm.eps, gq, gk, dm.g_bf16, v,
                                                     dm.v_bf16, states, bh_stride, blk_stride, out);
    return cudaGetLastError();
}

template <int DV>
cudaError_t launch_chunk_out_dv(const Dims &dm, bool causal, const void *gq, const void *gk, const void *v,
                                float *states, float *out, cudaStream_t st)
{
    switch (dm.C) {
    case 16: return launch_chunk_out_c<DV, 16>(dm, causal, gq, gk, v, states, out, st);
    case 32: return launch_chunk_out_c<DV, 32>(dm, causal, gq, gk, v, states, out, st);
    case 64: return launch_chunk_out_c<DV, 64>(dm, causal, gq, gk, v, states, out, st);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace

cudaError_t launch_block_state(const Dims &dm, const void *gk, const void *v, float *partial, cudaStream_t st)
{
    switch (dm.DV) {
    case 16: return launch_block_state_dv<16>(dm, gk, v, partial, st);
    case 32: return launch_block_state_dv<32>(dm, gk, v, partial, st);
    case 64: return launch_block_state_dv<64>(dm, gk, v, partial, st);
    case 128: return launch_block_state_dv<128>(dm, gk, v, partial, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_scan(const Dims &dm, float *partial, const float *state_in, float *total, bool exclusive,
                        cudaStream_t st, bool total_in_block_layout)
{
    const long long SZ = dm.state_size();
    dim3 grid((unsigned)((SZ + kThreads - 1) / kThreads), (unsigned)dm.BH());
    const bool tr = tc_path_applies(dm) && !total_in_block_layout;
    k_scan<<<grid, kThreads, 0, st>>>(SZ, dm.nblk(), partial, state_in, total, exclusive, tr ? dm.K : 0,
                                      tr ? dm.DV : 0);
    return cudaGetLastError();
}

cudaError_t launch_chunk_out(const Dims &dm, bool causal, const void *gq, const void *gk, const void *v,
                             float *states, float *out, cudaStream_t st)
{
    switch (dm.DV) {
    case 16: return launch_chunk_out_dv<16>(dm, causal, gq, gk, v, states, out, st);
    case 32: return launch_chunk_out_dv<32>(dm, causal, gq, gk, v, states, out, st);
    case 64: return launch_chunk_out_dv<64>(dm, causal, gq, gk, v, states, out, st);
    case 128: return launch_chunk_out_dv<128>(dm, causal, gq, gk, v, states, out, st);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace gma
