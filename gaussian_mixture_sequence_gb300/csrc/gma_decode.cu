// One recurrent decode step (S5): the causal GMA form advanced by one token.
//
// Per (b, h): gamma_q and gamma_k of the new token (the posterior of
// "핵심 메커니즘"), then the memory update Vt += gamma_k v^T, Z += gamma_k,
// then the read o = gamma_q Vt / (gamma_q Z + eps).  The memory of every head
// is a constant-size state, as the linear-attention page ("선형 어텐션 원리
// 정리", "쉽게 이해하기") describes for recurrent inference; streaming it once
// in and once out of HBM is the whole cost of the step.
#include "gma_internal.cuh"

#include <float.h>

namespace gma {
namespace {

__device__ __forceinline__ float block_reduce(float v, float *red, bool is_max)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float t = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmaxf(v, t) : v + t;
    }
    __syncthreads(); // red may still be read from a previous reduction
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float r = red[0];
    for (int w = 1; w < kThreads / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
    return r;
}

template <int DV>
__global__ void __launch_bounds__(kThreads)
    k_decode(int H, int D, int K, float eps, const void *__restrict__ qx, const void *__restrict__ kx, bool x_bf16,
             const void *__restrict__ v, bool v_bf16, const float4 *__restrict__ prm,
             const float *__restrict__ cst, float *__restrict__ state, float *__restrict__ out)
{
    extern __shared__ __align__(16) float sm[];
    float *xq = sm;            // [D]
    float *xk = xq + D;        // [D]
    float *vv = xk + D;        // [DV]
    float *gq = vv + DV;       // [K]
    float *gk = gq + K;        // [K]
    float *red = gk + K;       // [kThreads]

    const long long bh = blockIdx.x;
    const int h = (int)(bh % H), tid = threadIdx.x;
    for (int i = tid; i < D; i += kThreads) {
        xq[i] = load_elem(qx, bh * D + i, x_bf16);
        xk[i] = load_elem(kx, bh * D + i, x_bf16);
    }
    for (int i = tid; i < DV; i += kThreads) vv[i] = load_elem(v, bh * DV + i, v_bf16);
    __syncthreads();

    float mq = -FLT_MAX, mk = -FLT_MAX;
    for (int k = tid; k < K; k += kThreads) {
        const float4 *pk = prm + ((long long)h * K + k) * (D / 2);
        float aq = 0.f, ak = 0.f;
        for (int dp = 0; dp < D / 2; ++dp) {
            const float4 p = pk[dp];
            float y = fmaf(xq[2 * dp], p.x, p.z);
            aq = fmaf(y, y, aq);
            y = fmaf(xq[2 * dp + 1], p.y, p.w);
            aq = fmaf(y, y, aq);
            y = fmaf(xk[2 * dp], p.x, p.z);
            ak = fmaf(y, y, ak);
            y = fmaf(xk[2 * dp + 1], p.y, p.w);
            ak = fmaf(y, y, ak);
        }
        const float c = cst[(long long)h * K + k];
        gq[k] = fmaf(-0.5f, aq, c);
        gk[k] = fmaf(-0.5f, ak, c);
        mq = fmaxf(mq, gq[k]);
        mk = fmaxf(mk, gk[k]);
    }
    mq = block_reduce(mq, red, true);
    mk = block_reduce(mk, red, true);
    float sq = 0.f, sk = 0.f;
    for (int k = tid; k < K; k += kThreads) {
        gq[k] = expf(gq[k] - mq);
        gk[k] = expf(gk[k] - mk);
        sq += gq[k];
        sk += gk[k];
    }
    sq = block_reduce(sq, red, false);
    sk = block_reduce(sk, red, false);
    const float iq = 1.0f / sq, ik = 1.0f / sk;
    for (int k = tid; k < K; k += kThreads) {
        gq[k] *= iq;
        gk[k] *= ik;
    }
    __syncthreads();

    // Vt[k][c] += gk[k] v[c]; num[c] += gq[k] Vt_new[k][c].  Thread t always owns column t % DV.
    float *st = state + bh * ((long long)K * DV + K);
    const int c = tid % DV;
    const float vc = vv[c];
    float num = 0.f;
    const int total = K * DV;
    int e = tid;
    for (; e + 3 * kThreads < total; e += 4 * kThreads) {
        float s[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) s[u] = st[e + u * kThreads];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int k = (e + u * kThreads) / DV;
            s[u] = fmaf(gk[k], vc, s[u]);
            st[e + u * kThreads] = s[u];
            num = fmaf(gq[k], s[u], num);
        }
    }
    for (; e < total; e += kThreads) {
        const int k = e / DV;
        const float s = fmaf(gk[k], vc, st[e]);
        st[e] = s;
        num = fmaf(gq[k], s, num);
    }
    float den = 0.f;
    for (int k = tid; k < K; k += kThreads) {
        const float z = st[total + k] + gk[k];
        st[total + k] = z;
        den = fmaf(gq[k], z, den);
    }
    den = block_reduce(den, red, false);
    __syncthreads();
    red[tid] = num;
    __syncthreads();
    if (tid < DV) {
        float n = 0.f;
        for (int t = tid; t < kThreads; t += DV) n += red[t];
        out[bh * DV + tid] = n / (den + eps);
    }
}

template <int DV>
cudaError_t launch_decode_dv(const Dims &dm, const float4 *prm, const float *cst, const void *qx, const void *kx,
                             const void *v, float *state, float *out, cudaStream_t st)
{
    const size_t smem = (size_t)(2 * dm.D + DV + 2 * dm.K + kThreads) * 4;
    k_decode<DV><<<(unsigned)dm.BH(), kThreads, smem, st>>>(dm.H, dm.D, dm.K, dm.eps, qx, kx, dm.x_bf16, v,
                                                            dm.v_bf16, prm, cst, state, out);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_decode(const Dims &dm, const float4 *prm, const float *cst, const void *qx, const void *kx,
                          const void *v, float *state, float *out, cudaStream_t st)
{
    switch (dm.DV) {
    case 16: return launch_decode_dv<16>(dm, prm, cst, qx, kx, v, state, out, st);
    case 32: return launch_decode_dv<32>(dm, prm, cst, qx, kx, v, state, out, st);
    case 64: return launch_decode_dv<64>(dm, prm, cst, qx, kx, v, state, out, st);
    case 128: return launch_decode_dv<128>(dm, prm, cst, qx, kx, v, state, out, st);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace gma
