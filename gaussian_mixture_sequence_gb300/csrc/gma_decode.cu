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

// One CTA per (b, h).  The kernel is launched as a programmatic dependent of the
// parameter preparation, whose results it reads only after griddepcontrol.wait
// (the token rows it reads first were written before the preparation kernel
// started), so that the preparation overlaps its start.  The log-joints of the new
// token's q and k rows: a warp per component row of parameters at a time
// (coalesced, shared by both rows, sums over the warp by shuffles); then the two
// softmaxes, a warp each; then one pass over the state that updates and reads
// it, four columns per thread with 16-byte accesses (a scalar pass when K is not
// a multiple of 4, where the slices of the state are not 16-byte aligned).
template <int D, int DV>
__global__ void __launch_bounds__(kThreads, 6)
    k_decode(int H, int K, float eps, const void *__restrict__ qx, const void *__restrict__ kx, bool x_bf16,
             const void *__restrict__ v, bool v_bf16, const float4 *__restrict__ prm,
             const float *__restrict__ cst, float *__restrict__ state, float *__restrict__ out)
{
    extern __shared__ __align__(16) float sm[];
    float *xq = sm;            // [D]
    float *xk = xq + D;        // [D]
    float *vv = xk + D;        // [DV]
    float *gq = vv + DV;       // [K]
    float *gk = gq + K;        // [K]
    float *dz = gk + K;        // [kThreads / 32] den partials
    // then, 16-byte aligned: red4 [kThreads] followed by red [kThreads]
    float4 *red4 = reinterpret_cast<float4 *>((reinterpret_cast<uintptr_t>(dz + kThreads / 32) + 15) & ~uintptr_t(15));
    float *red = reinterpret_cast<float *>(red4 + kThreads);

    const long long bh = blockIdx.x;
    const int h = (int)(bh % H), tid = threadIdx.x;
    // the state of this slice: thread t updates column group t % G4 of rows t / G4 + j RP
    constexpr int G4 = DV / 4, RP = kThreads / G4, U = 4;
    const bool vec = (K & 3) == 0;   // 16-byte aligned slices
    const int c4 = tid % G4, r0 = tid / G4;
    float *st = state + bh * ((long long)K * DV + K);
    float4 *st4 = reinterpret_cast<float4 *>(st);
    const int total = K * DV;
    for (int i = tid; i < D; i += kThreads) {
        xq[i] = load_elem(qx, bh * D + i, x_bf16);
        xk[i] = load_elem(kx, bh * D + i, x_bf16);
    }
    for (int i = tid; i < DV; i += kThreads) vv[i] = load_elem(v, bh * DV + i, v_bf16);
    // the prepared parameters are written by the preceding kernel (programmatic launch)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __syncthreads();

    // log-joints -1/2 sum_d ((x_d - mu_d) / sigma_d)^2 + c_k of both rows.  A warp takes a
    // component's parameter row with consecutive lanes on consecutive words (one coalesced
    // read serves both rows), and its partial sums meet by shuffles.
    {
        constexpr int DP = D / 2;
        constexpr int LPC = DP < 32 ? DP : 32;   // lanes per component (a power of two)
        constexpr int CPW = 32 / LPC;            // components per warp and pass
        constexpr int WPL = DP / LPC;            // parameter words per lane
        constexpr int STEP = (kThreads / 32) * CPW, PB = WPL > 1 ? 2 : 4;   // passes whose reads overlap
        const int warp = tid >> 5, lane = tid & 31, sub = lane / LPC, l = lane % LPC;
        const float4 *ph = prm + (long long)h * K * DP;
        float2 xqr[WPL], xkr[WPL];   // this lane's features: the same for every component
#pragma unroll
        for (int w = 0; w < WPL; ++w) {
            const int dp = l + w * LPC;
            xqr[w] = *reinterpret_cast<const float2 *>(xq + 2 * dp);
            xkr[w] = *reinterpret_cast<const float2 *>(xk + 2 * dp);
        }
        for (int kb = warp * CPW + sub; kb < K + sub; kb += STEP * PB) {
            float4 pw[PB][WPL];
#pragma unroll
            for (int b = 0; b < PB; ++b)
#pragma unroll
                for (int w = 0; w < WPL; ++w) {
                    const int k = kb + b * STEP;
                    pw[b][w] = k < K ? ph[(long long)k * DP + l + w * LPC] : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            // the lane's partial sums: v[2 b] for the q row, v[2 b + 1] for the k row of pass b
            float v[2 * PB];
#pragma unroll
            for (int b = 0; b < PB; ++b) {
                float aq = 0.f, ak = 0.f;
#pragma unroll
                for (int w = 0; w < WPL; ++w) {
                    const float4 p = pw[b][w];
                    float y = fmaf(xqr[w].x, p.x, p.z);
                    aq = fmaf(y, y, aq);
                    y = fmaf(xqr[w].y, p.y, p.w);
                    aq = fmaf(y, y, aq);
                    y = fmaf(xkr[w].x, p.x, p.z);
                    ak = fmaf(y, y, ak);
                    y = fmaf(xkr[w].y, p.y, p.w);
                    ak = fmaf(y, y, ak);
                }
                v[2 * b] = aq;
                v[2 * b + 1] = ak;
            }
            if constexpr (LPC == 32) {
                // sums over the warp by recursive halving: each step a lane keeps half of its
                // values and adds the partner's copy of them, so that lane l ends with value
                // (l >> (5 - S)) over the lanes that differ in the top S bits, S = log2(2 PB),
                // and the last 5 - S steps add the rest
                constexpr int NV = 2 * PB, S = NV == 8 ? 3 : 2;
                int n = NV;
#pragma unroll
                for (int o = 16; o > (16 >> S); o >>= 1) {
                    const bool up = (lane & o) != 0;
                    n >>= 1;
#pragma unroll
                    for (int e = 0; e < NV / 2; ++e)
                        if (e < n) {
                            const float send = up ? v[e] : v[e + n], keep = up ? v[e + n] : v[e];
                            v[e] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                        }
                }
                float t = v[0];
#pragma unroll
                for (int o = 16 >> S; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                const int idx = lane >> (5 - S), k = kb + (idx >> 1) * STEP;
                if ((lane & ((32 >> S) - 1)) == 0 && k < K)
                    (idx & 1 ? gk : gq)[k] = fmaf(-0.5f, t, cst[(long long)h * K + k]);
            } else {
#pragma unroll
                for (int b = 0; b < PB; ++b) {
                    const int k = kb + b * STEP;
                    float aq = v[2 * b], ak = v[2 * b + 1];
#pragma unroll
                    for (int o = LPC / 2; o; o >>= 1) {
                        aq += __shfl_xor_sync(0xffffffffu, aq, o);
                        ak += __shfl_xor_sync(0xffffffffu, ak, o);
                    }
                    if (k < K && l == 0) {
                        const float c = cst[(long long)h * K + k];
                        gq[k] = fmaf(-0.5f, aq, c);
                        gk[k] = fmaf(-0.5f, ak, c);
                    }
                }
            }
        }
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < 2) {   // the two softmaxes: warp 0 the q row, warp 1 the k row
        float *gr = warp ? gk : gq;
        float m = -FLT_MAX;
        for (int k = lane; k < K; k += 32) m = fmaxf(m, gr[k]);
#pragma unroll
        for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float sum = 0.f;
        for (int k = lane; k < K; k += 32) {
            const float e = expf(gr[k] - m);
            gr[k] = e;
            sum += e;
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        const float inv = 1.0f / sum;
        for (int k = lane; k < K; k += 32) gr[k] *= inv;
    }
    __syncthreads();

    // Vt[k][c] += gk[k] v[c]; num[c] += gq[k] Vt_new[k][c]; Z[k] += gk[k]; den += gq[k] Z_new[k]
    // (den: a partial per warp, added up by the threads that write the output)
    {
        float dp = 0.f;
        for (int k = tid; k < K; k += kThreads) {
            const float z = st[total + k] + gk[k];
            st[total + k] = z;
            dp = fmaf(gq[k], z, dp);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) dp += __shfl_xor_sync(0xffffffffu, dp, o);
        if (lane == 0) dz[warp] = dp;
    }
    auto den_total = [&]() {   // after a barrier
        float d = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) d += dz[w];
        return d;
    };
    if (vec) {
        const float4 vc = reinterpret_cast<const float4 *>(vv)[c4];
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
        auto row = [&](int k, float4 t) {
            const float a = gk[k], b = gq[k];
            t.x = fmaf(a, vc.x, t.x);
            t.y = fmaf(a, vc.y, t.y);
            t.z = fmaf(a, vc.z, t.z);
            t.w = fmaf(a, vc.w, t.w);
            st4[k * G4 + c4] = t;
            num.x = fmaf(b, t.x, num.x);
            num.y = fmaf(b, t.y, num.y);
            num.z = fmaf(b, t.z, num.z);
            num.w = fmaf(b, t.w, num.w);
        };
        for (int k0 = r0; k0 < K; k0 += U * RP) {   // U rows at a time: the loads of a batch first
            float4 t[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (k0 + u * RP < K) t[u] = st4[(k0 + u * RP) * G4 + c4];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (k0 + u * RP < K) row(k0 + u * RP, t[u]);
        }
        red4[tid] = num;
        __syncthreads();
        if (tid < DV) {
            float n = 0.f;
            for (int r = 0; r < RP; ++r) {
                const float4 q = red4[r * G4 + tid / 4];
                n += (tid & 3) == 0 ? q.x : (tid & 3) == 1 ? q.y : (tid & 3) == 2 ? q.z : q.w;
            }
            out[bh * DV + tid] = n / (den_total() + eps);
        }
    } else {   // thread t owns column t % DV
        const int c = tid % DV;
        const float vc = vv[c];
        float num = 0.f;
        int e = tid;
        for (; e + 3 * kThreads < total; e += 4 * kThreads) {
            float sv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) sv[u] = st[e + u * kThreads];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int k = (e + u * kThreads) / DV;
                sv[u] = fmaf(gk[k], vc, sv[u]);
                st[e + u * kThreads] = sv[u];
                num = fmaf(gq[k], sv[u], num);
            }
        }
        for (; e < total; e += kThreads) {
            const int k = e / DV;
            const float sv = fmaf(gk[k], vc, st[e]);
            st[e] = sv;
            num = fmaf(gq[k], sv, num);
        }
        __syncthreads();
        red[tid] = num;
        __syncthreads();
        if (tid < DV) {
            float n = 0.f;
            for (int t = tid; t < kThreads; t += DV) n += red[t];
            out[bh * DV + tid] = n / (den_total() + eps);
        }
    }
}

template <int D, int DV>
cudaError_t launch_decode_dv(const Dims &dm, const float4 *prm, const float *cst, const void *qx, const void *kx,
                             const void *v, float *state, float *out, cudaStream_t st)
{
    // xq, xk, v, gq, gk, dz, then at a 16-byte aligned offset red4 and red
    const size_t head = ((size_t)(2 * dm.D + DV + 2 * dm.K + kThreads / 32) * 4 + 15) / 16 * 16;
    const size_t smem = head + (size_t)kThreads * 20;
    // a programmatic dependent of the preceding launch (the parameter preparation)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)dm.BH());
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_decode<D, DV>, dm.H, dm.K, dm.eps, qx, kx, dm.x_bf16, v, dm.v_bf16, prm, cst,
                              state, out);
}

template <int D>
cudaError_t launch_decode_d(const Dims &dm, const float4 *prm, const float *cst, const void *qx, const void *kx,
                            const void *v, float *state, float *out, cudaStream_t st)
{
    switch (dm.DV) {
    case 16: return launch_decode_dv<D, 16>(dm, prm, cst, qx, kx, v, state, out, st);
    case 32: return launch_decode_dv<D, 32>(dm, prm, cst, qx, kx, v, state, out, st);
    case 64: return launch_decode_dv<D, 64>(dm, prm, cst, qx, kx, v, state, out, st);
    case 128: return launch_decode_dv<D, 128>(dm, prm, cst, qx, kx, v, state, out, st);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace



cudaError_t launch_decode(const Dims &dm, const float4 *prm, const float *cst, const void *qx, const void *kx,
                          const void *v, float *state, float *out, cudaStream_t st)
{
    switch (dm.D) {
    case 16: return launch_decode_d<16>(dm, prm, cst, qx, kx, v, state, out, st);
    case 32: return launch_decode_d<32>(dm, prm, cst, qx, kx, v, state, out, st);
    case 64: return launch_decode_d<64>(dm, prm, cst, qx, kx, v, state, out, st);
    case 128: return launch_decode_d<128>(dm, prm, cst, qx, kx, v, state, out, st);
    default: return cudaErrorInvalidValue;
    }
}

} // namespace gma
