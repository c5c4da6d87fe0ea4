// Responsibility diagnostics: a reduction over Gamma.
//
// The explainer page ("Gaussian Mixture Attention: Linear-Time Sequence Mixing
// via Probabilistic Latent Routing", "결과 및 성능", interpretability) reads the
// learned responsibilities as a diagnostic object: how many components are in
// use, the entropy of their usage, and the hard assignment argmax_k gamma_ik of
// every token.  Per head h, over all B*N rows of that head:
//   usage[h][k]   = sum_i gamma_ik                    (soft usage)
//   counts[h][k]  = #{i : argmax_k gamma_ik = k}      (hard assignments, lowest k on ties)
//   entropy[h][0] = H(usage[h] / sum usage[h]) / log K, entropy[h][1] the same for counts
//   assign[b][h][i] = argmax_k gamma_ik               (optional)
// Every sum runs in a fixed order (per-thread serial sums over a block's rows,
// then over blocks and batch entries in order, then a fixed tree), so repeated
// calls give identical bits; the counts are integers.
#include "gma_internal.cuh"

#include <float.h>

namespace gma {
namespace {

constexpr int kStatRows = 1024;   // rows of one block of the partial pass

// Partial sums of one block of kStatRows rows of slice bh:
//   pu[bh][blk][k] = sum over the block's rows of gamma_ik
//   pc[bh][blk][k] = number of the block's rows whose argmax is k
// Thread t sums components t, t + 256 (coalesced row reads); warp w finds the
// argmax of rows w, w + 8, ... (lanes over components, then a shuffle reduction
// that keeps the lowest component among equal values).
__global__ void __launch_bounds__(kThreads) k_usage_partial(int N, int K, int ldg, const float *__restrict__ gamma,
                                                            float *__restrict__ pu, int *__restrict__ pc,
                                                            int *__restrict__ assign, int nblk)
{
    __shared__ int cnt[512];
    const long long bh = blockIdx.y;
    const int blk = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = blk * kStatRows, r1 = min(N, r0 + kStatRows);
    for (int k = tid; k < K; k += kThreads) cnt[k] = 0;
    __syncthreads();
    const float *g = gamma + (bh * N) * (long long)ldg;
    float s0 = 0.f, s1 = 0.f;
    for (int r = r0; r < r1; ++r) {
        const float *row = g + (long long)r * ldg;
        if (tid < K) s0 += row[tid];
        if (tid + kThreads < K) s1 += row[tid + kThreads];
    }
    for (int r = r0 + warp; r < r1; r += kThreads / 32) {
        const float *row = g + (long long)r * ldg;
        float best = -FLT_MAX;
        int arg = 0x7fffffff;
        for (int k = lane; k < K; k += 32) {
            const float v = row[k];
            if (v > best) {   // ascending k per lane: the first maximum is kept
                best = v;
                arg = k;
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            const float ob = __shfl_xor_sync(0xffffffffu, best, o);
            const int oa = __shfl_xor_sync(0xffffffffu, arg, o);
            if (ob > best || (ob == best && oa < arg)) {
                best = ob;
                arg = oa;
            }
        }
        if (lane == 0) {
            atomicAdd(&cnt[arg], 1);
            if (assign) assign[bh * N + r] = arg;
        }
    }
    __syncthreads();
    const long long o = (bh * nblk + blk) * (long long)K;
    if (tid < K) {
        pu[o + tid] = s0;
        pc[o + tid] = cnt[tid];
    }
    if (tid + kThreads < K) {
        pu[o + tid + kThreads] = s1;
        pc[o + tid + kThreads] = cnt[tid + kThreads];
    }
}

// Sum of one value per thread over the CTA in a fixed tree order.
__device__ float block_sum(float v, float *red)
{
    const int tid = threadIdx.x;
    red[tid] = v;
    __syncthreads();
    for (int s = kThreads / 2; s > 0; s >>= 1) {
        if (tid < s) red[tid] += red[tid + s];
        __syncthreads();
    }
    const float r = red[0];
    __syncthreads();
    return r;
}

// One CTA per head: the head's slices (b = 0 .. B-1) and blocks in order, then the
// two normalised entropies.
__global__ void __launch_bounds__(kThreads) k_usage_final(int B, int H, int K, int nblk, const float *__restrict__ pu,
                                                          const int *__restrict__ pc, float *__restrict__ usage,
                                                          long long *__restrict__ counts, float *__restrict__ entropy)
{
    __shared__ float red[kThreads];
    const int h = blockIdx.x, tid = threadIdx.x;
    float u[2] = {0.f, 0.f}, c[2] = {0.f, 0.f};
    for (int j = 0; j < 2; ++j) {
        const int k = tid + j * kThreads;
        if (k >= K) continue;
        long long n = 0;
        for (int b = 0; b < B; ++b) {
            const long long bh = (long long)b * H + h;
            for (int blk = 0; blk < nblk; ++blk) {
                const long long o = (bh * nblk + blk) * (long long)K + k;
                u[j] += pu[o];
                n += pc[o];
            }
        }
        usage[(long long)h * K + k] = u[j];
        counts[(long long)h * K + k] = n;
        c[j] = (float)n;
    }
    // entropy of w / sum w, divided by log K (0 for K = 1 or w = 0); 0 log 0 = 0
    const float su = block_sum(u[0] + u[1], red), sc = block_sum(c[0] + c[1], red);
    float eu = 0.f, ec = 0.f;
    for (int j = 0; j < 2; ++j) {
        if (su > 0.f && u[j] > 0.f) eu -= (u[j] / su) * logf(u[j] / su);
        if (sc > 0.f && c[j] > 0.f) ec -= (c[j] / sc) * logf(c[j] / sc);
    }
    eu = block_sum(eu, red);
    ec = block_sum(ec, red);
    if (tid == 0) {
        const float lk = K > 1 ? logf((float)K) : 1.f;
        entropy[2 * h] = K > 1 && su > 0.f ? eu / lk : 0.f;
        entropy[2 * h + 1] = K > 1 && sc > 0.f ? ec / lk : 0.f;
    }
}

} // namespace

int usage_blocks(const Dims &dm) { return (dm.N + kStatRows - 1) / kStatRows; }

cudaError_t launch_usage(const Dims &dm, const float *gamma, int ldg, float *pu, int *pc, int *assign, float *usage,
                         long long *counts, float *entropy, cudaStream_t st)
{
    const int nblk = usage_blocks(dm);
    if (dm.K > 2 * kThreads) return cudaErrorInvalidValue;
    if (nblk > 0) {
        k_usage_partial<<<dim3(nblk, (unsigned)dm.BH()), kThreads, 0, st>>>(dm.N, dm.K, ldg, gamma, pu, pc, assign,
                                                                          nblk);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    k_usage_final<<<dm.H, kThreads, 0, st>>>(dm.B, dm.H, dm.K, nblk, pu, pc, usage, counts, entropy);
    return cudaGetLastError();
}

} // namespace gma
