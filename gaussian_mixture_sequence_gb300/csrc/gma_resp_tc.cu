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
//   |l~_ik - l_ik| <= delta_i = U (1/2 A sum_d x_d^2 + M sum_d |x_d|) + 1e-3,
// U = 4e-3, A = max_kd a_kd, M = max_kd |a_kd mu_kd| over the head, and
// sum_d |x_d| <= 8 (sum_d x_d^2)^(1/2) (Cauchy-Schwarz, d = 64).  Component k
// is kept when l~_ik >= max_j l~_ij - T - 2 delta_i, which keeps every
// component within T of the true maximum.  The kept components get the same
// exact fp32 evaluation as the dense kernel (one packed FMA for (x - mu)/sigma,
// one for the square-accumulate, per feature pair).
//
// One persistent CTA per SM, 16 warps in two groups of 8 that take alternate
// tiles of 128 rows, so that one group's tensor-core, TMA and barrier waits
// overlap the other's arithmetic.  In a group, the two warps 4h + w' share the
// TMEM lanes 32 w' .. +31 (one row each) and take component half h.  The
// per-head bound matrix and constants are built once per call by
// k_prep_all and bulk-copied into shared memory (both groups work on the
// same head: the CTA's range is walked run by run); the exact parameters,
// needed only by rows with two or more kept components, are read from global
// memory (L2-resident).  Routing tiles arrive by TMA into one buffer that the
// groups consume in item order (the consumer of tile n fetches tile n + 1);
// each group assembles its output tile in its own buffer, which leaves by TMA
// stores.
#include "gma_internal.cuh"
#include "gma_tc.cuh"

#include <float.h>

namespace gma {
namespace {

using namespace tc;

constexpr int kPK = 128, kPD = 64, kPDP = kPD / 2;
constexpr int kPThreads = 512, kPRows = 128;
constexpr int kPGroups = 2, kPGThreads = kPThreads / kPGroups;
constexpr int kPRun = 16;                      // tiles of a slice taken in a row
constexpr int kPStride = kPDP + 1;            // padded float4 row of exact parameters
constexpr float kPT = 30.f;                   // log-joint window kept exactly
constexpr float kPU = 4.0e-3f;                // bf16 product + fp32 accumulation bound
// A tile is left to the dense kernel when at least kDenseRows of its (row, component half)
// pairs keep kDenseKept or more of the half's 64 components.
constexpr int kDenseKept = 8, kDenseRows = 64;

// Shared memory: the bound matrix, the routing tile, each group's output tile,
// the constants c, c', A, M, each group's exchange slots between the two
// halves of a row, the mbarriers (images, routing tile, each group's MMA), and
// each warp's copy of one component's exact parameters.
struct PrunedSmem {
    static constexpr uint32_t W = kPrunedWBytes;                        // bf16 [128][128], SW128
    static constexpr uint32_t X = kPRows * kPD * 4;                     // routing tile (fp32 worst case)
    static constexpr uint32_t O = kPRows * kPK * 4;                     // output tile (fp32 worst case)
    static constexpr uint32_t C = kPrunedCBytes;                        // c, c', A, M
    static constexpr uint32_t EX = 3 * 2 * kPK * 4;                     // [3][2][128] per group
    static constexpr uint32_t PW = kPDP * 16;                           // one component's parameters
    static constexpr size_t bytes =
        1024 + W + X + kPGroups * (size_t)O + C + kPGroups * (size_t)EX + 64 + (kPThreads / 32) * (size_t)PW;
};
static_assert(PrunedSmem::bytes <= 232448, "routing kernel: shared memory above the per-block limit");

// Named barrier of one group (ids 1, 2; id 0 is __syncthreads).
__device__ __forceinline__ void group_sync(int g)
{
    asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(kPGThreads) : "memory");
}
// Named barrier of one group that also returns the OR of `pred` over its threads.
__device__ __forceinline__ bool group_or(int g, bool pred)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)pred), "r"(1 + g), "r"(kPGThreads)
                 : "memory");
    return r != 0;
}

// Named barrier of one group that also returns how many of its threads have `pred` set.
__device__ __forceinline__ uint32_t group_popc(int g, bool pred)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.popc.u32 %0, %2, %3, p;\n\t}"
                 : "=r"(r)
                 : "r"((uint32_t)pred), "r"(1 + g), "r"(kPGThreads)
                 : "memory");
    return r;
}

__device__ __forceinline__ uint32_t pack2(float a, float b)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}


// The per-head parameters and the images of the bounded routing in one pass
// (K = 128, d = 64): CTA (h, q) takes the 32 components [32 q, 32 q + 32) of head h,
// 16 threads per component (4 features each).
//   prm[k][dp] = {s_2dp, s_2dp+1, -mu_2dp s_2dp, -mu_2dp+1 s_2dp+1}, s = 1/sigma, sigma^2 = softplus(r)
//   cst[k]     = log pi_k - 1/2 sum_d log sigma^2_kd, pi = softmax(logit_pi)
// and W, the padded parameters and c, c', A_k, M_k (the component's largest a = s^2 and
// |a mu|; the routing kernel takes the head-wide maxima when it loads the images), and W
// again as three bf16 planes in the operand order of the dense tensor-core pass (below).
constexpr int kPrepAllThreads = 512, kPrepAllComps = kPrepAllThreads / 16;

__device__ __forceinline__ float softplus_f(float r) { return fmaxf(r, 0.f) + log1pf(expf(-fabsf(r))); }

// v = p0 + p1 + p2 + r with p0, p1, p2 bf16 and |r| <= 2^-24 |v|: each plane is the
// round-to-nearest of what the previous ones leave, and each difference is exact in fp32.
__device__ __forceinline__ void split3(float v, unsigned short (&p)[3])
{
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        p[j] = __bfloat16_as_ushort(b);
        v -= __bfloat162float(b);
    }
}

// Operand position of feature f's square in the dense tensor-core pass; its value sits 16
// positions later.  Column quarter q of the operand holds the squares of features
// 16 q .. 16 q + 15, then their values.
__host__ __device__ constexpr int dtc_pos(int f) { return 32 * (f >> 4) + (f & 15); }

__global__ void __launch_bounds__(kPrepAllThreads)
    k_prep_all(const float *__restrict__ mu, const float *__restrict__ var_raw, const float *__restrict__ logit_pi,
               float4 *__restrict__ prm, float *__restrict__ cst, unsigned char *__restrict__ wimg,
               unsigned char *__restrict__ wimg3, float4 *__restrict__ pimg, float *__restrict__ cimg,
               float4 *__restrict__ pimg2, unsigned int *__restrict__ dctl)
{
    constexpr int NW = kPrepAllThreads / 32;
    __shared__ float red[2][NW];
    __shared__ float lmax_s, lse_s;
    const int h = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = blockIdx.y * kPrepAllComps + (tid >> 4), part = tid & 15;   // component, features 4 part ..
    const float *l = logit_pi + (long long)h * kPK;
    if (blockIdx.y == 0 && tid == 0) {   // no tile of this head listed for either dense pass yet
        dctl[h] = 0u;
        dctl[gridDim.x + h] = 0u;
    }

    // log-sum-exp of the head's logits (thread k < K holds logit k)
    const float lv = tid < kPK ? l[tid] : -FLT_MAX;
    float t = lv;
    for (int o = 16; o; o >>= 1) t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (lane == 0) red[0][warp] = t;
    __syncthreads();
    if (warp == 0) {
        float u = lane < NW ? red[0][lane] : -FLT_MAX;
        for (int o = 16; o; o >>= 1) u = fmaxf(u, __shfl_xor_sync(0xffffffffu, u, o));
        if (lane == 0) lmax_s = u;
    }
    __syncthreads();
    t = tid < kPK ? expf(lv - lmax_s) : 0.f;
    for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) red[1][warp] = t;
    __syncthreads();
    if (warp == 0) {
        float u = lane < NW ? red[1][lane] : 0.f;
        for (int o = 16; o; o >>= 1) u += __shfl_xor_sync(0xffffffffu, u, o);
        if (lane == 0) lse_s = lmax_s + logf(u);
    }

    // this thread's 4 features of component k: packed parameters, W, sums and maxima
    const long long row = (long long)h * kPK + k;
    const float4 r4 = *reinterpret_cast<const float4 *>(var_raw + row * kPD + 4 * part);
    const float4 u4 = *reinterpret_cast<const float4 *>(mu + row * kPD + 4 * part);
    const float rv[4] = {r4.x, r4.y, r4.z, r4.w}, uv[4] = {u4.x, u4.y, u4.z, u4.w};
    unsigned char *wh = wimg + (long long)h * kPrunedWBytes;
    float lsum = 0.f, amu2 = 0.f, amax = 0.f, mmax = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const int f = 4 * part + 2 * q, dp = f / 2;
        const float v0 = softplus_f(rv[2 * q]), v1 = softplus_f(rv[2 * q + 1]);
        const float s0 = 1.0f / sqrtf(v0), s1 = 1.0f / sqrtf(v1);
        const float4 p = make_float4(s0, s1, -uv[2 * q] * s0, -uv[2 * q + 1] * s1);
        prm[row * kPDP + dp] = p;
        pimg[row * kPStride + dp] = p;
        pimg2[row * kPDP + 8 * (dp % 4) + dp / 4] = p;   // pair 4 e + j at 8 j + e
        lsum += logf(v0) + logf(v1);
        amu2 = fmaf(p.z, p.z, fmaf(p.w, p.w, amu2));
        amax = fmaxf(amax, fmaxf(p.x * p.x, p.y * p.y));
        mmax = fmaxf(mmax, fmaxf(fabsf(p.x * p.z), fabsf(p.y * p.w)));
        // W row k: -1/2 s^2 at features f, f + 1 and -s (-mu s) at d + f, d + f + 1
        const float wa0 = -0.5f * p.x * p.x, wa1 = -0.5f * p.y * p.y, wb0 = -p.x * p.z, wb1 = -p.y * p.w;
        *reinterpret_cast<uint32_t *>(wh + sw128_offset(k, f, kPK, 2)) = pack2(wa0, wa1);
        *reinterpret_cast<uint32_t *>(wh + sw128_offset(k, kPD + f, kPK, 2)) = pack2(wb0, wb1);
        // the same row as three planes, squares' weights at dtc_pos(f), values' 16 later
        unsigned short a0[3], a1[3], b0[3], b1[3];
        split3(wa0, a0);
        split3(wa1, a1);
        split3(wb0, b0);
        split3(wb1, b1);
        unsigned char *w3 = wimg3 + (long long)h * kPrunedW3Bytes;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            unsigned char *pl = w3 + j * kPrunedWBytes;
            *reinterpret_cast<uint32_t *>(pl + sw128_offset(k, dtc_pos(f), kPK, 2)) =
                (uint32_t)a0[j] | ((uint32_t)a1[j] << 16);
            *reinterpret_cast<uint32_t *>(pl + sw128_offset(k, dtc_pos(f) + 16, kPK, 2)) =
                (uint32_t)b0[j] | ((uint32_t)b1[j] << 16);
        }
    }
    if (part == 15) pimg[row * kPStride + kPDP] = make_float4(0.f, 0.f, 0.f, 0.f);   // the row's padding word
    for (int o = 1; o < 16; o <<= 1) {   // the component's 16 threads
        lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
        amu2 += __shfl_xor_sync(0xffffffffu, amu2, o);
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
    }
    __syncthreads();   // lse_s
    if (part == 0) {
        float *ch = cimg + (long long)h * 4 * kPK;
        const float c = (l[k] - lse_s) - 0.5f * lsum;
        cst[row] = c;
        ch[k] = c;
        ch[kPK + k] = c - 0.5f * amu2;
        ch[2 * kPK + k] = amax;
        ch[3 * kPK + k] = mmax;
    }
}

// Persistent: CTA b handles the slots [b * per, (b + 1) * per) of the work order
// (runs of tiles of 128 rows, below), run by run; within a run group g takes the
// slots s + g, s + g + 2, ...  The output tile is assembled in shared memory and
// written by TMA stores that stop at the slice's last row.
__global__ void __launch_bounds__(kPThreads, 1)
    k_resp_pruned(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap gmap,
                  const __grid_constant__ CUtensorMap gmap_lo, int N, int H, int BH, bool x_bf16,
                  const unsigned char *__restrict__ wimg, const float4 *__restrict__ pimg,
                  const float *__restrict__ cimg, int layout, int pstride, unsigned int *timeout,
                  int2 *__restrict__ dlist, unsigned int *__restrict__ dctl, long long dcap, int src,
                  unsigned int *__restrict__ zq)
{
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    // a dense pass launched as a programmatic dependent of this kernel may be scheduled as soon as
    // SMs free up; it waits for this grid's completion before it reads the tiles listed here
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = warp >> 3;                    // group
    const int gt = tid - grp * kPGThreads;        // thread in the group
    const int hf = (warp >> 2) & 1;               // component half
    const uint32_t lane0 = 32 * (warp & 3);
    const int i = lane0 + lane;                   // row of the tile (TMEM lane)

    unsigned char *w_s = sm;                                                  // B operand W
    unsigned char *xb = sm + PrunedSmem::W;                                   // routing tile
    unsigned char *ob = xb + PrunedSmem::X + grp * PrunedSmem::O;             // this group's output tile
    float *f_s = reinterpret_cast<float *>(xb + PrunedSmem::X + kPGroups * PrunedSmem::O);
    const float *c_s = f_s, *cp_s = f_s + kPK, *a_s = f_s + 2 * kPK, *m_s = f_s + 3 * kPK;
    float *ex0 = f_s + 4 * kPK + grp * 6 * kPK;   // [2][128] exchange slots between the halves of a row
    float *ex1 = ex0 + 2 * kPK;
    float *ex2 = ex0 + 4 * kPK;
    // images, routing tile for group 0 / 1, MMA of group 0 / 1
    uint64_t *bar = reinterpret_cast<uint64_t *>(f_s + 4 * kPK + kPGroups * 6 * kPK);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 5);
    float4 *pw_s = reinterpret_cast<float4 *>(reinterpret_cast<unsigned char *>(bar) + 64) + warp * kPDP;
    const uint32_t BAR_I = smem_addr(bar), BAR_X = smem_addr(bar + 1 + grp), BAR_M = smem_addr(bar + 3 + grp);

    // Work order: runs of kPRun consecutive tiles of one slice; run r is run r / BH of
    // slice (r % BH) * pstride % BH (pstride coprime with BH), so that consecutive runs
    // come from slices far apart and a CTA's range mixes heads of unequal cost.  A
    // slot v of this order is tile (v % kPRun) of run v / kPRun; slots past a slice's
    // last tile are empty and skipped.
    const int tps = (N + kPRows - 1) / kPRows;    // tiles per slice
    const int rps = (tps + kPRun - 1) / kPRun;    // runs per slice
    const long long slots = (long long)BH * rps * kPRun;
    const long long per = (slots + gridDim.x - 1) / gridDim.x;
    const long long it0 = (long long)blockIdx.x * per;
    const long long it1 = it0 + per < slots ? it0 + per : slots;
    auto run_slice = [&](long long r) { return (int)((r % BH) * (long long)pstride % BH); };
    auto run_tiles = [&](long long r) { return min(kPRun, tps - (int)(r / BH) * kPRun); };   // filled slots
    auto tile_of = [&](long long v) { return (int)((v / kPRun) / BH) * kPRun + (int)(v % kPRun); };
    auto next_filled = [&](long long v) {   // the first filled slot at or after v
        const long long r = v / kPRun;
        return (v % kPRun) < run_tiles(r) ? v : (r + 1) * kPRun;
    };
    const uint32_t xbytes = kPRows * kPD * (x_bf16 ? 2 : 4);
    const bool g_f32 = layout == GL_F32, g_split = layout == GL_SPLIT;
    const int ge = g_f32 ? 4 : 2;
    constexpr uint32_t LO = kPRows * kPK * 2;   // split: the lo plane's tile follows the hi plane's
    // the routing of Q in the split layout records the tiles whose lo plane it leaves unwritten
    const bool zflag = g_split && zq != nullptr && src == 0;

    // one thread: TMA of slot it's rows, counted on the barrier of the group that takes it
    // (group 0 takes a run's first slot in the range, then the groups alternate)
    auto load_x = [&](long long it) {
        const int bh = run_slice(it / kPRun), t = tile_of(it);
        const long long first = max((it / kPRun) * kPRun, it0);
        const uint32_t bx = smem_addr(bar + 1 + (int)((it - first) & 1));
        mbar_expect_tx(bx, xbytes);
        tma_load_3d(smem_addr(xb), &xmap, 0, t * kPRows, bh, bx);
        if (!x_bf16) tma_load_3d(smem_addr(xb + kPRows * 128), &xmap, 32, t * kPRows, bh, bx);
    };
    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 5; ++b) mbar_init(smem_addr(bar + b), 1);
        mbar_init_fence();
        if (next_filled(it0) < it1) load_x(next_filled(it0));
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tcol = *tslot + 256u * grp;   // the group's 256 TMEM columns
    constexpr uint32_t A_COL = 0, D_COL = 128;
    const uint32_t id = idesc(128, kPK, kFmtBF16);
    bool ok = true;
    int head = -1, nimg = 0, j = 0;   // j: this group's items so far (its MMA and routing-tile phases)

    for (long long s0 = next_filled(it0); s0 < it1 && ok;) {
        const long long s1 = min(it1, (s0 / kPRun) * kPRun + run_tiles(s0 / kPRun));   // this run's tiles in the range
        const int hd = run_slice(s0 / kPRun) % H;
        if (hd != head) {   // both groups are done with the previous head: (re)load the images
            head = hd;
            fence_before_sync();
            __syncthreads();
            if (tid == 0) {
                fence_proxy_async();
                mbar_expect_tx(BAR_I, kPrunedWBytes + kPrunedCBytes);
                bulk_g2s(smem_addr(w_s), wimg + (long long)head * kPrunedWBytes, kPrunedWBytes, BAR_I);
                bulk_g2s(smem_addr(f_s), cimg + (long long)head * 4 * kPK, kPrunedCBytes, BAR_I);
            }
            ok = mbar_wait(BAR_I, (uint32_t)(nimg & 1)) && ok;
            ++nimg;
            if (warp == 0) {   // the head-wide maxima A, M of the per-component ones, into slot 0
                float a = 0.f, m = 0.f;
#pragma unroll
                for (int q = 0; q < kPK / 32; ++q) {
                    a = fmaxf(a, a_s[lane + 32 * q]);
                    m = fmaxf(m, m_s[lane + 32 * q]);
                }
                for (int o = 16; o; o >>= 1) {
                    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
                    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                }
                if (lane == 0) {
                    f_s[2 * kPK] = a;
                    f_s[3 * kPK] = m;
                }
            }
            __syncthreads();
        }
        const float4 *ph = pimg + (long long)head * kPK * kPStride;
        for (long long it = s0 + grp; it < s1; it += kPGroups, ++j) {
            const int bh = run_slice(it / kPRun), t = tile_of(it);
            // this group's routing tiles land in order on its own barrier; the consumer of
            // tile n fetches tile n + 1, so a group's next tile is never fetched before it
            // has consumed the previous one (its barrier runs at most one phase ahead)
            ok = mbar_wait(BAR_X, (uint32_t)(j & 1)) && ok;
            // the row (both halves hold all 64 features) and its sums for the bound
            float2 xr[kPDP];
            if (x_bf16) {
#pragma unroll
                for (int g = 0; g < kPD / 8; ++g) {
                    const uint4 u = *reinterpret_cast<const uint4 *>(xb + sw128_offset(i, 8 * g, kPRows, 2));
                    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        xr[4 * g + e] = make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
                }
            } else {
#pragma unroll
                for (int g = 0; g < kPD / 4; ++g) {
                    const float4 u = *reinterpret_cast<const float4 *>(xb + sw128_offset(i, 4 * g, kPRows, 4));
                    xr[2 * g] = make_float2(u.x, u.y);
                    xr[2 * g + 1] = make_float2(u.z, u.w);
                }
            }
            group_sync(grp);   // the routing tile has been read: the next item's tile may land in it
            if (gt == 0 && next_filled(it + 1) < it1) load_x(next_filled(it + 1));   // (read only: no proxy fence)
            float2 s2v = make_float2(0.f, 0.f);
#pragma unroll
            for (int g = 0; g < kPDP; ++g) s2v = __ffma2_rn(xr[g], xr[g], s2v);
            const float s2 = s2v.x + s2v.y;
            // per-row error bound of the bf16 log-joints (head-wide A = a_s[0], M = m_s[0], reduced
            // from the per-component values when the images were loaded)
            const float delta = fmaf(kPU, fmaf(0.5f * a_s[0], s2, m_s[0] * 8.f * sqrtf(s2)), 1e-3f);
            // A = [x^2 | x] in bf16: half 0 writes the squares (columns 0..31), half 1 the values (32..63)
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                uint32_t p[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const float2 v = xr[16 * b + jj];
                    p[jj] = hf == 0 ? pack2(v.x * v.x, v.y * v.y) : pack2(v.x, v.y);
                }
                tmem_st16(tmem_at(tcol, lane0, A_COL + 32 * hf + 16 * b), p);
            }
            tmem_wait_st();
            fence_before_sync();
            if (gt == 0) bulk_wait_read();   // this group's previous output tile has left shared memory
            group_sync(grp);   // A is in TMEM
            fence_after_sync();
            if (gt == 0) {
#pragma unroll 1
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t kb = kk * 32;
                    const uint32_t boff = (kb >> 7) * (kPK * 128) + (kb & 127);
                    mma_ts(0u, tcol + D_COL, tcol + A_COL + kk * 8, sdesc_sw128(smem_addr(w_s + boff)), id,
                           kk > 0 ? 1u : 0u);
                }
                mma_commit(BAR_M);
            }
            __syncwarp();
            // while the tensor core works: this half of the output row starts as zeros
            if (!g_f32) {
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const uint32_t off = sw128_offset(i, 64 * hf + 8 * g, kPRows, 2);
                    *reinterpret_cast<uint4 *>(ob + off) = make_uint4(0, 0, 0, 0);
                    if (g_split) *reinterpret_cast<uint4 *>(ob + LO + off) = make_uint4(0, 0, 0, 0);
                }
            } else {
#pragma unroll
                for (int g = 0; g < 16; ++g)
                    *reinterpret_cast<float4 *>(ob + sw128_offset(i, 64 * hf + 4 * g, kPRows, 4)) =
                        make_float4(0.f, 0.f, 0.f, 0.f);
            }
            ok = mbar_wait(BAR_M, (uint32_t)(j & 1)) && ok;
            fence_after_sync();

            // bound estimates of this half: l~_k = D_k + c'_k
            auto est = [&](int b, float (&lt)[16]) {
                uint32_t r[16];
                tmem_ld16(tmem_at(tcol, lane0, D_COL + 64 * hf + 16 * b), r);
                tmem_wait_ld();
                const float4 *c4 = reinterpret_cast<const float4 *>(cp_s + 64 * hf + 16 * b);
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const float4 c = c4[g];
                    lt[4 * g] = __uint_as_float(r[4 * g]) + c.x;
                    lt[4 * g + 1] = __uint_as_float(r[4 * g + 1]) + c.y;
                    lt[4 * g + 2] = __uint_as_float(r[4 * g + 2]) + c.z;
                    lt[4 * g + 3] = __uint_as_float(r[4 * g + 3]) + c.w;
                }
            };
            // best and second-best estimate of this half (and where the best is), without branches
            float e1 = -FLT_MAX, e2 = -FLT_MAX;
            int a1 = 0;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                float lt[16];
                est(b, lt);
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) {
                    const float v = lt[jj];
                    e2 = fmaxf(e2, fminf(v, e1));
                    a1 = v > e1 ? 16 * b + jj : a1;
                    e1 = fmaxf(e1, v);
                }
            }
            ex0[hf * kPK + i] = e1;
            ex2[hf * kPK + i] = e2;
            group_sync(grp);
            // the row's best m1 and second-best m2: the kept set is {k : l~_k >= m1 - T - 2 delta};
            // it is {argmax} alone iff m2 falls below that
            const float o1 = ex0[(1 - hf) * kPK + i], o2 = ex2[(1 - hf) * kPK + i];
            const float m1 = fmaxf(e1, o1), m2 = fmaxf(fmaxf(e2, o2), fminf(e1, o1));
            const float keep_from = m1 - kPT - 2.f * delta;
            const bool single = ok && m2 < keep_from;
            // single: a posterior of exactly 1 at the argmax (dropped mass < 128 e^-30)
            if (single && e1 == m1) {
                if (!g_f32)   // split: hi = 1, lo = 0
                    *reinterpret_cast<__nv_bfloat16 *>(ob + sw128_offset(i, 64 * hf + a1, kPRows, 2)) =
                        __float2bfloat16_rn(1.0f);
                else
                    *reinterpret_cast<float *>(ob + sw128_offset(i, 64 * hf + a1, kPRows, 4)) = 1.0f;
            }
            uint32_t xm0 = 0u, xm1 = 0u;   // the kept components of rows that need the softmax
            const bool any_multi = __any_sync(0xffffffffu, !single);
            if (any_multi) {   // tcgen05.ld is warp-collective: the whole warp reloads
                uint32_t mk[2] = {0u, 0u};
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    float lt[16];
                    est(b, lt);
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj)
                        mk[b >> 1] |= (uint32_t)(!ok || lt[jj] >= keep_from) << (16 * (b & 1) + jj);
                }
                if (!single) {
                    xm0 = mk[0];
                    xm1 = mk[1];
                }
            }
            // a tile where many rows keep many components goes to the dense passes (every
            // component of every row on the tensor cores, k_resp_dense_tc, and rows of large
            // magnitude exactly, k_resp_dense); walking the kept sets here one component at a
            // time would be bound by shared-memory reads
            if (group_popc(grp, __popc(xm0) + __popc(xm1) >= kDenseKept) >= kDenseRows) {
                if (gt == 0) dlist[(long long)head * dcap + atomicAdd(dctl + head, 1u)] = make_int2(bh | (src << 30), t);
                if (gt == 0 && zflag) zq[(long long)bh * tps + t] = 0u;   // the dense pass writes both planes
                continue;   // no exact pass and no output tile here
            }
            // per 32-component word: the union of the warp's kept sets, whether its lanes walk
            // their own sets, and the parameters of the union's first component (read here, so
            // that the read overlaps the group barrier below)
            uint32_t uni[2] = {0u, 0u};
            bool lanes[2] = {true, true};
            float4 wpre[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
            if (any_multi) {
#pragma unroll
                for (int wd = 0; wd < 2; ++wd) {
                    const uint32_t m = wd ? xm1 : xm0;
                    uni[wd] = __reduce_or_sync(0xffffffffu, m);
                    lanes[wd] = 16 * __reduce_max_sync(0xffffffffu, (uint32_t)__popc(m)) <= (uint32_t)__popc(uni[wd]);
                    if (!lanes[wd]) wpre[wd] = __ldg(ph + lane + (64 * hf + 32 * wd + __ffs(uni[wd]) - 1) * kPStride);
                }
            }
            // a tile whose rows all keep their argmax alone has a zero lo plane (posteriors 0 and 1)
            const bool any_exact = group_or(grp, (xm0 | xm1) != 0u);
            const bool zlo = zflag && !any_exact;
            if (any_exact) {
                // exact log-joint of a component for this lane's row (parameters from global
                // memory, L2-resident)
                auto exact = [&](int k) {
                    const float4 *pk = ph + k * kPStride;
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int dp = 0; dp < kPDP; dp += 2) {
                        const float4 p = __ldg(pk + dp), r = __ldg(pk + dp + 1);
                        const float2 y0 = __ffma2_rn(xr[dp], make_float2(p.x, p.y), make_float2(p.z, p.w));
                        acc0 = __ffma2_rn(y0, y0, acc0);
                        const float2 y1 = __ffma2_rn(xr[dp + 1], make_float2(r.x, r.y), make_float2(r.z, r.w));
                        acc1 = __ffma2_rn(y1, y1, acc1);
                    }
                    return fmaf(-0.5f, (acc0.x + acc0.y) + (acc1.x + acc1.y), c_s[k]);
                };
                // the same value for a component k common to the warp, every lane present: lane
                // dp holds the parameter word dp of k (one coalesced read per warp) and puts it in
                // the warp's shared copy, which every lane then reads as broadcasts
                auto exact_w = [&](int k, const float4 w) {
                    __syncwarp();   // the previous component's copy has been read
                    pw_s[lane] = w;
                    __syncwarp();
                    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int dp = 0; dp < kPDP; dp += 2) {
                        const float4 p = pw_s[dp], r = pw_s[dp + 1];
                        const float2 y0 = __ffma2_rn(xr[dp], make_float2(p.x, p.y), make_float2(p.z, p.w));
                        acc0 = __ffma2_rn(y0, y0, acc0);
                        const float2 y1 = __ffma2_rn(xr[dp + 1], make_float2(r.x, r.y), make_float2(r.z, r.w));
                        acc1 = __ffma2_rn(y1, y1, acc1);
                    }
                    return fmaf(-0.5f, (acc0.x + acc0.y) + (acc1.x + acc1.y), c_s[k]);
                };
                // Runs f(k, l_k) for every component k of the two masks, by 32-component word.
                // Lanes whose sets are small against their union (16 times or more) walk their
                // own sets; otherwise the warp walks the union one component at a time, reading
                // the next component's parameters while it evaluates the current one.
                // Warp-converged code only.
                auto for_kept = [&](auto &&f) {
#pragma unroll
                    for (int wd = 0; wd < 2; ++wd) {
                        const int k0 = 64 * hf + 32 * wd;
                        const uint32_t mk = wd ? xm1 : xm0;
                        if (lanes[wd]) {
                            for (uint32_t mm = mk; mm; mm &= mm - 1) {
                                const int k = k0 + __ffs(mm) - 1;
                                f(k, exact(k));
                            }
                        } else {
                            const float4 *pw = ph + lane;
                            uint32_t mm = uni[wd];
                            float4 w = wpre[wd];
                            while (mm) {
                                const int kq = __ffs(mm) - 1;
                                mm &= mm - 1;
                                const float4 wn = mm ? __ldg(pw + (k0 + __ffs(mm) - 1) * kPStride) : w;
                                const float l = exact_w(k0 + kq, w);
                                if ((mk >> kq) & 1u) f(k0 + kq, l);
                                w = wn;
                            }
                        }
                    }
                };
                // exact pass: online maximum and sum over the kept components of this half; the
                // log-joints wait in the output tile for the normalisation (fp32 tile: as floats;
                // 16-bit tiles: high half-word in the hi plane, low half-word in the lo plane, which
                // a single-plane tile has room for and never stores)
                float mt = -FLT_MAX, st = 0.f;
                for_kept([&](int k, float l) {
                    if (g_f32) {
                        *reinterpret_cast<float *>(ob + sw128_offset(i, k, kPRows, 4)) = l;
                    } else {
                        const uint32_t off = sw128_offset(i, k, kPRows, 2), u = __float_as_uint(l);
                        *reinterpret_cast<unsigned short *>(ob + off) = (unsigned short)(u >> 16);
                        *reinterpret_cast<unsigned short *>(ob + LO + off) = (unsigned short)(u & 0xffffu);
                    }
                    if (l > mt) {
                        st = st * expf(mt - l) + 1.f;
                        mt = l;
                    } else {
                        st += expf(l - mt);
                    }
                });
                ex1[hf * kPK + i] = mt;
                ex2[hf * kPK + i] = st;
                group_sync(grp);
                if (xm0 | xm1) {
                    const float q1 = ex1[(1 - hf) * kPK + i], q2 = ex2[(1 - hf) * kPK + i];
                    const float m = fmaxf(mt, q1);
                    const float inv = 1.0f / (st * expf(mt - m) + q2 * expf(q1 - m));
                    // the kept posteriors of this half into the output tile
#pragma unroll
                    for (int wd = 0; wd < 2; ++wd)
                        for (uint32_t mm = wd ? xm1 : xm0; mm; mm &= mm - 1) {
                            const int k = 64 * hf + 32 * wd + __ffs(mm) - 1;
                            if (g_f32) {
                                float *o = reinterpret_cast<float *>(ob + sw128_offset(i, k, kPRows, 4));
                                *o = expf(*o - m) * inv;
                            } else {
                                const uint32_t off = sw128_offset(i, k, kPRows, 2);
                                const float l = __uint_as_float(
                                    ((uint32_t)*reinterpret_cast<const unsigned short *>(ob + off) << 16) |
                                    *reinterpret_cast<const unsigned short *>(ob + LO + off));
                                __nv_bfloat16 hi, lo;
                                split_bf16(expf(l - m) * inv, hi, lo);
                                *reinterpret_cast<__nv_bfloat16 *>(ob + off) = hi;
                                if (g_split) *reinterpret_cast<__nv_bfloat16 *>(ob + LO + off) = lo;
                            }
                        }
                }
            }
            fence_proxy_async();   // the output tile, written by threads, is read by the TMA store
            fence_before_sync();
            group_sync(grp);
            fence_after_sync();
            if (gt == 0) {
                for (int a = 0; a < kPK * ge / 128; ++a) {
                    tma_store_3d(&gmap, a * (128 / ge), t * kPRows, bh, smem_addr(ob + a * (kPRows * 128)));
                    if (g_split && !zlo)
                        tma_store_3d(&gmap_lo, a * (128 / ge), t * kPRows, bh, smem_addr(ob + LO + a * (kPRows * 128)));
                }
                bulk_commit();
                if (zflag) zq[(long long)bh * tps + t] = zlo ? 1u : 0u;
            }
        }
        s0 = next_filled(s1);
        ok = __syncthreads_and(ok) != 0;   // both groups leave the loop together
    }
    // after a failed wait a routing tile may still be in flight for either group: let it land
    // (bounded) before the shared memory is released; after a normal end every fetched tile
    // has been consumed
    bool ok_end = ok;
    if (gt == 0) {
        if (!ok) ok_end = mbar_wait(BAR_X, (uint32_t)(j & 1)) && ok_end;
        bulk_wait_all();
    }
    fence_before_sync();
    if (__syncthreads_and(ok_end) == 0 && tid == 0) report_timeout(timeout);
    if (warp == 0) tmem_dealloc(*tslot, 512);
}

// ------------------------------------------------------------------------
// Dense exact responsibilities of the tiles the tensor-core dense pass leaves (rows
// of large magnitude among rows that keep many components): every one of the 128
// log-joints of every row, the same packed-FMA quadratic form ((x - mu) / sigma)^2,
// then the softmax.
//
// Two persistent CTAs of 8 warps per SM (one CTA's loads, softmax and stores
// overlap the other's FMAs), each taking a contiguous range of the listed tiles
// in head order, so that it works on one or two heads whose parameters stay in
// L1; every tile's result depends on that tile alone.  Warp w
// covers rows 32 (w % 4) .. + 31 and components 64 (w / 4) .. + 63; lane (g, e)
// holds rows 8 g .. 8 g + 7 of those and feature eighth e (features 8 e .. + 7)
// in registers and takes two components at a time: the parameter words of
// feature pair 4 e + j of both components are read through L1 with the
// evict-last hint (the eighths of one feature-pair slot are 128 contiguous bytes
// in the interleaved image; the routing rows are read L2-only so that they do
// not evict them), so every 16-byte read feeds 16 packed FMAs (8 rows, square
// and accumulate).  The 16 partial sums (2 components x 8 rows) meet over the
// eighth lanes by recursive halving (14 shuffles), each lane keeping one
// component for two rows.  Log-joints go to a shared [128][132] tile; 2 threads per row take the
// softmax (components strided by 2); rows then leave in the requested layout
// with coalesced stores.  The kernel
// is a programmatic dependent of the tensor-core dense pass: it reads its list
// only after griddepcontrol.wait.
constexpr int kDThreads = 256, kDPitch = 132;

// A read-only 16-byte load that L1 keeps in preference to other lines (the
// parameters of the head, reused by every tile of that head).
__device__ __forceinline__ float4 ld_keep(const float4 *p)
{
    float4 r;
    asm("ld.global.nc.L1::evict_last.v4.f32 {%0, %1, %2, %3}, [%4];"
        : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
        : "l"(p));
    return r;
}

struct DenseSrc {
    const void *x;
    void *gamma;
    int N;
    long long plane;   // elements of one plane of the split layout
};

__global__ void __launch_bounds__(kDThreads, 2)
    k_resp_dense(DenseSrc s0, DenseSrc s1, bool x_bf16, int H, const float4 *__restrict__ pimg2,
                 const float *__restrict__ cimg, int layout, const int2 *__restrict__ dlist,
                 const unsigned int *__restrict__ dctl, long long dcap)
{
    extern __shared__ float ell[];   // [128][kDPitch]
    __shared__ unsigned int s_red[kDThreads / 32];
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the routing launches have listed their tiles
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = lane & 7, rg = lane >> 3;      // q: feature eighth (pairs 4 q .. 4 q + 3)
    const int r0 = 32 * (warp & 3) + 8 * rg;     // this thread's rows r0 .. r0 + 7 of the tile
    const int k0 = 64 * (warp >> 2);             // its half of the components
    // the listed tiles in head order; this CTA takes a contiguous range of them, so that it
    // works on one or two heads (their parameters stay in L1) and needs no atomics
    unsigned int listed = 0;
    for (int h = tid; h < H; h += kDThreads) listed += dctl[h];
#pragma unroll
    for (int o = 16; o; o >>= 1) listed += __shfl_xor_sync(0xffffffffu, listed, o);
    if (lane == 0) s_red[warp] = listed;
    __syncthreads();
    listed = 0;
#pragma unroll
    for (int w = 0; w < kDThreads / 32; ++w) listed += s_red[w];
    if (listed == 0) return;   // nothing listed (peaked inputs)
    const unsigned int per = (listed + gridDim.x - 1) / gridDim.x;
    const unsigned int g0 = blockIdx.x * per, g1 = min(listed, g0 + per);
    int hc = 0;                // the head of position g: hbase = sum of the counts of heads < hc
    unsigned int hbase = 0, hcnt = g0 < g1 ? dctl[0] : 0;
    for (unsigned int g = g0; g < g1; ++g) {
        while (g >= hbase + hcnt) {   // uniform: every thread walks the same counts
            hbase += hcnt;
            hcnt = dctl[++hc];
        }
        const int2 e = dlist[(long long)hc * dcap + (g - hbase)];
        const DenseSrc src = (e.x >> 30) ? s1 : s0;
        const long long bh = e.x & 0x3fffffff;
        const int N = src.N, row0 = e.y * kPRows, h = (int)(bh % H);
        // the eight rows' feature eighth (zeros past the slice end)
        float2 xr[8][4];
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int row = row0 + r0 + r;
            const long long off = (bh * N + row) * kPD + 8 * q;
            if (row < N) {
                if (x_bf16) {
                    const uint4 w = __ldcg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(src.x) + off));
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        xr[r][c] = make_float2(__uint_as_float(ww[c] << 16), __uint_as_float(ww[c] & 0xffff0000u));
                } else {
                    const float4 *p4 = reinterpret_cast<const float4 *>(static_cast<const float *>(src.x) + off);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {   // routing rows: L2 only, L1 keeps the parameters
                        const float4 w = __ldcg(p4 + u);
                        xr[r][2 * u] = make_float2(w.x, w.y);
                        xr[r][2 * u + 1] = make_float2(w.z, w.w);
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) xr[r][j] = make_float2(0.f, 0.f);
            }
        }
        const float4 *ph = pimg2 + (long long)h * kPK * kPDP + q;
        const float *ch = cimg + (long long)h * 4 * kPK;   // c_k
#pragma unroll 1
        for (int kb = k0; kb < k0 + 64; kb += 2) {
            float2 acc[2][8];
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int r = 0; r < 8; ++r) acc[c][r] = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float4 pa = ld_keep(ph + kb * kPDP + 8 * j), pb = ld_keep(ph + (kb + 1) * kPDP + 8 * j);
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const float2 ya = __ffma2_rn(xr[r][j], make_float2(pa.x, pa.y), make_float2(pa.z, pa.w));
                    acc[0][r] = __ffma2_rn(ya, ya, acc[0][r]);
                    const float2 yb = __ffma2_rn(xr[r][j], make_float2(pb.x, pb.y), make_float2(pb.z, pb.w));
                    acc[1][r] = __ffma2_rn(yb, yb, acc[1][r]);
                }
            }
            // v[8 c + r]: this lane's partial sum of component kb + c, row r0 + r; recursive halving
            // over the eighth lanes: xor 1 keeps one component, xor 2 four of the rows, xor 4 two
            float v[16];
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int r = 0; r < 8; ++r) v[8 * c + r] = acc[c][r].x + acc[c][r].y;
#pragma unroll
            for (int o = 1, n = 8; o <= 4; o <<= 1, n >>= 1) {
                const bool up = (q & o) != 0;
#pragma unroll
                for (int e2 = 0; e2 < 8; ++e2)
                    if (e2 < n) {
                        const float send = up ? v[e2] : v[e2 + n], keep = up ? v[e2 + n] : v[e2];
                        v[e2] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                    }
            }
            // this lane now holds component kb + (q & 1) for rows r0 + 4 ((q >> 1) & 1) + 2 (q >> 2) + {0, 1}
            const int k = kb + (q & 1), rr = r0 + 4 * ((q >> 1) & 1) + 2 * (q >> 2);
            const float c = __ldg(ch + k);
            ell[rr * kDPitch + k] = fmaf(-0.5f, v[0], c);
            ell[(rr + 1) * kDPitch + k] = fmaf(-0.5f, v[1], c);
        }
        __syncthreads();
        // softmax of row tid / 2 over components 2 m + tid % 2 (in place)
        {
            float *er = ell + (tid >> 1) * kDPitch + (tid & 1);
            float m = -FLT_MAX;
#pragma unroll 8
            for (int i = 0; i < kPK / 2; ++i) m = fmaxf(m, er[2 * i]);
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            float sum = 0.f;
#pragma unroll 8
            for (int i = 0; i < kPK / 2; ++i) {
                const float ex = expf(er[2 * i] - m);
                er[2 * i] = ex;
                sum += ex;
            }
            sum += __shfl_xor_sync(0xffffffffu, sum, 1);
            const float inv = 1.0f / sum;
#pragma unroll 8
            for (int i = 0; i < kPK / 2; ++i) er[2 * i] *= inv;
        }
        __syncthreads();
        // rows out: warp w takes rows 16 w .. + 15, one row per instruction (fp32: 32 lanes x 16 B)
        // or two (16-bit planes: 16 lanes x 16 B each)
        if (layout == GL_F32) {
            float *g = static_cast<float *>(src.gamma);
#pragma unroll 4
            for (int rr = 0; rr < 16; ++rr) {
                const int r = 16 * warp + rr, row = row0 + r;
                if (row < N)
                    reinterpret_cast<float4 *>(g + (bh * N + row) * kPK)[lane] =
                        *reinterpret_cast<const float4 *>(ell + r * kDPitch + 4 * lane);
            }
        } else {
            __nv_bfloat16 *g = static_cast<__nv_bfloat16 *>(src.gamma);
#pragma unroll 2
            for (int rr = 0; rr < 16; rr += 2) {
                const int r = 16 * warp + rr + (lane >> 4), row = row0 + r, c8 = 8 * (lane & 15);
                if (row < N) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        __nv_bfloat16 h0, l0, h1, l1;
                        split_bf16(ell[r * kDPitch + c8 + 2 * u], h0, l0);
                        split_bf16(ell[r * kDPitch + c8 + 2 * u + 1], h1, l1);
                        hw[u] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                        lw[u] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
                    }
                    const long long o = (bh * N + row) * kPK + c8;
                    *reinterpret_cast<uint4 *>(g + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    if (layout == GL_SPLIT)
                        *reinterpret_cast<uint4 *>(g + src.plane + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
        }
        __syncthreads();   // the tile of log-joints is reused by the next tile
    }
}

// ------------------------------------------------------------------------
// Dense responsibilities of the listed tiles on the tensor cores.
//
// Expanding the square, the log-joint of the GMA explainer's posterior is
//   l_ik = c'_k + sum_d ( -1/2 a_kd x_id^2 + a_kd mu_kd x_id ),   a = 1/sigma^2,
// one product of [x^2 | x] (128 rows x 128) with W^T (128 x 128 components) per tile.
// Each fp32 operand is held as three bf16 planes, v = v0 + v1 + v2 up to 2^-24 |v| (each
// plane the round-to-nearest of what the previous ones leave), and the six plane products
// whose orders add up to at most two are accumulated in fp32, smallest first (A2 W0, A1 W1,
// A1 W0, A0 W2, A0 W1, A0 W0); each of the three dropped ones is below 2^-24 of its term.
// So every log-joint carries the rounding of an fp32 evaluation of the expanded form: a few
// fp32 units of
//   S_i = 1/2 A sum_d x_id^2 + M sum_d |x_id|   (A = max a, M = max |a mu| over the head),
// which bounds the sum of the terms' magnitudes.  The direct form (x - mu)^2 / sigma^2 of
// the exact kernels rounds at the scale of the log-joint itself, which on the rows these
// tiles hold (many components near the best one) is of the same order.  A tile with a row
// whose S_i exceeds kTSMax (|x| large against the components) goes on a second list, to
// the exact dense kernel; every other row's posteriors are the softmax of these log-joints.
// With bf16 routing rows the values are one plane and their squares two, and the products
// of the planes that are zero are skipped.
//
// One persistent CTA of 16 warps per SM over a contiguous range of the listed tiles in head
// order (the head's three planes, 96 KB, are loaded once per head).  Warp w owns TMEM lanes
// 32 (w % 4) .. + 31 (rows of the tile) and column quarter q = w / 4: operand positions
// 32 q .. 32 q + 31 (the squares, then the values, of features 16 q .. + 15; dtc_pos) and
// components 32 q .. + 31 of the result.  The operand planes are double-buffered in TMEM
// and the accumulator is read out before the next products are issued, so the products of
// item n + 1 run while the warps take the softmax of item n and split the routing tile of
// item n + 2; two CTA barriers per item.
constexpr int kTThreads = 512;
constexpr float kTSMax = 4096.f;
constexpr float kLog2e = 1.4426950408889634f;

struct DenseTcSmem {
    static constexpr uint32_t W3 = kPrunedW3Bytes;      // three planes of W, SW128 K-major
    static constexpr uint32_t X = kPRows * kPD * 4;     // routing tile (fp32 worst case)
    static constexpr uint32_t O = kPRows * kPK * 4;     // output tile (fp32 worst case)
    static constexpr uint32_t C = 2 * kPrunedCBytes;    // c, c', A, M of two heads
    static constexpr uint32_t EX = 4 * kPRows * 8;      // per quarter and row: (max, sum)
    static constexpr uint32_t SS = 2 * 4 * kPRows * 8;  // per item of two, quarter, row: (sum x^2, sum |x|)
    static constexpr size_t bytes = 1024 + (size_t)W3 + X + O + C + EX + SS + 64;
};
static_assert(DenseTcSmem::bytes <= 232448, "dense tensor-core routing: shared memory above the per-block limit");

struct DenseTcMaps {
    CUtensorMap x[2], g[2], glo[2];   // per source: routing rows, output (hi plane), lo plane
};

// 2^t by the SFU's base-2 exponential (relative error about 2^-22; 0 for t below -126).
__device__ __forceinline__ float ex2_sfu(float t)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

// The three bf16 planes of a pair of values, packed two per word (the first value in the
// low half): each plane the round-to-nearest of what the previous ones leave.
__device__ __forceinline__ void split3_pair(float2 v, uint32_t &p0, uint32_t &p1, uint32_t &p2)
{
    const float2 m1 = make_float2(-1.f, -1.f);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
    p0 = *reinterpret_cast<const uint32_t *>(&b);
    v = __ffma2_rn(make_float2(__uint_as_float(p0 << 16), __uint_as_float(p0 & 0xffff0000u)), m1, v);
    b = __floats2bfloat162_rn(v.x, v.y);
    p1 = *reinterpret_cast<const uint32_t *>(&b);
    v = __ffma2_rn(make_float2(__uint_as_float(p1 << 16), __uint_as_float(p1 & 0xffff0000u)), m1, v);
    b = __floats2bfloat162_rn(v.x, v.y);
    p2 = *reinterpret_cast<const uint32_t *>(&b);
}

__global__ void __launch_bounds__(kTThreads, 1)
    k_resp_dense_tc(const __grid_constant__ DenseTcMaps maps, bool x_bf16, int H,
                    const unsigned char *__restrict__ w3img, const float *__restrict__ cimg, int layout,
                    const int2 *__restrict__ dlist, unsigned int *__restrict__ dctl, int2 *__restrict__ dlist2,
                    long long dcap, unsigned int *timeout)
{
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the routing launches have listed their tiles
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    __shared__ unsigned int s_red[kTThreads / 32];
    __shared__ float2 am_s[2];   // A, M of the heads in the two constants' buffers
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, cq = warp >> 2;
    const int i = 32 * qd + lane;   // row of the tile (TMEM lane)

    // the listed tiles in head order; this CTA takes a contiguous range of them
    unsigned int listed = 0;
    for (int h = tid; h < H; h += kTThreads) listed += dctl[h];
#pragma unroll
    for (int o = 16; o; o >>= 1) listed += __shfl_xor_sync(0xffffffffu, listed, o);
    if (lane == 0) s_red[warp] = listed;
    __syncthreads();
    listed = 0;
#pragma unroll
    for (int w = 0; w < kTThreads / 32; ++w) listed += s_red[w];
    const unsigned int per = (listed + gridDim.x - 1) / gridDim.x;
    const unsigned int g0 = min(listed, blockIdx.x * per), g1 = min(listed, g0 + per);
    if (g0 >= g1) return;
    const int cnt = (int)(g1 - g0);
    // entry g of the list in head order, for g increasing: every thread walks the same counts
    int hc = 0;
    unsigned int hbase = 0, hcnt = dctl[0];
    auto entry_at = [&](unsigned int g, int &head) {
        while (g >= hbase + hcnt) {
            hbase += hcnt;
            hcnt = dctl[++hc];
        }
        head = hc;
        return dlist[(long long)hc * dcap + (g - hbase)];
    };

    unsigned char *w_s = sm;
    unsigned char *xb = w_s + DenseTcSmem::W3;
    unsigned char *ob = xb + DenseTcSmem::X;
    float *c_s = reinterpret_cast<float *>(ob + DenseTcSmem::O);                // [2][4][128]
    float2 *ex_s = reinterpret_cast<float2 *>(c_s + 2 * 4 * kPK);               // [4][128]
    float2 *ss_s = ex_s + 4 * kPRows;                                           // [2][4][128]
    uint64_t *bar = reinterpret_cast<uint64_t *>(ss_s + 2 * 4 * kPRows);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 3);
    const uint32_t BAR_I = smem_addr(bar), BAR_X = smem_addr(bar + 1), BAR_M = smem_addr(bar + 2);
    const uint32_t xbytes = kPRows * kPD * (x_bf16 ? 2 : 4);
    const bool g_f32 = layout == GL_F32, g_split = layout == GL_SPLIT;
    const int ge = g_f32 ? 4 : 2;
    constexpr uint32_t LO = kPRows * kPK * 2;   // split: the lo plane's tile follows the hi plane's
    constexpr uint32_t D_COL = 384;             // the accumulator; operand planes at 192 b + 64 j
    uint32_t tbase = 0;                         // TMEM base, once allocated
    auto load_x = [&](int2 e) {                 // one thread
        const int s = e.x >> 30, bh = e.x & 0x3fffffff;
        mbar_expect_tx(BAR_X, xbytes);
        tma_load_3d(smem_addr(xb), &maps.x[s], 0, e.y * kPRows, bh, BAR_X);
        if (!x_bf16) tma_load_3d(smem_addr(xb + kPRows * 128), &maps.x[s], 32, e.y * kPRows, bh, BAR_X);
    };
    int nimg = 0;
    // the planes of W and the constants of `head` into buffer `buf` (every thread; no
    // products may be running)
    auto load_head = [&](int head, int buf) {
        if (tid == 0) {
            fence_proxy_async();   // earlier thread reads of the constants' buffer come first
            mbar_expect_tx(BAR_I, (uint32_t)(kPrunedW3Bytes + kPrunedCBytes));
            bulk_g2s(smem_addr(w_s), w3img + (long long)head * kPrunedW3Bytes, kPrunedW3Bytes, BAR_I);
            bulk_g2s(smem_addr(c_s + buf * 4 * kPK), cimg + (long long)head * 4 * kPK, kPrunedCBytes, BAR_I);
        }
        const bool got = mbar_wait(BAR_I, (uint32_t)(nimg & 1));
        ++nimg;
        if (warp == 0) {   // the head-wide maxima of the per-component A_k, M_k
            float a = 0.f, m = 0.f;
#pragma unroll
            for (int q = 0; q < kPK / 32; ++q) {
                a = fmaxf(a, c_s[buf * 4 * kPK + 2 * kPK + lane + 32 * q]);
                m = fmaxf(m, c_s[buf * 4 * kPK + 3 * kPK + lane + 32 * q]);
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            }
            if (lane == 0) am_s[buf] = make_float2(a, m);
        }
        return got;
    };
    // item n's landed routing tile into operand buffer n % 2, and its rows' sums for S_i
    auto convert = [&](int n) {
        float2 xv[8];
        if (x_bf16) {
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const uint4 u = *reinterpret_cast<const uint4 *>(xb + sw128_offset(i, 16 * cq + 8 * g, kPRows, 2));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    xv[4 * g + e] = make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
            }
        } else {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float4 u = *reinterpret_cast<const float4 *>(xb + sw128_offset(i, 16 * cq + 4 * g, kPRows, 4));
                xv[2 * g] = make_float2(u.x, u.y);
                xv[2 * g + 1] = make_float2(u.z, u.w);
            }
        }
        uint32_t pw[3][16];
        float2 s2 = make_float2(0.f, 0.f), s1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const float2 q = __fmul2_rn(xv[c], xv[c]);
            s2 = __fadd2_rn(s2, q);
            s1 = __fadd2_rn(s1, make_float2(fabsf(xv[c].x), fabsf(xv[c].y)));
            split3_pair(q, pw[0][c], pw[1][c], pw[2][c]);
            split3_pair(xv[c], pw[0][8 + c], pw[1][8 + c], pw[2][8 + c]);
        }
        const uint32_t acol = 192u * (uint32_t)(n & 1) + 16u * (uint32_t)cq;
#pragma unroll
        for (int j = 0; j < 3; ++j) tmem_st16(tmem_at(tbase, 32 * qd, acol + 64 * j), pw[j]);
        ss_s[(n & 1) * 4 * kPRows + cq * kPRows + i] = make_float2(s2.x + s2.y, s1.x + s1.y);
        tmem_wait_st();
    };
    // one thread: item n's products (operand buffer n % 2) into the accumulator, smallest
    // first; with bf16 rows the values' higher planes and the squares' third plane are zero
    const uint32_t id = idesc(128, kPK, kFmtBF16);
    auto issue = [&](int n) {
        const uint32_t ab = 192u * (uint32_t)(n & 1);
        bool first = true;
#pragma unroll
        for (int q = 0; q < 6; ++q) {
            const uint32_t pa = q == 0 ? 2u : (q < 3 ? 1u : 0u);                // A plane
            const uint32_t pb = (q == 1 || q == 4) ? 1u : (q == 3 ? 2u : 0u);    // W plane
            if (x_bf16 && pa == 2) continue;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                if (x_bf16 && pa == 1 && (kk & 1)) continue;   // odd K steps: the values
                const uint32_t kb = kk * 32;   // byte offset of the K step in a row of W
                const uint32_t boff = pb * (uint32_t)kPrunedWBytes + (kb >> 7) * (kPK * 128) + (kb & 127);
                mma_ts(0u, tbase + D_COL, tbase + ab + 64u * pa + 8u * kk, sdesc_sw128(smem_addr(w_s + boff)), id,
                       first ? 0u : 1u);
                first = false;
            }
        }
        mma_commit(BAR_M);
    };

    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 512);
        tmem_relinquish();
    }
    int hcur = 0;
    int2 ecur = entry_at(g0, hcur);
    if (tid == 0) {
        for (int b = 0; b < 3; ++b) mbar_init(smem_addr(bar + b), 1);
        mbar_init_fence();
        load_x(ecur);
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    tbase = *tslot;
    bool ok = load_head(hcur, 0);
    int hp = 0;                        // constants' buffer of item n's head
    bool x_pending = true;             // tid 0: a routing tile in flight, and its phase
    uint32_t x_par = 0;
    int m_issued = -1;                 // tid 0: the last item whose products were issued
    {   // item 0: its operand planes, then its products and the next routing tile
        const bool landed = mbar_wait(BAR_X, 0u);
        ok = landed && ok;
        if (tid == 0 && landed) x_pending = false;
        convert(0);
        fence_before_sync();
        ok = __syncthreads_and(ok) != 0;   // the planes are in TMEM, am_s is written
        fence_after_sync();
    }
    int2 enext = ecur;
    int hnext = hcur;
    if (cnt > 1) enext = entry_at(g0 + 1, hnext);
    if (tid == 0 && ok) {
        issue(0);
        m_issued = 0;
        if (cnt > 1) {
            load_x(enext);
            x_pending = true;
            x_par = 1u;
        }
    }

    float2 acc[16];                    // the accumulator row of the previous item, 32 components
    int2 eprev = ecur;                 // the previous item: entry, head, constants' buffer
    int hprev = hcur, hpprev = hp;
    bool rel_prev = false;             // whether the previous item goes to the exact kernel

    // softmax of the previous item from acc: posteriors into the output tile unless a row is
    // beyond the magnitude limit; returns whether the item goes to the exact kernel
    auto softmax = [&](int m, int hpx) {
        const float2 *cp = reinterpret_cast<const float2 *>(c_s + hpx * 4 * kPK + kPK + 32 * cq);   // c'_k
        float mq = -FLT_MAX;
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            acc[p] = __fadd2_rn(acc[p], cp[p]);
            mq = fmaxf(mq, fmaxf(acc[p].x, acc[p].y));
        }
        const float2 mneg = make_float2(-mq, -mq), l2e = make_float2(kLog2e, kLog2e);
        float2 sq2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            const float2 t = __fmul2_rn(__fadd2_rn(acc[p], mneg), l2e);
            acc[p] = make_float2(ex2_sfu(t.x), ex2_sfu(t.y));
            sq2 = __fadd2_rn(sq2, acc[p]);
        }
        ex_s[cq * kPRows + i] = make_float2(mq, sq2.x + sq2.y);
        const float2 *sp = ss_s + (m & 1) * 4 * kPRows + i;
        const float2 am = am_s[hpx];
        const float sx2 = (sp[0].x + sp[kPRows].x) + (sp[2 * kPRows].x + sp[3 * kPRows].x);
        const float sx1 = (sp[0].y + sp[kPRows].y) + (sp[2 * kPRows].y + sp[3 * kPRows].y);
        const bool far = fmaf(0.5f * am.x, sx2, am.y * sx1) > kTSMax;
        if (tid == 0) bulk_wait_read();   // the output tile of the item before has left shared memory
        const bool relist = __syncthreads_or(far) != 0;
        if (!relist) {
            // merge the four quarters' (max, sum): the row's max, and this quarter's scale
            float2 e4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) e4[q] = ex_s[q * kPRows + i];
            const float mrow = fmaxf(fmaxf(e4[0].x, e4[1].x), fmaxf(e4[2].x, e4[3].x));
            float tot = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) tot = fmaf(e4[q].y, ex2_sfu((e4[q].x - mrow) * kLog2e), tot);
            const float sc = ex2_sfu((mq - mrow) * kLog2e) / tot;
            const float2 sc2 = make_float2(sc, sc);
            if (g_f32) {
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const float2 a = __fmul2_rn(acc[2 * g], sc2), b = __fmul2_rn(acc[2 * g + 1], sc2);
                    *reinterpret_cast<float4 *>(ob + sw128_offset(i, 32 * cq + 4 * g, kPRows, 4)) =
                        make_float4(a.x, a.y, b.x, b.y);
                }
            } else {
                const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 v = __fmul2_rn(acc[4 * g + u], sc2);
                        __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
                        hw[u] = *reinterpret_cast<const uint32_t *>(&b);
                        const float2 r = __ffma2_rn(
                            make_float2(__uint_as_float(hw[u] << 16), __uint_as_float(hw[u] & 0xffff0000u)), m1, v);
                        b = __floats2bfloat162_rn(r.x, r.y);
                        lw[u] = *reinterpret_cast<const uint32_t *>(&b);
                    }
                    const uint32_t off = sw128_offset(i, 32 * cq + 8 * g, kPRows, 2);
                    *reinterpret_cast<uint4 *>(ob + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    if (g_split) *reinterpret_cast<uint4 *>(ob + LO + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            fence_proxy_async();   // the output tile, written by threads, is read by the TMA store
        }
        return relist;
    };
    // one thread, after a CTA barrier that follows the softmax: the previous item's output
    // tile out by TMA stores, or the item onto the exact kernel's list
    auto finish = [&](int2 e, int h, bool relist) {
        if (relist) {
            dlist2[(long long)h * dcap + atomicAdd(dctl + H + h, 1u)] = e;
        } else {
            const int s = e.x >> 30, bh = e.x & 0x3fffffff;
            for (int a = 0; a < kPK * ge / 128; ++a) {
                tma_store_3d(&maps.g[s], a * (128 / ge), e.y * kPRows, bh, smem_addr(ob + a * (kPRows * 128)));
                if (g_split)
                    tma_store_3d(&maps.glo[s], a * (128 / ge), e.y * kPRows, bh,
                                 smem_addr(ob + LO + a * (kPRows * 128)));
            }
            bulk_commit();
        }
    };

    for (int n = 0; n < cnt && ok; ++n) {
        // item n's products are running; acc holds item n - 1's accumulator row
        if (n >= 1) rel_prev = softmax(n - 1, hpprev);
        if (n + 1 < cnt) {   // item n + 1's routing tile into the other operand buffer
            const bool landed = mbar_wait(BAR_X, (uint32_t)((n + 1) & 1));
            ok = landed && ok;
            if (tid == 0 && landed) x_pending = false;
            convert(n + 1);
        }
        // item n's accumulator row into registers (it is free for item n + 1's products after
        // the barrier below)
        ok = mbar_wait(BAR_M, (uint32_t)(n & 1)) && ok;
        fence_after_sync();
        {
            uint32_t r[2][16];
            tmem_ld16(tmem_at(tbase, 32 * qd, D_COL + 32 * cq), r[0]);
            tmem_ld16(tmem_at(tbase, 32 * qd, D_COL + 32 * cq + 16), r[1]);
            tmem_wait_ld();
#pragma unroll
            for (int p = 0; p < 16; ++p)
                acc[p] = make_float2(__uint_as_float(r[p >> 3][2 * (p & 7)]), __uint_as_float(r[p >> 3][2 * (p & 7) + 1]));
        }
        const int2 en = ecur;
        const int hn = hcur, hpn = hp;
        int2 e2 = enext;
        int h2 = hnext;
        if (n + 1 < cnt) {
            if (hnext != hcur) {   // item n + 1 is of another head (item n's products are done)
                hp ^= 1;           // the constants of item n's head stay for its softmax
                ok = load_head(hnext, hp) && ok;
            }
            if (n + 2 < cnt) e2 = entry_at(g0 + n + 2, h2);
        }
        fence_before_sync();
        ok = __syncthreads_and(ok) != 0;   // operand planes written, accumulator read, softmax done
        fence_after_sync();
        if (tid == 0 && ok) {
            if (n >= 1) finish(eprev, hprev, rel_prev);
            if (n + 1 < cnt) {
                issue(n + 1);
                m_issued = n + 1;
                if (n + 2 < cnt) {   // (the tile was only read by threads: no proxy fence)
                    load_x(e2);
                    x_pending = true;
                    x_par = (uint32_t)((n + 2) & 1);
                }
            }
        }
        eprev = en;
        hprev = hn;
        hpprev = hpn;
        ecur = enext;
        hcur = hnext;
        enext = e2;
        hnext = h2;
    }
    if (ok) {   // the last item's softmax and output
        rel_prev = softmax(cnt - 1, hpprev);
        ok = __syncthreads_and(ok) != 0;
        if (tid == 0 && ok) finish(eprev, hprev, rel_prev);
    }
    // after a failed wait a routing tile or products may still be in flight: let them finish
    // (bounded) before TMEM and shared memory are released
    bool ok_end = ok;
    if (tid == 0) {
        if (!ok) {
            if (x_pending) ok_end = mbar_wait(BAR_X, x_par) && ok_end;
            if (m_issued >= 0) ok_end = mbar_wait(BAR_M, (uint32_t)(m_issued & 1)) && ok_end;
        }
        bulk_wait_all();
    }
    fence_before_sync();
    if (__syncthreads_and(ok_end) == 0 && tid == 0) report_timeout(timeout);
    if (warp == 0) tmem_dealloc(tbase, 512);
}
} // namespace

bool resp_pruned_applies(const Dims &dm) { return dm.K == kPK && dm.D == kPD; }

cudaError_t launch_prep_all(const Dims &dm, const gma_params &p, float4 *prm, float *cst, const PrunedImages &img,
                            cudaStream_t st)
{
    if (!resp_pruned_applies(dm)) return cudaErrorInvalidValue;
    k_prep_all<<<dim3(dm.H, kPK / kPrepAllComps), kPrepAllThreads, 0, st>>>(p.mu, p.var_raw, p.logit_pi, prm, cst,
                                                                           img.w, img.w3, img.p, img.c, img.p2,
                                                                           img.ctl);
    return cudaGetLastError();
}

cudaError_t launch_resp_pruned(const Dims &dm, const PrunedImages &img, const void *x, void *gamma, int ldg,
                               int layout, cudaStream_t st, int src)
{
    constexpr size_t smem = PrunedSmem::bytes;
    static std::atomic<unsigned long long> smem_set{0};
    const cudaError_t attr = allow_smem(k_resp_pruned, smem, smem_set);
    if (attr != cudaSuccess) return attr;
    if (ldg != kPK) return cudaErrorInvalidValue;
    CUtensorMap xmap, gmap, gmap_lo;
    const bool g16 = layout != GL_F32;
    const long long plane = dm.BH() * dm.N * (long long)kPK;   // elements per plane (split)
    if (!make_tma_3d(&xmap, x, dm.x_bf16, kPD, dm.N, dm.BH(), kPRows) ||
        !make_tma_3d(&gmap, gamma, g16, kPK, dm.N, dm.BH(), kPRows))
        return cudaErrorInvalidValue;
    if (layout == GL_SPLIT) {
        if (!make_tma_3d(&gmap_lo, static_cast<__nv_bfloat16 *>(gamma) + plane, true, kPK, dm.N, dm.BH(), kPRows))
            return cudaErrorInvalidValue;
    } else {
        gmap_lo = gmap;
    }
    const long long items = dm.BH() * ((dm.N + kPRows - 1) / kPRows);
    const int grid = (int)(items < sm_count() ? items : sm_count());
    // run order stride: odd, near a fifth of the slices, coprime with their number
    const int nsl = (int)dm.BH();
    int pstride = (nsl / 5) | 1;
    auto gcd = [](int a, int b) { while (b) { const int t = a % b; a = b; b = t; } return a; };
    while (gcd(pstride, nsl) != 1) pstride += 2;
    unsigned int *flag = timeout_flag_dev();
    if (!flag) return cudaErrorMemoryAllocation;
    k_resp_pruned<<<grid, kPThreads, smem, st>>>(xmap, gmap, gmap_lo, dm.N, dm.H, nsl, dm.x_bf16, img.w, img.p,
                                                 img.c, layout, pstride, flag, img.list, img.ctl, img.cap, src, img.zq);
    return cudaGetLastError();
}

cudaError_t launch_resp_dense(const Dims &d0, const void *x0, void *g0, const Dims &d1, const void *x1, void *g1,
                              const PrunedImages &img, int layout, cudaStream_t st)
{
    const long long items = routing_tiles(d0.BH(), d0.N) + (x1 ? routing_tiles(d1.BH(), d1.N) : 0);
    if (items == 0) return cudaSuccess;   // no rows, nothing listed
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    {   // every listed tile on the tensor cores
        constexpr size_t smem = DenseTcSmem::bytes;
        static std::atomic<unsigned long long> smem_set{0};
        const cudaError_t e = allow_smem(k_resp_dense_tc, smem, smem_set);
        if (e != cudaSuccess) return e;
        DenseTcMaps maps;
        const bool g16 = layout != GL_F32;
        for (int s = 0; s < 2; ++s) {
            const bool one = s == 0 || !x1;   // without a second routing, source 1 repeats source 0
            const Dims &d = one ? d0 : d1;
            const void *x = one ? x0 : x1;
            void *g = one ? g0 : g1;
            const long long plane = d.BH() * d.N * (long long)kPK;   // elements of one plane (split)
            if (!make_tma_3d(&maps.x[s], x, d.x_bf16, kPD, d.N, d.BH(), kPRows) ||
                !make_tma_3d(&maps.g[s], g, g16, kPK, d.N, d.BH(), kPRows))
                return cudaErrorInvalidValue;
            if (layout == GL_SPLIT) {
                if (!make_tma_3d(&maps.glo[s], static_cast<__nv_bfloat16 *>(g) + plane, true, kPK, d.N, d.BH(),
                                 kPRows))
                    return cudaErrorInvalidValue;
            } else {
                maps.glo[s] = maps.g[s];
            }
        }
        unsigned int *flag = timeout_flag_dev();
        if (!flag) return cudaErrorMemoryAllocation;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(items < sm_count() ? items : sm_count()));   // one per SM
        cfg.blockDim = dim3(kTThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        const cudaError_t l = cudaLaunchKernelEx(&cfg, k_resp_dense_tc, maps, d0.x_bf16, d0.H,
                                                 (const unsigned char *)img.w3, (const float *)img.c, layout,
                                                 (const int2 *)img.list, img.ctl, img.list2, img.cap, flag);
        if (l != cudaSuccess) return l;
    }
    // the tiles it left (rows of large magnitude), exactly on the CUDA cores
    constexpr size_t smem = (size_t)kPRows * kDPitch * 4;
    static std::atomic<unsigned long long> smem_set{0};
    const cudaError_t e = allow_smem(k_resp_dense, smem, smem_set);
    if (e != cudaSuccess) return e;
    const DenseSrc s0{x0, g0, d0.N, d0.BH() * d0.N * (long long)kPK};
    const DenseSrc s1 = x1 ? DenseSrc{x1, g1, d1.N, d1.BH() * d1.N * (long long)kPK} : s0;
    cudaLaunchConfig_t cfg = {};
    const long long ctas = 2LL * sm_count();   // two resident per SM
    cfg.gridDim = dim3((unsigned)(items < ctas ? items : ctas));
    cfg.blockDim = dim3(kDThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_resp_dense, s0, s1, d0.x_bf16, d0.H, (const float4 *)img.p2,
                              (const float *)img.c, layout, (const int2 *)img.list2,
                              (const unsigned int *)(img.ctl + d0.H), img.cap);
}

} // namespace gma
