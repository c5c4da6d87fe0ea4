// Responsibilities (S1) on the tensor cores for 17 <= K <= 512 components (K = 128
// has the bounded routing of its own) and d_route = 64: every log-joint of every row,
// for any inputs.
//
// The posterior of the GMA explainer ("핵심 메커니즘": gamma_ik = p(z = k | x_i)
// under the diagonal GMM) is a softmax over the log-joints
//   l_ik = c_k - 1/2 sum_d ((x_id - mu_kd) / sigma_kd)^2
//        = c'_k + sum_d ( -1/2 a_kd x_id^2 + a_kd mu_kd x_id ),   a = 1/sigma^2,
// one product of [x^2 | x] (128 rows x 128) with W^T (128 x KN components) per
// tile of 128 rows, KN = K rounded up to 32, 64, 128, 256 or 512 (the components past K
// have W = 0 and c' = -1e30, so their posterior is 0).  As in the dense pass of the
// K = 128 routing, each fp32 operand is held as three bf16 planes (v = v0 + v1
// + v2 up to 2^-24 |v|) and the six plane products whose orders add up to at
// most two are accumulated in fp32, smallest first: every log-joint carries the
// rounding of an fp32 evaluation of the expanded form, a few fp32 units of
//   S_i = 1/2 A sum_d x_id^2 + M sum_d |x_id|   (A = max a, M = max |a mu| over the head).
// A row whose S_i exceeds kQSMax (|x| large against the components, where the
// expansion cancels) has its log-joints evaluated exactly instead, in the
// direct form, by the four threads that own the row.  With bf16 routing rows
// the values are one plane and their squares two, and the products of the zero
// planes are skipped.
//
// K <= 64: one persistent CTA of 16 warps per SM over a contiguous range of the
// (slice, tile) items of one routing; the head's planes of W (3 x KN x 256 B) are
// bulk-copied when the head changes.  Warp w owns TMEM lanes 32 (w % 4) .. + 31
// (rows) and quarter q = w / 4: operand positions 32 q .. 32 q + 31 (the squares,
// then the values, of features 16 q .. 16 q + 15) and components KN q / 4 .. of
// the result.  The operand planes are double-buffered in TMEM and the accumulator
// is read out before the next products are issued, so the products of item n + 1
// run while the warps take the softmax of item n and split the routing tile of
// item n + 2; the output tiles are double-buffered too, so a tile's TMA store
// drains while the next one is written.  Past 64 components the accumulator and a
// single operand buffer fill TMEM (k_resp_gtc_wide below, persistent too; past 256
// components a cluster of two CTAs per tile).
//
// Within each product the K steps of the values (odd) are issued before those of
// the squares (even): in ascending order some odd steps were measured to take W
// from the step before them (the products of the first tile of a CTA were exact,
// later ones not), and in this order every product matches its fp64 terms.
#include "gma_internal.cuh"
#include "gma_tc.cuh"

#include <float.h>

namespace gma {
namespace {

using namespace tc;

constexpr int kQD = 64, kQDP = kQD / 2;   // d_route, feature pairs
constexpr int kQRows = 128;
constexpr int kQThreads = 512;
constexpr float kQSMax = 4096.f;
constexpr float kQLog2e = 1.4426950408889634f;
constexpr float kQOff = -1.0e30f;         // c' of the components past K

// Operand position of feature f's square (its value sits 16 positions later):
// quarter q of the operand holds the squares of features 16 q .. 16 q + 15, then
// their values.
__host__ __device__ constexpr int gtc_pos(int f) { return 32 * (f >> 4) + (f & 15); }

// Per-head image: the three bf16 planes of W, each [KN][128] 128-byte-swizzled K-major
// (one bulk copy brings a plane), then c'[KN], then A and M.
template <int KN>
struct GtcImg {
    static constexpr uint32_t W = 3u * KN * 256u;
    static constexpr uint32_t C = KN * 4u + 16u;
    static constexpr uint32_t pitch = (W + C + 255u) & ~255u;
    // byte offset of operand position `pos` of component k in plane pl
    __host__ __device__ __forceinline__ static uint32_t off(int k, int pos, int pl)
    {
        return (uint32_t)pl * (KN * 256u) + sw128_offset(k, pos, KN, 2);
    }
};

size_t gtc_pitch(int KN)
{
    return KN <= 32    ? GtcImg<32>::pitch
           : KN <= 64  ? GtcImg<64>::pitch
           : KN <= 128 ? GtcImg<128>::pitch
                       : (size_t)(KN / 256) * GtcImg<256>::pitch;   // 512: two images of 256
}

// v = p0 + p1 + p2 + r with p0, p1, p2 bf16 and |r| <= 2^-24 |v|.
__device__ __forceinline__ void split3(float v, unsigned short (&p)[3])
{
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const __nv_bfloat16 b = __float2bfloat16_rn(v);
        p[j] = __bfloat16_as_ushort(b);
        v -= __bfloat162float(b);
    }
}

// Grid (H, images, KN / KB), KB * 4 threads (KB = min(KN, 64) components per block):
// component k = KN y + KB z + tid / 4 takes feature pairs 8 (tid % 4) .. + 7 from the packed
// parameters {s, s', -mu s, -mu' s'} and c_k that k_prep wrote, into image y of head h
// (past 256 components a head has two images of 256).  Every block of an image also
// takes the image's maxima A, M over all its components and writes them (the same
// values from each block).
template <int KN>
__global__ void __launch_bounds__((KN < 64 ? KN : 64) * 4)
    k_prep_gtc(int K, const float4 *__restrict__ prm, const float *__restrict__ cst, unsigned char *__restrict__ img)
{
    constexpr int KB = KN < 64 ? KN : 64, NT = KB * 4;
    __shared__ float red[2][NT / 32];
    const int h = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kl = KB * blockIdx.z + (tid >> 2), k = KN * blockIdx.y + kl, part = tid & 3;
    unsigned char *im = img + ((long long)h * gridDim.y + blockIdx.y) * GtcImg<KN>::pitch;
    float amu2 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int dp = 8 * part + j, f = 2 * dp;
        const float4 p = k < K ? prm[((long long)h * K + k) * kQDP + dp] : make_float4(0.f, 0.f, 0.f, 0.f);
        const float wa0 = -0.5f * p.x * p.x, wa1 = -0.5f * p.y * p.y, wb0 = -p.x * p.z, wb1 = -p.y * p.w;
        amu2 = fmaf(p.z, p.z, fmaf(p.w, p.w, amu2));
        unsigned short a0[3], a1[3], b0[3], b1[3];
        split3(wa0, a0);
        split3(wa1, a1);
        split3(wb0, b0);
        split3(wb1, b1);
#pragma unroll
        for (int pl = 0; pl < 3; ++pl) {
            *reinterpret_cast<uint32_t *>(im + GtcImg<KN>::off(kl, gtc_pos(f), pl)) =
                (uint32_t)a0[pl] | ((uint32_t)a1[pl] << 16);
            *reinterpret_cast<uint32_t *>(im + GtcImg<KN>::off(kl, gtc_pos(f) + 16, pl)) =
                (uint32_t)b0[pl] | ((uint32_t)b1[pl] << 16);
        }
    }
    for (int o = 1; o < 4; o <<= 1) amu2 += __shfl_xor_sync(0xffffffffu, amu2, o);   // the component's four threads
    float *c = reinterpret_cast<float *>(im + GtcImg<KN>::W);
    if (part == 0) c[kl] = k < K ? cst[(long long)h * K + k] - 0.5f * amu2 : kQOff;
    // the image's maxima of a and |a mu| over all its components
    float amax = 0.f, mmax = 0.f;
    const int k0 = KN * blockIdx.y, kend = min(K, k0 + KN);
    for (int e = tid; e < (kend - k0) * kQDP; e += NT) {
        const float4 p = prm[((long long)h * K + k0) * kQDP + e];
        amax = fmaxf(amax, fmaxf(p.x * p.x, p.y * p.y));
        mmax = fmaxf(mmax, fmaxf(fabsf(p.x * p.z), fabsf(p.y * p.w)));
    }
    for (int o = 1; o < 32; o <<= 1) {
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
    }
    if (lane == 0) {
        red[0][warp] = amax;
        red[1][warp] = mmax;
    }
    __syncthreads();
    if (tid == 0) {
        float a = 0.f, m = 0.f;
        for (int w = 0; w < NT / 32; ++w) {
            a = fmaxf(a, red[0][w]);
            m = fmaxf(m, red[1][w]);
        }
        c[KN] = a;
        c[KN + 1] = m;
        c[KN + 2] = 0.f;
        c[KN + 3] = 0.f;
    }
}

// One thread: the six plane products of a tile into the accumulator at d_tmem, smallest
// first, A's planes at a_tmem + 64 j and W's planes (K_N x 256 B each, 128-byte-swizzled
// K-major) described from bdesc; within each product the values' (odd) K steps before the
// squares' (even) ones (in ascending order some odd steps were measured to take W from the
// step before them).  XB16: bf16 rows, whose values' lower planes and squares' third plane
// are zero.  Every address and flag is fixed at compile time but for the three bases.
template <bool XB16, int KN>
__device__ __forceinline__ void issue_products(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t id)
{
#pragma unroll
    for (int q = 0; q < 6; ++q) {
        const uint32_t pa = q == 0 ? 2u : (q < 3 ? 1u : 0u);                // A plane
        const uint32_t pb = (q == 1 || q == 4) ? 1u : (q == 3 ? 2u : 0u);    // W plane
        if (XB16 && pa == 2) continue;
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) {
            const int kk = s8 < 4 ? 2 * s8 + 1 : 2 * (s8 - 4);
            if (XB16 && pa == 1 && (kk & 1)) continue;
            const uint32_t kb = kk * 32;   // byte offset of the K step in a row of W
            const uint32_t boff = pb * (uint32_t)(KN * 256) + (kb >> 7) * (KN * 128) + (kb & 127);
            const bool first = XB16 ? (q == 1 && s8 == 4) : (q == 0 && s8 == 0);
            mma_ts(0u, d_tmem, a_tmem + 64u * pa + 8u * kk, bdesc + (boff >> 4), id, first ? 0u : 1u);
        }
    }
}

// TMEM -> registers: 32 lanes x 32 bit, 8 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}

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

// The exact log-joints l_k = c_k - 1/2 sum_d ((x_d - mu_kd) / sigma_kd)^2 of components
// k0 .. k0 + n - 1 (those past K get kQOff) for routing row x (global memory), from the
// packed parameters {s, s', -mu s, -mu' s'} of head h: the path of rows too large for the
// expanded form, kept out of line.
__device__ __noinline__ void exact_row(const void *x, bool x_bf16, const float4 *__restrict__ prm,
                                       const float *__restrict__ cst, int h, int K, int k0, int n, float *l)
{
    float2 xr[kQDP];
    if (x_bf16) {
        const uint32_t *xw = static_cast<const uint32_t *>(x);
#pragma unroll
        for (int dp = 0; dp < kQDP; ++dp)
            xr[dp] = make_float2(__uint_as_float(xw[dp] << 16), __uint_as_float(xw[dp] & 0xffff0000u));
    } else {
        const float2 *x2 = static_cast<const float2 *>(x);
#pragma unroll
        for (int dp = 0; dp < kQDP; ++dp) xr[dp] = x2[dp];
    }
    for (int j = 0; j < n; ++j) {
        const int k = k0 + j;
        float v = kQOff;
        if (k < K) {
            const float4 *pk = prm + ((long long)h * K + k) * kQDP;
            float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int dp = 0; dp < kQDP; ++dp) {
                const float4 p = pk[dp];
                const float2 y = __ffma2_rn(xr[dp], make_float2(p.x, p.y), make_float2(p.z, p.w));
                a2 = __ffma2_rn(y, y, a2);
            }
            v = fmaf(-0.5f, a2.x + a2.y, cst[(long long)h * K + k]);
        }
        l[j] = v;
    }
}

template <int KN>
struct GtcSmem {
    static constexpr uint32_t W = GtcImg<KN>::W;        // three planes of W
    static constexpr uint32_t WA = (W + 1023u) & ~1023u;
    static constexpr uint32_t X = kQRows * kQD * 4;     // routing tile (fp32 worst case)
    static constexpr uint32_t O = kQRows * 128 * 4;     // one output tile (fp32 worst case, 128 columns)
    static constexpr uint32_t C = 2 * GtcImg<KN>::C;    // c', A, M of two heads
    static constexpr uint32_t EX = 4 * kQRows * 8;      // per quarter and row: (max, sum)
    static constexpr uint32_t SS = 2 * 4 * kQRows * 8;  // per item of two, quarter, row: (sum x^2, sum |x|)
    static constexpr size_t bytes = 1024 + (size_t)WA + X + 2 * (size_t)O + C + EX + SS + 64;
};
static_assert(GtcSmem<64>::bytes <= 232448, "small-K tensor-core routing: shared memory above the per-block limit");

template <int KN>
__global__ void __launch_bounds__(kQThreads, 1)
    k_resp_gtc(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap gmap,
               const __grid_constant__ CUtensorMap gmap_lo, int N, int H, int K, int tps, long long items,
               bool x_bf16, const void *__restrict__ xg, const unsigned char *__restrict__ img,
               const float4 *__restrict__ prm, const float *__restrict__ cst, int layout, int ow,
               unsigned int *timeout)
{
    constexpr int QC = KN / 4;   // components of a row per thread
    using SM = GtcSmem<KN>;
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    __shared__ float2 am_s[2];   // A, M of the heads in the two constants' buffers
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, cq = warp >> 2;
    const int i = 32 * qd + lane;   // row of the tile (TMEM lane)

    const long long per = (items + gridDim.x - 1) / gridDim.x;
    const long long it0 = min(items, (long long)blockIdx.x * per), it1 = min(items, it0 + per);
    if (it0 >= it1) return;
    const int cnt = (int)(it1 - it0);

    unsigned char *w_s = sm;
    unsigned char *xb = w_s + SM::WA;
    unsigned char *ob = xb + SM::X;   // two output tiles
    float *c_s = reinterpret_cast<float *>(ob + 2 * SM::O);   // [2][KN + 4]
    float2 *ex_s = reinterpret_cast<float2 *>(c_s + 2 * (KN + 4));
    float2 *ss_s = ex_s + 4 * kQRows;
    uint64_t *bar = reinterpret_cast<uint64_t *>(ss_s + 2 * 4 * kQRows);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 3);
    const uint32_t BAR_I = smem_addr(bar), BAR_X = smem_addr(bar + 1), BAR_M = smem_addr(bar + 2);
    const uint32_t xbytes = kQRows * kQD * (x_bf16 ? 2 : 4);
    const bool g_f32 = layout == GL_F32, g_split = layout == GL_SPLIT;
    const int ge = g_f32 ? 4 : 2;
    constexpr uint32_t LO = kQRows * 128 * 2;   // split: the lo plane's tile follows the hi plane's
    constexpr uint32_t D_COL = 384;             // the accumulator; operand planes at 192 b + 64 j
    uint32_t tbase = 0;
    auto slice_of = [&](int n) { return (int)((it0 + n) / tps); };
    auto tile_of = [&](int n) { return (int)((it0 + n) % tps); };
    auto load_x = [&](int n) {   // one thread
        mbar_expect_tx(BAR_X, xbytes);
        tma_load_3d(smem_addr(xb), &xmap, 0, tile_of(n) * kQRows, slice_of(n), BAR_X);
        if (!x_bf16) tma_load_3d(smem_addr(xb + kQRows * 128), &xmap, 32, tile_of(n) * kQRows, slice_of(n), BAR_X);
    };
    int nimg = 0;
    // the planes of W and the constants of `head` into buffer `buf` (every thread; no
    // products may be running)
    auto load_head = [&](int head, int buf) {
        if (tid == 0) {
            fence_proxy_async();   // earlier thread reads of the constants' buffer come first
            mbar_expect_tx(BAR_I, SM::W + GtcImg<KN>::C);
            const unsigned char *src = img + (long long)head * GtcImg<KN>::pitch;
            bulk_g2s(smem_addr(w_s), src, SM::W, BAR_I);
            bulk_g2s(smem_addr(c_s + buf * (KN + 4)), src + SM::W, GtcImg<KN>::C, BAR_I);
        }
        const bool got = mbar_wait(BAR_I, (uint32_t)(nimg & 1));
        ++nimg;
        if (tid == 0) am_s[buf] = make_float2(c_s[buf * (KN + 4) + KN], c_s[buf * (KN + 4) + KN + 1]);
        return got;
    };
    // item n's landed routing tile into operand buffer n % 2, and its rows' sums for S_i
    auto convert = [&](int n) {
        float2 xv[8];
        if (x_bf16) {
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const uint4 u = *reinterpret_cast<const uint4 *>(xb + sw128_offset(i, 16 * cq + 8 * g, kQRows, 2));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    xv[4 * g + e] = make_float2(__uint_as_float(w[e] << 16), __uint_as_float(w[e] & 0xffff0000u));
            }
        } else {
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float4 u = *reinterpret_cast<const float4 *>(xb + sw128_offset(i, 16 * cq + 4 * g, kQRows, 4));
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
        ss_s[(n & 1) * 4 * kQRows + cq * kQRows + i] = make_float2(s2.x + s2.y, s1.x + s1.y);
        tmem_wait_st();
    };
    // one thread: item n's products (operand buffer n % 2) into the accumulator
    const uint32_t id = idesc(128, KN, kFmtBF16);
    const uint64_t wdesc = sdesc_sw128(smem_addr(w_s));
    auto issue = [&](int n) {
        const uint32_t ab = tbase + 192u * (uint32_t)(n & 1);
        if (x_bf16)
            issue_products<true, KN>(tbase + D_COL, ab, wdesc, id);
        else
            issue_products<false, KN>(tbase + D_COL, ab, wdesc, id);
        mma_commit(BAR_M);
    };

    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 3; ++b) mbar_init(smem_addr(bar + b), 1);
        mbar_init_fence();
        load_x(0);
    }
    // both output tiles start as zeros: the columns past the components stay so
    for (int o = tid; o < (int)(2 * SM::O / 16); o += kQThreads)
        reinterpret_cast<uint4 *>(ob)[o] = make_uint4(0u, 0u, 0u, 0u);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    tbase = *tslot;
    int head = slice_of(0) % H;
    bool ok = load_head(head, 0);
    int hp = 0;                        // constants' buffer of item n's head
    uint32_t x_par = 0;                // tid 32: phase of the last routing tile fetched
    int m_issued = -1;                 // tid 0: the last item whose products were issued
    ok = mbar_wait(BAR_X, 0u) && ok;
    convert(0);
    fence_before_sync();
    ok = __syncthreads_and(ok) != 0;   // the planes are in TMEM, am_s is written
    fence_after_sync();
    if (tid == 0 && ok) {
        issue(0);
        m_issued = 0;
    }
    if (tid == 32 && ok && cnt > 1) {   // thread 32 moves the routing and output tiles from here on
        load_x(1);
        x_par = 1u;
    }

    float2 acc[QC / 2];                // the accumulator row of the previous item
    int hpprev = hp;
    // softmax of item m from acc into output tile m % 2 (rows beyond the magnitude limit
    // evaluated exactly first)
    auto softmax = [&](int m, int hpx) {
        const int bh = slice_of(m), row = tile_of(m) * kQRows + i;
        const float2 *sp = ss_s + (m & 1) * 4 * kQRows + i;
        const float sx2 = (sp[0].x + sp[kQRows].x) + (sp[2 * kQRows].x + sp[3 * kQRows].x);
        const float sx1 = (sp[0].y + sp[kQRows].y) + (sp[2 * kQRows].y + sp[3 * kQRows].y);
        const float2 am = am_s[hpx];
        const float *cb = c_s + hpx * (KN + 4) + QC * cq;   // c'_k of this thread's components
#pragma unroll
        for (int p = 0; p < QC / 2; ++p) acc[p] = __fadd2_rn(acc[p], make_float2(cb[2 * p], cb[2 * p + 1]));
        if (fmaf(0.5f * am.x, sx2, am.y * sx1) > kQSMax && row < N) {
            // the direct form ((x - mu) / sigma)^2 of this thread's components, from global memory
            const int h = bh % H;
            float2 xr[kQDP];
            if (x_bf16) {
                const uint32_t *xw = reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(xg) +
                                                                        ((long long)bh * N + row) * kQD);
#pragma unroll
                for (int dp = 0; dp < kQDP; ++dp)
                    xr[dp] = make_float2(__uint_as_float(xw[dp] << 16), __uint_as_float(xw[dp] & 0xffff0000u));
            } else {
                const float2 *x2 = reinterpret_cast<const float2 *>(static_cast<const float *>(xg) +
                                                                    ((long long)bh * N + row) * kQD);
#pragma unroll
                for (int dp = 0; dp < kQDP; ++dp) xr[dp] = x2[dp];
            }
#pragma unroll 1
            for (int j = 0; j < QC; ++j) {
                const int k = QC * cq + j;
                float l = kQOff;
                if (k < K) {
                    const float4 *pk = prm + ((long long)h * K + k) * kQDP;
                    float2 a2 = make_float2(0.f, 0.f);
#pragma unroll
                    for (int dp = 0; dp < kQDP; ++dp) {
                        const float4 p = pk[dp];
                        const float2 y = __ffma2_rn(xr[dp], make_float2(p.x, p.y), make_float2(p.z, p.w));
                        a2 = __ffma2_rn(y, y, a2);
                    }
                    l = fmaf(-0.5f, a2.x + a2.y, cst[(long long)h * K + k]);
                }
                if (j & 1) acc[j >> 1].y = l;
                else acc[j >> 1].x = l;
            }
        }
        float mq = -FLT_MAX;
#pragma unroll
        for (int p = 0; p < QC / 2; ++p) mq = fmaxf(mq, fmaxf(acc[p].x, acc[p].y));
        const float2 mneg = make_float2(-mq, -mq), l2e = make_float2(kQLog2e, kQLog2e);
        float2 sq2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < QC / 2; ++p) {
            const float2 t = __fmul2_rn(__fadd2_rn(acc[p], mneg), l2e);
            acc[p] = make_float2(ex2_sfu(t.x), ex2_sfu(t.y));
            sq2 = __fadd2_rn(sq2, acc[p]);
        }
        ex_s[cq * kQRows + i] = make_float2(mq, sq2.x + sq2.y);
        if (tid == 32)   // (the thread that stores the output tiles) item m - 2's has left shared memory
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
        __syncthreads();
        float2 e4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) e4[q] = ex_s[q * kQRows + i];
        const float mrow = fmaxf(fmaxf(e4[0].x, e4[1].x), fmaxf(e4[2].x, e4[3].x));
        float tot = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) tot = fmaf(e4[q].y, ex2_sfu((e4[q].x - mrow) * kQLog2e), tot);
        const float sc = ex2_sfu((mq - mrow) * kQLog2e) / tot;
        const float2 sc2 = make_float2(sc, sc);
        unsigned char *o = ob + (m & 1) * SM::O;
        if (g_f32) {
#pragma unroll
            for (int g = 0; g < QC / 4; ++g) {
                const float2 a = __fmul2_rn(acc[2 * g], sc2), b = __fmul2_rn(acc[2 * g + 1], sc2);
                *reinterpret_cast<float4 *>(o + sw128_offset(i, QC * cq + 4 * g, kQRows, 4)) =
                    make_float4(a.x, a.y, b.x, b.y);
            }
        } else {
            const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
            for (int g = 0; g < QC / 8; ++g) {
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
                const uint32_t off = sw128_offset(i, QC * cq + 8 * g, kQRows, 2);
                *reinterpret_cast<uint4 *>(o + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                if (g_split) *reinterpret_cast<uint4 *>(o + LO + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
            }
        }
        fence_proxy_async();   // the output tile, written by threads, is read by the TMA store
    };
    // one thread, after a CTA barrier that follows the softmax of item m: its output tile out
    auto finish = [&](int m) {
        const unsigned char *o = ob + (m & 1) * SM::O;
        const int bh = slice_of(m), t = tile_of(m);
        const int boxes = (ow * ge + 127) / 128;
        for (int a = 0; a < boxes; ++a) {
            tma_store_3d(&gmap, a * (128 / ge), t * kQRows, bh, smem_addr(o + a * (kQRows * 128)));
            if (g_split) tma_store_3d(&gmap_lo, a * (128 / ge), t * kQRows, bh, smem_addr(o + LO + a * (kQRows * 128)));
        }
        bulk_commit();
    };

    for (int n = 0; n < cnt && ok; ++n) {
        // item n's products are running; acc holds item n - 1's accumulator row
        if (n >= 1) softmax(n - 1, hpprev);
        if (n + 1 < cnt) {   // item n + 1's routing tile into the other operand buffer
            ok = mbar_wait(BAR_X, (uint32_t)((n + 1) & 1)) && ok;
            convert(n + 1);
        }
        // item n's accumulator row into registers (free for item n + 1's products after the
        // barrier below)
        ok = mbar_wait(BAR_M, (uint32_t)(n & 1)) && ok;
        fence_after_sync();
        {   // this thread's QC columns of the accumulator
            uint32_t r[QC];
            if constexpr (QC == 16)
                tmem_ld16(tmem_at(tbase, 32 * qd, D_COL + QC * cq), reinterpret_cast<uint32_t(&)[16]>(r));
            else
                tmem_ld8(tmem_at(tbase, 32 * qd, D_COL + QC * cq), reinterpret_cast<uint32_t(&)[8]>(r));
            tmem_wait_ld();
#pragma unroll
            for (int p = 0; p < QC / 2; ++p) acc[p] = make_float2(__uint_as_float(r[2 * p]), __uint_as_float(r[2 * p + 1]));
        }
        const int hpn = hp;
        if (n + 1 < cnt && slice_of(n + 1) % H != head) {   // item n + 1 is of another head
            head = slice_of(n + 1) % H;
            hp ^= 1;   // the constants of item n's head stay for its softmax
            ok = load_head(head, hp) && ok;
        }
        fence_before_sync();
        ok = __syncthreads_and(ok) != 0;   // operand planes written, accumulator read, softmax done
        fence_after_sync();
        if (tid == 0 && ok && n + 1 < cnt) {   // item n + 1's products
            issue(n + 1);
            m_issued = n + 1;
        }
        if (tid == 32 && ok) {
            // the routing tile was only read by threads (no proxy fence): item n + 2's comes in,
            // and item n - 1's output leaves
            if (n + 2 < cnt) {
                load_x(n + 2);
                x_par = (uint32_t)((n + 2) & 1);
            }
            if (n >= 1) finish(n - 1);
        }
        hpprev = hpn;
    }
    if (ok) {   // the last item's softmax and output
        softmax(cnt - 1, hpprev);
        ok = __syncthreads_and(ok) != 0;
        if (tid == 32 && ok) finish(cnt - 1);
    }
    // after a failed wait a routing tile or products may still be in flight: let them finish
    // (bounded) before TMEM and shared memory are released (a wait on a phase that has
    // completed returns at once)
    bool ok_end = ok;
    if (tid == 0 && !ok && m_issued >= 0) ok_end = mbar_wait(BAR_M, (uint32_t)(m_issued & 1)) && ok_end;
    if (tid == 32) {
        if (!ok) ok_end = mbar_wait(BAR_X, x_par) && ok_end;
        bulk_wait_all();
    }
    fence_before_sync();
    if (__syncthreads_and(ok_end) == 0 && tid == 0) report_timeout(timeout);
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ---- KN = 128 or 256 (65 <= K <= 256, d = 64): one product per plane pair, N = KN ----
// ---- and K up to 512 as clusters of two CTAs, 256 components each                   ----
//
// Persistent: one CTA (NH = 1), or a cluster of two (NH = 2, CTA r taking components
// 256 r ..), per SM pair, over a contiguous range of the (slice, tile) items.  The
// accumulator holds all KN log-joints of a row (TMEM columns 256 ..; the operand planes at
// 0 .. 191, the next tile's rows at 192 .. 255).  Plane 1 of the head's W stays in buffer
// P for all its tiles; for each tile plane 0 comes into O and plane 2 into Q (with one
// output half, Q keeps plane 2 for the head) as soon as the previous tile's output halves
// have left them.  The products run in the order the planes are at hand: (1,1), (0,1),
// then (2,0), (1,0), then (0,2) and last (0,0); every term before the last is at most
// 2^-8 of the log-joint, so the order keeps the rounding of one fp32 evaluation.  The routing rows go
// from global memory to registers, the next tile's while the products run, and wait in
// TMEM until that tile starts.  Each thread owns KN / 4 components of its row; with two
// CTAs each row's maximum and sum pass to the other CTA through distributed shared memory;
// the posteriors leave in halves of 128 components, the first from O, the second from Q,
// stored by thread 32 while thread 0 issues the next tile's products.
template <int KN>
struct GtcWSmem {
    static constexpr uint32_t WB = KN * 256;             // one plane of W
    static constexpr uint32_t O = kQRows * 128 * 4;      // plane 0, then half of the output tile (fp32
                                                         // worst case)
    static constexpr uint32_t C = GtcImg<KN>::C;         // c', A, M
    static constexpr uint32_t EX = 4 * kQRows * 8;       // per quarter and row: (max, sum)
    static constexpr uint32_t SS = 4 * kQRows * 8;       // per quarter and row: (sum x^2, sum |x|)
    static constexpr uint32_t XS = 2 * kQRows * 8;       // per tile parity and row: the CTA's (max, sum)
    static constexpr size_t bytes = 1024 + 2 * (size_t)WB + O + C + EX + SS + XS + 64;
};
static_assert(GtcWSmem<256>::bytes <= 232448, "wide tensor-core routing: shared memory above the per-block limit");

// All threads of both CTAs of the cluster (release / acquire of shared memory).
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// A float2 of the shared memory of CTA `rank` of the cluster, at this CTA's address p.
__device__ __forceinline__ float2 ld_cluster_f2(const void *p, uint32_t rank)
{
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(p)), "r"(rank));
    float2 v;
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(ra) : "memory");
    return v;
}

template <int KN, int NH>
__global__ void __launch_bounds__(kQThreads, 1)
    k_resp_gtc_wide(const __grid_constant__ CUtensorMap gmap, const __grid_constant__ CUtensorMap gmap_lo, int N,
                    int H, int K, int tps, long long items, bool x_bf16, const void *__restrict__ xg,
                    const unsigned char *__restrict__ img, const float4 *__restrict__ prm,
                    const float *__restrict__ cst, int layout, int ow, unsigned int *timeout)
{
    constexpr int QC = KN / 4;
    constexpr int HALVES = KN / 128, QPH = 4 / HALVES;   // output halves; quarters of a row per half
    constexpr bool QOUT = HALVES == 2;                   // the second half leaves through buffer Q
    using SM = GtcWSmem<KN>;
    using IM = GtcImg<KN>;
    static_assert(SM::O >= SM::WB, "plane 0 fits in the output tile's space");
    static_assert(!QOUT || SM::WB >= SM::O, "buffer Q holds the second half of the output tile");
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, cq = warp >> 2;
    const int i = 32 * qd + lane;   // row of the tile (TMEM lane)
    const uint32_t rank = NH == 1 ? 0u : cluster_rank();
    const int kbase = KN * (int)rank;   // this CTA's first component

    // the CTA (pair) takes a contiguous range of the (slice, tile) items
    const long long groups = gridDim.x / NH, grp = blockIdx.x / NH;
    const long long per = (items + groups - 1) / groups;
    const long long it0 = min(items, grp * per), it1 = min(items, it0 + per);
    if (it0 >= it1) return;   // (both CTAs of a pair alike)
    const int cnt = (int)(it1 - it0);

    unsigned char *wp = sm;              // buffer P: plane 1 of the head
    unsigned char *wq = sm + SM::WB;     // buffer Q: plane 2 while the products run, then (two
                                         // halves) the second output half
    unsigned char *ob = wq + SM::WB;     // plane 0 while the products run, then the (first) output half
    float *c_s = reinterpret_cast<float *>(ob + SM::O);       // [KN + 4]
    float2 *ex_s = reinterpret_cast<float2 *>(c_s + KN + 4);  // [4][128]
    float2 *ss_s = ex_s + 4 * kQRows;                         // [4][128]
    float2 *xs_s = ss_s + 4 * kQRows;                         // [2][128], by tile parity
    uint64_t *bar = reinterpret_cast<uint64_t *>(xs_s + 2 * kQRows);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 4);
    // the head's plane 1 (and plane 2 with one output half) and constants landed; the tile's
    // plane 0 landed; its plane 2 landed (two halves); products done
    const uint32_t BAR_W = smem_addr(bar), BAR_O = smem_addr(bar + 1), BAR_D = smem_addr(bar + 2);
    const uint32_t BAR_Q = smem_addr(bar + 3);
    const bool g_f32 = layout == GL_F32, g_split = layout == GL_SPLIT;
    const int ge = g_f32 ? 4 : 2;
    constexpr uint32_t LO = kQRows * 128 * 2;   // split: the lo plane's half tile follows the hi plane's
    constexpr uint32_t D_COL = 256, X_COL = 192;   // the accumulator; the next tile's rows (fp32)

    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 4; ++b) mbar_init(smem_addr(bar + b), 1);
        mbar_init_fence();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *tslot;

    // features 16 cq .. + 15 of row i of an item, straight from global memory (zeros past N)
    auto load_rows = [&](long long it, float2 (&xv)[8]) {
        const long long bh = it / tps;
        const int row = (int)(it % tps) * kQRows + i;
        if (row >= N) {
#pragma unroll
            for (int c = 0; c < 8; ++c) xv[c] = make_float2(0.f, 0.f);
            return;
        }
        const long long e = (bh * N + row) * kQD + 16 * cq;
        if (x_bf16) {
            const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(xg) + e);
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const uint4 u = __ldg(p + g);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    xv[4 * g + q] = make_float2(__uint_as_float(w[q] << 16), __uint_as_float(w[q] & 0xffff0000u));
            }
        } else {
            const float4 *p = reinterpret_cast<const float4 *>(static_cast<const float *>(xg) + e);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float4 u = __ldg(p + g);
                xv[2 * g] = make_float2(u.x, u.y);
                xv[2 * g + 1] = make_float2(u.z, u.w);
            }
        }
    };
    // one thread: the products of pa with the plane of W at w, the values' (odd) K steps first
    // (issued in ascending order, some odd steps were measured to take W from the step before
    // them); `first` clears the accumulator
    const uint32_t id = idesc(128, KN, kFmtBF16);
    bool first = true;
    auto prods = [&](uint32_t pa, const unsigned char *w) {
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int kk = s < 4 ? 2 * s + 1 : 2 * (s - 4);
            if (x_bf16 && pa == 1 && (kk & 1)) continue;   // bf16 rows: the values' plane 1 is zero
            const uint32_t kb = kk * 32;   // byte offset of the K step in a row of W
            const uint32_t boff = (kb >> 7) * (KN * 128) + (kb & 127);
            mma_ts(0u, tbase + D_COL, tbase + 64u * pa + 8u * kk, sdesc_sw128(smem_addr(w + boff)), id,
                   first ? 0u : 1u);
            first = false;
        }
    };

    float2 xv[8];
    load_rows(it0, xv);
    int head = -1;
    uint32_t nw = 0;                       // head loads so far
    const unsigned char *src = img;        // the head's image
    bool ok = true;
    // (thread 0) copies or products whose wait has not completed, and their phases; (thread 32,
    // which moves the output tiles and the per-tile planes) whether and with which phase it
    // last requested plane 0 and plane 2
    bool w_pend = false, d_pend = false;
    uint32_t w_par = 0, d_par = 0;
    bool o_req = false, q_req = false;
    uint32_t o_rpar = 0, q_rpar = 0;
    for (int j = 0; j < cnt; ++j) {
        const long long it = it0 + j;
        const int bh = (int)(it / tps), t = (int)(it % tps), h = bh % H;
        const int row = t * kQRows + i;
        if (j > 0) {   // this tile's rows, parked in TMEM while the previous tile's products ran
            uint32_t w[16];
            tmem_ld16(tmem_at(tbase, 32 * qd, X_COL + 16 * cq), w);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 8; ++c) xv[c] = make_float2(__uint_as_float(w[2 * c]), __uint_as_float(w[2 * c + 1]));
        }
        if (h != head) {   // the previous tile's products and softmax are done (the barriers below)
            head = h;
            src = img + ((long long)h * NH + rank) * IM::pitch;
            if (tid == 0 && ok) {
                fence_proxy_async();
                mbar_expect_tx(BAR_W, (QOUT ? 1 : 2) * SM::WB + SM::C);
                bulk_g2s(smem_addr(wp), src + IM::off(0, 0, 1), SM::WB, BAR_W);
                if (!QOUT) bulk_g2s(smem_addr(wq), src + IM::off(0, 0, 2), SM::WB, BAR_W);
                bulk_g2s(smem_addr(c_s), src + IM::W, SM::C, BAR_W);
                w_pend = true;
                w_par = nw & 1;
            }
            if (ok) ok = mbar_wait(BAR_W, nw & 1);
            if (tid == 0 && ok) w_pend = false;
            ++nw;
        }
        if (tid == 32 && ok) {   // the previous tile's output halves have left O (and Q): the
                                 // tile's plane 0 (and plane 2) come in
            if constexpr (QOUT)
                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");   // the first half's group
            else
                bulk_wait_read();
            mbar_expect_tx(BAR_O, SM::WB);
            bulk_g2s(smem_addr(ob), src + IM::off(0, 0, 0), SM::WB, BAR_O);
            o_req = true;
            o_rpar = j & 1;
            if constexpr (QOUT) {
                bulk_wait_read();
                mbar_expect_tx(BAR_Q, SM::WB);
                bulk_g2s(smem_addr(wq), src + IM::off(0, 0, 2), SM::WB, BAR_Q);
                q_req = true;
                q_rpar = j & 1;
            }
        }
        {   // the rows' squares and values into the three planes of A, and their sums for S_i
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
#pragma unroll
            for (int jj = 0; jj < 3; ++jj) tmem_st16(tmem_at(tbase, 32 * qd, 64 * jj + 16 * cq), pw[jj]);
            ss_s[cq * kQRows + i] = make_float2(s2.x + s2.y, s1.x + s1.y);
            tmem_wait_st();
        }
        fence_before_sync();
        ok = __syncthreads_and(ok) != 0;   // the planes are in TMEM, the accumulator was read
        fence_after_sync();
        if (tid == 0 && ok) {   // the products in the order the planes are at hand: plane 1 is
                                // resident, plane 0 lands in O, plane 2 in Q (or is resident)
            first = true;
            d_pend = true;
            d_par = j & 1;
            prods(1, wp);                          // (1,1)
            prods(0, wp);                          // (0,1)
            if (mbar_wait(BAR_O, (uint32_t)(j & 1))) {
                if (!x_bf16) prods(2, ob);         // (2,0); zero for bf16 rows
                prods(1, ob);                      // (1,0)
                if (!QOUT || mbar_wait(BAR_Q, (uint32_t)(j & 1))) {
                    prods(0, wq);                  // (0,2)
                    prods(0, ob);                  // (0,0), the largest last
                } else {
                    ok = false;
                }
            } else {
                ok = false;
            }
            mma_commit(BAR_D);                     // also after a failed wait: the products issued
        }
        if (j + 1 < cnt) {   // the next tile's rows, read while the products run, parked in TMEM
            float2 xn[8];
            load_rows(it + 1, xn);
            uint32_t w[16];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                w[2 * c] = __float_as_uint(xn[c].x);
                w[2 * c + 1] = __float_as_uint(xn[c].y);
            }
            tmem_st16(tmem_at(tbase, 32 * qd, X_COL + 16 * cq), w);
            tmem_wait_st();
        }
        if (ok) ok = mbar_wait(BAR_D, (uint32_t)(j & 1));
        if (tid == 0 && ok) d_pend = false;
        fence_after_sync();
        float2 acc[QC / 2];
#pragma unroll
        for (int b = 0; b < QC / 16; ++b) {
            uint32_t r[16];
            tmem_ld16(tmem_at(tbase, 32 * qd, D_COL + QC * cq + 16 * b), r);
            tmem_wait_ld();
#pragma unroll
            for (int p = 0; p < 8; ++p)
                acc[8 * b + p] = make_float2(__uint_as_float(r[2 * p]), __uint_as_float(r[2 * p + 1]));
        }
        // log-joints (rows beyond the magnitude limit exactly), then the softmax over the four
        // quarters of the row (and the other CTA's components)
        const float2 am = make_float2(c_s[KN], c_s[KN + 1]);
        const float2 *sp = ss_s + i;
        const float sx2 = (sp[0].x + sp[kQRows].x) + (sp[2 * kQRows].x + sp[3 * kQRows].x);
        const float sx1 = (sp[0].y + sp[kQRows].y) + (sp[2 * kQRows].y + sp[3 * kQRows].y);
        const float *cb = c_s + QC * cq;
#pragma unroll
        for (int p = 0; p < QC / 2; ++p) acc[p] = __fadd2_rn(acc[p], make_float2(cb[2 * p], cb[2 * p + 1]));
        if (fmaf(0.5f * am.x, sx2, am.y * sx1) > kQSMax && row < N) {
            float lex[QC];
            const long long xo = ((long long)bh * N + row) * kQD;
            exact_row(x_bf16 ? (const void *)(static_cast<const uint16_t *>(xg) + xo)
                             : (const void *)(static_cast<const float *>(xg) + xo),
                      x_bf16, prm, cst, h, K, kbase + QC * cq, QC, lex);
#pragma unroll
            for (int p = 0; p < QC / 2; ++p) acc[p] = make_float2(lex[2 * p], lex[2 * p + 1]);
        }
        float mq = -FLT_MAX;
#pragma unroll
        for (int p = 0; p < QC / 2; ++p) mq = fmaxf(mq, fmaxf(acc[p].x, acc[p].y));
        const float2 mneg = make_float2(-mq, -mq), l2e = make_float2(kQLog2e, kQLog2e);
        float2 sq2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < QC / 2; ++p) {
            const float2 tt = __fmul2_rn(__fadd2_rn(acc[p], mneg), l2e);
            acc[p] = make_float2(ex2_sfu(tt.x), ex2_sfu(tt.y));
            sq2 = __fadd2_rn(sq2, acc[p]);
        }
        ex_s[cq * kQRows + i] = make_float2(mq, sq2.x + sq2.y);
        ok = __syncthreads_and(ok) != 0;
        {
            float2 e4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) e4[q] = ex_s[q * kQRows + i];
            float mrow = fmaxf(fmaxf(e4[0].x, e4[1].x), fmaxf(e4[2].x, e4[3].x));
            float tot = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) tot = fmaf(e4[q].y, ex2_sfu((e4[q].x - mrow) * kQLog2e), tot);
            if constexpr (NH == 2) {   // the row's maximum and sum over the other CTA's components too
                float2 *xs = xs_s + (j & 1) * kQRows;   // by tile parity: the other CTA reads it before
                if (cq == 0) xs[i] = make_float2(mrow, tot);   // this CTA writes the slot again
                cluster_sync();
                const float2 pe = ld_cluster_f2(xs + i, rank ^ 1u);
                const float m2 = fmaxf(mrow, pe.x);
                tot = tot * ex2_sfu((mrow - m2) * kQLog2e) + pe.y * ex2_sfu((pe.x - m2) * kQLog2e);
                mrow = m2;
            }
            const float sc = ex2_sfu((mq - mrow) * kQLog2e) / tot;
            const float2 sc2 = make_float2(sc, sc);
#pragma unroll
            for (int p = 0; p < QC / 2; ++p) acc[p] = __fmul2_rn(acc[p], sc2);
        }
        // the posteriors in halves of 128 components, quarters QPH hf .. QPH hf + QPH - 1 writing
        // half hf: the first into O, the second into Q (both free: the products are done); thread
        // 32 stores them as two groups, which drain while the next tile is split and multiplied
        {
            const int hf = cq / QPH;
            unsigned char *hb = hf == 0 ? ob : wq;
            if (ok) {
                const int c0 = QC * (cq % QPH);   // this thread's columns in the half tile
                if (g_f32) {
#pragma unroll
                    for (int g = 0; g < QC / 4; ++g)
                        *reinterpret_cast<float4 *>(hb + sw128_offset(i, c0 + 4 * g, kQRows, 4)) =
                            make_float4(acc[2 * g].x, acc[2 * g].y, acc[2 * g + 1].x, acc[2 * g + 1].y);
                } else {
                    const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
                    for (int g = 0; g < QC / 8; ++g) {
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float2 v = acc[4 * g + u];
                            __nv_bfloat162 b = __floats2bfloat162_rn(v.x, v.y);
                            hw[u] = *reinterpret_cast<const uint32_t *>(&b);
                            const float2 r = __ffma2_rn(
                                make_float2(__uint_as_float(hw[u] << 16), __uint_as_float(hw[u] & 0xffff0000u)), m1, v);
                            b = __floats2bfloat162_rn(r.x, r.y);
                            lw[u] = *reinterpret_cast<const uint32_t *>(&b);
                        }
                        const uint32_t off = sw128_offset(i, c0 + 8 * g, kQRows, 2);
                        *reinterpret_cast<uint4 *>(hb + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        if (g_split) *reinterpret_cast<uint4 *>(hb + LO + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                }
                fence_proxy_async();   // the half tile, written by threads, is read by the TMA store
            }
        }
        fence_before_sync();
        __syncthreads();
        if (tid == 32 && ok) {
            const int pb = 128 / ge;   // columns of one 128-byte box
            for (int hf = 0; hf < HALVES; ++hf) {
                const unsigned char *hb = hf == 0 ? ob : wq;
                for (int a = 0; a < 128 / pb; ++a) {
                    const int x0 = kbase + 128 * hf + a * pb;
                    if (x0 >= ow) break;
                    tma_store_3d(&gmap, x0, t * kQRows, bh, smem_addr(hb + a * (kQRows * 128)));
                    if (g_split) tma_store_3d(&gmap_lo, x0, t * kQRows, bh, smem_addr(hb + LO + a * (kQRows * 128)));
                }
                bulk_commit();   // one group per half
            }
        }
    }
    if (tid == 0 && !ok) {
        // after a failed wait a copy or products may still be in flight: let them end (bounded;
        // a wait on a phase that has completed returns at once)
        if (w_pend) mbar_wait(BAR_W, w_par);
        if (d_pend) mbar_wait(BAR_D, d_par);
        report_timeout(timeout);
    }
    if (tid == 32) {
        if (!ok) {
            if (o_req) mbar_wait(BAR_O, o_rpar);
            if (q_req) mbar_wait(BAR_Q, q_rpar);
        }
        bulk_wait_read();   // the output tiles have left shared memory
    }
    fence_before_sync();
    __syncthreads();
    if constexpr (NH == 2) cluster_sync();   // the other CTA has read this one's last (max, sum)
    if (warp == 0) tmem_dealloc(tbase, 512);
}

int gtc_width(int K) { return K <= 32 ? 32 : (K <= 64 ? 64 : (K <= 128 ? 128 : (K <= 256 ? 256 : 512))); }

} // namespace

bool resp_gtc_applies(const Dims &dm)
{
    return dm.D == kQD && dm.K >= 17 && dm.K <= 512 && !resp_pruned_applies(dm);
}

size_t gtc_image_bytes(const Dims &dm) { return resp_gtc_applies(dm) ? dm.H * gtc_pitch(gtc_width(dm.K)) : 0; }

cudaError_t launch_prep_gtc(const Dims &dm, const float4 *prm, const float *cst, unsigned char *img, cudaStream_t st)
{
    if (!resp_gtc_applies(dm)) return cudaErrorInvalidValue;
    switch (gtc_width(dm.K)) {
    case 32: k_prep_gtc<32><<<dim3(dm.H, 1, 1), 32 * 4, 0, st>>>(dm.K, prm, cst, img); break;
    case 64: k_prep_gtc<64><<<dim3(dm.H, 1, 1), 64 * 4, 0, st>>>(dm.K, prm, cst, img); break;
    case 128: k_prep_gtc<128><<<dim3(dm.H, 1, 2), 64 * 4, 0, st>>>(dm.K, prm, cst, img); break;
    case 256: k_prep_gtc<256><<<dim3(dm.H, 1, 4), 64 * 4, 0, st>>>(dm.K, prm, cst, img); break;
    default: k_prep_gtc<256><<<dim3(dm.H, 2, 4), 64 * 4, 0, st>>>(dm.K, prm, cst, img); break;   // two images
    }
    return cudaGetLastError();
}

bool resp_gtc_output_ok(const Dims &dm, int ldg, int layout)
{
    // rows of the output start on 16-byte boundaries (a TMA store's strides); the output
    // tile covers 128 columns, or KN for the wide form
    const int KN = gtc_width(dm.K);
    return ldg <= (KN < 128 ? 128 : KN) && (layout == GL_F32 ? ldg % 4 == 0 : ldg % 8 == 0);
}

template <int KN>
cudaError_t launch_gtc(const Dims &dm, const unsigned char *img, const float4 *prm, const float *cst, const void *x,
                       void *gamma, int ldg, int layout, cudaStream_t st)
{
    constexpr bool wide = KN > 64;
    constexpr int NH = KN > 256 ? 2 : 1;   // CTAs per tile of the wide form
    constexpr int KC = wide ? KN / NH : 64;
    const size_t smem = wide ? GtcWSmem<KC>::bytes : GtcSmem<(wide ? 64 : KN)>::bytes;
    static std::atomic<unsigned long long> smem_set{0};
    cudaError_t attr;
    if constexpr (wide)
        attr = allow_smem(k_resp_gtc_wide<KC, NH>, smem, smem_set);
    else
        attr = allow_smem(k_resp_gtc<KN>, smem, smem_set);
    if (attr != cudaSuccess) return attr;
    const int tps = (dm.N + kQRows - 1) / kQRows;
    const long long items = dm.BH() * tps;
    if (items == 0) return cudaSuccess;
    CUtensorMap xmap, gmap, gmap_lo;
    const bool g16 = layout != GL_F32;
    const long long plane = dm.BH() * dm.N * (long long)ldg;   // elements per plane (split)
    if (!make_tma_3d(&xmap, x, dm.x_bf16, kQD, dm.N, dm.BH(), kQRows) ||
        !make_tma_3d(&gmap, gamma, g16, ldg, dm.N, dm.BH(), kQRows))
        return cudaErrorInvalidValue;
    if (layout == GL_SPLIT) {
        if (!make_tma_3d(&gmap_lo, static_cast<__nv_bfloat16 *>(gamma) + plane, true, ldg, dm.N, dm.BH(), kQRows))
            return cudaErrorInvalidValue;
    } else {
        gmap_lo = gmap;
    }
    unsigned int *flag = timeout_flag_dev();
    if (!flag) return cudaErrorMemoryAllocation;
    if (items * NH > 0x7fffffffLL) return cudaErrorInvalidValue;
    if constexpr (!wide) {   // persistent: one CTA per SM over a contiguous range of the tiles
        const int grid = (int)(items < sm_count() ? items : sm_count());
        k_resp_gtc<KN><<<grid, kQThreads, smem, st>>>(xmap, gmap, gmap_lo, dm.N, dm.H, dm.K, tps, items, dm.x_bf16, x,
                                                      img, prm, cst, layout, ldg, flag);
        return cudaGetLastError();
    } else if constexpr (NH == 1) {   // persistent too
        const int grid = (int)(items < sm_count() ? items : sm_count());
        k_resp_gtc_wide<KC, 1><<<grid, kQThreads, smem, st>>>(gmap, gmap_lo, dm.N, dm.H, dm.K, tps, items, dm.x_bf16,
                                                               x, img, prm, cst, layout, ldg, flag);
        return cudaGetLastError();
    } else {   // clusters of two CTAs, each pair over a range of the tiles
        const long long pairs = items < sm_count() / 2 ? items : sm_count() / 2;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(pairs * NH));
        cfg.blockDim = dim3(kQThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = NH;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, k_resp_gtc_wide<KC, NH>, gmap, gmap_lo, dm.N, dm.H, dm.K, tps, items,
                                  dm.x_bf16, x, img, prm, cst, layout, ldg, flag);
    }
}

cudaError_t launch_resp_gtc(const Dims &dm, const unsigned char *img, const float4 *prm, const float *cst,
                            const void *x, void *gamma, int ldg, int layout, cudaStream_t st)
{
    if (!resp_gtc_applies(dm) || !resp_gtc_output_ok(dm, ldg, layout)) return cudaErrorInvalidValue;
    switch (gtc_width(dm.K)) {
    case 32: return launch_gtc<32>(dm, img, prm, cst, x, gamma, ldg, layout, st);
    case 64: return launch_gtc<64>(dm, img, prm, cst, x, gamma, ldg, layout, st);
    case 128: return launch_gtc<128>(dm, img, prm, cst, x, gamma, ldg, layout, st);
    case 256: return launch_gtc<256>(dm, img, prm, cst, x, gamma, ldg, layout, st);
    default: return launch_gtc<512>(dm, img, prm, cst, x, gamma, ldg, layout, st);
    }
}

} // namespace gma
