// Tensor-core (tcgen05 / TMEM) path of the causal and bidirectional forms for K = 128.
//
// The causal variant of the GMA explainer ("변형 및 학습": prefix sums so that
// O_i depends on j <= i only) is evaluated in the chunkwise-parallel form of
// the linear-attention page ("선형 어텐션 원리 정리", "쉽게 이해하기"): chunks of
// C = 128 tokens, dense products inside a chunk, and a carried memory
// [Vt | Z] between chunks.
//
// K components are taken in groups of 128 (K = 256 .. 512: the contraction over
// components accumulates group by group into the same tensor-memory accumulator,
// and the chunk contribution is written group by group; K < 128: operands padded
// with zero components to 128).
//
//   k_chunk_state_tc : L_c = Gamma_K,c^T [V_c | 1]                 (chunk contribution)
//   k_scan_split     : S_{c-1} = state_in + sum_{c' < c} L_c'        (carried memory)
//   k_chunk_out_tc   : [P | U] = Gamma_Q,c [Gamma_K,c ; Vt_{c-1}^T]^T
//                      P_m = P with j > i zeroed;   U += P_m V_c
//                      O_i = U_i / (sum_j P_m[i][j] + Gamma_Q,i . Z_{c-1} + eps)
// The bidirectional read is k_chunk_out_tc without P: U = Gamma_Q [Vt | Z] with
// the sequence's total memory.
//
// Every contraction is a chain of tcgen05.mma kind::f16 instructions (M = 128,
// bf16 operands, fp32 accumulator in TMEM); B operands sit in shared memory in
// the K-major 128-byte-swizzled layout.  A tcgen05.mma costs about the same
// time for any N up to 256, and its k-step is 16 bf16 against 8 tf32, so the
// fp32-operand path holds every operand x as two bf16 planes
//   SPLIT = true :  hi = RN_bf16(x), lo = RN_bf16(x - hi)   (16 significant bits,
//                   |x - hi - lo| <= 2^-17 |x|);  a b ~ hi hi + hi lo + lo hi
//                   (three passes; the dropped lo lo is below 2^-16 |a b|),
//   SPLIT = false:  bf16 operands, one plane, one pass.
// Gamma_Q and Gamma_K arrive in this form from the routing kernels and the
// carried memory from k_scan_split; V and P_m are split by threads.  The row
// sums of P_m are taken on CUDA cores from the same split values the tensor
// core multiplies; Gamma_Q . Z is one more product, of both planes of Gamma_Q
// against the hi and lo rows of Z (all four cross terms, in two columns).
#include "gma_internal.cuh"
#include "gma_tc.cuh"

#include <cuda.h>

namespace gma {
namespace {

using namespace tc;

constexpr int kC = 128;                      // chunk rows (= MMA M)
constexpr int kK = 128;                      // components per group (the MMA M / contraction tile)
constexpr int kKSteps = kK * 2 / 32;         // MMA k-steps (16 bf16 each) of a 128-deep contraction
constexpr uint32_t kRowB = kK * 2;           // bytes of one 128-element bf16 row
constexpr uint32_t kAtom = kC * 128;         // bytes of one 128-row atom column

__device__ __forceinline__ uint32_t pack_bf16(__nv_bfloat16 a, __nv_bfloat16 b)
{
    return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// One MMA pass D (+)= A B^T over a 128-deep contraction.  B: K-major SW128 bf16
// tile of n rows whose 128-byte atom columns lie bstride bytes apart.  A: TMEM
// columns from a_col (two bf16 per column), or a K-major SW128 bf16 tile of
// 128 rows in shared memory (atom columns astride apart).
__device__ __forceinline__ void mma_pass_ss(uint32_t d, const unsigned char *a, uint32_t astride,
                                            const unsigned char *b, uint32_t n, uint32_t bstride, bool accumulate)
{
    const uint32_t id = idesc(128, n, kFmtBF16);
#pragma unroll 1
    for (int kk = 0; kk < kKSteps; ++kk) {
        const uint32_t kb = kk * 32;
        const uint32_t aoff = (kb >> 7) * astride + (kb & 127), boff = (kb >> 7) * bstride + (kb & 127);
        mma_ss(0u, d, sdesc_sw128(smem_addr(a + aoff)), sdesc_sw128(smem_addr(b + boff)), id,
               (accumulate || kk > 0) ? 1u : 0u);
    }
}

// 32 consecutive A-operand values of this thread's TMEM lane (operand columns
// j0 .. j0 + 31) as packed bf16: the hi parts at column a_hi + j0 / 2 and, for
// split operands, the lo parts at a_lo + j0 / 2.  Returns the sum of the values
// the tensor core will use (hi + lo).
template <bool SPLIT>
__device__ __forceinline__ float put_a32(uint32_t tbase, uint32_t lane0, uint32_t a_hi, uint32_t a_lo, int j0,
                                         const float (&x)[32])
{
    uint32_t ph[16], pl[16];
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        __nv_bfloat16 h0, l0, h1, l1;
        split_bf16(x[2 * j], h0, l0);
        split_bf16(x[2 * j + 1], h1, l1);
        ph[j] = pack_bf16(h0, h1);
        pl[j] = pack_bf16(l0, l1);
        sum += __bfloat162float(h0) + __bfloat162float(h1);
        if (SPLIT) sum += __bfloat162float(l0) + __bfloat162float(l1);
    }
    tmem_st16(tmem_at(tbase, lane0, a_hi + j0 / 2), ph);
    if (SPLIT) tmem_st16(tmem_at(tbase, lane0, a_lo + j0 / 2), pl);
    return sum;
}

// One element of a bf16 operand tile at byte offset off: hi image at `hi`, lo image at `lo`.
template <bool SPLIT>
__device__ __forceinline__ void put_split(unsigned char *hi, unsigned char *lo, uint32_t off, float x)
{
    __nv_bfloat16 h, l;
    split_bf16(x, h, l);
    *reinterpret_cast<__nv_bfloat16 *>(hi + off) = h;
    if (SPLIT) *reinterpret_cast<__nv_bfloat16 *>(lo + off) = l;
}

// ------------------------------------------------------------------------
// L_c = Gamma_K,c^T [V_c | 1]: M = components, contraction over the chunk's
// 128 tokens, with both operands MN-major in shared memory, so that no thread
// transposes anything:
//   A = Gamma_K^T: the chunk's Gamma_K planes as TMA lands them ([tokens][components]);
//   B = [V_hi | V_lo | 1] (split planes) or [V | 1]: token-major bf16 images that the
//       threads write from V, read from global memory one row per d_v / 4 lanes.
// One MMA chain per plane of A over the whole of B (N = value columns + 16), so with
// split planes D[:, c] + D[:, d_v + c] = (A_hi + A_lo)(V_hi + V_lo), and every column
// of the ones block holds Z_k = sum_j Gamma_K[j][k].  Rows past the sequence end
// land as zeros (3D maps; V rows are not read) and contribute nothing.
// Persistent: CTA b takes the chunks [b * per, (b + 1) * per) of the list (slice,
// chunk) in order.  Landing tiles, B images and accumulators are double-buffered:
// the MMA of chunk c runs while the threads write out chunk c - 1 and build the B
// image of chunk c + 1, whose Gamma_K planes are in flight.  The block is written
// transposed: d_v rows of K, then Z as row d_v.
constexpr int kStateThreads = 512;

template <bool SPLIT, int DV>
struct StateSmem {
    static constexpr int NP = SPLIT ? 2 : 1;               // planes of Gamma_K
    static constexpr int NBV = NP * DV / 64;               // 64-column value blocks of B
    static constexpr int N = NBV * 64 + 16;                // MMA N: the value columns, then 16 ones
    static constexpr uint32_t BLK = kC * 128;              // one 64-column block of 128 token rows
    static constexpr uint32_t G = kC * kRowB;              // one Gamma_K plane tile (two blocks)
    static constexpr uint32_t L = NP * G;                  // landing tiles of one chunk
    static constexpr uint32_t BI = (NBV + 1) * BLK;        // B image of one chunk (values, ones)
    static constexpr size_t bytes = 1024 + 2 * ((size_t)L + BI) + 64;
};

struct StateMaps {
    CUtensorMap gk[2];   // Gamma_K hi / lo planes as [slices][N][K], boxes of C rows x 64 components
};

template <bool SPLIT, int DV>
__global__ void __launch_bounds__(kStateThreads, 1)
    k_chunk_state_tc(const __grid_constant__ StateMaps maps, int N, int nblk, long long items, int K, int KH,
                     const void *__restrict__ v, bool v_bf16, float *__restrict__ partial, unsigned int *timeout)
{
    using Sm = StateSmem<SPLIT, DV>;
    constexpr int NP = Sm::NP, NBV = Sm::NBV;
    constexpr int F4 = DV / 4;                              // groups of four in a row of V
    constexpr int VPER = kC * F4 / kStateThreads;           // groups of V per thread
    static_assert(Sm::bytes <= 232448, "shared memory of one CTA");
    static_assert(Sm::N <= 256 && Sm::N % 16 == 0, "MMA N");
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *land = sm;                               // [2] Gamma_K landing tiles
    unsigned char *bimg = sm + 2 * Sm::L;                   // [2] B images
    uint64_t *bar = reinterpret_cast<uint64_t *>(bimg + 2 * Sm::BI);   // landing [2], MMA [2]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tg = warp >> 2;                   // column group of D
    const uint32_t lane0 = 32 * (warp & 3);
    const int k = lane0 + lane;                 // component (TMEM lane)
    const long long per = (items + gridDim.x - 1) / gridDim.x;
    const long long it0 = (long long)blockIdx.x * per;
    const long long it1 = it0 + per < items ? it0 + per : items;
    const long long SZ = (long long)K * DV + K;
    const float qnan = __int_as_float(0x7fc00000);
    // item it: component group it % KH of chunk it / KH (of the list (slice, chunk))

    // chunk and component group of item it (one group: no division)
    auto chunk_of = [&](long long it) { return KH == 1 ? it : it / KH; };
    auto group_of = [&](long long it) { return KH == 1 ? 0 : (int)(it % KH); };
    auto load = [&](long long it, int b) {   // one thread: the group's Gamma_K planes into landing buffer b
        const long long ch = chunk_of(it);
        const int sl = (int)(ch / nblk), c0 = (int)(ch % nblk) * kC, x0 = kK * group_of(it);
        const uint32_t bl = smem_addr(bar + b);
        mbar_expect_tx(bl, Sm::L);
        for (int pl = 0; pl < NP; ++pl)
            for (int a = 0; a < 2; ++a)
                tma_load_3d(smem_addr(land + b * Sm::L + pl * Sm::G + a * Sm::BLK), &maps.gk[pl], x0 + a * 64, c0, sl, bl);
    };
    // V of chunk it as raw words (fp32, or bf16 pairs in .x and .y); F4 consecutive threads read a row
    auto load_v = [&](long long it, uint4 (&r)[VPER]) {
        const long long ch = chunk_of(it);
        const int c0 = (int)(ch % nblk) * kC, nr = min(kC, N - c0);
        const long long rowbase = (ch / nblk) * N + c0;
#pragma unroll
        for (int u = 0; u < VPER; ++u) {
            const int f = tid + u * kStateThreads, j = f / F4, c4 = 4 * (f % F4);
            r[u] = make_uint4(0u, 0u, 0u, 0u);
            if (j < nr) {
                if (v_bf16) {
                    const uint2 w = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(v) + (rowbase + j) * DV + c4);
                    r[u].x = w.x;
                    r[u].y = w.y;
                } else {
                    r[u] = *reinterpret_cast<const uint4 *>(static_cast<const float *>(v) + (rowbase + j) * DV + c4);
                }
            }
        }
    };
    // the value columns of B image b: hi plane at column c, lo plane at column d_v + c
    auto put_b = [&](int b, const uint4 (&r)[VPER]) {
        unsigned char *bi = bimg + b * Sm::BI;
#pragma unroll
        for (int u = 0; u < VPER; ++u) {
            const int f = tid + u * kStateThreads, j = f / F4, c4 = 4 * (f % F4);
            const float x[4] = {v_bf16 ? __uint_as_float(r[u].x << 16) : __uint_as_float(r[u].x),
                                v_bf16 ? __uint_as_float(r[u].x & 0xffff0000u) : __uint_as_float(r[u].y),
                                v_bf16 ? __uint_as_float(r[u].y << 16) : __uint_as_float(r[u].z),
                                v_bf16 ? __uint_as_float(r[u].y & 0xffff0000u) : __uint_as_float(r[u].w)};
            uint32_t hw[2], lw[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                __nv_bfloat16 h0, l0, h1, l1;
                split_bf16(x[2 * e], h0, l0);
                split_bf16(x[2 * e + 1], h1, l1);
                hw[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                lw[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
            }
            *reinterpret_cast<uint2 *>(bi + sw128_offset(j, c4, kC, 2)) = make_uint2(hw[0], hw[1]);
            if (SPLIT) *reinterpret_cast<uint2 *>(bi + sw128_offset(j, DV + c4, kC, 2)) = make_uint2(lw[0], lw[1]);
        }
    };
    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 512);
        tmem_relinquish();
    }
    bool pend[2] = {false, false};   // landings in flight that the loop has not waited for (thread 0's record)
    uint32_t ph_l[2] = {0u, 0u};
    if (tid == 0) {
        for (int b = 0; b < 4; ++b) mbar_init(smem_addr(bar + b), 1);
        mbar_init_fence();
        for (int b = 0; b < 2; ++b)
            if (it0 + b < it1) {
                load(it0 + b, b);
                pend[b] = true;
            }
    }
    // the ones columns of both B images (they never change)
    for (int e = tid; e < 2 * kC * 2; e += kStateThreads) {
        const int b = e / (2 * kC), j = (e / 2) % kC, h = e % 2;
        *reinterpret_cast<uint4 *>(bimg + b * Sm::BI + sw128_offset(j, NBV * 64 + 8 * h, kC, 2)) =
            make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    }
    uint4 vr[VPER];
    if (it0 < it1) load_v(it0, vr);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *tslot;
    // L of chunk it from accumulator b (its MMA complete), into its block
    auto take = [&](long long it, int b, bool okv) {
        float *o = partial + chunk_of(it) * SZ;
        const int kg = kK * group_of(it) + k;    // this thread's component
        const bool kin = kg < K;                 // not a padding component
        const uint32_t d = 256u * b;
#pragma unroll
        for (int cb = 0; cb < DV / 4; cb += 16) {
            const int c = tg * (DV / 4) + cb;
            uint32_t r[16];
            tmem_ld16(tmem_at(tbase, lane0, d + c), r);
            float x[16];
            if constexpr (SPLIT) {
                uint32_t s[16];
                tmem_ld16(tmem_at(tbase, lane0, d + DV + c), s);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 16; ++q) x[q] = __uint_as_float(r[q]) + __uint_as_float(s[q]);
            } else {
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 16; ++q) x[q] = __uint_as_float(r[q]);
            }
            if (kin)
#pragma unroll
                for (int q = 0; q < 16; ++q) o[(long long)(c + q) * K + kg] = okv ? x[q] : qnan;
        }
        if (tg == 0) {   // Z: any column of the ones block
            uint32_t r[16];
            tmem_ld16(tmem_at(tbase, lane0, d + NBV * 64), r);
            tmem_wait_ld();
            if (kin) o[(long long)K * DV + kg] = okv ? __uint_as_float(r[0]) : qnan;
        }
    };

    const uint32_t id = idesc(128, Sm::N, kFmtBF16) | kAMajorMN | kBMajorMN;
    bool ok = true, okp = true;   // ok: agreed at the last barrier; okp: this thread's waits since
    int nm = 0;                   // MMA chains issued

    for (long long it = it0; it < it1 && ok; ++it) {
        const int j = (int)(it - it0), b = j & 1;
        bool okm = true;
        if (j > 0) {   // the previous chunk's MMA (issued a whole item ago): its landing buffer takes chunk j + 1
            okm = mbar_wait(smem_addr(bar + 2 + (b ^ 1)), (uint32_t)(((j - 1) >> 1) & 1));
            okp = okp && okm;
            fence_after_sync();
            if (tid == 0 && okm && it + 1 < it1) {
                load(it + 1, b ^ 1);
                pend[b ^ 1] = true;
                ph_l[b ^ 1] = (uint32_t)(((j + 1) >> 1) & 1);
            }
        }
        put_b(b, vr);   // its buffer was last read by the MMA of chunk j - 2, complete
        if (it + 1 < it1) load_v(it + 1, vr);   // in flight while this chunk's MMA runs
        const bool ok_l = mbar_wait(smem_addr(bar + b), (uint32_t)((j >> 1) & 1));
        if (tid == 0 && ok_l) pend[b] = false;
        okp = okp && ok_l;
        fence_proxy_async();   // the B image, written by threads, is read by the tensor core
        fence_before_sync();
        ok = __syncthreads_and(okp) != 0;
        fence_after_sync();
        if (!ok) break;
        if (tid == 0) {
            const uint32_t d = tbase + 256u * b;
            const unsigned char *a0 = land + b * Sm::L, *b0 = bimg + b * Sm::BI;
#pragma unroll 1
            for (int pl = 0; pl < NP; ++pl)
#pragma unroll 1
                for (int s = 0; s < kKSteps; ++s)
                    mma_ss(0u, d, sdesc_mn_sw128(smem_addr(a0 + pl * Sm::G + 2048 * s), Sm::BLK),
                           sdesc_mn_sw128(smem_addr(b0 + 2048 * s), Sm::BLK), id, (pl > 0 || s > 0) ? 1u : 0u);
            mma_commit(smem_addr(bar + 2 + b));
        }
        __syncwarp();
        ++nm;
        if (j > 0) take(it - 1, b ^ 1, okm);   // the previous chunk's accumulator goes out meanwhile
    }
    // the last chunk issued, once its MMA is done (chains complete in order, so this also
    // covers every earlier one after a failure)
    bool ok_end = ok;
    if (nm > 0) {
        const int jl = nm - 1, bl = jl & 1;
        const bool okm = mbar_wait(smem_addr(bar + 2 + bl), (uint32_t)((jl >> 1) & 1));
        fence_after_sync();
        take(it0 + jl, bl, ok && okm);
        ok_end = ok_end && okm;
    }
    // after a failed wait: let the landings in flight arrive before the shared memory is released
    if (tid == 0)
        for (int b = 0; b < 2; ++b)
            if (pend[b]) ok_end = mbar_wait(smem_addr(bar + b), ph_l[b]) && ok_end;
    fence_before_sync();
    if (__syncthreads_and(ok_end) == 0 && tid == 0) report_timeout(timeout);
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------------------
// Carried memory in operand form.  One thread per element of the operand-form
// block (d_v rows of KT components, then Z; KT = K padded to whole groups of 128,
// padding components written as zeros), serial over the chunks of its slice
// (fixed order, deterministic):
//   memory block c (exclusive prefix)  <- state_in + sum_{c' < c} L_c'
//   total (inclusive, bidirectional)   <- the sum over all chunks
//   state_out (caller layout)          <- state_in + the sum over all chunks
// The chunk contributions L are fp32 blocks of K d_v + K words (Vt^T as d_v rows of
// K, then Z).  A memory block in operand form holds the hi plane [d_v][KT] (bf16),
// the lo plane (split form only), then Z as a hi row and a lo row [KT] (bf16),
// within (d_v + 1) KT fp32 words.  state_in / state_out keep the caller layout (Vt
// as K rows of d_v, then Z).
__global__ void __launch_bounds__(256) k_scan_split(int DV, int K, int KT, int nblk, const float *__restrict__ partial,
                                                    const float *__restrict__ state_in, unsigned char *__restrict__ mem,
                                                    unsigned char *__restrict__ total, float *__restrict__ state_out,
                                                    bool lo_plane)
{
    const int MW = (DV + 1) * KT;                        // operand-form block (fp32 words)
    const int e = blockIdx.x * 256 + threadIdx.x;
    if (e >= MW) return;
    const long long bh = blockIdx.y;
    const long long SZ = (long long)K * DV + K;
    const int VT = KT * DV;
    const bool zrow = e >= VT;
    const int c = zrow ? DV : e / KT, k = zrow ? e - VT : e - c * KT;
    const bool pad = k >= K;
    const long long ep = zrow ? (long long)K * DV + k : (long long)c * K + k;   // element in the L blocks
    const long long eu = zrow ? ep : (long long)k * DV + c;                     // element in the caller layout
    auto put = [&](unsigned char *blk, float x) {
        __nv_bfloat16 hi, lo;
        split_bf16(x, hi, lo);
        __nv_bfloat16 *b16 = reinterpret_cast<__nv_bfloat16 *>(blk);
        if (!zrow) {
            b16[e] = hi;
            if (lo_plane) b16[VT + e] = lo;
        } else {   // Z: a hi row and a lo row after both planes
            b16[2 * VT + k] = hi;
            b16[2 * VT + KT + k] = lo;
        }
    };
    if (pad) {   // padding components: zeros in every block
        for (int b = 0; b < nblk; ++b)
            if (mem) put(mem + (bh * nblk + b) * MW * 4LL, 0.f);
        if (total) put(total + bh * MW * 4LL, 0.f);
        return;
    }
    float run = state_in ? state_in[bh * SZ + eu] : 0.f;
    const float *__restrict__ p = partial + bh * nblk * SZ + ep;
    constexpr int U = 32;   // loads in flight per thread
    int b = 0;
    for (; b + U <= nblk; b += U) {
        float t[U];
#pragma unroll
        for (int u = 0; u < U; ++u) t[u] = p[(long long)(b + u) * SZ];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (mem) put(mem + (bh * nblk + b + u) * MW * 4LL, run);
            run += t[u];
        }
    }
    for (; b < nblk; ++b) {
        const float t = p[(long long)b * SZ];
        if (mem) put(mem + (bh * nblk + b) * MW * 4LL, run);
        run += t;
    }
    if (total) put(total + bh * MW * 4LL, run);
    if (state_out) state_out[bh * SZ + eu] = run;
}

// ------------------------------------------------------------------------
// Chunk output, persistent: CTA b takes the items [b * per, (b + 1) * per) of
// the list (slice, chunk) in order.  16 warps: warp w owns TMEM lanes (rows)
// 32 (w % 4) + lane and column quarter w / 4 of every row-wise step.
//
// U = Gq Vt, P = Gq Gk^T and the denominator's Gq Z share the A operand Gq, so
// they are one MMA chain with N = C + d_v + 16 over the B tile [Gk ; Vt^T ; Z]
// (K-major, 128-byte swizzle; each 128-byte atom column holds the C rows of Gk,
// the d_v rows of Vt^T, then Z_hi, Z_lo and 14 zero rows, the lo image's Z rows
// all zero so that the three passes give (Gq_hi + Gq_lo)(Z_hi + Z_lo) in two
// columns); its accumulator is [P | U | Gq Z] in consecutive TMEM columns.  Gq
// is the A operand straight from shared memory.  Every operand plane arrives by
// TMA:
//   B images (hi, lo) <- Gk planes (rows 0 .. C-1), memory planes and Z rows
//   A images (hi, lo) <- Gq planes
// (with d_v = 128, N would pass 256: there the Z rows are a B operand of their
// own and one more chain of N = 16).
// Then P_m, split by threads, goes to TMEM as the A operand of P_m [V_hi | V_lo]:
// V, read with row-contiguous loads while the tensor core works, is split by
// threads into token-major bf16 images in the staging tile, the B operand
// (MN-major), and the two column halves of the product add up to
// (P_hi + P_lo)(V_hi + V_lo).  No thread reads the operand images, so the next
// item's Gamma tiles and memory are fetched as soon as the first chain has
// completed, while P_m and the V images are built.  The output tile is staged
// in shared memory and leaves by TMA stores.
constexpr int kOutThreads = 512;

template <bool SPLIT, int DV>
struct OutSmem {
    static constexpr int NP = SPLIT ? 2 : 1;                           // planes
    static constexpr uint32_t PART = kC * 128;                         // Gk rows of an atom column
    // the Z rows [Z_hi; Z_lo; 14 zero rows] join B when N stays within 256, else a B of their own
    static constexpr bool ZF = kC + DV + 16 <= 256;
    static constexpr uint32_t ATOM = (kC + DV + (ZF ? 16 : 0)) * 128;  // bytes of an atom column of B
    static constexpr uint32_t BIMG = 2 * ATOM;                         // one B image (two atom columns)
    static constexpr uint32_t AIMG = 2 * kAtom;                        // one A image
    static constexpr uint32_t OUT = kC * DV * 4;                       // output tile (fp32)
    static constexpr uint32_t ZATOM = 16 * 128;                        // atom column of the Z rows
    static constexpr uint32_t BZ = ZF ? 0 : 2 * ZATOM;                 // their own B operand
    static constexpr size_t bytes = 1024 + NP * ((size_t)BIMG + AIMG) + OUT + BZ + 4 * kK * 4 + 64;
};

struct OutMaps {
    CUtensorMap gq[2], gk[2];   // hi / lo planes of the responsibilities
    CUtensorMap s;              // memory blocks in operand form, as rows of 256 bytes
    CUtensorMap z;              // the same rows, boxes of the two Z rows
    CUtensorMap o;              // output [slices][N][d_v], boxes of 64 rows x 32 columns
};

// CAUSAL = false gives the bidirectional read: U = Gamma_Q [Vt | Z] with the
// total memory of the sequence (the same block for every chunk), no P.
template <bool SPLIT, int DV, bool CAUSAL>
__global__ void __launch_bounds__(kOutThreads, 1)
    k_chunk_out_tc(const __grid_constant__ OutMaps maps, int N, int nblk, long long items, int KH, float eps,
                   const void *__restrict__ v, bool v_bf16, float *__restrict__ out, unsigned int *timeout,
                   const unsigned int *__restrict__ zq)
{
    using Sm = OutSmem<SPLIT, DV>;
    constexpr int NP = Sm::NP;
    static_assert(OutSmem<SPLIT, DV>::bytes <= 232448, "shared memory of one CTA");
    constexpr int F4 = DV / 4;                              // groups of four in a row of V
    constexpr int VPER = kC * F4 / kOutThreads;             // groups of V per thread
    constexpr int NBV = NP * DV / 64;                       // 64-column blocks of the V images
    constexpr uint32_t AS = Sm::ATOM, PART = Sm::PART;
    constexpr int SROWS = 2 * DV + 2;                       // rows of a memory block (KH groups of 128)
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *const tb0 = sm, *const tb1 = sm + Sm::BIMG;                     // B images (hi, lo)
    unsigned char *const ta0 = sm + NP * Sm::BIMG, *const ta1 = ta0 + Sm::AIMG;    // A images (hi, lo)
    unsigned char *const os = sm + NP * (Sm::BIMG + Sm::AIMG);                     // output tile
    unsigned char *const bz = os + Sm::OUT;                                        // B operand of Gq Z (!ZF)
    float *part = reinterpret_cast<float *>(bz + Sm::BZ);           // [4][128]: row-sum quarters of P_m
    uint64_t *bar = reinterpret_cast<uint64_t *>(part + 4 * kK);    // [6]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 6);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = warp >> 2;                    // column quarter
    const uint32_t lane0 = 32 * (warp & 3);
    const int i = lane0 + lane;                 // row of the chunk owned in TMEM
    const long long per = (items + gridDim.x - 1) / gridDim.x;
    const long long it0 = (long long)blockIdx.x * per;
    const long long it1 = it0 + per < items ? it0 + per : items;
    // TMEM: P_m (hi, lo), then [P | U | Gq Z], P_m [V_hi | V_lo]; without ZF, Gq Z in the unused
    // lo half of P_m (bf16 operands only)
    constexpr bool ZF = Sm::ZF;
    constexpr uint32_t A_PM_HI = 0, A_PM_LO = 64, D_P = 128, D_U = D_P + kC, D_PV = D_U + DV + (ZF ? 64 : 0);
    constexpr uint32_t D_Z = ZF ? D_U + DV : A_PM_LO;
    static_assert(D_PV + NBV * 64 <= 512 && (ZF || !SPLIT), "TMEM columns");
    // G, S: loads of a group's tiles and memory; M: a chain that is not an item's last; L: an
    // item's last chain; V: P_m V; O: the output staging tile is free
    const uint32_t BAR_G = smem_addr(bar), BAR_S = smem_addr(bar + 1), BAR_M = smem_addr(bar + 2),
                   BAR_V = smem_addr(bar + 3), BAR_O = smem_addr(bar + 4), BAR_L = smem_addr(bar + 5);

    // block of the carried memory read by item it
    auto mem_block = [&](long long it) -> long long { return CAUSAL ? it : it / nblk; };
    // one thread: component group g (components 128 g .. + 127) of item it.  Returns whether the
    // lo plane of Gamma_Q is zero on this chunk (the routing of Q recorded it and did not write
    // it): then it is not loaded, and the product it takes is not issued (it would add zeros)
    auto load_gamma = [&](long long it, int g) {
        const int row0 = (int)((it / nblk) * N + (it % nblk) * kC), x0 = kK * g;
        const bool zl = SPLIT && zq != nullptr && zq[it] != 0u;   // (items are (slice, chunk), chunk = tile)
        mbar_expect_tx(BAR_G, (uint32_t)(((CAUSAL ? 2 : 1) * NP - (zl ? 1 : 0)) * kC * kRowB));
        for (int pl = 0; pl < NP; ++pl)
            for (int a = 0; a < 2; ++a) {
                if (CAUSAL) tma_load_2d(smem_addr((pl ? tb1 : tb0) + a * AS), &maps.gk[pl], x0 + a * 64, row0, BAR_G);
                if (!(pl && zl)) tma_load_2d(smem_addr((pl ? ta1 : ta0) + a * kAtom), &maps.gq[pl], x0 + a * 64, row0, BAR_G);
            }
        return zl;
    };
    auto load_memory = [&](long long it, int g) {
        const int srow = (int)(mem_block(it) * SROWS), x0 = kK * g;
        mbar_expect_tx(BAR_S, (uint32_t)((NP * DV + 2) * kRowB));
        for (int a = 0; a < 2; ++a) {
            for (int pl = 0; pl < NP; ++pl)
                tma_load_2d(smem_addr((pl ? tb1 : tb0) + a * AS + PART), &maps.s, x0 + a * 64, srow + pl * DV, BAR_S);
            tma_load_2d(smem_addr(ZF ? tb0 + a * AS + PART + DV * 128 : bz + a * Sm::ZATOM), &maps.z, x0 + a * 64,
                        srow + 2 * DV, BAR_S);   // Z_hi, Z_lo
        }
    };

    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 512);
        tmem_relinquish();
    }
    // loads in flight that the loop has not waited for (thread 0's record)
    bool pend_g = false, pend_s = false;
    uint32_t ph_g = 0, ph_s = 0;
    bool zq_l = false;   // (thread 0) the last loaded group's Gamma_Q lo plane is zero
    if (tid == 0) {
        for (int b = 0; b < 6; ++b) mbar_init(smem_addr(bar + b), 1);
        mbar_init_fence();
        if (it0 < it1) {
            zq_l = load_gamma(it0, 0);
            load_memory(it0, 0);
            pend_g = pend_s = true;
        }
    }
    // the Z rows that TMA never writes stay zero: rows 2 .. 15 of the hi image's (TMA writes
    // Z_hi, Z_lo), all 16 of the lo image's
    for (int e = tid; e < NP * 2 * 16 * 8; e += kOutThreads) {
        const int pl = e / (2 * 16 * 8), a = (e / (16 * 8)) % 2, r = (e / 8) % 16, c = e % 8;
        if (pl == 0 && r < 2) continue;
        unsigned char *zb = ZF ? (pl ? tb1 : tb0) + a * AS + PART + DV * 128 : bz + a * Sm::ZATOM;
        *reinterpret_cast<uint4 *>(zb + (r >> 3) * 1024 + (r & 7) * 128 + 16 * c) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async();   // read by the tensor core
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *tslot;
    bool ok = true;
    const float qnan = __int_as_float(0x7fc00000);
    uint32_t un = 0;   // component groups consumed (phases of the load barriers G, S)
    uint32_t um = 0;   // chains completed on M (thread 0)

    for (long long it = it0; it < it1 && ok; ++it) {
        const uint32_t ph = (uint32_t)((it - it0) & 1);   // phase of the item barriers L, V, O
        const long long bh = it / nblk;
        const int c0 = (int)(it % nblk) * kC;
        const int nr = min(kC, N - c0);
        const bool more = it + 1 < it1;
        // V of this chunk as raw words (fp32, or bf16 pairs in .x and .y), F4 consecutive threads
        // to a row, in flight while the tensor core works
        uint4 vr[CAUSAL ? VPER : 1];
        if constexpr (CAUSAL) {
            const long long rowbase = bh * N + c0;
#pragma unroll
            for (int u = 0; u < VPER; ++u) {
                const int f = tid + u * kOutThreads, j = f / F4, c4 = 4 * (f % F4);
                vr[u] = make_uint4(0u, 0u, 0u, 0u);
                if (j < nr) {
                    if (v_bf16) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(v) + (rowbase + j) * DV + c4);
                        vr[u].x = w.x;
                        vr[u].y = w.y;
                    } else {
                        vr[u] = *reinterpret_cast<const uint4 *>(static_cast<const float *>(v) + (rowbase + j) * DV + c4);
                    }
                }
            }
        }
        // [P | U | Gq Z] = Gq [Gk ; Vt^T ; Z]^T (bidirectional read: [U | Gq Z]), the contraction
        // over the components taken one group of 128 at a time into the same accumulator
        // Thread 0 alone waits for the loads (G, S) and for the chains before an item's last (M):
        // it re-arms those barriers for the next group or item as soon as a chain is done, with
        // no CTA barrier in between, so another thread waiting on them could find a barrier two
        // phases on (and wait for a phase that has passed) or start a phase early (and take the
        // phase before for it).  An item's last chain completes on L, one phase per item, waited
        // by every thread and committed again only after the item's closing barrier.
        for (int gr = 0; gr < KH; ++gr, ++un) {
            const uint32_t pu = un & 1u;   // phase of the per-group load barriers
            const bool last = gr + 1 == KH;
            if (tid == 0) {
                const bool ok_g = mbar_wait(BAR_G, pu), ok_s = mbar_wait(BAR_S, pu);
                ok = ok && ok_g && ok_s;
                // a load whose wait gave up is still in flight
                pend_g = pend_g && !ok_g;
                pend_s = pend_s && !ok_s;
                const uint32_t b0 = CAUSAL ? 0u : PART;
                const uint32_t d0 = CAUSAL ? D_P : D_U, nb = (CAUSAL ? kC + DV : DV) + (ZF ? 16 : 0);
                mma_pass_ss(tbase + d0, ta0, kAtom, tb0 + b0, nb, AS, gr > 0);
                if constexpr (SPLIT) {
                    mma_pass_ss(tbase + d0, ta0, kAtom, tb1 + b0, nb, AS, true);
                    if (!zq_l) mma_pass_ss(tbase + d0, ta1, kAtom, tb0 + b0, nb, AS, true);
                }
                if constexpr (!ZF)   // Gq [Z_hi | Z_lo] on its own
                    mma_pass_ss(tbase + D_Z, ta0, kAtom, bz, 16, Sm::ZATOM, gr > 0);
                mma_commit(last ? BAR_L : BAR_M);
                if (CAUSAL && gr == 0) {   // the previous output tile has left the staging tile, which takes V next
                    bulk_wait_read();
                    mbar_arrive(BAR_O);
                }
            }
            __syncwarp();
            if (last) {
                ok = mbar_wait(BAR_L, ph) && ok;
                fence_after_sync();
            } else if (tid == 0) {
                ok = mbar_wait(BAR_M, um & 1u) && ok;
                ++um;
                fence_after_sync();
            }
            if (tid == 0 && ok && (gr + 1 < KH || more)) {
                // the MMA has read B, the A images and the Z rows (no thread reads them): the next
                // group's (or the next item's first group's) tiles and memory may land in them
                const long long in = gr + 1 < KH ? it : it + 1;
                const int gn = gr + 1 < KH ? gr + 1 : 0;
                zq_l = load_gamma(in, gn);
                load_memory(in, gn);
                pend_g = pend_s = true;
                ph_g = ph_s = pu ^ 1u;
            }
        }
        if constexpr (CAUSAL) {
            // V into token-major images in the staging tile, the B operand (MN-major) of
            // U += P_m V: hi plane in columns [0, d_v), lo plane in [d_v, 2 d_v), once the
            // previous output tile has left it
            ok = mbar_wait(BAR_O, ph) && ok;
#pragma unroll
            for (int u = 0; u < VPER; ++u) {
                const int f = tid + u * kOutThreads, j = f / F4, c4 = 4 * (f % F4);
                const float x[4] = {v_bf16 ? __uint_as_float(vr[u].x << 16) : __uint_as_float(vr[u].x),
                                    v_bf16 ? __uint_as_float(vr[u].x & 0xffff0000u) : __uint_as_float(vr[u].y),
                                    v_bf16 ? __uint_as_float(vr[u].y << 16) : __uint_as_float(vr[u].z),
                                    v_bf16 ? __uint_as_float(vr[u].y & 0xffff0000u) : __uint_as_float(vr[u].w)};
                uint32_t hw[2], lw[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    __nv_bfloat16 h0, l0, h1, l1;
                    split_bf16(x[2 * e], h0, l0);
                    split_bf16(x[2 * e + 1], h1, l1);
                    hw[e] = (uint32_t)__bfloat16_as_ushort(h0) | ((uint32_t)__bfloat16_as_ushort(h1) << 16);
                    lw[e] = (uint32_t)__bfloat16_as_ushort(l0) | ((uint32_t)__bfloat16_as_ushort(l1) << 16);
                }
                *reinterpret_cast<uint2 *>(os + sw128_offset(j, c4, kC, 2)) = make_uint2(hw[0], hw[1]);
                if (SPLIT) *reinterpret_cast<uint2 *>(os + sw128_offset(j, DV + c4, kC, 2)) = make_uint2(lw[0], lw[1]);
            }
            // P_m = P with j > i zeroed, split, is the A operand of U += P_m V; the row sums
            // of the split values on CUDA cores
            {
                float x[32];
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    uint32_t r[16];
                    tmem_ld16(tmem_at(tbase, lane0, D_P + 32 * g + 16 * b), r);
                    tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int jj = 32 * g + 16 * b + j;
                        x[16 * b + j] = jj <= i ? __uint_as_float(r[j]) : 0.f;
                    }
                }
                part[g * kK + i] = put_a32<SPLIT>(tbase, lane0, A_PM_HI, A_PM_LO, 32 * g, x);
            }
            tmem_wait_st();
            fence_proxy_async();
            fence_before_sync();
            __syncthreads();   // the V images and P_m are in place
            fence_after_sync();
            if (tid == 0) {
                // U' = P_m [V_hi | V_lo] from both planes of P_m: (P_hi + P_lo)(V_hi + V_lo) in two halves
                const uint32_t idv = idesc(128, NBV * 64, kFmtBF16) | kBMajorMN;
#pragma unroll 1
                for (int pl = 0; pl < NP; ++pl)
#pragma unroll 1
                    for (int s = 0; s < kKSteps; ++s)
                        mma_ts(0u, tbase + D_PV, tbase + (pl ? A_PM_LO : A_PM_HI) + 8 * s,
                               sdesc_mn_sw128(smem_addr(os + 2048 * s), kC * 128), idv, (pl > 0 || s > 0) ? 1u : 0u);
                mma_commit(BAR_V);
            }
            __syncwarp();
            ok = mbar_wait(BAR_V, ph) && ok;
            fence_after_sync();
        } else {
            fence_before_sync();
            if (tid == 0) bulk_wait_read();   // the previous output tile has left shared memory
            __syncthreads();
            fence_after_sync();
        }

        // den = Gq . Z (two halves) + the row sum of P_m + eps
        float den;
        {
            uint32_t r[16];
            tmem_ld16(tmem_at(tbase, lane0, D_Z), r);
            tmem_wait_ld();
            den = eps + (__uint_as_float(r[0]) + __uint_as_float(r[1]));
        }
        if constexpr (CAUSAL) {
#pragma unroll
            for (int q = 0; q < 4; ++q) den += part[q * kK + i];
        }
        const float inv = 1.0f / den;
        // the output tile, in boxes of 64 rows x 32 columns (box (i / 64) (d_v / 32) + c / 32)
#pragma unroll
        for (int cb = 0; cb < DV / 64; ++cb) {
            const int c = g * (DV / 4) + 16 * cb;
            // U = Gamma_Q Vt_prev (+ the halves of P_m [V_hi | V_lo])
            uint32_t r[16];
            float y[16];
            tmem_ld16(tmem_at(tbase, lane0, D_U + c), r);
            if constexpr (CAUSAL) {
                uint32_t a[16], b2[16];
                tmem_ld16(tmem_at(tbase, lane0, D_PV + c), a);
                if constexpr (SPLIT) tmem_ld16(tmem_at(tbase, lane0, D_PV + DV + c), b2);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    y[q] = __uint_as_float(r[q]) +
                           (SPLIT ? __uint_as_float(a[q]) + __uint_as_float(b2[q]) : __uint_as_float(a[q]));
            } else {
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 16; ++q) y[q] = __uint_as_float(r[q]);
            }
            unsigned char *ob = os + ((i >> 6) * (DV / 32) + (c >> 5)) * 8192 + (i & 63) * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float4 o4 = ok ? make_float4(y[4 * q] * inv, y[4 * q + 1] * inv, y[4 * q + 2] * inv,
                                                   y[4 * q + 3] * inv)
                                     : make_float4(qnan, qnan, qnan, qnan);
                *reinterpret_cast<float4 *>(ob + ((((c & 31) >> 2) + q) ^ (i & 7)) * 16) = o4;
            }
        }
        fence_proxy_async();   // the staged tile is read by the TMA store
        fence_before_sync();
        ok = __syncthreads_and(ok) != 0;   // every thread leaves the loop together
        fence_after_sync();
        if (tid == 0) {
            for (int b = 0; b < 2 * (DV / 32); ++b)
                tma_store_3d(&maps.o, (b % (DV / 32)) * 32, c0 + (b / (DV / 32)) * 64, (int)bh,
                             smem_addr(os + b * 8192));
            bulk_commit();
        }
    }
    // after a failed wait: let the copies still in flight land before the shared memory is released
    bool ok_end = ok;
    if (tid == 0) {
        if (pend_g) ok_end = mbar_wait(BAR_G, ph_g) && ok_end;
        if (pend_s) ok_end = mbar_wait(BAR_S, ph_s) && ok_end;
        bulk_wait_all();
    }
    fence_before_sync();
    if (__syncthreads_and(ok_end) == 0 && tid == 0) report_timeout(timeout);
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------------------
// A kernel whose only work is one bounded wait that expires: it waits for the
// first phase of an mbarrier that nothing arrives on (no copy and no MMA is
// ever issued against it), gives up after `limit` SM cycles and records the
// timeout exactly as the kernels above do.  Nothing asynchronous is in flight
// when it returns.
__global__ void __launch_bounds__(32, 1) k_expire_wait(long long limit, unsigned int *timeout)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        mbar_init_fence();
    }
    __syncthreads();
    const bool ok = mbar_wait(smem_addr(&bar), 0u, limit);
    if (__syncthreads_and(ok) == 0 && threadIdx.x == 0) report_timeout(timeout);
}

} // namespace

cudaError_t launch_expire_wait(long long limit_cycles, cudaStream_t st)
{
    unsigned int *flag = timeout_flag_dev();
    if (!flag) return cudaErrorMemoryAllocation;
    k_expire_wait<<<1, 32, 0, st>>>(limit_cycles, flag);
    return cudaGetLastError();
}

bool tc_path_eligible(int K, int DV, bool g_bf16)
{
    return (K <= kK || (K % kK == 0 && K <= 4 * kK)) && (DV == 64 || (DV == 128 && g_bf16));
}

bool tc_path_applies(const Dims &dm) { return dm.C == kC && tc_path_eligible(dm.K, dm.DV, dm.g_bf16); }

template <bool SPLIT, int DV>
cudaError_t state_tc(const Dims &dm, const void *gk, const void *v, float *partial, cudaStream_t st)
{
    constexpr size_t smem = StateSmem<SPLIT, DV>::bytes;
    static std::atomic<unsigned long long> smem_set{0};
    const cudaError_t attr = allow_smem(k_chunk_state_tc<SPLIT, DV>, smem, smem_set);
    if (attr != cudaSuccess) return attr;
    StateMaps maps;
    const unsigned long long rows = (unsigned long long)dm.BH() * dm.N;
    const uint16_t *k16 = static_cast<const uint16_t *>(gk);
    const int KT = tc_kpad(dm.K), KH = KT / kK;   // component groups of 128
    for (int pl = 0; pl < (SPLIT ? 2 : 1); ++pl)
        if (!make_tma_3d(&maps.gk[pl], k16 + pl * (long long)rows * KT, true, KT, dm.N, dm.BH(), kC))
            return cudaErrorInvalidValue;
    if (!SPLIT) maps.gk[1] = maps.gk[0];
    const long long items = dm.BH() * (long long)dm.nblk() * KH;   // (chunk, component group)
    const int grid = (int)(items < sm_count() ? items : sm_count());
    unsigned int *flag = timeout_flag_dev();
    if (!flag) return cudaErrorMemoryAllocation;
    k_chunk_state_tc<SPLIT, DV><<<grid, kStateThreads, smem, st>>>(maps, dm.N, dm.nblk(), items, dm.K, KH, v,
                                                                   dm.v_bf16, partial, flag);
    return cudaGetLastError();
}

template <bool SPLIT, int DV, bool CAUSAL>
cudaError_t out_tc(const Dims &dm, const void *gq, const void *gk, const void *v, const unsigned char *mem,
                   float *out, cudaStream_t st, const unsigned int *zq)
{
    constexpr size_t smem = OutSmem<SPLIT, DV>::bytes;
    static std::atomic<unsigned long long> smem_set{0};
    const cudaError_t attr = allow_smem(k_chunk_out_tc<SPLIT, DV, CAUSAL>, smem, smem_set);
    if (attr != cudaSuccess) return attr;
    OutMaps maps;
    const unsigned long long rows = (unsigned long long)dm.BH() * dm.N;
    const int KT = tc_kpad(dm.K), KH = KT / kK;   // component groups of 128
    const long long plane = (long long)rows * KT;
    const unsigned long long blocks = (unsigned long long)dm.BH() * (CAUSAL ? dm.nblk() : 1);
    const uint16_t *q16 = static_cast<const uint16_t *>(gq), *k16 = static_cast<const uint16_t *>(gk);
    bool ok = true;
    for (int pl = 0; pl < (SPLIT ? 2 : 1); ++pl)
        ok = ok && make_tma_2d(&maps.gq[pl], q16 + pl * plane, true, rows, KT, kC) &&
             make_tma_2d(&maps.gk[pl], k16 + pl * plane, true, rows, KT, kC);
    if (!SPLIT) {
        maps.gq[1] = maps.gq[0];
        maps.gk[1] = maps.gk[0];
    }
    // memory blocks in operand form: rows of KT bf16 (hi plane, lo plane, Z), d_v rows per box
    ok = ok && make_tma_2d(&maps.s, mem, true, blocks * (2 * DV + 2), KT, DV) &&
         make_tma_2d(&maps.z, mem, true, blocks * (2 * DV + 2), KT, 2) &&
         make_tma_3d(&maps.o, out, false, DV, dm.N, dm.BH(), 64);
    if (!ok) return cudaErrorInvalidValue;
    const long long items = dm.BH() * (long long)dm.nblk();
    const int grid = (int)(items < sm_count() ? items : sm_count());
    unsigned int *flag = timeout_flag_dev();
    if (!flag) return cudaErrorMemoryAllocation;
    k_chunk_out_tc<SPLIT, DV, CAUSAL><<<grid, kOutThreads, smem, st>>>(
        maps, dm.N, dm.nblk(), items, KH, dm.eps, v, dm.v_bf16, out, flag, KH == 1 ? zq : nullptr);
    return cudaGetLastError();
}

cudaError_t launch_chunk_state_tc(const Dims &dm, const void *gk, const void *v, float *partial, cudaStream_t st)
{
    if (dm.g_bf16) {
        if (dm.DV == 64) return state_tc<false, 64>(dm, gk, v, partial, st);
        if (dm.DV == 128) return state_tc<false, 128>(dm, gk, v, partial, st);
    } else if (dm.DV == 64) {
        return state_tc<true, 64>(dm, gk, v, partial, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_scan_split(const Dims &dm, const float *partial, const float *state_in, unsigned char *mem,
                              unsigned char *total, float *state_out, cudaStream_t st)
{
    const long long MW = tc_mem_words(dm);
    dim3 grid((unsigned)((MW + 255) / 256), (unsigned)dm.BH());
    k_scan_split<<<grid, 256, 0, st>>>(dm.DV, dm.K, tc_kpad(dm.K), dm.nblk(), partial, state_in, mem, total,
                                       state_out, !dm.g_bf16);
    return cudaGetLastError();
}

cudaError_t launch_chunk_out_tc(const Dims &dm, bool causal, const void *gq, const void *gk, const void *v,
                                const unsigned char *mem, float *out, cudaStream_t st, const unsigned int *zq)
{
    if (dm.g_bf16) {
        if (dm.DV == 64)
            return causal ? out_tc<false, 64, true>(dm, gq, gk, v, mem, out, st, zq)
                          : out_tc<false, 64, false>(dm, gq, gk, v, mem, out, st, zq);
        if (dm.DV == 128)
            return causal ? out_tc<false, 128, true>(dm, gq, gk, v, mem, out, st, zq)
                          : out_tc<false, 128, false>(dm, gq, gk, v, mem, out, st, zq);
    } else if (dm.DV == 64) {
        return causal ? out_tc<true, 64, true>(dm, gq, gk, v, mem, out, st, zq)
                      : out_tc<true, 64, false>(dm, gq, gk, v, mem, out, st, zq);
    }
    return cudaErrorInvalidValue;
}

} // namespace gma
