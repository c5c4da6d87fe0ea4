// Tensor-core (tcgen05 / TMEM) path of the causal form for K = 128.
//
// The causal variant of the GMA explainer ("변형 및 학습": prefix sums so that
// O_i depends on j <= i only) is evaluated in the chunkwise-parallel form of
// the linear-attention page ("선형 어텐션 원리 정리", "쉽게 이해하기"): chunks of
// C = 128 tokens, dense products inside a chunk, and a carried memory
// [Vt | Z] between chunks.  Two kernels, one CTA (8 warps) per chunk:
//
//   k_chunk_state_tc : L_c = Gamma_K,c^T [V_c | 1]            (chunk contribution)
//   (k_scan, generic) : S_{c-1} = state_in + sum_{c' < c} L_c'   (carried memory)
//   k_chunk_out_tc   : [P | U] = Gamma_Q,c [Gamma_K,c^T | Vt_{c-1}]
//                      P_m = P with j > i zeroed;   U += P_m V_c
//                      O_i = U_i / (sum_j P_m[i][j] + Gamma_Q,i . Z_{c-1} + eps)
//
// Every contraction is one tcgen05.mma sequence with M = 128 and the fp32
// accumulator in TMEM.  The A operand (Gamma rows, or P_m) is written to TMEM by
// the warps that own the rows (two warps per 32-lane quarter, each taking half
// of the columns); B operands sit in shared memory in the K-major
// 128-byte-swizzled layout, staged with coalesced 16-byte loads that are all
// issued before the first store.  GEMM operand precision:
//   BF16 = false: each fp32 operand is split into a tf32 "hi" part and an
//                 exact remainder "lo"; a*b ~ hi*hi + hi*lo + lo*hi (three MMA
//                 passes, relative error ~1e-6), the fp32-operand path;
//   BF16 = true : operands rounded to bf16, one pass, fp32 accumulation.
// The normaliser Z and the row sums of P_m are accumulated on CUDA cores.
#include "gma_internal.cuh"
#include "gma_tc.cuh"

#include <cuda.h>
#include <type_traits>

namespace gma {
namespace {

using namespace tc;

constexpr int kC = 128;       // chunk rows (= MMA M)
constexpr int kK = 128;       // components handled by this path
constexpr int kTCThreads = 256;   // 8 warps: two per TMEM lane quarter

template <bool BF16>
struct Elem {
    static constexpr int E = BF16 ? 2 : 4;                 // bytes per operand element
    static constexpr int PASSES = BF16 ? 1 : 3;
    static constexpr uint32_t FMT = BF16 ? kFmtBF16 : kFmtTF32;
    static constexpr int COLS_PER_KSTEP = 8;               // TMEM columns per 32-byte K step
};

// Stores element (r, k) of a K-major SW128 tile (hi image, and lo image for fp32).
template <bool BF16>
__device__ __forceinline__ void put(unsigned char *hi, unsigned char *lo, uint32_t off, float x)
{
    if constexpr (BF16) {
        *reinterpret_cast<__nv_bfloat16 *>(hi + off) = __float2bfloat16_rn(x);
    } else {
        const float h = tf32_hi(x);
        *reinterpret_cast<float *>(hi + off) = h;
        *reinterpret_cast<float *>(lo + off) = x - h;
    }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}
__device__ __forceinline__ float bf16r(float a) { return __bfloat162float(__float2bfloat16_rn(a)); }

// Bytes of a K-major tile of `rows` x 128 elements.
template <bool BF16>
constexpr uint32_t tile_bytes(uint32_t rows) { return rows * kK * Elem<BF16>::E; }

// One MMA pass D (+)= A * B^T over the 128-deep contraction: A in TMEM
// (columns from a_col), B a K-major SW128 tile of `nrows` rows.
template <bool BF16>
__device__ __forceinline__ void mma_pass(uint32_t d_tmem, uint32_t a_col, const unsigned char *b, uint32_t nrows,
                                         bool accumulate)
{
    using El = Elem<BF16>;
    const uint32_t id = idesc(128, nrows, El::FMT);
    constexpr int ksteps = kK * El::E / 32;
#pragma unroll 1
    for (int kk = 0; kk < ksteps; ++kk) {
        const uint32_t kb = kk * 32;
        const uint32_t boff = (kb >> 7) * (nrows * 128) + (kb & 127);
        mma_ts(!BF16, d_tmem, a_col + kk * El::COLS_PER_KSTEP, sdesc_sw128(smem_addr(b + boff)), id,
               (accumulate || kk > 0) ? 1u : 0u);
    }
}

// All passes of D (+)= A * B^T: fp32 operands as hi*hi + hi*lo + lo*hi.
template <bool BF16>
__device__ __forceinline__ void mma_all(uint32_t d_tmem, uint32_t a_hi, uint32_t a_lo, const unsigned char *b_hi,
                                        const unsigned char *b_lo, uint32_t nrows, bool accumulate)
{
    mma_pass<BF16>(d_tmem, a_hi, b_hi, nrows, accumulate);
    if constexpr (!BF16) {
        mma_pass<BF16>(d_tmem, a_hi, b_lo, nrows, true);
        mma_pass<BF16>(d_tmem, a_lo, b_hi, nrows, true);
    }
}

// Writes 64 consecutive A-operand values of this thread's TMEM lane, starting
// at operand column j0 (a multiple of 64): fp32 -> tf32 part at a_hi and the
// exact remainder at a_lo (part = 0: parts only, 1: remainders only, 2: both);
// bf16 -> packed pairs at a_hi.
template <bool BF16>
__device__ __forceinline__ void put_a64(uint32_t tbase, uint32_t lane0, uint32_t a_hi, uint32_t a_lo, int j0,
                                        const float (&x)[64], int part = 2)
{
    if constexpr (BF16) {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            uint32_t p[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) p[j] = pack_bf16(x[32 * b + 2 * j], x[32 * b + 2 * j + 1]);
            tmem_st16(tmem_at(tbase, lane0, a_hi + j0 / 2 + 16 * b), p);
        }
    } else {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float v = x[16 * b + j];
                const float hv = tf32_hi(v);
                hi[j] = __float_as_uint(hv);
                lo[j] = __float_as_uint(v - hv);
            }
            if (part != 1) tmem_st16(tmem_at(tbase, lane0, a_hi + j0 + 16 * b), hi);
            if (part != 0) tmem_st16(tmem_at(tbase, lane0, a_lo + j0 + 16 * b), lo);
        }
    }
}

// B = V^T of the chunk: element (c, j) of a DV x 128 K-major tile, from
// V [tokens][DV].  Lanes run over tokens, so the transposed stores of a warp
// fall in one swizzled row (no bank conflicts).
template <bool BF16, int DV>
__device__ __forceinline__ void stage_vt(const void *v, bool v_bf16, long long row0, int nr, unsigned char *hi,
                                         unsigned char *lo, int tid)
{
    using El = Elem<BF16>;
    constexpr int PER = (kC * DV / 4) / kTCThreads;
    float4 t[PER];
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int f = tid + u * kTCThreads, j = f % kC, c4 = f / kC;
        t[u] = j < nr ? load4(v, (row0 + j) * DV + 4 * c4, v_bf16) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < PER; ++u) {
        const int f = tid + u * kTCThreads, j = f % kC, c4 = f / kC;
        put<BF16>(hi, lo, sw128_offset(4 * c4 + 0, j, DV, El::E), t[u].x);
        put<BF16>(hi, lo, sw128_offset(4 * c4 + 1, j, DV, El::E), t[u].y);
        put<BF16>(hi, lo, sw128_offset(4 * c4 + 2, j, DV, El::E), t[u].z);
        put<BF16>(hi, lo, sw128_offset(4 * c4 + 3, j, DV, El::E), t[u].w);
    }
}

// 64 consecutive Gamma values of one row (fp32 or bf16 storage) -> x[64].
template <bool BF16>
__device__ __forceinline__ void load_g64(const void *g, long long off, bool valid, float (&x)[64])
{
    if constexpr (BF16) {
        const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(g) + off);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint4 t = valid ? src[q] : make_uint4(0, 0, 0, 0);
            const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[8 * q + 2 * e] = __uint_as_float(w[e] << 16);
                x[8 * q + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
            }
        }
    } else {
        const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(g) + off);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float4 t = valid ? src[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            x[4 * q] = t.x; x[4 * q + 1] = t.y; x[4 * q + 2] = t.z; x[4 * q + 3] = t.w;
        }
    }
}

// ------------------------------------------------------------------------
// L_c = Gamma_K,c^T [V_c | 1]: M = components, N = d_v, contraction over the
// chunk's 128 tokens.  A = Gamma_K^T in TMEM: warp w owns components
// 32 (w % 4) + lane and tokens [64 (w / 4), +64).  For fp32 operands the
// 128 A columns first hold the tf32 parts (passes hi*hi, hi*lo), then the
// remainders (pass lo*hi), so that 256 TMEM columns suffice and two CTAs
// share an SM.  B = V^T in shared memory.
template <bool BF16, int DV>
struct StateSmem {
    static constexpr uint32_t VT = tile_bytes<BF16>(DV);
    static constexpr size_t bytes = 1024 + 2 * (size_t)VT + 2 * kK * 4 + 64;
};

template <bool BF16, int DV>
__global__ void __launch_bounds__(kTCThreads, 2)
    k_chunk_state_tc(int N, const void *__restrict__ gk, const void *__restrict__ v, bool v_bf16,
                     float *__restrict__ partial, int nblk)
{
    using Sm = StateSmem<BF16, DV>;
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *vt_hi = sm, *vt_lo = sm + Sm::VT;
    float *zp = reinterpret_cast<float *>(sm + 2 * Sm::VT);         // [2][128] partial Z
    uint64_t *bar = reinterpret_cast<uint64_t *>(zp + 2 * kK);      // [2]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, h = warp >> 2;
    const uint32_t lane0 = 32 * quarter;
    const int k = lane0 + lane;
    const long long bh = blockIdx.y;
    const int c0 = blockIdx.x * kC;
    const int nr = min(kC, N - c0);
    constexpr uint32_t A = 0, D_COL = 128;

    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(smem_addr(bar), 1);
        mbar_init(smem_addr(bar + 1), 1);
        mbar_init_fence();
    }
    // this thread's 64 A values: Gamma_K[c0 + 64h + jj][k] (coalesced across k)
    float x[64];
#pragma unroll
    for (int jj = 0; jj < 64; ++jj) {
        const int r = 64 * h + jj;
        x[jj] = r < nr ? load_elem(gk, (bh * N + c0 + r) * (long long)kK + k, BF16) : 0.f;
    }
    stage_vt<BF16, DV>(v, v_bf16, bh * N + c0, nr, vt_hi, vt_lo, tid);
    float z = 0.f;
#pragma unroll
    for (int jj = 0; jj < 64; ++jj) z += x[jj];
    zp[h * kK + k] = z;
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *tslot;
    put_a64<BF16>(tbase, lane0, A, A, 64 * h, x, 0);
    tmem_wait_st();
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
        mma_pass<BF16>(tbase + D_COL, tbase + A, vt_hi, DV, false);
        if constexpr (!BF16) mma_pass<BF16>(tbase + D_COL, tbase + A, vt_lo, DV, true);
        mma_commit(smem_addr(bar));
    }
    __syncwarp();
    bool ok = mbar_wait(smem_addr(bar), 0);
    fence_after_sync();
    if constexpr (!BF16) {
        put_a64<BF16>(tbase, lane0, A, A, 64 * h, x, 1);   // remainders into the same columns
        tmem_wait_st();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        if (tid == 0) {
            mma_pass<BF16>(tbase + D_COL, tbase + A, vt_hi, DV, true);
            mma_commit(smem_addr(bar + 1));
        }
        __syncwarp();
        ok = mbar_wait(smem_addr(bar + 1), 0) && ok;
        fence_after_sync();
    }
    // block layout on this path: Vt^T as DV rows of K, then Z as row DV
    const long long SZ = (long long)kK * DV + kK;
    float *o = partial + (bh * nblk + blockIdx.x) * SZ;
    const float qnan = __int_as_float(0x7fc00000);
#pragma unroll
    for (int cb = 0; cb < DV / 32; ++cb) {
        const int c = h * (DV / 2) + 16 * cb;
        uint32_t r[16];
        tmem_ld16(tmem_at(tbase, lane0, D_COL + c), r);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q) o[(long long)(c + q) * kK + k] = ok ? __uint_as_float(r[q]) : qnan;
    }
    if (h == 0) o[(long long)kK * DV + k] = ok ? zp[k] + zp[kK + k] : qnan;
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

// ------------------------------------------------------------------------
// Chunk output.  Warp w owns TMEM lanes (rows) 32 (w % 4) + lane and column
// half w / 4 of every row-wise step.  Every tile arrives by TMA (bulk tensor
// copies with the 128-byte swizzle) straight into the operand layout:
//   X_hi <- Gamma_K (B of P), X_lo <- Gamma_Q (moved to TMEM as the A operand),
//   Y_hi <- carried memory Vt^T (B of U = Gq Vt; fp32 operands only, the bf16
//           path converts it with threads), later X <- V (transposed by threads
//           into Y as the B of U += P_m V).
// For fp32 operands the raw fp32 tile is the tf32 "hi" image (the tensor core
// reads only the tf32 bits); threads derive the exact remainders in place.
template <bool BF16, int DV>
struct OutSmem {
    static constexpr uint32_t GK = tile_bytes<BF16>(kC);   // Gamma_K chunk, 128 x 128
    static constexpr uint32_t Y = tile_bytes<BF16>(DV);    // Vt^T, then V^T: DV x 128
    static constexpr size_t bytes = 1024 + 2 * (size_t)GK + 2 * (size_t)Y + kK * 4 + 4 * kK * 4 + 64;
};

struct OutMaps {
    CUtensorMap gq, gk, v, s;   // s: carried memory blocks (fp32 operands only)
};

// CAUSAL = false gives the bidirectional read: U = Gamma_Q [Vt | Z] with the
// total memory of the sequence (the same block for every chunk), no P.
template <bool BF16, int DV, bool CAUSAL>
__global__ void __launch_bounds__(kTCThreads, 1)
    k_chunk_out_tc(const __grid_constant__ OutMaps maps, int N, float eps, bool v_bf16,
                   const float *__restrict__ states, int nblk, float *__restrict__ out)
{
    using El = Elem<BF16>;
    using Sm = OutSmem<BF16, DV>;
    constexpr int EV_MAX = 4;
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *x_hi = sm, *x_lo = sm + Sm::GK;                  // Gamma_K / Gamma_Q, later V
    unsigned char *y_hi = sm + 2 * Sm::GK, *y_lo = y_hi + Sm::Y;    // Vt^T, later V^T
    float *z_s = reinterpret_cast<float *>(y_lo + Sm::Y);           // [128] Z of the carried memory
    float *part = z_s + kK;                                         // [4][128]: qz halves, row-sum halves
    uint64_t *bar = reinterpret_cast<uint64_t *>(part + 4 * kK);    // [5]: loads, U, P, V, final
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 5);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = warp >> 2;
    const uint32_t lane0 = 32 * (warp & 3);
    const int i = lane0 + lane;                 // row of the chunk owned in TMEM
    const long long bh = blockIdx.y;
    const int c0 = blockIdx.x * kC;
    const int nr = min(kC, N - c0);
    const int row0 = (int)(bh * N + c0);
    constexpr uint32_t A_HI = 0, A_LO = 128, D_P = 256, D_U = 384;
    constexpr int GBOX = 128 / El::E;                       // Gamma columns per TMA box
    const int ev = v_bf16 ? 2 : 4;
    const int vbox = 128 / ev;                              // V columns per TMA box
    (void)EV_MAX;

    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int b = 0; b < 5; ++b) mbar_init(smem_addr(bar + b), 1);
        mbar_init_fence();
        uint32_t bytes = (CAUSAL ? 2 : 1) * Sm::GK + (BF16 ? 0u : (uint32_t)Sm::Y);
        mbar_expect_tx(smem_addr(bar), bytes);
        for (int a = 0; a < kK / GBOX; ++a) {
            if (CAUSAL) tma_load_2d(smem_addr(x_hi + a * (kC * 128)), &maps.gk, a * GBOX, row0, smem_addr(bar));
            tma_load_2d(smem_addr(x_lo + a * (kC * 128)), &maps.gq, a * GBOX, row0, smem_addr(bar));
        }
        if constexpr (!BF16) {
            const int srow = (int)((CAUSAL ? bh * nblk + blockIdx.x : bh) * (DV + 1));
            for (int a = 0; a < kK / 32; ++a)
                tma_load_2d(smem_addr(y_hi + a * (DV * 128)), &maps.s, a * 32, srow, smem_addr(bar));
        }
    }
    const long long SZ = (long long)kK * DV + kK;
    const float *st = states + (CAUSAL ? bh * nblk + blockIdx.x : bh) * SZ;
    if (tid < kK) {
        const float zk = st[(long long)kK * DV + tid];
        z_s[tid] = BF16 ? bf16r(zk) : zk;
    }
    if constexpr (BF16) {
        // carried memory (block rows c of K) -> Y as bf16 Vt^T; lanes run over components
        constexpr int PER = (DV * kK / 4) / kTCThreads;
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int f = tid + u * kTCThreads, c = f / (kK / 4), k4 = 4 * (f % (kK / 4));
            const float4 t = reinterpret_cast<const float4 *>(st + (long long)c * kK)[k4 / 4];
            const uint2 p = make_uint2(pack_bf16(t.x, t.y), pack_bf16(t.z, t.w));
            *reinterpret_cast<uint2 *>(y_hi + sw128_offset(c, k4, DV, 2)) = p;
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *tslot;
    bool ok = mbar_wait(smem_addr(bar), 0);

    // A = Gamma_Q (row i, operand columns [64h, 64h + 64)) from its landing tile; partial Gamma_Q,i . Z
    {
        float xq[64];
#pragma unroll
        for (int q = 0; q < 64 / 4; ++q) {
            const int k = 64 * h + 4 * q;
            if constexpr (BF16) {
                const uint2 t = *reinterpret_cast<const uint2 *>(x_lo + sw128_offset(i, k, kC, 2));
                xq[4 * q] = __uint_as_float(t.x << 16);
                xq[4 * q + 1] = __uint_as_float(t.x & 0xffff0000u);
                xq[4 * q + 2] = __uint_as_float(t.y << 16);
                xq[4 * q + 3] = __uint_as_float(t.y & 0xffff0000u);
            } else {
                const float4 t = *reinterpret_cast<const float4 *>(x_lo + sw128_offset(i, k, kC, 4));
                xq[4 * q] = t.x; xq[4 * q + 1] = t.y; xq[4 * q + 2] = t.z; xq[4 * q + 3] = t.w;
            }
        }
        float qz = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) qz = fmaf(xq[j], z_s[64 * h + j], qz);
        part[h * kK + i] = qz;
        put_a64<BF16>(tbase, lane0, A_HI, A_LO, 64 * h, xq);
    }
    if constexpr (!BF16) {
        __syncthreads();   // Gamma_Q has been read from X_lo
        // exact remainders of Gamma_K (X_lo) and of the carried memory (Y_lo), in place
        constexpr int PX = Sm::GK / 16 / kTCThreads, PY = Sm::Y / 16 / kTCThreads;
#pragma unroll 4
        for (int u = 0; u < (CAUSAL ? PX : 0); ++u) {
            const uint32_t off = 16 * (tid + u * kTCThreads);
            const float4 t = *reinterpret_cast<const float4 *>(x_hi + off);
            *reinterpret_cast<float4 *>(x_lo + off) = make_float4(t.x - tf32_hi(t.x), t.y - tf32_hi(t.y),
                                                                  t.z - tf32_hi(t.z), t.w - tf32_hi(t.w));
        }
#pragma unroll 4
        for (int u = 0; u < PY; ++u) {
            const uint32_t off = 16 * (tid + u * kTCThreads);
            const float4 t = *reinterpret_cast<const float4 *>(y_hi + off);
            *reinterpret_cast<float4 *>(y_lo + off) = make_float4(t.x - tf32_hi(t.x), t.y - tf32_hi(t.y),
                                                                  t.z - tf32_hi(t.z), t.w - tf32_hi(t.w));
        }
    }
    tmem_wait_st();
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
        mma_all<BF16>(tbase + D_U, tbase + A_HI, tbase + A_LO, y_hi, y_lo, DV, false);    // U = Gq Vt
        mma_commit(smem_addr(bar + 1));
        if (CAUSAL) {
            mma_all<BF16>(tbase + D_P, tbase + A_HI, tbase + A_LO, x_hi, x_lo, kC, false);    // P = Gq Gk^T
            mma_commit(smem_addr(bar + 2));
        }
    }
    __syncwarp();
    if constexpr (!CAUSAL) {
        ok = mbar_wait(smem_addr(bar + 1), 0) && ok;
        fence_after_sync();
    } else {
    ok = mbar_wait(smem_addr(bar + 2), 0) && ok;   // P done (and U, committed earlier)
    fence_after_sync();
    if (tid == 0) {
        // X is free: bring V in while P_m is formed
        fence_proxy_async();
        mbar_expect_tx(smem_addr(bar + 3), (uint32_t)(kC * DV * ev));
        for (int a = 0; a < DV / vbox; ++a)
            tma_load_2d(smem_addr(x_hi + a * (kC * 128)), &maps.v, a * vbox, row0, smem_addr(bar + 3));
    }
    // P_m = P with j > i zeroed replaces Gamma_Q as the A operand; row sums on CUDA cores
    {
        float x[64];
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            uint32_t r[16];
            tmem_ld16(tmem_at(tbase, lane0, D_P + 64 * h + 16 * b), r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int jj = 64 * h + 16 * b + j;
                x[16 * b + j] = jj <= i ? __uint_as_float(r[j]) : 0.f;
            }
        }
        float ps = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) ps += BF16 ? bf16r(x[j]) : x[j];
        part[(2 + h) * kK + i] = ps;
        put_a64<BF16>(tbase, lane0, A_HI, A_LO, 64 * h, x);
    }
    ok = mbar_wait(smem_addr(bar + 3), 0) && ok;
    // V^T (element (c, j)) into Y from the V tile in X; lanes run over tokens
    {
        constexpr int PER = (kC * DV / 4) / kTCThreads;
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int f = tid + u * kTCThreads, j = f % kC, c4 = 4 * (f / kC);
            float4 t;
            if (j >= nr) {
                t = make_float4(0.f, 0.f, 0.f, 0.f);
            } else if (v_bf16) {
                const uint2 w = *reinterpret_cast<const uint2 *>(x_hi + sw128_offset(j, c4, kC, 2));
                t = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                                __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
            } else {
                t = *reinterpret_cast<const float4 *>(x_hi + sw128_offset(j, c4, kC, 4));
            }
            put<BF16>(y_hi, y_lo, sw128_offset(c4 + 0, j, DV, El::E), t.x);
            put<BF16>(y_hi, y_lo, sw128_offset(c4 + 1, j, DV, El::E), t.y);
            put<BF16>(y_hi, y_lo, sw128_offset(c4 + 2, j, DV, El::E), t.z);
            put<BF16>(y_hi, y_lo, sw128_offset(c4 + 3, j, DV, El::E), t.w);
        }
    }
    tmem_wait_st();
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
        mma_all<BF16>(tbase + D_U, tbase + A_HI, tbase + A_LO, y_hi, y_lo, DV, true);     // U += P_m V
        mma_commit(smem_addr(bar + 4));
    }
    __syncwarp();
    ok = mbar_wait(smem_addr(bar + 4), 0) && ok;
    fence_after_sync();
    }

    const float den = part[i] + part[kK + i] + (CAUSAL ? part[2 * kK + i] + part[3 * kK + i] : 0.f) + eps;
    const float qnan = __int_as_float(0x7fc00000);
#pragma unroll
    for (int cb = 0; cb < DV / 32; ++cb) {
        const int c = h * (DV / 2) + 16 * cb;
        uint32_t r[16];
        tmem_ld16(tmem_at(tbase, lane0, D_U + c), r);
        tmem_wait_ld();
        if (i < nr) {
            float4 *dst = reinterpret_cast<float4 *>(out + (bh * N + c0 + i) * (long long)DV + c);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                dst[q] = ok ? make_float4(__uint_as_float(r[4 * q]) / den, __uint_as_float(r[4 * q + 1]) / den,
                                          __uint_as_float(r[4 * q + 2]) / den, __uint_as_float(r[4 * q + 3]) / den)
                            : make_float4(qnan, qnan, qnan, qnan);
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

} // namespace

bool tc_path_eligible(int K, int DV, bool g_bf16) { return K == kK && (DV == 64 || (DV == 128 && g_bf16)); }

bool tc_path_applies(const Dims &dm) { return dm.C == kC && tc_path_eligible(dm.K, dm.DV, dm.g_bf16); }


template <bool BF16, int DV>
cudaError_t state_tc(const Dims &dm, const void *gk, const void *v, float *partial, cudaStream_t st)
{
    constexpr size_t smem = StateSmem<BF16, DV>::bytes;
    static cudaError_t attr = allow_smem(k_chunk_state_tc<BF16, DV>, smem);
    if (attr != cudaSuccess) return attr;
    dim3 grid(dm.nblk(), (unsigned)dm.BH());
    k_chunk_state_tc<BF16, DV><<<grid, kTCThreads, smem, st>>>(dm.N, gk, v, dm.v_bf16, partial, dm.nblk());
    return cudaGetLastError();
}

template <bool BF16, int DV, bool CAUSAL>
cudaError_t out_tc(const Dims &dm, const void *gq, const void *gk, const void *v, const float *states, float *out,
                   cudaStream_t st)
{
    constexpr size_t smem = OutSmem<BF16, DV>::bytes;
    static cudaError_t attr = allow_smem(k_chunk_out_tc<BF16, DV, CAUSAL>, smem);
    if (attr != cudaSuccess) return attr;
    OutMaps maps;
    const unsigned long long rows = (unsigned long long)dm.BH() * dm.N;
    bool ok = make_tma_2d(&maps.gq, gq, BF16, rows, kK, kC) && make_tma_2d(&maps.gk, gk, BF16, rows, kK, kC) &&
              make_tma_2d(&maps.v, v, dm.v_bf16, rows, DV, kC);
    if (!BF16)
        ok = ok && make_tma_2d(&maps.s, states, false,
                               (unsigned long long)dm.BH() * (CAUSAL ? dm.nblk() : 1) * (DV + 1), kK, DV);
    else
        maps.s = maps.gq;
    if (!ok) return cudaErrorInvalidValue;
    dim3 grid(dm.nblk(), (unsigned)dm.BH());
    k_chunk_out_tc<BF16, DV, CAUSAL><<<grid, kTCThreads, smem, st>>>(maps, dm.N, dm.eps, dm.v_bf16, states,
                                                                      dm.nblk(), out);
    return cudaGetLastError();
}

cudaError_t launch_chunk_state_tc(const Dims &dm, const void *gk, const void *v, float *partial, cudaStream_t st)
{
    if (dm.g_bf16) {
        if (dm.DV == 64) return state_tc<true, 64>(dm, gk, v, partial, st);
        if (dm.DV == 128) return state_tc<true, 128>(dm, gk, v, partial, st);
    } else if (dm.DV == 64) {
        return state_tc<false, 64>(dm, gk, v, partial, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_chunk_out_tc(const Dims &dm, bool causal, const void *gq, const void *gk, const void *v,
                                const float *states, float *out, cudaStream_t st)
{
    if (dm.g_bf16) {
        if (dm.DV == 64)
            return causal ? out_tc<true, 64, true>(dm, gq, gk, v, states, out, st)
                          : out_tc<true, 64, false>(dm, gq, gk, v, states, out, st);
        if (dm.DV == 128)
            return causal ? out_tc<true, 128, true>(dm, gq, gk, v, states, out, st)
                          : out_tc<true, 128, false>(dm, gq, gk, v, states, out, st);
    } else if (dm.DV == 64) {
        return causal ? out_tc<false, 64, true>(dm, gq, gk, v, states, out, st)
                      : out_tc<false, 64, false>(dm, gq, gk, v, states, out, st);
    }
    return cudaErrorInvalidValue;
}

} // namespace gma
