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
#include <climits>
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
// (columns from a_col), B a K-major SW128 tile of `nrows` rows whose 128-byte
// atom columns lie `atom_stride` bytes apart (nrows * 128 when packed).
template <bool BF16>
__device__ __forceinline__ void mma_pass_at(uint32_t d_tmem, uint32_t a_col, const unsigned char *b, uint32_t nrows,
                                            uint32_t atom_stride, bool accumulate)
{
    using El = Elem<BF16>;
    const uint32_t id = idesc(128, nrows, El::FMT);
    constexpr int ksteps = kK * El::E / 32;
#pragma unroll 1
    for (int kk = 0; kk < ksteps; ++kk) {
        const uint32_t kb = kk * 32;
        const uint32_t boff = (kb >> 7) * atom_stride + (kb & 127);
        mma_ts(!BF16, d_tmem, a_col + kk * El::COLS_PER_KSTEP, sdesc_sw128(smem_addr(b + boff)), id,
               (accumulate || kk > 0) ? 1u : 0u);
    }
}
template <bool BF16>
__device__ __forceinline__ void mma_pass(uint32_t d_tmem, uint32_t a_col, const unsigned char *b, uint32_t nrows,
                                         bool accumulate)
{
    mma_pass_at<BF16>(d_tmem, a_col, b, nrows, nrows * 128, accumulate);
}

// All passes of D (+)= A * B^T: fp32 operands as hi*hi + hi*lo + lo*hi.
template <bool BF16>
__device__ __forceinline__ void mma_all(uint32_t d_tmem, uint32_t a_hi, uint32_t a_lo, const unsigned char *b_hi,
                                        const unsigned char *b_lo, uint32_t nrows, uint32_t atom_stride,
                                        bool accumulate)
{
    mma_pass_at<BF16>(d_tmem, a_hi, b_hi, nrows, atom_stride, accumulate);
    if constexpr (!BF16) {
        mma_pass_at<BF16>(d_tmem, a_hi, b_lo, nrows, atom_stride, true);
        mma_pass_at<BF16>(d_tmem, a_lo, b_hi, nrows, atom_stride, true);
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
// Chunk output, persistent: CTA b takes the items [b * per, (b + 1) * per) of
// the list (slice, chunk) in order.  16 warps: warp w owns TMEM lanes (rows)
// 32 (w % 4) + lane and column quarter w / 4 of every row-wise step.
//
// A tcgen05.mma instruction costs about the same time for any N up to 256,
// so U = Gq Vt and P = Gq Gk^T, which share the A operand Gq, are one MMA
// chain with N = C + d_v: its B operand is the tile [Gk ; Vt^T] of C + d_v
// rows, K-major with the 128-byte swizzle, each 128-byte atom column holding
// the C rows of Gk followed by the d_v rows of Vt^T, and its accumulator is
// [P | U] in consecutive TMEM columns.  Shared memory holds two such tiles:
//   B <- Gk (TMA) and Vt^T (TMA for fp32 operands; bf16: converted by threads)
//        (raw fp32 = the tf32 part: the tensor core reads only the tf32 bits);
//   L <- Gq in its Gk rows (TMA; moved to TMEM as the A operand), then the exact
//        remainders of B (fp32 operands only).
// After P: the Vt^T rows of B and L take V^T (parts and remainders, written by
// threads from registers loaded while the tensor core works), the B operand
// of U += P_m V.  The next item's Gamma tiles are fetched into the Gk rows as
// soon as [P | U] is done, its carried memory as soon as U += P_m V is done,
// so that the loads overlap the rest of the item.
constexpr int kOutThreads = 512;

template <bool BF16, int DV>
struct OutSmem {
    static constexpr uint32_t ATOMS = kK * Elem<BF16>::E / 128;        // 128-byte atom columns
    static constexpr uint32_t PART = kC * 128;                         // Gk rows of an atom column
    static constexpr uint32_t ATOM = (kC + DV) * 128;                  // bytes of an atom column
    static constexpr uint32_t TILE = ATOMS * ATOM;                     // [Gk ; Vt^T]
    static constexpr size_t bytes = 1024 + 2 * (size_t)TILE + kK * 4 + 8 * kK * 4 + 64;
};

// Byte offset of element (r, k) in a tile whose atom columns are `stride` apart.
__device__ __forceinline__ uint32_t fused_off(uint32_t r, uint32_t k, uint32_t E, uint32_t stride)
{
    const uint32_t kb = k * E, inner = kb & 127u;
    return (kb >> 7) * stride + (r >> 3) * 1024u + (r & 7u) * 128u + (((inner >> 4) ^ (r & 7u)) << 4) + (inner & 15u);
}

struct OutMaps {
    CUtensorMap gq, gk, s;   // s: carried memory blocks (fp32 operands only)
    CUtensorMap o;           // output [slices][N][d_v], boxes of 64 rows x 32 columns (fp32 operands only)
};

// 32 consecutive A-operand values of this thread's TMEM lane from operand
// column j0 (a multiple of 32): fp32 -> tf32 part at a_hi, remainder at a_lo
// (part = 0: parts only, 1: remainders only, 2: both); bf16 -> packed pairs at a_hi.
template <bool BF16>
__device__ __forceinline__ void put_a32(uint32_t tbase, uint32_t lane0, uint32_t a_hi, uint32_t a_lo, int j0,
                                        const float (&x)[32], int part = 2)
{
    if constexpr (BF16) {
        uint32_t p[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) p[j] = pack_bf16(x[2 * j], x[2 * j + 1]);
        tmem_st16(tmem_at(tbase, lane0, a_hi + j0 / 2), p);
    } else {
#pragma unroll
        for (int b = 0; b < 2; ++b) {
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

// CAUSAL = false gives the bidirectional read: U = Gamma_Q [Vt | Z] with the
// total memory of the sequence (the same block for every chunk), no P.
template <bool BF16, int DV, bool CAUSAL>
__global__ void __launch_bounds__(kOutThreads, 1)
    k_chunk_out_tc(const __grid_constant__ OutMaps maps, int N, int nblk, long long items, float eps,
                   const void *__restrict__ v, bool v_bf16, const float *__restrict__ states, float *__restrict__ out)
{
    using El = Elem<BF16>;
    using Sm = OutSmem<BF16, DV>;
    static_assert(BF16 || DV == 64, "fp32 operands: d_v = 64 only (the output staging assumes it)");
    constexpr int VPER = (kC * DV / 4) / kOutThreads;       // float4 of V per thread
    constexpr uint32_t AS = Sm::ATOM, PART = Sm::PART;
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *tb = sm, *tl = sm + Sm::TILE;                     // B tile, L tile
    float *z_s = reinterpret_cast<float *>(tl + Sm::TILE);          // [128] Z of the carried memory
    float *part = z_s + kK;                                         // [8][128]: qz quarters, row-sum quarters
    uint64_t *bar = reinterpret_cast<uint64_t *>(part + 8 * kK);    // [4]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = warp >> 2;                    // column quarter
    const uint32_t lane0 = 32 * (warp & 3);
    const int i = lane0 + lane;                 // row of the chunk owned in TMEM
    const long long per = (items + gridDim.x - 1) / gridDim.x;
    const long long it0 = (long long)blockIdx.x * per;
    const long long it1 = it0 + per < items ? it0 + per : items;
    constexpr uint32_t A_HI = 0, A_LO = 128, D_P = 256, D_U = D_P + kC;
    constexpr int GBOX = 128 / El::E;                       // Gamma columns per TMA box
    const uint32_t BAR_G = smem_addr(bar), BAR_S = smem_addr(bar + 1), BAR_M = smem_addr(bar + 2),
                   BAR_V = smem_addr(bar + 3);
    const long long SZ = (long long)kK * DV + kK;

    // block of the carried memory read by item it
    auto mem_block = [&](long long it) -> long long { return CAUSAL ? it : it / nblk; };
    auto load_gamma = [&](long long it) {   // one thread
        const int row0 = (int)((it / nblk) * N + (it % nblk) * kC);
        mbar_expect_tx(BAR_G, (CAUSAL ? 2u : 1u) * (uint32_t)(kC * kK * El::E));
        for (int a = 0; a < (int)Sm::ATOMS; ++a) {
            if (CAUSAL) tma_load_2d(smem_addr(tb + a * AS), &maps.gk, a * GBOX, row0, BAR_G);
            tma_load_2d(smem_addr(tl + a * AS), &maps.gq, a * GBOX, row0, BAR_G);
        }
    };
    auto load_memory = [&](long long it) {   // one thread, fp32 operands
        const int srow = (int)(mem_block(it) * (DV + 1));
        mbar_expect_tx(BAR_S, (uint32_t)(DV * kK * 4));
        for (int a = 0; a < kK / 32; ++a)
            tma_load_2d(smem_addr(tb + a * AS + PART), &maps.s, a * 32, srow, BAR_S);
    };

    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 512);
        tmem_relinquish();
    }
    // loads in flight that the loop has not waited for (thread 0's record)
    bool pend_g = false, pend_s = false;
    uint32_t ph_g = 0, ph_s = 0;
    if (tid == 0) {
        for (int b = 0; b < 4; ++b) mbar_init(smem_addr(bar + b), 1);
        mbar_init_fence();
        if (it0 < it1) {
            load_gamma(it0);
            pend_g = true;
            if (!BF16) {
                load_memory(it0);
                pend_s = true;
            }
        }
    }
    // Z of the carried memory, loaded one item ahead
    float zreg = (tid < kK && it0 < it1) ? states[mem_block(it0) * SZ + (long long)kK * DV + tid] : 0.f;
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *tslot;
    bool ok = true;
    const float qnan = __int_as_float(0x7fc00000);

    for (long long it = it0; it < it1 && ok; ++it) {
        const uint32_t ph = (uint32_t)((it - it0) & 1);
        const long long bh = it / nblk;
        const int c0 = (int)(it % nblk) * kC;
        const int nr = min(kC, N - c0);
        const long long rowbase = bh * N + c0;
        const bool more = it + 1 < it1;
        if (tid < kK) z_s[tid] = BF16 ? bf16r(zreg) : zreg;
        if constexpr (BF16) {
            // carried memory (block rows c of K) -> Vt^T rows of B as bf16; lanes run over components
            const float *st = states + mem_block(it) * SZ;
            constexpr int PER = (DV * kK / 4) / kOutThreads;
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int f = tid + u * kOutThreads, c = f / (kK / 4), k4 = 4 * (f % (kK / 4));
                const float4 t = reinterpret_cast<const float4 *>(st + (long long)c * kK)[k4 / 4];
                const uint2 p = make_uint2(pack_bf16(t.x, t.y), pack_bf16(t.z, t.w));
                *reinterpret_cast<uint2 *>(tb + fused_off(kC + c, k4, 2, AS)) = p;
            }
        }
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        const bool ok_g = mbar_wait(BAR_G, ph), ok_s = BF16 || mbar_wait(BAR_S, ph);
        ok = ok && ok_g && ok_s;
        if (tid == 0) {   // a load whose wait gave up is still in flight
            pend_g = pend_g && !ok_g;
            pend_s = pend_s && !ok_s;
        }

        // A = Gamma_Q (row i, operand columns [32g, 32g + 32)) from its landing rows; partial Gamma_Q,i . Z
        {
            float xq[32];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int k = 32 * g + 4 * q;
                if constexpr (BF16) {
                    const uint2 t = *reinterpret_cast<const uint2 *>(tl + fused_off(i, k, 2, AS));
                    xq[4 * q] = __uint_as_float(t.x << 16);
                    xq[4 * q + 1] = __uint_as_float(t.x & 0xffff0000u);
                    xq[4 * q + 2] = __uint_as_float(t.y << 16);
                    xq[4 * q + 3] = __uint_as_float(t.y & 0xffff0000u);
                } else {
                    const float4 t = *reinterpret_cast<const float4 *>(tl + fused_off(i, k, 4, AS));
                    xq[4 * q] = t.x; xq[4 * q + 1] = t.y; xq[4 * q + 2] = t.z; xq[4 * q + 3] = t.w;
                }
            }
            float qz = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) qz = fmaf(xq[j], z_s[32 * g + j], qz);
            part[g * kK + i] = qz;
            put_a32<BF16>(tbase, lane0, A_HI, A_LO, 32 * g, xq);
        }
        tmem_wait_st();
        fence_proxy_async();
        fence_before_sync();
        if (!BF16 && tid == 0) bulk_wait_read();   // the previous output tile has left L
        __syncthreads();   // Gamma_Q has been read from L and is in TMEM
        fence_after_sync();
        // the passes that do not read the remainders of B start at once:
        // [P | U] = Gq [Gk ; Vt^T]^T (bidirectional read: U = Gq Vt)
        const unsigned char *b0 = CAUSAL ? tb : tb + PART, *l0 = CAUSAL ? tl : tl + PART;
        const uint32_t d0 = CAUSAL ? D_P : D_U, nb = CAUSAL ? kC + DV : DV;
        if (tid == 0) {
            mma_pass_at<BF16>(tbase + d0, tbase + A_HI, b0, nb, AS, false);
            if constexpr (!BF16) mma_pass_at<BF16>(tbase + d0, tbase + A_LO, b0, nb, AS, true);
            else mma_commit(BAR_M);
        }
        if constexpr (!BF16) {
            // exact remainders of B into L, in place (bidirectional read: the Vt^T rows only),
            // by warps 1..15 while warp 0 issues the passes above
            const int w0 = tid >= 32 ? tid - 32 : INT_MAX;   // warp 0 takes no words
            if constexpr (CAUSAL) {
#pragma unroll 1
                for (int w = w0; w < (int)(Sm::TILE / 16); w += kOutThreads - 32) {
                    const uint32_t off = 16 * w;
                    const float4 t = *reinterpret_cast<const float4 *>(tb + off);
                    *reinterpret_cast<float4 *>(tl + off) = make_float4(t.x - tf32_hi(t.x), t.y - tf32_hi(t.y),
                                                                        t.z - tf32_hi(t.z), t.w - tf32_hi(t.w));
                }
            } else {
                constexpr int PV16 = DV * 128 / 16;                       // 16-byte words per atom's Vt^T rows
#pragma unroll 4
                for (int w = w0; w < (int)Sm::ATOMS * PV16; w += kOutThreads - 32) {
                    const uint32_t off = (w / PV16) * AS + PART + 16 * (w % PV16);
                    const float4 t = *reinterpret_cast<const float4 *>(tb + off);
                    *reinterpret_cast<float4 *>(tl + off) = make_float4(t.x - tf32_hi(t.x), t.y - tf32_hi(t.y),
                                                                        t.z - tf32_hi(t.z), t.w - tf32_hi(t.w));
                }
            }
            fence_proxy_async();
            fence_before_sync();
            __syncthreads();
            fence_after_sync();
            if (tid == 0) {   // the pass that reads the remainders
                mma_pass_at<BF16>(tbase + d0, tbase + A_HI, l0, nb, AS, true);
                mma_commit(BAR_M);
            }
        }
        __syncwarp();
        // V of this chunk (lanes over tokens), loaded while the tensor core works, consumed after P
        float4 vr[CAUSAL ? VPER : 1];
        if constexpr (CAUSAL) {
#pragma unroll
            for (int u = 0; u < VPER; ++u) {
                const int f = tid + u * kOutThreads, j = f % kC, c4 = f / kC;
                vr[u] = j < nr ? load4(v, (rowbase + j) * DV + 4 * c4, v_bf16) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        ok = mbar_wait(BAR_M, ph) && ok;
        fence_after_sync();
        if constexpr (!CAUSAL) {
            if (tid == 0 && more && ok) {   // B and L are free: the next item's tiles
                fence_proxy_async();
                load_gamma(it + 1);
                pend_g = true;
                ph_g = ph ^ 1u;
                if (!BF16) {
                    load_memory(it + 1);
                    pend_s = true;
                    ph_s = ph ^ 1u;
                }
            }
        } else {
            if (tid == 0 && more && ok) {   // the Gamma rows are free: the next item's Gamma tiles
                fence_proxy_async();
                load_gamma(it + 1);
                pend_g = true;
                ph_g = ph ^ 1u;
            }
            // P_m = P with j > i zeroed replaces Gamma_Q as the A operand; row sums on CUDA cores
            auto load_pm = [&](float (&x)[32]) {
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
            };
            {
                float x[32];
                load_pm(x);
                float ps = 0.f;
#pragma unroll
                for (int j = 0; j < 32; ++j) ps += BF16 ? bf16r(x[j]) : x[j];
                part[(4 + g) * kK + i] = ps;
                // U += P_m V: the tf32 parts first (pass hi * hi), then the remainders (hi * lo, lo * hi)
                put_a32<BF16>(tbase, lane0, A_HI, A_LO, 32 * g, x, BF16 ? 2 : 0);
                // V^T (element (c, j)) into the Vt^T rows of B from registers; lanes run over tokens
#pragma unroll
                for (int u = 0; u < VPER; ++u) {
                    const int f = tid + u * kOutThreads, j = f % kC, c4 = 4 * (f / kC);
                    const float e4[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t off = fused_off(kC + c4 + e, j, El::E, AS);
                        if constexpr (BF16)
                            *reinterpret_cast<__nv_bfloat16 *>(tb + off) = __float2bfloat16_rn(e4[e]);
                        else
                            *reinterpret_cast<float *>(tb + off) = tf32_hi(e4[e]);
                    }
                }
                tmem_wait_st();
                fence_proxy_async();
                fence_before_sync();
                __syncthreads();
                fence_after_sync();
                if (tid == 0) {
                    mma_pass_at<BF16>(tbase + D_U, tbase + A_HI, tb + PART, DV, AS, true);
                    if constexpr (BF16) mma_commit(BAR_V);
                }
                if constexpr (!BF16) {
                    load_pm(x);   // P is still in TMEM: reloading beats keeping 32 values live
                    put_a32<BF16>(tbase, lane0, A_HI, A_LO, 32 * g, x, 1);
#pragma unroll
                    for (int u = 0; u < VPER; ++u) {
                        const int f = tid + u * kOutThreads, j = f % kC, c4 = 4 * (f / kC);
                        const float e4[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            *reinterpret_cast<float *>(tl + fused_off(kC + c4 + e, j, 4, AS)) = e4[e] - tf32_hi(e4[e]);
                    }
                    tmem_wait_st();
                    fence_proxy_async();
                    fence_before_sync();
                    __syncthreads();
                    fence_after_sync();
                    if (tid == 0) {
                        mma_pass_at<BF16>(tbase + D_U, tbase + A_HI, tl + PART, DV, AS, true);
                        mma_pass_at<BF16>(tbase + D_U, tbase + A_LO, tb + PART, DV, AS, true);
                        mma_commit(BAR_V);
                    }
                }
            }
            __syncwarp();
            ok = mbar_wait(BAR_V, ph) && ok;
            fence_after_sync();
            if (!BF16 && tid == 0 && more && ok) {   // the Vt^T rows are free: the next item's carried memory
                fence_proxy_async();
                load_memory(it + 1);
                pend_s = true;
                ph_s = ph ^ 1u;
            }
        }

        if (tid < kK && more) zreg = states[mem_block(it + 1) * SZ + (long long)kK * DV + tid];
        float den = eps;
#pragma unroll
        for (int q = 0; q < (CAUSAL ? 8 : 4); ++q) den += part[q * kK + i];
        const float inv = 1.0f / den;
#pragma unroll
        for (int cb = 0; cb < DV / 64; ++cb) {
            const int c = g * (DV / 4) + 16 * cb;
            uint32_t r[16];
            tmem_ld16(tmem_at(tbase, lane0, D_U + c), r);
            tmem_wait_ld();
            float4 o4[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                o4[q] = ok ? make_float4(__uint_as_float(r[4 * q]) * inv, __uint_as_float(r[4 * q + 1]) * inv,
                                         __uint_as_float(r[4 * q + 2]) * inv, __uint_as_float(r[4 * q + 3]) * inv)
                           : make_float4(qnan, qnan, qnan, qnan);
            if constexpr (!BF16) {
                // fp32 operands (d_v = 64): the output tile goes through the Vt^T rows of L
                // (free until the next item's remainders) and leaves by TMA stores, in
                // four boxes of 64 rows x 32 columns (box a: rows 64 (a / 2), columns 32 (a % 2))
                unsigned char *ob = tl + ((i >> 6) * 2 + (g >> 1)) * AS + PART + (i & 63) * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<float4 *>(ob + (((4 * (g & 1) + q) ^ (i & 7)) << 4)) = o4[q];
            } else if (i < nr) {
                float4 *dst = reinterpret_cast<float4 *>(out + (rowbase + i) * (long long)DV + c);
#pragma unroll
                for (int q = 0; q < 4; ++q) dst[q] = o4[q];
            }
        }
        if constexpr (!BF16) fence_proxy_async();   // the staged tile is read by the TMA store
        fence_before_sync();
        ok = __syncthreads_and(ok) != 0;   // every thread leaves the loop together
        fence_after_sync();
        if constexpr (!BF16) {
            if (tid == 0) {
                for (int a = 0; a < 4; ++a)
                    tma_store_3d(&maps.o, (a & 1) * 32, c0 + (a >> 1) * 64, (int)bh,
                                 smem_addr(tl + a * AS + PART));
                bulk_commit();
            }
        }
    }
    if (!BF16 && tid == 0) bulk_wait_all();
    // after a failed wait: let the copies still in flight land before the shared memory is released
    if (tid == 0) {
        if (pend_g) (void)mbar_wait(BAR_G, ph_g);
        if (pend_s) (void)mbar_wait(BAR_S, ph_s);
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
    bool ok = make_tma_2d(&maps.gq, gq, BF16, rows, kK, kC) && make_tma_2d(&maps.gk, gk, BF16, rows, kK, kC);
    if (!BF16)
        ok = ok && make_tma_2d(&maps.s, states, false,
                               (unsigned long long)dm.BH() * (CAUSAL ? dm.nblk() : 1) * (DV + 1), kK, DV) &&
             make_tma_3d(&maps.o, out, false, DV, dm.N, dm.BH(), 64);
    else
        maps.s = maps.o = maps.gq;
    if (!ok) return cudaErrorInvalidValue;
    const long long items = dm.BH() * (long long)dm.nblk();
    const int grid = (int)(items < sm_count() ? items : sm_count());
    k_chunk_out_tc<BF16, DV, CAUSAL><<<grid, kOutThreads, smem, st>>>(maps, dm.N, dm.nblk(), items, dm.eps, v,
                                                                       dm.v_bf16, states, out);
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
