// Tensor-core (tcgen05 / TMEM) path of the causal form for K = 128.
//
// The causal variant of the GMA explainer ("변형 및 학습": prefix sums so that
// O_i depends on j <= i only) is evaluated in the chunkwise-parallel form of
// the linear-attention page ("선형 어텐션 원리 정리", "쉽게 이해하기"): chunks of
// C = 128 tokens, dense products inside a chunk, and a carried memory
// [Vt | Z] between chunks.  Two kernels, one CTA (4 warps) per chunk:
//
//   k_chunk_state_tc : L_c = Gamma_K,c^T [V_c | 1]            (chunk contribution)
//   (k_scan, generic) : S_{c-1} = state_in + sum_{c' < c} L_c'   (carried memory)
//   k_chunk_out_tc   : [P | U] = Gamma_Q,c [Gamma_K,c^T | Vt_{c-1}]
//                      P_m = P with j > i zeroed;   U += P_m V_c
//                      O_i = U_i / (sum_j P_m[i][j] + Gamma_Q,i . Z_{c-1} + eps)
//
// Every contraction is one tcgen05.mma sequence with M = 128 and the fp32
// accumulator in TMEM.  The A operand (Gamma rows, or P_m) is written to TMEM by
// the thread that owns the row; B operands sit in shared memory in the K-major
// 128-byte-swizzled layout.  GEMM operand precision:
//   BF16 = false: each fp32 operand is split into a tf32 "hi" part and an
//                 exact remainder "lo"; a*b ~ hi*hi + hi*lo + lo*hi (three MMA
//                 passes, relative error ~1e-6), the fp32-operand path;
//   BF16 = true : operands rounded to bf16, one pass, fp32 accumulation.
// The normaliser Z and the row sums of P_m are accumulated on CUDA cores.
#include "gma_internal.cuh"
#include "gma_tc.cuh"

namespace gma {
namespace {

using namespace tc;

constexpr int kC = 128;       // chunk rows (= MMA M)
constexpr int kK = 128;       // components handled by this path
constexpr int kTCThreads = 128;

template <bool BF16>
struct Elem {
    static constexpr int E = BF16 ? 2 : 4;                 // bytes per operand element
    static constexpr int PASSES = BF16 ? 1 : 3;
    static constexpr uint32_t FMT = BF16 ? kFmtBF16 : kFmtTF32;
    static constexpr int COLS_PER_KSTEP = 8;               // TMEM columns per 32-byte K step
    static constexpr int ACOLS = BF16 ? kK / 2 : kK;        // TMEM columns of a 128-wide A row
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

// Writes a full 128-wide A row held in 32-value pieces via a callback get(j0, float[32]).
// Returns the sum of the (rounded, for bf16) values when `want_sum`.
template <bool BF16, typename Get>
__device__ __forceinline__ float put_a_row(uint32_t tbase, uint32_t lane0, uint32_t col_hi, uint32_t col_lo,
                                           Get get)
{
    float sum = 0.f;
#pragma unroll 1
    for (int j0 = 0; j0 < kK; j0 += 32) {
        float x[32];
        get(j0, x);
        if constexpr (BF16) {
            uint32_t p[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                p[j] = pack_bf16(x[2 * j], x[2 * j + 1]);
                sum += bf16r(x[2 * j]) + bf16r(x[2 * j + 1]);
            }
            tmem_st16(tmem_at(tbase, lane0, col_hi + j0 / 2), p);
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float v = x[16 * h + j];
                    const float hv = tf32_hi(v);
                    hi[j] = __float_as_uint(hv);
                    lo[j] = __float_as_uint(v - hv);
                    sum += v;
                }
                tmem_st16(tmem_at(tbase, lane0, col_hi + j0 + 16 * h), hi);
                tmem_st16(tmem_at(tbase, lane0, col_lo + j0 + 16 * h), lo);
            }
        }
    }
    return sum;
}

// Issues D (+)= A * B^T over a 128-deep contraction with A in TMEM and B a
// K-major SW128 tile of `nrows` rows (hi/lo images), PASSES passes.
template <bool BF16>
__device__ __forceinline__ void mma_tb(uint32_t d_tmem, uint32_t a_hi, uint32_t a_lo, unsigned char *b_hi,
                                       unsigned char *b_lo, uint32_t nrows, bool accumulate)
{
    using El = Elem<BF16>;
    const uint32_t id = idesc(128, nrows, El::FMT);
    bool acc = accumulate;
#pragma unroll 1
    for (int p = 0; p < El::PASSES; ++p) {
        const uint32_t a = (p == 2) ? a_lo : a_hi;
        unsigned char *b = (p == 1) ? b_lo : b_hi;
        const int ksteps = kK * El::E / 32;
#pragma unroll 1
        for (int kk = 0; kk < ksteps; ++kk) {
            const uint32_t kb = kk * 32;
            const uint32_t boff = (kb >> 7) * (nrows * 128) + (kb & 127);
            mma_ts(!BF16, d_tmem, a + kk * El::COLS_PER_KSTEP, sdesc_sw128(smem_addr(b + boff)), id, acc ? 1u : 0u);
            acc = true;
        }
    }
}

// Bytes of a K-major tile of `rows` x 128 elements.
template <bool BF16>
constexpr uint32_t tile_bytes(uint32_t rows) { return rows * kK * Elem<BF16>::E; }

// ------------------------------------------------------------------------
// L_c = Gamma_K,c^T [V_c | 1]: M = components, N = d_v, contraction over the
// chunk's tokens.  A = Gamma_K^T in TMEM (thread k owns component k's row of
// 128 token values), B = V^T in shared memory.
template <bool BF16, int DV>
struct StateSmem {
    static constexpr uint32_t VT = tile_bytes<BF16>(DV);
    static constexpr size_t bytes = 1024 + 2 * (size_t)VT + 64;
};

template <bool BF16, int DV>
__global__ void __launch_bounds__(kTCThreads, 1)
    k_chunk_state_tc(int N, const void *__restrict__ gk, const void *__restrict__ v, bool v_bf16,
                     float *__restrict__ partial, int nblk)
{
    using El = Elem<BF16>;
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *vt_hi = sm, *vt_lo = sm + StateSmem<BF16, DV>::VT;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + 2 * StateSmem<BF16, DV>::VT);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 1);

    const int tid = threadIdx.x, warp = tid >> 5;
    const long long bh = blockIdx.y;
    const int c0 = blockIdx.x * kC;
    const int nr = min(kC, N - c0);
    constexpr uint32_t A_HI = 0, A_LO = 128, D_COL = 256;

    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(smem_addr(bar), 1);
        mbar_init_fence();
    }
    // B = V^T: element (c, j) of a DV x 128 tile; thread j writes token j's values.
    {
        const int j = tid;
        const long long base = (bh * N + c0 + j) * (long long)DV;
#pragma unroll 4
        for (int c = 0; c < DV; ++c) {
            const float x = j < nr ? load_elem(v, base + c, v_bf16) : 0.f;
            put<BF16>(vt_hi, vt_lo, sw128_offset(c, j, DV, El::E), x);
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *tslot;
    const uint32_t lane0 = 32 * warp;

    // A = Gamma_K^T: thread k loads column k of the chunk's Gamma_K (coalesced across k).
    const int k = tid;
    const void *g = gk;
    float z = 0.f;
    {
        auto get = [&](int j0, float (&x)[32]) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int r = j0 + j;
                x[j] = r < nr ? load_elem(g, (bh * N + c0 + r) * (long long)kK + k, BF16) : 0.f;
            }
        };
        float zs = put_a_row<BF16>(tbase, lane0, A_HI, A_LO, get);
        z = zs;
    }
    tmem_wait_st();
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
        mma_tb<BF16>(tbase + D_COL, tbase + A_HI, tbase + A_LO, vt_hi, vt_lo, DV, false);
        mma_commit(smem_addr(bar));
    }
    __syncwarp();
    const bool ok = mbar_wait(smem_addr(bar), 0);
    fence_after_sync();
    const long long SZ = (long long)kK * DV + kK;
    float *o = partial + (bh * nblk + blockIdx.x) * SZ;
#pragma unroll 1
    for (int c = 0; c < DV; c += 16) {
        uint32_t r[16];
        tmem_ld16(tmem_at(tbase, lane0, D_COL + c), r);
        tmem_wait_ld();
        float4 *dst = reinterpret_cast<float4 *>(o + (long long)k * DV + c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float4 t = make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                   __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
            if (!ok) t = make_float4(__int_as_float(0x7fc00000), 0.f, 0.f, 0.f);
            dst[q] = t;
        }
    }
    o[(long long)kK * DV + k] = ok ? z : __int_as_float(0x7fc00000);
    fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------------------
template <bool BF16, int DV>
struct OutSmem {
    static constexpr uint32_t GK = tile_bytes<BF16>(kC);   // Gamma_K chunk, 128 x 128
    static constexpr uint32_t VT = tile_bytes<BF16>(DV);   // V^T, DV x 128
    static constexpr uint32_t ST = tile_bytes<BF16>(DV);   // Vt^T (memory), DV x 128
    static constexpr uint32_t X = GK > VT ? GK : VT;       // region reused: Gamma_K, then V^T
    static constexpr size_t bytes = 1024 + 2 * (size_t)X + 2 * (size_t)ST + kK * 4 + 64;
};

template <bool BF16, int DV>
__global__ void __launch_bounds__(kTCThreads, 1)
    k_chunk_out_tc(int N, float eps, const void *__restrict__ gq, const void *__restrict__ gk,
                   const void *__restrict__ v, bool v_bf16, const float *__restrict__ states, int nblk,
                   float *__restrict__ out)
{
    using El = Elem<BF16>;
    using Sm = OutSmem<BF16, DV>;
    extern __shared__ unsigned char sm_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    unsigned char *x_hi = sm, *x_lo = sm + Sm::X;                  // Gamma_K, later V^T
    unsigned char *s_hi = sm + 2 * Sm::X, *s_lo = s_hi + Sm::ST;   // memory Vt^T
    float *z_s = reinterpret_cast<float *>(s_lo + Sm::ST);         // Z of the carried memory
    uint64_t *bar = reinterpret_cast<uint64_t *>(z_s + kK);        // [2]
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 2);

    const int tid = threadIdx.x, warp = tid >> 5;
    const long long bh = blockIdx.y;
    const int c0 = blockIdx.x * kC;
    const int nr = min(kC, N - c0);
    const uint32_t lane0 = 32 * warp;
    // TMEM columns: A operand (Gamma_Q, later P_m) hi/lo, P accumulator, U accumulator.
    constexpr uint32_t A_HI = 0, A_LO = 128, D_P = 256, D_U = 384;

    if (warp == 0) {
        tmem_alloc(smem_addr(tslot), 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(smem_addr(bar), 1);
        mbar_init(smem_addr(bar + 1), 1);
        mbar_init_fence();
    }
    const long long SZ = (long long)kK * DV + kK;
    const float *st = states + (bh * nblk + blockIdx.x) * SZ;
    // carried memory: B = Vt^T (element (c, k)), thread k reads row k of Vt; Z to shared memory
    {
        const int k = tid;
        const float4 *src = reinterpret_cast<const float4 *>(st + (long long)k * DV);
#pragma unroll 4
        for (int c4 = 0; c4 < DV / 4; ++c4) {
            const float4 t = src[c4];
            put<BF16>(s_hi, s_lo, sw128_offset(4 * c4 + 0, k, DV, El::E), t.x);
            put<BF16>(s_hi, s_lo, sw128_offset(4 * c4 + 1, k, DV, El::E), t.y);
            put<BF16>(s_hi, s_lo, sw128_offset(4 * c4 + 2, k, DV, El::E), t.z);
            put<BF16>(s_hi, s_lo, sw128_offset(4 * c4 + 3, k, DV, El::E), t.w);
        }
        const float zk = st[(long long)kK * DV + k];
        z_s[k] = BF16 ? bf16r(zk) : zk;
    }
    // Gamma_K chunk as B (element (j, k)): thread j copies its row.
    {
        const int j = tid;
        if constexpr (BF16) {
            const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(gk) +
                                                               (bh * N + c0 + j) * (long long)kK);
#pragma unroll 4
            for (int q = 0; q < kK / 8; ++q) {
                const uint4 t = j < nr ? src[q] : make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(x_hi + sw128_offset(j, 8 * q, kC, 2)) = t;
            }
        } else {
            const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(gk) +
                                                                 (bh * N + c0 + j) * (long long)kK);
#pragma unroll 4
            for (int q = 0; q < kK / 4; ++q) {
                const float4 t = j < nr ? src[q] : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 h = make_float4(tf32_hi(t.x), tf32_hi(t.y), tf32_hi(t.z), tf32_hi(t.w));
                const float4 l = make_float4(t.x - h.x, t.y - h.y, t.z - h.z, t.w - h.w);
                const uint32_t off = sw128_offset(j, 4 * q, kC, 4);
                *reinterpret_cast<float4 *>(x_hi + off) = h;
                *reinterpret_cast<float4 *>(x_lo + off) = l;
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tbase = *tslot;

    // A = Gamma_Q chunk (thread i owns row i), and Gamma_Q,i . Z
    const int i = tid;
    float qz = 0.f;
    {
        auto get = [&](int j0, float (&x)[32]) {
            if constexpr (BF16) {
                const uint4 *src = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(gq) +
                                                                   (bh * N + c0 + i) * (long long)kK + j0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint4 t = i < nr ? src[q] : make_uint4(0, 0, 0, 0);
                    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        x[8 * q + 2 * e] = __uint_as_float(w[e] << 16);
                        x[8 * q + 2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
                    }
                }
            } else {
                const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(gq) +
                                                                     (bh * N + c0 + i) * (long long)kK + j0);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 t = i < nr ? src[q] : make_float4(0.f, 0.f, 0.f, 0.f);
                    x[4 * q] = t.x; x[4 * q + 1] = t.y; x[4 * q + 2] = t.z; x[4 * q + 3] = t.w;
                }
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) qz = fmaf(x[j], z_s[j0 + j], qz);
        };
        put_a_row<BF16>(tbase, lane0, A_HI, A_LO, get);
    }
    tmem_wait_st();
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
        mma_tb<BF16>(tbase + D_P, tbase + A_HI, tbase + A_LO, x_hi, x_lo, kC, false);   // P = Gq Gk^T
        mma_tb<BF16>(tbase + D_U, tbase + A_HI, tbase + A_LO, s_hi, s_lo, DV, false);   // U = Gq Vt
        mma_commit(smem_addr(bar));
    }
    __syncwarp();
    bool ok = mbar_wait(smem_addr(bar), 0);
    fence_after_sync();

    // P_m = P with j > i zeroed; it replaces Gamma_Q as the A operand.  Row sums on CUDA cores.
    float psum = 0.f;
    {
        auto get = [&](int j0, float (&x)[32]) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[16];
                tmem_ld16(tmem_at(tbase, lane0, D_P + j0 + 16 * h), r);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int jj = j0 + 16 * h + j;
                    x[16 * h + j] = jj <= i ? __uint_as_float(r[j]) : 0.f;
                }
            }
        };
        psum = put_a_row<BF16>(tbase, lane0, A_HI, A_LO, get);
    }
    // B = V^T (element (c, j)) into the region that held Gamma_K (its MMAs are complete).
    {
        const int j = tid;
        const long long base = (bh * N + c0 + j) * (long long)DV;
#pragma unroll 4
        for (int c = 0; c < DV; ++c) {
            const float x = j < nr ? load_elem(v, base + c, v_bf16) : 0.f;
            put<BF16>(x_hi, x_lo, sw128_offset(c, j, DV, El::E), x);
        }
    }
    tmem_wait_st();
    fence_proxy_async();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
        mma_tb<BF16>(tbase + D_U, tbase + A_HI, tbase + A_LO, x_hi, x_lo, DV, true);   // U += P_m V
        mma_commit(smem_addr(bar + 1));
    }
    __syncwarp();
    ok = mbar_wait(smem_addr(bar + 1), 0) && ok;
    fence_after_sync();

    const float den = psum + qz + eps;
    const float inv_nan = __int_as_float(0x7fc00000);
#pragma unroll 1
    for (int c = 0; c < DV; c += 16) {
        uint32_t r[16];
        tmem_ld16(tmem_at(tbase, lane0, D_U + c), r);
        tmem_wait_ld();
        if (i < nr) {
            float4 *dst = reinterpret_cast<float4 *>(out + (bh * N + c0 + i) * (long long)DV + c);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                dst[q] = ok ? make_float4(__uint_as_float(r[4 * q]) / den, __uint_as_float(r[4 * q + 1]) / den,
                                          __uint_as_float(r[4 * q + 2]) / den, __uint_as_float(r[4 * q + 3]) / den)
                            : make_float4(inv_nan, inv_nan, inv_nan, inv_nan);
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

template <bool BF16, int DV>
cudaError_t out_tc(const Dims &dm, const void *gq, const void *gk, const void *v, const float *states, float *out,
                   cudaStream_t st)
{
    constexpr size_t smem = OutSmem<BF16, DV>::bytes;
    static cudaError_t attr = allow_smem(k_chunk_out_tc<BF16, DV>, smem);
    if (attr != cudaSuccess) return attr;
    dim3 grid(dm.nblk(), (unsigned)dm.BH());
    k_chunk_out_tc<BF16, DV><<<grid, kTCThreads, smem, st>>>(dm.N, dm.eps, gq, gk, v, dm.v_bf16, states, dm.nblk(),
                                                             out);
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

cudaError_t launch_chunk_out_tc(const Dims &dm, const void *gq, const void *gk, const void *v, const float *states,
                                float *out, cudaStream_t st)
{
    if (dm.g_bf16) {
        if (dm.DV == 64) return out_tc<true, 64>(dm, gq, gk, v, states, out, st);
        if (dm.DV == 128) return out_tc<true, 128>(dm, gq, gk, v, states, out, st);
    } else if (dm.DV == 64) {
        return out_tc<false, 64>(dm, gq, gk, v, states, out, st);
    }
    return cudaErrorInvalidValue;
}

} // namespace gma
