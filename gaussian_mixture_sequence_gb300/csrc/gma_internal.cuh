// Internal declarations shared by the translation units of libgma.
//
// Data layout in device memory (all row-major):
//   routing rows     x[bh][n][d_route]      (fp32 or bf16)
//   values           v[bh][n][d_v]          (fp32 or bf16)
//   responsibilities g[bh][n][KP]           (workspace; fp32, bf16 or split, KP = K rounded up
//                                            to 8, the padding columns hold zeros; split = two
//                                            bf16 planes, hi then lo, see GLayout)
//   memory state     s[bh][K*d_v + K]       (Vt as K rows of d_v, then Z)
//   packed params    prm[h][k][d_route/2]   float4 {s_d, s_d+1, -mu_d s_d, -mu_d+1 s_d+1},
//                                            s = 1/sigma;  cst[h][k] = log pi_k - 1/2 sum_d log sigma^2
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/gma.h"

namespace gma {

constexpr int kThreads = 256;     // threads per CTA of every generic kernel
constexpr int kBlockRows = 256;   // rows per block of the block-state / causal-output kernels

struct Dims {
    int B, H, N, D, DV, K, KP, C;
    int KG;    // row length of the responsibilities in the workspace: KP, or on the tensor-core
               // path the components padded to whole groups of 128 (tc_kpad)
    int blk;   // rows per block of the memory scan (kBlockRows, or C on the tensor-core path)
    float eps;
    bool x_bf16, v_bf16, g_bf16;
    long long BH() const { return (long long)B * H; }
    long long state_size() const { return (long long)K * DV + K; }
    int nblk() const { return (N + blk - 1) / blk; }
};

__host__ __device__ constexpr inline long long round_up(long long a, long long b) { return (a + b - 1) / b * b; }

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }

// Element load from an fp32 or bf16 array (uniform runtime switch).
__device__ __forceinline__ float load_elem(const void *base, long long i, bool bf16)
{
    return bf16 ? bf16_bits_to_f32(static_cast<const uint16_t *>(base)[i])
                : static_cast<const float *>(base)[i];
}

// Four consecutive elements starting at i (i % 4 == 0, base 16-byte aligned).
__device__ __forceinline__ float4 load4(const void *base, long long i, bool bf16)
{
    if (bf16) {
        uint2 u = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(base) + i);
        return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                           __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
    }
    return *reinterpret_cast<const float4 *>(static_cast<const float *>(base) + i);
}

// Storage of the responsibilities in the workspace.  GL_SPLIT is the operand
// form of the fp32 tensor-core path: two bf16 planes hi = RN_bf16(g) and
// lo = RN_bf16(g - hi) (16 significant bits, |g - hi - lo| <= 2^-17 |g|); an
// array of R rows x ld holds the hi plane, then the lo plane.
enum GLayout : int { GL_F32 = 0, GL_BF16 = 1, GL_SPLIT = 2 };

__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16 &hi, __nv_bfloat16 &lo)
{
    hi = __float2bfloat16_rn(v);
    lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

__device__ __forceinline__ void store_elem(void *base, long long i, float v, bool bf16)
{
    if (bf16)
        static_cast<__nv_bfloat16 *>(base)[i] = __float2bfloat16_rn(v);
    else
        static_cast<float *>(base)[i] = v;
}

// Element i of a responsibility array of `plane` elements per plane, in `layout`.
__device__ __forceinline__ void store_g(void *base, long long i, long long plane, float v, int layout)
{
    if (layout == GL_F32) {
        static_cast<float *>(base)[i] = v;
    } else if (layout == GL_BF16) {
        static_cast<__nv_bfloat16 *>(base)[i] = __float2bfloat16_rn(v);
    } else {
        __nv_bfloat16 hi, lo;
        split_bf16(v, hi, lo);
        static_cast<__nv_bfloat16 *>(base)[i] = hi;
        static_cast<__nv_bfloat16 *>(base)[plane + i] = lo;
    }
}

// ---- launchers (each returns the launch's cudaError_t) ----
cudaError_t launch_prep(const Dims &dm, const gma_params &p, float4 *prm, float *cst, cudaStream_t st);
// gamma: responsibilities in `layout` (GLayout), ldg columns per row.  With the bounded
// routing (img non-null and resp_pruned_applies), tiles whose rows keep many components are
// listed for launch_resp_dense under source tag `src` (0 or 1) instead of being finished here.
cudaError_t launch_resp(const Dims &dm, const float4 *prm, const float *cst, const struct PrunedImages *img,
                        const void *x, void *gamma, int ldg, int layout, cudaStream_t st, int src = 0);
cudaError_t launch_block_state(const Dims &dm, const void *gk, const void *v, float *partial,
                               cudaStream_t st);
cudaError_t launch_scan(const Dims &dm, float *partial, const float *state_in, float *total,
                        bool exclusive, cudaStream_t st, bool total_in_block_layout = false);
cudaError_t launch_chunk_out(const Dims &dm, bool causal, const void *gq, const void *gk, const void *v,
                             float *states, float *out, cudaStream_t st);
cudaError_t launch_decode(const Dims &dm, const float4 *prm, const float *cst, const void *qx,
                          const void *kx, const void *v, float *state, float *out, cudaStream_t st);


// Row-major [rows][cols] tensor map with boxes of 128 bytes x box_rows and the
// 128-byte swizzle (gma_tma.cu).  Returns false if it cannot be encoded.
bool make_tma_2d(CUtensorMap *m, const void *base, bool bf16, unsigned long long rows, unsigned long long cols,
                 unsigned box_rows);

// Rank-3 variant: [d2][d1][d0] with boxes of 128 bytes x box1 x 1; coordinates
// past d1 are zero-filled on loads and skipped on stores.
bool make_tma_3d(CUtensorMap *m, const void *base, bool bf16, unsigned long long d0, unsigned long long d1,
                 unsigned long long d2, unsigned box1);
// Number of SMs of the current device (persistent grids).
int sm_count();

// Timeout flag of the current device: one word in page-locked host memory
// mapped into the device, set by a kernel whose bounded wait expired (device
// pointer, for kernels) and read / cleared by the host (host pointer).  The
// storage for all devices is allocated by the first call of timeout_flag_dev
// (nullptr if that fails); timeout_flag_host never allocates and returns
// nullptr until then.
unsigned int *timeout_flag_dev();
volatile unsigned int *timeout_flag_host();

// Per-head images the bounded routing kernel copies into shared memory.
struct PrunedImages {
    unsigned char *w;   // [H][32768 B]: bf16 bound matrix, 128-byte-swizzled K-major
    unsigned char *w3;  // [H][3][32768 B]: the log-joint matrix as three bf16 planes (hi, mid, lo)
                        // in the operand order of the dense tensor-core pass
    float4 *p;          // [H][128][33]: packed exact parameters, rows padded by one word
    float *c;           // [H][4][128]: c_k, c'_k, A_k, M_k
    float4 *p2;         // [H][128][32]: the packed exact parameters for the dense kernel, feature
                        // pair 4 e + j of a component at position 8 j + e (e = feature eighth)
    unsigned int *ctl;  // [2][H]: tiles of each head listed for the dense tensor-core pass, then
                        // those it leaves to the exact dense pass (both zeroed by k_prep_all)
    int2 *list;         // [H][cap]: (slice | source tag << 30, tile) of the tiles the routing left
    int2 *list2;        // [H][cap]: the same for the tiles the tensor-core pass leaves
    long long cap;      // list entries per head (the tiles of both routings of a head)
    unsigned int *zq;   // [BH][tiles] or null: 1 where the routing of Q (split layout) left the lo
                        // plane of a tile of 128 rows unwritten because every row kept its argmax
                        // alone (posterior 1: the plane is zero), else 0
};
constexpr size_t kPrunedWBytes = 32768, kPrunedW3Bytes = 3 * kPrunedWBytes, kPrunedPBytes = 128 * 33 * 16,
                 kPrunedCBytes = 4 * 128 * 4, kPrunedP2Bytes = 128 * 32 * 16;
// Routing tiles of 128 rows of a call with BH slices of N rows.
inline long long routing_tiles(long long BH, int N) { return BH * ((N + 127) / 128); }

// Responsibilities for K = 128, d_route = 64 with a tensor-core bound (gma_resp_tc.cu).
bool resp_pruned_applies(const Dims &dm);
// The per-head parameters (as launch_prep writes them) and the routing images in one
// kernel, for the shapes resp_pruned_applies accepts.
cudaError_t launch_prep_all(const Dims &dm, const gma_params &p, float4 *prm, float *cst, const PrunedImages &img,
                            cudaStream_t st);
cudaError_t launch_resp_pruned(const Dims &dm, const PrunedImages &img, const void *x, void *gamma, int ldg,
                               int layout, cudaStream_t st, int src = 0);
// The dense pass over the tiles the bounded routings listed: source 0 is (d0, x0, g0),
// source 1 (d1, x1, g1) (x1 may be null when only one routing ran).  The tensor-core pass
// takes every listed tile and leaves those with rows of large magnitude to the exact
// CUDA-core pass; both are launched as programmatic dependents of the preceding launch,
// and k_prep_all empties both lists at the start of every call that routes with the bound.
cudaError_t launch_resp_dense(const Dims &d0, const void *x0, void *g0, const Dims &d1, const void *x1, void *g1,
                              const PrunedImages &img, int layout, cudaStream_t st);

// Responsibilities on the tensor cores for 17 <= K <= 256 (K = 128 excepted: the bounded
// routing above takes it) and d_route = 64 (gma_resp_gtc.cu): per-head images (the three
// bf16 planes of the log-joint matrix, c', the head's maxima) built from k_prep's
// parameters into PrunedImages::w3, then every tile of a routing.
bool resp_gtc_applies(const Dims &dm);
size_t gtc_image_bytes(const Dims &dm);   // workspace for the images (0 where it does not apply)
bool resp_gtc_output_ok(const Dims &dm, int ldg, int layout);
cudaError_t launch_prep_gtc(const Dims &dm, const float4 *prm, const float *cst, unsigned char *img, cudaStream_t st);
cudaError_t launch_resp_gtc(const Dims &dm, const unsigned char *img, const float4 *prm, const float *cst,
                            const void *x, void *gamma, int ldg, int layout, cudaStream_t st);

// Tensor-core path of the causal and bidirectional forms (chunk 128; see gma_causal_tc.cu):
// K <= 128 (zero-padded to 128) or a multiple of 128 up to 512, d_v = 64, or d_v = 128 with
// bf16 products.
bool tc_path_eligible(int K, int DV, bool g_bf16);
bool tc_path_applies(const Dims &dm);
// Components of the tensor-core path's operands: K padded to 128 below 128, else K.
inline int tc_kpad(int K) { return K < 128 ? 128 : K; }
// fp32 words of one block of the carried memory in operand form (hi and lo planes of
// d_v rows of tc_kpad(K), then the Z rows).
inline long long tc_mem_words(const Dims &dm) { return (long long)(dm.DV + 1) * tc_kpad(dm.K); }
// Tensor-core path: gq / gk in GL_SPLIT (fp32 products) or GL_BF16 form; the
// carried memory in operand form (k_scan_split), one block per chunk (causal)
// or per slice (bidirectional total).
cudaError_t launch_chunk_state_tc(const Dims &dm, const void *gk, const void *v, float *partial, cudaStream_t st);
cudaError_t launch_scan_split(const Dims &dm, const float *partial, const float *state_in, unsigned char *mem,
                              unsigned char *total, float *state_out, cudaStream_t st);
// zq: the routing of Q's zero-lo-plane flags per (slice, chunk) (PrunedImages::zq), or null.
cudaError_t launch_chunk_out_tc(const Dims &dm, bool causal, const void *gq, const void *gk, const void *v,
                                const unsigned char *mem, float *out, cudaStream_t st,
                                const unsigned int *zq = nullptr);
// Responsibility diagnostics (gma_stats.cu): blocks of rows per slice of the partial
// pass, and the two launches (partial sums per block, then per head in fixed order).
int usage_blocks(const Dims &dm);
cudaError_t launch_usage(const Dims &dm, const float *gamma, int ldg, float *pu, int *pc, int *assign, float *usage,
                         long long *counts, float *entropy, cudaStream_t st);

// Gradients, CUDA-core path (gma_bwd.cu): Dims with C = 64 and blocks of kBlockRows rows,
// responsibilities fp32 [BH][N][KP].
size_t bwd_u_pitch(const Dims &dm);   // row pitch (floats) of u = dL/d[numerator | denominator]
cudaError_t launch_bwd_q(const Dims &dm, bool causal, const float *gq, const float *gk, const void *v,
                         const float *dout, float *states, float *u, float *dgq, cudaStream_t st);
cudaError_t launch_bwd_kv(const Dims &dm, bool causal, const float *gq, const float *gk, const void *v,
                          const float *u, float *mem, float *rtot, float *dgk, float *dv, cudaStream_t st);
cudaError_t launch_bwd_route(const Dims &dm, const void *x, const float4 *prm, const float *gamma, float *dgamma,
                             float *dx, float *pmu, float *pvar, float *plp, cudaStream_t st);
cudaError_t launch_bwd_final(const Dims &dm, const gma_params &p, const float *pmu, const float *pvar,
                             const float *plp, float *dmu, float *dvar, float *dlogit, cudaStream_t st);

// One kernel whose single bounded wait (limit_cycles SM cycles) expires and is reported
// through the timeout flag like the waits of the kernels above.
cudaError_t launch_expire_wait(long long limit_cycles, cudaStream_t st);

// Sets the dynamic shared-memory limit of a kernel on the current device, once
// per device (the attribute belongs to the kernel's module in that device's
// context).  `done` is the call site's record of the devices already set.
template <typename Kern>
inline cudaError_t allow_smem(Kern k, size_t bytes, std::atomic<unsigned long long> &done)
{
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_relaxed);
    return e;
}

} // namespace gma
