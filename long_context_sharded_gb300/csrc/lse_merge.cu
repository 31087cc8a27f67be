// lse_merge.cu -- exact log-sum-exp combine of per-step partial results.
//
// The shifted schedule leaves every query row with one partial (O_j, LSE_j)
// per step; combining them gives plain attention, as in the RingAttention-
// style schedules that Mercury reproduces (Mercury-SOSP25 paper notes,
// one-line summary and 实验与结果).  Per row:
//     L = ln sum_j exp(LSE_j),   O = sum_j exp(LSE_j - L) O_j.
//
// HBM-bound: every partial row is read once (R * (4d + 4) bytes per row) and
// the result written once.  A group of TPR lanes owns one row; each lane owns
// VEC consecutive float4 of it, so a part's row is one coalesced
// TPR*VEC*16-byte read.  The LSE values of a row are spread over the group's
// lanes, reduced with warp shuffles, and the weights broadcast back by
// shuffle.  Parts with LSE = -inf have weight 0 and are not read.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>

#include "internal.h"
#include "ptx.cuh"

namespace mercury {

// Device error word of this file's kernel (a module of its own): kErrBounds
// = the checked build skipped an out-of-range access; the first site.
__device__ unsigned int g_merge_err_word = 0;
__device__ unsigned int g_merge_err_site = 0;

namespace {

__device__ __forceinline__ void mrecord_bounds(uint32_t site)
{
    atomicOr(&g_merge_err_word, kErrBounds);
    atomicCAS(&g_merge_err_site, 0u, site);
}

constexpr int kMergeThreads = 256;

template <int TPR, int VEC>
__global__ void __launch_bounds__(kMergeThreads)
lse_merge_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part, int n_parts,
                 long long rows, int d, float *__restrict__ out, float *__restrict__ lse, int out_bf16)
{
    constexpr int kRowsPerWarp = 32 / TPR;
    const int lane = threadIdx.x % 32;
    const int g = lane % TPR;                 // lane inside the row group
    const int grp_base = lane - g;            // first lane of the row group
    const long long warp_id = ((long long)blockIdx.x * kMergeThreads + threadIdx.x) / 32;
    const long long row = warp_id * kRowsPerWarp + lane / TPR;
    const bool active = row < rows;
    const unsigned full = 0xffffffffu;
    const int nvec = d / 4;                   // float4 per row

    // 1. L = M + ln sum_j exp(l_j - M), lanes of the group striding over parts.
    float M = -INFINITY;
    if (active)
        for (int j = g; j < n_parts; j += TPR)
            M = fmaxf(M, lse_part[(long long)j * rows + row]);
#pragma unroll
    for (int off = TPR / 2; off > 0; off /= 2)
        M = fmaxf(M, __shfl_xor_sync(full, M, off));
    float Z = 0.f;
    if (active && M != -INFINITY)
        for (int j = g; j < n_parts; j += TPR)
            Z += expf(lse_part[(long long)j * rows + row] - M);
#pragma unroll
    for (int off = TPR / 2; off > 0; off /= 2)
        Z += __shfl_xor_sync(full, Z, off);
    const bool empty = (M == -INFINITY);
    const float L = empty ? -INFINITY : M + logf(Z);

    // 2. O = sum_j exp(l_j - L) O_j.
    float4 acc[VEC];
#pragma unroll
    for (int v = 0; v < VEC; ++v)
        acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    const long long part_stride = rows * (long long)d;
    const float4 *src = reinterpret_cast<const float4 *>(o_part + row * (long long)d);
    // checked build: every part's row read and the output row written lie
    // inside their arrays (element offsets of the row's first and last float4)
    bool row_ok = active;
    if (kChecked && active) {
        const long long first = row * (long long)d, last_read = (long long)(n_parts - 1) * part_stride + first + d;
        if (row < 0 || first + d > rows * (long long)d || last_read > (long long)n_parts * part_stride ||
            (d % 4) != 0) {
            mrecord_bounds(0x701);
            row_ok = false;
        }
    }
    for (int j0 = 0; j0 < n_parts; j0 += TPR) {
        // lane g of the group holds the weight of part j0 + g
        float w_mine = 0.f;
        if (active && !empty && j0 + g < n_parts)
            w_mine = expf(lse_part[(long long)(j0 + g) * rows + row] - L);
        const int cnt = min(TPR, n_parts - j0);
#pragma unroll 4
        for (int jj = 0; jj < cnt; ++jj) {
            const float w = __shfl_sync(full, w_mine, grp_base + jj);
            if (row_ok && w != 0.f) {
                const float4 *s = src + (long long)(j0 + jj) * (part_stride / 4);
#pragma unroll
                for (int v = 0; v < VEC; ++v) {
                    const int c = g + v * TPR;
                    if (c < nvec) {
                        const float4 x = __ldcs(s + c);  // streamed once: evict-first
                        acc[v].x = fmaf(w, x.x, acc[v].x);
                        acc[v].y = fmaf(w, x.y, acc[v].y);
                        acc[v].z = fmaf(w, x.z, acc[v].z);
                        acc[v].w = fmaf(w, x.w, acc[v].w);
                    }
                }
            }
        }
    }
    if (row_ok && out_bf16) {
        // out holds bf16: four elements (8 bytes) per float4 of the row
        uint2 *dst = reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(out) + row * (long long)d);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const int c = g + v * TPR;
            if (c < nvec) {
                __nv_bfloat162 lo = __floats2bfloat162_rn(acc[v].x, acc[v].y);
                __nv_bfloat162 hi = __floats2bfloat162_rn(acc[v].z, acc[v].w);
                dst[c] = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
            }
        }
    } else if (row_ok) {
        float4 *dst = reinterpret_cast<float4 *>(out + row * (long long)d);
#pragma unroll
        for (int v = 0; v < VEC; ++v) {
            const int c = g + v * TPR;
            if (c < nvec)
                dst[c] = acc[v];
        }
    }
    if (row_ok) {
        if (g == 0)
            lse[row] = L;
    }
}

template <int TPR, int VEC>
int launch(const float *o_part, const float *lse_part, int n_parts, long long rows, int d, float *out,
           float *lse, cudaStream_t stream, char *msg, size_t msg_len, int out_bf16)
{
    constexpr int kRowsPerBlock = (kMergeThreads / 32) * (32 / TPR);
    const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    if (blocks > 0x7fffffffLL) {
        snprintf(msg, msg_len, "too many rows for one merge launch (%lld)", rows);
        return MERCURY_EINVAL;
    }
    lse_merge_kernel<TPR, VEC><<<(unsigned)blocks, kMergeThreads, 0, stream>>>(o_part, lse_part, n_parts,
                                                                               rows, d, out, lse, out_bf16);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "merge kernel launch: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    return MERCURY_OK;
}

}  // namespace

int read_and_clear_merge_error(unsigned int *word, unsigned int *site, char *msg, size_t msg_len)
{
    unsigned int zero = 0, w = 0, st = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&w, g_merge_err_word, sizeof w);
    if (e == cudaSuccess)
        e = cudaMemcpyFromSymbol(&st, g_merge_err_site, sizeof st);
    if (e == cudaSuccess && (w || st)) {
        e = cudaMemcpyToSymbol(g_merge_err_word, &zero, sizeof zero);
        if (e == cudaSuccess)
            e = cudaMemcpyToSymbol(g_merge_err_site, &zero, sizeof zero);
    }
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "reading the merge error word: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    *word = w;
    *site = st;
    return MERCURY_OK;
}

int launch_lse_merge(const float *o_part, const float *lse_part, int n_parts, long long rows, int d,
                     float *out, float *lse, cudaStream_t stream, char *msg, size_t msg_len, int out_bf16)
{
    if (rows == 0)
        return MERCURY_OK;
    const int nvec = d / 4;
    if (nvec <= 4)
        return launch<4, 1>(o_part, lse_part, n_parts, rows, d, out, lse, stream, msg, msg_len, out_bf16);
    if (nvec <= 8)
        return launch<8, 1>(o_part, lse_part, n_parts, rows, d, out, lse, stream, msg, msg_len, out_bf16);
    // d = 64 and 128: half a warp per row, two float4 per lane per part (more
    // rows and more loads in flight per warp measured 3-5 % faster than a
    // whole warp per row with one float4 per lane)
    if (nvec <= 16)
        return launch<8, 2>(o_part, lse_part, n_parts, rows, d, out, lse, stream, msg, msg_len, out_bf16);
    if (nvec <= 32)
        return launch<16, 2>(o_part, lse_part, n_parts, rows, d, out, lse, stream, msg, msg_len, out_bf16);
    if (nvec <= 64)
        return launch<32, 2>(o_part, lse_part, n_parts, rows, d, out, lse, stream, msg, msg_len, out_bf16);
    return launch<32, 4>(o_part, lse_part, n_parts, rows, d, out, lse, stream, msg, msg_len, out_bf16);
}

}  // namespace mercury
