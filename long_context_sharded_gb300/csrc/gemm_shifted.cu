// gemm_shifted.cu -- the all-gather GEMM pattern of the pages under the
// shifted schedule, on sm_103a.
//
// Every rank owns a slice of A while all ranks need B; instead of first
// replicating B, a rank reads B's pieces from their owners in a
// rank-staggered order (Silicon & Systems, "The hidden cost of synchronized
// operators"; the all-gather GEMM results in "What Mercury finds that
// templates miss").  Here R virtual ranks share one GPU: rank i owns the row
// block A_i (M/R rows), B is cut into R column shards B_s (N/R columns), and
// rank i at step j computes C[block i, shard order[i][j]] = A_i B_s.  The
// result is C = A B, fp32, from bf16 inputs.
//
// Kernel: persistent, one CTA per SM walking output tiles of 256 x 256.  The
// shift fixes which shard each rank reads at each step; on one GPU the order
// in which the (rank, step) blocks run is free, since all R virtual ranks
// share one L2.  Blocks run shard-major -- for each B shard s, the R ranks
// that read it, in the order of the steps at which they do -- so a shard is
// fetched into L2 once and its R readers follow each other (step-major order
// fetched every shard and every A block again at every step).  Inside a block
// the tiles along a row of C are adjacent, so the CTAs resident together
// share the A rows too.  Warp 0: TMA producer (A tile 256 x 64 as two 128-row boxes, K-major;
// B tile 64 x 256 as four 64-column boxes, N-major) into a 3-stage ring:
// 64 KB per 1024 tensor cycles, two thirds of what 128 x 256 tiles pull from
// L2 per FLOP.  Warp 1 (one elected lane) issues tcgen05.mma kind::f16, M = 128,
// N = 256, K = 16 (128 tensor cycles per instruction, well above the issue
// cost of an MMA) into two 256-column TMEM accumulators, one per 128-row
// half.  Warps 4-7 and 8-11: epilogue of the two halves, TMEM -> fp32 global;
// the first half drains while the second half's last MMAs run.
#include <cuda.h>
#include <cuda_runtime.h>

#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "internal.h"
#include "ptx.cuh"
#include "work.h"

namespace mercury {

// Device error word of this file's kernel (a module of its own): kErrTimeout
// = a bounded wait ran out, kErrBounds = the checked build skipped an
// out-of-range access; the site of the first one recorded.
__device__ unsigned int g_gemm_err_word = 0;
__device__ unsigned int g_gemm_err_site = 0;

namespace {

constexpr int kGThreads = 384;
constexpr int kBM = 256, kBN = 256, kBK = 64;  // CTA tile (two 128-row halves)
constexpr int kMmaM = 128;                     // M of one tcgen05.mma (cta_group::1)
static_assert(kMmaM == 128, "cta_group::1 kind::f16 MMAs here are M = 128");
static_assert(kBM == 2 * kMmaM, "the CTA tile is two MMA halves");
constexpr int kStages = 3;
constexpr int kAHalf = kMmaM * kBK * 2;  // 16 KB: one 128-row half of A
constexpr int kABytes = 2 * kAHalf;      // 32 KB
constexpr int kBBytes = kBK * kBN * 2;   // 32 KB: four 64 x 64 boxes of 8 KB
constexpr int kBBox = kBK * 64 * 2;      // 8 KB
constexpr int kGOffBar = kStages * (kABytes + kBBytes);
constexpr int kGBytes = kGOffBar + 8 * (2 * kStages + 5) + 16;
constexpr uint32_t kGExitBarrier = 1;  // named barrier of all threads at exit
constexpr int kGAlloc = kGBytes + 1024;

struct GemmParams {
    int M, N, K, R;
    int Mr, Nr;        // rows per rank block, columns per shard
    int RT, CT;        // 128-row tiles per block, 256-column tiles per shard
    int KB;            // 64-wide K steps
    long long n_items;
    float *c;
    unsigned char reader[kMaxR * kMaxR];  // reader[s*R + p]: the p-th rank to read shard s (by step, then rank)
    int c_v8;          // c is 32-byte aligned (N % 8 == 0 keeps every row so)
    unsigned long long wait_ns;
};

__device__ __forceinline__ bool gwait(uint64_t *bar, uint32_t parity, unsigned long long budget,
                                      volatile uint32_t *abort, uint32_t site)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (*abort)
            return false;
        if (globaltimer_ns() - t0 > budget) {
            *abort = 1u;
            atomicOr(&g_gemm_err_word, kErrTimeout);
            atomicCAS(&g_gemm_err_site, 0u, site);
            return false;
        }
    }
}

// Bounded wait on the way out: not cut short by another role's abort (the
// operations it waits for complete on their own); a timeout is recorded.
__device__ __forceinline__ bool gdrain(uint64_t *bar, uint32_t parity, unsigned long long budget, uint32_t site)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > budget) {
            atomicOr(&g_gemm_err_word, kErrTimeout);
            atomicCAS(&g_gemm_err_site, 0u, site);
            return false;
        }
    }
    return true;
}

// Checked build: an out-of-range index found at `site`.
__device__ __forceinline__ void grecord_bounds(uint32_t site)
{
    atomicOr(&g_gemm_err_word, kErrBounds);
    atomicCAS(&g_gemm_err_site, 0u, site);
}

struct GTile {
    int m0, n0;        // first row / column of the tile
    int m_end, n_end;  // rows / columns of the tile's (rank, shard) block end here
};

// Item idx (shard-major): ct fastest, then rt, then the shard's readers in
// the order of their steps, shard s slowest.
__device__ __forceinline__ GTile decode_gtile(const GemmParams &p, long long idx)
{
    const int ct = (int)(idx % p.CT); idx /= p.CT;
    const int rt = (int)(idx % p.RT); idx /= p.RT;
    const int pos = (int)(idx % p.R); idx /= p.R;
    const int s = (int)idx;
    const int i = p.reader[s * p.R + pos];
    GTile t;
    t.m0 = i * p.Mr + rt * kBM;
    t.n0 = s * p.Nr + ct * kBN;
    t.m_end = (i + 1) * p.Mr;
    t.n_end = (s + 1) * p.Nr;
    return t;
}

__global__ void __launch_bounds__(kGThreads, 1)
gemm_shifted_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB)
{
    constexpr uint32_t kIdesc = idesc_bf16_f32(kMmaM, kBN, true);  // B is N-major
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sA = smem;
    uint8_t *sB = smem + kStages * kABytes;
    uint64_t *bars = (uint64_t *)(smem + kGOffBar);
    uint64_t *full = bars;
    uint64_t *empty = full + kStages;
    uint64_t *acc_full = empty + kStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *mma_done = acc_empty + 2;  // every MMA issued has completed (exit)
    uint32_t *tmem_slot = (uint32_t *)(mma_done + 1);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(acc_full + a, 1);
            mbar_init(acc_empty + a, 4);  // one arrive per warp of that half's epilogue
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // ----------------------------------------------------- TMA producer
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        int it = 0;
        bool ok = true;
        for (long long idx = blockIdx.x; idx < p.n_items && ok; idx += gridDim.x) {
            const GTile t = decode_gtile(p, idx);
            for (int kb = 0; kb < p.KB; ++kb, ++it) {
                const int st = it % kStages;
                if (it >= kStages &&
                    !gwait(empty + st, ((it / kStages) - 1) & 1, p.wait_ns, abort_flag, 0x401)) {
                    ok = false;
                    break;
                }
                if (kChecked) {
                    // A boxes at (k, m) and (k, m + 128): the second half may hang
                    // past M (zero fill); B boxes at (n + 64c, k)
                    bool good = tma_coords_ok(kb * kBK, t.m0, 0, p.K, p.M, 1, 0) &&
                                tma_coords_ok(kb * kBK, t.m0 + 128, 0, p.K, p.M, 1, kMmaM);
                    for (int c = 0; c < kBN / 64; ++c)
                        good = good && (t.n0 + c * 64 >= t.n_end ||
                                        tma_coords_ok(t.n0 + c * 64, kb * kBK, 0, p.N, p.K, 1, 0));
                    if (!good) {
                        grecord_bounds(0x601);
                        *abort_flag = 1u;
                        ok = false;
                        break;
                    }
                }
                mbar_arrive_expect_tx(full + st, (uint32_t)(kABytes + kBBytes));
                // A tile: [256 rows][64 k] as two boxes {64, 128} at (k, m), (k, m + 128)
                tma_load_2d(sA + st * kABytes, &tmA, full + st, kb * kBK, t.m0);
                tma_load_2d(sA + st * kABytes + kAHalf, &tmA, full + st, kb * kBK, t.m0 + 128);
                // B tile: [64 k][256 n] as four boxes {64 n, 64 k}
                for (int c = 0; c < kBN / 64; ++c)
                    tma_load_2d(sB + st * kBBytes + c * kBBox, &tmB, full + st, t.n0 + c * 64, kb * kBK);
            }
        }
        // every load issued into shared memory must land before the CTA
        // leaves (after an abort some may be in flight): the last load of a
        // stage is the newest phase of its barrier
        for (int s = 0; s < kStages; ++s)
            if (it > s) {
                const int last = it - 1 - ((it - 1 - s) % kStages);
                gdrain(full + s, (last / kStages) & 1, p.wait_ns, 0x411);
            }
    } else if (warp == 1) {
        // ----------------------------------------------------- MMA issuer
        // (the whole warp runs the loop; one elected lane issues)
        const uint32_t leader = elect_lane();  // the lane that issues
        const uint64_t da = smem_desc_sw128(smem_u32(sA), 16, 1024);
        // B N-major: 8 k-rows of 128 B per 1024-byte group; the four 64-column
        // boxes are kBBox bytes apart (leading-dimension offset)
        const uint64_t db = smem_desc_sw128(smem_u32(sB), kBBox, 1024);
        int it = 0, tile = 0;
        int released = 0;          // stage releases committed (iterations 0 .. released-1)
        int n_acc[2] = {0, 0};     // accumulator-ready commits per half
        bool ok = true;
        for (long long idx = blockIdx.x; idx < p.n_items && ok; idx += gridDim.x, ++tile) {
            for (int kb = 0; kb < p.KB && ok; ++kb, ++it) {
                const int st = it % kStages;
                if (!gwait(full + st, (it / kStages) & 1, p.wait_ns, abort_flag, 0x403)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t dbs = db + ((uint32_t)(st * kBBytes) >> 4);
                for (int h = 0; h < 2; ++h) {
                    // this half's accumulator must have been read out (previous tile)
                    if (kb == 0 && tile >= 1 &&
                        !gwait(acc_empty + h, (tile - 1) & 1, p.wait_ns, abort_flag, 0x402)) {
                        ok = false;
                        break;
                    }
                    if (kb == 0)
                        tc_fence_after();
                    const uint64_t das = da + ((uint32_t)(st * kABytes + h * kAHalf) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        umma_ss_w(tmem + h * kBN, das + (uint32_t)(kk * (32 >> 4)), dbs + (uint32_t)(kk * (2048 >> 4)),
                                kIdesc, (kb > 0 || kk > 0) ? 1u : 0u, leader);
                    if (kb == p.KB - 1) {
                        umma_commit_w(acc_full + h, leader);  // this half is final: its epilogue may start
                        ++n_acc[h];
                    }
                }
                if (ok) {
                    umma_commit_w(empty + st, leader);
                    ++released;
                }
            }
        }
        // Before the CTA leaves (and the tensor memory is freed) every MMA
        // issued must have completed and every commit's arrive have landed,
        // also after an abort.
        umma_commit_w(mma_done, leader);
        gdrain(mma_done, 0, p.wait_ns, 0x404);
        for (int m = (released > kStages ? released - kStages : 0); m < released; ++m)
            gdrain(empty + (m % kStages), (m / kStages) & 1, p.wait_ns, 0x406);
        for (int h = 0; h < 2; ++h)
            if (n_acc[h] > 0)
                gdrain(acc_full + h, (n_acc[h] - 1) & 1, p.wait_ns, 0x407);
    } else if (warp >= 4) {
        // ----------------------------------------------------- epilogue
        const int acc = (warp - 4) / 4;  // the 128-row half this warpgroup writes
        const int quarter = warp % 4;
        const int r = acc * 128 + quarter * 32 + lane;
        const uint32_t lane_field = (uint32_t)(quarter * 32) << 16;
        int tile = 0;
        bool ok = true;
        for (long long idx = blockIdx.x; idx < p.n_items && ok; idx += gridDim.x, ++tile) {
            const GTile t = decode_gtile(p, idx);
            bool got = gwait(acc_full + acc, tile & 1, p.wait_ns, abort_flag, 0x405);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int row = t.m0 + r;
            bool row_ok = row < t.m_end && row < p.M;
            const int n_lim = min(t.n_end, p.N) - t.n0;  // valid columns of this tile
            float *crow = p.c + (long long)row * p.N + t.n0;
            if (kChecked && row_ok) {
                // the row's stores cover columns [n0, n0 + min(n_lim, 256))
                const long long first = (long long)row * p.N + t.n0;
                const long long last = first + min(n_lim, kBN);
                if (row < 0 || t.n0 < 0 || n_lim < 0 || last > (long long)p.M * p.N) {
                    grecord_bounds(0x602);
                    row_ok = false;
                }
            }
#pragma unroll 1
            for (int c0 = 0; c0 < kBN; c0 += 32) {
                uint32_t v[32];
                tmem_ld_x32(tmem + lane_field + acc * kBN + c0, v);
                if (row_ok) {
                    if (c0 + 32 <= n_lim && p.c_v8) {
                        // 32 bytes per lane: half the store instructions and L1
                        // wavefronts of 16-byte stores
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            st_global_v8(crow + c0 + 8 * q, v[8 * q], v[8 * q + 1], v[8 * q + 2], v[8 * q + 3],
                                         v[8 * q + 4], v[8 * q + 5], v[8 * q + 6], v[8 * q + 7]);
                    } else if (c0 + 32 <= n_lim) {
                        float4 *dst = reinterpret_cast<float4 *>(crow + c0);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                    } else {
                        for (int q = 0; q < 32 && c0 + q < n_lim; ++q)
                            crow[c0 + q] = __uint_as_float(v[q]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(acc_empty + acc);
        }
    }
    tc_fence_before();
    named_barrier_sync(kGExitBarrier, kGThreads);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

// 2-D bf16 tensor [d1][d0] (d0 innermost), box {b0, b1}, 128-byte swizzle, zero fill.
int encode_2d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint32_t b0, uint32_t b1, char *msg,
              size_t msg_len)
{
    // looked up once (thread-safe static initialisation)
    static const EncodeFn fn = []() -> EncodeFn {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                                         cudaEnableDefault, &q);
        return (e == cudaSuccess && q == cudaDriverEntryPointSuccess) ? (EncodeFn)ptr : nullptr;
    }();
    if (!fn) {
        snprintf(msg, msg_len, "cuTensorMapEncodeTiled is not available from the driver");
        return MERCURY_ECUDA;
    }
    cuuint64_t dims[2] = {d0, d1};
    cuuint64_t strides[1] = {d0 * 2};
    cuuint32_t box[2] = {b0, b1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(msg, msg_len, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
        return MERCURY_ECUDA;
    }
    return MERCURY_OK;
}

}  // namespace

int launch_gemm_shifted(const void *a, const void *b, int M, int N, int K, int R, const int *order, float *c,
                        unsigned long long wait_ns, cudaStream_t stream, char *msg, size_t msg_len)
{
    static thread_local GemmParams p;
    memset(&p, 0, sizeof p);
    p.M = M;
    p.N = N;
    p.K = K;
    p.R = R;
    p.Mr = M / R;
    p.Nr = N / R;
    p.RT = (p.Mr + kBM - 1) / kBM;
    p.CT = (p.Nr + kBN - 1) / kBN;
    p.KB = (K + kBK - 1) / kBK;
    p.n_items = (long long)R * R * p.RT * p.CT;
    p.c = c;
    p.c_v8 = ((uintptr_t)c % 32 == 0 && N % 8 == 0) ? 1 : 0;
    p.wait_ns = wait_ns;
    // every rank reads every shard once (each row of the table is a
    // permutation); a shard's readers go by the step at which they read it,
    // ties (the unshifted order: all ranks at the same step) by rank
    for (int s = 0; s < R; ++s) {
        int n = 0;
        for (int j = 0; j < R; ++j)
            for (int i = 0; i < R; ++i)
                if (order[i * R + j] == s)
                    p.reader[s * R + n++] = (unsigned char)i;
    }
    CUtensorMap ma, mb;
    // A is loaded as two 128-row boxes per stage, B as four 64-column boxes:
    // the boxes must add up to the bytes each stage's barrier expects
    static_assert(kAHalf == kBK * kMmaM * 2 && kABytes == 2 * kAHalf, "A box");
    static_assert(kBBox == 64 * kBK * 2 && kBBytes == (kBN / 64) * kBBox, "B box");
    int rc = encode_2d(&ma, a, (uint64_t)K, (uint64_t)M, kBK, kMmaM, msg, msg_len);
    if (rc == MERCURY_OK)
        rc = encode_2d(&mb, b, (uint64_t)N, (uint64_t)K, 64, kBK, msg, msg_len);
    if (rc != MERCURY_OK)
        return rc;
    KernelInfo ki;
    rc = prepare_kernel((const void *)gemm_shifted_kernel, kGAlloc, &ki, msg, msg_len);
    if (rc != MERCURY_OK)
        return rc;
    const int sms = ki.sms;
    const long long grid = p.n_items < sms ? p.n_items : sms;
    if (grid < 1)
        return MERCURY_OK;
    gemm_shifted_kernel<<<(unsigned)grid, kGThreads, kGAlloc, stream>>>(p, ma, mb);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "GEMM kernel launch: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    return MERCURY_OK;
}

int read_and_clear_gemm_error(unsigned int *word, unsigned int *site, char *msg, size_t msg_len)
{
    unsigned int zero = 0, w = 0, st = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&w, g_gemm_err_word, sizeof w);
    if (e == cudaSuccess)
        e = cudaMemcpyFromSymbol(&st, g_gemm_err_site, sizeof st);
    if (e == cudaSuccess && (w || st)) {
        e = cudaMemcpyToSymbol(g_gemm_err_word, &zero, sizeof zero);
        if (e == cudaSuccess)
            e = cudaMemcpyToSymbol(g_gemm_err_site, &zero, sizeof zero);
    }
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "reading the GEMM error word: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    *word = w;
    *site = st;
    return MERCURY_OK;
}

}  // namespace mercury
