// api.cu -- the C ABI of libmercury_attn.so: argument validation, status
// codes and messages, the shift planner, and dispatch to the kernels.
// Declarations and the full contract are in include/mercury_attn.h.
#include <cuda_runtime.h>

#include <limits.h>
#include <atomic>
#include <map>
#include <mutex>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "internal.h"
#include "work.h"

using namespace mercury;

namespace {

thread_local char g_msg[512];

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

int ok()
{
    g_msg[0] = '\0';
    return MERCURY_OK;
}

bool aligned(const void *p, uintptr_t a)
{
    return ((uintptr_t)p % a) == 0;
}

unsigned long long wait_budget_ns()
{
    const char *e = getenv("MERCURY_WAIT_NS");
    if (e && *e) {
        char *end = nullptr;
        unsigned long long v = strtoull(e, &end, 10);
        if (end && *end == '\0' && v > 0)
            return v;
    }
    return 2000000000ull;  // 2 s
}

int fault_mode()
{
    const char *e = getenv("MERCURY_FAULT");
    if (e && strcmp(e, "drop_p_arrive") == 0)
        return 1;  // a softmax warp withholds its first P-ready arrive: the MMA issuer's wait runs out
    if (e && strcmp(e, "drop_kv_free") == 0)
        return 2;  // the first "iteration done" arrive is withheld: the TMA producer's wait runs out
    return 0;
}

bool sync_check()
{
    const char *e = getenv("MERCURY_SYNC_CHECK");
    return e && e[0] == '1';
}

// Overflow-checked product of non-negative factors; false if > 2^62.
bool mul_ok(long long &acc, long long f)
{
    if (f < 0)
        return false;
    if (f != 0 && acc > (1LL << 62) / f)
        return false;
    acc *= f;
    return true;
}

int check_shift(int R, int shift)
{
    if (R < 1 || R > kMaxR)
        return fail(MERCURY_EINVAL, "R must be in [1, %d] (got %d)", kMaxR, R);
    if (shift < 0)
        return fail(MERCURY_EINVAL, "shift must be >= 0 (got %d)", shift);
    if (shift >= 2 && R % shift != 0)
        return fail(MERCURY_EINVAL, "nested shift: inner size %d must divide R = %d", shift, R);
    return MERCURY_OK;
}

// The shape of an attention call (no pointers).
int check_attn_shape(int B, int Hq, int Hkv, int Sq, int Skv, int d, int R, int shift, int causal, int partial)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Skv < 1)
        return fail(MERCURY_EINVAL, "B, Hq, Hkv, Sq, Skv must be >= 1");
    if (Hq % Hkv != 0)
        return fail(MERCURY_EINVAL, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
    if (d != 64 && d != 128)
        return fail(MERCURY_EINVAL, "head dim must be 64 or 128 (got %d)", d);
    int rc = check_shift(R, shift);
    if (rc)
        return rc;
    if (Sq % R != 0 || Skv % R != 0)
        return fail(MERCURY_EINVAL, "R (%d) must divide Sq (%d) and Skv (%d)", R, Sq, Skv);
    if (causal && Sq > Skv)
        return fail(MERCURY_EINVAL, "causal attention needs Sq <= Skv (Sq %d, Skv %d)", Sq, Skv);
    long long nq = 1, nkv = 1;
    if (!mul_ok(nq, B) || !mul_ok(nq, Hq) || !mul_ok(nq, Sq) || !mul_ok(nq, d) ||
        (partial && !mul_ok(nq, R)) || !mul_ok(nkv, B) || !mul_ok(nkv, Hkv) || !mul_ok(nkv, Skv) ||
        !mul_ok(nkv, d))
        return fail(MERCURY_EINVAL, "tensor sizes overflow");
    if ((long long)B * Hq > INT_MAX || (long long)B * Hkv > INT_MAX)
        return fail(MERCURY_EINVAL, "B*H exceeds 2^31");
    return MERCURY_OK;
}

int check_attn_args(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq, int Skv,
                    int d, int R, int shift, int causal, const float *out, const float *lse, int partial)
{
    if (!q || !k || !v || !out || !lse)
        return fail(MERCURY_EINVAL, "null pointer argument");
    int rc = check_attn_shape(B, Hq, Hkv, Sq, Skv, d, R, shift, causal, partial);
    if (rc)
        return rc;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
        return fail(MERCURY_EALIGN, "q, k, v and the O output must be 16-byte aligned");
    if (!aligned(lse, 4))
        return fail(MERCURY_EALIGN, "the LSE output must be 4-byte aligned");
    return MERCURY_OK;
}

// Synchronise `stream` and collect the error words of every kernel module
// (bit 0: a bounded wait ran out; bit 1: the checked build skipped an
// out-of-range access).
int collect_device_errors(cudaStream_t stream)
{
    unsigned int w[3] = {0, 0, 0}, site[3] = {0, 0, 0};
    int rc = read_and_clear_device_error(stream, &w[0], &site[0], g_msg, sizeof g_msg);
    if (rc == MERCURY_OK)
        rc = read_and_clear_gemm_error(&w[1], &site[1], g_msg, sizeof g_msg);
    if (rc == MERCURY_OK)
        rc = read_and_clear_merge_error(&w[2], &site[2], g_msg, sizeof g_msg);
    if (rc != MERCURY_OK)
        return rc;
    for (int i = 0; i < 3; ++i)
        if (w[i] & 2u)
            return fail(MERCURY_EBOUNDS, "checked build: an out-of-range index was found and its access skipped "
                        "(site 0x%x)", site[i]);
    for (int i = 0; i < 3; ++i)
        if (w[i] & 1u)
            return fail(MERCURY_ETIMEOUT, "a bounded device wait ran out (site 0x%x)", site[i]);
    return MERCURY_OK;
}

int finish(int rc, cudaStream_t stream)
{
    if (rc != MERCURY_OK)
        return rc;
    if (sync_check()) {
        rc = collect_device_errors(stream);
        if (rc != MERCURY_OK)
            return rc;
    }
    return ok();
}

// Number of SMs of the current device (cached per device).
int sm_count(int *out)
{
    static std::atomic<int> cache[64];  // 0 until looked up
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(MERCURY_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *out = c;
            return MERCURY_OK;
        }
    }
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return fail(MERCURY_ECUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    if (dev >= 0 && dev < 64)
        cache[dev].store(n, std::memory_order_relaxed);
    *out = n;
    return MERCURY_OK;
}

long long env_ll(const char *name, long long dflt)
{
    const char *e = getenv(name);
    if (!e || !*e)
        return dflt;
    char *end = nullptr;
    long long v = strtoll(e, &end, 10);
    return (end && *end == '\0') ? v : dflt;
}

// Schedule chooser for mercury_attn_sharded: the fused schedule (one work
// item per rank's whole step sequence) unless it leaves the GPU short of
// work, in which case each rank's shifted step sequence is cut into runs
// whose partials are merged afterwards -- the latency / memory trade the
// pages describe (Silicon & Systems, "Memory capacity is part of
// performance"): more runs fill the SMs but cost scratch and merge traffic.
// The run count is the one schedule.cu's cost model predicts fastest among
// those whose scratch fits in MERCURY_SCRATCH_MAX_BYTES (default 4 GiB).
// Returns the number of runs (1 = fused).  MERCURY_SPLIT_GROUPS forces it.
// cap < 0: the scratch cap of mercury_attn_sharded (env or 4 GiB).
int choose_groups(int B, int Hq, int Hkv, int Sq, int Skv, int d, int R, int shift, int causal, int sms,
                  long long cap = -1)
{
    long long forced = env_ll("MERCURY_SPLIT_GROUPS", 0);
    if (forced >= 1)
        return (int)(forced < R ? forced : R);
    if (R == 1 || sms < 1)
        return 1;
    if (cap < 0)
        cap = env_ll("MERCURY_SCRATCH_MAX_BYTES", 4LL << 30);
    return best_run_count(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, sms, cap);
}

// Library-private stream-ordered pool for split-KV scratch (per device;
// memory is kept for reuse instead of being returned at every synchronise).
int scratch_pool(cudaMemPool_t *pool)
{
    static std::mutex mu;
    static cudaMemPool_t pools[64] = {};
    static bool made[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return fail(MERCURY_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64)
        return fail(MERCURY_ECUDA, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(mu);  // first calls from several threads create one pool
    if (!made[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        e = cudaMemPoolCreate(&pools[dev], &props);
        if (e != cudaSuccess)
            return fail(MERCURY_ECUDA, "cudaMemPoolCreate: %s", cudaGetErrorString(e));
        unsigned long long keep = ~0ull;
        e = cudaMemPoolSetAttribute(pools[dev], cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess)
            return fail(MERCURY_ECUDA, "cudaMemPoolSetAttribute: %s", cudaGetErrorString(e));
        made[dev] = true;
    }
    *pool = pools[dev];
    return MERCURY_OK;
}

// Run a validated call that produces the final O and LSE: the fused
// schedule writes them directly; a split schedule (per-step or grouped)
// writes one fp32 partial per slot into pooled scratch and merges the slots.
// out_bf16: out holds bf16 elements.
int run_to_output(AttnCall &c, float *out, float *lse, cudaStream_t s, int out_bf16 = 0)
{
    if (c.mode == kFused) {
        c.out = out;
        c.lse = lse;
        c.out_bf16 = out_bf16;
        return launch_attention(c, s, g_msg, sizeof g_msg);
    }
    c.out_bf16 = 0;  // the partials stay fp32
    Geom g;
    if (make_geom(g, c.B, c.Hq, c.Hkv, c.Sq, c.Skv, c.d, c.R, c.causal, c.mode, c.n_groups, c.Rq))
        return fail(MERCURY_EINVAL, "unsupported shape");
    const long long rows = (long long)c.B * c.Hq * c.Sq;
    const size_t o_bytes = (size_t)g.n_groups * rows * c.d * sizeof(float);
    const size_t l_bytes = (size_t)g.n_groups * rows * sizeof(float);
    cudaMemPool_t pool;
    int rc = scratch_pool(&pool);
    if (rc)
        return rc;
    void *scratch = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&scratch, o_bytes + l_bytes, pool, s);
    if (e != cudaSuccess)
        return fail(MERCURY_ECUDA, "split-KV scratch (%zu bytes): %s", o_bytes + l_bytes,
                    cudaGetErrorString(e));
    float *o_part = (float *)scratch;
    float *l_part = (float *)((char *)scratch + o_bytes);
    c.out = o_part;
    c.lse = l_part;
    rc = launch_attention(c, s, g_msg, sizeof g_msg);
    if (rc == MERCURY_OK)
        rc = launch_lse_merge(o_part, l_part, g.n_groups, rows, c.d, out, lse, s, g_msg, sizeof g_msg,
                              out_bf16);
    e = cudaFreeAsync(scratch, s);
    if (rc == MERCURY_OK && e != cudaSuccess)
        rc = fail(MERCURY_ECUDA, "cudaFreeAsync: %s", cudaGetErrorString(e));
    return rc;
}

int attn_common(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq, int Skv,
                int d, int R, int shift, int causal, float *out, float *lse, void *stream, int partial,
                int out_bf16 = 0)
{
    int rc = check_attn_args(q, k, v, B, Hq, Hkv, Sq, Skv, d, R, shift, causal, out, lse, partial);
    if (rc)
        return rc;
    cudaStream_t s = (cudaStream_t)stream;
    int groups = 1;
    if (!partial) {
        int sms = 0;
        rc = sm_count(&sms);
        if (rc)
            return rc;
        groups = choose_groups(B, Hq, Hkv, Sq, Skv, d, R, shift, causal, sms);
    }
    AttnCall c;
    c.q = q;
    c.k = k;
    c.v = v;
    c.B = B;
    c.Hq = Hq;
    c.Hkv = Hkv;
    c.Sq = Sq;
    c.Skv = Skv;
    c.d = d;
    c.R = R;
    c.causal = causal ? 1 : 0;
    // One run per step is the per-step split: use its shard-major item order
    // (resident CTAs then read the same shard, which matters once K/V
    // outgrow L2); the merge does not depend on the slot order.
    c.mode = (partial || groups >= R) ? kPerStep : (groups > 1 ? kGrouped : kFused);
    c.n_groups = (partial || groups >= R) ? R : groups;
    c.Rq = R;
    c.shift = shift;
    c.wait_ns = wait_budget_ns();
    c.fault = fault_mode();
    if (partial) {
        c.out = out;
        c.lse = lse;
        rc = launch_attention(c, s, g_msg, sizeof g_msg);
    } else {
        rc = run_to_output(c, out, lse, s, out_bf16);
    }
    return finish(rc, s);
}

}  // namespace

namespace mercury {

int set_error(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

int clear_error()
{
    return ok();
}

int device_sm_count(int *n)
{
    return sm_count(n);
}

int prepare_kernel(const void *func, int smem_bytes, KernelInfo *info, char *msg, size_t msg_len)
{
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, KernelInfo> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "cudaGetDevice: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find({func, dev});
    if (it != done.end()) {
        *info = it->second;
        return MERCURY_OK;
    }
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, func);
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "cudaFuncGetAttributes: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    KernelInfo ki{fa.numRegs, 0};
    e = cudaDeviceGetAttribute(&ki.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess || ki.sms < 1) {
        snprintf(msg, msg_len, "SM count: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    done[{func, dev}] = ki;
    *info = ki;
    return MERCURY_OK;
}

}  // namespace mercury

extern "C" {

int mercury_plan_shift(int R, int shift, int *order)
{
    if (!order)
        return fail(MERCURY_EINVAL, "order is NULL");
    int rc = check_shift(R, shift);
    if (rc)
        return rc;
    if (plan_shift(R, shift, order))
        return fail(MERCURY_EINVAL, "invalid (R, shift)");
    return ok();
}

int mercury_choose_runs(int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal, int R, int shift, int n_sms,
                        long long scratch_cap, int *n_runs)
{
    if (!n_runs)
        return fail(MERCURY_EINVAL, "n_runs is NULL");
    int rc = check_attn_shape(B, Hq, Hkv, Sq, Skv, d, R, shift, causal, 0);
    if (rc)
        return rc;
    if (n_sms < 1)
        return fail(MERCURY_EINVAL, "n_sms must be >= 1 (got %d)", n_sms);
    *n_runs = choose_groups(B, Hq, Hkv, Sq, Skv, d, R, shift, causal, n_sms, scratch_cap);
    return ok();
}

int mercury_attn_sharded(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq, int Skv,
                         int d, int R, int shift, int causal, float *out, float *lse, void *stream)
{
    CallRange range(__func__);
    return attn_common(q, k, v, B, Hq, Hkv, Sq, Skv, d, R, shift, causal, out, lse, stream, 0);
}

int mercury_attn_partial(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq, int Skv,
                         int d, int R, int shift, int causal, float *o_part, float *lse_part, void *stream)
{
    CallRange range(__func__);
    return attn_common(q, k, v, B, Hq, Hkv, Sq, Skv, d, R, shift, causal, o_part, lse_part, stream, 1);
}

int mercury_lse_merge(const float *o_part, const float *lse_part, int n_parts, long long rows, int d,
                      float *out, float *lse, void *stream)
{
    CallRange range(__func__);
    if (!o_part || !lse_part || !out || !lse)
        return fail(MERCURY_EINVAL, "null pointer argument");
    if (n_parts < 1 || n_parts > 4096)
        return fail(MERCURY_EINVAL, "n_parts must be in [1, 4096] (got %d)", n_parts);
    if (rows < 0)
        return fail(MERCURY_EINVAL, "rows must be >= 0");
    if (d < 4 || d > 512 || d % 4 != 0)
        return fail(MERCURY_EINVAL, "d must be a multiple of 4 in [4, 512] (got %d)", d);
    long long n = 1;
    if (!mul_ok(n, n_parts) || !mul_ok(n, rows) || !mul_ok(n, d))
        return fail(MERCURY_EINVAL, "tensor sizes overflow");
    if (!aligned(o_part, 16) || !aligned(out, 16))
        return fail(MERCURY_EALIGN, "o_part and out must be 16-byte aligned");
    if (!aligned(lse_part, 4) || !aligned(lse, 4))
        return fail(MERCURY_EALIGN, "lse_part and lse must be 4-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    int rc = launch_lse_merge(o_part, lse_part, n_parts, rows, d, out, lse, s, g_msg, sizeof g_msg);
    return finish(rc, s);
}

int mercury_attn_split_noalloc(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq,
                               int Skv, int d, int R, int shift, int causal, int n_runs, float *out,
                               float *lse, void *stream)
{
    CallRange range(__func__);
    cudaStream_t s = (cudaStream_t)stream;
    int rc = attn_split_noalloc(q, k, v, B, Hq, Hkv, Sq, Skv, d, R, shift, causal, n_runs, out, lse,
                                wait_budget_ns(), fault_mode(), s, g_msg, sizeof g_msg);
    return finish(rc, s);
}

int mercury_attn_sharded_bf16(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq,
                              int Skv, int d, int R, int shift, int causal, void *out, float *lse, void *stream)
{
    CallRange range(__func__);
    return attn_common(q, k, v, B, Hq, Hkv, Sq, Skv, d, R, shift, causal, (float *)out, lse, stream, 0, 1);
}

int mercury_attn_decode(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq, int Skv,
                        int d, int n_splits, int causal, float *out, float *lse, void *stream)
{
    CallRange range(__func__);
    if (n_splits < 0 || n_splits > kMaxR)
        return fail(MERCURY_EINVAL, "n_splits must be in [0, %d] (got %d)", kMaxR, n_splits);
    if (n_splits > 0 && Skv % n_splits != 0)
        return fail(MERCURY_EINVAL, "n_splits (%d) must divide Skv (%d)", n_splits, Skv);
    // the argument checks of a one-block call (Sq is not split)
    int rc = check_attn_args(q, k, v, B, Hq, Hkv, Sq, Skv, d, 1, 0, causal, out, lse, 0);
    if (rc)
        return rc;
    cudaStream_t s = (cudaStream_t)stream;
    int splits = n_splits;
    if (splits == 0) {
        // smallest divisor of Skv (<= 128) that gives every SM four work items
        int sms = 0;
        rc = sm_count(&sms);
        if (rc)
            return rc;
        Geom g1;
        if (make_geom(g1, B, Hq, Hkv, Sq, Skv, d, 1, causal, kFused, 1, 1))
            return fail(MERCURY_EINVAL, "unsupported shape");
        splits = 1;
        for (int c = 1; c <= kMaxR; ++c) {
            if (Skv % c)
                continue;
            splits = c;
            if (g1.n_items * c >= 4LL * sms)
                break;
        }
    }
    AttnCall c;
    c.q = q;
    c.k = k;
    c.v = v;
    c.B = B;
    c.Hq = Hq;
    c.Hkv = Hkv;
    c.Sq = Sq;
    c.Skv = Skv;
    c.d = d;
    c.R = splits;
    c.Rq = 1;
    c.causal = causal ? 1 : 0;
    c.mode = splits == 1 ? kFused : kPerStep;
    c.n_groups = splits;
    c.shift = 1;  // rank 0 reads shard j at step j
    c.wait_ns = wait_budget_ns();
    c.fault = fault_mode();
    rc = run_to_output(c, out, lse, s);
    return finish(rc, s);
}

int mercury_attn_run_schedule(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq,
                              int Skv, int d, int causal, const mercury_schedule *plan, float *out, float *lse,
                              void *stream)
{
    CallRange range(__func__);
    if (!plan)
        return fail(MERCURY_EINVAL, "plan is NULL");
    const int R = plan->R, Rq = plan->Rq, runs = plan->n_runs;
    // the argument checks of a one-block call, then the schedule's own
    int rc = check_attn_args(q, k, v, B, Hq, Hkv, Sq, Skv, d, 1, 0, causal, out, lse, 0);
    if (rc)
        return rc;
    rc = check_shift(R, plan->shift);
    if (rc)
        return rc;
    if (Skv % R != 0)
        return fail(MERCURY_EINVAL, "R (%d) must divide Skv (%d)", R, Skv);
    if (Rq != 1 && Rq != R)
        return fail(MERCURY_EINVAL, "Rq must be 1 or R (Rq %d, R %d)", Rq, R);
    if (Sq % Rq != 0)
        return fail(MERCURY_EINVAL, "Rq (%d) must divide Sq (%d)", Rq, Sq);
    if (runs < 1 || runs > R)
        return fail(MERCURY_EINVAL, "n_runs must be in [1, R] (n_runs %d, R %d)", runs, R);
    long long n = 1;
    if (!mul_ok(n, runs) || !mul_ok(n, B) || !mul_ok(n, Hq) || !mul_ok(n, Sq) || !mul_ok(n, d + 1) ||
        !mul_ok(n, 4))
        return fail(MERCURY_EINVAL, "scratch size overflows");
    AttnCall c;
    c.q = q;
    c.k = k;
    c.v = v;
    c.B = B;
    c.Hq = Hq;
    c.Hkv = Hkv;
    c.Sq = Sq;
    c.Skv = Skv;
    c.d = d;
    c.R = R;
    c.Rq = Rq;
    c.causal = causal ? 1 : 0;
    // as mercury_attn_sharded: one run per step takes the shard-major order
    c.mode = runs == 1 ? kFused : (runs >= R ? kPerStep : kGrouped);
    c.n_groups = runs >= R ? R : runs;
    c.shift = plan->shift;
    c.wait_ns = wait_budget_ns();
    c.fault = fault_mode();
    cudaStream_t s = (cudaStream_t)stream;
    rc = run_to_output(c, out, lse, s);
    return finish(rc, s);
}

int mercury_gemm_shifted(const void *a, const void *b, int M, int N, int K, int R, int shift, float *c,
                         void *stream)
{
    CallRange range(__func__);
    if (!a || !b || !c)
        return fail(MERCURY_EINVAL, "null pointer argument");
    if (M < 1 || N < 1 || K < 1)
        return fail(MERCURY_EINVAL, "M, N, K must be >= 1");
    int rc = check_shift(R, shift);
    if (rc)
        return rc;
    if (M % R != 0 || N % R != 0)
        return fail(MERCURY_EINVAL, "R (%d) must divide M (%d) and N (%d)", R, M, N);
    if ((N / R) % 8 != 0 || K % 8 != 0)
        return fail(MERCURY_EINVAL, "N/R and K must be multiples of 8 (N/R %d, K %d)", N / R, K);
    long long n = 1;
    if (!mul_ok(n, M) || !mul_ok(n, N) || !mul_ok(n, 4) || (long long)M * K > (1LL << 62) / 2 ||
        (long long)K * N > (1LL << 62) / 2)
        return fail(MERCURY_EINVAL, "tensor sizes overflow");
    if (!aligned(a, 16) || !aligned(b, 16) || !aligned(c, 16))
        return fail(MERCURY_EALIGN, "a, b and c must be 16-byte aligned");
    int order[kMaxR * kMaxR];
    plan_shift(R, shift, order);
    cudaStream_t s = (cudaStream_t)stream;
    rc = launch_gemm_shifted(a, b, M, N, K, R, order, c, wait_budget_ns(), s, g_msg, sizeof g_msg);
    return finish(rc, s);
}

int mercury_sync_status(void *stream)
{
    int rc = collect_device_errors((cudaStream_t)stream);
    if (rc != MERCURY_OK)
        return rc;
    return ok();
}

const char *mercury_last_error(void)
{
    return g_msg;
}

int mercury_work_decomposition(int B, int Hq, int Hkv, int Sq, int Skv, int d, int R, int causal, int partial,
                               long long *info)
{
    if (!info)
        return fail(MERCURY_EINVAL, "info is NULL");
    if (d != 64 && d != 128)
        return fail(MERCURY_EINVAL, "head dim must be 64 or 128 (got %d)", d);
    if (causal && Sq > Skv)
        return fail(MERCURY_EINVAL, "causal attention needs Sq <= Skv");
    if (partial < 0)
        return fail(MERCURY_EINVAL, "mode must be >= 0");
    Geom g;
    if (make_geom(g, B, Hq, Hkv, Sq, Skv, d, R, causal, partial >= 2 ? kGrouped : partial,
                  partial >= 2 ? partial : 1))
        return fail(MERCURY_EINVAL, "unsupported shape");
    info[0] = g.Mq;
    info[1] = g.Gp;
    info[2] = g.head_mode;
    info[3] = g.T_h;
    info[4] = g.T_r;
    info[5] = (long long)g.NHP * g.NRT;
    info[6] = g.n_items;
    info[7] = g.n_groups;
    return ok();
}

int mercury_work_item_rows(int B, int Hq, int Hkv, int Sq, int Skv, int d, int R, int shift, int causal,
                           int partial, long long item, long long *rows, int *n_rows, int *step)
{
    if (!rows || !n_rows || !step)
        return fail(MERCURY_EINVAL, "null pointer argument");
    if (d != 64 && d != 128)
        return fail(MERCURY_EINVAL, "head dim must be 64 or 128 (got %d)", d);
    if (causal && Sq > Skv)
        return fail(MERCURY_EINVAL, "causal attention needs Sq <= Skv");
    int rc = check_shift(R, shift);
    if (rc)
        return rc;
    Geom g;
    if (make_geom(g, B, Hq, Hkv, Sq, Skv, d, R, causal, partial >= 2 ? kGrouped : partial,
                  partial >= 2 ? partial : 1))
        return fail(MERCURY_EINVAL, "unsupported shape");
    if (item < 0 || item >= g.n_items)
        return fail(MERCURY_EINVAL, "item out of range");
    int order[kMaxR * kMaxR];
    plan_shift(R, shift, order);
    Item it = decode_item(g, item);
    int n = 0;
    for (int t = 0; t < 2; ++t) {
        if (!it.t[t].valid)
            continue;
        for (int r = 0; r < kTileRows; ++r) {
            if (r % g.Mq >= it.t[t].nq)
                continue;
            const long long head = it.t[t].h0 + r / g.Mq;
            const long long qi = it.t[t].q0 + r % g.Mq;
            rows[n++] = ((long long)it.b * Hq + head) * Sq + qi;
        }
    }
    *n_rows = n;
    *step = -1;
    if (g.partial == kPerStep) {
        for (int j = 0; j < R; ++j)
            if (order[it.rank * R + j] == it.shard)
                *step = j;
    } else if (g.partial == kGrouped) {
        *step = it.shard;
    }
    return ok();
}

}  // extern "C"
