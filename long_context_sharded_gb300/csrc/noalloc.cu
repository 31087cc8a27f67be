// noalloc.cu -- mercury_attn_split_noalloc: the split-KV schedule of
// mercury_attn_sharded for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc (or any routine that allocates) at the
// time they run attention: code inside a custom allocator or a memory
// manager that is itself servicing an allocation, real-time or serving loops
// that forbid allocator calls (and the synchronisation they can bring) on the
// hot path, and hosts that hand the library a fixed device-memory budget
// up front.  For them this entry point keeps the split-KV partials in a
// fixed-size array that lives in the library's own module: it is created when
// the library is loaded on a GPU and held by every GPU that loads the library
// until the process exits.
//
// Contract (also in include/mercury_attn.h):
//  * the scratch is kNoAllocScratchBytes (64 MiB) per device; a call whose
//    partials do not fit is rejected with MERCURY_EINVAL before any work;
//  * the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current.  With CUDA's lazy
//    module loading (the default) that lookup is also what loads this file's
//    module on the device and so reserves the 64 MiB: the first call can fail
//    for lack of device memory, and a caller that must not allocate makes one
//    warm-up call before it enters its allocation-free region (and before any
//    stream capture).  Calls after that allocate nothing;
//  * every call on a device uses the same array: calls that may overlap on
//    the GPU (different streams, or threads without ordering) race and give
//    wrong results; the array keeps the last call's contents, and nothing in
//    it has to start at zero because each call writes every partial slot it
//    later reads;
//  * no cudaMalloc, cudaFree or other allocating routine is called.
#include <cuda_runtime.h>

#include <mutex>
#include <stdint.h>
#include <stdio.h>

#include "internal.h"
#include "work.h"

namespace mercury {

// Maximum scratch of one call: n_runs * B*Hq*Sq*(d+1) * 4 bytes must fit.
constexpr size_t kNoAllocScratchBytes = 64ull << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_setup_mu;
void *g_scratch_ptr[64] = {};

// Device address of g_noalloc_scratch on the current device (looked up once
// per device).  In host code the array's name is only a host-side stand-in,
// so the kernels get the address returned here.
int scratch_address(void **out, char *msg, size_t msg_len)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "cudaGetDevice: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    if (dev < 0 || dev >= 64) {
        snprintf(msg, msg_len, "device ordinal %d out of range", dev);
        return MERCURY_ECUDA;
    }
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr) {
            snprintf(msg, msg_len, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
            return MERCURY_ECUDA;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return MERCURY_OK;
}

bool aligned(const void *p, uintptr_t a)
{
    return ((uintptr_t)p % a) == 0;
}

}  // namespace

int attn_split_noalloc(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq, int Skv,
                       int d, int R, int shift, int causal, int n_runs, float *out, float *lse,
                       unsigned long long wait_ns, int fault, cudaStream_t stream, char *msg, size_t msg_len)
{
    if (!q || !k || !v || !out || !lse) {
        snprintf(msg, msg_len, "null pointer argument");
        return MERCURY_EINVAL;
    }
    if (d != 64 && d != 128) {
        snprintf(msg, msg_len, "head dim must be 64 or 128 (got %d)", d);
        return MERCURY_EINVAL;
    }
    if (causal && Sq > Skv) {
        snprintf(msg, msg_len, "causal attention needs Sq <= Skv (Sq %d, Skv %d)", Sq, Skv);
        return MERCURY_EINVAL;
    }
    if (R < 1 || R > kMaxR || n_runs < 1 || n_runs > R) {
        snprintf(msg, msg_len, "need 1 <= R <= %d and 1 <= n_runs <= R (R %d, n_runs %d)", kMaxR, R, n_runs);
        return MERCURY_EINVAL;
    }
    if (shift < 0 || (shift >= 2 && R % shift != 0)) {
        snprintf(msg, msg_len, "invalid shift %d for R = %d", shift, R);
        return MERCURY_EINVAL;
    }
    Geom g;
    if (make_geom(g, B, Hq, Hkv, Sq, Skv, d, R, causal, kGrouped, n_runs)) {
        snprintf(msg, msg_len, "unsupported shape (B %d Hq %d Hkv %d Sq %d Skv %d R %d)", B, Hq, Hkv, Sq, Skv, R);
        return MERCURY_EINVAL;
    }
    if ((long long)B * Hq > 0x7fffffffLL || (long long)B * Hkv > 0x7fffffffLL) {
        snprintf(msg, msg_len, "B*H exceeds 2^31");
        return MERCURY_EINVAL;
    }
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 4)) {
        snprintf(msg, msg_len, "q, k, v, out must be 16-byte aligned and lse 4-byte aligned");
        return MERCURY_EALIGN;
    }
    // partials of every run: O [slots][rows][d] then LSE [slots][rows]
    const long long rows = (long long)B * Hq * Sq;
    const double need = (double)g.n_groups * (double)rows * (double)(d + 1) * 4.0;
    if (need > (double)kNoAllocScratchBytes) {
        snprintf(msg, msg_len,
                 "split-KV partials need %.0f bytes (%d runs x %lld rows x (d+1) x 4) but the "
                 "allocation-free scratch holds %zu bytes; use fewer runs or mercury_attn_sharded",
                 need, g.n_groups, rows, kNoAllocScratchBytes);
        return MERCURY_EINVAL;
    }
    void *scratch = nullptr;
    int rc = scratch_address(&scratch, msg, msg_len);
    if (rc != MERCURY_OK)
        return rc;
    const size_t o_bytes = (size_t)g.n_groups * rows * d * sizeof(float);
    float *o_part = (float *)scratch;
    float *l_part = (float *)((char *)scratch + o_bytes);

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
    c.mode = kGrouped;
    c.n_groups = n_runs;
    c.Rq = R;
    c.shift = shift;
    c.out = o_part;
    c.lse = l_part;
    c.wait_ns = wait_ns;
    c.fault = fault;
    rc = launch_attention(c, stream, msg, msg_len);
    if (rc == MERCURY_OK)
        rc = launch_lse_merge(o_part, l_part, g.n_groups, rows, d, out, lse, stream, msg, msg_len);
    return rc;
}

}  // namespace mercury
