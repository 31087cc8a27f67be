// internal.h -- declarations shared by the C-ABI layer and the kernel files.
#pragma once
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stddef.h>

#include "../../include/mercury_attn.h"

namespace mercury {

// An NVTX range around one C call, named after it, so that a profiler can
// pick the call's launches out of an application (for example
// `ncu --nvtx --nvtx-include "mercury_attn_sharded/"`).  Without an attached
// tool a range costs one well-predicted branch.
struct CallRange {
    explicit CallRange(const char *name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};

// One attention call, validated by the C-ABI layer.
struct AttnCall {
    const void *q = nullptr, *k = nullptr, *v = nullptr;
    int B = 0, Hq = 0, Hkv = 0, Sq = 0, Skv = 0, d = 0, R = 0, causal = 0;
    int mode = 0;            // kFused, kPerStep or kGrouped (work.h)
    int n_groups = 1;        // kGrouped: runs of steps per rank
    int Rq = 0;              // query blocks: R, or 1 for a decode split
    int shift = 1;           // shift order as in mercury_plan_shift (validated for R by the caller)
    float *out = nullptr, *lse = nullptr;  // fused: out/lse; otherwise [slots][B,Hq,Sq,(d)] partials
    unsigned long long wait_ns = 2000000000ull;
    int fault = 0;
    int out_bf16 = 0;        // fused only: out holds bf16 elements
};

int launch_attention(const AttnCall &c, cudaStream_t stream, char *msg, size_t msg_len);

// out_bf16: out holds bf16 elements (the merged fp32 values rounded to nearest).
int launch_lse_merge(const float *o_part, const float *lse_part, int n_parts, long long rows, int d,
                     float *out, float *lse, cudaStream_t stream, char *msg, size_t msg_len, int out_bf16 = 0);

// The split-KV schedule with its partials in the library's fixed-size
// device array instead of allocated scratch (noalloc.cu).  wait_ns and fault
// as in AttnCall.
int attn_split_noalloc(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq, int Skv,
                       int d, int R, int shift, int causal, int n_runs, float *out, float *lse,
                       unsigned long long wait_ns, int fault, cudaStream_t stream, char *msg, size_t msg_len);

// Shifted-shard GEMM: C [M,N] fp32 = A [M,K] bf16 x B [K,N] bf16; rank i's
// row block against B's column shards in the order order[i][*].
int launch_gemm_shifted(const void *a, const void *b, int M, int N, int K, int R, const int *order, float *c,
                        unsigned long long wait_ns, cudaStream_t stream, char *msg, size_t msg_len);

// Read and clear the GEMM kernel's device error word (no synchronisation).
int read_and_clear_gemm_error(unsigned int *word, unsigned int *site, char *msg, size_t msg_len);

// Read and clear the merge kernel's device error word (no synchronisation).
int read_and_clear_merge_error(unsigned int *word, unsigned int *site, char *msg, size_t msg_len);

// Synchronise `stream`, read and clear the kernels' device error word.
int read_and_clear_device_error(cudaStream_t stream, unsigned int *word, unsigned int *site, char *msg,
                                size_t msg_len);

// Status and message of the calling thread, shared by the C-ABI files.
int set_error(int code, const char *fmt, ...);
int clear_error();

// SMs of the current device (cached per device).
int device_sm_count(int *n);

// Launch preparation of a kernel on the current device, done once per
// (kernel, device): raises its dynamic shared-memory limit to smem_bytes and
// reports the registers per thread it was built with and the device's SM
// count.  Thread-safe.
struct KernelInfo {
    int regs;
    int sms;
};
int prepare_kernel(const void *func, int smem_bytes, KernelInfo *info, char *msg, size_t msg_len);

// Run count (1 = fused) with the least estimated time for a call with R
// virtual ranks each owning a query block, among those whose partials fit in
// scratch_cap bytes (schedule.cu's cost model, built-in device profile).
int best_run_count(int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal, int R, int shift, int n_sms,
                   long long scratch_cap);

}  // namespace mercury
