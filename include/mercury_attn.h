/*
 * mercury_attn.h -- C ABI of the GB300 (sm_103a) shifted-schedule sharded
 * attention library (libmercury_attn.so).
 *
 * The operation.  Mercury (SOSP 2025) keeps a shared KV buffer sharded across
 * ranks and lets every rank consume the shards in a rank-staggered order
 * instead of all at once (Silicon & Systems, "The hidden cost of synchronized
 * operators"); its shift primitive gives rank i at step j the piece
 * (j + i) mod J (Mercury-SOSP25 paper notes, section 核心方法).  The local
 * computation at every step is a fixed attention "patch" (FlashAttention) and
 * its result must equal single-device attention (Silicon & Systems,
 * "CommIR makes communication transformable" and "The tuning bill").
 *
 * Here R virtual ranks live in one GPU's memory.  Queries are split into R
 * contiguous blocks of Sq/R rows and keys/values into R contiguous shards of
 * Skv/R rows; virtual rank i owns query block i and, at step j, attends to KV
 * shard order[i][j] (see mercury_plan_shift).  The result equals
 *     O = softmax(Q K^T / sqrt(d)) V,   LSE = ln sum_k exp(q.k / sqrt(d))
 * for MHA, GQA and MQA (query head h uses KV head h / (Hq/Hkv)), causal
 * (key k allowed for query q iff k <= q + Skv - Sq) or not.
 *
 * Conventions for every call below.
 *   - Tensors are device pointers, row-major and contiguous, allocated and
 *     owned by the caller; the library keeps no reference after a call
 *     returns.  q [B,Hq,Sq,d] bf16; k, v [B,Hkv,Skv,d] bf16;
 *     out [B,Hq,Sq,d] fp32; lse [B,Hq,Sq] fp32 (natural log).
 *   - bf16 inputs and fp32 outputs must be 16-byte aligned (TMA and vector
 *     stores need it); lse arrays 4-byte aligned.
 *   - stream is a cudaStream_t passed as void* (NULL: the legacy default
 *     stream).  Compute calls are asynchronous on that stream.
 *   - Return value: MERCURY_OK (0) or a negative status; the message of the
 *     last non-zero status of the calling thread is mercury_last_error().
 *     No call throws, exits or traps.
 *   - Device waits are bounded (2 s by default, env MERCURY_WAIT_NS).  A wait
 *     that runs out makes the kernel record MERCURY_ETIMEOUT in a device
 *     error word and return early; that status is reported by
 *     mercury_sync_status().  With env MERCURY_SYNC_CHECK=1 every compute
 *     call synchronises its stream and returns the status itself.
 *   - Causal calls with more work items than the GPU has SMs let each CTA
 *     claim its next item from a counter: one of a fixed set of 4-byte slots
 *     in the library's module, taken in turn per launch and cleared by a
 *     memset on the call's stream (nothing is allocated; calls on different
 *     streams use different slots).  The first such call on a device looks
 *     up the slots' device address; make it before any stream capture.
 *   - Test hook (env MERCURY_FAULT, unset in normal use): drop_p_arrive or
 *     drop_kv_free makes the attention kernel withhold one internal arrive,
 *     so the MMA issuer's or the TMA producer's bounded wait runs out and the
 *     call ends with MERCURY_ETIMEOUT -- a timeout, never a GPU fault.
 */
#ifndef MERCURY_ATTN_H
#define MERCURY_ATTN_H

#if defined(__GNUC__)
#define MERCURY_API __attribute__((visibility("default")))
#else
#define MERCURY_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define MERCURY_OK        0
#define MERCURY_EINVAL   (-1)  /* bad argument: null pointer, bad size, bad shift, ... */
#define MERCURY_EALIGN   (-2)  /* a pointer is not aligned as required              */
#define MERCURY_ECUDA    (-3)  /* CUDA runtime / driver error (message has details) */
#define MERCURY_ETIMEOUT (-4)  /* a bounded device wait ran out                     */
#define MERCURY_ENOMEM   (-5)  /* host-side allocation failed                       */
#define MERCURY_EBUDGET  (-6)  /* no schedule fits the given device-memory budget   */
#define MERCURY_EBOUNDS  (-7)  /* checked build only: an out-of-range index was
                                  found in a kernel and its access skipped       */

/* Largest number of virtual ranks a compute call accepts. */
#define MERCURY_MAX_R 128

/*
 * mercury_plan_shift -- the shard/shift planner (pure host code, no GPU).
 *
 * Writes the [R][R] table order[i*R + j] = KV shard that virtual rank i reads
 * at step j.  shift selects the order:
 *   0      unshifted: order[i][j] = j (every rank reads the same shard at the
 *          same step: the synchronous, replicated schedule);
 *   1      flat shift: order[i][j] = (i + j) mod R, the shift primitive's
 *          "(j+i)%J" access (Mercury-SOSP25 paper notes, 核心方法);
 *   k >= 2 nested two-level shift for an Ro x Ri mesh with Ri = k inner
 *          (fast-link) ranks and Ro = R / k outer groups (hierarchical 2x4 /
 *          4x2 topologies, Silicon & Systems "What Mercury finds that
 *          templates miss"): rank i = a*Ri + b, step j = s*Ri + t,
 *          order = ((a + s) mod Ro)*Ri + (b + t) mod Ri.  k must divide R;
 *          k = R gives the flat order.
 * Every row and every column of the table is a permutation of 0..R-1.
 * order: host array of R*R ints, caller-owned.
 * Errors: MERCURY_EINVAL if R < 1, R > MERCURY_MAX_R, shift < 0, k does not
 * divide R, or order is NULL.
 */
MERCURY_API int mercury_plan_shift(int R, int shift, int *order);

/*
 * mercury_attn_sharded -- full attention through the shifted schedule, with
 * the per-step partials combined on the fly (online softmax across steps, the
 * same arithmetic as a log-sum-exp merge taken in step order).
 *
 * Passages: ranks consume the shared, sharded KV buffer in a rank-staggered
 * order (Silicon & Systems, "The hidden cost of synchronized operators"),
 * the shift primitive's (j+i)%J access gives the order (Mercury-SOSP25 paper
 * notes, 核心方法), every step runs the same local attention patch
 * (Silicon & Systems, "CommIR makes communication transformable"), and the
 * result is checked against single-device FlashAttention, i.e. plain
 * softmax attention (Silicon & Systems, "The tuning bill").
 *
 * Virtual rank i processes its query block against shards order[i][0..R-1]
 * (mercury_plan_shift(R, shift)); under causal masking a shard entirely in the
 * future of a block is skipped and the diagonal shard is masked per element.
 * Writes out [B,Hq,Sq,d] fp32 and lse [B,Hq,Sq] fp32.
 * Schedule: when one work item per rank's whole step sequence would leave the
 * GPU short of work (short query side, long KV), each rank's step sequence is
 * cut into g runs of consecutive steps; each run's partial (O, LSE) goes to
 * scratch memory and the runs are merged as by mercury_lse_merge.  g is the
 * run count that mercury_plan_schedules' cost model (built-in profile, this
 * R, Rq = R) predicts fastest among those whose scratch,
 * g * B*Hq*Sq*(d+1)*4 bytes, fits in 4 GiB (env MERCURY_SCRATCH_MAX_BYTES);
 * the scratch comes stream-ordered from a memory pool the library keeps per
 * device; env MERCURY_SPLIT_GROUPS=g forces g runs (1: no split).  The result
 * is the same up to rounding.
 * Requirements: B, Hq, Hkv, Sq, Skv >= 1; Hq % Hkv == 0; d in {64, 128};
 * 1 <= R <= MERCURY_MAX_R; Sq % R == 0 and Skv % R == 0; causal requires
 * Sq <= Skv; valid shift (as in mercury_plan_shift); every element count fits
 * in 63 bits and every sequence / head coordinate in 31 bits.
 * Errors: MERCURY_EINVAL, MERCURY_EALIGN, MERCURY_ECUDA, and
 * MERCURY_ETIMEOUT when MERCURY_SYNC_CHECK=1.
 */
MERCURY_API int mercury_attn_sharded(const void *q, const void *k, const void *v,
                         int B, int Hq, int Hkv, int Sq, int Skv, int d,
                         int R, int shift, int causal,
                         float *out, float *lse, void *stream);

/*
 * mercury_attn_sharded_bf16 -- mercury_attn_sharded with O written as bf16
 * (out [B,Hq,Sq,d] bf16, 16-byte aligned; lse stays fp32), halving the output
 * footprint.  Same schedule choice as mercury_attn_sharded; when it splits,
 * the partials stay fp32 in scratch and the merged O is rounded to bf16, so
 * the result is the fp32 call's O rounded to nearest.  Arguments,
 * requirements and errors as mercury_attn_sharded.
 */
MERCURY_API int mercury_attn_sharded_bf16(const void *q, const void *k, const void *v,
                                          int B, int Hq, int Hkv, int Sq, int Skv, int d,
                                          int R, int shift, int causal,
                                          void *out, float *lse, void *stream);

/*
 * mercury_attn_partial -- the per-step partials of the shifted schedule.
 *
 * Passages: each step's output is the local patch applied to one shard in
 * the shifted order (Mercury-SOSP25 paper notes, 核心方法: shift, shard and
 * the FlashAttention patch); combining the steps' partial results is what
 * the RingAttention-style asynchronous schedules that Mercury reproduces do
 * (Mercury-SOSP25 paper notes, one-line summary and 实验与结果).
 *
 * For every query row q (virtual rank i = q / (Sq/R)) and step j, slot j of
 * the outputs holds attention of that row over shard order[i][j] alone,
 * normalised within the shard:
 *   o_part  [R][B,Hq,Sq,d] fp32, lse_part [R][B,Hq,Sq] fp32.
 * A row with no allowed key in its shard (causal) gets O = 0, LSE = -inf.
 * mercury_lse_merge(o_part, lse_part, R, B*Hq*Sq, d, out, lse) then gives the
 * same result as mercury_attn_sharded.  Requirements and errors as for
 * mercury_attn_sharded.
 */
MERCURY_API int mercury_attn_partial(const void *q, const void *k, const void *v,
                         int B, int Hq, int Hkv, int Sq, int Skv, int d,
                         int R, int shift, int causal,
                         float *o_part, float *lse_part, void *stream);

/*
 * mercury_lse_merge -- exact log-sum-exp combine of n_parts partial results.
 *
 * Per row r:  L = ln sum_j exp(lse_part[j][r]),
 *             out[r][:] = sum_j exp(lse_part[j][r] - L) * o_part[j][r][:],
 *             lse[r] = L.
 * A part with lse = -inf has weight 0 and its o_part row is not read; a row
 * whose parts are all -inf gets out = 0 and lse = -inf.  The pages name no
 * combine formula; this is the standard exact one of the RingAttention-style
 * schedules that Mercury reproduces (Mercury-SOSP25 paper notes, one-line
 * summary).
 * o_part [n_parts][rows][d] fp32 (16-byte aligned), lse_part [n_parts][rows]
 * fp32, out [rows][d] fp32 (16-byte aligned), lse [rows] fp32.
 * Requirements: 1 <= n_parts <= 4096; rows >= 0; d % 4 == 0, 4 <= d <= 512;
 * n_parts*rows*d fits in 63 bits.  rows == 0 is a no-op.
 * Errors: MERCURY_EINVAL, MERCURY_EALIGN, MERCURY_ECUDA.
 */
MERCURY_API int mercury_lse_merge(const float *o_part, const float *lse_part, int n_parts,
                      long long rows, int d, float *out, float *lse, void *stream);

/*
 * mercury_attn_decode -- attention for a short query side against a long KV
 * (decode and chunked-prefill shapes), split across the KV.
 *
 * The whole query side [B,Hq,Sq,d] is one block (one rank); the KV is cut
 * into n_splits contiguous shards, each shard's partial (O, LSE) is computed
 * on its own work items (which fills the GPU when B*Hq*Sq is small) into
 * scratch memory from the library's per-device pool, and the partials are
 * combined by the log-sum-exp merge of mercury_lse_merge.  The result equals
 * softmax(QK^T/sqrt(d))V; causal alignment as elsewhere (k <= q + Skv - Sq).
 * n_splits: 1..128 dividing Skv, or 0 to choose the smallest divisor of Skv
 * that gives every SM four work items.  Scratch: n_splits * B*Hq*Sq*(d+1)*4
 * bytes.  Other arguments, layouts and errors as mercury_attn_sharded
 * (Sq need not be divisible by anything).
 */
MERCURY_API int mercury_attn_decode(const void *q, const void *k, const void *v,
                                    int B, int Hq, int Hkv, int Sq, int Skv, int d,
                                    int n_splits, int causal, float *out, float *lse,
                                    void *stream);

/*
 * mercury_gemm_shifted -- the all-gather GEMM pattern under the shifted
 * schedule (the pages' second operator family: every rank owns a slice of A
 * while all ranks need B, and B's pieces are read from their owners in a
 * rank-staggered order; Silicon & Systems, "The hidden cost of synchronized
 * operators" and "What Mercury finds that templates miss").
 *
 * R virtual ranks: rank i owns the row block A_i = rows [i*M/R, (i+1)*M/R) of
 * A; B is cut into R column shards B_s = columns [s*N/R, (s+1)*N/R); at step j
 * rank i computes C[block i, shard order[i][j]] = A_i B_s, order as in
 * mercury_plan_shift(R, shift).  The result is C = A B.
 * a [M,K] bf16, b [K,N] bf16, c [M,N] fp32, all row-major device pointers,
 * 16-byte aligned, caller-owned.  Requirements: M, N, K >= 1; R divides M and
 * N; N/R and K multiples of 8; valid (R, shift).
 * Errors: MERCURY_EINVAL, MERCURY_EALIGN, MERCURY_ECUDA, and
 * MERCURY_ETIMEOUT when MERCURY_SYNC_CHECK=1.
 */
MERCURY_API int mercury_gemm_shifted(const void *a, const void *b, int M, int N, int K,
                                     int R, int shift, float *c, void *stream);

/*
 * mercury_attn_split_noalloc -- mercury_attn_sharded's split-KV schedule for
 * callers that cannot allocate device memory.  (The pages have no
 * counterpart: this is a deployment convenience of this library.)
 *
 * Callers inside an allocator or memory manager, serving or real-time loops
 * that forbid allocator calls on their hot path, and hosts that give the
 * library a fixed device-memory budget cannot let a call allocate scratch.
 * This call cuts each rank's shifted step sequence into n_runs runs (as
 * mercury_attn_sharded does when it splits), keeps the runs' partial (O, LSE)
 * in a fixed 64 MiB array that the library's module holds on every GPU that
 * loads it (until the process exits), and merges them into out / lse.  It
 * calls no cudaMalloc, cudaFree or other allocating routine.
 * Arguments as mercury_attn_sharded, plus 1 <= n_runs <= R (rounded like the
 * run count of mercury_work_decomposition).  The partials need
 * runs * B*Hq*Sq*(d+1)*4 bytes; more than 64 MiB is rejected with
 * MERCURY_EINVAL before any work.
 * The first call on a device looks up the array's device address with that
 * device current.  Under CUDA's lazy module loading (the default) that
 * lookup also loads the array's module on the device, which reserves the
 * 64 MiB: the first call can fail with MERCURY_ECUDA for lack of device
 * memory.  A caller that must not allocate therefore makes one warm-up call
 * on each device before it enters its allocation-free region (and before
 * any stream capture); calls after that allocate nothing.  Waits and the
 * test fault hook follow MERCURY_WAIT_NS and MERCURY_FAULT as for every
 * other call.  All calls on a device
 * share the array: calls that can overlap on the GPU (other streams, other
 * threads) race and corrupt each other's results.  The array keeps the last
 * call's contents; nothing in it needs to start at zero, since each call
 * writes every partial it reads.
 * Errors: MERCURY_EINVAL, MERCURY_EALIGN, MERCURY_ECUDA, and
 * MERCURY_ETIMEOUT when MERCURY_SYNC_CHECK=1.
 */
MERCURY_API int mercury_attn_split_noalloc(const void *q, const void *k, const void *v,
                               int B, int Hq, int Hkv, int Sq, int Skv, int d,
                               int R, int shift, int causal, int n_runs,
                               float *out, float *lse, void *stream);

/*
 * mercury_sync_status -- synchronise `stream`, then read and clear the device
 * error words of this process's kernels.  Returns MERCURY_OK,
 * MERCURY_ETIMEOUT (a bounded device wait ran out in some earlier kernel),
 * MERCURY_EBOUNDS (only in the checked build, libmercury_attn.so built with
 * -DMERCURY_CHECK: a kernel found an out-of-range TMA coordinate or output
 * index and skipped that access) or MERCURY_ECUDA (the synchronise itself
 * failed).
 */
MERCURY_API int mercury_sync_status(void *stream);

/* Message for the last non-zero status returned to the calling thread
 * ("" if none).  The pointer stays valid until the thread's next call. */
MERCURY_API const char *mercury_last_error(void);

/*
 * mercury_work_decomposition -- host-side view of how a compute call splits
 * the work (no GPU needed; used to test the planner's coverage).
 * info[0..7] receives: rows per head in a query tile (Mq), heads per tile
 * (Gp), pairing mode (1: the two tiles of a work item are two head groups at
 * the same rows; 0: two consecutive row tiles of the same heads), head tiles
 * per KV group, row tiles per query block, work items per (batch, KV head,
 * rank), total work items, output slots.  mode: 0 the fused schedule of
 * mercury_attn_sharded, 1 mercury_attn_partial's per-step split, g >= 2 the
 * split into g runs of steps (g is rounded so every run but the last has
 * ceil(R/g) steps).
 * Errors: MERCURY_EINVAL for arguments a compute call would reject.
 */
MERCURY_API int mercury_work_decomposition(int B, int Hq, int Hkv, int Sq, int Skv, int d,
                               int R, int causal, int mode, long long *info);

/*
 * mercury_work_item_rows -- for work item `item` of that decomposition, writes
 * the flat rows ((b*Hq + h)*Sq + q) it computes and the output slot it writes
 * (mode 1: the step; mode >= 2: the run) or -1 (mode 0): rows[0..n-1],
 * *n_rows = n (at most 256), *step.  Pure host code, for coverage tests.
 * Errors: MERCURY_EINVAL.
 */
MERCURY_API int mercury_work_item_rows(int B, int Hq, int Hkv, int Sq, int Skv, int d,
                           int R, int shift, int causal, int mode,
                           long long item, long long *rows, int *n_rows, int *step);

/*
 * Schedule selection under a device-memory budget.
 *
 * The pages make memory capacity part of performance: a schedule that keeps
 * everything in one piece runs fastest when memory is plentiful, one that
 * splits its buffers pays extra traffic but can be the only one that fits,
 * and both should stay available (Silicon & Systems, "Memory capacity is
 * part of performance").  Candidates are filtered in stages -- a static check
 * of sizes and divisibility, a cost estimate, then profiling of the best few
 * on the target device -- and the tuned result is kept under a key of the
 * device, the library build and the shape, with a re-check when it stops
 * meeting its measured time (Silicon & Systems, "CommIR makes communication
 * transformable" and "The tuning bill").
 *
 * On one GPU a schedule is the tuple (R, Rq, n_runs, shift):
 *   R       KV shards (virtual ranks);
 *   Rq      query blocks: R (virtual rank i owns query block i) or 1 (the
 *           whole query side is one block that visits all R shards -- the
 *           query-tile split used for short query sides);
 *   n_runs  each rank's shifted step sequence is cut into n_runs runs of
 *           ceil(R / n_runs) consecutive steps; 1 is the fused schedule
 *           (partials combined on the fly, no scratch), n_runs > 1 writes one
 *           partial (O, LSE) per run to scratch and merges them as
 *           mercury_lse_merge does.  Scratch = n_runs * B*Hq*Sq*(d+1)*4 bytes.
 * The result is the same for every schedule up to rounding.
 */

/* Costs of this library's kernels on one device (microseconds, GB/s). */
typedef struct mercury_cost_profile {
    double tile_us;    /* one 128-key K/V tile through a work item holding two query tiles */
    double tile1_us;   /* the same for a work item holding one query tile */
    double item_us;    /* fixed cost of a work item (query load, epilogue) */
    double launch_us;  /* fixed cost of one attention launch */
    double merge_gbs;  /* LSE merge throughput: bytes read + written per second / 1e9 */
    double hbm_gbs;    /* device-to-device copy throughput, GB/s (bytes read + written) */
    int n_sms;         /* SMs the persistent attention kernel spreads its work items over */
    int measured;      /* 1: from mercury_measure_cost_profile; 0: built-in GB300 figures */
} mercury_cost_profile;

/* One candidate schedule and its estimated (and, once profiled, measured) cost. */
typedef struct mercury_schedule {
    int R;                    /* KV shards (virtual ranks) */
    int Rq;                   /* query blocks: R or 1 */
    int n_runs;               /* runs per rank's step sequence (1 = fused) */
    int shift;                /* shift order (as in mercury_plan_shift) */
    long long work_items;     /* attention work items of the launch */
    long long scratch_bytes;  /* partials of the runs; 0 when n_runs == 1 */
    long long hbm_bytes;      /* q, k, v, out, lse and scratch together */
    double predicted_us;      /* cost-model estimate of the whole call */
    double measured_us;       /* median device time when profiled, else -1 */
    int pareto;               /* 1: no other candidate of the same call is both
                                 smaller (hbm_bytes) and predicted faster */
} mercury_schedule;

/*
 * mercury_default_cost_profile -- the built-in cost figures (measured on a
 * GB300 with this library) for a device with n_sms SMs (n_sms >= 1).
 * Pure host code.  Errors: MERCURY_EINVAL (prof NULL or n_sms < 1).
 */
MERCURY_API int mercury_default_cost_profile(int n_sms, mercury_cost_profile *prof);

/*
 * mercury_measure_cost_profile -- measure the cost figures on the current
 * device: timed attention launches on synthetic inputs (one and two work
 * items per SM, two key lengths, one and two query tiles per item), one
 * timed merge and one timed device-to-device copy, each the median of five
 * runs after two warm-ups.  The
 * call allocates about 2 GB of device memory for its inputs, frees it
 * before returning, and synchronises `stream`.
 * Errors: MERCURY_EINVAL (prof NULL), MERCURY_ECUDA, MERCURY_ETIMEOUT.
 */
MERCURY_API int mercury_measure_cost_profile(mercury_cost_profile *prof, void *stream);

/*
 * mercury_plan_schedules -- the static filter and the cost estimate (pure
 * host code, no GPU).
 *
 * Enumerates the schedules of an attention call with the shape given: R
 * fixed (R >= 1) or, with R == 0, every R in 1..MERCURY_MAX_R that divides
 * Skv and suits `shift` (k >= 2 must divide R); Rq in {R, 1} (R only if it
 * divides Sq); every distinct n_runs in 1..R.  Drops those whose hbm_bytes
 * exceed budget_bytes (budget_bytes <= 0: no limit) and estimates the rest:
 * every work item costs item_us plus its K/V tiles times tile_us (tile1_us
 * for one query tile), items go to n_sms CTAs round robin in launch order
 * (in a causal launch with more items than CTAs, as the kernel does: each to
 * the CTA free earliest), and the attention launch costs launch_us plus the
 * larger of the busiest CTA's sum and its least memory traffic (q, k, v read
 * once, its outputs written once) at hbm_gbs; when n_runs > 1 a second launch and the merge's
 * bytes at merge_gbs are added.
 * Writes the min(count, max_plans) fastest candidates to plans[], fastest
 * first (ties: fewer hbm_bytes, then Rq == R, then smaller R, then fewer
 * runs), with the Pareto flag set over all candidates; *n_plans = count.  prof is required (from
 * mercury_default_cost_profile or mercury_measure_cost_profile).
 * Requirements: as mercury_attn_sharded for (B, Hq, Hkv, Sq, Skv, d, causal,
 * shift); max_plans >= 0 (plans may be NULL when it is 0).
 * Errors: MERCURY_EINVAL; MERCURY_EBUDGET when no candidate fits the budget
 * (the message states the smallest hbm_bytes of any candidate).
 */
MERCURY_API int mercury_plan_schedules(int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
                                       int R, int shift, long long budget_bytes,
                                       const mercury_cost_profile *prof,
                                       mercury_schedule *plans, int max_plans, int *n_plans);

/*
 * mercury_choose_runs -- the run count mercury_attn_sharded (and
 * mercury_attn_sharded_bf16) uses for a call of this shape on a device with
 * n_sms SMs: the n_runs that mercury_plan_schedules' estimate with the
 * built-in profile (this R, Rq = R) predicts fastest among those whose
 * scratch, n_runs * B*Hq*Sq*(d+1)*4 bytes, fits in scratch_cap bytes (ties:
 * fewer runs); scratch_cap < 0 takes mercury_attn_sharded's cap (env
 * MERCURY_SCRATCH_MAX_BYTES, default 4 GiB); env MERCURY_SPLIT_GROUPS=g
 * forces min(g, R) as it does for the call; R == 1 gives 1.  The search is
 * the pages' staged one -- a static memory check, then a cost estimate
 * (Mercury-SOSP25 paper notes, 核心方法 and 设计取舍) -- kept cheap because
 * a new shape's first call waits for it (time to first usable schedule:
 * Silicon & Systems, "The tuning bill"): a candidate whose lower bound (its
 * work items' summed cost spread over n_sms CTAs, its longest item, its
 * least memory traffic, plus the merge) is no better than the best so far is
 * not estimated further, which leaves the answer unchanged.  Pure host code,
 * no GPU; the answer is remembered per shape.
 * Requirements: as mercury_attn_sharded for the shape; n_sms >= 1; n_runs
 * not NULL.  Errors: MERCURY_EINVAL.
 */
MERCURY_API int mercury_choose_runs(int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal,
                                    int R, int shift, int n_sms, long long scratch_cap,
                                    int *n_runs);

/*
 * mercury_attn_run_schedule -- attention by a given schedule (one of
 * mercury_plan_schedules' candidates, or any valid tuple).  Arguments and
 * layouts as mercury_attn_sharded; the schedule's R, Rq, n_runs and shift
 * replace R and shift.  The scratch of n_runs > 1 comes stream-ordered from
 * the library's per-device pool.
 * Errors: MERCURY_EINVAL (invalid tuple for the shape), MERCURY_EALIGN,
 * MERCURY_ECUDA, and MERCURY_ETIMEOUT when MERCURY_SYNC_CHECK=1.
 */
MERCURY_API int mercury_attn_run_schedule(const void *q, const void *k, const void *v,
                                          int B, int Hq, int Hkv, int Sq, int Skv, int d,
                                          int causal, const mercury_schedule *plan,
                                          float *out, float *lse, void *stream);

/*
 * mercury_tune_schedule -- pick a schedule by measurement and compute the
 * attention with it.
 *
 * Plans the call (mercury_plan_schedules with the profile of
 * mercury_default_cost_profile for this device), runs the top_k predicted
 * candidates (1 <= top_k <= 16) on the caller's buffers -- one warm-up and
 * three timed launches each, CUDA events on `stream`, median -- and keeps the
 * fastest.  The choice is cached for the process under (device ordinal, SM
 * count, compute capability, library build, shape, R, shift, budget, top_k).
 * A later call with the same key runs the cached schedule twice, timed; if
 * the faster run takes more than 1.5 times its recorded time plus 20 us (an
 * allowance for host launch jitter on very short calls; env
 * MERCURY_TUNE_RECHECK sets the factor, 0 re-tunes on every call) the entry
 * is dropped and the call tunes again.  On return out / lse hold the attention result (from the
 * chosen schedule's last run) and *best (if not NULL) the chosen schedule
 * with measured_us set.  *cache_hit (if not NULL) is 1 when no tuning ran.
 * The call synchronises `stream`.
 * Errors: as mercury_plan_schedules and mercury_attn_run_schedule.
 */
MERCURY_API int mercury_tune_schedule(const void *q, const void *k, const void *v,
                                      int B, int Hq, int Hkv, int Sq, int Skv, int d,
                                      int R, int shift, int causal, long long budget_bytes,
                                      int top_k, float *out, float *lse, void *stream,
                                      mercury_schedule *best, int *cache_hit);

/* Drop every cached tuning result of mercury_tune_schedule. */
MERCURY_API void mercury_tune_cache_clear(void);

#ifdef __cplusplus
}
#endif

#endif /* MERCURY_ATTN_H */
