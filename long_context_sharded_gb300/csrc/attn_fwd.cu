// attn_fwd.cu -- the attention "patch" of the shifted schedule on sm_103a.
//
// Mercury keeps an optimised local attention kernel fixed and schedules the
// distributed loop around it (Silicon & Systems, "CommIR makes communication
// transformable"; Mercury-SOSP25 paper notes 核心方法, FlashAttention patch).
// This file is that patch for one GB300: a FlashAttention-style forward pass
// whose KV loop walks the shards in the shifted order, rank i reading shard
// order[i][j] at step j (the (j+i)%J access of the shift primitive, or its
// nested two-level form), with the R virtual ranks' data all in local HBM.
//
// One persistent CTA per SM takes work items in turn (a work item: up to two
// 128-row query tiles sharing a KV head, one (batch, KV head) at a time):
//   warp 0      TMA producer: decodes and publishes the CTA's work items,
//               loads Q tiles once, then K and V tiles into two
//               shared-memory rings, in the shifted shard order
//   warp 1      MMA issuer (the whole warp runs the loop, one elected lane
//               issues): S_t = Q_t K^T and O_t += P_t V on the tensor cores
//               (tcgen05.mma kind::f16, fp32 accumulators in tensor
//               memory); P_t is read straight from tensor memory
//   warps 4-7   softmax for tile 0, warps 8-11 for tile 1 (one query row per
//               thread): online softmax in the log2 domain, rescaling of O_t
//               in tensor memory when the running max moves by more than
//               2^8 (the row max is only taken when a tile's probabilities
//               could pass that), bf16 P_t written back over S_t, final O/l
//               and LSE
// Tensor memory (512 columns): S_0 [0,128) S_1 [128,256) O_0 [256,256+D)
// O_1 [256+D, 256+2D).
//
// The MMA issue order is PV_0(n-1), S_0(n), PV_1(n-1), S_1(n): the tensor
// pipe runs one tile's products while the other tile's softmax works.  A
// commit after S_t(n) therefore also covers PV_t(n-1), so the softmax may
// rescale O_t as soon as S_t(n) is ready.
//
// Every wait is bounded (%globaltimer); when one runs out the CTA records
// MERCURY_ETIMEOUT in a device error word, raises a shared abort flag so the
// other roles stop waiting too, and leaves: the producer first waits (bounded
// again) for the tile loads it has issued to land, the MMA issuer for the
// tensor-core operations it has issued to complete, then every thread meets
// at one exit barrier and the tensor memory is freed.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "internal.h"
#include "ptx.cuh"
#include "work.h"

namespace mercury {

// Device error word: kErrTimeout = a bounded wait ran out; kErrBounds = the
// checked build skipped an out-of-range access.  g_err_site keeps the first
// site recorded (for the error message).
__device__ unsigned int g_err_word = 0;
__device__ unsigned int g_err_site = 0;

// Work-item counters for dynamically scheduled launches: each launch takes
// the next slot (cycling) and zeroes it on its stream first, so launches on
// different streams never share one.
constexpr int kItemCounterSlots = 4096;
__device__ unsigned int g_item_counters[kItemCounterSlots];

// Kernel parameters.  The shift table's capacity TC (R <= TC) is a template
// parameter: the whole block travels with every launch, and a 128 x 128 table
// (16 KB) costs the host ~5 us per launch, so calls with R <= 32 take a 1 KB
// table.  (Computing the shard in the kernel instead was measured slower on
// short work items.)
template <int TC>
struct AttnParams {
    Geom g;
    float scale_log2;        // log2(e) / sqrt(d)
    int fault;               // test hook: 1 = drop the first P-ready arrive of tile 0,
                             // 2 = drop the first "iteration done" arrive (kv_free)
    int out_bf16;            // fused calls only: O is written as bf16 ([B,Hq,Sq,d], 2 bytes)
    int out_v8;              // O's base is 32-byte aligned: rows are stored 32 bytes per lane
    int o_tma;               // fp32 O: rows go out through shared memory and TMA tensor stores
    long long o_rows;        // rows of the O tensor map (all slots)
    float *out;              // fused: out; partial: o_part
    float *lse;              // fused: lse; partial: lse_part
    long long out_elems;     // elements of out / o_part (all slots); checked build only
    long long lse_elems;     // elements of lse / lse_part (all slots); checked build only
    long long slot_o;        // partial: elements between slots of o_part
    long long slot_lse;      // partial: elements between slots of lse_part
    unsigned long long wait_ns;
    // Dynamic work items: the producer claims item gridDim.x + atomicAdd(*item_counter)
    // after each CTA's first item (blockIdx.x); nullptr = static round robin.
    unsigned int *item_counter;
    // fused, grouped: tab[i*R + j] = shard of rank i at step j;
    // per step: tab[i*R + s] = step (slot) at which rank i reads shard s.
    unsigned char tab[TC * TC];
};
constexpr int kSmallTab = 32;  // table capacity of calls with R <= 32

namespace {

constexpr int kThreads = 384;
constexpr int kItemSlots = 4;  // work items published by the producer ahead of the other roles

// A work item as the producer publishes it to the MMA and softmax warps:
// decoded once, with its number of KV tiles, so that no consumer spends its
// way from one item to the next on the index arithmetic (a few thousand
// cycles of 64-bit division and a walk over the item's steps, measured on
// the item boundary).  has == 0 ends the CTA's work.
struct alignas(16) ItemSlot {
    int has;
    int ntot;   // KV tiles of the item's whole sequence
    Item it;
    int pad;
};
static_assert(sizeof(ItemSlot) == 64, "one 64-byte ring entry per item");
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale when max grows by > 2^8
constexpr float kRescaleFactor = 256.0f;   // 2^kRescaleThreshold

struct Ctl {
    unsigned long long budget;
    volatile uint32_t *abort;
};

// Exit barrier (named, all threads of the CTA; each role reaches it from its
// own branch).
constexpr uint32_t kExitBarrier = 1;

// Bounded wait on an mbarrier phase.  false: timed out here or elsewhere.
// Inlined: a call shared by warps with different setmaxnreg budgets does
// not register-allocate.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t parity, Ctl c, uint32_t site)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity))
                return true;
        if (*c.abort)
            return false;
        if (globaltimer_ns() - t0 > c.budget) {
            *c.abort = 1u;
            atomicOr(&g_err_word, kErrTimeout);
            atomicCAS(&g_err_site, 0u, site);
            return false;
        }
    }
}

// Checked build: an out-of-range index found at `site`.
__device__ __forceinline__ void record_bounds(uint32_t site)
{
    atomicOr(&g_err_word, kErrBounds);
    atomicCAS(&g_err_site, 0u, site);
}

// Bounded wait used on the way out: does not give up when another role
// aborted (the operations it waits for complete on their own), only when its
// own budget runs out, which it records like any other timeout.
__device__ __forceinline__ bool drain_phase(uint64_t *bar, uint32_t parity, Ctl c, uint32_t site)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > c.budget) {
            atomicOr(&g_err_word, kErrTimeout);
            atomicCAS(&g_err_site, 0u, site);
            return false;
        }
    }
    return true;
}

// Shard visited at step `step` of the item's sequence (fused: the rank's R
// steps; per step: the item's shard; grouped: the item's run of steps).
template <int TC>
__device__ __forceinline__ int shard_at(const AttnParams<TC> &p, const Item &it, int step)
{
    if (p.g.partial == kPerStep)
        return it.shard;
    const int j = p.g.partial == kGrouped ? it.shard * p.g.spg + step : step;
    return (int)p.tab[it.rank * p.g.R + j];
}

// Output slot of a non-fused item: the step (per step) or the run (grouped).
template <int TC>
__device__ __forceinline__ int out_slot(const AttnParams<TC> &p, const Item &it)
{
    return p.g.partial == kPerStep ? (int)p.tab[it.rank * p.g.R + it.shard] : it.shard;
}

template <int D, int NK, int NV>
struct Smem {
    static constexpr int kQBytes = kTileRows * D * 2;   // one query tile, bf16
    static constexpr int kKVBytes = kTileKeys * D * 2;  // one K or V tile, bf16
    static constexpr int kBoxBytes = 128 * 128;         // 128 rows x 128 B swizzle column
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = 2 * kQBytes;
    static constexpr int kOffV = kOffK + NK * kKVBytes;
    // O staging for the epilogue's tensor stores: 32 rows x 32 fp32 (4 KB,
    // 128-byte swizzle) per softmax warp
    static constexpr int kStageBytes = 32 * 32 * 4;
    static constexpr int kOffStage = kOffV + NV * kKVBytes;
    static constexpr int kOffBar = kOffStage + 8 * kStageBytes;
    static constexpr int NE = NK > NV ? NK : NV;  // ring of "iteration done" events
    static constexpr int kNumBars = 2 + NK + NV + NE + 8 + 1 + 2 * kItemSlots;
    static constexpr int kOffRing = (kOffBar + 8 * kNumBars + 15) / 16 * 16;  // kItemSlots published items
    static constexpr int kOffMisc = kOffRing + (int)sizeof(ItemSlot) * kItemSlots;  // tmem slot, abort flag
    static constexpr int kBytes = kOffMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

// Register split (setmaxnreg): the producer / MMA warpgroup gives registers
// to the two softmax warpgroups.  The launch must provide at least
// kMinLaunchRegs registers per thread (the host checks this before launching:
// with fewer, setmaxnreg.inc would wait for registers that do not exist).
constexpr uint32_t kRegsProducer = 104;
constexpr uint32_t kRegsSoftmax = 200;
constexpr int kMinLaunchRegs = (int)((kRegsProducer + 2 * kRegsSoftmax) * 128 + kThreads - 1) / kThreads;

// Key range [lo, hi) of step st of an item; returns its number of KV tiles.
template <int TC>
__device__ __forceinline__ int step_range(const AttnParams<TC> &p, const Item &it, int st, int &lo, int &hi)
{
    shard_range(p.g, it, shard_at(p, it, st), lo, hi);
    return n_kv_tiles(lo, hi);
}

// KV tiles of the item's whole shifted sequence.
template <int TC>
__device__ __forceinline__ int item_tiles(const AttnParams<TC> &p, const Item &it)
{
    int n = 0;
    const int ns = item_steps(p.g, it);
    for (int st = 0; st < ns; ++st) {
        int lo, hi;
        n += step_range(p, it, st, lo, hi);
    }
    return n;
}

// Persistent: each CTA (one per SM) takes work items blockIdx.x,
// blockIdx.x + gridDim.x, ...  (heaviest first for causal calls, which claim
// their items dynamically); its TMA producer decodes each item once and
// publishes it to the other roles.  Barrier phases run on across items; the
// MMA issuer starts the next item's Q K^T while the softmax warps still write
// out the previous item's O, and the softmax warps set up the next item
// before that epilogue.
template <int D, int NK, int NV, int TC>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ AttnParams<TC> p, const __grid_constant__ CUtensorMap tmQ,
                const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const __grid_constant__ CUtensorMap tmO)
{
    using L = Smem<D, NK, NV>;
    static_assert(L::kOffStage % 1024 == 0, "128-byte swizzled staging needs 1024-byte alignment");
    constexpr int NE = L::NE;
    constexpr int NBOX = D / 64;  // 128-byte swizzle columns per row
    // tensor-memory columns of S_t and O_t
    auto col_s = [](int t) { return (uint32_t)(t * 128); };
    auto col_o = [](int t) { return (uint32_t)(256 + t * D); };
    // cta_group::1 kind::f16: M = 128, N a multiple of 16 up to 256
    static_assert(kTileRows == 128 && kTileKeys % 16 == 0 && kTileKeys <= 256 && D % 16 == 0 && D <= 256,
                  "MMA shape");
    constexpr uint32_t kIdescQK = idesc_bf16_f32(kTileRows, kTileKeys, false);
    constexpr uint32_t kIdescPV = idesc_bf16_f32(kTileRows, D, true);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sQ = smem + L::kOffQ;
    uint8_t *sK = smem + L::kOffK;
    uint8_t *sV = smem + L::kOffV;
    uint64_t *bars = (uint64_t *)(smem + L::kOffBar);
    uint64_t *q_full = bars;  // [2]: Q tile t of the current item has landed
    uint64_t *k_full = q_full + 2;
    uint64_t *v_full = k_full + NK;
    // kv_free[g % NE], phase g / NE: the CTA's tile-iteration g (counted across
    // its items) is done -- S of the item's last tile is computed, so K(g) and
    // V(g-1) are no longer read, nor Q once g is an item's last iteration.
    // A softmax thread that waits on s_full anyway forwards it: a
    // tcgen05.commit costs the MMA issuer about as much as an MMA, so the
    // issuer commits only s_full and o_full.
    uint64_t *kv_free = v_full + NV;
    uint64_t *s_full = kv_free + NE;
    uint64_t *p_full = s_full + 2;
    uint64_t *o_full = p_full + 2;
    uint64_t *o_free = o_full + 2;  // O_t read out by the softmax warps
    uint64_t *mma_done = o_free + 2;  // every MMA the issuer issued has completed (exit)
    // work items: item_full[s] = the producer published ring slot s;
    // item_empty[s] = the MMA warp and the 8 softmax warps have read it
    uint64_t *item_full = mma_done + 1;
    uint64_t *item_empty = item_full + kItemSlots;
    ItemSlot *item_ring = (ItemSlot *)(smem + L::kOffRing);
    uint32_t *tmem_slot = (uint32_t *)(smem + L::kOffMisc);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const Ctl ctl{p.wait_ns, abort_flag};
    const long long n_items = p.g.n_items;
    const bool dyn = p.item_counter != nullptr;
    // Item k of this CTA on the consumer side, as the producer published it
    // in ring slot k % kItemSlots.  false past the end of the CTA's work, or
    // when the wait gave up (ok_ is then false).
    auto take_item = [&](int k, bool &ok_, uint32_t site, int lane_, ItemSlot &out) -> bool {
        const int slot = k % kItemSlots;
        const bool got = wait_phase(item_full + slot, (uint32_t)(k / kItemSlots) & 1u, ctl, site);
        if (!__all_sync(0xffffffffu, got)) {
            ok_ = false;
            return false;
        }
        out = item_ring[slot];
        __syncwarp();
        if (lane_ == 0)
            mbar_arrive(item_empty + slot);
        return out.has != 0;
    };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_full + 1, 1);
        for (int i = 0; i < NK; ++i)
            mbar_init(k_full + i, 1);
        for (int i = 0; i < NV; ++i)
            mbar_init(v_full + i, 1);
        for (int i = 0; i < NE; ++i)
            mbar_init(kv_free + i, 1);
        for (int t = 0; t < 2; ++t) {
            mbar_init(s_full + t, 1);
            mbar_init(p_full + t, 128);
            mbar_init(o_full + t, 1);
            mbar_init(o_free + t, 4);  // one arrive per softmax warp
        }
        mbar_init(mma_done, 1);
        for (int i = 0; i < kItemSlots; ++i) {
            mbar_init(item_full + i, 1);
            mbar_init(item_empty + i, 9);  // the MMA warp and the 8 softmax warps
        }
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // Each role sets its register budget inside its own branch and leaves
    // through its own copy of the exit barrier, so no code runs under two
    // budgets.  Warps 2-3 only give registers away.
    if (warp < 4) {
        regs_dec<kRegsProducer>();
        const uint32_t tmem = *tmem_slot;
        if (warp == 0 && lane == 0) {
            // --------------------------------------------------- TMA producer
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            int g = 0;  // tile-iterations issued so far by this CTA
            int nq0 = 0, nq1 = 0, nk = 0, nv = 0;  // Q tile 0 / 1, K and V loads issued (barrier phases)
            bool ok = true;
            for (int k = 0; ok; ++k) {
                // this CTA's item k: round robin, or (dynamic) claimed from the
                // launch's counter after the first and published to the other roles
                long long idx = blockIdx.x + (long long)k * gridDim.x;
                if (dyn && k > 0)
                    idx = (long long)gridDim.x + atomicAdd(p.item_counter, 1u);
                if (idx >= n_items)
                    idx = -1;
                const int slot = k % kItemSlots;
                if (k >= kItemSlots &&
                    !wait_phase(item_empty + slot, (uint32_t)(k / kItemSlots - 1) & 1u, ctl, 0x104)) {
                    ok = false;
                    break;
                }
                Item it{};
                int ntot = 0;
                if (idx >= 0) {
                    it = decode_item(p.g, idx);
                    ntot = item_tiles(p, it);
                }
                ItemSlot &pub = item_ring[slot];
                pub.has = idx >= 0 ? 1 : 0;
                pub.ntot = ntot;
                pub.it = it;
                mbar_arrive(item_full + slot);
                if (idx < 0)
                    break;
                if (ntot == 0)
                    continue;
                const int ntile = it.t[1].valid ? 2 : 1;
                // the Q buffer is free once the previous item's last iteration is done
                if (g > 0 && !wait_phase(kv_free + (g - 1) % NE, ((g - 1) / NE) & 1, ctl, 0x103)) {
                    ok = false;
                    break;
                }
                if (kChecked) {
                    // each Q box: Gp heads x Mq rows x 64 columns; its heads must
                    // be the item's batch's, its first row inside the sequence
                    bool good = true;
                    for (int t = 0; t < ntile; ++t)
                        good = good && it.t[t].h0 + p.g.Gp <= p.g.Hq &&
                               tma_coords_ok((NBOX - 1) * 64, it.t[t].q0, it.b * (long long)p.g.Hq + it.t[t].h0,
                                             D, p.g.Sq, (long long)p.g.B * p.g.Hq, 0);
                    if (!good) {
                        record_bounds(0x501);
                        *abort_flag = 1u;
                        ok = false;
                        break;
                    }
                }
                // Q tile 0 now and tile 1 right after the item's first K tile:
                // the item's first Q K^T then waits for one Q tile and one K tile
                // rather than both Q tiles ahead of the K tile
                mbar_arrive_expect_tx(q_full, (uint32_t)L::kQBytes);
                for (int c = 0; c < NBOX; ++c)
                    tma_load_3d(sQ + c * L::kBoxBytes, &tmQ, q_full, c * 64, it.t[0].q0,
                                it.b * p.g.Hq + it.t[0].h0);
                ++nq0;
                bool q1_pending = ntile == 2;
                const int bkv = it.b * p.g.Hkv + it.hkv;
                const int nsteps = item_steps(p.g, it);
                for (int st = 0; st < nsteps && ok; ++st) {
                    int lo, hi;
                    const int nt = step_range(p, it, st, lo, hi);
                    for (int tt = 0; tt < nt; ++tt, ++g) {
                        const int k0 = lo + tt * kTileKeys;
                        if (kChecked && !tma_coords_ok((NBOX - 1) * 64, k0, bkv, D, p.g.Skv,
                                                       (long long)p.g.B * p.g.Hkv, 0)) {
                            record_bounds(0x502);
                            *abort_flag = 1u;
                            ok = false;
                            break;
                        }
                        // stage g % NK held K(g - NK): free once iteration g - NK is done
                        const int ek = g - NK;
                        if (ek >= 0 && !wait_phase(kv_free + ek % NE, (ek / NE) & 1, ctl, 0x101)) {
                            ok = false;
                            break;
                        }
                        const int sk = g % NK;
                        mbar_arrive_expect_tx(k_full + sk, (uint32_t)L::kKVBytes);
                        for (int c = 0; c < NBOX; ++c)
                            tma_load_3d(sK + sk * L::kKVBytes + c * L::kBoxBytes, &tmK, k_full + sk, c * 64,
                                        k0, bkv);
                        ++nk;
                        if (q1_pending) {
                            mbar_arrive_expect_tx(q_full + 1, (uint32_t)L::kQBytes);
                            for (int c = 0; c < NBOX; ++c)
                                tma_load_3d(sQ + L::kQBytes + c * L::kBoxBytes, &tmQ, q_full + 1, c * 64,
                                            it.t[1].q0, it.b * p.g.Hq + it.t[1].h0);
                            ++nq1;
                            q1_pending = false;
                        }
                        // stage g % NV held V(g - NV): free once iteration g - NV + 1 is done
                        const int ev = g - NV + 1;
                        if (g >= NV && !wait_phase(kv_free + ev % NE, (ev / NE) & 1, ctl, 0x102)) {
                            ok = false;
                            break;
                        }
                        const int sv = g % NV;
                        mbar_arrive_expect_tx(v_full + sv, (uint32_t)L::kKVBytes);
                        for (int c = 0; c < NBOX; ++c)
                            tma_load_3d(sV + sv * L::kKVBytes + c * L::kBoxBytes, &tmV, v_full + sv, c * 64,
                                        k0, bkv);
                        ++nv;
                    }
                }
            }
            // Before the CTA may leave, every load issued into its shared
            // memory must have landed (after an abort some may still be in
            // flight).  The last load of a stage is the newest phase of its
            // barrier, so waiting for that phase covers the stage.
            for (int s = 0; s < NK; ++s)
                if (nk > s) {
                    const int last = nk - 1 - ((nk - 1 - s) % NK);
                    drain_phase(k_full + s, (last / NK) & 1, ctl, 0x111);
                }
            for (int s = 0; s < NV; ++s)
                if (nv > s) {
                    const int last = nv - 1 - ((nv - 1 - s) % NV);
                    drain_phase(v_full + s, (last / NV) & 1, ctl, 0x112);
                }
            if (nq0 > 0)
                drain_phase(q_full, (nq0 - 1) & 1, ctl, 0x113);
            if (nq1 > 0)
                drain_phase(q_full + 1, (nq1 - 1) & 1, ctl, 0x114);
        } else if (warp == 1) {
            // --------------------------------------------------- MMA issuer
            // The whole warp runs this loop (its waits and descriptor
            // arithmetic stay warp-uniform); one elected lane issues each
            // tcgen05 instruction.
            // Descriptors: the address field (bits 0-13, bytes >> 4) of a base
            // descriptor plus a constant offset never carries out of the field
            // (shared memory < 256 KB), so stepping is one add.
            const uint32_t leader = elect_lane();  // the lane that issues
            const uint64_t dq = smem_desc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dk = smem_desc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t dv = smem_desc_sw128(smem_u32(sV), L::kBoxBytes, 1024);
            // S_t = Q_t K^T over K = D: 16 elements (32 bytes) per MMA inside a
            // 128-byte swizzle column; 8-row groups 1024 bytes apart.
            auto issue_qk = [&](int t, int sk) {
                const uint64_t da = dq + ((uint32_t)(t * L::kQBytes) >> 4);
                const uint64_t db = dk + ((uint32_t)(sk * L::kKVBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk / 4) * L::kBoxBytes + (kk % 4) * 32) >> 4;
                    umma_ss_w(tmem + col_s(t), da + off, db + off, kIdescQK, kk > 0 ? 1u : 0u, leader);
                }
            };
            // O_t += P_t V over K = 128 keys: P_t from tensor memory (bf16 pairs,
            // 8 columns per 16 keys); V is MN-major (d contiguous): 16 keys =
            // two 8-row groups = 2048 bytes; the two 64-wide d halves are
            // kBoxBytes apart (leading-dimension offset).
            auto issue_pv = [&](int t, int sv, bool acc_in) {
                const uint64_t db = dv + ((uint32_t)(sv * L::kKVBytes) >> 4);
#pragma unroll
                for (int kk = 0; kk < kTileKeys / 16; ++kk)
                    umma_ts_w(tmem + col_o(t), tmem + col_s(t) + kk * 8, db + (uint32_t)(kk * (2048 >> 4)),
                            kIdescPV, (acc_in || kk > 0) ? 1u : 0u, leader);
            };
            int g = 0;                  // tile-iterations of this CTA so far
            int nq0 = 0, nq1 = 0;       // Q tile 0 / tile 1 loads consumed (q_full phases)
            int sp[2] = {0, 0};         // S_t / P_t phases so far, per tile
            int od[2] = {0, 0};         // O_t finalisations so far, per tile
            bool ok = true;
            for (int k = 0; ok; ++k) {
                ItemSlot cur;
                if (!take_item(k, ok, 0x206, lane, cur))
                    break;
                const int ntot = cur.ntot;
                if (ntot == 0)
                    continue;
                const int ntile = cur.it.t[1].valid ? 2 : 1;
                ok = wait_phase(q_full, nq0 & 1, ctl, 0x201);
                ++nq0;
                tc_fence_after();
                // iteration n issues P.V of n-1 (n >= 1) and Q K^T of n (n < ntot)
                for (int n = 0; n <= ntot && ok; ++n) {
                    const int sk = g % NK;
                    if (n < ntot) {
                        if (!wait_phase(k_full + sk, (g / NK) & 1, ctl, 0x202)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if (n == 0) {
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            if (t >= ntile || !ok)
                                break;
                            if (t == 1) {
                                // tile 1's Q follows the item's first K tile
                                if (!wait_phase(q_full + 1, nq1 & 1, ctl, 0x208)) {
                                    ok = false;
                                    break;
                                }
                                ++nq1;
                                tc_fence_after();
                            }
                            issue_qk(t, sk);
                            umma_commit_w(s_full + t, leader);
                            ++sp[t];
                        }
                    } else {
                        const int gv = g - 1;  // V of the previous iteration
                        const int sv = gv % NV;
                        if (!wait_phase(v_full + sv, (gv / NV) & 1, ctl, 0x204)) {
                            ok = false;
                            break;
                        }
                        // t unrolled: sp[] and od[] stay in registers
#pragma unroll
                        for (int t = 0; t < 2; ++t) {
                            if (t >= ntile || !ok)
                                break;
                            if (!wait_phase(p_full + t, (sp[t] - 1) & 1, ctl, 0x203)) {
                                ok = false;
                                break;
                            }
                            // the item's first P.V overwrites O_t: the softmax warps
                            // must have read out the previous item's O_t
                            if (n == 1 && od[t] > 0 &&
                                !wait_phase(o_free + t, (od[t] - 1) & 1, ctl, 0x205)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            issue_pv(t, sv, n > 1);
                            if (n < ntot) {
                                issue_qk(t, sk);
                                umma_commit_w(s_full + t, leader);
                                ++sp[t];
                            } else {
                                umma_commit_w(o_full + t, leader);
                                ++od[t];
                            }
                        }
                    }
                    if (n < ntot)
                        ++g;
                }
            }
            // Every MMA this warp issued must complete before the tensor
            // memory it writes is freed (after an abort some may be in flight).
            umma_commit_w(mma_done, leader);
            drain_phase(mma_done, 0, ctl, 0x211);
            // and the arrives of its earlier commits must have landed
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (sp[t] > 0)
                    drain_phase(s_full + t, (sp[t] - 1) & 1, ctl, 0x212);
                if (od[t] > 0)
                    drain_phase(o_full + t, (od[t] - 1) & 1, ctl, 0x213);
            }
        }
        tc_fence_before();
        named_barrier_sync(kExitBarrier, kThreads);
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, kTmemCols);
        }
    } else {
        regs_inc<kRegsSoftmax>();
        const uint32_t tmem = *tmem_slot;
        // ------------------------------------------------------- softmax
        const int t = (warp - 4) / 4;
        const int quarter = warp % 4;  // tcgen05.ld lane quarter of this warp
        const int r = quarter * 32 + lane;
        const uint32_t lane_field = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_field + col_s(t);
        const uint32_t tO = tmem + lane_field + col_o(t);
        const float scale = p.scale_log2;
        const uint64_t scale2 = f2_pack(scale, scale);
        int g = 0;   // tile-iterations of this CTA so far (all tiles)
        int sp = 0;  // S_t / P_t phases of this tile so far
        int od = 0;  // O_t finalisations of this tile so far
        bool ok = true;
        // Row set-up of this thread's row in a work item (its tile t).
        struct Rows {
            int ntot, ntile;
            float *orow;     // O row (nullptr: padding row, or skipped by the checked build)
            float *lrow;     // LSE element
            int causal_lim;  // last allowed key of the row (inclusive) under the causal mask
        };
        auto setup_rows = [&](const ItemSlot &c) -> Rows {
            Rows w;
            w.ntot = c.ntot;
            w.ntile = c.it.t[1].valid ? 2 : 1;
            w.orow = nullptr;
            w.lrow = nullptr;
            w.causal_lim = 0x7fffffff;
            if (t >= w.ntile)
                return w;
            const Tile T = t == 0 ? c.it.t[0] : c.it.t[1];
            const int head = T.h0 + r / p.g.Mq;
            const int qi = T.q0 + r % p.g.Mq;
            if ((r % p.g.Mq) < T.nq) {
                long long row = ((long long)c.it.b * p.g.Hq + head) * p.g.Sq + qi;
                long long so = 0, sl = 0;
                if (p.g.partial != kFused) {
                    const int slot = out_slot(p, c.it);
                    so = slot * p.slot_o;
                    sl = slot * p.slot_lse;
                }
                w.orow = p.out + so + row * D;
                w.lrow = p.lse + sl + row;
                if (kChecked) {
                    // element offsets (O may hold bf16 elements: same offsets)
                    const long long oo = so + row * D, lo_ = sl + row;
                    if (oo < 0 || oo + D > p.out_elems || lo_ < 0 || lo_ >= p.lse_elems) {
                        record_bounds(0x503);
                        w.orow = nullptr;
                        w.lrow = nullptr;
                    }
                }
            }
            if (p.g.causal)
                w.causal_lim = qi + (p.g.Skv - p.g.Sq);
            return w;
        };
        // The next item is taken and set up, and this item's LSE stored, while
        // the tensor cores finish the item's last P.V: the epilogue then runs
        // straight into the next item's first S.
        ItemSlot cur;
        bool have = take_item(0, ok, 0x303, lane, cur);
        Rows rw = have ? setup_rows(cur) : Rows{};
        for (int k = 0; have && ok; ++k) {
            // the fields the step loop reads: the rest of cur is not kept live
            // across the tiles
            Item it{};
            it.rank = cur.it.rank;
            it.shard = cur.it.shard;
            it.kv_end = cur.it.kv_end;
            const int ntot = rw.ntot;
            const int ntile = rw.ntile;
            if (t >= ntile) {
                g += ntot;
                have = take_item(k + 1, ok, 0x303, lane, cur);
                if (have)
                    rw = setup_rows(cur);
                continue;
            }
            if (ntot == 0) {
                // no allowed key for any row of this item in this shard
                if (rw.orow) {
                    float4 *dst = reinterpret_cast<float4 *>(rw.orow);
                    for (int c = 0; c < D / 4; ++c)
                        dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
                    *rw.lrow = -INFINITY;
                }
                have = take_item(k + 1, ok, 0x303, lane, cur);
                if (have)
                    rw = setup_rows(cur);
                continue;
            }
            const int causal_lim = rw.causal_lim;
            const bool forwards = (t == ntile - 1) && r == 0;  // reports iteration done
            float m = -INFINITY;  // running max (log2 domain), possibly stale by < 2^8
            float l = 0.f;        // running sum of 2^(y - m)
            int n = 0;
            const int nsteps = item_steps(p.g, it);
            for (int st = 0; st < nsteps && ok; ++st) {
                int lo, hi;
                const int nt = step_range(p, it, st, lo, hi);
                // allowed keys of this row in this step: k <= lim_abs
                const int lim_abs = min(hi - 1, causal_lim);
                for (int tt = 0; tt < nt; ++tt, ++n) {
                    const int lim = lim_abs - (lo + tt * kTileKeys);  // allowed columns c <= lim
                    bool got = wait_phase(s_full + t, sp & 1, ctl, 0x301);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        break;
                    }
                    ++sp;
                    tc_fence_after();
                    if (forwards && !(p.fault == 2 && g + n == 0))
                        mbar_arrive(kv_free + (g + n) % NE);
                    uint32_t sr[128];
                    tmem_ld_x32x4(tS, sr);
                    float *s = reinterpret_cast<float *>(sr);
                    if (lim < kTileKeys - 1) {
#pragma unroll
                        for (int c = 0; c < 128; ++c)
                            if (c > lim)
                                s[c] = -INFINITY;
                    }
                    // p = 2^(s*scale - mu): packed FMA, ex2 per element, packed
                    // partial sums in four chains; bf16 pairs for the P.V MMA are
                    // stored to tensor memory 16 columns (32 keys) at a time.
                    // Returns the tile's sum of p.
                    auto exp_pass = [&](float mu_) -> float {
                        const uint64_t nmu2 = f2_pack(-mu_, -mu_);
                        uint64_t acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
#pragma unroll
                        for (int cb = 0; cb < 64; cb += 16) {
                            uint32_t pk[16];
#pragma unroll
                            for (int c = 0; c < 16; c += 4) {
                                uint64_t pp[4];
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const int e = 2 * (cb + c + u);
                                    const uint64_t x = f2_fma(f2_pack(s[e], s[e + 1]), scale2, nmu2);
                                    float x0, x1;
                                    f2_unpack(x, x0, x1);
                                    const float p0 = ex2_approx(x0);
                                    const float p1 = ex2_approx(x1);
                                    pp[u] = f2_pack(p0, p1);
                                    __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);  // low half = p0
                                    pk[c + u] = *reinterpret_cast<uint32_t *>(&h2);
                                }
                                acc0 = f2_add(acc0, pp[0]);
                                acc1 = f2_add(acc1, pp[1]);
                                acc2 = f2_add(acc2, pp[2]);
                                acc3 = f2_add(acc3, pp[3]);
                            }
                            tmem_st_x16(tS + cb, pk);
                        }
                        float a0, a1, b0, b1, c0, c1, d0, d1;
                        f2_unpack(acc0, a0, a1);
                        f2_unpack(acc1, b0, b1);
                        f2_unpack(acc2, c0, c1);
                        f2_unpack(acc3, d0, d1);
                        return ((a0 + a1) + (b0 + b1)) + ((c0 + c1) + (d0 + d1));
                    };
                    // The running max m moves only when a tile's max exceeds it by
                    // more than 2^8.  After the first tile the exponentials are
                    // taken with the current m straight away: if every p <= 2^8
                    // (their sum <= 2^8 implies it) m would not have moved and the
                    // tile is done.  Otherwise (rare) the row max is taken, O and
                    // l are rescaled if m moves, and the tile is redone -- the
                    // same arithmetic as taking the max first, without the max on
                    // the common path.
                    float tile_l = 0.f;
                    bool exact = n == 0;
                    if (!exact) {
                        tile_l = exp_pass(m == -INFINITY ? 0.f : m);
                        exact = __any_sync(0xffffffffu, !(tile_l <= kRescaleFactor));
                        if (exact)
                            tmem_st_wait();  // the first pass's P stores land before they are replaced
                    }
                    if (exact) {
                        // row max: four independent 3-input chains
                        float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
                        float mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
                        for (int c = 8; c < 128; c += 8) {
                            mx0 = max3f(mx0, s[c], s[c + 1]);
                            mx1 = max3f(mx1, s[c + 2], s[c + 3]);
                            mx2 = max3f(mx2, s[c + 4], s[c + 5]);
                            mx3 = max3f(mx3, s[c + 6], s[c + 7]);
                        }
                        const float mx = max3f(mx0, mx1, fmaxf(mx2, mx3));
                        const float m_cand = fmaxf(m, mx * scale);
                        const bool need = (m == -INFINITY) ? (m_cand != -INFINITY)
                                                           : (m_cand - m > kRescaleThreshold);
                        const float m_new = need ? m_cand : m;
                        __syncwarp();
                        if (n > 0 && __any_sync(0xffffffffu, need)) {
                            const float alpha = need ? ex2_approx(m - m_new) : 1.f;
                            l *= alpha;
                            const uint64_t alpha2 = f2_pack(alpha, alpha);
#pragma unroll 1
                            for (int c0 = 0; c0 < D; c0 += 32) {
                                uint32_t o[32];
                                tmem_ld_x32(tO + c0, o);
#pragma unroll
                                for (int c = 0; c < 32; c += 2) {
                                    uint64_t v2 = f2_mul(f2_pack(__uint_as_float(o[c]), __uint_as_float(o[c + 1])),
                                                         alpha2);
                                    float a, b;
                                    f2_unpack(v2, a, b);
                                    o[c] = __float_as_uint(a);
                                    o[c + 1] = __float_as_uint(b);
                                }
                                tmem_st_x32(tO + c0, o);
                            }
                        }
                        m = m_new;
                        tile_l = exp_pass(m == -INFINITY ? 0.f : m);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    if (!(p.fault == 1 && t == 0 && n == 0))
                        mbar_arrive(p_full + t);
                    l += tile_l;
                }
            }
            g += ntot;
            if (!ok)
                break;
            if (rw.lrow)
                *rw.lrow = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
            float *const orow = rw.orow;
            have = take_item(k + 1, ok, 0x303, lane, cur);
            if (!ok)
                break;
            if (have)
                rw = setup_rows(cur);
            // ------------------------------------------------- epilogue
            bool got = wait_phase(o_full + t, od & 1, ctl, 0x302);
            ok = __all_sync(0xffffffffu, got);
            if (!ok)
                break;
            ++od;
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            // When this warp's 32 rows are 32 consecutive rows of O (one head,
            // all valid), each 32-column chunk goes through the warp's 4 KB of
            // shared memory (lane = row, 128-byte swizzle: conflict-free) and
            // one TMA tensor store, instead of 32 row-strided stores per
            // instruction -- the epilogue sits between two work items.
            const bool tma_rows = p.o_tma && p.g.Mq >= 32 && __all_sync(0xffffffffu, orow != nullptr);
            if (tma_rows) {
                const long long off0 = __shfl_sync(0xffffffffu, (long long)(orow - p.out), 0);
                const int y0 = (int)(off0 / D);
                uint8_t *stage = smem + L::kOffStage + (warp - 4) * L::kStageBytes;
                const uint32_t srow = smem_u32(stage) + lane * 128;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld_x32(tO + c0, o);
                    if (lane == 0)
                        bulk_wait_read_all();  // the previous store has read the staging rows
                    __syncwarp();
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_shared_v4(srow + ((c ^ (lane & 7)) << 4),
                                     __float_as_uint(__uint_as_float(o[4 * c]) * inv),
                                     __float_as_uint(__uint_as_float(o[4 * c + 1]) * inv),
                                     __float_as_uint(__uint_as_float(o[4 * c + 2]) * inv),
                                     __float_as_uint(__uint_as_float(o[4 * c + 3]) * inv));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (kChecked && (y0 < 0 || (long long)y0 + 32 > p.o_rows || c0 + 32 > D)) {
                            record_bounds(0x504);
                        } else {
                            tma_store_2d(&tmO, stage, c0, y0);
                            bulk_commit_group();
                        }
                    }
                }
            } else {
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld_x32(tO + c0, o);
                    // Each lane stores its own row; 32-byte stores (one whole sector
                    // per lane) need half the store instructions and L1 wavefronts
                    // of 16-byte ones, and this loop is bound by them.
                    if (orow && p.out_bf16) {
                        // the row's bf16 elements sit at half the fp32 offset
                        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + (orow - p.out) + c0;
                        uint32_t w[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(o[2 * e]) * inv,
                                                                      __uint_as_float(o[2 * e + 1]) * inv);
                            w[e] = *reinterpret_cast<uint32_t *>(&h2);
                        }
                        if (p.out_v8) {
#pragma unroll
                            for (int c = 0; c < 2; ++c)
                                st_global_v8(dst + 16 * c, w[8 * c], w[8 * c + 1], w[8 * c + 2], w[8 * c + 3],
                                             w[8 * c + 4], w[8 * c + 5], w[8 * c + 6], w[8 * c + 7]);
                        } else {
                            uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                d4[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
                        }
                    } else if (orow) {
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            o[c] = __float_as_uint(__uint_as_float(o[c]) * inv);
                        if (p.out_v8) {
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                st_global_v8(orow + c0 + 8 * c, o[8 * c], o[8 * c + 1], o[8 * c + 2], o[8 * c + 3],
                                             o[8 * c + 4], o[8 * c + 5], o[8 * c + 6], o[8 * c + 7]);
                        } else {
                            float4 *dst = reinterpret_cast<float4 *>(orow + c0);
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                dst[c] = make_float4(__uint_as_float(o[4 * c]), __uint_as_float(o[4 * c + 1]),
                                                     __uint_as_float(o[4 * c + 2]), __uint_as_float(o[4 * c + 3]));
                        }
                    }
                }
            }
            // O_t is read: the next item's first P.V may overwrite it
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(o_free + t);
        }
        // the O tensor stores this warp issued complete before the CTA leaves
        if (lane == 0)
            bulk_wait_all();
        tc_fence_before();
        named_barrier_sync(kExitBarrier, kThreads);
    }
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

EncodeFn get_encode_fn(char *msg, size_t msg_len)
{
    // looked up once (thread-safe static initialisation)
    static const EncodeFn fn = []() -> EncodeFn {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                                         cudaEnableDefault, &q);
        return (e == cudaSuccess && q == cudaDriverEntryPointSuccess) ? (EncodeFn)ptr : nullptr;
    }();
    if (!fn)
        snprintf(msg, msg_len, "cuTensorMapEncodeTiled is not available from the driver");
    return fn;
}

// 2-D fp32 tensor [d1][d0] (d0 innermost), box {b0, b1}, 128-byte swizzle:
// the epilogue's O stores.
int encode_2d_f32(CUtensorMap *m, void *base, uint64_t d0, uint64_t d1, uint32_t b0, uint32_t b1, char *msg,
                  size_t msg_len)
{
    EncodeFn fn = get_encode_fn(msg, msg_len);
    if (!fn)
        return MERCURY_ECUDA;
    cuuint64_t dims[2] = {d0, d1};
    cuuint64_t strides[1] = {d0 * 4};
    cuuint32_t box[2] = {b0, b1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(msg, msg_len, "cuTensorMapEncodeTiled (O) failed (CUresult %d)", (int)r);
        return MERCURY_ECUDA;
    }
    return MERCURY_OK;
}

// 3-D bf16 tensor [d2][d1][d0] (d0 innermost), 128-byte swizzle, zero fill.
int encode_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0,
              uint32_t b1, uint32_t b2, char *msg, size_t msg_len)
{
    EncodeFn fn = get_encode_fn(msg, msg_len);
    if (!fn)
        return MERCURY_ECUDA;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {d0 * 2, d0 * d1 * 2};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        snprintf(msg, msg_len, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
        return MERCURY_ECUDA;
    }
    return MERCURY_OK;
}

// A zeroed work-item counter for one launch on `stream`: the next slot of
// g_item_counters (cycling through kItemCounterSlots), cleared by a memset
// ordered before the launch.  The array's device address is looked up once
// per device.
int claim_item_counter(cudaStream_t stream, unsigned int **out, char *msg, size_t msg_len)
{
    static std::mutex mu;
    static unsigned int *base[64] = {};
    static std::atomic<unsigned int> next{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        snprintf(msg, msg_len, "cudaGetDevice: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    unsigned int *b = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!base[dev]) {
            void *ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_item_counters);
            if (e != cudaSuccess || !ptr) {
                snprintf(msg, msg_len, "cudaGetSymbolAddress(item counters): %s", cudaGetErrorString(e));
                return MERCURY_ECUDA;
            }
            base[dev] = (unsigned int *)ptr;
        }
        b = base[dev];
    }
    unsigned int *c = b + (next.fetch_add(1u, std::memory_order_relaxed) % kItemCounterSlots);
    e = cudaMemsetAsync(c, 0, sizeof(unsigned int), stream);
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "clearing the work-item counter: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    *out = c;
    return MERCURY_OK;
}

template <int D, int NK, int NV, int TC>
int launch_impl(AttnParams<TC> &p, const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                const CUtensorMap &mo, cudaStream_t stream, char *msg, size_t msg_len)
{
    using L = Smem<D, NK, NV>;
    auto kern = attn_fwd_kernel<D, NK, NV, TC>;
    KernelInfo ki;
    int rc = prepare_kernel((const void *)kern, L::kAlloc, &ki, msg, msg_len);
    if (rc != MERCURY_OK)
        return rc;
    // setmaxnreg.inc would wait for registers that the launch does not have
    if (ki.regs < kMinLaunchRegs) {
        snprintf(msg, msg_len, "kernel built with %d registers/thread, the register split needs %d", ki.regs,
                 kMinLaunchRegs);
        return MERCURY_ECUDA;
    }
    if (p.g.n_items > 0x7fffffffLL) {
        snprintf(msg, msg_len, "too many work items (%lld)", p.g.n_items);
        return MERCURY_EINVAL;
    }
    const int sms = ki.sms;
    // persistent: one CTA per SM (the shared memory and TMEM use allow one)
    const long long grid = p.g.n_items < sms ? p.g.n_items : sms;
    if (grid < 1)
        return MERCURY_OK;
    // Causal items differ in length (a block sees up to its diagonal): with
    // more items than CTAs, each CTA takes its next item when it is free
    // (items stay in their heaviest-first, head-by-head order), instead of
    // every grid-th one -- round robin left the busiest CTA 8-11 % above the
    // mean on 8K-32K causal shapes.
    p.item_counter = nullptr;
    if (p.g.causal && p.g.n_items > grid) {
        rc = claim_item_counter(stream, &p.item_counter, msg, msg_len);
        if (rc != MERCURY_OK)
            return rc;
    }
    kern<<<(unsigned)grid, kThreads, L::kAlloc, stream>>>(p, mq, mk, mv, mo);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "attention kernel launch: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    return MERCURY_OK;
}

}  // namespace

template <int TC>
int launch_with_table(const AttnCall &c, cudaStream_t stream, char *msg, size_t msg_len)
{
    // The parameter block and the planner's table live in thread-local
    // storage: the launch path makes no heap allocation.
    static thread_local AttnParams<TC> p;
    static thread_local int order[kMaxR * kMaxR];
    memset(&p, 0, sizeof p);
    if (c.R < 1 || c.R > TC || plan_shift(c.R, c.shift, order)) {
        snprintf(msg, msg_len, "invalid (R, shift) = (%d, %d)", c.R, c.shift);
        return MERCURY_EINVAL;
    }
    if (make_geom(p.g, c.B, c.Hq, c.Hkv, c.Sq, c.Skv, c.d, c.R, c.causal, c.mode, c.n_groups, c.Rq)) {
        snprintf(msg, msg_len, "unsupported shape");
        return MERCURY_EINVAL;
    }
    p.scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.d));
    p.fault = c.fault;
    p.out_bf16 = c.out_bf16;
    p.out_v8 = ((uintptr_t)c.out % 32) == 0 ? 1 : 0;
    p.out = c.out;
    p.lse = c.lse;
    p.slot_o = (long long)c.B * c.Hq * c.Sq * c.d;
    p.slot_lse = (long long)c.B * c.Hq * c.Sq;
    const int slots = c.mode == kFused ? 1 : p.g.n_groups;
    p.out_elems = slots * p.slot_o;
    p.lse_elems = slots * p.slot_lse;
    p.o_rows = slots * p.slot_lse;
    // fp32 O goes out through TMA tensor stores (32 fp32 = 128 bytes per box
    // row; every row starts 16-byte aligned since d is 64 or 128)
    p.o_tma = (!c.out_bf16 && p.o_rows < 0x7fffffffLL) ? 1 : 0;
    p.wait_ns = c.wait_ns;
    const int R = c.R;
    for (int i = 0; i < R; ++i)
        for (int j = 0; j < R; ++j) {
            const int s = order[i * R + j];
            if (c.mode == kPerStep)
                p.tab[i * R + s] = (unsigned char)j;
            else
                p.tab[i * R + j] = (unsigned char)s;
        }
    CUtensorMap mq, mk, mv;
    int rc = encode_3d(&mq, c.q, (uint64_t)c.d, (uint64_t)c.Sq, (uint64_t)c.B * c.Hq, 64, (uint32_t)p.g.Mq,
                       (uint32_t)p.g.Gp, msg, msg_len);
    if (rc == MERCURY_OK)
        rc = encode_3d(&mk, c.k, (uint64_t)c.d, (uint64_t)c.Skv, (uint64_t)c.B * c.Hkv, 64, kTileKeys, 1, msg,
                       msg_len);
    if (rc == MERCURY_OK)
        rc = encode_3d(&mv, c.v, (uint64_t)c.d, (uint64_t)c.Skv, (uint64_t)c.B * c.Hkv, 64, kTileKeys, 1, msg,
                       msg_len);
    CUtensorMap mo;
    memset(&mo, 0, sizeof mo);
    if (rc == MERCURY_OK && p.o_tma)
        rc = encode_2d_f32(&mo, c.out, (uint64_t)c.d, (uint64_t)p.o_rows, 32, 32, msg, msg_len);
    if (rc == MERCURY_OK) {
        if (c.d == 128)
            rc = launch_impl<128, 2, 2, TC>(p, mq, mk, mv, mo, stream, msg, msg_len);
        else
            rc = launch_impl<64, 4, 4, TC>(p, mq, mk, mv, mo, stream, msg, msg_len);
    }
    return rc;
}

int launch_attention(const AttnCall &c, cudaStream_t stream, char *msg, size_t msg_len)
{
    return c.R <= kSmallTab ? launch_with_table<kSmallTab>(c, stream, msg, msg_len)
                            : launch_with_table<kMaxR>(c, stream, msg, msg_len);
}

int read_and_clear_device_error(cudaStream_t stream, unsigned int *word, unsigned int *site, char *msg,
                                size_t msg_len)
{
    unsigned int zero = 0, w = 0, s = 0;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess)
        e = cudaMemcpyFromSymbol(&w, g_err_word, sizeof w);
    if (e == cudaSuccess)
        e = cudaMemcpyFromSymbol(&s, g_err_site, sizeof s);
    if (e == cudaSuccess && (w || s)) {
        e = cudaMemcpyToSymbol(g_err_word, &zero, sizeof zero);
        if (e == cudaSuccess)
            e = cudaMemcpyToSymbol(g_err_site, &zero, sizeof zero);
    }
    if (e != cudaSuccess) {
        snprintf(msg, msg_len, "reading the device error word: %s", cudaGetErrorString(e));
        return MERCURY_ECUDA;
    }
    *word = w;
    *site = s;
    return MERCURY_OK;
}

}  // namespace mercury
