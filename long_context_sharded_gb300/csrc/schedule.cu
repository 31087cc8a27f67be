// schedule.cu -- choosing a schedule of the sharded attention under a
// device-memory budget: the static filter, the cost estimate, the measured
// cost profile, and tuning by measurement with a per-process cache.
//
// The staged search follows the pages' description of how candidate
// schedules are narrowed (Silicon & Systems, "CommIR makes communication
// transformable": a static check of sizes and dependencies, then cost
// estimation, then profiling of the survivors on the target machine) and the
// latency / memory frontier they ask to keep (same page, "Memory capacity is
// part of performance"); the cache key and the re-check of a cached choice
// follow "The tuning bill".  Contracts are in include/mercury_attn.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <limits>
#include <map>
#include <mutex>
#include <stdio.h>
#include <stdlib.h>
#include <string>
#include <vector>

#include "internal.h"
#include "work.h"

using namespace mercury;

namespace {

long long input_output_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int d)
{
    const long long q = (long long)B * Hq * Sq * d * 2;
    const long long kv = 2LL * B * Hkv * Skv * d * 2;
    const long long o = (long long)B * Hq * Sq * d * 4;
    const long long l = (long long)B * Hq * Sq * 4;
    return q + kv + o + l;
}

long long scratch_bytes_of(int B, int Hq, int Sq, int d, int slots)
{
    return slots <= 1 ? 0 : (long long)slots * B * Hq * Sq * (d + 1) * 4;
}

// Mode of a run count, as mercury_attn_run_schedule maps it.
void mode_of(int R, int runs, int &mode, int &groups)
{
    mode = runs == 1 ? kFused : (runs >= R ? kPerStep : kGrouped);
    groups = runs >= R ? R : runs;
}

// K/V tiles of work item `it` over its steps (the kernel's own walk).
long long item_tiles(const Geom &g, const Item &it, const int *order)
{
    long long n = 0;
    const int ns = item_steps(g, it);
    for (int st = 0; st < ns; ++st) {
        int s;
        if (g.partial == kPerStep)
            s = it.shard;
        else
            s = order[it.rank * g.R + (g.partial == kGrouped ? it.shard * g.spg + st : st)];
        int lo, hi;
        shard_range(g, it, s, lo, hi);
        n += n_kv_tiles(lo, hi);
    }
    return n;
}

double item_cost(const Geom &g, const Item &it, const int *order, const mercury_cost_profile &p)
{
    const int valid = (it.t[0].valid ? 1 : 0) + (it.t[1].valid ? 1 : 0);
    const double per_tile = valid == 2 ? p.tile_us : p.tile1_us;
    return p.item_us + (double)item_tiles(g, it, order) * per_tile;
}

// Least HBM time of one launch: q, k, v read once; O and LSE (or every
// slot's partials) written once.
double traffic_floor_us(const Geom &g, const mercury_cost_profile &p)
{
    const double rows = (double)g.B * g.Hq * g.Sq;
    const double in = rows * g.d * 2.0 + 2.0 * g.B * g.Hkv * (double)g.Skv * g.d * 2.0;
    const double outb = (g.partial == kFused ? 1.0 : (double)g.n_groups) * rows * (g.d + 1) * 4.0;
    return (in + outb) / (p.hbm_gbs * 1e3);
}

// The costs of a launch's items in launch order, each computed once: an
// item's cost depends on its rows, rank, run and head pair but not on its
// batch or KV head, so fused items of one (batch, KV head) -- consecutive --
// repeat their costs with period NHP * NRT * Rq, and the other modes' items
// come in runs of NHP * Hkv * B that differ only by head pair.
class ItemCosts {
  public:
    ItemCosts(const Geom &g, const int *order, const mercury_cost_profile &p)
        : g_(g), order_(order), p_(p), fused_(g.partial == kFused),
          period_(fused_ ? (long long)g.NHP * g.NRT * g.Rq : 0),
          inner_((long long)g.NHP * g.Hkv * g.B), nhp_(std::min<int>(g.NHP, kMaxR))
    {
        if (fused_) {
            cost_.resize((size_t)std::min(period_, g.n_items));
            for (long long j = 0; j < (long long)cost_.size(); ++j)
                cost_[(size_t)j] = item_cost(g, decode_item(g, j), order, p);
        }
    }
    // cost of item i, called for i = 0, 1, 2, ... in turn
    double next(long long i)
    {
        double c;
        if (fused_) {
            c = cost_[(size_t)j_];
            if (++j_ == period_)
                j_ = 0;
            return c;
        }
        if (in_run_ < nhp_)
            run_cost_[in_run_] = item_cost(g_, decode_item(g_, i), order_, p_);
        c = hp_ < nhp_ ? run_cost_[hp_] : item_cost(g_, decode_item(g_, i), order_, p_);
        if (++hp_ == g_.NHP)
            hp_ = 0;
        if (++in_run_ == inner_) {
            in_run_ = 0;
            hp_ = 0;
        }
        return c;
    }

  private:
    const Geom &g_;
    const int *order_;
    const mercury_cost_profile &p_;
    bool fused_;
    long long period_, inner_;
    int nhp_;
    std::vector<double> cost_;
    double run_cost_[kMaxR];
    long long j_ = 0, in_run_ = 0;  // i % period, i % inner
    int hp_ = 0;                    // in_run % NHP
};

// A lower bound on launch_estimate: no launch ends before the average CTA's
// share of the item costs, its longest item or its least HBM traffic.
double launch_lower_bound(const Geom &g, const int *order, const mercury_cost_profile &p)
{
    const long long n = g.n_items;
    if (n <= 0)
        return p.launch_us;
    const long long grid = std::min<long long>(n, p.n_sms);
    ItemCosts ic(g, order, p);
    double sum = 0.0, longest = 0.0;
    for (long long i = 0; i < n; ++i) {
        const double c = ic.next(i);
        sum += c;
        longest = std::max(longest, c);
    }
    return p.launch_us + std::max(std::max(sum / (double)grid, longest), traffic_floor_us(g, p));
}

// Device time of one launch of geometry g on min(n_items, n_sms) persistent
// CTAs: the launch lasts as long as its busiest CTA, plus the launch cost.
// Items go round robin in launch order -- except in causal launches with
// more items than CTAs, where each CTA claims the next item when it becomes
// free (the kernel's dynamic scheduling): CTA i takes item i first, then each
// item goes to the CTA that is free earliest (ties: the lower index).
double launch_estimate(const Geom &g, const int *order, const mercury_cost_profile &p)
{
    const long long n = g.n_items;
    if (n <= 0)
        return p.launch_us;
    const long long grid = std::min<long long>(n, p.n_sms);
    if (g.causal && n > grid) {
        ItemCosts ic(g, order, p);
        // Winner tree over the CTAs: leaf c holds CTA c's busy-until time and
        // every inner node the CTA of its subtree that is free earliest (ties:
        // the lower index, which is always the left child's side).  The next
        // item goes to the root's CTA; only the path from that leaf up changes.
        // Padding leaves stay busy forever.
        int L = 1;
        while (L < grid)
            L <<= 1;
        std::vector<double> busy((size_t)L, std::numeric_limits<double>::infinity());
        std::vector<int> win(2 * (size_t)L);
        for (int c = 0; c < L; ++c) {
            if (c < grid)
                busy[(size_t)c] = 0.0;
            win[(size_t)(L + c)] = c;
        }
        auto better = [&](int a, int b) { return busy[(size_t)b] < busy[(size_t)a] ? b : a; };
        for (int k = L - 1; k >= 1; --k)
            win[(size_t)k] = better(win[(size_t)(2 * k)], win[(size_t)(2 * k + 1)]);
        double last = 0.0;
        for (long long i = 0; i < n; ++i) {
            const double c = ic.next(i);
            const int cta = win[1];
            const double t = busy[(size_t)cta] + c;
            busy[(size_t)cta] = t;
            last = std::max(last, t);
            for (int k = (L + cta) >> 1; k >= 1; k >>= 1)
                win[(size_t)k] = better(win[(size_t)(2 * k)], win[(size_t)(2 * k + 1)]);
        }
        return p.launch_us + std::max(last, traffic_floor_us(g, p));
    }
    std::vector<double> diff(grid + 1, 0.0);
    double everyone = 0.0;
    // Otherwise items sharing (row tile, rank, slot) sit in runs of NHP*Hkv*B
    // consecutive indices; their cost differs only through the head pair
    // (an odd number of head tiles leaves the last pair with one tile).
    const long long inner = (long long)g.NHP * g.Hkv * g.B;
    const bool uniform = !(g.head_mode && (g.T_h % 2));
    auto add_range = [&](long long start, long long count, double c) {
        // items start .. start+count-1, item i on CTA i % grid
        const long long full = count / grid, rem = count % grid;
        everyone += (double)full * c;
        if (rem == 0)
            return;
        const long long a = start % grid, b = a + rem;
        if (b <= grid) {
            diff[a] += c;
            diff[b] -= c;
        } else {
            diff[a] += c;
            diff[grid] -= c;
            diff[0] += c;
            diff[b - grid] -= c;
        }
    };
    if (g.partial == kFused) {
        // items of one (batch, KV head) are consecutive: the costs repeat with
        // period NHP * NRT * Rq
        const long long period = (long long)g.NHP * g.NRT * g.Rq;
        std::vector<double> c(period);
        for (long long j = 0; j < period; ++j)
            c[j] = item_cost(g, decode_item(g, j), order, p);
        for (long long i = 0; i < n; ++i)
            add_range(i, 1, c[i % period]);
    }
    for (long long start = 0; start < n && g.partial != kFused; start += inner) {
        if (uniform) {
            const Item it = decode_item(g, start);
            add_range(start, std::min(inner, n - start), item_cost(g, it, order, p));
        } else {
            double c[kMaxR];  // cost by head pair; pairs past kMaxR are costed one by one
            const int nhp = std::min<int>(g.NHP, kMaxR);
            for (int hp = 0; hp < nhp; ++hp)
                c[hp] = item_cost(g, decode_item(g, start + hp), order, p);
            for (long long i = start; i < std::min(n, start + inner); ++i) {
                const int hp = (int)((i - start) % g.NHP);
                add_range(i, 1, hp < nhp ? c[hp] : item_cost(g, decode_item(g, i), order, p));
            }
        }
    }
    double run = 0.0, best = 0.0;
    for (long long c = 0; c < grid; ++c) {
        run += diff[c];
        best = std::max(best, run);
    }
    return p.launch_us + std::max(everyone + best, traffic_floor_us(g, p));
}

int check_profile(const mercury_cost_profile *p)
{
    if (!p)
        return set_error(MERCURY_EINVAL, "cost profile is NULL");
    if (p->n_sms < 1 || !(p->tile_us >= 0) || !(p->tile1_us >= 0) || !(p->item_us >= 0) ||
        !(p->launch_us >= 0) || !(p->merge_gbs > 0) || !(p->hbm_gbs > 0))
        return set_error(MERCURY_EINVAL, "cost profile has a negative or missing figure");
    return MERCURY_OK;
}

// Estimate of one schedule, or a negative number if the shape does not
// admit it.
double estimate(int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal, int R, int Rq, int runs, int shift,
                const mercury_cost_profile &p, long long *items, bool lower_bound = false)
{
    int mode, groups;
    mode_of(R, runs, mode, groups);
    Geom g;
    if (make_geom(g, B, Hq, Hkv, Sq, Skv, d, R, causal, mode, groups, Rq))
        return -1.0;
    int order[kMaxR * kMaxR];
    if (plan_shift(R, shift, order))
        return -1.0;
    *items = g.n_items;
    double t = lower_bound ? launch_lower_bound(g, order, p) : launch_estimate(g, order, p);
    if (g.partial != kFused) {
        const double rows = (double)B * Hq * Sq;
        const double bytes = (g.n_groups + 1.0) * rows * (d + 1) * 4.0;
        t += p.launch_us + bytes / (p.merge_gbs * 1e3);
    }
    return t;
}

// Static filter + cost estimate over every candidate of a call.
int enumerate(int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal, int R_in, int shift,
              long long budget, const mercury_cost_profile &p, std::vector<mercury_schedule> &out,
              long long *smallest)
{
    const long long io = input_output_bytes(B, Hq, Hkv, Sq, Skv, d);
    *smallest = -1;
    const int r_lo = R_in > 0 ? R_in : 1, r_hi = R_in > 0 ? R_in : kMaxR;
    for (int R = r_lo; R <= r_hi; ++R) {
        if (Skv % R != 0)
            continue;
        if (shift >= 2 && R % shift != 0)
            continue;
        for (int qi = 0; qi < 2; ++qi) {
            const int Rq = qi == 0 ? R : 1;
            if (qi == 1 && R == 1)
                continue;
            if (Sq % Rq != 0)
                continue;
            for (int runs = 1; runs <= R; ++runs) {
                const int spg = (R + runs - 1) / runs;
                if ((R + spg - 1) / spg != runs)
                    continue;  // the same runs as a smaller count
                const long long scratch = scratch_bytes_of(B, Hq, Sq, d, runs >= R ? R : runs);
                const long long total = io + scratch;
                if (*smallest < 0 || total < *smallest)
                    *smallest = total;
                if (budget > 0 && total > budget)
                    continue;
                long long items = 0;
                const double t = estimate(B, Hq, Hkv, Sq, Skv, d, causal, R, Rq, runs, shift, p, &items);
                if (t < 0)
                    continue;
                mercury_schedule s = {};
                s.R = R;
                s.Rq = Rq;
                s.n_runs = runs;
                s.shift = shift;
                s.work_items = items;
                s.scratch_bytes = scratch;
                s.hbm_bytes = total;
                s.predicted_us = t;
                s.measured_us = -1.0;
                out.push_back(s);
            }
        }
    }
    // Pareto flag: nothing else both fits in no more memory and is faster
    // (or as fast in strictly less memory).
    for (auto &a : out) {
        a.pareto = 1;
        for (const auto &b : out) {
            if (b.hbm_bytes <= a.hbm_bytes && b.predicted_us <= a.predicted_us &&
                (b.hbm_bytes < a.hbm_bytes || b.predicted_us < a.predicted_us)) {
                a.pareto = 0;
                break;
            }
        }
    }
    std::stable_sort(out.begin(), out.end(), [](const mercury_schedule &a, const mercury_schedule &b) {
        if (a.predicted_us != b.predicted_us)
            return a.predicted_us < b.predicted_us;
        if (a.hbm_bytes != b.hbm_bytes)
            return a.hbm_bytes < b.hbm_bytes;
        if ((a.Rq == a.R) != (b.Rq == b.R))
            return a.Rq == a.R;
        if (a.R != b.R)
            return a.R < b.R;
        return a.n_runs < b.n_runs;
    });
    return MERCURY_OK;
}

int check_shape(int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal, int R, int shift)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Skv < 1)
        return set_error(MERCURY_EINVAL, "B, Hq, Hkv, Sq, Skv must be >= 1");
    if (Hq % Hkv != 0)
        return set_error(MERCURY_EINVAL, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
    if (d != 64 && d != 128)
        return set_error(MERCURY_EINVAL, "head dim must be 64 or 128 (got %d)", d);
    if (causal && Sq > Skv)
        return set_error(MERCURY_EINVAL, "causal attention needs Sq <= Skv (Sq %d, Skv %d)", Sq, Skv);
    if (R < 0 || R > kMaxR)
        return set_error(MERCURY_EINVAL, "R must be 0 (choose) or in [1, %d] (got %d)", kMaxR, R);
    if (shift < 0)
        return set_error(MERCURY_EINVAL, "shift must be >= 0 (got %d)", shift);
    if (R > 0 && shift >= 2 && R % shift != 0)
        return set_error(MERCURY_EINVAL, "nested shift: inner size %d must divide R = %d", shift, R);
    if (R > 0 && Skv % R != 0)
        return set_error(MERCURY_EINVAL, "R (%d) must divide Skv (%d)", R, Skv);
    // 63-bit products of every tensor and of the largest scratch
    const double worst = (double)kMaxR * B * Hq * Sq * (d + 1) * 4.0 + 2.0 * B * Hkv * (double)Skv * d * 2.0;
    if (worst > 4.0e18)
        return set_error(MERCURY_EINVAL, "tensor sizes overflow");
    if ((long long)B * Hq > 0x7fffffffLL || (long long)B * Hkv > 0x7fffffffLL)
        return set_error(MERCURY_EINVAL, "B*H exceeds 2^31");
    return MERCURY_OK;
}

// ------------------------------------------------------------ measurement

struct Events {
    cudaEvent_t a = nullptr, b = nullptr;
    ~Events()
    {
        if (a)
            cudaEventDestroy(a);
        if (b)
            cudaEventDestroy(b);
    }
};

struct DeviceBuffers {
    std::vector<void *> ptrs;
    ~DeviceBuffers()
    {
        for (void *p : ptrs)
            cudaFree(p);
    }
    int alloc(void **p, size_t bytes)
    {
        cudaError_t e = cudaMalloc(p, bytes);
        if (e != cudaSuccess)
            return set_error(MERCURY_ECUDA, "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
        ptrs.push_back(*p);
        return MERCURY_OK;
    }
};

// Median over `reps` timed launches of fn (after `warm` untimed ones), in us.
template <class F>
int time_median(F fn, int warm, int reps, cudaStream_t s, Events &ev, double *us)
{
    for (int i = 0; i < warm; ++i) {
        int rc = fn();
        if (rc)
            return rc;
    }
    std::vector<double> t;
    for (int i = 0; i < reps; ++i) {
        cudaEventRecord(ev.a, s);
        int rc = fn();
        if (rc)
            return rc;
        cudaEventRecord(ev.b, s);
        cudaError_t e = cudaEventSynchronize(ev.b);
        if (e != cudaSuccess)
            return set_error(MERCURY_ECUDA, "cudaEventSynchronize: %s", cudaGetErrorString(e));
        float ms = 0.f;
        cudaEventElapsedTime(&ms, ev.a, ev.b);
        t.push_back(ms * 1e3);
    }
    std::sort(t.begin(), t.end());
    *us = t[t.size() / 2];
    return MERCURY_OK;
}

int check_errors_after(cudaStream_t s)
{
    int rc = mercury_sync_status((void *)s);
    return rc;
}

// ------------------------------------------------------------ tuning cache

std::mutex g_cache_mu;
std::map<std::string, mercury_schedule> g_cache;

const char *kBuildId = __DATE__ " " __TIME__;

// A cached schedule is kept while the faster of two re-timed runs takes at
// most this factor of its recorded time (1.5; env MERCURY_TUNE_RECHECK
// overrides, 0 forces a re-tune on every call), plus kRecheckSlackUs: a
// single run of a call of a few tens of microseconds can take that much more
// when the host is late to launch it, which says nothing about the schedule.
constexpr double kRecheckSlackUs = 20.0;

double recheck_factor()
{
    const char *e = getenv("MERCURY_TUNE_RECHECK");
    if (e && *e) {
        char *end = nullptr;
        const double v = strtod(e, &end);
        if (end && *end == '\0' && v >= 0)
            return v;
    }
    return 1.5;
}

int cache_key(int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal, int R, int shift, long long budget,
              int top_k, std::string *key)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return set_error(MERCURY_ECUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    int sms = 0, major = 0, minor = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    char buf[512];
    snprintf(buf, sizeof buf, "dev%d sm%d cc%d.%d build[%s] B%d Hq%d Hkv%d Sq%d Skv%d d%d c%d R%d s%d b%lld k%d",
             dev, sms, major, minor, kBuildId, B, Hq, Hkv, Sq, Skv, d, causal, R, shift, budget, top_k);
    *key = buf;
    return MERCURY_OK;
}

}  // namespace

namespace mercury {

int best_run_count(int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal, int R, int shift, int n_sms,
                   long long scratch_cap)
{
    // The answer depends only on the arguments; remember it, so a repeated
    // call does not spend host time on the estimate in front of its launch.
    static std::mutex mu;
    static std::map<std::array<long long, 11>, int> memo;
    const std::array<long long, 11> key = {B, Hq, Hkv, Sq, Skv, d, causal, R, shift, n_sms, scratch_cap};
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = memo.find(key);
        if (it != memo.end())
            return it->second;
    }
    mercury_cost_profile p;
    mercury_default_cost_profile(n_sms, &p);
    clear_error();
    int best = 1;
    double best_t = -1.0;
    for (int runs = 1; runs <= R; ++runs) {
        const int spg = (R + runs - 1) / runs;
        if ((R + spg - 1) / spg != runs)
            continue;
        if (runs > 1 && scratch_bytes_of(B, Hq, Sq, d, runs >= R ? R : runs) > scratch_cap)
            break;
        long long items = 0;
        // A candidate whose lower bound is no better than the best so far
        // cannot win: skip its full estimate (the simulation of a causal
        // launch's dynamic scheduling costs ~70 ns per work item).  The margin
        // covers the different summation order of the bound.
        if (best_t >= 0 &&
            estimate(B, Hq, Hkv, Sq, Skv, d, causal, R, R, runs, shift, p, &items, true) * (1.0 - 1e-9) >= best_t)
            continue;
        const double t = estimate(B, Hq, Hkv, Sq, Skv, d, causal, R, R, runs, shift, p, &items);
        if (t >= 0 && (best_t < 0 || t < best_t)) {
            best_t = t;
            best = runs;
        }
    }
    std::lock_guard<std::mutex> lock(mu);
    if (memo.size() >= 4096)
        memo.clear();
    memo[key] = best;
    return best;
}

}  // namespace mercury

extern "C" {

int mercury_default_cost_profile(int n_sms, mercury_cost_profile *prof)
{
    if (!prof)
        return set_error(MERCURY_EINVAL, "prof is NULL");
    if (n_sms < 1)
        return set_error(MERCURY_EINVAL, "n_sms must be >= 1 (got %d)", n_sms);
    // GB300 figures of this library's kernels (mercury_measure_cost_profile
    // on one GB300, SM clock 2.07 GHz).
    prof->tile_us = 1.45;
    prof->tile1_us = 1.33;
    prof->item_us = 10.2;
    prof->launch_us = 14.3;
    prof->merge_gbs = 6320.0;
    prof->hbm_gbs = 6490.0;
    prof->n_sms = n_sms;
    prof->measured = 0;
    return clear_error();
}

int mercury_plan_schedules(int B, int Hq, int Hkv, int Sq, int Skv, int d, int causal, int R, int shift,
                           long long budget_bytes, const mercury_cost_profile *prof, mercury_schedule *plans,
                           int max_plans, int *n_plans)
{
    if (!n_plans)
        return set_error(MERCURY_EINVAL, "n_plans is NULL");
    if (max_plans < 0 || (max_plans > 0 && !plans))
        return set_error(MERCURY_EINVAL, "plans must hold max_plans >= 0 entries");
    int rc = check_profile(prof);
    if (rc)
        return rc;
    rc = check_shape(B, Hq, Hkv, Sq, Skv, d, causal, R, shift);
    if (rc)
        return rc;
    std::vector<mercury_schedule> all;
    long long smallest = -1;
    enumerate(B, Hq, Hkv, Sq, Skv, d, causal ? 1 : 0, R, shift, budget_bytes, *prof, all, &smallest);
    *n_plans = (int)all.size();
    if (all.empty()) {
        if (smallest < 0)
            return set_error(MERCURY_EINVAL, "no R in 1..%d divides Skv = %d and suits shift %d", kMaxR, Skv,
                             shift);
        return set_error(MERCURY_EBUDGET,
                         "no schedule fits %lld bytes: the smallest needs %lld (inputs, outputs and scratch)",
                         budget_bytes, smallest);
    }
    const int n = std::min<int>(max_plans, (int)all.size());
    for (int i = 0; i < n; ++i)
        plans[i] = all[i];
    return clear_error();
}

int mercury_measure_cost_profile(mercury_cost_profile *prof, void *stream)
{
    CallRange range(__func__);
    if (!prof)
        return set_error(MERCURY_EINVAL, "prof is NULL");
    int n = 0;
    int rc = device_sm_count(&n);
    if (rc)
        return rc;
    cudaStream_t s = (cudaStream_t)stream;
    const int d = 128;
    // Synthetic inputs: every bf16 element 0x3c3c (~0.0115), every float of
    // the merge's inputs 0x3c3c3c3c (~0.0115); timing does not depend on values.
    const size_t kv_elems = std::max<size_t>((size_t)2 * n * 2048, (size_t)n * 8192) * d;
    const size_t q_elems = (size_t)2 * n * 256 * d;
    const int parts = 8;
    const long long mrows = (long long)n * 1024;
    DeviceBuffers buf;
    void *q, *k, *v, *o, *l, *op, *lp;
    if ((rc = buf.alloc(&q, q_elems * 2)) || (rc = buf.alloc(&k, kv_elems * 2)) ||
        (rc = buf.alloc(&v, kv_elems * 2)) || (rc = buf.alloc(&o, (size_t)mrows * d * 4)) ||
        (rc = buf.alloc(&l, (size_t)mrows * 4)) || (rc = buf.alloc(&op, (size_t)parts * mrows * d * 4)) ||
        (rc = buf.alloc(&lp, (size_t)parts * mrows * 4)))
        return rc;
    cudaMemsetAsync(q, 0x3c, q_elems * 2, s);
    cudaMemsetAsync(k, 0x3c, kv_elems * 2, s);
    cudaMemsetAsync(v, 0x3c, kv_elems * 2, s);
    cudaMemsetAsync(op, 0x3c, (size_t)parts * mrows * d * 4, s);
    cudaMemsetAsync(lp, 0x3c, (size_t)parts * mrows * 4, s);
    Events ev;
    if (cudaEventCreate(&ev.a) != cudaSuccess || cudaEventCreate(&ev.b) != cudaSuccess)
        return set_error(MERCURY_ECUDA, "cudaEventCreate failed");
    mercury_schedule fused = {};
    fused.R = 1;
    fused.Rq = 1;
    fused.n_runs = 1;
    fused.shift = 0;
    auto attn = [&](int H, int Sq, int Skv) {
        return [=, &fused]() {
            return mercury_attn_run_schedule(q, k, v, 1, H, H, Sq, Skv, d, 0, &fused, (float *)o, (float *)l,
                                             (void *)s);
        };
    };
    // one work item per SM (two query tiles of 128 rows), 16 and 64 K/V
    // tiles; two items per SM; one query tile per item
    double t16 = 0, t64 = 0, t16x2 = 0, t64_1 = 0, tm = 0;
    if ((rc = time_median(attn(n, 256, 2048), 2, 5, s, ev, &t16)) ||
        (rc = time_median(attn(n, 256, 8192), 2, 5, s, ev, &t64)) ||
        (rc = time_median(attn(2 * n, 256, 2048), 2, 5, s, ev, &t16x2)) ||
        (rc = time_median(attn(n, 128, 8192), 2, 5, s, ev, &t64_1)))
        return rc;
    auto merge = [&]() {
        return mercury_lse_merge((const float *)op, (const float *)lp, parts, mrows, d, (float *)o, (float *)l,
                                 (void *)s);
    };
    if ((rc = time_median(merge, 2, 5, s, ev, &tm)))
        return rc;
    // device-to-device copy of the merge's partials into the K/V buffers
    const size_t copy_bytes = std::min<size_t>((size_t)parts * mrows * d * 4, kv_elems * 2);
    auto copy = [&]() {
        cudaError_t e = cudaMemcpyAsync(k, op, copy_bytes, cudaMemcpyDeviceToDevice, s);
        return e == cudaSuccess ? MERCURY_OK
                                : set_error(MERCURY_ECUDA, "cudaMemcpyAsync: %s", cudaGetErrorString(e));
    };
    double tc = 0;
    if ((rc = time_median(copy, 2, 5, s, ev, &tc)))
        return rc;
    if ((rc = check_errors_after(s)))
        return rc;
    const double tile = std::max(0.0, (t64 - t16) / 48.0);
    const double item = std::max(0.0, t16x2 - t16 - 16.0 * tile);
    const double launch = std::max(0.0, t16 - item - 16.0 * tile);
    const double tile1 = std::max(0.0, (t64_1 - launch - item) / 64.0);
    const double merge_bytes = (parts + 1.0) * (double)mrows * (d + 1) * 4.0;
    prof->tile_us = tile;
    prof->tile1_us = tile1;
    prof->item_us = item;
    prof->launch_us = launch;
    prof->merge_gbs = merge_bytes / (tm * 1e3);
    prof->hbm_gbs = 2.0 * (double)copy_bytes / (tc * 1e3);
    prof->n_sms = n;
    prof->measured = 1;
    return clear_error();
}

int mercury_tune_schedule(const void *q, const void *k, const void *v, int B, int Hq, int Hkv, int Sq, int Skv,
                          int d, int R, int shift, int causal, long long budget_bytes, int top_k, float *out,
                          float *lse, void *stream, mercury_schedule *best, int *cache_hit)
{
    CallRange range(__func__);
    if (top_k < 1 || top_k > 16)
        return set_error(MERCURY_EINVAL, "top_k must be in [1, 16] (got %d)", top_k);
    if (!q || !k || !v || !out || !lse)
        return set_error(MERCURY_EINVAL, "null pointer argument");
    causal = causal ? 1 : 0;
    cudaStream_t s = (cudaStream_t)stream;
    std::string key;
    int rc = cache_key(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, budget_bytes, top_k, &key);
    if (rc)
        return rc;
    Events ev;
    if (cudaEventCreate(&ev.a) != cudaSuccess || cudaEventCreate(&ev.b) != cudaSuccess)
        return set_error(MERCURY_ECUDA, "cudaEventCreate failed");
    auto runner = [&](const mercury_schedule &plan) {
        return [&, plan]() {
            return mercury_attn_run_schedule(q, k, v, B, Hq, Hkv, Sq, Skv, d, causal, &plan, out, lse, stream);
        };
    };
    mercury_schedule cached = {};
    bool have = false;
    {
        std::lock_guard<std::mutex> lock(g_cache_mu);
        auto it = g_cache.find(key);
        if (it != g_cache.end()) {
            cached = it->second;
            have = true;
        }
    }
    if (have) {
        double t = 0, t2 = 0;
        if ((rc = time_median(runner(cached), 0, 1, s, ev, &t)) ||
            (rc = time_median(runner(cached), 0, 1, s, ev, &t2)))
            return rc;
        t = std::min(t, t2);
        const double factor = recheck_factor();
        if (factor > 0 && t <= factor * cached.measured_us + kRecheckSlackUs) {
            if ((rc = check_errors_after(s)))
                return rc;
            if (best)
                *best = cached;
            if (cache_hit)
                *cache_hit = 1;
            return clear_error();
        }
        std::lock_guard<std::mutex> lock(g_cache_mu);
        g_cache.erase(key);  // no longer meets its measured time: tune again
    }
    int sms = 0;
    if ((rc = device_sm_count(&sms)))
        return rc;
    mercury_cost_profile prof;
    mercury_default_cost_profile(sms, &prof);
    std::vector<mercury_schedule> plans(top_k);
    int n_plans = 0;
    if ((rc = mercury_plan_schedules(B, Hq, Hkv, Sq, Skv, d, causal, R, shift, budget_bytes, &prof, plans.data(),
                                     top_k, &n_plans)))
        return rc;
    const int n = std::min(top_k, n_plans);
    int chosen = -1;
    for (int i = 0; i < n; ++i) {
        double t = 0;
        if ((rc = time_median(runner(plans[i]), 1, 3, s, ev, &t)))
            return rc;
        plans[i].measured_us = t;
        if (chosen < 0 || t < plans[chosen].measured_us)
            chosen = i;
    }
    // leave the chosen schedule's result in out / lse
    if (chosen != n - 1 && (rc = runner(plans[chosen])()))
        return rc;
    if ((rc = check_errors_after(s)))
        return rc;
    {
        std::lock_guard<std::mutex> lock(g_cache_mu);
        g_cache[key] = plans[chosen];
    }
    if (best)
        *best = plans[chosen];
    if (cache_hit)
        *cache_hit = 0;
    return clear_error();
}

void mercury_tune_cache_clear(void)
{
    std::lock_guard<std::mutex> lock(g_cache_mu);
    g_cache.clear();
}

}  // extern "C"
