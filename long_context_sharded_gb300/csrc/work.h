// work.h -- how one compute call is split into work items (host and device).
//
// A work item is (batch b, KV head hkv, virtual rank i, pair slot), plus the
// shard s in partial mode.  It covers up to two 128-row query tiles that
// share the KV head, so every K/V tile the CTA loads feeds two tensor-core
// tiles.  A tile is Gp query heads x Mq consecutive queries (Gp*Mq = 128):
// when a query block is short (Sq/R < 128) several heads of one GQA/MQA group
// are packed into the 128 rows, which is how the group's query heads reuse
// each KV tile (the pages note GQA/MQA head sharing changes how the work can
// be split: Silicon & Systems, "The hidden cost of synchronized operators";
// Mercury-SOSP25 paper notes, Critical Analysis).
//
// Queries are split into R contiguous blocks of Bq = Sq/R rows and keys into
// R contiguous shards of Bk = Skv/R rows; virtual rank i owns query block i
// (shard primitive, Mercury-SOSP25 paper notes 核心方法).
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define MERCURY_HD __host__ __device__ __forceinline__
#else
#define MERCURY_HD inline
#endif

namespace mercury {

constexpr int kMaxR = 128;      // largest R (shift table fits the kernel parameters)
constexpr int kTileRows = 128;  // M of the tcgen05 MMA: query rows per tile
constexpr int kTileKeys = 128;  // keys per K/V tile: N of S = Q K^T, K of O += P V

// Modes of a call: kFused runs all R steps of a rank in one work item (one
// output); kPerStep gives every (rank, shard) pair its own item and output
// slot (the step at which the rank reads that shard); kGrouped splits each
// rank's step sequence into n_groups runs of consecutive steps, one output
// slot per run, merged afterwards (split-KV for short query sides).
enum Mode { kFused = 0, kPerStep = 1, kGrouped = 2 };

struct Geom {
    int B, Hq, Hkv, Sq, Skv, d, R, causal, partial;  // partial: mode (Mode)
    int Rq;         // ranks that own query blocks: R, or 1 for a decode split
    int n_groups;   // kGrouped: runs per rank; else 1 (fused) or R (per step)
    int spg;        // steps per run (kGrouped), R (fused), 1 (per step)
    int G;          // query heads per KV head
    int Bq, Bk;     // rows per query block / keys per KV shard
    int Mq, Gp;     // queries per head in a tile, heads per tile (Mq*Gp = 128)
    int head_mode;  // 1: a pair = two head groups, same rows; 0: two row tiles
    int T_h;        // head tiles per KV group (G / Gp)
    int T_r;        // row tiles per query block (ceil(Bq / Mq))
    int NHP, NRT;   // pair slots along heads / along rows
    long long n_items;
};

// Choose the tile geometry.  mode: kFused, kPerStep or kGrouped (then
// n_groups in [1, R] runs; the run length is ceil(R / n_groups) steps and the
// run count is recomputed from it).  Returns 0, or -1 when unsupported.
// Rq: number of query blocks (ranks owning queries); R by default.  A decode
// split uses Rq = 1: the whole (short) query side is rank 0's, the KV is cut
// into R shards.
inline int make_geom(Geom &g, int B, int Hq, int Hkv, int Sq, int Skv, int d, int R,
                     int causal, int mode, int n_groups = 1, int Rq = -1)
{
    if (Rq < 0)
        Rq = R;
    if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Skv < 1 || R < 1 || R > kMaxR || Rq < 1 || Rq > R)
        return -1;
    if (Hq % Hkv != 0 || Sq % Rq != 0 || Skv % R != 0)
        return -1;
    if (mode != kFused && mode != kPerStep && mode != kGrouped)
        return -1;
    if (mode == kGrouped && (n_groups < 1 || n_groups > R))
        return -1;
    g.B = B; g.Hq = Hq; g.Hkv = Hkv; g.Sq = Sq; g.Skv = Skv; g.d = d; g.R = R; g.Rq = Rq;
    g.causal = causal ? 1 : 0;
    g.partial = mode;
    if (mode == kFused) {
        g.spg = R;
        g.n_groups = 1;
    } else if (mode == kPerStep) {
        g.spg = 1;
        g.n_groups = R;
    } else {
        g.spg = (R + n_groups - 1) / n_groups;
        g.n_groups = (R + g.spg - 1) / g.spg;
    }
    g.G = Hq / Hkv;
    g.Bq = Sq / Rq;
    g.Bk = Skv / R;
    int Mq = kTileRows;
    // pack heads of one group while a tile would otherwise run past its block
    while (Mq / 2 >= 16 && Mq / 2 >= g.Bq && g.G % (kTileRows / (Mq / 2)) == 0)
        Mq /= 2;
    g.Mq = Mq;
    g.Gp = kTileRows / Mq;
    g.T_h = g.G / g.Gp;
    g.T_r = (g.Bq + Mq - 1) / Mq;
    g.head_mode = g.T_h >= 2 ? 1 : 0;
    g.NHP = g.head_mode ? (g.T_h + 1) / 2 : 1;
    g.NRT = g.head_mode ? g.T_r : (g.T_r + 1) / 2;
    long long per_rank = (long long)g.NHP * g.Hkv * g.B * g.NRT;
    g.n_items = per_rank * Rq * (g.partial == kFused ? 1 : g.n_groups);
    return 0;
}

struct Tile {
    int valid;  // tile present in this work item
    int h0;     // first query head
    int q0;     // first query row
    int nq;     // valid queries per head (<= Mq)
};

struct Item {
    int b, hkv, rank;
    int shard;  // kPerStep: the KV shard; kGrouped: the run index; fused: -1
    Tile t[2];
    int kv_end; // keys [0, kv_end) can be attended by some row of the item
};

// Decode work item `idx`.  Fused causal items are ordered heaviest first
// (longest KV range first) so that a wave of CTAs ends together, with the
// items of one KV head's group next to each other; fused non-causal items
// (all of equal cost) take one (batch, KV head) at a time, so the CTAs
// resident together share K/V in L2.  Per-step items are ordered by shard
// first, so CTAs resident together read the same shard; grouped items by run
// first (neighbouring ranks' runs overlap in shards under the shift).
MERCURY_HD Item decode_item(const Geom &g, long long idx)
{
    Item it;
    int hp, rt, rank;
    if (g.partial == kFused) {
        // every item of one (batch, KV head) before the next, so the CTAs
        // resident together read a few heads' K/V from L2
        hp = (int)(idx % g.NHP); idx /= g.NHP;
        rt = (int)(idx % g.NRT); idx /= g.NRT;
        rank = (int)(idx % g.Rq); idx /= g.Rq;
        it.hkv = (int)(idx % g.Hkv); idx /= g.Hkv;
        it.b = (int)(idx % g.B); idx /= g.B;
    } else {
        hp = (int)(idx % g.NHP); idx /= g.NHP;
        it.hkv = (int)(idx % g.Hkv); idx /= g.Hkv;
        it.b = (int)(idx % g.B); idx /= g.B;
        rt = (int)(idx % g.NRT); idx /= g.NRT;
        rank = (int)(idx % g.Rq); idx /= g.Rq;
    }
    it.shard = g.partial != kFused ? (int)idx : -1;
    if (g.causal && g.partial == kFused) {
        rank = g.Rq - 1 - rank;
        rt = g.NRT - 1 - rt;
    }
    it.rank = rank;
    int last_q = -1;
    for (int t = 0; t < 2; ++t) {
        int ht, rtile;
        if (g.head_mode) {
            ht = 2 * hp + t;
            rtile = rt;
            it.t[t].valid = ht < g.T_h;
        } else {
            ht = 0;
            rtile = 2 * rt + t;
            it.t[t].valid = rtile < g.T_r;
        }
        it.t[t].h0 = it.hkv * g.G + ht * g.Gp;
        it.t[t].q0 = rank * g.Bq + rtile * g.Mq;
        int nq = g.Bq - rtile * g.Mq;
        it.t[t].nq = nq < g.Mq ? nq : g.Mq;
        if (it.t[t].valid) {
            int lq = it.t[t].q0 + it.t[t].nq - 1;
            if (lq > last_q)
                last_q = lq;
        }
    }
    if (g.causal) {
        long long e = (long long)last_q + (g.Skv - g.Sq) + 1;
        it.kv_end = e < g.Skv ? (int)e : g.Skv;
    } else {
        it.kv_end = g.Skv;
    }
    return it;
}

// Key range [lo, hi) of shard s that the item can attend (empty if hi <= lo).
MERCURY_HD void shard_range(const Geom &g, const Item &it, int s, int &lo, int &hi)
{
    lo = s * g.Bk;
    hi = lo + g.Bk;
    if (hi > it.kv_end)
        hi = it.kv_end;
}

// Steps in the item's sequence: all R (fused), one (per step), or the
// item's run of consecutive steps (grouped).
MERCURY_HD int item_steps(const Geom &g, const Item &it)
{
    if (g.partial == kFused)
        return g.R;
    if (g.partial == kPerStep)
        return 1;
    const int rest = g.R - it.shard * g.spg;
    return rest < g.spg ? rest : g.spg;
}

MERCURY_HD int n_kv_tiles(int lo, int hi)
{
    return hi > lo ? (hi - lo + kTileKeys - 1) / kTileKeys : 0;
}

// Shift table, shift encoding as in mercury_plan_shift.  Returns 0 or -1.
inline int plan_shift(int R, int shift, int *order)
{
    if (R < 1 || R > kMaxR || shift < 0 || order == nullptr)
        return -1;
    if (shift >= 2 && R % shift != 0)
        return -1;
    for (int i = 0; i < R; ++i) {
        for (int j = 0; j < R; ++j) {
            int s;
            if (shift == 0) {
                s = j;                         // synchronous: all ranks on shard j
            } else if (shift == 1) {
                s = (i + j) % R;               // flat (j+i)%J
            } else {
                const int Ri = shift, Ro = R / shift;
                const int outer = (i / Ri + j / Ri) % Ro;
                const int inner = (i % Ri + j % Ri) % Ri;
                s = outer * Ri + inner;        // nested: inner ring inside outer ring
            }
            order[i * R + j] = s;
        }
    }
    return 0;
}

}  // namespace mercury
