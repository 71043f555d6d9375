// dg_plan.h -- host-side choice of the LM-head kernel and its tiling, shared
// by every entry point that launches it.
#pragma once

#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "dg_kernels.h"

namespace dg {

constexpr int kMaxSlots = 256;       // upper bound on LM-head CTAs (>= SM count)

struct LmPlan {
    int M, V, d;
    bool pair;        // 2-CTA cluster kernel (lm_head_pair_kernel) or single-CTA kernel
    int BN;           // vocabulary columns per tile
    int ntn;          // vocabulary tiles per 256-row block
    int mblocks;      // 256-row blocks
    int total;        // tiles
    int units;        // CTAs (single) or clusters (pair): the tile schedule's
                      // slots, one partial state per (row, unit)
    int grid;         // CTAs launched
    int part_slots() const { return units; }
};

// Choose the kernel and tile width: fewest tile columns per SM on the busiest
// CTA, plus a per-tile overhead.  DG_LM_KERNEL=single|pair and DG_LM_BN
// force a choice.
inline LmPlan plan_lm_head(int M, int d, int V, int sms)
{
    LmPlan best{};
    best.M = M;
    best.V = V;
    best.d = d;
    best.mblocks = (M + kRowsPerBlock - 1) / kRowsPerBlock;
    const char *env_bn = std::getenv("DG_LM_BN");
    const int forced_bn = env_bn ? std::atoi(env_bn) : 0;
    const char *env_k = std::getenv("DG_LM_KERNEL");
    const bool only_single = env_k && std::strcmp(env_k, "single") == 0;
    const bool only_pair = env_k && std::strcmp(env_k, "pair") == 0;
    long best_cost = -1;
    auto consider = [&](bool pair, int bn) {
        if (forced_bn && bn != forced_bn) return;
        if ((pair && only_single) || (!pair && only_pair)) return;
        const int ntn = (V + bn - 1) / bn;
        const int total = ntn * best.mblocks;
        const int cap = pair ? std::max(1, sms / 2) : sms;
        const int units = std::min(std::min(total, cap), kMaxSlots / (pair ? 2 : 1));
        const long per_unit = (total + units - 1) / units;
        // per-SM columns of a tile: bn (single, 256 rows) or bn / 2 (pair, 128
        // rows each, and half the hidden-block traffic per tile)
        const long cost = per_unit * (pair ? bn / 2 + 30 : bn + 40);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best.pair = pair;
            best.BN = bn;
            best.ntn = ntn;
            best.total = total;
            best.units = units;
            best.grid = pair ? 2 * units : units;
        }
    };
    for (int bn = 128; bn >= 64; bn -= 16) consider(false, bn);
    consider(true, 256);
    consider(true, 128);
    return best;
}

// Upper bound on the partial-state slots of any plan for these shapes
// (workspace queries do not know the SM count).
inline int slot_bound(int M, int V)
{
    const long mblocks = (M + kRowsPerBlock - 1) / kRowsPerBlock;
    const long tiles = mblocks * ((V + 63) / 64);
    return static_cast<int>(std::min<long>(tiles, kMaxSlots));
}

}  // namespace dg
