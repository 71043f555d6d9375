// dg_plan.h -- host-side choice of the LM-head kernel and its tiling, shared
// by every entry point that launches it.
#pragma once

#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "dg_kernels.h"

namespace dg {

constexpr int kMaxSlots = 256;       // upper bound on LM-head CTAs (>= SM count)

// LM-head kernels
enum LmKind : int {
    kLmSingle = 0,    // lm_head_kernel: one CTA per tile, 256 rows x BN columns
                      // (kind 1 is not used)
    kLmDuo = 2,       // lm_head_duo_kernel: 2-CTA cluster, 2-SM UMMA
    kLmDuoFused = 3,  // lm_head_duo_kernel on 128-column schedule tiles, each
                      // adjacent pair in a cluster's range (same row block)
                      // run as one 256-column tile: a 256-column kernel whose
                      // tile count per cluster is balanced to half a tile
};

struct LmPlan {
    int M, V, d;
    int kind;         // LmKind
    int BN;           // vocabulary columns per tile
    int ntn;          // vocabulary tiles per 256-row block
    int mblocks;      // 256-row blocks
    int total;        // tiles
    int units;        // CTAs (single) or clusters (pair): the tile schedule's
                      // slots, one partial state per (row, unit)
    int grid;         // CTAs launched
    int sms;          // SMs of the device the plan was made for
    int epi_warps;    // epilogue warps of the 2-SM kernel (8 or 16, FP8 12; 0 otherwise)
    bool sc;          // the self-conditioning instance (lm_head_duo_sc_kernel)
    int part_slots() const { return units; }
    bool cluster() const { return kind != kLmSingle; }
    bool duo() const { return kind == kLmDuo || kind == kLmDuoFused; }
};

// Choose the kernel and tile width: fewest tile columns per SM on the busiest
// CTA, plus a per-tile overhead; the 2-SM kernel runs 8 epilogue warps on a
// single 256-row block of bf16 operands, else 16 (FP8: 12).  DG_LM_KERNEL=
// single|duo|fused, DG_LM_BN and DG_LM_EPI=8|16 (bf16) force a choice.  FP8
// operands have the 2-SM UMMA kernel only.
// only_kind >= 0 restricts the choice to that kernel (as DG_LM_KERNEL does).
// A packed weight (dg_pack_lm_weight) is read by the 2-SM kernels only.
inline LmPlan plan_lm_head(int M, int d, int V, int sms, bool fp8 = false, bool sc = false,
                           int only_kind = -1, bool packed = false)
{
    LmPlan best{};
    best.M = M;
    best.V = V;
    best.d = d;
    best.mblocks = (M + kRowsPerBlock - 1) / kRowsPerBlock;
    best.sms = sms;
    const char *env_bn = std::getenv("DG_LM_BN");
    int forced_bn = env_bn ? std::atoi(env_bn) : 0;
    const char *env_k = std::getenv("DG_LM_KERNEL");
    const int only_env = !env_k ? -1
                     : std::strcmp(env_k, "single") == 0 ? kLmSingle
                     : std::strcmp(env_k, "duo") == 0    ? kLmDuo
                     : std::strcmp(env_k, "fused") == 0  ? kLmDuoFused
                                                         : -1;
    // a forced kernel FP8 operands, the self-conditioning read-out or a
    // packed weight do not have is ignored
    const bool duo_only = fp8 || sc || packed;
    const int only_req = only_kind >= 0 ? only_kind : only_env;
    const int only = duo_only && only_req != kLmDuo && only_req != kLmDuoFused ? -1 : only_req;
    long best_cost = -1;
    auto consider = [&](int kind, int bn) {
        if (forced_bn && bn != forced_bn) return;
        if (only >= 0 && kind != only) return;
        if (duo_only && kind != kLmDuo && kind != kLmDuoFused) return;
        const bool pair = kind != kLmSingle;
        const int ntn = (V + bn - 1) / bn;
        const int total = ntn * best.mblocks;
        const int cap = pair ? std::max(1, sms / 2) : sms;
        const int units = std::min(std::min(total, cap), kMaxSlots / (pair ? 2 : 1));
        const long per_unit = (total + units - 1) / units;
        // per-SM columns of a tile: bn (single, 256 rows) or bn / 2 (clusters,
        // 128 rows each, and half the hidden-block traffic per tile), plus a
        // per-tile overhead
        const long over = kind == kLmSingle ? 40 : 25;
        // fused: the per-tile overhead is paid once per 256-column tile
        const long cost = kind == kLmDuoFused
                              ? per_unit * (bn / 2) + (per_unit + 1) / 2 * over
                              : per_unit * ((pair ? bn / 2 : bn) + over);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best.kind = kind;
            best.BN = bn;
            best.ntn = ntn;
            best.total = total;
            best.units = units;
            best.grid = pair ? 2 * units : units;
        }
    };
    for (int pass = 0; pass < 2 && best_cost < 0; ++pass) {
        // a forced width no candidate of the kernel has is ignored
        if (pass == 1) forced_bn = 0;
        for (int bn = 128; bn >= 64; bn -= 16) consider(kLmSingle, bn);
        consider(kLmDuo, 256);
        consider(kLmDuo, 128);
        consider(kLmDuoFused, 128);
    }
    best.sc = sc;
    if (best.duo()) {
        const char *env_e = std::getenv("DG_LM_EPI");
        const int forced_e = env_e ? std::atoi(env_e) : 0;
        best.epi_warps = fp8 ? 4 * kDuoCGFp8
                         : sc ? 4 * kDuoCGNarrow
                         : forced_e == 8 || forced_e == 16 ? forced_e
                         : best.mblocks == 1             ? 4 * kDuoCGNarrow
                                                         : 4 * kDuoCGWide;
    }
    return best;
}

inline int lm_smem_bytes(int kind)
{
    return kind == kLmSingle ? kLmSmemBytes : kDuoSmemBytes;
}

// Launch with programmatic stream serialization when `pdl` is set: the kernel
// may start while the previous kernel of the stream is still running (every
// kernel of the step waits, griddep_wait, before it touches memory).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t st, bool pdl, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Programmatic launches are used outside stream capture only.
inline bool use_pdl(cudaStream_t st)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return cs == cudaStreamCaptureStatusNone;
}

// Launch the planned LM-head kernel, not the self-conditioning instance,
// which takes a third map (maps: X box {64, 128} for the cluster
// kernels, {64, 256} otherwise; W box {64, 64}; FP8: X8 box {128, 128}, W8t
// box {128, BN / 2}).  a.fuse2 must be set for kLmDuoFused.
inline cudaError_t launch_lm_head(const LmPlan &plan, const CUtensorMap &mx, const CUtensorMap &mw,
                                  const LmHeadArgs &a, cudaStream_t st, bool pdl, bool fp8 = false)
{
    const int smem = lm_smem_bytes(plan.kind);
    const bool wide = plan.epi_warps == 4 * kDuoCGWide;
    auto kern = fp8                    ? lm_head_duo_fp8_kernel
                : plan.kind == kLmSingle ? lm_head_kernel
                : wide                   ? lm_head_duo_wide_kernel   // kLmDuo, kLmDuoFused
                                         : lm_head_duo_kernel;
    const int threads = fp8          ? DuoEpilogue<kDuoCGFp8>::Threads
                        : !plan.duo() ? kLmThreads
                        : wide        ? DuoEpilogue<kDuoCGWide>::Threads
                                      : DuoEpilogue<kDuoCGNarrow>::Threads;
    return launch_kernel(kern, dim3(plan.grid), dim3(threads), smem, st, pdl, mx, mw, a);
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
