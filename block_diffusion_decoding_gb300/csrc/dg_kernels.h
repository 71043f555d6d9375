// dg_kernels.h -- argument blocks and kernel declarations shared by the
// kernel files and the host-side entry points (dg_api.cu).
#pragma once

#include "dg_sampler.cuh"

namespace dg {

constexpr int kRowsPerBlock = 256;   // LM-head row block (two 128-row UMMAs)
constexpr int kMaxCanvas = 1024;     // largest canvas the acceptance kernel sorts
constexpr int kAcceptThreads = 1024; // threads of the combine / acceptance CTAs (>= kMaxCanvas)
// canvas rows merged per combine CTA, a warp each (the other warps of the
// CTA only take part in the acceptance): few merging warps per SM keep the
// merges' issue slots free, so a CTA merges kCombineRowsMin rows unless the
// B canvases then need more CTAs than the GPU has SMs
constexpr int kCombineRowsMin = 8;
inline int combine_rows_per_cta(int B, int L, int sms)
{
    const long need = (static_cast<long>(B) * L + sms - 1) / sms;
    return static_cast<int>(need < kCombineRowsMin ? kCombineRowsMin : need > 32 ? 32 : need);
}

// Host: whether the device-side checks are on (dg_set_device_checks).
int device_checks();

struct FoldArgs {
    int M, V, BN, ntn, total, n_slots;
    Partials part;
    StepSource src;
    uint64_t seed;
    int *counters;
    int ncounters;
};

struct CombineArgs {
    Partials part;
    int n_slots, ntn, total, M;   // slot s of a row = producer unit s (tile range tile_begin(s))
    float *H;
    int32_t *sample;
    int32_t *argmax;
    int *counters;      // [B] last-CTA counters, zeroed by the producer kernel
    int rows_per_cta;   // canvas rows merged per combine CTA (<= 32)
    // self-conditioning: per-(row, unit) parts [M][n_slots][kScDim] in, the
    // read-out sc [M][kScDim] out; both null without it
    const float *sc_part;
    float *sc_out;
};

struct AcceptArgs {
    int B, L, V;
    float bound;        // entropy bound b
    float threshold;    // stop threshold
    uint64_t seed;
    int step;           // single-step mode only
    int32_t *canvas;
    int32_t *prev_argmax;
    uint8_t *accepted;
    int32_t *n_accepted;
    float *mean_entropy;
    int32_t *stop;
    // block loop only (ctl == nullptr otherwise)
    LoopCtl *ctl;
    int32_t *done;
    int32_t *steps_taken;
    int32_t *out_argmax;
    int32_t *n_acc_hist;
    unsigned long long cond;   // cudaGraphConditionalHandle
    // device-side checks (dg_set_device_checks): the combine and acceptance
    // verify indices and finiteness and report DG_ERR_DEVICE to ws
    WsHeader *ws;
    int checks;
};

struct LmHeadArgs {
    int M, d, V;
    int BN;             // vocabulary columns per tile (multiple of 16)
    int ntn;            // vocabulary tiles per row block
    int total;          // tiles = row blocks * ntn
    int kblocks;        // k blocks of 128 bytes per row: d / 64 (bf16), d / 128 (FP8)
    int nbox_b;         // 64-column TMA boxes per W stage
    int x_3d;           // hidden states carry a step coordinate
    int fuse2;          // 2-SM UMMA kernel only: two adjacent tiles of a unit's
                        // range in one row block run as one tile of 2 BN columns
    // FP8 operands (E4M3 codes): logit = acc * row_scale[row] * col_scale[v];
    // both null for bf16 operands
    const float *row_scale;
    const float *col_scale;
    Partials part;
    StepSource src;
    uint64_t seed;
    WsHeader *ws;
    int *counters;
    int ncounters;
    // per-row lower bounds on the best Gumbel score, shared by the units of
    // one launch ([M] order-preserving keys, 0 = none; all 0 between
    // launches); null: not shared
    uint32_t *rowkey;
    int w_packed;       // W as [ceil(V / 128)][d][128] (2-SM kernels only)
    // self-conditioning read-out (lm_head_duo_sc_kernel only): table E
    // [V, kScDim] bf16 and the per-(row, unit) parts [M][units][kScDim] fp32
    const uint16_t *sc_table;
    float *sc_part;
};

// LM-head kernel geometry
constexpr int kLmStages = 4;
constexpr int kLmBK = 64;
constexpr int kLmABytes = kRowsPerBlock * kLmBK * 2;     // 32 KB
constexpr int kLmBBoxBytes = 64 * kLmBK * 2;             // 8 KB
constexpr int kLmBBytes = 2 * kLmBBoxBytes;              // 16 KB
constexpr int kLmStageBytes = kLmABytes + kLmBBytes;
constexpr int kLmEpiWarps = 16;                          // 2 per (row half, TMEM quadrant)
constexpr int kLmColGroups = kLmEpiWarps / 8;             // column groups per row
constexpr int kLmThreads = 128 + 32 * kLmEpiWarps;        // 640
constexpr int kLmMergeBytes = (kLmColGroups - 1) * 7 * kRowsPerBlock * 4;   // 7 KB
constexpr int kLmSmemBytes = kLmStages * kLmStageBytes + 1024 + 256 + kLmMergeBytes;

__global__ void lm_head_kernel(const __grid_constant__ CUtensorMap map_x,
                               const __grid_constant__ CUtensorMap map_w, LmHeadArgs a);

// Shared-memory geometry of the 2-CTA cluster kernels: each CTA of the pair
// stages its own 128 X rows per k block; the epilogue's column groups merge
// through up to (4 - 1) x 7 x 128 floats.
constexpr int kPairABytes = 128 * kLmBK * 2;             // 16 KB: X rows of this CTA
constexpr int kPairColGroups = 4;                        // largest epilogue column-group count
constexpr int kPairMergeBytes = (kPairColGroups - 1) * 7 * 128 * 4;     // 10.5 KB

// 2-SM UMMA variant (tcgen05 cta_group::2): each CTA of the pair loads its
// own 128 rows of X and 128 of the 256 W columns of a tile; the even CTA
// issues 256 x 256 x 16 UMMAs over both CTAs' shared memory.
constexpr int kDuoStages = 6;
// Epilogue of the 2-SM kernel: 4 x CG warps (CG column groups per TMEM lane
// quadrant).  With one 256-row block every tile brings new W columns from
// HBM, the stream sets the tile rate and the fold hides under it: 8 warps
// (CG = 2) suffice and leave the producer and MMA warps more issue slots.
// With several row blocks the W tiles come from L2, the tiles arrive at the
// MMA rate and the fold's latency shows: 16 warps (CG = 4).  FP8 tiles carry
// half the bytes and take the UMMA issue as their limit: 12 warps (CG = 3)
// fold a tile well inside the MMA's time for it and leave the MMA warp more
// issue slots than 16 do (measured: 8 warps fold too slowly, 16 slow the MMA).
constexpr int kDuoCGNarrow = 2;
constexpr int kDuoCGWide = 4;
constexpr int kDuoCGFp8 = 3;
template <int kCG>
struct DuoEpilogue {
    static constexpr int CG = kCG;
    static constexpr int Warps = 4 * kCG;
    static constexpr int Threads = 128 + 32 * Warps;
};
constexpr int kDuoStageBytes = kPairABytes + 2 * kLmBBoxBytes;      // 32 KB
constexpr int kDuoSmemBytes = kDuoStages * kDuoStageBytes + 1024 + 256 + kPairMergeBytes;
__global__ void lm_head_duo_kernel(const __grid_constant__ CUtensorMap map_x,
                                   const __grid_constant__ CUtensorMap map_w, LmHeadArgs a);
// the same kernel with 16 epilogue warps (several row blocks)
__global__ void lm_head_duo_wide_kernel(const __grid_constant__ CUtensorMap map_x,
                                        const __grid_constant__ CUtensorMap map_w, LmHeadArgs a);
// The 8-epilogue-warp kernel with the self-conditioning read-out folded in:
// its column groups merge kScDim more words per row through shared memory,
// and the TMA producer stages the table rows of each tile's columns (one
// box of kDuoScETileRows / 2 rows x kScDim bf16 per 128 columns) into one
// of two buffers, so the fold reads them from shared memory; every epilogue
// warp has a 1 KB staging buffer for its chunk's weights; the ring has
// kDuoScStages stages to make room.
constexpr int kDuoScStages = 5;
constexpr int kDuoScETileRows = 256;
constexpr int kDuoScSmemBytes = kDuoScStages * kDuoStageBytes + 1024 + 256 +
                                (kDuoCGNarrow - 1) * 7 * 128 * 4 +
                                (kDuoCGNarrow - 1) * kScDim * 128 * 4 +
                                2 * kDuoScETileRows * kScDim * 2 + 4 * kDuoCGNarrow * 32 * 16 * 2;
static_assert(kDuoScSmemBytes <= 227 * 1024, "self-conditioning LM head: shared memory");
__global__ void lm_head_duo_sc_kernel(const __grid_constant__ CUtensorMap map_x,
                                      const __grid_constant__ CUtensorMap map_w,
                                      const __grid_constant__ CUtensorMap map_e, LmHeadArgs a);
// FP8 (E4M3) operands of the 2-SM kernel: X8 [M, d] and W8t [V, d] (both
// K-major, 128-byte k blocks = 128 codes); same tiles, 256 x 256 x 32 UMMAs.
__global__ void lm_head_duo_fp8_kernel(const __grid_constant__ CUtensorMap map_x,
                                       const __grid_constant__ CUtensorMap map_w, LmHeadArgs a);
// Per-row E4M3 quantisation of bf16 rows [rows, cols] (one warp per row) and of
// the columns of W [d, V] into W8t [V, d] (column maxima, then 32 x 32 tiles).
__global__ void quantize_rows_e4m3_kernel(const uint16_t *__restrict__ x, int64_t rows, int cols,
                                          uint8_t *__restrict__ q, float *__restrict__ scale);
constexpr int kQuantVecs = 16;   // 16-byte vectors per thread of the vector row kernel
__global__ void quantize_rows_e4m3_vec_kernel(const uint16_t *__restrict__ x, int cols,
                                              uint8_t *__restrict__ q, float *__restrict__ scale);
__global__ void pack_lm_weight_kernel(const uint16_t *__restrict__ w, int d, int V,
                                      uint16_t *__restrict__ wp);
__global__ void column_amax_kernel(const uint16_t *__restrict__ w, int d, int V,
                                   float *__restrict__ amax);
__global__ void quantize_cols_e4m3_kernel(const uint16_t *__restrict__ w, int d, int V,
                                          const float *__restrict__ amax,
                                          uint8_t *__restrict__ w8t);
__global__ void scale_from_amax_kernel(float *__restrict__ s, int n);
__global__ void logits_fold_kernel(const float *__restrict__ logits, FoldArgs a);
__global__ void combine_accept_kernel(CombineArgs c, AcceptArgs a);
__global__ void accept_only_kernel(const float *__restrict__ H, const int32_t *__restrict__ sample,
                                   const int32_t *__restrict__ argmax, AcceptArgs a);
__global__ void loop_init_kernel(LoopCtl *ctl, int max_steps, double t0, double t1, int B,
                                 int32_t *done, int32_t *steps_taken, int32_t *canvas,
                                 int32_t *prev_argmax, int n, uint32_t V, uint32_t k0,
                                 uint32_t k1);
__global__ void gumbel_fill_kernel(uint32_t k0, uint32_t k1, uint32_t row, uint32_t step,
                                   uint32_t v0, int n, float *out);
__global__ void logf_eval_kernel(const float *x, float *y, int n);
__global__ void wait_probe_kernel(WsHeader *ws, uint64_t limit_ns);
__global__ void hidden_from_steps_kernel(const int32_t *step, const uint16_t *__restrict__ src,
                                         int64_t step_stride, int64_t n, uint16_t *__restrict__ out);
__global__ void hidden_embed_add_kernel(const int32_t *step, const int32_t *__restrict__ canvas,
                                        const uint16_t *__restrict__ base, int64_t base_step_stride,
                                        const uint16_t *__restrict__ table, int rows, int d, int V,
                                        uint16_t *__restrict__ out);

// ---------------------------------------------------------------- attention
struct AttnArgs {
    int B, L, P, Hq, Hkv, D;
    int G;              // Hq / Hkv
    int rows;           // folded query rows per (b, g): L * G
    int mtiles;         // ceil(rows / 128)
    int nsplit;         // key splits
    int nkt_p, nkt_c;   // key tiles in the prefix / canvas
    int tiles_per_split;
    float scale_log2;   // scale * log2(e)
    int checks;         // device-side checks (dg_set_device_checks)
    int causal;         // canvas keys after a query's position are masked (cache append)
    const uint16_t *q;  // [B, L, Hq, D]
    uint16_t *out;      // [B, L, Hq, D] (nsplit == 1)
    uint16_t *part_o;   // [nsplit][B*L*Hq][D] bf16, each split's rows normalised by its sum (nsplit > 1)
    float *part_ml;     // [nsplit][B*L*Hq][2] (row max in base 2, row sum)
    WsHeader *ws;
};

constexpr int kAttnThreads = 224;    // warp 0 K loads, 1 MMA, 2-5 softmax, 6 V loads

__global__ void attn_kernel_d128(const __grid_constant__ CUtensorMap map_kp,
                                 const __grid_constant__ CUtensorMap map_vp,
                                 const __grid_constant__ CUtensorMap map_kc,
                                 const __grid_constant__ CUtensorMap map_vc, AttnArgs a);
__global__ void attn_kernel_d256(const __grid_constant__ CUtensorMap map_kp,
                                 const __grid_constant__ CUtensorMap map_vp,
                                 const __grid_constant__ CUtensorMap map_kc,
                                 const __grid_constant__ CUtensorMap map_vc, AttnArgs a);
__global__ void attn_combine_kernel(AttnArgs a);
// 2-CTA clusters issuing 2-SM UMMAs: two consecutive query tiles share every
// 128-key tile (dg_attn_pair.cu)
__global__ void attn_pair_kernel_d128(const __grid_constant__ CUtensorMap map_q,
                                      const __grid_constant__ CUtensorMap map_kp,
                                      const __grid_constant__ CUtensorMap map_vp,
                                      const __grid_constant__ CUtensorMap map_kc,
                                      const __grid_constant__ CUtensorMap map_vc, AttnArgs a);
__global__ void attn_pair_kernel_d256(const __grid_constant__ CUtensorMap map_q,
                                      const __grid_constant__ CUtensorMap map_kp,
                                      const __grid_constant__ CUtensorMap map_vp,
                                      const __grid_constant__ CUtensorMap map_kc,
                                      const __grid_constant__ CUtensorMap map_vc, AttnArgs a);
int attn_pair_smem_bytes(int D);

int attn_smem_bytes(int D);

// ---------------------------------------------------------------- MoE FFN
constexpr int kMoeMaxExperts = 128;    // routed experts (plus one shared)
constexpr int kMoeMaxTopK = 8;
constexpr int kMoeMaxTokens = 2048;    // canvas rows per call
constexpr int kMoeChunk = 128;         // tokens per token tile of the expert GEMMs
constexpr int kMoeRouteThreads = 1024;
constexpr int kMoeRouterKSlice = 128;  // k values per router CTA (d % 128 == 0)
// token chunks of one call: every expert's tokens in chunks of kMoeChunk
constexpr int kMoeMaxChunks =
    kMoeMaxExperts + 1 + (kMoeMaxTokens * (kMoeMaxTopK + 1) + kMoeChunk - 1) / kMoeChunk;

struct MoeArgs {
    int M, d, f, E, top_k;
    int checks;                 // device-side checks (dg_set_device_checks)
    const uint16_t *x;          // [M, d] bf16
    float *logits;              // [M, E] router logits
    int32_t *sel_expert;        // [M, top_k] chosen experts, best first
    float *sel_gate;            // [M, top_k] their gates
    int32_t *pos_of;            // [M, top_k] row of each assignment in the sorted order
    int32_t *tok_of_pos;        // [M (top_k + 1)] token of each sorted row
    float *gate_of_pos;         // [M (top_k + 1)] gate of each sorted row (1: shared)
    int4 *items;                // work list (expert, tile | chunk << 8, first row, tokens)
    int32_t *counts;            // [4]: gate/up items, all items, sorted rows
    int32_t *next_item;         // work-list counter of the FFN kernel
    uint32_t *ready;            // [kMoeMaxChunks] H parts stored per chunk
    uint32_t *bits;             // [E][ceil(M / 32)] token bitmaps of the experts (0 between calls)
    float *router_part;         // [d / kMoeRouterKSlice][M][E] partial router logits
    uint16_t *x_sorted;         // [M (top_k + 1), d] bf16
    uint16_t *h_sorted;         // [M (top_k + 1), f] bf16
    float *y_sorted;            // [M (top_k + 1), d] fp32, gate applied
    float *out;                 // [M, d] fp32
    WsHeader *ws;
};

// router: maps of the router weight [E, d] and of x [M, d], box {64, 128}
__global__ void moe_router_kernel(const __grid_constant__ CUtensorMap map_wr,
                                  const __grid_constant__ CUtensorMap map_x, MoeArgs a);
int moe_router_smem_bytes();
__global__ void moe_topk_kernel(MoeArgs a, int nslices);
__global__ void moe_route_kernel(MoeArgs a);
__global__ void moe_gather_kernel(MoeArgs a);
__global__ void moe_combine_kernel(MoeArgs a);
// Tensor maps of the expert GEMMs: gate / up weights [E+1, f, d] as
// {d, f, E+1}, box {64, 128, 1}; down weights [E+1, d, f] as {f, d, E+1},
// box {64, 128, 1}; X_sorted / H_sorted as {d or f, rows} with boxes of
// {64, 16 << i} rows (a token chunk loads the smallest box that holds it).
constexpr int kMoeBoxes = 4;
struct MoeMaps {
    CUtensorMap wg, wu, wd;
    CUtensorMap xs[kMoeBoxes];
    CUtensorMap hs[kMoeBoxes];
};
__global__ void moe_ffn_kernel(const __grid_constant__ MoeMaps maps, MoeArgs a);
int moe_ffn_smem_bytes();

}  // namespace dg
