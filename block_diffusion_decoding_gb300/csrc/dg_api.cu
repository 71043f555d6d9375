// dg_api.cu -- the C ABI of libdg.so (declared in include/dg.h): argument
// validation, workspace layout, TMA tensor-map encoding, kernel launches and
// the CUDA graph of the block loop.  Host code only; kernels live in the
// other .cu files.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <vector>

#include "dg_kernels.h"
#include "dg_plan.h"

using namespace dg;

namespace {

// ---------------------------------------------------------------- small utilities
constexpr int kAssumedMaxSMs = 256;  // workspace queries do not touch the GPU

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }
inline uint64_t f2u(float f)
{
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return u;
}
inline uint64_t d2u(double f)
{
    uint64_t u;
    std::memcpy(&u, &f, 8);
    return u;
}

#define DG_CUDA_TRY(expr)                                  \
    do {                                                   \
        cudaError_t e_ = (expr);                           \
        if (e_ != cudaSuccess) {                           \
            (void)cudaGetLastError();                      \
            return DG_ERR_CUDA;                            \
        }                                                  \
    } while (0)

struct DeviceInfo {
    int sms = 0;
    bool attrs_set = false;
};

std::mutex g_mu;
// dg_set_device_checks: read when a call enqueues its kernels
std::atomic<int> g_checks{0};
std::map<int, DeviceInfo> g_dev;
std::atomic<uint64_t> g_launches{0};

// Every kernel launch goes through here so the library can count them.
#define DG_LAUNCHED() g_launches.fetch_add(1, std::memory_order_relaxed)

int current_device_info(DeviceInfo **out)
{
    int dev = 0;
    DG_CUDA_TRY(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo &di = g_dev[dev];
    if (di.sms == 0) {
        DG_CUDA_TRY(cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev));
    }
    if (!di.attrs_set) {
        DG_CUDA_TRY(cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kLmSmemBytes));
        DG_CUDA_TRY(cudaFuncSetAttribute(lm_head_duo_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kDuoSmemBytes));
        DG_CUDA_TRY(cudaFuncSetAttribute(lm_head_duo_wide_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kDuoSmemBytes));
        DG_CUDA_TRY(cudaFuncSetAttribute(lm_head_duo_sc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kDuoScSmemBytes));
        DG_CUDA_TRY(cudaFuncSetAttribute(lm_head_duo_fp8_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kDuoSmemBytes));
        DG_CUDA_TRY(cudaFuncSetAttribute(moe_router_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         moe_router_smem_bytes()));
        DG_CUDA_TRY(cudaFuncSetAttribute(moe_ffn_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         moe_ffn_smem_bytes()));
        DG_CUDA_TRY(cudaFuncSetAttribute(attn_kernel_d128,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         attn_smem_bytes(128)));
        DG_CUDA_TRY(cudaFuncSetAttribute(attn_kernel_d256,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         attn_smem_bytes(256)));
        DG_CUDA_TRY(cudaFuncSetAttribute(attn_pair_kernel_d128,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         attn_pair_smem_bytes(128)));
        DG_CUDA_TRY(cudaFuncSetAttribute(attn_pair_kernel_d256,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         attn_pair_smem_bytes(256)));
        di.attrs_set = true;
    }
    *out = &di;
    return DG_OK;
}

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

// Tensor map with 128-byte swizzle.  dims/strides innermost first;
// strides[i] is the byte stride of dimension i+1.
int make_map_sw128(CUtensorMap *map, CUtensorMapDataType dt, const void *base, int rank,
                   const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return DG_ERR_CUDA;
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    CUresult r = fn(map, dt, static_cast<cuuint32_t>(rank),
                    const_cast<void *>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DG_OK : DG_ERR_CUDA;
}

// bf16 rows without swizzle (the self-conditioning table's tiles).
int make_map_bf16_plain(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer)
{
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return DG_ERR_CUDA;
    const cuuint64_t d[2] = {inner, outer};
    const cuuint64_t st[1] = {inner * 2};
    const cuuint32_t b[2] = {box_inner, box_outer};
    const cuuint32_t e[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), d, st, b, e,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DG_OK : DG_ERR_CUDA;
}

int make_map_bf16(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                  const uint64_t *strides_bytes, const uint32_t *box)
{
    return make_map_sw128(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides_bytes,
                          box);
}

// E4M3 codes are moved as bytes.
int make_map_u8(CUtensorMap *map, const void *base, int rank, const uint64_t *dims,
                const uint64_t *strides_bytes, const uint32_t *box)
{
    return make_map_sw128(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rank, dims, strides_bytes, box);
}

// Workspace layout of one step: header | partials (7 x n_slots x M x 4 B) |
// counters (B ints) | row keys (M u32: the Gumbel lower bounds the LM-head
// units share within a launch).
struct StepWs {
    WsHeader *hdr;
    Partials part;
    int *counters;
    uint32_t *rowkey;
};

size_t step_ws_bytes(int M, int B, int slots)
{
    size_t b = sizeof(WsHeader);
    b += round_up(static_cast<size_t>(7) * slots * M * 4, 256);
    b += round_up(static_cast<size_t>(B) * 4, 256);
    b += round_up(static_cast<size_t>(M) * 4, 256);
    return b;
}

StepWs carve_step_ws(void *ws, int M, int B, int slots)
{
    StepWs w{};
    uint8_t *p = static_cast<uint8_t *>(ws);
    w.hdr = reinterpret_cast<WsHeader *>(p);
    p += sizeof(WsHeader);
    const size_t n = static_cast<size_t>(slots) * M;
    float *f = reinterpret_cast<float *>(p);
    w.part.m = f;
    w.part.S = f + n;
    w.part.A = f + 2 * n;
    w.part.gbest = f + 3 * n;
    w.part.amax = f + 4 * n;
    w.part.gidx = reinterpret_cast<int *>(f + 5 * n);
    w.part.aidx = reinterpret_cast<int *>(f + 6 * n);
    p += round_up(7 * n * 4, 256);
    w.counters = reinterpret_cast<int *>(p);
    p += round_up(static_cast<size_t>(B) * 4, 256);
    w.rowkey = reinterpret_cast<uint32_t *>(p);
    return w;
}

int check_step_params(const dg_step_params *p)
{
    if (p == nullptr) return DG_ERR_INVALID_ARG;
    if (p->B < 1 || p->L < 1 || p->V < 1 || p->d < 1) return DG_ERR_INVALID_ARG;
    if (!(p->temperature > 0.0) || !std::isfinite(p->temperature)) return DG_ERR_INVALID_ARG;
    if (!(p->entropy_bound >= 0.f) || !std::isfinite(p->entropy_bound)) return DG_ERR_INVALID_ARG;
    if (!std::isfinite(p->stop_threshold)) return DG_ERR_INVALID_ARG;
    if (p->step < 0) return DG_ERR_INVALID_ARG;
    if (p->w_layout != DG_W_ROWMAJOR && p->w_layout != DG_W_PACKED) return DG_ERR_INVALID_ARG;
    if (p->L > kMaxCanvas) return DG_ERR_UNSUPPORTED;
    if (p->V % 8 != 0 || p->V < 64) return DG_ERR_UNSUPPORTED;
    if (static_cast<long long>(p->B) * p->L > (1LL << 30)) return DG_ERR_UNSUPPORTED;
    return DG_OK;
}

int check_io(const dg_step_io *io, bool need_outputs)
{
    if (io == nullptr) return DG_ERR_INVALID_ARG;
    if (!io->canvas || !io->prev_argmax || !io->accepted || !io->n_accepted || !io->mean_entropy ||
        !io->stop)
        return DG_ERR_INVALID_ARG;
    if (need_outputs && (!io->argmax || !io->sample || !io->entropy)) return DG_ERR_INVALID_ARG;
    return DG_OK;
}

StepSource step_source(const dg_step_params *p)
{
    StepSource s{};
    s.ctl = nullptr;
    s.invT = static_cast<float>(1.0 / p->temperature);
    s.c2 = s.invT * 1.44269502162933349609375f;   // fp32(log2 e)
    s.step = p->step;
    return s;
}

AcceptArgs accept_args(const dg_step_params *p, const dg_step_io *io)
{
    AcceptArgs a{};
    a.B = p->B;
    a.L = p->L;
    a.V = p->V;
    a.bound = p->entropy_bound;
    a.threshold = p->stop_threshold;
    a.seed = p->seed;
    a.step = p->step;
    a.canvas = io->canvas;
    a.prev_argmax = io->prev_argmax;
    a.accepted = io->accepted;
    a.n_accepted = io->n_accepted;
    a.mean_entropy = io->mean_entropy;
    a.stop = io->stop;
    return a;
}

// E4M3 operands of the LM head: X8 [M, d] with row scales, W8t [V, d] with
// column scales.
struct Fp8Operands {
    const uint8_t *x8;
    const float *sx;
    const uint8_t *w8t;
    const float *sw;
};

// Self-conditioning read-out of the step: the table E [V, kScDim], the
// per-(row, unit) parts in the workspace and the read-out [M, kScDim].
struct ScOperands {
    const uint16_t *table;
    float *part;
    float *out;
};

// Enqueue LM head (or logits fold) + combine/accept for one step.
int enqueue_step(const uint16_t *hidden, int64_t hidden_stride, int x_steps, const float *logits,
                 const uint16_t *w, const dg_step_params *p, const LmPlan &plan, StepWs &ws,
                 const StepSource &src, float *H, int32_t *sample, int32_t *argmax,
                 const AcceptArgs &acc, cudaStream_t st, bool lm_only = false,
                 const Fp8Operands *f8 = nullptr, const ScOperands *sco = nullptr)
{
    const int M = p->B * p->L;
    const bool pdl = use_pdl(st);
    if (f8 != nullptr) {
        CUtensorMap mx, mw;
        {
            const uint64_t dims[2] = {static_cast<uint64_t>(p->d), static_cast<uint64_t>(M)};
            const uint64_t strides[1] = {static_cast<uint64_t>(p->d)};
            const uint32_t box[2] = {128, 128};
            int rc = make_map_u8(&mx, f8->x8, 2, dims, strides, box);
            if (rc != DG_OK) return rc;
        }
        {
            const uint64_t dims[2] = {static_cast<uint64_t>(p->d), static_cast<uint64_t>(p->V)};
            const uint64_t strides[1] = {static_cast<uint64_t>(p->d)};
            const uint32_t box[2] = {128, static_cast<uint32_t>(plan.BN / 2)};
            int rc = make_map_u8(&mw, f8->w8t, 2, dims, strides, box);
            if (rc != DG_OK) return rc;
        }
        LmHeadArgs a{};
        a.M = M;
        a.d = p->d;
        a.V = p->V;
        a.BN = plan.BN;
        a.ntn = plan.ntn;
        a.total = plan.total;
        a.kblocks = p->d / 128;
        a.nbox_b = 1;
        a.x_3d = 0;
        a.row_scale = f8->sx;
        a.col_scale = f8->sw;
        a.part = ws.part;
        a.src = src;
        a.seed = p->seed;
        a.ws = ws.hdr;
        a.counters = ws.counters;
        a.ncounters = p->B;
        a.rowkey = ws.rowkey;
        a.fuse2 = plan.kind == kLmDuoFused ? 1 : 0;
        DG_CUDA_TRY(launch_lm_head(plan, mx, mw, a, st, pdl, true));
        DG_LAUNCHED();
    } else if (logits == nullptr) {
        CUtensorMap mx, mw;
        {
            const uint64_t dims[3] = {static_cast<uint64_t>(p->d), static_cast<uint64_t>(M),
                                      static_cast<uint64_t>(x_steps)};
            const uint64_t strides[2] = {static_cast<uint64_t>(p->d) * 2,
                                         static_cast<uint64_t>(hidden_stride) * 2};
            const uint32_t box[3] = {64, plan.cluster() ? 128u : 256u, 1};
            const int rank = x_steps > 1 ? 3 : 2;
            int rc = make_map_bf16(&mx, hidden, rank, dims, strides, box);
            if (rc != DG_OK) return rc;
        }
        const bool packed = p->w_layout == DG_W_PACKED;
        if (packed) {
            // [ceil(V / 128)][d][128]: 64 x 64 boxes inside one 128-column tile
            const uint64_t dims[3] = {128, static_cast<uint64_t>(p->d),
                                      static_cast<uint64_t>((p->V + 127) / 128)};
            const uint64_t strides[2] = {256, static_cast<uint64_t>(p->d) * 256};
            const uint32_t box[3] = {64, 64, 1};
            int rc = make_map_bf16(&mw, w, 3, dims, strides, box);
            if (rc != DG_OK) return rc;
        } else {
            const uint64_t dims[2] = {static_cast<uint64_t>(p->V), static_cast<uint64_t>(p->d)};
            const uint64_t strides[1] = {static_cast<uint64_t>(p->V) * 2};
            const uint32_t box[2] = {64, 64};
            int rc = make_map_bf16(&mw, w, 2, dims, strides, box);
            if (rc != DG_OK) return rc;
        }
        LmHeadArgs a{};
        a.w_packed = packed ? 1 : 0;
        a.M = M;
        a.d = p->d;
        a.V = p->V;
        a.BN = plan.BN;
        a.ntn = plan.ntn;
        a.total = plan.total;
        a.kblocks = p->d / 64;
        a.nbox_b = (plan.BN + 63) / 64;
        a.x_3d = x_steps > 1 ? 1 : 0;
        a.part = ws.part;
        a.src = src;
        a.seed = p->seed;
        a.ws = ws.hdr;
        a.counters = ws.counters;
        a.ncounters = p->B;
        a.rowkey = ws.rowkey;
        a.fuse2 = plan.kind == kLmDuoFused ? 1 : 0;
        if (sco != nullptr) {
            a.sc_table = sco->table;
            a.sc_part = sco->part;
            CUtensorMap me;
            int rc = make_map_bf16_plain(&me, sco->table, kScDim, static_cast<uint64_t>(p->V),
                                         kScDim, kDuoScETileRows / 2);
            if (rc != DG_OK) return rc;
            DG_CUDA_TRY(launch_kernel(lm_head_duo_sc_kernel, dim3(plan.grid),
                                      dim3(DuoEpilogue<kDuoCGNarrow>::Threads), kDuoScSmemBytes,
                                      st, pdl, mx, mw, me, a));
        } else {
            DG_CUDA_TRY(launch_lm_head(plan, mx, mw, a, st, pdl));
        }
        DG_LAUNCHED();
    } else {
        FoldArgs f{};
        f.M = M;
        f.V = p->V;
        f.BN = plan.BN;
        f.ntn = plan.ntn;
        f.total = plan.total;
        f.n_slots = plan.units;
        f.part = ws.part;
        f.src = src;
        f.seed = p->seed;
        f.counters = ws.counters;
        f.ncounters = p->B;
        logits_fold_kernel<<<plan.units, 256, 0, st>>>(logits, f);
        DG_LAUNCHED();
    }
    DG_CUDA_TRY(cudaGetLastError());
    if (lm_only) return DG_OK;
    CombineArgs c{};
    c.part = ws.part;
    // one partial state per (row, producer unit)
    c.n_slots = plan.units;
    c.ntn = plan.ntn;
    c.total = plan.total;
    c.M = M;
    c.H = H;
    c.sample = sample;
    c.argmax = argmax;
    c.counters = ws.counters;
    c.rows_per_cta = combine_rows_per_cta(p->B, p->L, plan.sms);
    if (sco != nullptr) {
        c.sc_part = sco->part;
        c.sc_out = sco->out;
    }
    AcceptArgs acc_c = acc;
    acc_c.ws = ws.hdr;
    acc_c.checks = g_checks.load(std::memory_order_relaxed);
    DG_CUDA_TRY(launch_kernel(combine_accept_kernel, dim3((p->L + c.rows_per_cta - 1) / c.rows_per_cta, p->B), dim3(kAcceptThreads), 0, st,
                              pdl, c, acc_c));
    DG_LAUNCHED();
    DG_CUDA_TRY(cudaGetLastError());
    return DG_OK;
}

// ---------------------------------------------------------------- attention plan
struct AttnPlan {
    bool pair;   // 2-CTA clusters issuing 2-SM UMMAs (attn_pair_kernel_*)
    int BKV, nkt_p, nkt_c, nkt, mtiles, blocks, nsplit, tps;
};

// Largest split count any plan may take: enough CTAs for two waves on a GPU
// with kAssumedMaxSMs SMs, and at most one KV tile per split.  The workspace
// query sizes the split partials with it.
int attn_split_cap(int blocks, int nkt)
{
    const int cap = (2 * kAssumedMaxSMs + blocks - 1) / blocks;
    return std::max(1, std::min(cap, nkt));
}

// max_ctas > 0: no split count that would launch more CTAs than that.
AttnPlan plan_attn(int B, int L, int P, int Hq, int Hkv, int D, int sms, int max_ctas = 0)
{
    AttnPlan a{};
    // head dim 256: the 2-SM pair kernel (its 128-key S UMMAs replace 64-key
    // ones; measured 35.5 vs 39.6 us at 16/8 heads, 4096 cached keys); head
    // dim 128: one CTA per query tile (the pair measured 2 us slower there).
    // DG_ATTN_KERNEL=single|pair forces a choice.
    const char *envk = std::getenv("DG_ATTN_KERNEL");
    a.pair = envk ? std::strcmp(envk, "pair") == 0 : D == 256;
    a.BKV = (a.pair || D == 128) ? 128 : 64;
    a.nkt_p = (P + a.BKV - 1) / a.BKV;
    a.nkt_c = (L + a.BKV - 1) / a.BKV;
    a.nkt = a.nkt_p + a.nkt_c;
    const int G = Hq / Hkv;
    a.mtiles = (L * G + 127) / 128;
    if (a.pair) a.mtiles += a.mtiles & 1;   // query tiles in pairs
    a.blocks = a.mtiles * Hkv * B;
    // splits: minimise the estimated time in key-tile units -- waves x (tiles
    // per split + a fixed cost of about 3 tiles per CTA) + about 4 tiles for
    // the split combine -- preferring fewer splits; never more than two
    // waves' worth of CTAs on the largest GPU
    long best = -1;
    const char *env = std::getenv("DG_ATTN_SPLITS");
    const int forced = env ? std::atoi(env) : 0;
    const int cap = attn_split_cap(a.blocks, a.nkt);
    for (int ns = 1; ns <= cap; ++ns) {
        const int tps = (a.nkt + ns - 1) / ns;
        const int real = (a.nkt + tps - 1) / tps;
        if (real != ns) continue;
        if (forced && ns != std::min(forced, a.nkt)) continue;
        if (max_ctas > 0 && ns > 1 && static_cast<long>(a.blocks) * ns > max_ctas) continue;
        const long waves = (static_cast<long>(a.blocks) * ns + sms - 1) / sms;
        const long cost = (waves * (tps + 3) + (ns > 1 ? 4 : 0)) * 16 + ns;
        if (best < 0 || cost < best) {
            best = cost;
            a.nsplit = ns;
            a.tps = tps;
        }
    }
    if (best < 0) {   // forced split count not realisable: no split
        a.nsplit = 1;
        a.tps = a.nkt;
    }
    return a;
}

size_t attn_ws_bytes(int B, int L, int Hq, int D, int nsplit)
{
    size_t b = sizeof(WsHeader);
    if (nsplit > 1) {
        const size_t nr = static_cast<size_t>(B) * L * Hq;
        b += round_up(static_cast<size_t>(nsplit) * nr * D * 2, 256);
        b += round_up(static_cast<size_t>(nsplit) * nr * 8, 256);
    }
    return b;
}

// ---------------------------------------------------------------- block-loop graph cache
// One instantiated loop graph per key (pointers, shapes, parameters, plan,
// producer); beyond kMaxBlockGraphs the least recently used is dropped.  A
// call holds its own reference while it launches and records `done` after
// the launch; a dropped graph is freed once its last launch has completed.
struct BlockGraph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    cudaEvent_t done = nullptr;
};

void release_block_graph(BlockGraph *g)
{
    if (g->done) {
        cudaEventSynchronize(g->done);
        cudaEventDestroy(g->done);
    }
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    (void)cudaGetLastError();
    delete g;
}

struct BlockGraphEntry {
    std::shared_ptr<BlockGraph> g;
    uint64_t last_use = 0;
};

constexpr size_t kMaxBlockGraphs = 64;

// guarded by g_mu; never destroyed, so no CUDA call runs at process exit
std::map<std::vector<uint64_t>, BlockGraphEntry> &block_graphs()
{
    static auto *cache = new std::map<std::vector<uint64_t>, BlockGraphEntry>();
    return *cache;
}
uint64_t g_block_graph_clock = 0;

size_t block_ws_layout(const dg_step_params *p, int slots, size_t *off_ctl, size_t *off_scratch)
{
    const int M = p->B * p->L;
    size_t b = step_ws_bytes(M, p->B, slots);
    b = round_up(b, 256);
    *off_ctl = b;
    b += round_up(sizeof(LoopCtl), 256);
    *off_scratch = b;
    // H (M f32), sample, argmax, prev_argmax (M i32), accepted (M u8),
    // n_accepted, stop, done (B i32)
    b += round_up(static_cast<size_t>(M) * 4, 256) * 4;
    b += round_up(static_cast<size_t>(M), 256);
    b += round_up(static_cast<size_t>(p->B) * 4, 256) * 3;
    return b;
}

}  // namespace

// ====================================================================== C ABI
// Canvas attention over [prefix rows 0 .. P-1 ; canvas rows]; the prefix
// tensors hold prefix_alloc >= P rows per batch entry (a cache with room to
// grow); causal masks canvas keys after each query's position.
static int attn_run(const uint16_t *q, const uint16_t *k_prefix, const uint16_t *v_prefix,
             const uint16_t *k_canvas, const uint16_t *v_canvas, uint16_t *out, int B, int L, int P,
             int prefix_alloc, int Hq, int Hkv, int D, float scale, int causal, void *workspace,
             size_t workspace_bytes, void *stream, int max_ctas = 0)
{
    if (!q || !k_canvas || !v_canvas || !out) return DG_ERR_INVALID_ARG;
    if (B < 1 || L < 1 || P < 0 || Hq < 1 || Hkv < 1) return DG_ERR_INVALID_ARG;
    if (P > 0 && (!k_prefix || !v_prefix)) return DG_ERR_INVALID_ARG;
    if (!std::isfinite(scale)) return DG_ERR_INVALID_ARG;
    if (D != 128 && D != 256) return DG_ERR_UNSUPPORTED;
    if (Hq % Hkv != 0) return DG_ERR_UNSUPPORTED;
    const int G = Hq / Hkv;
    if (G > 16 || (G & (G - 1)) != 0) return DG_ERR_UNSUPPORTED;
    if (static_cast<long long>(B) * L * Hq > (1LL << 30) || P > (1 << 30)) return DG_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_canvas) || !aligned16(v_canvas) || !aligned16(out) ||
        (P > 0 && (!aligned16(k_prefix) || !aligned16(v_prefix))))
        return DG_ERR_ALIGNMENT;
    if (workspace == nullptr || workspace_bytes < dg_canvas_attn_workspace(B, L, P, Hq, Hkv, D))
        return DG_ERR_WORKSPACE;
    DeviceInfo *di = nullptr;
    int rc = current_device_info(&di);
    if (rc != DG_OK) return rc;
    const AttnPlan ap = plan_attn(B, L, P, Hq, Hkv, D, di->sms, max_ctas);
    cudaStream_t st = as_stream(stream);

    CUtensorMap mq, mkp, mvp, mkc, mvc;
    {
        // Q [B, L, Hq, D] as {D, G, Hkv, L, B}: a box is 64 dims x the G heads
        // of one kv head x 128 / G positions (one folded 128-row tile)
        const uint64_t dims[5] = {static_cast<uint64_t>(D), static_cast<uint64_t>(G),
                                  static_cast<uint64_t>(Hkv), static_cast<uint64_t>(L),
                                  static_cast<uint64_t>(B)};
        const uint64_t strides[4] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(G) * D * 2,
                                     static_cast<uint64_t>(Hq) * D * 2,
                                     static_cast<uint64_t>(L) * Hq * D * 2};
        const uint32_t box[5] = {64, static_cast<uint32_t>(G), 1, static_cast<uint32_t>(128 / G), 1};
        if ((rc = make_map_bf16(&mq, q, 5, dims, strides, box)) != DG_OK) return rc;
    }
    // K / V [B, rows, Hkv, D] as {D, Hkv, rows, B}; the pair kernel stages
    // half a key tile of K and a full key tile of half the dims of V per CTA
    const uint32_t k_rows = static_cast<uint32_t>(ap.pair ? ap.BKV / 2 : ap.BKV);
    const uint32_t v_rows = static_cast<uint32_t>(ap.BKV);
    auto kv_map = [&](CUtensorMap *m, const uint16_t *base, int rows, int rows_alloc,
                      uint32_t box_rows) -> int {
        const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hkv),
                                  static_cast<uint64_t>(rows), static_cast<uint64_t>(B)};
        const uint64_t strides[3] = {static_cast<uint64_t>(D) * 2,
                                     static_cast<uint64_t>(Hkv) * D * 2,
                                     static_cast<uint64_t>(rows_alloc) * Hkv * D * 2};
        const uint32_t box[4] = {64, 1, box_rows, 1};
        return make_map_bf16(m, base, 4, dims, strides, box);
    };
    if ((rc = kv_map(&mkc, k_canvas, L, L, k_rows)) != DG_OK) return rc;
    if ((rc = kv_map(&mvc, v_canvas, L, L, v_rows)) != DG_OK) return rc;
    if (P > 0) {
        if ((rc = kv_map(&mkp, k_prefix, P, prefix_alloc, k_rows)) != DG_OK) return rc;
        if ((rc = kv_map(&mvp, v_prefix, P, prefix_alloc, v_rows)) != DG_OK) return rc;
    } else {
        mkp = mkc;
        mvp = mvc;
    }
    AttnArgs a{};
    a.B = B;
    a.L = L;
    a.P = P;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.G = G;
    a.rows = L * G;
    a.mtiles = ap.mtiles;
    a.nsplit = ap.nsplit;
    a.nkt_p = ap.nkt_p;
    a.nkt_c = ap.nkt_c;
    a.tiles_per_split = ap.tps;
    a.scale_log2 = scale * 1.44269502162933349609375f;
    a.causal = causal;
    a.checks = g_checks.load(std::memory_order_relaxed);
    a.q = q;
    a.out = out;
    a.ws = static_cast<WsHeader *>(workspace);
    if (ap.nsplit > 1) {
        uint8_t *p = static_cast<uint8_t *>(workspace) + sizeof(WsHeader);
        const size_t nr = static_cast<size_t>(B) * L * Hq;
        a.part_o = reinterpret_cast<uint16_t *>(p);
        a.part_ml = reinterpret_cast<float *>(
            p + round_up(static_cast<size_t>(ap.nsplit) * nr * D * 2, 256));
    }
    const bool pdl = use_pdl(st);
    const dim3 grid(ap.mtiles, Hkv * B, ap.nsplit);
    if (ap.pair)
        DG_CUDA_TRY(launch_kernel(D == 128 ? attn_pair_kernel_d128 : attn_pair_kernel_d256, grid,
                                  dim3(kAttnThreads), attn_pair_smem_bytes(D), st, pdl, mq, mkp,
                                  mvp, mkc, mvc, a));
    else
        DG_CUDA_TRY(launch_kernel(D == 128 ? attn_kernel_d128 : attn_kernel_d256, grid,
                                  dim3(kAttnThreads), attn_smem_bytes(D), st, pdl, mkp, mvp, mkc,
                                  mvc, a));
    DG_LAUNCHED();
    if (ap.nsplit > 1) {
        const size_t nr = static_cast<size_t>(B) * L * Hq;
        DG_CUDA_TRY(launch_kernel(attn_combine_kernel, dim3(static_cast<unsigned>((nr + 7) / 8)),
                                  dim3(256), 0, st, pdl, a));
        DG_LAUNCHED();
    }
    return DG_OK;
}

namespace {

int check_fp8_step(const uint16_t *hidden, const uint8_t *w8t, const float *w_scale,
                   const dg_step_params *p)
{
    int rc = check_step_params(p);
    if (rc != DG_OK) return rc;
    if (!hidden || !w8t || !w_scale) return DG_ERR_INVALID_ARG;
    if (p->d % 128 != 0 || p->d > 16384) return DG_ERR_UNSUPPORTED;
    if (!aligned16(hidden) || !aligned16(w8t) || !aligned16(w_scale)) return DG_ERR_ALIGNMENT;
    return DG_OK;
}

// Row quantisation: the register-resident vector kernel where the shapes and
// alignments allow it, else one warp per row.
cudaError_t launch_quantize_rows(const uint16_t *x, int64_t rows, int cols, uint8_t *q, float *scale,
                                 cudaStream_t st, bool pdl)
{
    const bool vec = cols % 8 == 0 && cols <= 128 * 8 * kQuantVecs && aligned16(x) &&
                     (reinterpret_cast<uintptr_t>(q) & 7u) == 0 && rows <= 0x7FFFFFFF;
    cudaError_t e;
    if (vec)
        e = launch_kernel(quantize_rows_e4m3_vec_kernel, dim3(static_cast<unsigned>(rows)),
                          dim3(128), 0, st, pdl, x, cols, q, scale);
    else
        e = launch_kernel(quantize_rows_e4m3_kernel, dim3(static_cast<unsigned>((rows + 7) / 8)),
                          dim3(256), 0, st, pdl, x, rows, cols, q, scale);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e;
}

// Workspace of the FP8 step: the step's | X8 [M, d] | row scales [M].
size_t fp8_ws_bytes(const dg_step_params *p, size_t *off_x8, size_t *off_sx)
{
    const size_t M = static_cast<size_t>(p->B) * p->L;
    size_t off = round_up(step_ws_bytes(static_cast<int>(M), p->B, slot_bound(static_cast<int>(M), p->V)), 256);
    if (off_x8) *off_x8 = off;
    off += round_up(M * p->d, 256);
    if (off_sx) *off_sx = off;
    return off + round_up(M * 4, 256);
}

int fp8_step(const uint16_t *hidden, const uint8_t *w8t, const float *w_scale,
             const dg_step_params *p, const dg_step_io *io, void *workspace,
             size_t workspace_bytes, void *stream, bool lm_only)
{
    int rc = check_fp8_step(hidden, w8t, w_scale, p);
    if (rc != DG_OK) return rc;
    if (!lm_only && (rc = check_io(io, true)) != DG_OK) return rc;
    size_t off_x8 = 0, off_sx = 0;
    const size_t need = fp8_ws_bytes(p, &off_x8, &off_sx);
    if (workspace == nullptr || workspace_bytes < need) return DG_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DG_ERR_ALIGNMENT;
    DeviceInfo *di = nullptr;
    if ((rc = current_device_info(&di)) != DG_OK) return rc;
    const int M = p->B * p->L;
    const LmPlan plan = plan_lm_head(M, p->d, p->V, di->sms, true);
    StepWs ws = carve_step_ws(workspace, M, p->B, plan.part_slots());
    Fp8Operands f8{};
    f8.x8 = static_cast<uint8_t *>(workspace) + off_x8;
    f8.sx = reinterpret_cast<const float *>(static_cast<uint8_t *>(workspace) + off_sx);
    f8.w8t = w8t;
    f8.sw = w_scale;
    cudaStream_t st = as_stream(stream);
    // the hidden states of this step are quantised per canvas row first
    DG_CUDA_TRY(launch_quantize_rows(hidden, M, p->d, const_cast<uint8_t *>(f8.x8),
                                     const_cast<float *>(f8.sx), st, use_pdl(st)));
    DG_LAUNCHED();
    const StepSource src = step_source(p);
    if (lm_only) {
        AcceptArgs acc{};
        return enqueue_step(nullptr, 0, 1, nullptr, nullptr, p, plan, ws, src, nullptr, nullptr,
                            nullptr, acc, st, true, &f8);
    }
    const AcceptArgs acc = accept_args(p, io);
    return enqueue_step(nullptr, 0, 1, nullptr, nullptr, p, plan, ws, src, io->entropy, io->sample,
                        io->argmax, acc, st, false, &f8);
}

// Workspace of the self-conditioning step: the step's | SC parts
// [M][slots][kScDim] fp32.
size_t sc_ws_bytes(const dg_step_params *p, size_t *off_sc)
{
    const size_t M = static_cast<size_t>(p->B) * p->L;
    const int slots = slot_bound(static_cast<int>(M), p->V);
    const size_t off = round_up(step_ws_bytes(static_cast<int>(M), p->B, slots), 256);
    if (off_sc) *off_sc = off;
    return off + round_up(static_cast<size_t>(slots) * M * kScDim * 4, 256);
}

int sc_step(const uint16_t *hidden, const uint16_t *w, const uint16_t *sc_table,
            const dg_step_params *p, const dg_step_io *io, float *sc_out, void *workspace,
            size_t workspace_bytes, void *stream, bool lm_only)
{
    int rc = check_step_params(p);
    if (rc != DG_OK) return rc;
    if (!lm_only && (rc = check_io(io, true)) != DG_OK) return rc;
    if (!hidden || !w || !sc_table || (!lm_only && !sc_out)) return DG_ERR_INVALID_ARG;
    if (p->d % 64 != 0 || p->d < 64 || p->d > 16384) return DG_ERR_UNSUPPORTED;
    if (!aligned16(hidden) || !aligned16(w) || !aligned16(sc_table) ||
        (!lm_only && !aligned16(sc_out)))
        return DG_ERR_ALIGNMENT;
    size_t off_sc = 0;
    const size_t need = sc_ws_bytes(p, &off_sc);
    if (workspace == nullptr || workspace_bytes < need) return DG_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DG_ERR_ALIGNMENT;
    DeviceInfo *di = nullptr;
    if ((rc = current_device_info(&di)) != DG_OK) return rc;
    const int M = p->B * p->L;
    const LmPlan plan = plan_lm_head(M, p->d, p->V, di->sms, false, true, -1,
                                     p->w_layout == DG_W_PACKED);
    StepWs ws = carve_step_ws(workspace, M, p->B, plan.part_slots());
    ScOperands sco{sc_table, reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + off_sc),
                   sc_out};
    const StepSource src = step_source(p);
    if (lm_only) {
        AcceptArgs acc{};
        return enqueue_step(hidden, 0, 1, nullptr, w, p, plan, ws, src, nullptr, nullptr, nullptr,
                            acc, as_stream(stream), true, nullptr, &sco);
    }
    const AcceptArgs acc = accept_args(p, io);
    return enqueue_step(hidden, 0, 1, nullptr, w, p, plan, ws, src, io->entropy, io->sample,
                        io->argmax, acc, as_stream(stream), false, nullptr, &sco);
}

// ---------------------------------------------------------------- MoE FFN
int moe_chunks_cap(int M, int E, int K)
{
    return E + 1 + (M * (K + 1) + kMoeChunk - 1) / kMoeChunk;
}

struct MoeWs {
    size_t logits, sel_e, sel_g, pos_of, tok, gate, items, counts, next, ready, bits, rpart, xs, hs,
        ys, total;
};

MoeWs moe_ws_layout(const dg_moe_params *p)
{
    const size_t M = p->M, K = p->top_k, E = p->n_experts, d = p->d, f = p->f;
    const size_t R = M * (K + 1);
    const size_t items = static_cast<size_t>(moe_chunks_cap(p->M, p->n_experts, p->top_k)) *
                         (f / 128 + d / 128);
    MoeWs w{};
    size_t o = sizeof(WsHeader);
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o += round_up(bytes, 256);
        return at;
    };
    w.logits = take(M * E * 4);
    w.sel_e = take(M * K * 4);
    w.sel_g = take(M * K * 4);
    w.pos_of = take(M * K * 4);
    w.tok = take(R * 4);
    w.gate = take(R * 4);
    w.items = take(items * 16);
    w.counts = take(16);
    w.next = take(4);
    w.ready = take(static_cast<size_t>(kMoeMaxChunks) * 4);
    w.bits = take(E * ((M + 31) / 32) * 4);
    w.rpart = take((d / kMoeRouterKSlice) * M * E * 4);
    w.xs = take(R * d * 2);
    w.hs = take(R * f * 2);
    w.ys = take(R * d * 4);
    w.total = o;
    return w;
}

int check_moe_params(const dg_moe_params *p)
{
    if (p == nullptr) return DG_ERR_INVALID_ARG;
    if (p->M < 1 || p->d < 1 || p->f < 1 || p->n_experts < 1 || p->top_k < 1)
        return DG_ERR_INVALID_ARG;
    if (p->top_k > p->n_experts) return DG_ERR_INVALID_ARG;
    if (p->M > kMoeMaxTokens || p->n_experts > kMoeMaxExperts || p->top_k > kMoeMaxTopK)
        return DG_ERR_UNSUPPORTED;
    if (p->d % kMoeRouterKSlice != 0 || p->d > 16384 || p->f % 128 != 0 || p->f > 16384)
        return DG_ERR_UNSUPPORTED;
    return DG_OK;
}

}  // namespace

int dg::device_checks() { return g_checks.load(std::memory_order_relaxed); }

extern "C" {

const char *dg_status_string(int status)
{
    switch (status) {
    case DG_OK: return "ok";
    case DG_ERR_INVALID_ARG: return "invalid argument";
    case DG_ERR_UNSUPPORTED: return "unsupported shape";
    case DG_ERR_ALIGNMENT: return "tensor pointer not 16-byte aligned";
    case DG_ERR_WORKSPACE: return "workspace missing or too small";
    case DG_ERR_CUDA: return "CUDA runtime error";
    case DG_ERR_TIMEOUT: return "device wait timed out";
    case DG_ERR_DEVICE: return "device-side check failed";
    default: return "unknown status";
    }
}

int dg_version(void) { return 100; }

int dg_set_device_checks(int on)
{
    g_checks.store(on != 0 ? 1 : 0, std::memory_order_relaxed);
    return DG_OK;
}

int dg_device_checks(void) { return g_checks.load(std::memory_order_relaxed); }

int dg_read_device_status(const void *workspace, int *status_out, int clear, void *stream)
{
    if (workspace == nullptr || status_out == nullptr) return DG_ERR_INVALID_ARG;
    int32_t v = 0;
    cudaStream_t st = as_stream(stream);
    DG_CUDA_TRY(cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st));
    DG_CUDA_TRY(cudaStreamSynchronize(st));
    *status_out = v;
    if (clear) {
        DG_CUDA_TRY(cudaMemsetAsync(const_cast<void *>(workspace), 0, sizeof(WsHeader), st));
        DG_CUDA_TRY(cudaStreamSynchronize(st));
    }
    return DG_OK;
}

// ---------------------------------------------------------------- attention
size_t dg_canvas_attn_workspace(int B, int L, int P, int Hq, int Hkv, int D)
{
    if (B < 1 || L < 1 || P < 0 || Hq < 1 || Hkv < 1 || (D != 128 && D != 256) || Hq % Hkv)
        return 0;
    const int G = Hq / Hkv;
    if (G > 16 || (G & (G - 1)) != 0) return 0;
    // the split count depends on the SM count: size for the largest allowed
    const int BKV = (D == 128) ? 128 : 64;
    const int nkt = (P + BKV - 1) / BKV + (L + BKV - 1) / BKV;
    const long blocks = static_cast<long>((L * G + 127) / 128) * Hkv * B;
    const int cap = attn_split_cap(static_cast<int>(std::min<long>(blocks, 1 << 30)), nkt);
    return attn_ws_bytes(B, L, Hq, D, cap);
}

int dg_canvas_attn(const uint16_t *q, const uint16_t *k_prefix, const uint16_t *v_prefix,
                   const uint16_t *k_canvas, const uint16_t *v_canvas, uint16_t *out, int B, int L,
                   int P, int Hq, int Hkv, int D, float scale, void *workspace,
                   size_t workspace_bytes, void *stream)
{
    return attn_run(q, k_prefix, v_prefix, k_canvas, v_canvas, out, B, L, P, P, Hq, Hkv, D, scale,
                    0, workspace, workspace_bytes, stream);
}

size_t dg_encoder_append_workspace(int B, int L, int P, int Hq, int Hkv, int D)
{
    return dg_canvas_attn_workspace(B, L, P, Hq, Hkv, D);
}

int dg_encoder_append(const uint16_t *q, uint16_t *k_cache, uint16_t *v_cache, int P, int P_max,
                      const uint16_t *k_new, const uint16_t *v_new, uint16_t *out, int B, int L,
                      int Hq, int Hkv, int D, float scale, void *workspace,
                      size_t workspace_bytes, void *stream)
{
    if (!k_cache || !v_cache || !k_new || !v_new) return DG_ERR_INVALID_ARG;
    if (P < 0 || L < 1 || B < 1 || Hkv < 1 || P_max < P + L) return DG_ERR_INVALID_ARG;
    if (D != 128 && D != 256) return DG_ERR_UNSUPPORTED;
    if (static_cast<long long>(P_max) * Hkv * D > (1LL << 31)) return DG_ERR_UNSUPPORTED;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return DG_ERR_ALIGNMENT;
    if (workspace == nullptr || workspace_bytes < dg_encoder_append_workspace(B, L, P, Hq, Hkv, D))
        return DG_ERR_WORKSPACE;
    cudaStream_t st = as_stream(stream);
    // append: cache rows [P, P + L) of every batch entry <- the block's K / V
    const size_t row_bytes = static_cast<size_t>(Hkv) * D * 2;
    const size_t off = static_cast<size_t>(P) * Hkv * D;
    DG_CUDA_TRY(cudaMemcpy2DAsync(k_cache + off, static_cast<size_t>(P_max) * row_bytes, k_new,
                                  static_cast<size_t>(L) * row_bytes,
                                  static_cast<size_t>(L) * row_bytes, static_cast<size_t>(B),
                                  cudaMemcpyDeviceToDevice, st));
    DG_CUDA_TRY(cudaMemcpy2DAsync(v_cache + off, static_cast<size_t>(P_max) * row_bytes, v_new,
                                  static_cast<size_t>(L) * row_bytes,
                                  static_cast<size_t>(L) * row_bytes, static_cast<size_t>(B),
                                  cudaMemcpyDeviceToDevice, st));
    // the block attends causally to [cache rows 0 .. P-1 ; its own rows]
    return attn_run(q, k_cache, v_cache, k_new, v_new, out, B, L, P, P_max, Hq, Hkv, D, scale, 1,
                    workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- one step
size_t dg_denoise_step_workspace(const dg_step_params *p)
{
    if (check_step_params(p) != DG_OK) return 0;
    const int M = p->B * p->L;
    return step_ws_bytes(M, p->B, slot_bound(M, p->V));
}

int dg_denoise_step(const uint16_t *hidden, const uint16_t *w, const dg_step_params *p,
                    const dg_step_io *io, void *workspace, size_t workspace_bytes, void *stream)
{
    int rc = check_step_params(p);
    if (rc != DG_OK) return rc;
    if ((rc = check_io(io, true)) != DG_OK) return rc;
    if (!hidden || !w) return DG_ERR_INVALID_ARG;
    if (p->d % 64 != 0 || p->d < 64 || p->d > 16384) return DG_ERR_UNSUPPORTED;
    if (!aligned16(hidden) || !aligned16(w)) return DG_ERR_ALIGNMENT;
    if (workspace == nullptr || workspace_bytes < dg_denoise_step_workspace(p))
        return DG_ERR_WORKSPACE;
    DeviceInfo *di = nullptr;
    if ((rc = current_device_info(&di)) != DG_OK) return rc;
    const int M = p->B * p->L;
    const LmPlan plan = plan_lm_head(M, p->d, p->V, di->sms, false, false, -1,
                                     p->w_layout == DG_W_PACKED);
    StepWs ws = carve_step_ws(workspace, M, p->B, plan.part_slots());
    const StepSource src = step_source(p);
    const AcceptArgs acc = accept_args(p, io);
    return enqueue_step(hidden, 0, 1, nullptr, w, p, plan, ws, src, io->entropy, io->sample,
                        io->argmax, acc, as_stream(stream));
}

int dg_lm_head_fold(const uint16_t *hidden, const uint16_t *w, const dg_step_params *p,
                    void *workspace, size_t workspace_bytes, void *stream)
{
    int rc = check_step_params(p);
    if (rc != DG_OK) return rc;
    if (!hidden || !w) return DG_ERR_INVALID_ARG;
    if (p->d % 64 != 0 || p->d < 64 || p->d > 16384) return DG_ERR_UNSUPPORTED;
    if (!aligned16(hidden) || !aligned16(w)) return DG_ERR_ALIGNMENT;
    if (workspace == nullptr || workspace_bytes < dg_denoise_step_workspace(p))
        return DG_ERR_WORKSPACE;
    DeviceInfo *di = nullptr;
    if ((rc = current_device_info(&di)) != DG_OK) return rc;
    const int M = p->B * p->L;
    const LmPlan plan = plan_lm_head(M, p->d, p->V, di->sms, false, false, -1,
                                     p->w_layout == DG_W_PACKED);
    StepWs ws = carve_step_ws(workspace, M, p->B, plan.part_slots());
    const StepSource src = step_source(p);
    AcceptArgs acc{};
    return enqueue_step(hidden, 0, 1, nullptr, w, p, plan, ws, src, nullptr, nullptr, nullptr,
                        acc, as_stream(stream), true);
}

uint64_t dg_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

// ---------------------------------------------------------------- FP8 LM head
int dg_quantize_rows_e4m3(const uint16_t *x, int64_t rows, int cols, uint8_t *codes, float *scale,
                          void *stream)
{
    if (!x || !codes || !scale || rows < 1 || cols < 1) return DG_ERR_INVALID_ARG;
    if (rows > (1LL << 31) * 8 - 8) return DG_ERR_UNSUPPORTED;
    DG_CUDA_TRY(launch_quantize_rows(x, rows, cols, codes, scale, as_stream(stream), false));
    DG_LAUNCHED();
    return DG_OK;
}

int dg_quantize_weight_e4m3(const uint16_t *w, int d, int V, uint8_t *w8t, float *scale,
                            void *stream)
{
    if (!w || !w8t || !scale || d < 1 || V < 1) return DG_ERR_INVALID_ARG;
    if (d > 65535 * 32) return DG_ERR_UNSUPPORTED;
    cudaStream_t st = as_stream(stream);
    column_amax_kernel<<<(V + 255) / 256, 256, 0, st>>>(w, d, V, scale);
    DG_LAUNCHED();
    quantize_cols_e4m3_kernel<<<dim3((V + 31) / 32, (d + 31) / 32), 256, 0, st>>>(w, d, V, scale,
                                                                                 w8t);
    DG_LAUNCHED();
    scale_from_amax_kernel<<<(V + 255) / 256, 256, 0, st>>>(scale, V);
    DG_LAUNCHED();
    DG_CUDA_TRY(cudaGetLastError());
    return DG_OK;
}

size_t dg_lm_weight_packed_bytes(int d, int V)
{
    if (d < 1 || V < 1) return 0;
    return static_cast<size_t>((V + 127) / 128) * static_cast<size_t>(d) * 128 * 2;
}

int dg_pack_lm_weight(const uint16_t *w, int d, int V, uint16_t *w_packed, void *stream)
{
    if (!w || !w_packed) return DG_ERR_INVALID_ARG;
    if (d % 64 != 0 || d < 64 || d > 16384 || V % 8 != 0 || V < 64) return DG_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(w_packed)) return DG_ERR_ALIGNMENT;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(w);
    const uintptr_t a1 = a0 + static_cast<size_t>(d) * V * 2;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(w_packed);
    const uintptr_t b1 = b0 + dg_lm_weight_packed_bytes(d, V);
    if (a0 < b1 && b0 < a1) return DG_ERR_INVALID_ARG;
    const int64_t chunks = static_cast<int64_t>((V + 127) / 128) * d * 16;
    const unsigned grid = static_cast<unsigned>(std::min<int64_t>((chunks + 255) / 256, 8192));
    pack_lm_weight_kernel<<<grid, 256, 0, as_stream(stream)>>>(w, d, V, w_packed);
    DG_LAUNCHED();
    DG_CUDA_TRY(cudaGetLastError());
    return DG_OK;
}

size_t dg_denoise_step_fp8_workspace(const dg_step_params *p)
{
    if (check_step_params(p) != DG_OK) return 0;
    return fp8_ws_bytes(p, nullptr, nullptr);
}

int dg_denoise_step_fp8(const uint16_t *hidden, const uint8_t *w8t, const float *w_scale,
                        const dg_step_params *p, const dg_step_io *io, void *workspace,
                        size_t workspace_bytes, void *stream)
{
    return fp8_step(hidden, w8t, w_scale, p, io, workspace, workspace_bytes, stream, false);
}

int dg_lm_head_fold_fp8(const uint16_t *hidden, const uint8_t *w8t, const float *w_scale,
                        const dg_step_params *p, void *workspace, size_t workspace_bytes,
                        void *stream)
{
    return fp8_step(hidden, w8t, w_scale, p, nullptr, workspace, workspace_bytes, stream, true);
}

int dg_lm_head_plan(int rows, int d, int V, int *kind, int *bn, int *ctas, int *epilogue_warps)
{
    if (rows < 1 || d < 1 || V < 1) return DG_ERR_INVALID_ARG;
    if (rows > (1 << 20) || V % 8 != 0 || V < 64) return DG_ERR_UNSUPPORTED;
    if (d % 64 != 0 || d > 16384) return DG_ERR_UNSUPPORTED;
    DeviceInfo *di = nullptr;
    const int rc = current_device_info(&di);
    if (rc != DG_OK) return rc;
    const LmPlan plan = plan_lm_head(rows, d, V, di->sms);
    if (kind) *kind = plan.kind;
    if (bn) *bn = plan.BN;
    if (ctas) *ctas = plan.grid;
    if (epilogue_warps) *epilogue_warps = plan.epi_warps;
    return DG_OK;
}

// ---------------------------------------------------------------- the whole step
namespace {

// The second stream and the fork / join events of dg_canvas_step, one set per
// device, made at the first call on it.
struct ForkStreams {
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    // a step's fork, launches and join are enqueued under this lock, so calls
    // from several host threads cannot interleave their event records
    std::mutex mu;
};
std::map<int, ForkStreams> g_fork;

int fork_streams(ForkStreams **out)
{
    int dev = 0;
    DG_CUDA_TRY(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(g_mu);
    ForkStreams &f = g_fork[dev];
    if (f.side == nullptr) {
        DG_CUDA_TRY(cudaStreamCreateWithFlags(&f.side, cudaStreamNonBlocking));
        DG_CUDA_TRY(cudaEventCreateWithFlags(&f.fork, cudaEventDisableTiming));
        DG_CUDA_TRY(cudaEventCreateWithFlags(&f.join, cudaEventDisableTiming));
    }
    *out = &f;
    return DG_OK;
}

// SMs set aside for the attention of the step: when its query tiles need at
// most an eighth of the SMs (else a sixth) and, with its key splits limited
// to that many CTAs, each CTA has at most kReserveTiles key tiles (a short
// attention that hides under the LM head), its CTAs keep their SMs and the
// LM head is planned on the others; else none (a longer attention shares the GPU with the LM head
// instead).  Measured: an eighth for the small step (P = 256), a sixth for
// P = 2048 at one canvas (43.3 -> 41.6 us); none for 4 canvases or 32768
// cached keys, where every reservation tried was slower.
constexpr int kReserveTiles = 6;
int attn_reserve(int B, int L, int P, int Hq, int Hkv, int D, int sms)
{
    // DG_ATTN_RESERVE=n forces n SMs (0: none) for the attention
    if (const char *env = std::getenv("DG_ATTN_RESERVE")) {
        const int n = std::atoi(env);
        return n > 0 && n <= sms - 2 ? n & ~1 : 0;
    }
    for (const int cap : {sms / 8, sms / 6}) {
        // the attention's CTAs with its key splits capped at `cap`; the LM
        // head is planned on every other SM
        const AttnPlan ap = plan_attn(B, L, P, Hq, Hkv, D, sms, cap);
        const int ctas = ap.blocks * ap.nsplit;
        if (ctas <= cap && ap.tps <= kReserveTiles) return (ctas + 1) & ~1;
    }
    return 0;
}

// The LM head's plan for the canvas step on the SMs a reservation leaves.
LmPlan canvas_lm_plan(const dg_step_params *p, int sms, int reserve)
{
    const int M = p->B * p->L;
    const bool packed = p->w_layout == DG_W_PACKED;
    LmPlan plan = plan_lm_head(M, p->d, p->V, sms - reserve, false, false, -1, packed);
    if (reserve > 0 && !packed && plan.kind != kLmSingle && std::getenv("DG_LM_KERNEL") == nullptr) {
        // one tile per CTA on the SMs left: the single-CTA kernel (its 16
        // epilogue warps fold a 256-row tile; measured faster than the 2-SM
        // kernel's 8 at one tile per CTA)
        const LmPlan single = plan_lm_head(M, p->d, p->V, sms - reserve, false, false, kLmSingle);
        if (single.units >= single.total) plan = single;
    }
    return plan;
}

// The canvas step's plan on a GPU with `sms` SMs: the SMs set aside for the
// attention (attn_reserve), the attention's plan on them and the LM head's on
// the rest.
struct CanvasStepPlan {
    int reserve;
    AttnPlan ap;
    LmPlan lm;
};

CanvasStepPlan plan_canvas_step(const dg_step_params *p, int P, int Hq, int Hkv, int D, int sms)
{
    int reserve = attn_reserve(p->B, p->L, P, Hq, Hkv, D, sms);
    if (reserve > 0 && std::getenv("DG_ATTN_RESERVE") == nullptr) {
        // fewer SMs for the attention when that lets the LM head run more,
        // narrower tiles and each of them still has at most 2 kReserveTiles of
        // the attention's key tiles to run (small step: 4 instead of 8 SMs,
        // 147 LM-head CTAs of 112 columns instead of 128 of 128)
        const AttnPlan ap = plan_attn(p->B, p->L, P, Hq, Hkv, D, sms, reserve);
        const int ctas = ap.blocks * ap.nsplit;
        const int units = canvas_lm_plan(p, sms, reserve).units;
        for (int r = 2; r < reserve; r += 2) {
            if ((ctas + r - 1) / r * ap.tps > 2 * kReserveTiles) continue;
            if (canvas_lm_plan(p, sms, r).units > units) {
                reserve = r;
                break;
            }
        }
    }
    CanvasStepPlan sp{};
    sp.reserve = reserve;
    sp.ap = plan_attn(p->B, p->L, P, Hq, Hkv, D, sms, reserve);
    sp.lm = canvas_lm_plan(p, sms, reserve);
    return sp;
}

}  // namespace

size_t dg_canvas_step_workspace(const dg_step_params *p, int P, int Hq, int Hkv, int D)
{
    if (check_step_params(p) != DG_OK) return 0;
    const size_t a = dg_canvas_attn_workspace(p->B, p->L, P, Hq, Hkv, D);
    if (a == 0) return 0;
    return round_up(dg_denoise_step_workspace(p), 256) + a;
}

int dg_canvas_step_plan(const dg_step_params *p, int P, int Hq, int Hkv, int D, int sms,
                        dg_canvas_step_plan_info *out)
{
    int rc = check_step_params(p);
    if (rc != DG_OK) return rc;
    if (out == nullptr || sms > kAssumedMaxSMs) return DG_ERR_INVALID_ARG;
    if (p->d % 64 != 0 || p->d < 64 || p->d > 16384) return DG_ERR_UNSUPPORTED;
    if (dg_canvas_step_workspace(p, P, Hq, Hkv, D) == 0) return DG_ERR_UNSUPPORTED;
    if (sms <= 0) {
        DeviceInfo *di = nullptr;
        if ((rc = current_device_info(&di)) != DG_OK) return rc;
        sms = di->sms;
    }
    const CanvasStepPlan sp = plan_canvas_step(p, P, Hq, Hkv, D, sms);
    dg_canvas_step_plan_info o{};
    o.attn_reserved_sms = sp.reserve;
    o.attn_pair = sp.ap.pair ? 1 : 0;
    o.attn_ctas = sp.ap.blocks * sp.ap.nsplit;
    o.attn_splits = sp.ap.nsplit;
    o.attn_key_tiles = sp.ap.tps;
    o.attn_key_tile = sp.ap.BKV;
    o.lm_kind = sp.lm.kind;
    o.lm_bn = sp.lm.BN;
    o.lm_ctas = sp.lm.grid;
    o.lm_tiles = sp.lm.total;
    o.lm_epilogue_warps = sp.lm.epi_warps;
    o.lm_sms = sp.lm.sms;
    *out = o;
    return DG_OK;
}

int dg_canvas_step(const uint16_t *q, const uint16_t *k_prefix, const uint16_t *v_prefix,
                   const uint16_t *k_canvas, const uint16_t *v_canvas, uint16_t *attn_out, int P,
                   int Hq, int Hkv, int D, float scale, const uint16_t *hidden, const uint16_t *w,
                   const dg_step_params *p, const dg_step_io *io, void *workspace,
                   size_t workspace_bytes, void *stream)
{
    int rc = check_step_params(p);
    if (rc != DG_OK) return rc;
    if ((rc = check_io(io, true)) != DG_OK) return rc;
    if (!hidden || !w) return DG_ERR_INVALID_ARG;
    if (p->d % 64 != 0 || p->d < 64 || p->d > 16384) return DG_ERR_UNSUPPORTED;
    if (!aligned16(hidden) || !aligned16(w) || !aligned16(workspace)) return DG_ERR_ALIGNMENT;
    const size_t need = dg_canvas_step_workspace(p, P, Hq, Hkv, D);
    if (need == 0) return DG_ERR_UNSUPPORTED;
    if (workspace == nullptr || workspace_bytes < need) return DG_ERR_WORKSPACE;
    DeviceInfo *di = nullptr;
    if ((rc = current_device_info(&di)) != DG_OK) return rc;
    ForkStreams *fs = nullptr;
    if ((rc = fork_streams(&fs)) != DG_OK) return rc;
    std::lock_guard<std::mutex> fork_lock(fs->mu);
    const size_t step_bytes = round_up(dg_denoise_step_workspace(p), 256);
    uint8_t *aws = static_cast<uint8_t *>(workspace) + step_bytes;
    cudaStream_t st = as_stream(stream);
    // attention on the second stream, forked from and joined back into `stream`
    DG_CUDA_TRY(cudaEventRecord(fs->fork, st));
    DG_CUDA_TRY(cudaStreamWaitEvent(fs->side, fs->fork, 0));
    const int M = p->B * p->L;
    const CanvasStepPlan sp = plan_canvas_step(p, P, Hq, Hkv, D, di->sms);
    rc = attn_run(q, k_prefix, v_prefix, k_canvas, v_canvas, attn_out, p->B, p->L, P, P, Hq, Hkv, D,
                  scale, 0, aws, workspace_bytes - step_bytes, fs->side, sp.reserve);
    if (rc == DG_OK) {
        const LmPlan &plan = sp.lm;
        StepWs ws = carve_step_ws(workspace, M, p->B, plan.part_slots());
        const StepSource src = step_source(p);
        const AcceptArgs acc = accept_args(p, io);
        rc = enqueue_step(hidden, 0, 1, nullptr, w, p, plan, ws, src, io->entropy, io->sample,
                          io->argmax, acc, st);
    }
    // the join is recorded whatever happened, so `stream` never waits on a stale fork
    DG_CUDA_TRY(cudaEventRecord(fs->join, fs->side));
    DG_CUDA_TRY(cudaStreamWaitEvent(st, fs->join, 0));
    return rc;
}

// ---------------------------------------------------------------- whole step, FP8 / self-conditioning
namespace {

// The canvas attention on the library's second stream, forked from and joined
// back into `stream`, beside step(stream, ctx) (the LM-head step; it gets the
// first step_bytes of the workspace, the attention the rest from offset
// step_bytes).  No SMs are set aside: the attention shares the GPU.
typedef int (*ForkStepFn)(cudaStream_t st, void *ctx);
int canvas_fork_run(const uint16_t *q, const uint16_t *k_prefix, const uint16_t *v_prefix,
                    const uint16_t *k_canvas, const uint16_t *v_canvas, uint16_t *attn_out, int P,
                    int Hq, int Hkv, int D, float scale, const dg_step_params *p, size_t step_bytes,
                    void *workspace, size_t workspace_bytes, void *stream, ForkStepFn step,
                    void *ctx)
{
    ForkStreams *fs = nullptr;
    int rc = fork_streams(&fs);
    if (rc != DG_OK) return rc;
    std::lock_guard<std::mutex> fork_lock(fs->mu);
    uint8_t *aws = static_cast<uint8_t *>(workspace) + step_bytes;
    cudaStream_t st = as_stream(stream);
    DG_CUDA_TRY(cudaEventRecord(fs->fork, st));
    DG_CUDA_TRY(cudaStreamWaitEvent(fs->side, fs->fork, 0));
    rc = attn_run(q, k_prefix, v_prefix, k_canvas, v_canvas, attn_out, p->B, p->L, P, P, Hq, Hkv, D,
                  scale, 0, aws, workspace_bytes - step_bytes, fs->side, 0);
    if (rc == DG_OK) rc = step(st, ctx);
    // the join is recorded whatever happened, so `stream` never waits on a stale fork
    DG_CUDA_TRY(cudaEventRecord(fs->join, fs->side));
    DG_CUDA_TRY(cudaStreamWaitEvent(st, fs->join, 0));
    return rc;
}

struct Fp8StepArgs {
    const uint16_t *hidden;
    const uint8_t *w8t;
    const float *w_scale;
    const dg_step_params *p;
    const dg_step_io *io;
    void *workspace;
    size_t bytes;
};

int fp8_fork_step(cudaStream_t st, void *ctx)
{
    const Fp8StepArgs *a = static_cast<const Fp8StepArgs *>(ctx);
    return fp8_step(a->hidden, a->w8t, a->w_scale, a->p, a->io, a->workspace, a->bytes, st, false);
}

struct ScStepArgs {
    const uint16_t *hidden, *w, *sc_table;
    const dg_step_params *p;
    const dg_step_io *io;
    float *sc_out;
    void *workspace;
    size_t bytes;
};

int sc_fork_step(cudaStream_t st, void *ctx)
{
    const ScStepArgs *a = static_cast<const ScStepArgs *>(ctx);
    return sc_step(a->hidden, a->w, a->sc_table, a->p, a->io, a->sc_out, a->workspace, a->bytes,
                   st, false);
}

}  // namespace

size_t dg_canvas_step_fp8_workspace(const dg_step_params *p, int P, int Hq, int Hkv, int D)
{
    if (check_step_params(p) != DG_OK) return 0;
    const size_t a = dg_canvas_attn_workspace(p->B, p->L, P, Hq, Hkv, D);
    if (a == 0) return 0;
    return round_up(fp8_ws_bytes(p, nullptr, nullptr), 256) + a;
}

int dg_canvas_step_fp8(const uint16_t *q, const uint16_t *k_prefix, const uint16_t *v_prefix,
                       const uint16_t *k_canvas, const uint16_t *v_canvas, uint16_t *attn_out,
                       int P, int Hq, int Hkv, int D, float scale, const uint16_t *hidden,
                       const uint8_t *w8t, const float *w_scale, const dg_step_params *p,
                       const dg_step_io *io, void *workspace, size_t workspace_bytes, void *stream)
{
    int rc = check_fp8_step(hidden, w8t, w_scale, p);
    if (rc != DG_OK) return rc;
    if ((rc = check_io(io, true)) != DG_OK) return rc;
    if (!aligned16(workspace)) return DG_ERR_ALIGNMENT;
    const size_t need = dg_canvas_step_fp8_workspace(p, P, Hq, Hkv, D);
    if (need == 0) return DG_ERR_UNSUPPORTED;
    if (workspace == nullptr || workspace_bytes < need) return DG_ERR_WORKSPACE;
    const size_t step_bytes = round_up(fp8_ws_bytes(p, nullptr, nullptr), 256);
    Fp8StepArgs args{hidden, w8t, w_scale, p, io, workspace, step_bytes};
    return canvas_fork_run(q, k_prefix, v_prefix, k_canvas, v_canvas, attn_out, P, Hq, Hkv, D,
                           scale, p, step_bytes, workspace, workspace_bytes, stream, fp8_fork_step,
                           &args);
}

size_t dg_canvas_step_sc_workspace(const dg_step_params *p, int P, int Hq, int Hkv, int D)
{
    if (check_step_params(p) != DG_OK) return 0;
    const size_t a = dg_canvas_attn_workspace(p->B, p->L, P, Hq, Hkv, D);
    if (a == 0) return 0;
    return round_up(sc_ws_bytes(p, nullptr), 256) + a;
}

int dg_canvas_step_sc(const uint16_t *q, const uint16_t *k_prefix, const uint16_t *v_prefix,
                      const uint16_t *k_canvas, const uint16_t *v_canvas, uint16_t *attn_out, int P,
                      int Hq, int Hkv, int D, float scale, const uint16_t *hidden,
                      const uint16_t *w, const uint16_t *sc_table, const dg_step_params *p,
                      const dg_step_io *io, float *sc_out, void *workspace,
                      size_t workspace_bytes, void *stream)
{
    int rc = check_step_params(p);
    if (rc != DG_OK) return rc;
    if ((rc = check_io(io, true)) != DG_OK) return rc;
    if (!hidden || !w || !sc_table || !sc_out) return DG_ERR_INVALID_ARG;
    if (p->d % 64 != 0 || p->d < 64 || p->d > 16384) return DG_ERR_UNSUPPORTED;
    if (!aligned16(hidden) || !aligned16(w) || !aligned16(sc_table) || !aligned16(sc_out) ||
        !aligned16(workspace))
        return DG_ERR_ALIGNMENT;
    const size_t need = dg_canvas_step_sc_workspace(p, P, Hq, Hkv, D);
    if (need == 0) return DG_ERR_UNSUPPORTED;
    if (workspace == nullptr || workspace_bytes < need) return DG_ERR_WORKSPACE;
    const size_t step_bytes = round_up(sc_ws_bytes(p, nullptr), 256);
    ScStepArgs args{hidden, w, sc_table, p, io, sc_out, workspace, step_bytes};
    return canvas_fork_run(q, k_prefix, v_prefix, k_canvas, v_canvas, attn_out, P, Hq, Hkv, D,
                           scale, p, step_bytes, workspace, workspace_bytes, stream, sc_fork_step,
                           &args);
}

// ---------------------------------------------------------------- self-conditioning step
size_t dg_denoise_step_sc_workspace(const dg_step_params *p)
{
    if (check_step_params(p) != DG_OK) return 0;
    return sc_ws_bytes(p, nullptr);
}

int dg_denoise_step_sc(const uint16_t *hidden, const uint16_t *w, const uint16_t *sc_table,
                       const dg_step_params *p, const dg_step_io *io, float *sc_out,
                       void *workspace, size_t workspace_bytes, void *stream)
{
    return sc_step(hidden, w, sc_table, p, io, sc_out, workspace, workspace_bytes, stream, false);
}

int dg_lm_head_fold_sc(const uint16_t *hidden, const uint16_t *w, const uint16_t *sc_table,
                       const dg_step_params *p, void *workspace, size_t workspace_bytes,
                       void *stream)
{
    return sc_step(hidden, w, sc_table, p, nullptr, nullptr, workspace, workspace_bytes, stream,
                   true);
}

// ---------------------------------------------------------------- MoE FFN
size_t dg_moe_ffn_workspace(const dg_moe_params *p)
{
    if (check_moe_params(p) != DG_OK) return 0;
    return moe_ws_layout(p).total;
}

int dg_moe_ffn(const uint16_t *x, const uint16_t *w_router, const uint16_t *w_gate,
               const uint16_t *w_up, const uint16_t *w_down, float *out, int32_t *experts_out,
               float *gates_out, const dg_moe_params *p, void *workspace, size_t workspace_bytes,
               void *stream)
{
    int rc = check_moe_params(p);
    if (rc != DG_OK) return rc;
    if (!x || !w_router || !w_gate || !w_up || !w_down || !out) return DG_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_router) || !aligned16(w_gate) || !aligned16(w_up) ||
        !aligned16(w_down) || !aligned16(out))
        return DG_ERR_ALIGNMENT;
    const MoeWs L = moe_ws_layout(p);
    if (workspace == nullptr || workspace_bytes < L.total) return DG_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DG_ERR_ALIGNMENT;
    DeviceInfo *di = nullptr;
    if ((rc = current_device_info(&di)) != DG_OK) return rc;
    uint8_t *base = static_cast<uint8_t *>(workspace);
    const int M = p->M, K = p->top_k, E = p->n_experts, d = p->d, f = p->f;
    const uint64_t R = static_cast<uint64_t>(M) * (K + 1);
    MoeArgs a{};
    a.checks = g_checks.load(std::memory_order_relaxed);
    a.M = M;
    a.d = d;
    a.f = f;
    a.E = E;
    a.top_k = K;
    a.x = x;
    a.logits = reinterpret_cast<float *>(base + L.logits);
    a.sel_expert = experts_out ? experts_out : reinterpret_cast<int32_t *>(base + L.sel_e);
    a.sel_gate = gates_out ? gates_out : reinterpret_cast<float *>(base + L.sel_g);
    a.pos_of = reinterpret_cast<int32_t *>(base + L.pos_of);
    a.tok_of_pos = reinterpret_cast<int32_t *>(base + L.tok);
    a.gate_of_pos = reinterpret_cast<float *>(base + L.gate);
    a.items = reinterpret_cast<int4 *>(base + L.items);
    a.counts = reinterpret_cast<int32_t *>(base + L.counts);
    a.next_item = reinterpret_cast<int32_t *>(base + L.next);
    a.ready = reinterpret_cast<uint32_t *>(base + L.ready);
    a.bits = reinterpret_cast<uint32_t *>(base + L.bits);
    a.router_part = reinterpret_cast<float *>(base + L.rpart);
    a.x_sorted = reinterpret_cast<uint16_t *>(base + L.xs);
    a.h_sorted = reinterpret_cast<uint16_t *>(base + L.hs);
    a.y_sorted = reinterpret_cast<float *>(base + L.ys);
    a.out = out;
    a.ws = static_cast<WsHeader *>(workspace);

    MoeMaps maps;
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(d), static_cast<uint64_t>(f),
                                  static_cast<uint64_t>(E + 1)};
        const uint64_t strides[2] = {static_cast<uint64_t>(d) * 2, static_cast<uint64_t>(f) * d * 2};
        const uint32_t box[3] = {64, 128, 1};
        if ((rc = make_map_bf16(&maps.wg, w_gate, 3, dims, strides, box)) != DG_OK) return rc;
        if ((rc = make_map_bf16(&maps.wu, w_up, 3, dims, strides, box)) != DG_OK) return rc;
    }
    {
        const uint64_t dims[3] = {static_cast<uint64_t>(f), static_cast<uint64_t>(d),
                                  static_cast<uint64_t>(E + 1)};
        const uint64_t strides[2] = {static_cast<uint64_t>(f) * 2, static_cast<uint64_t>(d) * f * 2};
        const uint32_t box[3] = {64, 128, 1};
        if ((rc = make_map_bf16(&maps.wd, w_down, 3, dims, strides, box)) != DG_OK) return rc;
    }
    for (int i = 0; i < kMoeBoxes; ++i) {
        const uint32_t rows = 16u << i;
        {
            const uint64_t dims[2] = {static_cast<uint64_t>(d), R};
            const uint64_t strides[1] = {static_cast<uint64_t>(d) * 2};
            const uint32_t box[2] = {64, rows};
            if ((rc = make_map_bf16(&maps.xs[i], a.x_sorted, 2, dims, strides, box)) != DG_OK) return rc;
        }
        {
            const uint64_t dims[2] = {static_cast<uint64_t>(f), R};
            const uint64_t strides[1] = {static_cast<uint64_t>(f) * 2};
            const uint32_t box[2] = {64, rows};
            if ((rc = make_map_bf16(&maps.hs[i], a.h_sorted, 2, dims, strides, box)) != DG_OK) return rc;
        }
    }
    cudaStream_t st = as_stream(stream);
    const bool pdl = use_pdl(st);
    CUtensorMap mwr, mx;
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(E)};
        const uint64_t strides[1] = {static_cast<uint64_t>(d) * 2};
        const uint32_t box[2] = {64, 128};
        if ((rc = make_map_bf16(&mwr, w_router, 2, dims, strides, box)) != DG_OK) return rc;
    }
    {
        const uint64_t dims[2] = {static_cast<uint64_t>(d), static_cast<uint64_t>(M)};
        const uint64_t strides[1] = {static_cast<uint64_t>(d) * 2};
        const uint32_t box[2] = {64, 128};
        if ((rc = make_map_bf16(&mx, x, 2, dims, strides, box)) != DG_OK) return rc;
    }
    const int nslices = d / kMoeRouterKSlice;
    DG_CUDA_TRY(launch_kernel(moe_router_kernel, dim3(nslices, (M + 127) / 128), dim3(128),
                              moe_router_smem_bytes(), st, pdl, mwr, mx, a));
    DG_LAUNCHED();
    DG_CUDA_TRY(launch_kernel(moe_topk_kernel, dim3((M + 7) / 8), dim3(256), 0, st, pdl, a,
                              nslices));
    DG_LAUNCHED();
    DG_CUDA_TRY(launch_kernel(moe_route_kernel, dim3(1), dim3(kMoeRouteThreads), 0, st, pdl, a));
    DG_LAUNCHED();
    const unsigned fill = static_cast<unsigned>(std::max(1, di->sms * 8));
    const uint64_t gvec = R * static_cast<uint64_t>(d / 8);
    DG_CUDA_TRY(launch_kernel(moe_gather_kernel,
                              dim3(static_cast<unsigned>(std::min<uint64_t>((gvec + 255) / 256, fill))),
                              dim3(256), 0, st, pdl, a));
    DG_LAUNCHED();
    DG_CUDA_TRY(launch_kernel(moe_ffn_kernel, dim3(di->sms), dim3(192), moe_ffn_smem_bytes(), st,
                              pdl, maps, a));
    DG_LAUNCHED();
    const uint64_t cvec = static_cast<uint64_t>(M) * (d / 4);
    DG_CUDA_TRY(launch_kernel(moe_combine_kernel,
                              dim3(static_cast<unsigned>(std::min<uint64_t>((cvec + 255) / 256, fill))),
                              dim3(256), 0, st, pdl, a));
    DG_LAUNCHED();
    return DG_OK;
}

// ---------------------------------------------------------------- sampler on given logits
size_t dg_sampler_workspace(const dg_step_params *p)
{
    if (check_step_params(p) != DG_OK) return 0;
    const int M = p->B * p->L;
    return step_ws_bytes(M, p->B, slot_bound(M, p->V));
}

int dg_sampler_from_logits(const float *logits, const dg_step_params *p, const dg_step_io *io,
                           void *workspace, size_t workspace_bytes, void *stream)
{
    int rc = check_step_params(p);
    if (rc != DG_OK) return rc;
    if ((rc = check_io(io, true)) != DG_OK) return rc;
    if (!logits) return DG_ERR_INVALID_ARG;
    if (!aligned16(logits)) return DG_ERR_ALIGNMENT;
    if (workspace == nullptr || workspace_bytes < dg_sampler_workspace(p)) return DG_ERR_WORKSPACE;
    DeviceInfo *di = nullptr;
    if ((rc = current_device_info(&di)) != DG_OK) return rc;
    const int M = p->B * p->L;
    const LmPlan plan = plan_lm_head(M, 64, p->V, di->sms);
    StepWs ws = carve_step_ws(workspace, M, p->B, plan.part_slots());
    const StepSource src = step_source(p);
    const AcceptArgs acc = accept_args(p, io);
    return enqueue_step(nullptr, 0, 1, logits, nullptr, p, plan, ws, src, io->entropy, io->sample,
                        io->argmax, acc, as_stream(stream));
}

int dg_accept_renoise(const float *entropy, const int32_t *sample, const int32_t *argmax,
                      const dg_step_params *p, const dg_step_io *io, void *workspace,
                      size_t workspace_bytes, void *stream)
{
    int rc = check_step_params(p);
    if (rc != DG_OK) return rc;
    if ((rc = check_io(io, false)) != DG_OK) return rc;
    if (!entropy || !sample || !argmax) return DG_ERR_INVALID_ARG;
    if (workspace == nullptr || workspace_bytes < sizeof(WsHeader)) return DG_ERR_WORKSPACE;
    AcceptArgs acc = accept_args(p, io);
    acc.ws = static_cast<WsHeader *>(workspace);
    acc.checks = g_checks.load(std::memory_order_relaxed);
    accept_only_kernel<<<p->B, kAcceptThreads, 0, as_stream(stream)>>>(entropy, sample, argmax, acc);
    DG_LAUNCHED();
    DG_CUDA_TRY(cudaGetLastError());
    return DG_OK;
}

// ---------------------------------------------------------------- block loop
size_t dg_generate_block_workspace(const dg_step_params *p, const dg_block_params *bp)
{
    if (check_step_params(p) != DG_OK || bp == nullptr) return 0;
    const int M = p->B * p->L;
    size_t oc, os;
    return block_ws_layout(p, slot_bound(M, p->V), &oc, &os);
}

// The block loop; hidden states either from hidden_steps (+ k * stride) or,
// with fn != null, from the caller's producer writing hidden_buf each step.
static int block_run(const uint16_t *hidden_steps, dg_hidden_fn fn, void *user, uint16_t *hidden_buf,
                     const uint16_t *w, const dg_step_params *p, const dg_block_params *bp,
                     const dg_block_io *io, void *workspace, size_t workspace_bytes, void *stream)
{
    int rc = check_step_params(p);
    if (rc != DG_OK) return rc;
    if (bp == nullptr || io == nullptr) return DG_ERR_INVALID_ARG;
    if (bp->max_steps < 1 || bp->max_steps > kMaxLoopSteps) return DG_ERR_UNSUPPORTED;
    if (!(bp->t_start > 0.0) || !(bp->t_end > 0.0)) return DG_ERR_INVALID_ARG;
    if (bp->hidden_step_stride < 0) return DG_ERR_INVALID_ARG;
    if (!io->canvas || !io->argmax || !io->steps_taken || !io->mean_entropy)
        return DG_ERR_INVALID_ARG;
    const uint16_t *hidden = fn != nullptr ? hidden_buf : hidden_steps;
    if (!hidden || !w) return DG_ERR_INVALID_ARG;
    if (p->d % 64 != 0 || p->d < 64 || p->d > 16384) return DG_ERR_UNSUPPORTED;
    if (!aligned16(hidden) || !aligned16(w)) return DG_ERR_ALIGNMENT;
    if (fn == nullptr && (bp->hidden_step_stride * 2) % 16 != 0) return DG_ERR_ALIGNMENT;
    if (workspace == nullptr || workspace_bytes < dg_generate_block_workspace(p, bp))
        return DG_ERR_WORKSPACE;
    DeviceInfo *di = nullptr;
    if ((rc = current_device_info(&di)) != DG_OK) return rc;
    const int M = p->B * p->L;
    const LmPlan plan = plan_lm_head(M, p->d, p->V, di->sms, false, false, -1,
                                     p->w_layout == DG_W_PACKED);
    size_t off_ctl, off_scr;
    block_ws_layout(p, slot_bound(M, p->V), &off_ctl, &off_scr);
    uint8_t *base = static_cast<uint8_t *>(workspace);
    StepWs ws = carve_step_ws(workspace, M, p->B, plan.part_slots());
    LoopCtl *ctl = reinterpret_cast<LoopCtl *>(base + off_ctl);
    uint8_t *sp = base + off_scr;
    const size_t m4 = round_up(static_cast<size_t>(M) * 4, 256);
    const size_t b4 = round_up(static_cast<size_t>(p->B) * 4, 256);
    float *H = reinterpret_cast<float *>(sp);
    int32_t *sample = reinterpret_cast<int32_t *>(sp + m4);
    int32_t *argmax = reinterpret_cast<int32_t *>(sp + 2 * m4);
    int32_t *prev = reinterpret_cast<int32_t *>(sp + 3 * m4);
    uint8_t *accepted = sp + 4 * m4;
    uint8_t *sp2 = sp + 4 * m4 + round_up(static_cast<size_t>(M), 256);
    int32_t *n_acc = reinterpret_cast<int32_t *>(sp2);
    int32_t *stop = reinterpret_cast<int32_t *>(sp2 + b4);
    int32_t *done = reinterpret_cast<int32_t *>(sp2 + 2 * b4);

    cudaStream_t st = as_stream(stream);
    const int x_steps = (fn == nullptr && bp->hidden_step_stride > 0) ? bp->max_steps : 1;
    const int64_t stride = fn == nullptr ? bp->hidden_step_stride : 0;

    int dev = 0;
    DG_CUDA_TRY(cudaGetDevice(&dev));
    const std::vector<uint64_t> key = {
        reinterpret_cast<uint64_t>(hidden), reinterpret_cast<uint64_t>(w),
        reinterpret_cast<uint64_t>(workspace), reinterpret_cast<uint64_t>(io->canvas),
        reinterpret_cast<uint64_t>(io->argmax), reinterpret_cast<uint64_t>(io->steps_taken),
        reinterpret_cast<uint64_t>(io->mean_entropy),
        reinterpret_cast<uint64_t>(io->n_accepted_hist), static_cast<uint64_t>(p->B),
        static_cast<uint64_t>(p->L), static_cast<uint64_t>(p->d), static_cast<uint64_t>(p->V),
        f2u(p->entropy_bound), f2u(p->stop_threshold), d2u(bp->t_start), d2u(bp->t_end), p->seed,
        static_cast<uint64_t>(bp->max_steps), static_cast<uint64_t>(stride),
        static_cast<uint64_t>(plan.BN), static_cast<uint64_t>(plan.grid * 4 + plan.kind),
        static_cast<uint64_t>(plan.epi_warps), static_cast<uint64_t>(p->w_layout),
        static_cast<uint64_t>(dev), reinterpret_cast<uint64_t>(fn),
        reinterpret_cast<uint64_t>(user),
        static_cast<uint64_t>(g_checks.load(std::memory_order_relaxed))};

    std::shared_ptr<BlockGraph> bgp;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto &cache = block_graphs();
        auto it = cache.find(key);
        if (it != cache.end()) {
            it->second.last_use = ++g_block_graph_clock;
            bgp = it->second.g;
        }
    }
    if (!bgp) {
        BlockGraph bg;
        DG_CUDA_TRY(cudaGraphCreate(&bg.graph, 0));
        cudaGraphConditionalHandle cond;
        if (cudaGraphConditionalHandleCreate(&cond, bg.graph, 1, cudaGraphCondAssignDefault) !=
            cudaSuccess) {
            (void)cudaGetLastError();
            cudaGraphDestroy(bg.graph);
            return DG_ERR_CUDA;
        }
        cudaGraphNodeParams np = {};
        np.type = cudaGraphNodeTypeConditional;
        np.conditional.handle = cond;
        np.conditional.type = cudaGraphCondTypeWhile;
        np.conditional.size = 1;
        cudaGraphNode_t wnode;
        cudaStream_t cap = nullptr;
        if (cudaGraphAddNode(&wnode, bg.graph, nullptr, nullptr, 0, &np) != cudaSuccess ||
            cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking) != cudaSuccess) {
            (void)cudaGetLastError();
            cudaGraphDestroy(bg.graph);
            return DG_ERR_CUDA;
        }
        cudaGraph_t body = np.conditional.phGraph_out[0];
        if (cudaStreamBeginCaptureToGraph(cap, body, nullptr, nullptr, 0,
                                          cudaStreamCaptureModeRelaxed) != cudaSuccess) {
            (void)cudaGetLastError();
            cudaStreamDestroy(cap);
            cudaGraphDestroy(bg.graph);
            return DG_ERR_CUDA;
        }
        StepSource src{};
        src.ctl = ctl;
        AcceptArgs acc{};
        acc.B = p->B;
        acc.L = p->L;
        acc.V = p->V;
        acc.bound = p->entropy_bound;
        acc.threshold = p->stop_threshold;
        acc.seed = p->seed;
        acc.canvas = io->canvas;
        acc.prev_argmax = prev;
        acc.accepted = accepted;
        acc.n_accepted = n_acc;
        acc.mean_entropy = io->mean_entropy;
        acc.stop = stop;
        acc.ctl = ctl;
        acc.done = done;
        acc.steps_taken = io->steps_taken;
        acc.out_argmax = io->argmax;
        acc.n_acc_hist = io->n_accepted_hist;
        acc.cond = cond;
        // the producer's work for step k (it reads k from the control block on
        // the device), then the step itself
        int erc = fn != nullptr ? fn(&ctl->step, io->canvas, hidden_buf, cap, user) : DG_OK;
        if (erc == DG_OK)
            erc = enqueue_step(hidden, stride, x_steps, nullptr, w, p, plan, ws, src, H, sample,
                               argmax, acc, cap);
        cudaGraph_t captured = nullptr;
        cudaError_t ce = cudaStreamEndCapture(cap, &captured);
        cudaStreamDestroy(cap);
        if (erc != DG_OK || ce != cudaSuccess) {
            (void)cudaGetLastError();
            cudaGraphDestroy(bg.graph);
            return erc != DG_OK ? erc : DG_ERR_CUDA;
        }
        if (cudaGraphInstantiate(&bg.exec, bg.graph, 0) != cudaSuccess) {
            (void)cudaGetLastError();
            cudaGraphDestroy(bg.graph);
            return DG_ERR_CUDA;
        }
        if (cudaEventCreateWithFlags(&bg.done, cudaEventDisableTiming) != cudaSuccess) {
            (void)cudaGetLastError();
            cudaGraphExecDestroy(bg.exec);
            cudaGraphDestroy(bg.graph);
            return DG_ERR_CUDA;
        }
        // released after the lock below: a graph another thread built
        // meanwhile, or the one dropped from the cache
        std::shared_ptr<BlockGraph> made(new BlockGraph(bg), release_block_graph);
        std::shared_ptr<BlockGraph> dropped;
        std::lock_guard<std::mutex> lk(g_mu);
        auto &cache = block_graphs();
        // another thread may have built the same graph meanwhile: keep that
        // one (this one is released when `made` goes out of scope)
        auto ins = cache.emplace(key, BlockGraphEntry{made, 0});
        ins.first->second.last_use = ++g_block_graph_clock;
        bgp = ins.first->second.g;
        if (cache.size() > kMaxBlockGraphs) {
            auto lru = cache.end();
            for (auto e = cache.begin(); e != cache.end(); ++e)
                if (e != ins.first && (lru == cache.end() || e->second.last_use < lru->second.last_use))
                    lru = e;
            if (lru != cache.end()) {
                dropped = lru->second.g;
                cache.erase(lru);
            }
        }
    }
    loop_init_kernel<<<std::max(1, (M + 255) / 256), 256, 0, st>>>(
        ctl, bp->max_steps, bp->t_start, bp->t_end, p->B, done, io->steps_taken, io->canvas, prev,
        M, static_cast<uint32_t>(p->V), static_cast<uint32_t>(p->seed),
        static_cast<uint32_t>(p->seed >> 32));
    DG_LAUNCHED();
    DG_CUDA_TRY(cudaGetLastError());
    DG_CUDA_TRY(cudaGraphLaunch(bgp->exec, st));
    DG_CUDA_TRY(cudaEventRecord(bgp->done, st));
    return DG_OK;
}

int dg_generate_block(const uint16_t *hidden_steps, const uint16_t *w, const dg_step_params *p,
                      const dg_block_params *bp, const dg_block_io *io, void *workspace,
                      size_t workspace_bytes, void *stream)
{
    return block_run(hidden_steps, nullptr, nullptr, nullptr, w, p, bp, io, workspace,
                     workspace_bytes, stream);
}

int dg_generate_block_fn(dg_hidden_fn produce_hidden, void *user, uint16_t *hidden_buf,
                         const uint16_t *w, const dg_step_params *p, const dg_block_params *bp,
                         const dg_block_io *io, void *workspace, size_t workspace_bytes,
                         void *stream)
{
    if (produce_hidden == nullptr) return DG_ERR_INVALID_ARG;
    return block_run(nullptr, produce_hidden, user, hidden_buf, w, p, bp, io, workspace,
                     workspace_bytes, stream);
}

int dg_hidden_from_steps(const int32_t *step, const int32_t *canvas, uint16_t *hidden_out,
                         void *stream, void *user)
{
    (void)canvas;
    const dg_hidden_steps *u = static_cast<const dg_hidden_steps *>(user);
    if (u == nullptr || step == nullptr || hidden_out == nullptr || u->hidden_steps == nullptr)
        return DG_ERR_INVALID_ARG;
    if (u->n < 1 || u->step_stride < 0) return DG_ERR_INVALID_ARG;
    const int64_t n = u->n;
    hidden_from_steps_kernel<<<static_cast<unsigned>(std::min<int64_t>((n + 255) / 256, 65535)),
                               256, 0, as_stream(stream)>>>(step, u->hidden_steps, u->step_stride,
                                                            n, hidden_out);
    DG_LAUNCHED();
    DG_CUDA_TRY(cudaGetLastError());
    return DG_OK;
}

int dg_hidden_embed_add(const int32_t *step, const int32_t *canvas, uint16_t *hidden_out,
                        void *stream, void *user)
{
    const dg_hidden_embed *u = static_cast<const dg_hidden_embed *>(user);
    if (u == nullptr || step == nullptr || canvas == nullptr || hidden_out == nullptr ||
        u->base == nullptr || u->table == nullptr)
        return DG_ERR_INVALID_ARG;
    if (u->rows < 1 || u->d < 1 || u->V < 1 || u->base_step_stride < 0) return DG_ERR_INVALID_ARG;
    const int64_t n = static_cast<int64_t>(u->rows) * u->d;
    hidden_embed_add_kernel<<<static_cast<unsigned>(std::min<int64_t>((n + 255) / 256, 65535)),
                              256, 0, as_stream(stream)>>>(step, canvas, u->base,
                                                           u->base_step_stride, u->table, u->rows,
                                                           u->d, u->V, hidden_out);
    DG_LAUNCHED();
    DG_CUDA_TRY(cudaGetLastError());
    return DG_OK;
}

// ---------------------------------------------------------------- check entries
int dg_gumbel_fill(uint64_t seed, uint32_t row, uint32_t step, uint32_t v0, int n, float *out,
                   void *stream)
{
    if (n < 0 || (n > 0 && out == nullptr)) return DG_ERR_INVALID_ARG;
    if (n == 0) return DG_OK;
    gumbel_fill_kernel<<<(n + 255) / 256, 256, 0, as_stream(stream)>>>(
        static_cast<uint32_t>(seed), static_cast<uint32_t>(seed >> 32), row, step, v0, n, out);
    DG_LAUNCHED();
    DG_CUDA_TRY(cudaGetLastError());
    return DG_OK;
}

int dg_logf_eval(const float *x, float *y, int n, void *stream)
{
    if (n < 0 || (n > 0 && (x == nullptr || y == nullptr))) return DG_ERR_INVALID_ARG;
    if (n == 0) return DG_OK;
    logf_eval_kernel<<<(n + 255) / 256, 256, 0, as_stream(stream)>>>(x, y, n);
    DG_LAUNCHED();
    DG_CUDA_TRY(cudaGetLastError());
    return DG_OK;
}

int dg_wait_timeout_probe(void *workspace, size_t workspace_bytes, uint64_t limit_ns, void *stream)
{
    if (workspace == nullptr || workspace_bytes < sizeof(WsHeader)) return DG_ERR_WORKSPACE;
    if (limit_ns < 1000 || limit_ns > kWaitLimitNs) return DG_ERR_INVALID_ARG;
    if (!aligned16(workspace)) return DG_ERR_ALIGNMENT;
    wait_probe_kernel<<<1, 32, 0, as_stream(stream)>>>(static_cast<WsHeader *>(workspace), limit_ns);
    DG_LAUNCHED();
    DG_CUDA_TRY(cudaGetLastError());
    return DG_OK;
}

}  // extern "C"
