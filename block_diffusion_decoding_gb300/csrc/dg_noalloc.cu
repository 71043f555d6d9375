// dg_noalloc.cu -- dg_denoise_step_noalloc: the denoising step for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run a step: an
// inference engine that hands out all device memory from its own pool, code
// running inside a region where allocation is forbidden (a memory budget that
// is already fully committed, a driver-level allocator that must not be
// re-entered), or a host program that only receives device pointers for its
// inputs and outputs.  They have no workspace to pass.  This entry point runs
// the same two kernels as dg_denoise_step (LM head with the fused sampler
// epilogue, then combine + acceptance + stop) and keeps their scratch -- the
// per-CTA partial states, the per-canvas counters and the status header -- in
// one fixed array in the library's own device memory, declared below.  The
// array is part of the loaded module: every GPU that loads the library holds
// it until the process exits.
//
// Capacity: kNoAllocScratchBytes = 8 MiB.  A step needs 256 bytes of header,
// 7 x 4 bytes x (LM-head units) x B*L of partial states, 4 bytes per canvas
// and 4 bytes per canvas row (the per-row Gumbel bounds the 2-SM LM-head
// units share), each rounded up to 256 bytes.  With one unit per SM on a
// 152-SM GB300 (the most any plan uses) every step of up to B*L = 1968
// canvas rows fits (seven 256-token canvases); steps that need more are
// rejected with DG_ERR_UNSUPPORTED before anything is launched.
//
// Sharing: every call, from any thread or stream, uses the same array and
// leaves the last call's contents in it.  The counters that must start at
// zero are zeroed by the first kernel of each call (the row bounds by the
// LM head itself, under an epoch kept in the header); the status header is
// cleared at set-up and by dg_noalloc_read_device_status(clear != 0).  A
// kernel that meets a problem on the device (a bounded wait that ran out)
// records it in the header and returns early; the step's outputs are then
// not valid, and dg_noalloc_read_device_status reports it.  Calls whose kernels overlap on the GPU (two
// streams, two threads without ordering) race on the array and give wrong
// results: order them on one stream.
//
// Set-up: the first call on each device (with that device current) looks up
// the device address of the array with cudaGetSymbolAddress, sets the LM-head
// kernels' shared-memory limits and clears the status header (a synchronous
// cudaMemset).  Make that first call before any stream capture.  Nothing here
// calls cudaMalloc, cudaFree or any allocating library routine.  Kernels
// launched by this entry point are not counted by dg_kernel_launches.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <map>
#include <mutex>

#include "dg_kernels.h"
#include "dg_plan.h"

using namespace dg;

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

// The scratch of dg_denoise_step_noalloc.  In host code this name is only a
// stand-in for the symbol; kernels receive the device address obtained with
// cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

struct NoAllocDevice {
    unsigned char *scratch = nullptr;   // device address of g_noalloc_scratch
    int sms = 0;
};

std::mutex g_na_mu;
std::map<int, NoAllocDevice> g_na_dev;

inline size_t na_round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline bool na_aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int na_setup(NoAllocDevice **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return DG_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_na_mu);
    NoAllocDevice &st = g_na_dev[dev];
    if (st.scratch == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr ||
            cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kLmSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(lm_head_duo_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kDuoSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(lm_head_duo_wide_kernel,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kDuoSmemBytes) != cudaSuccess ||
            cudaMemset(ptr, 0, sizeof(WsHeader)) != cudaSuccess) {
            (void)cudaGetLastError();
            return DG_ERR_CUDA;
        }
        st.scratch = static_cast<unsigned char *>(ptr);
    }
    *out = &st;
    return DG_OK;
}

typedef CUresult (*NaEncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                               const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                               const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                               CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// A 2-D bf16 map [outer][inner], or with planes > 0 a 3-D one
// [planes][outer][inner] (the packed LM-head weight), 128-byte swizzle.
int na_map(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
           uint32_t box_outer, uint64_t planes = 0)
{
    static NaEncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<NaEncodeFn>(p);
        else
            (void)cudaGetLastError();
    });
    if (fn == nullptr) return DG_ERR_CUDA;
    const cuuint64_t dims[3] = {inner, outer, planes};
    const cuuint64_t strides[2] = {inner * 2, inner * 2 * outer};
    const cuuint32_t box[3] = {box_inner, box_outer, 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, planes > 0 ? 3 : 2, const_cast<void *>(base), dims,
                    strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DG_OK : DG_ERR_CUDA;
}

}  // namespace

extern "C" int dg_denoise_step_noalloc(const uint16_t *hidden, const uint16_t *w,
                                       const dg_step_params *p, const dg_step_io *io,
                                       void *stream)
{
    // ---- the same argument checks as dg_denoise_step
    if (p == nullptr || io == nullptr || hidden == nullptr || w == nullptr) return DG_ERR_INVALID_ARG;
    if (p->B < 1 || p->L < 1 || p->V < 1 || p->d < 1) return DG_ERR_INVALID_ARG;
    if (!(p->temperature > 0.0) || !std::isfinite(p->temperature)) return DG_ERR_INVALID_ARG;
    if (!(p->entropy_bound >= 0.f) || !std::isfinite(p->entropy_bound)) return DG_ERR_INVALID_ARG;
    if (!std::isfinite(p->stop_threshold) || p->step < 0) return DG_ERR_INVALID_ARG;
    if (p->w_layout != DG_W_ROWMAJOR && p->w_layout != DG_W_PACKED) return DG_ERR_INVALID_ARG;
    if (!io->canvas || !io->prev_argmax || !io->argmax || !io->sample || !io->entropy ||
        !io->accepted || !io->n_accepted || !io->mean_entropy || !io->stop)
        return DG_ERR_INVALID_ARG;
    if (p->L > kMaxCanvas || p->V % 8 != 0 || p->V < 64) return DG_ERR_UNSUPPORTED;
    if (p->d % 64 != 0 || p->d < 64 || p->d > 16384) return DG_ERR_UNSUPPORTED;
    if (static_cast<long long>(p->B) * p->L > (1LL << 20)) return DG_ERR_UNSUPPORTED;
    if (!na_aligned16(hidden) || !na_aligned16(w)) return DG_ERR_ALIGNMENT;

    NoAllocDevice *st = nullptr;
    int rc = na_setup(&st);
    if (rc != DG_OK) return rc;

    // ---- kernel and tile plan: the same choice as dg_denoise_step
    const int M = p->B * p->L;
    const bool packed = p->w_layout == DG_W_PACKED;
    const LmPlan plan = plan_lm_head(M, p->d, p->V, st->sms, false, false, -1, packed);
    const int BN = plan.BN, ntn = plan.ntn, total = plan.total;

    // ---- scratch layout (as a workspace): header | partials | counters | row keys
    const size_t npart = static_cast<size_t>(plan.part_slots()) * M;
    const size_t need = sizeof(WsHeader) + na_round_up(7 * npart * 4, 256) +
                        na_round_up(static_cast<size_t>(p->B) * 4, 256) +
                        na_round_up(static_cast<size_t>(M) * 4, 256);
    if (need > kNoAllocScratchBytes) return DG_ERR_UNSUPPORTED;
    unsigned char *base = st->scratch;
    WsHeader *hdr = reinterpret_cast<WsHeader *>(base);
    float *f = reinterpret_cast<float *>(base + sizeof(WsHeader));
    Partials part;
    part.m = f;
    part.S = f + npart;
    part.A = f + 2 * npart;
    part.gbest = f + 3 * npart;
    part.amax = f + 4 * npart;
    part.gidx = reinterpret_cast<int *>(f + 5 * npart);
    part.aidx = reinterpret_cast<int *>(f + 6 * npart);
    int *counters = reinterpret_cast<int *>(base + sizeof(WsHeader) + na_round_up(7 * npart * 4, 256));
    uint32_t *rowkey = reinterpret_cast<uint32_t *>(
        reinterpret_cast<unsigned char *>(counters) + na_round_up(static_cast<size_t>(p->B) * 4, 256));

    CUtensorMap mx, mw;
    if ((rc = na_map(&mx, hidden, static_cast<uint64_t>(p->d), static_cast<uint64_t>(M), 64,
                     plan.cluster() ? 128u : 256u)) != DG_OK)
        return rc;
    if (packed)
        rc = na_map(&mw, w, 128, static_cast<uint64_t>(p->d), 64, 64,
                    static_cast<uint64_t>((p->V + 127) / 128));
    else
        rc = na_map(&mw, w, static_cast<uint64_t>(p->V), static_cast<uint64_t>(p->d), 64, 64);
    if (rc != DG_OK) return rc;

    StepSource src{};
    src.ctl = nullptr;
    src.invT = static_cast<float>(1.0 / p->temperature);
    src.c2 = src.invT * 1.44269502162933349609375f;
    src.step = p->step;

    LmHeadArgs a{};
    a.w_packed = packed ? 1 : 0;
    a.M = M;
    a.d = p->d;
    a.V = p->V;
    a.BN = BN;
    a.ntn = ntn;
    a.total = total;
    a.kblocks = p->d / 64;
    a.nbox_b = (BN + 63) / 64;
    a.x_3d = 0;
    a.fuse2 = plan.kind == kLmDuoFused ? 1 : 0;
    a.part = part;
    a.src = src;
    a.seed = p->seed;
    a.ws = hdr;
    a.counters = counters;
    a.ncounters = p->B;
    a.rowkey = rowkey;

    CombineArgs c{};
    c.part = part;
    c.n_slots = plan.part_slots();
    c.ntn = ntn;
    c.total = total;
    c.M = M;
    c.H = io->entropy;
    c.sample = io->sample;
    c.argmax = io->argmax;
    c.counters = counters;
    c.rows_per_cta = combine_rows_per_cta(p->B, p->L, plan.sms);

    AcceptArgs acc{};
    acc.B = p->B;
    acc.L = p->L;
    acc.V = p->V;
    acc.bound = p->entropy_bound;
    acc.threshold = p->stop_threshold;
    acc.seed = p->seed;
    acc.step = p->step;
    acc.canvas = io->canvas;
    acc.prev_argmax = io->prev_argmax;
    acc.accepted = io->accepted;
    acc.n_accepted = io->n_accepted;
    acc.mean_entropy = io->mean_entropy;
    acc.stop = io->stop;
    acc.ws = hdr;
    acc.checks = device_checks();

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool pdl = use_pdl(s);
    if (launch_lm_head(plan, mx, mw, a, s, pdl) != cudaSuccess) return DG_ERR_CUDA;
    if (launch_kernel(combine_accept_kernel, dim3((p->L + c.rows_per_cta - 1) / c.rows_per_cta, p->B), dim3(kAcceptThreads), 0, s, pdl, c,
                      acc) != cudaSuccess)
        return DG_ERR_CUDA;
    return DG_OK;
}

// The status header of the scratch array: 0, or the DG_ERR_* code a kernel of
// dg_denoise_step_noalloc recorded on the device.  Synchronous on `stream`;
// clear != 0 resets the header afterwards (also on the stream).  Allocates
// nothing; the first call on a device may do the array's set-up.
extern "C" int dg_noalloc_read_device_status(int *status_out, int clear, void *stream)
{
    if (status_out == nullptr) return DG_ERR_INVALID_ARG;
    NoAllocDevice *st = nullptr;
    int rc = na_setup(&st);
    if (rc != DG_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, st->scratch, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        (void)cudaGetLastError();
        return DG_ERR_CUDA;
    }
    *status_out = v;
    if (clear && (cudaMemsetAsync(st->scratch, 0, sizeof(WsHeader), s) != cudaSuccess ||
                  cudaStreamSynchronize(s) != cudaSuccess)) {
        (void)cudaGetLastError();
        return DG_ERR_CUDA;
    }
    return DG_OK;
}
