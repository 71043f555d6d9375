// dg_moe.cu -- the mixture-of-experts FFN of a canvas forward on GB300.
//
// "DiffusionGemma: When the LLM Stops Writing Left to Right", section "What
// DiffusionGemma Actually Is": the body is a mixture of experts with 128
// experts, top-8 routing and one shared expert.  "Parallel Denoising From an
// Autoregressive Checkpoint", section "Finding": a canvas forward is 4.3x an
// AR step in its MoE layers because the 256 canvas tokens together touch about
// 84 distinct experts per layer, so a layer streams most of its expert
// weights from HBM.  The layer is bound by that stream: the kernels below read
// each touched expert's weights once.
//
// Per token t (readings: the pages give no formulas): router logits
// l = x_t Wr^T; the top_k experts by logit (ties to the lower index) with
// gates softmax(l_selected); out_t = shared(x_t) + sum_j gate_j expert_j(x_t),
// every expert a gated GELU FFN (gelu_tanh(x Wg^T) * (x Wu^T)) Wd^T whose
// intermediate activation is stored as bf16.
//
// Launches:
//   moe_router_kernel   router logits on the tensor cores, split over k
//                       (CTA = k slice x 128-token chunk, partial sums)
//   moe_topk_kernel     a warp per token: the slices summed in order, top-k
//                       experts and gates, a bit in each chosen expert's
//                       token bitmap
//   moe_route_kernel    one CTA: the tokens of each expert in token order
//                       (the bitmaps), their positions in the expert-sorted
//                       order, and the work list of the FFN kernel
//   moe_gather_kernel   X_sorted[pos] = x[token of pos] (bf16 rows)
//   moe_ffn_kernel      persistent tcgen05 GEMMs over the work list: gate/up
//                       items (expert, 128 rows of f, <= 128 tokens) write
//                       H_sorted = bf16(gelu(G) * U); down items (expert,
//                       128 rows of d, <= 128 tokens) write Y_sorted = gate *
//                       (H Wd^T) in fp32 once the expert's H is complete
//   moe_combine_kernel  out[t] = Y[shared pos] + sum_j Y[pos_j] (fixed order)
//
// The FFN GEMMs run weights-as-A ("swap AB"): a 128-row tile of an expert's
// weight (K-major, TMA, 128-byte swizzle) is the UMMA's A operand and the
// expert's tokens (K-major rows of X_sorted or H_sorted) its B operand with
// N = the chunk's token count rounded up to 16, so an expert with 20 tokens
// costs a 128 x 32 UMMA tile rather than a 128-row token tile, and the weight
// bytes set the time.
#include "dg_kernels.h"

namespace dg {

// ------------------------------------------------------------------ router
// Router logits on the tensor cores, split over k: CTA (ks, c) multiplies the
// router weight rows (experts, K-major, A) by the rows of token chunk c
// (K-major, B) over k slice ks (kMoeRouterKSlice values), one 128 x 128 x 16
// UMMA per 16 k into TMEM, and stores its partial logits [ks][t][e] (fp32);
// the top-k kernel sums the slices in order.  One thread loads the slice's
// operands with TMA (all of it at once) and issues the UMMAs; the four warps
// read TMEM (lane = expert, column = token) and store.
__global__ void __launch_bounds__(128, 1)
    moe_router_kernel(const __grid_constant__ CUtensorMap map_wr,
                      const __grid_constant__ CUtensorMap map_x, MoeArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    constexpr int kKB = kMoeRouterKSlice / 64;                 // k blocks of the slice
    constexpr int kTile = 128 * 64 * 2;                        // 16 KB per operand block
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + 2 * kKB * kTile);
    uint64_t *done = full + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    __shared__ int s_ok;
    const int ks = blockIdx.x, c = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        s_ok = 0;
        mbar_init(full, 1);
        mbar_init(done, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_wait();
    griddep_launch_dependents();
    bool ok = true;
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(full, 2 * kKB * kTile);
        for (int kb = 0; kb < kKB; ++kb) {
            const int k = ks * kMoeRouterKSlice + kb * 64;
            tma_load_2d(smem + kb * kTile, &map_wr, full, k, 0, policy_evict_last());
            tma_load_2d(smem + (kKB + kb) * kTile, &map_x, full, k, c * 128, policy_evict_last());
        }
        ok = mbar_wait(full, 0, a.ws, 731);
        if (ok) {
            tc_fence_after();
            const uint32_t idesc = make_idesc_bf16(128, 128, 0);
            const uint32_t sa = smem_u32(smem);
            for (int kb = 0; kb < kKB; ++kb)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = make_sdesc_sw128(sa + kb * kTile + kk * 32, 16, 1024);
                    const uint64_t bd = make_sdesc_sw128(sa + (kKB + kb) * kTile + kk * 32, 16, 1024);
                    umma_bf16(tmem, ad, bd, idesc, (kb | kk) != 0);
                }
        }
        s_ok = ok ? 1 : 0;
        umma_commit(done);
    }
    __syncwarp();
    const bool ok2 = __all_sync(0xFFFFFFFFu, mbar_wait(done, 0, a.ws, 732));
    __syncthreads();
    if (ok2 && s_ok != 0) {
        tc_fence_after();
        const int e = warp * 32 + lane;
        const uint32_t tb = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        float *part = a.router_part + static_cast<size_t>(ks) * a.M * a.E;
        for (int c0 = 0; c0 < 128; c0 += 16) {
            float v[16];
            tmem_ld16(tb + static_cast<uint32_t>(c0), v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int t = c * 128 + c0 + j;
                if (t < a.M && e < a.E) part[static_cast<size_t>(t) * a.E + e] = v[j];
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

int moe_router_smem_bytes() { return 2 * (kMoeRouterKSlice / 64) * 128 * 64 * 2 + 1024 + 256; }

// ------------------------------------------------------------------ top-k
// A warp per token: its logits are the sum of the k slices' parts in slice
// order; then the top_k (k rounds of the largest logit, ties to the lower
// expert index), their gates softmax(l[S]) and a bit in each chosen expert's
// token bitmap (zero between calls).
__global__ void __launch_bounds__(256) moe_topk_kernel(MoeArgs a, int nslices)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    const int E = a.E, K = a.top_k, M = a.M;
    griddep_wait();
    griddep_launch_dependents();
    if (t >= M) return;
    float v[kMoeMaxExperts / 32];
#pragma unroll
    for (int q = 0; q < kMoeMaxExperts / 32; ++q) v[q] = (q * 32 + lane < E) ? 0.f : -INFINITY;
    // the slices in order, eight slices' loads of every expert in flight together
    for (int k0 = 0; k0 < nslices; k0 += 8) {
        float part[8][kMoeMaxExperts / 32];
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int q = 0; q < kMoeMaxExperts / 32; ++q) {
                const int e = q * 32 + lane;
                part[u][q] = (k0 + u < nslices && e < E)
                                 ? __ldcg(a.router_part + (static_cast<size_t>(k0 + u) * M + t) * E + e)
                                 : 0.f;
            }
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
            for (int q = 0; q < kMoeMaxExperts / 32; ++q) v[q] += part[u][q];
    }
#pragma unroll
    for (int q = 0; q < kMoeMaxExperts / 32; ++q) {
        const int e = q * 32 + lane;
        if (e < E) a.logits[static_cast<size_t>(t) * E + e] = v[q];
    }
    const int words = (M + 31) >> 5;
    float mx = 0.f, s = 0.f, my_l = 0.f;
    int my_e = 0;
    for (int j = 0; j < K; ++j) {
        float bv = -INFINITY;
        int be = 0x7FFFFFFF;
#pragma unroll
        for (int q = 0; q < kMoeMaxExperts / 32; ++q) {
            const int e = q * 32 + lane;
            if (e < E && (v[q] > bv || (v[q] == bv && e < be))) { bv = v[q]; be = e; }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int oe = __shfl_xor_sync(0xFFFFFFFFu, be, o);
            if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
        }
#pragma unroll
        for (int q = 0; q < kMoeMaxExperts / 32; ++q)
            if (q * 32 + lane == be) v[q] = -INFINITY;
        if (j == 0) mx = bv;
        s += expf(bv - mx);          // the same sum in every lane, in selection order
        if (lane == j) {
            my_l = bv;
            my_e = be;
        }
    }
    if (lane < K) {
        const float gate = expf(my_l - mx) / s;
        if (a.checks && (!isfinite(gate) || my_e < 0 || my_e >= E)) {
            // device-side checks: a finite gate, an expert of the layer
            report_error(a.ws, DG_ERR_DEVICE, 825);
            if (my_e < 0 || my_e >= E) my_e = 0;
        }
        a.sel_expert[t * K + lane] = my_e;
        a.sel_gate[t * K + lane] = gate;
        atomicOr(a.bits + static_cast<size_t>(my_e) * words + (t >> 5), 1u << (t & 31));
    }
}

// ------------------------------------------------------------------ route
// One CTA of kMoeRouteThreads threads.  Positions in the expert-sorted order:
// experts 0 .. E-1, then the shared expert E (every token), each expert's
// tokens in increasing token order (their rank in the expert's bitmap); its
// chunks of <= kMoeChunk tokens are the FFN kernel's token tiles.  The
// bitmaps are cleared again for the next call.
__global__ void __launch_bounds__(kMoeRouteThreads) moe_route_kernel(MoeArgs a)
{
    __shared__ uint32_t bits[(kMoeMaxExperts + 1) * (kMoeMaxTokens / 32)];
    __shared__ int cnt[kMoeMaxExperts + 1];
    __shared__ int off[kMoeMaxExperts + 2];
    __shared__ int ch0[kMoeMaxExperts + 2];
    __shared__ int chunk_e[kMoeMaxChunks];
    __shared__ int nch_s;
    const int tid = threadIdx.x;
    const int M = a.M, E = a.E, K = a.top_k;
    const int words = (M + 31) >> 5;
    griddep_wait();
    griddep_launch_dependents();
    for (int i = tid; i < E * words; i += blockDim.x) {
        bits[i] = __ldcg(a.bits + i);
        a.bits[i] = 0u;
    }
    if (tid == 0) *a.next_item = 0;
    __syncthreads();
    // tokens per expert; the shared expert takes every token
    for (int e = tid; e <= E; e += blockDim.x) {
        int c = 0;
        if (e < E)
            for (int w = 0; w < words; ++w) c += __popc(bits[e * words + w]);
        else
            c = M;
        cnt[e] = c;
    }
    __syncthreads();
    if (a.checks && tid == 0) {
        // device-side check: every token chose top_k distinct experts
        int routed = 0;
        for (int e = 0; e < E; ++e) routed += cnt[e];
        if (routed != M * K) report_error(a.ws, DG_ERR_DEVICE, 821);
    }
    if (tid < 32) {
        // row offsets and chunk ids (chunks of <= kMoeChunk tokens), experts in
        // order: exclusive scans over the E + 1 experts, 32 at a time
        const int lane = tid;
        int o = 0, ch = 0;
        for (int e0 = 0; e0 <= E; e0 += 32) {
            const int e = e0 + lane;
            const int c = e <= E ? cnt[e] : 0;
            const int n = (c + kMoeChunk - 1) / kMoeChunk;
            int ic = c, in = n;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int uc = __shfl_up_sync(0xFFFFFFFFu, ic, d);
                const int un = __shfl_up_sync(0xFFFFFFFFu, in, d);
                if (lane >= d) {
                    ic += uc;
                    in += un;
                }
            }
            if (e <= E) {
                off[e] = o + ic - c;
                ch0[e] = ch + in - n;
            }
            o += __shfl_sync(0xFFFFFFFFu, ic, 31);
            ch += __shfl_sync(0xFFFFFFFFu, in, 31);
        }
        if (lane == 0) {
            off[E + 1] = o;
            ch0[E + 1] = ch;
            nch_s = ch;
            const int ft = a.f / 128, dt = a.d / 128;
            a.counts[0] = ch * ft;          // gate/up items
            a.counts[1] = ch * (ft + dt);   // all items
            a.counts[2] = o;                // rows of the sorted order
        }
    }
    __syncthreads();
    // the work list: every chunk x f tile of gate/up items, then every chunk x
    // d tile of down items, chunks in expert order; an item is (expert,
    // tile | chunk id << 8, first row, tokens)
    {
        const int nch = nch_s, ft = a.f / 128, dt = a.d / 128;
        for (int e = tid; e <= E; e += blockDim.x)
            for (int cid = ch0[e]; cid < ch0[e + 1]; ++cid) chunk_e[cid] = e;
        __syncthreads();
        for (int i = tid; i < nch * (ft + dt); i += blockDim.x) {
            const bool up = i < nch * ft;
            const int j = up ? i : i - nch * ft;
            const int per = up ? ft : dt;
            const int cid = j / per, tile = j % per;
            const int e = chunk_e[cid];
            const int r0 = off[e] + (cid - ch0[e]) * kMoeChunk;
            a.items[i] = make_int4(e, tile | (cid << 8), r0, min(kMoeChunk, off[e + 1] - r0));
        }
    }
    // readiness counters of the chunks' H blocks
    for (int i = tid; i < kMoeMaxChunks; i += blockDim.x) a.ready[i] = 0u;
    // positions of every assignment (token order within an expert)
    for (int i = tid; i < M * K; i += blockDim.x) {
        const int t = i / K;
        const int e = a.sel_expert[i];
        if (a.checks && (e < 0 || e >= E)) {
            report_error(a.ws, DG_ERR_DEVICE, 822);
            continue;
        }
        const int w = t >> 5;
        int r = __popc(bits[e * words + w] & ((1u << (t & 31)) - 1u));
        for (int q = 0; q < w; ++q) r += __popc(bits[e * words + q]);
        const int pos = off[e] + r;
        a.pos_of[i] = pos;
        a.tok_of_pos[pos] = t;
        a.gate_of_pos[pos] = a.sel_gate[i];
    }
    for (int t = tid; t < M; t += blockDim.x) {
        const int pos = off[E] + t;
        a.tok_of_pos[pos] = t;
        a.gate_of_pos[pos] = 1.0f;
    }
}

// ------------------------------------------------------------------ gather
// X_sorted[pos, :] = x[tok_of_pos[pos], :] for pos < counts[2]; 16-byte
// vectors, a grid-stride loop.
__global__ void moe_gather_kernel(MoeArgs a)
{
    griddep_wait();
    griddep_launch_dependents();
    const int rows = a.counts[2];
    const int vec = a.d / 8;
    const size_t n = static_cast<size_t>(rows) * vec;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t pos = i / vec, c = i % vec;
        const int t = a.tok_of_pos[pos];
        reinterpret_cast<uint4 *>(a.x_sorted)[pos * vec + c] =
            __ldg(reinterpret_cast<const uint4 *>(a.x) + static_cast<size_t>(t) * vec + c);
    }
}

// ------------------------------------------------------------------ combine
// out[t, :] = Y[shared pos] + sum_j Y[pos_of[t, j]] in that order (fp32).
__global__ void moe_combine_kernel(MoeArgs a)
{
    griddep_wait();
    griddep_launch_dependents();
    const int K = a.top_k;
    const int vec = a.d / 4;
    const int shared0 = a.M * K;          // the shared expert's rows start after the routed ones
    const size_t n = static_cast<size_t>(a.M) * vec;
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / vec);
        const size_t c = i % vec;
        const float4 *y = reinterpret_cast<const float4 *>(a.y_sorted);
        float4 s = __ldcg(y + static_cast<size_t>(shared0 + t) * vec + c);
        for (int j = 0; j < K; ++j) {
            const int pj = a.pos_of[t * K + j];
            if (a.checks && (pj < 0 || pj >= shared0)) {
                // device-side check: a routed row of the sorted order
                if (c == 0) report_error(a.ws, DG_ERR_DEVICE, 824);
                continue;
            }
            const float4 v = __ldcg(y + static_cast<size_t>(pj) * vec + c);
            s.x += v.x;
            s.y += v.y;
            s.z += v.z;
            s.w += v.w;
        }
        reinterpret_cast<float4 *>(a.out)[i] = s;
    }
}

// ------------------------------------------------------------------ expert GEMMs
namespace {

constexpr int kMoeStages = 4;
constexpr int kMoeATile = 128 * 64 * 2;           // 16 KB: 128 weight rows x 64 k
constexpr int kMoeBTile = kMoeChunk * 64 * 2;      // 16 KB: up to 128 token rows x 64 k
constexpr int kMoeStageBytes = 2 * kMoeATile + kMoeBTile;   // gate + up + tokens
constexpr int kMoeQueue = 4;                       // work items in flight in a CTA

DG_DEVICE void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

DG_DEVICE float gelu_tanh(float v)
{
    const float u = 0.7978845608028654f * fmaf(0.044715f * v, v * v, v);
    return 0.5f * v * (1.0f + tanhf(u));
}

}  // namespace

int moe_ffn_smem_bytes() { return kMoeStages * kMoeStageBytes + 1024 + 512; }

// Persistent: each CTA takes work items in list order (an atomic counter)
// until the list is exhausted.  Warp 0 fetches items and streams their
// operands through a 4-stage ring; warp 1 issues the UMMAs (one thread);
// warps 2-5 are the epilogue (one TMEM lane quadrant each).  Items travel
// from warp 0 to warps 1-5 through a small queue in shared memory.  A down
// item of expert e, chunk c waits (bounded) until every gate/up item of that
// (e, c) has stored its part of H_sorted.
__global__ void __launch_bounds__(192, 1) moe_ffn_kernel(const __grid_constant__ MoeMaps maps, MoeArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kMoeStages * kMoeStageBytes);
    uint64_t *empty = full + kMoeStages;
    uint64_t *acc_full = empty + kMoeStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *q_full = acc_empty + 2;
    uint64_t *q_empty = q_full + kMoeQueue;
    uint64_t *mma_done = q_empty + kMoeQueue;
    int *queue = reinterpret_cast<int *>(mma_done + 1);     // kMoeQueue item indices
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(queue + kMoeQueue);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kMoeStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], 4);
        }
        for (int q = 0; q < kMoeQueue; ++q) {
            mbar_init(&q_full[q], 1);
            mbar_init(&q_empty[q], 5);     // the MMA thread and the 4 epilogue warps
        }
        mbar_init(mma_done, 1);
        fence_barrier_init();
        tma_prefetch_desc(&maps.wg);
        tma_prefetch_desc(&maps.wu);
        tma_prefetch_desc(&maps.wd);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    griddep_wait();
    griddep_launch_dependents();
    const int n1 = a.counts[0], ntot = a.counts[1];
    const int ftiles = a.f / 128;

    if (warp == 0) {
        // ------------------------------------------------------------ fetch + producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_par = 0;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int q = it % kMoeQueue;
                const uint32_t qph = static_cast<uint32_t>(it / kMoeQueue) & 1u;
                if (!mbar_wait(&q_empty[q], qph ^ 1u, a.ws, 701)) break;
                const int idx = atomicAdd(a.next_item, 1);
                const int item = idx < ntot ? idx : -1;
                queue[q] = item;
                mbar_arrive(&q_full[q]);
                if (item < 0) break;
                const int4 w = a.items[item];
                const bool up = item < n1;
                if (!up) {
                    // the chunk's H rows must be complete: every gate/up item
                    // of the chunk counts once per epilogue warp
                    const uint32_t *rd = a.ready + (w.y >> 8);
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_gpu(rd) < static_cast<uint32_t>(4 * ftiles)) {
                        if (globaltimer_ns() - t0 > kWaitLimitNs) {
                            report_error(a.ws, DG_ERR_TIMEOUT, 702);
                            ok = false;
                            break;
                        }
                    }
                    if (!ok) break;
                    fence_proxy_async_global();
                }
                const int kblocks = (up ? a.d : a.f) / 64;
                // the smallest token box that holds the chunk: 16, 32, 64 or 128 rows
                const int bx = w.w <= 16 ? 0 : w.w <= 32 ? 1 : w.w <= 64 ? 2 : 3;
                const CUtensorMap *mb = up ? &maps.xs[bx] : &maps.hs[bx];
                const uint32_t tx = static_cast<uint32_t>((up ? 2 : 1) * kMoeATile + (16 << bx) * 128);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, a.ws, 703)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[s], tx);
                    uint8_t *sa = smem + s * kMoeStageBytes;
                    uint8_t *sb = sa + 2 * kMoeATile;
                    if (up) {
                        tma_load_3d(sa, &maps.wg, &full[s], kb * 64, (w.y & 255) * 128, w.x, pol_w);
                        tma_load_3d(sa + kMoeATile, &maps.wu, &full[s], kb * 64, (w.y & 255) * 128,
                                    w.x, pol_w);
                    } else {
                        tma_load_3d(sa, &maps.wd, &full[s], kb * 64, (w.y & 255) * 128, w.x, pol_w);
                    }
                    tma_load_2d(sb, mb, &full[s], kb * 64, w.z, pol_x);
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == kMoeStages) { s = 0; ph ^= 1u; }
                }
            }
            for (int q = 0; q < kMoeStages; ++q)
                if (armed >> q & 1u) mbar_wait(&full[q], armed_par >> q & 1u, a.ws, 704);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t sa0 = smem_u32(smem);
            const uint64_t adesc0 = make_sdesc_sw128(sa0, 16, 1024);
            const uint64_t bdesc0 = make_sdesc_sw128(sa0 + 2 * kMoeATile, 16, 1024);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int it = 0; ok; ++it) {
                const int q = it % kMoeQueue;
                const uint32_t qph = static_cast<uint32_t>(it / kMoeQueue) & 1u;
                if (!mbar_wait(&q_full[q], qph, a.ws, 711)) break;
                const int item = queue[q];
                mbar_arrive(&q_empty[q]);
                if (item < 0) break;
                const int4 w = a.items[item];
                const bool up = item < n1;
                const int nmma = (w.w + 15) & ~15;
                const uint32_t idesc = make_idesc_bf16(128, nmma, 0);
                const int acc = it & 1;
                const uint32_t use = static_cast<uint32_t>(it >> 1);
                if (!mbar_wait(&acc_empty[acc], (use & 1u) ^ 1u, a.ws, 712)) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * 256);
                const int kblocks = (up ? a.d : a.f) / 64;
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait(&full[s], ph, a.ws, 713)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t soff = static_cast<uint64_t>((s * kMoeStageBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // K-major A and B: +32 bytes (16 k) per step inside the 128-byte rows
                        const uint64_t adesc = adesc0 + soff + static_cast<uint64_t>(kk * 2);
                        const uint64_t bdesc = bdesc0 + soff + static_cast<uint64_t>(kk * 2);
                        umma_bf16(d0, adesc, bdesc, idesc, (kb | kk) != 0);
                        if (up)
                            umma_bf16(d0 + 128, adesc + static_cast<uint64_t>(kMoeATile >> 4), bdesc,
                                      idesc, (kb | kk) != 0);
                    }
                    umma_commit(&empty[s]);
                    if (++s == kMoeStages) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&acc_full[acc]);
            }
            umma_commit(mma_done);
            mbar_wait(mma_done, 0, a.ws, 714);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2-5)
        const int qd = warp & 3;                        // TMEM lane quadrant
        const int row = qd * 32 + lane;                 // row of the 128-row weight tile
        const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
        for (int it = 0;; ++it) {
            const int q = it % kMoeQueue;
            const uint32_t qph = static_cast<uint32_t>(it / kMoeQueue) & 1u;
            const bool okq = mbar_wait(&q_full[q], qph, a.ws, 721);
            if (!__all_sync(0xFFFFFFFFu, okq)) break;
            const int item = queue[q];
            __syncwarp();
            if (lane == 0) mbar_arrive(&q_empty[q]);
            if (item < 0) break;
            const int4 w = a.items[item];
            const bool up = item < n1;
            const int acc = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            const bool ok = mbar_wait(&acc_full[acc], use & 1u, a.ws, 722);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            const uint32_t tb = tmem_base + lane_off + static_cast<uint32_t>(acc * 256);
            const int n = w.w;
            for (int c0 = 0; c0 < n; c0 += 16) {
                float g[16];
                tmem_ld16(tb + static_cast<uint32_t>(c0), g);
                if (up) {
                    float u[16];
                    tmem_ld16(tb + 128u + static_cast<uint32_t>(c0), u);
                    const int fcol = (w.y & 255) * 128 + row;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < n) {
                            const float h = gelu_tanh(g[j]) * u[j];
                            const __nv_bfloat16 hb = __float2bfloat16_rn(h);
                            a.h_sorted[static_cast<size_t>(w.z + c0 + j) * a.f + fcol] =
                                *reinterpret_cast<const uint16_t *>(&hb);
                        }
                    }
                } else {
                    const int dcol = (w.y & 255) * 128 + row;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < n) {
                            const int pos = w.z + c0 + j;
                            a.y_sorted[static_cast<size_t>(pos) * a.d + dcol] =
                                g[j] * __ldg(a.gate_of_pos + pos);
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&acc_empty[acc]);
                if (up) {
                    // this warp's 32 rows of the chunk's H are stored: count
                    // them (fence, then a release at GPU scope)
                    __threadfence();
                    fence_proxy_async_global();
                    atomicAdd(a.ready + (w.y >> 8), 1u);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

}  // namespace dg
