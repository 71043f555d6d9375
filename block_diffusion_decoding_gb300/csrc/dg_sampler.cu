// dg_sampler.cu -- the sampler tail of a denoising step:
//   * combine: merge per-slot partial states into per-position entropy,
//     Gumbel-max sample and argmax;
//   * accept: per canvas, sort positions by entropy, commit the largest
//     prefix allowed by the entropy bound, renoise the rest, run the stop
//     test (fused behind the combine: the last combine CTA of a canvas runs
//     it, found with an atomic counter, no waiting);
//   * the logits-from-memory fold, the block-loop init and the small kernels
//     used to check Philox / log / Gumbel in isolation.
//
// "DiffusionGemma Lab", section 2: item 1 (uniform init), item 2 (sort by
// entropy ascending, commit the largest prefix with cumsum(H) - max(H) <=
// 0.1, at least one), item 3 (stop when the argmax canvas is unchanged and
// mean entropy < 0.005), item 5 (commit the sample, output the argmax).
// "Parallel Denoising From an Autoregressive Checkpoint", section "Finding",
// bullet "Entropy-bounded acceptance": the remainder is renoised uniformly.
#include "dg_kernels.h"

namespace dg {

// ---------------------------------------------------------------- fold of fp32 logits
// One thread per row of a 256-row block; CTA c folds the tiles of slot c.
__global__ void __launch_bounds__(256) logits_fold_kernel(const float *__restrict__ logits,
                                                          FoldArgs a)
{
    const int c = blockIdx.x;
    if (c == 0) {
        for (int i = threadIdx.x; i < a.ncounters; i += blockDim.x) a.counters[i] = 0;
    }
    const FoldConsts fc = fold_consts(a.src, a.seed);
    const int t0 = tile_begin(c, a.total, a.n_slots), t1 = tile_begin(c + 1, a.total, a.n_slots);
    RowState st;
    row_state_init(st);
    int cur_m = -1;
    for (int t = t0; t < t1; ++t) {
        const int m = t / a.ntn, n = t % a.ntn;
        const int row = m * kRowsPerBlock + threadIdx.x;
        if (m != cur_m) {
            if (cur_m >= 0) {
                const int prow = cur_m * kRowsPerBlock + threadIdx.x;
                row_state_finalize(st, fc);
                if (prow < a.M) partial_store(a.part, static_cast<size_t>(prow) * a.n_slots + c, st);
            }
            row_state_init(st);
            cur_m = m;
        }
        const bool live = row < a.M;
        const float *src = logits + static_cast<size_t>(live ? row : 0) * a.V;
        for (int c0 = 0; c0 < a.BN; c0 += 16) {
            const uint32_t v0 = static_cast<uint32_t>(n * a.BN + c0);
            if (v0 >= static_cast<uint32_t>(a.V)) break;
            float lg[16];
            if (!live) {
#pragma unroll
                for (int j = 0; j < 16; ++j) lg[j] = 0.f;
            } else if (v0 + 16u <= static_cast<uint32_t>(a.V)) {
                const float4 *p4 = reinterpret_cast<const float4 *>(src + v0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 f = __ldg(p4 + q);
                    lg[4 * q] = f.x; lg[4 * q + 1] = f.y; lg[4 * q + 2] = f.z; lg[4 * q + 3] = f.w;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    lg[j] = (v0 + j < static_cast<uint32_t>(a.V)) ? __ldg(src + v0 + j) : 0.f;
            }
            fold16(st, lg, v0, static_cast<uint32_t>(a.V), static_cast<uint32_t>(row), fc, live);
        }
    }
    if (cur_m >= 0) {
        const int prow = cur_m * kRowsPerBlock + threadIdx.x;
        row_state_finalize(st, fc);
        if (prow < a.M) partial_store(a.part, static_cast<size_t>(prow) * a.n_slots + c, st);
    }
}

// ---------------------------------------------------------------- accept (one canvas)
// Run by one CTA of kAcceptThreads threads (>= L).  Only the positions whose
// entropy is within the bound b (the set C) need an exact order: a sorted
// prefix that holds any larger entropy sums past b (an fp64 sum of
// non-negative terms is at least each of its terms), so the accepted
// positions are C's smallest keys (H, position) and at most one more, the
// smallest key outside C, which sorts right after all of C.  C is compacted
// in position order; the rank of every key of C among them gives the
// ascending order without a sorting network: each key is counted against up
// to kRankSplit slices of C's keys by separate threads, and the slice counts
// are summed.  The exclusive prefix sums of the sorted entropies (fp64)
// never decrease, so k* = #{j : sum of the first j sorted entropies <= b}
// (and k* >= 1); one warp scans them 32 at a time and stops at the first
// chunk that passes b.  Position i is accepted iff its rank is below k*.
constexpr int kRankSplit = 4;

__device__ void accept_canvas(const AcceptArgs &a, int b, int step, const float *__restrict__ H,
                              const int32_t *__restrict__ sample,
                              const int32_t *__restrict__ argmax)
{
    __shared__ __align__(16) uint64_t keys[kMaxCanvas];   // C's keys, in position order
    __shared__ float hsorted[kMaxCanvas];                 // C sorted, then the first key past C
    __shared__ int prank[kRankSplit * kMaxCanvas];
    __shared__ float hpos[kMaxCanvas];                    // the entropies, in position order
    __shared__ int wcnt[kAcceptThreads / 32];
    __shared__ uint64_t wmin[kAcceptThreads / 32];
    __shared__ double wsum[1];
    __shared__ int s_kstar;
    const int tid = threadIdx.x, nt = blockDim.x;
    const int lane = tid & 31, wid = tid >> 5, nw = nt >> 5;
    const int L = a.L;
    const size_t base = static_cast<size_t>(b) * L;
    const bool own = tid < L;    // this thread's position i = tid (nt >= L)

    // keys (H, position): H >= 0, so its bit pattern orders like the value;
    // the stop-test operands and the sample are fetched now, with the keys
    float h = 0.f;
    int32_t am = 0, pa = 0, smp = 0;
    if (own) {
        h = __ldcg(H + base + tid);
        am = __ldcg(argmax + base + tid);
        pa = a.prev_argmax[base + tid];
        smp = __ldcg(sample + base + tid);
        if (a.checks) {
            // device-side checks of the operands (the stage entry takes them from the caller)
            if (!(h >= 0.f) || !isfinite(h)) report_error(a.ws, DG_ERR_DEVICE, 804);
            if (smp < 0 || smp >= a.V) {
                report_error(a.ws, DG_ERR_DEVICE, 805);
                smp = 0;
            }
            if (am < 0 || am >= a.V) {
                report_error(a.ws, DG_ERR_DEVICE, 806);
                am = 0;
            }
        }
    }
    const uint64_t key = (static_cast<uint64_t>(__float_as_uint(h)) << 32) | static_cast<uint32_t>(tid);
    const bool inC = own && h <= a.bound;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, inC);
    // per warp: the smallest key outside C
    uint64_t mo = (own && !inC) ? key : ~0ull;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, mo, off);
        mo = o < mo ? o : mo;
    }
    if (own) hpos[tid] = h;
    if (lane == 0) {
        wcnt[wid] = __popc(bal);
        wmin[wid] = mo;
    }
    __syncthreads();
    // every warp combines the per-warp counts and minima (lane w: warp w's)
    const int cw = lane < nw ? wcnt[lane] : 0;
    int incl = cw;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
    }
    const int nC = __shfl_sync(0xFFFFFFFFu, incl, 31);
    const int ci = __shfl_sync(0xFFFFFFFFu, incl - cw, wid) + __popc(bal & ((1u << lane) - 1u));
    uint64_t mout = lane < nw ? wmin[lane] : ~0ull;
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, mout, off);
        mout = o < mout ? o : mout;
    }
    if (inC) keys[ci] = key;
    __syncthreads();
    // partial ranks within C: thread t counts key t % nC against slice
    // t / nC (slices start on even keys, two keys per 16-byte shared load)
    const int nq = nC > 0 ? max(1, min(kRankSplit, nt / nC)) : 0;
    if (tid < nq * nC) {
        const int i = tid % nC, q = tid / nC;
        const int j0 = (q * nC / nq) & ~1, j1 = (q + 1 == nq) ? nC : ((q + 1) * nC / nq) & ~1;
        const uint64_t k = keys[i];
        int cnt = 0;
        int j = j0;
#pragma unroll 4
        for (; j + 1 < j1; j += 2) {
            const ulonglong2 kk = *reinterpret_cast<const ulonglong2 *>(&keys[j]);
            cnt += (kk.x < k ? 1 : 0) + (kk.y < k ? 1 : 0);
        }
        if (j < j1) cnt += (keys[j] < k) ? 1 : 0;
        prank[q * nC + i] = cnt;
    }
    __syncthreads();
    int rank = L;    // outside C and not its smallest key: never accepted
    if (inC) {
        rank = 0;
        for (int q = 0; q < nq; ++q) rank += prank[q * nC + ci];
        if (a.checks && (rank < 0 || rank >= nC)) {
            report_error(a.ws, DG_ERR_DEVICE, 807);
            rank = nC - 1;
        }
        hsorted[rank] = h;
    } else if (own && key == mout) {
        rank = nC;
        hsorted[nC] = h;
    }
    const int nS = nC + (mout != ~0ull ? 1 : 0);   // entries of hsorted
    __syncthreads();
    // k*: warp 0 scans the sorted entropies in chunks of 32 (exclusive sums)
    if (wid == 0) {
        double carry = 0.0;
        int kcount = 0;
        for (int c0 = 0; c0 < nS; c0 += 32) {
            const int j = c0 + lane;
            const double hv = (j < nS) ? static_cast<double>(hsorted[j]) : 0.0;
            double inc = hv;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const double o = __shfl_up_sync(0xFFFFFFFFu, inc, off);
                if (lane >= off) inc += o;
            }
            const double prev = __shfl_up_sync(0xFFFFFFFFu, inc, 1);
            const double excl = carry + (lane == 0 ? 0.0 : prev);
            kcount += __popc(__ballot_sync(0xFFFFFFFFu, j < nS && excl <= static_cast<double>(a.bound)));
            const double last = __shfl_sync(0xFFFFFFFFu, excl, 31);
            carry += __shfl_sync(0xFFFFFFFFu, inc, 31);
            if (last > static_cast<double>(a.bound)) break;   // the sums only grow
        }
        if (lane == 0) s_kstar = max(1, kcount);
    } else if (wid == 1) {
        // fp64 total of the entropies (mean for the stop test), beside the
        // scan: lane l sums positions l, l + 32, ... in order, then a fixed
        // butterfly (fp64 is slow here: one warp does it)
        double t = 0.0;
        for (int j = lane; j < L; j += 32) t += static_cast<double>(hpos[j]);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, off);
        if (lane == 0) wsum[0] = t;
    }
    __syncthreads();
    const int kstar = s_kstar;
    const double total = wsum[0];
    const uint32_t k0 = static_cast<uint32_t>(a.seed), k1 = static_cast<uint32_t>(a.seed >> 32);
    if (own) {
        const size_t r = base + tid;
        if (rank < kstar) {
            a.canvas[r] = smp;
            a.accepted[r] = 1;
        } else {
            const uint4 x = philox4x32_10(make_uint4(0u, static_cast<uint32_t>(r),
                                                     static_cast<uint32_t>(step), kStreamRenoise),
                                          k0, k1);
            a.canvas[r] = static_cast<int32_t>(token_from_word(x.x, static_cast<uint32_t>(a.V)));
            a.accepted[r] = 0;
        }
    }
    // stop test: unchanged argmax and mean entropy below the threshold
    const int all_same = __syncthreads_and(own ? (am == pa) : 1);
    if (own) {
        a.prev_argmax[base + tid] = am;
        // freeze the block output: the argmax canvas of the latest live step
        if (a.ctl != nullptr) a.out_argmax[base + tid] = am;
    }
    if (tid == 0) {
        if (a.checks && !isfinite(total)) report_error(a.ws, DG_ERR_DEVICE, 808);
        const double mean = total / static_cast<double>(L);
        const int stop = (step >= 1 && all_same && mean < static_cast<double>(a.threshold)) ? 1 : 0;
        a.n_accepted[b] = kstar;
        a.mean_entropy[b] = static_cast<float>(mean);
        a.stop[b] = stop;
        if (a.ctl != nullptr) {   // block loop bookkeeping
            if (a.n_acc_hist != nullptr) a.n_acc_hist[static_cast<size_t>(step) * a.B + b] = kstar;
            a.steps_taken[b] = step + 1;
            if (stop || step + 1 >= a.ctl->max_steps) a.done[b] = 1;
        }
    }
}

// Block loop: the last canvas to finish its acceptance advances the loop.
__device__ void loop_advance(const AcceptArgs &a)
{
    __threadfence();
    LoopCtl *ctl = a.ctl;
    const int done_now = atomicAdd(&ctl->canvases_finished, 1) + 1;
    if (done_now < ctl->n_live) return;
    __threadfence();
    int live = 0;
    for (int b = 0; b < a.B; ++b) live += (__ldcg(a.done + b) == 0);
    const int next = ctl->step + 1;
    ctl->canvases_finished = 0;
    ctl->n_live = live;
    if (live == 0 || next >= ctl->max_steps) {
        cudaGraphSetConditional(a.cond, 0u);
    } else {
        ctl->step = next;
    }
    __threadfence();
}

// ---------------------------------------------------------------- combine + accept
// grid = (ceil(L / R), B) with R = c.rows_per_cta, kAcceptThreads threads:
// warp w < R of CTA (x, b) merges the partial states of canvas row
// b*L + R x + w; the last CTA of canvas b runs the acceptance for it.
__global__ void __launch_bounds__(kAcceptThreads) combine_accept_kernel(CombineArgs c, AcceptArgs a)
{
    griddep_wait();
    griddep_launch_dependents();
    const int b = blockIdx.y;
    if (a.ctl != nullptr && __ldcg(a.done + b) != 0) return;   // canvas already stopped
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * c.rows_per_cta + warp;
    if (warp < c.rows_per_cta && i < a.L) {
        const int r = b * a.L + i;
        const int m = r / kRowsPerBlock;
        // the producer units whose tile ranges meet row block m are contiguous
        const int u0 = tile_slot(m * c.ntn, c.total, c.n_slots);
        const int u1 = tile_slot(m * c.ntn + c.ntn - 1, c.total, c.n_slots);
        RowState st;
        row_state_init(st);
        const size_t base = static_cast<size_t>(r) * c.n_slots;
        for (int s = u0 + lane; s <= u1; s += 4 * 32) {
            // four slots per lane per pass, all loads in flight together
            RowState p[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (s + 32 * k <= u1) partial_load(c.part, base + s + 32 * k, p[k]);
                else row_state_init(p[k]);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) row_state_merge(st, p[k]);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
            RowState o;
            o.m = __shfl_xor_sync(0xFFFFFFFFu, st.m, off);
            o.S = __shfl_xor_sync(0xFFFFFFFFu, st.S, off);
            o.A = __shfl_xor_sync(0xFFFFFFFFu, st.A, off);
            o.gbest = __shfl_xor_sync(0xFFFFFFFFu, st.gbest, off);
            o.gidx = __shfl_xor_sync(0xFFFFFFFFu, st.gidx, off);
            o.amax = __shfl_xor_sync(0xFFFFFFFFu, st.amax, off);
            o.aidx = __shfl_xor_sync(0xFFFFFFFFu, st.aidx, off);
            row_state_merge(st, o);
        }
        if (lane == 0) {
            const float h_raw = 0.6931471805599453f * (log2f(st.S) - st.A / st.S);
            const float h = fmaxf(h_raw, 0.f);
            int gi = st.gidx, ai = st.aidx;
            if (a.checks) {
                // device-side checks: a finite entropy, indices inside the vocabulary
                if (!isfinite(h_raw)) report_error(a.ws, DG_ERR_DEVICE, 801);
                if (gi < 0 || gi >= a.V) {
                    report_error(a.ws, DG_ERR_DEVICE, 802);
                    gi = 0;
                }
                if (ai < 0 || ai >= a.V) {
                    report_error(a.ws, DG_ERR_DEVICE, 803);
                    ai = 0;
                }
            }
            c.H[r] = h;
            c.sample[r] = gi;
            c.argmax[r] = ai;
        }
        if (c.sc_out != nullptr) {
            // self-conditioning read-out: lane k sums component k of the
            // units' parts in unit order, each weighed by 2^(m_unit - m), then
            // divides by S (every lane holds the same merged m and S)
            float o = 0.f;
            for (int s = u0; s <= u1; ++s) {
                const size_t i = base + s;
                const float Ss = __ldcg(c.part.S + i);
                if (Ss > 0.f)
                    o = fmaf(fast_exp2(__ldcg(c.part.m + i) - st.m),
                             __ldcg(c.sc_part + i * kScDim + lane), o);
            }
            c.sc_out[static_cast<size_t>(r) * kScDim + lane] = o / st.S;
        }
    }
    // last CTA of this canvas?
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        // release this CTA's rows, acquire every other CTA's (acq_rel add)
        const int prev = atomic_add_acq_rel_gpu(&c.counters[b], 1);
        s_last = (prev == static_cast<int>(gridDim.x) - 1);
        if (s_last) c.counters[b] = 0;
    }
    __syncthreads();
    if (!s_last) return;
    const int step =
        (a.ctl != nullptr) ? *reinterpret_cast<volatile int32_t *>(&a.ctl->step) : a.step;
    accept_canvas(a, b, step, c.H, c.sample, c.argmax);
    if (a.ctl != nullptr) {
        __syncthreads();
        if (threadIdx.x == 0) loop_advance(a);
    }
}

// Acceptance alone on given entropy / sample / argmax (one CTA per canvas).
__global__ void __launch_bounds__(kAcceptThreads) accept_only_kernel(const float *__restrict__ H,
                                                          const int32_t *__restrict__ sample,
                                                          const int32_t *__restrict__ argmax,
                                                          AcceptArgs a)
{
    accept_canvas(a, blockIdx.x, a.step, H, sample, argmax);
}

// ---------------------------------------------------------------- block-loop init
__global__ void loop_init_kernel(LoopCtl *ctl, int max_steps, double t0, double t1, int B,
                                 int32_t *done, int32_t *steps_taken, int32_t *canvas,
                                 int32_t *prev_argmax, int n, uint32_t V, uint32_t k0,
                                 uint32_t k1)
{
    const int tid = blockIdx.x * blockDim.x + threadIdx.x;
    const int stride = gridDim.x * blockDim.x;
    if (tid == 0) {
        ctl->step = 0;
        ctl->max_steps = max_steps;
        ctl->canvases_finished = 0;
        ctl->n_live = B;
    }
    for (int k = tid; k < max_steps; k += stride) {
        // T_k = t0 + (t1 - t0) k / (N - 1), in fp64
        const double T = (max_steps <= 1) ? t0
                                          : t0 + (t1 - t0) * static_cast<double>(k) /
                                                     static_cast<double>(max_steps - 1);
        const float invT = static_cast<float>(1.0 / T);
        ctl->invT[k] = invT;
        ctl->c2[k] = __fmul_rn(invT, __uint_as_float(0x3FB8AA3Bu));   // * log2(e)
    }
    for (int b = tid; b < B; b += stride) {
        done[b] = 0;
        steps_taken[b] = 0;
    }
    for (int r = tid; r < n; r += stride) {
        // "DiffusionGemma Lab" section 2 item 1: uniform random init, not [MASK]
        const uint4 x = philox4x32_10(make_uint4(0u, static_cast<uint32_t>(r), 0u, kStreamInit),
                                      k0, k1);
        canvas[r] = static_cast<int32_t>(token_from_word(x.x, V));
        prev_argmax[r] = -1;
    }
}

// ---------------------------------------------------------------- hidden-state producers
// Slice k (= *step, read on the device) of precomputed hidden states.
__global__ void hidden_from_steps_kernel(const int32_t *step, const uint16_t *__restrict__ src,
                                         int64_t step_stride, int64_t n, uint16_t *__restrict__ out)
{
    const int64_t k = *reinterpret_cast<const volatile int32_t *>(step);
    const uint16_t *s = src + k * step_stride;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        out[i] = s[i];
}

// hidden[r, j] = bf16(base_k[r, j] + table[canvas[r], j]) (fp32 sum, nearest even).
__global__ void hidden_embed_add_kernel(const int32_t *step, const int32_t *__restrict__ canvas,
                                        const uint16_t *__restrict__ base, int64_t base_step_stride,
                                        const uint16_t *__restrict__ table, int rows, int d, int V,
                                        uint16_t *__restrict__ out)
{
    const int64_t k = *reinterpret_cast<const volatile int32_t *>(step);
    const uint16_t *b = base + k * base_step_stride;
    const int64_t n = static_cast<int64_t>(rows) * d;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / d, j = i % d;
        int tok = canvas[r];
        tok = tok < 0 ? 0 : (tok >= V ? V - 1 : tok);
        const float v = __uint_as_float(static_cast<uint32_t>(b[i]) << 16) +
                        __uint_as_float(static_cast<uint32_t>(table[static_cast<int64_t>(tok) * d + j]) << 16);
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        out[i] = *reinterpret_cast<const uint16_t *>(&h);
    }
}

// ---------------------------------------------------------------- check kernels
__global__ void gumbel_fill_kernel(uint32_t k0, uint32_t k1, uint32_t row, uint32_t step,
                                   uint32_t v0, int n, float *out)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < n) {
        const uint32_t v = v0 + static_cast<uint32_t>(t);
        const uint4 r = philox4x32_10(make_uint4(v >> 2, row, step, kStreamGumbel), k0, k1);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
        out[t] = gumbel_from_bits(w[v & 3u]);
    }
}

// The failure path of a bounded wait, on its own: one warp allocates TMEM,
// waits on an mbarrier that nothing arrives on, gives up after limit_ns
// (DG_ERR_TIMEOUT in the workspace header), frees its TMEM and returns.  A
// wait that completed would be a bug and is reported as DG_ERR_DEVICE.
__global__ void __launch_bounds__(32) wait_probe_kernel(WsHeader *ws, uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tslot;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    tmem_alloc(&tslot, 32);
    tmem_relinquish();
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    const uint32_t taddr = tslot;
    if (threadIdx.x == 0) {
        // phase 0 of a fresh barrier completes only after one arrival
        if (mbar_wait_limit(&bar, 0u, ws, 901, limit_ns)) report_error(ws, DG_ERR_DEVICE, 902);
    }
    tc_fence_before();
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(taddr, 32);
}

__global__ void logf_eval_kernel(const float *x, float *y, int n)
{
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t < n) y[t] = sampler_logf(x[t]);
}

}  // namespace dg
