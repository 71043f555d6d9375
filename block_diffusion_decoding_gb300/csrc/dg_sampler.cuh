// dg_sampler.cuh -- per-position sampler state folded over vocabulary tiles.
//
// "DiffusionGemma Lab", section 2 items 2 and 5: each canvas position needs
// the entropy of its sampling distribution softmax(logits / T) (the ranking
// key of the acceptance rule), a multinomial sample (what gets committed) and
// the argmax (the output canvas).  All three are folds over the vocabulary,
// so they are computed tile by tile as the LM-head accumulators come out of
// TMEM and merged afterwards; the logits themselves are never stored.
//
// Softmax statistics are kept in base 2: with t = logit * (log2(e) / T),
//   m = max t,  S = sum 2^(t - m),  A = sum 2^(t - m) (t - m),
// and the entropy in nats is  H = ln 2 * (log2 S - A / S).
// Two partial states merge exactly (up to rounding):
//   m = max(m1, m2), f_i = 2^(m_i - m),
//   S = f1 S1 + f2 S2,  A = f1 (A1 + (m1 - m) S1) + f2 (A2 + (m2 - m) S2).
// The Gumbel-max sample keeps the best fp32 score fmaf(logit, 1/T, G_v) and
// its index; the argmax keeps the best logit and its index; ties go to the
// lower vocabulary index in every merge.
#pragma once

#include "dg_device.cuh"

namespace dg {

struct RowState {
    float m;      // running max of t (base-2 scaled logits)
    float S;      // sum 2^(t - m)
    float A;      // sum 2^(t - m) (t - m)
    float gbest;  // best Gumbel score
    int gidx;     // its vocabulary index
    float amax;   // best logit
    int aidx;     // its vocabulary index
};

DG_DEVICE void row_state_init(RowState &s)
{
    s.m = -INFINITY;
    s.S = 0.f;
    s.A = 0.f;
    s.gbest = -INFINITY;
    s.gidx = 0x7FFFFFFF;
    s.amax = -INFINITY;
    s.aidx = 0x7FFFFFFF;
}

DG_DEVICE float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Per-step constants of the fold.
struct FoldConsts {
    float invT;      // fp32(1/T): the Gumbel score multiplier
    float c2;        // fp32(invT * log2(e)): softmax scale in base 2
    uint32_t k0, k1; // Philox key (seed lo, seed hi)
    uint32_t step;   // Philox counter word 2
};

// Fold 16 consecutive logits lg[0..15] of vocabulary entries v0 .. v0+15
// (v0 a multiple of 16) of canvas row `row` into the state.  Entries >= V
// are ignored.
DG_DEVICE void fold16(RowState &st, const float (&lg)[16], uint32_t v0, uint32_t V,
                      uint32_t row, const FoldConsts &fc)
{
    const bool full = v0 + 16u <= V;
    float t[16];
    float cmax = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const bool ok = full || (v0 + j < V);
        t[j] = ok ? __fmul_rn(lg[j], fc.c2) : -INFINITY;
        cmax = fmaxf(cmax, t[j]);
    }
    if (cmax > st.m) {
        if (st.S > 0.f) {
            const float f = fast_exp2(st.m - cmax);
            st.A = f * fmaf(st.m - cmax, st.S, st.A);
            st.S = f * st.S;
        }
        st.m = cmax;
    }
    if (full) {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const float dlt = t[j] - st.m;
            const float e = fast_exp2(dlt);
            st.S += e;
            st.A = fmaf(e, dlt, st.A);
            if (lg[j] > st.amax) { st.amax = lg[j]; st.aidx = static_cast<int>(v0 + j); }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (v0 + j < V) {
                const float dlt = t[j] - st.m;
                const float e = fast_exp2(dlt);
                st.S += e;
                st.A = fmaf(e, dlt, st.A);
                if (lg[j] > st.amax) { st.amax = lg[j]; st.aidx = static_cast<int>(v0 + j); }
            }
        }
    }
    // Gumbel-max: counter (v >> 2, row, step, 0), word v & 3.
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 r = philox4x32_10(make_uint4((v0 >> 2) + q, row, fc.step, kStreamGumbel),
                                      fc.k0, fc.k1);
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int j = 4 * q + b;
            if (full || (v0 + j < V)) {
                const float g = gumbel_from_bits(w[b]);
                const float sc = __fmaf_rn(lg[j], fc.invT, g);
                if (sc > st.gbest) { st.gbest = sc; st.gidx = static_cast<int>(v0 + j); }
            }
        }
    }
}

DG_DEVICE void row_state_merge(RowState &a, const RowState &b)
{
    if (b.S > 0.f) {
        if (a.S > 0.f) {
            const float m = fmaxf(a.m, b.m);
            const float fa = fast_exp2(a.m - m), fb = fast_exp2(b.m - m);
            const float S = fa * a.S + fb * b.S;
            const float A = fa * fmaf(a.m - m, a.S, a.A) + fb * fmaf(b.m - m, b.S, b.A);
            a.m = m;
            a.S = S;
            a.A = A;
        } else {
            a.m = b.m;
            a.S = b.S;
            a.A = b.A;
        }
    }
    if (b.gbest > a.gbest || (b.gbest == a.gbest && b.gidx < a.gidx)) {
        a.gbest = b.gbest;
        a.gidx = b.gidx;
    }
    if (b.amax > a.amax || (b.amax == a.amax && b.aidx < a.aidx)) {
        a.amax = b.amax;
        a.aidx = b.aidx;
    }
}

// Partial states in global memory: structure of arrays, slot-major
// ([n_slots][M]), so consecutive rows of one slot are contiguous.
struct Partials {
    float *m, *S, *A, *gbest, *amax;
    int *gidx, *aidx;
};

DG_DEVICE void partial_store(const Partials &p, size_t i, const RowState &s)
{
    p.m[i] = s.m;
    p.S[i] = s.S;
    p.A[i] = s.A;
    p.gbest[i] = s.gbest;
    p.gidx[i] = s.gidx;
    p.amax[i] = s.amax;
    p.aidx[i] = s.aidx;
}

DG_DEVICE void partial_load(const Partials &p, size_t i, RowState &s)
{
    s.m = __ldcg(p.m + i);
    s.S = __ldcg(p.S + i);
    s.A = __ldcg(p.A + i);
    s.gbest = __ldcg(p.gbest + i);
    s.gidx = __ldcg(p.gidx + i);
    s.amax = __ldcg(p.amax + i);
    s.aidx = __ldcg(p.aidx + i);
}

// Static schedule shared by the producers of partial states and the
// combine: `total` tiles, ordered row-block-major (tile t covers row block
// t / tiles_per_block and vocabulary tile t % tiles_per_block), are split
// into `n_slots` contiguous ranges; slot c owns [tile_begin(c), tile_begin(c+1)).
__host__ __device__ inline int tile_begin(int c, int total, int n_slots)
{
    const int q = total / n_slots, rem = total % n_slots;
    return c * q + (c < rem ? c : rem);
}

// Device-resident control block of the block loop (in the workspace).  The
// step index and the per-step temperature constants live here so that one
// captured graph body serves every step.
constexpr int kMaxLoopSteps = 1024;
struct LoopCtl {
    int32_t step;              // index k of the step being run
    int32_t max_steps;
    int32_t canvases_finished; // canvases whose acceptance ran this step
    int32_t n_live;            // canvases that have not stopped
    float invT[kMaxLoopSteps]; // fp32(1/T_k)
    float c2[kMaxLoopSteps];   // fp32(invT_k * log2 e)
};

// Where a kernel reads the step index and temperature from: the launch
// parameters (single step) or the loop control block (block loop).
struct StepSource {
    const LoopCtl *ctl;        // null: use the fields below
    float invT, c2;
    int32_t step;
};

DG_DEVICE FoldConsts fold_consts(const StepSource &src, uint64_t seed)
{
    FoldConsts fc;
    if (src.ctl != nullptr) {
        const int k = *reinterpret_cast<const volatile int32_t *>(&src.ctl->step);
        fc.invT = src.ctl->invT[k];
        fc.c2 = src.ctl->c2[k];
        fc.step = static_cast<uint32_t>(k);
    } else {
        fc.invT = src.invT;
        fc.c2 = src.c2;
        fc.step = static_cast<uint32_t>(src.step);
    }
    fc.k0 = static_cast<uint32_t>(seed);
    fc.k1 = static_cast<uint32_t>(seed >> 32);
    return fc;
}

}  // namespace dg
