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
    float gbest;  // best exact Gumbel score among the columns evaluated exactly
    int gidx;     // its vocabulary index
    float amax;   // best logit
    int aidx;     // its vocabulary index
    // fold only (not part of the stored partial): best approximate Gumbel
    // score seen, and the column holding it if it is still unevaluated
    float glb;    // a lower bound on the row's best exact score over the whole
                  // vocabulary, from other units of the same launch (-inf: none)
    float apb;    // best approximate score (-inf: none yet)
    float kx;     // kept column: logit
    uint32_t kw;  // kept column: Philox word
    int kj;       // kept column: vocabulary index, -1 = none
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
    s.glb = -INFINITY;
    s.apb = -INFINITY;
    s.kx = 0.f;
    s.kw = 0u;
    s.kj = -1;
}

// Self-conditioning read-out ("Parallel Denoising From an Autoregressive
// Checkpoint", section "Finding": a 7.8M-parameter block feeds the previous
// prediction back; its matmul runs in the sampling stage next to the
// full-vocabulary softmax).  Per canvas row, sc = sum_v softmax(logits /
// T)_v E[v, :] over a table E [V, kScDim] (bf16).  The fold keeps
// o = sum_v 2^(t_v - m) E[v, :] next to S, rescaled with it whenever the
// running maximum m moves; a merge weighs each part by 2^(m_part - m); the
// read-out is o / S.
//
// A warp folds 32 rows (one per lane) x 16 columns per chunk, so the chunk's
// part of o is a 32 x 16 x 32 product P E with P = 2^(t - m): it runs on the
// tensor cores as two m16 x four n8 mma.sync m16n8k16 (bf16 P and E, fp32
// accumulate).  P goes through a 1 KB per-warp shared buffer (ldmatrix gives
// the A fragments), E's 16 rows come from the tile's table rows in shared
// memory (ldmatrix.trans gives the B fragments).  The accumulator is held in
// the mma fragment layout: lane (g = lane / 4, t = lane % 4) holds rows g,
// g + 8 (first m16 tile) and g + 16, g + 24 (second) at columns 8 j + 2 t,
// 8 j + 2 t + 1 of n8 tile j.
constexpr int kScDim = 32;

struct ScAcc {
    float c[2][4][4];   // [m16 tile][n8 tile][fragment register]
};

DG_DEVICE void sc_init(ScAcc &a)
{
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) a.c[mt][j][r] = 0.f;
}

DG_DEVICE float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Multiply row r of the accumulator by the factor lane r holds.  All 32
// lanes call it together.
DG_DEVICE void sc_scale_rows(ScAcc &a, float f)
{
    if (!__any_sync(0xFFFFFFFFu, f != 1.0f)) return;
    const int g = (threadIdx.x & 31) >> 2;
    const float f0 = __shfl_sync(0xFFFFFFFFu, f, g), f1 = __shfl_sync(0xFFFFFFFFu, f, g + 8);
    const float f2 = __shfl_sync(0xFFFFFFFFu, f, g + 16), f3 = __shfl_sync(0xFFFFFFFFu, f, g + 24);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        a.c[0][j][0] *= f0;
        a.c[0][j][1] *= f0;
        a.c[0][j][2] *= f1;
        a.c[0][j][3] *= f1;
        a.c[1][j][0] *= f2;
        a.c[1][j][1] *= f2;
        a.c[1][j][2] *= f3;
        a.c[1][j][3] *= f3;
    }
}

DG_DEVICE uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// o += P E for one chunk: es[q] = (P[row][2q], P[row][2q + 1]) of this
// lane's row; Ec = the chunk's 16 table rows (bf16 [16][kScDim], shared,
// 16-byte aligned); pbuf = this warp's 32 x 16 bf16 staging buffer (shared).
// All 32 lanes call it together.
DG_DEVICE void sc_add_chunk(ScAcc &a, const float2 (&es)[8], const uint16_t *Ec, uint16_t *pbuf)
{
    const int lane = threadIdx.x & 31;
    uint4 lo, hi;
    lo.x = pack_bf16x2(es[0].x, es[0].y);
    lo.y = pack_bf16x2(es[1].x, es[1].y);
    lo.z = pack_bf16x2(es[2].x, es[2].y);
    lo.w = pack_bf16x2(es[3].x, es[3].y);
    hi.x = pack_bf16x2(es[4].x, es[4].y);
    hi.y = pack_bf16x2(es[5].x, es[5].y);
    hi.z = pack_bf16x2(es[6].x, es[6].y);
    hi.w = pack_bf16x2(es[7].x, es[7].y);
    __syncwarp();   // the previous chunk's fragments were read
    reinterpret_cast<uint4 *>(pbuf + lane * 16)[0] = lo;
    reinterpret_cast<uint4 *>(pbuf + lane * 16)[1] = hi;
    __syncwarp();
    uint32_t af[2][4], bf[4][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        // matrices: rows 0-7 / 8-15 of the m16 tile at columns 0-7, then 8-15
        const uint32_t addr = smem_u32(pbuf + (mt * 16 + (lane & 15)) * 16 + (lane >> 4) * 8);
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(af[mt][0]), "=r"(af[mt][1]), "=r"(af[mt][2]), "=r"(af[mt][3])
                     : "r"(addr)
                     : "memory");
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        // matrices: k 0-7 / 8-15 of n8 tile 2h, then of n8 tile 2h + 1
        const int mat = lane >> 3;
        const int k = (lane & 7) + 8 * (mat & 1);
        const int n0 = 16 * h + 8 * (mat >> 1);
        const uint32_t addr = smem_u32(Ec + k * kScDim + n0);
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(bf[2 * h][0]), "=r"(bf[2 * h][1]), "=r"(bf[2 * h + 1][0]),
                       "=r"(bf[2 * h + 1][1])
                     : "r"(addr)
                     : "memory");
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
                "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                : "+f"(a.c[mt][j][0]), "+f"(a.c[mt][j][1]), "+f"(a.c[mt][j][2]),
                  "+f"(a.c[mt][j][3])
                : "r"(af[mt][0]), "r"(af[mt][1]), "r"(af[mt][2]), "r"(af[mt][3]),
                  "r"(bf[j][0]), "r"(bf[j][1]));
}

// Before the softmax states of two parts merge (row_state_merge(sa, sb)),
// their read-out parts follow: a <- 2^(ma - m) a + 2^(mb - m) b per row
// (m = max(ma, mb); a part whose S is 0 holds nothing).  sa, sb are this
// lane's row; all 32 lanes call it together.
DG_DEVICE void sc_merge(ScAcc &a, const RowState &sa, const ScAcc &b, const RowState &sb)
{
    float fa = 1.f, fb = 0.f;
    if (sb.S > 0.f) {
        if (sa.S > 0.f) {
            const float m = fmaxf(sa.m, sb.m);
            fa = fast_exp2(sa.m - m);
            fb = fast_exp2(sb.m - m);
        } else {
            fa = 0.f;
            fb = 1.f;
        }
    }
    const int g = (threadIdx.x & 31) >> 2;
    float fA[4], fB[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        fA[i] = __shfl_sync(0xFFFFFFFFu, fa, g + 8 * i);
        fB[i] = __shfl_sync(0xFFFFFFFFu, fb, g + 8 * i);
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = 2 * mt + (r >> 1);   // rows g, g + 8, g + 16, g + 24
                a.c[mt][j][r] = fmaf(fA[i], a.c[mt][j][r], fB[i] * b.c[mt][j][r]);
            }
}

// The positions of this lane's fragment values: row (0..31 within the warp's
// rows) and column of register r of n8 tile j in m16 tile mt.
DG_DEVICE int sc_frag_row(int mt, int r) { return mt * 16 + ((threadIdx.x & 31) >> 2) + 8 * (r >> 1); }
DG_DEVICE int sc_frag_col(int j, int r) { return 8 * j + 2 * (threadIdx.x & 3) + (r & 1); }

// Per-step constants of the fold.
struct FoldConsts {
    float invT;      // fp32(1/T): the Gumbel score multiplier
    float c2;        // fp32(invT * log2(e)): softmax scale in base 2
    uint32_t k0, k1; // Philox key (seed lo, seed hi)
    uint32_t step;   // Philox counter word 2
};

DG_DEVICE float fast_log2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The exact fp32 score fmaf(logit, invT, G) of one column (rarely reached:
// kept out of line so the hot fold stays small).
static __device__ __noinline__ float exact_gumbel_score(float logit, float invT, uint32_t bits)
{
    return __fmaf_rn(logit, invT, gumbel_from_bits(bits));
}

// Pruning of the Gumbel-max search.  A column v can only replace the running
// best score B if its exact score fmaf(logit, invT, G_v) exceeds B, i.e. if
// G_v > B - logit * invT (up to the roundings of the score, a few ulp).
// G_v = -ln(-ln u) never exceeds -ln(-ln(1 - 2^-24)) = 16.636, so columns
// with B - logit * invT > 16.75 are out without drawing their noise (stage
// 1).  For the rest, G_v is estimated (stage 2): -ln u by its series when
// u > 0.99 (relative error < 3e-9) and by the hardware log2 otherwise
// (-ln u >= 0.01 there, so an absolute log2 error of 2^-22 is a relative
// error below 2e-5), then -ln of that by the hardware log2: the estimate is
// within 1e-4 of G_v.  Only columns whose estimated score is within
// 2 kGumbelSlack (= 20x that error) of the larger of B and the chunk's best
// estimate can be the chunk's exact best, so only those are evaluated with
// the exact fp32 sequence, in increasing column order with strict
// improvement: the result is the one of evaluating every column exactly.
constexpr float kGumbelMaxPlusSlack = 16.75f;
constexpr float kGumbelSlack = 1.0e-3f;

// Word threshold of stage 1b.  For a Philox word x the fold uses
// u = ((x >> 9) + 1/2) 2^-23, so 1 - u = ((~x >> 9) + 1/2) 2^-23 exactly.
// G = -ln(-ln u) <= t holds whenever -ln u >= e^-t, and -ln u >= 1 - u, so
// every word with (~x >> 9) >= K = ceil(e^-t 2^23) gives G <= t; in terms of
// x, only words x >= (2^23 - K) << 9 can give G > t.  The caller subtracts
// kGumbelSlack from t, which covers the error of the hardware exp2 here
// (relative 2^-22) and the roundings of the exact score many times over.
// Returns 0 (every word stays) for t = -inf or NaN and for K >= 2^23.
DG_DEVICE uint32_t gumbel_word_threshold(float t)
{
    const float ys = fast_exp2(fmaf(-t, 1.44269504f, 23.0f));   // e^-t 2^23
    if (!(ys < 8388608.0f)) return 0u;
    const uint32_t K = static_cast<uint32_t>(ceilf(ys));          // 0 .. 2^23
    return K == 0u ? 0xFFFFFFFFu : (8388608u - K) << 9;
}

// Fold 16 consecutive logits lg[0..15] of vocabulary entries v0 .. v0+15
// (v0 a multiple of 16, the same for every lane of the warp) of canvas row
// `row` into the state.  Entries >= V are ignored; a lane with live == false
// (a row past the end) leaves its state alone.  Must be called by all 32
// lanes of the warp together (it votes across the warp).
// With kSC, the self-conditioning part sc is folded along with S; E points
// at the table row of vocabulary entry v0 (rows kScDim floats apart).
template <bool kSC>
DG_DEVICE void fold16_t(RowState &st, const float (&lg)[16], uint32_t v0, uint32_t V,
                        uint32_t row, const FoldConsts &fc, bool live, ScAcc *sc,
                        const uint16_t *__restrict__ E, uint16_t *pbuf, uint32_t wtm = 0u)
{
    const bool full = v0 + 16u <= V;
    float x[16];
    float cmax = -INFINITY;
    if (live && full) {
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = lg[j];
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            // ignored entries get a finite sentinel: their exponentials
            // underflow to exactly 0 and no -inf * 0 can appear below
            x[j] = (live && (full || (v0 + j < V))) ? lg[j] : -1.0e30f;
        }
    }
#pragma unroll
    for (int j = 0; j < 16; j += 2) cmax = max3(cmax, x[j], x[j + 1]);
    if (!__any_sync(0xFFFFFFFFu, live)) return;
    // argmax: only a chunk whose maximum beats the running best can move it;
    // the first column holding that maximum wins ties
    if (cmax > st.amax) {
        int jj = 15;
#pragma unroll
        for (int j = 15; j >= 0; --j)
            if (x[j] == cmax) jj = j;
        st.amax = cmax;
        st.aidx = static_cast<int>(v0) + jj;
    }
    // softmax statistics in base 2 (c2 > 0, so the maximum maps through)
    const float mt = cmax * fc.c2;
    float fsc = 1.0f;      // the factor this row's read-out part is rescaled by
    if (mt > st.m) {
        if (st.S > 0.f) {
            const float f = fast_exp2(st.m - mt);
            st.A = f * fmaf(st.m - mt, st.S, st.A);
            st.S = f * st.S;
            fsc = f;
        }
        st.m = mt;
    }
    if constexpr (kSC) sc_scale_rows(*sc, fsc);
    // on pairs of columns (packed fp32: the same roundings as one column at
    // a time); the sums run as a fixed tree, column j with j + 8, then + 4,
    // + 2, + 1
    float2 es[8], as[8];
    const float2 c2v = make_float2(fc.c2, fc.c2), nm = make_float2(-st.m, -st.m);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float2 dlt = fma2(make_float2(x[2 * q], x[2 * q + 1]), c2v, nm);
        const float2 e = make_float2(fast_exp2(dlt.x), fast_exp2(dlt.y));   // 0 for ignored entries
        es[q] = e;
        as[q] = mul2(e, dlt);
    }
    // the chunk's read-out part (columns past V and rows past M weigh 0; the
    // table rows past V are zero-filled)
    if constexpr (kSC) sc_add_chunk(*sc, es, E, pbuf);
#pragma unroll
    for (int h = 4; h >= 1; h >>= 1) {
#pragma unroll
        for (int q = 0; q < h; ++q) {
            es[q] = add2(es[q], es[q + h]);
            as[q] = add2(as[q], as[q + h]);
        }
    }
    if (live) {
        st.S += es[0].x + es[0].y;
        st.A += as[0].x + as[0].y;
    }
    // Gumbel-max over the columns that can still win: counter (v >> 2, row,
    // step, 0), word v & 3.  lb is a lower bound on the exact best score of
    // the row: the best exact score found here, the best estimate less twice
    // its error margin, or the bound other units of the launch published.
    // Stage 1 (logits only) decides whether the warp draws the noise of this
    // chunk at all.
    const float lb = fmaxf(fmaxf(st.gbest, st.apb - 2.0f * kGumbelSlack), st.glb);
    // rounding is monotone, so the chunk's largest scaled logit is cmax * invT
    const float cz = cmax * fc.invT;
    if (!__any_sync(0xFFFFFFFFu, cz > lb - kGumbelMaxPlusSlack)) return;
    uint32_t w[16];
    if (wtm != 0u) {
        // the chunk's noise words, computed ahead into TMEM (same layout)
        tmem_ld16_issue(wtm, w);
        tmem_wait_ld16(w);
    } else {
        uint4 r[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) r[q] = make_uint4((v0 >> 2) + q, row, fc.step, kStreamGumbel);
        philox4x32_10_x4(r, fc.k0, fc.k1);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            w[4 * q] = r[q].x;
            w[4 * q + 1] = r[q].y;
            w[4 * q + 2] = r[q].z;
            w[4 * q + 3] = r[q].w;
        }
    }
    // Stage 1b (noise words only): a column of this chunk can reach lb only
    // if its Gumbel value exceeds lb - cz; the columns whose word is below the
    // threshold of gumbel_word_threshold cannot, and need no logarithm.
    const uint32_t wthr = gumbel_word_threshold(lb - cz - kGumbelSlack);
    // no column of the warp can win: stage 2 would change nothing (tested on
    // the chunk's largest word first; the per-column mask is built only for
    // a chunk that goes on)
    uint32_t wmax = w[0];
#pragma unroll
    for (int j = 1; j < 16; ++j) wmax = max(wmax, w[j]);
    if (!__any_sync(0xFFFFFFFFu, live && wmax >= wthr)) return;
    uint32_t in = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) in |= (w[j] >= wthr ? 1u : 0u) << j;
    if (!live) in = 0;
    // Stage 2: approximate scores lz + G~.  A column can end up as the chunk's
    // exact best only if its approximate score is within twice the estimate's
    // error of the chunk's best approximate score, and above the running best.
    // Columns stage 1 or 1b ruled out score below lb (they cannot be the
    // best); a group of four columns (one Philox block) that no lane of the
    // warp let through is skipped whole.
    float ap[16];
    float amax = -INFINITY;
    const uint32_t qin = ((in & 0x000Fu) ? 1u : 0u) | ((in & 0x00F0u) ? 2u : 0u) |
                         ((in & 0x0F00u) ? 4u : 0u) | ((in & 0xF000u) ? 8u : 0u);
    const uint32_t qany = __reduce_or_sync(0xFFFFFFFFu, qin);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if ((qany >> q) & 1u) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j0 = 4 * q + 2 * h;
                const float2 z = mul2(make_float2(x[j0], x[j0 + 1]), make_float2(fc.invT, fc.invT));
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    const int j = j0 + t;
                    // u = ((x >> 9) + 1/2) 2^-23 = (1 + (x >> 9) 2^-23) - (1 - 2^-24), exact
                    const float u = __fadd_rn(__uint_as_float(0x3F800000u | (w[j] >> 9)), -0.99999994f);
                    const float om = 1.0f - u;   // exact
                    // -ln u: series near u = 1 (relative error < 3e-9), hardware log2 below
                    const float e1 = (u > 0.99f) ? fmaf(om * om, 0.5f + om * (1.0f / 3.0f), om)
                                                 : -0.69314718f * fast_log2(u);
                    const float g = -0.69314718f * fast_log2(e1);
                    ap[j] = ((in >> j) & 1u) ? (t ? z.y : z.x) + g : -INFINITY;
                    amax = fmaxf(amax, ap[j]);
                }
            }
        } else {
#pragma unroll
            for (int t = 0; t < 4; ++t) ap[4 * q + t] = -INFINITY;
        }
    }
    // Deferred exact evaluation.  Invariant: the exact best of the columns
    // seen so far is either among those evaluated exactly (gbest, gidx) or is
    // the kept column (kj).  Every column whose estimate is more than
    // 2 kGumbelSlack below the best estimate seen (apb) is more than
    // kGumbelSlack below the exact score of the column holding apb, so it
    // cannot be the exact best and is dropped.
    const float apb_new = fmaxf(st.apb, amax);
    const float thr = apb_new - 2.0f * kGumbelSlack;
    uint32_t cand = 0;
    if (amax > thr) {   // only a chunk that reaches the contending range has candidates
#pragma unroll
        for (int j = 0; j < 16; ++j) cand |= (ap[j] > thr ? 1u : 0u) << j;
    }
    const bool keep_alive = st.kj >= 0 && st.apb > thr;   // the kept column still contends
    if (!keep_alive) st.kj = -1;
    st.apb = apb_new;
    const bool fast = (__popc(cand) <= 1) && !(keep_alive && cand != 0);
    if (fast) {
        // at most one contender in this chunk and none left over: keep it
        if (cand != 0) {
            const int j = __ffs(cand) - 1;
            uint32_t wj = w[0];
            float xj = x[0];
#pragma unroll
            for (int t = 1; t < 16; ++t)
                if (t == j) { wj = w[t]; xj = x[t]; }
            st.kj = static_cast<int>(v0) + j;
            st.kw = wj;
            st.kx = xj;
        }
    }
    // near ties (rare): evaluate every contender exactly, then nothing is kept
    uint32_t slow = fast ? 0u : cand;
    const bool flush_kept = !fast && st.kj >= 0;
    if (flush_kept) {
        const float sc = exact_gumbel_score(st.kx, fc.invT, st.kw);
        if (sc > st.gbest || (sc == st.gbest && st.kj < st.gidx)) { st.gbest = sc; st.gidx = st.kj; }
        st.kj = -1;
    }
    while (__any_sync(0xFFFFFFFFu, slow != 0)) {
        if (slow != 0) {
            const int j = __ffs(slow) - 1;
            slow &= slow - 1u;
            uint32_t wj = w[0];
            float xj = x[0];
#pragma unroll
            for (int t = 1; t < 16; ++t)
                if (t == j) { wj = w[t]; xj = x[t]; }
            const float sc = exact_gumbel_score(xj, fc.invT, wj);
            const int idx = static_cast<int>(v0) + j;
            if (sc > st.gbest || (sc == st.gbest && idx < st.gidx)) { st.gbest = sc; st.gidx = idx; }
        }
    }
}

DG_DEVICE void fold16(RowState &st, const float (&lg)[16], uint32_t v0, uint32_t V,
                      uint32_t row, const FoldConsts &fc, bool live, uint32_t wtm = 0u)
{
    fold16_t<false>(st, lg, v0, V, row, fc, live, nullptr, nullptr, nullptr, wtm);
}

// The noise words of the chunks fold_tile visits (first, first + stride,
// ... < BN, columns vbase + c), written to TMEM at wtb + c for this warp's
// lanes, so that the fold loads them instead of running Philox.  All 32
// lanes call it together.
DG_DEVICE void noise_to_tmem(uint32_t wtb, int first, int stride, int BN, uint32_t vbase,
                             uint32_t V, uint32_t row, const FoldConsts &fc)
{
#pragma unroll 1
    for (int c0 = first; c0 < BN; c0 += stride) {
        const uint32_t v0 = vbase + static_cast<uint32_t>(c0);
        if (v0 >= V) break;
        uint4 r[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) r[q] = make_uint4((v0 >> 2) + q, row, fc.step, kStreamGumbel);
        philox4x32_10_x4(r, fc.k0, fc.k1);
        uint32_t w[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            w[4 * q] = r[q].x;
            w[4 * q + 1] = r[q].y;
            w[4 * q + 2] = r[q].z;
            w[4 * q + 3] = r[q].w;
        }
        tmem_st16(wtb + static_cast<uint32_t>(c0), w);
    }
    tmem_wait_st();
}

// Resolve the kept column (evaluate it exactly) before the state is stored.
DG_DEVICE void row_state_finalize(RowState &st, const FoldConsts &fc)
{
    if (st.kj >= 0) {
        const float sc = exact_gumbel_score(st.kx, fc.invT, st.kw);
        if (sc > st.gbest || (sc == st.gbest && st.kj < st.gidx)) { st.gbest = sc; st.gidx = st.kj; }
        st.kj = -1;
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

// Fold one accumulator tile into a row's state: the 16-column chunks
// first, first + stride, ... < BN at TMEM address tb (this warp's lane
// quadrant, the buffer's first column) of vocabulary entries vbase + c.  All
// 32 lanes of the warp call it together.  (Loading the next chunk while one
// is folded needs 16 more live registers than the 96 a thread has here and
// spills; it measured slower.)
DG_DEVICE void fold_tile(RowState &st, uint32_t tb, int first, int stride, int BN, uint32_t vbase,
                         uint32_t V, uint32_t row, const FoldConsts &fc, bool live,
                         uint32_t wtb = 0u)
{
#pragma unroll 1
    for (int c0 = first; c0 < BN; c0 += stride) {
        float lg[16];
        tmem_ld16(tb + static_cast<uint32_t>(c0), lg);
        const uint32_t v0 = vbase + static_cast<uint32_t>(c0);
        // one call site of the (large) fold keeps the loop in the instruction cache
        if (v0 < V) fold16(st, lg, v0, V, row, fc, live, wtb ? wtb + static_cast<uint32_t>(c0) : 0u);
    }
}

// fold_tile with the self-conditioning part: Et holds the table rows of the
// tile's columns vbase, vbase + 1, ... (kScDim bf16 each, shared memory);
// pbuf is the warp's staging buffer.
DG_DEVICE void fold_tile_sc(RowState &st, ScAcc &sc, const uint16_t *__restrict__ Et, uint16_t *pbuf,
                            uint32_t tb, int first, int stride, int BN, uint32_t vbase, uint32_t V,
                            uint32_t row, const FoldConsts &fc, bool live)
{
#pragma unroll 1
    for (int c0 = first; c0 < BN; c0 += stride) {
        float lg[16];
        tmem_ld16(tb + static_cast<uint32_t>(c0), lg);
        const uint32_t v0 = vbase + static_cast<uint32_t>(c0);
        if (v0 < V) fold16_t<true>(st, lg, v0, V, row, fc, live, &sc, Et + c0 * kScDim, pbuf);
    }
}

// fold_tile for FP8 operands: the accumulator holds sum_k dec(x8) dec(w8);
// logit = (acc * rs) * cs[v] with the row's scale rs and the column scales
// cs (fp32 [V], 16-byte aligned).
DG_DEVICE void fold_tile_scaled(RowState &st, uint32_t tb, int first, int stride, int BN,
                                uint32_t vbase, uint32_t V, uint32_t row, const FoldConsts &fc,
                                bool live, float rs, const float *__restrict__ cs)
{
    const float2 rs2 = make_float2(rs, rs);
#pragma unroll 1
    for (int c0 = first; c0 < BN; c0 += stride) {
        float lg[16];
        tmem_ld16(tb + static_cast<uint32_t>(c0), lg);
        const uint32_t v0 = vbase + static_cast<uint32_t>(c0);
        if (v0 < V) {
            if (v0 + 16u <= V) {
                // (acc * rs) * cs on column pairs, the same roundings as one at a time
                const float4 *c4 = reinterpret_cast<const float4 *>(cs + v0);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 c = __ldg(c4 + j);
                    const float2 p0 = mul2(mul2(make_float2(lg[4 * j], lg[4 * j + 1]), rs2),
                                           make_float2(c.x, c.y));
                    const float2 p1 = mul2(mul2(make_float2(lg[4 * j + 2], lg[4 * j + 3]), rs2),
                                           make_float2(c.z, c.w));
                    lg[4 * j + 0] = p0.x;
                    lg[4 * j + 1] = p0.y;
                    lg[4 * j + 2] = p1.x;
                    lg[4 * j + 3] = p1.y;
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    lg[j] = (v0 + j < V) ? __fmul_rn(__fmul_rn(lg[j], rs), __ldg(cs + v0 + j)) : 0.f;
            }
            fold16(st, lg, v0, V, row, fc, live);
        }
    }
}

// Partial states in global memory: structure of arrays, row-major
// ([M][n_slots]), so the slots of one row are contiguous (the combine reads
// them with one lane per slot).
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

// The slot whose range holds tile t (0 <= t < total): the first `rem` slots
// own q + 1 tiles each, the others q.
__host__ __device__ inline int tile_slot(int t, int total, int n_slots)
{
    const int q = total / n_slots, rem = total % n_slots;
    const int big = rem * (q + 1);
    return t < big ? t / (q + 1) : rem + (t - big) / q;
}

// Merge of the column groups' states inside one LM-head CTA before the
// single store per (row, CTA).  The epilogue warps of group g > 0 put their
// finalized states into shared memory ([g - 1][field][row]) and arrive on
// `ready`; the group-0 warps wait, merge them into their own state, store,
// and arrive on `done`, which group g > 0 waits for before it writes the
// buffer again at the next row-block boundary.  `k` counts the merges of
// this CTA (the phase of both barriers).  All waits are bounded.
struct GroupMerge {
    float *buf;          // shared: (G - 1) x 7 x rows words
    uint64_t *ready;     // count: warps of groups 1 .. G-1
    uint64_t *done;      // count: warps of group 0
    int G;               // column groups
    int rows;            // rows of the CTA
};

// Self-conditioning parts of the column groups (kSC): (G - 1) x kScDim x
// rows words of shared memory after the states, and the per-(row, unit)
// parts in global memory ([M][n_slots][kScDim], unnormalised, relative to
// the stored state's m).
struct ScMerge {
    float *buf;          // shared
    float *part;         // global
};

template <bool kSC>
DG_DEVICE void group_merge_store_t(RowState &st, int cg, int rix, uint32_t k,
                                   const GroupMerge &gm, const Partials &p, size_t idx,
                                   bool store, WsHeader *ws, ScAcc *sc, const ScMerge &sm)
{
    const int lane = threadIdx.x & 31;
    if (cg != 0) {
        bool ok = true;
        if (k > 0) ok = mbar_wait(gm.done, (k - 1) & 1u, ws, 120);
        if (ok) {
            float *f = gm.buf + static_cast<size_t>(cg - 1) * 7 * gm.rows + rix;
            f[0 * gm.rows] = st.m;
            f[1 * gm.rows] = st.S;
            f[2 * gm.rows] = st.A;
            f[3 * gm.rows] = st.gbest;
            f[4 * gm.rows] = __int_as_float(st.gidx);
            f[5 * gm.rows] = st.amax;
            f[6 * gm.rows] = __int_as_float(st.aidx);
            if constexpr (kSC) {
                // [column][row] words; this lane's fragment positions
                float *o = sm.buf + static_cast<size_t>(cg - 1) * kScDim * gm.rows + (rix & ~31);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            o[sc_frag_col(j, r) * gm.rows + sc_frag_row(mt, r)] = sc->c[mt][j][r];
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(gm.ready);
        return;
    }
    // (warp-uniform: the read-out merge below exchanges values between lanes)
    const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(gm.ready, k & 1u, ws, 121));
    if (ok) {
        for (int g = 1; g < gm.G; ++g) {
            const float *f = gm.buf + static_cast<size_t>(g - 1) * 7 * gm.rows + rix;
            RowState o;
            o.m = f[0 * gm.rows];
            o.S = f[1 * gm.rows];
            o.A = f[2 * gm.rows];
            o.gbest = f[3 * gm.rows];
            o.gidx = __float_as_int(f[4 * gm.rows]);
            o.amax = f[5 * gm.rows];
            o.aidx = __float_as_int(f[6 * gm.rows]);
            if constexpr (kSC) {
                const float *ob =
                    sm.buf + static_cast<size_t>(g - 1) * kScDim * gm.rows + (rix & ~31);
                ScAcc b;
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            b.c[mt][j][r] = ob[sc_frag_col(j, r) * gm.rows + sc_frag_row(mt, r)];
                sc_merge(*sc, st, b, o);
            }
            row_state_merge(st, o);
        }
        if (store) partial_store(p, idx, st);
        if constexpr (kSC) {
            // the read-out part of row R sits in the lanes of its fragment
            // positions: each stores its values under row R's slot index
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int R = sc_frag_row(mt, 2 * h);
                    const unsigned long long iR = __shfl_sync(0xFFFFFFFFu,
                                                              static_cast<unsigned long long>(idx), R);
                    const int sR = __shfl_sync(0xFFFFFFFFu, store ? 1 : 0, R);
                    if (sR) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            *reinterpret_cast<float2 *>(sm.part + iR * kScDim + sc_frag_col(j, 0)) =
                                make_float2(sc->c[mt][j][2 * h], sc->c[mt][j][2 * h + 1]);
                    }
                }
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(gm.done);
}

DG_DEVICE void group_merge_store(RowState &st, int cg, int rix, uint32_t k,
                                 const GroupMerge &gm, const Partials &p, size_t idx, bool store,
                                 WsHeader *ws)
{
    group_merge_store_t<false>(st, cg, rix, k, gm, p, idx, store, ws, nullptr, ScMerge{});
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
