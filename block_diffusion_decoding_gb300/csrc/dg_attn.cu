// dg_attn.cu -- bidirectional canvas attention over [KV cache ; canvas].
//
// "DiffusionGemma Lab", section 2 item 6, and "Parallel Denoising From an
// Autoregressive Checkpoint", section "Finding": the decoder attends across
// the whole canvas with no mask and cross-attends to the causal encoder's
// append-only KV cache; the same page notes that this bidirectional
// attention over 256 tokens cannot use single-token decode kernels.
//
// GQA folding: the G = Hq / Hkv query heads that share kv head g are folded
// into the row dimension, so one 128-row tile holds 128 / G canvas positions
// x G heads (row = position * G + head in group) and every K/V tile is used
// by all of them.
//
// CTA (224 threads) = one 128-row query tile x one kv head x one batch
// entry x one split of the key tiles.  Operands that the tensor core reads
// from the A side live in tensor memory, so shared memory holds only the
// K/V rings (7 tiles of 32 KB) and the UMMAs read one operand from it:
//   TMEM        O [128 x D] fp32 | S0, S1 [128 x BKV] fp32 | Q [128 x D] bf16
//               (the bf16 P of a tile overwrites the first BKV/2 columns of
//               the S buffer it was computed from);
//   warp 0      TMA: K tiles (prefix tiles, then canvas tiles) into a
//               4-stage ring, released as soon as S = Q K^T has read them;
//   warp 6      TMA: V tiles into a 3-stage ring, released after O += P V;
//   warp 1      TMEM allocator + UMMA issuer, order S(0), S(1), PV(0), S(2),
//               PV(1), ...: S of tile j+1 is computed while the softmax
//               works on tile j, PV of tile j follows as soon as P(j) is in;
//   warps 2-5   load the Q rows into TMEM, then softmax, one query row per
//               thread: read S, keep a reference max that only moves when a
//               tile's max exceeds it by more than 2^8 (then O is rescaled in
//               TMEM, after the PV of the previous tile), write P as bf16
//               pairs into TMEM, and at the end normalise O (or write
//               unnormalised O, max and sum per split).
#include "dg_kernels.h"

namespace dg {

template <int D>
struct AttnGeom {
    static constexpr int BKV = (D == 128) ? 128 : 64;      // keys per tile
    static constexpr int NA = D / 64;                      // 64-dim atoms
    static constexpr int KVBytes = BKV * D * 2;            // 32 KB
    static constexpr int KVAtomBytes = BKV * 128;          // one 64-dim atom
    static constexpr int NK = 4;                           // K ring stages
    static constexpr int NV = 3;                           // V ring stages
    static constexpr int OffK = 0;
    static constexpr int OffV = OffK + NK * KVBytes;
    static constexpr int OffBar = OffV + NV * KVBytes;
    static constexpr int Smem = OffBar + 256 + 1024;
    static constexpr int ColO = 0;                         // O: [0, D)
    static constexpr int ColS = D;                         // S buffers: [D, D + 2 BKV)
    static constexpr int ColQ = D + 2 * BKV;               // Q: D / 2 columns
    static_assert(ColQ + D / 2 <= 512, "TMEM columns");
    static_assert(Smem <= 232448, "shared memory");
};

int attn_smem_bytes(int D)
{
    return D == 128 ? AttnGeom<128>::Smem : AttnGeom<256>::Smem;
}

// Loads kv tiles [j0, j1) of one ring (K or V) with TMA.  Returns after every
// copy it started has landed.
template <int D, int NS>
__device__ __forceinline__ void attn_ring_producer(uint8_t *ring, uint64_t *full, uint64_t *empty,
                                                   const CUtensorMap *map_p,
                                                   const CUtensorMap *map_c, const AttnArgs &a,
                                                   int j0, int nt, int g, int b, int where)
{
    using Gm = AttnGeom<D>;
    const uint64_t pol = policy_evict_first();
    uint32_t armed = 0, armed_par = 0;
    for (int it = 0; it < nt; ++it) {
        const int s = it % NS;
        const uint32_t use = static_cast<uint32_t>(it / NS);
        if (!mbar_wait(&empty[s], (use & 1u) ^ 1u, a.ws, where)) break;
        const int j = j0 + it;
        const bool pre = j < a.nkt_p;
        const CUtensorMap *m = pre ? map_p : map_c;
        const int row0 = (pre ? j : j - a.nkt_p) * Gm::BKV;
        mbar_arrive_expect_tx(&full[s], Gm::KVBytes);
        for (int at = 0; at < Gm::NA; ++at)
            tma_load_4d(ring + s * Gm::KVBytes + at * Gm::KVAtomBytes, m, &full[s], at * 64, g,
                        row0, b, pol);
        armed |= 1u << s;
        armed_par = (armed_par & ~(1u << s)) | ((use & 1u) << s);
    }
    for (int s = 0; s < NS; ++s)
        if (armed >> s & 1u) mbar_wait(&full[s], armed_par >> s & 1u, a.ws, where + 1);
}

template <int D>
__device__ __forceinline__ void attn_body(const CUtensorMap *map_kp, const CUtensorMap *map_vp,
                                          const CUtensorMap *map_kc, const CUtensorMap *map_vc,
                                          const AttnArgs &a)
{
    using Gm = AttnGeom<D>;
    constexpr int BKV = Gm::BKV;
    constexpr int NK = Gm::NK, NV = Gm::NV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Gm::OffBar);
    uint64_t *k_full = bars;                 // [NK]
    uint64_t *k_empty = k_full + NK;         // [NK]
    uint64_t *v_full = k_empty + NK;         // [NV]
    uint64_t *v_empty = v_full + NV;         // [NV]
    uint64_t *s_full = v_empty + NV;         // [2]
    uint64_t *pv_done = s_full + 2;          // [2]
    uint64_t *p_full = pv_done + 2;          // [2]
    uint64_t *q_ready = p_full + 2;
    uint64_t *o_full = q_ready + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(o_full + 1);

    // inputs may come from the previous kernel of the stream
    griddep_wait();
    griddep_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = blockIdx.x;
    const int bg = blockIdx.y;
    const int b = bg / a.Hkv, g = bg % a.Hkv;
    const int split = blockIdx.z;
    const int nkt = a.nkt_p + a.nkt_c;
    const int j0 = split * a.tiles_per_split;
    const int j1 = min(nkt, j0 + a.tiles_per_split);
    const int nt = j1 - j0;

    // softmax warps (2-5): thread = one query row of the tile; its Q row is
    // fetched now so that the loads overlap the set-up below
    const int q = warp & 3;                  // TMEM lane quadrant of the warp
    const int r = q * 32 + lane;             // row within the 128-row tile
    const int frow = mt * 128 + r;           // folded row = position * G + head
    const int i = frow / a.G, hj = frow % a.G;
    const bool live = i < a.L;
    const size_t flat =
        (static_cast<size_t>(b) * a.L + i) * a.Hq + static_cast<size_t>(g) * a.G + hj;
    uint4 qv[D / 8];
    if (warp >= 2 && warp < 6) {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.q + flat * D);
#pragma unroll
        for (int k = 0; k < D / 8; ++k) qv[k] = live ? __ldg(src + k) : make_uint4(0, 0, 0, 0);
    }

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < NK; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&s_full[s], 1);
            mbar_init(&pv_done[s], 1);
            mbar_init(&p_full[s], 4);
        }
        mbar_init(q_ready, 4);
        mbar_init(o_full, 1);
        fence_barrier_init();
        tma_prefetch_desc(map_kc);
        tma_prefetch_desc(map_vc);
        if (a.P > 0) {
            tma_prefetch_desc(map_kp);
            tma_prefetch_desc(map_vp);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // -------------------------------------------------------------- K loads
        if (lane == 0)
            attn_ring_producer<D, NK>(smem + Gm::OffK, k_full, k_empty, map_kp, map_kc, a, j0, nt,
                                      g, b, 201);
    } else if (warp == 6) {
        // -------------------------------------------------------------- V loads
        if (lane == 0)
            attn_ring_producer<D, NV>(smem + Gm::OffV, v_full, v_empty, map_vp, map_vc, a, j0, nt,
                                      g, b, 203);
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idesc_s = make_idesc_bf16(128, BKV, 0);
            const uint32_t idesc_o = make_idesc_bf16(128, D, 1);
            const uint32_t sk0 = smem_u32(smem + Gm::OffK);
            const uint32_t sv0 = smem_u32(smem + Gm::OffV);
            bool ok = mbar_wait(q_ready, 0, a.ws, 211);
            tc_fence_after();
            auto issue_s = [&](int it) -> bool {
                const int s = it % NK;
                if (!mbar_wait(&k_full[s], static_cast<uint32_t>((it / NK) & 1), a.ws, 212))
                    return false;
                tc_fence_after();
                const uint32_t sk = sk0 + s * Gm::KVBytes;
                const uint32_t d = tmem + Gm::ColS + (it & 1) * BKV;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // B = K: K-major, 64-dim atoms KVAtomBytes apart, +32 B per 16 dims
                    const uint64_t bdesc =
                        make_sdesc_sw128(sk + (kk >> 2) * Gm::KVAtomBytes + (kk & 3) * 32, 16, 1024);
                    umma_bf16_ts(d, tmem + Gm::ColQ + kk * 8, bdesc, idesc_s, kk != 0);
                }
                umma_commit(&k_empty[s]);
                umma_commit(&s_full[it & 1]);
                return true;
            };
            auto issue_pv = [&](int jt) -> bool {
                const int s = jt % NV;
                // one barrier per S buffer: the softmax cannot run two tiles ahead of a wait
                if (!mbar_wait(&p_full[jt & 1], static_cast<uint32_t>((jt >> 1) & 1), a.ws, 213))
                    return false;
                if (!mbar_wait(&v_full[s], static_cast<uint32_t>((jt / NV) & 1), a.ws, 214))
                    return false;
                tc_fence_after();
                const uint32_t sv = sv0 + s * Gm::KVBytes;
                const uint32_t pa = tmem + Gm::ColS + (jt & 1) * BKV;
#pragma unroll
                for (int kk = 0; kk < BKV / 16; ++kk) {
                    // B = V: MN-major, 64-dim atoms KVAtomBytes apart, 8-key groups 1 KB apart
                    const uint64_t bdesc = make_sdesc_sw128(sv + kk * 2048, Gm::KVAtomBytes, 1024);
                    umma_bf16_ts(tmem + Gm::ColO, pa + kk * 8, bdesc, idesc_o, (jt | kk) != 0);
                }
                umma_commit(&v_empty[s]);
                umma_commit(&pv_done[jt & 1]);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int it = 1; it < nt && ok; ++it) {
                // S(it) overwrites the buffer of P(it - 2), whose PV was issued before
                ok = issue_s(it) && issue_pv(it - 1);
            }
            if (ok) ok = issue_pv(nt - 1);
            umma_commit(o_full);
            mbar_wait(o_full, 0, a.ws, 215);
        }
    } else {
        // -------------------------------------------------------------- softmax
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        // ---- Q row into TMEM (rows past the canvas are zero)
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
            uint32_t w[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint4 v = qv[(c0 >> 2) + k];
                w[4 * k] = v.x;
                w[4 * k + 1] = v.y;
                w[4 * k + 2] = v.z;
                w[4 * k + 3] = v.w;
            }
            tmem_st32(tmem + lane_off + Gm::ColQ + c0, w);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_ready);
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int it = 0; it < nt; ++it) {
            const int sb = it & 1;
            ok = mbar_wait(&s_full[sb], static_cast<uint32_t>((it >> 1) & 1), a.ws, 221);
            if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
            tc_fence_after();
            const uint32_t ts = tmem + lane_off + Gm::ColS + sb * BKV;
            uint32_t sr[BKV];
#pragma unroll
            for (int c0 = 0; c0 < BKV; c0 += 32)
                tmem_ld32_nowait(ts + c0, *reinterpret_cast<uint32_t(*)[32]>(&sr[c0]));
            tmem_wait_ld();

            const int j = j0 + it;
            const bool pre = j < a.nkt_p;
            const int valid = pre ? min(BKV, a.P - j * BKV) : min(BKV, a.L - (j - a.nkt_p) * BKV);
            if (valid < BKV) {   // ragged tile: keys past the end weigh nothing
#pragma unroll
                for (int c = 0; c < BKV; ++c)
                    if (c >= valid) sr[c] = __float_as_uint(-INFINITY);
            }
            if (a.causal && !pre) {
                // cache-append forward: canvas keys after this row's position
                // weigh nothing (column c is canvas key (j - nkt_p) BKV + c)
                const int last = i - (j - a.nkt_p) * BKV;   // last visible column
                if (__any_sync(0xFFFFFFFFu, last < BKV - 1)) {
#pragma unroll
                    for (int c = 0; c < BKV; ++c)
                        if (c > last) sr[c] = __float_as_uint(-INFINITY);
                }
            }
            // the scale is positive, so the scaled maximum is the maximum scaled
            float rmax = -INFINITY;
#pragma unroll
            for (int c = 0; c < BKV; c += 2)
                rmax = max3(rmax, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            const float tmax = rmax * a.scale_log2;
            float factor = 1.f;
            bool rescale = false;
            if (m_ref == -INFINITY) {
                m_ref = tmax;
            } else if (tmax > m_ref + 8.f) {
                factor = fast_exp2(m_ref - tmax);
                l *= factor;
                m_ref = tmax;
                rescale = true;
            }
            // p = 2^(s scale - m), two columns per paired instruction; the row
            // sum is kept in fp32 (the MMA sees p rounded to bf16)
            const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
            // a row with no visible key yet (causal, later key split) keeps
            // m_ref = -inf and weighs every column 0
            const float mexp = (m_ref == -INFINITY) ? 0.f : m_ref;
            const float2 nm2 = make_float2(-mexp, -mexp);
            float2 acc = make_float2(0.f, 0.f);
            uint32_t pk[BKV / 2];
#pragma unroll
            for (int c = 0; c < BKV; c += 2) {
                const float2 d2 = fma2(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])),
                                       sc2, nm2);
                const float2 p2 = make_float2(fast_exp2(d2.x), fast_exp2(d2.y));
                acc = add2(acc, p2);
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(p2.x, p2.y);
                pk[c >> 1] = *reinterpret_cast<const uint32_t *>(&h2);
            }
            l += acc.x + acc.y;
            if (__any_sync(0xFFFFFFFFu, rescale)) {
                // O holds the PVs up to tile it - 1: wait for the last one (the
                // completed S(it) already implies every earlier PV is done)
                ok = mbar_wait(&pv_done[(it - 1) & 1], static_cast<uint32_t>(((it - 1) >> 1) & 1),
                               a.ws, 222);
                if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t o[32];
                    const uint32_t ta = tmem + lane_off + Gm::ColO + c0;
                    tmem_ld32_nowait(ta, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        o[k] = __float_as_uint(__uint_as_float(o[k]) * factor);
                    tmem_st32(ta, o);
                }
            }
            // P(it) as bf16 pairs over the first BKV / 2 columns of its S buffer
#pragma unroll
            for (int c0 = 0; c0 < BKV / 2; c0 += 32)
                tmem_st32(ts + c0, *reinterpret_cast<const uint32_t(*)[32]>(&pk[c0]));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[sb]);
        }
        // -------------------------------------------------------------- epilogue
        if (ok) ok = mbar_wait(o_full, 0, a.ws, 223);
        if (__all_sync(0xFFFFFFFFu, ok)) {
            tc_fence_after();
            const float inv_l = (l > 0.f) ? 1.f / l : 0.f;   // no visible key: zero row
            const size_t nrows = static_cast<size_t>(a.B) * a.L * a.Hq;
            // device-side checks: a finite softmax sum and output row
            bool bad = a.checks && live && !isfinite(l);
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld32_nowait(tmem + lane_off + Gm::ColO + c0, o);
                tmem_wait_ld();
                if (!live) continue;
                if (a.checks) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) bad |= !isfinite(__uint_as_float(o[k]));
                }
                // the output row, or (several key splits) this split's
                // normalised partial row, as bf16
                uint16_t *row_out = (a.nsplit == 1)
                                        ? a.out + flat * D
                                        : a.part_o + (static_cast<size_t>(split) * nrows + flat) * D;
                uint4 *dst = reinterpret_cast<uint4 *>(row_out + c0);
#pragma unroll
                for (int k = 0; k < 32; k += 8) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const __nv_bfloat162 h2 = __floats2bfloat162_rn(
                            __uint_as_float(o[k + 2 * e]) * inv_l,
                            __uint_as_float(o[k + 2 * e + 1]) * inv_l);
                        w4[e] = *reinterpret_cast<const uint32_t *>(&h2);
                    }
                    dst[k >> 3] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
            }
            if (live && a.nsplit > 1) {
                float2 *ml = reinterpret_cast<float2 *>(a.part_ml);
                ml[static_cast<size_t>(split) * nrows + flat] = make_float2(m_ref, l);
            }
            if (bad) report_error(a.ws, DG_ERR_DEVICE, 813);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel_d128(const __grid_constant__ CUtensorMap map_kp,
                     const __grid_constant__ CUtensorMap map_vp,
                     const __grid_constant__ CUtensorMap map_kc,
                     const __grid_constant__ CUtensorMap map_vc, AttnArgs a)
{
    attn_body<128>(&map_kp, &map_vp, &map_kc, &map_vc, a);
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel_d256(const __grid_constant__ CUtensorMap map_kp,
                     const __grid_constant__ CUtensorMap map_vp,
                     const __grid_constant__ CUtensorMap map_kc,
                     const __grid_constant__ CUtensorMap map_vc, AttnArgs a)
{
    attn_body<256>(&map_kp, &map_vp, &map_kc, &map_vc, a);
}

// Merge the key splits: one warp per query row, lanes over the head dim.
// Split z left its row normalised by its own sum l_z, with its reference max
// m_z (base 2); the row is sum_z 2^(m_z - M) l_z O_z / sum_z 2^(m_z - M) l_z,
// merged online four splits at a time (all their loads in flight together;
// the running sums are rescaled when a later split raises the maximum).
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgs a)
{
    griddep_wait();
    griddep_launch_dependents();
    const size_t nrows = static_cast<size_t>(a.B) * a.L * a.Hq;
    const size_t row = static_cast<size_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= nrows) return;
    const float2 *ml = reinterpret_cast<const float2 *>(a.part_ml);
    const int per = a.D / 32;   // 4 or 8 consecutive dims per lane
    float M = -INFINITY, den = 0.f;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int z0 = 0; z0 < a.nsplit; z0 += 4) {
        float2 v[4];
        uint32_t pw[4][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int z = z0 + k;
            if (z < a.nsplit) {
                v[k] = ml[z * nrows + row];
                const uint16_t *po = a.part_o + (z * nrows + row) * a.D + lane * per;
                if (per == 8) {
                    const uint4 q4 = *reinterpret_cast<const uint4 *>(po);
                    pw[k][0] = q4.x; pw[k][1] = q4.y; pw[k][2] = q4.z; pw[k][3] = q4.w;
                } else {
                    const uint2 q2 = *reinterpret_cast<const uint2 *>(po);
                    pw[k][0] = q2.x; pw[k][1] = q2.y; pw[k][2] = 0u; pw[k][3] = 0u;
                }
            } else {
                v[k] = make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int e = 0; e < 4; ++e) pw[k][e] = 0u;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            // a split with no visible key for this row has l = 0 (and a zero row)
            if (!(v[k].y > 0.f)) continue;
            if (v[k].x > M) {
                const float f = fast_exp2(M - v[k].x);   // 0 while M = -inf
                den *= f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] *= f;
                M = v[k].x;
            }
            const float wz = fast_exp2(v[k].x - M) * v[k].y;
            den += wz;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (2 * e < per) {
                    const float2 f2 =
                        __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pw[k][e]));
                    acc[2 * e] = fmaf(wz, f2.x, acc[2 * e]);
                    acc[2 * e + 1] = fmaf(wz, f2.y, acc[2 * e + 1]);
                }
            }
        }
    }
    const float inv = 1.f / den;
    if (a.checks) {
        // device-side checks: a positive finite sum over the splits, finite outputs
        bool bad = !(den > 0.f) || !isfinite(den);
#pragma unroll
        for (int e = 0; e < 8; ++e) bad |= !isfinite(acc[e]);
        if (bad) report_error(a.ws, DG_ERR_DEVICE, 811);
    }
    uint16_t *dst = a.out + row * a.D + lane * per;
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        if (e < per) {
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv);
            *reinterpret_cast<uint32_t *>(dst + e) = *reinterpret_cast<const uint32_t *>(&h2);
        }
    }
}

}  // namespace dg
