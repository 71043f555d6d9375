// dg_attn_pair.cu -- bidirectional canvas attention over [KV cache ; canvas]
// on 2-CTA clusters that issue 2-SM UMMAs (tcgen05 cta_group::2).
//
// "DiffusionGemma Lab", section 2 item 6, and "Parallel Denoising From an
// Autoregressive Checkpoint", section "Finding": every canvas query attends
// to every cached key and every canvas key, with no mask.
//
// The two CTAs of a cluster own two consecutive 128-row query tiles (GQA
// folded: row = position * G + head in group) of one kv head, batch entry and
// key split, and share every key tile of 128 keys: CTA r stages keys
// [64 r, 64 r + 64) of the K tile and dims [r D/2, (r + 1) D/2) of the V tile,
// and the even CTA issues the UMMAs over both CTAs' halves:
//   S = Q K^T   256 x 128 x 16 per k step (each CTA gets its 128 rows x 128
//               keys in its own TMEM);
//   O += P V    256 x D x 16 per 16 keys (each CTA's O: its rows x all D).
// Per SM this halves the shared memory written by TMA and read by the tensor
// core per key compared with one CTA per query tile, and every UMMA has
// N >= 128.  Q is a TMEM operand for D = 128 and a shared-memory one for
// D = 256 (TMEM holds O and the two S buffers there); P (bf16) overwrites the
// S buffer it came from and is the TMEM A operand of O += P V.
//
//   warp 0      Q (D = 256) then K halves into a ring; both CTAs' copies
//               complete on the even CTA's barriers;
//   warp 6      V halves into a ring, the same way;
//   warp 1      TMEM allocation (both CTAs, collectively); UMMA issue (even
//               CTA): S(0), S(1), PV(0), S(2), PV(1), ...; the commits are
//               multicast to both CTAs;
//   warps 2-5   softmax, one query row per thread, as in dg_attn.cu; the
//               arrivals that release a P or Q go to the even CTA's barriers.
#include "dg_kernels.h"

namespace dg {

template <int D>
struct PairGeom {
    static constexpr int BKV = 128;               // keys per tile of the pair
    static constexpr int HK = BKV / 2;            // keys this CTA stages
    static constexpr int NA = D / 64;             // 64-dim atoms of a key row
    static constexpr int NAV = NA / 2;            // 64-dim atoms of this CTA's V half
    static constexpr int KAtom = HK * 128;        // 64 keys x 64 dims
    static constexpr int KBytes = NA * KAtom;
    static constexpr int VAtom = BKV * 128;       // 128 keys x 64 dims
    static constexpr int VBytes = NAV * VAtom;
    static constexpr bool QInTmem = (D == 128);
    static constexpr int QBytes = QInTmem ? 0 : 128 * D * 2;
    static constexpr int NK = QInTmem ? 6 : 3;
    static constexpr int NV = QInTmem ? 5 : 2;
    static constexpr int OffQ = 0;
    static constexpr int OffK = QBytes;
    static constexpr int OffV = OffK + NK * KBytes;
    static constexpr int OffBar = OffV + NV * VBytes;
    static constexpr int Smem = OffBar + 256 + 1024;
    static constexpr int ColO = 0;                // O: [0, D)
    static constexpr int ColS = D;                // S buffers: [D, D + 2 BKV)
    static constexpr int ColQ = D + 2 * BKV;      // Q (D = 128 only): D / 2 columns
    static_assert(ColS + 2 * BKV <= 512, "TMEM columns");
    static_assert(!QInTmem || ColQ + D / 2 <= 512, "TMEM columns");
    static_assert(2 * (NK + NV) * 8 + 8 * 8 + 4 <= 256, "barrier area");
    static_assert(Smem <= 232448, "shared memory");
};

int attn_pair_smem_bytes(int D)
{
    return D == 128 ? PairGeom<128>::Smem : PairGeom<256>::Smem;
}

template <int D, int NS, int BYTES>
__device__ __forceinline__ void pair_ring_producer(uint8_t *ring, uint64_t *full, uint64_t *empty,
                                                   uint32_t lead_full, int r,
                                                   const CUtensorMap *map_p,
                                                   const CUtensorMap *map_c, const AttnArgs &a,
                                                   int j0, int nt, int g, int b, bool is_v,
                                                   int where)
{
    using Gm = PairGeom<D>;
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
        // the even CTA expects the bytes of both CTAs' halves
        if (r == 0) mbar_arrive_expect_tx(&full[s], 2 * BYTES);
        const uint32_t fb = lead_full + static_cast<uint32_t>(s * 8);
        uint8_t *dst = ring + s * BYTES;
        if (is_v) {
            for (int i = 0; i < Gm::NAV; ++i)
                tma_load_4d_pair(dst + i * Gm::VAtom, m, fb, (r * Gm::NAV + i) * 64, g, row0, b, pol);
        } else {
            for (int at = 0; at < Gm::NA; ++at)
                tma_load_4d_pair(dst + at * Gm::KAtom, m, fb, at * 64, g, row0 + r * Gm::HK, b, pol);
        }
        armed |= 1u << s;
        armed_par = (armed_par & ~(1u << s)) | ((use & 1u) << s);
    }
    // the even CTA: every copy of both CTAs has landed before the closing
    // cluster barrier lets either CTA leave
    if (r == 0)
        for (int s = 0; s < NS; ++s)
            if (armed >> s & 1u) mbar_wait(&full[s], armed_par >> s & 1u, a.ws, where + 1);
}

template <int D>
__device__ __forceinline__ void attn_pair_body(const CUtensorMap *map_q, const CUtensorMap *map_kp,
                                               const CUtensorMap *map_vp, const CUtensorMap *map_kc,
                                               const CUtensorMap *map_vc, const AttnArgs &a)
{
    using Gm = PairGeom<D>;
    constexpr int BKV = Gm::BKV;
    constexpr int NK = Gm::NK, NV = Gm::NV;
    // inputs may come from the previous kernel of the stream
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Gm::OffBar);
    uint64_t *k_full = bars;                 // [NK]  used in the even CTA
    uint64_t *k_empty = k_full + NK;         // [NK]
    uint64_t *v_full = k_empty + NK;         // [NV]  used in the even CTA
    uint64_t *v_empty = v_full + NV;         // [NV]
    uint64_t *s_full = v_empty + NV;         // [2]
    uint64_t *pv_done = s_full + 2;          // [2]
    uint64_t *p_full = pv_done + 2;          // [2]   used in the even CTA
    uint64_t *q_ready = p_full + 2;          //       used in the even CTA
    uint64_t *o_full = q_ready + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(o_full + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = static_cast<int>(cluster_ctarank());
    const int mt = blockIdx.x;                   // this CTA's query tile
    const int bg = blockIdx.y;
    const int b = bg / a.Hkv, g = bg % a.Hkv;
    const int split = blockIdx.z;
    const int nkt = a.nkt_p + a.nkt_c;
    const int j0 = split * a.tiles_per_split;
    const int j1 = min(nkt, j0 + a.tiles_per_split);
    const int nt = j1 - j0;

    // softmax warps (2-5): one query row per thread; D = 128 fetches its Q row
    // now, so the loads overlap the set-up
    const int q = warp & 3;
    const int rr = q * 32 + lane;
    const int frow = mt * 128 + rr;
    const int i = frow / a.G, hj = frow % a.G;
    const bool live = i < a.L;
    const size_t flat =
        (static_cast<size_t>(b) * a.L + i) * a.Hq + static_cast<size_t>(g) * a.G + hj;
    uint4 qv[Gm::QInTmem ? D / 8 : 1];
    if (Gm::QInTmem && warp >= 2 && warp < 6) {
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
            mbar_init(&p_full[s], 8);            // 4 softmax warps of each CTA
        }
        mbar_init(q_ready, Gm::QInTmem ? 8 : 1);
        mbar_init(o_full, 1);
        fence_barrier_init();
        if (!Gm::QInTmem) tma_prefetch_desc(map_q);
        tma_prefetch_desc(map_kc);
        tma_prefetch_desc(map_vc);
        if (a.P > 0) {
            tma_prefetch_desc(map_kp);
            tma_prefetch_desc(map_vp);
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // both CTAs' barriers exist before either signals the other
    cluster_sync_all();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lead = mapa_shared(smem_u32(bars), 0);   // the even CTA's barrier area
    auto lead_of = [&](const uint64_t *bar) -> uint32_t {
        return lead + static_cast<uint32_t>(reinterpret_cast<const uint8_t *>(bar) -
                                            reinterpret_cast<const uint8_t *>(bars));
    };

    if (warp == 0) {
        // -------------------------------------------------------------- Q (D = 256), K
        if (lane == 0) {
            if (!Gm::QInTmem) {
                if (r == 0) mbar_arrive_expect_tx(q_ready, 2 * Gm::QBytes);
                const int pos0 = mt * (128 / a.G);
                // Q map: {dim, head-in-group, group, pos, batch}
                for (int at = 0; at < Gm::NA; ++at)
                    tma_load_5d_pair(smem + Gm::OffQ + at * 128 * 128, map_q, lead_of(q_ready),
                                     at * 64, 0, g, pos0, b, policy_evict_first());
            }
            pair_ring_producer<D, NK, Gm::KBytes>(smem + Gm::OffK, k_full, k_empty,
                                                  lead_of(k_full), r, map_kp, map_kc, a, j0, nt,
                                                  g, b, false, 231);
            if (!Gm::QInTmem && r == 0) mbar_wait(q_ready, 0, a.ws, 233);
        }
    } else if (warp == 6) {
        // -------------------------------------------------------------- V
        if (lane == 0)
            pair_ring_producer<D, NV, Gm::VBytes>(smem + Gm::OffV, v_full, v_empty,
                                                  lead_of(v_full), r, map_vp, map_vc, a, j0, nt,
                                                  g, b, true, 234);
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMA (even CTA)
        if (lane == 0 && r == 0) {
            const uint32_t idesc_s = make_idesc_bf16(256, BKV, 0);
            const uint32_t idesc_o = make_idesc_bf16(256, D, 1);
            const uint32_t sq = smem_u32(smem + Gm::OffQ);
            const uint32_t sk0 = smem_u32(smem + Gm::OffK);
            const uint32_t sv0 = smem_u32(smem + Gm::OffV);
            bool ok = mbar_wait_cluster(q_ready, 0, a.ws, 241);
            tc_fence_after();
            auto issue_s = [&](int it) -> bool {
                const int s = it % NK;
                if (!mbar_wait(&k_full[s], static_cast<uint32_t>((it / NK) & 1), a.ws, 242))
                    return false;
                tc_fence_after();
                const uint32_t sk = sk0 + s * Gm::KBytes;
                const uint32_t d = tmem + Gm::ColS + (it & 1) * BKV;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    // B = K half: K-major, 64-dim atoms KAtom apart, +32 B per 16 dims
                    const uint64_t bdesc =
                        make_sdesc_sw128(sk + (kk >> 2) * Gm::KAtom + (kk & 3) * 32, 16, 1024);
                    if (Gm::QInTmem) {
                        umma_bf16_pair_ts(d, tmem + Gm::ColQ + kk * 8, bdesc, idesc_s, kk != 0);
                    } else {
                        // A = Q: K-major, 64-dim atoms of 128 rows x 128 B
                        const uint64_t adesc = make_sdesc_sw128(
                            sq + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024);
                        umma_bf16_pair(d, adesc, bdesc, idesc_s, kk != 0);
                    }
                }
                umma_commit_pair(&k_empty[s], 0x3);
                umma_commit_pair(&s_full[it & 1], 0x3);
                return true;
            };
            auto issue_pv = [&](int jt) -> bool {
                // both CTAs' softmax warps have written P(jt)
                if (!mbar_wait_cluster(&p_full[jt & 1], static_cast<uint32_t>((jt >> 1) & 1), a.ws,
                                       243))
                    return false;
                const int s = jt % NV;
                if (!mbar_wait(&v_full[s], static_cast<uint32_t>((jt / NV) & 1), a.ws, 244))
                    return false;
                tc_fence_after();
                const uint32_t sv = sv0 + s * Gm::VBytes;
                const uint32_t pa = tmem + Gm::ColS + (jt & 1) * BKV;
#pragma unroll
                for (int kk = 0; kk < BKV / 16; ++kk) {
                    // B = V half: MN-major, 64-dim atoms VAtom apart, 8-key groups 1 KB apart
                    const uint64_t bdesc = make_sdesc_sw128(sv + kk * 2048, Gm::VAtom, 1024);
                    umma_bf16_pair_ts(tmem + Gm::ColO, pa + kk * 8, bdesc, idesc_o, (jt | kk) != 0);
                }
                umma_commit_pair(&v_empty[s], 0x3);
                umma_commit_pair(&pv_done[jt & 1], 0x3);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int it = 1; it < nt && ok; ++it) {
                // S(it) overwrites the buffer of P(it - 2), whose PV was issued before
                ok = issue_s(it) && issue_pv(it - 1);
            }
            if (ok) ok = issue_pv(nt - 1);
            umma_commit_pair(o_full, 0x3);
            mbar_wait(o_full, 0, a.ws, 245);
        }
    } else if (warp >= 2 && warp < 6) {
        // -------------------------------------------------------------- softmax
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        if (Gm::QInTmem) {
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
            if (lane == 0) mbar_arrive_cluster_relaxed(lead_of(q_ready));
        }
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int it = 0; it < nt; ++it) {
            const int sb = it & 1;
            ok = mbar_wait(&s_full[sb], static_cast<uint32_t>((it >> 1) & 1), a.ws, 251);
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
                // O holds the PVs up to tile it - 1: wait for the last one
                ok = mbar_wait(&pv_done[(it - 1) & 1], static_cast<uint32_t>(((it - 1) >> 1) & 1),
                               a.ws, 252);
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
            if (lane == 0) mbar_arrive_cluster_relaxed(lead_of(&p_full[sb]));
        }
        // -------------------------------------------------------------- epilogue
        if (ok) ok = mbar_wait(o_full, 0, a.ws, 253);
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
            if (bad) report_error(a.ws, DG_ERR_DEVICE, 815);
        }
    }
    tc_fence_before();
    __syncthreads();
    // no CTA releases its TMEM or leaves while the pair's UMMAs, copies,
    // commits or remote arrivals may still reach it
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttnThreads, 1)
    attn_pair_kernel_d128(const __grid_constant__ CUtensorMap map_q,
                          const __grid_constant__ CUtensorMap map_kp,
                          const __grid_constant__ CUtensorMap map_vp,
                          const __grid_constant__ CUtensorMap map_kc,
                          const __grid_constant__ CUtensorMap map_vc, AttnArgs a)
{
    attn_pair_body<128>(&map_q, &map_kp, &map_vp, &map_kc, &map_vc, a);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttnThreads, 1)
    attn_pair_kernel_d256(const __grid_constant__ CUtensorMap map_q,
                          const __grid_constant__ CUtensorMap map_kp,
                          const __grid_constant__ CUtensorMap map_vp,
                          const __grid_constant__ CUtensorMap map_kc,
                          const __grid_constant__ CUtensorMap map_vc, AttnArgs a)
{
    attn_pair_body<256>(&map_q, &map_kp, &map_vp, &map_kc, &map_vc, a);
}

}  // namespace dg
