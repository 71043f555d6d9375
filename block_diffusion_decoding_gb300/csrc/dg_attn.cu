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
// x G heads and every K/V tile is used by all of them.  The 5-D TMA map of
// Q does the folding (box = 64 dims x G heads x 1 group x 128/G positions).
//
// CTA (192 threads) = one 128-row query tile x one kv head x one batch
// entry x one split of the key tiles:
//   warp 0     TMA: Q once, then K and V tiles (prefix tiles, then canvas
//              tiles) into a 2-stage ring, 128-byte swizzle;
//   warp 1     TMEM allocator + UMMA issuer: S = Q K^T (K-major B) into one
//              of two S buffers, and O += P V (V as MN-major B) into the O
//              accumulator, software-pipelined so that S of tile j+1 is
//              computed while the softmax works on tile j;
//   warps 2-5  softmax, one query row per thread: reads S from TMEM, keeps
//              a reference max that only moves when a tile's max exceeds it
//              by more than 2^8 (then O is rescaled in TMEM), writes P as
//              bf16 into shared memory in the UMMA A layout, and at the end
//              normalises O (or writes unnormalised O, max, sum per split).
#include "dg_kernels.h"

namespace dg {

template <int D>
struct AttnGeom {
    static constexpr int BKV = (D == 128) ? 128 : 64;      // keys per tile
    static constexpr int NA = D / 64;                      // 64-dim atoms
    static constexpr int QBytes = 128 * D * 2;
    static constexpr int KVBytes = BKV * D * 2;
    static constexpr int KVAtomBytes = BKV * 128;          // one 64-dim atom
    static constexpr int PBytes = 128 * BKV * 2;
    static constexpr int OffQ = 0;
    static constexpr int OffK = OffQ + QBytes;
    static constexpr int OffV = OffK + 2 * KVBytes;
    static constexpr int OffP = OffV + 2 * KVBytes;
    static constexpr int OffBar = OffP + PBytes;
    static constexpr int Smem = OffBar + 256 + 1024;
    static constexpr int ColS = 0;                         // S buffers: [0, 2 BKV)
    static constexpr int ColO = 2 * BKV;                   // O: [2 BKV, 2 BKV + D)
};

int attn_smem_bytes(int D)
{
    return D == 128 ? AttnGeom<128>::Smem : AttnGeom<256>::Smem;
}

template <int D>
__device__ __forceinline__ void attn_body(const CUtensorMap *map_q, const CUtensorMap *map_kp,
                                          const CUtensorMap *map_vp, const CUtensorMap *map_kc,
                                          const CUtensorMap *map_vc, const AttnArgs &a)
{
    using Gm = AttnGeom<D>;
    constexpr int BKV = Gm::BKV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Gm::OffBar);
    uint64_t *bar_q = bars + 0;
    uint64_t *k_full = bars + 1;     // [2]
    uint64_t *v_full = bars + 3;     // [2]
    uint64_t *kv_empty = bars + 5;   // [2]
    uint64_t *s_full = bars + 7;     // [2]
    uint64_t *s_empty = bars + 9;    // [2]
    uint64_t *p_full = bars + 11;
    uint64_t *pv_done = bars + 12;
    uint64_t *o_full = bars + 13;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 14);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = blockIdx.x;
    const int bg = blockIdx.y;
    const int b = bg / a.Hkv, g = bg % a.Hkv;
    const int split = blockIdx.z;
    const int nkt = a.nkt_p + a.nkt_c;
    const int j0 = split * a.tiles_per_split;
    const int j1 = min(nkt, j0 + a.tiles_per_split);
    const int nt = j1 - j0;

    if (warp == 0 && lane == 0) {
        mbar_init(bar_q, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&kv_empty[s], 1);
            mbar_init(&s_full[s], 1);
            mbar_init(&s_empty[s], 4);
        }
        mbar_init(p_full, 4);
        mbar_init(pv_done, 1);
        mbar_init(o_full, 1);
        fence_barrier_init();
        tma_prefetch_desc(map_q);
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
        // -------------------------------------------------------------- TMA
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            mbar_arrive_expect_tx(bar_q, Gm::QBytes);
            const int pos0 = mt * (128 / a.G);
            for (int at = 0; at < Gm::NA; ++at)   // Q map: {dim, head-in-group, group, pos, batch}
                tma_load_5d(smem + Gm::OffQ + at * 128 * 128, map_q, bar_q, at * 64, 0, g, pos0, b,
                            pol);
            uint32_t armed = 0, armed_par = 0;
            for (int it = 0; it < nt; ++it) {
                const int s = it & 1;
                const uint32_t use = static_cast<uint32_t>(it >> 1);
                if (!mbar_wait(&kv_empty[s], (use & 1u) ^ 1u, a.ws, 201)) break;
                const int j = j0 + it;
                const bool pre = j < a.nkt_p;
                const CUtensorMap *mk = pre ? map_kp : map_kc;
                const CUtensorMap *mv = pre ? map_vp : map_vc;
                const int row0 = (pre ? j : j - a.nkt_p) * BKV;
                mbar_arrive_expect_tx(&k_full[s], Gm::KVBytes);
                for (int at = 0; at < Gm::NA; ++at)
                    tma_load_4d(smem + Gm::OffK + s * Gm::KVBytes + at * Gm::KVAtomBytes, mk,
                                &k_full[s], at * 64, g, row0, b, pol);
                mbar_arrive_expect_tx(&v_full[s], Gm::KVBytes);
                for (int at = 0; at < Gm::NA; ++at)
                    tma_load_4d(smem + Gm::OffV + s * Gm::KVBytes + at * Gm::KVAtomBytes, mv,
                                &v_full[s], at * 64, g, row0, b, pol);
                armed |= 1u << s;
                armed_par = (armed_par & ~(1u << s)) | ((use & 1u) << s);
            }
            // every copy this thread started has landed before the CTA can exit
            mbar_wait(bar_q, 0, a.ws, 202);
            for (int s = 0; s < 2; ++s) {
                if (armed >> s & 1u) {
                    mbar_wait(&k_full[s], armed_par >> s & 1u, a.ws, 203);
                    mbar_wait(&v_full[s], armed_par >> s & 1u, a.ws, 204);
                }
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idesc_s = make_idesc_bf16(128, BKV, 0);
            const uint32_t idesc_o = make_idesc_bf16(128, D, 1);
            const uint32_t sq = smem_u32(smem + Gm::OffQ);
            const uint32_t sp = smem_u32(smem + Gm::OffP);
            bool ok = mbar_wait(bar_q, 0, a.ws, 211);
            auto issue_pv = [&](int jt) -> bool {
                const int s = jt & 1;
                if (!mbar_wait(p_full, static_cast<uint32_t>(jt & 1), a.ws, 212)) return false;
                if (!mbar_wait(&v_full[s], static_cast<uint32_t>((jt >> 1) & 1), a.ws, 213))
                    return false;
                tc_fence_after();
                const uint32_t sv = smem_u32(smem + Gm::OffV + s * Gm::KVBytes);
#pragma unroll
                for (int kk = 0; kk < BKV / 16; ++kk) {
                    // A = P: K-major, 64-key atoms of 128 rows x 128 B
                    const uint64_t adesc =
                        make_sdesc_sw128(sp + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024);
                    // B = V: MN-major, 64-dim atoms KVAtomBytes apart, 8-key groups 1 KB apart
                    const uint64_t bdesc = make_sdesc_sw128(sv + kk * 2048, Gm::KVAtomBytes, 1024);
                    umma_bf16(tmem + Gm::ColO, adesc, bdesc, idesc_o, (jt | kk) != 0);
                }
                umma_commit(&kv_empty[s]);
                umma_commit(pv_done);
                return true;
            };
            for (int it = 0; it < nt && ok; ++it) {
                const int s = it & 1;
                const uint32_t use = static_cast<uint32_t>(it >> 1);
                if (!mbar_wait(&k_full[s], use & 1u, a.ws, 214)) { ok = false; break; }
                if (!mbar_wait(&s_empty[s], (use & 1u) ^ 1u, a.ws, 215)) { ok = false; break; }
                tc_fence_after();
                const uint32_t sk = smem_u32(smem + Gm::OffK + s * Gm::KVBytes);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t adesc =
                        make_sdesc_sw128(sq + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024);
                    const uint64_t bdesc =
                        make_sdesc_sw128(sk + (kk >> 2) * Gm::KVAtomBytes + (kk & 3) * 32, 16, 1024);
                    umma_bf16(tmem + Gm::ColS + s * BKV, adesc, bdesc, idesc_s, kk != 0);
                }
                umma_commit(&s_full[s]);
                if (it >= 1 && !issue_pv(it - 1)) { ok = false; break; }
            }
            if (ok && nt >= 1) ok = issue_pv(nt - 1);
            umma_commit(o_full);
            mbar_wait(o_full, 0, a.ws, 216);
        }
    } else {
        // -------------------------------------------------------------- softmax
        const int q = warp & 3;                  // TMEM lane quadrant of this warp
        const int r = q * 32 + lane;             // row within the 128-row tile
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        uint8_t *sP = smem + Gm::OffP;
        for (int it = 0; it < nt; ++it) {
            const int s = it & 1;
            const uint32_t use = static_cast<uint32_t>(it >> 1);
            ok = mbar_wait(&s_full[s], use & 1u, a.ws, 221);
            if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
            tc_fence_after();
            uint32_t sr[BKV];
#pragma unroll
            for (int c0 = 0; c0 < BKV; c0 += 32)
                tmem_ld32_nowait(tmem + lane_off + Gm::ColS + s * BKV + c0,
                                 *reinterpret_cast<uint32_t(*)[32]>(&sr[c0]));
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[s]);

            const int j = j0 + it;
            const bool pre = j < a.nkt_p;
            const int valid = pre ? min(BKV, a.P - j * BKV) : min(BKV, a.L - (j - a.nkt_p) * BKV);
            float tmax = -INFINITY;
#pragma unroll
            for (int c = 0; c < BKV; ++c) {
                const float v = (c < valid) ? __uint_as_float(sr[c]) * a.scale_log2 : -INFINITY;
                sr[c] = __float_as_uint(v);
                tmax = fmaxf(tmax, v);
            }
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
            float psum = 0.f;
            uint32_t pk[BKV / 2];
#pragma unroll
            for (int c = 0; c < BKV; c += 2) {
                const float p0 = fast_exp2(__uint_as_float(sr[c]) - m_ref);
                const float p1 = fast_exp2(__uint_as_float(sr[c + 1]) - m_ref);
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
                // the row sum uses the bf16-rounded weights the MMA sees
                const float2 back = __bfloat1622float2(h2);
                psum += back.x + back.y;
                pk[c >> 1] = *reinterpret_cast<const uint32_t *>(&h2);
            }
            l += psum;
            if (it >= 1) {
                ok = mbar_wait(pv_done, static_cast<uint32_t>((it - 1) & 1), a.ws, 222);
                if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                tc_fence_after();
                if (__any_sync(0xFFFFFFFFu, rescale)) {
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
                    tmem_wait_st();
                }
            }
            // P row r, K-major 128B-swizzled: 64-key atoms of 128 rows x 128 B
#pragma unroll
            for (int at = 0; at < BKV / 64; ++at) {
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint32_t off = static_cast<uint32_t>(at * 128 * 128 + r * 128 +
                                                               ((ch ^ (r & 7)) << 4));
                    const int w0 = at * 32 + ch * 4;
                    *reinterpret_cast<uint4 *>(sP + off) =
                        make_uint4(pk[w0], pk[w0 + 1], pk[w0 + 2], pk[w0 + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        // -------------------------------------------------------------- epilogue
        if (ok) ok = mbar_wait(o_full, 0, a.ws, 223);
        if (__all_sync(0xFFFFFFFFu, ok)) {
            tc_fence_after();
            const int frow = mt * 128 + r;           // folded row = position * G + head
            const int i = frow / a.G, hj = frow % a.G;
            const bool live = i < a.L;
            const size_t flat =
                (static_cast<size_t>(b) * a.L + i) * a.Hq + static_cast<size_t>(g) * a.G + hj;
            const float inv_l = 1.f / l;
            const size_t nrows = static_cast<size_t>(a.B) * a.L * a.Hq;
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tmem_ld32_nowait(tmem + lane_off + Gm::ColO + c0, o);
                tmem_wait_ld();
                if (!live) continue;
                if (a.nsplit == 1) {
                    uint4 *dst = reinterpret_cast<uint4 *>(a.out + flat * D + c0);
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
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(
                        a.part_o + (static_cast<size_t>(split) * nrows + flat) * D + c0);
#pragma unroll
                    for (int k = 0; k < 32; k += 4)
                        dst[k >> 2] = make_float4(__uint_as_float(o[k]), __uint_as_float(o[k + 1]),
                                                  __uint_as_float(o[k + 2]),
                                                  __uint_as_float(o[k + 3]));
                }
            }
            if (live && a.nsplit > 1) {
                float2 *ml = reinterpret_cast<float2 *>(a.part_ml);
                ml[static_cast<size_t>(split) * nrows + flat] = make_float2(m_ref, l);
            }
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
    attn_kernel_d128(const __grid_constant__ CUtensorMap map_q,
                     const __grid_constant__ CUtensorMap map_kp,
                     const __grid_constant__ CUtensorMap map_vp,
                     const __grid_constant__ CUtensorMap map_kc,
                     const __grid_constant__ CUtensorMap map_vc, AttnArgs a)
{
    attn_body<128>(&map_q, &map_kp, &map_vp, &map_kc, &map_vc, a);
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_kernel_d256(const __grid_constant__ CUtensorMap map_q,
                     const __grid_constant__ CUtensorMap map_kp,
                     const __grid_constant__ CUtensorMap map_vp,
                     const __grid_constant__ CUtensorMap map_kc,
                     const __grid_constant__ CUtensorMap map_vc, AttnArgs a)
{
    attn_body<256>(&map_q, &map_kp, &map_vp, &map_kc, &map_vc, a);
}

// Merge the key splits: one warp per query row, lanes over the head dim.
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnArgs a)
{
    const size_t nrows = static_cast<size_t>(a.B) * a.L * a.Hq;
    const size_t row = static_cast<size_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= nrows) return;
    const float2 *ml = reinterpret_cast<const float2 *>(a.part_ml);
    float mx = -INFINITY;
    for (int z = 0; z < a.nsplit; ++z) mx = fmaxf(mx, ml[z * nrows + row].x);
    float den = 0.f;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    const int per = a.D / 32;   // 4 or 8 consecutive dims per lane
    for (int z = 0; z < a.nsplit; ++z) {
        const float2 v = ml[z * nrows + row];
        const float w = fast_exp2(v.x - mx);
        den = fmaf(w, v.y, den);
        const float *po = a.part_o + (z * nrows + row) * a.D + lane * per;
#pragma unroll
        for (int e = 0; e < 8; ++e)
            if (e < per) acc[e] = fmaf(w, po[e], acc[e]);
    }
    const float inv = 1.f / den;
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
