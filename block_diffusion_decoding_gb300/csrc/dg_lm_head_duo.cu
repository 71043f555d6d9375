// dg_lm_head_duo.cu -- the LM head of the denoising step on 2-CTA clusters
// that issue 2-SM UMMAs (tcgen05 cta_group::2), for large vocabularies (the
// full-vocabulary softmax the "Parallel Denoising From an Autoregressive
// Checkpoint" page, section "Finding", names as a per-step cost).
//
// A tile is 256 canvas rows x BN (256 or 128) vocabulary columns; with
// a.fuse2 (BN = 128) each pair of adjacent tiles of a cluster's range that
// lie in one row block runs as one 256-column tile, so the ranges balance to
// 128 columns while nearly every tile still has 256 (a range of odd length
// ends on a 128-column tile, whose epilogue is also the shorter tail).  CTA rank
// r of the pair streams rows [128 r, 128 r + 128) of the hidden block and
// columns [r BN/2, (r + 1) BN/2) of the W tile into its own shared memory;
// the even CTA issues one 256 x BN x 16 UMMA per 16-deep k step that reads
// both CTAs' halves, and each CTA receives its 128 rows x BN columns of the
// product in its own TMEM (double-buffered, 2 x BN columns).  Compared with
// a W tile multicast to both CTAs, every CTA writes and the tensor core reads
// a third less shared memory per k block, which is what bounds the single-CTA
// MMA at this shape.
//
//   warp 0      TMA producer (both CTAs): X[128 rows, 64] and W[64, BN/2] of
//               its own halves into a 6-stage ring (W from [d, V], or from
//               the packed layout [V/128][d][128] through a 3-D map: the
//               same boxes, each 64 x 64 pair one contiguous 16 KB); both
//               CTAs' copies
//               complete on the even CTA's full barrier (the even CTA expects
//               the bytes of both halves); a stage is free once the pair MMAs
//               that read it are done (the commit is multicast to both CTAs'
//               empty barriers);
//   warp 1      TMEM allocator (both CTAs, collectively); UMMA issuer (even
//               CTA); the accumulator is free once the epilogues of both
//               CTAs have read it (the odd CTA's warps arrive remotely);
//   warps 4..   epilogue (4 x CG warps: CG = 2 in lm_head_duo_kernel, 4 in
//               lm_head_duo_wide_kernel, 3 in the FP8 instance): warp w
//               reads TMEM lanes 32 (w % 4) .. +31, every CG-th 16-column
//               chunk starting at chunk (w - 4) / 4; the column groups merge
//               in shared memory and one partial state per (row, cluster)
//               is stored.
//
// The self-conditioning instance (lm_head_duo_sc_kernel, 8 epilogue warps)
// folds sc = sum_v softmax(logits / T)_v E[v, :] along with the softmax
// statistics (dg_sampler.cuh) and stores one unnormalised part per (row,
// cluster) next to the partial state.
//
// The FP8 instance (lm_head_duo_fp8_kernel) takes E4M3 codes of the hidden
// block X8 [M, d] and of the transposed weight W8t [V, d], both K-major: a
// k block is 128 codes (the same 128 bytes per row as 64 bf16 values), the
// W half tile is one box of BN/2 rows x 128 bytes, and the UMMA is
// kind::f8f6f4 with K = 32.  The epilogue applies the row and column scales
// before the fold.  Half the weight bytes per vocabulary column.
#include "dg_kernels.h"

namespace dg {

namespace {

// Tiles (of a.BN columns) that the tile starting at schedule tile t of a
// unit's range [t, t1) covers: 2 when a.fuse2 is set and tile t + 1 is in the
// range and in the same row block, else 1.
DG_DEVICE int duo_tile_span(const LmHeadArgs &a, int t, int t1)
{
    return (a.fuse2 && t + 1 < t1 && (t + 1) % a.ntn != 0) ? 2 : 1;
}

// TMEM columns between the two accumulator buffers (the widest tile)
constexpr int kDuoAccCols = 256;

template <bool kFp8, int kCG, bool kSC = false>
DG_DEVICE void lm_head_duo_body(const CUtensorMap &map_x, const CUtensorMap &map_w,
                                const LmHeadArgs &a, const CUtensorMap *map_e = nullptr)
{
    // the self-conditioning instance gives two stages of the ring to two
    // buffers of the table E for the tiles in the accumulators
    constexpr int Stages = kSC ? kDuoScStages : kDuoStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Stages * kDuoStageBytes);
    uint64_t *empty = full + Stages;
    uint64_t *acc_full = empty + Stages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *mma_done = acc_empty + 2;
    uint64_t *mrg_ready = mma_done + 1;
    uint64_t *mrg_done = mrg_ready + 1;
    uint64_t *e_full = mrg_done + 1;      // kSC: E buffer b holds the table rows of
    uint64_t *e_empty = e_full + 2;       // the tile in accumulator buffer b
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(e_empty + 2);
    constexpr int CG = DuoEpilogue<kCG>::CG;            // epilogue column groups
    constexpr int EpiWarps = DuoEpilogue<kCG>::Warps;
    const GroupMerge gm{reinterpret_cast<float *>(smem + Stages * kDuoStageBytes + 256),
                        mrg_ready, mrg_done, CG, 128};
    // the self-conditioning instance sizes the state merge for its 2 column
    // groups (the others for up to 4)
    constexpr int MergeBytes = kSC ? (kCG - 1) * 7 * 128 * 4 : kPairMergeBytes;
    const ScMerge sm{reinterpret_cast<float *>(smem + Stages * kDuoStageBytes + 256 + MergeBytes),
                     a.sc_part};
    // kSC: two E buffers of kDuoScETileRows x kScDim bf16 each, then a 1 KB
    // P staging buffer per epilogue warp
    uint16_t *ebuf = reinterpret_cast<uint16_t *>(smem + Stages * kDuoStageBytes + 256 +
                                                  MergeBytes + (kCG - 1) * kScDim * 128 * 4);
    uint16_t *pbuf_all = ebuf + 2 * kDuoScETileRows * kScDim;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = static_cast<int>(cluster_ctarank());          // row / column half
    const int cid = static_cast<int>(cluster_id_x());
    const int ncl = static_cast<int>(num_clusters_x());
    const int t0 = tile_begin(cid, a.total, ncl), t1 = tile_begin(cid + 1, a.total, ncl);
    // bytes of W one CTA stages per k block: BN / 2 columns (bf16, in boxes of
    // 64 columns) or BN / 2 rows of 128 codes (FP8, one box), per spanned tile
    const int w_half_bytes = a.BN * 64;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < Stages; ++s) {
            mbar_init(&full[s], 1);          // used in the even CTA only
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], 2 * EpiWarps);   // used in the even CTA only
        }
        mbar_init(mma_done, 1);
        mbar_init(mrg_ready, EpiWarps - EpiWarps / CG);
        mbar_init(mrg_done, EpiWarps / CG);
        if constexpr (kSC) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(&e_full[b], 1);
                mbar_init(&e_empty[b], EpiWarps);
            }
        }
        fence_barrier_init();
        tma_prefetch_desc(&map_x);
        tma_prefetch_desc(&map_w);
        if constexpr (kSC) tma_prefetch_desc(map_e);
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
    const uint32_t tmem_base = *tmem_slot;
    // set-up above overlaps the previous kernel of the stream; from here on
    // its outputs are visible and the memory it reads may be overwritten
    griddep_wait();
    griddep_launch_dependents();
    if (cid == 0 && r == 0 && warp == 2) {
        for (int i = lane; i < a.ncounters; i += 32) a.counters[i] = 0;
    }
    // Row-bound sharing (a.rowkey): the launch's tag is the epoch in the
    // workspace header.  Unit 0 clears the row keys, then publishes
    // ready = epoch + 1; a unit reads or raises keys only after it has seen
    // that.  The last unit to finish advances the epoch.
    const bool share = a.rowkey != nullptr;
    const uint32_t epoch = share ? ld_relaxed_gpu(&a.ws->lm_epoch) : 0u;
    if (share && cid == 0 && r == 0 && warp == 3) {
        for (int i = lane; i < a.M; i += 32) a.rowkey[i] = 0u;
        __threadfence();
        __syncwarp();
        if (lane == 0) st_release_gpu(&a.ws->lm_ready, epoch + 1u);
    }
    const FoldConsts fc = fold_consts(a.src, a.seed);
    const int xstep = a.x_3d ? static_cast<int>(fc.step) : 0;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            const uint32_t lead_full = mapa_shared(smem_u32(full), 0);
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_par = 0;
            uint32_t earmed = 0, earmed_par = 0;
            bool ok = true;
            int ti = 0;
            for (int t = t0, span = 1; t < t1 && ok; t += span, ++ti) {
                span = duo_tile_span(a, t, t1);
                const int m = t / a.ntn, n = t % a.ntn;
                const int bn = span * a.BN;                     // columns of this tile
                const uint32_t stage_tx =
                    static_cast<uint32_t>(kPairABytes + span * w_half_bytes);
                if constexpr (kSC) {
                    // this CTA's copy of the table rows of the tile's columns
                    const int b = ti & 1;
                    const uint32_t eu = static_cast<uint32_t>(ti >> 1);
                    if (!mbar_wait(&e_empty[b], (eu & 1u) ^ 1u, a.ws, 408)) { ok = false; break; }
                    const int nbox = (bn + kDuoScETileRows / 2 - 1) / (kDuoScETileRows / 2);
                    mbar_arrive_expect_tx(&e_full[b],
                                          static_cast<uint32_t>(nbox * (kDuoScETileRows / 2) * kScDim * 2));
                    for (int j = 0; j < nbox; ++j)
                        tma_load_2d(ebuf + (static_cast<size_t>(b) * kDuoScETileRows +
                                            j * (kDuoScETileRows / 2)) * kScDim,
                                    map_e, &e_full[b], 0, n * a.BN + j * (kDuoScETileRows / 2), pol_x);
                    earmed |= 1u << b;
                    earmed_par = (earmed_par & ~(1u << b)) | ((eu & 1u) << b);
                }
                for (int kb = 0; kb < a.kblocks; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, a.ws, 401)) { ok = false; break; }
                    if (r == 0) mbar_arrive_expect_tx(&full[s], 2 * stage_tx);
                    const uint32_t fb = lead_full + static_cast<uint32_t>(s * 8);
                    uint8_t *sa = smem + s * kDuoStageBytes;
                    uint8_t *sb = sa + kPairABytes;
                    // the block loop passes hidden states with a step coordinate (3-D map)
                    // 128 bytes of each row: 64 bf16 values or 128 codes
                    const int kx = kb * (kFp8 ? 128 : kLmBK);
                    if (a.x_3d)
                        tma_load_3d_pair(sa, &map_x, fb, kx, m * kRowsPerBlock + r * 128, xstep,
                                         pol_x);
                    else
                        tma_load_2d_pair(sa, &map_x, fb, kx, m * kRowsPerBlock + r * 128, pol_x);
                    if constexpr (kFp8) {
                        // W8t rows n BN + r bn/2 .., 128 codes of k block kb, in boxes
                        // of BN/2 rows (K-major: the boxes stack into one operand)
                        for (int j = 0; j < span; ++j)
                            tma_load_2d_pair(sb + j * w_half_bytes, &map_w, fb, kb * 128,
                                             n * a.BN + r * (bn / 2) + j * (a.BN / 2), pol_w);
                    } else if (a.w_packed) {
                        // packed W: the box of 64 columns x 64 rows starting at
                        // column c0 (a multiple of 64) lies in 128-column tile
                        // c0 / 128, at column c0 % 128 of its rows
                        for (int j = 0; j < bn / 128; ++j) {
                            const int c0 = n * a.BN + r * (bn / 2) + j * 64;
                            tma_load_3d_pair(sb + j * kLmBBoxBytes, &map_w, fb, c0 & 127,
                                             kb * kLmBK, c0 >> 7, pol_w);
                        }
                    } else {
                        for (int j = 0; j < bn / 128; ++j)
                            tma_load_2d_pair(sb + j * kLmBBoxBytes, &map_w, fb,
                                             n * a.BN + r * (bn / 2) + j * 64, kb * kLmBK, pol_w);
                    }
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == Stages) { s = 0; ph ^= 1u; }
                }
            }
            // the even CTA: every copy of both CTAs has landed before the
            // closing cluster barrier lets either CTA leave
            if (r == 0)
                for (int q = 0; q < Stages; ++q)
                    if (armed >> q & 1u) mbar_wait(&full[q], armed_par >> q & 1u, a.ws, 402);
            if constexpr (kSC)
                for (int b = 0; b < 2; ++b)
                    if (earmed >> b & 1u) mbar_wait(&e_full[b], earmed_par >> b & 1u, a.ws, 409);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        if (lane == 0 && r == 0) {
            const uint32_t idesc1 = kFp8 ? make_idesc_e4m3(256, a.BN) : make_idesc_bf16(256, a.BN, 1);
            const uint32_t idesc2 =
                kFp8 ? make_idesc_e4m3(256, 2 * a.BN) : make_idesc_bf16(256, 2 * a.BN, 1);
            const uint32_t sa0 = smem_u32(smem);
            const uint64_t adesc0 = make_sdesc_sw128(sa0, 16, 1024);
            // B: K-major 128-byte rows (FP8) or MN-major 64-column blocks (bf16)
            const uint64_t bdesc0 = kFp8 ? make_sdesc_sw128(sa0 + kPairABytes, 16, 1024)
                                         : make_sdesc_sw128(sa0 + kPairABytes, kLmBBoxBytes, 1024);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            int i = 0;
            for (int t = t0, span = 1; t < t1 && ok; t += span, ++i) {
                span = duo_tile_span(a, t, t1);
                const uint32_t idesc = span == 2 ? idesc2 : idesc1;
                const int acc = i & 1;
                const uint32_t use = static_cast<uint32_t>(i >> 1);
                if (!mbar_wait_cluster(&acc_empty[acc], (use & 1u) ^ 1u, a.ws, 404)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kDuoAccCols);
                for (int kb = 0; kb < a.kblocks; ++kb) {
                    if (!mbar_wait(&full[s], ph, a.ws, 405)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t soff = static_cast<uint64_t>((s * kDuoStageBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        // A: K-major 128-byte rows, 8-row groups 1 KB apart, +32 B per k step
                        // (16 bf16 or 32 codes)
                        const uint64_t adesc = adesc0 + soff + static_cast<uint64_t>(kk * 2);
                        if constexpr (kFp8) {
                            // B: K-major like A
                            const uint64_t bdesc = bdesc0 + soff + static_cast<uint64_t>(kk * 2);
                            umma_e4m3_pair(d, adesc, bdesc, idesc, (kb | kk) != 0);
                        } else {
                            // B: MN-major, 64-column blocks 8 KB apart, 8-row groups 1 KB
                            // apart, +16 rows (2 KB) per k step
                            const uint64_t bdesc =
                                bdesc0 + soff + static_cast<uint64_t>(kk * (2048 >> 4));
                            umma_bf16_pair(d, adesc, bdesc, idesc, (kb | kk) != 0);
                        }
                    }
                    umma_commit_pair(&empty[s], 0x3);
                    if (++s == Stages) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair(&acc_full[acc], 0x3);
            }
            umma_commit_pair(mma_done, 0x1);
            mbar_wait(mma_done, 0, a.ws, 406);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                  // TMEM lane quadrant of this warp
        const int cg = (warp - 4) >> 2;          // column group
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        const int rix = q * 32 + lane;           // row within this CTA's 128 rows
        const uint32_t lead_acc_empty = mapa_shared(smem_u32(acc_empty), 0);
        uint32_t merges = 0;
        RowState st;
        row_state_init(st);
        ScAcc sc;
        if constexpr (kSC) sc_init(sc);
        int cur_m = -1;
        int i = 0;
        for (int t = t0, span = 1; t < t1; t += span, ++i) {
            span = duo_tile_span(a, t, t1);
            const int bn = span * a.BN;
            const int m = t / a.ntn, n = t % a.ntn;
            const int acc = i & 1;
            const uint32_t use = static_cast<uint32_t>(i >> 1);
            if (m != cur_m) {
                if (cur_m >= 0) {
                    const int prow = cur_m * kRowsPerBlock + r * 128 + rix;
                    row_state_finalize(st, fc);
                    group_merge_store_t<kSC>(st, cg, rix, merges++, gm, a.part,
                                             static_cast<size_t>(prow) * ncl + cid, prow < a.M,
                                             a.ws, &sc, sm);
                }
                row_state_init(st);
                if constexpr (kSC) sc_init(sc);
                cur_m = m;
            }
            const int row = m * kRowsPerBlock + r * 128 + rix;
            const bool live = row < a.M;
            // the best scores other units have published for this row (read
            // before the wait for the accumulator, used after it)
            bool shared_ok = false;
            uint32_t key = 0u;
            if (share) {
                shared_ok = ld_acquire_gpu(&a.ws->lm_ready) == epoch + 1u;
                if (shared_ok && live) key = ld_relaxed_gpu(a.rowkey + row);
            }
            const bool ok = mbar_wait_cluster(&acc_full[acc], use & 1u, a.ws, 407);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            st.glb = fmaxf(st.glb, key_score(key));
            const uint32_t tb = tmem_base + lane_off + static_cast<uint32_t>(acc * kDuoAccCols);
            if constexpr (kSC) {
                const int b = i & 1;
                const bool eok = mbar_wait(&e_full[b], (use & 1u), a.ws, 410);
                if (!__all_sync(0xFFFFFFFFu, eok)) break;
                fold_tile_sc(st, sc, ebuf + static_cast<size_t>(b) * kDuoScETileRows * kScDim,
                             pbuf_all + (warp - 4) * 32 * 16, tb, 16 * cg, 16 * CG, bn,
                             static_cast<uint32_t>(n * a.BN), static_cast<uint32_t>(a.V),
                             static_cast<uint32_t>(row), fc, live);
                __syncwarp();
                if (lane == 0) mbar_arrive(&e_empty[b]);
            } else if constexpr (kFp8) {
                const float rs = live ? __ldg(a.row_scale + row) : 0.f;
                fold_tile_scaled(st, tb, 16 * cg, 16 * CG, bn,
                                 static_cast<uint32_t>(n * a.BN), static_cast<uint32_t>(a.V),
                                 static_cast<uint32_t>(row), fc, live, rs, a.col_scale);
            } else {
                fold_tile(st, tb, 16 * cg, 16 * CG, bn,
                          static_cast<uint32_t>(n * a.BN), static_cast<uint32_t>(a.V),
                          static_cast<uint32_t>(row), fc, live);
            }
            if (shared_ok && live) {
                // publish this unit's bound when it beats what is known
                const float lbv = fmaxf(st.gbest, st.apb - 2.0f * kGumbelSlack);
                if (lbv > st.glb) {
                    atomicMax(a.rowkey + row, score_key(lbv));
                    st.glb = lbv;
                }
            }
            tc_fence_before();
            __syncwarp();
            // the even CTA's MMA may overwrite this accumulator once both
            // CTAs' epilogues have read it
            if (lane == 0) mbar_arrive_cluster_relaxed(lead_acc_empty + static_cast<uint32_t>(acc * 8));
        }
        if (cur_m >= 0) {
            const int prow = cur_m * kRowsPerBlock + r * 128 + rix;
            row_state_finalize(st, fc);
            group_merge_store_t<kSC>(st, cg, rix, merges, gm, a.part,
                                     static_cast<size_t>(prow) * ncl + cid, prow < a.M, a.ws,
                                     &sc, sm);
        }
    }
    tc_fence_before();
    __syncthreads();
    // no CTA releases its TMEM or leaves while the pair's MMAs, commits or
    // remote arrivals may still reach it
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 512);
    }
    if (share) {
        // every key access of this unit is done before it is counted
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint32_t prev = atomicAdd(&a.ws->lm_done, 1u);
            if (prev == gridDim.x - 1u) {
                a.ws->lm_done = 0u;
                a.ws->lm_epoch = epoch + 1u;
            }
        }
    }
}

}  // namespace

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(DuoEpilogue<kDuoCGNarrow>::Threads, 1)
    lm_head_duo_kernel(const __grid_constant__ CUtensorMap map_x,
                       const __grid_constant__ CUtensorMap map_w, LmHeadArgs a)
{
    lm_head_duo_body<false, kDuoCGNarrow>(map_x, map_w, a);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(DuoEpilogue<kDuoCGWide>::Threads, 1)
    lm_head_duo_wide_kernel(const __grid_constant__ CUtensorMap map_x,
                            const __grid_constant__ CUtensorMap map_w, LmHeadArgs a)
{
    lm_head_duo_body<false, kDuoCGWide>(map_x, map_w, a);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(DuoEpilogue<kDuoCGNarrow>::Threads, 1)
    lm_head_duo_sc_kernel(const __grid_constant__ CUtensorMap map_x,
                          const __grid_constant__ CUtensorMap map_w,
                          const __grid_constant__ CUtensorMap map_e, LmHeadArgs a)
{
    lm_head_duo_body<false, kDuoCGNarrow, true>(map_x, map_w, a, &map_e);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(DuoEpilogue<kDuoCGFp8>::Threads, 1)
    lm_head_duo_fp8_kernel(const __grid_constant__ CUtensorMap map_x,
                           const __grid_constant__ CUtensorMap map_w, LmHeadArgs a)
{
    lm_head_duo_body<true, kDuoCGFp8>(map_x, map_w, a);
}

}  // namespace dg
