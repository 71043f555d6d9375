// dg_lm_head.cu -- the LM head of the denoising step as one persistent
// tcgen05 GEMM with the sampler fused into its epilogue.
//
// "Parallel Denoising From an Autoregressive Checkpoint", section "Finding":
// per step the sampling stage runs a full-vocabulary softmax over all 256
// canvas positions (3.06 ms on an H100 against 0.56 ms for an AR step).  Here
// the logits of a 256-row canvas block against a tile of BN vocabulary
// columns are accumulated in TMEM and folded straight into per-row partial
// states (softmax max / sum / entropy numerator, Gumbel-max sample, argmax);
// logits never reach HBM.  The vocabulary projection W [d, V] streams once
// from HBM through TMA; it is the bandwidth roofline of the step.
//
// CTA layout (640 threads, one CTA per SM, persistent over a contiguous
// range of tiles):
//   warp 0      TMA producer: per 64-deep k block, the hidden block
//               X[256 rows, 64] (K-major, 128B swizzle) and BN/64 boxes of
//               W[64, 64] (vocabulary-major = MN-major B, 128B swizzle) into
//               a 4-stage shared-memory ring;
//   warp 1      TMEM allocator + single-thread UMMA issuer: two 128 x BN x 16
//               MMAs (one per 128-row half) per 16-deep k step into a
//               double-buffered fp32 accumulator (2 buffers x 2 halves x 128
//               columns = 512 TMEM columns);
//   warps 4-19  epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 of half
//               ((w - 4) / 4) % 2, one canvas row per thread, every other
//               16-column chunk (two warps share a row's columns), and folds
//               them (dg_sampler.cuh) while the MMA fills the other buffer;
//               at each row-block boundary the two column groups merge
//               their states in shared memory and one partial state per
//               (row, CTA) goes to global memory (slot = CTA index).  A CTA
//               with a single tile leaves accumulator buffer 1 unused: its
//               epilogue warps fill it with the tile's Philox noise words
//               while the MMA runs, and the fold loads them from there.
#include "dg_kernels.h"

namespace dg {

__global__ void __launch_bounds__(kLmThreads, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap map_x,
                   const __grid_constant__ CUtensorMap map_w, LmHeadArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kLmStages * kLmStageBytes);
    uint64_t *empty = full + kLmStages;
    uint64_t *acc_full = empty + kLmStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *mma_done = acc_empty + 2;
    uint64_t *mrg_ready = mma_done + 1;
    uint64_t *mrg_done = mrg_ready + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mrg_done + 1);
    const GroupMerge gm{reinterpret_cast<float *>(smem + kLmStages * kLmStageBytes + 256),
                        mrg_ready, mrg_done, kLmColGroups, kRowsPerBlock};

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, n_slots = gridDim.x;
    const int t0 = tile_begin(c, a.total, n_slots), t1 = tile_begin(c + 1, a.total, n_slots);
    const int ntiles = t1 - t0;

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < kLmStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&acc_full[s], 1);
            mbar_init(&acc_empty[s], kLmEpiWarps);
        }
        mbar_init(mma_done, 1);
        mbar_init(mrg_ready, kLmEpiWarps - kLmEpiWarps / kLmColGroups);
        mbar_init(mrg_done, kLmEpiWarps / kLmColGroups);
        fence_barrier_init();
        tma_prefetch_desc(&map_x);
        tma_prefetch_desc(&map_w);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // set-up above overlaps the previous kernel of the stream; from here on
    // its outputs are visible and the memory it reads may be overwritten
    griddep_wait();
    griddep_launch_dependents();
    if (c == 0 && warp == 2) {
        for (int i = lane; i < a.ncounters; i += 32) a.counters[i] = 0;
    }
    const FoldConsts fc = fold_consts(a.src, a.seed);
    const int xstep = a.x_3d ? static_cast<int>(fc.step) : 0;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_x = policy_evict_last();
            const uint32_t tx = static_cast<uint32_t>(kLmABytes + a.nbox_b * kLmBBoxBytes);
            int s = 0;
            uint32_t ph = 0;
            uint32_t armed = 0, armed_par = 0;   // bit s: stage s armed, its parity
            bool ok = true;
            for (int t = t0; t < t1 && ok; ++t) {
                const int m = t / a.ntn, n = t % a.ntn;
                for (int kb = 0; kb < a.kblocks; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, a.ws, 101)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[s], tx);
                    uint8_t *sa = smem + s * kLmStageBytes;
                    uint8_t *sb = sa + kLmABytes;
                    if (a.x_3d)
                        tma_load_3d(sa, &map_x, &full[s], kb * kLmBK, m * kRowsPerBlock, xstep,
                                    pol_x);
                    else
                        tma_load_2d(sa, &map_x, &full[s], kb * kLmBK, m * kRowsPerBlock, pol_x);
                    for (int j = 0; j < a.nbox_b; ++j)
                        tma_load_2d(sb + j * kLmBBoxBytes, &map_w, &full[s], n * a.BN + j * 64,
                                    kb * kLmBK, pol_w);
                    armed |= 1u << s;
                    armed_par = (armed_par & ~(1u << s)) | (ph << s);
                    if (++s == kLmStages) { s = 0; ph ^= 1u; }
                }
            }
            // every copy this thread started has landed before the CTA can exit
            for (int q = 0; q < kLmStages; ++q)
                if (armed >> q & 1u) mbar_wait(&full[q], armed_par >> q & 1u, a.ws, 102);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = make_idesc_bf16(128, a.BN, 1);
            // descriptors of stage 0; stage s and k step kk only move the start
            // address field (bits 0-13, in 16-byte units)
            const uint32_t sa0 = smem_u32(smem);
            const uint64_t adesc0 = make_sdesc_sw128(sa0, 16, 1024);
            const uint64_t bdesc0 = make_sdesc_sw128(sa0 + kLmABytes, kLmBBoxBytes, 1024);
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int i = 0; i < ntiles && ok; ++i) {
                const int acc = i & 1;
                const uint32_t use = static_cast<uint32_t>(i >> 1);
                if (!mbar_wait(&acc_empty[acc], (use & 1u) ^ 1u, a.ws, 103)) break;
                tc_fence_after();
                const uint32_t d0 = tmem_base + static_cast<uint32_t>(acc * 256);
                for (int kb = 0; kb < a.kblocks; ++kb) {
                    if (!mbar_wait(&full[s], ph, a.ws, 104)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t soff = static_cast<uint64_t>((s * kLmStageBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kLmBK / 16; ++kk) {
                        // B: MN-major, 64-column blocks 8 KB apart (LBO), 8-row
                        // groups 1 KB apart (SBO); a 16-deep k step is 2 groups.
                        const uint64_t bdesc = bdesc0 + soff + static_cast<uint64_t>(kk * (2048 >> 4));
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            // A: K-major, 128-byte rows, 8-row groups 1 KB apart;
                            // a 16-deep k step advances 32 bytes inside the row.
                            const uint64_t adesc = adesc0 + soff +
                                static_cast<uint64_t>((h * (kLmABytes / 2) + kk * 32) >> 4);
                            umma_bf16(d0 + h * 128, adesc, bdesc, idesc, (kb | kk) != 0);
                        }
                    }
                    umma_commit(&empty[s]);
                    if (++s == kLmStages) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&acc_full[acc]);
            }
            umma_commit(mma_done);
            mbar_wait(mma_done, 0, a.ws, 105);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int e = warp - 4;
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int h = (e >> 2) & 1;             // 128-row half
        const int cg = e >> 3;                  // column group: chunks cg, cg + G, ...
        const int rix = h * 128 + q * 32 + lane;  // row within the 256-row block
        uint32_t merges = 0;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        RowState st;
        row_state_init(st);
        int cur_m = -1;
        // one tile: accumulator buffer 1 stays free, so the tile's noise words
        // are computed into it while the MMA runs and the fold loads them
        const bool pre = ntiles == 1;
        if (pre) {
            const int m = t0 / a.ntn, n = t0 % a.ntn;
            noise_to_tmem(tmem_base + lane_off + static_cast<uint32_t>(256 + h * 128), 16 * cg,
                          16 * kLmColGroups, a.BN, static_cast<uint32_t>(n * a.BN),
                          static_cast<uint32_t>(a.V),
                          static_cast<uint32_t>(m * kRowsPerBlock + h * 128 + q * 32 + lane), fc);
        }
        for (int i = 0; i < ntiles; ++i) {
            const int t = t0 + i;
            const int m = t / a.ntn, n = t % a.ntn;
            const int acc = i & 1;
            const uint32_t use = static_cast<uint32_t>(i >> 1);
            if (m != cur_m) {
                if (cur_m >= 0) {
                    const int prow = cur_m * kRowsPerBlock + rix;
                    row_state_finalize(st, fc);
                    group_merge_store(st, cg, rix, merges++, gm, a.part,
                                      static_cast<size_t>(prow) * n_slots + c, prow < a.M, a.ws);
                }
                row_state_init(st);
                cur_m = m;
            }
            const bool ok = mbar_wait(&acc_full[acc], use & 1u, a.ws, 106);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            const int row = m * kRowsPerBlock + h * 128 + q * 32 + lane;
            const uint32_t tb = tmem_base + lane_off + static_cast<uint32_t>(acc * 256 + h * 128);
            const bool live = row < a.M;
            fold_tile(st, tb, 16 * cg, 16 * kLmColGroups, a.BN, static_cast<uint32_t>(n * a.BN),
                      static_cast<uint32_t>(a.V), static_cast<uint32_t>(row), fc, live,
                      pre ? tb + 256u : 0u);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
        }
        if (cur_m >= 0) {
            const int prow = cur_m * kRowsPerBlock + rix;
            row_state_finalize(st, fc);
            group_merge_store(st, cg, rix, merges, gm, a.part,
                              static_cast<size_t>(prow) * n_slots + c, prow < a.M, a.ws);
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
