// dS and dB from one read of dY.
//
// LoRAFusion notes (papers.chlience.com), section 5 "FusedLoRA", and the
// article (juhe.plus) section 4.1, backward ③: the dS and dB computations are
// fused so the full-size dY is loaded once:
//     dS  = alpha dY B_a^T      (m x r; scaled by 1/(1-p) later: dSq)
//     dB  = S'^T dY             (r x n; S' = alpha S from the forward)
// Each unit is one (128-row tile, 128-wide n block) of dY, staged by TMA as two
// 128B-swizzled 128 x 64 boxes.  The same shared-memory tile is read twice by
// the tensor cores: K-major for dS (K = n) and MN-major for dB^T (M = n,
// K = tokens).
//
// Both products reduce over a different dimension of dY (dS over n, dB over
// the tokens), so whichever accumulator a CTA cannot keep must be flushed
// with fp32 reductions.  Two orders of the units:
//  - tile order (padded rank 16): tile by tile, each tile's n-blocks in
//    order.  dS stays in TMEM over the CTA's run of n-blocks and every unit's
//    128 x r dB^T partial is flushed.  At this rank the flushes are small.
//  - strip order (padded rank >= 32), where per-unit dB^T flushes would move
//    up to as many bytes as dY itself.  Units are walked in strips of `strip`
//    n-blocks; inside a strip, tile after tile in routing order, each tile's
//    n-blocks innermost.  TMEM holds one dB^T accumulator per n-block of the
//    strip for as long as the CTA stays in the strip with one adapter (a
//    segment), and a double-buffered dS accumulator per tile visit.  Per unit
//    of dY the reductions are then 128 x r floats divided by the strip width
//    (dS), plus one flush of the strip's dB^T accumulators per segment: at
//    rank 64 a sixth of the bytes of the tile order.
// In both orders two threads issue the MMAs of a stage (dS and dB^T): a small
// MMA costs its issuing thread a fixed time whatever its size.  The strip
// order up to padded rank 64 uses four (dsdb_strip4_kernel below).  Where two
// stages fit in half the shared memory (padded rank <= 32) two CTAs share each
// SM with two-stage rings; otherwise one CTA per SM holds the deepest ring.
// Either way finalize_bwd1 then scales and rounds the sums (dSq =
// bf16(alpha/(1-p) dS), dB = bf16(dB^T) transposed) and clears the
// accumulators, which start every call at zero.
#include "common.cuh"
#include "kernels.h"

namespace lora {

namespace {

constexpr int kThreads = 224;   // warp 0 TMA, warp 1 dS MMA issuer, warps 2-5 epilogue, warp 6 dB MMA issuer
constexpr int kThreads4 = 288;
constexpr uint32_t kDyBytes = 2u * 128u * 128u;   // 128 tokens x 128 n

// Walks units from u0 on in strip order (strip s of width w, active tile slot,
// n-block j of the strip), without a division per unit.  Every role of the
// kernel walks the same sequence with its own copy.
struct StripIter {
    int s, slot, j, w, tile, a;
    int J, nnb, n_active;
    __device__ __forceinline__ StripIter(int64_t u0, int J_, int nnb_, const Routing& rt)
        : J(J_), nnb(nnb_), n_active(rt.n_active) {
        const int64_t per = static_cast<int64_t>(n_active) * J;
        const int last = (nnb - 1) / J;
        s = static_cast<int>(u0 / per);
        if (s > last) s = last;
        w = min(J, nnb - s * J);
        const int64_t rem = u0 - static_cast<int64_t>(s) * per;
        slot = static_cast<int>(rem / w);
        j = static_cast<int>(rem - static_cast<int64_t>(slot) * w);
        load(rt);
    }
    __device__ __forceinline__ void load(const Routing& rt) {
        if (slot < n_active) {
            tile = rt.active_tiles[slot];
            a = rt.tile_adapter[tile];
        }
    }
    __device__ __forceinline__ int nb() const { return s * J + j; }
    // this unit is the last of its segment (strip and adapter) in the walk order
    __device__ __forceinline__ bool segment_ends(const Routing& rt) const {
        if (j != w - 1) return false;
        if (slot + 1 >= n_active) return true;
        return rt.tile_adapter[rt.active_tiles[slot + 1]] != a;
    }
    __device__ __forceinline__ void next(const Routing& rt) {
        if (++j == w) {
            j = 0;
            if (++slot == n_active) {
                slot = 0;
                ++s;
                w = min(J, nnb - s * J);
            }
            load(rt);
        }
    }
};

// Tile order (padded rank 16): units walked tile by tile, each tile's n-blocks
// in order; dS accumulates in TMEM over the CTA's run of n-blocks of a tile and
// each unit's dB^T partial is flushed from a double-buffered accumulator.
__global__ void __launch_bounds__(kThreads, 2) dsdb_tile_kernel(const __grid_constant__ DsDbParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const int S = p.stages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * p.stage_bytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;
    uint64_t* accS_full = bars + 2 * S;
    uint64_t* accS_empty = accS_full + 1;
    uint64_t* accB_full = accS_empty + 1;   // [2]
    uint64_t* accB_empty = accB_full + 2;   // [2]
    uint64_t* drain = accB_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rpad_max = p.rt.rpad_max;
    uint32_t tmem_cols = 32;
    while (tmem_cols < static_cast<uint32_t>(3 * rpad_max)) tmem_cols <<= 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);   // both issuers' commits
        }
        mbar_init(accS_full, 1);
        mbar_init(accS_empty, 128);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accB_full[b], 1);
            mbar_init(&accB_empty[b], 128);
        }
        mbar_init(drain, 2);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&p.mapDY);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem;
    const uint32_t tB = tmem + static_cast<uint32_t>(rpad_max);
    const WaitCtx w{&abort_flag, p.ctl.status, p.ctl.wait_ns, kKDsDb << 8};

    const int64_t U = p.units;
    const int64_t u0 = U * blockIdx.x / gridDim.x;
    const int64_t u1 = U * (blockIdx.x + 1) / gridDim.x;
    const uint32_t bbox = static_cast<uint32_t>(rpad_max) * 128u;   // spacing of the two B boxes

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            TileBlockIter it(u0, p.nnb, p.rt);
            for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
                const int nb = it.blk;
                const int tile = it.tile;
                const int a = it.a;
                const int rpad = p.rt.ad[a].rpad;
                if (!mbar_wait(&empty[s], ph ^ 1u, w, 1)) { ok = false; break; }
                uint8_t* st = smem + s * p.stage_bytes;
                mbar_arrive_expect_tx(&full[s], kDyBytes + 2u * 128u * rpad + 256u * rpad);
                tma_load_2d(st, &p.mapDY, &full[s], nb * 128, tile * kTileM);
                tma_load_2d(st + 16384, &p.mapDY, &full[s], nb * 128 + 64, tile * kTileM);
                tma_load_2d(st + p.off_b, &p.mapB[a], &full[s], nb * 128, 0);
                tma_load_2d(st + p.off_b + bbox, &p.mapB[a], &full[s], nb * 128 + 64, 0);
                tma_load_2d(st + p.off_s, &p.mapS[a], &full[s], 0, tile * kTileM);
                if (rpad > 64) tma_load_2d(st + p.off_s + 16384, &p.mapS[a], &full[s], 64, tile * kTileM);
                ++issued;
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            if (!ok) {
                const int64_t back = issued < S ? issued : S;
                for (int64_t i = issued - back; i < issued; ++i)
                    mbar_wait_drain(&full[i % S], static_cast<uint32_t>((i / S) & 1), p.ctl.wait_ns);
            }
        }
    } else if (warp == 1 || warp == 6) {
        // Two issuing threads: warp 1 issues the dS MMAs, warp 6 the dB^T MMAs of the same stage.  A small
        // MMA costs its issuing thread a fixed time whatever its size, so two issuers halve the issue time
        // per stage; each commits its own MMAs (a stage is free once both have).
        if (lane == 0) {
            const bool ds_role = warp == 1;
            int s = 0;
            uint32_t ph = 0;
            uint32_t units_done = 0, items_done = 0;
            // Operand descriptors of stage 0, built once: an MMA only moves the start-address
            // field (bytes / 16) by its stage and K step.  The rank-dependent ones (N = rpad,
            // S' layout) are rebuilt when the adapter's padded rank changes.
            const uint32_t sbase = smem_u32(smem);
            const uint64_t ds_a0 = make_smem_desc(sbase, 16, 1024, kSw128);              // dY, K-major
            const uint64_t ds_b0 = make_smem_desc(sbase + p.off_b, 16, 1024, kSw128);    // B_a, K-major
            const uint64_t db_a0 = make_smem_desc(sbase, 16384, 1024, kSw128);           // dY^T, MN-major
            const uint32_t bbox16 = bbox >> 4;
            int cur_rpad = -1;
            uint32_t idesc_s = 0, idesc_b = 0, rb = 0;
            uint64_t db_b0 = 0;
            TileBlockIter it(u0, p.nnb, p.rt);
            for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
                const int nb = it.blk;
                const int rpad = p.rt.ad[it.a].rpad;
                if (rpad != cur_rpad) {
                    cur_rpad = rpad;
                    idesc_s = make_idesc_bf16(128, rpad, false, false);
                    idesc_b = make_idesc_bf16(128, rpad, true, true);
                    rb = rank_row_bytes(rpad);
                    db_b0 = make_smem_desc(sbase + p.off_s, 16384, 8u * rb, rank_swizzle(rpad));   // S', MN-major
                }
                const bool first = (u == u0) || nb == 0;
                const bool last = (u == u1 - 1) || nb == p.nnb - 1;
                const uint32_t bb = units_done & 1u;
                if (ds_role) {
                    if (first) {
                        if (!mbar_wait(accS_empty, (items_done & 1u) ^ 1u, w, 2)) break;
                        tc_fence_after();
                    }
                } else {
                    if (!mbar_wait(&accB_empty[bb], ((units_done >> 1) & 1u) ^ 1u, w, 3)) break;
                    tc_fence_after();
                }
                if (!mbar_wait(&full[s], ph, w, 4)) break;
                tc_fence_after();
                const uint64_t so = (static_cast<uint32_t>(s) * p.stage_bytes) >> 4;
                if (ds_role) {
                    // dS (+)= dY_tile (128 x 128, K = n) * B_a^T (K = n, N = rpad): box h = ks / 4, 32 B per step
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t h = static_cast<uint64_t>(ks >> 2), kk = static_cast<uint64_t>(ks & 3);
                        umma_bf16(tS, ds_a0 + so + h * 1024u + kk * 2u, ds_b0 + so + h * bbox16 + kk * 2u, idesc_s,
                                  (first && ks == 0) ? 0u : 1u);
                    }
                    umma_commit(&empty[s]);
                    if (last) {
                        umma_commit(accS_full);
                        ++items_done;
                    }
                } else {
                    // dB^T = dY_tile^T (M = n: two 64-wide atoms, K = tokens) * S'_tile (K = tokens, N = rpad):
                    // 16 tokens per step = 2048 B of dY and 16 * rb B of S'
                    const uint32_t dB_acc = tB + bb * static_cast<uint32_t>(rpad_max);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        umma_bf16(dB_acc, db_a0 + so + ks * 128u, db_b0 + so + static_cast<uint64_t>(ks) * rb, idesc_b,
                                  ks != 0 ? 1u : 0u);
                    umma_commit(&empty[s]);
                    umma_commit(&accB_full[bb]);
                }
                ++units_done;
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            umma_commit(drain);
            mbar_wait_drain(drain, 0, p.ctl.wait_ns);
        }
    } else if (warp >= 2 && warp <= 5) {
        const int quad = warp & 3;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t units_done = 0, items_done = 0;
        TileBlockIter it(u0, p.nnb, p.rt);
        for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
            const int nb = it.blk;
            const int tile = it.tile;
            const AdapterDev ad = p.rt.ad[it.a];
            const bool last = (u == u1 - 1) || nb == p.nnb - 1;
            const uint32_t bb = units_done & 1u;
            bool ok = mbar_wait(&accB_full[bb], (units_done >> 1) & 1u, w, 5);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            if (p.parts & kPartDb) {
                const int64_t nidx = static_cast<int64_t>(nb) * 128 + quad * 32 + lane;
                float* dst = p.acc_base + ad.dB_off + nidx * ad.rpad;
                const uint32_t taddr = tB + lane_off + bb * static_cast<uint32_t>(rpad_max);
                for (int c0 = 0; c0 < ad.rpad; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(taddr + c0, v);
                    tmem_ld_wait();
                    if (nidx < p.n) {
#pragma unroll
                        for (int q = 0; q < 16; q += 4)
                            if (c0 + q < ad.rank)
                                red_add_v4(dst + c0 + q, __uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                                           __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&accB_empty[bb]);
            ++units_done;
            if (last) {
                ok = mbar_wait(accS_full, items_done & 1u, w, 6);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                tc_fence_after();
                const int64_t row = static_cast<int64_t>(tile) * kTileM + quad * 32 + lane;
                // deterministic mode: this CTA's partial of active tile it.slot goes to slot it.slot + CTA
                float* dst = p.sl.base ? p.sl.base + ((static_cast<int64_t>(it.slot) + blockIdx.x) * 128 + quad * 32 + lane) *
                                                         p.sl.ld
                                       : p.dS_acc + row * p.ld;
                for (int c0 = 0; (p.parts & kPartDs) && c0 < ad.rpad; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tS + lane_off + c0, v);
                    tmem_ld_wait();
                    if (row < p.m) {
#pragma unroll
                        for (int q = 0; q < 16; q += 4) {
                            if (c0 + q >= ad.rank) continue;
                            if (p.sl.base)
                                st_f4(dst + c0 + q, __uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                                      __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
                            else
                                red_add_v4(dst + c0 + q, __uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                                           __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(accS_empty);
                ++items_done;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

// Strip order (padded rank >= 32), described at the top of this file.
__global__ void __launch_bounds__(kThreads, 2) dsdb_strip_kernel(const __grid_constant__ DsDbParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const int S = p.stages;
    const int J = p.strip;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * p.stage_bytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;
    uint64_t* accS_full = bars + 2 * S;     // [2]
    uint64_t* accS_empty = accS_full + 2;   // [2]
    uint64_t* accB_full = accS_empty + 2;
    uint64_t* accB_empty = accB_full + 1;
    uint64_t* drain = accB_empty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rpad_max = p.rt.rpad_max;
    uint32_t tmem_cols = 32;
    while (tmem_cols < static_cast<uint32_t>((2 + J) * rpad_max)) tmem_cols <<= 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 2);   // both issuers' commits
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accS_full[b], 1);
            mbar_init(&accS_empty[b], 128);
        }
        mbar_init(accB_full, 1);
        mbar_init(accB_empty, 128);
        mbar_init(drain, 2);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&p.mapDY);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem;                                                   // dS: two buffers
    const uint32_t tB = tmem + 2u * static_cast<uint32_t>(rpad_max);            // dB^T: one per n-block of a strip
    const WaitCtx w{&abort_flag, p.ctl.status, p.ctl.wait_ns, kKDsDb << 8};

    const int64_t U = p.units;
    const int64_t u0 = U * blockIdx.x / gridDim.x;
    const int64_t u1 = U * (blockIdx.x + 1) / gridDim.x;
    const uint32_t bbox = static_cast<uint32_t>(rpad_max) * 128u;   // spacing of the two B boxes

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            StripIter it(u0, J, p.nnb, p.rt);
            for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
                const int nb = it.nb();
                const int tile = it.tile;
                const int a = it.a;
                const int rpad = p.rt.ad[a].rpad;
                if (!mbar_wait(&empty[s], ph ^ 1u, w, 1)) { ok = false; break; }
                uint8_t* st = smem + s * p.stage_bytes;
                mbar_arrive_expect_tx(&full[s], kDyBytes + 2u * 128u * rpad + 256u * rpad);
                tma_load_2d(st, &p.mapDY, &full[s], nb * 128, tile * kTileM);
                tma_load_2d(st + 16384, &p.mapDY, &full[s], nb * 128 + 64, tile * kTileM);
                tma_load_2d(st + p.off_b, &p.mapB[a], &full[s], nb * 128, 0);
                tma_load_2d(st + p.off_b + bbox, &p.mapB[a], &full[s], nb * 128 + 64, 0);
                tma_load_2d(st + p.off_s, &p.mapS[a], &full[s], 0, tile * kTileM);
                if (rpad > 64) tma_load_2d(st + p.off_s + 16384, &p.mapS[a], &full[s], 64, tile * kTileM);
                ++issued;
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            if (!ok) {
                const int64_t back = issued < S ? issued : S;
                for (int64_t i = issued - back; i < issued; ++i)
                    mbar_wait_drain(&full[i % S], static_cast<uint32_t>((i / S) & 1), p.ctl.wait_ns);
            }
        }
    } else if (warp == 1 || warp == 6) {
        // Two issuing threads, as in the tile order: warp 1 the dS MMAs, warp 6 the dB^T MMAs.
        if (lane == 0) {
            const bool ds_role = warp == 1;
            int s = 0;
            uint32_t ph = 0;
            uint32_t visits = 0, segs = 0, used = 0;
            bool new_seg = true;
            // Operand descriptors of stage 0, built once: an MMA only moves the start-address
            // field (bytes / 16) by its stage and K step.  The rank-dependent ones (N = rpad,
            // S' layout) are rebuilt when the adapter's padded rank changes.
            const uint32_t sbase = smem_u32(smem);
            const uint64_t ds_a0 = make_smem_desc(sbase, 16, 1024, kSw128);              // dY, K-major
            const uint64_t ds_b0 = make_smem_desc(sbase + p.off_b, 16, 1024, kSw128);    // B_a, K-major
            const uint64_t db_a0 = make_smem_desc(sbase, 16384, 1024, kSw128);           // dY^T, MN-major
            const uint32_t bbox16 = bbox >> 4;
            int cur_rpad = -1;
            uint32_t idesc_s = 0, idesc_b = 0, rb = 0;
            uint64_t db_b0 = 0;
            StripIter it(u0, J, p.nnb, p.rt);
            for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
                const int rpad = p.rt.ad[it.a].rpad;
                if (rpad != cur_rpad) {
                    cur_rpad = rpad;
                    idesc_s = make_idesc_bf16(128, rpad, false, false);
                    idesc_b = make_idesc_bf16(128, rpad, true, true);
                    rb = rank_row_bytes(rpad);
                    db_b0 = make_smem_desc(sbase + p.off_s, 16384, 8u * rb, rank_swizzle(rpad));   // S', MN-major
                }
                const bool visit_first = (u == u0) || it.j == 0;
                const bool visit_last = (u == u1 - 1) || it.j == it.w - 1;
                const bool seg_last = (u == u1 - 1) || it.segment_ends(p.rt);
                const uint32_t bs = visits & 1u;
                if (ds_role) {
                    if (visit_first) {
                        if (!mbar_wait(&accS_empty[bs], ((visits >> 1) & 1u) ^ 1u, w, 3)) break;
                        tc_fence_after();
                    }
                } else if (new_seg) {
                    // the previous segment's dB^T accumulators have been flushed
                    if (!mbar_wait(accB_empty, (segs & 1u) ^ 1u, w, 2)) break;
                    tc_fence_after();
                    used = 0;
                }
                if (!mbar_wait(&full[s], ph, w, 4)) break;
                tc_fence_after();
                const uint64_t so = (static_cast<uint32_t>(s) * p.stage_bytes) >> 4;
                if (ds_role) {
                    // dS (+)= dY_tile (128 x 128, K = n) * B_a^T (K = n, N = rpad): box h = ks / 4, 32 B per step
                    const uint32_t dS_acc = tS + bs * static_cast<uint32_t>(rpad_max);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t h = static_cast<uint64_t>(ks >> 2), kk = static_cast<uint64_t>(ks & 3);
                        umma_bf16(dS_acc, ds_a0 + so + h * 1024u + kk * 2u, ds_b0 + so + h * bbox16 + kk * 2u, idesc_s,
                                  (visit_first && ks == 0) ? 0u : 1u);
                    }
                    umma_commit(&empty[s]);
                    if (visit_last) {
                        umma_commit(&accS_full[bs]);
                        ++visits;
                    }
                } else {
                    // dB^T[n-block] (+)= dY_tile^T (M = n: two 64-wide atoms, K = tokens) * S'_tile (K = tokens,
                    // N = rpad): 16 tokens per step = 2048 B of dY and 16 * rb B of S'
                    const uint32_t dB_acc = tB + static_cast<uint32_t>(it.j * rpad_max);
                    const bool fresh = ((used >> it.j) & 1u) == 0u;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        umma_bf16(dB_acc, db_a0 + so + ks * 128u, db_b0 + so + static_cast<uint64_t>(ks) * rb, idesc_b,
                                  (fresh && ks == 0) ? 0u : 1u);
                    used |= 1u << it.j;
                    umma_commit(&empty[s]);
                    new_seg = seg_last;
                    if (seg_last) {
                        umma_commit(accB_full);
                        ++segs;
                    }
                }
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            umma_commit(drain);
            mbar_wait_drain(drain, 0, p.ctl.wait_ns);
        }
    } else if (warp >= 2 && warp <= 5) {
        const int quad = warp & 3;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t visits = 0, segs = 0, used = 0;
        StripIter it(u0, J, p.nnb, p.rt);
        for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
            const AdapterDev ad = p.rt.ad[it.a];
            const bool visit_last = (u == u1 - 1) || it.j == it.w - 1;
            const bool seg_last = (u == u1 - 1) || it.segment_ends(p.rt);
            used |= 1u << it.j;
            if (visit_last) {
                const uint32_t bs = visits & 1u;
                const bool ok = mbar_wait(&accS_full[bs], (visits >> 1) & 1u, w, 5);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                tc_fence_after();
                const int64_t row = static_cast<int64_t>(it.tile) * kTileM + quad * 32 + lane;
                float* dst = p.dS_acc + row * p.ld;
                const uint32_t taddr = tS + lane_off + bs * static_cast<uint32_t>(rpad_max);
                for (int c0 = 0; (p.parts & kPartDs) && c0 < ad.rpad; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(taddr + c0, v);
                    tmem_ld_wait();
                    if (row < p.m) {
#pragma unroll
                        for (int q = 0; q < 16; q += 4)
                            if (c0 + q < ad.rank)
                                red_add_v4(dst + c0 + q, __uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                                           __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
                    }
                }
                tc_fence_before();
                mbar_arrive(&accS_empty[bs]);
                ++visits;
            }
            if (seg_last) {
                const bool ok = mbar_wait(accB_full, segs & 1u, w, 6);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                tc_fence_after();
                for (int jj = 0; (p.parts & kPartDb) && jj < it.w; ++jj) {
                    if (!((used >> jj) & 1u)) continue;
                    const int64_t nidx = static_cast<int64_t>(it.s * J + jj) * 128 + quad * 32 + lane;
                    float* dst = p.acc_base + ad.dB_off + nidx * ad.rpad;
                    const uint32_t taddr = tB + lane_off + static_cast<uint32_t>(jj * rpad_max);
                    for (int c0 = 0; c0 < ad.rpad; c0 += 16) {
                        uint32_t v[16];
                        tmem_ld16(taddr + c0, v);
                        tmem_ld_wait();
                        if (nidx < p.n) {
#pragma unroll
                            for (int q = 0; q < 16; q += 4)
                                if (c0 + q < ad.rank)
                                    red_add_v4(dst + c0 + q, __uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                                               __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(accB_empty);
                ++segs;
                used = 0;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

// Strip order with four MMA-issuing threads (padded rank <= 64, even strip width).  One thread issues a
// small tcgen05 MMA about every 250-300 cycles however many accumulators it feeds, and independent issuing
// warps add up (measured on GB300 with M128 N64 K16 MMAs: 1, 2, 4 and 8 issuers gave one MMA per 318, 155,
// 79 and 49 cycles per SM).  So the dS MMAs of a unit are shared by two threads, each into its own
// accumulator (the 64-deep halves of the unit's n-block; the epilogue adds the two), and the dB^T MMAs of a
// unit go to one of two threads by the parity of its n-block within the strip, each n-block keeping one
// accumulator.  TMEM: two dS buffers per dS thread, then one dB^T accumulator per n-block of a strip.
__global__ void __launch_bounds__(kThreads4, 2) dsdb_strip4_kernel(const __grid_constant__ DsDbParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const int S = p.stages;
    const int J = p.strip;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * p.stage_bytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;             // all four issuers: both dS threads commit, the dB^T thread of the
                                            // unit's parity commits and the other one arrives
    uint64_t* accS_full = bars + 2 * S;     // [2]: both dS threads commit
    uint64_t* accS_empty = accS_full + 2;   // [2]
    uint64_t* accB_full = accS_empty + 2;   // [2]: per n-block parity
    uint64_t* accB_empty = accB_full + 2;   // [2]: per n-block parity
    uint64_t* drain = accB_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rpad_max = p.rt.rpad_max;
    uint32_t tmem_cols = 32;
    while (tmem_cols < static_cast<uint32_t>((4 + J) * rpad_max)) tmem_cols <<= 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accS_full[b], 2);
            mbar_init(&accS_empty[b], 128);
            mbar_init(&accB_full[b], 1);
            mbar_init(&accB_empty[b], 128);
        }
        mbar_init(drain, 4);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&p.mapDY);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem = *tmem_slot;
    const uint32_t rp = static_cast<uint32_t>(rpad_max);
    const uint32_t tB = tmem + 4u * rp;   // dB^T: one per n-block of a strip
    const WaitCtx w{&abort_flag, p.ctl.status, p.ctl.wait_ns, kKDsDb << 8};

    const int64_t U = p.units;
    const int64_t u0 = U * blockIdx.x / gridDim.x;
    const int64_t u1 = U * (blockIdx.x + 1) / gridDim.x;
    const uint32_t bbox = rp * 128u;   // spacing of the two B boxes

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            StripIter it(u0, J, p.nnb, p.rt);
            for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
                const int nb = it.nb();
                const int tile = it.tile;
                const int a = it.a;
                const int rpad = p.rt.ad[a].rpad;
                if (!mbar_wait(&empty[s], ph ^ 1u, w, 1)) { ok = false; break; }
                uint8_t* st = smem + s * p.stage_bytes;
                mbar_arrive_expect_tx(&full[s], kDyBytes + 2u * 128u * rpad + 256u * rpad);
                tma_load_2d(st, &p.mapDY, &full[s], nb * 128, tile * kTileM);
                tma_load_2d(st + 16384, &p.mapDY, &full[s], nb * 128 + 64, tile * kTileM);
                tma_load_2d(st + p.off_b, &p.mapB[a], &full[s], nb * 128, 0);
                tma_load_2d(st + p.off_b + bbox, &p.mapB[a], &full[s], nb * 128 + 64, 0);
                tma_load_2d(st + p.off_s, &p.mapS[a], &full[s], 0, tile * kTileM);
                if (rpad > 64) tma_load_2d(st + p.off_s + 16384, &p.mapS[a], &full[s], 64, tile * kTileM);
                ++issued;
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            if (!ok) {
                const int64_t back = issued < S ? issued : S;
                for (int64_t i = issued - back; i < issued; ++i)
                    mbar_wait_drain(&full[i % S], static_cast<uint32_t>((i / S) & 1), p.ctl.wait_ns);
            }
        }
    } else if (warp == 1 || warp == 7) {
        // dS (+)= dY_tile * B_a^T over one 64-deep half of the unit's n-block: warp 1 the first, warp 7 the second
        if (lane == 0) {
            const uint32_t h = warp == 1 ? 0u : 1u;
            const uint32_t tS = tmem + 2u * h * rp;
            int s = 0;
            uint32_t ph = 0;
            uint32_t visits = 0;
            const uint32_t sbase = smem_u32(smem);
            const uint64_t ds_a0 = make_smem_desc(sbase, 16, 1024, kSw128) + h * 1024u;                      // dY, K-major
            const uint64_t ds_b0 = make_smem_desc(sbase + p.off_b, 16, 1024, kSw128) + h * (bbox >> 4);      // B_a, K-major
            int cur_rpad = -1;
            uint32_t idesc_s = 0;
            StripIter it(u0, J, p.nnb, p.rt);
            for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
                const int rpad = p.rt.ad[it.a].rpad;
                if (rpad != cur_rpad) {
                    cur_rpad = rpad;
                    idesc_s = make_idesc_bf16(128, rpad, false, false);
                }
                const bool visit_first = (u == u0) || it.j == 0;
                const bool visit_last = (u == u1 - 1) || it.j == it.w - 1;
                const uint32_t bs = visits & 1u;
                if (visit_first) {
                    if (!mbar_wait(&accS_empty[bs], ((visits >> 1) & 1u) ^ 1u, w, 3)) break;
                    tc_fence_after();
                }
                if (!mbar_wait(&full[s], ph, w, 4)) break;
                tc_fence_after();
                const uint64_t so = (static_cast<uint32_t>(s) * p.stage_bytes) >> 4;
                const uint32_t dS_acc = tS + bs * rp;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(dS_acc, ds_a0 + so + kk * 2u, ds_b0 + so + kk * 2u, idesc_s, (visit_first && kk == 0) ? 0u : 1u);
                umma_commit(&empty[s]);
                if (visit_last) {
                    umma_commit(&accS_full[bs]);
                    ++visits;
                }
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            umma_commit(drain);
            mbar_wait_drain(drain, 0, p.ctl.wait_ns);
        }
    } else if (warp == 6 || warp == 8) {
        // dB^T[n-block] (+)= dY_tile^T * S'_tile for the units whose n-block has this thread's parity
        if (lane == 0) {
            const int par = warp == 6 ? 0 : 1;
            int s = 0;
            uint32_t ph = 0;
            uint32_t segs = 0, used = 0;
            bool had = false;   // this thread has MMAs in the current segment
            const uint32_t sbase = smem_u32(smem);
            const uint64_t db_a0 = make_smem_desc(sbase, 16384, 1024, kSw128);   // dY^T, MN-major
            int cur_rpad = -1;
            uint32_t idesc_b = 0, rb = 0;
            uint64_t db_b0 = 0;
            StripIter it(u0, J, p.nnb, p.rt);
            bool ok = true;
            for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
                const bool seg_last = (u == u1 - 1) || it.segment_ends(p.rt);
                // Every stage's phase is waited on, the other parity's too: a parity wait tells two phases apart
                // only if the waiter sees each one, and a thread that skipped stages could take an older
                // completion of this stage's barrier for the current one.
                if ((it.j & 1) != par) {
                    if (!mbar_wait(&full[s], ph, w, 4)) { ok = false; break; }
                    mbar_arrive(&empty[s]);
                } else {
                    const int rpad = p.rt.ad[it.a].rpad;
                    if (rpad != cur_rpad) {
                        cur_rpad = rpad;
                        idesc_b = make_idesc_bf16(128, rpad, true, true);
                        rb = rank_row_bytes(rpad);
                        db_b0 = make_smem_desc(sbase + p.off_s, 16384, 8u * rb, rank_swizzle(rpad));   // S', MN-major
                    }
                    if (!had) {
                        // the previous segment's dB^T accumulators of this parity have been flushed
                        if (!mbar_wait(&accB_empty[par], (segs & 1u) ^ 1u, w, 2)) { ok = false; break; }
                        tc_fence_after();
                        used = 0;
                        had = true;
                    }
                    if (!mbar_wait(&full[s], ph, w, 4)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t so = (static_cast<uint32_t>(s) * p.stage_bytes) >> 4;
                    const uint32_t dB_acc = tB + static_cast<uint32_t>(it.j) * rp;
                    const bool fresh = ((used >> it.j) & 1u) == 0u;
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks)
                        umma_bf16(dB_acc, db_a0 + so + ks * 128u, db_b0 + so + static_cast<uint64_t>(ks) * rb, idesc_b,
                                  (fresh && ks == 0) ? 0u : 1u);
                    used |= 1u << it.j;
                    umma_commit(&empty[s]);
                }
                if (seg_last && had) {
                    umma_commit(&accB_full[par]);
                    ++segs;
                    had = false;
                }
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            (void)ok;
            umma_commit(drain);
            mbar_wait_drain(drain, 0, p.ctl.wait_ns);
        }
    } else if (warp >= 2 && warp <= 5) {
        const int quad = warp & 3;
        const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
        uint32_t visits = 0, used = 0, present = 0;
        uint32_t segs[2] = {0u, 0u};
        StripIter it(u0, J, p.nnb, p.rt);
        for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
            const AdapterDev ad = p.rt.ad[it.a];
            const bool visit_last = (u == u1 - 1) || it.j == it.w - 1;
            const bool seg_last = (u == u1 - 1) || it.segment_ends(p.rt);
            used |= 1u << it.j;
            present |= 1u << (it.j & 1);
            if (visit_last) {
                const uint32_t bs = visits & 1u;
                const bool ok = mbar_wait(&accS_full[bs], (visits >> 1) & 1u, w, 5);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                tc_fence_after();
                const int64_t row = static_cast<int64_t>(it.tile) * kTileM + quad * 32 + lane;
                float* dst = p.dS_acc + row * p.ld;
                const uint32_t t0 = tmem + lane_off + bs * rp;             // first half's accumulator
                const uint32_t t1 = tmem + lane_off + (2u + bs) * rp;      // second half's
                for (int c0 = 0; (p.parts & kPartDs) && c0 < ad.rpad; c0 += 16) {
                    uint32_t v[16], x[16];
                    tmem_ld16(t0 + c0, v);
                    tmem_ld16(t1 + c0, x);
                    tmem_ld_wait();
                    if (row < p.m) {
#pragma unroll
                        for (int q = 0; q < 16; q += 4)
                            if (c0 + q < ad.rank)
                                red_add_v4(dst + c0 + q, __uint_as_float(v[q]) + __uint_as_float(x[q]),
                                           __uint_as_float(v[q + 1]) + __uint_as_float(x[q + 1]),
                                           __uint_as_float(v[q + 2]) + __uint_as_float(x[q + 2]),
                                           __uint_as_float(v[q + 3]) + __uint_as_float(x[q + 3]));
                    }
                }
                tc_fence_before();
                mbar_arrive(&accS_empty[bs]);
                ++visits;
            }
            if (seg_last) {
                bool ok = true;
                for (int par = 0; par < 2; ++par)
                    if ((present >> par) & 1u) ok = ok && mbar_wait(&accB_full[par], segs[par] & 1u, w, 6);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                tc_fence_after();
                for (int jj = 0; (p.parts & kPartDb) && jj < it.w; ++jj) {
                    if (!((used >> jj) & 1u)) continue;
                    const int64_t nidx = static_cast<int64_t>(it.s * J + jj) * 128 + quad * 32 + lane;
                    float* dst = p.acc_base + ad.dB_off + nidx * ad.rpad;
                    const uint32_t taddr = tB + lane_off + static_cast<uint32_t>(jj) * rp;
                    for (int c0 = 0; c0 < ad.rpad; c0 += 16) {
                        uint32_t v[16];
                        tmem_ld16(taddr + c0, v);
                        tmem_ld_wait();
                        if (nidx < p.n) {
#pragma unroll
                            for (int q = 0; q < 16; q += 4)
                                if (c0 + q < ad.rank)
                                    red_add_v4(dst + c0 + q, __uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                                               __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
                        }
                    }
                }
                tc_fence_before();
                for (int par = 0; par < 2; ++par)
                    if ((present >> par) & 1u) {
                        mbar_arrive(&accB_empty[par]);
                        ++segs[par];
                    }
                used = 0;
                present = 0;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

// dSq[t, c] = bf16(alpha_a / (1 - p_a) * dS_acc[t, c]) for c < r_a, else 0, on
// rows of active tiles (parts & kPartDs); dB_a[c, j] = bf16(dB^T_acc_a[j, c])
// (parts & kPartDb).  Every accumulator read is cleared.
__global__ void __launch_bounds__(256, 4) finalize_bwd1_kernel(float* __restrict__ dS_acc, uint16_t* __restrict__ dSq, int64_t m, int32_t ld,
                                     float* __restrict__ acc_base, int64_t n, const __grid_constant__ Routing rt,
                                     const __grid_constant__ AdapterPtrs dbp, int32_t parts, const Slots sl,
                                     int32_t nnb) {
    __shared__ RowRouting sr;
    load_row_routing(sr, rt);   // parameters only: before the wait on the previous kernel
    pdl_wait();
    pdl_trigger();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (parts & kPartDs) {
        // dS: one thread per 8 columns of a row (m * ld / 8 < 2^31: 32-bit index arithmetic)
        const uint32_t g8 = static_cast<uint32_t>(ld / 8);
        const uint32_t total_s = static_cast<uint32_t>(m) * g8;
        for (uint32_t i = static_cast<uint32_t>(tid); i < total_s; i += static_cast<uint32_t>(stride)) {
            const uint32_t t = i / g8;
            const int c0 = static_cast<int>(i - t * g8) * 8;
            const int a = sr.owner[t >> 7];
            if (a < 0) continue;
            const int valid = sr.rank[a];
            if (sl.base != nullptr) {
                // deterministic mode: the tile's slots added in CTA order
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = 0.f;
                const int64_t item = sr.active[t >> 7];
                if (c0 < valid) slot_sum8(sl, item, item * nnb, (item + 1) * nnb, static_cast<int>(t & 127), c0, v);
                store_row8(dSq + static_cast<int64_t>(t) * ld + c0, v, valid - c0, sr.scale[a]);
                continue;
            }
            float v[8];
            if (c0 < valid) {
                float* src = dS_acc + static_cast<int64_t>(t) * ld + c0;
                const float4 x = ld_l2_f4(src);
                const float4 y = ld_l2_f4(src + 4);
                v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w; v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
                st_zero_f4(src);
                st_zero_f4(src + 4);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = (c0 + e < valid) ? v[e] * sr.scale[a] : 0.f;
            uint4 pk;
            pk.x = pack_bf16x2(v[0], v[1]);
            pk.y = pack_bf16x2(v[2], v[3]);
            pk.z = pack_bf16x2(v[4], v[5]);
            pk.w = pack_bf16x2(v[6], v[7]);
            stg128(dSq + static_cast<int64_t>(t) * ld + c0, pk);
        }
    }
    if (!(parts & kPartDb)) return;
    // dB_a = (dB^T_acc_a)^T.  Lane i of a warp owns accumulator row j = 32 w + i (rpad floats, read 16 at a
    // time, contiguous across the warp) and writes those values down column j of dB, so every store of the
    // warp is 32 consecutive bf16 of one row of dB.  No shared memory and few registers, so these CTAs fit
    // beside the dX GEMM's CTAs on the same SMs.
    const int lane = threadIdx.x & 31;
    const int64_t n_warps = stride / 32, gw = tid / 32;
    const int64_t per_adapter = (n + 31) / 32;   // warp tasks of one adapter; tasks of all adapters share the warps
    int64_t tasks = 0;
    for (int a = 0; a < rt.n_adapters; ++a)
        if (rt.adapter_begin[a + 1] > rt.adapter_begin[a]) tasks += per_adapter;
    for (int64_t w = gw; w < tasks; w += n_warps) {
        int a = 0;
        int64_t rem = w;
        for (;; ++a) {
            if (rt.adapter_begin[a + 1] == rt.adapter_begin[a]) continue;
            if (rem < per_adapter) break;
            rem -= per_adapter;
        }
        const AdapterDev ad = rt.ad[a];
        const int64_t j = rem * 32 + lane;
        if (j >= n) continue;
        float* src = acc_base + ad.dB_off;
        uint16_t* dst = dbp.p[a];
        for (int c0 = 0; c0 < ad.rank; c0 += 16) {   // rpad is a power of two >= 16: whole float4 groups
            float* q = src + j * ad.rpad + c0;
            float v[16];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const float4 x = ld_l2_f4(q + 4 * g);
                v[4 * g + 0] = x.x;
                v[4 * g + 1] = x.y;
                v[4 * g + 2] = x.z;
                v[4 * g + 3] = x.w;
                st_zero_f4(q + 4 * g);
            }
#pragma unroll
            for (int e = 0; e < 16; ++e)
                if (c0 + e < ad.rank) dst[static_cast<int64_t>(c0 + e) * n + j] = bf16_bits(v[e]);
        }
    }
}

}  // namespace

size_t dsdb_smem_bytes(const DsDbParams& p) { return 1024 + p.stages * p.stage_bytes + (2 * p.stages + 9) * 8 + 16; }

cudaError_t dsdb_configure() {
    cudaError_t e = cudaFuncSetAttribute(dsdb_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dsdb_strip4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(dsdb_strip_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
}

cudaError_t launch_dsdb(const DsDbParams& p, int grid, cudaStream_t stream) {
    if (p.strip > 0 && strip_four_issuers(p.rt.rpad_max, p.parts))
        return launch_pdl(dsdb_strip4_kernel, dim3(grid), dim3(kThreads4), dsdb_smem_bytes(p), stream, p);
    if (p.strip > 0) return launch_pdl(dsdb_strip_kernel, dim3(grid), dim3(kThreads), dsdb_smem_bytes(p), stream, p);
    return launch_pdl(dsdb_tile_kernel, dim3(grid), dim3(kThreads), dsdb_smem_bytes(p), stream, p);
}

cudaError_t launch_finalize_bwd1(const DsDbParams& p, int parts, int sms, cudaStream_t stream, bool pdl) {
    if (parts < kPartDs || parts > (kPartDs | kPartDb)) return cudaErrorInvalidValue;
    return launch_k(pdl, finalize_bwd1_kernel, dim3(2 * sms), dim3(256), 0, stream, p.dS_acc, p.dSq, p.m, p.ld,
                    p.acc_base, p.n, p.rt, p.dB, static_cast<int32_t>(parts), p.sl, p.nnb);
}

}  // namespace lora
