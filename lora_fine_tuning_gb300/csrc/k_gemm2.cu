// The layer's two dense contractions on CTA pairs (tcgen05 cta_group::2).
//
// Products:
//   forward   Y  = [X | S'] [W ; B_a]                (article section 4.1, ②)
//   backward  dX = dY W^T + D .* (dSq A_a^T)         (article section 4.1, ⑤)
// but each output tile is 256 rows x BN columns computed by a cluster of two
// CTAs: CTA rank r stages rows [256 i + 128 r, +128) of the A operand and
// half of the B operand's BN columns; the leader (rank 0) issues one
// tcgen05.mma M=256 that reads both CTAs' shared memory and writes both CTAs'
// TMEM (each holds its own 128 rows x BN columns).  Per CTA and 64-deep K
// block that is 16 KB of A and BN/2 x 128 B of B for 128 x BN x 64 MACs,
// instead of 16 KB + BN x 128 B for a single CTA: fewer bytes in flight
// per FLOP, so the same shared memory holds a deeper stage ring (6 stages
// of 32 KB) and covers more load latency.
//
// The rank-r branch stays a K-tail of the same loop.  The two 128-row halves
// of a tile may belong to different adapters; each distinct adapter then gets
// its own tail pass, in which the rows of the other half load zeros (a TMA box
// placed wholly outside the tensor).
//
// Roles per CTA: warp 0 TMA producer (both CTAs; the leader also posts the
// expected bytes of both halves on its barrier), warp 1 MMA issue (leader
// only) and TMEM allocation, warps 2-5 epilogue (both CTAs, own rows): the
// output goes through a swizzled shared-memory block and a TMA tensor store,
// so global writes are whole 128-byte lines.
//
// Every role walks the same runs (plan.h): whole tiles, and where a last wave
// of tiles would leave most pairs idle, first a stream-K part in which tiles
// are cut into runs of K stages spread evenly over the pairs.  The rank-r
// tail goes with the run that ends a tile's K loop.  A run that does not start
// its tile hands its fp32 sum to the run that does through a partial slot and
// a flag in the workspace.
#include "cluster.cuh"
#include "kernels.h"

namespace lora {

namespace {

constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kGroupPairs = 8;   // rasterisation: pair-rows per group
constexpr int kBK = 64;          // K depth of one pipeline stage (a multiple of 64: one 128-byte swizzle row)
constexpr int kKB = kBK / 64;    // 64-deep TMA boxes per operand and stage

template <bool kBwd, int BN>
struct Cfg {
    static constexpr int BNH = BN / 2;                        // B columns (fwd) / rows (bwd) per CTA
    static constexpr uint32_t kA = 128u * 128u * kKB;          // 128 rows x kBK bf16 (kKB boxes of 16 KB)
    static constexpr uint32_t kBox = static_cast<uint32_t>(BNH) * 128u;   // B: BNH x 64 bf16
    static constexpr uint32_t kB = kBox * kKB;
    static constexpr uint32_t kStage = kA + kB;
    static constexpr int kStages = (192 * 1024) / kStage > 8 ? 8 : (192 * 1024) / kStage;
    static constexpr uint32_t kStaging = 2u * 16384u;           // two 128 x 64 bf16 output buffers
    static constexpr bool kDouble = !kBwd || BN <= 128;       // two accumulator buffers fit in TMEM
    static constexpr uint32_t kBufCols = kBwd ? 2u * BN : static_cast<uint32_t>(BN);
};

struct PairTile {
    int mp, np;
};

struct Tail {
    int a[2];    // adapter of each pass (-1: none)
    int nb[2];   // kBK-deep blocks of each pass
    int total;
    int half_adapter[2];   // adapter of each 128-row half
};

__device__ __forceinline__ Tail tail_of(int mp, const GemmParams& p) {
    Tail t;
    const int t0 = 2 * mp, t1 = 2 * mp + 1;
    const int a0 = t0 < p.rt.n_tiles ? p.rt.tile_adapter[t0] : -1;
    const int a1 = t1 < p.rt.n_tiles ? p.rt.tile_adapter[t1] : -1;
    t.half_adapter[0] = a0;
    t.half_adapter[1] = a1;
    t.a[0] = a0 >= 0 ? a0 : a1;
    t.a[1] = (a0 >= 0 && a1 >= 0 && a1 != a0) ? a1 : -1;
    for (int i = 0; i < 2; ++i) t.nb[i] = t.a[i] >= 0 ? (p.rt.ad[t.a[i]].rank + kBK - 1) / kBK : 0;
    t.total = t.nb[0] + t.nb[1];
    return t;
}

template <int BN>
__device__ __forceinline__ PairTile pair_tile(int tile, const GemmParams& p) {
    const int n_mp = static_cast<int>((p.M + 255) / 256);
    const int n_np = static_cast<int>((p.N + BN - 1) / BN);
    const int per_group = kGroupPairs * n_np;
    const int group = tile / per_group;
    const int first = group * kGroupPairs;
    const int gm = min(n_mp - first, kGroupPairs);
    const int in_group = tile - group * per_group;
    return PairTile{first + in_group % gm, in_group / gm};
}

__device__ __forceinline__ RunWalk pair_runs(const GemmParams& p, int pair, int npairs, int nk, int total) {
    return run_walk(p.sk_tiles, pair, npairs, nk, total);
}

// 16 accumulator columns of this thread's row; with the branch, plus the second accumulator's where the
// keep bits say the element was kept.
template <int BN>
__device__ __forceinline__ void acc_chunk(uint32_t t1, uint32_t t2, int c, bool branch, const uint32_t (&keep)[BN / 32],
                                          uint32_t (&v)[16]) {
    tmem_ld16(t1 + c * 16, v);
    if (branch) {
        uint32_t u[16];
        tmem_ld16(t2 + c * 16, u);
        tmem_ld_wait();
        const uint32_t kb = keep[c >> 1] >> ((c & 1) * 16);
#pragma unroll
        for (int e = 0; e < 16; ++e)
            if ((kb >> e) & 1u) v[e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(u[e]));
    } else {
        tmem_ld_wait();
    }
}

// DoRA: column j of the output times g_j (columns past N read nothing; the store clips them).
__device__ __forceinline__ void col_scale_chunk(const GemmParams& p, int col0, float* f) {
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        const int64_t col = static_cast<int64_t>(col0) + e;
        f[e] *= col < p.N ? __ldg(p.col_scale + col) : 0.f;
    }
}

// One 128 x 64 bf16 block of the output (this thread's row: 32 packed words) through a 128B-swizzled
// staging buffer and a TMA store; the two buffers alternate.
__device__ __forceinline__ void store_block(const CUtensorMap& map, uint8_t* staging, int& sb, bool issuer, int er,
                                            const uint32_t* pk, int x, int y) {
    uint8_t* buf = staging + sb * 16384;
    // the store that last read this buffer (two blocks ago) must be done with it
    if (issuer) bulk_wait_read<1>();
    named_barrier(1, 128);
    const uint32_t rowbase = smem_u32(buf) + er * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)   // 16-byte chunk j of the row's 128 bytes
        sts128(rowbase + ((j ^ (er & 7)) << 4), make_uint4(pk[j * 4], pk[j * 4 + 1], pk[j * 4 + 2], pk[j * 4 + 3]));
    fence_proxy_async_smem();
    named_barrier(1, 128);
    if (issuer) {
        tma_store_2d(&map, buf, x, y);
        bulk_commit();
    }
    sb ^= 1;
}

template <bool kBwd, int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm2_kernel(const __grid_constant__ GemmParams p) {
    using C = Cfg<kBwd, BN>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    uint8_t* staging = smem + S * C::kStage;   // epilogue: output blocks on their way to a TMA store
    uint64_t* bars = reinterpret_cast<uint64_t*>(staging + C::kStaging);
    uint64_t* full = bars;            // leader's are used: both halves' bytes land here
    uint64_t* empty = bars + S;       // per CTA: released by the leader's multicast commit
    uint64_t* acc_full = bars + 2 * S;
    uint64_t* acc_empty = acc_full + 2;   // leader's: 128 arrivals from each CTA
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 256);
        }
        mbar_init(drain, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.mapA);
        tma_prefetch_desc(&p.mapB);
    }
    tc_fence_before();
    cluster_sync();   // barriers initialised and TMEM allocated in both CTAs
    tc_fence_after();
    // Programmatic dependent launch: wait for the previous kernel before touching what it may write.  With
    // early_loads the producer first streams the first tile's main-loop stages (operands no earlier kernel of
    // the call writes) and waits afterwards; the MMA thread touches no global memory, and the epilogue waits
    // before its first global access.
    const bool early = p.early_loads != 0;
    if (!early) pdl_wait();
    pdl_trigger();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx w{&abort_flag, p.ctl.status, p.ctl.wait_ns, (kBwd ? kKGemmBwd : kKGemmFwd) << 8};

    const int n_mp = static_cast<int>((p.M + 255) / 256);
    const int n_np = static_cast<int>((p.N + BN - 1) / BN);
    const int total = n_mp * n_np;
    const int pair = blockIdx.x >> 1;
    const int npairs = gridDim.x >> 1;
    const int nkb = (p.nkb + kKB - 1) / kKB;   // kBK-deep stages of the main loop (p.nkb counts 64-deep blocks)

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            bool waited = !early;
            bool first_run = true;
            RunWalk rw = pair_runs(p, pair, npairs, nkb, total);
            for (Run run; ok && rw.next(run); first_run = false) {
                const PairTile pt = pair_tile<BN>(run.tile, p);
                const int m0 = pt.mp * 256 + static_cast<int>(rank) * 128;
                const int n0 = pt.np * BN + static_cast<int>(rank) * C::BNH;
                const Tail tl = tail_of(pt.mp, p);
                const int my_adapter = tl.half_adapter[rank];
                const int ntail = run.kb1 == nkb ? tl.total : 0;
                for (int j = run.kb0; j < run.kb1 + ntail; ++j) {
                    // only the first ring's worth of main-loop stages of the first run go before the wait
                    if (!waited && (!first_run || j >= run.kb1 || issued >= S)) {
                        pdl_wait();
                        waited = true;
                    }
                    if (!mbar_wait_cl(&empty[s], ph ^ 1u, w, 1)) { ok = false; break; }
                    uint8_t* as = smem + s * C::kStage;
                    uint8_t* bs = as + C::kA;
                    if (leader) mbar_arrive_expect_tx(&full[s], 2u * C::kStage);
                    const uint32_t fb = peer_addr(smem_u32(&full[s]), 0);
                    // kKB boxes of 64 K per operand; a box past the end of K reads zeros
                    if (j < run.kb1) {
#pragma unroll
                        for (int q = 0; q < kKB; ++q) {
                            const int x = j * kBK + 64 * q;
                            tma_load_2d_pair(as + q * 16384, &p.mapA, fb, x, m0);
                            if (kBwd) {
                                tma_load_2d_pair(bs + q * C::kBox, &p.mapB, fb, x, n0);
                            } else {
#pragma unroll
                                for (int j = 0; j < C::BNH / 64; ++j)
                                    tma_load_2d_pair(bs + q * C::kBox + j * 8192, &p.mapB, fb, n0 + 64 * j, x);
                            }
                        }
                    } else {
                        const int t = j - run.kb1;
                        const int pass = t < tl.nb[0] ? 0 : 1;
                        const int tb = pass == 0 ? t : t - tl.nb[0];
                        const int a = tl.a[pass];
#pragma unroll
                        for (int q = 0; q < kKB; ++q) {
                            const int x = tb * kBK + 64 * q;
                            // rows of the other adapter's half read zeros (box wholly outside the tensor)
                            tma_load_2d_pair(as + q * 16384, &p.mapTA, fb, x, my_adapter == a ? m0 : -256);
                            if (kBwd) {
                                tma_load_2d_pair(bs + q * C::kBox, &p.mapTB[a], fb, x, n0);
                            } else {
#pragma unroll
                                for (int j = 0; j < C::BNH / 64; ++j)
                                    tma_load_2d_pair(bs + q * C::kBox + j * 8192, &p.mapTB[a], fb, n0 + 64 * j, x);
                            }
                        }
                    }
                    ++issued;
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
            }
            if (!waited) pdl_wait();
            if (!ok && leader) {
                const int64_t back = issued < S ? issued : S;
                for (int64_t i = issued - back; i < issued; ++i)
                    mbar_wait_cl_drain(&full[i % S], static_cast<uint32_t>((i / S) & 1), p.ctl.wait_ns);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t use = 0;
            const uint32_t idesc = make_idesc_bf16(256, BN, false, !kBwd);
            // operand descriptors of stage 0 at K step 0; stage s and K step ks (16 deep) only move the
            // start-address field (bytes / 16): by s * stage bytes, by the 64-deep box ks / 4, and
            // within it by 32 B (K-major) or 2048 B (MN-major B: 16 rows of 128 B) per step;
            // shared-memory addresses stay below 256 KB, so the 14-bit field never carries
            const uint32_t sbase = smem_u32(smem);
            const uint64_t a_desc0 = make_smem_desc(sbase, 16, 1024, kSw128);
            const uint64_t b_desc0 = kBwd ? make_smem_desc(sbase + C::kA, 16, 1024, kSw128)
                                          : make_smem_desc(sbase + C::kA, 8192, 1024, kSw128);
            constexpr uint64_t kBStep = kBwd ? 2u : 128u;
            const auto a_step = [](int ks) -> uint64_t { return (ks >> 2) * (16384u >> 4) + (ks & 3) * 2u; };
            const auto b_step = [](int ks) -> uint64_t { return (ks >> 2) * (C::kBox >> 4) + (ks & 3) * kBStep; };
            bool ok = true;
            RunWalk rw = pair_runs(p, pair, npairs, nkb, total);
            for (Run run; ok && rw.next(run);) {
                const PairTile pt = pair_tile<BN>(run.tile, p);
                const Tail tl = tail_of(pt.mp, p);
                const int ntail = run.kb1 == nkb ? tl.total : 0;
                const uint32_t b = C::kDouble ? (use & 1u) : 0u;
                const uint32_t empty_parity = C::kDouble ? (((use >> 1) & 1u) ^ 1u) : ((use & 1u) ^ 1u);
                if (!mbar_wait_cl(&acc_empty[b], empty_parity, w, 2)) break;
                tc_fence_after();
                const uint32_t acc1 = tmem + b * C::kBufCols;
                const uint32_t acc2 = acc1 + BN;
                for (int kb = run.kb0; kb < run.kb1; ++kb) {
                    if (!mbar_wait_cl(&full[s], ph, w, 3)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t so = static_cast<uint64_t>(s) * (C::kStage >> 4);
                    umma_bf16_pair(acc1, a_desc0 + so, b_desc0 + so, idesc, kb != run.kb0 ? 1u : 0u);
#pragma unroll
                    for (int ks = 1; ks < 4 * kKB; ++ks)
                        umma_bf16_pair(acc1, a_desc0 + so + a_step(ks), b_desc0 + so + b_step(ks), idesc, 1u);
                    umma_commit_pair(&empty[s], 3);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
                for (int t = 0; t < ntail && ok; ++t) {
                    if (!mbar_wait_cl(&full[s], ph, w, 3)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t so = static_cast<uint64_t>(s) * (C::kStage >> 4);
                    const int pass = t < tl.nb[0] ? 0 : 1;
                    const int tb = pass == 0 ? t : t - tl.nb[0];
                    const int left = p.rt.ad[tl.a[pass]].rank - tb * kBK;
                    const int nks = left >= kBK ? 4 * kKB : (left + 15) / 16;
                    for (int ks = 0; ks < nks; ++ks) {
                        if (kBwd)
                            umma_bf16_pair(acc2, a_desc0 + so + a_step(ks), b_desc0 + so + b_step(ks), idesc,
                                           (t | ks) != 0 ? 1u : 0u);
                        else
                            umma_bf16_pair(acc1, a_desc0 + so + a_step(ks), b_desc0 + so + b_step(ks), idesc, 1u);
                    }
                    umma_commit_pair(&empty[s], 3);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair(&acc_full[b], 3);
                ++use;
            }
            umma_commit_pair(drain, 1);
            mbar_wait_cl_drain(drain, 0, p.ctl.wait_ns);
        }
    } else {
        // Epilogue.  While the tile's MMAs run: the keep bits of this thread's row
        // (backward).  Then TMEM -> registers (-> mask, add) -> packed bf16 for the
        // whole 128 x BN tile, and the accumulator goes back to the MMA warp before
        // anything is stored.  Then 128B-swizzled staging blocks of 128 rows x 64
        // columns, one TMA store each (two staging buffers, so storing one block
        // overlaps filling the next).
        //
        // Split tiles: a run that does not start its tile stores its fp32 sum (with the masked branch term
        // when it holds the tail) to its pair's partial slot and raises the pair's flag.  The run that starts
        // the tile waits for the flags of the pairs holding the rest, adds their partials to its own
        // accumulator in pair order (the same order on every call), clears the slots and stores the tile.
        const int quad = warp & 3;
        const int er = quad * 32 + lane;   // row within this CTA's 128 rows (= TMEM lane)
        const bool issuer = warp == 2 && lane == 0;
        if (early) pdl_wait();   // before the keep bits, the column scale and the stores
        const PhiloxKeys keys = philox_keys(p.seed_lo, p.seed_hi);
        const int64_t U = static_cast<int64_t>(p.sk_tiles) * nkb;
        uint32_t use = 0;
        int sb = 0;
        if (issuer) tma_prefetch_desc(&p.mapOut);
        RunWalk rw = pair_runs(p, pair, npairs, nkb, total);
        for (Run run; rw.next(run);) {
            const PairTile pt = pair_tile<BN>(run.tile, p);
            const Tail tl = tail_of(pt.mp, p);
            const int m0 = pt.mp * 256 + static_cast<int>(rank) * 128;
            const int n0 = pt.np * BN;
            const int a = tl.half_adapter[rank];
            const bool has_tail = run.kb1 == nkb;
            const bool split = run.kb0 > 0 || !has_tail;
            const bool branch = kBwd && a >= 0 && has_tail;
            const int64_t row = static_cast<int64_t>(m0) + er;
            uint32_t keep[BN / 32];
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) keep[c] = 0u;
            if (branch && p.keep_bits != nullptr) {
                // the forward's keep bits: 32 columns per little-endian word (bit e of byte g = column 8g + e)
                if (row < p.M) {
                    const uint32_t* kw = reinterpret_cast<const uint32_t*>(p.keep_bits + row * (p.N >> 3) + (n0 >> 3));
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c)
                        if (n0 + c * 32 < p.N) keep[c] = __ldg(kw + c);
                }
            } else if (branch) {
                const uint32_t T = p.rt.ad[a].T;
#pragma unroll
                for (int c = 0; c < BN / 32; ++c) {
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const uint32_t grp = static_cast<uint32_t>((n0 + c * 32 + g * 8) >> 3);
                        keep[c] |= keep_byte(philox_10(static_cast<uint32_t>(row), grp, keys), T) << (8 * g);
                    }
                }
                // hand the regenerated decisions to the dA pass (whole 16-byte groups: N % 128 == 0)
                if (p.keep_out != nullptr && row < p.M) {
                    uint8_t* kw = p.keep_out + row * (p.N >> 3) + (n0 >> 3);
#pragma unroll
                    for (int c = 0; c < BN / 32; c += 4)
                        if (n0 + c * 32 < p.N) stg128(kw + c * 4, make_uint4(keep[c], keep[c + 1], keep[c + 2], keep[c + 3]));
                }
            }
            // a split tile's first run: the pairs after this one whose first runs hold the rest of the tile
            const bool closing = split && run.kb0 == 0;
            int parts = 0;
            bool flags_ok = true;
            if (closing) {
                const int64_t tile_end = static_cast<int64_t>(run.tile + 1) * nkb;
                while (parts < kSkMaxParts && sk_unit_begin(pair + 1 + parts, U, npairs) < tile_end) ++parts;
                if (issuer) {
                    if (sk_unit_begin(pair + 1 + parts, U, npairs) < tile_end) {   // more runs than slots: refuse
                        abort_flag = 1;
                        if (p.ctl.status) atomicCAS(p.ctl.status, 0, w.code | 6);
                        flags_ok = false;
                    }
                    for (int j = 0; j < parts && flags_ok; ++j)
                        flags_ok = flag_wait(p.sk_flag + (pair + 1 + j) * 2 + rank, w, 5);
                }
            }
            const uint32_t b = C::kDouble ? (use & 1u) : 0u;
            const uint32_t full_parity = C::kDouble ? ((use >> 1) & 1u) : (use & 1u);
            const bool ok = mbar_wait_cl(&acc_full[b], full_parity, w, 4);
            // every epilogue thread has finished its (bounded) wait; all four warps
            // leave together if any of them timed out or the CTA is aborting
            if (named_barrier_or(1, 128, !ok || !flags_ok || abort_flag != 0)) break;
            tc_fence_after();
            const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
            const uint32_t t1 = tmem + lane_off + b * C::kBufCols;
            const uint32_t t2 = t1 + BN;
            if (split && !closing) {
                // the rest of a split tile: fp32 partial to this pair's slot, 16-byte pieces laid out so that a
                // warp's stores of one piece index cover 512 contiguous bytes
                float* slot = p.sk_part + (static_cast<size_t>(pair) * 2 + rank) * kSkSlotFloats;
#pragma unroll
                for (int c = 0; c < BN / 16; ++c) {
                    uint32_t v[16];
                    acc_chunk<BN>(t1, t2, c, branch, keep, v);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st_f4(slot + ((c * 4 + q) * 128 + er) * 4, __uint_as_float(v[4 * q]),
                              __uint_as_float(v[4 * q + 1]), __uint_as_float(v[4 * q + 2]),
                              __uint_as_float(v[4 * q + 3]));
                }
                tc_fence_before();
                mbar_arrive_cluster(peer_addr(smem_u32(&acc_empty[b]), 0));
                __threadfence();            // this thread's partial is visible at gpu scope ...
                named_barrier(1, 128);      // ... and so is every other thread's
                if (issuer) st_release_gpu(p.sk_flag + pair * 2 + rank, 1u);
            } else if (closing) {
                // own accumulator + the other runs' partials, in pair order; 64 columns at a time
#pragma unroll 1
                for (int j = 0; j < parts; ++j) (void)ld_acquire_gpu(p.sk_flag + (pair + 1 + j) * 2 + rank);
#pragma unroll
                for (int blk = 0; blk < BN / 64; ++blk) {
                    const float* src0 = p.sk_part + (static_cast<size_t>(pair + 1) * 2 + rank) * kSkSlotFloats;
                    float4 pf[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) pf[i] = ld_l2_f4(src0 + ((blk * 16 + i) * 128 + er) * 4);
                    float acc[64];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        uint32_t v[16];
                        tmem_ld16(t1 + (blk * 4 + c4) * 16, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 16; ++e) acc[c4 * 16 + e] = __uint_as_float(v[e]);
                    }
                    if (blk == BN / 64 - 1) {
                        // all of this tile's TMEM reads are done: hand the accumulator back
                        tc_fence_before();
                        mbar_arrive_cluster(peer_addr(smem_u32(&acc_empty[b]), 0));
                    }
                    for (int j = 0; j < parts; ++j) {
                        const float* src = p.sk_part + (static_cast<size_t>(pair + 1 + j) * 2 + rank) * kSkSlotFloats;
                        if (j > 0) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) pf[i] = ld_l2_f4(src + ((blk * 16 + i) * 128 + er) * 4);
                        }
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            acc[4 * i] += pf[i].x;
                            acc[4 * i + 1] += pf[i].y;
                            acc[4 * i + 2] += pf[i].z;
                            acc[4 * i + 3] += pf[i].w;
                            st_zero_f4(const_cast<float*>(src) + ((blk * 16 + i) * 128 + er) * 4);
                        }
                    }
                    uint32_t pk[32];
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        if (!kBwd && p.col_scale != nullptr) col_scale_chunk(p, n0 + blk * 64 + c4 * 16, acc + c4 * 16);
#pragma unroll
                        for (int e = 0; e < 8; ++e) pk[c4 * 8 + e] = pack_bf16x2(acc[c4 * 16 + 2 * e], acc[c4 * 16 + 2 * e + 1]);
                    }
                    store_block(p.mapOut, staging, sb, issuer, er, pk, n0 + blk * 64, m0);
                }
                if (issuer)
                    for (int j = 0; j < parts; ++j) p.sk_flag[(pair + 1 + j) * 2 + rank] = 0u;
            } else {
                uint32_t packed[BN / 2];
#pragma unroll
                for (int c = 0; c < BN / 16; ++c) {
                    uint32_t v[16];
                    acc_chunk<BN>(t1, t2, c, branch, keep, v);
                    float f[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(v[e]);
                    if (!kBwd && p.col_scale != nullptr) col_scale_chunk(p, n0 + c * 16, f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) packed[c * 8 + e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
                }
                // all of this tile's TMEM reads are done: hand the accumulator back
                tc_fence_before();
                mbar_arrive_cluster(peer_addr(smem_u32(&acc_empty[b]), 0));
#pragma unroll
                for (int blk = 0; blk < BN / 64; ++blk) store_block(p.mapOut, staging, sb, issuer, er, packed + blk * 32, n0 + blk * 64, m0);
            }
            ++use;
        }
        if (issuer) bulk_wait_all();
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();   // the leader's MMAs and both epilogues are finished
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

template <bool kBwd, int BN>
size_t smem_bytes() {
    using C = Cfg<kBwd, BN>;
    return 1024 + C::kStages * C::kStage + C::kStaging + (2 * C::kStages + 5) * 8 + 16;
}

}  // namespace

cudaError_t gemm2_configure() {
    cudaError_t e = cudaFuncSetAttribute(gemm2_kernel<false, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_bytes<false, 256>()));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gemm2_kernel<true, 256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem_bytes<true, 256>()));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemm2_kernel<true, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(smem_bytes<true, 128>()));
}

GemmSched plan_gemm2(const GemmParams& p, bool bwd, int bn, int sms, bool allow_split) {
    const bool single_acc = bwd ? !Cfg<true, 256>::kDouble && bn == 256 : false;
    return gemm_schedule(p.M, p.N, bn, (p.nkb + kKB - 1) / kKB, sms / 2, allow_split, single_acc);
}

cudaError_t launch_gemm2(const GemmParams& p, bool bwd, int bn, int pairs, cudaStream_t stream) {
    const dim3 grid(2 * pairs);
    if (!bwd) return launch_pdl(gemm2_kernel<false, 256>, grid, dim3(kThreads), smem_bytes<false, 256>(), stream, p);
    if (bn == 128) return launch_pdl(gemm2_kernel<true, 128>, grid, dim3(kThreads), smem_bytes<true, 128>(), stream, p);
    return launch_pdl(gemm2_kernel<true, 256>, grid, dim3(kThreads), smem_bytes<true, 256>(), stream, p);
}

}  // namespace lora
