// Down-projection with fused dropout: S_acc += (X .* D) A_a, per 128-row tile.
//
// LoRAFusion notes (papers.chlience.com), section 5 "FusedLoRA": dropout and
// the down-projection are one pass so the full-size X is read once; the
// article (juhe.plus) section 4.1 lists it as forward step ①.  Here:
//  - warp 0 streams X tiles (128 rows x 128 features: two TMA boxes, 128B
//    swizzle) and the matching 128-row block of A_a into a ring of
//    shared-memory stages;
//  - warps 2..9 regenerate the keep mask with Philox4x32-10 and zero the
//    dropped elements in place (16 bytes = 8 features = one Philox call per
//    access), then hand the stage to the MMA warp.  They form two groups of
//    four warps that take alternate stages, and a thread owns one whole row
//    of its stage: sixteen Philox calls per thread and stage, eight at a
//    time, with the counter's row word shared.  The first eight are computed
//    before the wait on the stage's data;
//  - warp 1 issues tcgen05.mma (M = 128 tokens, N = rank, K = 128 per stage)
//    into TMEM, one accumulator buffer per mask group;
//  - at the end of each tile range the group that owns the range's buffer
//    reads TMEM and adds the fp32 partial into S_acc with vector reductions
//    (ranges of one tile may be split over CTAs: units are spread evenly,
//    stream-K style).
// finalize_s then applies alpha/(1-p), writes S' in bf16 and clears S_acc,
// which starts every call at zero.
#include "common.cuh"
#include "kernels.h"

namespace lora {

namespace {

// Warps 2.. mask (and run the epilogue) in G groups of four; warp 0 is the TMA producer, warp 1 the MMA issuer.
constexpr int kGroupThreads = 128;                // a mask group: four warps, one per TMEM lane quadrant
constexpr int threads_of(int groups) { return 64 + kGroupThreads * groups; }
constexpr int kChunks = 16;                        // 16-byte chunks (8 features) of a row per stage: two 64-feature boxes
constexpr int kBatch = 8;                          // Philox calls computed before their chunks are masked
static_assert(kGroupThreads == 128, "a group is four warps: one thread per tile row, one warp per TMEM lane quadrant");
constexpr uint32_t kXBytes = 2u * 128u * 128u;   // 128 rows x 128 bf16 (two boxes); then 128 rows of A (rpad_max x 2 B each)

// The sixteen keep-bit bytes of a row's k-block (byte cc = chunk cc) to the caller's buffer: one 16-byte
// store when k is a multiple of 128, else byte by byte up to k.
__device__ __forceinline__ void store_row_bits(uint8_t* dst, uint4 v, int kb, int64_t k) {
    if ((k & 127) == 0) {
        *reinterpret_cast<uint4*>(dst) = v;
    } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < kChunks; ++i)
            if ((static_cast<int64_t>(kb) * kChunks + i) * 8 < k) dst[i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
    }
}

// Zeroes the dropped elements of one thread's row of a stage (16 chunks; the first kBatch keep masks come
// in `km`, computed before the data arrived), and with kBits also writes the row's keep bits.
template <bool kHalf, bool kBits>
__device__ __forceinline__ void apply_row(uint32_t xrow, int row, const PhiloxRow& prow, uint32_t g0,
                                          const PhiloxKeys& keys, const KeepForm& kf, uint4 (&km)[kBatch],
                                          uint8_t* bits, int kb, int64_t k) {
    uint32_t kw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int c0 = 0; c0 < kChunks; c0 += kBatch) {
        if (c0 > 0) {
#pragma unroll
            for (int i = 0; i < kBatch; ++i) km[i] = keep_chunk_mask<kHalf>(prow, g0 + c0 + i, keys, kf);
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int cc = c0 + i;                  // chunk of the row: box cc / 8, chunk cc % 8
            const uint32_t addr = xrow + (cc >> 3) * 16384 + (((cc & 7) ^ (row & 7)) << 4);
            sts128(addr, and4(lds128(addr), km[i]));
            if (kBits) kw[cc >> 2] |= chunk_mask_bits(km[i]) << (8 * (cc & 3));
        }
    }
    if (kBits) store_row_bits(bits, make_uint4(kw[0], kw[1], kw[2], kw[3]), kb, k);
}

// G mask groups take the ring's stages in turn (S % G == 0).
template <int G>
__global__ void __launch_bounds__(threads_of(G), 1) down_proj_kernel(const __grid_constant__ DownParams p) {
    constexpr int kGroups = G;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const int S = p.stages;
    if (S < kGroups || S % kGroups != 0) {
        // every stage must belong to one mask group (the host rounds the ring to a multiple of kGroups)
        if (threadIdx.x == 0 && p.ctl.status) atomicCAS(p.ctl.status, 0, (kKDown << 8) | 0xFF);
        return;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * p.stage_bytes);
    uint64_t* full = bars;
    uint64_t* masked = bars + S;
    uint64_t* empty = bars + 2 * S;
    uint64_t* acc_full = bars + 3 * S;
    uint64_t* acc_empty = acc_full + kGroups;
    uint64_t* drain = acc_empty + kGroups;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rpad_max = p.rt.rpad_max;
    // one accumulator buffer per mask group (see the epilogue)
    uint32_t tmem_cols = 32;
    while (tmem_cols < static_cast<uint32_t>(kGroups * rpad_max)) tmem_cols <<= 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&masked[s], kGroupThreads);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < kGroups; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], kGroupThreads);
        }
        mbar_init(drain, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) tma_prefetch_desc(&p.mapX);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx w{&abort_flag, p.ctl.status, p.ctl.wait_ns, kKDown << 8};

    const int64_t U = p.units;
    const int64_t u0 = U * blockIdx.x / gridDim.x;
    const int64_t u1 = U * (blockIdx.x + 1) / gridDim.x;

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            TileBlockIter it(u0, p.nkb, p.rt);
            for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
                const int kb = it.blk;
                const int tile = it.tile;
                const int a = it.a;
                const int rpad = p.rt.ad[a].rpad;
                if (!mbar_wait(&empty[s], ph ^ 1u, w, 1)) { ok = false; break; }
                uint8_t* xs = smem + s * p.stage_bytes;
                mbar_arrive_expect_tx(&full[s], kXBytes + 256u * static_cast<uint32_t>(rpad));
                tma_load_2d(xs, &p.mapX, &full[s], kb * 128, tile * kTileM);
                tma_load_2d(xs + 16384, &p.mapX, &full[s], kb * 128 + 64, tile * kTileM);
                tma_load_2d(xs + kXBytes, &p.mapA[a], &full[s], 0, kb * 128);
                if (rpad > 64) tma_load_2d(xs + kXBytes + 16384, &p.mapA[a], &full[s], 64, kb * 128);
                ++issued;
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            if (!ok) {
                // Let every copy still in flight land before the CTA can exit.
                const int64_t back = issued < S ? issued : S;
                for (int64_t i = issued - back; i < issued; ++i)
                    mbar_wait_drain(&full[i % S], static_cast<uint32_t>((i / S) & 1), p.ctl.wait_ns);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t use = 0;
            // Operand descriptors of stage 0, built once (the A_a block's when the padded
            // rank changes); an MMA only moves the start-address field (bytes / 16).
            const uint32_t sbase = smem_u32(smem);
            const uint64_t x_d0 = make_smem_desc(sbase, 16, 1024, kSw128);   // X tile, K-major
            int cur_rpad = -1;
            uint32_t idesc = 0, rb = 0;
            uint64_t a_d0 = 0;
            TileBlockIter it(u0, p.nkb, p.rt);
            for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
                const int kb = it.blk;
                const int rpad = p.rt.ad[it.a].rpad;
                if (rpad != cur_rpad) {
                    cur_rpad = rpad;
                    idesc = make_idesc_bf16(128, rpad, false, true);
                    rb = rank_row_bytes(rpad);
                    a_d0 = make_smem_desc(sbase + kXBytes, 16384, 8 * rb, rank_swizzle(rpad));   // A_a rows, MN-major
                }
                const bool first = (u == u0) || kb == 0;
                const bool last = (u == u1 - 1) || kb == p.nkb - 1;
                const uint32_t b = use % kGroups;
                if (first) {
                    if (!mbar_wait(&acc_empty[b], ((use / kGroups) & 1u) ^ 1u, w, 2)) break;
                    tc_fence_after();
                }
                if (!mbar_wait(&masked[s], ph, w, 3)) break;
                tc_fence_after();
                const uint64_t so = (static_cast<uint32_t>(s) * p.stage_bytes) >> 4;
                const uint32_t d = tmem + b * static_cast<uint32_t>(rpad_max);
                // 16 features per step: 32 B of the X row in box ks / 4, 16 rows (16 * rb B) of A_a
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint64_t xo = static_cast<uint64_t>(ks >> 2) * 1024u + static_cast<uint64_t>(ks & 3) * 2u;
                    umma_bf16(d, x_d0 + so + xo, a_d0 + so + static_cast<uint64_t>(ks) * rb, idesc,
                              (first && ks == 0) ? 0u : 1u);
                }
                umma_commit(&empty[s]);
                if (last) {
                    umma_commit(&acc_full[b]);
                    ++use;
                }
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            // Everything issued must complete before TMEM is released.
            umma_commit(drain);
            mbar_wait_drain(drain, 0, p.ctl.wait_ns);
        }
    } else {
        // mask warps: group g takes the units u0 + g, u0 + g + kGroups, ...; in
        // it thread -> row covers the row's kChunks 16-byte chunks, so the
        // Philox counter word is the row for all of them.  Each group also
        // runs the epilogue of every kGroups-th tile range (TMEM lane quadrant
        // = warp % 4; each group has one warp per quadrant).
        const int mt = threadIdx.x - 64;
        const int group = mt / kGroupThreads;
        const int row = mt & 127;
        const int quad = warp & 3;
        const PhiloxKeys keys = philox_keys(p.seed_lo, p.seed_hi);
        uint32_t prow_t = 0xFFFFFFFFu;   // row whose Philox words are in prow
        PhiloxRow prow{};
        int s = 0;
        uint32_t ph = 0;
        uint32_t use = 0;
        int turn = 0;                    // whose unit this is: the group with turn == group
        TileBlockIter it(u0, p.nkb, p.rt);
        for (int64_t u = u0; u < u1; ++u, it.next(p.rt)) {
            const int kb = it.blk;
            const bool last = (u == u1 - 1) || kb == p.nkb - 1;
            const bool mine = turn == group;
            if (++turn == kGroups) turn = 0;
            const int tile = it.tile;
            const int a = it.a;
            if (mine) {
                const uint32_t T = p.rt.ad[a].T;
                const int64_t t = static_cast<int64_t>(tile) * kTileM + row;
                // The first batch of keep masks depends only on (seed, row, feature): it is computed before
                // the wait on the stage's data, so that the Philox arithmetic overlaps the TMA load.
                uint4 km[kBatch];
                const KeepForm kf = keep_form(T);
                const uint32_t g0 = static_cast<uint32_t>(kb * kChunks);
                if (T != 0u) {
                    if (static_cast<uint32_t>(t) != prow_t) {
                        prow_t = static_cast<uint32_t>(t);
                        prow = philox_row(prow_t, keys);
                    }
                    if (kf.half) {
#pragma unroll
                        for (int i = 0; i < kBatch; ++i) km[i] = keep_chunk_mask<true>(prow, g0 + i, keys, kf);
                    } else {
#pragma unroll
                        for (int i = 0; i < kBatch; ++i) km[i] = keep_chunk_mask<false>(prow, g0 + i, keys, kf);
                    }
                }
                bool ok = mbar_wait(&full[s], ph, w, 4);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                if (T != 0u) {
                    const uint32_t xrow = smem_u32(smem + s * p.stage_bytes) + row * 128;
                    // the keep bits are packed only when the caller keeps them (it costs a quarter of the
                    // mask arithmetic)
                    uint8_t* bits = (p.mask_bits != nullptr && t < p.m)
                                        ? p.mask_bits + t * (p.k >> 3) + static_cast<int64_t>(kb) * kChunks
                                        : nullptr;
                    if (bits == nullptr) {
                        if (kf.half) apply_row<true, false>(xrow, row, prow, g0, keys, kf, km, nullptr, 0, 0);
                        else apply_row<false, false>(xrow, row, prow, g0, keys, kf, km, nullptr, 0, 0);
                    } else {
                        if (kf.half) apply_row<true, true>(xrow, row, prow, g0, keys, kf, km, bits, kb, p.k);
                        else apply_row<false, true>(xrow, row, prow, g0, keys, kf, km, bits, kb, p.k);
                    }
                } else if (p.mask_bits != nullptr && t < p.m) {
                    // p = 0 keeps everything: all bits set
                    uint8_t* bits = p.mask_bits + t * (p.k >> 3) + static_cast<int64_t>(kb) * kChunks;
                    store_row_bits(bits, make_uint4(~0u, ~0u, ~0u, ~0u), kb, p.k);
                }
                fence_proxy_async_smem();
                mbar_arrive(&masked[s]);
            }
            // The epilogue of tile range e is run by group e % kGroups, which is also the TMEM buffer the
            // range accumulated in: each buffer is waited on by one group only, in order, so a parity wait
            // never meets a phase two behind, whatever the lengths of the ranges.
            const uint32_t b = use % kGroups;
            if (last && b == static_cast<uint32_t>(group)) {
                const bool ok = mbar_wait(&acc_full[b], (use / kGroups) & 1u, w, 5);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                tc_fence_after();
                const AdapterDev ad = p.rt.ad[a];
                const int64_t orow = static_cast<int64_t>(tile) * kTileM + quad * 32 + lane;
                const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + b * static_cast<uint32_t>(rpad_max);
                // deterministic mode: this CTA's partial of active tile it.slot goes to slot it.slot + CTA
                float* const out = p.sl.base
                                       ? p.sl.base + ((static_cast<int64_t>(it.slot) + blockIdx.x) * 128 + quad * 32 + lane) * p.sl.ld
                                       : p.S_acc + orow * p.ld;
                for (int c0 = 0; c0 < ad.rpad; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(taddr + c0, v);
                    tmem_ld_wait();
                    if (orow < p.m) {
                        float* dst = out + c0;
#pragma unroll
                        for (int q = 0; q < 16; q += 4) {
                            if (c0 + q >= ad.rank) continue;
                            if (p.sl.base)
                                st_f4(dst + q, __uint_as_float(v[q]), __uint_as_float(v[q + 1]), __uint_as_float(v[q + 2]),
                                      __uint_as_float(v[q + 3]));
                            else
                                red_add_v4(dst + q, __uint_as_float(v[q]), __uint_as_float(v[q + 1]),
                                           __uint_as_float(v[q + 2]), __uint_as_float(v[q + 3]));
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&acc_empty[b]);
            }
            if (last) ++use;
            if (++s == S) { s = 0; ph ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

// S'[t, c] = bf16(alpha_a / (1 - p_a) * S_acc[t, c]) for c < r_a, 0 for
// r_a <= c < ld, on rows of tiles that have an adapter; S_acc is cleared.  In
// deterministic mode (sl.base set) the row's slots are added in CTA order instead.
__global__ void __launch_bounds__(256, 4) finalize_s_kernel(float* __restrict__ acc, uint16_t* __restrict__ out, int64_t m, int32_t ld,
                                  const __grid_constant__ Routing rt, const Slots sl, int32_t nkb) {
    __shared__ RowRouting sr;
    load_row_routing(sr, rt);   // parameters only: before the wait on the previous kernel
    pdl_wait();
    pdl_trigger();
    // m * ld / 8 stays below 2^31: 32-bit index arithmetic
    const uint32_t g8 = static_cast<uint32_t>(ld / 8);
    const uint32_t total = static_cast<uint32_t>(m) * g8;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const uint32_t t = i / g8;
        const int c0 = static_cast<int>(i - t * g8) * 8;
        const int a = sr.owner[t >> 7];
        if (a < 0) continue;
        if (sl.base == nullptr) {
            finish_row(acc + static_cast<int64_t>(t) * ld + c0, out + static_cast<int64_t>(t) * ld + c0,
                       sr.rank[a] - c0, 8, sr.scale[a]);
            continue;
        }
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = 0.f;
        const int64_t item = sr.active[t >> 7];
        if (c0 < sr.rank[a]) slot_sum8(sl, item, item * nkb, (item + 1) * nkb, static_cast<int>(t & 127), c0, v);
        store_row8(out + static_cast<int64_t>(t) * ld + c0, v, sr.rank[a] - c0, sr.scale[a]);
    }
}

}  // namespace

size_t down_smem_bytes(const DownParams& p) {
    return 1024 + static_cast<size_t>(p.stages) * p.stage_bytes + (3 * p.stages + 2 * p.groups + 1) * 8 + 16;
}

cudaError_t down_configure() {
    cudaError_t e = cudaFuncSetAttribute(down_proj_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(down_proj_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(down_proj_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    return e;
}

cudaError_t launch_down(const DownParams& p, int grid, cudaStream_t stream) {
    if (p.groups == 4) return launch_pdl(down_proj_kernel<4>, dim3(grid), dim3(threads_of(4)), down_smem_bytes(p), stream, p);
    if (p.groups == 3) return launch_pdl(down_proj_kernel<3>, dim3(grid), dim3(threads_of(3)), down_smem_bytes(p), stream, p);
    if (p.groups == 2) return launch_pdl(down_proj_kernel<2>, dim3(grid), dim3(threads_of(2)), down_smem_bytes(p), stream, p);
    return cudaErrorInvalidValue;
}

cudaError_t launch_finalize_s(const DownParams& p, int sms, cudaStream_t stream) {
    return launch_pdl(finalize_s_kernel, dim3(2 * sms), dim3(256), 0, stream, p.S_acc, p.S_out, p.m, p.ld, p.rt, p.sl,
                      p.nkb);
}

}  // namespace lora
