// dA_a = X_hat^T dS for each adapter, with the keep mask regenerated from the seed.
//
// The article (juhe.plus) section 4.1 numbers the backward kernels ③ and ⑤;
// the gradient of A is the one the list leaves out, and the definition gives
// it: dA = X_hat^T dS = (X .* D)^T (q dS) = (X .* D)^T dSq.
// Each unit is (adapter a, 128-feature block, one of a's 128-row tiles): two
// TMA boxes of X (128 tokens x 64 features, 128B swizzle) plus the tile's dSq
// rows.  Warps 2..9 zero the dropped X elements in shared memory (Philox,
// exactly as the forward) in two groups of four warps that take alternate
// stages, a thread one token row of its stage (sixteen independent Philox
// calls, eight at a time), warp 1 issues tcgen05.mma with both operands
// MN-major (M = 128 features, N = rank, K = 128 tokens) accumulating over a
// CTA's run of tiles of one (adapter, feature block), and the run's partial is
// added into the adapter's fp32 accumulator with vector reductions.
// finalize_da then writes dA in bf16 and clears the accumulators and dSq
// (dA is dSq's last reader), so the workspace ends the call all zeros.
#include "common.cuh"
#include "kernels.h"

namespace lora {

namespace {

// Warps 2.. mask (and run the epilogue) in G groups of four; warp 0 is the TMA producer, warp 1 the MMA issuer.
constexpr int kGroupThreads = 128;                // a mask group: four warps, one per TMEM lane quadrant
constexpr int threads_of(int groups) { return 64 + kGroupThreads * groups; }
constexpr int kChunks = 16;                        // 16-byte chunks of a token row (two 64-feature boxes)
constexpr int kBatch = 8;                          // Philox calls computed before their chunks are masked
static_assert(kGroupThreads == 128, "a group is four warps: one thread per token row, one warp per TMEM lane quadrant");
constexpr uint32_t kXBytes = 2u * 128u * 128u;   // 128 tokens x 128 features

struct DaUnit {
    int a, fb, ti, tile, n_a;
};

__device__ __forceinline__ DaUnit da_unit(int64_t u, const DaParams& p) {
    int a = 0;
    while (a + 1 < p.rt.n_adapters && p.unit_begin[a + 1] <= u) ++a;
    const int n_a = p.rt.adapter_begin[a + 1] - p.rt.adapter_begin[a];
    const int64_t r = u - p.unit_begin[a];
    DaUnit d;
    d.a = a;
    d.n_a = n_a;
    d.fb = static_cast<int>(r / n_a);
    d.ti = static_cast<int>(r % n_a);
    d.tile = p.rt.active_tiles[p.rt.adapter_begin[a] + d.ti];
    return d;
}

// The unit after d in the order of da_unit (tile fastest, then feature block,
// then adapter), without a division; adapters without tiles have no units.
__device__ __forceinline__ void da_next(DaUnit& d, const DaParams& p) {
    if (++d.ti == d.n_a) {
        d.ti = 0;
        if (++d.fb == p.nfb) {
            d.fb = 0;
            do {
                ++d.a;
            } while (d.a < p.rt.n_adapters && p.rt.adapter_begin[d.a + 1] == p.rt.adapter_begin[d.a]);
            if (d.a >= p.rt.n_adapters) return;   // past the last unit
            d.n_a = p.rt.adapter_begin[d.a + 1] - p.rt.adapter_begin[d.a];
        }
    }
    d.tile = p.rt.active_tiles[p.rt.adapter_begin[d.a] + d.ti];
}

// G mask groups take the ring's stages in turn (S % G == 0).
template <int G>
__global__ void __launch_bounds__(threads_of(G), 1) da_kernel(const __grid_constant__ DaParams p) {
    constexpr int kGroups = G;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    const int S = p.stages;
    if (S < kGroups || S % kGroups != 0) {
        // every stage must belong to one mask group (the host rounds the ring to a multiple of kGroups)
        if (threadIdx.x == 0 && p.ctl.status) atomicCAS(p.ctl.status, 0, (kKDa << 8) | 0xFF);
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
            mbar_init(&acc_empty[b], 128);
        }
        mbar_init(drain, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.mapX);
        if (p.use_bits) tma_prefetch_desc(&p.mapBits);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();
    pdl_trigger();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx w{&abort_flag, p.ctl.status, p.ctl.wait_ns, kKDa << 8};

    const int64_t U = p.units;
    const int64_t u0 = U * blockIdx.x / gridDim.x;
    const int64_t u1 = U * (blockIdx.x + 1) / gridDim.x;

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            DaUnit d = da_unit(u0, p);
            for (int64_t u = u0; u < u1; ++u, da_next(d, p)) {
                const int rpad = p.rt.ad[d.a].rpad;
                if (!mbar_wait(&empty[s], ph ^ 1u, w, 1)) { ok = false; break; }
                uint8_t* st = smem + s * p.stage_bytes;
                mbar_arrive_expect_tx(&full[s], kXBytes + 256u * static_cast<uint32_t>(rpad) + (p.use_bits ? 2048u : 0u));
                if (p.use_bits) tma_load_2d(st + p.off_bits, &p.mapBits, &full[s], d.fb * 16, d.tile * kTileM);
                tma_load_2d(st, &p.mapX, &full[s], d.fb * 128, d.tile * kTileM);
                tma_load_2d(st + 16384, &p.mapX, &full[s], d.fb * 128 + 64, d.tile * kTileM);
                tma_load_2d(st + p.off_d, &p.mapD[d.a], &full[s], 0, d.tile * kTileM);
                if (rpad > 64) tma_load_2d(st + p.off_d + 16384, &p.mapD[d.a], &full[s], 64, d.tile * kTileM);
                ++issued;
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            if (!ok) {
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
            // Operand descriptors of stage 0, built once (dSq's when the padded rank
            // changes); an MMA only moves the start-address field (bytes / 16).
            const uint32_t sbase = smem_u32(smem);
            const uint64_t x_d0 = make_smem_desc(sbase, 16384, 1024, kSw128);   // X^T, MN-major (two 64-wide atoms)
            int cur_rpad = -1;
            uint32_t idesc = 0, rb = 0;
            uint64_t d_d0 = 0;
            DaUnit d = da_unit(u0, p);
            for (int64_t u = u0; u < u1; ++u, da_next(d, p)) {
                const int rpad = p.rt.ad[d.a].rpad;
                if (rpad != cur_rpad) {
                    cur_rpad = rpad;
                    idesc = make_idesc_bf16(128, rpad, true, true);
                    rb = rank_row_bytes(rpad);
                    d_d0 = make_smem_desc(sbase + p.off_d, 16384, 8u * rb, rank_swizzle(rpad));   // dSq, MN-major
                }
                const bool first = (u == u0) || d.ti == 0;
                const bool last = (u == u1 - 1) || d.ti == d.n_a - 1;
                const uint32_t b = use % kGroups;
                if (first) {
                    if (!mbar_wait(&acc_empty[b], ((use / kGroups) & 1u) ^ 1u, w, 2)) break;
                    tc_fence_after();
                }
                if (!mbar_wait(&masked[s], ph, w, 3)) break;
                tc_fence_after();
                const uint64_t so = (static_cast<uint32_t>(s) * p.stage_bytes) >> 4;
                const uint32_t dacc = tmem + b * static_cast<uint32_t>(rpad_max);
                // 16 tokens per step: 2048 B of X (16 rows of 128 B), 16 * rb B of dSq
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    umma_bf16(dacc, x_d0 + so + ks * 128u, d_d0 + so + static_cast<uint64_t>(ks) * rb, idesc,
                              (first && ks == 0) ? 0u : 1u);
                umma_commit(&empty[s]);
                if (last) {
                    umma_commit(&acc_full[b]);
                    ++use;
                }
                if (++s == S) { s = 0; ph ^= 1u; }
            }
            umma_commit(drain);
            mbar_wait_drain(drain, 0, p.ctl.wait_ns);
        }
    } else {
        // mask warps: group g takes the units u0 + g, u0 + g + kGroups, ...; in
        // it thread -> token row covers the row's 16 chunks (8 per 64-feature
        // box).  Each group also runs the epilogue of every kGroups-th run
        // (TMEM lane quadrant = warp % 4; each group has one warp per quadrant).
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
        DaUnit d = da_unit(u0, p);
        for (int64_t u = u0; u < u1; ++u, da_next(d, p)) {
            const bool last = (u == u1 - 1) || d.ti == d.n_a - 1;
            const bool mine = turn == group;
            if (++turn == kGroups) turn = 0;
            const AdapterDev ad = p.rt.ad[d.a];
            if (mine) {
                const bool regen = ad.T != 0u && !p.use_bits;
                const uint32_t t = static_cast<uint32_t>(static_cast<int64_t>(d.tile) * kTileM + row);
                const uint32_t g0 = static_cast<uint32_t>(d.fb * 16);
                const KeepForm kf = keep_form(ad.T);
                // The first batch of keep masks depends only on (seed, row, feature): it is computed before
                // the wait on the stage's data, so that the Philox arithmetic overlaps the TMA load.
                uint4 km[kBatch];
                if (regen) {
                    if (t != prow_t) {
                        prow_t = t;
                        prow = philox_row(t, keys);
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
                // bits handed over by the dX GEMM live in the workspace: zero them once they are in shared memory
                if (p.bits_clear != nullptr && t < p.m)
                    stg128(p.bits_clear + static_cast<int64_t>(t) * (p.k >> 3) + static_cast<int64_t>(d.fb) * 16,
                           make_uint4(0u, 0u, 0u, 0u));
                if (ad.T != 0u && p.use_bits) {
                    // the forward's keep bits: byte cc of the row's 16 covers chunk cc (bit e = feature 8 cc + e)
                    const uint32_t sbase = smem_u32(smem + s * p.stage_bytes);
                    const uint32_t xrow = sbase + row * 128;
                    const uint4 kb4 = lds128(sbase + p.off_bits + row * 16);
                    const uint32_t kw[4] = {kb4.x, kb4.y, kb4.z, kb4.w};
#pragma unroll
                    for (int cc = 0; cc < kChunks; ++cc) {
                        const uint32_t byte = kw[cc >> 2] >> (8 * (cc & 3));
                        const uint32_t addr = xrow + (cc >> 3) * 16384 + (((cc & 7) ^ (row & 7)) << 4);
                        uint4 v = lds128(addr);
                        v.x &= keep_mask_word(byte, 0);
                        v.y &= keep_mask_word(byte, 1);
                        v.z &= keep_mask_word(byte, 2);
                        v.w &= keep_mask_word(byte, 3);
                        sts128(addr, v);
                    }
                } else if (regen) {
                    const uint32_t xrow = smem_u32(smem + s * p.stage_bytes) + row * 128;
#pragma unroll
                    for (int c0 = 0; c0 < kChunks; c0 += kBatch) {
                        if (c0 > 0) {
                            if (kf.half) {
#pragma unroll
                                for (int i = 0; i < kBatch; ++i) km[i] = keep_chunk_mask<true>(prow, g0 + c0 + i, keys, kf);
                            } else {
#pragma unroll
                                for (int i = 0; i < kBatch; ++i) km[i] = keep_chunk_mask<false>(prow, g0 + c0 + i, keys, kf);
                            }
                        }
#pragma unroll
                        for (int i = 0; i < kBatch; ++i) {
                            const int cc = c0 + i;                      // chunk of the row: box cc / 8, chunk cc % 8
                            const uint32_t addr = xrow + (cc >> 3) * 16384 + (((cc & 7) ^ (row & 7)) << 4);
                            sts128(addr, and4(lds128(addr), km[i]));
                        }
                    }
                }
                fence_proxy_async_smem();
                mbar_arrive(&masked[s]);
            }
            // The epilogue of run e is run by group e % kGroups, which is also the TMEM buffer the run
            // accumulated in: each buffer is waited on by one group only, in order, so a parity wait never
            // meets a phase two behind, however many tiles each adapter's runs have.
            const uint32_t b = use % kGroups;
            if (last && b == static_cast<uint32_t>(group)) {
                const bool ok = mbar_wait(&acc_full[b], (use / kGroups) & 1u, w, 5);
                if (!__all_sync(0xFFFFFFFFu, ok)) break;
                tc_fence_after();
                const int64_t j = static_cast<int64_t>(d.fb) * 128 + quad * 32 + lane;
                const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + b * static_cast<uint32_t>(rpad_max);
                // deterministic mode: this CTA's partial of item (adapter, feature block) goes to slot item + CTA
                const int64_t item = static_cast<int64_t>(d.a) * p.nfb + d.fb;
                float* dst = p.sl.base ? p.sl.base + ((item + blockIdx.x) * 128 + quad * 32 + lane) * p.sl.ld
                                       : p.acc_base + ad.dA_off + j * ad.rpad;
                for (int c0 = 0; c0 < ad.rpad; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(taddr + c0, v);
                    tmem_ld_wait();
                    if (j < p.k) {
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

// dA_a = bf16(acc_a) (k x r_a), accumulators cleared; dSq rows of active tiles cleared.
__global__ void __launch_bounds__(256, 4) finalize_da_kernel(float* __restrict__ acc_base, int64_t k, uint16_t* __restrict__ dsq, int64_t m,
                                   int32_t ld, const __grid_constant__ Routing rt, const __grid_constant__ AdapterPtrs dap,
                                   const Slots sl, int32_t nfb, const __grid_constant__ UnitBegin ub) {
    __shared__ RowRouting sr;
    load_row_routing(sr, rt);   // parameters only: before the wait on the previous kernel
    pdl_wait();
    pdl_trigger();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t tid = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    for (int a = 0; a < rt.n_adapters; ++a) {
        const AdapterDev ad = rt.ad[a];
        if (rt.adapter_begin[a + 1] == rt.adapter_begin[a]) continue;
        // k * rank / 8 and m * ld / 8 stay below 2^31: 32-bit index arithmetic
        const uint32_t g8 = static_cast<uint32_t>(ad.rank / 8);
        const uint32_t total = static_cast<uint32_t>(k) * g8;
        for (uint32_t i = static_cast<uint32_t>(tid); i < total; i += static_cast<uint32_t>(stride)) {
            const uint32_t j = i / g8;
            const int c0 = static_cast<int>(i - j * g8) * 8;
            if (sl.base == nullptr) {
                finish_row(acc_base + ad.dA_off + static_cast<int64_t>(j) * ad.rpad + c0,
                           dap.p[a] + static_cast<int64_t>(j) * ad.rank + c0, 8, 8, 1.0f);
                continue;
            }
            // deterministic mode: the item's slots added in CTA order; its units are the adapter's tiles
            // of feature block j / 128
            const int fb = static_cast<int>(j >> 7);
            const int64_t n_a = rt.adapter_begin[a + 1] - rt.adapter_begin[a];
            const int64_t b = ub.u[a] + static_cast<int64_t>(fb) * n_a;
            float v[8];
            slot_sum8(sl, static_cast<int64_t>(a) * nfb + fb, b, b + n_a, static_cast<int>(j & 127), c0, v);
            store_row8(dap.p[a] + static_cast<int64_t>(j) * ad.rank + c0, v, 8, 1.0f);
        }
    }
    const uint32_t g8 = static_cast<uint32_t>(ld / 8);
    const uint32_t total = static_cast<uint32_t>(m) * g8;
    for (uint32_t i = static_cast<uint32_t>(tid); i < total; i += static_cast<uint32_t>(stride)) {
        const uint32_t t = i / g8;
        if (sr.owner[t >> 7] < 0) continue;
        stg128(dsq + static_cast<int64_t>(t) * ld + (i - t * g8) * 8, make_uint4(0u, 0u, 0u, 0u));
    }
}

__global__ void stuck_wait_kernel(DevCtl ctl) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const WaitCtx w{&abort_flag, ctl.status, ctl.wait_ns, kKDebug << 8};
    // No thread ever arrives on `bar`: the wait can only end by running out of time.
    if (threadIdx.x == 0) mbar_wait(&bar, 0, w, 1);
    __syncthreads();
}

}  // namespace

size_t da_smem_bytes(const DaParams& p) { return 1024 + p.stages * p.stage_bytes + (3 * p.stages + 2 * p.groups + 1) * 8 + 16; }

cudaError_t da_configure() {
    cudaError_t e = cudaFuncSetAttribute(da_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(da_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    return e;
}

cudaError_t launch_da(const DaParams& p, int grid, cudaStream_t stream, bool pdl) {
    if (p.groups == 3) return launch_k(pdl, da_kernel<3>, dim3(grid), dim3(threads_of(3)), da_smem_bytes(p), stream, p);
    if (p.groups == 2) return launch_k(pdl, da_kernel<2>, dim3(grid), dim3(threads_of(2)), da_smem_bytes(p), stream, p);
    return cudaErrorInvalidValue;
}

cudaError_t launch_finalize_da(const DaParams& p, int sms, cudaStream_t stream, bool pdl) {
    UnitBegin ub;
    for (int a = 0; a <= kMaxAdapters; ++a) ub.u[a] = p.unit_begin[a];
    return launch_k(pdl, finalize_da_kernel, dim3(2 * sms), dim3(256), 0, stream, p.acc_base, p.k, p.dsq, p.m, p.ld,
                    p.rt, p.dA, p.sl, p.nfb, ub);
}

cudaError_t launch_stuck_wait(DevCtl ctl, cudaStream_t stream) {
    stuck_wait_kernel<<<1, 32, 0, stream>>>(ctl);
    return cudaGetLastError();
}

}  // namespace lora
