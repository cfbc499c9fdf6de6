// The two dense contractions of the layer on 5th-generation tensor cores.
//
// Forward (article section 4.1, forward ②: the frozen GEMM and the up-
// projection accumulate into one output so the partial Y is never written):
//     Y = X W + S' B_a = [X | S'] [W ; B_a],   S' = alpha S
// the rank-r branch is ceil(r/64) extra 64-deep K blocks of the same tile loop.
//
// Backward (article section 4.1, backward ⑤: the base-gradient path and the
// LoRA path are fused so the partial dX is never written):
//     dX = dY W^T + D .* (dSq A_a^T),   dSq = alpha/(1-p) dY B_a^T
// the branch product goes to a second TMEM accumulator (K = r), and the
// epilogue regenerates the keep mask D of each output element from the seed.
//
// Structure (one CTA per SM, persistent over 128 x 256 output tiles):
//   warp 0    TMA producer: A tile 128 x 64 (K-major, 128B swizzle) and
//             B tile 64 x 256 into a 4-stage ring;
//   warp 1    one thread issues tcgen05.mma M=128 N=256 K=16 and commits
//             stage releases / accumulator hand-offs to mbarriers;
//   warps 2-5 epilogue: tcgen05.ld from TMEM, (mask, add,) bf16, store.
// Forward keeps two accumulators (512 TMEM columns) so a tile's epilogue
// overlaps the next tile's main loop; backward uses both halves for the two
// accumulators of one tile.
#include "common.cuh"
#include "kernels.h"

namespace lora {

namespace {

constexpr int kThreads = 192;
constexpr uint32_t kABytes = 128u * 128u;       // 128 rows x 64 bf16
constexpr uint32_t kBBytes = 256u * 128u;       // 256 x 64 bf16
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = 512;

struct TileCoord {
    int m_blk, n_blk;
};

__device__ __forceinline__ TileCoord tile_coord(int tile, const GemmParams& p) {
    const int per_group = p.group_m * p.n_ntiles;
    const int group = tile / per_group;
    const int first_m = group * p.group_m;
    const int gm = min(p.n_mtiles - first_m, p.group_m);
    const int in_group = tile - group * per_group;
    return TileCoord{first_m + in_group % gm, in_group / gm};
}

template <bool kBwd>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align_1024(smem_raw);
    constexpr int S = kGemmStages;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * kStageBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + S;
    uint64_t* acc_full = bars + 2 * S;
    uint64_t* acc_empty = acc_full + 2;
    uint64_t* drain = acc_empty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 128);
        }
        mbar_init(drain, 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.mapA);
        tma_prefetch_desc(&p.mapB);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx w{&abort_flag, p.ctl.status, p.ctl.wait_ns, (kBwd ? kKGemmBwd : kKGemmFwd) << 8};

    const int total_tiles = p.n_mtiles * p.n_ntiles;

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
                const TileCoord tc = tile_coord(tile, p);
                const int m0 = tc.m_blk * kTileM;
                const int n0 = tc.n_blk * 256;
                const int a = p.rt.tile_adapter[tc.m_blk];
                const int ntail = a >= 0 ? (p.rt.ad[a].rank + 63) / 64 : 0;
                for (int kb = 0; kb < p.nkb + ntail; ++kb) {
                    if (!mbar_wait(&empty[s], ph ^ 1u, w, 1)) { ok = false; break; }
                    uint8_t* as = smem + s * kStageBytes;
                    uint8_t* bs = as + kABytes;
                    mbar_arrive_expect_tx(&full[s], kStageBytes);
                    if (kb < p.nkb) {
                        tma_load_2d(as, &p.mapA, &full[s], kb * 64, m0);
                        if (kBwd) {
                            tma_load_2d(bs, &p.mapB, &full[s], kb * 64, n0);
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j) tma_load_2d(bs + j * 8192, &p.mapB, &full[s], n0 + 64 * j, kb * 64);
                        }
                    } else {
                        const int tb = kb - p.nkb;
                        tma_load_2d(as, &p.mapTA, &full[s], tb * 64, m0);
                        if (kBwd) {
                            tma_load_2d(bs, &p.mapTB[a], &full[s], tb * 64, n0);
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                tma_load_2d(bs + j * 8192, &p.mapTB[a], &full[s], n0 + 64 * j, tb * 64);
                        }
                    }
                    ++issued;
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
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
            const uint32_t idesc = make_idesc_bf16(128, 256, false, !kBwd);
            bool ok = true;
            for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
                const TileCoord tc = tile_coord(tile, p);
                const int a = p.rt.tile_adapter[tc.m_blk];
                const int rank = a >= 0 ? p.rt.ad[a].rank : 0;
                const int ntail = (rank + 63) / 64;
                const uint32_t b = kBwd ? 0u : (use & 1u);
                const uint32_t empty_parity = kBwd ? ((use & 1u) ^ 1u) : (((use >> 1) & 1u) ^ 1u);
                if (!mbar_wait(&acc_empty[b], empty_parity, w, 2)) break;
                tc_fence_after();
                const uint32_t acc1 = tmem + b * 256u;
                const uint32_t acc2 = tmem + 256u;
                for (int kb = 0; kb < p.nkb + ntail; ++kb) {
                    if (!mbar_wait(&full[s], ph, w, 3)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t as = smem_u32(smem + s * kStageBytes);
                    const uint32_t bs = as + kABytes;
                    if (kb < p.nkb) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint64_t ad = make_smem_desc(as + ks * 32, 16, 1024, kSw128);
                            const uint64_t bd = kBwd ? make_smem_desc(bs + ks * 32, 16, 1024, kSw128)
                                                     : make_smem_desc(bs + ks * 2048, 8192, 1024, kSw128);
                            umma_bf16(acc1, ad, bd, idesc, (kb | ks) != 0 ? 1u : 0u);
                        }
                    } else {
                        const int tb = kb - p.nkb;
                        const int left = rank - tb * 64;
                        const int nks = left >= 64 ? 4 : (left + 15) / 16;
                        for (int ks = 0; ks < nks; ++ks) {
                            const uint64_t ad = make_smem_desc(as + ks * 32, 16, 1024, kSw128);
                            if (kBwd) {
                                const uint64_t bd = make_smem_desc(bs + ks * 32, 16, 1024, kSw128);
                                umma_bf16(acc2, ad, bd, idesc, (tb | ks) != 0 ? 1u : 0u);
                            } else {
                                const uint64_t bd = make_smem_desc(bs + ks * 2048, 8192, 1024, kSw128);
                                umma_bf16(acc1, ad, bd, idesc, 1u);
                            }
                        }
                    }
                    umma_commit(&empty[s]);
                    if (++s == S) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                umma_commit(&acc_full[b]);
                ++use;
            }
            umma_commit(drain);
            mbar_wait_drain(drain, 0, p.ctl.wait_ns);
        }
    } else {
        const int quad = warp & 3;
        const PhiloxKeys keys = philox_keys(p.seed_lo, p.seed_hi);
        uint32_t use = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
            const TileCoord tc = tile_coord(tile, p);
            const int m0 = tc.m_blk * kTileM;
            const int n0 = tc.n_blk * 256;
            const int a = p.rt.tile_adapter[tc.m_blk];
            const bool branch = kBwd && a >= 0;
            const uint32_t T = a >= 0 ? p.rt.ad[a].T : 0u;
            const uint32_t b = kBwd ? 0u : (use & 1u);
            const uint32_t full_parity = kBwd ? (use & 1u) : ((use >> 1) & 1u);
            const bool ok = mbar_wait(&acc_full[b], full_parity, w, 4);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            const int64_t row = static_cast<int64_t>(m0) + quad * 32 + lane;
            const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
            const uint32_t t1 = tmem + lane_off + b * 256u;
            const uint32_t t2 = tmem + lane_off + 256u;
            uint16_t* out_row = p.out + row * p.N;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
                uint32_t v[32];
                tmem_ld32(t1 + c * 32, v);
                if (branch) {
                    uint32_t u[32];
                    tmem_ld32(t2 + c * 32, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const int64_t col0 = static_cast<int64_t>(n0) + c * 32 + g * 8;
                        const uint4 wv = philox_10(static_cast<uint32_t>(row), static_cast<uint32_t>(col0 >> 3), keys);
                        const uint32_t keep = keep_byte(wv, T);
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            if ((keep >> e) & 1u)
                                v[g * 8 + e] = __float_as_uint(__uint_as_float(v[g * 8 + e]) + __uint_as_float(u[g * 8 + e]));
                    }
                } else {
                    tmem_ld_wait();
                }
                if (row < p.M) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int64_t col = static_cast<int64_t>(n0) + c * 32 + q * 8;
                        if (col < p.N) {
                            uint4 pk;
                            pk.x = pack_bf16x2(__uint_as_float(v[q * 8 + 0]), __uint_as_float(v[q * 8 + 1]));
                            pk.y = pack_bf16x2(__uint_as_float(v[q * 8 + 2]), __uint_as_float(v[q * 8 + 3]));
                            pk.z = pack_bf16x2(__uint_as_float(v[q * 8 + 4]), __uint_as_float(v[q * 8 + 5]));
                            pk.w = pack_bf16x2(__uint_as_float(v[q * 8 + 6]), __uint_as_float(v[q * 8 + 7]));
                            stg128(out_row + col, pk);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[b]);
            ++use;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t gemm_smem_bytes() { return 1024 + kGemmStages * kStageBytes + (2 * kGemmStages + 5) * 8 + 16; }

cudaError_t gemm_configure() {
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(gemm_smem_bytes()));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(gemm_smem_bytes()));
}

cudaError_t launch_gemm_fwd(const GemmParams& p, int grid, cudaStream_t stream) {
    gemm_kernel<false><<<grid, kThreads, gemm_smem_bytes(), stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_gemm_bwd(const GemmParams& p, int grid, cudaStream_t stream) {
    gemm_kernel<true><<<grid, kThreads, gemm_smem_bytes(), stream>>>(p);
    return cudaGetLastError();
}

}  // namespace lora
