// Launch plans shared by the host driver (api.cu) and the kernels.
//
// Routing for the multi-adapter form travels as kernel parameters (no device
// tables, no host->device copies): every 128-row tile carries one adapter id
// (LoRAFusion notes, section 5 "FusedMultiLoRA": each input tile carries its
// adapter id and that adapter's rank, scale and dropout rate).
#pragma once

#include <algorithm>
#include <cstdint>
#include <cuda.h>

namespace lora {

constexpr int kTileM = 128;          // rows per routing tile (= GEMM M tile)
constexpr int kMaxAdapters = 16;
constexpr int kMaxTiles = 2048;      // m <= 262144
constexpr int kMaxRank = 128;

// Kernel ids for device status codes (code = id << 8 | call site).
enum KernelId : int { kKDown = 1, kKGemmFwd = 2, kKGemmBwd = 3, kKDsDb = 4, kKDa = 5, kKDebug = 6 };

struct AdapterDev {
    int32_t rank;      // r_i
    int32_t rpad;      // power of two >= max(16, r_i): the MMA N (or M) extent of the rank
    uint32_t T;        // keep threshold: a 16-bit lane >= T keeps its element
    float scale;       // alpha_i / (1 - p_i): applied to (X.*D) A and to dY B^T
    int64_t dB_off;    // float offset of this adapter's dB^T accumulator (n x rpad)
    int64_t dA_off;    // float offset of this adapter's dA accumulator (k x rpad)
};

struct Routing {
    int32_t n_tiles;                         // ceil(m / 128)
    int32_t n_active;                        // tiles that have an adapter
    int32_t n_adapters;
    int32_t rpad_max;                        // max rpad over adapters (16 if none)
    int32_t adapter_begin[kMaxAdapters + 1]; // active_tiles[adapter_begin[a] .. adapter_begin[a+1]) = tiles of a
    AdapterDev ad[kMaxAdapters];
    int8_t tile_adapter[kMaxTiles];          // -1: no adapter
    uint16_t active_tiles[kMaxTiles];        // tile ids grouped by adapter, ascending within a group
};

// Per-adapter output pointers for the finalize kernels.
struct AdapterPtrs {
    uint16_t* p[kMaxAdapters];
};

struct DevCtl {
    int* status;        // device status word (workspace)
    uint64_t wait_ns;   // bounded-wait limit
};

// Fixed-order sums of stream-K partials (the library's deterministic mode).
// A pass splits its U units into G contiguous CTA ranges [U c / G, U (c+1) / G)
// with G <= U, so no range is empty.  An output item whose units are [b, e) is
// then summed by the CTAs slot_cta(b) .. slot_cta(e - 1), and CTA c writes its
// partial of item i, 128 rows of `ld` floats, to slot i + c: an item starts in
// the CTA where the one before it ends or later, so slots never collide, and
// the finalize kernel adds an item's slots in CTA order, the same order on every
// call, clearing them as it reads.  At most n_items + G - 1 slots are written.
struct Slots {
    float* base;     // null: partials are added into the accumulator with fp32 reductions
    int64_t units;   // U
    int32_t grid;    // G
    int32_t ld;      // floats per slot row
};

// The CTA whose range holds unit u: the largest c with floor(U c / G) <= u.
__host__ __device__ __forceinline__ int slot_cta(int64_t u, int64_t U, int32_t G) {
    return static_cast<int>(((u + 1) * G - 1) / U);
}

// Down-projection: S_acc[t, c] += sum_j (X .* D)[t, j] A_a[j, c] over stream-K
// ranges of (active tile, 128-wide k-block) units.
struct DownParams {
    CUtensorMap mapX;                  // X: dims {k, m}, box {64, 128}, 128B swizzle
    CUtensorMap mapA[kMaxAdapters];    // A_i: dims {r_i, k}, box {min(rpad,64), 128}, swizzle by rpad
    Routing rt;
    DevCtl ctl;
    float* S_acc;                      // m x ld fp32 (zero on entry; cleared by finalize_s)
    uint16_t* S_out;                   // S' = bf16(alpha/(1-p) S), m x ld
    uint8_t* mask_bits;                // optional, m x k/8
    int64_t m, k;
    int32_t ld;                        // s_ld
    int32_t nkb;                       // ceil(k / 128)
    int64_t units;                     // n_active * nkb
    uint32_t seed_lo, seed_hi;
    int32_t stages;
    uint32_t stage_bytes;              // X tile (two 16 KB boxes) + 128 rows of A (256 * rpad_max bytes)
    int32_t groups;                    // mask groups of four warps (2 or 4); stages % groups == 0
    Slots sl;                          // deterministic mode: S partials per (active tile, CTA) slot
};

// CTA-pair GEMM with the rank-r tail (k_gemm2.cu).
//  forward:  Y = [X | S'] [W ; B_a]           (B operand MN-major)
//  backward: dX = dY W^T + D .* (dSq A_a^T)   (B operand K-major; second accumulator)
// Each CTA of a pair stages half of the B tile, so B boxes are BN/2 wide.
struct GemmParams {
    CUtensorMap mapA;                  // fwd: X {k, m}; bwd: dY {n, m}; box {64, 128}
    CUtensorMap mapB;                  // fwd: W {n, k} box {64, 64}; bwd: W {n, k} box {64, BN/2}
    CUtensorMap mapTA;                 // tail A: fwd S' / bwd dSq, {s_ld, m}, box {64, 128}
    CUtensorMap mapTB[kMaxAdapters];   // tail B: fwd B_i {n, r_i} box {64, 64}; bwd A_i {r_i, k} box {64, BN/2}
    CUtensorMap mapOut;                // output Y / dX {N, M}, box {64, 128}, 128B swizzle (TMA store)
    Routing rt;
    DevCtl ctl;
    uint16_t* out;                     // Y (m x n) or dX (m x k), bf16
    int64_t M, N, K;                   // GEMM sizes: fwd (m, n, k), bwd (m, k, n)
    int32_t nkb;                       // 64-deep K blocks of the main product
    uint32_t seed_lo, seed_hi;
    const float* col_scale;            // forward only, optional: output column j is multiplied by col_scale[j] (DoRA)
    const uint8_t* keep_bits;          // backward only, optional: the forward's keep bits (m x N/8 bytes, N % 32 == 0),
                                       // read instead of regenerating the mask
    uint8_t* keep_out;                 // backward only, optional: where the regenerated keep bits of every branch row go
                                       // (same layout; N % 128 == 0), for the dA pass to read
    int32_t early_loads;               // 1: the producer may load the first tile's main-loop stages before waiting on
                                       // the previous kernel (no kernel of this call writes the main-loop operands, and
                                       // an earlier kernel of the call has already waited on the caller's work)
    int32_t sk_tiles;                  // stream-K: tiles [0, sk_tiles) are cut into runs of K stages spread evenly over
                                       // the pairs (0: every tile goes whole to one pair)
    float* sk_part;                    // per pair and CTA rank: the fp32 partial of the pair's first run when that run
                                       // is not the start of its tile (kSkSlotFloats each)
    uint32_t* sk_flag;                 // per pair and CTA rank: 1 once that partial is stored; reset by its reader
};

// Stream-K split tiles of the pair GEMM.  A pair's runs cover the contiguous units (tile, K stage)
// [U c / P, U (c+1) / P) of the first sk_tiles tiles, U = sk_tiles * stages, then whole tiles.  Only a pair's
// first run can start inside a tile, so one partial slot per pair and CTA suffices.  The run that starts a
// split tile adds the other runs' partials to its own accumulator in pair order and stores the tile.
constexpr int kSkSlotFloats = 128 * 256;   // 128 rows x up to 256 columns
constexpr int kSkMaxParts = 2;             // other runs per split tile (the schedule keeps U / P >= stages / 2)
constexpr int kSkMinStages = 32;           // below this many K stages no tile is split

struct GemmSched {
    int32_t pairs;      // CTA pairs in the grid
    int32_t sk_tiles;   // tiles split by K (GemmParams::sk_tiles)
};

// Tiles T of 256 rows x bn columns, `stages` K stages each, `max_pairs` pairs that fit the device.  Whole
// tiles go to pairs in turn (min(T, max_pairs) pairs).  Splitting costs a partial store and read per split
// tile (a closing run's epilogue takes about as long as 26 stages of main loop), and the split runs start at
// staggered K offsets, which shares fewer operand lines in L2.  So tiles are split only where a last wave
// leaves most pairs idle and tiles have at least kSkMinStages stages (on GB300 splitting lost at 16):
//  - 2T <= max_pairs: every tile split in two, over 2T pairs;
//  - W = T / max_pairs full waves and R = T mod max_pairs > 0 tiles left: the first R + max_pairs tiles are
//    split (between one and two tiles of stages a pair) when R <= max_pairs / 4; or when R <= max_pairs / 2,
//    the closing runs are followed by whole tiles whose main loops hide them (W >= 2, two accumulator
//    sets) and the tiles are at most 64 stages deep (measured: a gain at 64 stages, none at 128).
// The split runs come first in every pair's order, so a split tile's closing run (which reads the other
// runs' partials) is followed by whole tiles.
inline GemmSched gemm_schedule(int64_t M, int64_t N, int bn, int stages, int max_pairs, bool allow_split,
                               bool single_acc) {
    const int64_t T = ((M + 255) / 256) * ((N + bn - 1) / bn);
    if (max_pairs < 1) max_pairs = 1;
    GemmSched s{static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(T, max_pairs))), 0};
    if (!allow_split || T == 0 || stages < kSkMinStages) return s;
    if (2 * T <= max_pairs) {
        s.pairs = static_cast<int32_t>(2 * T);
        s.sk_tiles = static_cast<int32_t>(T);
        return s;
    }
    if (T < max_pairs) return s;
    const int64_t W = T / max_pairs, R = T % max_pairs;
    const bool hidden = W >= 2 && !single_acc && stages <= 64;
    if (R != 0 && (hidden ? 2 * R <= max_pairs : 4 * R <= max_pairs)) s.sk_tiles = static_cast<int32_t>(R + max_pairs);
    return s;
}

// One run of a pair's work: main-loop stages [kb0, kb1) of a tile.  A run that ends at the last stage also
// takes the tile's rank-r tail; a run that is not the whole tile is part of a split tile.
struct Run {
    int tile, kb0, kb1;
};

__host__ __device__ __forceinline__ int64_t sk_unit_begin(int pair, int64_t U, int npairs) {
    return U * pair / npairs;
}

// A pair's runs in order: its units [U c / P, U (c+1) / P) of the first sk_tiles tiles (one run per tile
// touched), then whole tiles sk_tiles + c, + P, ...
struct RunWalk {
    int64_t u, u_end;
    int tile, total, step, nk;

    __host__ __device__ __forceinline__ bool next(Run& r) {
        if (u < u_end) {
            const int t = static_cast<int>(u / nk);
            const int kb0 = static_cast<int>(u - static_cast<int64_t>(t) * nk);
            const int64_t left = u_end - u;
            const int kb1 = left < nk - kb0 ? kb0 + static_cast<int>(left) : nk;
            r = Run{t, kb0, kb1};
            u += kb1 - kb0;
            return true;
        }
        if (tile < total) {
            r = Run{tile, 0, nk};
            tile += step;
            return true;
        }
        return false;
    }
};

__host__ __device__ __forceinline__ RunWalk run_walk(int sk_tiles, int pair, int npairs, int nk, int total) {
    const int64_t U = static_cast<int64_t>(sk_tiles) * nk;
    return RunWalk{sk_unit_begin(pair, U, npairs), sk_unit_begin(pair + 1, U, npairs), sk_tiles + pair, total,
                   npairs, nk};
}

// dS / dB from one read of dY: per (active tile, 128-wide n-block) unit,
//   acc_dS[tile]  += dY_tile B_a^T
//   acc_dBt[nblk] += dY_tile^T S'_tile
// strip == 0 (tile order): units tile by tile, n-blocks in order; dS is kept in
// TMEM over a CTA's run of n-blocks, each unit's dB^T is flushed.  strip > 0:
// units strip by strip (strip = `strip` consecutive n-blocks), tiles in routing
// order inside a strip, n-blocks innermost; dS is flushed per tile visit and a
// strip's dB^T accumulators stay in TMEM while the CTA stays in the strip.
struct DsDbParams {
    CUtensorMap mapDY;                 // dY {n, m}, box {64, 128}, 128B swizzle
    CUtensorMap mapB[kMaxAdapters];    // B_i {n, r_i}, box {64, rpad}, 128B swizzle (K-major, K = n)
    CUtensorMap mapS[kMaxAdapters];    // S' {s_ld, m}, box {min(rpad,64), 128}, swizzle by rpad (MN-major)
    Routing rt;
    DevCtl ctl;
    float* dS_acc;                     // m x ld fp32 (zero on entry; cleared by finalize_bwd1)
    float* acc_base;                   // adapter accumulators (dB_off; same)
    uint16_t* dSq;                     // bf16(alpha/(1-p) dS), m x ld (written by finalize_bwd1)
    AdapterPtrs dB;                    // per adapter: dB_i (r_i x n)
    int64_t m, n;
    int32_t ld;
    int32_t nnb;                       // ceil(n / 128)
    int32_t strip;                     // 0: tile order; else n-blocks per strip (one dB^T accumulator each in TMEM)
    int64_t units;                     // n_active * nnb
    int32_t stages;
    uint32_t stage_bytes, off_b, off_s; // stage layout
    int32_t parts;                     // kPartDs: flush dS; kPartDb: flush dB^T (the other product is computed, not kept)
    Slots sl;                          // deterministic mode (tile order): dS partials per (active tile, CTA) slot
};

// First unit of each adapter in the dA pass's order (the last entry: the unit count).
struct UnitBegin {
    int64_t u[kMaxAdapters + 1];
};

// dA = (X .* D)^T dSq per adapter: per (adapter, 128-feature block, tile) unit.
struct DaParams {
    CUtensorMap mapX;                  // X {k, m}, box {64, 128}, 128B swizzle
    CUtensorMap mapD[kMaxAdapters];    // dSq {s_ld, m}, box {min(rpad,64), 128}, swizzle by rpad (MN-major)
    Routing rt;
    DevCtl ctl;
    float* acc_base;                   // adapter accumulators (dA_off; zero on entry; cleared by finalize_da)
    AdapterPtrs dA;                    // per adapter: dA_i (k x r_i)
    uint16_t* dsq;                     // dSq (m x ld): cleared by finalize_da after its last read
    int32_t ld;
    int64_t m, k;
    int32_t nfb;                       // ceil(k / 128)
    int64_t units;                     // nfb * n_active
    int64_t unit_begin[kMaxAdapters + 1];  // first unit of each adapter
    uint32_t seed_lo, seed_hi;
    int32_t stages;
    uint32_t stage_bytes, off_d;
    CUtensorMap mapBits;               // optional: the forward's keep bits {k/8, m} bytes, box {16, 128}, no swizzle
    int32_t use_bits;                  // 1: the stage's keep bits come with X (at off_bits) instead of from Philox
    uint32_t off_bits;
    uint8_t* bits_clear;               // optional: the bits tensor of mapBits, whose bytes this pass zeroes once read
    int32_t groups;                    // mask groups of four warps (2 or 3); stages % groups == 0
    Slots sl;                          // deterministic mode: dA partials per (adapter * nfb + feature block, CTA) slot
};

}  // namespace lora
