// C ABI of the LoRA linear layer: validation, routing tables, tensor maps,
// workspace layout and the launch sequence of each call.  See include/lora.h
// for the contract of every entry point.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "kernels.h"
#include "lora.h"
#include "plan.h"

namespace lora {
namespace {

// ---------------------------------------------------------------------------
// per-device setup
// ---------------------------------------------------------------------------

struct DeviceState {
    bool ready = false;
    lora_status status = LORA_OK;
    int sms = 0;
};

// The backward's dA pass runs on a side stream, forked from and joined back to
// the caller's stream, so that it can use the SMs the dX GEMM's last wave of
// tiles leaves idle.  Each caller stream (per device) gets its own side stream
// and fork / join events, so that callers on different streams stay
// independent of one another.
struct SideStream {
    int device;
    cudaStream_t caller;
    cudaStream_t side;
    cudaEvent_t fork, join;
};

std::mutex g_mu;
thread_local const char* g_last_error = "no error";

bool cuda_ok(cudaError_t e) {
    if (e == cudaSuccess) return true;
    g_last_error = cudaGetErrorString(e);
    return false;
}
DeviceState g_dev[64];
uint64_t g_wait_ns = 2000000000ull;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// ---------------------------------------------------------------------------
// optional per-kernel timing (measurement tools): events around each launch
// ---------------------------------------------------------------------------

enum Kind : int {
    kDownProj = 0, kFinalizeS, kGemmFwd, kDsDb, kFinalize, kGemmBwd, kDa, kFinalizeDa, kMemset,
    kDoraU, kDoraNorm, kDoraDz, kDoraDmag, kKinds
};
const char* const kKindNames[kKinds] = {"down_proj", "finalize_s", "gemm_fwd", "ds_db", "finalize_ds_db",
                                        "gemm_bwd", "da", "finalize_da", "memset",
                                        "dora_u", "dora_norm", "dora_dz", "dora_dmag"};

struct TimingRec {
    int kind;
    cudaEvent_t a, b;
};
std::mutex g_timing_mu;
bool g_timing_on = false;
std::vector<TimingRec> g_timing;
std::vector<cudaEvent_t> g_event_pool;
size_t g_pool_next = 0;

cudaEvent_t pool_event() {
    if (g_pool_next == g_event_pool.size()) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        g_event_pool.push_back(e);
    }
    return g_event_pool[g_pool_next++];
}

// Runs `launch` (which enqueues work on `s`); when timing is on, brackets it with events.
template <class F>
cudaError_t timed(int kind, cudaStream_t s, F&& launch) {
    if (!g_timing_on) return launch();
    std::lock_guard<std::mutex> lock(g_timing_mu);
    cudaEvent_t a = pool_event(), b = pool_event();
    if (a) cudaEventRecord(a, s);
    const cudaError_t e = launch();
    if (b) cudaEventRecord(b, s);
    if (a && b) g_timing.push_back(TimingRec{kind, a, b});
    return e;
}

lora_status device_setup(int* sms_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LORA_ECUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& d = g_dev[dev];
    if (!d.ready) {
        d.ready = true;
        int major = 0, minor = 0, sms = 0;
        if (!cuda_ok(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) ||
            !cuda_ok(cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
            !cuda_ok(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))) {
            d.status = LORA_ECUDA;
        } else if (major != 10 || minor != 3) {
            d.status = LORA_EARCH;
        } else {
            d.sms = sms;
            if (!cuda_ok(down_configure()) || !cuda_ok(gemm2_configure()) ||
                !cuda_ok(dsdb_configure()) ||
                !cuda_ok(da_configure()) || !cuda_ok(dora_configure()))
                d.status = LORA_ECUDA;
        }
        if (d.status == LORA_OK && g_encode == nullptr) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (!cuda_ok(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q)) ||
                q != cudaDriverEntryPointSuccess || fn == nullptr) {
                if (q != cudaDriverEntryPointSuccess) g_last_error = "cuTensorMapEncodeTiled entry point not found";
                d.status = LORA_ECUDA;
            }
            else
                g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    if (d.status != LORA_OK) return d.status;
    *sms_out = d.sms;
    return LORA_OK;
}

std::vector<SideStream> g_side;   // guarded by g_mu

// The side stream and fork / join events of `caller` on the current device, created on first use (the first
// backward call on a stream therefore creates a stream and two events: make it before any stream capture).
bool side_stream(cudaStream_t caller, cudaStream_t* side, cudaEvent_t* fork, cudaEvent_t* join) {
    int dev = 0;
    if (!cuda_ok(cudaGetDevice(&dev))) return false;
    std::lock_guard<std::mutex> lock(g_mu);
    for (const SideStream& e : g_side)
        if (e.device == dev && e.caller == caller) {
            *side = e.side;
            *fork = e.fork;
            *join = e.join;
            return true;
        }
    SideStream e{dev, caller, nullptr, nullptr, nullptr};
    if (!cuda_ok(cudaStreamCreateWithFlags(&e.side, cudaStreamNonBlocking)) ||
        !cuda_ok(cudaEventCreateWithFlags(&e.fork, cudaEventDisableTiming)) ||
        !cuda_ok(cudaEventCreateWithFlags(&e.join, cudaEventDisableTiming)))
        return false;
    g_side.push_back(e);
    *side = e.side;
    *fork = e.fork;
    *join = e.join;
    return true;
}

// 2-D bf16 tensor map: `inner` contiguous elements per row, `outer` rows,
// `ld` elements between rows.
bool make_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
              uint32_t box_outer, CUtensorMapSwizzle swz) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) g_last_error = "cuTensorMapEncodeTiled rejected a tensor map";
    return r == CUDA_SUCCESS;
}

// 2-D byte tensor map (keep bits): `inner` bytes per row, `outer` rows, `ld` bytes between rows, no swizzle.
bool make_map_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld, uint32_t box_inner,
                 uint32_t box_outer) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
                                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) g_last_error = "cuTensorMapEncodeTiled rejected a tensor map";
    return r == CUDA_SUCCESS;
}

CUtensorMapSwizzle rank_swizzle_host(int rpad) {
    return rpad <= 16 ? CU_TENSOR_MAP_SWIZZLE_32B : (rpad <= 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B);
}

// ---------------------------------------------------------------------------
// validation helpers
// ---------------------------------------------------------------------------

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int rank_pad(int r) {
    int p = 16;
    while (p < r) p <<= 1;
    return p;
}

uint32_t keep_threshold(float p) {
    return static_cast<uint32_t>(std::floor(static_cast<double>(p) * 65536.0 + 0.5));
}

lora_status check_dims(int64_t m, int64_t k, int64_t n) {
    if (m < 0 || k <= 0 || n <= 0) return LORA_ESHAPE;
    if (k % 8 || n % 8) return LORA_ESHAPE;
    if (m > LORA_MAX_ROWS) return LORA_ESHAPE;
    // at most 2^24 features: every per-feature count (k * rank / 8, n blocks, units) then fits 32 bits
    if (k > LORA_MAX_FEATURES || n > LORA_MAX_FEATURES) return LORA_ESHAPE;
    return LORA_OK;
}

lora_status check_adapter(const lora_adapter& a, bool need_grads) {
    if (a.rank < 8 || a.rank > LORA_MAX_RANK || a.rank % 8) return LORA_EINVAL;
    if (!(a.p >= 0.f && a.p < 1.f)) return LORA_EINVAL;
    if (!std::isfinite(a.alpha)) return LORA_EINVAL;
    if (!a.A || !a.B) return LORA_EINVAL;
    if (!aligned16(a.A) || !aligned16(a.B)) return LORA_EALIGN;
    if (need_grads) {
        if (!a.dA || !a.dB) return LORA_EINVAL;
        if (!aligned16(a.dA) || !aligned16(a.dB)) return LORA_EALIGN;
    }
    return LORA_OK;
}

// Segment table -> per-tile adapter (the routing table of the multi-adapter form).
lora_status tile_table(const lora_segment* seg, int32_t nseg, int32_t nad, int64_t m, int8_t* owner, int64_t n_tiles) {
    for (int64_t i = 0; i < n_tiles; ++i) owner[i] = -1;
    if (nseg < 0 || (nseg > 0 && !seg)) return LORA_EINVAL;
    for (int32_t s = 0; s < nseg; ++s) {
        const lora_segment& g = seg[s];
        if (g.rows == 0) continue;
        if (g.row_start < 0 || g.rows < 0 || g.row_start + g.rows > m) return LORA_ETABLE;
        if (g.row_start % LORA_TILE_ROWS) return LORA_ETABLE;
        if (g.rows % LORA_TILE_ROWS && g.row_start + g.rows != m) return LORA_ETABLE;
        if (g.adapter < 0 || g.adapter >= nad) return LORA_ETABLE;
        const int64_t t0 = g.row_start / LORA_TILE_ROWS;
        const int64_t t1 = (g.row_start + g.rows + LORA_TILE_ROWS - 1) / LORA_TILE_ROWS;
        for (int64_t t = t0; t < t1; ++t) {
            if (owner[t] != -1) return LORA_ETABLE;
            owner[t] = static_cast<int8_t>(g.adapter);
        }
    }
    return LORA_OK;
}

// ---------------------------------------------------------------------------
// workspace
// ---------------------------------------------------------------------------

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Every byte below is zero between calls: each finalize kernel clears the
// accumulators it reads, and finalize_da (after dSq's last reader) clears dSq.
struct Layout {
    size_t status = 0;      // int32 device status word
    size_t s_acc = 0;       // m x s_ld fp32 (forward S, backward dS)
    size_t dsq = 0;         // m x s_ld bf16
    size_t acc = 0;         // per-adapter dB^T (n x rpad) and dA (k x rpad) fp32
    size_t acc_floats = 0;
    size_t slots = 0;       // deterministic mode only: partial sums of split items (cleared by their finalize)
    size_t fwd_total = 0;   // bytes a forward call needs (the regions above)
    size_t bits = 0;        // backward only: m x k/8 keep bits from the dX GEMM to the dA pass (k % 128 == 0;
                            // zeroed by dA)
    size_t grads_total = 0; // bytes a backward call needs (the regions above)
    size_t sk = 0;          // optional: the pair GEMMs' split-tile flags, then their partial slots (plan.h); the
                            // closing run of a split tile resets the flags and zeroes the slots it reads
    int32_t sk_pairs = 0;   // pairs with a slot
    size_t total = 0;
};

// Pairs that may hold a split-tile partial: a GEMM splits tiles over at most twice its tile count of pairs,
// and never over more pairs than kSkSlotPairs (on a device with more SMs the GEMMs split no tiles).
constexpr int kSkSlotPairs = 80;

int32_t sk_slot_pairs(int64_t m, int64_t k, int64_t n) {
    const int64_t tiles = ((m + 255) / 256) * ((std::max(k, n) + 127) / 128);   // 128 wide: an upper bound
    return static_cast<int32_t>(std::min<int64_t>(kSkSlotPairs, 2 * tiles));
}

size_t sk_flag_bytes(int32_t pairs) { return up(static_cast<size_t>(pairs) * 2 * 4); }

// Deterministic mode: bytes of the slot region, whose slots (128 rows each) hold the partial sums of output
// items split over CTAs (plan.h, Slots): S' and dS items are active tiles (s_ld floats a row), dA items are
// (adapter, 128-feature block) pairs (rpad_max floats a row).  `ctas` bounds the grid of every such pass.
size_t det_slot_bytes(int64_t m, int64_t k, int s_ld, int rpad_max, int nad, int ctas) {
    const int64_t n_tiles = (m + kTileM - 1) / kTileM;
    const int64_t nfb = (k + 127) / 128;
    const size_t s = static_cast<size_t>(n_tiles + ctas) * 128 * s_ld * 4;
    const size_t d = static_cast<size_t>(std::max(nad, 1) * nfb + ctas) * 128 * rpad_max * 4;
    return std::max(s, d);
}

// Deterministic mode (lora_set_deterministic): split sums go through the slot region in a fixed order.
std::atomic<int> g_deterministic{0};

Layout layout(int64_t m, int64_t k, int64_t n, int s_ld, const int* rpads, int nad, int det_ctas = 0) {
    Layout L;
    size_t off = 0;
    L.status = off;
    off += kAlign;
    L.s_acc = off;
    off = up(off + static_cast<size_t>(m) * s_ld * 4);
    L.dsq = off;
    off = up(off + static_cast<size_t>(m) * s_ld * 2);
    L.acc = off;
    size_t floats = 0;
    for (int a = 0; a < nad; ++a) floats += static_cast<size_t>(n + k) * rpads[a];
    L.acc_floats = floats;
    off = up(off + floats * 4);
    if (det_ctas > 0) {
        int rpad_max = 16;
        for (int a = 0; a < nad; ++a) rpad_max = std::max(rpad_max, rpads[a]);
        L.slots = off;
        off = up(off + det_slot_bytes(m, k, std::max(s_ld, 8), rpad_max, nad, det_ctas));
    }
    L.fwd_total = off;   // the forward needs nothing after this
    L.bits = off;
    if (k % 128 == 0) off = up(off + static_cast<size_t>(m) * static_cast<size_t>(k / 8));
    L.grads_total = off;
    L.sk = off;
    L.sk_pairs = sk_slot_pairs(m, k, n);
    off = up(off + sk_flag_bytes(L.sk_pairs) + static_cast<size_t>(L.sk_pairs) * 2 * kSkSlotFloats * 4);
    L.total = off;
    return L;
}

// ---------------------------------------------------------------------------
// one prepared call
// ---------------------------------------------------------------------------

struct Call {
    Routing rt;
    int s_ld = 0;
    int rpads[kMaxAdapters] = {};
    Layout L;
    uint8_t* ws = nullptr;
    int sms = 0;
    bool det = false;    // deterministic mode for this call
    bool sk = false;     // the workspace holds the split-tile region
    cudaStream_t stream = nullptr;
};

lora_status prepare(Call& c, const lora_adapter* ads, int32_t nad, const lora_segment* seg, int32_t nseg, int64_t m,
                    int64_t k, int64_t n, bool need_grads, void* workspace, size_t ws_bytes, void* stream) {
    lora_status st = check_dims(m, k, n);
    if (st) return st;
    if (nad < 0 || nad > kMaxAdapters) return LORA_EINVAL;
    if (nad == 0 && nseg != 0) return LORA_ETABLE;
    if (nad > 0 && !ads) return LORA_EINVAL;
    std::memset(&c.rt, 0, sizeof(c.rt));
    c.rt.n_adapters = nad;
    c.rt.rpad_max = 16;
    int s_ld = 0;
    for (int a = 0; a < nad; ++a) {
        st = check_adapter(ads[a], need_grads);
        if (st) return st;
        AdapterDev& d = c.rt.ad[a];
        d.rank = ads[a].rank;
        d.rpad = rank_pad(ads[a].rank);
        d.T = keep_threshold(ads[a].p);
        d.scale = static_cast<float>(static_cast<double>(ads[a].alpha) / (1.0 - static_cast<double>(ads[a].p)));
        c.rpads[a] = d.rpad;
        c.rt.rpad_max = std::max(c.rt.rpad_max, d.rpad);
        s_ld = std::max(s_ld, d.rank);
    }
    c.s_ld = s_ld;
    const int64_t n_tiles = (m + kTileM - 1) / kTileM;
    if (n_tiles > kMaxTiles) return LORA_ESHAPE;
    c.rt.n_tiles = static_cast<int32_t>(n_tiles);
    st = tile_table(seg, nseg, nad, m, c.rt.tile_adapter, n_tiles);
    if (st) return st;
    // group active tiles by adapter (ascending tile id within a group)
    int count[kMaxAdapters + 1] = {};
    for (int64_t t = 0; t < n_tiles; ++t)
        if (c.rt.tile_adapter[t] >= 0) ++count[c.rt.tile_adapter[t]];
    c.rt.adapter_begin[0] = 0;
    for (int a = 0; a < kMaxAdapters; ++a) c.rt.adapter_begin[a + 1] = c.rt.adapter_begin[a] + (a < nad ? count[a] : 0);
    int fill[kMaxAdapters] = {};
    for (int64_t t = 0; t < n_tiles; ++t) {
        const int a = c.rt.tile_adapter[t];
        if (a >= 0) c.rt.active_tiles[c.rt.adapter_begin[a] + fill[a]++] = static_cast<uint16_t>(t);
    }
    c.rt.n_active = c.rt.adapter_begin[nad > 0 ? nad : 0];
    // workspace (the deterministic mode's slot region is sized by the device's grid: device set-up first)
    c.det = g_deterministic.load() != 0;
    int det_ctas = 0;
    if (c.det) {
        st = device_setup(&c.sms);
        if (st) return st;
        det_ctas = 2 * c.sms;
    }
    c.L = layout(m, k, n, s_ld, c.rpads, nad, det_ctas);
    int64_t off = 0;
    for (int a = 0; a < nad; ++a) {
        c.rt.ad[a].dB_off = off;
        off += n * c.rpads[a];
        c.rt.ad[a].dA_off = off;
        off += k * c.rpads[a];
    }
    if (!workspace) return LORA_EWORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return LORA_EWORKSPACE;
    if (ws_bytes < (need_grads ? c.L.grads_total : c.L.fwd_total)) return LORA_EWORKSPACE;
    c.sk = ws_bytes >= c.L.total;
    c.ws = static_cast<uint8_t*>(workspace);
    st = device_setup(&c.sms);
    if (st) return st;
    c.stream = static_cast<cudaStream_t>(stream);
    return LORA_OK;
}

DevCtl ctl_of(const Call& c) { return DevCtl{reinterpret_cast<int*>(c.ws + c.L.status), g_wait_ns}; }

// Grid of a pair GEMM and its split tiles: splits only where the workspace holds slots for every pair.
GemmSched gemm_plan(const Call& c, GemmParams& g, bool bwd, int bn) {
    GemmSched sc = plan_gemm2(g, bwd, bn, c.sms, c.sk);
    if (sc.sk_tiles > 0 && sc.pairs > c.L.sk_pairs) sc = plan_gemm2(g, bwd, bn, c.sms, false);
    g.sk_tiles = sc.sk_tiles;
    g.sk_flag = reinterpret_cast<uint32_t*>(c.ws + c.L.sk);
    g.sk_part = reinterpret_cast<float*>(c.ws + c.L.sk + sk_flag_bytes(c.L.sk_pairs));
    return sc;
}

#define LORA_CUDA(expr)                          \
    do {                                         \
        if (!cuda_ok(expr)) return LORA_ECUDA;   \
    } while (0)

// DoRA's extra inputs and scratch for one forward (single adapter).
struct DoraFwd {
    const float* mag;     // n
    const float* wn2;     // n: ||W[:, j]||^2
    float* g_out;         // n: the column scale (saved for the backward)
    float* U;             // workspace: n x rpad fp32 (zero between calls)
    float* G;             // workspace: r x r fp32
};

lora_status run_dora_norm(const Call& c, const DoraFwd& d, const uint16_t* W, const lora_adapter& ad, int64_t k,
                          int64_t n);

lora_status run_fwd(const Call& c, const uint16_t* X, const uint16_t* W, const lora_adapter* ads, uint64_t seed,
                    int64_t m, int64_t k, int64_t n, uint16_t* Y, uint16_t* S_saved, uint8_t* mask_bits,
                    const DoraFwd* dora = nullptr) {
    if (m == 0) return LORA_OK;
    const uint32_t seed_lo = static_cast<uint32_t>(seed), seed_hi = static_cast<uint32_t>(seed >> 32);
    const int nad = c.rt.n_adapters;

    if (nad > 0 && c.rt.n_active > 0) {
        thread_local DownParams p;  // large: off the stack, one per calling thread
        std::memset(&p, 0, sizeof(p));
        if (!make_map(&p.mapX, X, k, m, k, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
        for (int a = 0; a < nad; ++a) {
            const int rp = c.rpads[a];
            if (!make_map(&p.mapA[a], ads[a].A, ads[a].rank, k, ads[a].rank, std::min(rp, 64), 128,
                          rank_swizzle_host(rp)))
                return LORA_ECUDA;
        }
        p.rt = c.rt;
        p.ctl = ctl_of(c);
        p.S_acc = reinterpret_cast<float*>(c.ws + c.L.s_acc);
        p.S_out = S_saved;
        p.mask_bits = mask_bits;
        p.m = m;
        p.k = k;
        p.ld = c.s_ld;
        p.nkb = static_cast<int32_t>((k + 127) / 128);
        p.units = static_cast<int64_t>(c.rt.n_active) * p.nkb;
        p.seed_lo = seed_lo;
        p.seed_hi = seed_hi;
        p.stage_bytes = 32768u + 256u * static_cast<uint32_t>(c.rt.rpad_max);
        // Three mask groups (twelve warps; two if the ring held fewer than three stages): the mask's
        // Philox arithmetic is the pass's limit, and more warps keep more of it in flight.  Measured on the
        // m = 16384 square 4096 layer: two groups 47.6 us, three 45.2 us, four (at 96 registers) 45.3 us.
        p.groups = mask_ring_stages(p.stage_bytes, 8, 3) >= 3 ? 3 : 2;
        p.stages = mask_ring_stages(p.stage_bytes, 8, p.groups);
        const int grid = static_cast<int>(std::min<int64_t>(p.units, c.sms));
        if (c.det) p.sl = Slots{reinterpret_cast<float*>(c.ws + c.L.slots), p.units, grid, c.s_ld};
        LORA_CUDA(timed(kDownProj, c.stream, [&] { return launch_down(p, grid, c.stream); }));
        LORA_CUDA(timed(kFinalizeS, c.stream, [&] { return launch_finalize_s(p, c.sms, c.stream); }));
    }

    thread_local GemmParams g;
    std::memset(&g, 0, sizeof(g));
    if (!make_map(&g.mapA, X, k, m, k, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
    if (!make_map(&g.mapB, W, n, k, n, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
    if (nad > 0) {
        if (!make_map(&g.mapTA, S_saved, c.s_ld, m, c.s_ld, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
        for (int a = 0; a < nad; ++a)
            if (!make_map(&g.mapTB[a], ads[a].B, n, ads[a].rank, n, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
                return LORA_ECUDA;
    }
    if (!make_map(&g.mapOut, Y, n, m, n, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
    g.rt = c.rt;
    g.ctl = ctl_of(c);
    g.out = Y;
    g.M = m;
    g.N = n;
    g.K = k;
    g.nkb = static_cast<int32_t>((k + 63) / 64);
    g.seed_lo = seed_lo;
    g.seed_hi = seed_hi;
    // the down-projection, launched first, has waited on the caller's earlier work; no kernel of this call
    // writes X or W, so the GEMM may start loading them before it waits on finalize_s
    g.early_loads = (nad > 0 && c.rt.n_active > 0) ? 1 : 0;
    if (dora) {
        const lora_status st = run_dora_norm(c, *dora, W, ads[0], k, n);
        if (st) return st;
        g.col_scale = dora->g_out;
    }
    const GemmSched sc = gemm_plan(c, g, false, 256);
    LORA_CUDA(timed(kGemmFwd, c.stream, [&] { return launch_gemm2(g, false, 256, sc.pairs, c.stream); }));
    return LORA_OK;
}

// Padded rank from which the dS/dB pass walks its units in strip order (see run_bwd).
constexpr uint32_t kStripMinRank = 32;

// Output tile width of the backward (dX) GEMM: 256 columns with one accumulator set (dY W^T and the
// branch's dSq A^T fill TMEM), or 128 with two sets, so that a tile's epilogue overlaps the next tile's MMAs.
int bwd_tile_width(int64_t m, int64_t k, int64_t n) {
    (void)m;
    (void)k;
    (void)n;
    return kBwdPairBN;
}

// dy_from_call: dY was written by an earlier kernel of the same call (DoRA's dZ), so the dX GEMM must not
// read it before waiting on its predecessor.
lora_status run_bwd(const Call& c, const uint16_t* dY, const uint16_t* X, const uint16_t* W, const lora_adapter* ads,
                    uint64_t seed, int64_t m, int64_t k, int64_t n, const uint16_t* S_saved, const uint8_t* mask_bits,
                    uint16_t* dX, bool dy_from_call = false) {
    const uint32_t seed_lo = static_cast<uint32_t>(seed), seed_hi = static_cast<uint32_t>(seed >> 32);
    const int nad = c.rt.n_adapters;
    uint16_t* dsq = reinterpret_cast<uint16_t*>(c.ws + c.L.dsq);
    float* acc = reinterpret_cast<float*>(c.ws + c.L.acc);

    // Adapters that own no rows get zero gradients (no kernel finishes them).
    for (int a = 0; a < nad; ++a) {
        if (c.rt.adapter_begin[a + 1] > c.rt.adapter_begin[a]) continue;
        LORA_CUDA(timed(kMemset, c.stream, [&] {
            return cudaMemsetAsync(ads[a].dA, 0, static_cast<size_t>(k) * ads[a].rank * 2, c.stream);
        }));
        LORA_CUDA(timed(kMemset, c.stream, [&] {
            return cudaMemsetAsync(ads[a].dB, 0, static_cast<size_t>(n) * ads[a].rank * 2, c.stream);
        }));
    }

    if (nad > 0 && c.rt.n_active > 0) {
        thread_local DsDbParams p;
        std::memset(&p, 0, sizeof(p));
        if (!make_map(&p.mapDY, dY, n, m, n, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
        for (int a = 0; a < nad; ++a) {
            const int rp = c.rpads[a];
            if (!make_map(&p.mapB[a], ads[a].B, n, ads[a].rank, n, 64, rp, CU_TENSOR_MAP_SWIZZLE_128B))
                return LORA_ECUDA;
            if (!make_map(&p.mapS[a], S_saved, c.s_ld, m, c.s_ld, std::min(rp, 64), 128, rank_swizzle_host(rp)))
                return LORA_ECUDA;
            p.dB.p[a] = ads[a].dB;
        }
        p.rt = c.rt;
        p.ctl = ctl_of(c);
        p.dS_acc = reinterpret_cast<float*>(c.ws + c.L.s_acc);
        p.acc_base = acc;
        p.dSq = dsq;
        p.m = m;
        p.n = n;
        p.ld = c.s_ld;
        p.nnb = static_cast<int32_t>((n + 127) / 128);
        p.units = static_cast<int64_t>(c.rt.n_active) * p.nnb;
        const uint32_t rpm = static_cast<uint32_t>(c.rt.rpad_max);
        p.off_b = 32768;
        p.off_s = p.off_b + 2 * 128 * rpm;
        p.stage_bytes = p.off_s + 256 * rpm;
        // Two issuing threads per CTA (dS and dB^T) share the small MMAs' fixed per-instruction cost.  When
        // two stages fit in half the shared memory (padded rank <= 32), two CTAs share each SM, each with a
        // two-stage ring; larger ranks keep one CTA per SM with the deepest ring that fits.
        const bool two_per_sm = 2u * p.stage_bytes <= kStageBudget / 2 - 2048;
        p.stages = two_per_sm ? 2 : static_cast<int32_t>(std::min<size_t>(8, kStageBudget / p.stage_bytes));
        // From padded rank 32 on, the strip order: TMEM of a CTA (512 columns, 256 when two CTAs share the
        // SM) holds two dS buffers and one dB^T accumulator per n-block of a strip, each rpad_max columns
        // wide, so dB^T is flushed once per strip segment instead of once per unit.  At padded rank 16 the
        // tile order with per-unit dB^T flushes is faster: its flushes are small.  Measured (us): rank 16 on
        // the Llama-3.1-8B up-proj 52 tile / 61 strip; rank 32 on the square 4096 layer at m = 16384
        // 52.3 tile / 46.5 strip, at m = 4096 21.9 tile / 23.7 strip.
        p.strip = rpm >= kStripMinRank ? std::max(1, std::min<int>(p.nnb, (two_per_sm ? 256 : 512) / static_cast<int>(rpm) - 2)) : 0;
        p.parts = kPartDs | kPartDb;
        const int64_t ctas = static_cast<int64_t>(two_per_sm ? 2 : 1) * c.sms;
        if (!c.det) {
            // up to padded rank 64 four threads issue the strip order's MMAs: two dS accumulators per buffer
            // leave TMEM for four n-blocks a strip (k_dsdb.cu, dsdb_strip4_kernel).  Measured on the 70B up-proj at
            // rank 64: 257 -> 213 us for the pass, 9.245 -> 9.155 ms for the step.
            if (p.strip > 0 && strip_four_issuers(static_cast<int>(rpm), p.parts))
                p.strip = std::max(1, std::min<int>(p.nnb, (two_per_sm ? 256 : 512) / static_cast<int>(rpm) - 4));
            const int grid = static_cast<int>(std::min<int64_t>(p.units, ctas));
            LORA_CUDA(timed(kDsDb, c.stream, [&] { return launch_dsdb(p, grid, c.stream); }));
            LORA_CUDA(timed(kFinalize, c.stream, [&] { return launch_finalize_bwd1(p, kPartDs | kPartDb, c.sms, c.stream); }));
        } else {
            // Deterministic mode, two reads of dY.  dS: tile order, each CTA's partial of a tile in its own slot,
            // added in CTA order by finalize_bwd1.  dB: strips of one n-block, each split between at most two CTAs,
            // so every dB^T element is the sum of at most two reductions onto zero, which commute exactly.
            p.strip = 0;
            p.parts = kPartDs;
            const int grid = static_cast<int>(std::min<int64_t>(p.units, ctas));
            p.sl = Slots{reinterpret_cast<float*>(c.ws + c.L.slots), p.units, grid, c.s_ld};
            LORA_CUDA(timed(kDsDb, c.stream, [&] { return launch_dsdb(p, grid, c.stream); }));
            LORA_CUDA(timed(kFinalize, c.stream, [&] { return launch_finalize_bwd1(p, kPartDs, c.sms, c.stream); }));
            p.strip = 1;
            p.parts = kPartDb;
            p.sl = Slots{};
            const int grid_db = p.nnb * (c.rt.n_active >= 2 ? 2 : 1);
            LORA_CUDA(timed(kDsDb, c.stream, [&] { return launch_dsdb(p, grid_db, c.stream); }));
            LORA_CUDA(timed(kFinalize, c.stream, [&] { return launch_finalize_bwd1(p, kPartDb, c.sms, c.stream); }));
        }
    }

    // The dA pass needs the keep mask.  When the backward regenerates it (no caller bits) and k % 128 == 0, the
    // dX GEMM's epilogue, which regenerates it for its own tiles anyway, writes the bits to the workspace and
    // the dA pass reads them after the GEMM: an HBM-bound pass instead of a second Philox pass.  Otherwise dA
    // regenerates (or reads the caller's bits) and is forked onto the side stream, launched after the dX GEMM
    // so that the GEMM's CTAs take the SMs first, and joined back before finalize_da.
    // Measured against the forked Philox pass (step time): Llama-3.1-8B up-proj 1.1523 -> 1.1481 ms, square 4096
    // layer at m = 16384 0.7609 -> 0.7542 ms, Llama-3.1-70B up-proj at rank 64 9.491 -> 9.469 ms.
    const bool gemm_bits = mask_bits == nullptr && k % 128 == 0 && nad > 0 && c.rt.n_active > 0;
    uint8_t* const ws_bits = gemm_bits ? c.ws + c.L.bits : nullptr;
    const bool fork_da = nad > 0 && c.rt.n_active > 0 && !gemm_bits;
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    if (fork_da) {
        if (!side_stream(c.stream, &side, &ev_fork, &ev_join)) return LORA_ECUDA;
        LORA_CUDA(cudaEventRecord(ev_fork, c.stream));
        LORA_CUDA(cudaStreamWaitEvent(side, ev_fork, 0));
    }

    if (m > 0) {
        thread_local GemmParams g;
        std::memset(&g, 0, sizeof(g));
        if (!make_map(&g.mapA, dY, n, m, n, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
        const int bn = bwd_tile_width(m, k, n);
        if (!make_map(&g.mapB, W, n, k, n, 64, bn / 2, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
        if (nad > 0) {
            if (!make_map(&g.mapTA, dsq, c.s_ld, m, c.s_ld, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
            for (int a = 0; a < nad; ++a)
                if (!make_map(&g.mapTB[a], ads[a].A, ads[a].rank, k, ads[a].rank, 64, bn / 2,
                              CU_TENSOR_MAP_SWIZZLE_128B))
                    return LORA_ECUDA;
        }
        if (!make_map(&g.mapOut, dX, k, m, k, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
        g.rt = c.rt;
        g.ctl = ctl_of(c);
        g.out = dX;
        g.M = m;
        g.N = k;
        g.K = n;
        g.nkb = static_cast<int32_t>((n + 63) / 64);
        g.seed_lo = seed_lo;
        g.seed_hi = seed_hi;
        // the forward's keep bits, when given, replace the epilogue's Philox (whole 32-bit words per row)
        g.keep_bits = (mask_bits != nullptr && k % 32 == 0) ? mask_bits : nullptr;
        g.keep_out = ws_bits;
        // the dS/dB pass, launched first, has waited on the caller's earlier work; dY and W are written by no
        // kernel of this call (unless dY is DoRA's dZ)
        g.early_loads = (nad > 0 && c.rt.n_active > 0 && !dy_from_call) ? 1 : 0;
        const GemmSched sc = gemm_plan(c, g, true, bn);
        LORA_CUDA(timed(kGemmBwd, c.stream, [&] { return launch_gemm2(g, true, bn, sc.pairs, c.stream); }));
    }

    if (fork_da || gemm_bits) {
        thread_local DaParams p;
        std::memset(&p, 0, sizeof(p));
        if (!make_map(&p.mapX, X, k, m, k, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
        for (int a = 0; a < nad; ++a) {
            const int rp = c.rpads[a];
            if (!make_map(&p.mapD[a], dsq, c.s_ld, m, c.s_ld, std::min(rp, 64), 128, rank_swizzle_host(rp)))
                return LORA_ECUDA;
            p.dA.p[a] = ads[a].dA;
        }
        p.rt = c.rt;
        p.ctl = ctl_of(c);
        p.acc_base = acc;
        p.dsq = dsq;
        p.ld = c.s_ld;
        p.m = m;
        p.k = k;
        p.nfb = static_cast<int32_t>((k + 127) / 128);
        int64_t u = 0;
        for (int a = 0; a <= nad; ++a) {
            p.unit_begin[a] = u;
            if (a < nad) u += static_cast<int64_t>(p.nfb) * (c.rt.adapter_begin[a + 1] - c.rt.adapter_begin[a]);
        }
        for (int a = nad + 1; a <= kMaxAdapters; ++a) p.unit_begin[a] = u;
        p.units = u;
        p.seed_lo = seed_lo;
        p.seed_hi = seed_hi;
        const uint32_t rpm = static_cast<uint32_t>(c.rt.rpad_max);
        p.off_d = 32768;
        p.stage_bytes = p.off_d + 256 * rpm;
        // the forward's keep bits, when given, come with each X stage (16 bytes a row; rows of whole 16 bytes)
        p.use_bits = ((mask_bits != nullptr && k % 128 == 0) || gemm_bits) ? 1 : 0;
        p.bits_clear = ws_bits;
        if (p.use_bits) {
            if (!make_map_u8(&p.mapBits, gemm_bits ? ws_bits : mask_bits, k / 8, m, k / 8, 16, 128)) return LORA_ECUDA;
            p.off_bits = p.stage_bytes;
            p.stage_bytes += 2048;
        }
        // three mask groups where the ring holds three stages (as the down-projection), else two
        p.groups = mask_ring_stages(p.stage_bytes, 8, 3) >= 3 ? 3 : 2;
        p.stages = mask_ring_stages(p.stage_bytes, 8, p.groups);
        const int grid = static_cast<int>(std::min<int64_t>(p.units, c.sms));
        if (c.det) p.sl = Slots{reinterpret_cast<float*>(c.ws + c.L.slots), p.units, grid, static_cast<int32_t>(rpm)};
        // plain launches on both sides of the event waits: a programmatic launch could start before the
        // other stream's work it waits for is done
        if (fork_da) {
            LORA_CUDA(timed(kDa, side, [&] { return launch_da(p, grid, side, false); }));
            LORA_CUDA(cudaEventRecord(ev_join, side));
            LORA_CUDA(cudaStreamWaitEvent(c.stream, ev_join, 0));
            LORA_CUDA(timed(kFinalizeDa, c.stream, [&] { return launch_finalize_da(p, c.sms, c.stream, false); }));
        } else {
            LORA_CUDA(timed(kDa, c.stream, [&] { return launch_da(p, grid, c.stream); }));
            LORA_CUDA(timed(kFinalizeDa, c.stream, [&] { return launch_finalize_da(p, c.sms, c.stream); }));
        }
    }
    return LORA_OK;
}

// DoRA column scale g_j = mag_j / ||W_j + alpha (A B)_j|| from the factored norm: U = W^T A by the dA
// kernel (W's k rows stand in for the tokens, A for dSq, no mask), G = A^T A, then one thread per column.
lora_status run_dora_norm(const Call& c, const DoraFwd& d, const uint16_t* W, const lora_adapter& ad, int64_t k,
                          int64_t n) {
    const int r = ad.rank, rp = rank_pad(r);
    const int64_t n_tiles = (k + kTileM - 1) / kTileM;
    if (n_tiles > kMaxTiles) return LORA_ESHAPE;
    thread_local DaParams pu;
    std::memset(&pu, 0, sizeof(pu));
    if (!make_map(&pu.mapX, W, n, k, n, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) return LORA_ECUDA;
    if (!make_map(&pu.mapD[0], ad.A, r, k, r, std::min(rp, 64), 128, rank_swizzle_host(rp))) return LORA_ECUDA;
    Routing& rt = pu.rt;
    rt.n_tiles = static_cast<int32_t>(n_tiles);
    rt.n_active = static_cast<int32_t>(n_tiles);
    rt.n_adapters = 1;
    rt.rpad_max = rp;
    rt.adapter_begin[0] = 0;
    for (int a = 1; a <= kMaxAdapters; ++a) rt.adapter_begin[a] = static_cast<int32_t>(n_tiles);
    rt.ad[0].rank = r;
    rt.ad[0].rpad = rp;
    rt.ad[0].T = 0;          // no dropout: the plain contraction W^T A
    rt.ad[0].scale = 1.f;
    rt.ad[0].dA_off = 0;
    for (int64_t t = 0; t < n_tiles; ++t) {
        rt.tile_adapter[t] = 0;
        rt.active_tiles[t] = static_cast<uint16_t>(t);
    }
    pu.ctl = ctl_of(c);
    pu.acc_base = d.U;
    pu.ld = r;
    pu.m = k;
    pu.k = n;
    pu.nfb = static_cast<int32_t>((n + 127) / 128);
    pu.units = static_cast<int64_t>(pu.nfb) * n_tiles;
    pu.unit_begin[0] = 0;
    for (int a = 1; a <= kMaxAdapters; ++a) pu.unit_begin[a] = pu.units;
    pu.off_d = 32768;
    pu.stage_bytes = pu.off_d + 256 * static_cast<uint32_t>(rp);
    pu.groups = mask_ring_stages(pu.stage_bytes, 8, 3) >= 3 ? 3 : 2;
    pu.stages = mask_ring_stages(pu.stage_bytes, 8, pu.groups);
    const int grid = static_cast<int>(std::min<int64_t>(pu.units, c.sms));
    LORA_CUDA(timed(kDoraU, c.stream, [&] { return launch_da(pu, grid, c.stream); }));
    LORA_CUDA(timed(kDoraNorm, c.stream, [&] {
        cudaError_t e = launch_dora_gram(ad.A, k, r, d.G, c.stream);
        if (e != cudaSuccess) return e;
        return launch_dora_scale(d.U, rp, ad.B, d.G, r, d.wn2, d.mag, ad.alpha, n, d.g_out, c.stream);
    }));
    // G's last reader is done: back to zero, like every other accumulator of the workspace
    LORA_CUDA(cudaMemsetAsync(d.G, 0, static_cast<size_t>(r) * r * 4, c.stream));
    return LORA_OK;
}

// DoRA accumulators after the LoRA workspace: U (n x rpad fp32), G (r x r fp32), dmag (n fp32).  Like the
// rest of the workspace they are zero between calls: their last readers clear them.
struct DoraLayout {
    size_t u = 0, g = 0, dmag = 0, total = 0;
};

DoraLayout dora_layout(size_t base, int64_t n, int r) {
    DoraLayout D;
    size_t off = up(base);
    D.u = off;
    off = up(off + static_cast<size_t>(n) * rank_pad(r) * 4);
    D.g = off;
    off = up(off + static_cast<size_t>(r) * r * 4);
    D.dmag = off;
    off = up(off + static_cast<size_t>(n) * 4);
    D.total = off;
    return D;
}


// Scratch for lora_fwd_static_scratch, for callers that cannot hand the
// library any device memory of their own.  Every GPU that loads the library
// holds this array until the process exits; all calls on one GPU share it.
constexpr size_t kStaticScratchBytes = 8u << 20;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];
void* g_static_scratch_ptr[64] = {};   // device address of the array, per device
std::mutex g_static_mu;

}  // namespace
}  // namespace lora

using namespace lora;

// The layout lora_workspace_size sizes: every adapter at rank r_max (upper bounds for any call with these sizes).
Layout workspace_layout(int64_t m, int64_t k, int64_t n, int32_t r_max, int32_t n_adapters) {
    if (m < 0 || k < 0 || n < 0 || r_max < 0 || n_adapters < 0) return Layout{};
    int rp[kMaxAdapters];
    const int nad = std::min<int32_t>(std::max<int32_t>(n_adapters, 1), kMaxAdapters);
    for (int a = 0; a < nad; ++a) rp[a] = rank_pad(std::max(r_max, 8));
    int det_ctas = 0;
    if (g_deterministic.load() != 0) {
        // the slot region grows with the grid: two CTAs per SM of the current device (1024 if none answers)
        int dev = 0, sms = 0;
        det_ctas = (cudaGetDevice(&dev) == cudaSuccess &&
                    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms > 0)
                       ? 2 * sms
                       : 1024;
        cudaGetLastError();   // a failed query leaves no sticky error behind
    }
    return layout(m, k, n, std::max(r_max, 8), rp, nad, det_ctas);
}

extern "C" {

size_t lora_workspace_size(int64_t m, int64_t k, int64_t n, int32_t r_max, int32_t n_adapters) {
    return workspace_layout(m, k, n, r_max, n_adapters).total;
}

lora_status lora_set_deterministic(int32_t on) {
    if (on != 0 && on != 1) return LORA_EINVAL;
    g_deterministic.store(on);
    return LORA_OK;
}

int32_t lora_get_deterministic(void) { return g_deterministic.load(); }

lora_status multi_lora_fwd(const lora_bf16* X, const lora_bf16* W, const lora_adapter* adapters, int32_t n_adapters,
                           const lora_segment* segments, int32_t n_segments, uint64_t seed, int64_t m, int64_t k,
                           int64_t n, lora_bf16* Y, lora_bf16* S_saved, uint8_t* mask_bits, void* workspace,
                           size_t workspace_bytes, void* stream) {
    if (!W || (m > 0 && (!X || !Y))) return LORA_EINVAL;
    if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || !aligned16(S_saved) || !aligned16(mask_bits))
        return LORA_EALIGN;
    if (n_adapters > 0 && m > 0 && !S_saved) return LORA_EINVAL;
    thread_local Call c;
    lora_status st = prepare(c, adapters, n_adapters, segments, n_segments, m, k, n, false, workspace,
                             workspace_bytes, stream);
    if (st) return st;
    return run_fwd(c, X, W, adapters, seed, m, k, n, Y, S_saved, mask_bits);
}

lora_status multi_lora_bwd(const lora_bf16* dY, const lora_bf16* X, const lora_bf16* W, const lora_adapter* adapters,
                           int32_t n_adapters, const lora_segment* segments, int32_t n_segments, uint64_t seed,
                           int64_t m, int64_t k, int64_t n, const lora_bf16* S_saved, const uint8_t* mask_bits,
                           lora_bf16* dX, void* workspace, size_t workspace_bytes, void* stream) {
    if (!W || (m > 0 && (!X || !dY || !dX))) return LORA_EINVAL;
    if (!aligned16(dY) || !aligned16(X) || !aligned16(W) || !aligned16(dX) || !aligned16(S_saved) ||
        !aligned16(mask_bits))
        return LORA_EALIGN;
    if (n_adapters > 0 && m > 0 && !S_saved) return LORA_EINVAL;
    thread_local Call c;
    lora_status st = prepare(c, adapters, n_adapters, segments, n_segments, m, k, n, true, workspace,
                             workspace_bytes, stream);
    if (st) return st;
    return run_bwd(c, dY, X, W, adapters, seed, m, k, n, S_saved, mask_bits, dX);
}

lora_status lora_fwd(const lora_bf16* X, const lora_bf16* W, const lora_bf16* A, const lora_bf16* B, float alpha,
                     float p, uint64_t seed, int64_t m, int64_t k, int64_t n, int32_t r, lora_bf16* Y,
                     lora_bf16* S_saved, uint8_t* mask_bits, void* workspace, size_t workspace_bytes, void* stream) {
    lora_adapter ad{r, alpha, p, A, B, nullptr, nullptr};
    lora_segment seg{0, m, 0, 0};
    return multi_lora_fwd(X, W, &ad, 1, &seg, m > 0 ? 1 : 0, seed, m, k, n, Y, S_saved, mask_bits, workspace,
                          workspace_bytes, stream);
}

lora_status lora_bwd(const lora_bf16* dY, const lora_bf16* X, const lora_bf16* W, const lora_bf16* A,
                     const lora_bf16* B, const lora_bf16* S_saved, const uint8_t* mask_bits, float alpha, float p,
                     uint64_t seed, int64_t m, int64_t k, int64_t n, int32_t r, lora_bf16* dX, lora_bf16* dA,
                     lora_bf16* dB, void* workspace, size_t workspace_bytes, void* stream) {
    lora_adapter ad{r, alpha, p, A, B, dA, dB};
    lora_segment seg{0, m, 0, 0};
    return multi_lora_bwd(dY, X, W, &ad, 1, &seg, m > 0 ? 1 : 0, seed, m, k, n, S_saved, mask_bits, dX, workspace,
                          workspace_bytes, stream);
}

lora_status lora_fwd_static_scratch(const lora_bf16* X, const lora_bf16* W, const lora_bf16* A, const lora_bf16* B,
                                    float alpha, float p, uint64_t seed, int64_t m, int64_t k, int64_t n, int32_t r,
                                    lora_bf16* Y, lora_bf16* S_saved, uint8_t* mask_bits, void* stream) {
    // Every check lora_fwd makes comes first, so that a call that fails enqueues nothing (not even the
    // first call's clearing of the array) and reports the same status lora_fwd would.
    if (!W || (m > 0 && (!X || !Y || !S_saved))) return LORA_EINVAL;
    if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || !aligned16(S_saved) || !aligned16(mask_bits))
        return LORA_EALIGN;
    lora_status st = check_dims(m, k, n);
    if (st) return st;
    const lora_adapter ad{r, alpha, p, A, B, nullptr, nullptr};
    st = check_adapter(ad, false);
    if (st) return st;
    if ((m + kTileM - 1) / kTileM > kMaxTiles) return LORA_ESHAPE;
    const size_t need = workspace_layout(m, k, n, r, 1).fwd_total;   // a forward needs no backward-only region
    if (need > kStaticScratchBytes) {
        g_last_error = "lora_fwd_static_scratch: these sizes need more scratch than the 8 MiB static buffer";
        return LORA_EWORKSPACE;
    }
    int sms = 0;
    st = device_setup(&sms);
    if (st) return st;
    int dev = 0;
    if (!cuda_ok(cudaGetDevice(&dev)) || dev < 0 || dev >= 64) return LORA_ECUDA;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_mu);
        if (g_static_scratch_ptr[dev] == nullptr) {
            // Once per device, with that device current: the host name of the
            // array is only a stand-in, so look up its device address.
            void* ptr = nullptr;
            if (!cuda_ok(cudaGetSymbolAddress(&ptr, g_static_scratch))) return LORA_ECUDA;
            // The status word, accumulators and counters must start at zero.
            if (!cuda_ok(cudaMemsetAsync(ptr, 0, kStaticScratchBytes, static_cast<cudaStream_t>(stream))))
                return LORA_ECUDA;
            g_static_scratch_ptr[dev] = ptr;
        }
        scratch = g_static_scratch_ptr[dev];
    }
    return lora_fwd(X, W, A, B, alpha, p, seed, m, k, n, r, Y, S_saved, mask_bits, scratch, kStaticScratchBytes, stream);
}

lora_status lora_tile_table(const lora_segment* segments, int32_t n_segments, int32_t n_adapters, int64_t m,
                            int32_t* tile_adapter, int64_t n_tiles) {
    if (m < 0 || m > LORA_MAX_ROWS || n_adapters < 0 || n_adapters > kMaxAdapters) return LORA_EINVAL;
    const int64_t need = (m + kTileM - 1) / kTileM;
    if (!tile_adapter || n_tiles < need) return LORA_EINVAL;
    thread_local int8_t owner[kMaxTiles];
    lora_status st = tile_table(segments, n_segments, n_adapters, m, owner, need);
    if (st) return st;
    for (int64_t t = 0; t < need; ++t) tile_adapter[t] = owner[t];
    return LORA_OK;
}

lora_status lora_keep_threshold(float p, uint32_t* T) {
    if (!T || !(p >= 0.f && p < 1.f)) return LORA_EINVAL;
    *T = keep_threshold(p);
    return LORA_OK;
}

lora_status lora_device_status(void* workspace, void* stream, int32_t* code) {
    if (!workspace || !code) return LORA_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return LORA_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return LORA_ECUDA;
    if (v != 0) {
        const int32_t zero = 0;
        if (cudaMemcpyAsync(workspace, &zero, sizeof(zero), cudaMemcpyHostToDevice, s) != cudaSuccess)
            return LORA_ECUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return LORA_ECUDA;
    }
    *code = v;
    return v != 0 ? LORA_EDEVICE_TIMEOUT : LORA_OK;
}

void lora_set_wait_limit_ns(uint64_t ns) { g_wait_ns = ns > 0 ? ns : 1; }

lora_status lora_debug_stuck_wait(void* workspace, size_t workspace_bytes, void* stream) {
    if (!workspace || workspace_bytes < kAlign || reinterpret_cast<uintptr_t>(workspace) % kAlign)
        return LORA_EWORKSPACE;
    int sms = 0;
    lora_status st = device_setup(&sms);
    if (st) return st;
    DevCtl ctl{static_cast<int*>(workspace), g_wait_ns};
    if (!cuda_ok(launch_stuck_wait(ctl, static_cast<cudaStream_t>(stream)))) return LORA_ECUDA;
    return LORA_OK;
}

lora_status lora_debug_gemm_runs(int64_t M, int64_t N, int32_t bn, int32_t stages, int32_t max_pairs,
                                 int32_t allow_split, int32_t single_acc, int32_t* pairs, int32_t* split_tiles,
                                 int32_t* runs, int64_t cap, int64_t* n_runs) {
    if (!pairs || !split_tiles || !n_runs || (cap > 0 && !runs)) return LORA_EINVAL;
    if (M < 1 || N < 1 || bn < 1 || stages < 1 || max_pairs < 1 || cap < 0) return LORA_EINVAL;
    const int64_t T = ((M + 255) / 256) * ((N + bn - 1) / bn);
    if (T > (int64_t{1} << 30)) return LORA_EINVAL;
    const GemmSched sc = gemm_schedule(M, N, bn, stages, max_pairs, allow_split != 0, single_acc != 0);
    *pairs = sc.pairs;
    *split_tiles = sc.sk_tiles;
    int64_t n = 0;
    for (int c = 0; c < sc.pairs; ++c) {
        RunWalk w = run_walk(sc.sk_tiles, c, sc.pairs, stages, static_cast<int>(T));
        for (Run r; w.next(r); ++n) {
            if (n >= cap) continue;
            runs[4 * n] = c;
            runs[4 * n + 1] = r.tile;
            runs[4 * n + 2] = r.kb0;
            runs[4 * n + 3] = r.kb1;
        }
    }
    *n_runs = n;
    return LORA_OK;
}

const char* lora_last_error_string(void) { return g_last_error; }

lora_status lora_timing_begin(void) {
    std::lock_guard<std::mutex> lock(g_timing_mu);
    g_timing.clear();
    g_pool_next = 0;
    g_timing_on = true;
    return LORA_OK;
}

lora_status lora_timing_end(float* total_ms, int32_t* launches, int32_t n_kinds) {
    std::lock_guard<std::mutex> lock(g_timing_mu);
    g_timing_on = false;
    if (!total_ms || !launches || n_kinds < 0) return LORA_EINVAL;
    for (int i = 0; i < n_kinds; ++i) {
        total_ms[i] = 0.f;
        launches[i] = 0;
    }
    lora_status st = LORA_OK;
    for (const TimingRec& r : g_timing) {
        float ms = 0.f;
        if (!cuda_ok(cudaEventSynchronize(r.b)) || !cuda_ok(cudaEventElapsedTime(&ms, r.a, r.b))) {
            st = LORA_ECUDA;
            continue;
        }
        if (r.kind < n_kinds) {
            total_ms[r.kind] += ms;
            launches[r.kind] += 1;
        }
    }
    g_timing.clear();
    g_pool_next = 0;
    return st;
}

const char* lora_kernel_name(int32_t kind) { return (kind >= 0 && kind < kKinds) ? kKindNames[kind] : "unknown"; }

const char* lora_status_string(lora_status s) {
    switch (s) {
        case LORA_OK: return "ok";
        case LORA_EINVAL: return "invalid argument";
        case LORA_EALIGN: return "pointer not 16-byte aligned";
        case LORA_ESHAPE: return "unsupported shape";
        case LORA_EARCH: return "device is not sm_103";
        case LORA_ECUDA: return "CUDA call failed";
        case LORA_EWORKSPACE: return "workspace missing, misaligned or too small";
        case LORA_EDEVICE_TIMEOUT: return "a kernel gave up on a bounded wait";
        case LORA_ETABLE: return "invalid segment table";
    }
    return "unknown status";
}

size_t dora_workspace_size(int64_t m, int64_t k, int64_t n, int32_t r) {
    if (m < 0 || k < 0 || n < 0 || r < 0) return 0;
    return dora_layout(lora_workspace_size(m, k, n, r, 1), n, std::max(r, 8)).total;
}

lora_status dora_weight_norm2(const lora_bf16* W, int64_t k, int64_t n, float* w_norm2, void* stream) {
    if (!W || !w_norm2) return LORA_EINVAL;
    if (k <= 0 || n <= 0 || n % 8 || k > LORA_MAX_FEATURES || n > LORA_MAX_FEATURES) return LORA_ESHAPE;
    if (!aligned16(W) || !aligned16(w_norm2)) return LORA_EALIGN;
    int sms = 0;
    const lora_status st = device_setup(&sms);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!cuda_ok(cudaMemsetAsync(w_norm2, 0, static_cast<size_t>(n) * 4, s))) return LORA_ECUDA;
    if (!cuda_ok(launch_dora_norm2(W, k, n, w_norm2, sms, s))) return LORA_ECUDA;
    return LORA_OK;
}

lora_status dora_fwd(const lora_bf16* X, const lora_bf16* W, const lora_bf16* A, const lora_bf16* B, const float* mag,
                     const float* w_norm2, float alpha, float p, uint64_t seed, int64_t m, int64_t k, int64_t n,
                     int32_t r, lora_bf16* Y, lora_bf16* S_saved, float* g_saved, uint8_t* mask_bits, void* workspace,
                     size_t workspace_bytes, void* stream) {
    if (!W || !mag || !w_norm2 || !g_saved || (m > 0 && (!X || !Y || !S_saved))) return LORA_EINVAL;
    if (!aligned16(X) || !aligned16(W) || !aligned16(Y) || !aligned16(S_saved) || !aligned16(mag) ||
        !aligned16(w_norm2) || !aligned16(g_saved) || !aligned16(mask_bits))
        return LORA_EALIGN;
    lora_adapter ad{r, alpha, p, A, B, nullptr, nullptr};
    lora_segment seg{0, m, 0, 0};
    thread_local Call c;
    lora_status st = prepare(c, &ad, 1, &seg, m > 0 ? 1 : 0, m, k, n, false, workspace, workspace_bytes, stream);
    if (st) return st;
    const DoraLayout D = dora_layout(c.L.total, n, r);
    if (workspace_bytes < D.total) return LORA_EWORKSPACE;
    DoraFwd d{mag, w_norm2, g_saved, reinterpret_cast<float*>(c.ws + D.u), reinterpret_cast<float*>(c.ws + D.g)};
    if (m == 0) {
        // no tokens: the column scale is still defined (the backward reads it)
        return run_dora_norm(c, d, W, ad, k, n);
    }
    return run_fwd(c, X, W, &ad, seed, m, k, n, Y, S_saved, mask_bits, &d);
}

lora_status dora_bwd(const lora_bf16* dY, const lora_bf16* X, const lora_bf16* W, const lora_bf16* A,
                     const lora_bf16* B, const lora_bf16* S_saved, const uint8_t* mask_bits, const lora_bf16* Y,
                     const float* mag,
                     const float* g_saved, float alpha, float p, uint64_t seed, int64_t m, int64_t k, int64_t n,
                     int32_t r, lora_bf16* dX, lora_bf16* dA, lora_bf16* dB, float* dmag, lora_bf16* dZ,
                     void* workspace, size_t workspace_bytes, void* stream) {
    if (!W || !mag || !g_saved || !dmag || (m > 0 && (!X || !dY || !dX || !Y || !S_saved || !dZ)))
        return LORA_EINVAL;
    if (!aligned16(dY) || !aligned16(X) || !aligned16(W) || !aligned16(dX) || !aligned16(S_saved) ||
        !aligned16(Y) || !aligned16(mag) || !aligned16(g_saved) || !aligned16(dmag) || !aligned16(dZ) ||
        !aligned16(mask_bits))
        return LORA_EALIGN;
    lora_adapter ad{r, alpha, p, A, B, dA, dB};
    lora_segment seg{0, m, 0, 0};
    thread_local Call c;
    lora_status st = prepare(c, &ad, 1, &seg, m > 0 ? 1 : 0, m, k, n, true, workspace, workspace_bytes, stream);
    if (st) return st;
    const DoraLayout D = dora_layout(c.L.total, n, r);
    if (workspace_bytes < D.total) return LORA_EWORKSPACE;
    float* dmag_acc = reinterpret_cast<float*>(c.ws + D.dmag);
    if (m > 0)
        LORA_CUDA(timed(kDoraDz, c.stream, [&] { return launch_dora_dz(dY, Y, g_saved, m, n, dZ, dmag_acc, c.sms,
                                                                      c.stream); }));
    st = run_bwd(c, dZ, X, W, &ad, seed, m, k, n, S_saved, mask_bits, dX, /*dy_from_call=*/true);
    if (st) return st;
    LORA_CUDA(timed(kDoraDmag, c.stream, [&] { return launch_dora_dmag(dmag_acc, mag, n, dmag, c.stream); }));
    return LORA_OK;
}

}  // extern "C"
