// Device-side building blocks shared by the LoRA kernels (sm_103a only):
// mbarrier / TMA / tcgen05 wrappers written as inline PTX, shared-memory and
// instruction descriptors for tcgen05.mma kind::f16, bounded waits, and the
// Philox4x32-10 keep-mask generator.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "plan.h"

namespace lora {

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

__device__ __forceinline__ bool elect_lane0() { return (threadIdx.x & 31u) == 0u; }

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits that find their phase still open suspend the thread in hardware for
// up to this long (it wakes as soon as the phase completes): a role that only
// waits (the TMA producer, the MMA issuer, an idle mask group) then takes no
// issue slots from the warps that share its scheduler.
constexpr uint32_t kWaitSuspendNs = 20000;

__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kWaitSuspendNs)
        : "memory");
    return done != 0;
}

// Per-CTA failure state for bounded waits.  `abort` lives in shared memory;
// once any thread of the CTA times out, every later wait returns false at
// once and the roles wind down.
struct WaitCtx {
    volatile int* abort;   // shared
    int* status;           // global status word (workspace), may be null
    uint64_t limit_ns;
    int code;              // kernel id << 8, ORed with the call site
};

static __device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, const WaitCtx& w, int site) {
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 4; ++i)
            if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*w.abort) return false;
        if (global_timer_ns() - t0 > w.limit_ns) {
            *w.abort = 1;
            if (w.status) atomicCAS(w.status, 0, w.code | site);
            return false;
        }
    }
}

// Returns true once the phase with the given parity has completed; false if
// the CTA is aborting (this wait or another one ran out of time).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtx& w, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, w, site);
}

// Waits for a phase regardless of the CTA's abort state (used while winding
// down, so that copies and MMAs in flight finish before the CTA exits and
// TMEM is released).  Gives up after limit_ns.
static __device__ __noinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait_sleep(bar, parity))
        if (global_timer_ns() - t0 > limit_ns) return false;
    return true;
}

// Flags between CTAs of one grid, in global memory (gpu scope).
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Bounded wait until *flag is non-zero (acquire).  The flag is set by another CTA of the same grid that
// needs nothing from this one; false if the CTA is aborting or the wait ran out of time.
static __device__ __noinline__ bool flag_wait(const uint32_t* flag, const WaitCtx& w, int site) {
    const uint64_t t0 = global_timer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i) {
            if (ld_acquire_gpu(flag) != 0) return true;
            __nanosleep(100);
        }
        if (*w.abort) return false;
        if (global_timer_ns() - t0 > w.limit_ns) {
            *w.abort = 1;
            if (w.status) atomicCAS(w.status, 0, w.code | site);
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies global -> shared, completion on an mbarrier)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// Generic-proxy writes to shared memory become visible to the async proxy
// (tcgen05.mma operand reads) after this fence.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, loads
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Programmatic dependent launch.  pdl_wait: returns once the kernels this grid
// depends on have completed and their memory is visible (immediately when it
// was launched without the attribute); every global access of a kernel comes
// after it.  pdl_trigger: lets the next kernel on the stream start its CTAs
// (their prologue) on SMs this grid leaves free.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulator, one CTA.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Thread i of the warp receives row (lane base + i), 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Thread i of the warp receives row (lane base + i), 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// ---------------------------------------------------------------------------
// descriptors
// ---------------------------------------------------------------------------

// Swizzle modes of the tcgen05 shared-memory descriptor (bits 61..63).
enum : uint32_t { kSwNone = 0, kSw128 = 2, kSw64 = 4, kSw32 = 6 };

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (both in bytes here, stored >> 4), fixed version bit 46, swizzle.
// K-major swizzled operands: rows of the swizzle width along K, 8-row groups
// `sbo` bytes apart (lbo unused).  MN-major swizzled operands: `lbo` = bytes
// between swizzle atoms along M/N, `sbo` = bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t make_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;
    d |= static_cast<uint64_t>(swizzle & 7u) << 61;
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, dense.
// a_mn / b_mn select the MN-major ("transposed") operand layout.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4)                                      // D format: f32
           | (1u << 7)                                    // A format: bf16
           | (1u << 10)                                   // B format: bf16
           | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16)
           | (static_cast<uint32_t>(N >> 3) << 17)        // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);       // M / 16
}

// MN-major operand whose MN extent is the (padded) rank: the swizzle width
// follows the row bytes rpad*2 (32, 64 or 128; rank 128 uses two 128-byte atoms).
__device__ __forceinline__ uint32_t rank_swizzle(int rpad) {
    return rpad <= 16 ? kSw32 : (rpad <= 32 ? kSw64 : kSw128);
}
__device__ __forceinline__ uint32_t rank_row_bytes(int rpad) { return rpad >= 64 ? 128u : static_cast<uint32_t>(rpad) * 2u; }

// ---------------------------------------------------------------------------
// misc memory ops
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(addr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void stg128(void* ptr, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    // round to nearest even, low element in the low half
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// ---------------------------------------------------------------------------
// Philox4x32-10 keep mask (Salmon, Moraes, Dror, Shaw, SC'11)
// ---------------------------------------------------------------------------

// Round keys of one seed: round r uses (k0 + r*W0, k1 + r*W1).
struct PhiloxKeys {
    uint32_t k0[10], k1[10];
};

__device__ __forceinline__ PhiloxKeys philox_keys(uint32_t k0, uint32_t k1) {
    PhiloxKeys K;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        K.k0[r] = k0 + static_cast<uint32_t>(r) * 0x9E3779B9u;
        K.k1[r] = k1 + static_cast<uint32_t>(r) * 0xBB67AE85u;
    }
    return K;
}

// Counter (c0, c1, 0, 0); ten rounds.  Each round is two 32x32->64 products
// (one IMAD.WIDE each: high and low words come out as a register pair) and
// two three-input XORs.
__device__ __forceinline__ uint4 philox_10(uint32_t c0, uint32_t c1, const PhiloxKeys& K) {
    uint32_t x0 = c0, x1 = c1, x2 = 0u, x3 = 0u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = static_cast<uint64_t>(x0) * 0xD2511F53u;
        const uint64_t p1 = static_cast<uint64_t>(x2) * 0xCD9E8D57u;
        x0 = static_cast<uint32_t>(p1 >> 32) ^ x1 ^ K.k0[r];
        x1 = static_cast<uint32_t>(p1);
        x2 = static_cast<uint32_t>(p0 >> 32) ^ x3 ^ K.k1[r];
        x3 = static_cast<uint32_t>(p0);
    }
    return make_uint4(x0, x1, x2, x3);
}

__device__ __forceinline__ uint4 philox_10(uint32_t c0, uint32_t c1, uint32_t k0, uint32_t k1) {
    return philox_10(c0, c1, philox_keys(k0, k1));
}

// The same generator for many counters (t, c1) of one row t.  With x2 = x3 = 0
// at the start, the words that rounds 1-3 compute from t alone are the same for
// every c1; they are computed once per row here, and philox_10_row finishes the
// rest (two products and four XORs fewer per call than philox_10).
struct PhiloxRow {
    uint32_t a2, b3, c0, d1k, e2, f3;   // round 1: x2, x3; round 2: x0, x1 ^ k0[2]; round 3: x2 part, x3
};

__device__ __forceinline__ PhiloxRow philox_row(uint32_t t, const PhiloxKeys& K) {
    PhiloxRow R;
    const uint64_t p0 = static_cast<uint64_t>(t) * 0xD2511F53u;              // round 1: x0 * M0
    R.a2 = static_cast<uint32_t>(p0 >> 32) ^ K.k1[0];                        // round 1: x2
    R.b3 = static_cast<uint32_t>(p0);                                         // round 1: x3
    const uint64_t p1 = static_cast<uint64_t>(R.a2) * 0xCD9E8D57u;           // round 2: x2 * M1
    R.c0 = static_cast<uint32_t>(p1 >> 32) ^ K.k0[1];                        // round 2: x0 (x1 was 0)
    R.d1k = static_cast<uint32_t>(p1) ^ K.k0[2];                             // round 2: x1, with round 3's key
    const uint64_t q0 = static_cast<uint64_t>(R.c0) * 0xD2511F53u;           // round 3: x0 * M0
    R.e2 = static_cast<uint32_t>(q0 >> 32) ^ K.k1[2];                        // round 3: x2 = this ^ x3
    R.f3 = static_cast<uint32_t>(q0);                                         // round 3: x3
    return R;
}

__device__ __forceinline__ uint4 philox_10_row(const PhiloxRow& R, uint32_t c1, const PhiloxKeys& K) {
    // round 1: x0 = c1 ^ k0[0], x1 = 0, x2 = a2, x3 = b3
    const uint32_t y0 = c1 ^ K.k0[0];
    // round 2: x2 = hi(y0 * M0) ^ b3 ^ k1[1], x3 = lo(y0 * M0); x0, x1 per row
    const uint64_t p0 = static_cast<uint64_t>(y0) * 0xD2511F53u;
    const uint32_t z2 = static_cast<uint32_t>(p0 >> 32) ^ R.b3 ^ K.k1[1];
    const uint32_t z3 = static_cast<uint32_t>(p0);
    // round 3: x0 = hi(z2 * M1) ^ x1 ^ k0[2], x1 = lo(z2 * M1), x2 = e2 ^ z3, x3 = f3
    const uint64_t p1 = static_cast<uint64_t>(z2) * 0xCD9E8D57u;
    uint32_t x0 = static_cast<uint32_t>(p1 >> 32) ^ R.d1k;
    uint32_t x1 = static_cast<uint32_t>(p1);
    uint32_t x2 = R.e2 ^ z3;
    uint32_t x3 = R.f3;
#pragma unroll
    for (int r = 3; r < 10; ++r) {
        const uint64_t q0 = static_cast<uint64_t>(x0) * 0xD2511F53u;
        const uint64_t q1 = static_cast<uint64_t>(x2) * 0xCD9E8D57u;
        x0 = static_cast<uint32_t>(q1 >> 32) ^ x1 ^ K.k0[r];
        x1 = static_cast<uint32_t>(q1);
        x2 = static_cast<uint32_t>(q0 >> 32) ^ x3 ^ K.k1[r];
        x3 = static_cast<uint32_t>(q0);
    }
    return make_uint4(x0, x1, x2, x3);
}

// Constants of the keep test lane >= T (0 < T <= 65536) written as a carry:
// lane + (65536 - T) carries out of the lane's 16 bits exactly when it keeps.
struct KeepTest {
    uint32_t low, top;   // low 15 bits and top bit of 65536 - T, in both 16-bit lanes
};

__device__ __forceinline__ KeepTest keep_test(uint32_t T) {
    const uint32_t c = 65536u - T;
    return KeepTest{(c & 0x7FFFu) * 0x10001u, (c & 0x8000u) * 0x10001u};
}

// The keep decisions of one Philox word as a carry: bit 15 set iff the low
// lane is >= T, bit 31 iff the high lane is (see apply_keep_fast).
__device__ __forceinline__ uint32_t keep_carry(uint32_t w, const KeepTest& kt) {
    const uint32_t s = (w & 0x7FFF7FFFu) + kt.low;
    return (w & kt.top) | (w & s) | (kt.top & s);
}

// AND mask of a packed bf16 pair from keep_carry: each carry bit spread over its lane.
__device__ __forceinline__ uint32_t carry_mask(uint32_t carry) {
    uint32_t m;
    asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(m) : "r"(carry));
    return m;
}

// The two keep bits of keep_carry, or of an AND mask (bits 15 and 31 mark the
// lanes that keep in both): bit 0 the low lane, bit 1 the high lane.
__device__ __forceinline__ uint32_t carry_bits(uint32_t carry) { return ((carry >> 15) & 1u) | ((carry >> 30) & 2u); }

// Zeroes the dropped elements of a packed bf16 pair: the low 15 bits of both
// lanes are added without crossing lanes, the carry out of each lane is the
// majority of its top bits and the carry into them, and a byte permute spreads
// each carry (bits 15, 31) over its lane.
__device__ __forceinline__ uint32_t apply_keep_fast(uint32_t data, uint32_t w, const KeepTest& kt) {
    const uint32_t s = (w & 0x7FFF7FFFu) + kt.low;
    const uint32_t carry = (w & kt.top) | (w & s) | (kt.top & s);
    uint32_t m;
    asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(m) : "r"(carry));
    return data & m;
}

// The keep test lane >= T in one of two exact forms, picked per adapter.
//  - half form, for 1 <= T <= 0x7BFF (drop rates up to 0.484): a lane whose
//    top bit is set keeps (it is >= 0x8000 > T); any other lane, read as an
//    IEEE half, is a positive number, +inf or a NaN, and keeps iff it compares
//    greater-or-equal-or-unordered with T read as a half: finite positive
//    halves order like their bit patterns, and +inf and every NaN pattern lie
//    above 0x7BFF.  One f16x2 compare (set.geu gives 0xFFFF per true half)
//    and one byte permute that spreads each lane's top bit.
//  - carry form (keep_carry), for every other T.
struct KeepForm {
    KeepTest kt;       // carry form constants
    uint32_t TT;       // T in both 16-bit halves (half form)
    bool half;
};

__device__ __forceinline__ KeepForm keep_form(uint32_t T) {
    KeepForm f;
    f.kt = keep_test(T);
    f.TT = T * 0x10001u;
    f.half = T >= 1u && T <= 0x7BFFu;
    return f;
}

// AND mask of one Philox word: 0xFFFF over each 16-bit lane that keeps.
template <bool kHalf>
__device__ __forceinline__ uint32_t keep_word_mask(uint32_t w, const KeepForm& f) {
    uint32_t m;
    if (kHalf) {
        uint32_t ge;
        asm("set.geu.u32.f16x2 %0, %1, %2;" : "=r"(ge) : "r"(w), "r"(f.TT));
        asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(m) : "r"(w));
        m |= ge;
    } else {
        m = carry_mask(keep_carry(w, f.kt));
    }
    return m;
}

// AND masks of the eight features of one Philox call (row t, counter word g).
template <bool kHalf>
__device__ __forceinline__ uint4 keep_chunk_mask(const PhiloxRow& R, uint32_t g, const PhiloxKeys& K,
                                                 const KeepForm& f) {
    const uint4 w = philox_10_row(R, g, K);
    return make_uint4(keep_word_mask<kHalf>(w.x, f), keep_word_mask<kHalf>(w.y, f), keep_word_mask<kHalf>(w.z, f),
                      keep_word_mask<kHalf>(w.w, f));
}

// The eight keep bits of a chunk's AND masks (bit e = element e).
__device__ __forceinline__ uint32_t chunk_mask_bits(uint4 m) {
    return carry_bits(m.x) | (carry_bits(m.y) << 2) | (carry_bits(m.z) << 4) | (carry_bits(m.w) << 6);
}

__device__ __forceinline__ uint4 and4(uint4 v, uint4 m) { return make_uint4(v.x & m.x, v.y & m.y, v.z & m.z, v.w & m.w); }

// AND mask of 32-bit word w (elements 2w, 2w + 1) of a 16-byte chunk whose
// eight keep bits are the low byte of `bits` (bit e = element e).
__device__ __forceinline__ uint32_t keep_mask_word(uint32_t bits, int w) {
    const uint32_t lo = 0u - ((bits >> (2 * w)) & 1u);
    const uint32_t hi = 0u - ((bits >> (2 * w + 1)) & 1u);
    return (lo & 0x0000FFFFu) | (hi & 0xFFFF0000u);
}

// One Philox word covers two bf16 elements: the low 16-bit lane decides the
// element in the low half of a packed pair, the high lane the high half.
// Returns an AND mask that keeps the element bits where lane >= T.
__device__ __forceinline__ uint32_t keep_pair_mask(uint32_t w, uint32_t T) {
    const uint32_t lo = ((w & 0xFFFFu) >= T) ? 0x0000FFFFu : 0u;
    const uint32_t hi = ((w >> 16) >= T) ? 0xFFFF0000u : 0u;
    return lo | hi;
}

// Zeroes the dropped elements of a packed bf16 pair.
__device__ __forceinline__ uint32_t apply_keep(uint32_t data, uint32_t w, uint32_t T) {
    if ((w & 0xFFFFu) < T) data &= 0xFFFF0000u;
    if ((w >> 16) < T) data &= 0x0000FFFFu;
    return data;
}

// Walks units u = slot * nblk + blk (slot: an active tile, blk: a block of the
// other dimension) from u0 on, in order, without a division per unit; the
// slot's tile and adapter are looked up once per slot.  Every role of a kernel
// walks the same sequence with its own copy.
struct TileBlockIter {
    int slot, blk, nblk, tile, a;
    __device__ __forceinline__ TileBlockIter(int64_t u0, int nblk_, const Routing& rt) : nblk(nblk_) {
        slot = static_cast<int>(u0 / nblk_);
        blk = static_cast<int>(u0 - static_cast<int64_t>(slot) * nblk_);
        load(rt);
    }
    __device__ __forceinline__ void load(const Routing& rt) {
        if (slot < rt.n_active) {
            tile = rt.active_tiles[slot];
            a = rt.tile_adapter[tile];
        }
    }
    __device__ __forceinline__ void next(const Routing& rt) {
        if (++blk == nblk) {
            blk = 0;
            ++slot;
            load(rt);
        }
    }
};

// Eight keep bits (bit e = element e of the 8-group).
__device__ __forceinline__ uint32_t keep_byte(uint4 w, uint32_t T) {
    uint32_t b = 0;
    b |= ((w.x & 0xFFFFu) >= T) ? 0x01u : 0u;
    b |= ((w.x >> 16) >= T) ? 0x02u : 0u;
    b |= ((w.y & 0xFFFFu) >= T) ? 0x04u : 0u;
    b |= ((w.y >> 16) >= T) ? 0x08u : 0u;
    b |= ((w.z & 0xFFFFu) >= T) ? 0x10u : 0u;
    b |= ((w.z >> 16) >= T) ? 0x20u : 0u;
    b |= ((w.w & 0xFFFFu) >= T) ? 0x40u : 0u;
    b |= ((w.w >> 16) >= T) ? 0x80u : 0u;
    return b;
}

// ---------------------------------------------------------------------------
// finishing fp32 accumulators
// ---------------------------------------------------------------------------

// The per-row routing the finalize kernels look up for every element: the adapter of each tile and each
// adapter's rank and scale, copied once per CTA from the kernel's parameters into shared memory (a lookup
// with a per-thread index in parameter space is far slower than one in shared memory).
struct RowRouting {
    int8_t owner[kMaxTiles];
    int16_t active[kMaxTiles];   // tile -> its index in the active tile list (tiles with an adapter)
    int32_t rank[kMaxAdapters];
    float scale[kMaxAdapters];
};

__device__ __forceinline__ void load_row_routing(RowRouting& s, const Routing& rt) {
    for (int i = threadIdx.x; i < rt.n_tiles; i += blockDim.x) s.owner[i] = rt.tile_adapter[i];
    for (int i = threadIdx.x; i < rt.n_active; i += blockDim.x) s.active[rt.active_tiles[i]] = static_cast<int16_t>(i);
    if (threadIdx.x < kMaxAdapters) {
        s.rank[threadIdx.x] = rt.ad[threadIdx.x].rank;
        s.scale[threadIdx.x] = rt.ad[threadIdx.x].scale;
    }
    __syncthreads();
}

// Four fp32 accumulators read from L2 (written there by reductions).
__device__ __forceinline__ float4 ld_l2_f4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

__device__ __forceinline__ void st_zero_f4(float* p) {
    *reinterpret_cast<float4*>(p) = make_float4(0.f, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ void st_f4(float* p, float a, float b, float c, float d) {
    *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}

// Row `row` (of 128), columns c0 .. c0 + 7, of item `item` whose units are [b, e): its slots added in CTA
// order.  Each slot element read is cleared (the producers wrote exactly the elements their finalize reads),
// so the workspace is zero again after the call, whatever layout the next call puts over these bytes.
__device__ __forceinline__ void slot_sum8(const Slots& sl, int64_t item, int64_t b, int64_t e, int row, int c0,
                                          float (&v)[8]) {
#pragma unroll
    for (int x = 0; x < 8; ++x) v[x] = 0.f;
    const int c_lo = slot_cta(b, sl.units, sl.grid), c_hi = slot_cta(e - 1, sl.units, sl.grid);
    for (int c = c_lo; c <= c_hi; ++c) {
        float* src = sl.base + ((item + c) * 128 + row) * static_cast<int64_t>(sl.ld) + c0;
        const float4 x = ld_l2_f4(src);
        const float4 y = ld_l2_f4(src + 4);
        st_zero_f4(src);
        st_zero_f4(src + 4);
        v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w; v[4] += y.x; v[5] += y.y; v[6] += y.z; v[7] += y.w;
    }
}

__device__ __forceinline__ uint16_t bf16_bits(float v) { return static_cast<uint16_t>(pack_bf16x2(v, 0.f) & 0xFFFFu); }

// Eight sums -> bf16: out[e] = scale * v[e] for e < valid, 0 for valid <= e < 8.
__device__ __forceinline__ void store_row8(uint16_t* out, const float (&v)[8], int valid, float scale) {
    float w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) w[e] = e < valid ? v[e] * scale : 0.f;
    stg128(out, make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]), pack_bf16x2(w[4], w[5]),
                           pack_bf16x2(w[6], w[7])));
}

// Row of an fp32 accumulator -> bf16 row: out[c] = scale * acc[c] for c < valid,
// 0 for valid <= c < width; the accumulator row is zeroed.  width % 8 == 0.
__device__ __forceinline__ void finish_row(float* acc, uint16_t* out, int valid, int width, float scale) {
    for (int c0 = 0; c0 < width; c0 += 8) {
        float v[8];
        if (c0 < valid) {
            const float4 a = ld_l2_f4(acc + c0);
            const float4 b = ld_l2_f4(acc + c0 + 4);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            st_zero_f4(acc + c0);
            st_zero_f4(acc + c0 + 4);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = (c0 + e < valid) ? v[e] * scale : 0.f;
        uint4 pk;
        pk.x = pack_bf16x2(v[0], v[1]);
        pk.y = pack_bf16x2(v[2], v[3]);
        pk.z = pack_bf16x2(v[4], v[5]);
        pk.w = pack_bf16x2(v[6], v[7]);
        stg128(out + c0, pk);
    }
}

// ---------------------------------------------------------------------------
// CTA prologue / epilogue helpers shared by the warp-specialised kernels
// ---------------------------------------------------------------------------

// Rounds a dynamic shared-memory pointer up to 1024 bytes (swizzle atoms).
__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
    const uint32_t a = smem_u32(p);
    return p + ((1024u - (a & 1023u)) & 1023u);
}

}  // namespace lora
