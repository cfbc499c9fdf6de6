// Host-side launchers of the kernels (one translation unit per kernel family).
#pragma once
#include <algorithm>

#include <cstddef>
#include <utility>
#include <cuda_runtime.h>

#include "plan.h"

namespace lora {

// Launches a kernel on `stream` with programmatic stream serialization: it may
// start while the previous kernel on the stream finishes, and waits for it with
// griddepcontrol.wait before touching global memory.
//
// `pdl` false gives a plain launch.  A kernel whose stream waits on another
// stream's event just before it is launched plainly: with the attribute it
// could start once the previous kernel of its own stream triggers, before the
// other stream's work is done.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    return launch_k(true, kernel, grid, block, smem, stream, std::forward<Args>(args)...);
}

// Dynamic shared memory a kernel may request; leaves room for its few bytes
// of static shared memory under the 227 KB per-block limit.
constexpr int kMaxDynSmem = 225 * 1024;
// Stage ring budget of the rank-r kernels (stages * stage bytes).
constexpr int kStageBudget = 220 * 1024;
// down_proj and da mask their stages in groups of four warps that take the ring's stages in turn.  Their
// rings hold a multiple of the group count, so that every stage belongs to one group: a group then never
// waits on a stage another group may still be working through, and a parity wait can never see the
// completion of a phase two behind.
constexpr int kMaskGroups = 2;

inline int mask_ring_stages(size_t stage_bytes, int max_stages, int groups = kMaskGroups) {
    int s = static_cast<int>(std::min<size_t>(static_cast<size_t>(max_stages), kStageBudget / stage_bytes));
    return s - s % groups;
}

size_t down_smem_bytes(const DownParams& p);
cudaError_t down_configure();
cudaError_t launch_down(const DownParams& p, int grid, cudaStream_t stream);
cudaError_t launch_finalize_s(const DownParams& p, int sms, cudaStream_t stream);

// CTA-pair GEMM (cta_group::2): forward 256 x 256 tiles (two accumulator
// buffers); backward 256 x kBwdPairBN (acc1 + acc2 fill TMEM: one buffer).
constexpr int kBwdPairBN = 256;
cudaError_t gemm2_configure();
// Grid and split tiles for a call (p.M, p.N, p.nkb set); `allow_split` false when the workspace has no
// partial slots.  The launch takes p.sk_tiles as set from it and the schedule's pair count.
GemmSched plan_gemm2(const GemmParams& p, bool bwd, int bn, int sms, bool allow_split);
cudaError_t launch_gemm2(const GemmParams& p, bool bwd, int bn, int pairs, cudaStream_t stream);

size_t dsdb_smem_bytes(const DsDbParams& p);
cudaError_t dsdb_configure();
cudaError_t launch_dsdb(const DsDbParams& p, int grid, cudaStream_t stream);
// finalize_bwd1 parts: dSq from dS (the dX GEMM and dA need it) and dB from dB^T (an output only).
constexpr int kPartDs = 1, kPartDb = 2;
// The strip order issues its MMAs from four threads up to padded rank 64 when it flushes both products: two
// dS accumulators per buffer leave TMEM for four n-blocks a strip (columns / rpad - 4) instead of six
// (columns / rpad - 2).  The host sizes the strip and launch_dsdb picks the kernel by the same test.
inline bool strip_four_issuers(int rpad_max, int parts) { return rpad_max <= 64 && parts == (kPartDs | kPartDb); }
cudaError_t launch_finalize_bwd1(const DsDbParams& p, int parts, int sms, cudaStream_t stream, bool pdl = true);

size_t da_smem_bytes(const DaParams& p);
cudaError_t da_configure();
cudaError_t launch_da(const DaParams& p, int grid, cudaStream_t stream, bool pdl = true);
cudaError_t launch_finalize_da(const DaParams& p, int sms, cudaStream_t stream, bool pdl = true);

cudaError_t launch_stuck_wait(DevCtl ctl, cudaStream_t stream);

// DoRA pieces (k_dora.cu); the dA kernel also computes DoRA's U = W^T A.
cudaError_t dora_configure();
cudaError_t launch_dora_norm2(const uint16_t* W, int64_t k, int64_t n, float* out, int sms, cudaStream_t stream);
cudaError_t launch_dora_gram(const uint16_t* A, int64_t k, int r, float* G, cudaStream_t stream);
cudaError_t launch_dora_scale(float* U, int rpad, const uint16_t* B, const float* G, int r, const float* wn2,
                              const float* mag, float alpha, int64_t n, float* g_out, cudaStream_t stream);
cudaError_t launch_dora_dz(const uint16_t* dY, const uint16_t* Y, const float* g, int64_t m, int64_t n, uint16_t* dZ,
                           float* dmag_acc, int sms, cudaStream_t stream);
cudaError_t launch_dora_dmag(float* dmag_acc, const float* mag, int64_t n, float* dmag, cudaStream_t stream);

}  // namespace lora
