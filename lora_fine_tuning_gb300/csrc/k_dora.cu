// DoRA: the magnitude / direction split of the adapted weight ("Scaling DoRA",
// paper.rainbus.top, method).  In this layer's orientation (Y = X W, W k x n)
//     g_j = mag_j / ||W[:, j] + alpha (A B)[:, j]||,   Y = g * (X W + alpha S B).
// The column norm is never formed from the dense k x n update: with the
// pages' factored identity
//     ||W_j + a (AB)_j||^2 = ||W_j||^2 + 2 a B_j . U_j + a^2 B_j^T G B_j,
//     U = W^T A (n x r),  G = A^T A (r x r),
// it needs ||W_j||^2 (W is frozen: computed once, dora_norm2_kernel), U (the
// dA kernel's contraction with W in the place of X and no mask), and G
// (dora_gram_kernel).  dora_scale_kernel assembles g.  The forward GEMM then
// scales column j of its output by g_j in the epilogue.
//
// Backward, with the norm held constant: dZ = dY * g feeds the LoRA backward,
// and dmag_j = sum_t dY[t, j] Z[t, j] / ||.||_j = sum_t dY[t, j] Y[t, j] / mag_j
// (Y = g Z and g ||.|| = mag).  dora_dz_kernel writes dZ and the column sums
// in one pass over dY and Y; dora_dmag_kernel divides by mag.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace lora {

namespace {

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// ||W[:, j]||^2 += sum over this block's rows; two columns per thread.  out is zeroed first.
__global__ void __launch_bounds__(256) dora_norm2_kernel(const uint16_t* __restrict__ W, int64_t k, int64_t n,
                                                         int64_t rows_per_block, float* __restrict__ out) {
    const int64_t j = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 2;
    if (j >= n) return;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_block;
    const int64_t r1 = min(k, r0 + rows_per_block);
    float s0 = 0.f, s1 = 0.f;
    for (int64_t r = r0; r < r1; ++r) {
        const uint32_t w2 = *reinterpret_cast<const uint32_t*>(W + r * n + j);   // n is even: j, j+1 in range
        const float a = __uint_as_float(w2 << 16), b = __uint_as_float(w2 & 0xFFFF0000u);
        s0 = fmaf(a, a, s0);
        s1 = fmaf(b, b, s1);
    }
    atomicAdd(out + j, s0);
    atomicAdd(out + j + 1, s1);
}

// G += A_blk^T A_blk over this block's 64 rows of A (k x r).  G (r x r) is zeroed first.
__global__ void __launch_bounds__(256) dora_gram_kernel(const uint16_t* __restrict__ A, int64_t k, int r,
                                                        float* __restrict__ G) {
    pdl_wait();
    pdl_trigger();
    __shared__ float a_s[64][kMaxRank + 1];
    const int64_t k0 = static_cast<int64_t>(blockIdx.x) * 64;
    const int rows = static_cast<int>(min(static_cast<int64_t>(64), k - k0));
    for (int i = threadIdx.x; i < 64 * r; i += blockDim.x) {
        const int row = i / r, c = i - row * r;
        a_s[row][c] = row < rows ? bf16_to_f32(A[(k0 + row) * r + c]) : 0.f;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < r * r; e += blockDim.x) {
        const int c = e / r, d = e - c * r;
        float s = 0.f;
        for (int row = 0; row < rows; ++row) s = fmaf(a_s[row][c], a_s[row][d], s);
        atomicAdd(G + e, s);
    }
}

// g_j = mag_j / sqrt(||W_j||^2 + 2 alpha B_j . U_j + alpha^2 B_j^T G B_j).  A block of 256 threads takes
// kScaleCols columns, eight threads per column: thread `part` of column j sums the terms c = part, part + 8,
// ... of  B_cj U_jc  and  B_cj (G B_j)_c , and the eight partial sums meet by warp shuffles.  U's row j is
// cleared (the workspace is zero between calls).  Dynamic shared memory: G (r x r) and the block's columns
// of B (r x kScaleCols), both fp32.
constexpr int kScaleCols = 32;

__global__ void __launch_bounds__(256) dora_scale_kernel(float* __restrict__ U, int rpad, const uint16_t* __restrict__ B,
                                                         const float* __restrict__ G, int r, const float* __restrict__ wn2,
                                                         const float* __restrict__ mag, float alpha, int64_t n,
                                                         float* __restrict__ g_out) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ float sh[];
    float* g_s = sh;              // r x r
    float* b_s = sh + r * r;      // r x kScaleCols (column-local)
    const int64_t j0 = static_cast<int64_t>(blockIdx.x) * kScaleCols;
    for (int i = threadIdx.x; i < r * r; i += blockDim.x) g_s[i] = G[i];
    for (int i = threadIdx.x; i < r * kScaleCols; i += blockDim.x) {
        const int c = i / kScaleCols, jj = i - c * kScaleCols;
        b_s[i] = (j0 + jj < n) ? bf16_to_f32(B[c * n + j0 + jj]) : 0.f;
    }
    __syncthreads();
    const int jj = threadIdx.x >> 3;
    const int part = threadIdx.x & 7;
    const int64_t j = j0 + jj;
    const bool valid = j < n;   // all eight threads of a column agree
    float cross = 0.f, quad = 0.f;
    if (valid) {
        float* u = U + j * rpad;
        for (int c = part; c < r; c += 8) {
            const float bc = b_s[c * kScaleCols + jj];
            cross = fmaf(bc, u[c], cross);
            const float* gc = g_s + c * r;
            float gb0 = 0.f, gb1 = 0.f;
            int d = 0;
            for (; d + 1 < r; d += 2) {
                gb0 = fmaf(gc[d], b_s[d * kScaleCols + jj], gb0);
                gb1 = fmaf(gc[d + 1], b_s[(d + 1) * kScaleCols + jj], gb1);
            }
            if (d < r) gb0 = fmaf(gc[d], b_s[d * kScaleCols + jj], gb0);
            quad = fmaf(bc, gb0 + gb1, quad);
        }
    }
    __syncwarp();   // the column's eight threads have read U's row before any of it is cleared
    if (valid)
        for (int c = 4 * part; c < rpad; c += 32) st_zero_f4(U + j * rpad + c);
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
        cross += __shfl_xor_sync(0xFFFFFFFFu, cross, o);
        quad += __shfl_xor_sync(0xFFFFFFFFu, quad, o);
    }
    if (valid && part == 0) {
        const float norm2 = wn2[j] + 2.f * alpha * cross + alpha * alpha * quad;
        g_out[j] = mag[j] * rsqrtf(fmaxf(norm2, 1e-30f));
    }
}

// dZ = dY * g (bf16) and dmag_acc_j += sum_t dY[t, j] Y[t, j] over this block's rows; eight columns per
// thread (16-byte loads and stores, contiguous across the warp).
__global__ void __launch_bounds__(256) dora_dz_kernel(const uint16_t* __restrict__ dY, const uint16_t* __restrict__ Y,
                                                      const float* __restrict__ g, int64_t m, int64_t n,
                                                      int64_t rows_per_block, uint16_t* __restrict__ dZ,
                                                      float* __restrict__ dmag_acc) {
    pdl_wait();
    pdl_trigger();
    const int64_t j = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
    if (j >= n) return;   // n is a multiple of 8
    float gj[8], acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        gj[e] = g[j + e];
        acc[e] = 0.f;
    }
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per_block;
    const int64_t r1 = min(m, r0 + rows_per_block);
    for (int64_t t = r0; t < r1; ++t) {
        const uint4 dy = __ldcs(reinterpret_cast<const uint4*>(dY + t * n + j));
        const uint4 y = __ldcs(reinterpret_cast<const uint4*>(Y + t * n + j));
        const uint32_t dyw[4] = {dy.x, dy.y, dy.z, dy.w}, yw[4] = {y.x, y.y, y.z, y.w};
        uint32_t out[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float d0 = __uint_as_float(dyw[q] << 16), d1 = __uint_as_float(dyw[q] & 0xFFFF0000u);
            const float y0 = __uint_as_float(yw[q] << 16), y1 = __uint_as_float(yw[q] & 0xFFFF0000u);
            acc[2 * q] = fmaf(d0, y0, acc[2 * q]);
            acc[2 * q + 1] = fmaf(d1, y1, acc[2 * q + 1]);
            out[q] = pack_bf16x2(d0 * gj[2 * q], d1 * gj[2 * q + 1]);
        }
        stg128(dZ + t * n + j, make_uint4(out[0], out[1], out[2], out[3]));
    }
    red_add_v4(dmag_acc + j, acc[0], acc[1], acc[2], acc[3]);
    red_add_v4(dmag_acc + j + 4, acc[4], acc[5], acc[6], acc[7]);
}

// dmag_j = dmag_acc_j / mag_j; the accumulator is cleared.
__global__ void __launch_bounds__(256) dora_dmag_kernel(float* __restrict__ dmag_acc, const float* __restrict__ mag,
                                                        int64_t n, float* __restrict__ dmag) {
    pdl_wait();
    pdl_trigger();
    const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (j >= n) return;
    dmag[j] = dmag_acc[j] / mag[j];
    dmag_acc[j] = 0.f;
}

}  // namespace

cudaError_t dora_configure() {
    return cudaFuncSetAttribute(dora_scale_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (kMaxRank * kMaxRank + kMaxRank * kScaleCols) * 4);
}

cudaError_t launch_dora_norm2(const uint16_t* W, int64_t k, int64_t n, float* out, int sms, cudaStream_t stream) {
    const int cols = static_cast<int>((n / 2 + 255) / 256);
    const int64_t chunks = std::max<int64_t>(1, std::min<int64_t>(k, (4 * sms + cols - 1) / cols));
    const int64_t rows_per = (k + chunks - 1) / chunks;
    dora_norm2_kernel<<<dim3(cols, static_cast<unsigned>((k + rows_per - 1) / rows_per)), 256, 0, stream>>>(
        W, k, n, rows_per, out);
    return cudaGetLastError();
}

cudaError_t launch_dora_gram(const uint16_t* A, int64_t k, int r, float* G, cudaStream_t stream) {
    return launch_pdl(dora_gram_kernel, dim3(static_cast<unsigned>((k + 63) / 64)), dim3(256), 0, stream, A, k, r, G);
}

cudaError_t launch_dora_scale(float* U, int rpad, const uint16_t* B, const float* G, int r, const float* wn2,
                              const float* mag, float alpha, int64_t n, float* g_out, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(r * r + r * kScaleCols) * 4;
    return launch_pdl(dora_scale_kernel, dim3(static_cast<unsigned>((n + kScaleCols - 1) / kScaleCols)), dim3(256), smem, stream, U,
                      rpad, B, G, r, wn2, mag, alpha, n, g_out);
}

cudaError_t launch_dora_dz(const uint16_t* dY, const uint16_t* Y, const float* g, int64_t m, int64_t n, uint16_t* dZ,
                           float* dmag_acc, int sms, cudaStream_t stream) {
    const int cols = static_cast<int>((n / 8 + 255) / 256);
    const int64_t chunks = std::max<int64_t>(1, std::min<int64_t>(m, (8 * sms + cols - 1) / cols));
    const int64_t rows_per = (m + chunks - 1) / chunks;
    return launch_pdl(dora_dz_kernel, dim3(cols, static_cast<unsigned>((m + rows_per - 1) / rows_per)), dim3(256), 0,
                      stream, dY, Y, g, m, n, rows_per, dZ, dmag_acc);
}

cudaError_t launch_dora_dmag(float* dmag_acc, const float* mag, int64_t n, float* dmag, cudaStream_t stream) {
    return launch_pdl(dora_dmag_kernel, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, stream, dmag_acc,
                      mag, n, dmag);
}

}  // namespace lora
