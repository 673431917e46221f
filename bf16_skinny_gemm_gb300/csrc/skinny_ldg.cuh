// Weight-streaming BF16 skinny GEMM for sm_103a: y[M,N] = x[M,K] . W[N,K]^T.
//
// The operation and its cost model come from vLLM PR #62949 ("SM121
// skinny-GEMM plans for the GLM-5.3-Flash BF16 decode projections", Validation:
// decode reads each weight once per step, so the GEMM is a stream over W) and
// vLLM PR #65306 ("Add SM90 skinny GEMM plans ...", Details: the kernel
// launches N / outputs_per_block CTAs and needs no reduce kernel, unlike the
// library GEMM's split-K + reduce).  The design here is our own for GB300:
//
//  * W is read exactly once, with 128-bit non-allocating loads
//    (ld.global.nc.L1::no_allocate), U loads per row per lane in flight so that
//    enough bytes are outstanding to cover HBM latency.
//  * x (all M rows of this CTA's K range) is staged once per CTA in shared
//    memory and re-read from there for every row: it is tiny next to W.
//  * A warp is split into 32/LPR lane groups; each group owns R rows and walks
//    their K range with stride LPR chunks of 8 elements.  Each lane keeps M*R
//    FP32 accumulators; products are exact in FP32 and added with FMA.
//  * Lane partial sums are combined with an xor-butterfly of warp shuffles
//    (fixed order).  With split-K (gridDim.y > 1) each split writes FP32
//    partials and a second kernel adds them in split order.
//  * The grid is sized for the GPU (SMs x resident CTAs) and each CTA takes a
//    balanced contiguous range of row groups, so every SM streams an equal
//    share of W.
//
// Accumulation order for one output is a function of (K range, LPR) only: it
// never depends on M, R, U, the CTA size or the grid, which makes results
// deterministic and row-wise independent of M.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"

namespace sk {

// 16 bytes of W, streamed: no L1 allocation, 256-byte L2 prefetch granule.
__device__ __forceinline__ uint4 ldg_stream(const uint16_t *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// BF16 -> FP32 is exact: the BF16 bits are the top half of the FP32 bits.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// acc[m] += sum over the 8 elements of one chunk, in element order.
template <int M, int R>
__device__ __forceinline__ void fma_chunk(float (&acc)[M][R], const float (&xf)[M][8],
                                          const uint4 &w, int r) {
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float w0 = bf16_lo(ww[i]);
        const float w1 = bf16_hi(ww[i]);
#pragma unroll
        for (int m = 0; m < M; ++m) {
            acc[m][r] = fmaf(xf[m][2 * i], w0, acc[m][r]);
            acc[m][r] = fmaf(xf[m][2 * i + 1], w1, acc[m][r]);
        }
    }
}

template <int M>
__device__ __forceinline__ void unpack_x(float (&xf)[M][8], const uint4 *xs, int nchunk, int c) {
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint4 v = xs[m * nchunk + c];
        const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            xf[m][2 * i] = bf16_lo(vv[i]);
            xf[m][2 * i + 1] = bf16_hi(vv[i]);
        }
    }
}

template <int M, int R, int LPR, int U>
__global__ void __launch_bounds__(kMaxThreads) skinny_ldg_kernel(const __grid_constant__ Params p) {
    static_assert(LPR == 32 || LPR == 16 || LPR == 8, "lanes per row");
    constexpr int G = 32 / LPR;  // lane groups per warp
    extern __shared__ uint4 xs[];  // [M][nchunk] chunks of 8 BF16

    const Item &it = p.item[blockIdx.z];
    const int s = blockIdx.y;
    const int k0 = s * p.kps;
    const int kc = min(p.K - k0, p.kps);
    const int nchunk = kc >> 3;

    // stage x[:, k0:k0+kc] in shared memory
    for (int i = threadIdx.x; i < M * nchunk; i += blockDim.x) {
        const int m = i / nchunk;
        const int c = i - m * nchunk;
        xs[i] = *reinterpret_cast<const uint4 *>(it.x + m * it.ldx + k0 + 8 * c);
    }
    __syncthreads();

    const int warps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gi = lane / LPR;  // lane group
    const int li = lane % LPR;  // lane in group

    // balanced contiguous range of row groups for this CTA
    const long long RG = p.row_groups;
    const int g_begin = static_cast<int>(RG * blockIdx.x / gridDim.x);
    const int g_end = static_cast<int>(RG * (blockIdx.x + 1) / gridDim.x);
    const int jfull = nchunk / LPR;      // iterations with every lane of the group busy
    const int rem = nchunk - jfull * LPR;  // chunks of the final partial iteration

    for (int g = g_begin + warp; g < g_end; g += warps) {
        const int n0 = (g * G + gi) * R;
        const uint16_t *wr[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int n = min(n0 + r, p.N - 1);  // rows past N re-read row N-1; result dropped
            wr[r] = it.W + static_cast<long long>(n) * p.K + k0 + 8 * li;
        }
        float acc[M][R];
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) acc[m][r] = 0.0f;

        int j = 0;
        for (; j + U <= jfull; j += U) {
            uint4 w[U][R];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int r = 0; r < R; ++r) w[u][r] = ldg_stream(wr[r] + 8 * LPR * (j + u));
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float xf[M][8];
                unpack_x<M>(xf, xs, nchunk, li + LPR * (j + u));
#pragma unroll
                for (int r = 0; r < R; ++r) fma_chunk<M, R>(acc, xf, w[u][r], r);
            }
        }
        for (; j < jfull; ++j) {
            uint4 w[R];
#pragma unroll
            for (int r = 0; r < R; ++r) w[r] = ldg_stream(wr[r] + 8 * LPR * j);
            float xf[M][8];
            unpack_x<M>(xf, xs, nchunk, li + LPR * j);
#pragma unroll
            for (int r = 0; r < R; ++r) fma_chunk<M, R>(acc, xf, w[r], r);
        }
        if (li < rem) {
            uint4 w[R];
#pragma unroll
            for (int r = 0; r < R; ++r) w[r] = ldg_stream(wr[r] + 8 * LPR * jfull);
            float xf[M][8];
            unpack_x<M>(xf, xs, nchunk, li + LPR * jfull);
#pragma unroll
            for (int r = 0; r < R; ++r) fma_chunk<M, R>(acc, xf, w[r], r);
        }

        // xor-butterfly over the LPR lanes of the group (fixed tree order)
#pragma unroll
        for (int m = 0; m < M; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float v = acc[m][r];
#pragma unroll
                for (int off = LPR / 2; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                acc[m][r] = v;
            }

        if (li == 0) {
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const int n = n0 + r;
                if (n < p.N) {
#pragma unroll
                    for (int m = 0; m < M; ++m) {
                        if (p.split == 1) {
                            it.y[m * it.ldy + n] = f32_to_bf16_rn(acc[m][r]);
                        } else {
                            const long long slot =
                                ((static_cast<long long>(blockIdx.z) * p.split + s) * M + m);
                            p.ws[slot * p.N + n] = acc[m][r];
                        }
                    }
                }
            }
        }
    }
}

// Second pass of split-K: y = RNE_bf16(sum over splits, in split order).
template <int M>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const __grid_constant__ Params p,
                                                             int batch) {
    const long long per_item = static_cast<long long>(M) * p.N;
    const long long total = per_item * batch;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int b = static_cast<int>(i / per_item);
        const long long mn = i - b * per_item;
        const int m = static_cast<int>(mn / p.N);
        const int n = static_cast<int>(mn - static_cast<long long>(m) * p.N);
        const float *src = p.ws + (static_cast<long long>(b) * p.split * M + m) * p.N + n;
        float acc = 0.0f;
        for (int s = 0; s < p.split; ++s) acc += src[static_cast<long long>(s) * M * p.N];
        const Item &it = p.item[b];
        it.y[m * it.ldy + n] = f32_to_bf16_rn(acc);
    }
}

}  // namespace sk
