// Tensor-core skinny GEMM with warp-owned tiles (sm_103a):
// y[M,N] = x[M,K] . W[N,K]^T, M <= 8, BF16 in, FP32 accumulation, BF16 out.
//
// The math is that of skinny_mmat.cuh: x is the A operand of mma.sync
// m16n8k16 (rows m < M, zero-padded to 16), 8 rows of W the B operand, and
// lane (g, c) streams W[row g][kb + 8c .. +8] (16 contiguous bytes) for each
// 32-element k-block kb; its 8 physical k are mapped onto the fragment's k
// slots and x uses the same map.  D's lane (g, c) ends up with y[m = g][tile
// rows 2c, 2c+1], so a warp that owns a whole tile writes y straight from its
// fragment.
//
// What differs is who owns what.  In skinny_mma(t).cuh every warp of a CTA
// takes a share of each tile's k-blocks and the CTA meets at a barrier at
// every tile end, so it advances at the pace of its slowest warp's memory
// latency.  Here the warps of a CTA form groups of KS (= p.split: 1, 2, 4 or 8)
// warps; the tiles are shared out evenly over all groups of the grid, and
// warp `part` of a group streams k-blocks [J*part/KS, J*(part+1)/KS) of each of
// its group's tiles, a contiguous stretch of K.  With KS = 1 a warp owns whole
// tiles and never waits for another warp after x is staged; with KS > 1 the KS
// partial fragments of a tile meet in shared memory at a named barrier of the
// group only (double-buffered, so one barrier per tile) and part 0 adds them
// in part order.  Like the CUDA-core streaming kernel, warps run on their own:
// the grid is balanced per warp, not per SM.
//
// No scratch, no second pass, no waits outside the CTA.  The accumulation
// order depends on (K, KS) only, never on M, the grid or the data.
#pragma once

#include <cuda_bf16.h>

#include "skinny_mma.cuh"

namespace sk {

template <int M, int U, bool DB>
__global__ void __launch_bounds__(kMaxThreads) skinny_mmatw_kernel(const __grid_constant__ Params p) {
    static_assert(M >= 1 && M <= 8, "x rows fill the upper half of the A fragment");
    constexpr int TILE = 8;
    extern __shared__ uint4 smem[];

    const bool pdl = (p.flags & kFlagPdl) != 0;
    if (pdl) pdl_launch_dependents();

    const Item &it = p.item[blockIdx.z];
    const int nchunk = p.K >> 3;     // 16-byte chunks of a row
    const int xstride = nchunk + 1;  // x row stride in chunks (+1: rows start in different banks)
    uint4 *xs = smem;                // [M][xstride]
    float *red = reinterpret_cast<float *>(smem + M * xstride);  // [2][NW][32 lanes][2]

    const int NW = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int c = lane & 3;

    const int KS = p.split;  // warps sharing each tile's K range (divides NW, <= J)
    const int group = warp / KS;
    const int part = warp - group * KS;
    const int groups = NW / KS;

    const int J = (nchunk + 3) >> 2;            // 32-element k-blocks of a row
    const int j0 = J * part / KS;               // this warp's k-blocks of every tile
    const int I = J * (part + 1) / KS - j0;     // >= 1 since KS <= J
    const long long T = (p.N + TILE - 1) / TILE;
    const long long GG = static_cast<long long>(gridDim.x) * groups;
    const long long gg = static_cast<long long>(blockIdx.x) * groups + group;
    const int t_begin = static_cast<int>(T * gg / GG);
    const int t_end = static_cast<int>(T * (gg + 1) / GG);
    const int total = (t_end - t_begin) * I;    // this warp's steps

    int lt = t_begin, li_ = 0;
    const uint16_t *wrow = nullptr;
    auto row_of = [&](int t) {
        const int n = min(t * TILE + g, p.N - 1);  // rows past N re-read row N-1; dropped
        wrow = it.W + static_cast<long long>(n) * p.K + 8 * c + 32 * j0;
    };
    if (total > 0) row_of(lt);

    using Batch = uint4[U];
    auto issue_batch = [&](Batch &w, int base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (base + u < total) {
                const bool ok = 4 * (j0 + li_) + c < nchunk;
                w[u] = ok ? ldg_stream(wrow + 32 * li_) : make_uint4(0u, 0u, 0u, 0u);
                if (++li_ == I) {
                    li_ = 0;
                    if (++lt < t_end) row_of(lt);
                }
            }
        }
    };

    Batch wA, wB;
    const bool early_w = !pdl || (p.flags & kFlagWeightsReadOnly);
    // with read-only weights, both batches of a double-buffered plan go out before
    // the wait for the previous kernel (the same order the loop below would use)
    const bool pre_b = DB && early_w && U < total;
    if (early_w) issue_batch(wA, 0);
    if (pre_b) issue_batch(wB, U);
    if (pdl) pdl_wait();
    if (!early_w) issue_batch(wA, 0);

    for (int i = threadIdx.x; i < M * nchunk; i += blockDim.x) {
        const int m = i / nchunk;
        const int q = i - m * nchunk;
        xs[m * xstride + q] = *reinterpret_cast<const uint4 *>(it.x + m * it.ldx + 8 * q);
    }
    __syncthreads();

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int ct = t_begin, ci = 0, rb = 0;
    auto consume_batch = [&](const Batch &w, int base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (base + u < total) {
                const int j = j0 + ci;
                uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                if (g < M && 4 * j + c < nchunk) xv = xs[g * xstride + 4 * j + c];
                const uint32_t a0[4] = {xv.x, 0u, xv.y, 0u};
                const uint32_t a1[4] = {xv.z, 0u, xv.w, 0u};
                mma_bf16_16816(acc, a0, w[u].x, w[u].y);
                mma_bf16_16816(acc, a1, w[u].z, w[u].w);
                if (++ci == I) {
                    // tile done: lane (g < M, c) holds y[g][8t + 2c], y[g][8t + 2c + 1]
                    float v0 = acc[0], v1 = acc[1];
                    bool write = true;
                    if (KS > 1) {
                        float *rw = red + ((rb * NW + warp) * 32 + lane) * 2;
                        rw[0] = acc[0];
                        rw[1] = acc[1];
                        asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "r"(KS * 32) : "memory");
                        write = part == 0;
                        if (write) {
                            const float *rr = red + ((rb * NW + group * KS) * 32 + lane) * 2;
                            v0 = rr[0];
                            v1 = rr[1];
                            for (int q = 1; q < KS; ++q) {
                                v0 += rr[q * 64];
                                v1 += rr[q * 64 + 1];
                            }
                        }
                        rb ^= 1;
                    }
                    if (write && g < M) {
                        const int n = ct * TILE + 2 * c;
                        if (n < p.N) store_out(p, it, g, n, v0);
                        if (n + 1 < p.N) store_out(p, it, g, n + 1, v1);
                    }
                    acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
                    ci = 0;
                    ++ct;
                }
            }
        }
    };

    if (DB) {
        for (int base = 0; base < total; base += 2 * U) {
            if (base + U < total && !(base == 0 && pre_b)) issue_batch(wB, base + U);
            consume_batch(wA, base);
            if (base + U >= total) break;
            if (base + 2 * U < total) issue_batch(wA, base + 2 * U);
            consume_batch(wB, base + U);
        }
    } else {
        for (int base = 0; base < total; base += U) {
            consume_batch(wA, base);
            if (base + U < total) issue_batch(wA, base + U);
        }
    }
}

}  // namespace sk
