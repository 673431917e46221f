// Tensor-core variant with the roles of x and W swapped: y^T = W . x^T.
//
// One mma.sync m16n8k16 (BF16 in, FP32 accumulation) computes
// D[16 x 8] += A[16 x 16] . B[16 x 8] with A = x (rows m < M, zero-padded to
// 16) and B = a 16-k slice of 8 consecutive rows of W.  Compared with the
// W-as-A kernel (skinny_mma.cuh) a tile is 8 rows instead of 16, which halves
// the granularity of the work split on the 2048..4096-row decode shapes, and
// each lane streams 16 contiguous bytes of a single row per step.
//
// One warp step covers a k-block of 32 elements of the tile's 8 rows (512 B):
//  * lane = 4*g + c loads W[row g][kb + 8c .. +8].  The 8 physical k are
//    mapped onto the fragment's logical k slots: MMA 0 takes kb+8c+{0,1} as
//    slots {2c,2c+1} and kb+8c+{2,3} as {2c+8,2c+9}; MMA 1 the same with
//    kb+8c+{4..7}.  B's fragment of lane (g, c) is exactly column g at those
//    slots, i.e. the lane's own 16 bytes.
//  * A's fragment of lane (g, c) holds x[g][same slots] (rows g < M) and
//    x[g+8][...] (zero here, since M <= 8): one 16-byte shared-memory load.
//  * D's lane (g, c) ends up with y[m = g][rows 2c, 2c+1 of the tile].
// A CTA of NW warps works on one tile at a time; warp w takes the k-blocks
// w, w+NW, ... and the NW partial tiles are added in shared memory in warp
// order.  Loads go in batches of U steps over the warp's flat sequence of
// (tile, k-block) steps; with DB two batches alternate between register sets,
// the next issued before the current one is consumed.
//
// The accumulation order depends on (K range, NW) only, never on M.
#pragma once

#include <cuda_bf16.h>

#include "skinny_mma.cuh"

namespace sk {

template <int M, int U, bool DB>
__global__ void __launch_bounds__(kMaxThreads) skinny_mmat_kernel(const __grid_constant__ Params p) {
    static_assert(M >= 1 && M <= 8, "x rows fill the upper half of the A fragment");
    constexpr int TILE = 8;
    extern __shared__ uint4 smem[];

    const bool pdl = (p.flags & kFlagPdl) != 0;
    if (pdl) pdl_launch_dependents();

    const Item &it = p.item[blockIdx.z];
    const int s = blockIdx.y;
    const int k0 = s * p.kps;
    const int kc = min(p.K - k0, p.kps);
    const int nchunk = kc >> 3;
    const int xstride = nchunk + 1;  // +1 chunk: rows of x start in different banks
    uint4 *xs = smem;                // [M][xstride]
    float *red = reinterpret_cast<float *>(smem + M * xstride);  // [2][NW][TILE][M]

    const int NW = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int c = lane & 3;

    const int J = (nchunk + 3) >> 2;  // k-blocks of 32 elements (the last may be partial)
    const int I = (J + NW - 1) / NW;  // steps per warp per tile (uniform over warps)
    const long long T = (p.N + TILE - 1) / TILE;
    const int t_begin = static_cast<int>(T * blockIdx.x / gridDim.x);
    const int t_end = static_cast<int>(T * (blockIdx.x + 1) / gridDim.x);
    const int total = (t_end - t_begin) * I;

    int lt = t_begin, li_ = 0;
    const uint16_t *wrow = nullptr;
    auto row_of = [&](int t) {
        const int n = min(t * TILE + g, p.N - 1);  // rows past N re-read row N-1; dropped
        wrow = it.W + static_cast<long long>(n) * p.K + k0 + 8 * c;
    };
    if (total > 0) row_of(lt);

    using Batch = uint4[U];
    auto issue_batch = [&](Batch &w, int base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (base + u < total) {
                const int jb = warp + li_ * NW;
                const bool ok = jb < J && (4 * jb + c) < nchunk;
                w[u] = ok ? ldg_stream(wrow + 32 * jb) : make_uint4(0u, 0u, 0u, 0u);
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
        xs[m * xstride + q] = *reinterpret_cast<const uint4 *>(it.x + m * it.ldx + k0 + 8 * q);
    }
    __syncthreads();

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int ct = t_begin, ci = 0, rb = 0;
    auto consume_batch = [&](const Batch &w, int base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (base + u < total) {
                const int jb = warp + ci * NW;
                if (jb < J) {
                    uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                    if (g < M && (4 * jb + c) < nchunk) xv = xs[g * xstride + 4 * jb + c];
                    const uint32_t a0[4] = {xv.x, 0u, xv.y, 0u};
                    const uint32_t a1[4] = {xv.z, 0u, xv.w, 0u};
                    mma_bf16_16816(acc, a0, w[u].x, w[u].y);
                    mma_bf16_16816(acc, a1, w[u].z, w[u].w);
                }
                if (++ci == I) {
                    // tile done: this warp's partial y[m][8 rows] -> shared memory, then
                    // the first 8*M threads add the NW partials in warp order
                    float *rw = red + (rb * NW + warp) * TILE * M;
                    if (g < M) {
                        rw[(2 * c) * M + g] = acc[0];
                        rw[(2 * c + 1) * M + g] = acc[1];
                    }
                    __syncthreads();
                    if (threadIdx.x < TILE * M) {
                        const int row = threadIdx.x / M;
                        const int m = threadIdx.x - row * M;
                        const int n = ct * TILE + row;
                        const float *rr = red + rb * NW * TILE * M + row * M + m;
                        float v = 0.0f;
                        for (int ww = 0; ww < NW; ++ww) v += rr[ww * TILE * M];
                        if (n < p.N) {
                            if (p.split == 1) {
                                store_out(p, it, m, n, v);
                            } else {
                                const long long slot =
                                    (static_cast<long long>(blockIdx.z) * p.split + s) * M + m;
                                p.ws[slot * p.N + n] = v;
                            }
                        }
                    }
                    acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
                    ci = 0;
                    ++ct;
                    rb ^= 1;
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
