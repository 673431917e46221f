// Tensor-core variant of the weight-streaming skinny GEMM (sm_103a):
// y[M,N] = x[M,K] . W[N,K]^T with M <= 8 padded to the 8 columns of one
// mma.sync m16n8k16 (BF16 inputs, FP32 accumulation).
//
// Why: at M = 4 the CUDA-core kernel spends about 100 instructions per KiB of
// W (operand handling, 4x FMA per element, bookkeeping) and runs at 50-55 %
// issue utilisation on GB300 (ncu: high "not selected" stalls), while two
// m16n8k16 MMAs do a 16-row x 32-k tile in two instructions.  The problem is
// still HBM-bound: the tensor core only removes instruction pressure.
//
// Layout of one warp step (a "k-block" of 32 elements of 16 rows = 1 KiB):
//  * lane = 4*g + c (g = 0..7, c = 0..3) loads 16 contiguous bytes of row g
//    and of row g+8 at k = kb + 8c.  Since the contraction may use any order
//    of k, those 8 physical k are mapped onto the MMA fragment's logical k
//    slots: MMA 0 takes k = kb+8c+{0,1} as slots {2c,2c+1} and kb+8c+{2,3} as
//    {2c+8,2c+9}; MMA 1 the same with kb+8c+{4..7}.  x uses the same map, so
//    one 16-byte shared-memory load of x[g][kb+8c..] gives both B fragments
//    (lanes with g >= M feed zeros).  Each load instruction reads 8 rows x 64
//    contiguous bytes, whole 32-byte sectors.
//  * a CTA of NW warps works on one 16-row tile at a time; warp w takes the
//    k-blocks w, w+NW, w+2NW, ... (the CTA sweeps each row contiguously), and
//    the NW partial tiles are added in shared memory in warp order.
//  * loads are issued in batches of U k-blocks (2U loads per lane) over the
//    warp's flat sequence of (tile, k-block) steps, consumed together; with DB
//    two batches alternate, so a batch is in flight during the tile-end
//    barrier and reduction.
//
// The order of accumulation depends on (K range, NW) only, never on M, so the
// result is deterministic and row-wise independent of M for a given plan.
#pragma once

#include <cuda_bf16.h>

#include "skinny_ldg.cuh"

namespace sk {

template <int M, int U, bool DB = false>
__global__ void __launch_bounds__(kMaxThreads) skinny_mma_kernel(const __grid_constant__ Params p) {
    constexpr int TILE = 16;
    constexpr int MC = M <= 4 ? 4 : 8;  // columns of a partial tile in shared memory
    extern __shared__ uint4 smem[];

    const bool pdl = (p.flags & kFlagPdl) != 0;
    if (pdl) pdl_launch_dependents();

    const Item &it = p.item[blockIdx.z];
    const int s = blockIdx.y;
    const int k0 = s * p.kps;
    const int kc = min(p.K - k0, p.kps);
    const int nchunk = kc >> 3;            // 16-byte chunks of this split's K range
    const int xstride = nchunk + 1;        // x row stride in chunks (+1 avoids bank conflicts)
    uint4 *xs = smem;                      // [M][xstride]
    float *red = reinterpret_cast<float *>(smem + M * xstride);  // [2][NW][TILE][MC]

    const int NW = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int c = lane & 3;

    const int J = (nchunk + 3) >> 2;       // k-blocks of 32 elements (the last may be partial)
    const int I = (J + NW - 1) / NW;       // k-block steps per warp per tile (uniform)
    const long long T = (p.N + TILE - 1) / TILE;
    const int t_begin = static_cast<int>(T * blockIdx.x / gridDim.x);
    const int t_end = static_cast<int>(T * (blockIdx.x + 1) / gridDim.x);
    const int total = (t_end - t_begin) * I;  // this warp's steps (same for every warp)

    // load cursor: tile lt, step li_
    int lt = t_begin, li_ = 0;
    const uint16_t *row_lo = nullptr, *row_hi = nullptr;
    auto rows_of = [&](int t) {
        const int n_lo = min(t * TILE + g, p.N - 1);  // rows past N re-read row N-1; dropped
        const int n_hi = min(t * TILE + g + 8, p.N - 1);
        row_lo = it.W + static_cast<long long>(n_lo) * p.K + k0 + 8 * c;
        row_hi = it.W + static_cast<long long>(n_hi) * p.K + k0 + 8 * c;
    };
    if (total > 0) rows_of(lt);

    struct Batch {
        uint4 lo[U], hi[U];
    };
    auto issue_batch = [&](Batch &b, int base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (base + u < total) {
                const int jb = warp + li_ * NW;
                const bool ok = jb < J && (4 * jb + c) < nchunk;
                b.lo[u] = ok ? ldg_stream(row_lo + 32 * jb) : make_uint4(0u, 0u, 0u, 0u);
                b.hi[u] = ok ? ldg_stream(row_hi + 32 * jb) : make_uint4(0u, 0u, 0u, 0u);
                if (++li_ == I) {
                    li_ = 0;
                    if (++lt < t_end) rows_of(lt);
                }
            }
        }
    };

    Batch bA, bB;
    const bool early_w = !pdl || (p.flags & kFlagWeightsReadOnly);
    // with read-only weights, both batches of a double-buffered plan go out before
    // the wait for the previous kernel (the same order the loop below would use)
    const bool pre_b = DB && early_w && U < total;
    if (early_w) issue_batch(bA, 0);
    if (pre_b) issue_batch(bB, U);
    if (pdl) pdl_wait();
    if (!early_w) issue_batch(bA, 0);

    for (int i = threadIdx.x; i < M * nchunk; i += blockDim.x) {
        const int m = i / nchunk;
        const int q = i - m * nchunk;
        xs[m * xstride + q] = *reinterpret_cast<const uint4 *>(it.x + m * it.ldx + k0 + 8 * q);
    }
    __syncthreads();

    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    int ct = t_begin, ci = 0, rb = 0;  // consume cursor: tile, step, reduction buffer
    auto consume_batch = [&](const Batch &b, int base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (base + u < total) {
                const int jb = warp + ci * NW;
                if (jb < J) {
                    uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                    if (g < M && (4 * jb + c) < nchunk) xv = xs[g * xstride + 4 * jb + c];
                    const uint32_t a0[4] = {b.lo[u].x, b.hi[u].x, b.lo[u].y, b.hi[u].y};
                    const uint32_t a1[4] = {b.lo[u].z, b.hi[u].z, b.lo[u].w, b.hi[u].w};
                    mma_bf16_16816(acc, a0, xv.x, xv.y);
                    mma_bf16_16816(acc, a1, xv.z, xv.w);
                }
                if (++ci == I) {
                    // tile done: partial sums of this warp -> shared memory, then the
                    // first 16*M threads add the NW partials in warp order
                    float *rw = red + (rb * NW + warp) * TILE * MC;
                    if (2 * c < M) {
                        rw[g * MC + 2 * c] = acc[0];
                        rw[(g + 8) * MC + 2 * c] = acc[2];
                        if (2 * c + 1 < M) {
                            rw[g * MC + 2 * c + 1] = acc[1];
                            rw[(g + 8) * MC + 2 * c + 1] = acc[3];
                        }
                    }
                    __syncthreads();
                    if (threadIdx.x < TILE * M) {
                        const int row = threadIdx.x / M;
                        const int m = threadIdx.x - row * M;
                        const int n = ct * TILE + row;
                        const float *rr = red + rb * NW * TILE * MC + row * MC + m;
                        float v = 0.0f;
                        for (int w = 0; w < NW; ++w) v += rr[w * TILE * MC];
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
        // the next batch is in flight while this one is consumed, including the
        // tile-end barrier and reduction
        for (int base = 0; base < total; base += 2 * U) {
            if (base + U < total && !(base == 0 && pre_b)) issue_batch(bB, base + U);
            consume_batch(bA, base);
            if (base + U >= total) break;
            if (base + 2 * U < total) issue_batch(bA, base + 2 * U);
            consume_batch(bB, base + U);
        }
    } else {
        for (int base = 0; base < total; base += U) {
            consume_batch(bA, base);
            if (base + U < total) issue_batch(bA, base + U);
        }
    }
}

}  // namespace sk
