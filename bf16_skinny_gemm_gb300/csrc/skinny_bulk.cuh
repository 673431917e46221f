// Bulk-copy pipelined variant (sm_103a): y[M,N] = x[M,K] . W[N,K]^T, M <= 8.
//
// One persistent CTA per SM (or two) owns a balanced, contiguous range of rows
// of W (within one row of the fair share), so every SM streams the same number
// of bytes.  The range is cut into 8-row tiles (the last one partial) and each
// tile's K range into stages of 8 rows x KS columns.
//
//  * Warp 0, lane 0 is the producer: for every stage it copies the 8 row
//    segments with cp.async.bulk (the TMA engine's 1-D bulk copy) into a ring
//    of S shared-memory slots, completing a "full" mbarrier per slot with
//    complete_tx.  It refills a slot once all consumer warps have arrived on
//    that slot's "empty" mbarrier.  With S slots the number of bytes in flight
//    per SM is S x 8 x KS x 2, independent of registers and warp counts (a
//    GB300 probe of this scheme streamed 7.0-7.3 TB/s).
//  * Warps 1..NW are consumers.  They split each stage's 32-element k-blocks
//    (warp w takes blocks w, w+NW, ...) and run the x-as-A m16n8k16 MMA of
//    skinny_mmat.cuh on them: B = 8 rows of W straight from the ring (each row
//    padded by 16 bytes so the 8 rows of a fragment hit different banks),
//    A = x from shared memory.  At the end of a tile the NW partial tiles are
//    added in shared memory in warp order (a named barrier over the consumer
//    warps, double-buffered partials).
//  * Every wait is bounded: after about 0.2 s on %globaltimer a wait gives up,
//    sets bit 0 of *p.err (if given), and the CTA stops computing, writes NaN
//    to the outputs it owns and returns once its own copies have landed (the
//    producer waits, again bounded, for every copy it issued).  The flag
//    kFlagTestStall makes the producer issue nothing, so tests can exercise
//    this path without any fault.
//
// The accumulation order depends on (K, KS, NW) only, never on M.
#pragma once

#include <cuda_bf16.h>

#include "skinny_mma.cuh"

namespace sk {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *b, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *b, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *b, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase of the given parity; false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *b, unsigned parity) {
    if (mbar_try_wait(b, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(b, parity)) {
        if (static_cast<long long>(global_ns() - t0) > kWaitLimitNs) return false;
    }
    return true;
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void consumer_barrier(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

template <int M>
__global__ void __launch_bounds__(kMaxThreadsBulk, 1)
    skinny_bulk_kernel(const __grid_constant__ Params p) {
    static_assert(M >= 1 && M <= 8, "x rows fill the upper half of the A fragment");
    extern __shared__ __align__(128) unsigned char sm[];
    constexpr int TILE = 8;

    const bool pdl = (p.flags & kFlagPdl) != 0;
    if (pdl) pdl_launch_dependents();

    const Item &it = p.item[blockIdx.z];
    const int K = p.K;
    const int KS = p.kps;                    // stage width in elements (multiple of 32)
    const int S = p.ring;                    // ring depth
    const int NW = (blockDim.x >> 5) - 1;    // consumer warps
    const BulkLayout L(M, K, KS, S, NW);
    uint64_t *full = reinterpret_cast<uint64_t *>(sm);
    uint64_t *empty = full + S;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // balanced contiguous row range of this CTA, cut into 8-row tiles and KS-wide stages
    const long long Nl = p.N;
    const int n_begin = static_cast<int>(Nl * blockIdx.x / gridDim.x);
    const int n_end = static_cast<int>(Nl * (blockIdx.x + 1) / gridDim.x);
    const int ntiles = (n_end - n_begin + TILE - 1) / TILE;
    const int nparts = (K + KS - 1) / KS;    // stages per tile
    const int nstages = ntiles * nparts;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const bool stall = (p.flags & kFlagTestStall) != 0;
    const bool early_w = !pdl || (p.flags & kFlagWeightsReadOnly);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        auto issue = [&](int st) {
            const int tile = st / nparts;
            const int part = st - tile * nparts;
            const int slot = st % S;
            const int r0 = n_begin + tile * TILE;
            const int rows = min(TILE, n_end - r0);
            const int k0 = part * KS;
            const int kw = min(KS, K - k0);
            const unsigned bytes = static_cast<unsigned>(rows) * kw * 2;
            unsigned char *dst = sm + L.ring_off + slot * L.slot_bytes;
            mbar_arrive_expect_tx(&full[slot], bytes);
            for (int r = 0; r < rows; ++r)
                bulk_g2s(dst + r * L.row_stride, it.W + static_cast<long long>(r0 + r) * K + k0,
                         static_cast<unsigned>(kw) * 2, &full[slot]);
        };
        int issued = 0;
        bool ok = true;
        if (!stall) {
            if (!early_w && pdl) pdl_wait();
            for (int st = 0; st < nstages && ok; ++st) {
                if (st >= S) {
                    // slot reuse: wait until every consumer warp released round st/S - 1
                    ok = mbar_wait_bounded(&empty[st % S], ((st / S) - 1) & 1);
                    if (!ok || *reinterpret_cast<volatile int *>(&abort_flag)) break;
                }
                issue(st);
                ++issued;
            }
        }
        if (!ok) {
            if (p.err) atomicOr(p.err, 1);
            abort_flag = 1;
        }
        // never leave while a copy of ours may still be landing in shared memory
        for (int st = issued > S ? issued - S : 0; st < issued; ++st)
            mbar_wait_bounded(&full[st % S], (st / S) & 1);
        return;
    }

    // -------------------------------------------------------------- consumers
    const int cw = warp - 1;  // consumer warp index
    const int g = lane >> 2;
    const int c = lane & 3;
    if (pdl) pdl_wait();
    // stage x (all M rows, all of K) in shared memory
    {
        const int nchunk = K >> 3;
        for (int i = threadIdx.x - 32; i < M * nchunk; i += NW * 32) {
            const int m = i / nchunk;
            const int q = i - m * nchunk;
            *reinterpret_cast<uint4 *>(sm + L.x_off + m * L.x_stride + 16 * q) =
                *reinterpret_cast<const uint4 *>(it.x + m * it.ldx + 8 * q);
        }
    }
    consumer_barrier(NW * 32);

    float *red = reinterpret_cast<float *>(sm + L.red_off);
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    bool aborted = false;
    int rb = 0;
    for (int st = 0; st < nstages; ++st) {
        const int tile = st / nparts;
        const int part = st - tile * nparts;
        const int slot = st % S;
        const int r0 = n_begin + tile * TILE;
        const int rows = min(TILE, n_end - r0);
        const int k0 = part * KS;
        const int kw = min(KS, K - k0);
        if (!aborted) {
            // every lane waits (acquiring the copied bytes); the outcome is made
            // warp-uniform so that the MMAs below run converged
            const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[slot], (st / S) & 1));
            const bool flagged =
                __any_sync(0xffffffffu, *reinterpret_cast<volatile int *>(&abort_flag) != 0);
            if (!ok || flagged) {
                aborted = true;
                if (!ok && lane == 0 && p.err) atomicOr(p.err, 1);
                abort_flag = 1;
            }
        }
        if (!aborted) {
            const unsigned char *ws = sm + L.ring_off + slot * L.slot_bytes;
            const int nkb = (kw + 31) >> 5;  // k-blocks in this stage
            for (int jb = cw; jb < nkb; jb += NW) {
                const int kk = 32 * jb + 8 * c;  // element offset of this lane's chunk
                uint4 w = make_uint4(0u, 0u, 0u, 0u), xv = make_uint4(0u, 0u, 0u, 0u);
                if (kk < kw) {
                    if (g < rows)
                        w = *reinterpret_cast<const uint4 *>(ws + g * L.row_stride + 2 * kk);
                    if (g < M)
                        xv = *reinterpret_cast<const uint4 *>(sm + L.x_off + g * L.x_stride +
                                                              2 * (k0 + kk));
                }
                const uint32_t a0[4] = {xv.x, 0u, xv.y, 0u};
                const uint32_t a1[4] = {xv.z, 0u, xv.w, 0u};
                mma_bf16_16816(acc, a0, w.x, w.y);
                mma_bf16_16816(acc, a1, w.z, w.w);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);  // release the slot (also when aborted)

        if (part == nparts - 1) {
            // tile done: partial tiles -> shared memory, add them in warp order
            float *rw = red + (rb * NW + cw) * TILE * M;
            if (g < M) {
                rw[(2 * c) * M + g] = acc[0];
                rw[(2 * c + 1) * M + g] = acc[1];
            }
            consumer_barrier(NW * 32);
            const int t = threadIdx.x - 32;
            if (t < TILE * M) {
                const int row = t / M;
                const int m = t - row * M;
                const int n = r0 + row;
                if (row < rows) {
                    const float *rr = red + rb * NW * TILE * M + row * M + m;
                    float v = 0.0f;
                    for (int w2 = 0; w2 < NW; ++w2) v += rr[w2 * TILE * M];
                    const bool bad = *reinterpret_cast<volatile int *>(&abort_flag) != 0;
                    store_out(p, it, m, n, bad ? __int_as_float(0x7fc00000) : v);
                }
            }
            acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
            rb ^= 1;
        }
    }
}

}  // namespace sk
