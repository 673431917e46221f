// Tensor-core skinny GEMM on the Blackwell data path (sm_103a):
//
//     y[M,N] = x[M,K] . W[N,K]^T,   M <= 8,   BF16 in, FP32 accumulation
//
// The operation is the decode projection of vLLM PR #62949 ("SM121 skinny-GEMM
// plans for the GLM-5.3-Flash BF16 decode projections", Validation: each
// weight is read once per step) and PR #65306 ("Add SM90 skinny GEMM plans
// ...", Details: a library GEMM spends a split-K reduce kernel on these
// shapes).  This kernel is our own design for GB300:
//
//  * W never passes through registers.  A producer thread streams boxes of
//    128 rows x 64 elements of W (16 KiB) with cp.async.bulk.tensor into a
//    ring of S shared-memory stages of NB boxes each, 128-byte swizzled, with
//    the matching 16 x 64 box of x (2 KiB; rows >= M and columns >= K are
//    zero-filled by the copy engine, so they cost no memory traffic).  Each
//    stage completes on its "full" mbarrier.
//  * One thread issues, per box, four tcgen05.mma.kind::f16 of 128 (rows of
//    W) x 16 (rows of x, padded) x 16 (k), both operands K-major in shared
//    memory, FP32 accumulator in tensor memory, then tcgen05.commit onto the
//    stage's "empty" mbarrier, which hands the stage back to the producer.
//    At a tile's end it commits onto the tile's accumulator barrier.
//  * Four epilogue warps read the 128 x 16 accumulator with tcgen05.ld (warp
//    w reads tensor-memory lanes 32(w%4) .. +31, the tile's rows) and write y
//    through the library's common epilogue (BF16, FP32, or the fused decode-
//    chain step).  Two accumulators alternate, so the epilogue of one tile
//    overlaps the MMAs of the next.
//  * Work split, one of two forms (both one launch, no scratch memory):
//     - split == 1: a persistent grid; each CTA takes a balanced contiguous
//       range of 128-row tiles and walks each tile's whole K;
//     - split > 1: the `split` CTAs of a thread-block cluster share one tile,
//       each a contiguous range of K boxes.  At the end every CTA but rank 0
//       pushes its FP32 partial tile into rank 0's shared memory with
//       st.async (distributed shared memory), each store counted in bytes on
//       rank 0's reduction mbarrier, and exits; rank 0 waits for those bytes,
//       adds the partials in rank order and writes y.  (A cluster barrier in
//       place of the mbarrier cost about 0.5 us more per GEMM.)
//
// The accumulation order of an output depends on (K, boxes per split) only:
// never on M (the columns of one MMA are independent), the ring depth, the
// boxes per stage or the grid.  So results are deterministic and row m of an
// M-row call equals the 1-row call.
//
// Every wait on an mbarrier is bounded on the global timer.  A wait that runs
// out sets bit 0 of the device error word; the CTA stops issuing, writes NaN
// to its outputs, waits (bounded) for the copies and MMAs it issued and frees
// its tensor memory before it returns, so the context stays usable.  The
// test-only flag kFlagTestStall makes the producer issue no copies, so the
// waits run out without any fault.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "skinny_ldg.cuh"
#include "tc05_consts.h"

namespace sk {
namespace tc05 {

// Shared-memory matrix descriptor of a K-major operand stored in 128-byte
// swizzle atoms (8 rows x 128 bytes; atoms 1024 bytes apart along the rows):
// start address >> 4 (bits 0-13), leading byte offset 1 (unused by this
// layout, bits 16-29), stride byte offset 1024 >> 4 (bits 32-45), descriptor
// version 1 (bits 46-47), base offset 0, layout 128-byte swizzle = 2 (bits
// 61-63).  Advancing K by 16 elements inside the atom adds 32 bytes to the
// start address; the swizzle is applied to the generated addresses.
constexpr uint64_t kDescHi = (static_cast<uint64_t>(1024 >> 4) << 32) |
                             (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return kDescHi | (static_cast<uint64_t>(1) << 16) |
           static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
}

// Instruction descriptor of tcgen05.mma.kind::f16: FP32 accumulator (bits 4-5
// = 1), A and B BF16 (bits 7-9 and 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            (static_cast<uint32_t>(kCols >> 3) << 17) |
                            (static_cast<uint32_t>(kRows >> 4) << 24);

__device__ __forceinline__ void bar_arrive(uint32_t b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(b) : "memory");
}

__device__ __forceinline__ bool bar_try(uint32_t b, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(b), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of parity `parity` of mbarrier b to complete, at most
// kWaitLimitNs; false when the wait ran out.
__device__ __forceinline__ bool bar_wait(uint32_t b, unsigned parity) {
    if (bar_try(b, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!bar_try(b, parity)) {
        if (static_cast<long long>(global_ns() - t0) > kWaitLimitNs) return false;
    }
    return true;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void mma_f16(uint32_t tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

// Arrive on mbarrier b once every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::
                     "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive FP32 columns of this thread's tensor-memory lane (warp-wide).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}


__device__ __forceinline__ int read_flag(const int *f) {
    return *reinterpret_cast<const volatile int *>(f);
}

template <int M>
__global__ void __launch_bounds__(kThreads) skinny_tc05_kernel(const __grid_constant__ Tc05Params p) {
    static_assert(M >= 1 && M <= 8, "x rows fill the first M columns of the MMA");
    extern __shared__ uint8_t smem_raw[];
    // full[S], empty[S], accumulator full[2], accumulator empty[2], MMAs done, partials in
    __shared__ __align__(8) uint64_t bars[2 * kMaxRingSlots + 6];
    __shared__ uint32_t tmem_slot;
    __shared__ int abort_flag;

    // swizzled stages want 1024-byte aligned shared addresses; the host adds 1 KiB of slack
    uint8_t *ring = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
    const int S = p.ring;
    const int NB = p.nb;
    const int stage_bytes = NB * kBoxBytes;
    float *red = reinterpret_cast<float *>(ring + S * stage_bytes);  // [split-1][M][128]

    const Params &bp = p.base;
    const int bi = blockIdx.y;  // problem of a batched call
    const Item &it = bp.item[bi];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool pdl = (bp.flags & kFlagPdl) != 0;
    if (pdl) pdl_launch_dependents();

    // this CTA's tiles and K boxes
    const int split = p.split;
    int t_begin, t_end, kb0, kb1;
    uint32_t rank = 0;
    if (split > 1) {
        rank = cluster_rank();
        t_begin = static_cast<int>(blockIdx.x) / split;
        t_end = t_begin + 1;
        kb0 = static_cast<int>(rank) * p.per;
        kb1 = min(p.kbox, kb0 + p.per);
    } else {
        t_begin = static_cast<int>(static_cast<long long>(p.tiles) * blockIdx.x / gridDim.x);
        t_end = static_cast<int>(static_cast<long long>(p.tiles) * (blockIdx.x + 1) / gridDim.x);
        kb0 = 0;
        kb1 = p.kbox;
    }
    const int nbox = kb1 - kb0;
    const int nst = (nbox + NB - 1) / NB;  // stages per tile
    const int ntile = t_end - t_begin;
    const int total = ntile * nst;         // stages of this CTA

    const uint32_t full0 = saddr(&bars[0]);
    const uint32_t empty0 = full0 + 8 * S;
    const uint32_t accf0 = full0 + 8 * 2 * kMaxRingSlots;
    const uint32_t acce0 = accf0 + 16;
    const uint32_t fin = acce0 + 16;
    const uint32_t redb = fin + 8;  // rank 0: the other ranks' partial tiles have landed

    // The producer is thread 0.  Its tensor maps, and the stage -> (rows, boxes) map.
    const CUtensorMap *tw = &p.tw[bi];
    const CUtensorMap *tx = &p.tx[bi];
    const bool stall = (bp.flags & kFlagTestStall) != 0;
    auto stage_of = [&](int g, int &row, int &kb, int &cnt) {
        const int t = g / nst;
        const int st = g - t * nst;
        row = (t_begin + t) * kRows;
        kb = kb0 + st * NB;
        cnt = min(NB, kb1 - kb);
    };
    auto issue_w = [&](int g) {
        int row, kb, cnt;
        stage_of(g, row, kb, cnt);
        const int slot = g % S;
        const uint32_t fb = full0 + 8 * slot;
        bar_expect_tx(fb, static_cast<unsigned>(cnt * kBoxBytes));
        if (stall) return;
        const uint32_t st0 = saddr(ring + slot * stage_bytes);
        for (int b = 0; b < cnt; ++b) tma_load_2d(st0 + b * kWBox, tw, (kb + b) * kBoxK, row, fb);
    };
    auto issue_x = [&](int g) {
        if (stall) return;
        int row, kb, cnt;
        stage_of(g, row, kb, cnt);
        const int slot = g % S;
        const uint32_t x0 = saddr(ring + slot * stage_bytes) + NB * kWBox;
        for (int b = 0; b < cnt; ++b)
            tma_load_2d(x0 + b * kXBox, tx, (kb + b) * kBoxK, 0, full0 + 8 * slot);
    };
    // W of the first ring's worth of stages may stream before the previous kernel
    // on the stream finishes (PDL with read-only weights); x may not
    const bool early_w = !pdl || (bp.flags & kFlagWeightsReadOnly);
    const int pre = early_w ? min(S, total) : 0;

    if (warp == 0) {
        // The lanes of warp 0 set up the mbarriers in parallel, then each issues one stage
        // of the first ring of W, before the tensor-memory allocation and the CTA barrier.
        // (One thread doing all of it took about 2 us from kernel entry to the last copy
        // of an 8-stage ring: each copy costs its issuing thread about 0.1-0.2 us.)
        if (lane == 0) {
            prefetch_tmap(tw);
            prefetch_tmap(tx);
            abort_flag = 0;
        }
        for (int i = lane; i < 2 * S; i += 32) bar_init(full0 + 8 * i, 1);  // full[S], empty[S]
        // accf[2], acce[2], fin, redb
        if (lane < 6) bar_init(accf0 + 8 * lane, (lane == 2 || lane == 3) ? 4 : 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the copy engine
        __syncwarp();
        for (int g = lane; g < pre; g += 32) issue_w(g);
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         saddr(&tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (split > 1) cluster_arrive_relaxed();  // this CTA has started (paired with the wait below)

    float v[M];  // split > 1: this thread's partial sums of its row, kept for the cluster reduce
#pragma unroll
    for (int m = 0; m < M; ++m) v[m] = 0.0f;

    int issued = 0;  // stages the producer issued
    Out o{};         // epilogue warps: the output parameters, in registers
    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        if (total > 0) {
            if (pdl) pdl_wait();
            for (int g = lane; g < pre; g += 32) issue_x(g);  // the first ring's x, one stage per lane
            __syncwarp();
        }
        if (lane == 0 && total > 0) {
            issued = pre;
            for (int g = pre; g < total; ++g) {
                const int slot = g % S;
                if (g >= S && !bar_wait(empty0 + 8 * slot, ((g / S) - 1) & 1)) {
                    atomicExch(&abort_flag, 1);
                    break;
                }
                if (read_flag(&abort_flag)) break;
                issue_w(g);
                issue_x(g);
                issued = g + 1;
            }
            if (stall) issued = 0;  // nothing is in flight
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        if (lane == 0) {
            bool ok = true;
            int g = 0;
            for (int i = 0; i < ntile && ok; ++i) {
                const int b = i & 1;
                if (i >= 2 && !bar_wait(acce0 + 8 * b, ((i >> 1) - 1) & 1)) {
                    atomicExch(&abort_flag, 1);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(b * kCols);
                for (int st = 0; st < nst; ++st, ++g) {
                    const int slot = g % S;
                    if (!bar_wait(full0 + 8 * slot, (g / S) & 1) || read_flag(&abort_flag)) {
                        atomicExch(&abort_flag, 1);  // before the commit below releases the epilogue
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int cnt = min(NB, nbox - st * NB);
                    const uint32_t a0 = saddr(ring + slot * stage_bytes);
                    const uint32_t x0 = a0 + NB * kWBox;
                    for (int bx = 0; bx < cnt; ++bx) {
#pragma unroll
                        for (int j = 0; j < kBoxK / 16; ++j)
                            mma_f16(d, sw128_desc(a0 + bx * kWBox + 32 * j),
                                    sw128_desc(x0 + bx * kXBox + 32 * j),
                                    (st | bx | j) != 0 ? 1u : 0u);
                    }
                    mma_commit(empty0 + 8 * slot);
                }
                // also on failure, so that the epilogue's wait for this tile ends
                mma_commit(accf0 + 8 * b);
            }
            // every MMA issued has completed before the tensor memory is freed
            mma_commit(fin);
            if (!bar_wait(fin, 0)) atomicExch(&abort_flag, 1);
        }
    } else {
        // --------------------------------------------------------------- epilogue
        o = out_pinned(bp, it);  // read the output parameters while the copies stream
        if (pdl) pdl_wait();  // y (and the fused next input) may be read by the previous kernel
        const int q = warp & 3;  // tensor-memory lane quarter this warp may access
        const int row = q * 32 + lane;
        for (int i = 0; i < ntile; ++i) {
            const int b = i & 1;
            bool good = !read_flag(&abort_flag) && bar_wait(accf0 + 8 * b, (i >> 1) & 1) &&
                        !read_flag(&abort_flag);
            good = __all_sync(0xffffffffu, good);  // tcgen05.ld is warp-wide
            uint32_t r[16];
            if (good) {
                tc_fence_after();
                tmem_ld16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * kCols), r);
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) bar_arrive(acce0 + 8 * b);
            if (!good && lane == 0) atomicExch(&abort_flag, 1);
#pragma unroll
            for (int m = 0; m < M; ++m) v[m] = good ? __uint_as_float(r[m]) : __int_as_float(0x7fc00000);
            if (split == 1) {
                const int n = (t_begin + i) * kRows + row;
                if (n < o.N) {
#pragma unroll
                    for (int m = 0; m < M; ++m) store_out(o, m, n, v[m]);
                }
            }
        }
    }
    __syncwarp();

    if (split > 1) {
        // Deterministic K reduction across the cluster.  Ranks 1.. push their partial tile
        // into rank 0's shared memory with st.async, every byte counted on rank 0's mbarrier
        // redb, and are done; rank 0 waits for all of them and adds the partials in rank
        // order.  The only cluster barrier before this is the one that shows every CTA of
        // the cluster has started (so redb exists), which is long past by now.
        cluster_wait_acquire();
        if (warp >= 2 && ntile > 0) {
            const int row = (warp & 3) * 32 + lane;
            if (rank > 0) {
                // [rank-1][m][row]: each store of a warp is 128 contiguous bytes
                const uint32_t dst = cluster_addr(saddr(red + (rank - 1) * M * kRows + row), 0u);
                const uint32_t bar = cluster_addr(redb, 0u);
#pragma unroll
                for (int m = 0; m < M; ++m) st_async1(dst + 4u * static_cast<uint32_t>(m * kRows), v[m], bar);
            } else {
                if (warp == 2 && lane == 0)
                    bar_expect_tx(redb, static_cast<unsigned>((split - 1) * kRows * M * sizeof(float)));
                const bool got = bar_wait_cluster(redb, 0);
                if (!got) atomicExch(&abort_flag, 1);
                const int n = t_begin * kRows + row;
                if (n < o.N) {
                    float s[M];
#pragma unroll
                    for (int m = 0; m < M; ++m) s[m] = v[m];
                    // unrolled to the largest cluster (loads predicated on the rank count,
                    // so they issue back to back); the additions stay in rank order
#pragma unroll
                    for (int rr = 1; rr < kMaxSplit; ++rr) {
                        if (rr < split) {
#pragma unroll
                            for (int m = 0; m < M; ++m) s[m] += red[((rr - 1) * M + m) * kRows + row];
                        }
                    }
#pragma unroll
                    for (int m = 0; m < M; ++m) store_out(o, m, n, got ? s[m] : __int_as_float(0x7fc00000));
                }
            }
        }
    }

    // abort path: the producer's copies must have landed before the CTA's shared
    // memory goes (bounded waits); the MMAs are known complete (the "done" barrier)
    if (warp == 0 && lane == 0 && read_flag(&abort_flag)) {
        for (int g = max(0, issued - S); g < issued; ++g)
            (void)bar_wait(full0 + 8 * (g % S), (g / S) & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && abort_flag && bp.err) atomicOr(bp.err, 1);
    if (split > 1 && abort_flag) {
        // A CTA that gave up a wait may have got here before the other ranks issued their
        // stores into rank 0.  This cluster barrier waits for every thread of the cluster
        // that has not exited (ranks that finished normally have exited, stores issued);
        // then rank 0 waits, bounded, for those stores to land before its shared memory goes.
        cluster_arrive_release();
        cluster_wait_acquire();
        if (rank == 0 && warp == 2 && lane == 0) (void)bar_wait_cluster(redb, 0);
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace tc05
}  // namespace sk
