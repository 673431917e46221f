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
//    (ld.global.nc.L1::no_allocate).  Each lane walks a flat sequence of
//    (row group, K chunk) iterations that runs across row boundaries, issuing
//    U loads at once and consuming them together.  Batches rather than a
//    rolling ring: measured on GB300, a register ring of loads consumed one at
//    a time keeps only about one load per warp in flight, while a batch keeps
//    all U in flight (5.1 vs 1.3 TB/s at 8 warps per SM).  With DB, two
//    batches alternate between two register sets, the next one issued before
//    the current one is consumed, so loads stay in flight while the warp
//    computes.  The number of bytes in flight does not depend on K.
//  * The first U loads are issued before x is staged, so the latency of the
//    W stream and of the x staging overlap.
//  * x (all M rows of this CTA's K range) is staged once per CTA in shared
//    memory and re-read from there for every row: it is tiny next to W.
//  * A warp is split into 32/LPR lane groups; each group owns R rows at a time
//    and walks their K range with stride LPR chunks of 8 elements.  Each lane
//    keeps M*R FP32 accumulators.  Products are exact in FP32 and are added
//    with FMA (see XChunk: widened FMA, mixed-precision FMA, or packed FP32x2
//    FMA over even/odd k).
//  * Lane partial sums are combined with an xor-butterfly of warp shuffles
//    (fixed order).  With split-K (gridDim.y > 1) each split writes FP32
//    partials and a second kernel adds them in split order.
//  * The grid is sized for the GPU (SMs x resident CTAs) and each CTA takes a
//    balanced contiguous range of row groups.
//  * Optional programmatic dependent launch: the kernel lets the next kernel
//    on the stream launch early, and waits for the previous one before it
//    reads x or writes y (and, unless told that W is read-only with respect to
//    the previous kernel, before it reads W).
//
// Accumulation order for one output is a function of (K range, LPR, FMODE
// pairing) only: it never depends on M, R, U, the CTA size or the grid, which
// makes results deterministic and row-wise independent of M.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"

namespace sk {

// 16 bytes of W, streamed: no L1 allocation, 256-byte L2 prefetch granule.
__device__ __forceinline__ uint4 ldg_stream(const uint16_t *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Returns at once when the kernel was not launched as a programmatic dependent.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Every wait of a kernel on something outside its own CTA is bounded on the
// global nanosecond timer; a wait that runs out reports it in the device error
// word instead of hanging the GPU.
constexpr long long kWaitLimitNs = 200LL * 1000 * 1000;  // 0.2 s per wait
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// Shared-memory mbarriers and thread-block-cluster primitives (used by the
// tcgen05 kernel and by the streaming kernel's cluster split).

__device__ __forceinline__ uint32_t saddr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void bar_init(uint32_t b, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(b), "r"(count) : "memory");
}

__device__ __forceinline__ void bar_expect_tx(uint32_t b, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(bytes)
                 : "memory");
}

// Whether the phase of parity `parity` of mbarrier b has completed, with
// cluster-scope acquire: for a barrier that other CTAs of the cluster complete
// with st.async.
__device__ __forceinline__ bool bar_try_cluster(uint32_t b, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(b), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool bar_wait_cluster(uint32_t b, unsigned parity) {
    if (bar_try_cluster(b, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!bar_try_cluster(b, parity)) {
        if (static_cast<long long>(global_ns() - t0) > kWaitLimitNs) return false;
    }
    return true;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// The shared::cluster address of CTA-local shared address `local` in the
// cluster's CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    return remote;
}

// Asynchronous store of one word into another CTA's shared memory (shared::cluster
// addresses); it completes its 4 bytes on mbarrier `bar` there.
__device__ __forceinline__ void st_async1(uint32_t dst, float a, uint32_t bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(dst),
                 "r"(__float_as_uint(a)), "r"(bar)
                 : "memory");
}

// BF16 -> FP32 is exact: the BF16 bits are the top half of the FP32 bits.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// The epilogue of every kernel: output (m, n) of problem `it`, FP32 sum v.
//  - BF16 output: y = RNE_bf16(v).  With the fused chain epilogue, the next
//    GEMM's input also gets xn[m][k] = RNE_bf16(float(y) * scale) for every
//    k < xn_len with k = n (mod N): the elementwise step between the decode
//    chain's GEMMs, done on the value just rounded, so the result is bitwise
//    that of the separate step.
//  - FP32 output: y = v, no rounding.
// `Out` holds what the epilogue reads of the parameters.
struct Out {
    uint16_t *y;
    uint16_t *xn;
    long long ldy;
    long long ldxn;
    int out_f32;
    int xn_len;
    int N;
    float xn_scale;
};

__device__ __forceinline__ Out out_of(const Params &p, const Item &it) {
    return Out{it.y, it.xn, it.ldy, it.ldxn, p.out_f32, p.xn_len, p.N, p.xn_scale};
}

// The same, read into registers now: a kernel whose epilogue would first touch
// these parameters at its very end (a constant-cache miss on the critical
// path) reads them when it starts.  The moves are opaque, so the compiler
// cannot sink the reads back to the use.
__device__ __forceinline__ Out out_pinned(const Params &p, const Item &it) {
    Out o = out_of(p, it);
    asm volatile("mov.b64 %0, %0;" : "+l"(o.y));
    asm volatile("mov.b64 %0, %0;" : "+l"(o.xn));
    asm volatile("mov.b64 %0, %0;" : "+l"(o.ldy));
    asm volatile("mov.b64 %0, %0;" : "+l"(o.ldxn));
    asm volatile("mov.b32 %0, %0;" : "+r"(o.out_f32));
    asm volatile("mov.b32 %0, %0;" : "+r"(o.xn_len));
    asm volatile("mov.b32 %0, %0;" : "+r"(o.N));
    asm volatile("mov.b32 %0, %0;" : "+f"(o.xn_scale));
    return o;
}

__device__ __forceinline__ void store_out(const Out &o, int m, int n, float v) {
    if (o.out_f32) {
        reinterpret_cast<float *>(o.y)[m * o.ldy + n] = v;
        return;
    }
    const uint16_t b = f32_to_bf16_rn(v);
    o.y[m * o.ldy + n] = b;
    if (o.xn) {
        const uint16_t q = f32_to_bf16_rn(__uint_as_float(static_cast<uint32_t>(b) << 16) * o.xn_scale);
        for (int k = n; k < o.xn_len; k += o.N) o.xn[m * o.ldxn + k] = q;
    }
}

__device__ __forceinline__ void store_out(const Params &p, const Item &it, int m, int n, float v) {
    store_out(out_of(p, it), m, n, v);
}

// acc += lo(x)*lo(w), then acc += hi(x)*hi(w): BF16 operands, FP32 addend,
// one round-to-nearest per FMA.
__device__ __forceinline__ float fma2_bf16(uint32_t xw, uint32_t ww, float acc) {
    asm("{\n\t.reg .b16 xl, xh, wl, wh;\n\t"
        "mov.b32 {xl, xh}, %1;\n\t"
        "mov.b32 {wl, wh}, %2;\n\t"
        "fma.rn.f32.bf16 %0, xl, wl, %0;\n\t"
        "fma.rn.f32.bf16 %0, xh, wh, %0;\n\t}"
        : "+f"(acc)
        : "r"(xw), "r"(ww));
    return acc;
}

// D[16x8] += A[16x16] . B[16x8], BF16 inputs, FP32 accumulation (mma.sync).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4],
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 16 bytes of x: from shared memory (staged), or straight from global memory
// through the L1 cache (x is a few KiB and stays there after the first touch).
template <bool XG>
__device__ __forceinline__ uint4 load_x(const uint4 *p) {
    if (XG) return __ldg(p);
    return *p;
}

// x operand of one chunk (8 elements) for all M rows, and how a chunk of W is
// multiplied into the accumulators.  FMODE selects the arithmetic:
//   0: widen both operands to FP32, one FMA per element;
//   1: the mixed-precision FMA (BF16 operands, FP32 addend) per element;
//   2: packed FP32x2 FMA (fma.rn.f32x2, sm_100+): each accumulator is a pair
//      {even k, odd k} of FP32 partial sums, one instruction per two elements;
//      the pair is added (even + odd) when the row is finished.
//   3: the tensor core on the same data layout (LPR = 32, so lane l holds
//      k = 8l .. 8l+7 of each 256-element chunk of a row): in one mma.sync
//      m16n8k16 the 8 columns of B are the chunk's 8 segments of 32 elements
//      (lanes 4g .. 4g+3 hold segment g, each lane its own 16 bytes, the
//      first 8 bytes in one MMA and the last 8 in a second), and row g (g+8)
//      of A is x row m (m+1) at the k of segment g -- which are exactly the k
//      of the lane's own x chunk.  So D[g][g] (D[g+8][g]) accumulates x_m
//      (x_{m+1}) . W over segment g; the off-diagonal entries are not used.
//      Two MMAs per 16 bytes of W and pair of x rows instead of 8 FMAs per x
//      row; the 8 diagonal entries are added by the butterfly at row end.
// Modes 0 and 1 round identically (one rounding per element); modes 2 and 3
// each keep their own, equally fixed, summation order.
template <int M, int FMODE>
struct XChunk;

template <int M>
struct XChunk<M, 0> {
    using Acc = float;
    float v[M][8];
    static __device__ __forceinline__ float total(Acc a) { return a; }
    template <bool XG>
    __device__ __forceinline__ void load(const uint4 *xs, long long stride, int c) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const uint4 q = load_x<XG>(xs + m * stride + c);
            const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[m][2 * i] = bf16_lo(qq[i]);
                v[m][2 * i + 1] = bf16_hi(qq[i]);
            }
        }
    }
    template <int R>
    __device__ __forceinline__ void fma(Acc (&acc)[M][R], const uint4 &w, int r) const {
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float w0 = bf16_lo(ww[i]);
            const float w1 = bf16_hi(ww[i]);
#pragma unroll
            for (int m = 0; m < M; ++m) {
                acc[m][r] = fmaf(v[m][2 * i], w0, acc[m][r]);
                acc[m][r] = fmaf(v[m][2 * i + 1], w1, acc[m][r]);
            }
        }
    }
};

template <int M>
struct XChunk<M, 1> {
    using Acc = float;
    uint32_t v[M][4];
    static __device__ __forceinline__ float total(Acc a) { return a; }
    template <bool XG>
    __device__ __forceinline__ void load(const uint4 *xs, long long stride, int c) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const uint4 q = load_x<XG>(xs + m * stride + c);
            v[m][0] = q.x;
            v[m][1] = q.y;
            v[m][2] = q.z;
            v[m][3] = q.w;
        }
    }
    template <int R>
    __device__ __forceinline__ void fma(Acc (&acc)[M][R], const uint4 &w, int r) const {
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int m = 0; m < M; ++m) acc[m][r] = fma2_bf16(v[m][i], ww[i], acc[m][r]);
    }
};

// {lo, hi} FP32 pair in one 64-bit register pair
__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(c) : "l"(a), "l"(b));
    return c;
}

template <int M>
struct XChunk<M, 2> {
    using Acc = unsigned long long;  // {sum over even k, sum over odd k}
    unsigned long long v[M][4];
    static __device__ __forceinline__ float total(Acc a) {
        float lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(a));
        return lo + hi;
    }
    template <bool XG>
    __device__ __forceinline__ void load(const uint4 *xs, long long stride, int c) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const uint4 q = load_x<XG>(xs + m * stride + c);
            const uint32_t qq[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) v[m][i] = pack_f32x2(bf16_lo(qq[i]), bf16_hi(qq[i]));
        }
    }
    template <int R>
    __device__ __forceinline__ void fma(Acc (&acc)[M][R], const uint4 &w, int r) const {
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const unsigned long long wp = pack_f32x2(bf16_lo(ww[i]), bf16_hi(ww[i]));
#pragma unroll
            for (int m = 0; m < M; ++m) acc[m][r] = ffma2(v[m][i], wp, acc[m][r]);
        }
    }
};

template <int M>
struct XChunk<M, 3> {
    struct Acc {
        float d[4];  // D fragment of the x-row pair (m, m+1), kept at even m
    };
    uint32_t v[M][4];
    // this lane's share of row m's sum: its diagonal entry of D, if it holds one
    template <int R>
    static __device__ __forceinline__ float diag(const Acc (&acc)[M][R], int m, int r) {
        const int lane = threadIdx.x & 31;
        const int g = lane >> 2, c = lane & 3;
        if (c != (g >> 1)) return 0.0f;  // D[g][g] sits in lane (g, g/2), element g%2
        const Acc &a = acc[m & ~1][r];
        return (m & 1) ? ((g & 1) ? a.d[3] : a.d[2]) : ((g & 1) ? a.d[1] : a.d[0]);
    }
    template <bool XG>
    __device__ __forceinline__ void load(const uint4 *xs, long long stride, int c) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const uint4 q = load_x<XG>(xs + m * stride + c);
            v[m][0] = q.x;
            v[m][1] = q.y;
            v[m][2] = q.z;
            v[m][3] = q.w;
        }
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int m = 0; m < M; ++m) v[m][0] = v[m][1] = v[m][2] = v[m][3] = 0u;
    }
    // called by all 32 lanes together (mma.sync), never under a lane-dependent branch
    template <int R>
    __device__ __forceinline__ void fma(Acc (&acc)[M][R], const uint4 &w, int r) const {
#pragma unroll
        for (int m = 0; m < M; m += 2) {
            const uint32_t y0 = m + 1 < M ? v[m + 1][0] : 0u, y1 = m + 1 < M ? v[m + 1][1] : 0u;
            const uint32_t y2 = m + 1 < M ? v[m + 1][2] : 0u, y3 = m + 1 < M ? v[m + 1][3] : 0u;
            const uint32_t a0[4] = {v[m][0], y0, v[m][1], y1};
            const uint32_t a1[4] = {v[m][2], y2, v[m][3], y3};
            mma_bf16_16816(acc[m][r].d, a0, w.x, w.y);
            mma_bf16_16816(acc[m][r].d, a1, w.z, w.w);
        }
    }
};

template <int M, int R, int LPR, int U, int FMODE, bool DB, bool XG = false, bool CL = false>
__global__ void __launch_bounds__(kMaxThreads) skinny_ldg_kernel(const __grid_constant__ Params p) {
    static_assert(LPR == 32 || LPR == 16 || LPR == 8, "lanes per row");
    static_assert(FMODE != 3 || LPR == 32, "the tensor-core mode spreads a row over the warp");
    constexpr int G = 32 / LPR;  // lane groups per warp
    extern __shared__ uint4 xs[];  // [M][nchunk] chunks of 8 BF16

    const bool pdl = (p.flags & kFlagPdl) != 0;
    if (pdl) pdl_launch_dependents();

    const Item &it = p.item[blockIdx.z];
    const int s = blockIdx.y;
    const int k0 = s * p.kps;
    const int kc = min(p.K - k0, p.kps);
    const int nchunk = kc >> 3;

    const int warps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int gi = lane / LPR;  // lane group
    const int li = lane % LPR;  // lane in group

    // balanced contiguous range of row groups for this CTA; warps interleave
    const long long RG = p.row_groups;
    const int g_begin = static_cast<int>(RG * blockIdx.x / gridDim.x);
    const int g_end = static_cast<int>(RG * (blockIdx.x + 1) / gridDim.x);
    const int g0 = g_begin + warp;
    const int ntask = g0 < g_end ? (g_end - g0 + warps - 1) / warps : 0;

    // Split across a thread-block cluster (CL, compiled only for the cluster-split plans,
    // so the other plans' code is unchanged): the p.split CTAs of this row range form a
    // cluster, rank r having K split r.  Rank 0 keeps its own partial sums and takes
    // the other ranks' through st.async into red [split][cl_rows][M], every byte counted on
    // its mbarrier cl_bar; it adds them in split order once they have landed.
    __shared__ __align__(8) uint64_t cl_bar;
    const bool cl = CL && p.split > 1;
    const int crank = cl ? static_cast<int>(cluster_rank()) : 0;
    const int row0 = g_begin * G * R;
    const int rows_valid = max(0, min(p.N, g_end * G * R) - row0);
    // after the x slice of a full split (the last split's is shorter), the same offset on
    // every rank
    float *red = reinterpret_cast<float *>(xs + (XG ? 0 : M * (p.kps >> 3)));
    bool cl_waited = false;
    if (cl) {
        if (threadIdx.x == 0) {
            bar_init(saddr(&cl_bar), 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            if (crank == 0)  // the only arrival: the bytes the other ranks will send
                bar_expect_tx(saddr(&cl_bar),
                              static_cast<unsigned>((p.split - 1) * rows_valid * M * sizeof(float)));
        }
        cluster_arrive_relaxed();  // this CTA has started (its mbarrier exists)
    }
    const int jtot = (nchunk + LPR - 1) / LPR;          // iterations per task
    const int last_lanes = nchunk - (jtot - 1) * LPR;   // lanes busy in a task's last iteration
    const int total = ntask * jtot;                     // iterations of this warp

    // Load cursor (task lt, iteration lj) and consume cursor (task ct, iteration cj)
    // walk the same flat sequence of this warp's iterations.  Loads are issued in
    // batches of U iterations (which may span tasks) and the whole batch is consumed
    // before the next batch is issued: every load of a batch is in flight at once.
    int lt = 0, lj = 0;
    const uint16_t *lrow[R];
    auto rows_of = [&](int t) {
        const int n0 = ((g0 + t * warps) * G + gi) * R;
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int n = min(n0 + r, p.N - 1);  // rows past N re-read row N-1; result dropped
            lrow[r] = it.W + static_cast<long long>(n) * p.K + k0 + 8 * li;
        }
    };
    rows_of(0);

    using Batch = uint4[U][R];
    auto issue_batch = [&](Batch &buf, int base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (base + u < total) {
                const bool ok = (lj < jtot - 1) || (li < last_lanes);
#pragma unroll
                for (int r = 0; r < R; ++r)
                    buf[u][r] = ok ? ldg_stream(lrow[r] + 8 * LPR * lj) : make_uint4(0u, 0u, 0u, 0u);
                if (++lj == jtot) {
                    lj = 0;
                    if (++lt < ntask) rows_of(lt);
                }
            }
        }
    };

    Batch bufA, bufB;
    const bool early_w = !pdl || (p.flags & kFlagWeightsReadOnly);
    // with read-only weights, both batches of a double-buffered plan go out before
    // the wait for the previous kernel (the same order the loop below would use)
    const bool pre_b = DB && early_w && U < total;
    if (early_w) issue_batch(bufA, 0);
    if (pre_b) issue_batch(bufB, U);
    if (pdl) pdl_wait();
    if (!early_w) issue_batch(bufA, 0);

    // x: staged in shared memory (overlaps the first batch's latency), or read
    // from global memory at each use (no staging, no CTA barrier)
    const uint4 *xsrc = XG ? reinterpret_cast<const uint4 *>(it.x + k0) : xs;
    const long long xstride = XG ? it.ldx / 8 : nchunk;
    if (!XG) {
        for (int i = threadIdx.x; i < M * nchunk; i += blockDim.x) {
            const int m = i / nchunk;
            const int c = i - m * nchunk;
            xs[i] = *reinterpret_cast<const uint4 *>(it.x + m * it.ldx + k0 + 8 * c);
        }
        __syncthreads();
    }

    using XC = XChunk<M, FMODE>;
    using Acc = typename XC::Acc;
    Acc acc[M][R];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
        for (int r = 0; r < R; ++r) acc[m][r] = Acc{};

    int ct = 0, cj = 0;
    auto consume_batch = [&](const Batch &buf, int base) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (base + u < total) {
                const bool active = (cj < jtot - 1) || (li < last_lanes);
                if constexpr (FMODE == 3) {
                    // mma.sync is a warp-wide instruction: every lane takes part, and
                    // the lanes past the end of the row bring zero x (their W is zero)
                    XC xc;
                    if (active) {
                        xc.template load<XG>(xsrc, xstride, li + LPR * cj);
                    } else {
                        xc.zero();
                    }
#pragma unroll
                    for (int r = 0; r < R; ++r) xc.template fma<R>(acc, buf[u][r], r);
                } else if (active) {
                    XC xc;
                    xc.template load<XG>(xsrc, xstride, li + LPR * cj);
#pragma unroll
                    for (int r = 0; r < R; ++r) xc.template fma<R>(acc, buf[u][r], r);
                }
                if (++cj == jtot) {
                    // task done: xor-butterfly over the LPR lanes (fixed tree order)
                    float tot[M][R];
#pragma unroll
                    for (int m = 0; m < M; ++m)
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            float v;
                            if constexpr (FMODE == 3) {
                                v = XC::diag(acc, m, r);
                            } else {
                                v = XC::total(acc[m][r]);
                            }
#pragma unroll
                            for (int off = LPR / 2; off >= 1; off >>= 1)
                                v += __shfl_xor_sync(0xffffffffu, v, off);
                            tot[m][r] = v;
                        }
                    if (li == 0) {
                        const int n0 = ((g0 + ct * warps) * G + gi) * R;
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const int n = n0 + r;
                            if (n < p.N) {
#pragma unroll
                                for (int m = 0; m < M; ++m) {
                                    if (p.split == 1) {
                                        store_out(p, it, m, n, tot[m][r]);
                                    } else if (cl) {
                                        const int rl = n - row0;
                                        if (crank == 0) {
                                            red[rl * M + m] = tot[m][r];
                                        } else if (!(p.flags & kFlagTestStall)) {
                                            if (!cl_waited) {
                                                cluster_wait_acquire();  // rank 0 has started
                                                cl_waited = true;
                                            }
                                            st_async1(cluster_addr(saddr(red + (crank * p.cl_rows + rl) * M + m), 0u),
                                                      tot[m][r], cluster_addr(saddr(&cl_bar), 0u));
                                        }
                                    } else {
                                        const long long slot =
                                            (static_cast<long long>(blockIdx.z) * p.split + s) * M + m;
                                        p.ws[slot * p.N + n] = tot[m][r];
                                    }
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int m = 0; m < M; ++m)
#pragma unroll
                        for (int r = 0; r < R; ++r) acc[m][r] = Acc{};
                    cj = 0;
                    ++ct;
                }
            }
        }
    };

    if (DB) {
        // two batches in flight: the next batch is issued before the current one is
        // consumed (the two buffers are distinct registers, so consuming one does not
        // wait for the other's loads)
        for (int base = 0; base < total; base += 2 * U) {
            if (base + U < total && !(base == 0 && pre_b)) issue_batch(bufB, base + U);
            consume_batch(bufA, base);
            if (base + U >= total) break;
            if (base + 2 * U < total) issue_batch(bufA, base + 2 * U);
            consume_batch(bufB, base + U);
        }
    } else {
        for (int base = 0; base < total; base += U) {
            consume_batch(bufA, base);
            if (base + U < total) issue_batch(bufA, base + U);
        }
    }

    if (cl) {
        // every thread waits once on the start barrier it arrived on (long complete)
        if (!cl_waited) cluster_wait_acquire();
        if (crank == 0) {
            __syncthreads();  // this CTA's own partial sums are in red
            const bool got = bar_wait_cluster(saddr(&cl_bar), 0);
            const bool bad = __syncthreads_or(!got) != 0;
            for (int i = threadIdx.x; i < rows_valid * M; i += blockDim.x) {
                const int rl = i / M;
                const int m = i - rl * M;
                // split order from 0.0f, as the second-pass kernel adds: the same bits
                float acc = 0.0f;
                for (int q = 0; q < p.split; ++q) acc += red[(q * p.cl_rows + rl) * M + m];
                store_out(p, it, m, row0 + rl, bad ? __int_as_float(0x7fc00000) : acc);
            }
            if (bad) {
                // a rank's partials did not all land in time: report it, then wait until
                // every other rank has issued its stores (this barrier waits for the
                // threads of the cluster that have not exited), and for those to land,
                // before this CTA's shared memory goes
                if (threadIdx.x == 0 && p.err) atomicOr(p.err, 1);
                cluster_arrive_release();
                cluster_wait_acquire();
                if (threadIdx.x == 0) (void)bar_wait_cluster(saddr(&cl_bar), 0);
            }
        }
    }
}

// Second pass of split-K: y = RNE_bf16(sum over splits, in split order).
template <int M>
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const __grid_constant__ Params p,
                                                             int batch) {
    if (p.flags & kFlagPdl) {
        pdl_launch_dependents();
        pdl_wait();
    }
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
        store_out(p, it, m, n, acc);
    }
}

}  // namespace sk
