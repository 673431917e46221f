// Tensor-core skinny GEMM on the Blackwell data path (sm_103a) -- a draft.
//
//     y[M,N] = x[M,K] . W[N,K]^T,   M <= 16,   BF16 in, FP32 accumulation
//
// STATUS: compiled for sm_103a by the CPU test-suite (tests/test_abi.py), so
// ptxas checks every instruction form below and the host launch compiles; not
// yet part of the library (no translation unit of it includes this file) and
// never run on a GPU.  It becomes a plan variant only after parity tests
// against the oracle pass.
//
// Why: the mma.sync kernels of this library load W through registers in the
// fragment layout (8 rows x 64 bytes per warp instruction) and stop at 0.66 to
// 0.73 of the HBM peak for M = 4..8, while a library GEMM reaches about 0.8 at
// M = 8 on the same shapes.  Here W never passes through registers:
//  * a producer thread streams boxes of 128 rows x 64 elements of W (16 KiB)
//    and the matching 16 x 64 box of x (2 KiB; rows >= M and columns >= K are
//    zero-filled by the copy engine) with cp.async.bulk.tensor into a ring of
//    S shared-memory stages, 128-byte swizzled; each stage completes on its
//    "full" mbarrier;
//  * an MMA thread issues, per stage, four tcgen05.mma.kind::f16 of
//    M = 128 (rows of W) x N = 16 (rows of x) x K = 16, both operands K-major
//    in shared memory (128-byte-swizzle descriptors, advanced 32 bytes per K
//    step), FP32 accumulator in tensor memory, then tcgen05.commit onto the
//    stage's "empty" mbarrier, which hands the stage back to the producer;
//    after the last stage a commit onto "done";
//  * four warps read the 128 x 16 accumulator with tcgen05.ld (warp w owns
//    tensor-memory lanes 32w .. 32w+31, the tile's rows) and store y, or FP32
//    split-K partials for the library's second pass.
// Every wait is bounded on the global timer.  A wait that runs out sets bit 2
// of the error word; the CTA stops issuing, waits (bounded) for the copies it
// issued, writes NaN to its outputs and frees its tensor memory before it
// returns.  The accumulation order depends on (K range, stage width) only.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "skinny_ldg.cuh"

namespace sk {
namespace tc05 {

constexpr int kRows = 128;                        // rows of W per tile (MMA M)
constexpr int kCols = 16;                         // columns of the MMA (rows of x, padded)
constexpr int kBoxK = 64;                         // K elements per stage (128 bytes of a row)
constexpr int kWBytes = kRows * kBoxK * 2;        // 16 KiB
constexpr int kXBytes = kCols * kBoxK * 2;        // 2 KiB
constexpr int kStageBytes = kWBytes + kXBytes;    // multiple of 1024 (swizzle atoms)
constexpr int kTmemCols = 32;                     // smallest allocation
constexpr int kThreads = 128;                     // four warps

struct Tc05Params {
    CUtensorMap tw;   // W [N][K]: dims {K, N}, box {64, 128}, 128-byte swizzle
    CUtensorMap tx;   // x [M][K]: dims {K, M}, box {64, 16}, 128-byte swizzle
    uint16_t *y;      // [M][ldy] BF16, written when split == 1
    long long ldy;
    float *ws;        // [split][M][N] FP32 partials when split > 1
    int M, N, K;
    int kps;          // K elements per split, a multiple of 64
    int split;
    int stages;       // ring depth S
    int flags;
    int *err;
};

// Shared-memory matrix descriptor of a K-major operand laid out in 128-byte
// swizzle atoms (8 rows x 128 bytes, 1024 bytes apart along the rows):
// start address >> 4 (bits 0-13), leading byte offset (unused by this layout,
// 1), stride byte offset 1024 >> 4 (bits 32-45), descriptor version 1 (bits
// 46-47), layout 128-byte swizzle = 2 (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16: FP32 accumulator (bits 4-5
// = 1), A and B BF16 (bits 7-9 and 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 at bits 17-22, M >> 4 at bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                            (static_cast<uint32_t>(kCols >> 3) << 17) |
                            (static_cast<uint32_t>(kRows >> 4) << 24);

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

// Wait for phase `parity` of mbarrier b, at most kWaitLimitNs.
__device__ __forceinline__ bool bar_wait(uint32_t b, unsigned parity) {
    if (bar_try(b, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!bar_try(b, parity)) {
        if (static_cast<long long>(global_ns() - t0) > kWaitLimitNs) return false;
    }
    return true;
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
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::
                     "r"(bar)
                 : "memory");
}

template <int M>
__global__ void __launch_bounds__(kThreads) skinny_tc05_kernel(const __grid_constant__ Tc05Params p) {
    static_assert(M >= 1 && M <= kCols, "x rows fill the N columns of the MMA");
    extern __shared__ uint8_t smem_raw[];
    // the swizzled stages want 1024-byte alignment of their shared-memory
    // addresses; the host adds 1 KiB of slack
    uint8_t *smem = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
    const int S = p.stages;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S * kStageBytes);  // full[S], empty[S], done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 1);
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool pdl = (p.flags & kFlagPdl) != 0;
    if (pdl) pdl_launch_dependents();

    const int n0 = blockIdx.x * kRows;
    const int k0 = blockIdx.y * p.kps;
    const int kc = min(p.K - k0, p.kps);
    const int nst = (kc + kBoxK - 1) / kBoxK;  // stages of this CTA

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < 2 * S + 1; ++s) bar_init(saddr(bars + s), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         saddr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = *tmem_slot;

    if (pdl) pdl_wait();  // x (and y) belong to the stream's previous kernel

    int issued = 0;  // stages the producer issued
    if (warp == 0 && lane == 0) {
        // producer: stage st goes to slot st % S; refilling a slot waits for the
        // MMAs that read it (phase (st / S - 1) & 1 of its "empty" barrier)
        for (int st = 0; st < nst; ++st) {
            const int slot = st % S;
            if (st >= S && !bar_wait(saddr(bars + S + slot), ((st / S) - 1) & 1)) {
                atomicExch(&abort_flag, 1);
                break;
            }
            if (atomicAdd(&abort_flag, 0)) break;
            uint8_t *stage = smem + slot * kStageBytes;
            const uint32_t full = saddr(bars + slot);
            bar_expect_tx(full, kStageBytes);
            tma_load_2d(saddr(stage), &p.tw, k0 + st * kBoxK, n0, full);
            tma_load_2d(saddr(stage + kWBytes), &p.tx, k0 + st * kBoxK, 0, full);
            ++issued;
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: four K = 16 steps per stage, 32 bytes apart in the swizzled rows
        bool ok = true;
        for (int st = 0; st < nst; ++st) {
            const int slot = st % S;
            if (!bar_wait(saddr(bars + slot), (st / S) & 1)) {
                ok = false;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            uint8_t *stage = smem + slot * kStageBytes;
            const uint32_t a0 = saddr(stage), b0 = saddr(stage + kWBytes);
#pragma unroll
            for (int j = 0; j < kBoxK / 16; ++j)
                mma_f16(tmem, sw128_desc(a0 + 32 * j), sw128_desc(b0 + 32 * j), kIdesc,
                        (st > 0 || j > 0) ? 1u : 0u);
            mma_commit(saddr(bars + S + slot));
        }
        if (!ok) atomicExch(&abort_flag, 1);
        mma_commit(saddr(bars + 2 * S));  // "done" once every issued MMA has completed
    }

    // epilogue: every warp waits for "done", then reads its 32 rows x 16 columns.
    // tcgen05.ld is warp-wide: the warp reconverges first (lane 0 of warps 0 and 1
    // comes from its own loop, and each lane leaves the bounded wait on its own).
    bool done_ok = bar_wait(saddr(bars + 2 * S), 0);
    __syncwarp();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(tmem + (static_cast<uint32_t>(warp * 32) << 16)));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");

    const bool bad = !done_ok || atomicAdd(&abort_flag, 0) != 0;
    if (bad && threadIdx.x == 0 && p.err) atomicOr(p.err, 4);
    const int n = n0 + warp * 32 + lane;  // this thread's row of the tile
    if (n < p.N) {
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const float v = bad ? __int_as_float(0x7fc00000) : __uint_as_float(r[m]);
            if (p.split == 1) {
                p.y[m * p.ldy + n] = f32_to_bf16_rn(v);
            } else {
                p.ws[(static_cast<long long>(blockIdx.y) * M + m) * p.N + n] = v;
            }
        }
    }

    // on the abort path: the producer's copies must have landed before the CTA's
    // shared memory goes, and the issued MMAs must be done before their tensor
    // memory is freed (both bounded)
    if (warp == 0 && lane == 0 && bad) {
        for (int st = max(0, issued - S); st < issued; ++st)
            (void)bar_wait(saddr(bars + st % S), (st / S) & 1);
    }
    if (warp == 1 && lane == 0 && !done_ok) (void)bar_wait(saddr(bars + 2 * S), 0);
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

// Dynamic shared memory of a CTA with S stages: the ring, 2S+1 mbarriers, the
// tensor-memory address slot, and 1 KiB of alignment slack.
inline size_t smem_bytes(int stages) {
    return static_cast<size_t>(stages) * kStageBytes + (2 * stages + 1) * 8 + 16 + 1024;
}

// Host: the two tensor maps of one problem.  The driver's encoder is looked up
// through the runtime once, so the library needs no link against the driver
// library.  W [N][K] row-major: dims {K, N}, row stride 2K bytes, box {64, 128};
// x [M][K] with row stride ldx: dims {K, M}, box {64, 16}.  Both 128-byte
// swizzled (a box row is exactly 128 bytes), out-of-range elements read as 0.
// The preconditions of the library's calls (16-byte aligned x and W, K and ldx
// multiples of 8) are those of the encoder.
inline cudaError_t encode_maps(Tc05Params &p, const uint16_t *x, long long ldx, const uint16_t *W,
                               int M, int N, int K) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint32_t estride[2] = {1, 1};
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t box[2] = {kBoxK, kRows};
        if (encode(&p.tw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(W), dims,
                   strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ldx) * 2};
        const cuuint32_t box[2] = {kBoxK, kCols};
        if (encode(&p.tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(x), dims,
                   strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

// Host: one launch of the kernel for y = x . W^T (one problem), M <= 16.
// grid = (ceil(N / 128) tiles, split); split > 1 writes FP32 partials to ws
// ([split][M][N], caller-provided) for the library's split-K second pass,
// which the caller launches after this.  kps (K per split) is rounded up to
// whole 64-element stages, so the splits actually used (stored in *split_used
// when given; the second pass must use that count) may be fewer than asked.
// Flags as Params::flags (PDL launch attribute when kFlagPdl is set).  Returns
// the launch's CUDA status.
template <int M>
inline cudaError_t launch(const uint16_t *x, long long ldx, const uint16_t *W, uint16_t *y,
                          long long ldy, int N, int K, int split, int stages, float *ws,
                          int *err, int flags, cudaStream_t stream, int *split_used = nullptr) {
    Tc05Params p;
    cudaError_t e = encode_maps(p, x, ldx, W, M, N, K);
    if (e != cudaSuccess) return e;
    const int nst = (K + kBoxK - 1) / kBoxK;
    const int per = (nst + split - 1) / split;
    p.y = y;
    p.ldy = ldy;
    p.ws = ws;
    p.M = M;
    p.N = N;
    p.K = K;
    p.kps = per * kBoxK;
    p.split = (nst + per - 1) / per;  // every split non-empty
    if (split_used) *split_used = p.split;
    p.stages = stages;
    p.flags = flags;
    p.err = err;
    const size_t smem = smem_bytes(stages);
    e = cudaFuncSetAttribute(skinny_tc05_kernel<M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((N + kRows - 1) / kRows),
                       static_cast<unsigned>(p.split), 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (flags & kFlagPdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, skinny_tc05_kernel<M>, p);
}

}  // namespace tc05
}  // namespace sk
