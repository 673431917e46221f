// Internal declarations shared by the host library and the kernel translation
// units of the BF16 skinny GEMM (y[M,N] = x[M,K] . W[N,K]^T, M <= 8).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sgemm_skinny.h"

namespace sk {

constexpr int kMaxBatch = SGEMM_MAX_BATCH;
constexpr int kMaxM = 8;
constexpr int kMaxThreads = 256;
constexpr size_t kMaxSmemOptin = 227 * 1024;  // shared memory a CTA may opt in to

// One problem of a (possibly batched) launch.  Row strides in elements.
struct Item {
    const uint16_t *x;
    const uint16_t *W;
    uint16_t *y;       // BF16 outputs, or FP32 outputs (reinterpreted) when Params::out_f32
    long long ldx;
    long long ldy;
    uint16_t *xn;      // fused chain epilogue: the next GEMM's input, or null
    long long ldxn;
};

// Params::flags bits (the launch flags of the C ABI, SGEMM_FLAG_*).
constexpr int kFlagPdl = SGEMM_FLAG_PDL;
constexpr int kFlagWeightsReadOnly = SGEMM_FLAG_WEIGHTS_READONLY;
constexpr int kFlagTestStall = SGEMM_FLAG_TEST_STALL;

// Kernel parameters (passed by value; about 350 bytes).
struct Params {
    Item item[kMaxBatch];
    float *ws;       // split-K partial sums, laid out [batch][split][M][N]; null when split == 1
    int N;
    int K;
    int kps;         // K elements per split (a multiple of 8); the last split may be shorter
    int split;       // number of K splits (gridDim.y)
    int row_groups;  // ceil(N / rows per warp task)
    int flags;       // SGEMM_FLAG_* bits
    int *err;        // device error word (bit 0: a bounded wait gave up); may be null
    int out_f32;     // 1: y holds FP32 outputs (no BF16 rounding)
    int xn_len;      // fused chain epilogue: xn[m][k] for 0 <= k < xn_len ...
    float xn_scale;  // ... = RNE_bf16(float(y[m][k mod N]) * xn_scale)
    int cl_rows;     // cluster-split streaming plans: rows per CTA that rank 0's buffer
                     // holds per split
};

// Kernel parameters of the TMA + tcgen05 kernel (skinny_tc05.cuh): the common
// parameters plus one pair of tensor maps (W and x) per problem, which the
// copy engine reads from the kernel's parameter space.  About 2.6 KB.
struct Tc05Params {
    CUtensorMap tw[kMaxBatch];  // W [N][K]: dims {K, N}, box {64, 128}, 128-byte swizzle
    CUtensorMap tx[kMaxBatch];  // x [M][K] (row stride ldx): dims {K, M}, box {64, 16}
    Params base;                // y, strides, epilogue, flags, error word (ws unused)
    int tiles;                  // ceil(N / 128)
    int kbox;                   // ceil(K / 64): 64-element boxes along K
    int per;                    // boxes per K split
    int split;                  // CTAs per cluster sharing a tile (1 = persistent grid)
    int ring;                   // shared-memory stages
    int nb;                     // boxes per stage
};

// A compiled instantiation of a kernel template.
struct KernelInfo {
    int variant;  // SGEMM_VARIANT_*
    int M;
    int R;        // rows per lane group
    int LPR;      // lanes per row
    int U;        // loads (CUDA cores) or 32-element k-blocks (tensor cores) per batch
    int stages;   // batches in flight: 1, or 2 when double-buffered
    const void *fn;
};

// Kernel tables, one per M (defined in the inst_m*.cu translation units).
extern const KernelInfo kKernelsM1[];
extern const KernelInfo kKernelsM2[];
extern const KernelInfo kKernelsM3[];
extern const KernelInfo kKernelsM4[];
extern const KernelInfo kKernelsM5[];
extern const KernelInfo kKernelsM6[];
extern const KernelInfo kKernelsM7[];
extern const KernelInfo kKernelsM8[];
extern const int kKernelCountPerM;

// Deterministic split-K reduction kernels, one per M.
extern const void *const kReduceKernels[kMaxM + 1];

// Launch geometry shared by every entry point (defined in api.cpp).
// K elements per split: a multiple of 8, every split non-empty.
int split_kps(int K, int split);
// Dynamic shared memory of one CTA of this plan.
size_t smem_bytes(const sgemm_plan_t &plan, int M, int kps);
// Rows per CTA of a cluster-split streaming plan (SGEMM_VARIANT_LDG_CLUSTER).
int cluster_rows(const sgemm_plan_t &plan);
// Work units of this plan (row groups for the CUDA-core kernel, 16-row tiles
// for the tensor-core kernel) and the CTAs that can use them.
int work_units(const sgemm_plan_t &plan, int N);
long long ctas_wanted(const sgemm_plan_t &plan, int N);
// Let a kernel use all the dynamic shared memory its static part leaves.
cudaError_t allow_max_dynamic_smem(const void *fn);

// The device error word of the current device (a static device variable of
// the library; bit 0: a kernel gave up a bounded wait).  Defined in
// tc05_launch.cu, which owns the variable.
cudaError_t device_error_word(int **out);

// The TMA + tcgen05 kernel (defined in tc05_launch.cu).  K boxes per split and
// the splits actually used for K and `split` CTAs requested: every split
// non-empty, so fewer may be used.
int tc05_boxes_per_split(int K, int split);
int tc05_splits_used(int K, int split);
// Dynamic shared memory of one CTA.
size_t tc05_smem_bytes(int M, int ring, int nb, int splits_used);
// Launch y = x . W^T for the problems in `base` (batch of them, all (M, N, K))
// with this plan; `fn` is the kernel for M, `ctas` the persistent grid's CTAs
// per problem when the plan does not split K.  Returns the CUDA status.
cudaError_t tc05_launch(const Params &base, int batch, int M, const sgemm_plan_t &plan,
                        long long ctas, const void *fn, cudaStream_t stream);

}  // namespace sk
