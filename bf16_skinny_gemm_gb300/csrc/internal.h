// Internal declarations shared by the host library and the kernel translation
// units of the BF16 skinny GEMM (y[M,N] = x[M,K] . W[N,K]^T, M <= 4).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "sgemm_skinny.h"

namespace sk {

constexpr int kMaxBatch = SGEMM_MAX_BATCH;
constexpr int kMaxM = 4;
constexpr int kMaxThreads = 256;

// One problem of a (possibly batched) launch.  Row strides in elements.
struct Item {
    const uint16_t *x;
    const uint16_t *W;
    uint16_t *y;
    long long ldx;
    long long ldy;
};

// Params::flags bits (the launch flags of the C ABI, SGEMM_FLAG_*).
constexpr int kFlagPdl = SGEMM_FLAG_PDL;
constexpr int kFlagWeightsReadOnly = SGEMM_FLAG_WEIGHTS_READONLY;

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
};

// A compiled instantiation of a kernel template.
struct KernelInfo {
    int variant;  // SGEMM_VARIANT_*
    int M;
    int R;        // rows per lane group
    int LPR;      // lanes per row
    int U;        // 16-byte loads per row per lane in flight
    const void *fn;
};

// Kernel tables, one per M (defined in the inst_m*.cu translation units).
extern const KernelInfo kKernelsM1[];
extern const KernelInfo kKernelsM2[];
extern const KernelInfo kKernelsM3[];
extern const KernelInfo kKernelsM4[];
extern const int kKernelCountPerM;

// Deterministic split-K reduction kernels, one per M.
extern const void *const kReduceKernels[kMaxM + 1];

// Launch geometry shared by every entry point (defined in api.cpp).
// K elements per split: a multiple of 8, every split non-empty.
int split_kps(int K, int split);
// Dynamic shared memory of one CTA of this plan.
size_t smem_bytes(const sgemm_plan_t &plan, int M, int kps);
// Work units of this plan (row groups for the CUDA-core kernel, 16-row tiles
// for the tensor-core kernel) and the CTAs that can use them.
int work_units(const sgemm_plan_t &plan, int N);
long long ctas_wanted(const sgemm_plan_t &plan, int N);

}  // namespace sk
