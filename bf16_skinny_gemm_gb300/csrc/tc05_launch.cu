// Host side of the TMA + tcgen05 kernel (skinny_tc05.cuh), and the library's
// device error word.
//
// The error word is a static device variable, so reporting a failed bounded
// wait needs no allocated memory: every kernel that can give up a wait gets
// its device address as a parameter.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "tc05_consts.h"

namespace {

__device__ __align__(16) int g_device_error_word;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// A 2-D BF16 tensor map over rows x cols (row stride ld elements) with a box of
// box_rows x 64 elements, 128-byte swizzled; elements outside the tensor read
// as zero.  The library's preconditions (16-byte aligned base, ld a multiple
// of 8) are those of the encoder.
cudaError_t encode(CUtensorMap *map, const uint16_t *base, long long rows, long long cols,
                   long long ld, int box_rows, CUtensorMapL2promotion promo) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(sk::tc05::kBoxK),
                               static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(base),
                           dims, strides, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

std::mutex g_attr_mu;

}  // namespace

namespace sk {

cudaError_t device_error_word(int **out) {
    return cudaGetSymbolAddress(reinterpret_cast<void **>(out), g_device_error_word);
}

int tc05_boxes_per_split(int K, int split) {
    const int kbox = (K + tc05::kBoxK - 1) / tc05::kBoxK;
    return (kbox + split - 1) / split;
}

int tc05_splits_used(int K, int split) {
    const int kbox = (K + tc05::kBoxK - 1) / tc05::kBoxK;
    const int per = tc05_boxes_per_split(K, split);
    return (kbox + per - 1) / per;
}

size_t tc05_smem_bytes(int M, int ring, int nb, int splits_used) {
    // the ring, the cluster-reduction buffer of rank 0, and 1 KiB of alignment slack
    return static_cast<size_t>(ring) * nb * tc05::kBoxBytes +
           static_cast<size_t>(splits_used - 1) * M * tc05::kRows * sizeof(float) + 1024;
}

cudaError_t tc05_launch(const Params &base, int batch, int M, const sgemm_plan_t &plan,
                        long long ctas, const void *fn, cudaStream_t stream) {
    static_assert(sizeof(Tc05Params) <= 4096, "kernel parameters must fit 4 KB");
    const int N = base.N, K = base.K;
    Tc05Params tp;
    std::memset(&tp, 0, sizeof(tp));
    tp.base = base;
    for (int b = 0; b < batch; ++b) {
        const Item &it = base.item[b];
        cudaError_t e = encode(&tp.tw[b], it.W, N, K, K, tc05::kRows, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (e != cudaSuccess) return e;
        e = encode(&tp.tx[b], it.x, M, K, it.ldx, tc05::kCols, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
        if (e != cudaSuccess) return e;
    }
    const int used = tc05_splits_used(K, plan.split_k);
    tp.tiles = (N + tc05::kRows - 1) / tc05::kRows;
    tp.kbox = (K + tc05::kBoxK - 1) / tc05::kBoxK;
    tp.per = tc05_boxes_per_split(K, plan.split_k);
    tp.split = used;
    tp.ring = plan.stages;
    tp.nb = plan.k_unroll;

    if (used > 8) {
        std::lock_guard<std::mutex> lk(g_attr_mu);
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    long long gx;
    if (used > 1) {
        gx = static_cast<long long>(tp.tiles) * used;  // one tile per cluster
    } else {
        gx = std::max<long long>(1, std::min<long long>(tp.tiles, ctas));
    }

    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(batch), 1);
    cfg.blockDim = dim3(tc05::kThreads, 1, 1);
    cfg.dynamicSmemBytes = tc05_smem_bytes(M, plan.stages, plan.k_unroll, used);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (used > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(used);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (base.flags & kFlagPdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = static_cast<unsigned>(na);
    void *args[] = {&tp};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace sk
