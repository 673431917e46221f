// The small elementwise step between consecutive GEMMs of a decode chain.
//
// vLLM PR #65306 ("Add SM90 skinny GEMM plans for the BF16 decode projections",
// Validation) times its GEMMs as a chain "with a small kernel between GEMMs"
// and subtracts that kernel's time.  Here that kernel forms the next GEMM's
// input row from the previous GEMM's output:
//     x[k] = RNE_bf16( float(y[k mod n_src]) * scale ),  0 <= k < n_dst,
// which lets a chain of projections of different shapes run back to back with
// x kept near N(0,1) (scale = 1 / (0.02 sqrt(K_prev)) for W ~ N(0, 0.02^2)).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "internal.h"

namespace sk {

__global__ void __launch_bounds__(256) rescale_wrap_kernel(const uint16_t *__restrict__ y,
                                                           long long n_src,
                                                           uint16_t *__restrict__ x,
                                                           long long n_dst, float scale,
                                                           int flags) {
    if (flags & kFlagPdl) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n_dst;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const float v = __uint_as_float(static_cast<uint32_t>(y[i % n_src]) << 16);
        x[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v * scale));
    }
}

}  // namespace sk

extern "C" sgemm_status_t sgemm_bf16_rescale(const sgemm_bf16_t *y, long long n_src,
                                             sgemm_bf16_t *x, long long n_dst, float scale,
                                             unsigned flags, sgemm_stream_t stream) {
    if (!y || !x || n_src < 1 || n_dst < 1) return SGEMM_ERR_INVALID_ARG;
    if (flags & ~(SGEMM_FLAG_PDL | SGEMM_FLAG_WEIGHTS_READONLY)) return SGEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(x)) & 1u)
        return SGEMM_ERR_MISALIGNED;
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return SGEMM_ERR_CUDA;
    if (major != 10 || minor != 3) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    const long long blocks = (n_dst + 255) / 256 < 1024 ? (n_dst + 255) / 256 : 1024;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    if (flags & SGEMM_FLAG_PDL) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    const uint16_t *yy = y;
    uint16_t *xx = x;
    int fl = static_cast<int>(flags);
    void *args[] = {&yy, &n_src, &xx, &n_dst, &scale, &fl};
    if (cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(&sk::rescale_wrap_kernel), args) !=
        cudaSuccess)
        return SGEMM_ERR_CUDA;
    return SGEMM_OK;
}
