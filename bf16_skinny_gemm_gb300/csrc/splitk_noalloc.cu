// Split-K skinny GEMM whose scratch is a fixed array in device memory, so a
// call allocates nothing.
//
// Why it exists: some callers cannot call cudaMalloc (or any allocating
// routine) at the point where they run a GEMM -- for example code that runs
// under a memory manager that owns all device memory and forbids other
// allocations, plugins and embedded runtimes that are not allowed to grow
// their footprint after start-up, or latency-critical loops where a
// cudaMalloc (which may synchronize the device) is not acceptable.  The
// regular split-K path allocates its scratch on first use; this entry point
// instead uses the file-scope array below, which is part of the library's
// device image and is created when the library's code is loaded on a device.
//
// The kernels are the regular ones of the plan sgemm_splitk_noalloc_plan
// returns: the selected plan with split_k splits (the kernel with gridDim.y
// splits, then splitk_reduce_kernel), or a plan that splits K the same way
// when the selected one does not (see that function); only where the FP32
// partial sums live differs, so results are bitwise equal to
// sgemm_bf16_skinny_ex with that plan.
#include <cuda_runtime.h>

#include <mutex>
#include <set>

#include "internal.h"

namespace {

constexpr size_t kScratchFloats = SGEMM_NOALLOC_SCRATCH_BYTES / sizeof(float);

// Shared by every call of sgemm_bf16_skinny_splitk_noalloc on a device; it keeps
// whatever the last call left in it.  Held by every GPU that loads the library
// until the process exits.
static __device__ __align__(256) float g_splitk_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool done = false;
    bool supported = false;
    int sms = 0;
    float *scratch = nullptr;  // device address of g_splitk_scratch on this device
    std::set<const void *> smem_attr_set;  // kernels already allowed their shared memory
};

std::mutex g_mu;
DeviceSetup g_dev[kMaxDevices];

const sk::KernelInfo *find(int M, const sgemm_plan_t &p) {
    const sk::KernelInfo *t = nullptr;
    switch (M) {
        case 1: t = sk::kKernelsM1; break;
        case 2: t = sk::kKernelsM2; break;
        case 3: t = sk::kKernelsM3; break;
        case 4: t = sk::kKernelsM4; break;
        case 5: t = sk::kKernelsM5; break;
        case 6: t = sk::kKernelsM6; break;
        case 7: t = sk::kKernelsM7; break;
        case 8: t = sk::kKernelsM8; break;
        default: return nullptr;
    }
    const int stages = p.stages == 0 ? 1 : p.stages;
    for (int i = 0; i < sk::kKernelCountPerM; ++i)
        if (t[i].variant == p.variant && t[i].R == p.rows_per_warp &&
            t[i].LPR == p.lanes_per_row && t[i].U == p.k_unroll && t[i].stages == stages)
            return &t[i];
    return nullptr;
}

// Once per device, with that device current: look up the array's device
// address (the host-side name g_splitk_scratch is only a stand-in and must
// never be handed to a kernel).  Refused while `stream` is capturing, so that
// the one-time set-up never lands inside a graph.  Then allow the kernel `fn`
// its shared memory (once per kernel and device).
sgemm_status_t setup_current_device(cudaStream_t stream, const void *fn, DeviceSetup **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceSetup &st = g_dev[dev];
    if (!st.done) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return SGEMM_ERR_CUDA;
        if (cap != cudaStreamCaptureStatusNone) return SGEMM_ERR_INVALID_ARG;
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SGEMM_ERR_CUDA;
        st.supported = (major == 10 && minor == 3);
        st.sms = sms;
        if (st.supported) {
            void *ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_splitk_scratch) != cudaSuccess || ptr == nullptr)
                return SGEMM_ERR_CUDA;
            st.scratch = static_cast<float *>(ptr);
        }
        st.done = true;
    }
    if (!st.supported) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    if (!st.smem_attr_set.count(fn)) {
        if (sk::allow_max_dynamic_smem(fn) != cudaSuccess) return SGEMM_ERR_CUDA;
        st.smem_attr_set.insert(fn);
    }
    *out = &st;
    return SGEMM_OK;
}

sgemm_plan_t streaming_plan(int split_k) {
    sgemm_plan_t p;
    p.variant = SGEMM_VARIANT_LDG_MIXFMA;
    p.threads = 256;
    p.rows_per_warp = 1;
    p.lanes_per_row = 32;
    p.k_unroll = 8;
    p.vec_bytes = 16;
    p.split_k = split_k;
    p.stages = 1;
    p.ctas_per_sm = 0;
    p.id = -1;
    return p;
}

}  // namespace

extern "C" sgemm_status_t sgemm_splitk_noalloc_plan(int N, int K, int M, int split_k,
                                                    const sgemm_plan_t *selected,
                                                    sgemm_plan_t *out) {
    if (!out || split_k < 2) return SGEMM_ERR_INVALID_ARG;
    sgemm_plan_t plan = selected ? *selected : sgemm_plan_select(N, K, M);
    plan.split_k = split_k;
    if (plan.variant == SGEMM_VARIANT_TC05) {
        // the tcgen05 kernel reduces its split inside a cluster, without scratch: the
        // CUDA-core streaming kernel with split_k splits
        plan = streaming_plan(split_k);
    } else if (plan.variant == SGEMM_VARIANT_LDG_CLUSTER) {
        plan.variant = SGEMM_VARIANT_LDG_MIXFMA;  // the same kernel, split through the array
    }
    *out = plan;
    return sgemm_plan_check(out, M, N, K);
}

extern "C" sgemm_status_t sgemm_bf16_skinny_splitk_noalloc(
    const sgemm_bf16_t *x, long long ldx, const sgemm_bf16_t *W, sgemm_bf16_t *y, long long ldy,
    int M, int N, int K, int split_k, sgemm_stream_t stream) {
    if (M < 1 || M > sk::kMaxM || N < 1 || K < 1) return SGEMM_ERR_INVALID_ARG;
    if (!x || !W || !y || ldx < K || ldy < N) return SGEMM_ERR_INVALID_ARG;
    if (split_k < 2) return SGEMM_ERR_INVALID_ARG;
    if (K % 8) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(W)) & 15u)
        return SGEMM_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(y) & 1u) || ldx % 8) return SGEMM_ERR_MISALIGNED;
    // the partial sums [split][M][N] must fit the fixed scratch
    if (static_cast<unsigned long long>(split_k) * M * N > kScratchFloats)
        return SGEMM_ERR_UNSUPPORTED_SHAPE;

    sgemm_plan_t plan;
    sgemm_status_t s = sgemm_splitk_noalloc_plan(N, K, M, split_k, nullptr, &plan);
    if (s != SGEMM_OK) return s;
    const sk::KernelInfo *ki = find(M, plan);
    if (!ki) return SGEMM_ERR_UNSUPPORTED_SHAPE;

    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    DeviceSetup *st = nullptr;
    s = setup_current_device(cs, ki->fn, &st);
    if (s != SGEMM_OK) return s;

    const int kps = sk::split_kps(K, split_k);
    const size_t smem = sk::smem_bytes(plan, M, kps);

    sk::Params prm = {};
    prm.item[0].x = x;
    prm.item[0].W = W;
    prm.item[0].y = y;
    prm.item[0].ldx = ldx;
    prm.item[0].ldy = ldy;
    prm.ws = st->scratch;  // every slot the reduce reads is written earlier in this call
    prm.N = N;
    prm.K = K;
    prm.kps = kps;
    prm.split = split_k;
    prm.row_groups = sk::work_units(plan, N);

    // CTAs per SM as the regular path sizes them: the plan's, else the occupancy
    int occ = plan.ctas_per_sm;
    if (occ < 1 &&
        (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, ki->fn, plan.threads, smem) !=
             cudaSuccess ||
         occ < 1))
        occ = 1;
    const long long need = sk::ctas_wanted(plan, N);
    long long slots = static_cast<long long>(st->sms) * occ / split_k;
    if (slots < 1) slots = 1;
    const int grid_x = static_cast<int>(need < slots ? need : slots);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid_x), static_cast<unsigned>(split_k), 1);
    cfg.blockDim = dim3(static_cast<unsigned>(plan.threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = cs;
    void *args[] = {&prm};
    if (cudaLaunchKernelExC(&cfg, ki->fn, args) != cudaSuccess) return SGEMM_ERR_CUDA;

    const long long total = static_cast<long long>(M) * N;
    long long blocks = (total + 255) / 256;
    if (blocks > 8LL * st->sms) blocks = 8LL * st->sms;
    cudaLaunchConfig_t rc = {};
    rc.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    rc.blockDim = dim3(256, 1, 1);
    rc.stream = cs;
    int batch = 1;
    void *rargs[] = {&prm, &batch};
    if (cudaLaunchKernelExC(&rc, sk::kReduceKernels[M], rargs) != cudaSuccess)
        return SGEMM_ERR_CUDA;
    return SGEMM_OK;
}
