// Host side of the BF16 skinny GEMM library: argument checks, plan selection,
// launch.  The C ABI is declared (and documented) in include/sgemm_skinny.h.
//
// Dispatch follows the plan tables of vLLM PR #62949 (Details: per-shape
// configs from a sweep, keyed by the local (N, K) and M) and vLLM PR #65306
// (Details: table keyed by capability and local (N, K)).  Here the table is
// compiled in for sm_103 only, and shapes without an entry get a heuristic
// plan instead of another library's GEMM.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "internal.h"
#include "tc05_consts.h"

namespace {

using sk::KernelInfo;

struct TableEntry {
    int N, K, M;
    int variant, threads, R, LPR, U, split, stages, ctas_per_sm;
};

// Plans from the offline sweep (generated file; see the package's sweep module).
const TableEntry kTable[] = {
#include "plan_table.inc"
    {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0}  // sentinel
};
const int kTableSize = static_cast<int>(sizeof(kTable) / sizeof(kTable[0])) - 1;

constexpr int kThreadChoices[] = {256, 128};
constexpr int kNumThreadChoices = 2;
constexpr size_t kMaxSmem = sk::kMaxSmemOptin;
constexpr size_t kDefaultWorkspace = 16u << 20;

const KernelInfo *table_for_m(int M) {
    switch (M) {
        case 1: return sk::kKernelsM1;
        case 2: return sk::kKernelsM2;
        case 3: return sk::kKernelsM3;
        case 4: return sk::kKernelsM4;
        case 5: return sk::kKernelsM5;
        case 6: return sk::kKernelsM6;
        case 7: return sk::kKernelsM7;
        case 8: return sk::kKernelsM8;
        default: return nullptr;
    }
}

// stages 0 is accepted as 1 (single batch in flight).
const KernelInfo *find_kernel(int variant, int M, int R, int LPR, int U, int stages) {
    const KernelInfo *t = table_for_m(M);
    if (!t) return nullptr;
    if (variant == SGEMM_VARIANT_TC05) {
        // one kernel per M; the rest are launch parameters
        for (int i = 0; i < sk::kKernelCountPerM; ++i)
            if (t[i].variant == variant && t[i].R == R && t[i].LPR == LPR) return &t[i];
        return nullptr;
    }
    if (stages == 0) stages = 1;
    for (int i = 0; i < sk::kKernelCountPerM; ++i)
        if (t[i].variant == variant && t[i].R == R && t[i].LPR == LPR && t[i].U == U &&
            t[i].stages == stages)
            return &t[i];
    return nullptr;
}

struct DeviceState {
    bool probed = false;
    bool supported = false;
    int sms = 0;
    int *err = nullptr;  // device error word (a static device variable of the library)
    float *ws = nullptr;
    size_t ws_bytes = 0;
    std::map<std::tuple<const void *, int, size_t>, int> occupancy;
    std::map<const void *, bool> smem_attr_set;
};

std::mutex g_mu;
std::map<int, DeviceState> g_dev;


sgemm_status_t check_tc05_plan(const sgemm_plan_t &p, int M, int K) {
    if (p.threads != sk::tc05::kThreads || p.rows_per_warp != sk::tc05::kRows ||
        p.lanes_per_row != 0 || p.vec_bytes != 16)
        return SGEMM_ERR_UNSUPPORTED_SHAPE;
    if (p.k_unroll < 1 || p.k_unroll > sk::tc05::kMaxNb) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    if (p.stages < 2 || p.stages > sk::tc05::kMaxRingSlots) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    if (p.ctas_per_sm < 0 || p.ctas_per_sm > 8) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    const int kbox = (K + sk::tc05::kBoxK - 1) / sk::tc05::kBoxK;
    if (p.split_k < 1 || p.split_k > sk::tc05::kMaxSplit || p.split_k > kbox)
        return SGEMM_ERR_UNSUPPORTED_SHAPE;
    if (!find_kernel(p.variant, M, p.rows_per_warp, p.lanes_per_row, 0, 0))
        return SGEMM_ERR_UNSUPPORTED_SHAPE;
    // leave 1 KiB for the kernel's static shared memory (mbarriers, flags)
    const size_t smem = sk::tc05_smem_bytes(M, p.stages, p.k_unroll, sk::tc05_splits_used(K, p.split_k));
    if (smem + 1024 > kMaxSmem) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    return SGEMM_OK;
}

sgemm_status_t check_plan(const sgemm_plan_t &p, int M, int N, int K) {
    (void)N;
    if (p.variant == SGEMM_VARIANT_TC05) return check_tc05_plan(p, M, K);
    if (p.variant != SGEMM_VARIANT_LDG && p.variant != SGEMM_VARIANT_LDG_MIXFMA &&
        p.variant != SGEMM_VARIANT_LDG_FFMA2 && p.variant != SGEMM_VARIANT_MMA &&
        p.variant != SGEMM_VARIANT_LDGX_MIXFMA && p.variant != SGEMM_VARIANT_LDGX_FFMA2 &&
        p.variant != SGEMM_VARIANT_LDG_MMA && p.variant != SGEMM_VARIANT_LDG_CLUSTER)
        return SGEMM_ERR_UNSUPPORTED_SHAPE;
    // a cluster holds at most 8 CTAs portably
    if (p.variant == SGEMM_VARIANT_LDG_CLUSTER && p.split_k > 8) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    if (p.threads < 32 || p.threads > sk::kMaxThreads || p.threads % 32) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    if (p.vec_bytes != 16 || p.stages < 0 || p.stages > 2) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    if (p.split_k < 1 || p.split_k > 64) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    if (p.ctas_per_sm < 0 || p.ctas_per_sm > 32) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    if (!find_kernel(p.variant, M, p.rows_per_warp, p.lanes_per_row, p.k_unroll, p.stages))
        return SGEMM_ERR_UNSUPPORTED_SHAPE;
    if (p.variant == SGEMM_VARIANT_MMA && p.threads < 64)
        return SGEMM_ERR_UNSUPPORTED_SHAPE;
    const int kps = sk::split_kps(K, p.split_k);
    if (static_cast<long long>(p.split_k - 1) * kps >= K) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    if (sk::smem_bytes(p, M, kps) > kMaxSmem) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    return SGEMM_OK;
}

sgemm_plan_t make_plan(int variant, int threads, int R, int LPR, int U, int split, int stages,
                       int ctas, int id) {
    sgemm_plan_t p;
    p.variant = variant;
    p.threads = threads;
    p.rows_per_warp = R;
    p.lanes_per_row = LPR;
    p.k_unroll = U;
    p.vec_bytes = 16;
    p.split_k = split;
    p.stages = stages;
    p.ctas_per_sm = ctas;
    p.id = id;
    return p;
}

// A plan for shapes the table does not hold.  M <= 4: the mixed-precision FMA
// streaming kernel; M >= 5: the 16-row tensor-core kernel (eight FMAs per
// element and x row would make the CUDA-core kernel issue-bound).  K is split
// when the x slice would not leave room for two CTAs per SM, and further while
// the rows alone give fewer than two CTAs per SM of a GB300 (152 SMs) and each
// split keeps at least 512 elements of K.
// SM count of the current device (cached per device); 152, a GB300's count,
// when no device can be queried (plan selection is a host function).
int current_sm_count() {
    static std::mutex mu;
    static std::map<int, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 152;
    }
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
        (void)cudaGetLastError();
        sms = 152;
    }
    cache[dev] = sms;
    return sms;
}

sgemm_plan_t heuristic_plan(int N, int K, int M) {
    int variant = SGEMM_VARIANT_LDG_MIXFMA;
    int R, LPR, U, rows_per_cta;
    if (M >= 5) {
        variant = SGEMM_VARIANT_MMA;
        R = 16, LPR = 4, U = 4;
        rows_per_cta = 16;
    } else if (K <= 128) {
        R = 2, LPR = 16, U = 2;
        rows_per_cta = 8 * 2 * R;
    } else if (M <= 2) {
        R = 1, LPR = 32, U = 8;
        rows_per_cta = 8 * R;
    } else {
        R = 2, LPR = 32, U = 4;
        rows_per_cta = 8 * R;
    }
    int split = 1;
    const size_t budget = 96 * 1024;  // x slice per CTA, leaves room for two CTAs per SM
    if (M >= 1 && K >= 8) {
        const size_t xbytes = static_cast<size_t>(M) * K * 2;
        split = static_cast<int>((xbytes + budget - 1) / budget);
        split = std::max(1, std::min(split, 64));
        const long long ctas = (static_cast<long long>(std::max(N, 1)) + rows_per_cta - 1) / rows_per_cta;
        const long long sms = current_sm_count();
        while (split < 16 && ctas * split < 2 * sms && K / (2 * split) >= 512) split *= 2;
    }
    return make_plan(variant, 256, R, LPR, U, split, 1, 0, -1);
}

sgemm_status_t probe_device(int *dev_out, DeviceState **st_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &st = g_dev[dev];
    if (!st.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SGEMM_ERR_CUDA;
        st.supported = (major == 10 && minor == 3);
        st.sms = sms;
        if (st.supported && sk::device_error_word(&st.err) != cudaSuccess) return SGEMM_ERR_CUDA;
        st.probed = true;
    }
    if (!st.supported) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    *dev_out = dev;
    *st_out = &st;
    return SGEMM_OK;
}

// Requires g_mu held.  `bytes` is the partial-sum space needed.
sgemm_status_t ensure_workspace(DeviceState &st, size_t bytes, cudaStream_t stream) {
    if (st.ws && st.ws_bytes >= bytes) return SGEMM_OK;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return SGEMM_ERR_NO_WORKSPACE;
    if (cap != cudaStreamCaptureStatusNone) return SGEMM_ERR_NO_WORKSPACE;
    size_t want = std::max(bytes, kDefaultWorkspace);
    if (st.ws) {
        // older launches may still read the old scratch
        if (cudaDeviceSynchronize() != cudaSuccess) return SGEMM_ERR_CUDA;
        cudaFree(st.ws);
        st.ws = nullptr;
        st.ws_bytes = 0;
    }
    void *p = nullptr;
    if (cudaMalloc(&p, want) != cudaSuccess) return SGEMM_ERR_CUDA;
    st.ws = static_cast<float *>(p);
    st.ws_bytes = want;
    return SGEMM_OK;
}

// Requires g_mu held.
int occupancy(DeviceState &st, const void *fn, int threads, size_t smem) {
    auto key = std::make_tuple(fn, threads, smem);
    auto it = st.occupancy.find(key);
    if (it != st.occupancy.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess) n = 1;
    n = std::max(n, 1);
    st.occupancy[key] = n;
    return n;
}

sgemm_status_t validate_common(int M, int N, int K, int batch) {
    if (M < 1 || M > sk::kMaxM || N < 1 || K < 1) return SGEMM_ERR_INVALID_ARG;
    if (batch < 1 || batch > sk::kMaxBatch) return SGEMM_ERR_INVALID_ARG;
    if (K % 8) return SGEMM_ERR_UNSUPPORTED_SHAPE;
    return SGEMM_OK;
}

sgemm_status_t validate_item(const sgemm_pair_t &it, int N, int K) {
    if (!it.x || !it.W || !it.y) return SGEMM_ERR_INVALID_ARG;
    if (it.ldx < K || it.ldy < N) return SGEMM_ERR_INVALID_ARG;
    const uintptr_t ax = reinterpret_cast<uintptr_t>(it.x);
    const uintptr_t aw = reinterpret_cast<uintptr_t>(it.W);
    const uintptr_t ay = reinterpret_cast<uintptr_t>(it.y);
    if ((ax | aw) & 15u) return SGEMM_ERR_MISALIGNED;  // 128-bit loads
    if (ay & 1u) return SGEMM_ERR_MISALIGNED;          // 16-bit stores
    if (it.ldx % 8) return SGEMM_ERR_MISALIGNED;
    return SGEMM_OK;
}

// What the kernels' epilogue writes besides BF16 y (see store_out in skinny_ldg.cuh).
struct Epilogue {
    bool out_f32 = false;     // y is FP32
    uint16_t *xn = nullptr;   // fused chain step: the next GEMM's input (single problem only)
    long long ldxn = 0;
    long long xn_len = 0;
    float xn_scale = 1.0f;
};

// Byte ranges [a, a + na) and [b, b + nb) overlap.
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

sgemm_status_t validate_epilogue(const Epilogue &ep, const sgemm_pair_t &it, int M, int N, int K) {
    if (ep.out_f32 && (reinterpret_cast<uintptr_t>(it.y) & 3u)) return SGEMM_ERR_MISALIGNED;
    if (!ep.xn) return SGEMM_OK;
    if (ep.xn_len < 1 || ep.xn_len > 0x7fffffffLL || ep.ldxn < ep.xn_len) return SGEMM_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(ep.xn) & 1u) return SGEMM_ERR_MISALIGNED;
    // the next input is written while this GEMM still reads x and W and writes y
    const size_t xn_bytes = (static_cast<size_t>(M - 1) * ep.ldxn + ep.xn_len) * 2;
    const size_t x_bytes = (static_cast<size_t>(M - 1) * it.ldx + K) * 2;
    const size_t y_bytes = (static_cast<size_t>(M - 1) * it.ldy + N) * 2;
    const size_t w_bytes = static_cast<size_t>(N) * K * 2;
    if (overlaps(ep.xn, xn_bytes, it.x, x_bytes) || overlaps(ep.xn, xn_bytes, it.y, y_bytes) ||
        overlaps(ep.xn, xn_bytes, it.W, w_bytes))
        return SGEMM_ERR_INVALID_ARG;
    return SGEMM_OK;
}

// The common kernel parameters of one launch (no split-K scratch).
sk::Params make_params(const sgemm_pair_t *items, int batch, int N, int K, unsigned flags,
                       const Epilogue &ep) {
    sk::Params prm;
    std::memset(&prm, 0, sizeof(prm));
    for (int b = 0; b < batch; ++b) {
        prm.item[b].x = items[b].x;
        prm.item[b].W = items[b].W;
        prm.item[b].y = items[b].y;
        prm.item[b].ldx = items[b].ldx;
        prm.item[b].ldy = items[b].ldy;
        prm.item[b].xn = ep.xn;
        prm.item[b].ldxn = ep.ldxn;
    }
    prm.out_f32 = ep.out_f32 ? 1 : 0;
    prm.xn_len = static_cast<int>(ep.xn_len);
    prm.xn_scale = ep.xn_scale;
    prm.N = N;
    prm.K = K;
    prm.split = 1;
    prm.flags = static_cast<int>(flags);
    return prm;
}

// The TMA + tcgen05 kernel: one launch, no scratch (its K split reduces inside
// a thread-block cluster).
sgemm_status_t run_tc05(const sgemm_pair_t *items, int batch, int M, int N, int K,
                        const sgemm_plan_t &plan, unsigned flags, cudaStream_t stream,
                        const Epilogue &ep, DeviceState &st, const void *fn) {
    sk::Params prm = make_params(items, batch, N, K, flags, ep);
    prm.err = st.err;
    long long ctas = 1;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!st.smem_attr_set[fn]) {
            if (sk::allow_max_dynamic_smem(fn) != cudaSuccess) return SGEMM_ERR_CUDA;
            st.smem_attr_set[fn] = true;
        }
        const size_t smem = sk::tc05_smem_bytes(M, plan.stages, plan.k_unroll, 1);
        const int occ = plan.ctas_per_sm > 0 ? plan.ctas_per_sm
                                             : occupancy(st, fn, sk::tc05::kThreads, smem);
        ctas = std::max<long long>(1, static_cast<long long>(st.sms) * occ / batch);
    }
    if (sk::tc05_launch(prm, batch, M, plan, ctas, fn, stream) != cudaSuccess) return SGEMM_ERR_CUDA;
    return SGEMM_OK;
}

sgemm_status_t run(const sgemm_pair_t *items, int batch, int M, int N, int K,
                   const sgemm_plan_t *plan_in, unsigned flags, cudaStream_t stream,
                   const Epilogue &ep = Epilogue()) {
    sgemm_status_t s = validate_common(M, N, K, batch);
    if (s != SGEMM_OK) return s;
    if (flags & ~(SGEMM_FLAG_PDL | SGEMM_FLAG_WEIGHTS_READONLY | SGEMM_FLAG_TEST_STALL))
        return SGEMM_ERR_INVALID_ARG;
    if (!items) return SGEMM_ERR_INVALID_ARG;
    for (int b = 0; b < batch; ++b) {
        s = validate_item(items[b], N, K);
        if (s != SGEMM_OK) return s;
        s = validate_epilogue(ep, items[b], M, N, K);
        if (s != SGEMM_OK) return s;
    }
    if (ep.xn && batch != 1) return SGEMM_ERR_INVALID_ARG;
    const sgemm_plan_t plan = plan_in ? *plan_in : sgemm_plan_select(N, K, M);
    s = check_plan(plan, M, N, K);
    if (s != SGEMM_OK) return s;

    int dev = 0;
    DeviceState *st = nullptr;
    s = probe_device(&dev, &st);
    if (s != SGEMM_OK) return s;

    const KernelInfo *ki = find_kernel(plan.variant, M, plan.rows_per_warp, plan.lanes_per_row,
                                       plan.k_unroll, plan.stages);
    if (plan.variant == SGEMM_VARIANT_TC05) return run_tc05(items, batch, M, N, K, plan, flags,
                                                            stream, ep, *st, ki->fn);
    const int split = plan.split_k;
    const int kps = sk::split_kps(K, split);
    const size_t smem = sk::smem_bytes(plan, M, kps);
    // the split CTAs of a row range form a cluster and reduce in rank 0's shared memory
    const bool clv = plan.variant == SGEMM_VARIANT_LDG_CLUSTER && split > 1;

    sk::Params prm;
    std::memset(&prm, 0, sizeof(prm));
    for (int b = 0; b < batch; ++b) {
        prm.item[b].x = items[b].x;
        prm.item[b].W = items[b].W;
        prm.item[b].y = items[b].y;
        prm.item[b].ldx = items[b].ldx;
        prm.item[b].ldy = items[b].ldy;
        prm.item[b].xn = ep.xn;
        prm.item[b].ldxn = ep.ldxn;
    }
    prm.out_f32 = ep.out_f32 ? 1 : 0;
    prm.xn_len = static_cast<int>(ep.xn_len);
    prm.xn_scale = ep.xn_scale;
    prm.N = N;
    prm.K = K;
    prm.kps = kps;
    prm.split = split;
    prm.row_groups = sk::work_units(plan, N);
    prm.flags = static_cast<int>(flags);
    prm.cl_rows = clv ? sk::cluster_rows(plan) : 0;

    int grid_x = 0;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (split > 1 && !clv) {
            const size_t need = static_cast<size_t>(batch) * split * M * N * sizeof(float);
            s = ensure_workspace(*st, need, stream);
            if (s != SGEMM_OK) return s;
            prm.ws = st->ws;
        }
        prm.err = st->err;
        if (!st->smem_attr_set[ki->fn]) {
            if (sk::allow_max_dynamic_smem(ki->fn) != cudaSuccess) return SGEMM_ERR_CUDA;
            st->smem_attr_set[ki->fn] = true;
        }
        const int occ = plan.ctas_per_sm > 0 ? plan.ctas_per_sm
                                             : occupancy(*st, ki->fn, plan.threads, smem);
        const long long need_ctas = sk::ctas_wanted(plan, N);
        const long long slots = std::max<long long>(
            1, static_cast<long long>(st->sms) * occ / (static_cast<long long>(split) * batch));
        // a cluster-split grid gives each warp one task at most (the size of rank 0's buffer)
        grid_x = static_cast<int>(std::max<long long>(1, clv ? need_ctas : std::min(need_ctas, slots)));
    }

    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(grid_x), static_cast<unsigned>(split),
                       static_cast<unsigned>(batch));
    cfg.blockDim = dim3(static_cast<unsigned>(plan.threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (flags & SGEMM_FLAG_PDL) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (clv) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = static_cast<unsigned>(split);
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = static_cast<unsigned>(na);
    void *args[] = {&prm};
    if (cudaLaunchKernelExC(&cfg, ki->fn, args) != cudaSuccess) return SGEMM_ERR_CUDA;

    if (split > 1 && !clv) {
        const long long total = static_cast<long long>(batch) * M * N;
        int blocks = static_cast<int>(std::min<long long>((total + 255) / 256, 8LL * st->sms));
        cudaLaunchConfig_t rc;
        std::memset(&rc, 0, sizeof(rc));
        rc.gridDim = dim3(static_cast<unsigned>(std::max(blocks, 1)), 1, 1);
        rc.blockDim = dim3(256, 1, 1);
        rc.dynamicSmemBytes = 0;
        rc.stream = stream;
        if (flags & SGEMM_FLAG_PDL) {
            rc.attrs = attr;
            rc.numAttrs = 1;
        }
        int batch_arg = batch;
        void *rargs[] = {&prm, &batch_arg};
        if (cudaLaunchKernelExC(&rc, sk::kReduceKernels[M], rargs) != cudaSuccess)
            return SGEMM_ERR_CUDA;
    }
    return SGEMM_OK;
}

}  // namespace

namespace sk {

int split_kps(int K, int split) {
    const int chunks = K / 8;
    const int per = (chunks + split - 1) / split;
    return per * 8;
}

// Rows of a CTA of a cluster-split plan, whose grid gives each warp one task (one
// row group of R * 32 / lanes_per_row rows) at most.
int cluster_rows(const sgemm_plan_t &plan) {
    return plan.threads / 32 * (32 / plan.lanes_per_row) * plan.rows_per_warp;
}

size_t smem_bytes(const sgemm_plan_t &plan, int M, int kps) {
    const size_t chunks = static_cast<size_t>(kps) / 8;
    if (plan.variant == SGEMM_VARIANT_LDGX_MIXFMA || plan.variant == SGEMM_VARIANT_LDGX_FFMA2)
        return 0;  // x is read from global memory
    if (plan.variant == SGEMM_VARIANT_MMA) {
        // x rows padded by one chunk, plus two reduction buffers [NW][16][4 or 8] floats
        return static_cast<size_t>(M) * (chunks + 1) * 16 +
               2 * static_cast<size_t>(plan.threads / 32) * 16 * (M <= 4 ? 4 : 8) * sizeof(float);
    }
    size_t bytes = static_cast<size_t>(M) * chunks * 16;
    if (plan.variant == SGEMM_VARIANT_LDG_CLUSTER && plan.split_k > 1)
        bytes += static_cast<size_t>(plan.split_k) * cluster_rows(plan) * M * sizeof(float);
    return bytes;
}

int work_units(const sgemm_plan_t &plan, int N) {
    if (plan.variant == SGEMM_VARIANT_TC05) return (N + tc05::kRows - 1) / tc05::kRows;
    if (plan.variant == SGEMM_VARIANT_MMA) return (N + 15) / 16;
    const int rows_per_task = (32 / plan.lanes_per_row) * plan.rows_per_warp;
    return (N + rows_per_task - 1) / rows_per_task;
}

cudaError_t allow_max_dynamic_smem(const void *fn) {
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, fn);
    if (e != cudaSuccess) return e;
    const int dyn = static_cast<int>(kMaxSmemOptin) - static_cast<int>(a.sharedSizeBytes);
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
}

long long ctas_wanted(const sgemm_plan_t &plan, int N) {
    const long long units = work_units(plan, N);
    if (plan.variant == SGEMM_VARIANT_MMA || plan.variant == SGEMM_VARIANT_TC05)
        return units;  // one tile per CTA at most
    const int warps = plan.threads / 32;
    return (units + warps - 1) / warps;
}

}  // namespace sk

extern "C" {

sgemm_plan_t sgemm_plan_select(int N, int K, int M) {
    for (int i = 0; i < kTableSize; ++i) {
        const TableEntry &e = kTable[i];
        if (e.N == N && e.K == K && e.M == M) {
            sgemm_plan_t p = make_plan(e.variant, e.threads, e.R, e.LPR, e.U, e.split, e.stages,
                                       e.ctas_per_sm, i);
            if (check_plan(p, M, N, K) == SGEMM_OK) return p;
        }
    }
    return heuristic_plan(N, K, M);
}

int sgemm_plan_count(void) { return sk::kKernelCountPerM * kNumThreadChoices; }

sgemm_status_t sgemm_plan_get(int index, sgemm_plan_t *plan) {
    if (!plan || index < 0 || index >= sgemm_plan_count()) return SGEMM_ERR_INVALID_ARG;
    const KernelInfo &k = sk::kKernelsM1[index / kNumThreadChoices];
    if (k.variant == SGEMM_VARIANT_TC05) {
        // six single-box stages, or three stages of two boxes (the same bytes in flight)
        const bool first = (index % kNumThreadChoices) == 0;
        *plan = make_plan(k.variant, sk::tc05::kThreads, sk::tc05::kRows, 0, first ? 1 : 2, 1,
                          first ? 6 : 3, 0, -1);
        return SGEMM_OK;
    }
    *plan = make_plan(k.variant, kThreadChoices[index % kNumThreadChoices], k.R, k.LPR, k.U, 1,
                      k.stages, 0, -1);
    return SGEMM_OK;
}

sgemm_status_t sgemm_plan_check(const sgemm_plan_t *plan, int M, int N, int K) {
    if (!plan) return SGEMM_ERR_INVALID_ARG;
    sgemm_status_t s = validate_common(M, N, K, 1);
    if (s != SGEMM_OK) return s;
    return check_plan(*plan, M, N, K);
}

sgemm_status_t sgemm_bf16_skinny_ex(const sgemm_bf16_t *x, long long ldx, const sgemm_bf16_t *W,
                                    sgemm_bf16_t *y, long long ldy, int M, int N, int K,
                                    const sgemm_plan_t *plan, unsigned flags,
                                    sgemm_stream_t stream) {
    sgemm_pair_t it;
    it.x = x;
    it.W = W;
    it.y = y;
    it.ldx = ldx;
    it.ldy = ldy;
    return run(&it, 1, M, N, K, plan, flags, reinterpret_cast<cudaStream_t>(stream));
}

sgemm_status_t sgemm_bf16_skinny_f32out_ex(const sgemm_bf16_t *x, long long ldx,
                                           const sgemm_bf16_t *W, float *y, long long ldy, int M,
                                           int N, int K, const sgemm_plan_t *plan, unsigned flags,
                                           sgemm_stream_t stream) {
    sgemm_pair_t it;
    it.x = x;
    it.W = W;
    it.y = reinterpret_cast<sgemm_bf16_t *>(y);
    it.ldx = ldx;
    it.ldy = ldy;
    Epilogue ep;
    ep.out_f32 = true;
    return run(&it, 1, M, N, K, plan, flags, reinterpret_cast<cudaStream_t>(stream), ep);
}

sgemm_status_t sgemm_bf16_skinny_rescale_ex(const sgemm_bf16_t *x, long long ldx,
                                            const sgemm_bf16_t *W, sgemm_bf16_t *y, long long ldy,
                                            int M, int N, int K, sgemm_bf16_t *x_next,
                                            long long ld_next, long long n_next, float scale,
                                            const sgemm_plan_t *plan, unsigned flags,
                                            sgemm_stream_t stream) {
    if (!x_next) return SGEMM_ERR_INVALID_ARG;
    sgemm_pair_t it;
    it.x = x;
    it.W = W;
    it.y = y;
    it.ldx = ldx;
    it.ldy = ldy;
    Epilogue ep;
    ep.xn = x_next;
    ep.ldxn = ld_next;
    ep.xn_len = n_next;
    ep.xn_scale = scale;
    return run(&it, 1, M, N, K, plan, flags, reinterpret_cast<cudaStream_t>(stream), ep);
}

sgemm_status_t sgemm_bf16_skinny(const sgemm_bf16_t *x, const sgemm_bf16_t *W, sgemm_bf16_t *y,
                                 int M, int N, int K, sgemm_stream_t stream) {
    return sgemm_bf16_skinny_ex(x, K, W, y, N, M, N, K, nullptr, 0u, stream);
}

sgemm_status_t sgemm_bf16_skinny_batched_ex(const sgemm_pair_t *items, int batch, int M, int N,
                                            int K, const sgemm_plan_t *plan, unsigned flags,
                                            sgemm_stream_t stream) {
    return run(items, batch, M, N, K, plan, flags, reinterpret_cast<cudaStream_t>(stream));
}

sgemm_status_t sgemm_bf16_skinny_batched(const sgemm_pair_t *items, int batch, int M, int N, int K,
                                         sgemm_stream_t stream) {
    return run(items, batch, M, N, K, nullptr, 0u, reinterpret_cast<cudaStream_t>(stream));
}

sgemm_status_t sgemm_init(void) {
    int dev = 0;
    DeviceState *st = nullptr;
    sgemm_status_t s = probe_device(&dev, &st);
    if (s != SGEMM_OK) return s;
    std::lock_guard<std::mutex> lk(g_mu);
    return ensure_workspace(*st, kDefaultWorkspace, nullptr);
}

sgemm_status_t sgemm_device_errors(int *flags) {
    if (!flags) return SGEMM_ERR_INVALID_ARG;
    *flags = 0;
    int dev = 0;
    DeviceState *st = nullptr;
    sgemm_status_t s = probe_device(&dev, &st);
    if (s != SGEMM_OK) return s;
    std::lock_guard<std::mutex> lk(g_mu);
    if (cudaDeviceSynchronize() != cudaSuccess) return SGEMM_ERR_CUDA;
    int *w = st->err;
    if (cudaMemcpy(flags, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(w, 0, sizeof(int)) != cudaSuccess)
        return SGEMM_ERR_CUDA;
    return SGEMM_OK;
}

const char *sgemm_status_string(sgemm_status_t status) {
    switch (status) {
        case SGEMM_OK: return "ok";
        case SGEMM_ERR_INVALID_ARG: return "invalid argument";
        case SGEMM_ERR_UNSUPPORTED_SHAPE: return "unsupported shape or plan";
        case SGEMM_ERR_MISALIGNED: return "misaligned pointer or row stride";
        case SGEMM_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
        case SGEMM_ERR_NO_WORKSPACE: return "split-K scratch missing during stream capture";
        case SGEMM_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

const char *sgemm_version(void) { return "0.1.0"; }

}  // extern "C"
