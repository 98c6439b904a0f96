// status.cu -- per-device status word, size helpers and diagnostics of libnvfp4.
//
// The library allocates nothing: the status word is a module-scope __device__
// variable (one per device and CUDA context that loads the library), reached by
// kernels through the address cached here per device and context.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace nvfp4 {

__device__ unsigned g_status_words[2];   // [0] first nvfp4_status recorded, [1] detail

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceCtx g_ctx[kMaxDevices];
nvfp4_status g_ctx_state[kMaxDevices];
bool g_ctx_init[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id (for the process's lifetime, unlike the handle, which a new
// context may reuse) of the context current on this thread; 0 if none is
// current yet or the driver does not provide it.  The driver entry points come
// through the runtime, so loading the library needs no libcuda.
unsigned long long current_ctx_id() {
    static const CtxGetCurrentFn get_current = []() -> CtxGetCurrentFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<CtxGetCurrentFn>(p);
    }();
    static const CtxGetIdFn get_id = []() -> CtxGetIdFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<CtxGetIdFn>(p);
    }();
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext c = nullptr;
    if (get_current(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    unsigned long long id = 0;
    if (get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}
}  // namespace

nvfp4_status device_ctx(DeviceCtx* ctx) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    const unsigned long long id = current_ctx_id();
    if (!g_ctx_init[dev] || id == 0 || id != g_ctx[dev].ctx_id) {
        int major = 0, minor = 0, sms = 0;
        nvfp4_status st = NVFP4_OK;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            st = NVFP4_ERR_CUDA;
        } else if (major != 10 || minor != 3) {
            st = NVFP4_ERR_UNSUPPORTED_DEVICE;
        }
        void* addr = nullptr;
        if (st == NVFP4_OK && cudaGetSymbolAddress(&addr, g_status_words) != cudaSuccess) {
            st = NVFP4_ERR_CUDA;
        }
        // the lookup above made the runtime's context current if none was
        g_ctx[dev] = DeviceCtx{static_cast<unsigned*>(addr), sms, dev, current_ctx_id()};
        g_ctx_state[dev] = st;
        g_ctx_init[dev] = true;
    }
    *ctx = g_ctx[dev];
    return g_ctx_state[dev];
}

TensorMapEncodeTiledFn tensor_map_encode_fn() {
    static const TensorMapEncodeTiledFn fn = []() -> TensorMapEncodeTiledFn {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<TensorMapEncodeTiledFn>(ptr);
    }();
    return fn;
}

// ---------------------------------------------------------------------------
// Exhaustive conversion probe
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cvt_probe_kernel(uint32_t* first, uint32_t* last,
                                                        uint32_t* counters, uint32_t end,
                                                        uint32_t per_thread) {
    __shared__ uint32_t s_first[144], s_last[144], s_cnt[4];
    for (int i = threadIdx.x; i < 144; i += blockDim.x) {
        s_first[i] = 0xFFFFFFFFu;
        s_last[i] = 0u;
    }
    if (threadIdx.x < 4) s_cnt[threadIdx.x] = 0u;
    __syncthreads();

    const uint64_t tid = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const uint64_t lo64 = tid * per_thread;
    if (lo64 <= end) {
        const uint32_t lo = static_cast<uint32_t>(lo64);
        const uint32_t hi = static_cast<uint32_t>((lo64 + per_thread - 1) < end ? (lo64 + per_thread - 1) : end);
        uint32_t nonmono2 = 0, nonmono4 = 0, asym = 0, nan4 = 0;
        // codes of the pattern just before the range (for the monotonicity check)
        uint32_t prev2 = 0, prev4 = 0;
        if (lo > 0) {
            float xp = __uint_as_float(lo - 1);
            prev2 = cvt_e2m1x2(xp, xp) & 15u;
            prev4 = cvt_e4m3(xp);
        }
        uint32_t run2 = 0xFFFFFFFFu, run4 = 0xFFFFFFFFu, start2 = lo, start4 = lo;
        for (uint32_t p = lo;; ++p) {
            float x = __uint_as_float(p);
            uint32_t c2 = cvt_e2m1x2(x, x) & 15u;
            uint32_t c4 = cvt_e4m3(x);
            uint32_t n2 = cvt_e2m1x2(-x, -x) & 15u;
            if (n2 != (c2 | 8u)) ++asym;
            if ((c4 & 0x7Fu) == 0x7Fu) ++nan4;
            if (c2 < prev2) ++nonmono2;
            if (c4 < prev4) ++nonmono4;
            if (c2 != run2) {
                if (run2 != 0xFFFFFFFFu) {
                    atomicMin(&s_first[run2 & 15u], start2);
                    atomicMax(&s_last[run2 & 15u], p - 1);
                }
                run2 = c2;
                start2 = p;
            }
            if (c4 != run4) {
                if (run4 != 0xFFFFFFFFu) {
                    atomicMin(&s_first[16 + (run4 & 127u)], start4);
                    atomicMax(&s_last[16 + (run4 & 127u)], p - 1);
                }
                run4 = c4;
                start4 = p;
            }
            prev2 = c2;
            prev4 = c4;
            if (p == hi) break;
        }
        atomicMin(&s_first[run2 & 15u], start2);
        atomicMax(&s_last[run2 & 15u], hi);
        atomicMin(&s_first[16 + (run4 & 127u)], start4);
        atomicMax(&s_last[16 + (run4 & 127u)], hi);
        atomicAdd(&s_cnt[0], nonmono2);
        atomicAdd(&s_cnt[1], nonmono4);
        atomicAdd(&s_cnt[2], asym);
        atomicAdd(&s_cnt[3], nan4);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 144; i += blockDim.x) {
        if (s_first[i] != 0xFFFFFFFFu) atomicMin(&first[i], s_first[i]);
        if (s_last[i] != 0u) atomicMax(&last[i], s_last[i]);
    }
    if (threadIdx.x < 4 && s_cnt[threadIdx.x]) atomicAdd(&counters[threadIdx.x], s_cnt[threadIdx.x]);
}

// Self-check of the scale recipe's two forms: block i takes the row amax with
// bf16 bits i (every positive finite bf16 and zero: i = 0 .. 0x7F7F); the row's
// S, T, 1/T and FMA-range decision must equal the IEEE recipe's, and for a row
// in the FMA range its threads take every block amax a <= amax (bf16 bits
// j <= i), whose code and multiplier must equal the IEEE form's, bit for bit.
// counters[0] = pairs compared (rows in the FMA range), counters[1] = mismatches;
// mismatch[0] = how many were recorded, then up to 8 (i, j) pairs.
__global__ void __launch_bounds__(256) recipe_check_kernel(unsigned long long* counters, uint32_t* mismatch) {
    const uint32_t i = blockIdx.x;
    const float amax = __uint_as_float(i << 16);
    const ScaleRecipe rec(amax);
    const ScaleRecipe ref = ScaleRecipe::ieee(amax);
    // the row's own quantities: the FMA range decision, S, T and 1/T
    if (threadIdx.x == 0 && (rec.fast != ref.fast || __float_as_uint(rec.S) != __float_as_uint(ref.S) ||
                             __float_as_uint(rec.T) != __float_as_uint(ref.T) ||
                             __float_as_uint(rec.rcpT) != __float_as_uint(ref.rcpT))) {
        atomicAdd(&counters[1], 1ull);
        const uint32_t k = atomicAdd(mismatch, 1u);
        if (k < 8) {
            mismatch[1 + 2 * k] = i;
            mismatch[2 + 2 * k] = 0xFFFFFFFFu;   // the row's recipe, not a block
        }
    }
    if (!rec.fast) return;
    unsigned long long n = 0, bad = 0;
    for (uint32_t j = threadIdx.x; j <= i; j += blockDim.x) {
        const float a = __uint_as_float(j << 16);
        float r_fma, r_ieee;
        const uint32_t s_fma = rec.block_as<true>(a, &r_fma);
        const uint32_t s_ieee = ref.block_as<false>(a, &r_ieee);
        ++n;
        if (s_fma != s_ieee || __float_as_uint(r_fma) != __float_as_uint(r_ieee)) {
            ++bad;
            const uint32_t k = atomicAdd(mismatch, 1u);
            if (k < 8) {
                mismatch[1 + 2 * k] = i;
                mismatch[2 + 2 * k] = j;
            }
        }
    }
    atomicAdd(&counters[0], n);
    if (bad) atomicAdd(&counters[1], bad);
}

__global__ void cvt_probe_init_kernel(uint32_t* first, uint32_t* last, uint32_t* counters) {
    for (int i = threadIdx.x; i < 144; i += blockDim.x) {
        first[i] = 0xFFFFFFFFu;
        last[i] = 0u;
    }
    if (threadIdx.x < 4) counters[threadIdx.x] = 0u;
}

// ---------------------------------------------------------------------------
// Bounded-wait failure check
// ---------------------------------------------------------------------------
__global__ void wait_timeout_kernel(unsigned* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives: phase 0 never completes and the wait must give up.
        if (!mbar_wait_bounded(&bar, 0u, limit_ns, nullptr))
            record_error(status, NVFP4_ERR_TIMEOUT, DETAIL_DEBUG_WAIT);
    }
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

size_t nvfp4_packed_bytes(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 0) return 0;
    return static_cast<size_t>(rows * (cols / 2));
}

size_t nvfp4_sf_bytes(int64_t rows, int64_t cols) {
    if (rows < 0 || cols < 0) return 0;
    return static_cast<size_t>(round_up(rows, 128) * round_up(cols / 16, 4));
}

nvfp4_status nvfp4_get_device_status(nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    unsigned words[2] = {0u, 0u};
    if (cudaMemcpyFromSymbol(words, g_status_words, sizeof(words)) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (words[0] != 0u) {
        const unsigned zero[2] = {0u, 0u};
        if (cudaMemcpyToSymbol(g_status_words, zero, sizeof(zero)) != cudaSuccess)
            return NVFP4_ERR_CUDA;
    }
    return static_cast<nvfp4_status>(words[0]);
}

const char* nvfp4_status_string(nvfp4_status s) {
    switch (s) {
        case NVFP4_OK: return "NVFP4_OK";
        case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG";
        case NVFP4_ERR_ALIGNMENT: return "NVFP4_ERR_ALIGNMENT";
        case NVFP4_ERR_SHAPE: return "NVFP4_ERR_SHAPE";
        case NVFP4_ERR_UNSUPPORTED_DEVICE: return "NVFP4_ERR_UNSUPPORTED_DEVICE";
        case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
        case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT";
        case NVFP4_ERR_DEVICE_INPUT: return "NVFP4_ERR_DEVICE_INPUT";
        case NVFP4_ERR_WORKSPACE: return "NVFP4_ERR_WORKSPACE";
    }
    return "NVFP4_ERR_UNKNOWN";
}

nvfp4_status nvfp4_debug_scale_recipe_check(unsigned long long* counters, uint32_t* mismatch,
                                            nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (!counters || !mismatch) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(counters, 8) || !aligned(mismatch, 4)) return NVFP4_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(counters, 0, 2 * sizeof(unsigned long long), s) != cudaSuccess ||
        cudaMemsetAsync(mismatch, 0, 17 * sizeof(uint32_t), s) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    recipe_check_kernel<<<0x7F80, 256, 0, s>>>(counters, mismatch);
    NVFP4_CHECK_LAUNCH();
    return NVFP4_OK;
}

nvfp4_status nvfp4_debug_cvt_probe(uint32_t* first, uint32_t* last, uint32_t* counters,
                                   nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (!first || !last || !counters) return NVFP4_ERR_INVALID_ARG;
    if (!aligned(first, 4) || !aligned(last, 4) || !aligned(counters, 4)) return NVFP4_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cvt_probe_init_kernel<<<1, 256, 0, s>>>(first, last, counters);
    NVFP4_CHECK_LAUNCH();
    const uint32_t end = 0x7F800000u;        // +0 .. +inf inclusive
    const int threads = 256;
    const int blocks = ctx.sm_count * 8;
    const uint64_t total = static_cast<uint64_t>(end) + 1;
    const uint64_t nthreads = static_cast<uint64_t>(threads) * blocks;
    const uint32_t per_thread = static_cast<uint32_t>((total + nthreads - 1) / nthreads);
    cvt_probe_kernel<<<blocks, threads, 0, s>>>(first, last, counters, end, per_thread);
    NVFP4_CHECK_LAUNCH();
    return NVFP4_OK;
}

nvfp4_status nvfp4_debug_wait_timeout(int64_t timeout_ns, nvfp4_stream_t stream) {
    DeviceCtx ctx;
    nvfp4_status st = device_ctx(&ctx);
    if (st != NVFP4_OK) return st;
    if (timeout_ns < 1000000 || timeout_ns > 10000000000LL) return NVFP4_ERR_INVALID_ARG;
    wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        ctx.status, static_cast<uint64_t>(timeout_ns));
    NVFP4_CHECK_LAUNCH();
    return NVFP4_OK;
}

}  // extern "C"
