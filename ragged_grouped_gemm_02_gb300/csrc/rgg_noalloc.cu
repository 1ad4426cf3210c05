// rgg_noalloc.cu -- rgg_grouped_gemm_noalloc: the grouped GEMM for callers
// that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc at the point where they run
// the GEMM: an inference-engine plugin whose execute step runs inside the
// engine's own memory budget and must not allocate, or a process whose device
// memory is entirely owned by a pool allocator that other code may not go
// around.  rgg_grouped_gemm needs a handle, and rgg_create allocates the
// handle's device status word with cudaMalloc.  This entry point needs no
// handle: the only scratch the kernels use beyond their inputs and outputs --
// the status word that records bad offsets or a timed-out wait, and the mixed
// launch's tile counters -- lives in a file-scope device array instead.
//
// The array is small and fixed: every GPU that loads librgg.so holds it until
// the process exits.  All calls share it, so calls that run at the same time
// on the GPU (on different streams, or from different threads) race on the
// status word; serialise them if you read status_out.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "rgg.h"
#include "rgg_internal.h"

namespace {

// 256 bytes of device scratch per GPU.  The kernels use the first int32 as
// the status word (zero = OK) and, for the mixed launch, the three int32 at
// byte 64 as its tile counters (zero here at load, and zero again after every
// mixed launch); the rest is reserved.
constexpr int kNoallocScratchWords = 64;
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoallocScratchWords];

constexpr size_t kStatusWordBytes = sizeof(int32_t);
static_assert(kStatusWordBytes <= sizeof(int32_t) * kNoallocScratchWords, "status word must fit the scratch");

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool ready = false;
    int32_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
    int smem_optin = 0;
};

std::mutex g_setup_mutex;
DeviceSetup g_setup[kMaxDevices];

// Once per device, with that device current: find the device address of the
// scratch array (host code cannot use the array's name as a device pointer),
// and read the SM count and shared-memory limit the planner needs.  The
// address is kept for the life of the process, so the entry point must not be
// used on a device after cudaDeviceReset() on it.
rgg_status setup_device(int device, DeviceSetup* out) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup& s = g_setup[device];
    if (!s.ready) {
        int major = 0, minor = 0;
        cudaError_t err;
        if ((err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device)) != cudaSuccess ||
            (err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device)) != cudaSuccess ||
            (err = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess ||
            (err = cudaDeviceGetAttribute(&s.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device)) !=
                cudaSuccess)
            return rgg::host_cuda_failure(err, "rgg_grouped_gemm_noalloc: cudaDeviceGetAttribute");
        if (major != 10 || minor != 3) {
            rgg::host_set_last_error("rgg_grouped_gemm_noalloc: librgg is built for sm_103a only");
            return RGG_ERR_UNSUPPORTED;
        }
        void* addr = nullptr;
        err = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
        if (err != cudaSuccess) return rgg::host_cuda_failure(err, "rgg_grouped_gemm_noalloc: cudaGetSymbolAddress");
        s.scratch = static_cast<int32_t*>(addr);
        s.ready = true;
    }
    *out = s;
    return RGG_OK;
}

}  // namespace

extern "C" rgg_status rgg_grouped_gemm_noalloc(const void* X, const void* W, const int32_t* group_offsets, void* Y,
                                               int E, int64_t M_tot, int K, int N, int32_t* status_out,
                                               void* stream) {
    rgg_status s = rgg::host_check_gemm_args(X, W, group_offsets, Y, E, M_tot, K, N);
    if (s != RGG_OK) return s;
    if (status_out && (reinterpret_cast<uintptr_t>(status_out) % 4) != 0) return RGG_ERR_INVALID_ARG;
    // The kernels' scratch need does not grow with the problem: the status
    // word and three counters.  Sizes the kernels cannot take (E > 4096,
    // M_tot >= 2^31, K or N not a multiple of 8) were rejected above.
    if (kStatusWordBytes > sizeof(g_noalloc_scratch) || 19 * sizeof(int32_t) > sizeof(g_noalloc_scratch)) {
        rgg::host_set_last_error("rgg_grouped_gemm_noalloc: request needs more than the 256-byte scratch");
        return RGG_ERR_UNSUPPORTED;
    }

    int device = -1;
    cudaError_t err = cudaGetDevice(&device);
    if (err != cudaSuccess) return rgg::host_cuda_failure(err, "rgg_grouped_gemm_noalloc: cudaGetDevice");
    if (device < 0 || device >= kMaxDevices) return RGG_ERR_UNSUPPORTED;
    DeviceSetup dev;
    s = setup_device(device, &dev);
    if (s != RGG_OK) return s;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The status word must start at zero: the kernel only records the first error.
    err = cudaMemsetAsync(dev.scratch, 0, kStatusWordBytes, st);
    if (err != cudaSuccess) return rgg::host_cuda_failure(err, "rgg_grouped_gemm_noalloc: cudaMemsetAsync");
    // The same plan, kernels and launch as rgg_grouped_gemm with default options.
    s = rgg::host_grouped_gemm(dev.num_sms, dev.smem_optin, dev.scratch, X, W, group_offsets, Y, E, M_tot, K, N, st,
                               nullptr);
    if (s != RGG_OK) return s;
    if (status_out) {
        err = cudaMemcpyAsync(status_out, dev.scratch, kStatusWordBytes, cudaMemcpyDefault, st);
        if (err != cudaSuccess) return rgg::host_cuda_failure(err, "rgg_grouped_gemm_noalloc: status copy");
    }
    return RGG_OK;
}
