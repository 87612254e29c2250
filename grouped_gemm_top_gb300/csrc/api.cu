// Library-wide entry points: init, status strings, sizes.
#include <mutex>

#include "common.cuh"

namespace moe {

static constexpr int kMaxDevices = 64;
static int g_sm_count[kMaxDevices] = {0};
static bool g_init[kMaxDevices] = {false};
static std::mutex g_mu;

cudaError_t gemm_set_attributes();   // gemm.cu
cudaError_t quant_set_attributes();  // quant.cu
cudaError_t gemm_init_driver();      // gemm.cu
void route_scratch_forget(int device);  // route.cu

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
    return g_sm_count[dev];
}

bool device_initialized() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    return g_init[dev];
}

}  // namespace moe

extern "C" int moe_abi_version(void) { return 200; }

extern "C" const char* moe_status_string(int s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape";
        case MOE_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_NOT_INITIALIZED: return "moe_init was not called for this device";
        case MOE_ERR_BAD_EXPERT: return "expert index out of range or repeated within a token";
        case MOE_ERR_BAD_OFFSETS: return "group offsets not monotone, not 128-aligned or beyond the buffer";
        case MOE_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel timed out";
        case MOE_ERR_CAPACITY: return "padded rows exceed the buffer capacity";
        default: return "unknown status";
    }
}

// Every call redoes the per-device set-up (kernel attributes, SM count) in
// the context that is current now, so a caller that reset the device
// (cudaDeviceReset) calls moe_init again and the library works in the new
// primary context; the address of the no-allocation routing scratch is
// looked up again on its next call for the same reason.
extern "C" moe_status_t moe_init(int device) {
    using namespace moe;
    if (device < 0 || device >= kMaxDevices) return MOE_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    if (cudaSetDevice(device) != cudaSuccess) return MOE_ERR_CUDA;
    g_init[device] = false;
    route_scratch_forget(device);
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return MOE_ERR_CUDA;
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;   // built for sm_103a only
    if (gemm_init_driver() != cudaSuccess) return MOE_ERR_CUDA;
    if (gemm_set_attributes() != cudaSuccess) return MOE_ERR_CUDA;
    if (quant_set_attributes() != cudaSuccess) return MOE_ERR_CUDA;
    g_sm_count[device] = sms;
    g_init[device] = true;
    return MOE_OK;
}

extern "C" int64_t moe_row_capacity(int T, int E, int k) {
    if (T < 0 || E <= 0 || k <= 0) return -1;
    const int64_t R = (int64_t)T * k;
    const int64_t pad = 127 * (R < E ? R : (int64_t)E);
    return (R + pad + 127) / 128 * 128;
}

extern "C" size_t moe_workspace_size(int op, int T, int d, int E, int k, int f) {
    if (T < 0 || d < 1 || E < 1 || k < 1 || f < 1) return (size_t)-1;
    switch (op) {
        case MOE_OP_ROUTE_TOPK: return moe_route_workspace_size(T, E);
        case MOE_OP_PERMUTE: return moe_permute_workspace_size(T, E);
        case MOE_OP_GROUP_QUANTIZE:
        case MOE_OP_GATHER_QUANTIZE:
        case MOE_OP_GROUPED_GEMM:
        case MOE_OP_UNPERMUTE_COMBINE:
        case MOE_OP_COMBINE_BWD:
        case MOE_OP_ROUTE_BWD: return 0;
        default: return (size_t)-1;
    }
}
