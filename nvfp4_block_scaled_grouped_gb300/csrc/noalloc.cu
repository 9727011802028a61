// noalloc.cu -- the grouped GEMM for callers that cannot allocate device memory.
//
// nvfp4_grouped_gemm keeps its scratch (tile prefix sum, group table, TMA
// descriptors, status word) in a buffer it cudaMalloc's on the first call for
// each (device, stream). Some callers must not have the library allocate at
// all: frameworks that hand out every byte of device memory from their own
// pre-planned arena and account for it, and latency-critical callers for whom
// a cudaMalloc / cudaFree -- which may synchronise the whole device -- in the
// middle of their work is not acceptable. nvfp4_grouped_gemm_noalloc runs the
// same GEMM kernel with its scratch in the fixed array below
// instead, and never allocates.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace nvfp4 {
namespace {

constexpr size_t kNoallocWorkspaceBytes = workspace_bytes(NVFP4_NOALLOC_MAX_GROUPS);

// The scratch of every nvfp4_grouped_gemm_noalloc call on a device. Each GPU
// that loads the library holds these bytes until the process exits.
static __device__ __align__(256) uint8_t g_noalloc_workspace[kNoallocWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

}  // namespace

// Device address of g_noalloc_workspace on `device` (the current device).
// In host code the array's name is only a host-side stand-in, so the address
// is looked up once per device, at the device's first call, and cached; after
// a cudaDeviceReset the cached address is stale, so the entry point must not
// be used again in that process.
int noalloc_workspace(int device, void **out) {
    if (device < 0 || device >= kMaxDevices)
        return fail(NVFP4_ERR_UNSUPPORTED, "device ordinal %d out of range", device);
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[device]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_workspace);
        if (e != cudaSuccess || p == nullptr)
            return cuda_fail(e, "cudaGetSymbolAddress(static workspace)");
        g_noalloc_ptr[device] = p;
    }
    *out = g_noalloc_ptr[device];
    return NVFP4_OK;
}

// The static array's address on `device` if a call has set it up there, else
// null (nothing is looked up or allocated).
void *noalloc_workspace_if_ready(int device) {
    if (device < 0 || device >= kMaxDevices)
        return nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    return g_noalloc_ptr[device];
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" int nvfp4_grouped_gemm_noalloc(int group_count, const nvfp4_problem_size *problem_sizes,
                                          const void *const *A, const void *const *B, const void *const *SFA,
                                          const void *const *SFB, void *const *C, nvfp4_stream_t stream) {
    if (group_count > NVFP4_NOALLOC_MAX_GROUPS)
        return fail(NVFP4_ERR_INVALID_ARG,
                    "group_count %d exceeds the %d groups the static workspace of nvfp4_grouped_gemm_noalloc holds",
                    group_count, NVFP4_NOALLOC_MAX_GROUPS);
    const int block_n = current_block_n();
    GroupArgs args[NVFP4_NOALLOC_MAX_GROUPS];
    long long total = 0;
    int s = check_groups(group_count, NVFP4_NOALLOC_MAX_GROUPS, problem_sizes, A, B, SFA, SFB, C, block_n, args,
                         &total);
    if (s != NVFP4_OK || total == 0)
        return s;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    void *ws = nullptr;
    s = noalloc_workspace(device, &ws);
    if (s != NVFP4_OK)
        return s;
    // The array keeps the previous call's contents. Each call rewrites the
    // descriptors it reads; the call counters of the header (bytes 64..127:
    // the descriptor-publication counter, the count of CTAs past it, the
    // epoch) must start at zero. The status word (byte 0) is left alone: it
    // collects the bits of every call until nvfp4_device_status reads and
    // clears it.
    e = cudaMemsetAsync(static_cast<uint8_t *>(ws) + 64, 0, 64, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "clearing the static workspace header");
    WorkspaceState state;  // empty slot cache: every descriptor is patched
    return launch_on_workspace(group_count, args, total, block_n, ws, NVFP4_NOALLOC_MAX_GROUPS, 0, 0, 1, &state,
                               reinterpret_cast<cudaStream_t>(stream));
}
