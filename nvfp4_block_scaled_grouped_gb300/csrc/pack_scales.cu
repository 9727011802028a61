// pack_scales.cu -- row-major e4m3 scales -> the reordered atom layout read by
// the block-scaled MMA.
//
// Layout ("nvfp4 group gemm" submission 385043, kernel body where the scale
// tensors are built; the same layout in submission 499344): 512-byte atoms of
// 128 rows x 4 scale blocks. Inside an atom, row r and block kb sit at byte
// 16*(r%32) + 4*((r/32)%4) + kb%4, i.e. 32 lines of 16 bytes, line l holding
// rows l, l+32, l+64, l+96 (4 blocks each) -- the 32x128-bit shape tcgen05.cp
// copies into TMEM. Atoms run K-atom fastest: atom (r/128)*ceil(k/64) + kb/4.
// Rows pad to a multiple of 128 and blocks to a multiple of 4 with zeros.
//
// A warp takes one task: a 128-row block and 8 consecutive atoms of it. Lane
// l reads the 32 scale bytes (8 atoms x 4 blocks) of rows l, l+32, l+64, l+96
// -- a whole 32-byte sector of each row when the rows are 16-byte aligned --
// and writes line l of each of the 8 atoms, so every store instruction of the
// warp writes one whole 512-byte atom.
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kAtomsPerTask = 8;

// Tasks of one matrix: 128-row blocks x groups of kAtomsPerTask atoms.
__host__ __device__ inline long long pack_task_count(int rows, int k) {
    const long long k_atoms = (k + 63) / 64;
    return (long long)((rows + 127) / 128) * ((k_atoms + kAtomsPerTask - 1) / kAtomsPerTask);
}

// Tasks t0, t0 + step, ... of one matrix (tasks = row blocks x atom groups).
__device__ __forceinline__ void pack_tasks(const uint8_t *__restrict__ src, int rows, int k, uint8_t *__restrict__ dst,
                                           long long tasks, long long t0, long long step) {
    const int lane = threadIdx.x & 31;
    const int kbs = k / 16;
    const int k_atoms = (k + 63) / 64;
    const int groups = (k_atoms + kAtomsPerTask - 1) / kAtomsPerTask;
    const uintptr_t base = reinterpret_cast<uintptr_t>(src);
    const bool vec = (kbs % 16) == 0 && (base % 16) == 0;
    const bool words = (kbs % 4) == 0 && (base % 4) == 0;
    for (long long t = t0; t < tasks; t += step) {
        const int rb = (int)(t / groups);
        const int ka0 = (int)(t - (long long)rb * groups) * kAtomsPerTask;
        const int na = k_atoms - ka0 < kAtomsPerTask ? k_atoms - ka0 : kAtomsPerTask;
        uint32_t w[4][kAtomsPerTask];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int j = 0; j < kAtomsPerTask; ++j)
                w[c][j] = 0u;
            const int r = rb * 128 + 32 * c + lane;
            if (r < rows) {
                const uint8_t *s = src + (size_t)r * kbs + 4 * ka0;
                const int avail = kbs - 4 * ka0;  // this row's bytes from block 4 * ka0 on (> 0)
                if (vec && avail >= 4 * kAtomsPerTask) {
                    const uint4 a = __ldg(reinterpret_cast<const uint4 *>(s));
                    const uint4 b = __ldg(reinterpret_cast<const uint4 *>(s) + 1);
                    w[c][0] = a.x, w[c][1] = a.y, w[c][2] = a.z, w[c][3] = a.w;
                    w[c][4] = b.x, w[c][5] = b.y, w[c][6] = b.z, w[c][7] = b.w;
                } else if (words) {
#pragma unroll
                    for (int j = 0; j < kAtomsPerTask; ++j)
                        if (4 * j < avail)
                            w[c][j] = __ldg(reinterpret_cast<const uint32_t *>(s) + j);
                } else {
#pragma unroll
                    for (int j = 0; j < kAtomsPerTask; ++j)
#pragma unroll
                        for (int bb = 0; bb < 4; ++bb)
                            if (4 * j + bb < avail)
                                w[c][j] |= (uint32_t)__ldg(s + 4 * j + bb) << (8 * bb);
                }
            }
        }
        uint4 *out = reinterpret_cast<uint4 *>(dst) + ((size_t)rb * k_atoms + ka0) * 32 + lane;
#pragma unroll
        for (int j = 0; j < kAtomsPerTask; ++j)
            if (j < na)
                out[(size_t)j * 32] = make_uint4(w[0][j], w[1][j], w[2][j], w[3][j]);
    }
}

__global__ void __launch_bounds__(256) pack_scales_kernel(const uint8_t *__restrict__ src, int rows, int k,
                                                          uint8_t *__restrict__ dst, long long tasks) {
    pack_tasks(src, rows, k, dst, tasks, (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5),
               (long long)gridDim.x * (blockDim.x / 32));
}

// Several matrices in one launch: CTA row blockIdx.y packs matrix blockIdx.y.
struct PackBatch {
    const uint8_t *src[kPackBatchMax];
    uint8_t *dst[kPackBatchMax];
    int rows[kPackBatchMax];
    int k[kPackBatchMax];
};

__global__ void __launch_bounds__(256) pack_scales_batched_kernel(const __grid_constant__ PackBatch b) {
    const int i = blockIdx.y;
    const int rows = b.rows[i], k = b.k[i];
    const long long tasks = pack_task_count(rows, k);
    pack_tasks(b.src[i], rows, k, b.dst[i], tasks, (long long)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5),
               (long long)gridDim.x * (blockDim.x / 32));
}

}  // namespace

cudaError_t launch_pack_scales(const uint8_t *src, int rows, int k, uint8_t *dst, cudaStream_t stream) {
    const long long tasks = pack_task_count(rows, k);
    if (tasks == 0)
        return cudaSuccess;
    int device = 0, sms = 148;
    cudaGetDevice(&device);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    long long blocks = (tasks + 7) / 8;  // 8 warps per CTA, one task each
    const long long cap = (long long)sms * 8;
    if (blocks > cap)
        blocks = cap;
    pack_scales_kernel<<<(unsigned)blocks, 256, 0, stream>>>(src, rows, k, dst, tasks);
    return cudaGetLastError();
}

cudaError_t launch_pack_scales_batched(int count, const uint8_t *const *src, const int *rows, const int *k,
                                       uint8_t *const *dst, cudaStream_t stream) {
    if (count <= 0)
        return cudaSuccess;
    if (count > kPackBatchMax)
        return cudaErrorInvalidValue;
    PackBatch b;
    long long max_tasks = 0, total_tasks = 0;
    for (int i = 0; i < count; ++i) {
        b.src[i] = src[i];
        b.dst[i] = dst[i];
        b.rows[i] = rows[i];
        b.k[i] = k[i];
        const long long tasks = pack_task_count(rows[i], k[i]);
        max_tasks = tasks > max_tasks ? tasks : max_tasks;
        total_tasks += tasks;
    }
    if (max_tasks == 0)
        return cudaSuccess;
    int device = 0, sms = 148;
    cudaGetDevice(&device);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    // about 8 CTAs per SM over the whole batch, spread in proportion to the
    // largest matrix (smaller ones finish early in their row)
    long long per_row = (8LL * sms * max_tasks + total_tasks - 1) / total_tasks;
    const long long need = (max_tasks + 7) / 8;
    if (per_row > need)
        per_row = need;
    if (per_row < 1)
        per_row = 1;
    pack_scales_batched_kernel<<<dim3((unsigned)per_row, (unsigned)count), 256, 0, stream>>>(b);
    return cudaGetLastError();
}

}  // namespace nvfp4
