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
// One thread writes one 16-byte line of one atom: a single 16-byte store per
// thread, consecutive threads writing consecutive lines, so the output stream
// is fully coalesced; the 16 source bytes come from 4 rows.
#include "internal.h"

namespace nvfp4 {
namespace {

// Lines q0, q0 + step, ... of one matrix.
__device__ __forceinline__ void pack_lines(const uint8_t *__restrict__ src, int rows, int k, uint8_t *__restrict__ dst,
                                           long long lines, long long q0, long long step) {
    const int kbs = k / 16;
    const int k_atoms = (k + 63) / 64;
    const bool words = (kbs % 4) == 0 && (reinterpret_cast<uintptr_t>(src) % 4) == 0;
    for (long long q = q0; q < lines; q += step) {
        const long long atom = q >> 5;
        const int l = (int)(q & 31);
        const int row_block = (int)(atom / k_atoms);
        const int ka = (int)(atom % k_atoms);
        uint32_t w[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int r = row_block * 128 + 32 * c + l;
            uint32_t word = 0;
            if (r < rows) {
                const uint8_t *s = src + (size_t)r * kbs + 4 * ka;
                if (words) {
                    word = __ldg(reinterpret_cast<const uint32_t *>(s));
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (4 * ka + j < kbs)
                            word |= (uint32_t)__ldg(s + j) << (8 * j);
                }
            }
            w[c] = word;
        }
        reinterpret_cast<uint4 *>(dst)[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

__global__ void __launch_bounds__(256) pack_scales_kernel(const uint8_t *__restrict__ src, int rows, int k,
                                                          uint8_t *__restrict__ dst, long long lines) {
    pack_lines(src, rows, k, dst, lines, (long long)blockIdx.x * blockDim.x + threadIdx.x,
               (long long)gridDim.x * blockDim.x);
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
    const long long lines = (long long)((rows + 127) / 128) * ((k + 63) / 64) * 32;
    pack_lines(b.src[i], rows, k, b.dst[i], lines, (long long)blockIdx.x * blockDim.x + threadIdx.x,
               (long long)gridDim.x * blockDim.x);
}

}  // namespace

cudaError_t launch_pack_scales(const uint8_t *src, int rows, int k, uint8_t *dst, cudaStream_t stream) {
    const long long row_blocks = (rows + 127) / 128;
    const long long k_atoms = (k + 63) / 64;
    const long long lines = row_blocks * k_atoms * 32;
    if (lines == 0)
        return cudaSuccess;
    int device = 0, sms = 148;
    cudaGetDevice(&device);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    long long blocks = (lines + 255) / 256;
    const long long cap = (long long)sms * 8;
    if (blocks > cap)
        blocks = cap;
    pack_scales_kernel<<<(unsigned)blocks, 256, 0, stream>>>(src, rows, k, dst, lines);
    return cudaGetLastError();
}

cudaError_t launch_pack_scales_batched(int count, const uint8_t *const *src, const int *rows, const int *k,
                                       uint8_t *const *dst, cudaStream_t stream) {
    if (count <= 0)
        return cudaSuccess;
    if (count > kPackBatchMax)
        return cudaErrorInvalidValue;
    PackBatch b;
    long long max_lines = 0, total_lines = 0;
    for (int i = 0; i < count; ++i) {
        b.src[i] = src[i];
        b.dst[i] = dst[i];
        b.rows[i] = rows[i];
        b.k[i] = k[i];
        const long long lines = (long long)((rows[i] + 127) / 128) * ((k[i] + 63) / 64) * 32;
        max_lines = lines > max_lines ? lines : max_lines;
        total_lines += lines;
    }
    if (max_lines == 0)
        return cudaSuccess;
    int device = 0, sms = 148;
    cudaGetDevice(&device);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    // about 8 CTAs per SM over the whole batch, spread in proportion to the
    // largest matrix (smaller ones finish early in their row)
    long long per_row = (8LL * sms * max_lines + total_lines - 1) / total_lines;
    const long long need = (max_lines + 255) / 256;
    if (per_row > need)
        per_row = need;
    if (per_row < 1)
        per_row = 1;
    pack_scales_batched_kernel<<<dim3((unsigned)per_row, (unsigned)count), 256, 0, stream>>>(b);
    return cudaGetLastError();
}

}  // namespace nvfp4
