// quantize.cu -- fused NVFP4 quantise-and-pack of an activation matrix.
//
// x [rows][k] bf16 or fp16 (row-major, k % 16 == 0) becomes the operand pair
// the grouped GEMM reads: e2m1 codes [rows][k/2] (two per byte, the even k in
// the low nibble) and e4m3fn scales, one per 16 K-elements, written directly
// in the 512-byte atom layout (128 rows x 4 scale blocks per atom; byte
// 16*(r%32) + 4*((r/32)%4) + kb%4 of atom (r/128)*ceil(k/64) + kb/4, the
// reordered scale layout of the "nvfp4 group gemm" submission 385043) with
// the padding rows and blocks zero.
//
// The quantisation is the one the grouped-GEMM task states for its operands,
// per row and 16-element block:
//   amax = max|x|;  sf = e4m3fn(amax / 6), round to nearest even, saturating
//   at 448;  code = e2m1(x / dec(sf)), round to nearest even, saturating at
//   6, sign of x kept;  all codes +0 when dec(sf) == 0.
// amax / 6 is formed exactly on every e4m3 rounding midpoint and within
// about 2 ulps elsewhere, then converted exactly to e4m3. The e2m1 codes come
// from the hardware conversion (cvt.rn.satfinite.e2m1x2.f32) of quotients
// x / dec that are exact on the rounding boundaries of the e2m1 grid and
// within about 2 ulps elsewhere (see quantize16): for bf16 and fp16 inputs
// that decides the scale and every code as the exact quotients would.
//
// Layout of the work: a unit is one row and 32 consecutive scale blocks (512
// K-elements); a warp takes a unit with one lane per 16-element block, so each
// of its loads reads 512 contiguous bytes of the row and each code store
// writes 256 contiguous bytes. Lanes kb % 4 == 0 gather the four scale bytes
// of their atom column with shuffles and store them as one 32-bit word. Units
// cover the padded rows (a multiple of 128) and the padded scale blocks (a
// multiple of 4), whose scale bytes are written as zero. Warps walk the units
// grid-stride, two units per step so that two loads of each lane are in
// flight. The quotients are formed two at a time with the packed fp32
// instructions (mul / fma .f32x2, each lane the IEEE operation of its scalar
// form). The kernel streams its input once (bound by HBM bandwidth for large
// inputs).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kQuantThreads = 256;  // 8 warps per CTA
constexpr int kUnitBlocks = 32;     // scale blocks per unit (one per lane)

// e4m3fn code of s >= 0 (finite), round to nearest even, 448 for s >= 448:
// the hardware conversion (cvt.rn.satfinite.e4m3x2.f32, round to nearest
// even on the e4m3 grid including its subnormals, saturating at the largest
// finite value), low byte.
__device__ __forceinline__ uint32_t e4m3_code(float s) {
    uint32_t out;
    asm("{\n\t.reg .b16 h;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 h, %2, %1;\n\t"
        "cvt.u32.u16 %0, h;\n\t}"
        : "=r"(out)
        : "f"(s), "f"(0.0f));
    return out & 0xFFu;
}

// Value of a non-negative e4m3fn code (not NaN), exact in fp32.
__device__ __forceinline__ float e4m3_decode(uint32_t c) {
    const uint32_t e = c >> 3, m = c & 7u;
    if (e == 0)
        return (float)m * 0.001953125f;  // m * 2^-9
    return __uint_as_float(((e + 120u) << 23) | (m << 20));  // (1 + m/8) * 2^(e-7)
}

// The 16 elements of one block (two 16-byte loads) as fp32 (exact).
template <bool BF16>
__device__ __forceinline__ void unpack16(const uint4 (&v)[2], float (&f)[16]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t w[4] = {v[h].x, v[h].y, v[h].z, v[h].w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (BF16) {
                f[8 * h + 2 * q] = __uint_as_float(w[q] << 16);
                f[8 * h + 2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
            } else {
                const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&w[q]));
                f[8 * h + 2 * q] = t.x;
                f[8 * h + 2 * q + 1] = t.y;
            }
        }
    }
}

// Four e2m1 codes pairs -> one 32-bit word: byte i holds (q[2i+1] << 4) | q[2i],
// each code round-to-nearest-even with saturation at +-6 (hardware cvt).
__device__ __forceinline__ uint32_t cvt_e2m1x8(const float (&q)[8]) {
    uint32_t out;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(out)
        : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
    return out;
}

// x / d (d > 0) from an estimate r of 1/d by one corrected-quotient step of
// Markstein's division method: q0 = x * r, q = q0 + (x - q0 * d) * r, the
// residual x - q0 * d exact (FMA). With r within a few ulps of 1/d, q is
// exactly x / d whenever that quotient is representable (the correction
// moves q0 by (x/d - q0)(1 + O(ulp)), far less than half an ulp away from the
// exact value) and within about 2 ulps of it otherwise.
__device__ __forceinline__ float div_corrected(float x, float d, float r) {
    const float q0 = x * r;
    return fmaf(fmaf(-q0, d, x), r, q0);
}

// The same step for two dividends x0, x1 over one divisor d (nd = -d), with
// the packed fp32 instructions: q0 = x * r, e = q0 * (-d) + x, q = e * r + q0,
// each rounded to nearest even per lane as the scalar mul / fma are.
__device__ __forceinline__ void div_corrected2(float x0, float x1, float nd, float r, float &q0, float &q1) {
    asm("{\n\t.reg .b64 xx, rr, dd, q, e;\n\t"
        "mov.b64 xx, {%2, %3};\n\t"
        "mov.b64 rr, {%4, %4};\n\t"
        "mov.b64 dd, {%5, %5};\n\t"
        "mul.rn.f32x2 q, xx, rr;\n\t"
        "fma.rn.f32x2 e, q, dd, xx;\n\t"
        "fma.rn.f32x2 q, e, rr, q;\n\t"
        "mov.b64 {%0, %1}, q;\n\t}"
        : "=f"(q0), "=f"(q1)
        : "f"(x0), "f"(x1), "f"(r), "f"(nd));
}

// Hardware reciprocal estimate (PTX rcp.approx, about 1 ulp); d here is an
// e4m3 value in [2^-9, 448], a normal fp32 number.
__device__ __forceinline__ float rcp_estimate(float d) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// Quantise one 16-element block: its e4m3 scale code, and its 16 e2m1 codes
// packed into 8 bytes (element j in bits 4j..4j+3).
//
// amax / 6 and the quotients x / dec come from div_corrected(2): exact on every
// quotient that is representable -- in particular on every e4m3 rounding
// midpoint amax / 6 and every e2m1 rounding boundary x / dec = t -- so those
// ties are decided by round-to-nearest-even as for the exact quotient; every
// other quotient is within about 2 ulps of the exact one, and for bf16 / fp16
// inputs none lies within 2^-10 (relative) of a boundary, so the scale and the
// codes are those of the exact quotients.
__device__ __forceinline__ uint32_t quantize16(const float (&f)[16], uint2 &packed) {
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
        amax = fmaxf(amax, fabsf(f[j]));
    const uint32_t sc = e4m3_code(div_corrected(amax, 6.0f, 1.0f / 6.0f));
    const float dec = e4m3_decode(sc);
    uint32_t w[2] = {0u, 0u};
    if (dec != 0.0f) {
        const float r = rcp_estimate(dec);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float q[8];
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                div_corrected2(f[8 * h + j], f[8 * h + j + 1], -dec, r, q[j], q[j + 1]);
                // (the correction turns x = -0 into +0; the quotient has x's sign)
                q[j] = copysignf(q[j], f[8 * h + j]);
                q[j + 1] = copysignf(q[j + 1], f[8 * h + j + 1]);
            }
            w[h] = cvt_e2m1x8(q);
        }
    }
    packed = make_uint2(w[0], w[1]);
    return sc;
}

// chunks_m, chunks_s: the host's multiplier and shift that divide a unit
// index by the units per row (see launch_quantize_pack).
template <bool BF16>
__global__ void __launch_bounds__(kQuantThreads) quantize_pack_kernel(const uint16_t *__restrict__ x, int rows, int k,
                                                                      uint8_t *__restrict__ codes,
                                                                      uint8_t *__restrict__ sf_atoms,
                                                                      uint32_t chunks_m, int chunks_s) {
    const int lane = threadIdx.x & 31;
    const int k_blocks = k / 16;
    const int k_atoms = (k + 63) / 64;
    const int blocks_pad = 4 * k_atoms;
    const int chunks = (blocks_pad + kUnitBlocks - 1) / kUnitBlocks;
    const int units = ((rows + 127) / 128) * 128 * chunks;
    const int stride = gridDim.x * (kQuantThreads / 32);
    const unsigned full = 0xffffffffu;
    for (int u0 = blockIdx.x * (kQuantThreads / 32) + (threadIdx.x >> 5); u0 < units; u0 += 2 * stride) {
        int r[2], kb[2];
        bool real[2];
        uint4 raw[2][2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int u = u0 + i * stride;
            r[i] = (int)(((uint64_t)(uint32_t)u * chunks_m) >> chunks_s);  // u / chunks
            kb[i] = (u - r[i] * chunks) * kUnitBlocks + lane;
            real[i] = u < units && r[i] < rows && kb[i] < k_blocks;
            const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)r[i] * (size_t)k + (size_t)kb[i] * 16);
            raw[i][0] = real[i] ? __ldg(src) : make_uint4(0, 0, 0, 0);
            raw[i][1] = real[i] ? __ldg(src + 1) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            if (u0 + i * stride >= units)
                break;  // warp-uniform
            uint32_t sc = 0;
            if (real[i]) {
                float f[16];
                unpack16<BF16>(raw[i], f);
                uint2 packed;
                sc = quantize16(f, packed);
                *reinterpret_cast<uint2 *>(codes + (size_t)r[i] * (size_t)(k / 2) + (size_t)kb[i] * 8) = packed;
            }
            // the scale bytes of blocks kb..kb+3 (one atom column) -> one word
            uint32_t word = sc;
            word |= __shfl_down_sync(full, sc, 1) << 8;
            word |= __shfl_down_sync(full, sc, 2) << 16;
            word |= __shfl_down_sync(full, sc, 3) << 24;
            if ((lane & 3) == 0 && kb[i] < blocks_pad) {
                const uint32_t rr = (uint32_t)r[i];
                uint8_t *atom = sf_atoms + ((size_t)(rr >> 7) * (size_t)k_atoms + (size_t)((uint32_t)kb[i] >> 2)) * kSfAtomBytes;
                *reinterpret_cast<uint32_t *>(atom + 16 * (rr & 31u) + 4 * ((rr >> 5) & 3u)) = word;
            }
        }
    }
}

}  // namespace

cudaError_t launch_quantize_pack(const void *x, bool bf16, int rows, int k, void *codes, void *sf_atoms,
                                 cudaStream_t stream) {
    const long long chunks = ((long long)(k + 63) / 64 * 4 + kUnitBlocks - 1) / kUnitBlocks;
    const long long units = ((long long)(rows + 127) / 128) * 128 * chunks;
    if (units > 0x7fffffffLL - 2LL * 65535 * 8)
        return cudaErrorInvalidValue;
    int device = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess)
        return e;
    // enough resident warps to keep two 512-byte loads each in flight
    const long long want = (units + kQuantThreads / 32 - 1) / (kQuantThreads / 32);
    const int grid = (int)(want < 8LL * sms ? want : 8LL * sms);
    // unit u's row u / chunks by multiplication: with l = ceil(log2 chunks)
    // and m = ceil(2^(31+l) / chunks), floor(u / chunks) = (u * m) >> (31 + l)
    // for every u < 2^31 (Granlund and Montgomery, "Division by Invariant
    // Integers using Multiplication", Theorem 4.2); m < 2^32
    int l = 0;
    while ((1LL << l) < chunks)
        ++l;
    const uint32_t chunks_m = (uint32_t)((((uint64_t)1 << (31 + l)) + (uint64_t)chunks - 1) / (uint64_t)chunks);
    const uint16_t *xs = static_cast<const uint16_t *>(x);
    uint8_t *c = static_cast<uint8_t *>(codes);
    uint8_t *s = static_cast<uint8_t *>(sf_atoms);
    if (bf16)
        quantize_pack_kernel<true><<<grid, kQuantThreads, 0, stream>>>(xs, rows, k, c, s, chunks_m, 31 + l);
    else
        quantize_pack_kernel<false><<<grid, kQuantThreads, 0, stream>>>(xs, rows, k, c, s, chunks_m, 31 + l);
    return cudaGetLastError();
}

}  // namespace nvfp4
