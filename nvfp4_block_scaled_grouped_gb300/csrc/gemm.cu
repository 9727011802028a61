// gemm.cu -- the grouped NVFP4 block-scaled GEMM for sm_103a.
//
// Two kernels per call, in stream order:
//
//  1. prologue_kernel (one CTA): per-group tile counts and their exclusive
//     prefix sum, a compact per-group table, and per-group TMA descriptors for
//     A and B patched from a host-encoded template with tensormap.replace
//     (the per-group descriptor patching of "nvfp4 group gemm" submission
//     506336, TMA warp, and the one-off descriptor initialisation kernel of
//     submission 499344; here the tile prefix sum also moves to the device).
//     It triggers programmatic dependent launch at once so the GEMM kernel's
//     set-up overlaps it.
//
//  2. grouped_gemm_kernel<BN> (persistent, one CTA per SM, 192 threads):
//       warp 4   TMA producer: A and B tiles (128-byte swizzle) plus the 2 KiB
//                scale runs of each k-tile (1-D bulk copies: a 128-row x 256-K
//                slice of the reordered scale layout is 4 consecutive 512-byte
//                atoms) into a multi-stage shared-memory ring;
//       warp 5   MMA issuer: tcgen05.cp of the scale atoms into TMEM, then
//                tcgen05.mma kind::mxf4nvf4 block_scale (scale_vec::4X = one
//                e4m3 scale per 16 elements) 128 x BN x 64, four per k-tile,
//                into a TMEM accumulator; commits free the smem stage and
//                publish the finished accumulator;
//       warps 0-3 epilogue: tcgen05.ld of the accumulator lanes they own,
//                fp32 -> fp16 round-to-nearest-even, 16-byte stores, rows
//                >= m skipped, column chunks >= n skipped.
//     The persistent schedule walks tiles blockIdx.x, blockIdx.x + gridDim.x,
//     ...; a tile maps to its group by a binary search of the prefix sum
//     (correct across empty groups) and to (m-tile, n-tile) with M fastest,
//     so CTAs working at the same time share a B panel in L2.
//     Roles follow submission 506336 (kernel roles and pipelines), re-sized
//     for GB300: deeper ring, per-stage scale TMEM, bounded waits.
//
// Every mbarrier wait is bounded (%globaltimer); a wait that gives up sets a
// bit in the workspace status word and a CTA-wide abort flag, the other roles
// leave their loops, the producer waits (bounded) for the copies it issued,
// and the CTA frees its TMEM and exits.
#include <cuda_fp16.h>

#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

template <int BN>
struct Cfg {
    static_assert(BN == 128 || BN == 256, "BLOCK_N");
    static constexpr int kStages = (BN == 128) ? 6 : 4;
    static constexpr int kAccStages = (BN == 128) ? 2 : 1;
    static constexpr int kABytes = kBlockM * 128;                  // 128 rows x 256 fp4
    static constexpr int kBBytes = BN * 128;                       // BN rows x 256 fp4
    static constexpr int kSfaBytes = 4 * kSfAtomBytes;             // 4 atoms (one per k-block)
    static constexpr int kSfbRowBlocks = BN / 128;
    static constexpr int kSfbBytes = kSfbRowBlocks * 4 * kSfAtomBytes;
    static constexpr int kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
    static_assert(kStageBytes % 1024 == 0, "stage alignment for the 128-byte swizzle");
    // TMEM columns: accumulators first, then one scale region per smem stage.
    static constexpr int kAccCols = BN;
    static constexpr int kSfaCols = 4 * 4;                         // 4 k-blocks x 4 columns
    static constexpr int kSfbCols = 4 * 4 * kSfbRowBlocks;
    static constexpr int kSfColsPerStage = kSfaCols + kSfbCols;
    static constexpr int kSfColBase = kAccStages * kAccCols;
    static constexpr int kTmemCols = 512;
    static_assert(kSfColBase + kStages * kSfColsPerStage <= kTmemCols, "TMEM budget");
    static constexpr int kThreads = 192;
    static constexpr int kBarrierBytes = 256;
    static constexpr uint32_t kIdesc = ptx::idesc_mxf4nvf4(kBlockM, BN);

    static size_t smem_bytes(int capacity) {
        return 1024 + (size_t)kStages * kStageBytes + kBarrierBytes + round_up(sizeof(int32_t) * (capacity + 1), 16);
    }
};

// Group of `tile`: the g with prefix[g] <= tile < prefix[g + 1].
__device__ __forceinline__ int find_group(const int32_t *prefix, int group_count, int tile) {
    int lo = 0, hi = group_count;  // prefix[lo] <= tile < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= tile)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             uint64_t timeout_ns, uint32_t *status, uint32_t bit) {
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = ptx::globaltimer();
    uint32_t spins = 0;
    while (true) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if ((++spins & 15u) == 0) {
            if (*abort_flag)
                return false;
            if (ptx::globaltimer() - t0 > timeout_ns) {
                *abort_flag = 1;
                atomicOr(status, bit);
                return false;
            }
        }
    }
}

template <int BN>
__global__ void __launch_bounds__(192, 1)
    grouped_gemm_kernel(const WorkspaceView ws, const int group_count, const int total_tiles,
                        const uint64_t timeout_ns) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem_base = ptx::smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    uint8_t *bar_area = smem + C::kStages * C::kStageBytes;
    const uint32_t bars = ptx::smem_addr(bar_area);
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (C::kStages + s); };
    auto accf_bar = [&](int a) { return bars + 8u * (2 * C::kStages + a); };
    auto acce_bar = [&](int a) { return bars + 8u * (2 * C::kStages + C::kAccStages + a); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_area + 192);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 196);
    int32_t *s_prefix = reinterpret_cast<int32_t *>(bar_area + C::kBarrierBytes);

    // ---- set-up that does not depend on the prologue -----------------------
    if (warp == 4 && lane == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < C::kAccStages; ++a) {
            ptx::mbar_init(accf_bar(a), 1);
            ptx::mbar_init(acce_bar(a), 4);
        }
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 5) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish();
    }

    // ---- wait for the prologue's prefix sum, group table and descriptors ---
    ptx::griddep_wait();
    for (int i = threadIdx.x; i <= group_count; i += blockDim.x)
        s_prefix[i] = ws.prefix[i];
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 4) {
        // ===================== TMA producer =====================
        if (lane == 0) {
            const uint64_t pol_a = ptx::l2_policy_evict_last();
            const uint64_t pol_b = ptx::l2_policy_evict_normal();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            int prev_g = -1;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                const int g = find_group(s_prefix, group_count, tile);
                const GroupInfo &gi = ws.groups[g];
                const int local = tile - s_prefix[g];
                const int tiles_m = gi.tiles_m;
                const int tm = local % tiles_m;
                const int tn = local / tiles_m;
                const int k_tiles = gi.k_tiles;
                const int k_blocks = gi.k_blocks;
                const uint8_t *tmap_a = ws.tmaps + (size_t)g * 256;
                const uint8_t *tmap_b = tmap_a + 128;
                if (g != prev_g) {
                    ptx::tmap_acquire(tmap_a);
                    ptx::tmap_acquire(tmap_b);
                    prev_g = g;
                }
                const uint8_t *sfa = gi.sfa + (size_t)tm * k_blocks * kSfAtomBytes;
                int sfb_blocks = gi.sf_row_blocks_b - tn * C::kSfbRowBlocks;
                sfb_blocks = sfb_blocks < C::kSfbRowBlocks ? sfb_blocks : C::kSfbRowBlocks;
                const uint8_t *sfb = gi.sfb + (size_t)tn * C::kSfbRowBlocks * k_blocks * kSfAtomBytes;
                for (int kt = 0; kt < k_tiles; ++kt) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, timeout_ns, ws.status,
                                      kStatusProducerTimeout)) {
                        ok = false;
                        break;
                    }
                    const int nkb = (k_blocks - 4 * kt) < 4 ? (k_blocks - 4 * kt) : 4;
                    const uint32_t sf_bytes = (uint32_t)nkb * kSfAtomBytes;
                    const uint32_t st = smem_base + stage * C::kStageBytes;
                    const uint32_t fb = full_bar(stage);
                    ptx::mbar_arrive_expect_tx(fb, C::kABytes + C::kBBytes + sf_bytes * (1 + sfb_blocks));
                    ptx::tma_load_2d(st, tmap_a, kt * 128, tm * kBlockM, fb, pol_a);
                    ptx::tma_load_2d(st + C::kABytes, tmap_b, kt * 128, tn * BN, fb, pol_b);
                    ptx::bulk_load(st + C::kABytes + C::kBBytes, sfa + (size_t)(4 * kt) * kSfAtomBytes, sf_bytes,
                                   fb, pol_a);
                    for (int j = 0; j < sfb_blocks; ++j)
                        ptx::bulk_load(st + C::kABytes + C::kBBytes + C::kSfaBytes + j * 4 * kSfAtomBytes,
                                       sfb + ((size_t)j * k_blocks + 4 * kt) * kSfAtomBytes, sf_bytes, fb, pol_b);
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok || *abort_flag) {
                // Let every copy this thread issued land before the CTA exits.
                for (int s = 0; s < C::kStages; ++s) {
                    if (!(armed & (1u << s)))
                        continue;
                    const uint32_t par = (armed_parity >> s) & 1u;
                    const uint64_t t0 = ptx::globaltimer();
                    while (!ptx::mbar_try_wait(full_bar(s), par) && ptx::globaltimer() - t0 < timeout_ns) {
                    }
                }
            }
        }
    } else if (warp == 5) {
        // ===================== MMA issuer =====================
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                const int g = find_group(s_prefix, group_count, tile);
                const int k_tiles = ws.groups[g].k_tiles;
                const int k_blocks = ws.groups[g].k_blocks;
                if (!wait_bounded(acce_bar(acc), acc_phase ^ 1u, abort_flag, timeout_ns, ws.status,
                                  kStatusMmaTimeout))
                    break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::kAccCols);
                for (int kt = 0; kt < k_tiles; ++kt) {
                    if (!wait_bounded(full_bar(stage), phase, abort_flag, timeout_ns, ws.status,
                                      kStatusMmaTimeout)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const int nkb = (k_blocks - 4 * kt) < 4 ? (k_blocks - 4 * kt) : 4;
                    const uint32_t st = smem_base + stage * C::kStageBytes;
                    const uint32_t st_sfa = st + C::kABytes + C::kBBytes;
                    const uint32_t st_sfb = st_sfa + C::kSfaBytes;
                    const uint32_t sfa_t = tmem_base + (uint32_t)(C::kSfColBase + stage * C::kSfColsPerStage);
                    const uint32_t sfb_t = sfa_t + C::kSfaCols;
                    for (int kb = 0; kb < nkb; ++kb) {
                        ptx::tc_cp_32x128b_warpx4(sfa_t + 4 * kb, ptx::sdesc_sf_atom(st_sfa + kb * kSfAtomBytes));
#pragma unroll
                        for (int j = 0; j < C::kSfbRowBlocks; ++j)
                            ptx::tc_cp_32x128b_warpx4(
                                sfb_t + kb * (BN / 32) + 4 * j,
                                ptx::sdesc_sf_atom(st_sfb + j * 4 * kSfAtomBytes + kb * kSfAtomBytes));
                    }
                    const uint64_t adesc = ptx::sdesc_kmajor_sw128(st);
                    const uint64_t bdesc = ptx::sdesc_kmajor_sw128(st + C::kABytes);
                    for (int kb = 0; kb < nkb; ++kb) {
                        // +32 bytes per 64-element k-block inside the swizzled row
                        ptx::tc_mma_mxf4nvf4(d_tmem, adesc + 2u * kb, bdesc + 2u * kb, C::kIdesc, sfa_t + 4 * kb,
                                             sfb_t + kb * (BN / 32), (kt | kb) != 0 ? 1u : 0u);
                    }
                    ptx::tc_commit(empty_bar(stage));
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                ptx::tc_commit(accf_bar(acc));
                if (++acc == C::kAccStages) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
        }
    } else {
        // ===================== epilogue (warps 0..3) =====================
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
            const int g = find_group(s_prefix, group_count, tile);
            const GroupInfo &gi = ws.groups[g];
            const int local = tile - s_prefix[g];
            const int tm = local % gi.tiles_m;
            const int tn = local / gi.tiles_m;
            const int m = gi.m, n = gi.n;
            const bool zero = gi.k == 0;
            // One lane waits so the warp leaves (or stays) as a whole: the
            // TMEM loads below are warp-collective.
            int ok = 0;
            if (lane == 0)
                ok = wait_bounded(accf_bar(acc), acc_phase, abort_flag, timeout_ns, ws.status,
                                  kStatusEpilogueTimeout) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok)
                break;
            ptx::tc_fence_after();
            const int row = tm * kBlockM + warp * 32 + lane;
            const uint32_t t_row = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(acc * C::kAccCols);
            __half *c_row = static_cast<__half *>(gi.c) + (size_t)row * (size_t)n;
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; ++cc) {
                const int col = tn * BN + cc * 32;
                if (col >= n)
                    break;
                uint32_t v[32];
                ptx::tmem_ld_32x32b_x32(t_row + cc * 32, v);
                ptx::tmem_ld_wait();
                if (row < m) {
                    uint32_t h[16];
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        __half2 p = __floats2half2_rn(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
                        h[q] = zero ? 0u : *reinterpret_cast<uint32_t *>(&p);
                    }
                    uint4 *dst = reinterpret_cast<uint4 *>(c_row + col);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(acce_bar(acc));
            if (++acc == C::kAccStages) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    // ---- teardown ----------------------------------------------------------
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// Prologue: tile counts, prefix sum, group table, per-group TMA descriptors.

template <int CAP>
struct PrologueParams {
    alignas(64) uint8_t tmpl_a[128];
    alignas(64) uint8_t tmpl_b[128];
    WorkspaceView ws;
    int32_t group_count;
    int32_t block_n;
    GroupArgs groups[CAP];
};

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

template <int CAP>
__global__ void __launch_bounds__(CAP < 32 ? 32 : CAP)
    prologue_kernel(const __grid_constant__ PrologueParams<CAP> p) {
    // The GEMM kernel may start its set-up now; it waits for this grid's
    // completion before it reads anything written here.
    ptx::griddep_launch_dependents();
    __shared__ int32_t warp_sums[32];
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    const int G = p.group_count;

    int tiles = 0;
    if (tid < G) {
        const GroupArgs &a = p.groups[tid];
        if (a.m > 0 && a.n > 0)
            tiles = ceil_div_i(a.m, kBlockM) * ceil_div_i(a.n, p.block_n);
    }
    // block-wide inclusive scan of `tiles`
    int v = tiles;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off)
            v += y;
    }
    if (lane == 31)
        warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off)
                w += y;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const int inclusive = v + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (tid < G) {
        p.ws.prefix[tid] = inclusive - tiles;
        if (tid == G - 1)
            p.ws.prefix[G] = inclusive;
    }
    if (G == 0 && tid == 0)
        p.ws.prefix[0] = 0;

    if (tid < G) {
        const GroupArgs &a = p.groups[tid];
        GroupInfo gi;
        gi.m = a.m;
        gi.n = a.n;
        gi.k = a.k;
        gi.tiles_m = ceil_div_i(a.m > 0 ? a.m : 0, kBlockM);
        gi.k_tiles = ceil_div_i(a.k > 0 ? a.k : 0, kBlockK);
        gi.k_blocks = ceil_div_i(a.k > 0 ? a.k : 0, kMmaK);
        gi.sf_row_blocks_b = ceil_div_i(a.n > 0 ? a.n : 0, 128);
        gi.pad0 = 0;
        gi.sfa = static_cast<const uint8_t *>(a.sfa);
        gi.sfb = static_cast<const uint8_t *>(a.sfb);
        gi.c = a.c;
        gi.pad1 = 0;
        p.ws.groups[tid] = gi;
        if (a.m > 0 && a.n > 0 && a.k > 0) {
            uint8_t *ta = p.ws.tmaps + (size_t)tid * 256;
            uint8_t *tb = ta + 128;
            const uint4 *src_a = reinterpret_cast<const uint4 *>(p.tmpl_a);
            const uint4 *src_b = reinterpret_cast<const uint4 *>(p.tmpl_b);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                reinterpret_cast<uint4 *>(ta)[q] = src_a[q];
                reinterpret_cast<uint4 *>(tb)[q] = src_b[q];
            }
            const uint32_t row_bytes = (uint32_t)(a.k / 2);
            ptx::tmap_set_address(ta, a.a);
            ptx::tmap_set_dims(ta, row_bytes, (uint32_t)a.m);
            ptx::tmap_set_stride1(ta, row_bytes);
            ptx::tmap_set_address(tb, a.b);
            ptx::tmap_set_dims(tb, row_bytes, (uint32_t)a.n);
            ptx::tmap_set_stride1(tb, row_bytes);
            ptx::tmap_release();
        }
    }
}

template <int CAP>
cudaError_t launch_prologue(const GemmLaunch &cfg, const GroupArgs *groups, const WorkspaceView &ws,
                            const void *tmpl_a, const void *tmpl_b, cudaStream_t stream) {
    PrologueParams<CAP> p;
    std::memcpy(p.tmpl_a, tmpl_a, 128);
    std::memcpy(p.tmpl_b, tmpl_b, 128);
    p.ws = ws;
    p.group_count = cfg.group_count;
    p.block_n = cfg.block_n;
    std::memcpy(p.groups, groups, sizeof(GroupArgs) * (size_t)cfg.group_count);
    if (cfg.group_count < CAP)
        std::memset(p.groups + cfg.group_count, 0, sizeof(GroupArgs) * (size_t)(CAP - cfg.group_count));
    prologue_kernel<CAP><<<1, CAP < 32 ? 32 : CAP, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int BN>
cudaError_t launch_main(const GemmLaunch &cfg, const WorkspaceView &ws, cudaStream_t stream) {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)cfg.grid, 1, 1);
    lc.blockDim = dim3(Cfg<BN>::kThreads, 1, 1);
    lc.dynamicSmemBytes = Cfg<BN>::smem_bytes(ws.capacity);
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, grouped_gemm_kernel<BN>, ws, cfg.group_count, cfg.total_tiles, cfg.timeout_ns);
}

}  // namespace

size_t gemm_smem_bytes(int block_n) {
    return block_n == 256 ? Cfg<256>::smem_bytes(NVFP4_MAX_GROUPS) : Cfg<128>::smem_bytes(NVFP4_MAX_GROUPS);
}

cudaError_t prepare_gemm_kernels(int /*device*/) {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Cfg<128>::smem_bytes(NVFP4_MAX_GROUPS));
    if (e != cudaSuccess)
        return e;
    return cudaFuncSetAttribute(grouped_gemm_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Cfg<256>::smem_bytes(NVFP4_MAX_GROUPS));
}

cudaError_t launch_grouped(const GemmLaunch &cfg, const GroupArgs *groups, const WorkspaceView &ws,
                           const void *tmpl_a, const void *tmpl_b, cudaStream_t stream) {
    if (ws.capacity < cfg.group_count || ws.capacity > NVFP4_MAX_GROUPS)
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (cfg.group_count <= 8)
        e = launch_prologue<8>(cfg, groups, ws, tmpl_a, tmpl_b, stream);
    else if (cfg.group_count <= 64)
        e = launch_prologue<64>(cfg, groups, ws, tmpl_a, tmpl_b, stream);
    else
        e = launch_prologue<NVFP4_MAX_GROUPS>(cfg, groups, ws, tmpl_a, tmpl_b, stream);
    if (e != cudaSuccess)
        return e;
    return cfg.block_n == 256 ? launch_main<256>(cfg, ws, stream) : launch_main<128>(cfg, ws, stream);
}

}  // namespace nvfp4
