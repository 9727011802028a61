// gemm.cu -- the grouped NVFP4 block-scaled GEMM for sm_103a.
//
// Two kernels per call, in stream order:
//
//  1. prologue_kernel (one CTA): per-group output-tile counts and schedule-unit
//     counts with their exclusive prefix sums, a compact per-group table, and
//     per-group TMA descriptors for A and B patched from a host-encoded
//     template with tensormap.replace (the per-group descriptor patching of
//     "nvfp4 group gemm" submission 506336, TMA warp, and the one-off descriptor
//     initialisation kernel of submission 499344; here the tile prefix sum also
//     moves to the device). It triggers programmatic dependent launch at once so
//     the GEMM kernel's set-up overlaps it.
//
//  2. grouped_gemm_kernel<BN> (persistent, one CTA per SM, 320 threads):
//       warp 4    TMA producer: A and B tiles (128-byte swizzle) plus the scale
//                 runs of each 256-K k-tile (1-D bulk copies: a 128-row x 256-K
//                 slice of the reordered scale layout is 4 consecutive 512-byte
//                 atoms) into a multi-stage shared-memory ring;
//       warps 6-9 scale writers: each copies the stage's scale atoms into its
//                 own 32-lane quarter of TMEM with tcgen05.st (the layout the
//                 block-scaled MMA reads: lane l, column c of a k-block holds
//                 the 4 scales of row 32c + l, the same in every quarter);
//       warp 5    MMA issuer: tcgen05.mma kind::mxf4nvf4 block_scale
//                 (scale_vec::4X = one e4m3 scale per 16 elements),
//                 128 x BN x 64, four per k-tile, into a TMEM accumulator;
//                 commits free the smem stage and publish the accumulator;
//       warps 0-3 epilogue: tcgen05.ld of the accumulator lanes they own,
//                 fp32 -> fp16 round-to-nearest-even, 16-byte stores, rows
//                 >= m skipped, column chunks >= n skipped.
//
// Schedule. The work of a call is a sequence of schedule units: for every
// output tile (group-major, M fastest inside a group, so neighbouring units
// share a B panel) its k-tiles, at least one per tile (a k == 0 tile has one
// unit and produces zeros). Each CTA takes one contiguous range of units:
//   * whole-tile ranges (tiles split evenly over the CTAs) when there are many
//     tiles per SM;
//   * equal ranges of units (stream-K) when there are few: a tile may then be
//     split along K between consecutive CTAs. The CTA holding the tile's first
//     k-tile finishes it; every later piece is the first segment of its CTA,
//     so it is computed without waiting, stored as an fp32 partial tile in the
//     CTA's workspace slot and published with an epoch flag (release); the
//     finishing CTA acquires the flags, adds the partials and writes C.
//
// Every wait is bounded (%globaltimer): a wait that gives up sets a bit in
// the workspace status word and a CTA-wide abort flag, the other roles leave
// their loops, the producer waits (bounded) for the copies it issued, and the
// CTA frees its TMEM and exits.
#include <cuda_fp16.h>

#include <cstring>

#include "internal.h"
#include "ptx.cuh"

namespace nvfp4 {
namespace {

constexpr uint32_t kStatusFlagTimeout = 8u;

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
    static constexpr int kThreads = 320;                           // 10 warps
    static constexpr int kBarrierBytes = 256;
    static_assert((3 * kStages + 2 * kAccStages) * 8 <= 192, "barrier area");
    static constexpr uint32_t kIdesc = ptx::idesc_mxf4nvf4(kBlockM, BN);

    static size_t smem_bytes(int capacity) {
        return 1024 + (size_t)kStages * kStageBytes + kBarrierBytes +
               2 * round_up(sizeof(int32_t) * (capacity + 1), 16);
    }
};

// Index g with prefix[g] <= x < prefix[g + 1] (groups with no entries skipped).
__device__ __forceinline__ int find_group(const int32_t *prefix, int group_count, int x) {
    int lo = 0, hi = group_count;  // prefix[lo] <= x < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (prefix[mid] <= x)
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

// A run of one tile's k-tiles [kt0, kt1) (out of ktg schedule units) that one
// CTA processes.
struct Segment {
    int g, tm, tn;
    int kt0, kt1, ktg;
    int w_tile_end;  // schedule index one past the tile's last unit
};

__device__ __forceinline__ Segment segment_at(int w, int w_end, const int32_t *wprefix, int group_count,
                                              const GroupInfo *groups) {
    Segment s;
    s.g = find_group(wprefix, group_count, w);
    const int ktg = groups[s.g].work_tiles;
    const int local = w - wprefix[s.g];
    const int t = local / ktg;
    s.kt0 = local - t * ktg;
    const int rest = w_end - w;
    s.kt1 = s.kt0 + ((ktg - s.kt0) < rest ? (ktg - s.kt0) : rest);
    s.ktg = ktg;
    const int tiles_m = groups[s.g].tiles_m;
    s.tm = t % tiles_m;
    s.tn = t / tiles_m;
    s.w_tile_end = wprefix[s.g] + (t + 1) * ktg;
    return s;
}

// First schedule unit of CTA c out of p in a split (stream-K) schedule.
__device__ __forceinline__ int split_begin(int c, int p, int total_work) {
    return (int)(((long long)c * total_work) / p);
}

template <int BN>
__global__ void __launch_bounds__(320, 1)
    grouped_gemm_kernel(const WorkspaceView ws, const int group_count, const int total_tiles, const int total_work,
                        const int split, const uint32_t epoch, const uint64_t timeout_ns) {
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
    auto sff_bar = [&](int s) { return bars + 8u * (2 * C::kStages + s); };
    auto accf_bar = [&](int a) { return bars + 8u * (3 * C::kStages + a); };
    auto acce_bar = [&](int a) { return bars + 8u * (3 * C::kStages + C::kAccStages + a); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_area + 192);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 196);
    int *s_range = reinterpret_cast<int *>(bar_area + 200);           // [w_begin, w_end)
    volatile int *s_epi_ok = reinterpret_cast<volatile int *>(bar_area + 208);
    const size_t prefix_bytes = round_up(sizeof(int32_t) * (group_count + 1), 16);
    int32_t *s_prefix = reinterpret_cast<int32_t *>(bar_area + C::kBarrierBytes);
    int32_t *s_wprefix = reinterpret_cast<int32_t *>(bar_area + C::kBarrierBytes + prefix_bytes);

    // ---- set-up that does not depend on the prologue -----------------------
    if (warp == 4 && lane == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
            ptx::mbar_init(sff_bar(s), 4);
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

    // ---- wait for the prologue's prefix sums, group table and descriptors --
    ptx::griddep_wait();
    for (int i = threadIdx.x; i <= group_count; i += blockDim.x) {
        s_prefix[i] = ws.prefix[i];
        s_wprefix[i] = ws.wprefix[i];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const int c = blockIdx.x, p = gridDim.x;
        if (split) {
            s_range[0] = split_begin(c, p, total_work);
            s_range[1] = split_begin(c + 1, p, total_work);
        } else {
            // whole tiles: [c*T/p, (c+1)*T/p) mapped to schedule units
            for (int e = 0; e < 2; ++e) {
                const int t = (int)(((long long)(c + e) * total_tiles) / p);
                if (t >= total_tiles) {
                    s_range[e] = total_work;
                } else {
                    const int g = find_group(s_prefix, group_count, t);
                    s_range[e] = s_wprefix[g] + (t - s_prefix[g]) * ws.groups[g].work_tiles;
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int w_begin = s_range[0];
    const int w_end = s_range[1];

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
            for (int w = w_begin; ok && w < w_end;) {
                const Segment sg = segment_at(w, w_end, s_wprefix, group_count, ws.groups);
                w += sg.kt1 - sg.kt0;
                const GroupInfo &gi = ws.groups[sg.g];
                const int k_tiles = gi.k_tiles;
                const int kend = sg.kt1 < k_tiles ? sg.kt1 : k_tiles;
                if (sg.kt0 >= kend)
                    continue;  // k == 0 tile: nothing to load
                const int k_blocks = gi.k_blocks;
                const uint8_t *tmap_a = ws.tmaps + (size_t)sg.g * 256;
                const uint8_t *tmap_b = tmap_a + 128;
                if (sg.g != prev_g) {
                    ptx::tmap_acquire(tmap_a);
                    ptx::tmap_acquire(tmap_b);
                    prev_g = sg.g;
                }
                const uint8_t *sfa = gi.sfa + (size_t)sg.tm * k_blocks * kSfAtomBytes;
                int sfb_blocks = gi.sf_row_blocks_b - sg.tn * C::kSfbRowBlocks;
                sfb_blocks = sfb_blocks < C::kSfbRowBlocks ? sfb_blocks : C::kSfbRowBlocks;
                const uint8_t *sfb = gi.sfb + (size_t)sg.tn * C::kSfbRowBlocks * k_blocks * kSfAtomBytes;
                for (int kt = sg.kt0; kt < kend; ++kt) {
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
                    ptx::tma_load_2d(st, tmap_a, kt * 128, sg.tm * kBlockM, fb, pol_a);
                    ptx::tma_load_2d(st + C::kABytes, tmap_b, kt * 128, sg.tn * BN, fb, pol_b);
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
            for (int w = w_begin; ok && w < w_end;) {
                const Segment sg = segment_at(w, w_end, s_wprefix, group_count, ws.groups);
                w += sg.kt1 - sg.kt0;
                const int k_tiles = ws.groups[sg.g].k_tiles;
                const int k_blocks = ws.groups[sg.g].k_blocks;
                const int kend = sg.kt1 < k_tiles ? sg.kt1 : k_tiles;
                if (!wait_bounded(acce_bar(acc), acc_phase ^ 1u, abort_flag, timeout_ns, ws.status,
                                  kStatusMmaTimeout))
                    break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::kAccCols);
                for (int kt = sg.kt0; kt < kend; ++kt) {
                    if (!wait_bounded(full_bar(stage), phase, abort_flag, timeout_ns, ws.status,
                                      kStatusMmaTimeout) ||
                        !wait_bounded(sff_bar(stage), phase, abort_flag, timeout_ns, ws.status,
                                      kStatusMmaTimeout)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const int nkb = (k_blocks - 4 * kt) < 4 ? (k_blocks - 4 * kt) : 4;
                    const uint32_t st = smem_base + stage * C::kStageBytes;
                    const uint32_t sfa_t = tmem_base + (uint32_t)(C::kSfColBase + stage * C::kSfColsPerStage);
                    const uint32_t sfb_t = sfa_t + C::kSfaCols;
                    const uint64_t adesc = ptx::sdesc_kmajor_sw128(st);
                    const uint64_t bdesc = ptx::sdesc_kmajor_sw128(st + C::kABytes);
                    for (int kb = 0; kb < nkb; ++kb) {
                        // +32 bytes per 64-element k-block inside the swizzled row
                        ptx::tc_mma_mxf4nvf4(d_tmem, adesc + 2u * kb, bdesc + 2u * kb, C::kIdesc, sfa_t + 4 * kb,
                                             sfb_t + kb * (BN / 32), (kt != sg.kt0 || kb != 0) ? 1u : 0u);
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
    } else if (warp >= 6) {
        // ===================== scale writers (warps 6..9) =====================
        // Warp w owns TMEM lanes 32*(w % 4) .. +31 and writes the scale atoms
        // of every stage into that quarter.
        const uint32_t quarter = (uint32_t)((warp & 3) * 32) << 16;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int w = w_begin; ok && w < w_end;) {
            const Segment sg = segment_at(w, w_end, s_wprefix, group_count, ws.groups);
            w += sg.kt1 - sg.kt0;
            const int k_tiles = ws.groups[sg.g].k_tiles;
            const int k_blocks = ws.groups[sg.g].k_blocks;
            const int kend = sg.kt1 < k_tiles ? sg.kt1 : k_tiles;
            for (int kt = sg.kt0; kt < kend; ++kt) {
                int got = 0;
                if (lane == 0)
                    got = wait_bounded(full_bar(stage), phase, abort_flag, timeout_ns, ws.status, kStatusMmaTimeout)
                              ? 1
                              : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                (void)ptx::mbar_try_wait(full_bar(stage), phase);  // every lane acquires the landed stage
                const int nkb = (k_blocks - 4 * kt) < 4 ? (k_blocks - 4 * kt) : 4;
                const uint8_t *st_sfa = smem + stage * C::kStageBytes + C::kABytes + C::kBBytes;
                const uint8_t *st_sfb = st_sfa + C::kSfaBytes;
                const uint32_t sfa_t = tmem_base + quarter + (uint32_t)(C::kSfColBase + stage * C::kSfColsPerStage);
                const uint32_t sfb_t = sfa_t + C::kSfaCols;
                for (int kb = 0; kb < nkb; ++kb) {
                    ptx::tmem_st_32x32b_x4(sfa_t + 4 * kb,
                                           *reinterpret_cast<const uint4 *>(st_sfa + kb * kSfAtomBytes + 16 * lane));
#pragma unroll
                    for (int j = 0; j < C::kSfbRowBlocks; ++j)
                        ptx::tmem_st_32x32b_x4(sfb_t + kb * (BN / 32) + 4 * j,
                                               *reinterpret_cast<const uint4 *>(
                                                   st_sfb + (j * 4 + kb) * kSfAtomBytes + 16 * lane));
                }
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    ptx::mbar_arrive(sff_bar(stage));
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else {
        // ===================== epilogue (warps 0..3) =====================
        const int cta = blockIdx.x, ncta = gridDim.x;
        const int r_local = warp * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int w = w_begin; w < w_end;) {
            const Segment sg = segment_at(w, w_end, s_wprefix, group_count, ws.groups);
            w += sg.kt1 - sg.kt0;
            const GroupInfo &gi = ws.groups[sg.g];
            const int m = gi.m, n = gi.n;
            const bool zero = gi.k == 0;
            const bool cont = sg.kt0 > 0;                                       // a later piece of a split tile
            const bool finish_split = split && sg.kt0 == 0 && sg.kt1 < sg.ktg;  // first piece of a split tile
            // One thread waits (for the accumulator and, when finishing a split
            // tile, for the later pieces' flags); the four warps leave or stay
            // together: the TMEM loads below are warp-collective.
            if (threadIdx.x == 0) {
                int ok = wait_bounded(accf_bar(acc), acc_phase, abort_flag, timeout_ns, ws.status,
                                      kStatusEpilogueTimeout)
                             ? 1
                             : 0;
                if (ok && finish_split) {
                    for (int c2 = cta + 1; c2 < ncta && split_begin(c2, ncta, total_work) < sg.w_tile_end; ++c2) {
                        const uint64_t t0 = ptx::globaltimer();
                        while (ptx::ld_acquire_gpu(ws.flags + c2) != epoch) {
                            if (ptx::globaltimer() - t0 > timeout_ns) {
                                *abort_flag = 1;
                                atomicOr(ws.status, kStatusFlagTimeout);
                                ok = 0;
                                break;
                            }
                        }
                        if (!ok)
                            break;
                    }
                }
                *s_epi_ok = ok;
            }
            ptx::named_barrier(1, 128);
            if (!*s_epi_ok)
                break;
            ptx::tc_fence_after();
            const int row = sg.tm * kBlockM + r_local;
            const uint32_t t_row = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(acc * C::kAccCols);
            __half *c_row = static_cast<__half *>(gi.c) + (size_t)row * (size_t)n;
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; ++cc) {
                const int col = sg.tn * BN + cc * 32;
                if (col >= n)
                    break;
                uint32_t v[32];
                ptx::tmem_ld_32x32b_x32(t_row + cc * 32, v);
                ptx::tmem_ld_wait();
                if (row >= m)
                    continue;
                const size_t part_off = ((size_t)cc * kBlockM + r_local) * 32;
                if (cont) {
                    float4 *dst = reinterpret_cast<float4 *>(ws.partials + (size_t)cta * (kPartialSlotBytes / 4) +
                                                             part_off);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                             __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                    continue;
                }
                float f[32];
#pragma unroll
                for (int q = 0; q < 32; ++q)
                    f[q] = zero ? 0.0f : __uint_as_float(v[q]);
                if (finish_split) {
                    for (int c2 = cta + 1; c2 < ncta && split_begin(c2, ncta, total_work) < sg.w_tile_end; ++c2) {
                        const float4 *src = reinterpret_cast<const float4 *>(
                            ws.partials + (size_t)c2 * (kPartialSlotBytes / 4) + part_off);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 p4 = __ldcg(src + q);
                            f[4 * q] += p4.x;
                            f[4 * q + 1] += p4.y;
                            f[4 * q + 2] += p4.z;
                            f[4 * q + 3] += p4.w;
                        }
                    }
                }
                uint32_t h[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    __half2 p2 = __floats2half2_rn(f[2 * q], f[2 * q + 1]);
                    h[q] = *reinterpret_cast<uint32_t *>(&p2);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(c_row + col);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[q] = make_uint4(h[4 * q], h[4 * q + 1], h[4 * q + 2], h[4 * q + 3]);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                ptx::mbar_arrive(acce_bar(acc));
            if (cont) {
                // publish this CTA's partial tile
                ptx::named_barrier(1, 128);
                if (threadIdx.x == 0) {
                    __threadfence();
                    ptx::st_release_gpu(ws.flags + cta, epoch);
                }
            }
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
// Prologue: tile and schedule-unit counts, prefix sums, group table, per-group
// TMA descriptors.

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

// Exclusive prefix sum over the block (blockDim.x <= 1024); returns this
// thread's exclusive value and writes the block total to *total.
__device__ __forceinline__ int block_exclusive_scan(int x, int32_t *warp_sums, int *total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    int v = x;
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
        int s = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off)
                s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    const int inclusive = v + (warp > 0 ? warp_sums[warp - 1] : 0);
    *total = warp_sums[31];
    __syncthreads();
    return inclusive - x;
}

template <int CAP>
__global__ void __launch_bounds__(CAP < 32 ? 32 : CAP)
    prologue_kernel(const __grid_constant__ PrologueParams<CAP> p) {
    // The GEMM kernel may start its set-up now; it waits for this grid's
    // completion before it reads anything written here.
    ptx::griddep_launch_dependents();
    __shared__ int32_t warp_sums[32];
    const int tid = threadIdx.x;
    const int G = p.group_count;

    int tiles = 0, work = 0;
    if (tid < G) {
        const GroupArgs &a = p.groups[tid];
        if (a.m > 0 && a.n > 0) {
            tiles = ceil_div_i(a.m, kBlockM) * ceil_div_i(a.n, p.block_n);
            const int kt = ceil_div_i(a.k > 0 ? a.k : 0, kBlockK);
            work = tiles * (kt > 1 ? kt : 1);
        }
    }
    int total_tiles = 0, total_work = 0;
    const int t_ex = block_exclusive_scan(tiles, warp_sums, &total_tiles);
    const int w_ex = block_exclusive_scan(work, warp_sums, &total_work);
    if (tid < G) {
        p.ws.prefix[tid] = t_ex;
        p.ws.wprefix[tid] = w_ex;
    }
    if (tid == 0) {
        p.ws.prefix[G] = total_tiles;
        p.ws.wprefix[G] = total_work;
    }

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
        gi.work_tiles = gi.k_tiles > 1 ? gi.k_tiles : 1;
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
    return cudaLaunchKernelEx(&lc, grouped_gemm_kernel<BN>, ws, cfg.group_count, cfg.total_tiles, cfg.total_work,
                              cfg.split, cfg.epoch, cfg.timeout_ns);
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
    if (cfg.split && ws.partial_slots < cfg.grid)
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
