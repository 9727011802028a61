// internal.h -- structures shared by the host layer (api.cu, noalloc.cu) and
// the kernels (gemm.cu, pack_scales.cu).
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "nvfp4_grouped.h"

namespace nvfp4 {

// Tile shape of one CTA: BLOCK_M rows of C (one 128-lane MMA), BLOCK_N columns
// (a template parameter, 128 or 256), BLOCK_K = 256 fp4 elements = one
// 128-byte swizzle row of packed codes = four MMAs of K = 64.
constexpr int kBlockM = 128;
constexpr int kBlockK = 256;
constexpr int kMmaK = 64;
constexpr int kSfAtomBytes = 512;  // 128 rows x 4 scale blocks

// A group's arguments, passed to the GEMM kernel as a kernel parameter.
// l is the group's batch count: batch b of A starts l-major at row b*m of a
// [l*m][k/2] stack (likewise B, C and the per-batch scale-atom blocks).
// `patch` tells the kernel which of the group's descriptors (bit 0: A, bit 1:
// B, bit 2: SFB) must be rewritten; the others already hold this group's
// pointer and shape.
struct GroupArgs {
    int32_t m, n, k;
    uint16_t l, patch;
    const void *a, *b, *sfa, *sfb;
    void *c;
};
static_assert(sizeof(GroupArgs) == 56, "kernel parameter budget");
constexpr int kMaxBatch = 65535;  // largest l

// A call whose group table stays in device memory: the caller's arrays of
// group_count sizes and pointers, read by the kernel (nothing on the host).
struct DeviceTable {
    const nvfp4_problem_size *sizes;
    const void *const *a;
    const void *const *b;
    const void *const *sfa;
    const void *const *sfb;
    void *const *c;
};

// Group counts with a kernel instantiation (the parameter block holds
// GroupArgs[CAP]); calls use the smallest that fits.
constexpr int kSmallGroups = 8;
constexpr int kMediumGroups = 64;

__host__ __device__ constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr size_t kPartialSlotBytes = sizeof(float) * 128 * 256;
constexpr int kDescBytes = 128;
// Descriptor slots per group: A, B and the B scales (SFB).
constexpr int kDescPerGroup = 3;

// Per-CTA prefix-sum scratch in global memory, used when the group count is
// too large for the kernel's spare shared memory: [tiles prefix | units prefix].
__host__ __device__ constexpr size_t cta_prefix_bytes(int capacity) { return 2 * round_up(sizeof(int32_t) * (size_t)(capacity + 1), 128); }

// Device workspace, carved from one allocation at 128-byte aligned offsets.
//   header      128 B: status word (bit flags of bounded waits that gave up or
//               of rejected device-table groups) at byte 0; at byte 64 the
//               descriptor-publication counter (CTAs that have published their
//               patched descriptors in the running call), at 96 the count of
//               CTAs whose producer has passed the running call's descriptor
//               wait and read the epoch, at 100 the epoch of the last call.
//               The last CTA to get there resets both counters and advances
//               the epoch, so nothing on the host tracks them (calls replayed
//               from a CUDA graph included).
//   tmaps       TMA descriptors [regions][capacity][A, B, SFB], 128 B each. Region
//               0 serves eager host-table calls (its contents are cached on
//               the host); region 1, where present, serves calls whose
//               launch may run at another time or patches slots the host
//               cannot see: captured launches and device-table calls. Those
//               rewrite every slot they use on every run.
//   cta_prefix  [prefix_slots][cta_prefix_bytes(capacity)]  (capacity > 64 only)
//   flags       uint32 [partial_slots]   epoch of the partial tile a CTA published
//   partials    [partial_slots][128 x 256 fp32]  split-schedule partial tiles
struct WorkspaceView {
    uint32_t *status;
    uint32_t *desc_count;
    uint32_t *done;
    uint32_t *epoch;
    uint8_t *tmaps;
    int32_t *cta_prefix;
    uint32_t *flags;
    float *partials;
    int32_t capacity;
    int32_t prefix_slots;
    int32_t partial_slots;
    int32_t regions;
};

constexpr size_t workspace_bytes(int capacity, int prefix_slots = 0, int partial_slots = 0, int regions = 1) {
    return 128 + (size_t)kDescBytes * kDescPerGroup * (size_t)capacity * (size_t)regions +
           (capacity > kMediumGroups ? cta_prefix_bytes(capacity) * (size_t)prefix_slots : 0) +
           (partial_slots > 0 ? round_up(sizeof(uint32_t) * (size_t)partial_slots, 128) +
                                    kPartialSlotBytes * (size_t)partial_slots
                              : 0);
}

inline WorkspaceView workspace_view(void *base, int capacity, int prefix_slots = 0, int partial_slots = 0,
                                    int regions = 1) {
    uint8_t *p = static_cast<uint8_t *>(base);
    WorkspaceView v;
    v.status = reinterpret_cast<uint32_t *>(p);
    v.desc_count = reinterpret_cast<uint32_t *>(p + 64);
    v.done = reinterpret_cast<uint32_t *>(p + 96);
    v.epoch = reinterpret_cast<uint32_t *>(p + 100);
    p += 128;
    v.tmaps = p;
    p += (size_t)kDescBytes * kDescPerGroup * (size_t)capacity * (size_t)regions;
    v.cta_prefix = nullptr;
    v.prefix_slots = 0;
    if (capacity > kMediumGroups) {
        v.cta_prefix = reinterpret_cast<int32_t *>(p);
        v.prefix_slots = prefix_slots;
        p += cta_prefix_bytes(capacity) * (size_t)prefix_slots;
    }
    v.flags = nullptr;
    v.partials = nullptr;
    if (partial_slots > 0) {
        v.flags = reinterpret_cast<uint32_t *>(p);
        p += round_up(sizeof(uint32_t) * (size_t)partial_slots, 128);
        v.partials = reinterpret_cast<float *>(p);
    }
    v.capacity = capacity;
    v.partial_slots = partial_slots;
    v.regions = regions;
    return v;
}

// The same workspace with descriptor region 1 in place of region 0.
inline WorkspaceView second_region(WorkspaceView v) {
    v.tmaps += (size_t)kDescBytes * kDescPerGroup * (size_t)v.capacity;
    return v;
}

// Status bits written by the GEMM kernel when a bounded wait gives up.
constexpr uint32_t kStatusProducerTimeout = 1u;
constexpr uint32_t kStatusMmaTimeout = 2u;
constexpr uint32_t kStatusEpilogueTimeout = 4u;
constexpr uint32_t kStatusFlagTimeout = 8u;
constexpr uint32_t kStatusDescTimeout = 16u;
constexpr uint32_t kStatusBadGroup = 32u;  // a device-table group failed validation and was skipped
constexpr uint32_t kStatusTimeoutMask = 31u;

// Schedule of a call with T output tiles on P CTAs (the host applies it to
// host-table calls, the kernel to device-table calls; integer arithmetic, so
// both agree). Tiles [0, F) are whole tiles dealt round-robin; the schedule
// units of tiles [F, T) are cut into P equal contiguous ranges, one per CTA
// (stream-K: a tile may be split along K between consecutive CTAs). Returns
// F (T: no split range). Automatic choice: 0 (all split) when whole tiles
// would waste >= ~30% of the time in their last wave (ceil(T/P) >= 1.4 T/P),
// else T. Splitting costs an fp32 partial tile per piece through the SM's
// store port (about two fp16 epilogues), so the whole-waves-plus-split-rest
// form (F = P * floor(T/P)) is measured slower than whole tiles on every
// workload here and is only taken when forced.
// `forced`: -1 automatic, 0 no split, 1 all split, 2 whole waves + split rest.
__host__ __device__ inline int choose_split_tile(int T, int P, int forced) {
    const int full = T / P, rem = T - full * P;
    const long long waves = full + (rem ? 1 : 0);
    if (forced == 0 || T == 0)
        return T;
    if (forced == 1)
        return 0;
    if (forced == 2)
        return full * P;
    if (rem != 0 && 10ll * waves * P >= 14ll * T)
        return 0;
    return T;
}

// Launch configuration chosen by the host for one call.
struct GemmLaunch {
    int block_n;            // 128 or 256
    int group_count;
    int desc_maps;          // descriptors the kernel patches (bits set in GroupArgs::patch)
    int total_tiles;        // output tiles (host-table calls)
    int total_work;         // schedule units: sum over tiles of max(k-tiles, 1) (host-table calls)
    int grid;               // persistent CTAs (all resident: cooperative launch)
    int split;              // 1: tiles >= split_tile form a split range (see choose_split_tile);
                            // device-table calls: the `forced` argument of choose_split_tile
    int split_tile;         // first tile of the split range (host-table calls)
    int capacity;           // workspace descriptor capacity (groups)
    uint64_t timeout_ns;    // bound of every wait
    bool device_table;      // the group table is `dt` (device memory), not the host array
    int cluster;            // clusters of two CTAs (256 x 256 tiles, whole tiles only; grid = 2 x clusters):
                            // 0 none, 1 CTA pair with cta_group::2 MMAs, 2 multicast cluster
    bool pair_launch = false;  // cluster == 0: launch the CTAs as clusters of two all the same (placement
                               // only: the two CTAs of an SM pair take neighbouring tiles, which share
                               // a B panel; measured 1-2% faster on the ring-bound workloads)
    DeviceTable dt;
};

// Host launcher (gemm.cu). `tmpl_a` / `tmpl_b` / `tmpl_sfb` are 128-byte
// encoded TMA descriptors the kernel patches per group.
cudaError_t launch_grouped(const GemmLaunch &cfg, const GroupArgs *groups, const WorkspaceView &ws,
                           const void *tmpl_a, const void *tmpl_b, const void *tmpl_sfb, cudaStream_t stream);
cudaError_t prepare_gemm_kernels(int device);
// Clusters of two CTAs of the cluster kernels that are resident at once on
// the current device (0: the cluster kernels cannot run).
int pair_capacity(int device);

// Host layer (api.cu), shared by the entry points.
int fail(int status, const char *fmt, ...);
int cuda_fail(cudaError_t e, const char *what);
// Check one call's arguments (at most max_groups groups); fills args[0..G)
// and the tile count for a BLOCK_N of block_n.
int check_groups(int group_count, int max_groups, const nvfp4_problem_size *problem_sizes, const void *const *A,
                 const void *const *B, const void *const *SFA, const void *const *SFB, void *const *C, int block_n,
                 GroupArgs *args, long long *total_tiles);
int current_block_n();
// What one descriptor slot holds: base address, rows, k and the box height.
struct DescKey {
    const void *ptr = nullptr;
    int32_t rows = 0, k = 0, box = 0;
    bool operator==(const DescKey &o) const { return ptr == o.ptr && rows == o.rows && k == o.k && box == o.box; }
};
// Per-workspace host state of the calls that share it (in stream order).
struct WorkspaceState {
    std::vector<DescKey> descs;    // [group][A, B]: what each descriptor slot holds (empty: unknown)
};
// Set up the current device on first use and launch a checked call whose
// scratch is the workspace at ws_base. With partial_slots > 0 the call may use
// a split schedule.
int launch_on_workspace(int group_count, GroupArgs *args, long long total_tiles, int block_n, void *ws_base,
                        int capacity, int prefix_slots, int partial_slots, int regions, WorkspaceState *state,
                        cudaStream_t stream);
// Launch a device-table call on the workspace (every group's descriptors are
// patched by the kernel, in descriptor region 1).
int launch_device_table(int group_count, const DeviceTable &dt, int block_n, void *ws_base, int capacity,
                        int slots, WorkspaceState *state, cudaStream_t stream);

// The static scratch array of nvfp4_grouped_gemm_noalloc on `device` once a
// call has set it up there, else null (noalloc.cu).
void *noalloc_workspace_if_ready(int device);

// Quantise-and-pack launcher (quantize.cu).
cudaError_t launch_quantize_pack(const void *x, bool bf16, int rows, int k, void *codes, void *sf_atoms,
                                 cudaStream_t stream);

// Packer launcher (pack_scales.cu).
cudaError_t launch_pack_scales(const uint8_t *src, int rows, int k, uint8_t *dst, cudaStream_t stream);
// Matrices per nvfp4_pack_scales_batched launch (kernel parameter budget).
constexpr int kPackBatchMax = NVFP4_PACK_MAX_BATCH;
cudaError_t launch_pack_scales_batched(int count, const uint8_t *const *src, const int *rows, const int *k,
                                       uint8_t *const *dst, cudaStream_t stream);

}  // namespace nvfp4
