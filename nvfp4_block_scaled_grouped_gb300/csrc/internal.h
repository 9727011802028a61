// internal.h -- structures shared by the host layer (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

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

// One group as the prologue writes it for the GEMM kernel (64 bytes).
struct GroupInfo {
    int32_t m, n, k;
    int32_t tiles_m;          // ceil(m / BLOCK_M)
    int32_t k_tiles;          // ceil(k / BLOCK_K)
    int32_t k_blocks;         // ceil(k / 64): MMA k-blocks = scale atoms along K
    int32_t sf_row_blocks_b;  // ceil(n / 128): 128-row scale blocks that exist for B
    int32_t work_tiles;       // max(k_tiles, 1): schedule units per output tile
    const uint8_t *sfa;
    const uint8_t *sfb;
    void *c;
    uint64_t pad1;
};
static_assert(sizeof(GroupInfo) == 64, "GroupInfo layout");

// A group's raw arguments (host -> prologue, by kernel parameter).
struct GroupArgs {
    int32_t m, n, k, l;
    const void *a, *b, *sfa, *sfb;
    void *c;
};

// Device workspace, carved from one allocation at 128-byte aligned offsets.
//   status    uint32 (bit flags of bounded waits that gave up)
//   prefix    int32 [capacity + 1]  exclusive prefix sum of output tiles per group
//   wprefix   int32 [capacity + 1]  exclusive prefix sum of schedule units
//                                   (tiles x max(k-tiles, 1)) per group
//   groups    GroupInfo [capacity]
//   tmaps     128-byte TMA descriptors [capacity][2] (A, B)
//   flags     uint32 [slots]        epoch of the partial sum a CTA published
//   partials  fp32 [slots][BLOCK_M x 256]  split-K partial tiles, one slot per CTA
// The last two exist only when partial_slots > 0 (split schedules allowed).
struct WorkspaceView {
    uint32_t *status;
    int32_t *prefix;
    int32_t *wprefix;
    GroupInfo *groups;
    uint8_t *tmaps;
    uint32_t *flags;
    float *partials;
    int32_t capacity;
    int32_t partial_slots;
};

__host__ __device__ constexpr size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr size_t kPartialSlotBytes = sizeof(float) * 128 * 256;

constexpr size_t workspace_bytes(int capacity, int partial_slots = 0) {
    return 128 + 2 * round_up(sizeof(int32_t) * (size_t)(capacity + 1), 128) +
           round_up(sizeof(GroupInfo) * (size_t)capacity, 128) + 256 * (size_t)capacity +
           (partial_slots > 0 ? round_up(sizeof(uint32_t) * (size_t)partial_slots, 128) +
                                    kPartialSlotBytes * (size_t)partial_slots
                              : 0);
}

inline WorkspaceView workspace_view(void *base, int capacity, int partial_slots = 0) {
    uint8_t *p = static_cast<uint8_t *>(base);
    WorkspaceView v;
    v.status = reinterpret_cast<uint32_t *>(p);
    p += 128;
    v.prefix = reinterpret_cast<int32_t *>(p);
    p += round_up(sizeof(int32_t) * (size_t)(capacity + 1), 128);
    v.wprefix = reinterpret_cast<int32_t *>(p);
    p += round_up(sizeof(int32_t) * (size_t)(capacity + 1), 128);
    v.groups = reinterpret_cast<GroupInfo *>(p);
    p += round_up(sizeof(GroupInfo) * (size_t)capacity, 128);
    v.tmaps = p;
    p += 256 * (size_t)capacity;
    v.flags = nullptr;
    v.partials = nullptr;
    if (partial_slots > 0) {
        v.flags = reinterpret_cast<uint32_t *>(p);
        p += round_up(sizeof(uint32_t) * (size_t)partial_slots, 128);
        v.partials = reinterpret_cast<float *>(p);
    }
    v.capacity = capacity;
    v.partial_slots = partial_slots;
    return v;
}

// Status bits written by the GEMM kernel when a bounded wait gives up.
constexpr uint32_t kStatusProducerTimeout = 1u;
constexpr uint32_t kStatusMmaTimeout = 2u;
constexpr uint32_t kStatusEpilogueTimeout = 4u;

// Launch configuration chosen by the host for one call.
struct GemmLaunch {
    int block_n;          // 128 or 256
    int group_count;
    int total_tiles;      // output tiles
    int total_work;       // schedule units: sum over tiles of max(k-tiles, 1)
    int grid;             // persistent CTAs
    int split;            // 1: CTAs take equal ranges of schedule units (tiles may be split along K)
    uint32_t epoch;       // tag of this call's partial-sum flags (split schedules)
    uint64_t timeout_ns;  // bound of every wait
};

// Host launchers (gemm.cu). `tmpl_a` / `tmpl_b` are 128-byte encoded TMA
// descriptors used as templates by the prologue.
cudaError_t launch_grouped(const GemmLaunch &cfg, const GroupArgs *groups, const WorkspaceView &ws,
                           const void *tmpl_a, const void *tmpl_b, cudaStream_t stream);
cudaError_t prepare_gemm_kernels(int device);
size_t gemm_smem_bytes(int block_n);

// Host layer (api.cu), shared by the entry points.
int fail(int status, const char *fmt, ...);
int cuda_fail(cudaError_t e, const char *what);
// Check one call's arguments (at most max_groups groups); fills args[0..G)
// and the tile count for a BLOCK_N of block_n.
int check_groups(int group_count, int max_groups, const nvfp4_problem_size *problem_sizes, const void *const *A,
                 const void *const *B, const void *const *SFA, const void *const *SFB, void *const *C, int block_n,
                 GroupArgs *args, long long *total_tiles);
int current_block_n();
// Set up the current device on first use and launch a checked call whose
// scratch is the workspace at ws_base (capacity groups).
// With partial_slots > 0 and a non-null epoch counter the call may use a
// split schedule (the counter tags its partial-sum flags).
int launch_on_workspace(int group_count, const GroupArgs *args, long long total_tiles, int block_n, void *ws_base,
                        int capacity, int partial_slots, uint32_t *epoch, cudaStream_t stream);

// Packer launcher (pack_scales.cu).
cudaError_t launch_pack_scales(const uint8_t *src, int rows, int k, uint8_t *dst, cudaStream_t stream);

}  // namespace nvfp4
