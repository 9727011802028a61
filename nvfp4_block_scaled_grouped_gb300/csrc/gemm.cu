// gemm.cu -- the grouped NVFP4 block-scaled GEMM for sm_103a.
//
// One persistent kernel per call, grouped_gemm_kernel<BN, CAP, DEV> (one CTA
// per SM, 448 threads, cooperative launch so every CTA is resident). The group
// table (sizes, batch counts and pointers of up to CAP groups) arrives as a
// __grid_constant__ kernel parameter, or (DEV) stays in the caller's device
// arrays and is read, and checked, by the kernel. At start-up every CTA
//   * computes the per-group output-tile counts and schedule-unit counts and
//     their exclusive prefix sums (the tile prefix sum that the "nvfp4 group
//     gemm" submissions build on the host is built here), and from them the
//     schedule when the host could not choose it (DEV);
//   * patches the TMA descriptors of its share of the groups (group g by CTA
//     g mod gridDim) from a host-encoded template with tensormap.replace,
//     releases them and adds 1 to a publication counter; producers wait for
//     all CTAs before their first copy (the per-group descriptor patching of
//     submission 506336, TMA warp, and the descriptor initialisation kernel of
//     submission 499344, done inside the one launch). Once past that wait
//     and its first copies, each producer counts its CTA as done; the last
//     one resets the call counters for the next call.
// Set-up is split across warps: 4 initialises the barriers and patches
// descriptors, 5 allocates TMEM, 6 builds the prefix sums, 7 reads the call
// epoch; the producer starts as soon as 4, 6 and 7 are done.
// Roles:
//       warp 4    TMA producer: A and B tiles (128-byte swizzle) plus the scale
//                 runs of each 256-K k-tile (1-D bulk copies: a 128-row x 256-K
//                 slice of the reordered scale layout is 4 consecutive 512-byte
//                 atoms) into a multi-stage shared-memory ring; the scale runs
//                 are issued first and land on their own mbarrier; A panels
//                 (re-read per n-tile) are kept in L2 with evict-last, B
//                 panels only when the group has more than one m-tile;
//       warps 6-9 scale writers: each copies the stage's scale atoms into its
//                 own 32-lane quarter of TMEM with two wide tcgen05.st (the
//                 layout the block-scaled MMA reads: lane l, column c of a
//                 k-block holds the 4 scales of row 32c + l, the same in every
//                 quarter);
//       warp 5    MMA issuer: tcgen05.mma kind::mxf4nvf4 block_scale
//                 (scale_vec::4X = one e4m3 scale per 16 elements),
//                 128 x BN x 64, four per k-tile, into a TMEM accumulator;
//                 commits free the smem stage and publish the accumulator;
//       warps 0-3 and 10-13: epilogue of every segment but the CTA's last
//                 (two warps per TMEM lane quarter, each half of the column
//                 chunks): tcgen05.ld of the accumulator lanes they own,
//                 fp32 -> fp16 round-to-nearest-even; a whole tile is moved
//                 into registers first and the accumulator released to the
//                 next tile's MMAs before the stores, which a warp-shuffle
//                 transpose turns into 8 rows x 128 B per store instruction
//                 (whole lines: few write requests, which would otherwise
//                 hold up the next tile's copies); rows >= m and column
//                 chunks >= n skipped;
//       warps 0-7 epilogue of the CTA's last segment, once every role has
//                 left its loop (the last epilogue is on the critical path).
//
// Schedule. The work of a call is a sequence of schedule units: for every
// output tile (group-major, batch-major inside a group, then M fastest, so
// neighbouring units share a B panel) its k-tiles, at least one per tile (a
// k == 0 tile has one unit and produces zeros). CTAs take
//   * whole tiles round-robin (tile blockIdx.x, + gridDim.x, ...) when there
//     are many tiles per SM, so the CTAs running at one time work on
//     neighbouring tiles and share their A and B panels in L2;
//   * equal contiguous ranges of units (stream-K) when there are few: a tile
//     may then be split along K between consecutive CTAs. The CTA holding the
//     tile's first k-tile finishes it; every later piece is the first segment
//     of its CTA, so it is computed without waiting, stored as an fp32 partial
//     tile in the CTA's workspace slot and published with an epoch flag
//     (release); the finishing CTA's producer acquires the flags and copies
//     the next piece's partial tile into the ring as the final MMAs free it,
//     and the last epilogue adds it (any further pieces from L2).
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

constexpr int kPartialChunkBytes = 8 * kBlockM * 16;  // one 32-column chunk of an fp32 partial tile

// CLU: how CTAs cooperate on a tile.
//   0  one CTA per 128 x BN tile.
//   1  CTA pair: a cluster of two CTAs computes 256 x BN tiles with
//      cta_group::2 MMAs (M = 256) issued by the even CTA: each CTA stages its
//      own 128 rows of A and its half (BN / 2 rows) of B, and holds its 128
//      rows of the accumulator.
//   2  multicast cluster: a cluster of two CTAs computes the two 128 x BN
//      tiles of a 256 x BN block, each with its own cta_group::1 MMAs; the
//      B tile and its scales, which both need, are fetched once per cluster
//      by TMA multicast into both CTAs (B by the even CTA, the B scales by the
//      odd one), so each CTA issues three copies per k-tile instead of four.
template <int BN, int CAP, int CLU = 0>
struct Cfg {
    static_assert(BN == 128 || BN == 256, "BLOCK_N");
    static_assert(CLU >= 0 && CLU <= 2, "cluster mode");
    static_assert(CLU == 0 || BN == 256, "clusters use 256-column tiles");
    static constexpr bool kCluster = CLU != 0;
    static constexpr bool kPairMma = CLU == 1;
    static constexpr bool kMcast = CLU == 2;
    static constexpr int kTileM = kCluster ? 2 * kBlockM : kBlockM;  // rows of C per schedule tile
    static constexpr int kBRows = kPairMma ? BN / 2 : BN;            // rows of B in this CTA's stage
    static constexpr int kStages = kPairMma ? 5 : ((BN == 128) ? 6 : 4);
    static constexpr int kAccStages = (BN == 128) ? 2 : 1;
    static constexpr int kABytes = kBlockM * 128;                  // 128 rows x 256 fp4
    static constexpr int kBBytes = kBRows * 128;                   // kBRows rows x 256 fp4
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
    // 14 warps: 0-3 and 10-13 epilogue, 4 producer, 5 MMA, 6-9 scale writers
    static constexpr int kThreads = 448;
    static constexpr int kMaxLoopChunks = BN / 64;  // column chunks per epilogue warp in the loop
    // barrier area: full / empty / scales-written per stage and the
    // accumulator barriers from 0, scratch from 176, scales-landed per stage
    // from 384, the epilogue warps' schedule cursor (64 bytes), two segment
    // slots (2 x 32) and three flags from 448
    static constexpr int kBarrierBytes = 640;
    static constexpr int kEpiCursorOffset = 448;
    static_assert((3 * kStages + 2 * kAccStages) * 8 <= 176 && kStages <= 8, "barrier area");
    // A finishing CTA receives the next piece's partial tile in ring stages,
    // kPartialChunksPerStage 16 KiB chunks (32 columns x 128 rows fp32) per
    // stage from offset 0.
    static constexpr int kPartialChunksPerStage = kStageBytes / kPartialChunkBytes;
    static_assert(kStages >= 4 && kPartialChunksPerStage * kStages >= BN / 32, "partial tile in the ring");
    // Prefix sums live in shared memory for up to kMediumGroups groups, else
    // in the CTA's global scratch slot.
    static constexpr bool kSmemPrefix = CAP <= kMediumGroups;
    static constexpr int kPrefixInts = (int)round_up(CAP + 1, 4);
    static constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kBarrierBytes +
                                         (kSmemPrefix ? 2 * sizeof(int32_t) * kPrefixInts : 0);
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static constexpr uint32_t kIdesc = ptx::idesc_mxf4nvf4(kPairMma ? 2 * kBlockM : kBlockM, BN);
    static constexpr int kCtaGroup = kPairMma ? 2 : 1;
};

// DEV: the group table is the caller's device arrays (`dt`), else `groups`.
template <int CAP, bool DEV>
struct GemmParams {
    alignas(64) uint8_t tmpl_a[128];
    alignas(64) uint8_t tmpl_b[128];
    alignas(64) uint8_t tmpl_sfb[128];
    WorkspaceView ws;
    DeviceTable dt;
    int32_t group_count, block_n, total_tiles, total_work, split, split_tile, desc_maps;
    uint64_t timeout_ns;
    GroupArgs groups[DEV ? 1 : CAP];
};

__device__ __forceinline__ bool aligned16(const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

// Largest m, n or k, and l*m or l*n, of a device-table group (keeps every
// tile and unit count of a call inside int32).
constexpr int kDeviceTableMaxDim = 1 << 24;
constexpr long long kDeviceTableMaxRows = 1ll << 30;

// Group g's arguments: the kernel parameter's entry, or the caller's device
// arrays checked against the same rules as the host entry point; a group that
// breaks one is skipped (sizes read as 0) and *bad is set.
template <int CAP, bool DEV>
__device__ __forceinline__ GroupArgs load_group(const GemmParams<CAP, DEV> &p, int g, bool *bad = nullptr) {
    if constexpr (!DEV) {
        return p.groups[g];
    } else {
        const int4 sz = __ldg(reinterpret_cast<const int4 *>(p.dt.sizes) + g);
        GroupArgs a;
        a.m = sz.x;
        a.n = sz.y;
        a.k = sz.z;
        a.l = (uint16_t)(sz.w >= 0 && sz.w <= kMaxBatch ? sz.w : 0);
        a.patch = 7;
        a.a = p.dt.a[g];
        a.b = p.dt.b[g];
        a.sfa = p.dt.sfa[g];
        a.sfb = p.dt.sfb[g];
        a.c = p.dt.c[g];
        bool ok = a.m >= 0 && a.n >= 0 && a.k >= 0 && sz.w >= 0 && a.m <= kDeviceTableMaxDim &&
                  a.n <= kDeviceTableMaxDim && a.k <= kDeviceTableMaxDim && sz.w <= kMaxBatch;
        if (ok && a.m > 0 && a.n > 0 && sz.w > 0) {
            ok = (long long)sz.w * a.m <= kDeviceTableMaxRows && (long long)sz.w * a.n <= kDeviceTableMaxRows &&
                 a.k % 32 == 0 && a.n % 32 == 0 && a.c && aligned16(a.c);
            if (ok && a.k > 0)
                ok = a.a && a.b && a.sfa && a.sfb && aligned16(a.a) && aligned16(a.b) && aligned16(a.sfa) &&
                     aligned16(a.sfb);
        }
        if (!ok) {
            if (bad)
                *bad = true;
            a.m = a.n = a.k = 0;
        }
        return a;
    }
}

__device__ __forceinline__ int ceil_div_i(int a, int b) { return (a + b - 1) / b; }

// Derived sizes of one group (m, n, k >= 0).
struct GInfo {
    int m, n, k, l;
    int tiles_m, tiles_mn;    // ceil(m / TM), ceil(m / TM) * ceil(n / BN) (0 for an empty group), TM the
                              // schedule tile's rows (128, or 256 for CTA pairs)
    int sf_row_blocks_a;      // ceil(m / 128): 128-row scale blocks of A
    int tiles;                // tiles_mn * l
    int k_tiles, k_blocks;    // ceil(k / 256), ceil(k / 64)
    int work_tiles;           // max(k_tiles, 1): schedule units per output tile
    int sf_row_blocks_b;      // ceil(n / 128): 128-row scale blocks of B
    size_t sfa_batch, sfb_batch;  // bytes of one batch's scale atoms
    const uint8_t *sfa, *sfb;
    void *c;
};

// CLUSTER: schedule tiles of 256 rows (clusters of two CTAs).
template <int BN, bool CLUSTER = false>
__device__ __forceinline__ GInfo group_info(const GroupArgs &a) {
    GInfo g;
    g.m = a.m;
    g.n = a.n;
    g.k = a.k;
    g.l = a.l;
    g.tiles_m = ceil_div_i(a.m, CLUSTER ? 2 * kBlockM : kBlockM);
    g.sf_row_blocks_a = ceil_div_i(a.m, kBlockM);
    g.tiles_mn = (a.m > 0 && a.n > 0) ? g.tiles_m * ceil_div_i(a.n, BN) : 0;
    g.tiles = g.tiles_mn * (int)a.l;
    g.k_tiles = ceil_div_i(a.k, kBlockK);
    g.k_blocks = ceil_div_i(a.k, kMmaK);
    g.work_tiles = g.k_tiles > 1 ? g.k_tiles : 1;
    g.sf_row_blocks_b = ceil_div_i(a.n, 128);
    g.sfa_batch = (size_t)g.sf_row_blocks_a * g.k_blocks * kSfAtomBytes;
    g.sfb_batch = (size_t)g.sf_row_blocks_b * g.k_blocks * kSfAtomBytes;
    g.sfa = static_cast<const uint8_t *>(a.sfa);
    g.sfb = static_cast<const uint8_t *>(a.sfb);
    g.c = a.c;
    return g;
}

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

// CL: acquire at cluster scope (barriers that threads of the other CTA of a
// pair arrive on). spin: poll without suspending the thread (barriers that
// the other CTA completes, whose completion may not wake a suspended
// waiter at once). On giving up, `peer_abort` (a shared::cluster address, 0
// for none) is the other CTA's abort flag, set too so that both CTAs of a
// pair leave their loops.
template <bool CL = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             uint64_t timeout_ns, uint32_t *status, uint32_t bit,
                                             uint32_t peer_abort = 0, bool spin = false) {
    // Each attempt suspends the thread for at most the bound (capped at
    // 1 ms), and the bound is checked after every failed one.
    const uint32_t hint = timeout_ns < 1000000ull ? (uint32_t)timeout_ns : 1000000u;
    auto attempt = [&]() {
        if (spin)
            return ptx::mbar_test_wait<CL>(bar, parity);
        return CL ? ptx::mbar_try_wait_hint_cluster(bar, parity, hint) : ptx::mbar_try_wait_hint(bar, parity, hint);
    };
    if (attempt())
        return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (attempt())
            return true;
        if (*abort_flag)
            return false;
        if (ptx::globaltimer() - t0 > timeout_ns) {
            *abort_flag = 1;
            if (peer_abort)
                ptx::st_cluster_u32(peer_abort, 1u);
            atomicOr(status, bit);
            return false;
        }
    }
}

// Wait until the global counter reaches `target` (modulo 2^32), acquire.
__device__ __forceinline__ bool wait_counter(const uint32_t *counter, uint32_t target, volatile int *abort_flag,
                                             uint64_t timeout_ns, uint32_t *status) {
    const uint64_t t0 = ptx::globaltimer();
    while ((int32_t)(ptx::ld_acquire_gpu(counter) - target) < 0) {
        if (*abort_flag)
            return false;
        if (ptx::globaltimer() - t0 > timeout_ns) {
            *abort_flag = 1;
            atomicOr(status, kStatusDescTimeout);
            return false;
        }
    }
    return true;
}

// A run of one tile's k-tiles [kt0, kt1) (out of ktg schedule units) that one
// CTA processes.
struct Segment {
    int g, b, tm, tn;  // group, batch, m-tile, n-tile
    int kt0, kt1, ktg;
    int w_tile_end;  // schedule index one past the tile's last unit
};

// First schedule unit of CTA c out of p in a split (stream-K) schedule
// (0 <= c <= p); 32-bit arithmetic whenever c * total_work fits.
__device__ __forceinline__ int split_begin(int c, int p, int total_work) {
    if ((unsigned)total_work <= 0xffffffffu / (unsigned)p)
        return (int)(((unsigned)c * (unsigned)total_work) / (unsigned)p);
    return (int)(((long long)c * total_work) / p);
}

// The sequence of segments one CTA processes; every role walks the same one:
// first the head of its split range when that range starts inside a tile (a
// later piece of a split tile, computed before anything else so its partial
// tile is published early), then its whole tiles (blockIdx, + P, ... below
// the first split tile), then the rest of its split range (ending, when the
// range ends inside a tile, with that tile's first piece, which this CTA
// finishes as its last segment).
template <int BN, int CAP, bool DEV, bool CLUSTER = false>
struct Cursor {
    // (the kernel parameters are passed to next() by reference rather than
    // kept here: through a stored pointer they would be read with generic
    // loads instead of from the constant bank, about 1 us per segment)
    const int32_t *prefix, *wprefix;
    int group_count;
    int tile, tile_end, step;  // whole tiles
    int w, w_end;              // split range [w, w_end) of schedule units
    int phase;                 // 0: head, 1: whole tiles, 2: rest of the split range
    int rank;                  // clusters: this CTA's rank in its cluster (segments carry its own 128-row m-tile)

    __device__ __forceinline__ void split_segment(const GemmParams<CAP, DEV> &p, Segment &s, const int limit) {
        s.g = find_group(wprefix, group_count, w);
        const GInfo gi = group_info<BN, CLUSTER>(load_group(p, s.g));
        const int local = w - wprefix[s.g];
        const int t = local / gi.work_tiles;
        s.ktg = gi.work_tiles;
        s.kt0 = local - t * gi.work_tiles;
        const int rest = limit - w;
        s.kt1 = s.kt0 + ((s.ktg - s.kt0) < rest ? (s.ktg - s.kt0) : rest);
        s.b = t / gi.tiles_mn;
        const int tb = t - s.b * gi.tiles_mn;
        s.tm = CLUSTER ? 2 * (tb % gi.tiles_m) + rank : tb % gi.tiles_m;
        s.tn = tb / gi.tiles_m;
        s.w_tile_end = wprefix[s.g] + (t + 1) * s.ktg;
        w += s.kt1 - s.kt0;
    }

    // Whether next() would return another segment.
    __device__ __forceinline__ bool more() const { return tile < tile_end || w < w_end; }

    __device__ __forceinline__ bool next(const GemmParams<CAP, DEV> &p, Segment &s) {
        if (phase == 0) {
            phase = 1;
            if (w < w_end) {
                // the range's first segment is the head when it is a later
                // piece of a tile (its first unit is not a tile's first
                // k-tile); otherwise it waits for phase 2. Only the group and
                // its k-tile count are needed to tell, not the whole segment,
                // which lies on the path to the first copy.
                const int g = find_group(wprefix, group_count, w);
                const int kt = ceil_div_i(load_group(p, g).k, kBlockK);
                if ((w - wprefix[g]) % (kt > 1 ? kt : 1) != 0) {
                    split_segment(p, s, w_end);
                    return true;
                }
            }
        }
        if (phase == 1) {
            if (tile < tile_end) {
                s.g = find_group(prefix, group_count, tile);
                const GInfo gi = group_info<BN, CLUSTER>(load_group(p, s.g));
                const int t = tile - prefix[s.g];
                s.b = t / gi.tiles_mn;
                const int tb = t - s.b * gi.tiles_mn;
                s.tm = CLUSTER ? 2 * (tb % gi.tiles_m) + rank : tb % gi.tiles_m;
                s.tn = tb / gi.tiles_m;
                s.ktg = gi.work_tiles;
                s.kt0 = 0;
                s.kt1 = s.ktg;
                s.w_tile_end = wprefix[s.g] + (t + 1) * s.ktg;
                tile += step;
                return true;
            }
            phase = 2;
        }
        if (w < w_end) {
            split_segment(p, s, w_end);
            return true;
        }
        return false;
    }
};

// Schedule unit index of the first unit of tile `tile` (total_work for
// tile == total_tiles).
template <int BN, int CAP, bool DEV>
__device__ __forceinline__ int tile_first_unit(const GemmParams<CAP, DEV> &p, const int32_t *prefix,
                                               const int32_t *wprefix, int group_count, int tile, int total_tiles,
                                               int total_work) {
    if (tile >= total_tiles)
        return total_work;
    const int g = find_group(prefix, group_count, tile);
    return wprefix[g] + (tile - prefix[g]) * group_info<BN>(load_group(p, g)).work_tiles;
}

// What the epilogue does with a segment's accumulator.
enum : int {
    kEpiWhole = 0,   // whole tile: fp16 to C
    kEpiCont = 1,    // later piece of a split tile: fp32 partial tile to this CTA's workspace slot
    kEpiFinish = 2,  // first piece of a split tile: add the later pieces' partial tiles, fp16 to C
};

// Hand-over of a CTA's last segment, which is finished after every role has
// left its loop by the epilogue warps together with warps 4..7.
struct TailState {
    Segment seg;
    int32_t valid, acc, acc_phase;
    int32_t part_state;   // 1: the producer issued the next piece's partial-tile copies on partial_bar
    int32_t part_ok;      // ... and every one of them
    int32_t part_stage0;  // ring stage of the first partial chunk
    int32_t pieces;       // later pieces of the finishing tile (CTAs blockIdx + 1 ..)
};

// Column chunks (32 columns) of a tile that hold columns < n.
template <int BN>
__device__ __forceinline__ int tile_chunks(const GInfo &gi, const Segment &sg) {
    const int c = (gi.n - sg.tn * BN) / 32;
    return c < BN / 32 ? c : BN / 32;
}

// One warp's share of a segment's epilogue: accumulator lanes 32 * quarter ..
// +31 (tile rows), column chunks [c0, c1) (at most kMaxLoopChunks). TMEM loads
// run half a chunk (16 columns) ahead of the arithmetic. `smem` is the CTA's
// ring (holding the next piece's partial tile from stage part_stage0 when
// finishing a split tile). A whole tile is moved from TMEM into registers
// first; with `release_bar` (the main loop) the warp then arrives on it, so
// the next tile's MMAs may start, before the stores. CTA pairs
// (CLU 1): `release_bar` is the shared::cluster address of the
// accumulator-empty barrier of the pair's even CTA. In clusters, a CTA whose
// 128 rows all lie past m (its half of a 256-row tile over a short group)
// only releases.
template <int BN, int CAP, bool DEV, int CLU = 0>
__device__ __forceinline__ void epilogue_warp(const GemmParams<CAP, DEV> &p, const Segment &sg, const GInfo &gi,
                                              const int kind, const int quarter, const int lane,
                                              const uint32_t t_acc, const int c0, const int c1,
                                              const uint8_t *smem, const int part_stage0, const int pieces,
                                              const uint32_t release_bar = 0) {
    using C = Cfg<BN, CAP, CLU>;
    auto release = [&]() {
        if constexpr (CLU == 1)
            ptx::mbar_arrive_cluster(release_bar);
        else
            ptx::mbar_arrive(release_bar);
    };
    if (c0 >= c1 || sg.tm * kBlockM >= gi.m) {
        // no chunks for this warp (a narrow tile, or no rows), but its release
        // still counts
        if (release_bar != 0) {
            __syncwarp();
            if (lane == 0)
                release();
        }
        return;
    }
    const int m = gi.m, n = gi.n;
    const int cta = blockIdx.x;
    const int r_local = quarter * 32 + lane;
    const int row = sg.tm * kBlockM + r_local;
    const uint32_t t_row = t_acc + ((uint32_t)(quarter * 32) << 16);
    __half *c_base = static_cast<__half *>(gi.c) + (size_t)sg.b * (size_t)m * (size_t)n;
    // Two chunks of fp16 row segments held in registers (chunks c0 + 2cp and
    // c0 + 2cp + 1 in h2[0], h2[1]; lane = row) go out as whole 128-byte
    // lines: for each group q of 8 rows, lane 4x + p gathers by shuffles the
    // 32-byte part p of row 8q + x (four rounds, one per part, in which the
    // eight lanes of the row group send that part), so each store instruction
    // writes 8 rows x 128 B -- a quarter of the write requests of one 16-byte
    // piece per row, which is what the next tile's operand copies compete
    // with. (The q loop stays rolled: unrolled, it costs tens of KB of code
    // per kernel, which every call fetches cold.)
    auto store_pair = [&](const int cp, const uint32_t (&h2)[2][16]) {
        const int x = lane >> 2, part = lane & 3;
        const bool wide = (reinterpret_cast<uintptr_t>(c_base) & 31u) == 0;
        const int cc = c0 + 2 * cp + (part >> 1);
        const int col = sg.tn * BN + cc * 32 + 16 * (part & 1);
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
            uint32_t o[8];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t got = __shfl_sync(0xffffffffu, h2[r >> 1][8 * (r & 1) + j], 8 * q + x);
                    if (r == 0 || part == r)
                        o[j] = got;
                }
            }
            const int grow = sg.tm * kBlockM + quarter * 32 + 8 * q + x;
            if (grow < m && cc < c1) {
                __half *dst = c_base + (size_t)grow * (size_t)n + col;
                if (wide) {
                    ptx::st_global_v8(dst, o);
                } else {
                    reinterpret_cast<uint4 *>(dst)[0] = make_uint4(o[0], o[1], o[2], o[3]);
                    reinterpret_cast<uint4 *>(dst)[1] = make_uint4(o[4], o[5], o[6], o[7]);
                }
            }
        }
    };
    auto pack = [](float x0, float x1) {
        __half2 h2 = __floats2half2_rn(x0, x1);
        return *reinterpret_cast<uint32_t *>(&h2);
    };
    // Partial tiles: [chunk][quad q][row] of float4, so a warp's stores and
    // loads of one (chunk, q) cover 512 contiguous bytes.
    uint32_t va[16], vb[16];
    if (kind != kEpiWhole)
        ptx::tmem_ld_32x32b_x16(t_row + c0 * 32, va);
    if (kind == kEpiCont) {
        float4 *dst = reinterpret_cast<float4 *>(p.ws.partials) + (size_t)cta * (kPartialSlotBytes / 16) + r_local;
        auto put = [&](const uint32_t (&v)[16], float4 *d) {
            if (row < m) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    d[q * kBlockM] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
        };
#pragma unroll 1
        for (int cc = c0; cc < c1; ++cc) {
            ptx::tmem_ld_wait();
            ptx::tmem_ld_32x32b_x16(t_row + cc * 32 + 16, vb);
            put(va, dst + (size_t)cc * 8 * kBlockM);
            ptx::tmem_ld_wait();
            if (cc + 1 < c1)
                ptx::tmem_ld_32x32b_x16(t_row + (cc + 1) * 32, va);
            put(vb, dst + ((size_t)cc * 8 + 4) * kBlockM);
        }
    } else if (kind == kEpiFinish) {
        // the first piece of a split tile (always the CTA's last segment):
        // plus the next piece's partial from the ring, and any further ones
        // (a tile spanning 3+ CTAs) from L2
        const float4 *gpart = reinterpret_cast<const float4 *>(p.ws.partials) + r_local;
        auto add_half = [&](const uint32_t (&v)[16], const int cc, const int q0, uint32_t *h) {
            const float4 *sp =
                reinterpret_cast<const float4 *>(
                    smem + ((part_stage0 + cc / C::kPartialChunksPerStage) % C::kStages) * C::kStageBytes +
                    (cc % C::kPartialChunksPerStage) * kPartialChunkBytes) +
                r_local;
            // (rows >= m hold no partial values; their sums are never stored)
            float4 a[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                a[q] = sp[(q0 + q) * kBlockM];
            for (int c2 = cta + 2; c2 <= cta + pieces; ++c2) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 b =
                        __ldcg(gpart + (size_t)c2 * (kPartialSlotBytes / 16) + ((size_t)cc * 8 + q0 + q) * kBlockM);
                    a[q].x += b.x;
                    a[q].y += b.y;
                    a[q].z += b.z;
                    a[q].w += b.w;
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                h[2 * q] = pack(__uint_as_float(v[4 * q]) + a[q].x, __uint_as_float(v[4 * q + 1]) + a[q].y);
                h[2 * q + 1] = pack(__uint_as_float(v[4 * q + 2]) + a[q].z, __uint_as_float(v[4 * q + 3]) + a[q].w);
            }
        };
#pragma unroll 1
        for (int cp = 0; c0 + 2 * cp < c1; ++cp) {
            uint32_t h2[2][16];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int cc = c0 + 2 * cp + i;
                if (cc < c1) {
                    ptx::tmem_ld_wait();
                    ptx::tmem_ld_32x32b_x16(t_row + cc * 32 + 16, vb);
                    add_half(va, cc, 0, h2[i]);
                    ptx::tmem_ld_wait();
                    if (cc + 1 < c1)
                        ptx::tmem_ld_32x32b_x16(t_row + (cc + 1) * 32, va);
                    add_half(vb, cc, 4, h2[i] + 8);
                }
            }
            store_pair(cp, h2);
        }
    } else {
        // whole tile: every chunk into registers; in the main loop the
        // accumulator is then released to the next tile's MMAs before the
        // stores. The pairs of chunks go out through one store_pair (the
        // second pair moved down after the first is stored): a last segment
        // runs this code once per call from a cold instruction cache.
        const bool zero = gi.k == 0;
        uint32_t hs[C::kMaxLoopChunks][16];
        // one 32-column load per chunk: the drain is a chain of TMEM load
        // round trips, which gate the release of the accumulator
#pragma unroll
        for (int i = 0; i < C::kMaxLoopChunks; ++i) {
            const int cc = c0 + i;
            if (cc < c1) {
                uint32_t v[32];
                ptx::tmem_ld_32x32b_x32(t_row + cc * 32, v);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    hs[i][q] = zero ? 0u : pack(__uint_as_float(v[2 * q]), __uint_as_float(v[2 * q + 1]));
            }
        }
        if (release_bar != 0) {
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0)
                release();
        }
#pragma unroll 1
        for (int cp = 0; cp < C::kMaxLoopChunks / 2 && c0 + 2 * cp < c1; ++cp) {
            store_pair(cp, reinterpret_cast<const uint32_t(&)[2][16]>(hs[0]));
#pragma unroll
            for (int i = 0; i + 2 < C::kMaxLoopChunks; ++i)
#pragma unroll
                for (int w = 0; w < 16; ++w)
                    hs[i][w] = hs[i + 2][w];
        }
    }
}

template <int BN, int CAP, bool DEV, int CLU>
__global__ void __launch_bounds__(448, 1) grouped_gemm_kernel(const __grid_constant__ GemmParams<CAP, DEV> p) {
    using C = Cfg<BN, CAP, CLU>;
    constexpr bool CLUSTER = C::kCluster;  // clusters of two CTAs (either mode)
    constexpr bool PAIR = C::kPairMma;     // CTA pair with cta_group::2 MMAs
    constexpr bool MCAST = C::kMcast;      // multicast cluster
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t smem_base = ptx::smem_addr(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int group_count = p.group_count;
    // Clusters of two: this CTA's rank in its cluster; the schedule deals
    // tiles to clusters (slot = cluster index), and both CTAs of a cluster walk
    // the same 256-row tiles, each its own 128 rows
    const uint32_t rank = CLUSTER ? ptx::cluster_ctarank() : 0u;
    const int slot = CLUSTER ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int nslots = CLUSTER ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    // descriptors are patched in this call (host table: only those that changed)
    const bool publish = DEV || p.desc_maps != 0;
    // Tag of this call's partial-tile flags: one more than the last completed
    // call's on this workspace (never 0, the value of a fresh flag).
    auto call_epoch = [&]() {
        const uint32_t e = *reinterpret_cast<const volatile uint32_t *>(p.ws.epoch) + 1u;
        return e ? e : 1u;
    };

    uint8_t *bar_area = smem + C::kStages * C::kStageBytes;
    const uint32_t bars = ptx::smem_addr(bar_area);
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (C::kStages + s); };
    auto sff_bar = [&](int s) { return bars + 8u * (2 * C::kStages + s); };
    auto sfl_bar = [&](int s) { return bars + 384u + 8u * s; };  // the stage's scale atoms landed
    auto accf_bar = [&](int a) { return bars + 8u * (3 * C::kStages + a); };
    auto acce_bar = [&](int a) { return bars + 8u * (3 * C::kStages + C::kAccStages + a); };
    // CTA pairs, even CTA: the odd CTA's stage s is ready (A / B landed, its
    // scales written to its TMEM)
    // where the epilogue releases accumulator a: the even CTA's barrier in a pair
    auto acce_release = [&](int a) { return PAIR ? ptx::mapa(acce_bar(a), 0u) : acce_bar(a); };
    const uint32_t drain_bar = bars + 176;    // the MMA thread's issued MMAs have completed
    const uint32_t partial_bar = bars + 184;  // partial tile of a split tile landed in smem
    // Bound of the waits that let this CTA's own asynchronous copies and MMAs
    // finish before it frees TMEM and exits: never shorter than 1 s, whatever
    // the watchdog, so an abort never leaves work in flight.
    const uint64_t drain_ns = p.timeout_ns > 1000000000ull ? p.timeout_ns : 1000000000ull;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_area + 192);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bar_area + 196);
    volatile int *s_epi_ok = reinterpret_cast<volatile int *>(bar_area + 208);  // [3]: by segment parity, tail
    volatile uint32_t *s_epoch = reinterpret_cast<volatile uint32_t *>(bar_area + 224);  // this call's epoch
    TailState *s_tail = reinterpret_cast<TailState *>(bar_area + 256);
    // the other CTA's abort flag (clusters), set with this CTA's
    const uint32_t peer_abort = CLUSTER ? ptx::mapa(ptx::smem_addr(bar_area + 196), rank ^ 1u) : 0u;
    // barriers completed by the other CTA's tcgen05 commits: the odd CTA of a
    // pair (stage-empty, accumulator-full); both CTAs of a multicast cluster
    // (stage-empty: a stage is refilled once both CTAs' MMAs are done with it)
    const bool remote_empty = (PAIR && rank != 0) || MCAST;
    const bool remote_accf = PAIR && rank != 0;
    static_assert(256 + sizeof(TailState) <= 384, "barrier area");
    int32_t *prefix;
    if constexpr (C::kSmemPrefix)
        prefix = reinterpret_cast<int32_t *>(bar_area + C::kBarrierBytes);
    else
        prefix = p.ws.cta_prefix + (size_t)blockIdx.x * (cta_prefix_bytes(CAP) / sizeof(int32_t));
    int32_t *wprefix = prefix + (C::kSmemPrefix ? C::kPrefixInts : (int)(cta_prefix_bytes(CAP) / 8));

    // ---- set-up -------------------------------------------------------------
    // Clusters: every thread arrives on the cluster barrier (warp 4 once the
    // mbarriers are initialised) and waits on it before its first access to
    // the other CTA
    if constexpr (CLUSTER) {
        if (warp != 4 && warp != 5)
            ptx::cluster_arrive();
    }
    if (warp == 4) {
        if (lane == 0) {
            for (int s = 0; s < C::kStages; ++s) {
                ptx::mbar_init(full_bar(s), 1);
                ptx::mbar_init(empty_bar(s), MCAST ? 2 : 1);  // multicast: both CTAs' MMAs
                // CTA pairs: the even CTA's also takes the odd CTA's relay
                ptx::mbar_init(sff_bar(s), (PAIR && rank == 0) ? 5 : 4);
                ptx::mbar_init(sfl_bar(s), 1);
            }
            for (int a = 0; a < C::kAccStages; ++a) {
                ptx::mbar_init(accf_bar(a), 1);
                ptx::mbar_init(acce_bar(a), PAIR ? 16 : 8);  // the epilogue warps of both CTAs of a pair
            }
            ptx::mbar_init(partial_bar, 1);
            ptx::mbar_init(drain_bar, 1);
            *abort_flag = 0;
            s_tail->valid = 0;
            s_tail->part_state = 0;
            s_tail->part_ok = 0;
            s_tail->part_stage0 = 0;
            s_tail->pieces = 0;
            ptx::fence_mbar_init();
        }
        if constexpr (CLUSTER) {
            __syncwarp();
            ptx::cluster_arrive();
        }
        // Patch the descriptors of this CTA's share of the groups.
        uint32_t patched = 0;
        for (int g = blockIdx.x + lane * gridDim.x; g < group_count; g += 32 * gridDim.x) {
            const GroupArgs a = load_group(p, g);
            if (a.m <= 0 || a.n <= 0 || a.k <= 0 || a.l == 0)
                continue;
            const uint32_t row_bytes = (uint32_t)(a.k / 2);
            // SFB as a 2-D array of 8-byte words: one row per 128-row block
            // of B (all batches stacked), ceil(k / 64) atoms of 512 B per row
            const uint32_t sf_row_words = (uint32_t)ceil_div_i(a.k, kMmaK) * (kSfAtomBytes / 8);
            const uint32_t sf_rows = (uint32_t)a.l * (uint32_t)ceil_div_i(a.n, kBlockM);
            for (int which = 0; which < kDescPerGroup; ++which) {
                if (!(a.patch & (1 << which)))
                    continue;
                uint8_t *t = p.ws.tmaps + ((size_t)g * kDescPerGroup + which) * kDescBytes;
                const uint4 *src =
                    reinterpret_cast<const uint4 *>(which == 0 ? p.tmpl_a : which == 1 ? p.tmpl_b : p.tmpl_sfb);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    reinterpret_cast<uint4 *>(t)[q] = src[q];
                if (which < 2) {
                    ptx::tmap_set_address(t, which ? a.b : a.a);
                    ptx::tmap_set_dims(t, row_bytes, (uint32_t)a.l * (uint32_t)(which ? a.n : a.m));
                    ptx::tmap_set_stride1(t, row_bytes);
                } else {
                    ptx::tmap_set_address(t, a.sfb);
                    ptx::tmap_set_dims(t, sf_row_words, sf_rows);
                    ptx::tmap_set_stride1(t, (uint64_t)sf_row_words * 8u);
                }
                ++patched;
            }
        }
        // Publication: every CTA adds 1 once its lanes' descriptors are
        // released; producers wait for all gridDim.x.
        if (patched)
            ptx::tmap_release();
        __syncwarp();
        if (publish && lane == 0)
            ptx::red_release_add_gpu(p.ws.desc_count, 1u);
        // When no descriptor changes in this call, start fetching those of
        // the first 10 groups (lane: group lane / 3, A, B or SFB) into the
        // descriptor cache while set-up goes on (non-empty groups only: the
        // slots of the others may hold anything).
        if (!publish && lane < kDescPerGroup * group_count && lane < 30) {
            const GroupArgs a = load_group(p, lane / kDescPerGroup);
            if (a.m > 0 && a.n > 0 && a.k > 0 && a.l > 0)
                ptx::tmap_prefetch(p.ws.tmaps + (size_t)lane * kDescBytes);
        }
        // The producer needs the barriers, the prefix sums and the epoch, not
        // TMEM: it starts once warp 6 has the prefix sums and warp 7 the
        // epoch, while the TMEM allocation may still be in progress.
        __syncwarp();
        ptx::named_barrier(2, 96);
        ptx::named_barrier_arrive(3, C::kThreads);
        if constexpr (CLUSTER)
            ptx::cluster_wait();
    } else if (warp == 5) {
        // a pair's allocation is made by this warp of both CTAs together
        if constexpr (CLUSTER) {
            ptx::cluster_arrive();
            ptx::cluster_wait();
        }
        ptx::tmem_alloc<C::kCtaGroup>(ptx::smem_addr(tmem_slot), C::kTmemCols);
        ptx::tmem_relinquish<C::kCtaGroup>();
    } else if (warp == 7) {
        // This call's epoch, for the producer, the partial-tile flags and the
        // counter reset (read before the producer counts this CTA as done).
        if (lane == 0)
            *s_epoch = call_epoch();
        __syncwarp();
        ptx::named_barrier_arrive(2, 96);
    } else if (warp == 6) {
        // Exclusive prefix sums of output tiles and schedule units per group.
        if constexpr (DEV) {
            // The caller's table in global memory: 32 groups per step, one per
            // lane (independent loads), then a warp scan. A call whose unit
            // count overflows int32 does nothing and is reported.
            const unsigned full = 0xffffffffu;
            long long bt = 0, bw = 0;
            bool bad = false;
            for (int g0 = 0; g0 < group_count; g0 += 32) {
                const int g = g0 + lane;
                long long t = 0, w = 0;
                if (g < group_count) {
                    const GroupArgs a = load_group(p, g, &bad);
                    t = (a.m > 0 && a.n > 0) ? (long long)ceil_div_i(a.m, C::kTileM) * ceil_div_i(a.n, BN) * a.l : 0;
                    const int kt = ceil_div_i(a.k, kBlockK);
                    w = t * (kt > 1 ? kt : 1);
                }
                long long it = t, iw = w;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const long long ut = __shfl_up_sync(full, it, o), uw = __shfl_up_sync(full, iw, o);
                    if (lane >= o) {
                        it += ut;
                        iw += uw;
                    }
                }
                if (g < group_count) {
                    prefix[g] = (int32_t)(bt + it - t);
                    wprefix[g] = (int32_t)(bw + iw - w);
                }
                bt += __shfl_sync(full, it, 31);
                bw += __shfl_sync(full, iw, 31);
            }
            if (bw > 0x7fffffffLL) {
                for (int g = lane; g < group_count; g += 32)
                    prefix[g] = wprefix[g] = 0;
                bt = bw = 0;
                bad = true;
            }
            if (lane == 0) {
                prefix[group_count] = (int32_t)bt;
                wprefix[group_count] = (int32_t)bw;
            }
            if (__any_sync(full, bad) && blockIdx.x == 0 && lane == 0)
                atomicOr(p.ws.status, kStatusBadGroup);
        } else {
            // The group table lives in the constant bank, where a warp
            // reading different addresses is serialised, so every lane walks
            // all groups with the same index (broadcast reads) and lane g % 32
            // stores entry g.
            int bt = 0, bw = 0;
#pragma unroll 4
            for (int g = 0; g < group_count; ++g) {
                const GroupArgs &a = p.groups[g];
                const int tiles = (a.m > 0 && a.n > 0) ? ceil_div_i(a.m, C::kTileM) * ceil_div_i(a.n, BN) * a.l : 0;
                const int kt = ceil_div_i(a.k, kBlockK);
                if (lane == (g & 31)) {
                    prefix[g] = bt;
                    wprefix[g] = bw;
                }
                bt += tiles;
                bw += tiles * (kt > 1 ? kt : 1);
            }
            if (lane == 0) {
                prefix[group_count] = bt;
                wprefix[group_count] = bw;
            }
        }
        __syncwarp();
        ptx::named_barrier_arrive(2, 96);
    }
    uint32_t tmem_base = 0;  // warp 4 reads it after the role loops
    if (warp != 4) {
        if constexpr (CLUSTER) {
            if (warp != 5)
                ptx::cluster_wait();
        }
        ptx::tc_fence_before();
        ptx::named_barrier(3, C::kThreads);
        ptx::tc_fence_after();
        tmem_base = *tmem_slot;
    }
    // Schedule of the call (choose_split_tile): given by the host, or (device
    // table) derived here by every CTA from the same prefix sums with the
    // host's rule. Whole tiles go round-robin over P CTAs; the split range --
    // the schedule units of tiles >= split_tile, from unit sk0 -- is cut into
    // P equal parts. An all-split schedule uses the first P = min(units, grid)
    // CTAs.
    const int total_tiles = DEV ? prefix[group_count] : p.total_tiles;
    const int total_work = DEV ? wprefix[group_count] : p.total_work;
    int split_tile = p.split_tile;
    if constexpr (DEV)
        split_tile = choose_split_tile(total_tiles, nslots, p.ws.partial_slots >= nslots ? p.split : 0);
    if constexpr (CLUSTER)
        split_tile = total_tiles;  // clusters run whole tiles only
    const int split = split_tile < total_tiles ? 1 : 0;
    const int P = (split && split_tile == 0 && total_work < nslots) ? total_work : nslots;
    const int sk0 = split_tile == 0 ? 0
                                    : tile_first_unit<BN>(p, prefix, wprefix, group_count, split_tile, total_tiles,
                                                          total_work);
    // The split range goes to the first Psk CTAs, at least one unit each (an
    // empty part would hold no piece, yet a finishing CTA counts the CTAs
    // after it whose part starts inside its tile as holding pieces).
    const int Psk = split ? (total_work - sk0 < P ? total_work - sk0 : P) : 0;
    // first schedule unit of CTA c's part of the split range
    auto sk_begin = [&](int c) { return sk0 + split_begin(c, Psk, total_work - sk0); };
    Cursor<BN, CAP, DEV, CLUSTER> cursor0{prefix, wprefix, group_count, slot, split_tile, P, 0, 0, 0, (int)rank};
    if (split && slot < Psk) {
        cursor0.w = sk_begin(slot);
        cursor0.w_end = sk_begin(slot + 1);
    }
    if (slot >= P)
        cursor0.tile = cursor0.tile_end;  // no whole tiles either

    if (warp == 4) {
        // ===================== TMA producer =====================
        if (lane == 0) {
            const uint64_t pol_a = ptx::l2_policy_evict_last();
            const uint64_t pol_keep = ptx::l2_policy_evict_last();
            const uint64_t pol_once = ptx::l2_policy_evict_first();
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            int prev_g = -1;
            const uint32_t epoch = *s_epoch;
            // every group's descriptors are patched by some CTA at start-up
            bool ok = !publish || wait_counter(p.ws.desc_count, gridDim.x, abort_flag, p.timeout_ns, p.ws.status);
            // Once every CTA is past its descriptor wait and has read the
            // epoch (set-up, warp 6), the last one resets the call counters
            // for the next call. Counted after this CTA's first copies are
            // issued (or when it has none), off the path to its first MMA.
            bool counted = false;
            auto count_done = [&]() {
                counted = true;
                if (atomicAdd(p.ws.done, 1u) == gridDim.x - 1) {
                    *p.ws.desc_count = 0;
                    *p.ws.done = 0;
                    *p.ws.epoch = *s_epoch;
                }
            };
            auto cur = cursor0;
            Segment sg;
            bool any = false;
            while (ok && cur.next(p, sg)) {
                any = true;
                const GInfo gi = group_info<BN, CLUSTER>(load_group(p, sg.g));
                const int k_tiles = gi.k_tiles;
                const int kend = sg.kt1 < k_tiles ? sg.kt1 : k_tiles;
                if (sg.kt0 >= kend)
                    continue;  // k == 0 tile: nothing to load
                const int k_blocks = gi.k_blocks;
                // B panels read by one m-tile stream through L2; the others stay
                const uint64_t pol_b = gi.tiles_m > 1 ? pol_keep : pol_once;
                const uint8_t *tmap_a = p.ws.tmaps + (size_t)sg.g * (kDescPerGroup * kDescBytes);
                const uint8_t *tmap_b = tmap_a + kDescBytes;
                const uint8_t *tmap_sfb = tmap_b + kDescBytes;
                if (sg.g != prev_g) {
                    ptx::tmap_acquire(tmap_a);
                    ptx::tmap_acquire(tmap_b);
                    if constexpr (BN == 256)
                        ptx::tmap_acquire(tmap_sfb);
                    prev_g = sg.g;
                }
                // a CTA of a pair whose 128 rows all lie past m loads no A and
                // no A scales (its accumulator rows are never stored)
                const bool a_live = !CLUSTER || sg.tm * kBlockM < gi.m;
                const uint8_t *sfa = gi.sfa + (size_t)sg.b * gi.sfa_batch + (size_t)sg.tm * k_blocks * kSfAtomBytes;
                int sfb_blocks = gi.sf_row_blocks_b - sg.tn * C::kSfbRowBlocks;
                sfb_blocks = sfb_blocks < C::kSfbRowBlocks ? sfb_blocks : C::kSfbRowBlocks;
                const uint8_t *sfb =
                    gi.sfb + (size_t)sg.b * gi.sfb_batch + (size_t)sg.tn * C::kSfbRowBlocks * k_blocks * kSfAtomBytes;
                for (int kt = sg.kt0; kt < kend; ++kt) {
                    // (the odd CTA of a pair is released by the even CTA's commits)
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, p.timeout_ns, p.ws.status,
                                      kStatusProducerTimeout, peer_abort, remote_empty)) {
                        ok = false;
                        break;
                    }
                    const int nkb = (k_blocks - 4 * kt) < 4 ? (k_blocks - 4 * kt) : 4;
                    const uint32_t sf_bytes = (uint32_t)nkb * kSfAtomBytes;
                    const uint32_t st = smem_base + stage * C::kStageBytes;
                    const uint32_t fb = full_bar(stage);
                    // The scale atoms go first, on their own barrier: they land
                    // well before the operand tiles, so the scale writers move
                    // them into TMEM while A and B are still in flight.
                    const uint32_t sb = sfl_bar(stage);
                    if constexpr (BN == 256) {
                        // both 128-row blocks of SFB in one 2-D copy (4 atoms x
                        // 2 rows, zero beyond k and n; a last n-tile with one
                        // row block reads the next rows, which only reach
                        // accumulator columns >= n): one copy operation fewer
                        // per stage, which the ring's round trip pays for
                        ptx::mbar_arrive_expect_tx(sb, (a_live ? sf_bytes : 0u) + C::kSfbBytes);
                        if (a_live)
                            ptx::bulk_load(st + C::kABytes + C::kBBytes, sfa + (size_t)(4 * kt) * kSfAtomBytes,
                                           sf_bytes, sb, pol_a);
                        // (multicast cluster: the odd CTA fetches the B scales for both)
                        if constexpr (MCAST) {
                            if (rank == 1)
                                ptx::tma_load_2d_multicast(st + C::kABytes + C::kBBytes + C::kSfaBytes, tmap_sfb,
                                                           kt * (4 * kSfAtomBytes / 8),
                                                           sg.b * gi.sf_row_blocks_b + sg.tn * 2, sb, 3, pol_b);
                        } else {
                            ptx::tma_load_2d(st + C::kABytes + C::kBBytes + C::kSfaBytes, tmap_sfb,
                                             kt * (4 * kSfAtomBytes / 8), sg.b * gi.sf_row_blocks_b + sg.tn * 2, sb,
                                             pol_b);
                        }
                    } else {
                        ptx::mbar_arrive_expect_tx(sb, sf_bytes * (1 + sfb_blocks));
                        ptx::bulk_load(st + C::kABytes + C::kBBytes, sfa + (size_t)(4 * kt) * kSfAtomBytes, sf_bytes,
                                       sb, pol_a);
                        for (int j = 0; j < sfb_blocks; ++j)
                            ptx::bulk_load(st + C::kABytes + C::kBBytes + C::kSfaBytes + j * 4 * kSfAtomBytes,
                                           sfb + ((size_t)j * k_blocks + 4 * kt) * kSfAtomBytes, sf_bytes, sb, pol_b);
                    }
                    ptx::mbar_arrive_expect_tx(fb, (a_live ? (uint32_t)C::kABytes : 0u) + C::kBBytes);
                    // batch b's rows start at b * m (b * n) of the group's stack;
                    // rows a tile reads past its batch only reach accumulator
                    // rows / columns that the epilogue does not store. A CTA of
                    // a pair loads its half of the tile's B rows.
                    if (a_live)
                        ptx::tma_load_2d(st, tmap_a, kt * 128, sg.b * gi.m + sg.tm * kBlockM, fb, pol_a);
                    if constexpr (MCAST) {
                        // the even CTA fetches the B tile for both
                        if (rank == 0)
                            ptx::tma_load_2d_multicast(st + C::kABytes, tmap_b, kt * 128, sg.b * gi.n + sg.tn * BN, fb,
                                                       3, pol_b);
                    } else {
                        ptx::tma_load_2d(st + C::kABytes, tmap_b, kt * 128,
                                         sg.b * gi.n + sg.tn * BN + (PAIR ? (int)rank * C::kBRows : 0), fb, pol_b);
                    }
                    armed |= 1u << stage;
                    armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (!counted)
                        count_done();
                }
            }
            if (!counted)
                count_done();
            if (ok && any && split && sg.kt0 == 0 && sg.kt1 < sg.ktg && !*abort_flag) {
                // The last segment is the first piece of a split tile. Once the
                // later pieces are published (they are their CTAs' first
                // segments, so usually long before), the next piece's partial
                // tile is copied into the ring, each stage as soon as the MMAs
                // reading it have completed, oldest stage first.
                const int cta = blockIdx.x;
                int pieces = 0;
                while (cta + pieces + 1 < Psk && sk_begin(cta + pieces + 1) < sg.w_tile_end)
                    ++pieces;
                bool flags_ok = true;
                for (int c2 = cta + 1; c2 <= cta + pieces && flags_ok; ++c2) {
                    const uint64_t t0 = ptx::globaltimer();
                    while (ptx::ld_acquire_gpu(p.ws.flags + c2) != epoch) {
                        if (*abort_flag) {
                            flags_ok = false;
                            break;
                        }
                        if (ptx::globaltimer() - t0 > p.timeout_ns) {
                            *abort_flag = 1;
                            atomicOr(p.ws.status, kStatusFlagTimeout);
                            flags_ok = false;
                            break;
                        }
                    }
                }
                s_tail->pieces = pieces;
                if (flags_ok) {
                    ptx::fence_proxy_async_global();
                    const int nch = tile_chunks<BN>(group_info<BN, CLUSTER>(load_group(p, sg.g)), sg);
                    const char *src =
                        reinterpret_cast<const char *>(p.ws.partials) + (size_t)(cta + 1) * kPartialSlotBytes;
                    bool good = true;
                    // one copy per ring stage: the chunks of a stage are
                    // contiguous in the workspace slot and in the stage
                    for (int cc = 0; cc < nch; cc += C::kPartialChunksPerStage) {
                        const int s = (stage + cc / C::kPartialChunksPerStage) % C::kStages;
                        if (((armed >> s) & 1u) &&
                            !wait_bounded(empty_bar(s), (armed_parity >> s) & 1u, abort_flag, p.timeout_ns,
                                          p.ws.status, kStatusProducerTimeout, peer_abort)) {
                            good = false;
                            break;
                        }
                        const int nc = (nch - cc) < C::kPartialChunksPerStage ? (nch - cc) : C::kPartialChunksPerStage;
                        ptx::mbar_expect_tx(partial_bar, (uint32_t)nc * kPartialChunkBytes);
                        ptx::bulk_load(smem_base + s * C::kStageBytes, src + (size_t)cc * kPartialChunkBytes,
                                       (uint32_t)nc * kPartialChunkBytes, partial_bar, ptx::l2_policy_evict_first());
                    }
                    ptx::mbar_arrive(partial_bar);
                    s_tail->part_stage0 = stage;
                    s_tail->part_ok = good ? 1 : 0;
                    s_tail->part_state = 1;
                }
            }
            if (!ok || *abort_flag) {
                // Let every copy this thread issued land before the CTA exits.
                for (int s = 0; s < C::kStages; ++s) {
                    if (!(armed & (1u << s)))
                        continue;
                    const uint32_t par = (armed_parity >> s) & 1u;
                    const uint64_t t0 = ptx::globaltimer();
                    while (!ptx::mbar_try_wait(full_bar(s), par) && ptx::globaltimer() - t0 < drain_ns) {
                    }
                    while (!ptx::mbar_try_wait(sfl_bar(s), par) && ptx::globaltimer() - t0 < drain_ns) {
                    }
                }
            }
        }
    } else if (warp == 5) {
        if (PAIR && rank != 0) {
            // ============ relay (odd CTA of a pair) ============
            // Tells the even CTA's MMA thread when this CTA's stage is ready
            // (its A / B tiles have landed and its scale writers are done) by
            // arriving on the even CTA's scales-written barrier of the stage.
            if (lane == 0) {
                int stage = 0;
                uint32_t phase = 0;
                bool ok = true;
                auto cur = cursor0;
                Segment sg;
                while (ok && cur.next(p, sg)) {
                    const GInfo gi = group_info<BN, CLUSTER>(load_group(p, sg.g));
                    const int kend = sg.kt1 < gi.k_tiles ? sg.kt1 : gi.k_tiles;
                    for (int kt = sg.kt0; kt < kend; ++kt) {
                        if (!wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns, p.ws.status,
                                                kStatusMmaTimeout, peer_abort) ||
                            !wait_bounded(sff_bar(stage), phase, abort_flag, p.timeout_ns, p.ws.status,
                                                kStatusMmaTimeout, peer_abort)) {
                            ok = false;
                            break;
                        }
                        ptx::mbar_arrive_cluster(ptx::mapa(sff_bar(stage), 0u));
                        if (++stage == C::kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
        } else if (lane == 0) {
            // ===================== MMA issuer =====================
            // (CTA pairs: the even CTA issues the pair's MMAs and commits to
            // both CTAs' barriers)
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            auto cur = cursor0;
            Segment sg;
            while (ok && cur.next(p, sg)) {
                const GInfo gi = group_info<BN, CLUSTER>(load_group(p, sg.g));
                const int k_tiles = gi.k_tiles;
                const int k_blocks = gi.k_blocks;
                const int kend = sg.kt1 < k_tiles ? sg.kt1 : k_tiles;
                if (!wait_bounded<PAIR>(acce_bar(acc), acc_phase ^ 1u, abort_flag, p.timeout_ns, p.ws.status,
                                        kStatusMmaTimeout, peer_abort, PAIR))
                    break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * C::kAccCols);
                // (multicast cluster: a CTA whose rows all lie past m computes
                // nothing, but still releases its stages)
                const bool mma_live = !MCAST || sg.tm * kBlockM < gi.m;
                for (int kt = sg.kt0; kt < kend; ++kt) {
                    // (CTA pairs: one wait. The even CTA's scales-written
                    // barrier completes once its tiles have landed too -- its
                    // scale writer warp 6 waits for them -- and the odd CTA's
                    // stage is ready, which the odd CTA's relay reports on it.)
                    if ((!PAIR && !wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns, p.ws.status,
                                                kStatusMmaTimeout, peer_abort)) ||
                        !wait_bounded<PAIR>(sff_bar(stage), phase, abort_flag, p.timeout_ns, p.ws.status,
                                            kStatusMmaTimeout, peer_abort)) {
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
                    // (+32 bytes per 64-element k-block inside the swizzled row)
                    if (nkb == 4 && mma_live) {
                        // a whole k-tile: straight-line issue (a loop with a
                        // run-time trip count between the MMAs costs issue rate)
                        ptx::tc_mma_mxf4nvf4<C::kCtaGroup>(d_tmem, adesc, bdesc, C::kIdesc, sfa_t, sfb_t,
                                                           kt != sg.kt0 ? 1u : 0u);
                        ptx::tc_mma_mxf4nvf4<C::kCtaGroup>(d_tmem, adesc + 2u, bdesc + 2u, C::kIdesc, sfa_t + 4,
                                                           sfb_t + (BN / 32), 1u);
                        ptx::tc_mma_mxf4nvf4<C::kCtaGroup>(d_tmem, adesc + 4u, bdesc + 4u, C::kIdesc, sfa_t + 8,
                                                           sfb_t + 2 * (BN / 32), 1u);
                        ptx::tc_mma_mxf4nvf4<C::kCtaGroup>(d_tmem, adesc + 6u, bdesc + 6u, C::kIdesc, sfa_t + 12,
                                                           sfb_t + 3 * (BN / 32), 1u);
                    } else {
                        for (int kb = 0; kb < (mma_live ? nkb : 0); ++kb)
                            ptx::tc_mma_mxf4nvf4<C::kCtaGroup>(d_tmem, adesc + 2u * kb, bdesc + 2u * kb, C::kIdesc,
                                                               sfa_t + 4 * kb, sfb_t + kb * (BN / 32),
                                                               (kt != sg.kt0 || kb != 0) ? 1u : 0u);
                    }
                    if constexpr (MCAST) {
                        // the stage is refilled (by multicasts into both CTAs)
                        // once both CTAs' MMAs are done with it
                        ptx::tc_commit_multicast(empty_bar(stage), 3);
                    } else {
                        ptx::tc_commit<C::kCtaGroup>(empty_bar(stage));
                        if constexpr (PAIR)
                            ptx::tc_commit<C::kCtaGroup>(ptx::mapa(empty_bar(stage), 1u));
                    }
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                ptx::tc_commit<C::kCtaGroup>(accf_bar(acc));
                if constexpr (PAIR)
                    ptx::tc_commit<C::kCtaGroup>(ptx::mapa(accf_bar(acc), 1u));
                if (++acc == C::kAccStages) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            // Every MMA this thread issued completes before the CTA can free
            // TMEM -- on the normal path the epilogue already waits for them,
            // after an abort nothing else would.
            ptx::tc_commit<C::kCtaGroup>(drain_bar);
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(drain_bar, 0) && ptx::globaltimer() - t0 < drain_ns) {
            }
        }
    } else if (warp >= 6 && warp < 10) {
        // ===================== scale writers (warps 6..9) =====================
        // Warp w owns TMEM lanes 32*(w % 4) .. +31 and writes the scale atoms
        // of every stage into that quarter.
        const uint32_t quarter = (uint32_t)((warp & 3) * 32) << 16;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        auto cur = cursor0;
        Segment sg;
        while (ok && cur.next(p, sg)) {
            const GInfo gi = group_info<BN, CLUSTER>(load_group(p, sg.g));
            const int k_tiles = gi.k_tiles;
            const int k_blocks = gi.k_blocks;
            const int kend = sg.kt1 < k_tiles ? sg.kt1 : k_tiles;
            for (int kt = sg.kt0; kt < kend; ++kt) {
                int got = 0;
                if (lane == 0)
                    got = wait_bounded(sfl_bar(stage), phase, abort_flag, p.timeout_ns, p.ws.status, kStatusMmaTimeout, peer_abort)
                              ? 1
                              : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                (void)ptx::mbar_try_wait(sfl_bar(stage), phase);  // every lane acquires the landed scales
                const int nkb = (k_blocks - 4 * kt) < 4 ? (k_blocks - 4 * kt) : 4;
                const uint8_t *st_sfa = smem + stage * C::kStageBytes + C::kABytes + C::kBBytes;
                const uint8_t *st_sfb = st_sfa + C::kSfaBytes;
                const uint32_t sfa_t = tmem_base + quarter + (uint32_t)(C::kSfColBase + stage * C::kSfColsPerStage);
                const uint32_t sfb_t = sfa_t + C::kSfaCols;
                // The stage's SFA columns (4 per k-block) and SFB columns
                // (BN/32 per k-block) are each one contiguous run: all of a
                // lane's words go out in one wide store per operand. Columns
                // of k-blocks past the K tail get zeros (no MMA reads them).
                uint32_t va[C::kSfaCols], vb[C::kSfbCols];
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
                    const uint4 w = kb < nkb ? *reinterpret_cast<const uint4 *>(st_sfa + kb * kSfAtomBytes + 16 * lane)
                                             : make_uint4(0, 0, 0, 0);
                    va[4 * kb] = w.x;
                    va[4 * kb + 1] = w.y;
                    va[4 * kb + 2] = w.z;
                    va[4 * kb + 3] = w.w;
#pragma unroll
                    for (int j = 0; j < C::kSfbRowBlocks; ++j) {
                        const uint4 u = kb < nkb ? *reinterpret_cast<const uint4 *>(
                                                       st_sfb + (j * 4 + kb) * kSfAtomBytes + 16 * lane)
                                                 : make_uint4(0, 0, 0, 0);
                        const int c = kb * (BN / 32) + 4 * j;
                        vb[c] = u.x;
                        vb[c + 1] = u.y;
                        vb[c + 2] = u.z;
                        vb[c + 3] = u.w;
                    }
                }
                ptx::tmem_st_32x32b_x16(sfa_t, va);
                if constexpr (C::kSfbCols == 32)
                    ptx::tmem_st_32x32b_x32(sfb_t, vb);
                else
                    ptx::tmem_st_32x32b_x16(sfb_t, reinterpret_cast<const uint32_t(&)[16]>(vb));
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                __syncwarp();
                // (the even CTA of a pair: warp 6 first waits for the stage's
                // A and B tiles, so that the barrier stands for the whole
                // stage and the pair's MMA thread waits on it alone)
                int fine = 1;
                if (lane == 0) {
                    if (PAIR && rank == 0 && warp == 6)
                        fine = wait_bounded(full_bar(stage), phase, abort_flag, p.timeout_ns, p.ws.status,
                                            kStatusMmaTimeout, peer_abort)
                                   ? 1
                                   : 0;
                    if (fine)
                        ptx::mbar_arrive(sff_bar(stage));
                }
                if (PAIR && !__shfl_sync(0xffffffffu, fine, 0)) {
                    ok = false;
                    break;
                }
                if (++stage == C::kStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else {
        // ================= epilogue (warps 0..3 and 10..13) =================
        // Every segment but the CTA's last; the last is finished below, once
        // every role has left its loop, by warps 0..7. Warp w takes TMEM lane
        // quarter w % 4; warps 0..3 the first half of the column chunks,
        // warps 10..13 the second.
        const int cta = blockIdx.x;
        const bool first_half = warp < 4;
        const int quarter = warp & 3;
        int acc = 0, it = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        // The eight warps' schedule cursor is one copy in shared memory,
        // advanced by thread 0 (segments in two slots by parity, each with
        // whether another segment follows it), so that no epilogue register
        // holds it across the accumulator drain.
        static_assert(sizeof(Cursor<BN, CAP, DEV, CLUSTER>) <= 64 && 2 * sizeof(Segment) <= 64, "cursor area");
        auto *ecur = reinterpret_cast<Cursor<BN, CAP, DEV, CLUSTER> *>(bar_area + C::kEpiCursorOffset);
        Segment *eseg = reinterpret_cast<Segment *>(bar_area + C::kEpiCursorOffset + 64);
        volatile int *emore = reinterpret_cast<volatile int *>(bar_area + C::kEpiCursorOffset + 128);
        if (threadIdx.x == 0) {
            *ecur = cursor0;
            emore[2] = ecur->next(p, eseg[0]) ? 1 : 0;
            emore[0] = ecur->more() ? 1 : 0;
        }
        ptx::named_barrier(4, 256);
        const bool have = emore[2] != 0;
        while (have && emore[it & 1]) {
            const Segment sg = eseg[it & 1];
            const GInfo gi = group_info<BN, CLUSTER>(load_group(p, sg.g));
            // a first piece of a split tile is always a CTA's last segment
            const int kind = sg.kt0 > 0 ? kEpiCont : kEpiWhole;
            // One thread takes the next segment and waits for the
            // accumulator; the eight warps leave or stay together (the TMEM
            // loads are warp-collective).
            if (threadIdx.x == 0) {
                (void)ecur->next(p, eseg[(it + 1) & 1]);
                emore[(it + 1) & 1] = ecur->more() ? 1 : 0;
                s_epi_ok[it & 1] = wait_bounded(accf_bar(acc), acc_phase, abort_flag, p.timeout_ns, p.ws.status,
                                                kStatusEpilogueTimeout, peer_abort, remote_accf)
                                       ? 1
                                       : 0;
            }
            ptx::named_barrier(4, 256);
            if (!s_epi_ok[it & 1]) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const int nch = tile_chunks<BN>(gi, sg);
            const int half = (nch + 1) / 2;
            // a whole tile releases the accumulator once its chunks are in
            // registers; a partial tile (fp32) goes out chunk by chunk first
            const uint32_t t_acc = tmem_base + (uint32_t)(acc * C::kAccCols);
            epilogue_warp<BN, CAP, DEV, CLU>(p, sg, gi, kind, quarter, lane, t_acc, first_half ? 0 : half,
                                             first_half ? half : nch, smem, 0, 0,
                                             kind == kEpiWhole ? acce_release(acc) : 0u);
            if (kind != kEpiWhole) {
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR)
                        ptx::mbar_arrive_cluster(acce_release(acc));
                    else
                        ptx::mbar_arrive(acce_bar(acc));
                }
            }
            if (kind == kEpiCont) {
                // publish this CTA's partial tile
                ptx::named_barrier(4, 256);
                if (threadIdx.x == 0) {
                    __threadfence();
                    ptx::st_release_gpu(p.ws.flags + cta, *s_epoch);
                }
            }
            if (++acc == C::kAccStages) {
                acc = 0;
                acc_phase ^= 1u;
            }
            ++it;
        }
        if (threadIdx.x == 0) {
            s_tail->seg = eseg[it & 1];
            s_tail->valid = (have && ok) ? 1 : 0;
            s_tail->acc = acc;
            s_tail->acc_phase = (int32_t)acc_phase;
        }
    }

    // ---- the last segment: warps 0..7 ------------------------------------------
    // Its MMAs are the CTA's last, so the ring holds nothing but the partial
    // tile the producer may have prefetched.
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    tmem_base = *tmem_slot;
    if (warp < 8) {
        const TailState ts = *s_tail;
        const Segment sg = ts.seg;
        const GInfo gi = group_info<BN, CLUSTER>(load_group(p, ts.valid ? sg.g : 0));
        const int kind = sg.kt0 > 0 ? kEpiCont : ((split && sg.kt1 < sg.ktg) ? kEpiFinish : kEpiWhole);
        if (threadIdx.x == 0) {
            int ok = ts.valid && wait_bounded(accf_bar(ts.acc), (uint32_t)ts.acc_phase, abort_flag, p.timeout_ns,
                                              p.ws.status, kStatusEpilogueTimeout, peer_abort, remote_accf);
            if (ts.part_state) {
                // the partial-tile copies must land before the CTA exits, even
                // after an abort
                const uint64_t t0 = ptx::globaltimer();
                bool landed;
                while (!(landed = ptx::mbar_try_wait(partial_bar, 0)) && ptx::globaltimer() - t0 < drain_ns) {
                }
                if (!landed) {
                    *abort_flag = 1;
                    atomicOr(p.ws.status, kStatusFlagTimeout);
                }
                ok = ok && landed && ts.part_ok;
            } else if (kind == kEpiFinish) {
                ok = 0;  // the producer gave up before copying the partial tile
            }
            s_epi_ok[2] = ok;
        }
        ptx::named_barrier(1, 256);
        if (ts.valid && s_epi_ok[2]) {
            if (kind == kEpiFinish)
                (void)ptx::mbar_try_wait(partial_bar, 0);  // every thread acquires the landed partial tile
            ptx::tc_fence_after();
            const int nch = tile_chunks<BN>(gi, sg);
            const int half = (nch + 1) / 2;
            const int quarter = warp & 3;
            epilogue_warp<BN, CAP, DEV, CLU>(p, sg, gi, kind, quarter, lane, tmem_base + (uint32_t)(ts.acc * C::kAccCols),
                                             warp < 4 ? 0 : half, warp < 4 ? half : nch, smem, ts.part_stage0,
                                             ts.pieces);
            if (kind == kEpiCont) {
                ptx::named_barrier(1, 256);
                if (threadIdx.x == 0) {
                    __threadfence();
                    ptx::st_release_gpu(p.ws.flags + blockIdx.x, *s_epoch);
                }
            }
        }
    }

    // ---- teardown ----------------------------------------------------------
    // Clusters: neither CTA leaves (or frees a pair's TMEM, which both free
    // together) while the other may still touch its shared memory, barriers
    // or TMEM
    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (CLUSTER) {
        ptx::cluster_arrive();
        ptx::cluster_wait();
    }
    if (warp == 5) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc<C::kCtaGroup>(tmem_base, C::kTmemCols);
    }
}

template <int BN, int CAP, bool DEV, int CLU = 0>
cudaError_t launch_cap(const GemmLaunch &cfg, const GroupArgs *groups, const WorkspaceView &ws,
                       const void *tmpl_a, const void *tmpl_b, const void *tmpl_sfb, cudaStream_t stream) {
    static_assert(sizeof(GemmParams<CAP, DEV>) <= 32000, "kernel parameter limit");
    GemmParams<CAP, DEV> prm;
    std::memcpy(prm.tmpl_a, tmpl_a, 128);
    std::memcpy(prm.tmpl_b, tmpl_b, 128);
    std::memcpy(prm.tmpl_sfb, tmpl_sfb, 128);
    prm.ws = ws;
    prm.group_count = cfg.group_count;
    prm.block_n = cfg.block_n;
    prm.total_tiles = cfg.total_tiles;
    prm.total_work = cfg.total_work;
    prm.split = cfg.split;
    prm.split_tile = cfg.split_tile;
    prm.desc_maps = cfg.desc_maps;
    prm.timeout_ns = cfg.timeout_ns;
    if constexpr (DEV) {
        prm.dt = cfg.dt;
        std::memset(prm.groups, 0, sizeof(prm.groups));
    } else {
        prm.dt = DeviceTable{};
        std::memcpy(prm.groups, groups, sizeof(GroupArgs) * (size_t)cfg.group_count);
        if (cfg.group_count < CAP)
            std::memset(prm.groups + cfg.group_count, 0, sizeof(GroupArgs) * (size_t)(CAP - cfg.group_count));
    }
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)cfg.grid, 1, 1);
    lc.blockDim = dim3(Cfg<BN, CAP, CLU>::kThreads, 1, 1);
    lc.dynamicSmemBytes = Cfg<BN, CAP, CLU>::kSmemBytes;
    lc.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = (CLU || cfg.pair_launch) ? 2 : 1;
    return cudaLaunchKernelEx(&lc, grouped_gemm_kernel<BN, CAP, DEV, CLU>, prm);
}

}  // namespace

cudaError_t prepare_gemm_kernels(int /*device*/) {
    cudaError_t e = cudaSuccess;
#define NVFP4_SET_SMEM(BN, CAP, DEV, CLU)                                                           \
    if (e == cudaSuccess)                                                                           \
        e = cudaFuncSetAttribute(grouped_gemm_kernel<BN, CAP, DEV, CLU>,                            \
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<BN, CAP, CLU>::kSmemBytes);
    NVFP4_SET_SMEM(128, kSmallGroups, false, 0)
    NVFP4_SET_SMEM(128, kMediumGroups, false, 0)
    NVFP4_SET_SMEM(128, NVFP4_MAX_GROUPS, false, 0)
    NVFP4_SET_SMEM(256, kSmallGroups, false, 0)
    NVFP4_SET_SMEM(256, kMediumGroups, false, 0)
    NVFP4_SET_SMEM(256, NVFP4_MAX_GROUPS, false, 0)
    NVFP4_SET_SMEM(128, kMediumGroups, true, 0)
    NVFP4_SET_SMEM(128, NVFP4_MAX_GROUPS, true, 0)
    NVFP4_SET_SMEM(256, kMediumGroups, true, 0)
    NVFP4_SET_SMEM(256, NVFP4_MAX_GROUPS, true, 0)
    NVFP4_SET_SMEM(256, kSmallGroups, false, 1)
    NVFP4_SET_SMEM(256, kMediumGroups, false, 1)
    NVFP4_SET_SMEM(256, NVFP4_MAX_GROUPS, false, 1)
    NVFP4_SET_SMEM(256, kSmallGroups, false, 2)
    NVFP4_SET_SMEM(256, kMediumGroups, false, 2)
    NVFP4_SET_SMEM(256, NVFP4_MAX_GROUPS, false, 2)
#undef NVFP4_SET_SMEM
    return e;
}

int pair_capacity(int /*device*/) {
    // The pair instantiation with the most shared memory (group table prefix
    // sums in shared memory) bounds how many pairs are resident at once.
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(2, 1, 1);
    lc.blockDim = dim3(Cfg<256, kMediumGroups, 2>::kThreads, 1, 1);
    lc.dynamicSmemBytes = Cfg<256, kMediumGroups, 2>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, (void *)grouped_gemm_kernel<256, kMediumGroups, false, 2>, &lc) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return clusters;
}

cudaError_t launch_grouped(const GemmLaunch &cfg, const GroupArgs *groups, const WorkspaceView &ws,
                           const void *tmpl_a, const void *tmpl_b, const void *tmpl_sfb, cudaStream_t stream) {
    if (ws.capacity < cfg.group_count || ws.capacity > NVFP4_MAX_GROUPS)
        return cudaErrorInvalidValue;
    if (cfg.split && ws.partial_slots < cfg.grid)
        return cudaErrorInvalidValue;
    if (cfg.group_count > kMediumGroups && ws.prefix_slots < cfg.grid)
        return cudaErrorInvalidValue;
    const bool wide = cfg.block_n == 256;
    if (cfg.cluster != 0) {
        if (!wide || cfg.device_table || cfg.split || (cfg.grid & 1) || cfg.cluster > 2)
            return cudaErrorInvalidValue;
#define NVFP4_LAUNCH_CLUSTER(CLU)                                                                                   \
    if (cfg.group_count <= kSmallGroups)                                                                          \
        return launch_cap<256, kSmallGroups, false, CLU>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream);     \
    if (cfg.group_count <= kMediumGroups)                                                                         \
        return launch_cap<256, kMediumGroups, false, CLU>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream);    \
    return launch_cap<256, NVFP4_MAX_GROUPS, false, CLU>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream);
        if (cfg.cluster == 1) {
            NVFP4_LAUNCH_CLUSTER(1)
        }
        NVFP4_LAUNCH_CLUSTER(2)
#undef NVFP4_LAUNCH_CLUSTER
    }
    if (cfg.device_table) {
        // shared-memory prefix sums up to kMediumGroups groups
        if (cfg.group_count <= kMediumGroups)
            return wide ? launch_cap<256, kMediumGroups, true>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream)
                        : launch_cap<128, kMediumGroups, true>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream);
        return wide ? launch_cap<256, NVFP4_MAX_GROUPS, true>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream)
                    : launch_cap<128, NVFP4_MAX_GROUPS, true>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream);
    }
    if (cfg.group_count <= kSmallGroups)
        return wide ? launch_cap<256, kSmallGroups, false>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream)
                    : launch_cap<128, kSmallGroups, false>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream);
    if (cfg.group_count <= kMediumGroups)
        return wide ? launch_cap<256, kMediumGroups, false>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream)
                    : launch_cap<128, kMediumGroups, false>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream);
    return wide ? launch_cap<256, NVFP4_MAX_GROUPS, false>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream)
                : launch_cap<128, NVFP4_MAX_GROUPS, false>(cfg, groups, ws, tmpl_a, tmpl_b, tmpl_sfb, stream);
}

}  // namespace nvfp4
