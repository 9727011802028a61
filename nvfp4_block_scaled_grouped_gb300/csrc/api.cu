// api.cu -- the C ABI: argument checks, per-device TMA descriptor templates,
// per-(device, stream) workspaces, launch configuration.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "internal.h"

namespace nvfp4 {

namespace {
thread_local char g_last_error[512] = "";
}  // namespace

int fail(int status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return status;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(NVFP4_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int pairs = 0;            // CTA pairs of the pair kernel resident at once (0: not used)
    CUtensorMap tmpl_a;       // box 128 B x 128 rows
    CUtensorMap tmpl_b128;    // box 128 B x 128 rows
    CUtensorMap tmpl_b256;    // box 128 B x 256 rows
    CUtensorMap tmpl_sfb;     // 8-byte words, box 256 words (4 scale atoms) x 2 rows, no swizzle
};

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
// One workspace per (device, stream): base pointer, per-CTA slots and what
// its descriptor slots hold.
struct StreamWorkspace {
    void *base = nullptr;
    int slots = 0;  // CTA slots for prefix scratch and partial tiles
    WorkspaceState state;
};
std::map<std::pair<int, cudaStream_t>, StreamWorkspace> g_workspaces;
int g_tile_n_override = 0;

// Encode a 2-D uint8 tensor map with 128-byte swizzle: dims {row_bytes, rows},
// box {128 bytes, box_rows}. Out-of-bounds elements read as zero.
int encode_template(EncodeTiledFn encode, CUtensorMap *out, void *addr, uint32_t box_rows) {
    const cuuint64_t dims[2] = {128, 256};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, addr, dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return NVFP4_OK;
}

// Encode the template of the B-scale map: a 2-D array of 8-byte words, dims
// {words per 128-row block, row blocks} (patched per group in the kernel), box
// {256 words = 4 scale atoms, 2 row blocks}, no swizzle. Out-of-bounds words
// read as zero.
int encode_sfb_template(EncodeTiledFn encode, CUtensorMap *out, void *addr) {
    const cuuint64_t dims[2] = {256, 2};
    const cuuint64_t strides[1] = {2048};
    const cuuint32_t box[2] = {256, 2};
    const cuuint32_t elem[2] = {1, 1};
    CUresult r = encode(out, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, addr, dims, strides, box, elem,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled failed for the scale map (CUresult %d)", (int)r);
    return NVFP4_OK;
}

// Caller holds g_mutex.
int device_state(int device, void *any_device_buffer, DeviceState **out) {
    if (device < 0 || device >= kMaxDevices)
        return fail(NVFP4_ERR_UNSUPPORTED, "device ordinal %d out of range", device);
    DeviceState &st = g_devices[device];
    if (!st.ready) {
        cudaDeviceProp prop;
        cudaError_t e = cudaGetDeviceProperties(&prop, device);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaGetDeviceProperties");
        if (prop.major != 10 || prop.minor != 3)
            return fail(NVFP4_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", device,
                        prop.major, prop.minor);
        st.sm_count = prop.multiProcessorCount;
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || fn == nullptr || q != cudaDriverEntryPointSuccess)
            return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
        auto encode = reinterpret_cast<EncodeTiledFn>(fn);
        int s = encode_template(encode, &st.tmpl_a, any_device_buffer, 128);
        if (s == NVFP4_OK)
            s = encode_template(encode, &st.tmpl_b128, any_device_buffer, 128);
        if (s == NVFP4_OK)
            s = encode_template(encode, &st.tmpl_b256, any_device_buffer, 256);
        if (s == NVFP4_OK)
            s = encode_sfb_template(encode, &st.tmpl_sfb, any_device_buffer);
        if (s != NVFP4_OK)
            return s;
        e = prepare_gemm_kernels(device);
        if (e != cudaSuccess)
            return cuda_fail(e, "cudaFuncSetAttribute");
        st.pairs = pair_capacity(device);
        if (st.pairs > st.sm_count / 2)
            st.pairs = st.sm_count / 2;
        st.ready = true;
    }
    *out = &st;
    return NVFP4_OK;
}

// Caller holds g_mutex. Allocates the workspace with `slots` per-CTA slots
// (prefix scratch, partial tiles) on first use for (device, stream).
int stream_workspace(int device, cudaStream_t stream, int slots, StreamWorkspace **out) {
    auto key = std::make_pair(device, stream);
    auto it = g_workspaces.find(key);
    if (it != g_workspaces.end()) {
        *out = &it->second;
        return NVFP4_OK;
    }
    void *p = nullptr;
    const size_t bytes = workspace_bytes(NVFP4_MAX_GROUPS, slots, slots, 2);
    cudaError_t e = cudaMalloc(&p, bytes);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaMalloc(workspace)");
    // header (status word, descriptor counter), descriptors, prefix scratch
    // and flags start at zero; partial tiles are written before they are read
    const size_t head = bytes - kPartialSlotBytes * (size_t)slots;
    e = cudaMemset(p, 0, head);
    if (e != cudaSuccess) {
        cudaFree(p);
        return cuda_fail(e, "cudaMemset(workspace)");
    }
    StreamWorkspace &w = g_workspaces[key];
    w.base = p;
    w.slots = slots;
    w.state = WorkspaceState();
    *out = &w;
    return NVFP4_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Bound of every wait in the GEMM kernel: NVFP4_WATCHDOG_MS milliseconds
// (fractions allowed), default 4000.
uint64_t watchdog_ns() {
    const char *s = std::getenv("NVFP4_WATCHDOG_MS");
    double ms = s ? std::strtod(s, nullptr) : 0.0;
    if (!(ms > 0.0) || ms > 3.6e6)
        ms = 4000.0;
    const double ns = ms * 1e6;
    return ns < 1.0 ? 1ull : (uint64_t)ns;
}

// BLOCK_N for a call: an explicit nvfp4_set_tile_n() value or NVFP4_TILE_N,
// else 256 (a 128 x 256 x 64 MMA does twice the work of a 128 x 128 x 64 one
// for about the same issue cost).
int choose_block_n() {
    if (g_tile_n_override == 128 || g_tile_n_override == 256)
        return g_tile_n_override;
    const char *s = std::getenv("NVFP4_TILE_N");
    if (s && std::atoi(s) == 128)
        return 128;
    return 256;
}

}  // namespace

int check_groups(int group_count, int max_groups, const nvfp4_problem_size *problem_sizes, const void *const *A,
                 const void *const *B, const void *const *SFA, const void *const *SFB, void *const *C, int block_n,
                 GroupArgs *args, long long *total_tiles) {
    *total_tiles = 0;
    if (group_count < 0)
        return fail(NVFP4_ERR_INVALID_ARG, "group_count %d < 0", group_count);
    if (group_count == 0)
        return NVFP4_OK;
    if (group_count > max_groups)
        return fail(NVFP4_ERR_INVALID_ARG, "group_count %d > %d", group_count, max_groups);
    if (!problem_sizes || !A || !B || !SFA || !SFB || !C)
        return fail(NVFP4_ERR_INVALID_ARG, "null problem_sizes or pointer array");
    long long total = 0;
    for (int g = 0; g < group_count; ++g) {
        const nvfp4_problem_size &s = problem_sizes[g];
        if (s.m < 0 || s.n < 0 || s.k < 0 || s.l < 0)
            return fail(NVFP4_ERR_INVALID_ARG, "group %d: negative size (%d, %d, %d, %d)", g, s.m, s.n, s.k, s.l);
        args[g] = GroupArgs{s.m, s.n, s.k, (uint16_t)(s.l <= kMaxBatch ? s.l : 0), 3, A[g], B[g], SFA[g], SFB[g],
                            C[g]};
        if (s.m == 0 || s.n == 0 || s.l == 0) {
            args[g].m = args[g].n = 0;  // empty: nothing is read or written
            continue;
        }
        if (s.l > kMaxBatch || (long long)s.l * s.m > 0x7fffffffLL || (long long)s.l * s.n > 0x7fffffffLL)
            return fail(NVFP4_ERR_UNSUPPORTED, "group %d: l = %d with m = %d, n = %d is too large", g, s.l, s.m,
                        s.n);
        if (s.k % 32 != 0 || s.n % 32 != 0)
            return fail(NVFP4_ERR_UNSUPPORTED, "group %d: k = %d and n = %d must be multiples of 32", g, s.k, s.n);
        if (!C[g])
            return fail(NVFP4_ERR_INVALID_ARG, "group %d: null C", g);
        if (!aligned16(C[g]))
            return fail(NVFP4_ERR_MISALIGNED, "group %d: C not 16-byte aligned", g);
        if (s.k > 0) {
            if (!A[g] || !B[g] || !SFA[g] || !SFB[g])
                return fail(NVFP4_ERR_INVALID_ARG, "group %d: null A/B/SFA/SFB", g);
            if (!aligned16(A[g]) || !aligned16(B[g]) || !aligned16(SFA[g]) || !aligned16(SFB[g]))
                return fail(NVFP4_ERR_MISALIGNED, "group %d: A/B/SFA/SFB not 16-byte aligned", g);
        }
        total += (long long)((s.m + kBlockM - 1) / kBlockM) * (long long)((s.n + block_n - 1) / block_n) * s.l;
        if (total > 0x7fffffffLL)
            return fail(NVFP4_ERR_UNSUPPORTED, "more than 2^31 - 1 tiles");
    }
    *total_tiles = total;
    return NVFP4_OK;
}

int current_block_n() { return choose_block_n(); }

// NVFP4_SPLIT forces the schedule: -1 if unset (automatic), else 0 (whole
// tiles), 1 (all tiles in the split range) or 2 (whole waves + split rest).
int split_override() {
    const char *s = std::getenv("NVFP4_SPLIT");
    if (s && *s) {
        const int v = std::atoi(s);
        return v == 1 ? 1 : (v == 2 ? 2 : 0);
    }
    return -1;
}

// NVFP4_PAIR selects a cluster kernel for calls that run whole tiles: 1 the
// CTA pair (cta_group::2 MMAs), 2 the multicast cluster, 0 neither; unset:
// the library's choice.
int pair_override() {
    const char *s = std::getenv("NVFP4_PAIR");
    if (s && *s) {
        const int v = std::atoi(s);
        return v == 1 || v == 2 ? v : 0;
    }
    return -1;
}

// Whether `stream` is capturing into a CUDA graph (the launch is then
// replayed later, possibly after other calls changed the descriptor slots).
bool capturing(cudaStream_t stream) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    return cudaStreamIsCapturing(stream, &cs) == cudaSuccess && cs != cudaStreamCaptureStatusNone;
}

int launch_on_workspace(int group_count, GroupArgs *args, long long total_tiles, int block_n, void *ws_base,
                        int capacity, int prefix_slots, int partial_slots, int regions, WorkspaceState *state,
                        cudaStream_t stream) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    // schedule units of the one-CTA tiling (128 x block_n tiles) and of the
    // CTA-pair tiling (256 x 256 tiles)
    long long total_work = 0, pair_tiles = 0, pair_work = 0;
    for (int g = 0; g < group_count; ++g) {
        const GroupArgs &a = args[g];
        if (a.m <= 0 || a.n <= 0)
            continue;
        const long long tiles =
            (long long)((a.m + kBlockM - 1) / kBlockM) * ((a.n + block_n - 1) / block_n) * (long long)a.l;
        const long long kt = (a.k + kBlockK - 1) / kBlockK;
        total_work += tiles * (kt > 1 ? kt : 1);
        const long long ptiles = (long long)((a.m + 2 * kBlockM - 1) / (2 * kBlockM)) * ((a.n + 255) / 256) * a.l;
        pair_tiles += ptiles;
        pair_work += ptiles * (kt > 1 ? kt : 1);
    }
    if (total_work > 0x7fffffffLL)
        return fail(NVFP4_ERR_UNSUPPORTED, "more than 2^31 - 1 k-tiles in one call");
    DeviceState *st = nullptr;
    GemmLaunch cfg;
    int desc_maps = 0, b_box = block_n;
    const bool graph = capturing(stream);
    // One lock over set-up, launch and bookkeeping: calls that share a
    // workspace must reach the GPU in the order their descriptor-cache
    // updates were taken.
    std::lock_guard<std::mutex> lock(g_mutex);
    {
        int s = device_state(device, ws_base, &st);
        if (s != NVFP4_OK)
            return s;
        const int sms = st->sm_count;
        int forced = split_override();
        if (partial_slots < sms)
            forced = 0;  // no partial-tile slots: whole tiles only
        const int split_tile = choose_split_tile((int)total_tiles, sms, forced);
        cfg.split = split_tile < total_tiles ? 1 : 0;
        cfg.split_tile = split_tile;
        if (!cfg.split)
            cfg.grid = (int)(total_tiles < sms ? total_tiles : sms);
        else if (split_tile == 0)
            cfg.grid = (int)(total_work < sms ? total_work : sms);
        else
            cfg.grid = sms;  // whole waves use every SM
        // Clusters of two (256 x 256 tiles, whole tiles only): when selected
        // with NVFP4_PAIR, and not with a split schedule forced.
        const int pmode = pair_override();
        cfg.cluster = (block_n == 256 && st->pairs > 0 && pmode > 0 && pair_work <= 0x7fffffffLL && forced <= 0)
                          ? pmode
                          : 0;
        if (cfg.cluster) {
            cfg.split = 0;
            cfg.split_tile = (int)pair_tiles;
            cfg.grid = 2 * (int)(pair_tiles < st->pairs ? pair_tiles : st->pairs);
            total_tiles = pair_tiles;
            total_work = pair_work;
        }
        cfg.pair_launch = cfg.cluster == 0 && cfg.grid % 2 == 0 && cfg.grid / 2 <= st->pairs;
        if (group_count > kMediumGroups && prefix_slots < cfg.grid)
            return fail(NVFP4_ERR_UNSUPPORTED, "workspace has %d CTA slots, the launch needs %d", prefix_slots,
                        cfg.grid);
        // rows of B per TMA box: a CTA of a pair loads half of a 256-row tile
        b_box = cfg.cluster == 1 ? 128 : block_n;
        // Descriptors to patch: those whose region-0 slot does not already
        // hold this group's pointer and shape (region 0 is written only by
        // this workspace's eager calls, in stream order). A captured launch
        // runs whenever it is replayed: it uses region 1 (when the workspace
        // has one, else region 0 with the cache dropped) and patches every
        // slot it uses.
        if (state->descs.size() < kDescPerGroup * (size_t)capacity || (graph && regions < 2))
            state->descs.assign(kDescPerGroup * (size_t)capacity, DescKey());
        desc_maps = 0;
        for (int g = 0; g < group_count; ++g) {
            GroupArgs &a = args[g];
            a.patch = 0;
            if (a.m <= 0 || a.n <= 0 || a.k <= 0)
                continue;
            const DescKey ka{a.a, (int32_t)a.l * a.m, a.k, kBlockM}, kb{a.b, (int32_t)a.l * a.n, a.k, b_box},
                ks{a.sfb, (int32_t)a.l * ((a.n + kBlockM - 1) / kBlockM), a.k, 2};
            if (graph || !(state->descs[kDescPerGroup * g] == ka)) {
                a.patch |= 1;
                ++desc_maps;
            }
            if (graph || !(state->descs[kDescPerGroup * g + 1] == kb)) {
                a.patch |= 2;
                ++desc_maps;
            }
            if (graph || !(state->descs[kDescPerGroup * g + 2] == ks)) {
                a.patch |= 4;
                ++desc_maps;
            }
        }
    }
    cfg.block_n = block_n;
    cfg.group_count = group_count;
    cfg.desc_maps = desc_maps;
    cfg.total_tiles = (int)total_tiles;
    cfg.total_work = (int)total_work;
    cfg.capacity = capacity;
    cfg.timeout_ns = watchdog_ns();
    cfg.device_table = false;
    cfg.dt = DeviceTable{};
    WorkspaceView ws = workspace_view(ws_base, capacity, prefix_slots, partial_slots, regions);
    if (graph && regions > 1)
        ws = second_region(ws);
    const void *tmpl_b = b_box == 256 ? (const void *)&st->tmpl_b256 : (const void *)&st->tmpl_b128;
    e = launch_grouped(cfg, args, ws, &st->tmpl_a, tmpl_b, &st->tmpl_sfb, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "grouped GEMM launch");  // nothing ran, no slot was written
    if (graph)
        return NVFP4_OK;
    for (int g = 0; g < group_count; ++g) {
        const GroupArgs &a = args[g];
        if (a.patch & 1)
            state->descs[kDescPerGroup * g] = DescKey{a.a, (int32_t)a.l * a.m, a.k, kBlockM};
        if (a.patch & 2)
            state->descs[kDescPerGroup * g + 1] = DescKey{a.b, (int32_t)a.l * a.n, a.k, b_box};
        if (a.patch & 4)
            state->descs[kDescPerGroup * g + 2] =
                DescKey{a.sfb, (int32_t)a.l * ((a.n + kBlockM - 1) / kBlockM), a.k, 2};
    }
    return NVFP4_OK;
}

int launch_device_table(int group_count, const DeviceTable &dt, int block_n, void *ws_base, int capacity,
                        int slots, WorkspaceState *state, cudaStream_t stream) {
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState *st = nullptr;
    int s = device_state(device, ws_base, &st);
    if (s != NVFP4_OK)
        return s;
    GemmLaunch cfg;
    cfg.block_n = block_n;
    cfg.group_count = group_count;
    cfg.desc_maps = kDescPerGroup * group_count;  // every group's slots are rewritten
    cfg.total_tiles = 0;              // derived by the kernel
    cfg.total_work = 0;
    cfg.grid = st->sm_count < slots ? st->sm_count : slots;
    cfg.split = split_override();  // the kernel chooses with the same rule
    cfg.split_tile = 0;
    cfg.capacity = capacity;
    cfg.timeout_ns = watchdog_ns();
    cfg.device_table = true;
    cfg.cluster = 0;
    cfg.pair_launch = cfg.grid % 2 == 0 && cfg.grid / 2 <= st->pairs;
    cfg.dt = dt;
    (void)state;  // region 0 and its host cache are left alone
    const WorkspaceView ws = second_region(workspace_view(ws_base, capacity, slots, slots, 2));
    const void *tmpl_b = block_n == 256 ? (const void *)&st->tmpl_b256 : (const void *)&st->tmpl_b128;
    e = launch_grouped(cfg, nullptr, ws, &st->tmpl_a, tmpl_b, &st->tmpl_sfb, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "grouped GEMM launch");
    return NVFP4_OK;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

const char *nvfp4_status_string(int status) {
    switch (status) {
    case NVFP4_OK: return "NVFP4_OK";
    case NVFP4_ERR_INVALID_ARG: return "NVFP4_ERR_INVALID_ARG";
    case NVFP4_ERR_UNSUPPORTED: return "NVFP4_ERR_UNSUPPORTED";
    case NVFP4_ERR_MISALIGNED: return "NVFP4_ERR_MISALIGNED";
    case NVFP4_ERR_CUDA: return "NVFP4_ERR_CUDA";
    case NVFP4_ERR_TIMEOUT: return "NVFP4_ERR_TIMEOUT";
    default: return "NVFP4_ERR_UNKNOWN";
    }
}

const char *nvfp4_last_error_message(void) { return g_last_error; }

size_t nvfp4_scale_bytes(int rows, int k) {
    if (rows <= 0 || k <= 0)
        return 0;
    return (size_t)((rows + 127) / 128) * 128u * (size_t)((k + 63) / 64) * 4u;
}

int nvfp4_set_tile_n(int block_n) {
    if (block_n != 0 && block_n != 128 && block_n != 256)
        return fail(NVFP4_ERR_INVALID_ARG, "tile N must be 0 (automatic), 128 or 256, got %d", block_n);
    std::lock_guard<std::mutex> lock(g_mutex);
    g_tile_n_override = block_n;
    return NVFP4_OK;
}

int nvfp4_grouped_gemm(int group_count, const nvfp4_problem_size *problem_sizes, const void *const *A,
                       const void *const *B, const void *const *SFA, const void *const *SFB, void *const *C,
                       nvfp4_stream_t stream) {
    const int block_n = choose_block_n();
    GroupArgs args[NVFP4_MAX_GROUPS];
    long long total = 0;
    int s = check_groups(group_count, NVFP4_MAX_GROUPS, problem_sizes, A, B, SFA, SFB, C, block_n, args, &total);
    if (s != NVFP4_OK || total == 0)
        return s;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    StreamWorkspace *w = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        s = stream_workspace(device, reinterpret_cast<cudaStream_t>(stream), sms, &w);
        if (s != NVFP4_OK)
            return s;
    }
    return launch_on_workspace(group_count, args, total, block_n, w->base, NVFP4_MAX_GROUPS, w->slots, w->slots, 2,
                               &w->state, reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_grouped_gemm_batched(int problem_count, const int *group_counts, const nvfp4_problem_size *problem_sizes,
                               const void *const *A, const void *const *B, const void *const *SFA,
                               const void *const *SFB, void *const *C, nvfp4_stream_t stream) {
    if (problem_count < 0)
        return fail(NVFP4_ERR_INVALID_ARG, "problem_count %d < 0", problem_count);
    if (problem_count == 0)
        return NVFP4_OK;
    if (!group_counts)
        return fail(NVFP4_ERR_INVALID_ARG, "null group_counts");
    long long total = 0;
    for (int p = 0; p < problem_count; ++p) {
        if (group_counts[p] < 0)
            return fail(NVFP4_ERR_INVALID_ARG, "problem %d: group count %d < 0", p, group_counts[p]);
        total += group_counts[p];
    }
    if (total > NVFP4_MAX_GROUPS)
        return fail(NVFP4_ERR_INVALID_ARG, "%lld groups in all; at most %d fit one launch", total, NVFP4_MAX_GROUPS);
    return nvfp4_grouped_gemm((int)total, problem_sizes, A, B, SFA, SFB, C, stream);
}

int nvfp4_grouped_gemm_device(int group_count, const nvfp4_problem_size *problem_sizes, const void *const *A,
                              const void *const *B, const void *const *SFA, const void *const *SFB, void *const *C,
                              nvfp4_stream_t stream) {
    if (group_count < 0)
        return fail(NVFP4_ERR_INVALID_ARG, "group_count %d < 0", group_count);
    if (group_count == 0)
        return NVFP4_OK;
    if (group_count > NVFP4_MAX_GROUPS)
        return fail(NVFP4_ERR_INVALID_ARG, "group_count %d > %d", group_count, NVFP4_MAX_GROUPS);
    if (!problem_sizes || !A || !B || !SFA || !SFB || !C)
        return fail(NVFP4_ERR_INVALID_ARG, "null problem_sizes or pointer array");
    if (!aligned16(problem_sizes))
        return fail(NVFP4_ERR_MISALIGNED, "problem_sizes not 16-byte aligned");
    const void *arrays[5] = {A, B, SFA, SFB, C};
    for (const void *q : arrays)
        if ((reinterpret_cast<uintptr_t>(q) & 7u) != 0)
            return fail(NVFP4_ERR_MISALIGNED, "pointer array not 8-byte aligned");
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaDeviceGetAttribute");
    StreamWorkspace *w = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        int s = stream_workspace(device, reinterpret_cast<cudaStream_t>(stream), sms, &w);
        if (s != NVFP4_OK)
            return s;
    }
    const DeviceTable dt{problem_sizes, A, B, SFA, SFB, C};
    return launch_device_table(group_count, dt, choose_block_n(), w->base, NVFP4_MAX_GROUPS, w->slots, &w->state,
                               reinterpret_cast<cudaStream_t>(stream));
}

int nvfp4_pack_scales(const void *sf_rowmajor, int rows, int k, void *sf_atoms, nvfp4_stream_t stream) {
    if (rows < 0 || k < 0)
        return fail(NVFP4_ERR_INVALID_ARG, "negative rows (%d) or k (%d)", rows, k);
    if (k % 16 != 0)
        return fail(NVFP4_ERR_UNSUPPORTED, "k = %d is not a multiple of 16", k);
    if (rows == 0 || k == 0)
        return NVFP4_OK;
    if (!sf_rowmajor || !sf_atoms)
        return fail(NVFP4_ERR_INVALID_ARG, "null scale pointer");
    if (!aligned16(sf_atoms))
        return fail(NVFP4_ERR_MISALIGNED, "sf_atoms not 16-byte aligned");
    cudaError_t e = launch_pack_scales(static_cast<const uint8_t *>(sf_rowmajor), rows, k,
                                       static_cast<uint8_t *>(sf_atoms), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "scale packer launch");
    return NVFP4_OK;
}

int nvfp4_pack_scales_batched(int count, const void *const *sf_rowmajor, const int *rows, const int *k,
                              void *const *sf_atoms, nvfp4_stream_t stream) {
    if (count < 0 || count > NVFP4_PACK_MAX_BATCH)
        return fail(NVFP4_ERR_INVALID_ARG, "count = %d outside [0, %d]", count, NVFP4_PACK_MAX_BATCH);
    if (count == 0)
        return NVFP4_OK;
    if (!sf_rowmajor || !rows || !k || !sf_atoms)
        return fail(NVFP4_ERR_INVALID_ARG, "null array");
    std::vector<const uint8_t *> src;
    std::vector<uint8_t *> dst;
    std::vector<int> rs, ks;
    for (int i = 0; i < count; ++i) {
        if (rows[i] < 0 || k[i] < 0)
            return fail(NVFP4_ERR_INVALID_ARG, "entry %d: negative rows (%d) or k (%d)", i, rows[i], k[i]);
        if (k[i] % 16 != 0)
            return fail(NVFP4_ERR_UNSUPPORTED, "entry %d: k = %d is not a multiple of 16", i, k[i]);
        if (rows[i] == 0 || k[i] == 0)
            continue;
        if (!sf_rowmajor[i] || !sf_atoms[i])
            return fail(NVFP4_ERR_INVALID_ARG, "entry %d: null scale pointer", i);
        if (!aligned16(sf_atoms[i]))
            return fail(NVFP4_ERR_MISALIGNED, "entry %d: sf_atoms not 16-byte aligned", i);
        src.push_back(static_cast<const uint8_t *>(sf_rowmajor[i]));
        dst.push_back(static_cast<uint8_t *>(sf_atoms[i]));
        rs.push_back(rows[i]);
        ks.push_back(k[i]);
    }
    cudaError_t e = launch_pack_scales_batched((int)src.size(), src.data(), rs.data(), ks.data(), dst.data(),
                                               reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "batched scale packer launch");
    return NVFP4_OK;
}

int nvfp4_quantize_pack(const void *x, int x_dtype, int rows, int k, void *codes, void *sf_atoms,
                        nvfp4_stream_t stream) {
    if (rows < 0 || k < 0)
        return fail(NVFP4_ERR_INVALID_ARG, "negative rows (%d) or k (%d)", rows, k);
    if (x_dtype != NVFP4_DTYPE_BF16 && x_dtype != NVFP4_DTYPE_F16)
        return fail(NVFP4_ERR_INVALID_ARG, "x_dtype %d is neither NVFP4_DTYPE_BF16 nor NVFP4_DTYPE_F16", x_dtype);
    if (k % 16 != 0)
        return fail(NVFP4_ERR_UNSUPPORTED, "k = %d is not a multiple of 16", k);
    if (rows > 65535 * 128)
        return fail(NVFP4_ERR_UNSUPPORTED, "rows = %d exceeds %d", rows, 65535 * 128);
    if (rows == 0 || k == 0)
        return NVFP4_OK;
    if (!x || !codes || !sf_atoms)
        return fail(NVFP4_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(x) || !aligned16(codes) || !aligned16(sf_atoms))
        return fail(NVFP4_ERR_MISALIGNED, "x, codes and sf_atoms must be 16-byte aligned");
    cudaError_t e = launch_quantize_pack(x, x_dtype == NVFP4_DTYPE_BF16, rows, k, codes, sf_atoms,
                                         reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "quantise-and-pack launch");
    return NVFP4_OK;
}

int nvfp4_device_status(nvfp4_stream_t stream, int *status) {
    if (!status)
        return fail(NVFP4_ERR_INVALID_ARG, "null status");
    *status = NVFP4_OK;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaGetDevice");
    // The status words to read: the (device, stream) workspace's, and the
    // static array of nvfp4_grouped_gemm_noalloc (one per device, shared by
    // every stream) once a call has set it up.
    uint32_t *words[2] = {nullptr, nullptr};
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        auto it = g_workspaces.find(std::make_pair(device, reinterpret_cast<cudaStream_t>(stream)));
        if (it != g_workspaces.end())
            words[0] = workspace_view(it->second.base, NVFP4_MAX_GROUPS).status;
    }
    if (void *na = noalloc_workspace_if_ready(device))
        words[1] = workspace_view(na, NVFP4_NOALLOC_MAX_GROUPS).status;
    uint32_t word = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    for (uint32_t *w : words) {
        if (!w)
            continue;
        uint32_t v = 0;
        e = cudaMemcpyAsync(&v, w, sizeof(v), cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess)
            e = cudaStreamSynchronize(s);
        if (e == cudaSuccess && v != 0) {
            e = cudaMemsetAsync(w, 0, sizeof(v), s);
            if (e == cudaSuccess)
                e = cudaStreamSynchronize(s);
        }
        if (e != cudaSuccess)
            return cuda_fail(e, "reading the device status word");
        word |= v;
    }
    if (word & kStatusTimeoutMask) {
        *status = NVFP4_ERR_TIMEOUT;
        fail(NVFP4_ERR_TIMEOUT,
             "a bounded wait gave up (status bits 0x%x: 1 producer, 2 MMA, 4 epilogue, 8 partial tile, 16 descriptors)",
             word);
    } else if (word & kStatusBadGroup) {
        *status = NVFP4_ERR_INVALID_ARG;
        fail(NVFP4_ERR_INVALID_ARG, "a device-table call skipped a group that breaks the group rules");
    }
    return NVFP4_OK;
}

}  // extern "C"
