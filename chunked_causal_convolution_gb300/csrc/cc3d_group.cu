// cc3d_group.cu -- layer groups run frame batch by frame batch ("SwiftVR Inference Optimization"
// (LightX2V blog), section "ReAE Frame Batching": a small batch of frames passes through a whole
// group of consecutive layers before the next batch starts, so only that batch's intermediate
// features are held, and the group's last layer writes into one output buffer; layers with a
// temporal history keep their state rules).
//
// Host code only: every step runs in the kernels of the plans' own launches.  For batch j of a
// chunk and layer l, the layer reads batch j's frames (the chunk's input for l = 0, the previous
// layer's batch otherwise), its history is the one it left after batch j - 1 (cache_in for the
// first batch), and it writes the next layer's batch into the caller's workspace (the group's
// output y for the last layer).  A layer's histories alternate between cache_out and one buffer in
// the workspace, arranged so that the last batch leaves it in cache_out.  The library's result does
// not depend on how frames are grouped into launches, so the output equals the layer-by-layer
// chunk loop bit for bit.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "cc3d.h"
#include "cc3d_internal.h"

using namespace cc3d;

// Workspace for cc3d_group_forward_chunk_static: a fixed array in device memory that exists on
// every GPU where this library's device code is loaded, so that callers who cannot allocate device
// memory still get frame batching.  In host code the name is only a stand-in, not a device
// address: static_scratch() below looks the address up once per device, with that device current.
static constexpr size_t kStaticScratchBytes = CC3D_GROUP_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_group_scratch[kStaticScratchBytes];

struct cc3d_group_s {
    std::vector<cc3d_plan_t> plans;
    std::vector<PlanShape> shapes;
    int frame_batch = 0;  // 0: the whole chunk in one batch
};

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t n) { return (n + kAlign - 1) & ~(kAlign - 1); }

size_t frame_in_bytes(const PlanShape& s) { return (size_t)s.H * s.W * s.Cin * s.esize; }
size_t frame_out_bytes(const PlanShape& s) { return (size_t)s.Ho * s.Wo * s.Cout * s.esize; }

int batch_frames(const cc3d_group_s& g, int T) { return g.frame_batch == 0 ? T : (T < g.frame_batch ? T : g.frame_batch); }
int batches(const cc3d_group_s& g, int T)
{
    if (T == 0) return 0;
    const int fb = batch_frames(g, T);
    return (T + fb - 1) / fb;
}

// Workspace layout for a chunk of T frames: two buffers for the intermediate batches between
// consecutive layers, then (when the chunk takes more than one batch) one history buffer per layer
// with a history.
struct Layout {
    std::vector<size_t> act;   // offset of layer l's output batch (l < nlayers - 1)
    std::vector<size_t> hist;  // offset of layer l's second history buffer, or SIZE_MAX
    size_t bytes = 0;
};

Layout layout(const cc3d_group_s& g, int T)
{
    Layout L;
    const int n = (int)g.plans.size();
    const int fb = batch_frames(g, T);
    // the intermediate batches alternate between two buffers: layer l writes buffer l % 2 while it
    // reads buffer (l - 1) % 2, each buffer as large as the largest batch it holds
    size_t side[2] = {0, 0};
    for (int l = 0; l + 1 < n; ++l) {
        const size_t need = round_up((size_t)fb * frame_out_bytes(g.shapes[l]));
        if (need > side[l % 2]) side[l % 2] = need;
    }
    for (int l = 0; l + 1 < n; ++l) L.act.push_back(l % 2 == 0 ? 0 : side[0]);
    size_t off = side[0] + side[1];
    const bool ping_pong = batches(g, T) > 1;
    for (int l = 0; l < n; ++l) {
        const int P = g.shapes[l].kt - 1;
        if (ping_pong && P > 0) {
            L.hist.push_back(off);
            off += round_up((size_t)P * frame_in_bytes(g.shapes[l]));
        } else {
            L.hist.push_back(SIZE_MAX);
        }
    }
    L.bytes = off;
    return L;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxScratchDevices] = {};

// The device address of g_group_scratch on the current device (looked up on the first call there).
cc3d_status static_scratch(void** out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) {
        cudaGetLastError();
        return CC3D_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_group_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return CC3D_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return CC3D_OK;
}

}  // namespace

extern "C" {

cc3d_status cc3d_group_create(int nlayers, const cc3d_plan_t* plans, int frame_batch, cc3d_group_t* out)
{
    if (out == nullptr) return CC3D_ERR_INVALID_ARG;
    *out = nullptr;
    if (nlayers < 1 || nlayers > 64 || plans == nullptr || frame_batch < 0) return CC3D_ERR_INVALID_ARG;
    cc3d_group_s* g = new (std::nothrow) cc3d_group_s;
    if (g == nullptr) return CC3D_ERR_OOM;
    try {
        for (int l = 0; l < nlayers; ++l) {
            PlanShape s;
            if (!plan_shape(plans[l], &s)) {
                delete g;
                return CC3D_ERR_INVALID_ARG;
            }
            if (l > 0) {
                const PlanShape& p = g->shapes.back();
                if (s.Cin != p.Cout || s.H != p.Ho || s.W != p.Wo || s.esize != p.esize) {
                    delete g;
                    return CC3D_ERR_INVALID_ARG;
                }
            }
            g->plans.push_back(plans[l]);
            g->shapes.push_back(s);
        }
    } catch (...) {
        delete g;
        return CC3D_ERR_OOM;
    }
    g->frame_batch = frame_batch;
    *out = g;
    return CC3D_OK;
}

void cc3d_group_destroy(cc3d_group_t g) { delete g; }

cc3d_status cc3d_group_workspace_bytes(cc3d_group_t g, int T_max, size_t* bytes)
{
    if (g == nullptr || T_max < 0 || bytes == nullptr) return CC3D_ERR_INVALID_ARG;
    *bytes = layout(*g, T_max).bytes;
    return CC3D_OK;
}

cc3d_status cc3d_group_forward_chunk(cc3d_group_t g, int T, const void* x, const void* const* w, const void* const* b,
                                     const void* const* cache_in, void* const* cache_out, void* y, void* workspace,
                                     size_t workspace_bytes, void* stream)
{
    if (g == nullptr || T < 0 || w == nullptr) return CC3D_ERR_INVALID_ARG;
    const int n = (int)g->plans.size();
    bool any_history = false;
    for (int l = 0; l < n; ++l) any_history |= g->shapes[l].kt > 1;
    if (any_history && cache_out == nullptr) return CC3D_ERR_INVALID_ARG;
    const Layout L = layout(*g, T);
    if (L.bytes > 0 && (workspace == nullptr || workspace_bytes < L.bytes)) return CC3D_ERR_INVALID_ARG;
    if (L.bytes > 0 && (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return CC3D_ERR_ALIGNMENT;
    // the workspace is the group's own: it must not overlap anything the caller passes
    const PlanShape& s0 = g->shapes[0];
    const PlanShape& sl = g->shapes[n - 1];
    if (T > 0 && (overlaps(workspace, L.bytes, x, (size_t)T * frame_in_bytes(s0)) ||
                  overlaps(workspace, L.bytes, y, (size_t)T * frame_out_bytes(sl))))
        return CC3D_ERR_ALIAS;
    for (int l = 0; l < n; ++l) {
        const PlanShape& s = g->shapes[l];
        const size_t nh = (size_t)(s.kt - 1) * frame_in_bytes(s);
        const size_t nw = (size_t)s.Cout * s.kt * s.kh * s.kw * s.Cin * s.esize;
        if (overlaps(workspace, L.bytes, cache_in ? cache_in[l] : nullptr, nh) ||
            overlaps(workspace, L.bytes, cache_out ? cache_out[l] : nullptr, nh) ||
            overlaps(workspace, L.bytes, w[l], nw))
            return CC3D_ERR_ALIAS;
    }
    char* ws = static_cast<char*>(workspace);
    const int fb = batch_frames(*g, T);
    const int nb = batches(*g, T);
    // pass 0 checks every launch of the chunk (nothing is launched if one fails), pass 1 launches
    for (int pass = 0; pass < 2; ++pass) {
        const bool dry = pass == 0;
        if (T == 0) {
            for (int l = 0; l < n; ++l) {
                const cc3d_status st = forward_impl(g->plans[l], 0, nullptr, w[l], b ? b[l] : nullptr, nullptr,
                                                    cache_in ? cache_in[l] : nullptr,
                                                    cache_out ? cache_out[l] : nullptr, nullptr, stream, false, dry);
                if (st != CC3D_OK) return st;
            }
            continue;
        }
        for (int j = 0; j < nb; ++j) {
            const int t0 = j * fb;
            const int c = (T - t0) < fb ? (T - t0) : fb;
            const void* in = static_cast<const char*>(x) + (size_t)t0 * frame_in_bytes(s0);
            for (int l = 0; l < n; ++l) {
                const PlanShape& s = g->shapes[l];
                void* out = (l == n - 1) ? static_cast<void*>(static_cast<char*>(y) + (size_t)t0 * frame_out_bytes(sl))
                                         : static_cast<void*>(ws + L.act[l]);
                const void* hin = nullptr;
                void* hout = nullptr;
                if (s.kt > 1) {
                    // batch j writes cache_out when nb - 1 - j is even, the workspace buffer otherwise,
                    // so the histories alternate and the last batch leaves the layer's in cache_out
                    void* mine[2] = {cache_out[l], L.hist[l] == SIZE_MAX ? nullptr : ws + L.hist[l]};
                    hout = mine[(nb - 1 - j) % 2];
                    hin = j == 0 ? (cache_in ? cache_in[l] : nullptr) : mine[(nb - j) % 2];
                }
                const cc3d_status st = forward_impl(g->plans[l], c, in, w[l], b ? b[l] : nullptr, nullptr, hin, hout,
                                                    out, stream, false, dry);
                if (st != CC3D_OK) return st;
                in = out;
            }
        }
    }
    return CC3D_OK;
}

cc3d_status cc3d_group_forward_chunk_static(cc3d_group_t g, int T, const void* x, const void* const* w,
                                            const void* const* b, const void* const* cache_in, void* const* cache_out,
                                            void* y, void* stream)
{
    if (g == nullptr || T < 0) return CC3D_ERR_INVALID_ARG;
    // the first call on a device looks up the array's address there
    void* scratch = nullptr;
    const cc3d_status st = static_scratch(&scratch);
    if (st != CC3D_OK) return st;
    // nothing in the array has to start at zero: every intermediate batch and history the chunk
    // reads from it is written earlier in the same chunk, so the previous call's contents never
    // matter
    if (layout(*g, T).bytes > kStaticScratchBytes) return CC3D_ERR_SCRATCH_TOO_SMALL;
    return cc3d_group_forward_chunk(g, T, x, w, b, cache_in, cache_out, y, scratch, kStaticScratchBytes, stream);
}

}  // extern "C"
