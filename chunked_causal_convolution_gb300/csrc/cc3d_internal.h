// cc3d_internal.h -- launch descriptors shared between the C-ABI layer and the kernels.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "cc3d.h"

namespace cc3d {

// Device status word bits (or-ed by kernels, read and cleared by cc3d_get_status).
enum : unsigned {
    STATUS_TIMEOUT_LOADER = 1u << 0,
    STATUS_TIMEOUT_MMA = 1u << 1,
    STATUS_TIMEOUT_EPILOGUE = 1u << 2,
    STATUS_TIMEOUT_DRAIN = 1u << 3,
    STATUS_TIMEOUT_COPY = 1u << 4,
};

// Geometry of the tensor-core kernel's tiles.
//
// The frame is cut into column blocks of S pixels.  Inside a column block the
// pixels are numbered in a "padded flat" order f = h * Sp + j with Sp = S + 2:
// j = 0 and j = S + 1 are the zero columns left and right of the block, so
// every spatial tap (dh, dw) of every output position f reads the input at
// f + (dh - 1) * Sp + (dw - 1) -- a pure shift (1x1 spatial kernels read f itself).  A tile is SUB groups of 128
// consecutive output positions (one MMA row block each); in row-aligned mode
// (S == 128) each group is exactly one row segment, otherwise groups are
// consecutive 128-blocks of f and the positions on padding columns or beyond
// the last row are computed but not stored.
struct TcGeometry {
    int S, Sp, ncolblk;
    int halo;           // (ks - 1) / 2: spatial taps reach this far from the output position
    int row_aligned;
    int sub;            // 128-row groups per tile
    int sub_stride;     // f distance between groups (Sp or 128)
    int tile_f;         // f distance between consecutive tiles of a column block
    int tiles_per_cb;   // tiles per (frame, column block)
    int nrows;          // padded rows loaded per input window
};

struct TcLaunch {
    // tensor maps (encoded on the host)
    CUtensorMap map_x;      // x_chunk   [T][H][W][Cin]   box (CB, Sp, nrows, 1)
    CUtensorMap map_cache;  // cache_in  [P][H][W][Cin]   same box (unused if no cache)
    CUtensorMap map_w;      // w viewed as (Cin, Cout, taps) box (CB, NT, ks * rb)
    CUtensorMap map_w2;     // two-frame SM-pair schedule: the same view, box (CB, Cout, ks)
    int T, H, W, Cin, Cout;
    int kt, ks;             // temporal extent (1..3) and spatial extent kh = kw (1 or 3)
    int up2;                // nearest-2x upsampling fused: H x W source frames, 2H x 2W outputs
    int NT, nsplit, acc_stages;
    int ncoblk;                       // output-channel blocks handled by separate tiles
    int na, nb;                       // A / B ring stages
    int prefetch;                     // temporal taps of the next tile warmed in L2 (0..3)
    int issuers;                      // MMA-issuing warps (1 or 2)
    int rb;                           // kernel rows (of ks taps) per B stage: 1 or 3 (1 when ks == 1)
    int pair;                         // 1: SM-pair kernel (cta_group::2), weight rows split in two
    int tstack;                       // 1: SM pairs with two output frames stacked into N per MMA
    // one-SM kernel work units: units [0, nfull) are whole tiles; the rest split tiles nfull, ...
    // into their two 128-row groups, two units per tile, each computed by both MMA warps (one half
    // of the output channels each), so that a short last wave spreads over all blocks (nunits =
    // tiles when nothing is split)
    int nfull, nunits;
    int v32;                          // y and the residual are 32-byte aligned: 32-byte epilogue accesses
    int split_n;                      // with 2 issuers: split by N slice (else by 128-row group)
    int a_stage_bytes, b_stage_bytes;
    int tmem_cols;                    // allocated columns (power of two)
    TcGeometry g;
    int has_cache;
    const void* bias;                 // bf16 [Cout] or null
    const void* res;                  // bf16 [T][H][W][Cout] or null
    void* y;                          // bf16 [T][H][W][Cout]
    // temporal cache update: history slots hist_from .. P-1 are copied by otherwise idle warps
    // when copy_hist is set, the slots before hist_from by a copy engine beside the kernel
    int copy_hist;
    int hist_from;
    const void* x;
    const void* cache_in;
    void* cache_out;
    unsigned* status;
    unsigned long long wait_ns;
    int fault;
    int grid;
    size_t smem_bytes;
};

// Schedule overrides of one plan (cc3d_debug_set_schedule): one value per CC3D_SCHED_* knob of
// cc3d.h, -1 = the measured default.  They change how the work is tiled, never the result.
constexpr int kMaxRingStages = 8;  // deepest window / weight ring of the tensor-core kernels
constexpr int kMaxAccStages = 2;   // accumulator buffers in tensor memory
struct TcOverrides {
    int v[CC3D_SCHED_COUNT];
    int get(int knob, int dflt) const { return v[knob] >= 0 ? v[knob] : dflt; }
};

// Pick tiles / pipeline depths for a tensor-core launch.  Returns false if the
// shape has no configuration.  ov may be null (every knob at its default).
bool tc_configure(int CB, int T, int H, int W, int Cin, int Cout, int kt, int ks, bool has_residual, bool up2,
                  const TcOverrides* ov, TcLaunch* L);
cudaError_t tc_launch(int CB, const TcLaunch& L, cudaStream_t stream);
cudaError_t tc2_launch(int CB, const TcLaunch& L, cudaStream_t stream);
cudaError_t tc2s_launch(int CB, const TcLaunch& L, cudaStream_t stream);

// Narrow-output kernel (Cout <= 5): the nine spatial taps stacked into N, rows streamed once.
struct HeadLaunch {
    CUtensorMap map_x;          // x_chunk   [T][H][W][Cin]  box (32, 128, 1, 1)
    CUtensorMap map_cache;      // cache_in  [2][H][W][Cin]  same box (unused if no cache)
    CUtensorMap map_w;          // w viewed as (Cin, Cout, 27 taps)  box (32, Cout, 9)
    CUtensorMap map_cache_out;  // cache_out [2][H][W][Cin]  box (32, 120, 1, 1), stored from shared memory
    int T, H, W, Cin, Cout;
    int gmax;               // output frames per pass over the rows
    int ncolblk;            // column strips of 126 output pixels
    long long units;        // (frame group, strip, output row) units, dealt out in equal runs
    int nstages;            // input-row stages in shared memory
    int w_bytes, x_stage_bytes;
    int tmem_cols;
    int has_cache;
    const void* bias;       // bf16 [Cout] or null
    const void* res;        // bf16 [T][H][W][Cout] or null
    void* y;                // bf16 [T][H][W][Cout], or uint8 when out_u8
    int out_u8;             // store clamp(round((y + 1) * 127.5), 0, 255) of the bf16 output instead
    const void* x;
    const void* cache_in;
    void* cache_out;
    unsigned* status;
    unsigned long long wait_ns;
    int fault;
    int grid;
    size_t smem_bytes;
};
bool head_configure(int T, int H, int W, int Cin, int Cout, int sms, HeadLaunch* L);
cudaError_t head_launch(const HeadLaunch& L, cudaStream_t stream);

// Streaming kernel for 1x1 spatial kernels (kt x 1 x 1): frames as [H*W][Cin] matrices.
struct StreamLaunch {
    CUtensorMap map_x;          // x_chunk   viewed as (Cin, H*W, T)  box (32, 128, 1)
    CUtensorMap map_cache;      // cache_in  viewed as (Cin, H*W, P)  same box (unused if no cache)
    CUtensorMap map_w;          // w         viewed as (Cin, Cout, kt)  box (32, Cout, 1)
    CUtensorMap map_cache_out;  // cache_out viewed as (Cin, H*W, P)  box (32, 128, 1), stored from shared memory
    int T, H, W, Cin, Cout, kt;
    int gmax;                   // output frames per unit (tensor-memory slots of Cout columns)
    int npb;                    // 128-position blocks per frame
    long long units;            // (frame group, position block) units, dealt out in equal runs
    int nstages, w_bytes, x_stage_bytes, tmem_cols;
    int has_cache;
    const void* bias;           // bf16 [Cout] or null
    const void* res;            // bf16 [T][H][W][Cout] or null
    void* y;                    // bf16 [T][H][W][Cout]
    int v32;                    // y and the residual 32-byte aligned: 32-byte epilogue accesses
    unsigned* status;
    unsigned long long wait_ns;
    int fault;
    int grid;
    size_t smem_bytes;
};
bool stream_configure(int T, int H, int W, int Cin, int Cout, int kt, int sms, StreamLaunch* L);
cudaError_t stream_launch(const StreamLaunch& L, cudaStream_t stream);

// fp32 direct kernel (CUDA cores, fixed accumulation order).
struct SimtLaunch {
    int T, H, W, Cin, Cout, kt, kh, kw;
    const float* x;
    const float* cache_in;
    const float* w;
    const float* bias;
    const float* res;
    float* y;
};
cudaError_t simt_f32_launch(const SimtLaunch& L, cudaStream_t stream);

// cache_out[j] = frame (T + j) of concat(cache_in or zeros, x), j < P; plain 16-byte copies.
cudaError_t cache_update_launch(const void* x, const void* cache_in, void* cache_out, int T, int P,
                                size_t frame_bytes, cudaStream_t stream);
cudaError_t zero_fill_launch(void* p, size_t bytes, cudaStream_t stream);

// One chunk of a plan (cc3d_forward_chunk, or cc3d_forward_chunk_u8 with out_u8).  With dry_run
// every check of the call runs (arguments, device, launch configuration) and nothing is launched.
cc3d_status forward_impl(cc3d_plan_t plan, int T, const void* x, const void* w, const void* b, const void* res,
                         const void* cache_in, void* cache_out, void* y, void* stream, bool out_u8, bool dry_run);

// A plan's shape, for the layer-group runtime (cc3d_group_*): input frames H x W x Cin, output
// frames Ho x Wo x Cout, the kernel extent and the element size.
struct PlanShape {
    int Cin, Cout, H, W, Ho, Wo, kt, kh, kw, esize;
};
bool plan_shape(cc3d_plan_t plan, PlanShape* out);

}  // namespace cc3d
