/*
 * cc3d.h -- C ABI of the chunked causal 3-D convolution library (libcc3d.so).
 *
 * The operation (NDHWC activations, batch 1):
 *
 *   y[t,h,w,co] = b[co] + sum_{dt<kt, dh<kh, dw<kw, ci<Cin}
 *                   w[co,dt,dh,dw,ci] * xe[t+dt, h+dh-(kh-1)/2, w+dw-(kw-1)/2, ci]
 *                 (+ residual[t,h,w,co])
 *
 *   xe = concat_t(cache_in, x_chunk) is the chunk preceded by the kt-1 input
 *   frames of the previous chunk (all zeros for the first chunk of a video);
 *   spatial positions outside the frame read zero.  After the call,
 *   cache_out holds the last kt-1 frames of xe, which is the history the next
 *   chunk needs.
 *
 * Sources: "SwiftVR Inference Optimization" (LightX2V blog), section "ReAE:
 * Causal Halo Exchange" -- a causal layer convolves the current frame's input
 * features together with the preceding frames' input features; across chunks
 * only the previous chunk's last input frames are carried; a video's opening
 * chunk starts from an all-zero history.  Section "From Pixels to Latents and
 * Back" -- long videos are processed in temporal chunks while the per-layer
 * boundary features are kept.  "SGLang-Diffusion advanced optimizations",
 * section 3 "Parallel VAE" -- the VAE's cost is dense 3-D convolution, and
 * chunked or halo-split evaluation must stay equal to the unsplit result.
 * The state conventions (validate everything before touching any buffer,
 * caller-owned state buffers that swap roles between calls, reset without
 * reallocation, one instance per shape, no host synchronisation per call)
 * follow the "pixtreme-infer-cda-vsr" package page, section "Frame, state and
 * stream requirements" and "CUDA Graph inference".
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    never frees, retains or reallocates them.  Alignment: float32 plans need
 *    4 bytes for every pointer; bfloat16 plans need 16 bytes for x_chunk, w,
 *    cache_in and cache_out (tensor-memory-accelerator copies), 16 bytes for
 *    y and residual when Cout is a multiple of 16 (2 bytes for the narrow
 *    head, Cout < 16), and 2 bytes for b.  (y and residual 32-byte aligned
 *    let the SM-pair kernels use 32-byte accesses; results are the same.)
 *  - Layouts are dense row-major (channels innermost):
 *      x_chunk, residual, y : [T_chunk][H][W][C]
 *      cache_in, cache_out  : [kt-1][H][W][Cin]
 *      w                    : [Cout][kt][kh][kw][Cin]
 *      b                    : [Cout]
 *    with the element type of the plan (float32 or bfloat16) for all of them.
 *  - Work is enqueued on the given CUDA stream (a cudaStream_t passed as
 *    void*; NULL means the legacy default stream).  No call except
 *    cc3d_get_status synchronises the host.
 *  - Every argument is checked before anything is launched or written; a
 *    failed check returns an error code and leaves every buffer untouched.
 *    Device pointers must belong to the device current at the call (or be
 *    managed memory): host memory gives CC3D_ERR_NOT_DEVICE_MEMORY, another
 *    device's memory CC3D_ERR_INVALID_ARG.
 *  - Kernel waits are bounded.  A wait that runs out records an error in a
 *    per-device status word and the kernel returns; cc3d_get_status reports
 *    it.
 *  - A plan is used from one host thread at a time (its side stream and
 *    events, see cc3d_forward_chunk, are per plan); different plans may be
 *    used from different threads concurrently.
 */
#ifndef CC3D_H
#define CC3D_H

#include <stddef.h> /* size_t */

#ifdef __cplusplus
extern "C" {
#endif

typedef struct cc3d_plan_s* cc3d_plan_t;     /* opaque, owned by the library */
typedef struct cc3d_writer_s* cc3d_writer_t; /* opaque, owned by the library */

typedef enum { CC3D_F32 = 0, CC3D_BF16 = 1 } cc3d_dtype;

typedef enum {
    CC3D_OK = 0,
    CC3D_ERR_INVALID_ARG = 1,     /* null / negative / inconsistent argument        */
    CC3D_ERR_UNSUPPORTED = 2,     /* shape or dtype this build has no kernel for     */
    CC3D_ERR_ALIGNMENT = 3,       /* pointer not aligned (see Conventions)          */
    CC3D_ERR_ALIAS = 4,           /* an output overlaps another buffer              */
    CC3D_ERR_CUDA = 5,            /* a CUDA runtime call failed                     */
    CC3D_ERR_OOM = 6,             /* host allocation failed                         */
    CC3D_ERR_DEVICE_TIMEOUT = 7,  /* a bounded wait inside a kernel ran out          */
    CC3D_ERR_NOT_DEVICE_MEMORY = 8, /* a tensor pointer is not device-accessible      */
    CC3D_ERR_IO = 9,               /* a host file could not be opened or written      */
    CC3D_ERR_SCRATCH_TOO_SMALL = 10 /* the call needs more than the library's fixed
                                       device scratch array holds                   */
} cc3d_status;

/*
 * Create a plan for one layer shape.  Host-only: no CUDA call, no device
 * allocation.  kh and kw must be odd.  Supported in this build:
 *   CC3D_F32  : any Cin, Cout >= 1; 1 <= kt <= 4; kh, kw in {1, 3, 5}.
 *   CC3D_BF16 : 1 <= kt <= 3 and kh = kw in {1, 3} (the decoder's 3x3x3 layers,
 *               a 2x3x3 MemoryBlock, a 3x1x1 TemporalGrow, 1x1x1 projections);
 *               Cin a multiple of 16 (<= 1024); Cout a multiple of 16 (<= 512)
 *               or Cout < 16 (narrow output head).
 * When kt = 1 there is no history: cache_in is ignored and cache_out may be
 * NULL.
 * Anything else returns CC3D_ERR_UNSUPPORTED.  On error *out is set to NULL
 * and nothing is leaked.
 */
cc3d_status cc3d_plan_create(int Cin, int Cout, int H, int W, int kt, int kh, int kw, cc3d_dtype dtype,
                             cc3d_plan_t* out);

/*
 * A plan for a causal conv that reads its input through a nearest-2x spatial upsample
 * (the decoder's upsampling stage: every input pixel becomes a 2x2 block, then a
 * kt x 3 x 3 conv with zero padding 1), fused so that the 2H x 2W upsampled frames are
 * never stored:
 *   y[t, 2h+a, 2w+b, co] = conv(U(x))[...] with U(x)[t, i, j, c] = x[t, i/2, j/2, c].
 * H and W are the input (source) frames; x_chunk and the histories are [..][H][W][Cin],
 * y and the residual [T_chunk][2H][2W][Cout].  The history holds the last kt-1 *source*
 * frames (the upsample is per frame).  The results are bit-identical to a
 * cc3d_plan_create plan run on the materialised U(x).  bf16 only: Cin and Cout
 * multiples of 16 (<= 1024), 1 <= kt <= 3; the plan's kernel family is "tc_bf16_up2".
 * Otherwise as cc3d_plan_create.
 */
cc3d_status cc3d_plan_create_upsample2x(int Cin, int Cout, int H, int W, int kt, cc3d_dtype dtype,
                                        cc3d_plan_t* out);

/*
 * One temporal chunk of T_chunk frames (see the formula above).
 *   x_chunk  [T_chunk][H][W][Cin]  input frames of this chunk.
 *   w, b     weights and bias; b may be NULL (zero bias).
 *   residual [T_chunk][H][W][Cout] added after the bias, or NULL.
 *   cache_in [kt-1][H][W][Cin] history, or NULL for zero history (first chunk).
 *   cache_out[kt-1][H][W][Cin] receives the new history.  It must not overlap
 *            cache_in, x_chunk, y or residual (ping-pong two buffers).
 *   y        [T_chunk][H][W][Cout] output; must not overlap any input.
 * T_chunk may be 0: then only cache_out is written (it receives cache_in, or
 * zeros), and x_chunk, residual and y may be NULL.  A chunk of more than 2^33
 * positions (T_chunk * H * W) returns CC3D_ERR_UNSUPPORTED.
 * The result of every output element does not depend on how the video is
 * split into chunks (bit-identical across chunkings).  (The chunk sees the
 * previous chunk's last kt-1 input frames before its own: "SwiftVR Inference
 * Optimization" (LightX2V blog), section "ReAE: Causal Halo Exchange"; chunked
 * and whole-sequence results agree: "SGLang-Diffusion advanced optimizations",
 * section 3 "Parallel VAE".)
 * Returns CC3D_OK once the work is enqueued; asynchronous failures surface in
 * cc3d_get_status.
 * Stream use: all work is ordered after what the caller enqueued earlier on
 * `stream`, and everything the caller enqueues on it afterwards sees y and
 * cache_out complete.  For the SM-pair tensor-core kernels part of the
 * cache_out copy runs on a copy engine, on a side stream the plan creates on
 * its first such call (with two events; freed by cc3d_destroy): an event
 * forks it from `stream` before the kernel and `stream` waits for it after.
 * The call therefore stays capturable into a CUDA graph on `stream`.
 */
cc3d_status cc3d_forward_chunk(cc3d_plan_t plan, int T_chunk, const void* x_chunk, const void* w, const void* b,
                               const void* residual_or_null, const void* cache_in, void* cache_out, void* y,
                               void* stream);

/*
 * The same chunk with 8-bit pixels out, for narrow-output plans (cc3d_plan_kernel
 * "tc_bf16_head", e.g. the RGB head of a video decoder): the device-side half of an
 * asynchronous frame output path (AWS / Synthesia, "How Synthesia optimizes
 * generative AI video inference on Amazon EC2 G7e instances": chunks are copied to
 * the host and written while the next chunk computes; 8-bit frames halve those
 * copies).  Every output value is first rounded to bf16 exactly as
 * cc3d_forward_chunk stores it (v), then
 *   y_u8 = clamp(round_to_nearest_even((v + 1) * 127.5), 0, 255)
 * computed in fp32 (one rounding after the add, one after the multiply): decoder
 * outputs in [-1, 1] map onto [0, 255].
 *   y_u8  [T_chunk][H][W][Cout] uint8, any alignment; must not overlap any input.
 * Other arguments, checks and the history are as in cc3d_forward_chunk.  Plans of
 * any other kernel family return CC3D_ERR_UNSUPPORTED.
 */
cc3d_status cc3d_forward_chunk_u8(cc3d_plan_t plan, int T_chunk, const void* x_chunk, const void* w, const void* b,
                                  const void* residual_or_null, const void* cache_in, void* cache_out, void* y_u8,
                                  void* stream);

/*
 * Asynchronous chunk output (the host half of the frame output path of AWS /
 * Synthesia, "How Synthesia optimizes generative AI video inference on Amazon EC2
 * G7e instances": a copy stream beside the compute stream, double buffers in device
 * and pinned host memory with events as barriers, and a worker thread that writes
 * the host buffers to storage while the next chunk computes).
 *
 * cc3d_writer_create: opens (truncates) the file at `path` and allocates two pinned
 *   host slots of slot_bytes, a copy stream and events; starts the worker thread.
 * cc3d_writer_submit: once the work already enqueued on compute_stream is done, copy
 *   `bytes` (<= slot_bytes) from the device buffer `src` into the next pinned slot on
 *   the copy stream; the worker appends the slot to the file, in submission order.
 *   Returns at once unless that slot still holds an unwritten chunk (then it waits for
 *   the worker).  *seq_out (may be NULL) receives the submission's number (0, 1, ...).
 *   `src` is read asynchronously: before the caller overwrites it, it calls
 * cc3d_writer_wait_copied(w, seq, stream): `stream` waits (stream-ordered, no host
 *   block) until the copy of submission `seq` is done.  seq < 0 is a no-op.
 * cc3d_writer_close: writes everything submitted, stops the worker, frees the writer
 *   (also on error); *bytes_written (may be NULL) receives the bytes written.
 * Errors: CC3D_ERR_INVALID_ARG (also: src on another device than the one current at
 * create), CC3D_ERR_NOT_DEVICE_MEMORY (src), CC3D_ERR_CUDA, CC3D_ERR_OOM, CC3D_ERR_IO
 * (open or write failed; reported by the next submit and by close).  After the first
 * failed copy or write, the chunks still queued are dropped, not written: the file
 * holds the chunks before the failure and nothing after it.  A writer is used from
 * one host thread at a time.
 */
cc3d_status cc3d_writer_create(const char* path, size_t slot_bytes, cc3d_writer_t* out);
cc3d_status cc3d_writer_submit(cc3d_writer_t w, const void* src, size_t bytes, void* compute_stream,
                               long long* seq_out);
cc3d_status cc3d_writer_wait_copied(cc3d_writer_t w, long long seq, void* stream);
cc3d_status cc3d_writer_close(cc3d_writer_t w, long long* bytes_written);

/*
 * Layer groups run frame batch by frame batch ("SwiftVR Inference Optimization"
 * (LightX2V blog), section "ReAE Frame Batching": consecutive layers pass a small
 * batch of frames through the whole group before the next batch starts, so only
 * one batch's intermediate features exist at a time and the last layer writes into
 * one output buffer; layers with a temporal history keep their state rules).
 *
 * cc3d_group_create: a group of nlayers (1..64) consecutive plans, run in order
 *   on each batch of frame_batch frames (0: the whole chunk as one batch).  Layer
 *   l + 1 reads what layer l writes: its input frames must be layer l's output
 *   frames (channels and size; an upsampling plan doubles them) in the same dtype,
 *   else CC3D_ERR_INVALID_ARG.  The host array is copied; the plans are not owned
 *   and must outlive the group.
 * cc3d_group_workspace_bytes: device bytes of workspace that a chunk of up to T_max
 *   frames needs: two buffers that the intermediate batches alternate between
 *   (each one batch of the largest layer output it holds), and, when a chunk takes
 *   more than one batch, one more history buffer [kt-1][H][W][Cin] per layer with
 *   a history.  0 for a one-layer group taking its chunk in one batch.
 * cc3d_group_forward_chunk: one chunk of T_chunk frames through the group.
 *   x_chunk   the first layer's input [T_chunk][H][W][Cin].
 *   w, b      host arrays of nlayers device pointers (b, and any b[l], may be NULL).
 *   cache_in  host array of nlayers history pointers, or NULL; an entry is NULL
 *             for a zero history (and for kt = 1 layers).
 *   cache_out host array of nlayers history buffers (entries of kt = 1 layers may
 *             be NULL); each receives its layer's history after the chunk, as
 *             cc3d_forward_chunk would leave it.
 *   y         the last layer's output [T_chunk][Ho][Wo][Cout].
 *   workspace device memory owned by the caller, 256-byte aligned, at least
 *             cc3d_group_workspace_bytes(T_chunk) bytes (workspace_bytes gives its
 *             size), overlapping nothing else; its contents need no initialisation
 *             and are undefined afterwards.  May be NULL when 0 bytes are needed.
 *   No residual inputs.  Every launch of the chunk is checked (as in
 *   cc3d_forward_chunk) before the first one is enqueued; a failed check launches
 *   nothing.  All work is enqueued on `stream`, in order.  The outputs and
 *   histories equal those of running each layer's chunk loop over the whole chunk,
 *   bit for bit.
 */
typedef struct cc3d_group_s* cc3d_group_t;
cc3d_status cc3d_group_create(int nlayers, const cc3d_plan_t* plans, int frame_batch, cc3d_group_t* out);
cc3d_status cc3d_group_workspace_bytes(cc3d_group_t g, int T_max, size_t* bytes);
cc3d_status cc3d_group_forward_chunk(cc3d_group_t g, int T_chunk, const void* x_chunk, const void* const* w,
                                     const void* const* b, const void* const* cache_in, void* const* cache_out,
                                     void* y, void* workspace, size_t workspace_bytes, void* stream);
void cc3d_group_destroy(cc3d_group_t g);

/*
 * cc3d_group_forward_chunk without a caller-provided workspace; it allocates
 * nothing.  (The pages have no counterpart of this call: it is an addition for
 * callers that cannot allocate device memory themselves -- for example a plugin
 * running inside a host framework whose allocator owns the GPU's memory and hands
 * the plugin only its input and output buffers, or a processing loop that must
 * not allocate once it is running, since cudaMalloc and cudaFree can synchronise
 * the device and take an unbounded time.)
 *
 * The workspace is instead a fixed array of CC3D_GROUP_STATIC_SCRATCH_BYTES
 * (64 MiB) in device memory, declared in the library itself: every GPU on which
 * the library's device code is loaded holds it until the process exits.  A chunk
 * whose workspace (cc3d_group_workspace_bytes(g, T_chunk)) exceeds it is refused
 * with CC3D_ERR_SCRATCH_TOO_SMALL before anything is launched; use
 * cc3d_group_forward_chunk with your own workspace for such groups.  The caller
 * still provides the inputs, outputs and histories, exactly as for
 * cc3d_group_forward_chunk (same arguments without the workspace, same checks,
 * same results).
 *
 * The first call on each device looks up the array's device address there (one
 * CUDA runtime query with that device current; later calls reuse it), so make
 * the first call on a device before any stream capture on it.  The array keeps
 * whatever the last call left in it; nothing in it needs to start at zero, as a
 * chunk writes every part of it that it reads.  All calls on one device share
 * the one array: two calls whose work overlaps on the GPU (e.g. on two streams
 * without an event between them) race and corrupt each other's intermediates;
 * order them on one stream or with events.
 */
#define CC3D_GROUP_STATIC_SCRATCH_BYTES (64u * 1024u * 1024u)
cc3d_status cc3d_group_forward_chunk_static(cc3d_group_t g, int T_chunk, const void* x_chunk, const void* const* w,
                                            const void* const* b, const void* const* cache_in,
                                            void* const* cache_out, void* y, void* stream);

/* Zero a cache buffer ([kt-1][H][W][Cin]) on the stream: the history of a new
 * video.  Stream-ordered, no allocation.  Same alignment rule as cache_out.
 * (A new stream restarts from a clean state without reallocating its buffers:
 * "pixtreme-infer-cda-vsr" package page, section "Frame, state and stream
 * requirements"; the first chunk's history is zeros: "SwiftVR Inference
 * Optimization", section "ReAE: Causal Halo Exchange".) */
cc3d_status cc3d_reset(cc3d_plan_t plan, void* cache, void* stream);

/* Synchronise the stream, then report (and clear) the device status word and
 * any pending CUDA error: CC3D_OK, CC3D_ERR_DEVICE_TIMEOUT or CC3D_ERR_CUDA.
 * The word is read and cleared in one atomic exchange on the device (a bit set
 * meanwhile by a kernel still running elsewhere is kept for the next call).  It
 * is one word per device, shared by every plan on it: a timeout in one plan's
 * kernel is reported to whichever caller polls that device first. */
cc3d_status cc3d_get_status(cc3d_plan_t plan, void* stream);

/* Release the plan (NULL is accepted). */
void cc3d_destroy(cc3d_plan_t plan);

/* Text naming the CUDA call (or CUDA error) behind the last CC3D_ERR_CUDA
 * returned on the calling thread; "none" before any.  Static storage. */
const char* cc3d_last_error_detail(void);

/* Static, human-readable text of a status code. */
const char* cc3d_status_string(cc3d_status s);

/* Name of the kernel family the plan will launch ("tc_bf16", "tc_bf16_pair" -- SM
 * pairs, "tc_bf16_head" -- narrow outputs with the spatial taps stacked into N,
 * "tc_bf16_stream" -- 1x1 spatial kernels, "tc_bf16_up2" -- fused nearest-2x
 * upsampling, "tc_bf16_narrow", "simt_f32"); a static
 * string, NULL for a NULL plan. */
const char* cc3d_plan_kernel(cc3d_plan_t plan);

/* Number of kernel launches one cc3d_forward_chunk call of this plan makes
 * (T_chunk >= 1). */
int cc3d_plan_launches_per_chunk(cc3d_plan_t plan);

/* The launch configuration cc3d_forward_chunk would use for a chunk of T_chunk
 * frames (with a residual when has_residual != 0), as one line of
 * space-separated key=value pairs, NUL-terminated, written into buf (len bytes,
 * owned by the caller).  Host-only: no device is needed and nothing is
 * launched.  Keys for the tensor-core families: kernel (the CUDA kernel:
 * tc_bf16_kernel on one SM, tc2_bf16_kernel on SM pairs, tc2s_bf16_kernel on
 * SM pairs with two output frames per MMA), pair, two_frame, up2,
 * channel_block, NT (output channels per tile), row_groups (128-row groups per
 * tile), window_stages / weight_stages and their bytes, tap_rows_per_weight_stage,
 * acc_stages, smem_bytes, tiles (per chunk) and history_frames_on_copy_engine;
 * the head, streaming and fp32 families report their own keys.  Returns
 * CC3D_ERR_INVALID_ARG for a NULL plan or buf, T_chunk < 1, or a line longer
 * than len - 1 (buf is then the empty string); CC3D_ERR_UNSUPPORTED when the
 * chunk has no configuration. */
cc3d_status cc3d_plan_describe(cc3d_plan_t plan, int T_chunk, int has_residual, char* buf, size_t len);

/*
 * Test hooks (used by the fault tests; never needed in normal use).
 * cc3d_debug_set_wait_budget_ns: wall-clock budget of every bounded wait in
 *   this plan's kernels (default 2e9 ns).
 * cc3d_debug_set_fault: 0 = none; 1 = the tensor-core kernel's loader skips
 *   its first copy so that the consumer's bounded wait runs out (the kernel
 *   then records CC3D_ERR_DEVICE_TIMEOUT and returns); 2 = fail host-side
 *   tensor-map encoding (CC3D_ERR_CUDA, nothing launched).
 */
cc3d_status cc3d_debug_set_wait_budget_ns(cc3d_plan_t plan, unsigned long long ns);
cc3d_status cc3d_debug_set_fault(cc3d_plan_t plan, int mode);

/*
 * Schedule overrides of the bf16 tensor-core families "tc_bf16", "tc_bf16_pair",
 * "tc_bf16_narrow" and "tc_bf16_up2" (for tuning sweeps and for the tests that
 * compare two schedules bit for bit; never needed in normal use).  Every knob
 * starts at -1, the measured default for the chunk's shape.  A knob other than
 * CC3D_SCHED_CHANNEL_BLOCK changes only how the work is tiled: the accumulation
 * order of every output is fixed, so every schedule gives the same bits.  A combination with no configuration makes
 * cc3d_forward_chunk return CC3D_ERR_UNSUPPORTED (nothing launched); one whose
 * shared memory does not fit the SM is refused by the launch (CC3D_ERR_CUDA).
 * The plan's settings are its own: nothing is read from the environment.
 * cc3d_debug_set_schedule returns CC3D_ERR_INVALID_ARG for a NULL plan, an
 * unknown knob or a value outside the knob's range (given beside it; -1 restores
 * the default).
 */
typedef enum {
    CC3D_SCHED_PAIR = 0,           /* 0..1: SM pairs (cta_group::2) where the geometry allows */
    CC3D_SCHED_TWO_FRAME = 1,      /* 0..1: two output frames per MMA on SM pairs (chunks of >= 2 frames) */
    CC3D_SCHED_SPLIT_TAIL = 2,     /* 0..1: split the tiles of a short last wave between both MMA warps */
    CC3D_SCHED_CHANNEL_BLOCKS = 3, /* 0..1: outputs wider than 256 channels as channel-block tiles */
    CC3D_SCHED_MMA_WARPS = 4,      /* 1..2: MMA-issuing warps */
    CC3D_SCHED_ROW_GROUPS = 5,     /* 1, 2 or 4: 128-row groups per tile */
    CC3D_SCHED_ACC_STAGES = 6,     /* 1..2: accumulator buffers in tensor memory */
    CC3D_SCHED_TAP_ROWS = 7,       /* 1 or 3: kernel rows per weight stage */
    CC3D_SCHED_WINDOW_STAGES = 8,  /* 2..8: input-window ring depth */
    CC3D_SCHED_WEIGHT_STAGES = 9,  /* 2..8: upper bound of the weight ring depth */
    CC3D_SCHED_PREFETCH = 10,      /* 0..3: temporal taps of the next tile warmed in L2 */
    CC3D_SCHED_CHANNEL_BLOCK = 11, /* 16 or 32: input channels per K block (where Cin allows).  Unlike
                                      the other knobs it changes the order in which each output's
                                      products are summed (so the low bits of the result), the same
                                      way for every chunk: set it before a video's first chunk */
    CC3D_SCHED_COUNT = 12
} cc3d_schedule_knob;
cc3d_status cc3d_debug_set_schedule(cc3d_plan_t plan, int knob, int value);

#ifdef __cplusplus
}
#endif
#endif /* CC3D_H */
