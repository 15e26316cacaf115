// cc3d_api.cu -- the C ABI declared in include/cc3d.h: plans, argument checks, tensor-map
// encoding and kernel dispatch.  Nothing here computes on the host; every step of the
// convolution runs in the kernels of cc3d_tc.cu, cc3d_tc2.cu, cc3d_head.cu, cc3d_stream.cu and
// cc3d_simt.cu.
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "cc3d.h"
#include "cc3d_internal.h"

namespace cc3d {

// Per-device status word: kernels or-in STATUS_* bits, cc3d_get_status reads and clears it.  It is
// shared by every plan on the device: a timeout of one plan is reported to whichever caller of
// cc3d_get_status on that device comes first.
__device__ unsigned g_status_word;
// cc3d_get_status's read of the word, taken and cleared in one atomic exchange
__device__ unsigned g_status_taken;

__global__ void status_take_kernel() { g_status_taken = atomicExch(&g_status_word, 0u); }

cudaError_t status_take_launch(cudaStream_t stream)
{
    status_take_kernel<<<1, 1, 0, stream>>>();
    return cudaGetLastError();
}

namespace {

enum KernelKind {
    K_SIMT_F32 = 0,
    K_TC_BF16 = 1,
    K_TC_BF16_NARROW = 2,
    K_TC_BF16_PAIR = 3,
    K_TC_BF16_HEAD = 4,
    K_TC_BF16_STREAM = 5,
    K_TC_BF16_UP2 = 6
};

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    bool sm103 = false;
    int sms = 0;
    unsigned* status = nullptr;
};

std::mutex g_mutex;
std::mutex g_status_mutex;
thread_local const char* g_last_detail = "none";

// Record what failed (for cc3d_last_error_detail) and return CC3D_ERR_CUDA.
cc3d_status cuda_fail(const char* what, cudaError_t e = cudaSuccess)
{
    g_last_detail = (e != cudaSuccess) ? cudaGetErrorName(e) : what;
    return CC3D_ERR_CUDA;
}
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cc3d_status device_info(DeviceInfo** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cuda_fail("cudaGetDevice", e);
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cuda_fail("cudaDeviceGetAttribute", cudaGetLastError());
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return cuda_fail("cudaGetSymbolAddress", e);
        if (g_encode == nullptr) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                fn == nullptr)
                return cuda_fail("cuTensorMapEncodeTiled entry point unavailable");
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.sm103 = (major == 10 && minor == 3);
        d.sms = sms;
        d.status = static_cast<unsigned*>(p);
        d.ready = true;
    }
    *out = &d;
    return CC3D_OK;
}

// Where a tensor pointer lives: CC3D_OK for memory the current device's kernels may use (its own
// device memory, or managed memory), CC3D_ERR_NOT_DEVICE_MEMORY for host or unknown memory, and
// CC3D_ERR_INVALID_ARG for another device's memory (the kernels, tensor maps and status word are
// those of the current device, and without peer access such a read faults).
cc3d_status pointer_check(const void* p)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();  // clear the non-sticky error
        return CC3D_ERR_NOT_DEVICE_MEMORY;
    }
    if (a.type == cudaMemoryTypeManaged) return CC3D_OK;
    if (a.type != cudaMemoryTypeDevice) return CC3D_ERR_NOT_DEVICE_MEMORY;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return CC3D_ERR_NOT_DEVICE_MEMORY;
    }
    return a.device == dev ? CC3D_OK : CC3D_ERR_INVALID_ARG;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
}

bool aligned_to(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace cc3d

using namespace cc3d;

struct cc3d_plan_s {
    int Cin, Cout, H, W, kt, kh, kw;  // H, W: the input frames (an upsampling plan writes 2H x 2W)
    int up2 = 0;
    cc3d_dtype dtype;
    int kind;
    int CB;
    unsigned long long wait_ns;
    int fault;
    TcOverrides ov;  // schedule knobs (cc3d_debug_set_schedule), all -1 = measured defaults
    // Part of the new history is copied by a copy engine on a side stream, forked from the
    // caller's stream before the launch and joined to it after (created on first use, on the
    // device current then; on another device the kernel copies the whole history itself): all of
    // it for the one-frame SM-pair kernel, the first of the two frames for the two-frame kernel,
    // none for the one-SM kernel.  Measured on GB300 against the kernel's own copy warp: 2x3x3 at
    // 96 channels 1400 against 1315 TFLOP/s, 3x3x3 at 96 channels 1587 against 1558; the one-SM
    // kernel lost 1.5-2.5 %.  A copy engine moves about 0.3 TB/s (more streams did not add to
    // it), so a larger share outlasts the launch.
    static constexpr int kSide = 1;
    cudaStream_t side[kSide] = {};
    cudaEvent_t fork = nullptr;
    cudaEvent_t join[kSide] = {};
    int side_device = -1;
    ~cc3d_plan_s()
    {
        for (int i = 0; i < kSide; ++i) {
            if (side[i] != nullptr) cudaStreamDestroy(side[i]);
            if (join[i] != nullptr) cudaEventDestroy(join[i]);
        }
        if (fork != nullptr) cudaEventDestroy(fork);
    }
};

namespace {

// The side streams and their events for this plan on the current device; false if they cannot be
// had (then the kernel copies the history).
bool side_stream_ready(cc3d_plan_s* p)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (p->fork != nullptr) return p->side_device == dev;
    bool ok = cudaEventCreateWithFlags(&p->fork, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < cc3d_plan_s::kSide; ++i)
        ok = cudaStreamCreateWithFlags(&p->side[i], cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&p->join[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        for (int i = 0; i < cc3d_plan_s::kSide; ++i) {
            if (p->side[i] != nullptr) cudaStreamDestroy(p->side[i]);
            if (p->join[i] != nullptr) cudaEventDestroy(p->join[i]);
            p->side[i] = nullptr;
            p->join[i] = nullptr;
        }
        if (p->fork != nullptr) cudaEventDestroy(p->fork);
        p->fork = nullptr;
        return false;
    }
    p->side_device = dev;
    return true;
}

}  // namespace

// Narrow-output launch: tensor maps with one-row boxes for the staged input rows (loads) and the
// new history (stores, from staged row 8 on), and a (32 channels, Cout, 9 taps) box for the weights of one (dt,
// channel block).
static cc3d_status head_forward(const cc3d_plan_s& p, const DeviceInfo& d, int T, const void* x, const void* w,
                                const void* b, const void* res, const void* cache_in, void* cache_out, void* y,
                                cudaStream_t stream, bool out_u8)
{
    HeadLaunch L;
    memset(&L, 0, sizeof(L));
    if (!head_configure(T, p.H, p.W, p.Cin, p.Cout, d.sms, &L)) return CC3D_ERR_UNSUPPORTED;
    if (p.fault == 2) return cuda_fail("injected tensor-map encode failure");  // nothing launched
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const cuuint64_t strides[3] = {(cuuint64_t)p.Cin * 2, (cuuint64_t)p.W * p.Cin * 2,
                                   (cuuint64_t)p.H * p.W * p.Cin * 2};
    const cuuint32_t box[4] = {32, 128, 1, 1};  // the 128 input positions of a strip
    const cuuint64_t dims[4] = {(cuuint64_t)p.Cin, (cuuint64_t)p.W, (cuuint64_t)p.H, (cuuint64_t)T};
    if (g_encode(&L.map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cuda_fail("cuTensorMapEncodeTiled (x_chunk)");
    if (cache_in != nullptr) {
        const cuuint64_t cdims[4] = {(cuuint64_t)p.Cin, (cuuint64_t)p.W, (cuuint64_t)p.H, 2};
        if (g_encode(&L.map_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache_in), cdims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_fail("cuTensorMapEncodeTiled (cache_in)");
    }
    {
        const cuuint64_t cdims[4] = {(cuuint64_t)p.Cin, (cuuint64_t)p.W, (cuuint64_t)p.H, 2};
        const cuuint32_t sbox[4] = {32, 120, 1, 1};  // staged rows 8 .. 127 (positions w0 + 7 .. w0 + 126)
        if (g_encode(&L.map_cache_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, cache_out, cdims, strides, sbox, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_fail("cuTensorMapEncodeTiled (cache_out)");
    }
    {
        // weights [Cout][27][Cin] seen as (ci, co, tap): one box = the 9 spatial taps of one dt
        const cuuint64_t wdims[3] = {(cuuint64_t)p.Cin, (cuuint64_t)p.Cout, 27};
        const cuuint64_t wstrides[2] = {(cuuint64_t)27 * p.Cin * 2, (cuuint64_t)p.Cin * 2};
        const cuuint32_t wbox[3] = {32, (cuuint32_t)p.Cout, 9};
        if (g_encode(&L.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), wdims, wstrides, wbox, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_fail("cuTensorMapEncodeTiled (w)");
    }
    L.has_cache = cache_in != nullptr;
    L.bias = b;
    L.res = res;
    L.y = y;
    L.x = x;
    L.cache_in = cache_in;
    L.cache_out = cache_out;
    L.out_u8 = out_u8 ? 1 : 0;
    L.status = d.status;
    L.wait_ns = p.wait_ns;
    L.fault = p.fault;
    const cudaError_t e = head_launch(L, stream);
    return e == cudaSuccess ? CC3D_OK : cuda_fail("narrow-output kernel launch", e);
}

// Streaming launch for 1x1 spatial kernels: frames seen as (Cin, H*W) matrices.
static cc3d_status stream_forward(const cc3d_plan_s& p, const DeviceInfo& d, int T, const void* x, const void* w,
                                  const void* b, const void* res, const void* cache_in, void* cache_out, void* y,
                                  cudaStream_t stream)
{
    StreamLaunch L;
    memset(&L, 0, sizeof(L));
    if (!stream_configure(T, p.H, p.W, p.Cin, p.Cout, p.kt, d.sms, &L)) return CC3D_ERR_UNSUPPORTED;
    if (p.fault == 2) return cuda_fail("injected tensor-map encode failure");  // nothing launched
    const int P = p.kt - 1;
    const cuuint64_t HW = (cuuint64_t)p.H * p.W;
    const cuuint32_t estr[3] = {1, 1, 1};
    const cuuint64_t strides[2] = {(cuuint64_t)p.Cin * 2, HW * p.Cin * 2};
    const cuuint32_t box[3] = {32, 128, 1};
    const cuuint64_t dims[3] = {(cuuint64_t)p.Cin, HW, (cuuint64_t)T};
    if (g_encode(&L.map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(x), dims, strides, box, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cuda_fail("cuTensorMapEncodeTiled (x_chunk)");
    if (P > 0) {
        const cuuint64_t cdims[3] = {(cuuint64_t)p.Cin, HW, (cuuint64_t)P};
        if (cache_in != nullptr &&
            g_encode(&L.map_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(cache_in), cdims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_fail("cuTensorMapEncodeTiled (cache_in)");
        if (g_encode(&L.map_cache_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, cache_out, cdims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_fail("cuTensorMapEncodeTiled (cache_out)");
    }
    {
        // weights [Cout][kt][1][1][Cin] seen as (ci, co, dt): one box = all output channels of one tap
        const cuuint64_t wdims[3] = {(cuuint64_t)p.Cin, (cuuint64_t)p.Cout, (cuuint64_t)p.kt};
        const cuuint64_t wstrides[2] = {(cuuint64_t)p.kt * p.Cin * 2, (cuuint64_t)p.Cin * 2};
        const cuuint32_t wbox[3] = {32, (cuuint32_t)p.Cout, 1};
        if (g_encode(&L.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), wdims, wstrides, wbox, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_fail("cuTensorMapEncodeTiled (w)");
    }
    L.has_cache = P > 0 && cache_in != nullptr;
    L.bias = b;
    L.res = res;
    L.y = y;
    L.v32 = ((reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(res)) & 31) == 0 ? 1 : 0;
    L.status = d.status;
    L.wait_ns = p.wait_ns;
    L.fault = p.fault;
    const cudaError_t e = stream_launch(L, stream);
    return e == cudaSuccess ? CC3D_OK : cuda_fail("streaming kernel launch", e);
}

// The plan's input-channel block (the K step of the tensor-core kernels), 16 or 32 channels; the
// CC3D_SCHED_CHANNEL_BLOCK knob may choose 16 for a plan whose Cin allows 32 (it changes the order
// in which the products of every output are summed, the same way for every chunk of the plan).
static int plan_cb(const cc3d_plan_s& p)
{
    const int v = p.ov.get(CC3D_SCHED_CHANNEL_BLOCK, 0);
    if (v == 16 && p.Cin % 16 == 0) return 16;
    if (v == 32 && p.Cin % 32 == 0) return 32;
    return p.CB;
}

extern "C" {

const char* cc3d_status_string(cc3d_status s)
{
    switch (s) {
    case CC3D_OK: return "ok";
    case CC3D_ERR_INVALID_ARG: return "invalid argument";
    case CC3D_ERR_UNSUPPORTED: return "unsupported shape, dtype or device";
    case CC3D_ERR_ALIGNMENT: return "pointer not aligned as the plan requires";
    case CC3D_ERR_ALIAS: return "output buffer overlaps another buffer";
    case CC3D_ERR_CUDA: return "CUDA runtime error";
    case CC3D_ERR_OOM: return "out of host memory";
    case CC3D_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel ran out";
    case CC3D_ERR_NOT_DEVICE_MEMORY: return "pointer is not device memory";
    case CC3D_ERR_IO: return "host file could not be opened or written";
    case CC3D_ERR_SCRATCH_TOO_SMALL: return "the call needs more than the library's fixed device scratch array";
    }
    return "unknown status";
}

cc3d_status cc3d_plan_create(int Cin, int Cout, int H, int W, int kt, int kh, int kw, cc3d_dtype dtype,
                             cc3d_plan_t* out)
{
    if (out == nullptr) return CC3D_ERR_INVALID_ARG;
    *out = nullptr;
    if (Cin < 1 || Cout < 1 || H < 1 || W < 1 || kt < 1 || kh < 1 || kw < 1) return CC3D_ERR_INVALID_ARG;
    if (kh % 2 == 0 || kw % 2 == 0) return CC3D_ERR_INVALID_ARG;
    if (dtype != CC3D_F32 && dtype != CC3D_BF16) return CC3D_ERR_INVALID_ARG;
    if ((long long)H * W > (1LL << 30) || Cin > 65536 || Cout > 65536) return CC3D_ERR_UNSUPPORTED;
    int kind, CB = 0;
    if (dtype == CC3D_F32) {
        if (kt > 4 || kh > 5 || kw > 5) return CC3D_ERR_UNSUPPORTED;
        kind = K_SIMT_F32;
    } else {
        // tensor cores: kt in 1..3 with a square 3x3 or 1x1 spatial kernel (the decoder's 3x3x3,
        // MemoryBlock 2x3x3, TemporalGrow 3x1x1 and pointwise 1x1x1 layers)
        if (kt > 3 || kh != kw || (kh != 1 && kh != 3)) return CC3D_ERR_UNSUPPORTED;
        if (Cin % 16 != 0 || Cin > 1024) return CC3D_ERR_UNSUPPORTED;
        if (!(Cout < 16 || (Cout % 16 == 0 && Cout <= 512))) return CC3D_ERR_UNSUPPORTED;
        CB = (Cin % 32 == 0) ? 32 : 16;
        HeadLaunch hprobe;
        memset(&hprobe, 0, sizeof(hprobe));
        StreamLaunch sprobe;
        memset(&sprobe, 0, sizeof(sprobe));
        if (kt == 3 && kh == 3 && head_configure(1, H, W, Cin, Cout, 1, &hprobe)) {
            kind = K_TC_BF16_HEAD;  // narrow output: taps stacked into N
        } else if (kh == 1 && stream_configure(1, H, W, Cin, Cout, kt, 1, &sprobe)) {
            kind = K_TC_BF16_STREAM;  // no spatial taps: HBM-bound, streamed
        } else {
            TcLaunch probe;
            memset(&probe, 0, sizeof(probe));
            if (!tc_configure(CB, 1, H, W, Cin, Cout, kt, kh, false, false, nullptr, &probe) ||
                !tc_configure(CB, 1, H, W, Cin, Cout, kt, kh, true, false, nullptr, &probe))
                return CC3D_ERR_UNSUPPORTED;
            kind = Cout < 16 ? K_TC_BF16_NARROW : (probe.pair ? K_TC_BF16_PAIR : K_TC_BF16);
        }
    }
    cc3d_plan_s* p = new (std::nothrow) cc3d_plan_s;
    if (p == nullptr) return CC3D_ERR_OOM;
    p->Cin = Cin;
    p->Cout = Cout;
    p->H = H;
    p->W = W;
    p->kt = kt;
    p->kh = kh;
    p->kw = kw;
    p->dtype = dtype;
    p->kind = kind;
    p->CB = CB;
    p->wait_ns = 2000000000ull;
    p->fault = 0;
    for (int& v : p->ov.v) v = -1;
    *out = p;
    return CC3D_OK;
}

cc3d_status cc3d_plan_create_upsample2x(int Cin, int Cout, int H, int W, int kt, cc3d_dtype dtype,
                                        cc3d_plan_t* out)
{
    if (out == nullptr) return CC3D_ERR_INVALID_ARG;
    *out = nullptr;
    if (Cin < 1 || Cout < 1 || H < 1 || W < 1 || kt < 1) return CC3D_ERR_INVALID_ARG;
    if (dtype != CC3D_F32 && dtype != CC3D_BF16) return CC3D_ERR_INVALID_ARG;
    if (dtype != CC3D_BF16 || kt > 3) return CC3D_ERR_UNSUPPORTED;
    if ((long long)H * W > (1LL << 28) || Cin % 16 != 0 || Cin > 1024 || Cout % 16 != 0 || Cout > 1024)
        return CC3D_ERR_UNSUPPORTED;
    const int CB = (Cin % 32 == 0) ? 32 : 16;
    TcLaunch probe;
    memset(&probe, 0, sizeof(probe));
    if (!tc_configure(CB, 1, H, W, Cin, Cout, kt, 3, false, true, nullptr, &probe) ||
        !tc_configure(CB, 1, H, W, Cin, Cout, kt, 3, true, true, nullptr, &probe))
        return CC3D_ERR_UNSUPPORTED;
    cc3d_plan_s* p = new (std::nothrow) cc3d_plan_s;
    if (p == nullptr) return CC3D_ERR_OOM;
    p->Cin = Cin;
    p->Cout = Cout;
    p->H = H;
    p->W = W;
    p->kt = kt;
    p->kh = 3;
    p->kw = 3;
    p->up2 = 1;
    p->dtype = dtype;
    p->kind = K_TC_BF16_UP2;
    p->CB = CB;
    p->wait_ns = 2000000000ull;
    p->fault = 0;
    for (int& v : p->ov.v) v = -1;
    *out = p;
    return CC3D_OK;
}

void cc3d_destroy(cc3d_plan_t plan) { delete plan; }

const char* cc3d_last_error_detail(void) { return g_last_detail; }

const char* cc3d_plan_kernel(cc3d_plan_t plan)
{
    if (plan == nullptr) return nullptr;
    switch (plan->kind) {
    case K_SIMT_F32: return "simt_f32";
    case K_TC_BF16: return "tc_bf16";
    case K_TC_BF16_PAIR: return "tc_bf16_pair";
    case K_TC_BF16_HEAD: return "tc_bf16_head";
    case K_TC_BF16_STREAM: return "tc_bf16_stream";
    case K_TC_BF16_UP2: return "tc_bf16_up2";
    default: return "tc_bf16_narrow";
    }
}

int cc3d_plan_launches_per_chunk(cc3d_plan_t plan)
{
    if (plan == nullptr) return 0;
    return plan->kind == K_SIMT_F32 ? 2 : 1;  // the tensor-core kernel also writes the new cache
}

cc3d_status cc3d_plan_describe(cc3d_plan_t plan, int T, int has_residual, char* buf, size_t len)
{
    if (plan == nullptr || buf == nullptr || len == 0 || T < 1) return CC3D_ERR_INVALID_ARG;
    buf[0] = 0;
    const cc3d_plan_s& p = *plan;
    const int P = p.kt - 1;
    int n = 0;
    if (p.kind == K_SIMT_F32) {
        n = snprintf(buf, len, "kernel=simt_f32_kernel launches=%d", P > 0 ? 2 : 1);
    } else if (p.kind == K_TC_BF16_HEAD) {
        HeadLaunch hl;
        memset(&hl, 0, sizeof(hl));
        if (!head_configure(T, p.H, p.W, p.Cin, p.Cout, 1, &hl)) return CC3D_ERR_UNSUPPORTED;
        n = snprintf(buf, len,
                     "kernel=head_bf16_kernel frames_per_pass=%d column_strips=%d row_stages=%d row_stage_bytes=%d "
                     "weight_bytes=%d tmem_cols=%d smem_bytes=%zu units=%lld",
                     hl.gmax, hl.ncolblk, hl.nstages, hl.x_stage_bytes, hl.w_bytes, hl.tmem_cols, hl.smem_bytes,
                     hl.units);
    } else if (p.kind == K_TC_BF16_STREAM) {
        StreamLaunch sl;
        memset(&sl, 0, sizeof(sl));
        if (!stream_configure(T, p.H, p.W, p.Cin, p.Cout, p.kt, 1, &sl)) return CC3D_ERR_UNSUPPORTED;
        n = snprintf(buf, len,
                     "kernel=stream_bf16_kernel frames_per_unit=%d position_blocks=%d stages=%d stage_bytes=%d "
                     "weight_bytes=%d tmem_cols=%d smem_bytes=%zu units=%lld",
                     sl.gmax, sl.npb, sl.nstages, sl.x_stage_bytes, sl.w_bytes, sl.tmem_cols, sl.smem_bytes, sl.units);
    } else {
        TcLaunch L;
        memset(&L, 0, sizeof(L));
        if (!tc_configure(plan_cb(p), T, p.H, p.W, p.Cin, p.Cout, p.kt, p.kh, has_residual != 0, p.up2 != 0, &p.ov,
                          &L))
            return CC3D_ERR_UNSUPPORTED;
        const int tiles = L.g.tiles_per_cb * L.g.ncolblk * (L.tstack ? (T + 1) / 2 : T) * L.ncoblk;
        // history frames the forward call hands to a copy engine (when the side stream is available)
        const int n_ce = P == 0 ? 0 : (L.pair && !L.tstack ? P : (L.tstack ? 1 : 0));
        n = snprintf(buf, len,
                     "kernel=%s pair=%d two_frame=%d up2=%d channel_block=%d NT=%d nsplit=%d cout_blocks=%d "
                     "row_groups=%d column_block=%d row_aligned=%d window_rows=%d tap_rows_per_weight_stage=%d "
                     "window_stages=%d weight_stages=%d window_stage_bytes=%d weight_stage_bytes=%d acc_stages=%d "
                     "mma_warps=%d split_n=%d tmem_cols=%d smem_bytes=%zu tiles=%d history_frames_on_copy_engine=%d",
                     L.tstack ? "tc2s_bf16_kernel" : (L.pair ? "tc2_bf16_kernel" : "tc_bf16_kernel"), L.pair,
                     L.tstack, L.up2, plan_cb(p), L.NT, L.nsplit, L.ncoblk, L.g.sub, L.g.S, L.g.row_aligned, L.g.nrows,
                     L.rb, L.na, L.nb, L.a_stage_bytes, L.b_stage_bytes, L.acc_stages, L.issuers, L.split_n,
                     L.tmem_cols, L.smem_bytes, tiles, n_ce);
    }
    if (n < 0 || (size_t)n >= len) {
        buf[0] = 0;
        return CC3D_ERR_INVALID_ARG;
    }
    return CC3D_OK;
}

cc3d_status cc3d_debug_set_wait_budget_ns(cc3d_plan_t plan, unsigned long long ns)
{
    if (plan == nullptr || ns == 0) return CC3D_ERR_INVALID_ARG;
    plan->wait_ns = ns;
    return CC3D_OK;
}

cc3d_status cc3d_debug_set_fault(cc3d_plan_t plan, int mode)
{
    if (plan == nullptr || mode < 0 || mode > 2) return CC3D_ERR_INVALID_ARG;
    plan->fault = mode;
    return CC3D_OK;
}

cc3d_status cc3d_debug_set_schedule(cc3d_plan_t plan, int knob, int value)
{
    // [lo, hi] of every knob; value -1 restores the measured default
    static const int range[CC3D_SCHED_COUNT][2] = {
        {0, 1}, {0, 1}, {0, 1}, {0, 1}, {1, 2}, {1, 4}, {1, kMaxAccStages}, {1, 3}, {2, kMaxRingStages},
        {2, kMaxRingStages}, {0, 3}, {16, 32}};
    if (plan == nullptr || knob < 0 || knob >= CC3D_SCHED_COUNT) return CC3D_ERR_INVALID_ARG;
    if (value != -1) {
        if (value < range[knob][0] || value > range[knob][1]) return CC3D_ERR_INVALID_ARG;
        if (knob == CC3D_SCHED_ROW_GROUPS && value == 3) return CC3D_ERR_INVALID_ARG;
        if (knob == CC3D_SCHED_TAP_ROWS && value == 2) return CC3D_ERR_INVALID_ARG;
        if (knob == CC3D_SCHED_CHANNEL_BLOCK && value != 16 && value != 32) return CC3D_ERR_INVALID_ARG;
    }
    plan->ov.v[knob] = value;
    return CC3D_OK;
}

static size_t esize(const cc3d_plan_s* p) { return p->dtype == CC3D_F32 ? 4 : 2; }



cc3d_status cc3d_reset(cc3d_plan_t plan, void* cache, void* stream)
{
    if (plan == nullptr || cache == nullptr) return CC3D_ERR_INVALID_ARG;
    if (!aligned_to(cache, plan->dtype == CC3D_F32 ? 4 : 16)) return CC3D_ERR_ALIGNMENT;
    const cc3d_status where = pointer_check(cache);
    if (where != CC3D_OK) return where;
    const size_t bytes = (size_t)(plan->kt - 1) * plan->H * plan->W * plan->Cin * esize(plan);
    if (bytes == 0) return CC3D_OK;
    DeviceInfo* d = nullptr;
    cc3d_status st = device_info(&d);
    if (st != CC3D_OK) return st;
    if (!d->sm103) return CC3D_ERR_UNSUPPORTED;
    const cudaError_t e = zero_fill_launch(cache, bytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CC3D_OK : cuda_fail("zero fill launch", e);
}

cc3d_status cc3d_get_status(cc3d_plan_t plan, void* stream)
{
    if (plan == nullptr) return CC3D_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    cc3d_status st = device_info(&d);
    if (st != CC3D_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
    // one atomic exchange on the device reads and clears the word, so a bit that a kernel still
    // running elsewhere ors in is either in this read or left for the next one; the snapshot word
    // is shared, so the exchange and its read-back are serialised across host threads
    unsigned word = 0;
    {
        std::lock_guard<std::mutex> lock(g_status_mutex);
        e = status_take_launch(s);
        if (e == cudaSuccess) e = cudaMemcpyFromSymbolAsync(&word, g_status_taken, sizeof(word), 0,
                                                            cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    }
    if (e != cudaSuccess) return cuda_fail("read and clear the status word", e);
    return word != 0 ? CC3D_ERR_DEVICE_TIMEOUT : CC3D_OK;
}

}  // extern "C"

bool cc3d::plan_shape(cc3d_plan_t plan, PlanShape* out)
{
    if (plan == nullptr || out == nullptr) return false;
    out->Cin = plan->Cin;
    out->Cout = plan->Cout;
    out->H = plan->H;
    out->W = plan->W;
    out->Ho = plan->up2 ? 2 * plan->H : plan->H;
    out->Wo = plan->up2 ? 2 * plan->W : plan->W;
    out->kt = plan->kt;
    out->kh = plan->kh;
    out->kw = plan->kw;
    out->esize = (int)esize(plan);
    return true;
}

// Both forward entry points: y in the plan's dtype, or (out_u8, narrow-head plans) 8-bit pixels.
// With dry_run every check runs (arguments, device, configuration) and nothing is launched.
cc3d_status cc3d::forward_impl(cc3d_plan_t plan, int T, const void* x, const void* w, const void* b,
                               const void* res, const void* cache_in, void* cache_out, void* y, void* stream_,
                               bool out_u8, bool dry_run)
{
    if (plan == nullptr || T < 0) return CC3D_ERR_INVALID_ARG;
    const cc3d_plan_s& p = *plan;
    if (out_u8 && p.kind != K_TC_BF16_HEAD) return CC3D_ERR_UNSUPPORTED;
    cudaStream_t stream = static_cast<cudaStream_t>(stream_);
    const size_t es = esize(&p);
    const int P = p.kt - 1;
    const size_t frame_in = (size_t)p.H * p.W * p.Cin * es;
    // an upsampling plan's outputs (and residual) are 2H x 2W frames
    const size_t out_px = (size_t)p.H * p.W * (p.up2 ? 4 : 1);
    const size_t frame_out = out_px * p.Cout * (out_u8 ? 1 : es);
    const size_t n_x = (size_t)T * frame_in, n_y = (size_t)T * frame_out;
    const size_t n_cache = (size_t)P * frame_in;
    const size_t n_w = (size_t)p.Cout * p.kt * p.kh * p.kw * p.Cin * es, n_b = (size_t)p.Cout * es;

    // ---- presence
    if (P > 0 && cache_out == nullptr) return CC3D_ERR_INVALID_ARG;
    if (T > 0 && (x == nullptr || w == nullptr || y == nullptr)) return CC3D_ERR_INVALID_ARG;
    // every tile and unit index of the kernels stays within int (2^33 positions of even 16 bf16
    // channels are 275 GB, more than the device holds)
    if ((long long)T * p.H * p.W > (1LL << 33)) return CC3D_ERR_UNSUPPORTED;
    // ---- alignment.  fp32: one element.  bf16: 16 bytes for everything the tensor-core kernel
    // moves with TMA or 16-byte vectors (x, w, caches, and y / residual when Cout is a multiple
    // of 16); the narrow head stores y and reads the residual and bias per element.
    const void* all[] = {x, w, b, res, cache_in, cache_out, y};
    if (p.dtype == CC3D_F32) {
        for (const void* q : all)
            if (q != nullptr && !aligned_to(q, 4)) return CC3D_ERR_ALIGNMENT;
    } else {
        const uintptr_t out_align = (p.Cout % 16 == 0) ? 16 : 2;
        if (out_u8 && res && !aligned_to(res, 2)) return CC3D_ERR_ALIGNMENT;
        const void* a16[] = {x, w, cache_in, cache_out};
        for (const void* q : a16)
            if (q != nullptr && !aligned_to(q, 16)) return CC3D_ERR_ALIGNMENT;
        if ((y && !out_u8 && !aligned_to(y, out_align)) || (res && !aligned_to(res, out_align)) ||
            (b && !aligned_to(b, 2)))
            return CC3D_ERR_ALIGNMENT;
    }
    // ---- overlaps: outputs against everything else
    struct Span {
        const void* p;
        size_t n;
    };
    const size_t n_res = (size_t)T * out_px * p.Cout * es;
    const Span ins[] = {{T > 0 ? x : nullptr, n_x}, {T > 0 ? w : nullptr, n_w}, {T > 0 ? b : nullptr, n_b},
                        {T > 0 ? res : nullptr, n_res}, {cache_in, n_cache}};
    for (const Span& s : ins) {
        if (T > 0 && overlaps(y, n_y, s.p, s.n)) return CC3D_ERR_ALIAS;
        if (P > 0 && overlaps(cache_out, n_cache, s.p, s.n)) return CC3D_ERR_ALIAS;
    }
    if (T > 0 && P > 0 && overlaps(y, n_y, cache_out, n_cache)) return CC3D_ERR_ALIAS;
    // ---- device memory, of the current device
    for (const void* q : all) {
        if (q == nullptr) continue;
        const cc3d_status where = pointer_check(q);
        if (where != CC3D_OK) return where;
    }
    DeviceInfo* d = nullptr;
    cc3d_status st = device_info(&d);
    if (st != CC3D_OK) return st;
    if (!d->sm103) return CC3D_ERR_UNSUPPORTED;

    if (T == 0) {
        // only the history moves: cache_out = last P frames of cache_in (or zeros)
        if (P == 0 || dry_run) return CC3D_OK;
        const cudaError_t e = cache_update_launch(nullptr, cache_in, cache_out, 0, P, frame_in, stream);
        return e == cudaSuccess ? CC3D_OK : cuda_fail("cache update launch", e);
    }

    if (p.kind == K_SIMT_F32) {
        if (dry_run) return CC3D_OK;
        SimtLaunch L;
        L.T = T;
        L.H = p.H;
        L.W = p.W;
        L.Cin = p.Cin;
        L.Cout = p.Cout;
        L.kt = p.kt;
        L.kh = p.kh;
        L.kw = p.kw;
        L.x = static_cast<const float*>(x);
        L.cache_in = static_cast<const float*>(cache_in);
        L.w = static_cast<const float*>(w);
        L.bias = static_cast<const float*>(b);
        L.res = static_cast<const float*>(res);
        L.y = static_cast<float*>(y);
        cudaError_t e = simt_f32_launch(L, stream);
        if (e != cudaSuccess) return cuda_fail("fp32 kernel launch", e);
        if (P > 0 && (e = cache_update_launch(x, cache_in, cache_out, T, P, frame_in, stream)) != cudaSuccess)
            return cuda_fail("cache update launch", e);
        return CC3D_OK;
    }

    if (p.kind == K_TC_BF16_HEAD) {
        if (dry_run) {
            HeadLaunch hl;
            memset(&hl, 0, sizeof(hl));
            return head_configure(T, p.H, p.W, p.Cin, p.Cout, d->sms, &hl) ? CC3D_OK : CC3D_ERR_UNSUPPORTED;
        }
        return head_forward(p, *d, T, x, w, b, res, cache_in, cache_out, y, stream, out_u8);
    }
    if (p.kind == K_TC_BF16_STREAM) {
        if (dry_run) {
            StreamLaunch sl;
            memset(&sl, 0, sizeof(sl));
            return stream_configure(T, p.H, p.W, p.Cin, p.Cout, p.kt, d->sms, &sl) ? CC3D_OK : CC3D_ERR_UNSUPPORTED;
        }
        return stream_forward(p, *d, T, x, w, b, res, cache_in, cache_out, y, stream);
    }

    // ---- tensor-core path
    TcLaunch L;
    memset(&L, 0, sizeof(L));
    const int CB = plan_cb(p);
    if (!tc_configure(CB, T, p.H, p.W, p.Cin, p.Cout, p.kt, p.kh, res != nullptr, p.up2 != 0, &p.ov, &L))
        return CC3D_ERR_UNSUPPORTED;
    if (dry_run) return CC3D_OK;
    if (p.fault == 2) return cuda_fail("injected tensor-map encode failure");  // nothing launched
    const CUtensorMapSwizzle sw = CB == 64   ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : CB == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                               : CU_TENSOR_MAP_SWIZZLE_32B;
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    {
        const cuuint64_t dims[4] = {(cuuint64_t)p.Cin, (cuuint64_t)p.W, (cuuint64_t)p.H, (cuuint64_t)T};
        const cuuint64_t strides[3] = {(cuuint64_t)p.Cin * 2, (cuuint64_t)p.W * p.Cin * 2,
                                       (cuuint64_t)p.H * p.W * p.Cin * 2};
        const cuuint32_t box[4] = {(cuuint32_t)CB, (cuuint32_t)L.g.Sp, (cuuint32_t)L.g.nrows, 1};
        if (g_encode(&L.map_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_fail("cuTensorMapEncodeTiled (x_chunk)");
        if (cache_in != nullptr && P > 0) {
            const cuuint64_t cdims[4] = {(cuuint64_t)p.Cin, (cuuint64_t)p.W, (cuuint64_t)p.H, (cuuint64_t)P};
            if (g_encode(&L.map_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache_in), cdims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cuda_fail("cuTensorMapEncodeTiled (cache_in)");
        }
    }
    {
        // weights [Cout][kt*ks*ks][Cin] seen as (ci, co, tap) so one box holds ks * rb K-major tap tiles
        const int taps = p.kt * p.kh * p.kw;
        const cuuint64_t dims[3] = {(cuuint64_t)p.Cin, (cuuint64_t)p.Cout, (cuuint64_t)taps};
        const cuuint64_t strides[2] = {(cuuint64_t)taps * p.Cin * 2, (cuuint64_t)p.Cin * 2};
        const cuuint32_t box[3] = {(cuuint32_t)CB, (cuuint32_t)(L.pair ? L.NT / 2 : L.NT),
                                   (cuuint32_t)(p.kh * L.rb)};
        if (g_encode(&L.map_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cuda_fail("cuTensorMapEncodeTiled (w)");
        if (L.tstack) {
            // the two-frame schedule's stacked stages: all NT rows of rb tap rows per block
            const cuuint32_t box2[3] = {(cuuint32_t)CB, (cuuint32_t)L.NT, (cuuint32_t)(p.kh * L.rb)};
            if (g_encode(&L.map_w2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), dims, strides, box2,
                         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return cuda_fail("cuTensorMapEncodeTiled (w, two-frame stages)");
        }
    }
    L.has_cache = cache_in != nullptr && P > 0;
    L.bias = b;
    L.res = res;
    L.y = y;
    L.v32 = ((reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(res)) & 31) == 0 ? 1 : 0;
    L.x = x;
    L.cache_in = P > 0 ? cache_in : nullptr;
    L.cache_out = cache_out;
    L.status = d->status;
    L.wait_ns = p.wait_ns;
    L.fault = p.fault;
    // tiles: one per output frame, or per pair of output frames in the two-frame schedule
    const int ntiles = L.g.tiles_per_cb * L.g.ncolblk * (L.tstack ? (T + 1) / 2 : T) * L.ncoblk;
    L.nfull = ntiles;
    L.nunits = ntiles;
    if (L.pair) {
        const int npairs = (ntiles + 1) / 2;
        L.grid = 2 * (npairs < d->sms / 2 ? npairs : d->sms / 2);
    } else {
        // A short last wave (at most half the SMs busy) of two-row-group tiles with one
        // accumulator buffer: split those tiles into one-row-group units, each computed by both
        // MMA warps on half of the output channels, so every block gets about the same work
        // (c384 -> 192 at 90 x 160: 228 tiles = 152 whole + 76 split over 152 SMs).
        const bool allow = p.ov.get(CC3D_SCHED_SPLIT_TAIL, 1) != 0;
        const int R = ntiles % d->sms;
        if (allow && L.acc_stages == 1 && L.issuers == 2 && !L.split_n && !L.up2 && L.nsplit == 1 &&
            L.g.sub == 2 && L.NT % 32 == 0 && R > 0 && 2 * R <= d->sms) {
            L.nfull = ntiles - R;
            L.nunits = L.nfull + 2 * R;
        }
        L.grid = L.nunits < d->sms ? L.nunits : d->sms;
    }
    // ---- the new history: cache_out slot j = frame T + j of the stack (cache_in frames, then x
    // frames; zeros for a missing cache_in), moved by the copy engines while the kernel runs
    // Slots [0, n_ce) go to the copy engine: all of them for the one-frame pair kernel, the first
    // of the two-frame kernel's (one 2-frame history would outlast its launch on one engine), none
    // for the one-SM kernel.
    const int n_ce = P == 0 ? 0 : (L.pair && !L.tstack ? P : (L.tstack ? 1 : 0));
    const bool side_copy = n_ce > 0 && side_stream_ready(plan);
    L.hist_from = side_copy ? n_ce : 0;
    L.copy_hist = L.hist_from < P ? 1 : 0;
    if (side_copy) {
        // slots [0, n_ce) of cache_out as one byte range: the first jx slots from cache_in (or
        // zeros), the rest from x; each side stream moves an equal share of it
        const int jx = P > T ? P - T : 0;
        const size_t n_in = (size_t)(jx < n_ce ? jx : n_ce) * frame_in, n_all = (size_t)n_ce * frame_in;
        const char* src_in = static_cast<const char*>(cache_in) + (size_t)T * frame_in;
        const char* src_x = static_cast<const char*>(x) + (size_t)(T + jx - P) * frame_in - n_in;
        char* dst = static_cast<char*>(cache_out);
        const size_t share = ((n_all + cc3d_plan_s::kSide - 1) / cc3d_plan_s::kSide + 255) & ~size_t(255);
        cudaError_t e = cudaEventRecord(plan->fork, stream);
        for (int i = 0; e == cudaSuccess && i < cc3d_plan_s::kSide; ++i) {
            cudaStream_t ss = plan->side[i];
            e = cudaStreamWaitEvent(ss, plan->fork, 0);
            const size_t a0 = (size_t)i * share < n_all ? (size_t)i * share : n_all;
            const size_t a1 = a0 + share < n_all ? a0 + share : n_all;
            // [a0, a1) split at n_in into its cache_in part and its x part
            const size_t m = a1 < n_in ? a1 : (a0 > n_in ? a0 : n_in);
            if (e == cudaSuccess && m > a0)
                e = cache_in != nullptr ? cudaMemcpyAsync(dst + a0, src_in + a0, m - a0, cudaMemcpyDeviceToDevice, ss)
                                        : cudaMemsetAsync(dst + a0, 0, m - a0, ss);
            if (e == cudaSuccess && a1 > m) e = cudaMemcpyAsync(dst + m, src_x + m, a1 - m, cudaMemcpyDeviceToDevice, ss);
            if (e == cudaSuccess) e = cudaEventRecord(plan->join[i], ss);
        }
        if (e != cudaSuccess) return cuda_fail("history copy on the side streams", e);
    }
    cudaError_t e = tc_launch(CB, L, stream);
    if (e != cudaSuccess) return cuda_fail("tensor-core kernel launch", e);
    for (int i = 0; side_copy && i < cc3d_plan_s::kSide; ++i)
        if ((e = cudaStreamWaitEvent(stream, plan->join[i], 0)) != cudaSuccess)
            return cuda_fail("join of the history copy", e);
    return CC3D_OK;
}

extern "C" {

cc3d_status cc3d_forward_chunk(cc3d_plan_t plan, int T, const void* x, const void* w, const void* b,
                               const void* res, const void* cache_in, void* cache_out, void* y, void* stream)
{
    return forward_impl(plan, T, x, w, b, res, cache_in, cache_out, y, stream, false, false);
}

cc3d_status cc3d_forward_chunk_u8(cc3d_plan_t plan, int T, const void* x, const void* w, const void* b,
                                  const void* res, const void* cache_in, void* cache_out, void* y_u8, void* stream)
{
    return forward_impl(plan, T, x, w, b, res, cache_in, cache_out, y_u8, stream, true, false);
}

}  // extern "C"
