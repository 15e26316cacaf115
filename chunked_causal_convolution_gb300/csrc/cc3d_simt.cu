// cc3d_simt.cu -- float32 causal conv on the CUDA cores, and the small copy kernels.
//
// The float32 path needs true fp32 products: TF32 tensor-core inputs keep 10
// mantissa bits, which puts the error of a 27*Cin-term sum far above a 1e-4
// relative bound.  Each thread owns one output position and 16 output
// channels and accumulates with fmaf in a fixed order (dt, dh, dw, ci), so the
// result does not depend on the chunking.  History frames come from the cache
// (or are zero without one) through the same arithmetic as frames of the chunk.
#include <cuda_runtime.h>

#include "cc3d_internal.h"

namespace cc3d {
namespace {

constexpr int kCoGroup = 16;
constexpr int kThreads = 128;

__global__ void __launch_bounds__(kThreads) simt_f32_kernel(SimtLaunch L)
{
    const int P = L.kt - 1;
    const int ph = (L.kh - 1) / 2, pw = (L.kw - 1) / 2;
    const long long npos = (long long)L.T * L.H * L.W;
    const int ngroups = (L.Cout + kCoGroup - 1) / kCoGroup;
    const long long item = (long long)blockIdx.x * kThreads + threadIdx.x;
    if (item >= npos * ngroups) return;
    const int g = (int)(item / npos);
    const long long pos = item - (long long)g * npos;
    const int w = (int)(pos % L.W);
    const int h = (int)((pos / L.W) % L.H);
    const int t = (int)(pos / ((long long)L.W * L.H));
    const int co0 = g * kCoGroup;
    const int nco = min(kCoGroup, L.Cout - co0);
    const size_t frame = (size_t)L.H * L.W * L.Cin;
    const size_t wtap = (size_t)L.Cin;
    const size_t wco = (size_t)L.kt * L.kh * L.kw * L.Cin;

    float acc[kCoGroup];
#pragma unroll
    for (int k = 0; k < kCoGroup; ++k) acc[k] = 0.0f;

    for (int dt = 0; dt < L.kt; ++dt) {
        // frame t + dt of the extended stack concat(cache, x)
        const int te = t + dt;
        const float* src = nullptr;
        if (te >= P)
            src = L.x + (size_t)(te - P) * frame;
        else if (L.cache_in != nullptr)
            src = L.cache_in + (size_t)te * frame;
        for (int dh = 0; dh < L.kh; ++dh) {
            const int hs = h + dh - ph;
            if (hs < 0 || hs >= L.H) continue;
            for (int dw = 0; dw < L.kw; ++dw) {
                const int ws = w + dw - pw;
                if (ws < 0 || ws >= L.W) continue;
                const float* xp = src ? src + ((size_t)hs * L.W + ws) * L.Cin : nullptr;
                const float* wp = L.w + (size_t)co0 * wco + (((size_t)dt * L.kh + dh) * L.kw + dw) * wtap;
                for (int ci = 0; ci < L.Cin; ++ci) {
                    const float xv = xp ? __ldg(xp + ci) : 0.0f;
#pragma unroll
                    for (int k = 0; k < kCoGroup; ++k)
                        if (k < nco) acc[k] = fmaf(__ldg(wp + (size_t)k * wco + ci), xv, acc[k]);
                }
            }
        }
    }
    const size_t out = (((size_t)t * L.H + h) * L.W + w) * L.Cout + co0;
#pragma unroll
    for (int k = 0; k < kCoGroup; ++k) {
        if (k >= nco) break;
        float v = acc[k];
        if (L.bias) v = __fadd_rn(v, __ldg(L.bias + co0 + k));
        if (L.res) v = __fadd_rn(v, __ldg(L.res + out + k));
        L.y[out + k] = v;
    }
}

template <typename V>
__global__ void cache_update_kernel(const V* __restrict__ x, const V* __restrict__ cache_in, V* __restrict__ cache_out,
                                    int T, int P, size_t frame_chunks)
{
    const size_t total = (size_t)P * frame_chunks;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int j = (int)(i / frame_chunks);
        const size_t o = i - (size_t)j * frame_chunks;
        const int src = T + j;  // index in concat(cache_in, x)
        V v{};
        if (src >= P)
            v = __ldg(x + (size_t)(src - P) * frame_chunks + o);
        else if (cache_in != nullptr)
            v = __ldg(cache_in + (size_t)src * frame_chunks + o);
        cache_out[i] = v;
    }
}

template <typename V>
__global__ void zero_fill_kernel(V* p, size_t n)
{
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        p[i] = V{};
}

int grid_for(size_t n, int threads)
{
    size_t b = (n + threads - 1) / threads;
    if (b > 152 * 16) b = 152 * 16;
    if (b < 1) b = 1;
    return (int)b;
}

}  // namespace

cudaError_t simt_f32_launch(const SimtLaunch& L, cudaStream_t stream)
{
    const long long npos = (long long)L.T * L.H * L.W;
    const long long items = npos * ((L.Cout + kCoGroup - 1) / kCoGroup);
    if (items <= 0) return cudaSuccess;
    const long long blocks = (items + kThreads - 1) / kThreads;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
    simt_f32_kernel<<<(unsigned)blocks, kThreads, 0, stream>>>(L);
    return cudaGetLastError();
}

cudaError_t cache_update_launch(const void* x, const void* cache_in, void* cache_out, int T, int P,
                                size_t frame_bytes, cudaStream_t stream)
{
    if (P <= 0) return cudaSuccess;
    const uintptr_t a = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(cache_in) |
                        reinterpret_cast<uintptr_t>(cache_out);
    if (frame_bytes % 16 == 0 && (a & 15u) == 0) {
        const size_t chunks = frame_bytes / 16;
        cache_update_kernel<uint4><<<grid_for((size_t)P * chunks, 256), 256, 0, stream>>>(
            static_cast<const uint4*>(x), static_cast<const uint4*>(cache_in), static_cast<uint4*>(cache_out), T, P,
            chunks);
    } else {
        const size_t words = frame_bytes / 4;  // element sizes are 2 or 4 bytes and frames hold whole words
        cache_update_kernel<uint32_t><<<grid_for((size_t)P * words, 256), 256, 0, stream>>>(
            static_cast<const uint32_t*>(x), static_cast<const uint32_t*>(cache_in),
            static_cast<uint32_t*>(cache_out), T, P, words);
    }
    return cudaGetLastError();
}

cudaError_t zero_fill_launch(void* p, size_t bytes, cudaStream_t stream)
{
    if (bytes == 0) return cudaSuccess;
    if (bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0)
        zero_fill_kernel<uint4><<<grid_for(bytes / 16, 256), 256, 0, stream>>>(static_cast<uint4*>(p), bytes / 16);
    else
        zero_fill_kernel<uint32_t><<<grid_for(bytes / 4, 256), 256, 0, stream>>>(static_cast<uint32_t*>(p), bytes / 4);
    return cudaGetLastError();
}

}  // namespace cc3d
