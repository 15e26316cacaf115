// cc3d_tc_common.cuh -- pieces shared by the one-SM and the SM-pair tensor-core kernels: tile
// coordinates, failure recording and the epilogue's bias / residual / bf16 store helpers.
#pragma once
#include <cuda_bf16.h>

#include "cc3d_internal.h"
#include "cc3d_ptx.cuh"

namespace cc3d {
namespace tcc {
using namespace ptx;

constexpr int kThreads = 256;
constexpr int kMaxStages = kMaxRingStages;
constexpr int kMaxAcc = kMaxAccStages;
// sleep between polls of waits that usually last long (the epilogue waits for a whole tile), so
// that those warps leave issue slots to the MMA warps sharing their schedulers; the loader polls
// without sleeping (a late refill costs more than the issue slots)
constexpr uint32_t kLoaderSleepNs = 0;
constexpr uint32_t kEpilogueSleepNs = 256;

struct TileCoord {
    int t, w0, f0, hstart, co0;
};

__device__ __forceinline__ int floor_div(int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); }

__device__ __forceinline__ TileCoord tile_coord(const TcLaunch& L, int tile)
{
    // order: frame fastest, then output-channel block (both reuse the same input windows), then
    // the position inside the column block, then the column block
    TileCoord c;
    c.t = tile % L.T;
    const int r0 = tile / L.T;
    c.co0 = (r0 % L.ncoblk) * L.nsplit * L.NT;
    const int r = r0 / L.ncoblk;
    const int i = r % L.g.tiles_per_cb;
    const int cbk = r / L.g.tiles_per_cb;
    c.w0 = cbk * L.g.S;
    c.f0 = i * L.g.tile_f + (L.g.row_aligned ? 1 : 0);
    c.hstart = floor_div(c.f0 - L.g.halo * (L.g.Sp + 1), L.g.Sp);  // padded row of the first input read
    return c;
}

__device__ __forceinline__ void record_failure(const TcLaunch& L, unsigned bit, volatile int* abort_flag)
{
    *abort_flag = 1;
    atomicOr(L.status, bit);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat16 l = __float2bfloat16_rn(lo);
    const __nv_bfloat16 h = __float2bfloat16_rn(hi);
    return (uint32_t)__bfloat16_as_ushort(l) | ((uint32_t)__bfloat16_as_ushort(h) << 16);
}

// 16 bias values from shared memory as four 16-byte broadcast loads (co0 is a multiple of 16 and
// the bias array is 16-byte aligned): a quarter of the shared-memory wavefronts of scalar loads,
// which share the data path with the tensor core's operand reads.
__device__ __forceinline__ void load_bias16(const float* s_bias, int co0, float* b)
{
    const float4* p = reinterpret_cast<const float4*>(s_bias + co0);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float4 q = p[k];
        b[4 * k] = q.x;
        b[4 * k + 1] = q.y;
        b[4 * k + 2] = q.z;
        b[4 * k + 3] = q.w;
    }
}

// 16 accumulator columns of one output position: + bias (+ residual) -> bf16 -> global.
__device__ __forceinline__ void store16(const uint32_t* r, const float* s_bias, int co0, size_t px, int Cout,
                                        bool wide, const __nv_bfloat16* res, __nv_bfloat16* y)
{
    float v[16];
    load_bias16(s_bias, co0, v);
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = __fadd_rn(__uint_as_float(r[k]), v[k]);
    if (wide) {
        const size_t off = px * Cout + co0;
        if (res != nullptr) {
            const uint4 r0 = __ldg(reinterpret_cast<const uint4*>(res + off));
            const uint4 r1 = __ldg(reinterpret_cast<const uint4*>(res + off + 8));
            const uint32_t rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                v[2 * k] = __fadd_rn(v[2 * k], bf16_lo(rr[k]));
                v[2 * k + 1] = __fadd_rn(v[2 * k + 1], bf16_hi(rr[k]));
            }
        }
        uint4 o0, o1;
        o0.x = pack_bf16x2(v[0], v[1]);
        o0.y = pack_bf16x2(v[2], v[3]);
        o0.z = pack_bf16x2(v[4], v[5]);
        o0.w = pack_bf16x2(v[6], v[7]);
        o1.x = pack_bf16x2(v[8], v[9]);
        o1.y = pack_bf16x2(v[10], v[11]);
        o1.z = pack_bf16x2(v[12], v[13]);
        o1.w = pack_bf16x2(v[14], v[15]);
        *reinterpret_cast<uint4*>(y + off) = o0;
        *reinterpret_cast<uint4*>(y + off + 8) = o1;
    } else {
        // narrow output head: fewer than 16 channels, element stores
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const int co = co0 + k;
            if (co < Cout) {
                const size_t off = px * Cout + co;
                float o = v[k];
                if (res != nullptr) o = __fadd_rn(o, __bfloat162float(res[off]));
                y[off] = __float2bfloat16_rn(o);
            }
        }
    }
}

// 16 accumulator columns + bias + residual held in registers (8 bf16 pairs) -> bf16 -> global
__device__ __forceinline__ void store16_res(const uint32_t* r, const float* s_bias, int co0, __nv_bfloat16* yp,
                                            const uint4 ra, const uint4 rb)
{
    const uint32_t rr[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
    float bv[16];
    load_bias16(s_bias, co0, bv);
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float lo = __fadd_rn(__fadd_rn(__uint_as_float(r[2 * k]), bv[2 * k]), bf16_lo(rr[k]));
        const float hi = __fadd_rn(__fadd_rn(__uint_as_float(r[2 * k + 1]), bv[2 * k + 1]), bf16_hi(rr[k]));
        o[k] = pack_bf16x2(lo, hi);
    }
    reinterpret_cast<uint4*>(yp)[0] = make_uint4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<uint4*>(yp)[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// 32-byte global accesses (8 x 32 bits; the address must be 32-byte aligned): half the load /
// store instructions of 16-byte ones for the same bytes
__device__ __forceinline__ void ld_nc_v8(const void* p, uint32_t* r)
{
    asm volatile("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "l"(p));
}

__device__ __forceinline__ void st_v8(void* p, const uint32_t* v)
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]), "r"(v[2]),
                 "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

// 16 accumulator columns + bias (+ 16 bf16 residual values when RES) -> bf16 -> one 32-byte store
template <bool RES>
__device__ __forceinline__ void store16_v8(const uint32_t* r, const float* s_bias, int co0, __nv_bfloat16* yp,
                                           const uint32_t* rr)
{
    float bv[16];
    load_bias16(s_bias, co0, bv);
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        float lo = __fadd_rn(__uint_as_float(r[2 * k]), bv[2 * k]);
        float hi = __fadd_rn(__uint_as_float(r[2 * k + 1]), bv[2 * k + 1]);
        if (RES) {
            lo = __fadd_rn(lo, bf16_lo(rr[k]));
            hi = __fadd_rn(hi, bf16_hi(rr[k]));
        }
        o[k] = pack_bf16x2(lo, hi);
    }
    st_v8(yp, o);
}

// The temporal cache update done by otherwise idle warps: cache_out[j] = frame T + j of the
// stack (the P cache_in frames, then the T frames of x; zeros for a missing cache_in), for
// hist_from <= j < P (the host has a copy engine move the slots before hist_from).
// `nwarps` warps of every block take part (this one is number `cw`).  In each 16-byte step the
// 32 lanes of a warp cover 512 contiguous bytes, and each thread has 16 loads in flight before
// its stores.
__device__ __forceinline__ void copy_history(const TcLaunch& L, int P, int cw, int nwarps, int lane)
{
    const size_t frame_chunks = (size_t)L.H * L.W * L.Cin * 2 / 16;
    const size_t total = (size_t)P * frame_chunks;
    const size_t first = (size_t)L.hist_from * frame_chunks;  // slots before hist_from: copy engine
    const uint4* xin = reinterpret_cast<const uint4*>(L.x);
    const uint4* cin = reinterpret_cast<const uint4*>(L.cache_in);
    uint4* cout_ = reinterpret_cast<uint4*>(L.cache_out);
    constexpr int U = 16;
    const size_t span = (size_t)32 * U;  // 16-byte elements of one warp step
    const size_t stride = (size_t)gridDim.x * nwarps * span;
    for (size_t base = first + ((size_t)blockIdx.x * nwarps + cw) * span; base < total; base += stride) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t i = base + (size_t)u * 32 + lane;
            v[u] = make_uint4(0, 0, 0, 0);
            if (i < total) {
                const int j = (int)(i / frame_chunks);
                const size_t o = i - (size_t)j * frame_chunks;
                const int src = L.T + j;  // index in the stack of cache_in and x frames
                if (src >= P)
                    v[u] = __ldg(xin + (size_t)(src - P) * frame_chunks + o);
                else if (cin != nullptr)
                    v[u] = __ldg(cin + (size_t)src * frame_chunks + o);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const size_t i = base + (size_t)u * 32 + lane;
            if (i < total) __stcs(cout_ + i, v[u]);
        }
    }
}

// Epilogues that hand accumulators back before touching memory: read NT <= MAXC columns of this
// thread's lane into registers (tmem_read_quarter, then tmem_ld_wait), optionally zero them
// (tmem_zero_quarter, then tmem_st_wait), release them, and only then add bias / residual and
// store (store_quarter): the MMA warps wait for tensor-memory reads only, never for memory.
template <int MAXC>
__device__ __forceinline__ void tmem_read_quarter(uint32_t tbase, int NT, uint32_t* r)
{
#pragma unroll
    for (int g = 0; g < MAXC / 32; ++g) {
        if (g * 32 + 32 <= NT)
            tmem_ld_32x32b_x32(tbase + (uint32_t)(g * 32), r + g * 32);
        else if (g * 32 + 16 == NT)
            tmem_ld_32x32b_x16(tbase + (uint32_t)(g * 32), r + g * 32);
    }
}

template <int MAXC>
__device__ __forceinline__ void tmem_zero_quarter(uint32_t tbase, int NT)
{
#pragma unroll
    for (int g = 0; g < MAXC / 32; ++g) {
        if (g * 32 + 32 <= NT)
            tmem_st_32x32b_x32_zero(tbase + (uint32_t)(g * 32));
        else if (g * 32 + 16 == NT)
            tmem_st_32x32b_x16_zero(tbase + (uint32_t)(g * 32));
    }
}

// bias (+ residual) and the bf16 stores of NT <= MAXC accumulator columns held in registers, output
// channels co0 .. co0 + NT - 1 of position px, 32 columns at a time; with `v32` every 16 channels
// move as one 32-byte load / store
template <int MAXC>
__device__ __forceinline__ void store_quarter(const uint32_t* r, int NT, int co0, size_t px, const float* s_bias,
                                              int Cout, const __nv_bfloat16* res, __nv_bfloat16* y, bool v32)
{
    __nv_bfloat16* yp = y + px * Cout + co0;
    const __nv_bfloat16* rq = res + px * Cout + co0;
    if (v32) {
#pragma unroll
        for (int g = 0; g < MAXC / 32; ++g) {
            if (g * 32 + 16 > NT) break;
            const bool two = g * 32 + 32 <= NT;
            if (res != nullptr) {
                uint32_t rr[16];
                ld_nc_v8(rq + g * 32, rr);
                if (two) ld_nc_v8(rq + g * 32 + 16, rr + 8);
                store16_v8<true>(r + g * 32, s_bias, co0 + g * 32, yp + g * 32, rr);
                if (two) store16_v8<true>(r + g * 32 + 16, s_bias, co0 + g * 32 + 16, yp + g * 32 + 16, rr + 8);
            } else {
                store16_v8<false>(r + g * 32, s_bias, co0 + g * 32, yp + g * 32, nullptr);
                if (two) store16_v8<false>(r + g * 32 + 16, s_bias, co0 + g * 32 + 16, yp + g * 32 + 16, nullptr);
            }
        }
        return;
    }
    const uint4* rp = reinterpret_cast<const uint4*>(rq);
#pragma unroll
    for (int g = 0; g < MAXC / 32; ++g) {
        if (g * 32 + 16 > NT) break;
        const bool two = g * 32 + 32 <= NT;
        if (res != nullptr) {
            uint4 rv[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) rv[k] = (k < 2 || two) ? __ldg(rp + 4 * g + k) : make_uint4(0, 0, 0, 0);
            store16_res(r + g * 32, s_bias, co0 + g * 32, yp + g * 32, rv[0], rv[1]);
            if (two) store16_res(r + g * 32 + 16, s_bias, co0 + g * 32 + 16, yp + g * 32 + 16, rv[2], rv[3]);
        } else {
            store16(r + g * 32, s_bias, co0 + g * 32, px, Cout, true, nullptr, y);
            if (two) store16(r + g * 32 + 16, s_bias, co0 + g * 32 + 16, px, Cout, true, nullptr, y);
        }
    }
}

// the epilogue warp is done reading this accumulator stage: let the MMA warps overwrite it
__device__ __forceinline__ void release_acc(uint64_t* bar, int lane)
{
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// One accumulator slice of the epilogue: NT fp32 columns of this thread's output position,
// read from tensor memory 32 (or 16) at a time, + bias (+ residual), rounded to bf16 and stored.
// `release()` runs once, right after the last columns are in registers, when `last` is set (the
// accumulators may then be overwritten).  With a residual and NT <= 128 the whole residual row is
// fetched in one batch first, so the thread waits for memory once per slice.  With `v32` (y and
// the residual 32-byte aligned, Cout a multiple of 16) every 16 channels move as one 32-byte
// access instead of two 16-byte ones.
template <typename Release>
__device__ __forceinline__ void epilogue_slice(uint32_t tbase, int NT, int co_base, size_t px, bool valid, bool last,
                                               const float* s_bias, int Cout, bool wide,
                                               const __nv_bfloat16* res, __nv_bfloat16* y, bool v32,
                                               Release release)
{
    if (res != nullptr && wide && NT <= 128 && v32) {
        uint32_t rr[64];
        const __nv_bfloat16* rp = res + px * Cout + co_base;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (valid && k * 16 < NT) {
                ld_nc_v8(rp + k * 16, rr + 8 * k);
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) rr[8 * k + u] = 0u;
            }
        }
        __nv_bfloat16* yp = y + px * Cout + co_base;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            if (g * 32 + 32 <= NT) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(g * 32), r);
                tmem_ld_wait();
                if (last && g * 32 + 32 == NT) release();
                if (valid) {
                    store16_v8<true>(r, s_bias, co_base + g * 32, yp + g * 32, rr + 16 * g);
                    store16_v8<true>(r + 16, s_bias, co_base + g * 32 + 16, yp + g * 32 + 16, rr + 16 * g + 8);
                }
            } else if (g * 32 + 16 == NT) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(tbase + (uint32_t)(g * 32), r);
                tmem_ld_wait();
                if (last) release();
                if (valid) store16_v8<true>(r, s_bias, co_base + g * 32, yp + g * 32, rr + 16 * g);
            }
        }
        return;
    }
    if (res != nullptr && wide && NT <= 128) {
        uint4 rv[16];
        const uint4* rp = reinterpret_cast<const uint4*>(res + px * Cout + co_base);
#pragma unroll
        for (int k = 0; k < 16; ++k) rv[k] = (valid && k * 8 < NT) ? __ldg(rp + k) : make_uint4(0, 0, 0, 0);
        __nv_bfloat16* yp = y + px * Cout + co_base;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            if (g * 32 + 32 <= NT) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + (uint32_t)(g * 32), r);
                tmem_ld_wait();
                if (last && g * 32 + 32 == NT) release();
                if (valid) {
                    store16_res(r, s_bias, co_base + g * 32, yp + g * 32, rv[4 * g], rv[4 * g + 1]);
                    store16_res(r + 16, s_bias, co_base + g * 32 + 16, yp + g * 32 + 16, rv[4 * g + 2],
                                rv[4 * g + 3]);
                }
            } else if (g * 32 + 16 == NT) {
                uint32_t r[16];
                tmem_ld_32x32b_x16(tbase + (uint32_t)(g * 32), r);
                tmem_ld_wait();
                if (last) release();
                if (valid) store16_res(r, s_bias, co_base + g * 32, yp + g * 32, rv[4 * g], rv[4 * g + 1]);
            }
        }
        return;
    }
    const bool wide32 = v32 && wide && res == nullptr;
    int cc = 0;
    for (; cc + 32 <= NT; cc += 32) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tbase + (uint32_t)cc, r);
        tmem_ld_wait();
        if (last && cc + 32 == NT) release();
        if (valid) {
            if (wide32) {
                store16_v8<false>(r, s_bias, co_base + cc, y + px * Cout + co_base + cc, nullptr);
                store16_v8<false>(r + 16, s_bias, co_base + cc + 16, y + px * Cout + co_base + cc + 16, nullptr);
            } else {
                store16(r, s_bias, co_base + cc, px, Cout, wide, res, y);
                store16(r + 16, s_bias, co_base + cc + 16, px, Cout, wide, res, y);
            }
        }
    }
    if (cc < NT) {  // NT % 32 == 16
        uint32_t r[16];
        tmem_ld_32x32b_x16(tbase + (uint32_t)cc, r);
        tmem_ld_wait();
        if (last) release();
        if (valid) {
            if (wide32)
                store16_v8<false>(r, s_bias, co_base + cc, y + px * Cout + co_base + cc, nullptr);
            else
                store16(r, s_bias, co_base + cc, px, Cout, wide, res, y);
        }
    }
}

}  // namespace tcc
}  // namespace cc3d
