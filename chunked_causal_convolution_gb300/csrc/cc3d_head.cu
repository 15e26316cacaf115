// cc3d_head.cu -- the causal 3x3x3 convolution for narrow outputs (Cout <= 5, e.g. an RGB head).
//
// With a handful of output channels the implicit GEMM of the wide kernels pads N to 16 and
// re-reads every staged activation tile once per tap: it is bound by shared-memory operand
// reads at a fraction of HBM bandwidth.  This kernel stacks the nine spatial taps into N:
//
//   D[h, t][p][(dh, dw, co)] = sum_{dt, ci} x[frame t + dt - 2][row h][position p][ci] * W[co][dt][dh][dw][ci]
//   y[t][h][w][co]           = sum_{dh, dw} D[h + dh - 1, t][w + dw - 1][(dh, dw, co)]   (+ bias, + residual)
//
// One MMA (M = 128 input positions, N = 32 or 48 >= 9 * Cout, K = 16 channels) reads a staged
// input row once per temporal tap.  The epilogue combines neighbouring positions (warp shuffles)
// and neighbouring rows (running sums kept in registers).  A block walks a contiguous run of rows
// of one column strip (126 output pixels = 128 input positions with the halo), input row by input
// row; every input row (all channels, the chunk's frames and the two history frames) is loaded
// into shared memory once -- exactly the 128 positions the MMA reads -- and the new history (the
// last two input frames) is written back from there (TMA stores from a swizzle-atom boundary on,
// a warp copy for the strip's first pixels).  Rows are dealt out to the blocks in equal runs, so
// there is no tail wave.
//
// Accumulation order of one output (t, h, w, co), fixed whatever the chunking: inside the tensor
// core dt, channel block, 16-channel step; then ((dh = 0) + (dh = 1)) + (dh = 2), each dh term
// being ((dw = 0) + (dw = 1)) + (dw = 2); then the bias, then the residual.
#include <cuda_bf16.h>

#include "cc3d_internal.h"
#include "cc3d_ptx.cuh"
#include "cc3d_tc_common.cuh"

namespace cc3d {
using namespace ptx;
using namespace tcc;

namespace {

constexpr int kHeadCB = 32;              // channels per staged block: 64-byte rows, 64-byte swizzle
constexpr int kHeadMaxStages = 8;        // input-row stages
constexpr int kHeadSlots = 2;            // input rows whose sums sit in tensor memory at once
constexpr int kHeadPos = 128;            // input positions per strip (the MMA's M)
constexpr int kHeadOut = kHeadPos - 2;   // output pixels per strip
constexpr int kHeadLead = 1;             // staged positions before the strip's first output pixel
constexpr int kHeadBox = 128;            // staged positions: w0 - 1 .. w0 + 126 (the MMA's rows)
// the history of staged rows kHeadStoreRow .. kHeadBox - 1 (positions w0 + 7 .. w0 + 126) is stored
// by TMA, whose shared-memory source must start on a 512-byte swizzle atom (row 8); a warp copies
// rows 1 .. 7 (positions w0 .. w0 + 6).  Position w0 + 126 is the next strip's first pixel: both
// strips write the same bytes there.
constexpr int kHeadStoreRow = 8;
constexpr int kHeadEdge = 16;            // floats per (frame, warp, side) in the edge exchange

template <int COUT>
struct HeadShape {
    static constexpr int NCOL = 9 * COUT <= 32 ? 32 : 48;  // MMA N
    static constexpr int GMAX = NCOL == 32 ? 8 : 5;         // output frames per pass
    static constexpr int SLOT = GMAX * NCOL;                // tensor-memory columns per input row
};

int head_ncol(int Cout) { return 9 * Cout <= 32 ? 32 : 48; }
int head_gmax(int Cout) { return head_ncol(Cout) == 32 ? 8 : 5; }

// A run of output rows [h0, h1) of one column strip and one group of output frames.
struct HeadSeg {
    int t0, G, w0, h0, h1;
};

// Units are (frame group, strip, output row), row fastest; the block owns [ubeg, uend).
__device__ __forceinline__ HeadSeg head_segment(const HeadLaunch& L, long long u, long long uend)
{
    HeadSeg s;
    const int h = (int)(u % L.H);
    const long long r = u / L.H;
    const int cbk = (int)(r % L.ncolblk);
    const int fg = (int)(r / L.ncolblk);
    s.h0 = h;
    s.h1 = (int)((uend - u) < (long long)(L.H - h) ? h + (uend - u) : L.H);
    s.w0 = cbk * kHeadOut;
    s.t0 = fg * L.gmax;
    s.G = min(L.gmax, L.T - s.t0);
    return s;
}

__device__ __forceinline__ void head_fail(const HeadLaunch& L, unsigned bit, volatile int* abort_flag)
{
    *abort_flag = 1;
    atomicOr(L.status, bit);
}

template <int NCOL>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* v)
{
    tmem_ld_32x32b_x32(taddr, v);
    if constexpr (NCOL == 48) tmem_ld_32x32b_x16(taddr + 32, v + 32);
    tmem_ld_wait();
}

// The 8-bit output of a pixel value: the bf16 result mapped from [-1, 1] to [0, 255] in fp32
// (add, multiply, round to nearest even, clamp).
__device__ __forceinline__ uint8_t quant_u8(float o)
{
    const float v = __bfloat162float(__float2bfloat16_rn(o));
    const float t = __fmul_rn(__fadd_rn(v, 1.0f), 127.5f);
    return (uint8_t)rintf(fminf(fmaxf(t, 0.0f), 255.0f));
}

template <int COUT>
__global__ void __launch_bounds__(kThreads, 1) head_bf16_kernel(const __grid_constant__ HeadLaunch L)
{
    using Shape = HeadShape<COUT>;
    constexpr int NCOL = Shape::NCOL, GMAX = Shape::GMAX;
    constexpr uint32_t SLOT = Shape::SLOT;
    constexpr uint32_t ROWB = kHeadCB * 2;
    constexpr uint32_t SBO = 8 * ROWB;
    constexpr int KSTEPS = kHeadCB / 16;
    constexpr int EBUF = GMAX * 6 * 2 * kHeadEdge;  // floats per edge buffer: [frame][slot 0..5][side]

    extern __shared__ uint8_t dsm_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smW = sm;                                 // [dt][channel block] tiles of NCOL rows x 64 B
    uint8_t* smX = sm + (size_t)L.w_bytes;             // stages of [channel block][128 positions] x 64 B
    float* s_edge = reinterpret_cast<float*>(smX + (size_t)L.nstages * L.x_stage_bytes);  // [2][EBUF]

    __shared__ uint64_t x_full[kHeadMaxStages], x_empty[kHeadMaxStages], w_full, acc_full[kHeadSlots],
        acc_empty[kHeadSlots], mma_drain[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;
    __shared__ int s_ok[2][4];
    __shared__ float s_bias[8];

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int ncb = L.Cin / kHeadCB;
    const int nst = L.nstages;
    const unsigned long long budget = L.wait_ns;
    const long long ubeg = L.units * blockIdx.x / gridDim.x;
    const long long uend = L.units * (blockIdx.x + 1) / gridDim.x;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < nst; ++s) { mbar_init(&x_full[s], 1); mbar_init(&x_empty[s], 3); }  // 2 MMA warps + copy
        mbar_init(&w_full, 1);
        for (int s = 0; s < kHeadSlots; ++s) { mbar_init(&acc_full[s], 2); mbar_init(&acc_empty[s], 4); }
        mbar_init(&mma_drain[0], 1);
        mbar_init(&mma_drain[1], 1);
        fence_mbar_init();
    }
    {
        // weight rows 9 * COUT .. NCOL - 1 of every tile (the N padding) are zero; the TMA loads
        // fill the rows before them, so the two never touch the same bytes
        constexpr int pad16 = (NCOL - 9 * COUT) * ROWB / 16;
        const int ntiles = 3 * ncb;
        for (int i = threadIdx.x; i < ntiles * pad16; i += kThreads) {
            uint8_t* tile = smW + (size_t)(i / pad16) * NCOL * ROWB + 9 * COUT * ROWB;
            reinterpret_cast<uint4*>(tile)[i % pad16] = make_uint4(0, 0, 0, 0);
        }
    }
    for (int i = threadIdx.x; i < 2 * EBUF; i += kThreads) s_edge[i] = 0.0f;  // slots 0 and 5 stay zero
    if (threadIdx.x < 8) {
        const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(L.bias);
        s_bias[threadIdx.x] = (b != nullptr && (int)threadIdx.x < COUT) ? __bfloat162float(b[threadIdx.x]) : 0.0f;
    }
    if (warp == 2) {
        tmem_alloc(&tmem_base_sh, (uint32_t)L.tmem_cols);
        tmem_relinquish();
    }
    fence_proxy_async_smem();  // the zero padding is visible to the tensor core's reads
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA loader
        if (lane == 0) {
            prefetch_tensormap(&L.map_x);
            prefetch_tensormap(&L.map_w);
            if (L.has_cache) prefetch_tensormap(&L.map_cache);
            // all weights once: per (dt, channel block) a box of [9 taps (dh, dw)][COUT][32 channels]
            mbar_arrive_expect_tx(&w_full, (uint32_t)(3 * ncb * 9 * COUT * ROWB));
            for (int dt = 0; dt < 3; ++dt)
                for (int cb = 0; cb < ncb; ++cb)
                    tma_load_3d(smW + (size_t)(dt * ncb + cb) * NCOL * ROWB, &L.map_w, &w_full, cb * kHeadCB, 0,
                                dt * 9);
            int s = 0, ph = 0;
            int last_ph[kHeadMaxStages];
            for (int k = 0; k < kHeadMaxStages; ++k) last_ph[k] = -1;
            const uint32_t x_tx = (uint32_t)(ncb * kHeadBox * ROWB);
            bool skip_first = (L.fault == 1);
            bool ok = true;
            for (long long u = ubeg; ok && u < uend;) {
                const HeadSeg g = head_segment(L, u, uend);
                for (int hin = g.h0 - 1; ok && hin <= g.h1; ++hin) {
                    for (int j = 0; j < g.G + 2; ++j) {
                        const int tin = g.t0 - 2 + j;
                        if (!bounded_wait(&x_empty[s], ph ^ 1, budget, &abort_flag)) {
                            if (!abort_flag) head_fail(L, STATUS_TIMEOUT_LOADER, &abort_flag);
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&x_full[s], x_tx);
                        // history frames come from the cache (or the zero fill of an out-of-range frame)
                        const CUtensorMap* map = &L.map_x;
                        int tc = tin;
                        if (tin < 0 && L.has_cache) { map = &L.map_cache; tc = tin + 2; }
                        if (!skip_first)
                            for (int cb = 0; cb < ncb; ++cb)
                                tma_load_4d(smX + (size_t)s * L.x_stage_bytes + (size_t)cb * kHeadBox * ROWB, map,
                                            &x_full[s], cb * kHeadCB, g.w0 - kHeadLead, hin, tc);
                        skip_first = false;
                        last_ph[s] = ph;
                        if (++s == nst) { s = 0; ph ^= 1; }
                    }
                }
                u += g.h1 - g.h0;
            }
            // never leave while a copy into this block's shared memory may still be in flight
            for (int k = 0; k < nst; ++k)
                if (last_ph[k] >= 0 && !bounded_wait(&x_full[k], (uint32_t)last_ph[k], budget, nullptr))
                    atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
            if (!bounded_wait(&w_full, 0, budget, nullptr)) atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------ MMA warps
        // warp 1 owns the even output frames of a pass, warp 2 the odd ones: every accumulator
        // (input row, output frame) has one writer, in the order dt, channel block, k step.
        const int k = warp - 1;
        const bool lead = lane == 0;  // issues every MMA and commit: the lane that polls the barriers
        const uint32_t idesc = make_idesc_bf16_f32(128, NCOL);
        // the A operand starts at staged row 7 (position w0 - 1); the swizzle follows the address bits
        const uint64_t x_desc0 = make_sdesc(smem_u32(smX) + (kHeadLead - 1) * ROWB, 16, SBO, LAYOUT_SW64, 0);
        const uint64_t w_desc0 = make_sdesc(smem_u32(smW), 16, SBO, LAYOUT_SW64, 0);
        const uint32_t x_inc = (uint32_t)L.x_stage_bytes >> 4;
        const uint32_t cb_inc = (uint32_t)(kHeadBox * ROWB) >> 4;
        const uint32_t w_inc = (uint32_t)(NCOL * ROWB) >> 4;
        bool ok = warp_bounded_wait(&w_full, 0, budget, &abort_flag);
        if (!ok && lane == 0 && !abort_flag) head_fail(L, STATUS_TIMEOUT_MMA, &abort_flag);
        tc_fence_after();
        int s = 0, ph = 0;
        uint32_t rs = 0;  // input rows started by this block
        for (long long u = ubeg; ok && u < uend;) {
            const HeadSeg g = head_segment(L, u, uend);
            for (int hin = g.h0 - 1; ok && hin <= g.h1; ++hin, ++rs) {
                const uint32_t slot = rs % kHeadSlots;
                if (!warp_bounded_wait(&acc_empty[slot], ((rs / kHeadSlots) & 1) ^ 1, budget, &abort_flag)) {
                    if (lane == 0 && !abort_flag) head_fail(L, STATUS_TIMEOUT_MMA, &abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                bool wrote = false;
                for (int j = 0; j < g.G + 2; ++j) {
                    if (!warp_bounded_wait(&x_full[s], ph, budget, &abort_flag)) {
                        if (lane == 0 && !abort_flag) head_fail(L, STATUS_TIMEOUT_MMA, &abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t xs = desc_add(x_desc0, s * x_inc);
                    bool any = false;
                    for (int dt = 0; dt < 3; ++dt) {
                        const int tout = j - dt;  // input frame t0 - 2 + j is tap dt of output frame t0 + tout
                        if (tout < 0 || tout >= g.G || (tout & 1) != k) continue;
                        const uint32_t d = tmem + slot * SLOT + (uint32_t)(tout * NCOL);
                        const uint64_t wd = desc_add(w_desc0, dt * ncb * w_inc);
                        for (int cb = 0; cb < ncb; ++cb) {
#pragma unroll
                            for (int ks = 0; ks < KSTEPS; ++ks) {
                                const uint64_t ad = desc_add(xs, cb * cb_inc + ks * 2);
                                const uint64_t bd = desc_add(wd, cb * w_inc + ks * 2);
                                const uint32_t acc = (dt == 0 && cb == 0 && ks == 0) ? 0u : 1u;
                                if (lead) umma_bf16_ss(d, ad, bd, idesc, acc);
                            }
                        }
                        any = true;
                    }
                    // a warp that read nothing from this stage releases it at once
                    if (lead) {
                        if (any) umma_commit(&x_empty[s]);
                        else mbar_arrive(&x_empty[s]);
                    }
                    __syncwarp();
                    wrote = wrote || any;
                    if (++s == nst) { s = 0; ph ^= 1; }
                }
                if (!ok) break;
                if (lead) {
                    if (wrote) umma_commit(&acc_full[slot]);
                    else mbar_arrive(&acc_full[slot]);
                }
                __syncwarp();
            }
            u += g.h1 - g.h0;
        }
        if (lead) umma_commit(&mma_drain[k]);
        __syncwarp();
        if (!warp_bounded_wait(&mma_drain[k], 0, budget, nullptr) && lane == 0)
            atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
    } else if (warp == 3) {
        // ------------------------------------------------------------ temporal cache update
        // cache_out[k] is frame T - 2 + k of (cache_in or zeros) ++ x_chunk: the input frame that
        // the last frame group stages as j = G + k.  This warp follows the stage ring and writes
        // the segment's output rows of those stages to cache_out from shared memory, so x is not
        // read a second time: the TMA unit stores staged rows 8 .. 127 (a store must start on a
        // swizzle atom), and the warp's lanes copy rows 1 .. 7 themselves, undoing the 64-byte
        // swizzle (16-byte chunk c of staged row r sits at chunk c ^ ((r >> 1) & 3)).
        __nv_bfloat16* hist = reinterpret_cast<__nv_bfloat16*>(L.cache_out);
        int s = 0, ph = 0;
        bool ok = true;
        for (long long u = ubeg; ok && u < uend;) {
            const HeadSeg g = head_segment(L, u, uend);
            const bool last_group = g.t0 + g.G == L.T;
            for (int hin = g.h0 - 1; ok && hin <= g.h1; ++hin) {
                for (int j = 0; j < g.G + 2; ++j) {
                    if (!warp_bounded_wait(&x_full[s], ph, budget, &abort_flag)) {
                        if (lane == 0 && !abort_flag) head_fail(L, STATUS_TIMEOUT_COPY, &abort_flag);
                        ok = false;
                        break;
                    }
                    if (last_group && j >= g.G && hin >= g.h0 && hin < g.h1) {
                        const uint8_t* stage = smX + (size_t)s * L.x_stage_bytes;
                        constexpr int NLEAD = kHeadStoreRow - kHeadLead;  // positions w0 .. w0 + 6
                        for (int i = lane; i < NLEAD * ncb * 4; i += 32) {
                            const int c = i & 3, rest = i >> 2;
                            const int r = kHeadLead + rest % NLEAD, cb = rest / NLEAD;
                            const int w = g.w0 + r - kHeadLead;
                            if (w < L.W) {
                                const uint4 v = *reinterpret_cast<const uint4*>(
                                    stage + (size_t)(cb * kHeadBox + r) * ROWB + ((c ^ ((r >> 1) & 3)) << 4));
                                *reinterpret_cast<uint4*>(
                                    hist + (((size_t)(j - g.G) * L.H + hin) * L.W + w) * L.Cin + cb * kHeadCB + c * 8) = v;
                            }
                        }
                        // (frames narrower than 8 pixels have nothing in the TMA store's box)
                        if (lane == 0 && g.w0 + kHeadStoreRow - kHeadLead < L.W) {
                            fence_proxy_async_smem();
                            for (int cb = 0; cb < ncb; ++cb)
                                tma_store_4d(&L.map_cache_out, stage + (size_t)(cb * kHeadBox + kHeadStoreRow) * ROWB,
                                             cb * kHeadCB, g.w0 + kHeadStoreRow - kHeadLead, hin, j - g.G);
                            bulk_commit_group();
                            bulk_wait_group_read<0>();  // the stage may be refilled once the store has read it
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&x_empty[s]);
                    if (++s == nst) { s = 0; ph ^= 1; }
                }
            }
            u += g.h1 - g.h0;
        }
        if (lane == 0) bulk_wait_group<0>();  // every store has landed before the block exits
    } else {
        // ------------------------------------------------------------ epilogue
        // Thread (q, lane) holds tensor-memory lane p = 32 q + lane: input position w0 - 1 + p,
        // which is output pixel w0 - 1 + p for p in 1..126.  Its left neighbour's dw = 0 terms and
        // its right neighbour's dw = 2 terms come by shuffles; across warps through shared memory.
        const int q = warp - 4;
        const int p = q * 32 + lane;
        const __nv_bfloat16* res = reinterpret_cast<const __nv_bfloat16*>(L.res);
        __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(L.y);
        uint8_t* yu8 = reinterpret_cast<uint8_t*>(L.y);
        const bool out_u8 = L.out_u8 != 0;
        float bias[COUT];
#pragma unroll
        for (int c = 0; c < COUT; ++c) bias[c] = s_bias[c];
        // edge lanes publish into slot q + 1; a lane 0 reads its left terms from slot q and a lane 31
        // its right terms from slot q + 2 (slots 0 and 5 stay zero: there is no warp -1 or 4)
        const bool edge_lane = lane == 0 || lane == 31;
        const int side = lane == 0 ? 1 : 0;
        uint32_t rs = 0;
        bool ok = true;
        for (long long u = ubeg; ok && u < uend;) {
            const HeadSeg g = head_segment(L, u, uend);
            const int w = g.w0 - 1 + p;
            const bool wvalid = p >= 1 && p <= kHeadOut && w < L.W;
            // running sums: P = row hin - 1 (dh 0 and 1 added), Q = row hin (dh 0 added)
            float P[GMAX][COUT], Q[GMAX][COUT];
#pragma unroll
            for (int t = 0; t < GMAX; ++t)
#pragma unroll
                for (int c = 0; c < COUT; ++c) P[t][c] = Q[t][c] = 0.0f;
            for (int hin = g.h0 - 1; hin <= g.h1; ++hin, ++rs) {
                const uint32_t slot = rs % kHeadSlots;
                const int buf = (int)(rs & 1);
                int ready = 0;
                if (lane == 0) {
                    ready = bounded_wait(&acc_full[slot], (rs / kHeadSlots) & 1, budget, &abort_flag,
                                         kEpilogueSleepNs);
                    if (!ready && !abort_flag) head_fail(L, STATUS_TIMEOUT_EPILOGUE, &abort_flag);
                    s_ok[buf][q] = ready;
                }
                ready = __shfl_sync(0xffffffffu, ready, 0);
                float* eb = s_edge + buf * EBUF;
                const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + slot * SLOT;
                if (ready) {
                    tc_fence_after();
                    // publish the edge lanes' terms (lane 31: dw = 0, lane 0: dw = 2) for the neighbours
#pragma unroll
                    for (int t = 0; t < GMAX; ++t) {
                        if (t < g.G) {
                            uint32_t v[NCOL];
                            tmem_ld_cols<NCOL>(trow + (uint32_t)(t * NCOL), v);
                            float* e = eb + ((t * 6 + q + 1) * 2 + side) * kHeadEdge;
#pragma unroll
                            for (int dh = 0; dh < 3; ++dh)
#pragma unroll
                                for (int c = 0; c < COUT; ++c) {
                                    const uint32_t val = lane == 0 ? v[(dh * 3 + 2) * COUT + c] : v[(dh * 3) * COUT + c];
                                    if (edge_lane) e[dh * COUT + c] = __uint_as_float(val);
                                }
                        }
                    }
                }
                named_barrier_sync(1, 128);
                // every epilogue warp reads the same four verdicts, so all leave together
                if (!(s_ok[buf][0] && s_ok[buf][1] && s_ok[buf][2] && s_ok[buf][3])) {
                    ok = false;
                    break;
                }
                const int h = hin - 1;  // the output row this input row completes
                const bool store = wvalid && h >= g.h0 && h < g.h1;
#pragma unroll
                for (int t = 0; t < GMAX; ++t) {
                    if (t < g.G) {
                        const long long px = ((long long)(g.t0 + t) * L.H + h) * L.W + w;  // used only if store
                        float rr[COUT];
#pragma unroll
                        for (int c = 0; c < COUT; ++c)
                            rr[c] = (store && res != nullptr) ? __bfloat162float(res[px * COUT + c]) : 0.0f;
                        uint32_t v[NCOL];
                        tmem_ld_cols<NCOL>(trow + (uint32_t)(t * NCOL), v);
                        if (t == g.G - 1) {
                            // every column of this slot is in registers: the MMA warps may reuse it
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&acc_empty[slot]);
                        }
                        // the neighbours' edge terms: same address in every lane (a broadcast read)
                        float el[16], er[16];  // 3 * COUT <= 15 terms per side
                        const float4* el4 = reinterpret_cast<const float4*>(eb + ((t * 6 + q) * 2 + 0) * kHeadEdge);
                        const float4* er4 = reinterpret_cast<const float4*>(eb + ((t * 6 + q + 2) * 2 + 1) * kHeadEdge);
#pragma unroll
                        for (int k4 = 0; k4 < (3 * COUT + 3) / 4; ++k4) {
                            const float4 a = el4[k4], b = er4[k4];
                            el[4 * k4] = a.x; el[4 * k4 + 1] = a.y; el[4 * k4 + 2] = a.z; el[4 * k4 + 3] = a.w;
                            er[4 * k4] = b.x; er[4 * k4 + 1] = b.y; er[4 * k4 + 2] = b.z; er[4 * k4 + 3] = b.w;
                        }
                        float sdh[3][COUT];
#pragma unroll
                        for (int dh = 0; dh < 3; ++dh) {
#pragma unroll
                            for (int c = 0; c < COUT; ++c) {
                                float l = __shfl_up_sync(0xffffffffu, __uint_as_float(v[(dh * 3 + 0) * COUT + c]), 1);
                                float r = __shfl_down_sync(0xffffffffu, __uint_as_float(v[(dh * 3 + 2) * COUT + c]), 1);
                                l = lane == 0 ? el[dh * COUT + c] : l;
                                r = lane == 31 ? er[dh * COUT + c] : r;
                                sdh[dh][c] = __fadd_rn(__fadd_rn(l, __uint_as_float(v[(dh * 3 + 1) * COUT + c])), r);
                            }
                        }
#pragma unroll
                        for (int c = 0; c < COUT; ++c) {
                            const float done = __fadd_rn(P[t][c], sdh[2][c]);
                            P[t][c] = __fadd_rn(Q[t][c], sdh[1][c]);
                            Q[t][c] = sdh[0][c];
                            const float o = __fadd_rn(__fadd_rn(done, bias[c]), rr[c]);
                            if (store) {
                                if (out_u8) yu8[px * COUT + c] = quant_u8(o);
                                else y[px * COUT + c] = __float2bfloat16_rn(o);
                            }
                        }
                    }
                }
            }
            u += g.h1 - g.h0;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem, (uint32_t)L.tmem_cols);
}

int cdiv(int a, int b) { return (a + b - 1) / b; }

}  // namespace

bool head_configure(int T, int H, int W, int Cin, int Cout, int sms, HeadLaunch* L)
{
    if (Cout < 1 || Cout > 5 || T < 1 || H < 1 || W < 1 || sms < 1) return false;
    if (Cin % kHeadCB != 0 || Cin > 256) return false;
    const int ncol = head_ncol(Cout);
    L->T = T;
    L->H = H;
    L->W = W;
    L->Cin = Cin;
    L->Cout = Cout;
    L->gmax = head_gmax(Cout);
    L->ncolblk = cdiv(W, kHeadOut);
    L->units = (long long)cdiv(T, L->gmax) * L->ncolblk * H;
    const int ncb = Cin / kHeadCB;
    L->w_bytes = (3 * ncb * ncol * kHeadCB * 2 + 1023) & ~1023;
    L->x_stage_bytes = ncb * kHeadBox * kHeadCB * 2;  // a multiple of 512 B (the 64-byte swizzle atom)
    const int edge_bytes = 2 * L->gmax * 6 * 2 * kHeadEdge * 4;
    const int fixed = L->w_bytes + edge_bytes + 1024;  // + alignment slack
    int nst = (227 * 1024 - fixed) / L->x_stage_bytes;
    if (nst > kHeadMaxStages) nst = kHeadMaxStages;
    if (nst < 2) return false;
    L->nstages = nst;
    L->smem_bytes = (size_t)fixed + (size_t)nst * L->x_stage_bytes;
    if (L->smem_bytes < 120 * 1024) L->smem_bytes = 120 * 1024;  // one block per SM: it owns all tensor memory
    L->tmem_cols = 512;
    L->grid = L->units < sms ? (int)L->units : sms;
    return true;
}

cudaError_t head_launch(const HeadLaunch& L, cudaStream_t stream)
{
    void* kern = nullptr;
    switch (L.Cout) {
    case 1: kern = reinterpret_cast<void*>(head_bf16_kernel<1>); break;
    case 2: kern = reinterpret_cast<void*>(head_bf16_kernel<2>); break;
    case 3: kern = reinterpret_cast<void*>(head_bf16_kernel<3>); break;
    case 4: kern = reinterpret_cast<void*>(head_bf16_kernel<4>); break;
    case 5: kern = reinterpret_cast<void*>(head_bf16_kernel<5>); break;
    default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem_bytes);
    if (e != cudaSuccess) return e;
    void* args[] = {const_cast<HeadLaunch*>(&L)};
    return cudaLaunchKernel(kern, dim3(L.grid), dim3(kThreads), args, L.smem_bytes, stream);
}

}  // namespace cc3d
