// cc3d_tc.cu -- implicit-GEMM causal 3x3x3 convolution on the sm_103a tensor cores.
//
// GEMM view: rows (M) = output positions of one frame, columns (N) = output
// channels, reduction (K) = 27 taps x Cin.  Accumulators live in tensor memory
// (fp32), operands are staged in shared memory by TMA:
//
//   * A: for every (temporal tap dt, channel block cb) one input window of
//     `nrows` padded rows x Sp pixels x CB channels is loaded once; the nine
//     spatial taps (dh, dw) of every 128-row group are row-shifted views of
//     that window (see TcGeometry): the tensor core applies the swizzle on
//     absolute shared-memory addresses, so a descriptor that starts any number
//     of rows into the swizzled window is valid.  The TMA box starts one pixel
//     left of the column block and may start above the frame; everything
//     outside the frame is filled with zeros by the copy engine, which is the
//     spatial zero padding.  Frames before the chunk come from the caller's
//     cache (or read as zeros through a negative frame coordinate when there is
//     no cache), which is the causal history.
//   * B: one stage = the weights of the taps of one or all three (dt, dh) kernel
//     rows for one channel block and one N slice, K-major.
//
// Warp roles (256 threads): warp 0 = TMA loader, warp 1 = MMA issuer, warp 2
// = tensor-memory allocator and, with warp 3, the copy of the new temporal
// cache, warps 4-7 = epilogue (tensor memory -> registers -> + bias
// [+ residual] -> bf16 -> global), one output position per thread.
//
// The MMA warp keeps the shared-memory descriptors of stage 0 and advances
// them by 32-bit additions on the low word (the start-address field is the low
// 14 bits and every address stays below 2^18 bytes), with the tap / row-group /
// K-step loops unrolled at compile time.  All 32 lanes walk the issue loop, so
// the descriptors stay warp-uniform, and lane 0 -- the lane that polls the
// barriers -- issues every MMA (an elect.sync before every MMA made the warp
// reconverge each time and cost about 10 % end to end).
//
// The accumulation order of every output is fixed: dt, channel block, dh, dw,
// 16-channel step -- it depends neither on the tile an output falls in nor on
// how the video is cut into chunks, so chunked and unchunked results are
// bit-identical.
#include <cuda_bf16.h>

#include "cc3d_internal.h"
#include "cc3d_ptx.cuh"
#include "cc3d_tc_common.cuh"

namespace cc3d {
using namespace ptx;
using namespace tcc;

namespace {

// Work unit u of the one-SM kernel: its tile, and the mask of its 128-row groups (bit m: row
// group m of the tile; a split tile's two units hold one row group each).
__device__ __forceinline__ int unit_tile(const TcLaunch& L, int u)
{
    return u < L.nfull ? u : L.nfull + ((u - L.nfull) >> 1);
}

__device__ __forceinline__ int unit_mask(const TcLaunch& L, int u)
{
    return u < L.nfull ? 0xF : 1 << ((u - L.nfull) & 1);
}

template <int CB, int SUBI, int RB>
__global__ void __launch_bounds__(kThreads, 1) tc_bf16_kernel(const __grid_constant__ TcLaunch L)
{
    constexpr uint32_t ROWB = CB * 2;     // bytes of one pixel row of a channel block = swizzle span
    constexpr uint32_t ROWU = ROWB / 16;  // the same in descriptor address units
    constexpr uint32_t LAYOUT = CB == 64 ? LAYOUT_SW128 : (CB == 32 ? LAYOUT_SW64 : LAYOUT_SW32);
    constexpr uint32_t SBO = 8 * ROWB;
    constexpr int KSTEPS = CB / 16;

    extern __shared__ uint8_t dsm_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smA = sm;
    uint8_t* smB = sm + (size_t)L.na * L.a_stage_bytes;
    float* s_bias = reinterpret_cast<float*>(smB + (size_t)L.nb * L.b_stage_bytes);

    __shared__ uint64_t a_full[kMaxStages], a_empty[kMaxStages], b_full[kMaxStages], b_empty[kMaxStages];
    __shared__ uint64_t acc_full[kMaxAcc], acc_empty[kMaxAcc], mma_drain[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int Sp = L.g.Sp;
    const int NT = L.NT;
    const int nsplit = L.nsplit;
    const int ncb = L.Cin / CB;
    const int cout_pad = L.ncoblk * nsplit * NT;
    const int SUB = L.g.sub;                   // 128-row groups per tile (all MMA warps together)
    const int nissue = L.issuers;              // MMA-issuing warps (1 or 2)
    const uint32_t acc_cols = (uint32_t)(SUB * nsplit * NT * (L.up2 ? 4 : 1));
    const unsigned long long budget = L.wait_ns;
    const int KSZ = L.ks;     // spatial kernel extent (kh = kw): 3, or 1 for temporal / pointwise kernels
    const int P = L.kt - 1;   // history frames in the cache
    // one accumulator buffer shared by two MMA warps that own disjoint 128-row groups (or
    // output classes): each warp waits only for its own part to be drained
    const bool per_warp_release = L.acc_stages == 1 && nissue == 2 && !L.split_n;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        // stage releases and accumulator completions come from every MMA warp
        for (int s = 0; s < L.na; ++s) { mbar_init(&a_full[s], 1); mbar_init(&a_empty[s], nissue); }
        for (int s = 0; s < L.nb; ++s) { mbar_init(&b_full[s], 1); mbar_init(&b_empty[s], nissue); }
        for (int a = 0; a < L.acc_stages; ++a) mbar_init(&acc_full[a], nissue);
        // released by the 4 epilogue warps; with one accumulator stage and two MMA warps that
        // split the rows (or an upsampling layer's classes), each MMA warp's part is released
        // separately, on acc_empty[0] and acc_empty[1]
        for (int a = 0; a < (per_warp_release ? 2 : L.acc_stages); ++a) mbar_init(&acc_empty[a], 4);
        mbar_init(&mma_drain[0], 1);
        mbar_init(&mma_drain[1], 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&L.map_x);
        prefetch_tensormap(&L.map_w);
        if (L.has_cache) prefetch_tensormap(&L.map_cache);
    }
    if (warp == 2) {
        tmem_alloc(&tmem_base_sh, (uint32_t)L.tmem_cols);
        tmem_relinquish();
    }
    if (warp >= 4) {
        const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(L.bias);
        for (int i = threadIdx.x - 128; i < cout_pad; i += 128)
            s_bias[i] = (b != nullptr && i < L.Cout) ? __bfloat162float(b[i]) : 0.0f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA loader
        if (lane == 0) {
            int sa = 0, pa = 0, sb = 0, pb = 0;
            int last_pa[kMaxStages], last_pb[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) last_pa[s] = last_pb[s] = -1;
            const uint32_t a_tx = (uint32_t)(ROWB * Sp * L.g.nrows);
            const uint32_t b_tx = (uint32_t)(ROWB * NT * KSZ * RB);
            bool skip_first = (L.fault == 1);
            bool ok = true;
            for (int u = blockIdx.x; ok && u < L.nunits; u += gridDim.x) {
                const TileCoord c = tile_coord(L, unit_tile(L, u));
                // optionally warm L2 with the input windows of this block's next tile
                const int next = u + (int)gridDim.x;
                if (L.prefetch && next < L.nunits) {
                    const TileCoord n = tile_coord(L, unit_tile(L, next));
                    for (int dt = L.kt > L.prefetch ? L.kt - L.prefetch : 0; dt < L.kt; ++dt) {
                        const int tin = n.t + dt - P;
                        const bool from_cache = tin < 0 && L.has_cache;
                        for (int cb = 0; cb < ncb; ++cb)
                            tma_prefetch_4d(from_cache ? &L.map_cache : &L.map_x, cb * CB, n.w0 - 1, n.hstart,
                                            from_cache ? tin + P : tin);
                    }
                }
                for (int dt = 0; ok && dt < L.kt; ++dt) {
                    const int tin = c.t + dt - P;
                    const CUtensorMap* map = &L.map_x;
                    int tc = tin;
                    if (tin < 0 && L.has_cache) { map = &L.map_cache; tc = tin + P; }
                    for (int cb = 0; ok && cb < ncb; ++cb) {
                        if (!bounded_wait(&a_empty[sa], pa ^ 1, budget, &abort_flag, kLoaderSleepNs)) {
                            if (!abort_flag) record_failure(L, STATUS_TIMEOUT_LOADER, &abort_flag);
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&a_full[sa], a_tx);
                        if (!skip_first)
                            tma_load_4d(smA + (size_t)sa * L.a_stage_bytes, map, &a_full[sa], cb * CB, c.w0 - 1,
                                        c.hstart, tc);
                        skip_first = false;
                        last_pa[sa] = pa;
                        if (++sa == L.na) { sa = 0; pa ^= 1; }
                        for (int dg = 0; ok && dg < KSZ / RB; ++dg) {
                            for (int ns = 0; ns < nsplit; ++ns) {
                                if (!bounded_wait(&b_empty[sb], pb ^ 1, budget, &abort_flag, kLoaderSleepNs)) {
                                    if (!abort_flag) record_failure(L, STATUS_TIMEOUT_LOADER, &abort_flag);
                                    ok = false;
                                    break;
                                }
                                mbar_arrive_expect_tx(&b_full[sb], b_tx);
                                tma_load_3d(smB + (size_t)sb * L.b_stage_bytes, &L.map_w, &b_full[sb], cb * CB,
                                            c.co0 + ns * NT, dt * KSZ * KSZ + dg * RB * KSZ);
                                last_pb[sb] = pb;
                                if (++sb == L.nb) { sb = 0; pb ^= 1; }
                            }
                        }
                    }
                }
            }
            // never leave while a copy into this block's shared memory may still be in flight
            for (int s = 0; s < L.na; ++s)
                if (last_pa[s] >= 0 && !bounded_wait(&a_full[s], (uint32_t)last_pa[s], budget, nullptr))
                    atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
            for (int s = 0; s < L.nb; ++s)
                if (last_pb[s] >= 0 && !bounded_wait(&b_full[s], (uint32_t)last_pb[s], budget, nullptr))
                    atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
        }
    } else if (warp == 1 || (warp == 2 && nissue == 2)) {
        // ------------------------------------------------------------ MMA issuers
        // The whole warp walks the loop so that every descriptor stays warp-uniform (the MMA takes
        // its operands from uniform registers); lane 0 issues the tcgen05 instructions.
        // With two MMA warps each one owns its own accumulators (half of the 128-row groups, or one
        // of two N slices) and both consume every stage: while one polls a barrier or does its
        // bookkeeping the other keeps the tensor core fed.  Every accumulator is still written by
        // one warp in program order, so the accumulation order is unchanged.
        const int k = warp - 1;
        // Lane 0 issues every MMA and commit of this warp: it is the lane that polls the full
        // barriers (warp_bounded_wait), so the thread that observes a stage's completion is the one
        // whose MMAs read it, and a commit tracks the MMAs of the thread that issues it.  (An
        // elect.sync per MMA made the warp reconverge before every instruction and was measured
        // 10 % slower; a lane elected once need not be the polling lane, and that form gave wrong
        // results on first launches.)
        const bool lead = lane == 0;
        // first 128-row group of this warp (all of them when the warps split N slices or classes)
        const int m0 = (L.split_n || L.up2) ? 0 : k * SUBI;
        // upsampling layers: four output classes per row group, two per MMA warp
        const int ncls = L.up2 ? 4 : 1;
        const int ns_lo = L.split_n ? k : 0, ns_hi = L.split_n ? k + 1 : nsplit;
        const uint32_t idesc = make_idesc_bf16_f32(128, NT);
        const uint32_t idesc_h = make_idesc_bf16_f32(128, NT >= 32 ? NT / 2 : NT);  // split tiles: half of N
        const uint32_t idesc2 = make_idesc_bf16_f32(128, L.up2 ? 2 * NT : NT);  // two classes side by side
        const uint64_t a_desc0 = make_sdesc(smem_u32(smA), 16, SBO, LAYOUT, 0);
        const uint64_t b_desc0 = make_sdesc(smem_u32(smB), 16, SBO, LAYOUT, 0);
        const uint32_t a_inc = (uint32_t)L.a_stage_bytes >> 4;
        const uint32_t b_inc = (uint32_t)L.b_stage_bytes >> 4;
        const uint32_t b_tap_inc = (uint32_t)NT * ROWU;  // next tap inside a B stage
        const uint32_t row_shift = (uint32_t)Sp * ROWU;  // next padded row inside the A window
        const uint32_t m_cols = (uint32_t)(nsplit * NT * ncls);  // tensor-memory columns per row group
        int sa = 0, pa = 0, sb = 0, pb = 0;
        bool ok = true;
        int it = 0;
        for (int u = blockIdx.x; ok && u < L.nunits; u += gridDim.x, ++it) {
            const TileCoord c = tile_coord(L, unit_tile(L, u));
            const int umask = unit_mask(L, u);
            // a split tile's unit: one row group (hrg), whose output channels the two MMA warps
            // share, NT / 2 each (each output's accumulation order is unchanged)
            const bool half = umask != 0xF;
            const int hrg = umask >> 1;
            const int as = it % L.acc_stages;
            const int aph = (it / L.acc_stages) & 1;
            bool freed = warp_bounded_wait(&acc_empty[per_warp_release ? k : as], aph ^ 1, budget, &abort_flag);
            if (freed && half) freed = warp_bounded_wait(&acc_empty[1 - k], aph ^ 1, budget, &abort_flag);
            if (!freed) {
                if (lane == 0 && !abort_flag) record_failure(L, STATUS_TIMEOUT_MMA, &abort_flag);
                break;
            }
            tc_fence_after();
            const uint32_t dbase = tmem + (uint32_t)as * acc_cols;
            const int mrow = half ? hrg : m0;  // first row group this warp issues
            const uint32_t hcol = half ? (uint32_t)(k * (NT / 2)) : 0u;  // its columns / weight rows
            const uint32_t idesc_u = half ? idesc_h : idesc;
            // window row of the (dh = 0, dw = 0) view of each 128-row group, in descriptor units
            uint32_t rowu[SUBI];
#pragma unroll
            for (int m = 0; m < SUBI; ++m)
                rowu[m] = (uint32_t)(c.f0 + (mrow + m) * L.g.sub_stride - c.hstart * Sp - L.g.halo * (Sp + 1)) * ROWU;
            for (int dt = 0; ok && dt < L.kt; ++dt) {
                for (int cb = 0; ok && cb < ncb; ++cb) {
                    if (!warp_bounded_wait(&a_full[sa], pa, budget, &abort_flag)) {
                        if (lane == 0 && !abort_flag) record_failure(L, STATUS_TIMEOUT_MMA, &abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_st = a_desc0 + (uint64_t)(sa * a_inc);
                    for (int dg = 0; ok && dg < KSZ / RB; ++dg) {
                        for (int ns = 0; ns < nsplit; ++ns) {
                            if (!warp_bounded_wait(&b_full[sb], pb, budget, &abort_flag)) {
                                if (lane == 0 && !abort_flag) record_failure(L, STATUS_TIMEOUT_MMA, &abort_flag);
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            const uint64_t b_st = b_desc0 + (uint64_t)(sb * b_inc);
                            const uint32_t dcol = dbase + (uint32_t)(ns * NT) + (uint32_t)mrow * m_cols + hcol;
                            const bool mine = ns >= ns_lo && ns < ns_hi;
                            if (L.up2) {
                                // Output class (a, b) of source position (i, j) is the upsampled
                                // pixel (2i + a, 2j + b): its tap (dh, dw) reads source pixel
                                // (i + floor((a + dh - 1) / 2), j + floor((b + dw - 1) / 2)), a view
                                // of the same window shifted by 0..2 rows and 0..2 pixels.  MMA
                                // warp k owns class row a = k; its two classes (slots 2a: b = 1,
                                // 2a + 1: b = 0, in that column order) read the same view for
                                // taps (dw = 0 of b = 1, dw = 1 of b = 0) and (dw = 1 of b = 1,
                                // dw = 2 of b = 0), whose weight taps lie side by side in the
                                // stage: those pairs go through one MMA with N = 2 NT.  Per tap row:
                                //   b = 0, dw = 0 (view 0)   N = NT
                                //   both, dw = 0 | 1 (view 1) N = 2 NT
                                //   both, dw = 1 | 2 (view 1) N = 2 NT
                                //   b = 1, dw = 2 (view 2)   N = NT
                                // which keeps each class's order dh, dw, 16-channel step.  The
                                // first stacked MMA of a tile is issued as its two halves, so that
                                // class (a, 1) starts from zero while (a, 0) accumulates.
                                const int a = k;
                                const uint32_t slot1 = dcol + (uint32_t)(2 * a * NT);  // class (a, 1), then (a, 0)
                                const uint32_t slot0 = slot1 + (uint32_t)NT;
                                for (int dr = 0; dr < RB; ++dr) {
                                    const int dh = dg * RB + dr;
                                    const bool first_row = (dt | cb | dh) == 0;
                                    const uint64_t vrow = desc_add(a_st, ((a + dh + 1) >> 1) * row_shift);
                                    const uint64_t btap = desc_add(b_st, (dr * 3) * b_tap_inc);
#pragma unroll
                                    for (int m = 0; m < SUBI; ++m) {
#pragma unroll
                                        for (int kind = 0; kind < 4; ++kind) {
                                            const int sw1 = kind == 0 ? 0 : (kind == 3 ? 2 : 1);
                                            const int dw0 = kind == 0 ? 0 : (kind == 3 ? 2 : kind - 1);  // first weight tap
                                            const uint32_t dst = (kind == 0 ? slot0 : slot1) + (uint32_t)m * m_cols;
#pragma unroll
                                            for (int ks = 0; ks < KSTEPS; ++ks) {
                                                const uint64_t ad = desc_add(vrow, sw1 * ROWU + rowu[m] + ks * 2);
                                                const uint64_t bd = desc_add(btap, dw0 * b_tap_inc + ks * 2);
                                                if (kind == 1 || kind == 2) {
                                                    if (kind == 1 && first_row && ks == 0) {
                                                        // halves: (a, 1) tap dw = 0 from zero, (a, 0) tap dw = 1
                                                        if (lead) umma_bf16_ss(dst, ad, bd, idesc, 0u);
                                                        if (lead)
                                                            umma_bf16_ss(dst + (uint32_t)NT, ad, desc_add(bd, b_tap_inc), idesc, 1u);
                                                    } else if (lead) {
                                                        umma_bf16_ss(dst, ad, bd, idesc2, 1u);
                                                    }
                                                } else {
                                                    const uint32_t acc = (kind == 0 && first_row && ks == 0) ? 0u : 1u;
                                                    if (lead) umma_bf16_ss(dst, ad, bd, idesc, acc);
                                                }
                                            }
                                        }
                                    }
                                }
                            } else {
#pragma unroll
                            for (int dr = 0; dr < RB; ++dr) {
                                const int dh = dg * RB + dr;
                                const uint64_t a_row = desc_add(a_st, dh * row_shift);
                                const bool first_row = (dt | cb | dh) == 0;
#pragma unroll
                                for (int dw = 0; dw < 3; ++dw) {
                                    if (dw >= KSZ) continue;  // 1x1 spatial kernels: the single tap
#pragma unroll
                                    for (int m = 0; m < SUBI; ++m) {
#pragma unroll
                                        for (int ks = 0; ks < KSTEPS; ++ks) {
                                            const uint64_t ad = desc_add(a_row, rowu[m] + dw * ROWU + ks * 2);
                                            const uint64_t bd =
                                                desc_add(b_st, (dr * KSZ + dw) * b_tap_inc + hcol * ROWU + ks * 2);
                                            const uint32_t acc = (first_row && dw == 0 && ks == 0) ? 0u : 1u;
                                            if (mine && lead)
                                                umma_bf16_ss(dcol + (uint32_t)m * m_cols, ad, bd, idesc_u, acc);
                                        }
                                    }
                                }
                            }
                            }
                            if (lead) umma_commit(&b_empty[sb]);
                            __syncwarp();
                            if (++sb == L.nb) { sb = 0; pb ^= 1; }
                        }
                    }
                    if (!ok) break;
                    if (lead) umma_commit(&a_empty[sa]);
                    if (++sa == L.na) { sa = 0; pa ^= 1; }
                }
            }
            if (!ok) break;
            if (lead) umma_commit(&acc_full[as]);
        }
        // wait until every MMA this warp issued has finished writing tensor memory
        if (lead) umma_commit(&mma_drain[k]);
        __syncwarp();
        if (!warp_bounded_wait(&mma_drain[k], 0, budget, nullptr) && lane == 0)
            atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
    } else if (warp == 2 || warp == 3) {
        // ------------------------------------------------------------ temporal cache update
        // Warps 2-3, or warp 3 alone when warp 2 issues MMAs.
        const int nw = nissue == 2 ? 1 : 2;
        if (L.copy_hist) copy_history(L, P, warp - (nissue == 2 ? 3 : 2), nw, lane);
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp - 4;  // tensor-memory lanes 32q .. 32q+31
        const __nv_bfloat16* res = reinterpret_cast<const __nv_bfloat16*>(L.res);
        __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(L.y);
        const bool wide = (L.Cout % 16) == 0;
        int it = 0;
        for (int u = blockIdx.x; u < L.nunits; u += gridDim.x, ++it) {
            const int umask = unit_mask(L, u);  // row groups of this unit (all of a whole tile)
            const bool half = umask != 0xF;
            const int hrg = umask >> 1;
            const int as = it % L.acc_stages;
            const int aph = (it / L.acc_stages) & 1;
            const TileCoord c = tile_coord(L, unit_tile(L, u));
            // while the accumulators fill, pull this thread's residual lines into L2
            if (res != nullptr && wide && !L.up2) {
                for (int m = 0; m < SUB; ++m) {
                    const int f = c.f0 + m * L.g.sub_stride + q * 32 + lane;
                    const int h = f / Sp;
                    const int jcol = f - h * Sp;
                    const int w = c.w0 + jcol - 1;
                    if (h < L.H && jcol >= 1 && jcol <= L.g.S && w < L.W) {
                        const char* p = reinterpret_cast<const char*>(
                            res + (((size_t)c.t * L.H + h) * L.W + w) * L.Cout);
                        for (int o = 0; o < L.Cout * 2; o += 128) prefetch_l2(p + o);
                    }
                }
            }
            // one lane waits and the verdict is shared: tcgen05.ld below needs the whole warp
            int ready = 0;
            if (lane == 0) {
                ready = bounded_wait(&acc_full[as], aph, budget, &abort_flag, kEpilogueSleepNs);
                if (!ready && !abort_flag) record_failure(L, STATUS_TIMEOUT_EPILOGUE, &abort_flag);
            }
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) break;
            tc_fence_after();
            if (L.up2) {
                // class (a, b) of source pixel (h, w) is output pixel (2h + a, 2w + b) of the
                // 2H x 2W frame.  Class pair kp belongs to MMA warp kp and is released on
                // acc_empty[kp] once its columns of the last row group are in registers: with NT
                // <= 96 each class is read whole before its stores, so an MMA warp waits for its
                // own classes only, and for the stores of one of them.
                for (int kp = 0; kp < 2; ++kp) {
                    for (int m = 0; m < SUB; ++m) {
                        const int f = c.f0 + m * L.g.sub_stride + q * 32 + lane;
                        const int h = f / Sp;
                        const int jcol = f - h * Sp;
                        const int w = c.w0 + jcol - 1;
                        const bool valid = h < L.H && jcol >= 1 && jcol <= L.g.S && w < L.W;
                        const bool last_m = m == SUB - 1;
                        // output position of the class in column slot 2 kp + u: class (kp, 1 - u)
                        auto out_px = [&](int u) {
                            const size_t oh = valid ? 2 * (size_t)h + kp : 0;
                            const size_t ow = valid ? 2 * (size_t)w + (1 - u) : 0;
                            return ((size_t)c.t * 2 * L.H + oh) * 2 * L.W + ow;
                        };
                        const uint32_t tb = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)as * acc_cols +
                                            (uint32_t)((m * 4 + 2 * kp) * NT);
                        if (NT <= 96 && wide) {
                            for (int u = 0; u < 2; ++u) {
                                uint32_t r[96];
                                tmem_read_quarter<96>(tb + (uint32_t)(u * NT), NT, r);
                                tmem_ld_wait();
                                if (last_m && u == 1) release_acc(&acc_empty[kp], lane);
                                if (valid) store_quarter<96>(r, NT, c.co0, out_px(u), s_bias, L.Cout, res, y, L.v32 != 0);
                            }
                        } else {
                            for (int u = 0; u < 2; ++u)
                                epilogue_slice(tb + (uint32_t)(u * NT), NT, c.co0, out_px(u), valid, last_m && u == 1, s_bias,
                                               L.Cout, wide, res, y, L.v32 != 0,
                                               [&]() { release_acc(&acc_empty[kp], lane); });
                        }
                    }
                }
                continue;
            }
            for (int m = 0; m < SUB; ++m) {
                const int f = c.f0 + m * L.g.sub_stride + q * 32 + lane;
                const int h = f / Sp;
                const int jcol = f - h * Sp;
                const int w = c.w0 + jcol - 1;
                const bool valid = h < L.H && jcol >= 1 && jcol <= L.g.S && w < L.W;
                const size_t px = ((size_t)c.t * L.H + (valid ? h : 0)) * L.W + (valid ? w : 0);
                if (per_warp_release && half) {
                    // a split tile's unit: only row group hrg, written by both MMA warps, which
                    // both wait for both releases
                    if (m != hrg) continue;
                    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(m * nsplit * NT);
                    epilogue_slice(tbase, NT, c.co0, px, valid, true, s_bias, L.Cout, wide, res, y, L.v32 != 0,
                                   [&]() {
                                       release_acc(&acc_empty[0], lane);
                                       release_acc(&acc_empty[1], lane);
                                   });
                    continue;
                }
                if (per_warp_release) {
                    // row group m belongs to MMA warp m / SUBI; the read of its last row group of
                    // the tile releases that warp's part (the other warp's part may still be
                    // waiting for the epilogue)
                    const int owner = m / SUBI;
                    const bool last_of_owner = (m % SUBI) == SUBI - 1;
                    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(m * nsplit * NT);
                    for (int ns = 0; ns < nsplit; ++ns)
                        epilogue_slice(tbase + (uint32_t)(ns * NT), NT, c.co0 + ns * NT, px, valid,
                                       last_of_owner && ns == nsplit - 1, s_bias, L.Cout, wide, res, y, L.v32 != 0,
                                       [&]() { release_acc(&acc_empty[owner], lane); });
                    continue;
                }
                for (int ns = 0; ns < nsplit; ++ns) {
                    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)as * acc_cols +
                                           (uint32_t)((m * nsplit + ns) * NT);
                    const bool last_slice = (m == SUB - 1) && (ns == nsplit - 1);
                    epilogue_slice(tbase, NT, c.co0 + ns * NT, px, valid, last_slice, s_bias, L.Cout, wide, res, y, L.v32 != 0,
                                   [&]() { release_acc(&acc_empty[as], lane); });
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem, (uint32_t)L.tmem_cols);
}

int cdiv(int a, int b) { return (a + b - 1) / b; }


template <int CB, int RB>
void* kernel_for(int sub)
{
    // sub = 128-row groups owned by one MMA warp
    switch (sub) {
    case 1: return reinterpret_cast<void*>(tc_bf16_kernel<CB, 1, RB>);
    case 2: return reinterpret_cast<void*>(tc_bf16_kernel<CB, 2, RB>);
    case 4: return reinterpret_cast<void*>(tc_bf16_kernel<CB, 4, RB>);
    default: return nullptr;
    }
}

}  // namespace

namespace {

// One attempt at a configuration with at most sub_cap row groups per tile.
bool tc_configure_capped(int CB, int T, int H, int W, int Cin, int Cout, int kt, int ks, bool has_residual, bool up2,
                         int sub_cap, int smax, const TcOverrides* O, TcLaunch* L)
{
    (void)has_residual;  // the measured best configuration does not depend on it today
    auto ov = [O](int knob, int dflt) { return O != nullptr ? O->get(knob, dflt) : dflt; };
    if (CB != 16 && CB != 32) return false;
    if (Cin % CB != 0) return false;
    if (kt < 1 || kt > 3 || (ks != 1 && ks != 3)) return false;
    L->kt = kt;
    L->ks = ks;
    L->T = T;
    L->H = H;
    L->W = W;
    L->Cin = Cin;
    L->Cout = Cout;
    L->up2 = up2 ? 1 : 0;
    if (up2 && (ks != 3 || Cout % 16 != 0)) return false;
    // output channels per MMA (N) and number of N slices
    // Output channels: NT per MMA, nsplit N slices per tile (they share the input windows), and
    // ncoblk channel blocks handled by different tiles.  Wide layers (more than 256 channels) are
    // cut into channel blocks by default: the tiles then hold two 128-row groups each and load
    // only their block's weights.
    L->ncoblk = 1;
    if (up2) {
        // four output classes per row group share the accumulator budget: channel blocks of at
        // most 128, each its own tiles
        int nb = cdiv(Cout, 128);
        while (nb <= 8 && !(Cout % nb == 0 && (Cout / nb) % 16 == 0)) ++nb;
        if (nb > 8) return false;
        L->ncoblk = nb;
        L->nsplit = 1;
        L->NT = Cout / nb;
    } else if (Cout < 16) {
        L->NT = 16;
        L->nsplit = 1;
    } else {
        if (Cout % 16 != 0) return false;
        int ns = cdiv(Cout, 256);
        while (ns <= 4 && !(Cout % ns == 0 && (Cout / ns) % 16 == 0)) ++ns;
        if (ns > 4) return false;
        L->nsplit = ns;
        L->NT = Cout / ns;
        if (ns > 1 && ov(CC3D_SCHED_CHANNEL_BLOCKS, 1)) {
            L->ncoblk = ns;
            L->nsplit = 1;
        }
    }
    const int ntot = L->NT * L->nsplit * (up2 ? 4 : 1);  // accumulator columns of a row group
    // 128-row groups per tile (sub) and accumulator stages (acc), within the 512 tensor-memory
    // columns (sub * ntot * acc <= 512).  Measured on GB300: more rows per tile share each weight
    // stage and amortise the per-stage work of the MMA warps, which outweighs double-buffering
    // the accumulators (the epilogue is short: it reads each residual row once and frees the
    // accumulators as soon as their last columns are in registers).
    int sub, acc;
    if (ntot <= 64) {
        sub = 4;
        acc = 2;
    } else if (ntot <= 128) {
        sub = 4;
        acc = 1;
    } else if (ntot <= 256) {
        sub = 2;
        acc = 1;
    } else if (ntot <= 512) {
        sub = 1;
        acc = 1;
    } else {
        return false;
    }
    if (up2) {
        sub = ntot <= 128 ? 4 : (ntot <= 256 ? 2 : 1);
        acc = 1;
    }
    sub = ov(CC3D_SCHED_ROW_GROUPS, sub);
    acc = ov(CC3D_SCHED_ACC_STAGES, acc);
    if (sub > sub_cap) sub = sub_cap;
    // SM pairs (cta_group::2): both tiles of a pair must use the same window offsets (row-aligned
    // geometry) and the same weights (one output-channel block); then each block holds half of
    // every weight stage and the tensor core reads less shared memory per MMA.  Two row groups
    // per block with double-buffered accumulators, measured best for narrow layers.
    // Tiles are ordered frame fastest, so with an even number of frames the two tiles of a pair
    // are consecutive frames at one spatial position (and one output-channel block): they share
    // window offsets and weights in any geometry.  With an odd number the row-aligned geometry
    // (W a multiple of 128, equal offsets everywhere) still pairs a single channel block.
    L->pair = 0;
    const bool pair_tiles_match = T % 2 == 0 || (W % 128 == 0 && L->ncoblk == 1);
    if (!up2 && pair_tiles_match && L->nsplit == 1 && L->NT >= 32 && L->NT <= 192 && ov(CC3D_SCHED_PAIR, 1)) {
        L->pair = 1;
        sub = ov(CC3D_SCHED_ROW_GROUPS, 2);
        acc = ov(CC3D_SCHED_ACC_STAGES, 2 * 2 * L->NT <= 512 ? 2 : 1);
    }
    // two output frames per pair tile, stacked into N where an input frame is a tap of both
    // (chunks of two or more frames of a kt x 3 x 3 kernel with kt >= 2, up to 96 output channels;
    // with kt = 2 one of three input frames is shared, measured 1 % faster): two row groups per
    // block, one accumulator buffer of 2 frames x 2 row groups x NT columns
    L->tstack = 0;
    if (L->pair && W % 128 == 0 && L->ncoblk == 1 && kt >= 2 && ks == 3 && T >= 2 && L->NT <= 96 && sub_cap >= 2 &&
        ov(CC3D_SCHED_TWO_FRAME, 1)) {
        L->tstack = 1;
        sub = 2;
        acc = 1;
    }
    if ((sub != 1 && sub != 2 && sub != 4) || acc < 1 || acc > kMaxAcc || sub * ntot * acc > 512) return false;
    if (L->pair && sub > 2) return false;
    L->acc_stages = acc;
    // two MMA warps when the accumulators split evenly: by 128-row groups, else by N slices
    L->issuers = 1;
    L->split_n = 0;
    if (up2) {
        L->issuers = 2;  // each MMA warp owns two of the four output classes
    } else if (ov(CC3D_SCHED_MMA_WARPS, 2) == 2) {
        if (sub >= 2) {
            L->issuers = 2;
        } else if (L->nsplit == 2) {
            L->issuers = 2;
            L->split_n = 1;
        }
    }
    int cols = 32;
    while (cols < (L->tstack ? 4 * L->NT : sub * ntot * acc)) cols *= 2;
    L->tmem_cols = cols;
    // column blocks and padded-flat geometry
    TcGeometry& g = L->g;
    g.sub = sub;
    if (W % 128 == 0) {
        g.S = 128;
        g.row_aligned = 1;
    } else {
        const int nblk = cdiv(W, smax);
        g.S = cdiv(W, nblk);
        g.row_aligned = 0;
    }
    g.Sp = g.S + 2;
    g.halo = (ks - 1) / 2;
    g.ncolblk = cdiv(W, g.S);
    if (g.row_aligned) {
        g.sub_stride = g.Sp;
        g.tile_f = sub * g.Sp;
        g.tiles_per_cb = cdiv(H, sub);
        g.nrows = sub + 2 * g.halo;
    } else {
        g.sub_stride = 128;
        g.tile_f = sub * 128;
        g.tiles_per_cb = cdiv(H * g.Sp, g.tile_f);
        // the reads of a tile span sub*128 positions plus halo*(Sp+1) on each side, which starts
        // anywhere in the window's first row
        g.nrows = 2 + 2 * g.halo + (sub * 128) / g.Sp;
    }
    if (g.nrows > 256 || g.Sp > 256) return false;
    // pipeline stages
    const int rowb = CB * 2;
    const int a_bytes = rowb * g.Sp * g.nrows;
    L->a_stage_bytes = (a_bytes + 1023) & ~1023;
    // a B stage holds the taps of `rb` kernel rows (3 or 9 taps) for one N slice: the larger
    // stage amortises the per-stage work of the MMA warps for narrow N with four row groups
    // (measured faster there; with two row groups the deeper 3-tap ring wins)
    L->rb = (ks == 3 && 9 * L->NT * rowb <= 64 * 1024 && (sub >= 4 || up2)) ? 3 : 1;
    L->rb = ov(CC3D_SCHED_TAP_ROWS, L->rb);
    if (L->rb != 1 && L->rb != 3) return false;
    // weight rows of one block (the two-frame schedule's stacked stages hold a whole tap)
    const int b_rows = L->pair && !L->tstack ? L->NT / 2 : L->NT;
    // pairs: 9-tap weight stages in the row-aligned geometry (c96), 3-tap ones in the flat
    // geometry, whose wide windows leave room for only two 9-tap stages (the weight ring was the
    // wait there: c384 1960 against 1837 TFLOP/s)
    if (L->pair) L->rb = ov(CC3D_SCHED_TAP_ROWS, ks == 3 && W % 128 == 0 ? 3 : 1);
    if (L->tstack) L->rb = ov(CC3D_SCHED_TAP_ROWS, 3);  // 9-tap stages: measured 8 % faster than 3-tap on c96
    if ((L->rb != 1 && L->rb != 3) || ks % L->rb != 0) return false;
    L->b_stage_bytes = (ks * L->rb * b_rows * rowb + 1023) & ~1023;
    const int budget = 220 * 1024 - 4 * ntot * L->ncoblk;
    L->na = (L->a_stage_bytes > 40 * 1024) ? 2 : 3;
    L->na = ov(CC3D_SCHED_WINDOW_STAGES, L->na);
    if (L->na < 2 || L->na > kMaxStages) return false;
    int nb = (budget - L->na * L->a_stage_bytes) / L->b_stage_bytes;
    if (nb > kMaxStages) nb = kMaxStages;
    const int nb_env = ov(CC3D_SCHED_WEIGHT_STAGES, 0);
    if (nb_env >= 2 && nb_env < nb) nb = nb_env;
    if (nb < 2) {
        L->na = 2;
        nb = (budget - L->na * L->a_stage_bytes) / L->b_stage_bytes;
        if (nb > kMaxStages) nb = kMaxStages;
    }
    if (nb < 2 && L->rb == 3 && ov(CC3D_SCHED_TAP_ROWS, 0) == 0) {
        // the 9-tap weight stages do not fit beside two windows: 3-tap stages
        L->rb = 1;
        L->b_stage_bytes = (ks * b_rows * rowb + 1023) & ~1023;
        nb = (budget - L->na * L->a_stage_bytes) / L->b_stage_bytes;
        if (nb > kMaxStages) nb = kMaxStages;
    }
    if (nb < 2) return false;
    L->nb = nb;
    // L2 prefetch of the next tile's windows: 0 none, 1..3 = that many temporal taps (newest first);
    // off by default: measured slower on every decoder shape (it competes with the live working set)
    L->prefetch = ov(CC3D_SCHED_PREFETCH, 0);
    if (L->prefetch < 0 || L->prefetch > 3) L->prefetch = 0;
    L->smem_bytes =
        (size_t)L->na * L->a_stage_bytes + (size_t)L->nb * L->b_stage_bytes + 4 * ntot * L->ncoblk + 1024;
    // one block per SM: a second resident block would wait inside its tensor-memory allocation
    if (L->smem_bytes < 120 * 1024) L->smem_bytes = 120 * 1024;
    return true;
}

}  // namespace

bool tc_configure(int CB, int T, int H, int W, int Cin, int Cout, int kt, int ks, bool has_residual, bool up2,
                  const TcOverrides* ov, TcLaunch* L)
{
    // the preferred tile height and column blocks of up to 254 pixels first; wide flat windows may
    // need fewer row groups, then narrower column blocks, to leave room for two windows and two
    // weight stages in shared memory
    for (int smax : {254, 128})
        for (int cap = 4; cap >= 1; cap /= 2)
            if (tc_configure_capped(CB, T, H, W, Cin, Cout, kt, ks, has_residual, up2, cap, smax, ov, L)) return true;
    return false;
}

cudaError_t tc_launch(int CB, const TcLaunch& L, cudaStream_t stream)
{
    if (L.tstack) return tc2s_launch(CB, L, stream);
    if (L.pair) return tc2_launch(CB, L, stream);
    const int subi = (L.issuers == 2 && !L.split_n && !L.up2) ? L.g.sub / 2 : L.g.sub;
    void* kern = CB == 16 ? (L.rb == 3 ? kernel_for<16, 3>(subi) : kernel_for<16, 1>(subi))
                          : (L.rb == 3 ? kernel_for<32, 3>(subi) : kernel_for<32, 1>(subi));
    if (kern == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem_bytes);
    if (e != cudaSuccess) return e;
    void* args[] = {const_cast<TcLaunch*>(&L)};
    return cudaLaunchKernel(kern, dim3(L.grid), dim3(kThreads), args, L.smem_bytes, stream);
}

}  // namespace cc3d
