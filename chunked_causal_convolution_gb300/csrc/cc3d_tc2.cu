// cc3d_tc2.cu -- the causal 3x3x3 convolution on SM pairs (tcgen05 cta_group::2).
//
// Same tiling, operand layout and accumulation order as the one-SM kernel in cc3d_tc.cu, with
// two blocks of a 2-block cluster working as one unit:
//   * block r of the pair owns its own output tile (tile 2p + r) and its own input windows;
//   * every weight stage is split: block r holds output channels [r*NT/2, (r+1)*NT/2) of the
//     stage's taps, so each block stores and reads half of the weights;
//   * the leader block (rank 0) issues M = 256 MMAs: rows 0-127 come from the leader's window
//     view, rows 128-255 from the same shared-memory offset in the peer's window, B comes half
//     from each block, and each block's tensor memory receives its own 128 rows x NT columns;
//   * copies of both blocks are counted on the leader's "full" barriers; the leader's commits
//     are multicast to both blocks' "empty" and accumulator barriers; the epilogues of both
//     blocks release the accumulators on the leader's barrier.
// Per block and 128x96x16 step the tensor core reads 4 KB of activations and 1.5 KB of weights
// from shared memory instead of 4 + 3 KB, and one issued instruction does twice the work.
//
// Requirement: both tiles of a pair must use the same window offsets and weights.  Tiles are
// ordered frame fastest, so with an even number of frames the pair's tiles are two frames at one
// spatial position and output-channel block, in any geometry; with an odd number the host
// selects this kernel only for one channel block in the row-aligned geometry (W a multiple of
// 128), where every tile has the same offsets.  Up to 192 output channels per block (96 weight
// rows in each block of the pair).
#include <cuda_bf16.h>

#include "cc3d_internal.h"
#include "cc3d_ptx.cuh"
#include "cc3d_tc_common.cuh"

namespace cc3d {
using namespace ptx;
using namespace tcc;

namespace {

template <int CB, int SUBI, int RB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc2_bf16_kernel(const __grid_constant__ TcLaunch L)
{
    constexpr uint32_t ROWB = CB * 2;
    constexpr uint32_t ROWU = ROWB / 16;
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
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int Sp = L.g.Sp;
    const int NT = L.NT;
    const int NH = NT / 2;  // weight rows of each block
    const int nsplit = L.nsplit;
    const int ncb = L.Cin / CB;
    const int SUB = L.g.sub;
    const int nissue = L.issuers;
    const int ntiles = L.g.tiles_per_cb * L.g.ncolblk * L.T * L.ncoblk;
    const int npairs = (ntiles + 1) / 2;
    const int pair0 = blockIdx.x / 2, pstride = gridDim.x / 2;
    const int cout_pad = L.ncoblk * nsplit * NT;
    const uint32_t acc_cols = (uint32_t)(SUB * nsplit * NT);
    const unsigned long long budget = L.wait_ns;
    const int KSZ = L.ks;     // spatial kernel extent (kh = kw): 3, or 1 for temporal / pointwise kernels
    const int P = L.kt - 1;   // history frames in the cache

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < L.na; ++s) { mbar_init(&a_full[s], 1); mbar_init(&a_empty[s], nissue); }
        for (int s = 0; s < L.nb; ++s) { mbar_init(&b_full[s], 1); mbar_init(&b_empty[s], nissue); }
        for (int a = 0; a < L.acc_stages; ++a) { mbar_init(&acc_full[a], nissue); mbar_init(&acc_empty[a], 8); }
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
        tmem_alloc_pair(&tmem_base_sh, (uint32_t)L.tmem_cols);
        tmem_relinquish_pair();
    }
    if (warp >= 4) {
        const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(L.bias);
        for (int i = threadIdx.x - 128; i < cout_pad; i += 128)
            s_bias[i] = (b != nullptr && i < L.Cout) ? __bfloat162float(b[i]) : 0.0f;
    }
    tc_fence_before();
    __syncthreads();
    // both blocks' barriers must exist before either block signals the other
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA loader (both blocks)
        // Copies of both blocks complete on the leader's full barriers; the leader announces the
        // bytes of the pair.  A block refills a stage once the leader's MMAs released it (the
        // release is multicast to this block's empty barrier).
        if (lane == 0) {
            int sa = 0, pa = 0, sb = 0, pb = 0;
            int last_pa[kMaxStages], last_pb[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) last_pa[s] = last_pb[s] = -1;
            const uint32_t a_tx = (uint32_t)(ROWB * Sp * L.g.nrows);
            const uint32_t b_tx = (uint32_t)(ROWB * NH * KSZ * RB);
            bool skip_first = (L.fault == 1);
            bool ok = true;
            for (int p = pair0; ok && p < npairs; p += pstride) {
                const TileCoord c = tile_coord(L, 2 * p + (int)rank);
                for (int dt = 0; ok && dt < L.kt; ++dt) {
                    const int tin = c.t + dt - P;
                    const CUtensorMap* map = &L.map_x;
                    int tc = tin;
                    if (tin < 0 && L.has_cache) { map = &L.map_cache; tc = tin + P; }
                    for (int cb = 0; ok && cb < ncb; ++cb) {
                        if (!bounded_wait(&a_empty[sa], pa ^ 1, budget, &abort_flag)) {
                            if (!abort_flag) record_failure(L, STATUS_TIMEOUT_LOADER, &abort_flag);
                            ok = false;
                            break;
                        }
                        if (leader) mbar_arrive_expect_tx(&a_full[sa], 2 * a_tx);
                        if (!skip_first)
                            tma_load_4d_pair(smA + (size_t)sa * L.a_stage_bytes, map,
                                             mapa_shared(smem_u32(&a_full[sa]), 0), cb * CB, c.w0 - 1, c.hstart, tc);
                        skip_first = false;
                        last_pa[sa] = pa;
                        if (++sa == L.na) { sa = 0; pa ^= 1; }
                        for (int dg = 0; ok && dg < KSZ / RB; ++dg) {
                            for (int ns = 0; ns < nsplit; ++ns) {
                                if (!bounded_wait(&b_empty[sb], pb ^ 1, budget, &abort_flag)) {
                                    if (!abort_flag) record_failure(L, STATUS_TIMEOUT_LOADER, &abort_flag);
                                    ok = false;
                                    break;
                                }
                                if (leader) mbar_arrive_expect_tx(&b_full[sb], 2 * b_tx);
                                tma_load_3d_pair(smB + (size_t)sb * L.b_stage_bytes, &L.map_w,
                                                 mapa_shared(smem_u32(&b_full[sb]), 0), cb * CB,
                                                 c.co0 + ns * NT + (int)rank * NH, dt * KSZ * KSZ + dg * RB * KSZ);
                                last_pb[sb] = pb;
                                if (++sb == L.nb) { sb = 0; pb ^= 1; }
                            }
                        }
                    }
                }
            }
            // the leader's full barriers count the copies of both blocks: once they have landed,
            // nothing more is in flight into either block (the peer waits for this at the cluster
            // barrier below before it may exit)
            if (leader) {
                for (int s = 0; s < L.na; ++s)
                    if (last_pa[s] >= 0 && !bounded_wait(&a_full[s], (uint32_t)last_pa[s], budget, nullptr))
                        atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
                for (int s = 0; s < L.nb; ++s)
                    if (last_pb[s] >= 0 && !bounded_wait(&b_full[s], (uint32_t)last_pb[s], budget, nullptr))
                        atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
            }
        }
    } else if (leader && (warp == 1 || (warp == 2 && nissue == 2))) {
        // ------------------------------------------------------------ MMA issuers (leader only)
        const int k = warp - 1;
        // Lane 0 issues every MMA and commit of this warp: it is the lane that polls the full
        // barriers (warp_bounded_wait), so the thread that observes a stage's completion is the one
        // whose MMAs read it, and a commit tracks the MMAs of the thread that issues it.  (An
        // elect.sync per MMA made the warp reconverge before every instruction and was measured
        // 10 % slower; a lane elected once need not be the polling lane, and that form gave wrong
        // results on first launches.)
        const bool lead = lane == 0;
        const int m0 = L.split_n ? 0 : k * SUBI;
        const int ns_lo = L.split_n ? k : 0, ns_hi = L.split_n ? k + 1 : nsplit;
        const uint32_t idesc = make_idesc_bf16_f32(256, NT);
        const uint64_t a_desc0 = make_sdesc(smem_u32(smA), 16, SBO, LAYOUT, 0);
        const uint64_t b_desc0 = make_sdesc(smem_u32(smB), 16, SBO, LAYOUT, 0);
        const uint32_t a_inc = (uint32_t)L.a_stage_bytes >> 4;
        const uint32_t b_inc = (uint32_t)L.b_stage_bytes >> 4;
        const uint32_t b_tap_inc = (uint32_t)NH * ROWU;  // next tap inside a (half) B stage
        const uint32_t row_shift = (uint32_t)Sp * ROWU;
        const uint32_t m_cols = (uint32_t)(nsplit * NT);
        int sa = 0, pa = 0, sb = 0, pb = 0;
        bool ok = true;
        int it = 0;
        for (int p = pair0; ok && p < npairs; p += pstride, ++it) {
            const TileCoord c = tile_coord(L, 2 * p);
            const int as = it % L.acc_stages;
            const int aph = (it / L.acc_stages) & 1;
            if (!warp_bounded_wait(&acc_empty[as], aph ^ 1, budget, &abort_flag)) {
                if (lane == 0 && !abort_flag) record_failure(L, STATUS_TIMEOUT_MMA, &abort_flag);
                break;
            }
            tc_fence_after();
            const uint32_t dbase = tmem + (uint32_t)as * acc_cols;
            // row-aligned tiles: the window offsets are the same in both blocks of the pair
            uint32_t rowu[SUBI];
#pragma unroll
            for (int m = 0; m < SUBI; ++m)
                rowu[m] = (uint32_t)(c.f0 + (m0 + m) * L.g.sub_stride - c.hstart * Sp - L.g.halo * (Sp + 1)) * ROWU;
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
                            const uint32_t dcol = dbase + (uint32_t)(ns * NT) + (uint32_t)m0 * m_cols;
                            const bool mine = ns >= ns_lo && ns < ns_hi;
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
                                            const uint64_t bd = desc_add(b_st, (dr * KSZ + dw) * b_tap_inc + ks * 2);
                                            const uint32_t acc = (first_row && dw == 0 && ks == 0) ? 0u : 1u;
                                            if (mine && lead)
                                                umma_bf16_ss_pair(dcol + (uint32_t)m * m_cols, ad, bd, idesc, acc);
                                        }
                                    }
                                }
                            }
                            if (lead) umma_commit_pair(&b_empty[sb], 3);
                            __syncwarp();
                            if (++sb == L.nb) { sb = 0; pb ^= 1; }
                        }
                    }
                    if (!ok) break;
                    if (lead) umma_commit_pair(&a_empty[sa], 3);
                    if (++sa == L.na) { sa = 0; pa ^= 1; }
                }
            }
            if (!ok) break;
            if (lead) umma_commit_pair(&acc_full[as], 3);
        }
        if (lead) umma_commit_pair(&mma_drain[k], 1);
        __syncwarp();
        if (!warp_bounded_wait(&mma_drain[k], 0, budget, nullptr) && lane == 0)
            atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
    } else if (warp == 3) {
        // ------------------------------------------------------------ temporal cache update
        if (L.copy_hist) copy_history(L, P, 0, 1, lane);
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue (both blocks)
        const int q = warp - 4;
        const __nv_bfloat16* res = reinterpret_cast<const __nv_bfloat16*>(L.res);
        __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(L.y);
        const bool wide = (L.Cout % 16) == 0;
        int it = 0;
        for (int p = pair0; p < npairs; p += pstride, ++it) {
            const int as = it % L.acc_stages;
            const int aph = (it / L.acc_stages) & 1;
            const TileCoord c = tile_coord(L, 2 * p + (int)rank);
            if (res != nullptr && wide) {
                for (int m = 0; m < SUB; ++m) {
                    const int f = c.f0 + m * L.g.sub_stride + q * 32 + lane;
                    const int h = f / Sp;
                    const int jcol = f - h * Sp;
                    const int w = c.w0 + jcol - 1;
                    if (c.t < L.T && h < L.H && jcol >= 1 && jcol <= L.g.S && w < L.W) {
                        const char* pp = reinterpret_cast<const char*>(
                            res + (((size_t)c.t * L.H + h) * L.W + w) * L.Cout);
                        for (int o = 0; o < L.Cout * 2; o += 128) prefetch_l2(pp + o);
                    }
                }
            }
            int ready = 0;
            if (lane == 0) {
                ready = bounded_wait(&acc_full[as], aph, budget, &abort_flag, kEpilogueSleepNs);
                if (!ready && !abort_flag) record_failure(L, STATUS_TIMEOUT_EPILOGUE, &abort_flag);
            }
            ready = __shfl_sync(0xffffffffu, ready, 0);
            if (!ready) break;
            tc_fence_after();
            const uint32_t rel = leader ? 0u : mapa_shared(smem_u32(&acc_empty[as]), 0);
            for (int m = 0; m < SUB; ++m) {
                const int f = c.f0 + m * L.g.sub_stride + q * 32 + lane;
                const int h = f / Sp;
                const int jcol = f - h * Sp;
                const int w = c.w0 + jcol - 1;
                // a phantom tile (odd tile count) lies outside the video: nothing is stored
                const bool valid = (2 * p + (int)rank) < ntiles && h < L.H && jcol >= 1 && jcol <= L.g.S && w < L.W;
                const size_t px = ((size_t)(valid ? c.t : 0) * L.H + (valid ? h : 0)) * L.W + (valid ? w : 0);
                for (int ns = 0; ns < nsplit; ++ns) {
                    const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)as * acc_cols +
                                           (uint32_t)((m * nsplit + ns) * NT);
                    const bool last_slice = (m == SUB - 1) && (ns == nsplit - 1);
                    // the release goes to the leader, whose MMA warps wait on it
                    epilogue_slice(tbase, NT, c.co0 + ns * NT, px, valid, last_slice, s_bias, L.Cout, wide, res, y, L.v32 != 0,
                                   [&]() {
                                       tc_fence_before();
                                       __syncwarp();
                                       if (lane == 0) {
                                           if (leader)
                                               mbar_arrive(&acc_empty[as]);
                                           else
                                               mbar_arrive_remote(rel);
                                       }
                                   });
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // neither block frees its tensor memory or leaves while the pair may still use its shared
    // memory, barriers or tensor memory
    cluster_sync_all();
    tc_fence_after();
    if (warp == 2) tmem_dealloc_pair(tmem, (uint32_t)L.tmem_cols);
}

template <int CB, int RB>
void* kernel2_for(int sub)
{
    switch (sub) {
    case 1: return reinterpret_cast<void*>(tc2_bf16_kernel<CB, 1, RB>);
    case 2: return reinterpret_cast<void*>(tc2_bf16_kernel<CB, 2, RB>);
    default: return nullptr;
    }
}

}  // namespace

cudaError_t tc2_launch(int CB, const TcLaunch& L, cudaStream_t stream)
{
    const int subi = (L.issuers == 2 && !L.split_n) ? L.g.sub / 2 : L.g.sub;
    void* kern = CB == 16 ? (L.rb == 3 ? kernel2_for<16, 3>(subi) : kernel2_for<16, 1>(subi))
                          : (L.rb == 3 ? kernel2_for<32, 3>(subi) : kernel2_for<32, 1>(subi));
    if (kern == nullptr) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem_bytes);
    if (e != cudaSuccess) return e;
    // as many pairs as can be resident at once, at most one per two SMs and per pair of tiles
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L.smem_bytes;
    cfg.stream = stream;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
        cudaGetLastError();
        clusters = L.grid / 2;
    }
    int grid = L.grid;
    if (grid > 2 * clusters) grid = 2 * clusters;
    if (grid < 2) grid = 2;
    void* args[] = {const_cast<TcLaunch*>(&L)};
    return cudaLaunchKernel(kern, dim3(grid), dim3(kThreads), args, L.smem_bytes, stream);
}

}  // namespace cc3d
