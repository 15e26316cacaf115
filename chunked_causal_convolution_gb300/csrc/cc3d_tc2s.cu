// cc3d_tc2s.cu -- the causal kt x 3 x 3 convolution on SM pairs with two output frames stacked
// into the N dimension of every MMA whose input frame is a tap of both.
//
// Output frame t reads input frames t - P .. t (P = kt - 1, temporal tap dt = input - t + P).  A
// tile here is a pair of output frames (t, t + 1) at one spatial position, and its input frames
// j = 0 .. kt are input t - P + j:
//   * j = 0 is a tap of frame t only (dt = 0):                   N = NT,  into frame t's columns
//   * 0 < j < kt is a tap of both (dt = j for t, j - 1 for t + 1): N = 2NT, into both
//   * j = kt is a tap of frame t + 1 only (dt = kt - 1):           N = NT,  into frame t + 1's
// so each staged input window is read by the tensor core kt + 1 times per two output frames
// instead of 2 kt times (a third fewer operand reads from shared memory for kt = 3), while the
// accumulation order of every output (dt, channel block, dh, dw, 16-channel step) and therefore
// every result bit is that of the one-frame kernels.
//
// SM-pair layout (cta_group::2, M = 256): block r owns tile 2p + r (its own two 128-row groups,
// one per MMA warp); A comes from each block's own window at the same offset.  B is split by N
// across the pair: for the stacked stages block 0 holds the NT weight rows of frame t's tap and
// block 1 those of frame t + 1's, for the one-frame stages each block holds half of the tap's rows.
// The stacked columns of frame t + 1 accumulate onto zeros (the MMA's accumulate flag covers all
// N columns and frame t's columns already hold the j = 0 sums): the epilogue writes zeros into
// them after reading them out.
//
// Tensor memory: per block 2 row groups x 2 frames x NT columns, one buffer.  Frame t's columns
// are complete after stage kt - 1 and are drained while stage kt runs; frame t + 1's after stage
// kt, drained while the next tile's stage 0 runs, each within one stage's time.  Each (frame, row
// group) quarter is released on its own barrier, which the MMA warp of that row group waits for
// before its first write; the epilogue reads both row groups of a frame into registers and
// releases them before any memory access (so NT <= 96: 192 accumulator registers a thread).
#include <cuda_bf16.h>

#include "cc3d_internal.h"
#include "cc3d_ptx.cuh"
#include "cc3d_tc_common.cuh"

namespace cc3d {
using namespace ptx;
using namespace tcc;

namespace {

constexpr int kSub = 2;  // 128-row groups per block, one per MMA warp
// warps: 0 loader, 1-2 MMA issuers (leader block), 3 history copy, 4-7 epilogue (warp 4 + q drains
// lane quadrant q, the quadrant a warp may access being its index mod 4, of both row groups)
constexpr int kThreads2s = 256;

__device__ __forceinline__ TileCoord frame_pair_tile(const TcLaunch& L, int tile)
{
    // order: frame pair fastest, then the row group position inside the column block, then the
    // column block (row-aligned geometry: every tile starts at padded column 1 of a row)
    const int T2 = (L.T + 1) / 2;
    TileCoord c;
    c.t = 2 * (tile % T2);
    const int r = tile / T2;
    c.co0 = 0;
    const int i = r % L.g.tiles_per_cb;
    const int cbk = r / L.g.tiles_per_cb;
    c.w0 = cbk * L.g.S;
    c.f0 = i * L.g.tile_f + 1;
    c.hstart = floor_div(c.f0 - L.g.halo * (L.g.Sp + 1), L.g.Sp);
    return c;
}

// the residual rows of this thread's output position, warmed in L2 while the accumulators fill
__device__ __forceinline__ void prefetch_residual(const __nv_bfloat16* res, size_t px, int Cout, bool valid)
{
    if (res == nullptr || !valid) return;
    const char* p = reinterpret_cast<const char*>(res + px * Cout);
    for (int o = 0; o < Cout * 2; o += 128) prefetch_l2(p + o);
}

template <int CB, int RB>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads2s, 1)
    tc2s_bf16_kernel(const __grid_constant__ TcLaunch L)
{
    constexpr uint32_t ROWB = CB * 2;
    constexpr uint32_t ROWU = ROWB / 16;
    constexpr uint32_t LAYOUT = CB == 32 ? LAYOUT_SW64 : LAYOUT_SW32;
    constexpr uint32_t SBO = 8 * ROWB;
    constexpr int KSTEPS = CB / 16;
    constexpr int KSZ = 3;

    extern __shared__ uint8_t dsm_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smA = sm;
    uint8_t* smB = sm + (size_t)L.na * L.a_stage_bytes;
    float* s_bias = reinterpret_cast<float*>(smB + (size_t)L.nb * L.b_stage_bytes);

    __shared__ uint64_t a_full[kMaxStages], a_empty[kMaxStages], b_full[kMaxStages], b_empty[kMaxStages];
    // accumulator handshakes: frame t ("A") and frame t + 1 ("B") complete separately; each
    // (frame, row group) quarter is released separately
    __shared__ uint64_t accA_full, accB_full, accA_empty[kSub], accB_empty[kSub], mma_drain[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int Sp = L.g.Sp;
    const int NT = L.NT;
    const int NH = NT / 2;
    const int ncb = L.Cin / CB;
    const int P = L.kt - 1;
    const int nj = L.kt + 1;  // input frames of a frame pair
    const int T2 = (L.T + 1) / 2;
    const int ntiles = L.g.tiles_per_cb * L.g.ncolblk * T2;
    const int npairs = (ntiles + 1) / 2;
    const int pair0 = blockIdx.x / 2, pstride = gridDim.x / 2;
    const unsigned long long budget = L.wait_ns;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int s = 0; s < L.na; ++s) { mbar_init(&a_full[s], 1); mbar_init(&a_empty[s], kSub); }
        for (int s = 0; s < L.nb; ++s) { mbar_init(&b_full[s], 1); mbar_init(&b_empty[s], kSub); }
        mbar_init(&accA_full, kSub);
        mbar_init(&accB_full, kSub);
        for (int m = 0; m < kSub; ++m) {
            mbar_init(&accA_empty[m], 8);  // 4 epilogue warps in each block of the pair
            mbar_init(&accB_empty[m], 8);
        }
        mbar_init(&mma_drain[0], 1);
        mbar_init(&mma_drain[1], 1);
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&L.map_x);
        prefetch_tensormap(&L.map_w);
        prefetch_tensormap(&L.map_w2);
        if (L.has_cache) prefetch_tensormap(&L.map_cache);
    }
    if (warp == 2) {
        tmem_alloc_pair(&tmem_base_sh, (uint32_t)L.tmem_cols);
        tmem_relinquish_pair();
    }
    if (warp >= 4) {
        const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(L.bias);
        for (int i = threadIdx.x - 128; i < NT; i += kThreads2s - 128)
            s_bias[i] = (b != nullptr && i < L.Cout) ? __bfloat162float(b[i]) : 0.0f;
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA loader (both blocks)
        if (lane == 0) {
            int sa = 0, pa = 0, sb = 0, pb = 0;
            int last_pa[kMaxStages], last_pb[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) last_pa[s] = last_pb[s] = -1;
            const uint32_t a_tx = (uint32_t)(ROWB * Sp * L.g.nrows);
            const uint32_t b_tx_half = (uint32_t)(ROWB * NH * KSZ * RB);
            const uint32_t b_tx_full = (uint32_t)(ROWB * NT * KSZ * RB);
            bool skip_first = (L.fault == 1);
            bool ok = true;
            for (int p = pair0; ok && p < npairs; p += pstride) {
                const TileCoord c = frame_pair_tile(L, 2 * p + (int)rank);
                for (int j = 0; ok && j < nj; ++j) {
                    // input frame t - P + j: from the history when negative; past the chunk's end
                    // (an odd chunk's last pair) the copy reads the zero fill
                    const int tin = c.t + j - P;
                    const CUtensorMap* map = &L.map_x;
                    int tc = tin;
                    if (tin < 0 && L.has_cache) { map = &L.map_cache; tc = tin + P; }
                    const bool stacked = j > 0 && j < L.kt;
                    const int dt = j == 0 ? 0 : (j == L.kt ? L.kt - 1 : j - (int)rank);
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
                        for (int dg = 0; dg < KSZ / RB; ++dg) {
                            if (!bounded_wait(&b_empty[sb], pb ^ 1, budget, &abort_flag)) {
                                if (!abort_flag) record_failure(L, STATUS_TIMEOUT_LOADER, &abort_flag);
                                ok = false;
                                break;
                            }
                            if (leader) mbar_arrive_expect_tx(&b_full[sb], 2 * (stacked ? b_tx_full : b_tx_half));
                            const uint32_t bar = mapa_shared(smem_u32(&b_full[sb]), 0);
                            uint8_t* dst = smB + (size_t)sb * L.b_stage_bytes;
                            if (stacked)
                                tma_load_3d_pair(dst, &L.map_w2, bar, cb * CB, 0, dt * 9 + dg * RB * KSZ);
                            else
                                tma_load_3d_pair(dst, &L.map_w, bar, cb * CB, (int)rank * NH, dt * 9 + dg * RB * KSZ);
                            last_pb[sb] = pb;
                            if (++sb == L.nb) { sb = 0; pb ^= 1; }
                        }
                    }
                }
            }
            // the leader's full barriers count the copies of both blocks (see the pair kernel)
            if (leader) {
                for (int s = 0; s < L.na; ++s)
                    if (last_pa[s] >= 0 && !bounded_wait(&a_full[s], (uint32_t)last_pa[s], budget, nullptr))
                        atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
                for (int s = 0; s < L.nb; ++s)
                    if (last_pb[s] >= 0 && !bounded_wait(&b_full[s], (uint32_t)last_pb[s], budget, nullptr))
                        atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
            }
        }
    } else if (leader && (warp == 1 || warp == 2)) {
        // ------------------------------------------------------------ MMA issuers (leader only)
        // warp 1 + k issues the MMAs of row group k of both blocks; lane 0 polls and issues (the
        // thread that observes a stage's completion is the one whose MMAs read it)
        const int k = warp - 1;
        const bool lead = lane == 0;
        const uint32_t idesc1 = make_idesc_bf16_f32(256, NT);
        const uint32_t idesc2 = make_idesc_bf16_f32(256, 2 * NT);
        const uint64_t a_desc0 = make_sdesc(smem_u32(smA), 16, SBO, LAYOUT, 0);
        const uint64_t b_desc0 = make_sdesc(smem_u32(smB), 16, SBO, LAYOUT, 0);
        const uint32_t a_inc = (uint32_t)L.a_stage_bytes >> 4;
        const uint32_t b_inc = (uint32_t)L.b_stage_bytes >> 4;
        const uint32_t row_shift = (uint32_t)Sp * ROWU;
        const uint32_t colA = tmem + (uint32_t)(k * 2 * NT);
        const uint32_t colB = colA + (uint32_t)NT;
        int sa = 0, pa = 0, sb = 0, pb = 0;
        bool ok = true;
        int it = 0;
        for (int p = pair0; ok && p < npairs; p += pstride, ++it) {
            const TileCoord c = frame_pair_tile(L, 2 * p);
            const uint32_t ph = (uint32_t)(it & 1);
            const uint32_t rowu =
                (uint32_t)(c.f0 + k * L.g.sub_stride - c.hstart * Sp - L.g.halo * (Sp + 1)) * ROWU;
            for (int j = 0; ok && j < nj; ++j) {
                // frame t's quarter must be drained before stage 0 writes it, frame t + 1's (and
                // zeroed) before stage 1; the B barrier completes once at start-up, after the
                // first zeroing
                if (j <= 1) {
                    uint64_t* bar = j == 0 ? &accA_empty[k] : &accB_empty[k];
                    if (!warp_bounded_wait(bar, j == 0 ? ph ^ 1u : ph, budget, &abort_flag)) {
                        if (lane == 0 && !abort_flag) record_failure(L, STATUS_TIMEOUT_MMA, &abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                const bool stacked = j > 0 && j < L.kt;
                const uint32_t dcol = j == L.kt ? colB : colA;
                const uint32_t idesc = stacked ? idesc2 : idesc1;
                const uint32_t b_tap_inc = (uint32_t)(stacked ? NT : NH) * ROWU;
                for (int cb = 0; ok && cb < ncb; ++cb) {
                    if (!warp_bounded_wait(&a_full[sa], pa, budget, &abort_flag)) {
                        if (lane == 0 && !abort_flag) record_failure(L, STATUS_TIMEOUT_MMA, &abort_flag);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t a_st = a_desc0 + (uint64_t)(sa * a_inc);
                    for (int dg = 0; dg < KSZ / RB; ++dg) {
                        if (!warp_bounded_wait(&b_full[sb], pb, budget, &abort_flag)) {
                            if (lane == 0 && !abort_flag) record_failure(L, STATUS_TIMEOUT_MMA, &abort_flag);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint64_t b_st = b_desc0 + (uint64_t)(sb * b_inc);
#pragma unroll
                        for (int dr = 0; dr < RB; ++dr) {
                            const int dh = dg * RB + dr;
                            const uint64_t a_row = desc_add(a_st, dh * row_shift + rowu);
                            const bool first = (j | cb | dh) == 0;
#pragma unroll
                            for (int dw = 0; dw < KSZ; ++dw) {
#pragma unroll
                                for (int ks = 0; ks < KSTEPS; ++ks) {
                                    const uint64_t ad = desc_add(a_row, dw * ROWU + ks * 2);
                                    const uint64_t bd = desc_add(b_st, (dr * KSZ + dw) * b_tap_inc + ks * 2);
                                    const uint32_t acc = (first && dw == 0 && ks == 0) ? 0u : 1u;
                                    if (lead) umma_bf16_ss_pair(dcol, ad, bd, idesc, acc);
                                }
                            }
                        }
                        if (lead) umma_commit_pair(&b_empty[sb], 3);
                        __syncwarp();
                        if (++sb == L.nb) { sb = 0; pb ^= 1; }
                    }
                    if (!ok) break;
                    if (lead) umma_commit_pair(&a_empty[sa], 3);
                    if (++sa == L.na) { sa = 0; pa ^= 1; }
                }
                if (!ok) break;
                if (j == L.kt - 1 && lead) umma_commit_pair(&accA_full, 3);
                if (j == L.kt && lead) umma_commit_pair(&accB_full, 3);
            }
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
        const int q = warp - 4;  // lane quadrant of tensor memory this warp may access
        const __nv_bfloat16* res = reinterpret_cast<const __nv_bfloat16*>(L.res);
        __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(L.y);
        const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16);
        auto release_to = [&](uint64_t* bar) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(bar);
                else
                    mbar_arrive_remote(mapa_shared(smem_u32(bar), 0));
            }
        };
        // frame t + 1's columns start at zero (the stacked MMAs accumulate onto them)
        for (int m = 0; m < kSub; ++m) {
            const uint32_t tb = lane_base + (uint32_t)(m * 2 * NT + NT);
            int cc = 0;
            for (; cc + 32 <= NT; cc += 32) tmem_st_32x32b_x32_zero(tb + (uint32_t)cc);
            if (cc < NT) tmem_st_32x32b_x16_zero(tb + (uint32_t)cc);
            tmem_st_wait();
            release_to(&accB_empty[m]);
        }
        int it = 0;
        for (int p = pair0; p < npairs; p += pstride, ++it) {
            const uint32_t ph = (uint32_t)(it & 1);
            const int tile = 2 * p + (int)rank;
            const TileCoord c = frame_pair_tile(L, tile);
            for (int half = 0; half < 2; ++half) {
                const int t = c.t + half;
                // this lane's output position in row group m; a phantom tile (odd tile count) and
                // the second frame of an odd chunk's last pair lie outside the output: nothing is
                // stored there
                auto position = [&](int m, size_t* px) {
                    const int f = c.f0 + m * L.g.sub_stride + q * 32 + lane;
                    const int h = f / Sp;
                    const int jcol = f - h * Sp;
                    const int w = c.w0 + jcol - 1;
                    const bool valid =
                        tile < ntiles && t < L.T && h < L.H && jcol >= 1 && jcol <= L.g.S && w < L.W;
                    *px = ((size_t)(valid ? t : 0) * L.H + (valid ? h : 0)) * L.W + (valid ? w : 0);
                    return valid;
                };
                // both frames' residual rows are warmed at the start of the tile: frame t + 1's
                // are read right after its columns are released, too soon after frame t's stores
                // for a prefetch issued there to have landed
                if (half == 0) {
                    for (int m = 0; m < kSub; ++m) {
                        size_t px;
                        const bool valid = position(m, &px);
                        prefetch_residual(res, px, L.Cout, valid);
                        prefetch_residual(res, px + (size_t)L.H * L.W, L.Cout, valid && t + 1 < L.T);
                    }
                }
                int ready = 0;
                if (lane == 0) {
                    ready = bounded_wait(half == 0 ? &accA_full : &accB_full, ph, budget, &abort_flag,
                                         kEpilogueSleepNs);
                    if (!ready && !abort_flag) record_failure(L, STATUS_TIMEOUT_EPILOGUE, &abort_flag);
                }
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (!ready) break;
                tc_fence_after();
                uint32_t r0[96], r1[96];
                const uint32_t tb0 = lane_base + (uint32_t)(half * NT);
                const uint32_t tb1 = tb0 + (uint32_t)(2 * NT);
                tmem_read_quarter<96>(tb0, NT, r0);
                tmem_read_quarter<96>(tb1, NT, r1);
                tmem_ld_wait();
                if (half == 1) {
                    tmem_zero_quarter<96>(tb0, NT);
                    tmem_zero_quarter<96>(tb1, NT);
                    tmem_st_wait();
                }
                release_to(half == 0 ? &accA_empty[0] : &accB_empty[0]);
                release_to(half == 0 ? &accA_empty[1] : &accB_empty[1]);
                size_t px;
                if (position(0, &px)) store_quarter<96>(r0, NT, 0, px, s_bias, L.Cout, res, y, L.v32 != 0);
                if (position(1, &px)) store_quarter<96>(r1, NT, 0, px, s_bias, L.Cout, res, y, L.v32 != 0);
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

}  // namespace

cudaError_t tc2s_launch(int CB, const TcLaunch& L, cudaStream_t stream)
{
    void* kern = CB == 32 ? (L.rb == 3 ? reinterpret_cast<void*>(tc2s_bf16_kernel<32, 3>)
                                       : reinterpret_cast<void*>(tc2s_bf16_kernel<32, 1>))
                          : (L.rb == 3 ? reinterpret_cast<void*>(tc2s_bf16_kernel<16, 3>)
                                       : reinterpret_cast<void*>(tc2s_bf16_kernel<16, 1>));
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.grid);
    cfg.blockDim = dim3(kThreads2s);
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
    return cudaLaunchKernel(kern, dim3(grid), dim3(kThreads2s), args, L.smem_bytes, stream);
}

}  // namespace cc3d
