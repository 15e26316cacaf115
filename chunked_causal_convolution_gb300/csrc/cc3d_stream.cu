// cc3d_stream.cu -- causal convolutions with a 1x1 spatial kernel (kt x 1 x 1: TemporalGrow,
// pointwise projections) as a streaming kernel.
//
// Without spatial taps these layers do little arithmetic per byte (2 * kt * Cin * Cout FLOP
// against about 2 * (Cin + Cout) bytes per output position), so HBM bandwidth bounds them and
// the tile machinery of the 3x3x3 kernels (windows per tap, weights streamed per tile) only adds
// traffic and per-stage work.  Here:
//
//   * a frame is a [H*W][Cin] matrix; a unit of work is one 128-position block of it (the MMA's
//     M) for one group of up to G output frames;
//   * the weights of every temporal tap stay in shared memory for the whole kernel;
//   * each input frame of the unit (the P = kt-1 history frames, then the chunk's) is staged once,
//     all channels, and multiplied into the accumulators of every output frame it is a tap of:
//     D[t_out] += X[t_out + dt - P] * W[dt]^T, dt = 0 .. kt-1;
//   * tensor memory holds one Cout-column accumulator per output frame of the unit; a frame's
//     accumulator is complete after its last tap (the input frame t_out itself), so the epilogue
//     drains frame 0 while the MMAs still run on later frames, and the next unit's frame 0 only
//     needs frame 0's columns back;
//   * two MMA warps take the output frames of a unit by parity (each accumulator has one writer),
//     so that one warp's issue stalls are covered by the other's MMAs, and two sets of four
//     epilogue warps drain them by the same parity;
//   * the new history (the last P input frames) is stored from the staged blocks by the copy
//     engine.
//
// Accumulation order of every output: dt, channel block, 16-channel step (in the tensor core),
// then bias, then residual -- independent of the chunking.
#include <cuda_bf16.h>

#include "cc3d_internal.h"
#include "cc3d_ptx.cuh"
#include "cc3d_tc_common.cuh"

namespace cc3d {
using namespace ptx;
using namespace tcc;

namespace {

constexpr int kSCB = 32;          // channels per staged block: 64-byte rows, 64-byte swizzle
constexpr int kSPos = 128;        // positions per unit (the MMA's M)
constexpr int kSMaxStages = 8;    // input-frame stages
constexpr int kSMaxFrames = 8;    // output frames per unit (tensor-memory slots)
// warps: 0 loader, 1-2 MMA, 3 history stores, 4-7 and 8-11 the two epilogue sets (warp w reads
// tensor-memory lanes 32 * (w % 4) ..)
constexpr int kSThreads = 384;

struct SUnit {
    int t0, G;   // output frames [t0, t0 + G)
    int p0;      // first position of the block in the flattened frame
};

__device__ __forceinline__ SUnit s_unit(const StreamLaunch& L, long long u)
{
    SUnit s;
    const int pb = (int)(u % L.npb);
    const int fg = (int)(u / L.npb);
    s.t0 = fg * L.gmax;
    s.G = min(L.gmax, L.T - s.t0);
    s.p0 = pb * kSPos;
    return s;
}

__device__ __forceinline__ void s_fail(const StreamLaunch& L, unsigned bit, volatile int* abort_flag)
{
    *abort_flag = 1;
    atomicOr(L.status, bit);
}

__global__ void __launch_bounds__(kSThreads, 1) stream_bf16_kernel(const __grid_constant__ StreamLaunch L)
{
    constexpr uint32_t ROWB = kSCB * 2;
    constexpr uint32_t SBO = 8 * ROWB;
    constexpr int KSTEPS = kSCB / 16;

    extern __shared__ uint8_t dsm_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsm_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* smW = sm;                          // [dt][channel block] tiles of Cout rows x 64 B
    uint8_t* smX = sm + (size_t)L.w_bytes;      // stages of [channel block][128 positions] x 64 B
    float* s_bias = reinterpret_cast<float*>(smX + (size_t)L.nstages * L.x_stage_bytes);

    __shared__ uint64_t x_full[kSMaxStages], x_empty[kSMaxStages], w_full, acc_full[kSMaxFrames],
        acc_empty[kSMaxFrames], mma_drain[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int ncb = L.Cin / kSCB;
    const int nst = L.nstages;
    const int P = L.kt - 1;
    const int Cout = L.Cout;
    const unsigned long long budget = L.wait_ns;
    const long long ubeg = L.units * blockIdx.x / gridDim.x;
    const long long uend = L.units * (blockIdx.x + 1) / gridDim.x;

    if (threadIdx.x == 0) {
        abort_flag = 0;
        // a stage is released by both MMA warps and, when there is a history to write, the copy warp
        for (int s = 0; s < nst; ++s) { mbar_init(&x_full[s], 1); mbar_init(&x_empty[s], P > 0 ? 3 : 2); }
        mbar_init(&w_full, 1);
        for (int f = 0; f < L.gmax; ++f) { mbar_init(&acc_full[f], 1); mbar_init(&acc_empty[f], 4); }
        mbar_init(&mma_drain[0], 1);
        mbar_init(&mma_drain[1], 1);
        fence_mbar_init();
    }
    if (warp >= 4) {
        const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(L.bias);
        for (int i = threadIdx.x - 128; i < Cout; i += kSThreads - 128)
            s_bias[i] = b != nullptr ? __bfloat162float(b[i]) : 0.0f;
    }
    if (warp == 2) {
        tmem_alloc(&tmem_base_sh, (uint32_t)L.tmem_cols);
        tmem_relinquish();
    }
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
            // all weights once: per (dt, channel block) a box of [Cout][32 channels]
            mbar_arrive_expect_tx(&w_full, (uint32_t)(L.kt * ncb * Cout * ROWB));
            for (int dt = 0; dt < L.kt; ++dt)
                for (int cb = 0; cb < ncb; ++cb)
                    tma_load_3d(smW + (size_t)(dt * ncb + cb) * Cout * ROWB, &L.map_w, &w_full, cb * kSCB, 0, dt);
            int s = 0, ph = 0;
            int last_ph[kSMaxStages];
            for (int k = 0; k < kSMaxStages; ++k) last_ph[k] = -1;
            const uint32_t x_tx = (uint32_t)(ncb * kSPos * ROWB);
            bool skip_first = (L.fault == 1);
            bool ok = true;
            for (long long u = ubeg; ok && u < uend; ++u) {
                const SUnit g = s_unit(L, u);
                for (int j = 0; j < g.G + P; ++j) {
                    const int tin = g.t0 - P + j;
                    if (!bounded_wait(&x_empty[s], ph ^ 1, budget, &abort_flag)) {
                        if (!abort_flag) s_fail(L, STATUS_TIMEOUT_LOADER, &abort_flag);
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&x_full[s], x_tx);
                    // history frames come from the cache (or the zero fill of an out-of-range frame)
                    const CUtensorMap* map = &L.map_x;
                    int tc = tin;
                    if (tin < 0 && L.has_cache) { map = &L.map_cache; tc = tin + P; }
                    if (!skip_first)
                        for (int cb = 0; cb < ncb; ++cb)
                            tma_load_3d(smX + (size_t)s * L.x_stage_bytes + (size_t)cb * kSPos * ROWB, map, &x_full[s],
                                        cb * kSCB, g.p0, tc);
                    skip_first = false;
                    last_ph[s] = ph;
                    if (++s == nst) { s = 0; ph ^= 1; }
                }
            }
            // never leave while a copy into this block's shared memory may still be in flight
            for (int k = 0; k < nst; ++k)
                if (last_ph[k] >= 0 && !bounded_wait(&x_full[k], (uint32_t)last_ph[k], budget, nullptr))
                    atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
            if (!bounded_wait(&w_full, 0, budget, nullptr)) atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------ MMA warps
        // warp 1 owns the unit's even output frames, warp 2 the odd ones; lane 0 of each polls the
        // barriers and issues its MMAs and commits
        const int k = warp - 1;
        const bool lead = lane == 0;
        const uint32_t idesc = make_idesc_bf16_f32(128, Cout);
        const uint64_t x_desc0 = make_sdesc(smem_u32(smX), 16, SBO, LAYOUT_SW64, 0);
        const uint64_t w_desc0 = make_sdesc(smem_u32(smW), 16, SBO, LAYOUT_SW64, 0);
        const uint32_t x_inc = (uint32_t)L.x_stage_bytes >> 4;
        const uint32_t cb_inc = (uint32_t)(kSPos * ROWB) >> 4;
        const uint32_t w_inc = (uint32_t)(Cout * ROWB) >> 4;
        bool ok = warp_bounded_wait(&w_full, 0, budget, &abort_flag);
        if (!ok && lane == 0 && !abort_flag) s_fail(L, STATUS_TIMEOUT_MMA, &abort_flag);
        tc_fence_after();
        int s = 0, ph = 0;
        uint32_t slot_phase = 0;  // bit f: parity of the uses of output-frame slot f so far
        for (long long u = ubeg; ok && u < uend; ++u) {
            const SUnit g = s_unit(L, u);
            for (int j = 0; ok && j < g.G + P; ++j) {
                if (!warp_bounded_wait(&x_full[s], ph, budget, &abort_flag)) {
                    if (lane == 0 && !abort_flag) s_fail(L, STATUS_TIMEOUT_MMA, &abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t xs = desc_add(x_desc0, s * x_inc);
                bool any = false;
                for (int dt = 0; dt < L.kt; ++dt) {
                    const int tout = j - dt;  // input frame t0 - P + j is tap dt of output frame t0 + tout
                    if (tout < 0 || tout >= g.G || (tout & 1) != k) continue;
                    any = true;
                    if (dt == 0) {
                        // first tap of this frame: its slot must have been drained by the epilogue
                        const uint32_t par = ((slot_phase >> tout) & 1u) ^ 1u;
                        if (!warp_bounded_wait(&acc_empty[tout], par, budget, &abort_flag)) {
                            if (lane == 0 && !abort_flag) s_fail(L, STATUS_TIMEOUT_MMA, &abort_flag);
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    const uint32_t d = tmem + (uint32_t)(tout * Cout);
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
                    if (dt == L.kt - 1) {
                        // last tap of this frame: its accumulator is complete once these MMAs finish
                        if (lead) umma_commit(&acc_full[tout]);
                        slot_phase ^= 1u << tout;
                    }
                }
                if (!ok) break;
                // a warp that read nothing from this stage releases it at once
                if (lead) {
                    if (any) umma_commit(&x_empty[s]);
                    else mbar_arrive(&x_empty[s]);
                }
                __syncwarp();
                if (++s == nst) { s = 0; ph ^= 1; }
            }
        }
        if (lead) umma_commit(&mma_drain[k]);
        __syncwarp();
        if (!warp_bounded_wait(&mma_drain[k], 0, budget, nullptr) && lane == 0) atomicOr(L.status, STATUS_TIMEOUT_DRAIN);
    } else if (warp == 3) {
        // ------------------------------------------------------------ temporal cache update
        // cache_out[k] is input frame T - P + k, which the last frame group stages as j = G + k:
        // TMA stores write those blocks straight from shared memory
        if (P > 0) {
            int s = 0, ph = 0;
            bool ok = true;
            for (long long u = ubeg; ok && u < uend; ++u) {
                const SUnit g = s_unit(L, u);
                const bool last_group = g.t0 + g.G == L.T;
                for (int j = 0; j < g.G + P; ++j) {
                    if (!warp_bounded_wait(&x_full[s], ph, budget, &abort_flag)) {
                        if (lane == 0 && !abort_flag) s_fail(L, STATUS_TIMEOUT_COPY, &abort_flag);
                        ok = false;
                        break;
                    }
                    if (lane == 0 && last_group && j >= g.G) {
                        const uint8_t* stage = smX + (size_t)s * L.x_stage_bytes;
                        fence_proxy_async_smem();
                        for (int cb = 0; cb < ncb; ++cb)
                            tma_store_3d(&L.map_cache_out, stage + (size_t)cb * kSPos * ROWB, cb * kSCB, g.p0, j - g.G);
                        bulk_commit_group();
                        bulk_wait_group_read<0>();  // the stage may be refilled once the store has read it
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&x_empty[s]);
                    if (++s == nst) { s = 0; ph ^= 1; }
                }
            }
            if (lane == 0) bulk_wait_group<0>();  // every store has landed before the block exits
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = (warp - 4) % 4;  // tensor-memory lanes 32q .. 32q+31 = positions p0 + 32q + lane
        const int set = (warp - 4) / 4;  // this set drains the output frames of its parity
        const __nv_bfloat16* res = reinterpret_cast<const __nv_bfloat16*>(L.res);
        __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(L.y);
        const bool wide = (Cout % 16) == 0;
        const long long HW = (long long)L.H * L.W;
        uint32_t slot_phase = 0;
        bool ok = true;
        for (long long u = ubeg; ok && u < uend; ++u) {
            const SUnit g = s_unit(L, u);
            const long long p = (long long)g.p0 + q * 32 + lane;
            const bool pvalid = p < HW;
            for (int tout = set; tout < g.G; tout += 2) {
                int ready = 0;
                if (lane == 0) {
                    ready = bounded_wait(&acc_full[tout], (slot_phase >> tout) & 1u, budget, &abort_flag,
                                         kEpilogueSleepNs);
                    if (!ready && !abort_flag) s_fail(L, STATUS_TIMEOUT_EPILOGUE, &abort_flag);
                }
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (!ready) { ok = false; break; }
                slot_phase ^= 1u << tout;
                tc_fence_after();
                const size_t px = pvalid ? (size_t)(g.t0 + tout) * (size_t)HW + (size_t)p : 0;
                const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(tout * Cout);
                epilogue_slice(tbase, Cout, 0, px, pvalid, true, s_bias, Cout, wide, res, y, L.v32 != 0,
                               [&]() { release_acc(&acc_empty[tout], lane); });
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) tmem_dealloc(tmem, (uint32_t)L.tmem_cols);
}

int cdiv(int a, int b) { return (a + b - 1) / b; }

}  // namespace

bool stream_configure(int T, int H, int W, int Cin, int Cout, int kt, int sms, StreamLaunch* L)
{
    if (T < 1 || H < 1 || W < 1 || sms < 1 || kt < 1 || kt > 3) return false;
    if (Cin % kSCB != 0 || Cout % 16 != 0 || Cout < 16 || Cout > 256) return false;
    const long long HW = (long long)H * W;
    if (HW > (1LL << 30)) return false;
    const int ncb = Cin / kSCB;
    L->T = T;
    L->H = H;
    L->W = W;
    L->Cin = Cin;
    L->Cout = Cout;
    L->kt = kt;
    int gmax = 512 / Cout;
    if (gmax > kSMaxFrames) gmax = kSMaxFrames;
    L->gmax = gmax;
    L->npb = (int)((HW + kSPos - 1) / kSPos);
    L->units = (long long)cdiv(T, gmax) * L->npb;
    L->w_bytes = (kt * ncb * Cout * kSCB * 2 + 1023) & ~1023;
    L->x_stage_bytes = ncb * kSPos * kSCB * 2;  // a multiple of 8 KB
    const int fixed = L->w_bytes + 4 * 256 + 1024;  // weights, bias, alignment slack
    int nst = (227 * 1024 - fixed) / L->x_stage_bytes;
    if (nst > kSMaxStages) nst = kSMaxStages;
    if (nst < 2) return false;
    L->nstages = nst;
    L->smem_bytes = (size_t)fixed + (size_t)nst * L->x_stage_bytes;
    if (L->smem_bytes < 120 * 1024) L->smem_bytes = 120 * 1024;  // one block per SM: it owns all tensor memory
    int cols = 32;
    while (cols < gmax * Cout) cols *= 2;
    L->tmem_cols = cols;
    L->grid = L->units < sms ? (int)L->units : sms;
    return true;
}

cudaError_t stream_launch(const StreamLaunch& L, cudaStream_t stream)
{
    void* kern = reinterpret_cast<void*>(stream_bf16_kernel);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem_bytes);
    if (e != cudaSuccess) return e;
    void* args[] = {const_cast<StreamLaunch*>(&L)};
    return cudaLaunchKernel(kern, dim3(L.grid), dim3(kSThreads), args, L.smem_bytes, stream);
}

}  // namespace cc3d
