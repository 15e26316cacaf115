/*
 * cc3d_oracle.c -- plain fp64 CPU oracle for the chunked causal 3-D convolution.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the package smoke check and the
 * CPU-baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA path.
 *
 * What it computes (sources are the pages this project is built from):
 *
 *   SwiftVR Inference Optimization (LightX2V blog), section "ReAE: Causal Halo
 *   Exchange": a causal layer concatenates the current frame's input features
 *   with those of the preceding frame(s) and convolves the stack; across a
 *   chunk boundary the only state needed is the *input* features of the
 *   previous chunk's last frame(s); a video's opening chunk starts from an
 *   all-zero history.  Section "From Pixels to Latents and Back": long videos are
 *   split into temporal chunks and the autoencoder keeps per-layer boundary
 *   features across chunks.
 *
 *   SGLang-Diffusion advanced optimizations, section 3 "Parallel VAE": VAE
 *   encode/decode is dominated by dense 3-D convolutions; splitting the work
 *   with a halo of boundary pixels keeps the result mathematically equal to
 *   the unsplit convolution.
 *
 *   The kernel shape (kt x kh x kw, stride 1), the spatial zero padding of
 *   (kh-1)/2, (kw-1)/2 and the causal zero left-padding of kt-1 frames are the
 *   plain reading of those passages for a "same"-size causal video conv, the
 *   form PyTorch's Conv3d computes (cross-correlation, no kernel flip).
 *
 * Definition (NDHWC, batch 1):
 *
 *   Y[t,h,w,co] = b[co]
 *               + sum_{dt<kt} sum_{dh<kh} sum_{dw<kw} sum_{ci<Cin}
 *                   Wt[co,dt,dh,dw,ci] * Xz[t+dt-(kt-1), h+dh-ph, w+dw-pw, ci]
 *               (+ R[t,h,w,co] when a residual is given)
 *   Xz[tau,i,j,c] = X[tau,i,j,c] inside the video, 0 outside it,
 *   ph = (kh-1)/2, pw = (kw-1)/2.
 *
 *   So the tap dt = kt-1 multiplies the current frame and dt = 0 the oldest
 *   one (the current frame is paired with its *previous* frames, never with a
 *   future frame).
 *
 * Chunked form: a chunk of Tc frames is processed with a cache holding the
 * kt-1 input frames that precede it (zeros before the first chunk).  The
 * oracle builds the extended stack concat(cache_in, x_chunk) physically,
 * convolves it without any temporal padding, and returns the last kt-1 frames
 * of that stack as the next cache.
 *
 * Everything is evaluated in double precision, one product and one add at a
 * time, in the loop order written below.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

static int valid_kernel(int kt, int kh, int kw)
{
    /* odd spatial extents so that "same" padding is symmetric; any kt >= 1 */
    return kt >= 1 && kh >= 1 && kw >= 1 && (kh % 2) == 1 && (kw % 2) == 1;
}

/* ------------------------------------------------------------------------ */
/* Work splitting: a tiny static thread pool over an index range.            */

typedef void (*range_fn)(void* ctx, long lo, long hi);

typedef struct {
    range_fn fn;
    void* ctx;
    long lo, hi;
} range_job;

static void* range_thread(void* p)
{
    range_job* j = (range_job*)p;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

static void run_range(range_fn fn, void* ctx, long n, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((long)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    if (nthreads == 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t th[256];
    int ok[256];
    range_job jobs[256];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].fn = fn;
        jobs[i].ctx = ctx;
        jobs[i].lo = n * i / nthreads;
        jobs[i].hi = n * (i + 1) / nthreads;
        ok[i] = pthread_create(&th[i], NULL, range_thread, &jobs[i]) == 0;
        if (!ok[i]) fn(ctx, jobs[i].lo, jobs[i].hi); /* no thread: do the slice here */
    }
    for (int i = 0; i < nthreads; ++i)
        if (ok[i]) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------------ */
/* Whole-sequence form.                                                       */

typedef struct {
    int T, H, W, Cin, Cout, kt, kh, kw;
    const double *x, *w, *b, *r;
    double* y;
} whole_ctx;

/* one output row (t, h): all w and co */
static void whole_rows(void* p, long lo, long hi)
{
    const whole_ctx* c = (const whole_ctx*)p;
    const int H = c->H, W = c->W, Cin = c->Cin, Cout = c->Cout;
    const int kt = c->kt, kh = c->kh, kw = c->kw;
    const int ph = (kh - 1) / 2, pw = (kw - 1) / 2;
    for (long row = lo; row < hi; ++row) {
        const int t = (int)(row / H), h = (int)(row % H);
        for (int w = 0; w < W; ++w) {
            for (int co = 0; co < Cout; ++co) {
                double acc = 0.0;
                for (int dt = 0; dt < kt; ++dt) {
                    const int ts = t + dt - (kt - 1);
                    if (ts < 0 || ts >= c->T) continue; /* Xz = 0 outside the video */
                    for (int dh = 0; dh < kh; ++dh) {
                        const int hs = h + dh - ph;
                        if (hs < 0 || hs >= H) continue;
                        for (int dw = 0; dw < kw; ++dw) {
                            const int ws = w + dw - pw;
                            if (ws < 0 || ws >= W) continue;
                            const double* xp = c->x + (((size_t)ts * H + hs) * W + ws) * Cin;
                            const double* wp =
                                c->w + ((((size_t)co * kt + dt) * kh + dh) * kw + dw) * Cin;
                            for (int ci = 0; ci < Cin; ++ci) acc += wp[ci] * xp[ci];
                        }
                    }
                }
                const size_t o = (((size_t)t * H + h) * W + w) * Cout + co;
                double v = acc;
                if (c->b) v += c->b[co];
                if (c->r) v += c->r[o];
                c->y[o] = v;
            }
        }
    }
}

/*
 * Y = causal conv of the whole sequence X[T][H][W][Cin].
 * w: [Cout][kt][kh][kw][Cin]; b: [Cout] or NULL; r: [T][H][W][Cout] or NULL.
 */
int cc3d_oracle_whole(int T, int H, int W, int Cin, int Cout, int kt, int kh, int kw,
                      const double* x, const double* w, const double* b, const double* r,
                      double* y, int nthreads)
{
    if (T < 0 || H < 1 || W < 1 || Cin < 1 || Cout < 1 || !valid_kernel(kt, kh, kw))
        return ORACLE_EINVAL;
    if (T == 0) return ORACLE_OK;
    if (!x || !w || !y) return ORACLE_EINVAL;
    whole_ctx c = {T, H, W, Cin, Cout, kt, kh, kw, x, w, b, r, y};
    run_range(whole_rows, &c, (long)T * H, nthreads);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Chunked form: physical concat(cache, chunk), conv without temporal pad.    */

typedef struct {
    int Tc, H, W, Cin, Cout, kt, kh, kw;
    const double* xe; /* [Tc + kt - 1][H][W][Cin] */
    const double *w, *b, *r;
    double* y;
} chunk_ctx;

static void chunk_rows(void* p, long lo, long hi)
{
    const chunk_ctx* c = (const chunk_ctx*)p;
    const int H = c->H, W = c->W, Cin = c->Cin, Cout = c->Cout;
    const int kt = c->kt, kh = c->kh, kw = c->kw;
    const int ph = (kh - 1) / 2, pw = (kw - 1) / 2;
    for (long row = lo; row < hi; ++row) {
        const int t = (int)(row / H), h = (int)(row % H);
        for (int w = 0; w < W; ++w) {
            for (int co = 0; co < Cout; ++co) {
                double acc = 0.0;
                for (int dt = 0; dt < kt; ++dt) {
                    /* frame t of the chunk sits at index t + kt - 1 of the stack,
                       so its tap dt reads stack frame t + dt */
                    const int te = t + dt;
                    for (int dh = 0; dh < kh; ++dh) {
                        const int hs = h + dh - ph;
                        if (hs < 0 || hs >= H) continue;
                        for (int dw = 0; dw < kw; ++dw) {
                            const int ws = w + dw - pw;
                            if (ws < 0 || ws >= W) continue;
                            const double* xp = c->xe + (((size_t)te * H + hs) * W + ws) * Cin;
                            const double* wp =
                                c->w + ((((size_t)co * kt + dt) * kh + dh) * kw + dw) * Cin;
                            for (int ci = 0; ci < Cin; ++ci) acc += wp[ci] * xp[ci];
                        }
                    }
                }
                const size_t o = (((size_t)t * H + h) * W + w) * Cout + co;
                double v = acc;
                if (c->b) v += c->b[co];
                if (c->r) v += c->r[o];
                c->y[o] = v;
            }
        }
    }
}

/*
 * One chunk of Tc frames.
 * cache_in: [kt-1][H][W][Cin], or NULL for zero history (first chunk).
 * cache_out: [kt-1][H][W][Cin] receives the last kt-1 frames of
 *            concat(cache_in, x_chunk) (may be NULL when kt == 1).
 */
int cc3d_oracle_chunk(int Tc, int H, int W, int Cin, int Cout, int kt, int kh, int kw,
                      const double* x_chunk, const double* w, const double* b, const double* r,
                      const double* cache_in, double* cache_out, double* y, int nthreads)
{
    if (Tc < 1 || H < 1 || W < 1 || Cin < 1 || Cout < 1 || !valid_kernel(kt, kh, kw))
        return ORACLE_EINVAL;
    if (!x_chunk || !w || !y) return ORACLE_EINVAL;
    const int P = kt - 1;
    const size_t frame = (size_t)H * W * Cin;
    double* xe = (double*)malloc(sizeof(double) * frame * (size_t)(Tc + P) + 1);
    if (!xe) return ORACLE_ENOMEM;
    /* the extended stack: history first, then the chunk */
    if (P > 0) {
        if (cache_in)
            memcpy(xe, cache_in, sizeof(double) * frame * P);
        else
            memset(xe, 0, sizeof(double) * frame * P); /* zero history */
    }
    memcpy(xe + frame * P, x_chunk, sizeof(double) * frame * Tc);

    chunk_ctx c = {Tc, H, W, Cin, Cout, kt, kh, kw, xe, w, b, r, y};
    run_range(chunk_rows, &c, (long)Tc * H, nthreads);

    /* the next chunk's history: the last P frames of the stack */
    if (P > 0 && cache_out) memcpy(cache_out, xe + frame * Tc, sizeof(double) * frame * P);
    free(xe);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Point form: Y at chosen output positions of the whole sequence.            */

typedef struct {
    int T, H, W, Cin, Cout, kt, kh, kw;
    const int* pts;
    const double *xwin, *w, *b, *rpts;
    double* ypts;
} pts_ctx;

static void pts_range(void* p, long lo, long hi)
{
    const pts_ctx* c = (const pts_ctx*)p;
    const int H = c->H, W = c->W, Cin = c->Cin, Cout = c->Cout;
    const int kt = c->kt, kh = c->kh, kw = c->kw;
    const int ph = (kh - 1) / 2, pw = (kw - 1) / 2;
    const size_t win = (size_t)kt * kh * kw * Cin;
    for (long i = lo; i < hi; ++i) {
        const int t = c->pts[3 * i], h = c->pts[3 * i + 1], w = c->pts[3 * i + 2];
        const double* xw = c->xwin + win * (size_t)i;
        for (int co = 0; co < Cout; ++co) {
            double acc = 0.0;
            for (int dt = 0; dt < kt; ++dt) {
                const int ts = t + dt - (kt - 1);
                if (ts < 0 || ts >= c->T) continue;
                for (int dh = 0; dh < kh; ++dh) {
                    const int hs = h + dh - ph;
                    if (hs < 0 || hs >= H) continue;
                    for (int dw = 0; dw < kw; ++dw) {
                        const int ws = w + dw - pw;
                        if (ws < 0 || ws >= W) continue;
                        const double* xp = xw + (((size_t)dt * kh + dh) * kw + dw) * Cin;
                        const double* wp =
                            c->w + ((((size_t)co * kt + dt) * kh + dh) * kw + dw) * Cin;
                        for (int ci = 0; ci < Cin; ++ci) acc += wp[ci] * xp[ci];
                    }
                }
            }
            double v = acc;
            if (c->b) v += c->b[co];
            if (c->rpts) v += c->rpts[(size_t)i * Cout + co];
            c->ypts[(size_t)i * Cout + co] = v;
        }
    }
}

/*
 * Y[t,h,w,:] of the whole-sequence definition at npts positions.
 * pts: [npts][3] = (t, h, w), 0 <= t < T, 0 <= h < H, 0 <= w < W.
 * xwin: [npts][kt][kh][kw][Cin]; entry (dt,dh,dw) holds X at
 *       (t+dt-(kt-1), h+dh-ph, w+dw-pw) when that position is inside the
 *       video; entries outside the video are ignored (taken as zero).
 * rpts: [npts][Cout] residual values at the points, or NULL.
 * ypts: [npts][Cout] output.
 */
int cc3d_oracle_points(int T, int H, int W, int Cin, int Cout, int kt, int kh, int kw, int npts,
                       const int* pts, const double* xwin, const double* w, const double* b,
                       const double* rpts, double* ypts, int nthreads)
{
    if (T < 1 || H < 1 || W < 1 || Cin < 1 || Cout < 1 || npts < 0 || !valid_kernel(kt, kh, kw))
        return ORACLE_EINVAL;
    if (npts == 0) return ORACLE_OK;
    if (!pts || !xwin || !w || !ypts) return ORACLE_EINVAL;
    for (int i = 0; i < npts; ++i) {
        const int t = pts[3 * i], h = pts[3 * i + 1], w = pts[3 * i + 2];
        if (t < 0 || t >= T || h < 0 || h >= H || w < 0 || w >= W) return ORACLE_EINVAL;
    }
    pts_ctx c = {T, H, W, Cin, Cout, kt, kh, kw, pts, xwin, w, b, rpts, ypts};
    run_range(pts_range, &c, npts, nthreads);
    return ORACLE_OK;
}

int cc3d_oracle_version(void) { return 1; }
