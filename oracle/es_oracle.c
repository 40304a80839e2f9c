/*
 * es_oracle.c -- plain CPU oracle for `element-scan` (TEST INFRASTRUCTURE).
 *
 * This file is test infrastructure, not part of the product.  Only the test
 * suite, the smoke check and the bench's CPU-baseline / reference arm may load
 * it.  It shares no code, header or constant with the CUDA library: it is the
 * independent statement of what the library must compute.
 *
 * Source of truth: "Nonlinear element scans" (sx.041.io/docs/element-scan.md).
 *   - intro: h[t] = f(h[t-1], x[t], ...) at every position outside one axis,
 *     from h[-1] = initial; every output position holds the state after its
 *     own trip.
 *   - TANH_DECAY: the page's first example, h = tanh(x + a*h).
 *   - NORMCAP: the `:state-axis` example, y = a*h + x, h = y / max(1, |y|)
 *     over the whole state vector, `a` a per-trip gate of width one.
 *   - MAXPLUS: the `:reverse true` example, the max-plus sweep
 *     h = maximum(h - c, x).
 *   - `:reverse true`: trips run from the last position of the axis to the
 *     first, from h[time] = initial (section intro, reverse paragraph).
 *   - "Arguments and body": initial is the sequence shape with the axis
 *     removed; with `:state-axis` every sequence has the same shape except its
 *     own last width, and a width-one sequence broadcasts over the state.
 *   - "Precision and gradients": the recurrence computes in f32.
 * Layout: C-contiguous row-major arrays ("lucid.tensor" page, contiguity and
 * reshape paragraphs).
 *
 * Readings taken where the pages are silent (each one is also listed in the
 * design notes):
 *   - every body operation is one f32 operation rounded to nearest, in the
 *     order the body is written; no fused multiply-add (build with
 *     -ffp-contract=off);
 *   - tanh of an f32 argument is the f32 rounding of the double tanh;
 *   - `sum` over the state adds w = 0, 1, ..., W-1 in order, in f32;
 *   - `maximum` is IEEE 754-2019 maximum: the larger value, +0 above -0, NaN
 *     if either operand is NaN;
 *   - with `:state-axis`, TANH_DECAY and MAXPLUS act element by element on
 *     the state (their bodies are pointwise), and NORMCAP requires a vector
 *     state (a scalar state's body cannot reduce).
 *
 * The oracle is deliberately a plain lane-by-lane, trip-by-trip loop: no
 * blocking, no threading, no reordering.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_TANH_DECAY 0
#define ORACLE_NORMCAP 1
#define ORACLE_MAXPLUS 2
#define ORACLE_MAX_STATE 16

/* IEEE 754-2019 maximum(a, b): larger value; +0 is above -0; NaN wins. */
static float oracle_maximum(float a, float b)
{
    if (a != a) return a;
    if (b != b) return b;
    if (a > b) return a;
    if (b > a) return b;
    /* equal values: only the sign of a zero can differ */
    return signbit(a) ? b : a;
}

/* tanh of an f32 value, rounded once to f32 */
static float oracle_tanh(float v)
{
    return (float)tanh((double)v);
}

/*
 * Run the scan.  Arguments mirror the library's entry point, with host
 * pointers:
 *   body        0 TANH_DECAY (seqs x, a), 1 NORMCAP (x, a), 2 MAXPLUS (x, c)
 *   initial     f32, the output shape with `axis` removed
 *   seqs        n_seqs f32 arrays (must be 2)
 *   shape/rank  the output shape (equal to the full-width sequence shape)
 *   axis        sequence axis, negative counts from the end
 *   state_width 0: scalar state; W in 1..16: vector state along the last axis
 *   seq_widths  NULL, or per sequence its own last width (1 or W)
 *   reverse     0 forward, 1 reverse
 *   out         f32 array of `shape`
 * Returns 0, or -1 for arguments the oracle cannot interpret.
 */
int es_oracle_f32(int body, const float *initial, const float *const *seqs,
                  int n_seqs, const int64_t *shape, int rank, int axis,
                  int state_width, const int64_t *seq_widths, int reverse,
                  float *out)
{
    if (n_seqs != 2 || rank < 1) return -1;
    if (axis < 0) axis += rank;
    if (axis < 0 || axis >= rank) return -1;
    if (state_width < 0 || state_width > ORACLE_MAX_STATE) return -1;
    if (state_width > 0 && (axis == rank - 1 || shape[rank - 1] != state_width))
        return -1;
    if (body == ORACLE_NORMCAP && state_width == 0) return -1;
    if (body != ORACLE_TANH_DECAY && body != ORACLE_NORMCAP && body != ORACLE_MAXPLUS)
        return -1;

    /* canonical view: [O, T, J, W] with J lanes after the axis */
    int64_t O = 1, T = shape[axis], after = 1;
    for (int d = 0; d < axis; d++) O *= shape[d];
    for (int d = axis + 1; d < rank; d++) after *= shape[d];
    int64_t W = state_width > 0 ? state_width : 1;
    int64_t J = after / W;

    /* each sequence's own width along the state axis (1 broadcasts) */
    int64_t sw[2];
    for (int k = 0; k < 2; k++) {
        sw[k] = W;
        if (state_width > 0 && seq_widths != NULL) sw[k] = seq_widths[k];
        if (sw[k] != 1 && sw[k] != W) return -1;
    }

    const float *x = seqs[0];
    const float *a = seqs[1];
    float h[ORACLE_MAX_STATE];
    float y[ORACLE_MAX_STATE];

    for (int64_t o = 0; o < O; o++) {
        for (int64_t j = 0; j < J; j++) {
            /* h[-1] (forward) or h[T] (reverse) = initial */
            for (int64_t w = 0; w < W; w++)
                h[w] = initial[(o * J + j) * W + w];

            for (int64_t s = 0; s < T; s++) {
                int64_t t = reverse ? T - 1 - s : s;
                /* element (o, t, j, w) of sequence k lives at
                   ((o*T + t)*J + j)*sw[k] + (sw[k] == 1 ? 0 : w) */
                const float *xt = x + ((o * T + t) * J + j) * sw[0];
                const float *at = a + ((o * T + t) * J + j) * sw[1];

                if (body == ORACLE_TANH_DECAY) {
                    /* h = tanh(x + a*h) */
                    for (int64_t w = 0; w < W; w++) {
                        float xv = xt[sw[0] == 1 ? 0 : w];
                        float av = at[sw[1] == 1 ? 0 : w];
                        float ah = av * h[w];
                        float v = xv + ah;
                        h[w] = oracle_tanh(v);
                    }
                } else if (body == ORACLE_MAXPLUS) {
                    /* h = maximum(h - c, x) */
                    for (int64_t w = 0; w < W; w++) {
                        float xv = xt[sw[0] == 1 ? 0 : w];
                        float cv = at[sw[1] == 1 ? 0 : w];
                        float v = h[w] - cv;
                        h[w] = oracle_maximum(v, xv);
                    }
                } else {
                    /* y = a*h + x;  h = y / maximum(1, sqrt(sum(y*y))) */
                    float ss = 0.0f;
                    for (int64_t w = 0; w < W; w++) {
                        float xv = xt[sw[0] == 1 ? 0 : w];
                        float av = at[sw[1] == 1 ? 0 : w];
                        float ah = av * h[w];
                        y[w] = ah + xv;
                    }
                    for (int64_t w = 0; w < W; w++) {
                        float sq = y[w] * y[w];
                        ss = ss + sq;
                    }
                    float d = oracle_maximum(1.0f, sqrtf(ss));
                    for (int64_t w = 0; w < W; w++)
                        h[w] = y[w] / d;
                }

                float *ot = out + ((o * T + t) * J + j) * W;
                for (int64_t w = 0; w < W; w++)
                    ot[w] = h[w];
            }
        }
    }
    return 0;
}

/* Same computation in double precision, for error diagnostics only. */
int es_oracle_f64(int body, const double *initial, const double *const *seqs,
                  int n_seqs, const int64_t *shape, int rank, int axis,
                  int state_width, const int64_t *seq_widths, int reverse,
                  double *out)
{
    if (n_seqs != 2 || rank < 1) return -1;
    if (axis < 0) axis += rank;
    if (axis < 0 || axis >= rank) return -1;
    if (state_width < 0 || state_width > ORACLE_MAX_STATE) return -1;
    if (state_width > 0 && (axis == rank - 1 || shape[rank - 1] != state_width))
        return -1;
    if (body == ORACLE_NORMCAP && state_width == 0) return -1;
    if (body != ORACLE_TANH_DECAY && body != ORACLE_NORMCAP && body != ORACLE_MAXPLUS)
        return -1;

    int64_t O = 1, T = shape[axis], after = 1;
    for (int d = 0; d < axis; d++) O *= shape[d];
    for (int d = axis + 1; d < rank; d++) after *= shape[d];
    int64_t W = state_width > 0 ? state_width : 1;
    int64_t J = after / W;
    int64_t sw[2];
    for (int k = 0; k < 2; k++) {
        sw[k] = W;
        if (state_width > 0 && seq_widths != NULL) sw[k] = seq_widths[k];
        if (sw[k] != 1 && sw[k] != W) return -1;
    }

    const double *x = seqs[0];
    const double *a = seqs[1];
    double h[ORACLE_MAX_STATE];
    double y[ORACLE_MAX_STATE];

    for (int64_t o = 0; o < O; o++) {
        for (int64_t j = 0; j < J; j++) {
            for (int64_t w = 0; w < W; w++)
                h[w] = initial[(o * J + j) * W + w];
            for (int64_t s = 0; s < T; s++) {
                int64_t t = reverse ? T - 1 - s : s;
                const double *xt = x + ((o * T + t) * J + j) * sw[0];
                const double *at = a + ((o * T + t) * J + j) * sw[1];
                if (body == ORACLE_TANH_DECAY) {
                    for (int64_t w = 0; w < W; w++)
                        h[w] = tanh(xt[sw[0] == 1 ? 0 : w] + at[sw[1] == 1 ? 0 : w] * h[w]);
                } else if (body == ORACLE_MAXPLUS) {
                    for (int64_t w = 0; w < W; w++) {
                        double v = h[w] - at[sw[1] == 1 ? 0 : w];
                        double xv = xt[sw[0] == 1 ? 0 : w];
                        h[w] = v > xv ? v : xv;
                    }
                } else {
                    double ss = 0.0;
                    for (int64_t w = 0; w < W; w++) {
                        y[w] = at[sw[1] == 1 ? 0 : w] * h[w] + xt[sw[0] == 1 ? 0 : w];
                        ss += y[w] * y[w];
                    }
                    double n = sqrt(ss);
                    double d = n > 1.0 ? n : 1.0;
                    for (int64_t w = 0; w < W; w++)
                        h[w] = y[w] / d;
                }
                double *ot = out + ((o * T + t) * J + j) * W;
                for (int64_t w = 0; w < W; w++)
                    ot[w] = h[w];
            }
        }
    }
    return 0;
}

/*
 * Backward pass ("Nonlinear element scans", "Precision and gradients"):
 * gradients flow to `initial` and to every sequence; the gradient of a scan
 * is another scan that runs the trips in the opposite order and applies the
 * body's vector-Jacobian product once a trip.  The forward states are given
 * (`states`, the forward output); `grad_out` is dL/d(states).
 *
 * In scan order s = 0..T-1 (trip t(s) = reverse ? T-1-s : s) the state before
 * trip s is initial for s = 0, else states[t(s-1)].  The cotangent lam of the
 * state starts at zero; for s = T-1 down to 0: lam += grad_out[t(s)], then
 * the body's VJP at trip s gives (lam_prev, dx[t], da[t]), and lam = lam_prev.
 * At the end grad_initial = lam.
 *
 * Per body, with h the trip's output and p the state before it:
 *   TANH_DECAY  mu = lam * (1 - h*h);  dx = mu;  da = mu * p;  lam_prev = mu * a
 *   MAXPLUS     v = p - c: v > x routes lam to the state (lam_prev = lam,
 *               dc = -lam), x > v routes it to x (dx = lam); a tie splits it
 *               evenly (the usual tie rule for maximum)
 *   NORMCAP     y = a*p + x recomputed, n = sqrt(sum y*y); if n <= 1,
 *               mu = lam, else mu = (lam - h * (h . lam)) / n; dx = mu;
 *               da = mu * p (summed over the state for a width-one gate);
 *               lam_prev = a * mu
 * A width-one sequence receives the sum over the state of its gradients.
 * Readings: the MAXPLUS tie rule (even split) and the NORMCAP branch at
 * n == 1 (the unscaled side) are not fixed by the pages.
 */
int es_oracle_backward_f32(int body, const float *initial, const float *const *seqs, int n_seqs,
                           const int64_t *shape, int rank, int axis, int state_width,
                           const int64_t *seq_widths, int reverse, const float *states,
                           const float *grad_out, float *grad_initial, float *const *grad_seqs)
{
    if (n_seqs != 2 || rank < 1) return -1;
    if (axis < 0) axis += rank;
    if (axis < 0 || axis >= rank) return -1;
    if (state_width < 0 || state_width > ORACLE_MAX_STATE) return -1;
    if (state_width > 0 && (axis == rank - 1 || shape[rank - 1] != state_width))
        return -1;
    if (body == ORACLE_NORMCAP && state_width == 0) return -1;
    if (body != ORACLE_TANH_DECAY && body != ORACLE_NORMCAP && body != ORACLE_MAXPLUS)
        return -1;

    int64_t O = 1, T = shape[axis], after = 1;
    for (int d = 0; d < axis; d++) O *= shape[d];
    for (int d = axis + 1; d < rank; d++) after *= shape[d];
    int64_t W = state_width > 0 ? state_width : 1;
    int64_t J = after / W;
    int64_t sw[2];
    for (int k = 0; k < 2; k++) {
        sw[k] = W;
        if (state_width > 0 && seq_widths != NULL) sw[k] = seq_widths[k];
        if (sw[k] != 1 && sw[k] != W) return -1;
    }

    const float *x = seqs[0];
    const float *a = seqs[1];
    float *gx = grad_seqs[0];
    float *ga = grad_seqs[1];
    float lam[ORACLE_MAX_STATE], p[ORACLE_MAX_STATE], mu[ORACLE_MAX_STATE], y[ORACLE_MAX_STATE];
    float dx[ORACLE_MAX_STATE], da[ORACLE_MAX_STATE];

    for (int64_t o = 0; o < O; o++) {
        for (int64_t j = 0; j < J; j++) {
            for (int64_t w = 0; w < W; w++) lam[w] = 0.0f;

            /* scan order backwards: s = T-1 .. 0 */
            for (int64_t s = T - 1; s >= 0; s--) {
                int64_t t = reverse ? T - 1 - s : s;
                const float *ht = states + ((o * T + t) * J + j) * W;
                const float *gt = grad_out + ((o * T + t) * J + j) * W;
                /* the state before this trip */
                if (s == 0) {
                    for (int64_t w = 0; w < W; w++) p[w] = initial[(o * J + j) * W + w];
                } else {
                    int64_t tp = reverse ? t + 1 : t - 1;
                    const float *hp = states + ((o * T + tp) * J + j) * W;
                    for (int64_t w = 0; w < W; w++) p[w] = hp[w];
                }
                for (int64_t w = 0; w < W; w++) lam[w] = lam[w] + gt[w];
                const float *xt = x + ((o * T + t) * J + j) * sw[0];
                const float *at = a + ((o * T + t) * J + j) * sw[1];

                if (body == ORACLE_TANH_DECAY) {
                    /* h = tanh(v), v = x + a*p:  dh/dv = 1 - h*h */
                    for (int64_t w = 0; w < W; w++) {
                        float av = at[sw[1] == 1 ? 0 : w];
                        float hh = ht[w] * ht[w];
                        float om = 1.0f - hh;
                        float m = lam[w] * om;
                        dx[w] = m;
                        da[w] = m * p[w];
                        lam[w] = m * av;
                    }
                } else if (body == ORACLE_MAXPLUS) {
                    /* h = maximum(p - c, x): the larger operand takes the
                       cotangent, a tie splits it evenly */
                    for (int64_t w = 0; w < W; w++) {
                        float v = p[w] - at[sw[1] == 1 ? 0 : w];
                        float xv = xt[sw[0] == 1 ? 0 : w];
                        if (v > xv) {
                            dx[w] = 0.0f;
                            da[w] = -lam[w];
                        } else if (xv > v) {
                            dx[w] = lam[w];
                            da[w] = 0.0f;
                            lam[w] = 0.0f;
                        } else {
                            float half = lam[w] * 0.5f;
                            dx[w] = half;
                            da[w] = -half;
                            lam[w] = half;
                        }
                    }
                } else {
                    /* y = a*p + x recomputed; h = y / max(1, |y|) */
                    float ss = 0.0f;
                    for (int64_t w = 0; w < W; w++) {
                        float ap = at[sw[1] == 1 ? 0 : w] * p[w];
                        y[w] = ap + xt[sw[0] == 1 ? 0 : w];
                    }
                    for (int64_t w = 0; w < W; w++) {
                        float sq = y[w] * y[w];
                        ss = ss + sq;
                    }
                    float nrm = sqrtf(ss);
                    if (nrm <= 1.0f) {
                        /* inside the unit ball h = y */
                        for (int64_t w = 0; w < W; w++) mu[w] = lam[w];
                    } else {
                        /* h = y/n: d h = (I - h h^T) d y / n */
                        float hl = 0.0f;
                        for (int64_t w = 0; w < W; w++) {
                            float q = ht[w] * lam[w];
                            hl = hl + q;
                        }
                        for (int64_t w = 0; w < W; w++) {
                            float r = ht[w] * hl;
                            float dlt = lam[w] - r;
                            mu[w] = dlt / nrm;
                        }
                    }
                    for (int64_t w = 0; w < W; w++) {
                        dx[w] = mu[w];
                        da[w] = mu[w] * p[w];
                        lam[w] = at[sw[1] == 1 ? 0 : w] * mu[w];
                    }
                }

                /* a width-one sequence gets the sum over the state, in order */
                float *gxt = gx + ((o * T + t) * J + j) * sw[0];
                float *gat = ga + ((o * T + t) * J + j) * sw[1];
                if (sw[0] == 1 && W > 1) {
                    float acc = 0.0f;
                    for (int64_t w = 0; w < W; w++) acc = acc + dx[w];
                    gxt[0] = acc;
                } else {
                    for (int64_t w = 0; w < W; w++) gxt[w] = dx[w];
                }
                if (sw[1] == 1 && W > 1) {
                    float acc = 0.0f;
                    for (int64_t w = 0; w < W; w++) acc = acc + da[w];
                    gat[0] = acc;
                } else {
                    for (int64_t w = 0; w < W; w++) gat[w] = da[w];
                }
            }
            for (int64_t w = 0; w < W; w++) grad_initial[(o * J + j) * W + w] = lam[w];
        }
    }
    return 0;
}
