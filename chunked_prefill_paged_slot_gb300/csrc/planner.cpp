// planner.cpp -- host-side dynamic chunk planner and latency-model fits
// (vllm-ascend design page "Dynamic Chunked Pipeline Parallel (CPP)": quadratic
// latency model f(l) = a l^2 + b l + c, target T = f(base) - f(0), chunk size
// from f(L + x) - f(L) = T, smoothing / page alignment / caps, and the
// two-variable model f(C, H) = a C (C + H) + b (C + H) + c for calibration).
#include <math.h>
#include <stdint.h>

#include <new>
#include <vector>

#include "../../include/cpsa.h"

namespace {

// Positive root of a x^2 + lin x - T = 0 written without the cancellation of
// (-lin + sqrt(lin^2 + 4aT)) / 2a at large lin.
double next_chunk_root(double a, double b, double T, double L, double base)
{
    if (a <= 0.0)
        return b > 0.0 ? T / b : base;
    const double lin = 2.0 * a * L + b;
    return 2.0 * T / (lin + sqrt(lin * lin + 4.0 * a * T));
}

// Solve the 3x3 normal equations (X^T X) c = X^T t by Gaussian elimination with
// partial pivoting, on column-scaled features for conditioning.
int least_squares3(const double *x0, const double *x1, const double *x2, const double *t, int n, double *coef)
{
    if (n < 3)
        return CPSA_ERR_BAD_SHAPE;
    const double *cols[3] = {x0, x1, x2};
    double scale[3];
    for (int j = 0; j < 3; ++j) {
        double m = 0.0;
        for (int i = 0; i < n; ++i)
            m = fmax(m, fabs(cols[j][i]));
        scale[j] = m > 0.0 ? m : 1.0;
    }
    double A[3][4] = {{0}};
    for (int i = 0; i < n; ++i) {
        double f[3] = {x0[i] / scale[0], x1[i] / scale[1], x2[i] / scale[2]};
        for (int r = 0; r < 3; ++r) {
            for (int c = 0; c < 3; ++c)
                A[r][c] += f[r] * f[c];
            A[r][3] += f[r] * t[i];
        }
    }
    for (int c = 0; c < 3; ++c) {
        int piv = c;
        for (int r = c + 1; r < 3; ++r)
            if (fabs(A[r][c]) > fabs(A[piv][c]))
                piv = r;
        if (fabs(A[piv][c]) < 1e-300)
            return CPSA_ERR_BAD_SHAPE;
        if (piv != c)
            for (int k = 0; k < 4; ++k) {
                double tmp = A[c][k];
                A[c][k] = A[piv][k];
                A[piv][k] = tmp;
            }
        for (int r = 0; r < 3; ++r) {
            if (r == c)
                continue;
            double f = A[r][c] / A[c][c];
            for (int k = c; k < 4; ++k)
                A[r][k] -= f * A[c][k];
        }
    }
    for (int j = 0; j < 3; ++j)
        coef[j] = A[j][3] / A[j][j] / scale[j];
    return CPSA_OK;
}

// Page alignment, minimum and caps of a solved chunk size (shared by the
// planner and the online controller).
int64_t postprocess_chunk(double x, int64_t L, int64_t remaining, double base, int page_size, int64_t min_chunk,
                          int64_t max_model_len, int64_t max_num_scheduled_tokens, double smooth_factor)
{
    const double xs = smooth_factor * x + (1.0 - smooth_factor) * base;
    int64_t units = (int64_t)floor(xs / (double)page_size * (1.0 + 1e-9));
    int64_t sz = units * page_size;
    if (sz < min_chunk)
        sz = min_chunk;
    if (max_model_len > 0 && sz > max_model_len - L)
        sz = max_model_len - L;
    if (max_num_scheduled_tokens > 0 && sz > max_num_scheduled_tokens)
        sz = max_num_scheduled_tokens;
    if (sz > remaining)
        sz = remaining;
    if (sz < 1)
        sz = 1;
    return sz;
}

// Positive root C of f(C, H) - f(0, H) = T under f(C, H) = a C (C + H) + b (C + H) + c,
// i.e. a C^2 + (aH + b) C - T = 0, in the same cancellation-free form.
double next_chunk_root_two_var(double a, double b, double T, double H, double base)
{
    if (a <= 0.0)
        return b > 0.0 ? T / b : base;
    const double lin = a * H + b;
    return 2.0 * T / (lin + sqrt(lin * lin + 4.0 * a * T));
}

}  // namespace

// Online chunk-size controller: the startup model until enough batches are
// recorded, then the two-variable model refitted over a sliding window.
struct cpsa_online {
    double a, b, c;             // current coefficients
    bool calibrated;            // two-variable model in use
    double base;
    int page_size;
    int64_t min_chunk, max_model_len, max_num_scheduled_tokens;
    double smooth_factor;
    int window, min_points;
    std::vector<double> x0, x1, x2, t;   // per recorded batch
};

extern "C" {

cpsa_online *cpp_online_create(double a, double b, double c, int64_t base_chunk_size, int page_size,
                               int64_t min_chunk, int64_t max_model_len, int64_t max_num_scheduled_tokens,
                               double smooth_factor, int window, int min_points)
{
    if (base_chunk_size <= 0 || page_size <= 0 || min_chunk < 1 || window < 3 || min_points < 3 ||
        min_points > window)
        return nullptr;
    cpsa_online *h = new (std::nothrow) cpsa_online();
    if (!h)
        return nullptr;
    h->a = a;
    h->b = b;
    h->c = c;
    h->calibrated = false;
    h->base = (double)base_chunk_size;
    h->page_size = page_size;
    h->min_chunk = min_chunk;
    h->max_model_len = max_model_len;
    h->max_num_scheduled_tokens = max_num_scheduled_tokens;
    h->smooth_factor = smooth_factor;
    h->window = window;
    h->min_points = min_points;
    return h;
}

void cpp_online_destroy(cpsa_online *h) { delete h; }

int cpp_online_next_chunk(const cpsa_online *h, int64_t history, int64_t remaining, int64_t *chunk)
{
    if (!h || !chunk || history < 0 || remaining < 1)
        return CPSA_ERR_BAD_SHAPE;
    const double base = h->base;
    const double T = h->a * base * base + h->b * base;   // f(base, 0) - f(0, 0), same for both models
    const double x = h->calibrated ? next_chunk_root_two_var(h->a, h->b, T, (double)history, base)
                                   : next_chunk_root(h->a, h->b, T, (double)history, base);
    *chunk = postprocess_chunk(x, history, remaining, base, h->page_size, h->min_chunk, h->max_model_len,
                               h->max_num_scheduled_tokens, h->smooth_factor);
    return CPSA_OK;
}

int cpp_online_record(cpsa_online *h, const int64_t *chunks, const int64_t *histories, int n_chunks,
                      double time_ms)
{
    if (!h || n_chunks < 1 || !chunks || !histories)
        return CPSA_ERR_BAD_SHAPE;
    double f0 = 0.0, f1 = 0.0;
    for (int i = 0; i < n_chunks; ++i) {
        const double C = (double)chunks[i], H = (double)histories[i];
        f0 += C * (C + H);
        f1 += C + H;
    }
    h->x0.push_back(f0);
    h->x1.push_back(f1);
    h->x2.push_back((double)n_chunks);
    h->t.push_back(time_ms);
    const int n = (int)h->t.size();
    if (n < h->min_points)
        return CPSA_OK;
    const int m = n < h->window ? n : h->window;
    const int o = n - m;
    double coef[3];
    if (least_squares3(h->x0.data() + o, h->x1.data() + o, h->x2.data() + o, h->t.data() + o, m, coef) == CPSA_OK) {
        h->a = coef[0];
        h->b = coef[1];
        h->c = coef[2];
        h->calibrated = true;
    }
    return CPSA_OK;
}

int cpp_online_model(const cpsa_online *h, double *coef, int *n_samples, int *calibrated)
{
    if (!h || !coef)
        return CPSA_ERR_NULL_ARG;
    coef[0] = h->a;
    coef[1] = h->b;
    coef[2] = h->c;
    if (n_samples)
        *n_samples = (int)h->t.size();
    if (calibrated)
        *calibrated = h->calibrated ? 1 : 0;
    return CPSA_OK;
}

int cpp_plan_chunk_sizes(double a, double b, double c, int64_t prompt_len, int64_t base_chunk_size, int page_size,
                         int64_t min_chunk, int64_t max_model_len, int64_t max_num_scheduled_tokens,
                         double smooth_factor, int64_t *chunks, int64_t max_chunks, int64_t *n_chunks)
{
    if (prompt_len < 0 || base_chunk_size <= 0 || page_size <= 0 || min_chunk < 1 || !n_chunks ||
        (max_chunks > 0 && !chunks))
        return CPSA_ERR_BAD_SHAPE;
    const double base = (double)base_chunk_size;
    const double T = (a * base * base + b * base + c) - c;   // f(base) - f(0)
    int64_t L = 0, n = 0;
    while (L < prompt_len) {
        const double x = next_chunk_root(a, b, T, (double)L, base);
        const int64_t sz = postprocess_chunk(x, L, prompt_len - L, base, page_size, min_chunk, max_model_len,
                                             max_num_scheduled_tokens, smooth_factor);
        if (n < max_chunks)
            chunks[n] = sz;
        ++n;
        L += sz;
    }
    *n_chunks = n;
    return n <= max_chunks ? CPSA_OK : CPSA_ERR_BAD_SHAPE;
}

int cpp_fit_latency_quadratic(const double *l, const double *t, int n, double *coef)
{
    if (!l || !t || !coef || n < 3)
        return CPSA_ERR_BAD_SHAPE;
    double *x0 = new double[n];
    double *x2 = new double[n];
    for (int i = 0; i < n; ++i) {
        x0[i] = l[i] * l[i];
        x2[i] = 1.0;
    }
    int st = least_squares3(x0, l, x2, t, n, coef);
    delete[] x0;
    delete[] x2;
    return st;
}

int cpp_fit_latency_two_var(const double *x0, const double *x1, const double *x2, const double *t, int n,
                            double *coef)
{
    if (!x0 || !x1 || !x2 || !t || !coef)
        return CPSA_ERR_BAD_SHAPE;
    return least_squares3(x0, x1, x2, t, n, coef);
}

}  // extern "C"
