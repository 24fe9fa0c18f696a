// Host-only parts of the library: error text, the greedy RoPE-block bit
// allocator and the Gaussian Lloyd-Max codebooks.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <limits>
#include <vector>

#include "../../include/kvq.h"

namespace {
thread_local char g_err[512] = "";
}

kvq_status kvq_set_error(kvq_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

kvq_status kvq_check_cuda(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return KVQ_OK;
    return kvq_set_error(KVQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

extern "C" const char* kvq_last_error(void) { return g_err; }

// ---------------------------------------------------------------------------
// Greedy allocation ("RoPE-Aware Bit Allocation for KV-Cache Quantization",
// prerequisites: greedy allocation and Theorem 1; method step (2)).  The
// marginal gain of one more bit on block i is (3/4) s_i 4^-b_i; the factor
// 3/4 is common to all blocks, so s_i 4^-b_i (an exact power-of-two scaling)
// is compared, ties going to the lowest index.
// ---------------------------------------------------------------------------
extern "C" kvq_status bgtq_allocate(const double* scores, int n_blocks, int b_min, int b_max, int64_t total_bits,
                                    int8_t* widths_out) {
    if (!scores || !widths_out || n_blocks <= 0)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_allocate: null pointer or n_blocks=%d", n_blocks);
    if (b_min < 1 || b_max > 8 || b_min > b_max)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_allocate: need 1 <= b_min=%d <= b_max=%d <= 8", b_min, b_max);
    if (total_bits < (int64_t)n_blocks * b_min)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_allocate: total_bits=%lld below n_blocks*b_min",
                             (long long)total_bits);
    for (int i = 0; i < n_blocks; ++i)
        if (!std::isfinite(scores[i]) || scores[i] < 0.0)
            return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_allocate: score %d is not finite and >= 0", i);
    std::vector<int> w(n_blocks, b_min);
    int64_t budget = total_bits - (int64_t)n_blocks * b_min;
    while (budget > 0) {
        int best = -1;
        double best_gain = 0.0;
        for (int i = 0; i < n_blocks; ++i) {
            if (w[i] >= b_max) continue;
            const double gain = std::ldexp(scores[i], -2 * w[i]);
            if (best < 0 || gain > best_gain) {
                best = i;
                best_gain = gain;
            }
        }
        if (best < 0) break;
        ++w[best];
        --budget;
    }
    for (int i = 0; i < n_blocks; ++i) widths_out[i] = (int8_t)w[i];
    return KVQ_OK;
}

// ---------------------------------------------------------------------------
// Lloyd-Max quantiser of N(0,1) with 2^b levels.  The optimum satisfies
// c_i = E[X | t_{i-1} < X < t_i] with t_i = (c_i + c_{i+1}) / 2.  A few
// Lloyd sweeps from the quantile midpoints give a starting point; Newton's
// method on F_i(c) = E[X | cell_i] - c_i (tridiagonal Jacobian) then
// converges quadratically.
// ---------------------------------------------------------------------------
namespace {

const double kInvSqrt2Pi = 0.39894228040143267794;

double pdf(double x) { return std::isinf(x) ? 0.0 : kInvSqrt2Pi * std::exp(-0.5 * x * x); }
double upper_tail(double x) { return 0.5 * std::erfc(x / std::sqrt(2.0)); }  // P(X > x)
double lower_tail(double x) { return 0.5 * std::erfc(-x / std::sqrt(2.0)); } // P(X < x)

// P(a < X < b), evaluated on the side where it is a difference of small tails
double cell_mass(double a, double b) {
    if (a >= 0) return upper_tail(a) - upper_tail(b);
    if (b <= 0) return lower_tail(b) - lower_tail(a);
    return 1.0 - lower_tail(a) - upper_tail(b);
}

void cells(const std::vector<double>& c, std::vector<double>& lo, std::vector<double>& hi) {
    const size_t n = c.size();
    lo.resize(n);
    hi.resize(n);
    for (size_t i = 0; i < n; ++i) {
        lo[i] = i == 0 ? -std::numeric_limits<double>::infinity() : 0.5 * (c[i - 1] + c[i]);
        hi[i] = i + 1 == n ? std::numeric_limits<double>::infinity() : 0.5 * (c[i] + c[i + 1]);
    }
}

// inverse standard normal CDF by bisection on erfc (start values only)
double probit(double p) {
    double a = -10, b = 10;
    for (int it = 0; it < 200; ++it) {
        const double m = 0.5 * (a + b);
        if (lower_tail(m) < p) a = m; else b = m;
    }
    return 0.5 * (a + b);
}

}  // namespace

extern "C" kvq_status bgtq_lloyd_max_codebook(int b, double* out) {
    if (b < 1 || b > 8 || !out)
        return kvq_set_error(KVQ_ERR_INVALID_ARG, "bgtq_lloyd_max_codebook: b=%d (1..8), out=%p", b, (void*)out);
    const int n = 1 << b;
    std::vector<double> c(n), lo, hi, mu(n), F(n), dl(n), dd(n), du(n);
    for (int i = 0; i < n; ++i) c[i] = probit((i + 0.5) / n);
    for (int it = 0; it < 300; ++it) {  // Lloyd sweeps
        cells(c, lo, hi);
        for (int i = 0; i < n; ++i) c[i] = (pdf(lo[i]) - pdf(hi[i])) / cell_mass(lo[i], hi[i]);
    }
    for (int it = 0; it < 100; ++it) {  // Newton
        cells(c, lo, hi);
        for (int i = 0; i < n; ++i) {
            const double m = cell_mass(lo[i], hi[i]);
            mu[i] = (pdf(lo[i]) - pdf(hi[i])) / m;
            F[i] = mu[i] - c[i];
            const double dmu_da = std::isinf(lo[i]) ? 0.0 : pdf(lo[i]) * (mu[i] - lo[i]) / m;
            const double dmu_db = std::isinf(hi[i]) ? 0.0 : pdf(hi[i]) * (hi[i] - mu[i]) / m;
            dl[i] = 0.5 * dmu_da;
            du[i] = 0.5 * dmu_db;
            dd[i] = 0.5 * dmu_da + 0.5 * dmu_db - 1.0;
        }
        // solve J delta = -F (Thomas algorithm)
        std::vector<double> cp(n), dp(n);
        cp[0] = du[0] / dd[0];
        dp[0] = -F[0] / dd[0];
        for (int i = 1; i < n; ++i) {
            const double den = dd[i] - dl[i] * cp[i - 1];
            cp[i] = du[i] / den;
            dp[i] = (-F[i] - dl[i] * dp[i - 1]) / den;
        }
        double step = 0.0;
        std::vector<double> delta(n);
        delta[n - 1] = dp[n - 1];
        for (int i = n - 2; i >= 0; --i) delta[i] = dp[i] - cp[i] * delta[i + 1];
        for (int i = 0; i < n; ++i) {
            c[i] += delta[i];
            step = std::fmax(step, std::fabs(delta[i]));
        }
        if (step < 1e-15) break;
    }
    for (int i = 0; i < n; ++i) out[i] = c[i];
    return KVQ_OK;
}

extern "C" size_t bgtq_tile_bytes(int total_bits, int v_bits) {
    if (total_bits < 64 || total_bits > 512 || v_bits < 1 || v_bits > 8) return 0;
    const size_t kb = 4 * ((2 * (size_t)total_bits + 31) / 32);
    const size_t vb = 16 * (size_t)v_bits;
    return 16 * (kb + 16 + vb + 2);
}
