// Format constants derived by the library itself, once per process, on the host:
//  - TBQ4 centroids and decision boundaries: 16-level Lloyd-Max quantizer of N(0, 1/128), and
//    turbo3's 8-level one by the same construction
//    (KV cache math, "How a 4-bit cache gets away with it": 16 Lloyd-Max centroids fitted
//    to N(0, 1/sqrt(128)), read as a standard deviation of 1/sqrt(128)), computed in fp64
//    by Lloyd iteration with closed-form Gaussian cell means and rounded to fp32;
//  - the two 128-entry sign vectors of the randomized Walsh-Hadamard transform, as the
//    first four outputs of splitmix64 (Steele, Lea & Flood 2014) from state 0x54425134.
#include <cmath>
#include <mutex>
#include "kvq_internal.h"

namespace kvq {
namespace {

uint64_t splitmix_next(uint64_t& state) {
    state += 0x9E3779B97F4A7C15ULL;
    uint64_t z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

double normal_pdf(double x) { return std::exp(-0.5 * x * x) / std::sqrt(2.0 * M_PI); }
double normal_upper(double x) { return 0.5 * std::erfc(x / std::sqrt(2.0)); }

// Positive half of the symmetric 16-level optimum for N(0,1), by 50,000 Lloyd steps
// from c_k = (k + 0.5) * 2.5 / 8. Cell k of the positive half is (b_k, b_{k+1}], with
// b_0 = 0, b_k = (c_{k-1} + c_k) / 2, b_8 = infinity; its mean is
// (pdf(b_k) - pdf(b_{k+1})) / (upper(b_k) - upper(b_{k+1})).
// The same with h = 4 half-levels gives turbo3's 8-level table.
void lloyd_half(double c[8], int h = 8) {
    for (int k = 0; k < h; ++k) c[k] = (k + 0.5) * 2.5 / h;
    for (int it = 0; it < 50000; ++it) {
        double b[9];
        b[0] = 0.0;
        for (int k = 1; k < h; ++k) b[k] = (c[k - 1] + c[k]) / 2.0;
        double nc[8];
        for (int k = 0; k < h; ++k) {
            const bool last = (k == h - 1);
            double num = normal_pdf(b[k]) - (last ? 0.0 : normal_pdf(b[k + 1]));
            double den = normal_upper(b[k]) - (last ? 0.0 : normal_upper(b[k + 1]));
            nc[k] = num / den;
        }
        for (int k = 0; k < h; ++k) c[k] = nc[k];
    }
}

FormatTables build() {
    FormatTables t{};
    double half[8];
    lloyd_half(half);
    double C[16];
    for (int j = 0; j < 8; ++j) {
        C[j] = -half[7 - j];
        C[8 + j] = half[j];
    }
    const double sigma = 1.0 / std::sqrt(128.0);
    for (int j = 0; j < 16; ++j) t.cent[j] = (float)(sigma * C[j]);
    for (int k = 1; k < 16; ++k) t.bnd[k - 1] = (float)(sigma * (C[k - 1] + C[k]) / 2.0);
    double h3[8];
    lloyd_half(h3, 4);
    double C3[8];
    for (int j = 0; j < 4; ++j) {
        C3[j] = -h3[3 - j];
        C3[4 + j] = h3[j];
    }
    for (int j = 0; j < 8; ++j) t.cent3[j] = (float)(sigma * C3[j]);
    for (int k = 1; k < 8; ++k) t.bnd3[k - 1] = (float)(sigma * (C3[k - 1] + C3[k]) / 2.0);
    uint64_t st = 0x54425134ULL;
    for (int i = 0; i < 4; ++i) t.sign_words[i] = splitmix_next(st);
    return t;
}

}  // namespace

const FormatTables& host_tables() {
    static FormatTables t;
    static std::once_flag once;
    std::call_once(once, [] { t = build(); });
    return t;
}

}  // namespace kvq
