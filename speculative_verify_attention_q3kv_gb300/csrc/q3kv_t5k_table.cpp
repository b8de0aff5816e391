// The turbo5k K codebook: the 32-level Lloyd-Max quantizer of N(0, 1).
//
// Source: "Quasar" (q27 wiki), turbo5k bullet of the stack list (32 Lloyd-Max
// centroids over the WHT rotation).  Lloyd-Max: every centroid is the mean of
// the normal over its cell, every boundary the midpoint of its two centroids.
// Found by Max's shooting method in double precision: the quantizer is
// symmetric, so the positive half is fixed by its first centroid y0 (the cell
// (0, t1) whose mean is y0 gives t1, the next centroid is 2 t1 - y0, and so on
// outward); bisection on y0 until the outermost centroid equals the mean of
// its unbounded cell.  The centroids are then rounded to float32 and the
// boundaries taken as float32 midpoints.
#include <cmath>

#include "q3kv_internal.h"

namespace q3kv {
namespace {

double upper_tail(double x) { return 0.5 * std::erfc(x / std::sqrt(2.0)); }
double pdf(double x) { return std::exp(-0.5 * x * x) / std::sqrt(2.0 * 3.141592653589793); }

// E[X | a < X < b], X ~ N(0, 1), 0 <= a < b <= inf
double cell_mean(double a, double b) {
    if (std::isinf(b)) return pdf(a) / upper_tail(a);
    return (pdf(a) - pdf(b)) / (upper_tail(a) - upper_tail(b));
}

// Positive half from y0 into ys[16]; returns how far the last centroid lies
// above the mean of its cell (+inf when a cell cannot reach its centroid).
double shoot(double y0, double* ys) {
    double t = 0.0;
    ys[0] = y0;
    for (int k = 0; k < 15; ++k) {
        const double y = ys[k];
        if (cell_mean(t, INFINITY) <= y) return INFINITY;
        double lo = t, hi = t + 1.0;
        while (cell_mean(t, hi) < y) hi = t + 2.0 * (hi - t);
        for (int it = 0; it < 200; ++it) {
            const double mid = 0.5 * (lo + hi);
            if (mid <= lo || mid >= hi) break;
            if (cell_mean(t, mid) < y) lo = mid;
            else hi = mid;
        }
        const double tn = 0.5 * (lo + hi);
        ys[k + 1] = 2.0 * tn - y;
        t = tn;
    }
    return ys[15] - cell_mean(t, INFINITY);
}

T5kTable build_table() {
    double ys[16];
    double lo = 1e-3, hi = 0.5;
    for (int it = 0; it < 200; ++it) {
        const double mid = 0.5 * (lo + hi);
        if (mid <= lo || mid >= hi) break;
        if (shoot(mid, ys) > 0.0) hi = mid;
        else lo = mid;
    }
    shoot(0.5 * (lo + hi), ys);
    T5kTable t{};
    for (int j = 0; j < 16; ++j) {
        t.c[16 + j] = static_cast<float>(ys[j]);
        t.c[15 - j] = -static_cast<float>(ys[j]);
    }
    for (int j = 0; j < 31; ++j) t.b[j] = (t.c[j] + t.c[j + 1]) * 0.5f;
    return t;
}

}  // namespace

const T5kTable& t5k_table() {
    static const T5kTable table = build_table();
    return table;
}

}  // namespace q3kv
