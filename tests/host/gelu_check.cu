// Host-side check of the GELU of fno_gelu.cuh against the exact form in double
// precision, v/2 (1 + erf(v / sqrt 2)), on a dense grid of v in [-12, 12].
// Prints "<max abs error> <max abs error / max(1, |v|)> <points>".
#include <cmath>
#include <cstdio>

#include "fno_gelu.cuh"

int main() {
    double worst = 0.0, worst_rel = 0.0;
    int n = 0;
    for (int i = -1200000; i <= 1200000; ++i, ++n) {
        const float v = (float)(i * 1e-5);
        const double exact = 0.5 * (double)v * (1.0 + std::erf((double)v / std::sqrt(2.0)));
        const double err = std::fabs((double)fno::gelu_erf(v) - exact);
        if (err > worst) worst = err;
        const double rel = err / std::fmax(1.0, std::fabs((double)v));
        if (rel > worst_rel) worst_rel = rel;
    }
    std::printf("%.3e %.3e %d\n", worst, worst_rel, n);
    return 0;
}
