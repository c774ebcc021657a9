// Host check of the boundary-count tables (csrc/grid.cpp), built and run by
// tests/test_grid_tables.py.  Usage: grid_harness guard b0 b1 ... (sorted).
// For the table build_grid returns, checks on many fp32 values v (every
// boundary and its neighbours, every cell edge and its neighbours, a dense
// sweep) that
//   (1) code[g(v)] + (v > bnd[g(v)]) == #{k : v > b_k}, and
//   (2) no boundary outside v's cell lies within `guard` of v.
// Prints "OK <checked>" or a failure description; exit code 0 only on OK.
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "launch.h"

using namespace vq;

static int count_above(float v, const std::vector<float> &b)
{
    int c = 0;
    for (float x : b) c += v > x;
    return c;
}

int main(int argc, char **argv)
{
    if (argc < 3) return 2;
    const float guard = std::strtof(argv[1], nullptr);
    std::vector<float> b;
    for (int i = 2; i < argc; ++i) b.push_back(std::strtof(argv[i], nullptr));
    GridTable t;
    if (!build_grid(b.data(), (int)b.size(), guard, t)) {
        std::printf("NOTABLE\n");
        return 1;
    }
    std::vector<float> vals;
    for (float x : b) {
        float lo = x, hi = x;
        vals.push_back(x);
        for (int i = 0; i < 8; ++i) {
            lo = std::nextafterf(lo, -INFINITY);
            hi = std::nextafterf(hi, INFINITY);
            vals.push_back(lo);
            vals.push_back(hi);
        }
        vals.push_back(x - guard);
        vals.push_back(x + guard);
    }
    // cell edges: binary search for the first value of every cell
    for (int g = 1; g < 32; ++g) {
        float lo = -1e30f, hi = 1e30f;
        for (int it = 0; it < 200; ++it) {
            const float mid = 0.5f * (lo + hi);
            if (grid_cell_host(mid, t.a, t.bc) >= g) hi = mid; else lo = mid;
        }
        vals.push_back(lo);
        vals.push_back(hi);
        vals.push_back(std::nextafterf(hi, INFINITY));
    }
    const double span = (double)b.back() - (double)b.front() + 1e-3;
    for (int i = 0; i <= 200000; ++i)
        vals.push_back((float)((double)b.front() - span + 3.0 * span * i / 200000.0));
    vals.push_back(0.0f);
    vals.push_back(-0.0f);
    vals.push_back(1e30f);
    vals.push_back(-1e30f);
    long checked = 0;
    for (float v : vals) {
        const int g = grid_cell_host(v, t.a, t.bc);
        const int code = t.code[g] + (v > t.bnd[g] ? 1 : 0);
        const int ref = count_above(v, b);
        if (code != ref) {
            std::printf("COUNT v=%.9g g=%d table=%d direct=%d\n", v, g, code, ref);
            return 1;
        }
        for (size_t k = 0; k < b.size(); ++k) {
            if (grid_cell_host(b[k], t.a, t.bc) == g) continue;
            if (std::fabs((double)v - (double)b[k]) < guard) {
                std::printf("MARGIN v=%.9g b=%.9g g=%d\n", v, b[k], g);
                return 1;
            }
        }
        ++checked;
    }
    std::printf("OK %ld a=%.9g bc=%.9g\n", checked, t.a, t.bc);
    return 0;
}
