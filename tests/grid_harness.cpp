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
#include <cstring>
#include <string>
#include <vector>

#include "launch.h"

using namespace vq;

static int count_above(float v, const std::vector<float> &b)
{
    int c = 0;
    for (float x : b) c += v > x;
    return c;
}

// The exact two-stage pair of the fp32 value v (binary64 arithmetic).
static unsigned pair_exact(float v, const float *c1, const float *b1, const float *b2, int L)
{
    int i1 = 0, i2 = 0;
    for (int k = 0; k < L - 1; ++k) i1 += (double)v > (double)b1[k];
    const double r = (double)v - (double)c1[i1];
    for (int j = 0; j < L - 1; ++j) i2 += r > (double)b2[j];
    return (unsigned)(i1 | (i2 << 4));
}

// Usage: grid_harness pair guard c1[16] b1[15] c2[16] b2[15].  For the table
// build_pair_table returns, checks on many fp32 values v that the looked-up
// pair equals the exact pair whenever v is at least `guard` from its cell's
// boundary (closer values are flagged on the device and recomputed), and that
// no step of the pair function outside v's cell lies within `guard` of v.
static int pair_main(int argc, char **argv)
{
    if (argc != 3 + 62) return 2;
    const float guard = std::strtof(argv[2], nullptr);
    float c1[16], b1[15], c2[16], b2[15];
    int a = 3;
    for (int i = 0; i < 16; ++i) c1[i] = std::strtof(argv[a++], nullptr);
    for (int i = 0; i < 15; ++i) b1[i] = std::strtof(argv[a++], nullptr);
    for (int i = 0; i < 16; ++i) c2[i] = std::strtof(argv[a++], nullptr);
    for (int i = 0; i < 15; ++i) b2[i] = std::strtof(argv[a++], nullptr);
    static PairTable t;
    if (!build_pair_table(c1, b1, c2, b2, 4, guard, t)) {
        std::printf("NOTABLE\n");
        return 1;
    }
    // the steps, recomputed here by brute force: every fp32 value where the
    // exact pair changes between neighbours, found on a dense sweep and refined
    std::vector<float> vals;
    std::vector<double> steps;
    const float lo = -0.6f, hi = 0.6f;
    float prev = lo;
    unsigned pp = pair_exact(prev, c1, b1, b2, 16);
    for (int i = 1; i <= 400000; ++i) {
        const float v = lo + (hi - lo) * (float)i / 400000.0f;
        const unsigned pv = pair_exact(v, c1, b1, b2, 16);
        vals.push_back(v);
        if (pv != pp) {
            float l = prev, h = v;  // pair changes in (l, h]: bisect to adjacent floats
            while (std::nextafterf(l, INFINITY) < h) {
                const float m = l + 0.5f * (h - l);
                if (m <= l || m >= h) break;
                if (pair_exact(m, c1, b1, b2, 16) == pp) l = m; else h = m;
            }
            steps.push_back((double)l);
            for (int k = 0; k < 6; ++k) {
                vals.push_back(l);
                vals.push_back(h);
                l = std::nextafterf(l, -INFINITY);
                h = std::nextafterf(h, INFINITY);
            }
        }
        prev = v;
        pp = pv;
    }
    for (double sv : steps) {
        vals.push_back((float)(sv - guard));
        vals.push_back((float)(sv + guard));
        vals.push_back((float)(sv - 2.0 * guard));
        vals.push_back((float)(sv + 2.0 * guard));
    }
    vals.push_back(0.0f);
    vals.push_back(-0.0f);
    vals.push_back(1e30f);
    vals.push_back(-1e30f);
    long checked = 0, flagged = 0;
    for (float v : vals) {
        const int g = pair_cell_host(v, t.a, t.bc);
        float bnd;
        std::memcpy(&bnd, &t.ent[g].x, 4);
        const unsigned sel = v > bnd ? 1u : 0u;
        const unsigned got = (t.ent[g].y >> (8 * sel)) & 0xffu;
        const unsigned ref = pair_exact(v, c1, b1, b2, 16);
        const bool near = std::fabs((double)bnd - (double)v) < guard;
        if (near) {
            ++flagged;
        } else if (got != ref) {
            std::printf("PAIR v=%.9g g=%d table=%02x exact=%02x\n", v, g, got, ref);
            return 1;
        }
        for (double sv : steps) {
            if (pair_cell_host((float)sv, t.a, t.bc) == g) continue;
            if (std::fabs((double)v - sv) < guard - 1e-12) {
                std::printf("MARGIN v=%.9g step=%.9g g=%d\n", v, sv, g);
                return 1;
            }
        }
        ++checked;
    }
    std::printf("OK %ld flagged %ld steps %zu\n", checked, flagged, steps.size());
    return 0;
}

int main(int argc, char **argv)
{
    if (argc >= 2 && std::string(argv[1]) == "pair") return pair_main(argc, argv);
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
