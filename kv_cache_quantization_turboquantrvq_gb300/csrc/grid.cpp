// grid.cpp - host construction of the boundary-count lookup tables
// (GridTable in launch.h).
//
// The device maps a value v to one of 32 cells with two correctly rounded
// fp32 FMAs and a saturation:
//   g(v) = RN(31 * sat(fma(v, a, bc)))   (the result's low 5 bits)
// which is monotone in v.  The host evaluates the same fp32 map, so it knows
// exactly which fp32 values share a cell.  A table is accepted when every
// boundary has a cell of its own and sits at least `guard` away from that
// cell's edges; then, for v in cell g,
//   #{k : v > b_k} = code[g] + (v > bnd[g])
// exactly, and no boundary outside the cell is within `guard` of v.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "launch.h"

namespace vq {
namespace {

int32_t ordered(float f)
{
    int32_t i;
    std::memcpy(&i, &f, 4);
    return i >= 0 ? i : (int32_t)(0x80000000u - (uint32_t)i);
}

float from_ordered(int32_t o)
{
    const int32_t i = o >= 0 ? o : (int32_t)(0x80000000u - (uint32_t)o);
    float f;
    std::memcpy(&f, &i, 4);
    return f;
}

// Smallest finite float v with grid_cell_host(v) >= g.
double cell_lower_edge(int g, float a, float bc)
{
    if (g <= 0) return -INFINITY;
    int64_t lo = ordered(-3.0e38f), hi = ordered(3.0e38f);
    if (grid_cell_host(from_ordered((int32_t)hi), a, bc) < g) return INFINITY;
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (grid_cell_host(from_ordered((int32_t)mid), a, bc) >= g) hi = mid;
        else lo = mid + 1;
    }
    return (double)from_ordered((int32_t)lo);
}

}  // namespace

int grid_cell_host(float v, float a, float bc)
{
    float u = std::fmaf(v, a, bc);
    if (!(u > 0.0f)) u = 0.0f;  // NaN -> 0 as the device saturation
    if (u > 1.0f) u = 1.0f;
    const float gf = std::fmaf(u, 31.0f, 12582912.0f);
    uint32_t bits;
    std::memcpy(&bits, &gf, 4);
    return (int)(bits & 31u);
}

bool build_grid(const float *b, int nb, float guard, GridTable &t)
{
    if (nb < 1 || nb > 31) return false;
    const double span = nb > 1 ? (double)b[nb - 1] - (double)b[0]
                               : std::fmax(std::fabs((double)b[0]), 1e-3);
    // Try widths (padding around the outer boundaries) and phases (shifts of a
    // fraction of a cell); a symmetric codebook puts its middle boundary on a
    // cell edge at phase 0, which the margin check rejects.
    for (int trial = 0; trial < 64; ++trial) {
        for (int ph = 0; ph < 8; ++ph) {
            const double pad = span * (0.6 / 31.0 + 0.0071 * trial);
            const double width = (nb > 1 ? span : 0.0) + 2.0 * pad;
            const double phase = (0.5 + 0.37 * ph) / 31.0;
            t.a = (float)(1.0 / width);
            t.bc = (float)(-((double)b[0] - pad) / width + phase - 0.5 / 31.0);
            int cell[32];
            bool ok = true;
            for (int k = 0; k < nb && ok; ++k) {
                cell[k] = grid_cell_host(b[k], t.a, t.bc);
                if (k > 0 && cell[k] <= cell[k - 1]) ok = false;
            }
            for (int k = 0; k < nb && ok; ++k) {
                const double lo = cell_lower_edge(cell[k], t.a, t.bc);
                const double hi = cell[k] == 31 ? INFINITY : cell_lower_edge(cell[k] + 1, t.a, t.bc);
                if (!((double)b[k] - lo >= guard) || !(hi - (double)b[k] > guard)) ok = false;
            }
            if (!ok) continue;
            int k = 0;
            for (int g = 0; g < 32; ++g) {
                while (k < nb && cell[k] < g) ++k;
                const bool has = k < nb && cell[k] == g;
                t.bnd[g] = has ? b[k] : -INFINITY;
                t.code[g] = has ? k : k - 1;
            }
            return true;
        }
    }
    return false;
}

int pair_cell_host(float v, float a, float bc)
{
    float u = std::fmaf(v, a, bc);
    if (!(u > 0.0f)) u = 0.0f;
    if (u > 1.0f) u = 1.0f;
    const float gf = std::fmaf(u, (float)(PT_CELLS - 1), 12582912.0f);
    uint32_t bits;
    std::memcpy(&bits, &gf, 4);
    return (int)(bits - 0x4B400000u);
}

// The code pair (i1 | i2 << 4) of a binary64 value y, by the definition:
// i1 = #{k : y > b1_k}, i2 = #{j : y - c1[i1] > b2_j}.
static uint32_t pair_of(double y, const float *c1, const float *b1, const float *b2, int L)
{
    int i1 = 0, i2 = 0;
    for (int k = 0; k < L - 1; ++k) i1 += y > (double)b1[k];
    const double r = y - (double)c1[i1];
    for (int j = 0; j < L - 1; ++j) i2 += r > (double)b2[j];
    return (uint32_t)(i1 | (i2 << 4));
}

// Largest fp32 not above x / smallest fp32 not below x.
static float f32_down(double x)
{
    float f = (float)x;
    if ((double)f > x) f = std::nextafterf(f, -INFINITY);
    return f;
}
static float f32_up(double x)
{
    float f = (float)x;
    if ((double)f < x) f = std::nextafterf(f, INFINITY);
    return f;
}

bool build_pair_table(const float *c1, const float *b1, const float *c2, const float *b2, int bits,
                      float guard, PairTable &t)
{
    (void)c2;
    if (bits != 4) return false;
    const int L = 1 << bits;
    // every step of the pair function: stage-1 boundaries, and the stage-2
    // boundaries shifted by c1[k] that fall strictly inside stage-1 cell k
    // (exact sums in binary64; compared on the device as fp32)
    std::vector<double> steps;
    for (int k = 0; k < L - 1; ++k) steps.push_back((double)b1[k]);
    for (int k = 0; k < L; ++k) {
        const double lo = k > 0 ? (double)b1[k - 1] : -INFINITY;
        const double hi = k < L - 1 ? (double)b1[k] : INFINITY;
        for (int j = 0; j < L - 1; ++j) {
            const double s = (double)c1[k] + (double)b2[j];
            if (s > lo && s < hi) steps.push_back(s);
        }
    }
    std::sort(steps.begin(), steps.end());
    const int nb = (int)steps.size();
    std::vector<float> bnd(nb);
    for (int i = 0; i < nb; ++i) {
        bnd[i] = (float)steps[i];
        if (!std::isfinite(bnd[i])) return false;
        // two steps that no fp32 value separates by more than the guard band
        if (i > 0 && !((double)bnd[i] - (double)bnd[i - 1] > 2.0 * guard)) return false;
    }
    // the pair on each open interval between consecutive steps (segment s
    // lies between steps s-1 and s), evaluated at its midpoint
    std::vector<uint32_t> seg(nb + 1);
    for (int s = 0; s <= nb; ++s) {
        const double y = s == 0 ? steps[0] - 1.0
                         : s == nb ? steps[nb - 1] + 1.0
                                   : 0.5 * (steps[s - 1] + steps[s]);
        seg[s] = pair_of(y, c1, b1, b2, L);
    }
    const double span = (double)bnd[nb - 1] - (double)bnd[0];
    std::vector<int> cell(nb);
    for (int trial = 0; trial < 64; ++trial) {
        for (int ph = 0; ph < 16; ++ph) {
            const double pad = span * (2.0 / (PT_CELLS - 1) + 0.0013 * trial);
            const double width = span + 2.0 * pad;
            const double phase = (0.5 + 0.0613 * ph) / (PT_CELLS - 1);
            t.a = (float)(1.0 / width);
            t.bc = (float)(-((double)bnd[0] - pad) / width + phase - 0.5 / (PT_CELLS - 1));
            bool ok = true;
            for (int i = 0; i < nb && ok; ++i) {
                cell[i] = pair_cell_host(bnd[i], t.a, t.bc);
                // own cell, and every fp32 value within three guard bands of
                // the boundary in that same cell (the map is monotone)
                if (i > 0 && cell[i] <= cell[i - 1]) ok = false;
                if (pair_cell_host(f32_down((double)bnd[i] - 3.0 * guard), t.a, t.bc) != cell[i] ||
                    pair_cell_host(f32_up((double)bnd[i] + 3.0 * guard), t.a, t.bc) != cell[i])
                    ok = false;
            }
            if (!ok) continue;
            int i = 0;
            for (int g = 0; g < PT_CELLS; ++g) {
                while (i < nb && cell[i] < g) ++i;
                const bool has = i < nb && cell[i] == g;
                float b = has ? bnd[i] : -INFINITY;
                uint32_t bb;
                std::memcpy(&bb, &b, 4);
                const uint32_t below = seg[i];
                const uint32_t above = has ? seg[i + 1] : seg[i];
                t.ent[g].x = bb;
                t.ent[g].y = below | (above << 8);
            }
            return true;
        }
    }
    return false;
}

}  // namespace vq
