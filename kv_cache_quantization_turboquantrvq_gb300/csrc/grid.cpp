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
#include <cmath>
#include <cstdint>
#include <cstring>

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

}  // namespace vq
