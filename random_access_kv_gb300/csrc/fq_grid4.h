// Candidate grid of the k = 4 block search [FibQuant §2.3, encoder: the nearest codeword of the
// shared codebook], built on the host in double precision.
//
// Each coordinate of a block maps to a fine lattice index j = round(u * fs + fo) (fp32 on the
// device: one fused multiply-add whose result is rounded to an integer), and a byte table maps
// j to a coarse cell index along that axis (0xFF for the two outer lattice cells, which catch
// points outside the grid). The four coarse indices select one cell of a G^4 grid. Coarse cells
// are narrow near the origin and wide in the tails, following the density of the blocks of a
// rotated unit vector (each coordinate about N(0, 1/d)); the coarse edges sit at the lattice
// boundaries nearest to Gaussian quantiles of standard deviation 1.6 / sqrt(d).
//
// A cell lists every codeword that is the nearest one to some point of the cell's box (widened
// by a small margin), by two exact tests on the box, applied in turn:
//   1. c_n stays only if its distance to the box is at most min_m (distance from c_m to the
//      box's farthest corner): that bound holds at every point of the box, so the nearest
//      codeword of any point passes;
//   2. c_n is dropped if another listed c_m is strictly closer at every point of the box:
//      |x - c_n|^2 - |x - c_m|^2 = 2 x.(c_m - c_n) + |c_n|^2 - |c_m|^2 is linear in x, so its
//      minimum over the box is at the corner picked coordinate by coordinate; the nearest
//      codeword of a point is never dropped, since no codeword is strictly closer there.
// Test 1 runs first on super-cells of 2^4 cells (a codeword that fails on a super-cell fails on
// each of its cells, and the super-cell's survivors give an upper bound for each cell's bound).
//
// Record of a cell: 16 uint16 (one 32-byte sector), e[0] = the number of listed codewords; up to
// 15 indices (ascending) in e[1..15], unused slots zero. A cell with more than 15 lists them all
// in the overflow pool at the 32-bit offset held in e[2] (low half) and e[3] (high half).
#pragma once

#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <thread>
#include <vector>

namespace fq {

constexpr int kRec = 16;         // uint16 per cell record

struct Grid4 {
    int G = 0;                   // coarse cells per axis
    int F = 512;                 // fine lattice entries per axis (0 and F - 1: outside)
    int fo = 256;                // lattice index of u = 0
    float fs = 0.f;              // lattice cells per unit of u
    std::vector<uint8_t> axis;   // [F] coarse index of each lattice entry, 0xFF outside
    std::vector<uint16_t> rec;   // [G^4][16] cell records
    std::vector<uint16_t> pool;  // overflow lists
    double mean_listed = 0;      // average list length over the cells (for diagnostics)
    int max_listed = 0;
};

namespace grid4_detail {

inline double norm_quantile(double p) {
    // Inverse of Phi(x) = erfc(-x / sqrt 2) / 2 by bisection (the grid's edges need no more).
    double lo = -40, hi = 40;
    for (int i = 0; i < 200; ++i) {
        const double mid = 0.5 * (lo + hi);
        if (0.5 * erfc(-mid / sqrt(2.0)) < p)
            lo = mid;
        else
            hi = mid;
    }
    return 0.5 * (lo + hi);
}

struct Box {
    double lo[4], hi[4];
};

// Plain comparisons (libm's fmax / fmin are calls unless the compiler may ignore NaNs).
inline double dmax(double a, double b) { return a > b ? a : b; }
inline double dmin(double a, double b) { return a < b ? a : b; }

// Codewords n of `from` that pass test 1 on box b (every codeword when from is empty).
inline void pass_bound(const double *C, int N, const std::vector<int> &from, const Box &b, std::vector<int> &out) {
    const int M = from.empty() ? N : (int)from.size();
    const int *ix = from.empty() ? nullptr : from.data();
    double U2 = INFINITY;
    for (int q = 0; q < M; ++q) {
        const double *c = C + 4 * (ix ? ix[q] : q);
        double s = 0;
        for (int i = 0; i < 4; ++i) {
            const double f = dmax(fabs(c[i] - b.lo[i]), fabs(c[i] - b.hi[i]));
            s += f * f;
        }
        U2 = dmin(U2, s);
    }
    U2 *= 1.0 + 1e-12;
    out.clear();
    for (int q = 0; q < M; ++q) {
        const int n = ix ? ix[q] : q;
        const double *c = C + 4 * n;
        double s = 0;
        for (int i = 0; i < 4; ++i) {
            const double e = dmax(0.0, dmax(b.lo[i] - c[i], c[i] - b.hi[i]));
            s += e * e;
        }
        if (s <= U2) out.push_back(n);
    }
}

// Test 2 on the survivors s of test 1: drop c_n when some c_m is strictly closer on all of b.
// The challengers c_m are tried nearest to the box's centre first, the likeliest to dominate.
inline void drop_dominated(const double *C, const double *cc, const Box &b, const std::vector<int> &s,
                           std::vector<std::pair<double, int>> &order, std::vector<int> &out) {
    double mid[4];
    for (int i = 0; i < 4; ++i) mid[i] = 0.5 * (b.lo[i] + b.hi[i]);
    order.clear();
    for (int n : s) {
        double q = 0;
        for (int i = 0; i < 4; ++i) q += (C[4 * n + i] - mid[i]) * (C[4 * n + i] - mid[i]);
        order.emplace_back(q, n);
    }
    std::sort(order.begin(), order.end());
    out.clear();
    for (int n : s) {
        const double *cn = C + 4 * n;
        bool dominated = false;
        for (size_t q = 0; q < order.size() && !dominated; ++q) {
            const int m = order[q].second;
            if (m == n) continue;
            const double *cm = C + 4 * m;
            double f = cc[n] - cc[m], mag = cc[n] + cc[m];
            for (int i = 0; i < 4; ++i) {
                const double dl = 2.0 * (cm[i] - cn[i]);
                f += dmin(dl * b.lo[i], dl * b.hi[i]);
                mag += fabs(dl) * dmax(fabs(b.lo[i]), fabs(b.hi[i]));
            }
            dominated = f > 1e-12 * mag;
        }
        if (!dominated) out.push_back(n);
    }
}

}  // namespace grid4_detail

// Builds the grid of codebook C [N x 4] for blocks of a d-dimensional unit vector.
inline void build_grid4(const float *Cf, int N, int d, Grid4 &g) {
    using namespace grid4_detail;
    std::vector<double> C((size_t)N * 4), cc(N);
    double cmax = 0;
    for (int n = 0; n < N; ++n) {
        double s = 0;
        for (int i = 0; i < 4; ++i) {
            C[4 * n + i] = Cf[4 * n + i];
            s += C[4 * n + i] * C[4 * n + i];
            cmax = fmax(cmax, fabs(C[4 * n + i]));
        }
        cc[n] = s;
    }
    // Coarse resolution: about 40 cells per axis for 1024 codewords, scaled with N^(1/4), at most
    // 40 (an 82 MB table of 32-byte records, which stays in L2 beside the streamed input).
    g.G = (int)lround(40.0 * pow(N / 1024.0, 0.25));
    g.G = std::min(40, std::max(4, g.G));
    const int G = g.G, F = g.F, fo = g.fo;
    // Extent: the codebook's, or 4.9 standard deviations of a coordinate (1 / sqrt d).
    const double R = fmax(1.05 * cmax, 4.9 / sqrt((double)d));
    g.fs = (float)((F / 2 - 2) / R);
    const double fs = g.fs;
    // Lattice entry j covers u * fs in [j - fo - 1/2, j - fo + 1/2] (round to nearest, either way
    // at the midpoint); entries 1 .. F-2 are inside. Boundary t (t = 0 .. F-2) sits at
    // u = (t + 1/2 - fo) / fs: the upper edge of entry t and the lower edge of entry t + 1.
    const int T = F - 2;   // the last boundary
    auto bound_u = [&](int t) { return (t + 0.5 - fo) / fs; };
    // Coarse cell i holds entries e[i] + 1 .. e[i+1], with 0 = e[0] < e[1] < ... < e[G] = T.
    const double sg = 1.6 / sqrt((double)d);
    const double qhi = 0.5 * erfc(-(bound_u(T) / sg) / sqrt(2.0));
    const double qlo = 0.5 * erfc(-(bound_u(0) / sg) / sqrt(2.0));
    std::vector<int> e(G + 1);
    e[0] = 0;
    e[G] = T;
    for (int i = 1; i < G; ++i) {
        const double x = sg * norm_quantile(qlo + (qhi - qlo) * i / G);
        int t = (int)lround(x * fs - 0.5 + fo);
        t = std::max(t, e[i - 1] + 1);
        t = std::min(t, T - (G - i));
        e[i] = t;
    }
    g.axis.assign(F, 0xFF);
    for (int i = 0; i < G; ++i)
        for (int j = e[i] + 1; j <= e[i + 1]; ++j) g.axis[j] = (uint8_t)i;
    // Coarse boxes along an axis, widened against rounding in these bounds.
    std::vector<double> lo(G), hi(G);
    for (int i = 0; i < G; ++i) {
        const double w = bound_u(e[i + 1]) - bound_u(e[i]);
        lo[i] = bound_u(e[i]) - 1e-6 * w;
        hi[i] = bound_u(e[i + 1]) + 1e-6 * w;
    }
    const int SG = (G + 1) / 2;   // super-cells per axis
    const size_t ncell = (size_t)G * G * G * G;
    g.rec.assign(ncell * kRec, 0);
    // Work split over super-cells; each thread keeps its overflow lists and totals.
    const int nsuper = SG * SG * SG * SG;
    unsigned nth = std::thread::hardware_concurrency();
    nth = std::max(1u, std::min(nth, 32u));
    struct Part {
        std::vector<std::pair<size_t, std::vector<uint16_t>>> ovf;
        double listed = 0;
        int maxl = 0;
    };
    std::vector<Part> parts(nth);
    auto work = [&](unsigned tid) {
        std::vector<int> none, sup, s1, s2;
        std::vector<std::pair<double, int>> order;
        Part &pt = parts[tid];
        for (int sc = (int)tid; sc < nsuper; sc += (int)nth) {
            int si[4], r = sc;
            for (int a = 3; a >= 0; --a) {
                si[a] = r % SG;
                r /= SG;
            }
            Box sb;
            int c0[4], c1[4];
            for (int a = 0; a < 4; ++a) {
                c0[a] = 2 * si[a];
                c1[a] = std::min(G, c0[a] + 2);
                sb.lo[a] = lo[c0[a]];
                sb.hi[a] = hi[c1[a] - 1];
            }
            pass_bound(C.data(), N, none, sb, sup);
            for (int i0 = c0[0]; i0 < c1[0]; ++i0)
                for (int i1 = c0[1]; i1 < c1[1]; ++i1)
                    for (int i2 = c0[2]; i2 < c1[2]; ++i2)
                        for (int i3 = c0[3]; i3 < c1[3]; ++i3) {
                            Box b;
                            const int ii[4] = {i0, i1, i2, i3};
                            for (int a = 0; a < 4; ++a) {
                                b.lo[a] = lo[ii[a]];
                                b.hi[a] = hi[ii[a]];
                            }
                            pass_bound(C.data(), N, sup, b, s1);
                            drop_dominated(C.data(), cc.data(), b, s1, order, s2);
                            std::sort(s2.begin(), s2.end());
                            const size_t cell = (((size_t)i0 * G + i1) * G + i2) * G + i3;
                            uint16_t *rr = &g.rec[cell * kRec];
                            rr[0] = (uint16_t)s2.size();
                            pt.listed += (double)s2.size();
                            pt.maxl = std::max(pt.maxl, (int)s2.size());
                            if (s2.size() <= (size_t)(kRec - 1)) {
                                for (size_t q = 0; q < s2.size(); ++q) rr[1 + q] = (uint16_t)s2[q];
                            } else {
                                pt.ovf.emplace_back(cell, std::vector<uint16_t>(s2.begin(), s2.end()));
                            }
                        }
        }
    };
    std::vector<std::thread> th;
    for (unsigned t = 1; t < nth; ++t) th.emplace_back(work, t);
    work(0);
    for (auto &t : th) t.join();
    g.pool.clear();
    double listed = 0;
    int maxl = 0;
    for (auto &pt : parts) {
        listed += pt.listed;
        maxl = std::max(maxl, pt.maxl);
        for (auto &o : pt.ovf) {
            const uint32_t off = (uint32_t)g.pool.size();
            uint16_t *rr = &g.rec[o.first * kRec];
            rr[2] = (uint16_t)(off & 0xFFFFu);
            rr[3] = (uint16_t)(off >> 16);
            g.pool.insert(g.pool.end(), o.second.begin(), o.second.end());
        }
    }
    if (g.pool.empty()) g.pool.push_back(0);
    g.mean_listed = listed / (double)ncell;
    g.max_listed = maxl;
}

}  // namespace fq
