// Test helper: builds the k = 4 candidate grid of a codebook with the library's host builder and
// checks, by brute force in double precision, that for every probe point the cell the device would
// pick (the same fp32 lattice arithmetic: one fused multiply-add rounded to an integer, clamped)
// lists the exact nearest codeword, or the point falls outside the grid (the device then scans the
// whole codebook). Probe points: Gaussian blocks of a d-dimensional unit vector, uniform points,
// points near codewords and points within 1e-4 of midpoints between two codewords.
// Usage: grid4_check <codebook.f32> N d n_points seed [drop]
//        -> prints "checked C misses M outside O ..."
// With drop = 1 the check ignores each list's first entry (a planted builder error), so that a
// test can see the check fail.
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cmath>
#include <random>
#include <vector>

#include "../random_access_kv_gb300/csrc/fq_grid4.h"

int main(int argc, char **argv) {
    if (argc != 6 && argc != 7) return 2;
    const bool drop = argc == 7 && atoi(argv[6]) != 0;
    const int N = atoi(argv[2]), d = atoi(argv[3]);
    const long npts = atol(argv[4]);
    std::vector<float> C((size_t)N * 4);
    FILE *f = fopen(argv[1], "rb");
    if (!f || fread(C.data(), 4, C.size(), f) != C.size()) return 3;
    fclose(f);
    fq::Grid4 g;
    fq::build_grid4(C.data(), N, d, g);
    std::mt19937_64 rng((uint64_t)atoll(argv[5]));
    std::normal_distribution<float> gauss(0.f, 1.f / std::sqrt((float)d));
    std::uniform_real_distribution<float> unif(-0.8f, 0.8f);
    std::normal_distribution<float> jitter(0.f, 1.f);
    const float magic = 12582912.f;             // 1.5 * 2^23
    long misses = 0, outside = 0, checked = 0;
    for (long it = 0; it < npts; ++it) {
        float u[4];
        const int mode = (int)(it % 4);
        const int a = (int)(rng() % (uint64_t)N), b = (int)(rng() % (uint64_t)N);
        for (int i = 0; i < 4; ++i) {
            if (mode == 0) u[i] = gauss(rng);
            else if (mode == 1) u[i] = unif(rng);
            else if (mode == 2) u[i] = C[4 * a + i] + 0.01f * jitter(rng);
            else u[i] = 0.5f * (C[4 * a + i] + C[4 * b + i]) + 1e-4f * jitter(rng);
        }
        uint32_t cell = 0, orv = 0;
        for (int i = 0; i < 4; ++i) {
            const float t = std::fmaf(u[i], g.fs, (float)g.fo + magic);
            int32_t bits;
            memcpy(&bits, &t, 4);
            uint32_t j = (uint32_t)(bits - 0x4B400000);
            if (j > (uint32_t)(g.F - 1)) j = (uint32_t)(g.F - 1);
            const uint32_t cv = g.axis[j];
            cell = cell * (uint32_t)g.G + cv;
            orv |= cv;
        }
        if (orv >= 0x80u) {
            ++outside;
            continue;
        }
        const uint16_t *rec = &g.rec[(size_t)cell * fq::kRec];
        const int cnt = rec[0];
        const uint16_t *lst = rec + 1;
        if (cnt > fq::kRec - 1) lst = &g.pool[(uint32_t)rec[2] | ((uint32_t)rec[3] << 16)];
        double best = INFINITY;
        int bi = -1;
        for (int n = 0; n < N; ++n) {
            double s = 0;
            for (int i = 0; i < 4; ++i) {
                const double e = (double)u[i] - (double)C[4 * n + i];
                s += e * e;
            }
            if (s < best) {
                best = s;
                bi = n;
            }
        }
        bool found = false;
        for (int q = drop ? 1 : 0; q < cnt; ++q) found = found || lst[q] == bi;
        // Lists are ascending and hold valid indices.
        for (int q = 1; q < cnt; ++q)
            if (lst[q] <= lst[q - 1]) found = false;
        ++checked;
        if (!found) ++misses;
    }
    printf("checked %ld misses %ld outside %ld G %d mean_listed %.3f max_listed %d\n", checked, misses, outside, g.G,
           g.mean_listed, g.max_listed);
    return 0;
}
