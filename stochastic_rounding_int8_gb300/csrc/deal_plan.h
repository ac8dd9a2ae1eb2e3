// Static deal of a persistent GEMM launch's tiles to its CTAs.
//
// A launch runs its problems' tiles on G persistent CTAs.  Problem i has n[i]
// tiles of cost c[i] each (its 128-wide contraction blocks plus a per-tile
// share of the epilogue).  Its tiles are dealt in two phases (the kernel's
// next_tile walks the same plan): first m rounds over the w CTAs s, s + 1, ...
// (cyclic), then round robin over all G CTAs starting at s.  With m = 0 and s
// the CTA after the previous problem's last tile this is plain round robin
// over the whole launch.
//
// Round robin leaves the CTAs that took the last, partial round of a problem
// with long tiles one long tile ahead of the rest; the first phase of the next
// problem hands that deficit to the CTAs behind.  The plan is chosen greedily,
// problem by problem (the launch orders them longest tile first): among plain
// round robin and the catch-up deals over a low run of CTAs it takes the one
// with the smallest maximum load, then the smallest sum of squared loads.
#pragma once

#include <cstdint>
#include <vector>

#if defined(__CUDACC__)
#define S3R_DEAL_HD __host__ __device__ __forceinline__
#else
#define S3R_DEAL_HD inline
#endif

namespace s3r {
namespace deal {

struct Plan {
    int s, w, m;
};

// The k-th tile (k = 0, 1, ...; within the problem, in increasing order) that
// CTA b of G takes from a problem of n tiles under the plan (s, w, m); false
// past its last.  Tile counts stay below 2^30, so int arithmetic holds.
S3R_DEAL_HD bool kth_tile(int n, int s, int w, int m, int b, int G, int k, int& t) {
    const int rel = b >= s ? b - s : b - s + G;   // b's place counted from s
    const int my1 = rel < w ? m : 0;               // b's tiles of the first phase
    if (k < my1) {
        t = rel + k * w;
        return true;
    }
    const int t2 = m * w + rel + (k - my1) * G;
    if (t2 < n) {
        t = t2;
        return true;
    }
    return false;
}

// Tiles CTA b (of G) takes from a problem of n tiles under plan p.
inline int64_t tiles_of(int64_t n, const Plan& p, int b, int G) {
    const int rel = b >= p.s ? b - p.s : b - p.s + G;
    const int64_t n1 = (int64_t)p.m * p.w;
    const int64_t my1 = rel < p.w ? p.m : 0;
    const int64_t my2 = n - n1 > rel ? (n - n1 - rel + G - 1) / G : 0;
    return my1 + my2;
}

// The CTA after the last one that takes a tile under plan p.
inline int next_start(int64_t n, const Plan& p, int G) {
    const int64_t n2 = n - (int64_t)p.m * p.w;
    if (n2 > 0) return (int)((p.s + n2) % G);
    return (p.s + p.w) % G;
}

// Plans for problems 0 .. nprob (n[i] tiles of cost c[i]) on G CTAs.
inline void plan(int nprob, const int64_t* n, const double* c, int G, Plan* out) {
    std::vector<double> L(G, 0.0);   // load per CTA so far
    int next = 0;
    constexpr int kMaxEvals = 1024;
    for (int i = 0; i < nprob; ++i) {
        Plan best{next, G, 0};
        if (n[i] <= 0 || G <= 1) {
            out[i] = best;
            continue;
        }
        double best_max = 0.0, best_ss = 0.0;
        auto score = [&](const Plan& p, double& mx, double& ss) {
            mx = 0.0;
            ss = 0.0;
            for (int b = 0; b < G; ++b) {
                const double v = L[b] + c[i] * (double)tiles_of(n[i], p, b, G);
                mx = v > mx ? v : mx;
                ss += v * v;
            }
        };
        score(best, best_max, best_ss);
        // low runs of CTAs: [s, e) cyclic, s where the load drops, e where it rises
        std::vector<int> drops, rises;
        double lo = L[0], hi = L[0];
        for (int b = 0; b < G; ++b) {
            const double prev = L[(b + G - 1) % G];
            if (L[b] < prev) drops.push_back(b);
            if (L[b] > prev) rises.push_back(b);
            lo = L[b] < lo ? L[b] : lo;
            hi = L[b] > hi ? L[b] : hi;
        }
        // rounds that can close the gap between the lowest and the highest CTA
        const int64_t mcap = (int64_t)((hi - lo) / c[i]) + 1;
        int evals = 0;
        for (int s : drops) {
            for (int e : rises) {
                const int w = (e - s + G) % G;
                if (w == 0) continue;
                for (int64_t m = 1; m <= mcap && m * w <= n[i] && evals < kMaxEvals; ++m, ++evals) {
                    const Plan p{s, w, (int)m};
                    double mx, ss;
                    score(p, mx, ss);
                    const double tol = 1e-9 * (best_max > 1.0 ? best_max : 1.0);
                    if (mx < best_max - tol || (mx <= best_max + tol && ss < best_ss * (1.0 - 1e-12))) {
                        best = p;
                        best_max = mx;
                        best_ss = ss;
                    }
                }
            }
        }
        out[i] = best;
        for (int b = 0; b < G; ++b) L[b] += c[i] * (double)tiles_of(n[i], best, b, G);
        next = next_start(n[i], best, G);
    }
}

}  // namespace deal
}  // namespace s3r
