// Host check of the GEMM's static tile deal (the header the kernel walks).
// Reads launches from stdin, one per line: G nprob n_0 c_0 ... n_{nprob-1} c_{nprob-1}.
// Prints one line per launch: "ok <max load, deal> <max load, round robin> <mean load> s w m ..."
// or "FAIL <reason>".
#include <cstdio>
#include <vector>

#include "../stochastic_rounding_int8_gb300/csrc/deal_plan.h"

using namespace s3r::deal;

int main() {
    int G, np;
    while (std::scanf("%d %d", &G, &np) == 2) {
        std::vector<int64_t> n(np);
        std::vector<double> c(np);
        for (int i = 0; i < np; ++i) {
            long long ni = 0;
            if (std::scanf("%lld %lf", &ni, &c[i]) != 2) return 2;
            n[i] = ni;
        }
        std::vector<Plan> p(np);
        plan(np, n.data(), c.data(), G, p.data());
        std::vector<double> L(G, 0.0), Lrr(G, 0.0);
        double total = 0.0;
        int64_t base = 0;
        const char* fail = nullptr;
        for (int i = 0; i < np && !fail; ++i) {
            if (p[i].s < 0 || p[i].s >= G || p[i].w < 1 || p[i].w > G || p[i].m < 0 ||
                (int64_t)p[i].m * p[i].w > n[i])
                fail = "plan out of range";
            std::vector<int> seen(n[i] > 0 ? n[i] : 0, 0);
            for (int b = 0; b < G && !fail; ++b) {
                int64_t cnt = 0;
                int last = -1, t = 0;
                for (int k = 0; kth_tile((int)n[i], p[i].s, p[i].w, p[i].m, b, G, k, t); ++k) {
                    if (t < 0 || t >= n[i]) { fail = "tile out of range"; break; }
                    if (t <= last) { fail = "tiles not increasing"; break; }
                    last = t;
                    ++seen[t];
                    ++cnt;
                }
                if (!fail && cnt != tiles_of(n[i], p[i], b, G)) fail = "count differs from tiles_of";
                L[b] += c[i] * (double)cnt;
            }
            for (int64_t t = 0; t < n[i] && !fail; ++t)
                if (seen[t] != 1) fail = "a tile not dealt exactly once";
            for (int64_t t = 0; t < n[i]; ++t) Lrr[(base + t) % G] += c[i];
            base += n[i];
            total += c[i] * (double)n[i];
        }
        if (fail) {
            std::printf("FAIL %s\n", fail);
            continue;
        }
        double mx = 0.0, mrr = 0.0;
        for (int b = 0; b < G; ++b) {
            mx = L[b] > mx ? L[b] : mx;
            mrr = Lrr[b] > mrr ? Lrr[b] : mrr;
        }
        std::printf("ok %.6f %.6f %.6f", mx, mrr, total / G);
        for (int i = 0; i < np; ++i) std::printf(" %d %d %d", p[i].s, p[i].w, p[i].m);
        std::printf("\n");
    }
    return 0;
}
