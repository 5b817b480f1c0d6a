// sequoia_tree.cpp -- tree construction on the host: the draft-tree shape with the
// largest expected number of generated tokens per verification step, and the
// hardware-aware choice of its size and depth.
//
// Sequoia summary, sections "Scalable Speculative Decoding" and "Dynamic Programming":
// the speculated tokens form a tree whose shape is found by dynamic programming over
// smaller subproblems; figure of forward-pass time against input length: the size
// trades draft time against verification time.  The objective and the recurrence are
// not on the pages; the reading used here (positional acceptance vector, E(tree) =
// sum over nodes of the probability that the walk reaches them) is stated in tsv.h.
// The acceptance vector itself is estimated from verification outputs by
// tsv_sequoia_accept_counts (per rank: reached nodes with that many children, and how
// often the child of that rank was the accepted one).
//
// Recurrence.  With F(n, d) the best E of an n-node tree of depth <= d:
//   F(1, d) = 1;  F(n > 1, 0) = -inf;
//   F(n, d) = 1 + G_d(1, n - 1)  for d >= 1, where G_d(i, m) is the best value of m
//   nodes hung below a node as children of rank i, i+1, ... (each child of rank j with
//   its own subtree of a nodes and depth <= d - 1 adds accept[j-1] * F(a, d - 1)):
//     G_d(i, 0) = 0;   G_d(K + 1, m) = 0 (the m nodes become children of rank > K,
//     leaves, never accepted);   G_d(i, m) = max over 1 <= a <= m with
//     F(a, d - 1) > -inf of accept[i-1] * F(a, d - 1) + G_d(i + 1, m - a).
// The ranks are filled in order, so a node's children occupy ranks 1, 2, ... with no
// gap.  Cost O(D K n^2) for D = min(d_max, n_max - 1) levels and K = min(K, n_max - 1)
// ranks: about 10^8 multiply-adds at n = 128, D = K = 127, a fraction of a second.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#include "../../include/tsv.h"

namespace tsv {
tsv_status report_error(tsv_status s, const char* fmt, ...);
}

namespace {

constexpr int kMaxTreeNodes = 128;

// The DP over levels d = 1..D for trees of up to n_max nodes.  F is kept for every
// level; the choice table records, per level, rank and budget, the size of the
// rank's subtree (0: no child, or the leftover nodes become never-accepted leaves).
struct SequoiaDP {
    int n_max = 0, D = 0, K = 0;
    std::vector<double> F;          // [(D + 1) * (n_max + 1)]
    std::vector<uint8_t> choice;    // [D][K + 1][n_max]   (level d >= 1, rank i in 1..K, budget m)

    double f(int n, int d) const { return F[(size_t)d * (n_max + 1) + n]; }
    uint8_t& pick(int d, int i, int m) { return choice[((size_t)(d - 1) * (K + 1) + i) * n_max + m]; }
    uint8_t pick(int d, int i, int m) const { return choice[((size_t)(d - 1) * (K + 1) + i) * n_max + m]; }

    void run(const double* accept, int K_in, int n_max_in, int d_max) {
        n_max = n_max_in;
        D = d_max < n_max - 1 ? d_max : n_max - 1;
        K = K_in < n_max - 1 ? K_in : n_max - 1;
        F.assign((size_t)(D + 1) * (n_max + 1), -INFINITY);
        choice.assign((size_t)(D > 0 ? D : 1) * (K + 1) * n_max, 0);
        for (int d = 0; d <= D; ++d) F[(size_t)d * (n_max + 1) + 0] = 0.0;
        for (int d = 0; d <= D; ++d) F[(size_t)d * (n_max + 1) + 1] = 1.0;
        std::vector<double> g_next(n_max), g_cur(n_max);  // G_d(i + 1, .), G_d(i, .)
        for (int d = 1; d <= D; ++d) {
            const double* Fprev = &F[(size_t)(d - 1) * (n_max + 1)];
            for (int m = 0; m < n_max; ++m) g_next[m] = 0.0;  // rank K + 1: leftover leaves
            for (int i = K; i >= 1; --i) {
                const double p = accept[i - 1];
                g_cur[0] = 0.0;
                pick(d, i, 0) = 0;
                for (int m = 1; m < n_max; ++m) {
                    double best = -INFINITY;
                    int best_a = 0;
                    for (int a = 1; a <= m; ++a) {
                        const double fa = Fprev[a];
                        if (fa == -INFINITY) continue;
                        const double v = p * fa + g_next[m - a];
                        if (v > best) {
                            best = v;
                            best_a = a;
                        }
                    }
                    g_cur[m] = best;
                    pick(d, i, m) = static_cast<uint8_t>(best_a);
                }
                g_next.swap(g_cur);
            }
            double* Fd = &F[(size_t)d * (n_max + 1)];
            for (int n = 2; n <= n_max; ++n) Fd[n] = 1.0 + g_next[n - 1];  // g_next = G_d(1, .)
        }
    }
};

// Children (by rank) of a subtree of s nodes with depth budget r, rooted at `node`,
// appended to the ordered child lists `kids`.
void build_subtree(const SequoiaDP& dp, int node, int s, int r, std::vector<std::vector<int>>& kids, int& next_id) {
    if (s <= 1 || r <= 0) return;
    const int d = r < dp.D ? r : dp.D;  // a deeper budget than D changes nothing
    int m = s - 1;
    for (int i = 1; i <= dp.K && m > 0; ++i) {
        const int a = dp.pick(d, i, m);
        if (a == 0) break;
        const int c = next_id++;
        kids[node].push_back(c);
        kids.emplace_back();
        build_subtree(dp, c, a, r - 1, kids, next_id);
        m -= a;
    }
    for (; m > 0; --m) {  // leftover: never-accepted leaves of rank > K
        const int c = next_id++;
        kids[node].push_back(c);
        kids.emplace_back();
    }
}

bool check_accept(const double* accept, int K) {
    double sum = 0.0;
    for (int k = 0; k < K; ++k) {
        if (!(accept[k] >= 0.0) || !std::isfinite(accept[k])) return false;
        sum += accept[k];
    }
    return sum <= 1.0 + 1e-9;
}

}  // namespace

extern "C" {

tsv_status tsv_sequoia_values(const double* accept, int K, int n_max, int d_max, double* values) {
    if (!accept || !values) return tsv::report_error(TSV_ERR_ARG, "null pointer");
    if (K < 1 || n_max < 1 || n_max > kMaxTreeNodes || d_max < 0)
        return tsv::report_error(TSV_ERR_ARG, "bad sizes K=%d n_max=%d d_max=%d", K, n_max, d_max);
    if (!check_accept(accept, K)) return tsv::report_error(TSV_ERR_ARG, "accept must be >= 0 with sum <= 1");
    SequoiaDP dp;
    dp.run(accept, K, n_max, d_max);
    for (int n = 0; n <= n_max; ++n)
        for (int d = 0; d <= d_max; ++d) values[(size_t)n * (d_max + 1) + d] = dp.f(n, d < dp.D ? d : dp.D);
    return TSV_OK;
}

tsv_status tsv_sequoia_tree(const double* accept, int K, int n, int max_depth, int32_t* parent, double* expected) {
    if (!accept || !parent || !expected) return tsv::report_error(TSV_ERR_ARG, "null pointer");
    if (K < 1 || n < 1 || n > kMaxTreeNodes || max_depth < 0 || (n > 1 && max_depth < 1))
        return tsv::report_error(TSV_ERR_ARG, "bad sizes K=%d n=%d max_depth=%d", K, n, max_depth);
    if (!check_accept(accept, K)) return tsv::report_error(TSV_ERR_ARG, "accept must be >= 0 with sum <= 1");
    SequoiaDP dp;
    dp.run(accept, K, n, max_depth);
    std::vector<std::vector<int>> kids(1);
    int next_id = 1;
    build_subtree(dp, 0, n, max_depth, kids, next_id);
    // breadth-first relabelling: children in rank order get increasing indices
    std::vector<int> order{0}, label(n, -1);
    label[0] = 0;
    parent[0] = -1;
    for (size_t h = 0; h < order.size(); ++h) {
        const int u = order[h];
        for (int c : kids[u]) {
            label[c] = static_cast<int>(order.size());
            parent[label[c]] = label[u];
            order.push_back(c);
        }
    }
    *expected = dp.f(n, max_depth < dp.D ? max_depth : dp.D);
    return TSV_OK;
}

tsv_status tsv_sequoia_plan(const double* accept, int K, int n_max, int d_max, const double* t_verify,
                            double t_draft, int* n_best, int* d_best, double* speedup) {
    if (!accept || !t_verify || !n_best || !d_best || !speedup) return tsv::report_error(TSV_ERR_ARG, "null pointer");
    if (K < 1 || n_max < 1 || n_max > kMaxTreeNodes || d_max < 0)
        return tsv::report_error(TSV_ERR_ARG, "bad sizes K=%d n_max=%d d_max=%d", K, n_max, d_max);
    if (!check_accept(accept, K)) return tsv::report_error(TSV_ERR_ARG, "accept must be >= 0 with sum <= 1");
    if (!(t_draft >= 0.0) || !std::isfinite(t_draft)) return tsv::report_error(TSV_ERR_ARG, "t_draft must be >= 0");
    for (int n = 1; n <= n_max; ++n)
        if (!(t_verify[n] > 0.0) || !std::isfinite(t_verify[n]))
            return tsv::report_error(TSV_ERR_ARG, "t_verify[%d] must be > 0", n);
    SequoiaDP dp;
    dp.run(accept, K, n_max, d_max);
    double best = -INFINITY;
    int bn = 1, bd = 0;
    for (int n = 1; n <= n_max; ++n)
        for (int d = 0; d <= d_max; ++d) {
            const double e = dp.f(n, d < dp.D ? d : dp.D);
            if (e == -INFINITY) continue;
            const double s = e * t_verify[1] / (t_verify[n] + d * t_draft);
            if (s > best) {
                best = s;
                bn = n;
                bd = d;
            }
        }
    *n_best = bn;
    *d_best = bd;
    *speedup = best;
    return TSV_OK;
}

tsv_status tsv_sequoia_accept_counts(const int32_t* parent, const int32_t* accepted_nodes, const int32_t* accept_len,
                                     int B, int N, int K, int64_t* reached, int64_t* accepted) {
    if (!parent || !accepted_nodes || !accept_len || !reached || !accepted)
        return tsv::report_error(TSV_ERR_ARG, "null pointer");
    if (B < 0 || N < 1 || N > kMaxTreeNodes || K < 1)
        return tsv::report_error(TSV_ERR_ARG, "bad sizes B=%d N=%d K=%d", B, N, K);
    std::vector<int> nkids(N), rank(N);
    for (int b = 0; b < B; ++b) {
        const int A = accept_len[b];
        if (A < 0) continue;
        const int32_t* par = parent + (size_t)b * N;
        const int32_t* path = accepted_nodes + (size_t)b * N;
        if (par[0] != -1) return tsv::report_error(TSV_ERR_ARG, "sequence %d: parent[0] != -1", b);
        std::fill(nkids.begin(), nkids.end(), 0);
        for (int i = 1; i < N; ++i) {
            if (par[i] < 0 || par[i] >= i) return tsv::report_error(TSV_ERR_ARG, "sequence %d: bad parent[%d]", b, i);
            rank[i] = ++nkids[par[i]];  // children in index order: the order the walk tries them
        }
        if (A >= N || path[0] != 0) return tsv::report_error(TSV_ERR_ARG, "sequence %d: bad accepted path", b);
        for (int j = 0; j <= A; ++j) {
            const int v = path[j];
            for (int k = 0; k < nkids[v] && k < K; ++k) ++reached[k];
            if (j < A) {
                const int c = path[j + 1];
                if (c <= 0 || c >= N || par[c] != v)
                    return tsv::report_error(TSV_ERR_ARG, "sequence %d: accepted path leaves the tree", b);
                if (rank[c] <= K) ++accepted[rank[c] - 1];
            }
        }
    }
    return TSV_OK;
}

}  // extern "C"
