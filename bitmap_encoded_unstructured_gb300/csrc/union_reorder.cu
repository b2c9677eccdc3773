// Bitmap-aware row reordering for IE-BME ("UnionSparse", sections "Grouped
// Cost Formulation" and "Grouped Subset Dynamic Programming"): host code,
// offline.
//
// The rows of a local tile are partitioned into groups of R_A rows (one
// group per logical row of the union mask); a group's cost is the number of
// grouped columns in which one of its rows has a nonzero (the union-mask
// entries the group activates).  Two solvers of the same objective:
//  - the page's subset DP: F(S) over the set S of rows not yet grouped,
//    F(empty) = 0, F(S) = min over the groups g of size R_A that contain the
//    smallest row of S of cost(g) + F(S \ g), groups enumerated in
//    lexicographic order and the first minimum kept.  2^H states: used for
//    H <= 20 rows.
//  - for the 64-row tiles of the union format with R_A = 2 (a minimum-cost
//    pairing, where the DP's 2^64 states are out of reach): the better of
//    the identity pairing and a greedy pairing (the smallest free row with
//    its cheapest free partner), each improved by pair swaps ((a, b), (c,
//    d) -> (a, c), (b, d) or (a, d), (b, c)) while a swap lowers the cost.
// Either result is made canonical as on the page: rows ascending inside a
// group, groups in lexicographic order, and the permutation taken
// partition-wise (the p-th row of every group, for p = 0 .. R_A - 1).
#include "bsp_internal.cuh"

#include <algorithm>
#include <cstdint>
#include <vector>

namespace {

int popc64(uint64_t x) { return __builtin_popcountll(x); }

// the page's subset DP; act[r] = grouped activity of row r (bit j = grouped
// column j); groups of RA rows
int64_t solve_dp(const uint64_t* act, int H, int RA, std::vector<std::vector<int>>& groups)
{
    const uint32_t full = (1u << H) - 1u;  // H <= 20
    std::vector<int64_t> F((size_t)full + 1, -1);
    std::vector<uint32_t> choice((size_t)full + 1, 0);  // chosen group as a row mask
    F[0] = 0;
    // states by increasing popcount: every proper subset is solved first
    std::vector<uint32_t> states;
    for (uint32_t S = 1; S <= full; ++S)
        if (__builtin_popcount(S) % RA == 0) states.push_back(S);
    std::stable_sort(states.begin(), states.end(),
                     [](uint32_t x, uint32_t y) { return __builtin_popcount(x) < __builtin_popcount(y); });
    std::vector<int> rows;
    std::vector<int> idx;
    for (uint32_t S : states) {
        rows.clear();
        for (int r = 0; r < H; ++r)
            if ((S >> r) & 1u) rows.push_back(r);
        const int r0 = rows[0];
        const int n = (int)rows.size() - 1;
        // combinations of RA - 1 of rows[1..n] in lexicographic order
        idx.assign(RA - 1, 0);
        for (int k = 0; k < RA - 1; ++k) idx[k] = k;
        int64_t best = -1;
        uint32_t bestg = 0;
        while (true) {
            uint64_t a = act[r0];
            uint32_t g = 1u << r0;
            for (int k = 0; k < RA - 1; ++k) {
                a |= act[rows[1 + idx[k]]];
                g |= 1u << rows[1 + idx[k]];
            }
            const int64_t c = popc64(a) + F[S & ~g];
            if (best < 0 || c < best) {
                best = c;
                bestg = g;
            }
            int k = RA - 2;
            while (k >= 0 && idx[k] == n - (RA - 1) + k) --k;
            if (k < 0) break;
            ++idx[k];
            for (int l = k + 1; l < RA - 1; ++l) idx[l] = idx[l - 1] + 1;
        }
        F[S] = best;
        choice[S] = bestg;
    }
    groups.clear();
    for (uint32_t S = full; S;) {
        std::vector<int> g;
        for (int r = 0; r < H; ++r)
            if ((choice[S] >> r) & 1u) g.push_back(r);
        groups.push_back(g);
        S &= ~choice[S];
    }
    return F[full];
}

int64_t pair_cost(const uint64_t* act, const std::vector<std::pair<int, int>>& P)
{
    int64_t c = 0;
    for (auto& p : P) c += popc64(act[p.first] | act[p.second]);
    return c;
}

// pair swaps while one lowers the cost
void improve_pairs(const uint64_t* act, std::vector<std::pair<int, int>>& P)
{
    const int np = (int)P.size();
    for (int pass = 0; pass < 4 * np; ++pass) {
        bool changed = false;
        for (int x = 0; x < np; ++x)
            for (int y = x + 1; y < np; ++y) {
                const int a = P[x].first, b = P[x].second, c = P[y].first, d = P[y].second;
                const int now = popc64(act[a] | act[b]) + popc64(act[c] | act[d]);
                const int s1 = popc64(act[a] | act[c]) + popc64(act[b] | act[d]);
                const int s2 = popc64(act[a] | act[d]) + popc64(act[b] | act[c]);
                if (s1 < now && s1 <= s2) {
                    P[x] = {a, c};
                    P[y] = {b, d};
                    changed = true;
                } else if (s2 < now) {
                    P[x] = {a, d};
                    P[y] = {b, c};
                    changed = true;
                }
            }
        if (!changed) break;
    }
}

int64_t solve_pairs(const uint64_t* act, int H, std::vector<std::vector<int>>& groups)
{
    const int h = H / 2;
    std::vector<std::pair<int, int>> ident, greedy;
    for (int i = 0; i < h; ++i) ident.push_back({i, h + i});
    std::vector<char> used(H, 0);
    for (int r = 0; r < H; ++r) {
        if (used[r]) continue;
        used[r] = 1;
        int best = -1, bc = 1 << 30;
        for (int q = r + 1; q < H; ++q) {
            if (used[q]) continue;
            const int c = popc64(act[r] | act[q]);
            if (c < bc) {
                bc = c;
                best = q;
            }
        }
        used[best] = 1;
        greedy.push_back({r, best});
    }
    improve_pairs(act, ident);
    improve_pairs(act, greedy);
    const int64_t ci = pair_cost(act, ident), cg = pair_cost(act, greedy);
    const auto& P = cg < ci ? greedy : ident;
    groups.clear();
    for (auto& p : P) groups.push_back({p.first, p.second});
    return cg < ci ? cg : ci;
}

}  // namespace

int64_t bsp_reorder_rows_act(const uint64_t* act, int H, int RA, int exact, int32_t* perm)
{
    std::vector<std::vector<int>> groups;
    const int64_t cost = exact ? solve_dp(act, H, RA, groups) : solve_pairs(act, H, groups);
    for (auto& g : groups) std::sort(g.begin(), g.end());
    std::sort(groups.begin(), groups.end());
    int k = 0;
    for (int p = 0; p < RA; ++p)
        for (auto& g : groups) perm[k++] = g[p];
    return cost;
}

extern "C" bsp_status_t bsp_reorder_rows(const int8_t* tile, int H, int KL, int RA, int CA, int exact,
                                         int32_t* perm, int64_t* cost)
{
    if (!tile || !perm || !cost || H < 1 || KL < 1 || RA < 1 || CA < 1) return BSP_ERR_INVALID_ARG;
    if (H % RA || KL % CA || KL / CA > 64) return BSP_ERR_SHAPE;
    if (exact ? H > 20 : (RA != 2)) return BSP_ERR_SHAPE;
    const int w = KL / CA;
    std::vector<uint64_t> act(H, 0);
    for (int r = 0; r < H; ++r)
        for (int ca = 0; ca < CA; ++ca)
            for (int j = 0; j < w; ++j)
                if (tile[(int64_t)r * KL + ca * w + j] != 0) act[r] |= 1ull << j;
    *cost = bsp_reorder_rows_act(act.data(), H, RA, exact, perm);
    return BSP_OK;
}
