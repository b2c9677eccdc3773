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
//    d) -> (a, c), (b, d) or (a, d), (b, c)) while a swap lowers the cost,
//    then an iterated local search (re-pair a few random pairs, descend
//    again, keep what is cheaper).
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

// cost of every row pair of a tile: popcount(act[a] | act[b]), computed once
struct PairCosts {
    int H;
    std::vector<uint8_t> c;
    PairCosts(const uint64_t* act, int h) : H(h), c((size_t)h * h)
    {
        for (int a = 0; a < H; ++a)
            for (int b = a; b < H; ++b)
                c[(size_t)a * H + b] = c[(size_t)b * H + a] = (uint8_t)popc64(act[a] | act[b]);
    }
    int operator()(int a, int b) const { return c[(size_t)a * H + b]; }
};

int64_t pair_cost(const PairCosts& C, const std::vector<std::pair<int, int>>& P)
{
    int64_t c = 0;
    for (auto& p : P) c += C(p.first, p.second);
    return c;
}

// pair swaps ((a, b), (c, d) -> (a, c), (b, d) or (a, d), (b, c)) that
// involve a pair of the worklist, until none lowers the cost; a pair that
// changes joins the worklist, and a pair x whose scan made a swap scans
// every other pair again (its new partner may now improve with a pair
// checked before the swap).  Started with every pair listed, it ends in a
// grouping where no swap helps; started from such a grouping with only the
// pairs changed since listed, it ends in one again.  Every swap lowers an
// integer cost, so it ends.
void improve_from(const PairCosts& C, std::vector<std::pair<int, int>>& P, std::vector<int>& work)
{
    const int np = (int)P.size();
    std::vector<char> queued(np, 0);
    for (int x : work) queued[x] = 1;
    for (size_t it = 0; it < work.size(); ++it) {
        const int x = work[it];
        queued[x] = 0;
        for (int y = 0; y < np; ++y) {
            if (y == x) continue;
            const int a = P[x].first, b = P[x].second, c = P[y].first, d = P[y].second;
            const int now = C(a, b) + C(c, d);
            const int s1 = C(a, c) + C(b, d);
            const int s2 = C(a, d) + C(b, c);
            if (s1 >= now && s2 >= now) continue;
            if (s1 <= s2) {
                P[x] = {a, c};
                P[y] = {b, d};
            } else {
                P[x] = {a, d};
                P[y] = {b, c};
            }
            if (!queued[y]) {
                queued[y] = 1;
                work.push_back(y);
            }
            y = -1;  // P[x] changed: rescan from the first pair
        }
    }
}

// iterated local search of the pairing heuristic: rounds, pairs re-paired per round
#ifndef BSP_REORDER_ROUNDS
#define BSP_REORDER_ROUNDS 192
#endif
#ifndef BSP_REORDER_KICK
#define BSP_REORDER_KICK 3
#endif

int64_t solve_pairs(const uint64_t* act, int H, std::vector<std::vector<int>>& groups)
{
    const int h = H / 2;
    const PairCosts C(act, H);
    std::vector<std::pair<int, int>> ident, greedy;
    for (int i = 0; i < h; ++i) ident.push_back({i, h + i});
    std::vector<char> used(H, 0);
    for (int r = 0; r < H; ++r) {
        if (used[r]) continue;
        used[r] = 1;
        int best = -1, bc = 1 << 30;
        for (int q = r + 1; q < H; ++q) {
            if (used[q]) continue;
            if (C(r, q) < bc) {
                bc = C(r, q);
                best = q;
            }
        }
        used[best] = 1;
        greedy.push_back({r, best});
    }
    std::vector<int> all(h);
    for (int i = 0; i < h; ++i) all[i] = i;
    std::vector<int> work = all;
    improve_from(C, ident, work);
    work = all;
    improve_from(C, greedy, work);
    const int64_t ci = pair_cost(C, ident), cg = pair_cost(C, greedy);
    std::vector<std::pair<int, int>> best = cg < ci ? greedy : ident;
    int64_t best_cost = cg < ci ? cg : ci;
    // iterated local search: re-pair the rows of KICK random pairs of the
    // best grouping, descend again from those pairs, keep the result if it
    // is cheaper.  The random source is a fixed-seed xorshift, so the
    // grouping is a function of the tile alone.
    constexpr int ROUNDS = BSP_REORDER_ROUNDS, KICK = BSP_REORDER_KICK;
    if (h > KICK) {
        uint64_t rs = 0x9E3779B97F4A7C15ull;
        auto next = [&rs]() {
            rs ^= rs << 13;
            rs ^= rs >> 7;
            rs ^= rs << 17;
            return rs;
        };
        std::vector<std::pair<int, int>> P;
        for (int round = 0; round < ROUNDS && best_cost > 0; ++round) {
            P = best;
            int pick[KICK], rows[2 * KICK];
            for (int k = 0; k < KICK; ++k) {
                bool fresh;
                do {  // KICK distinct pairs
                    pick[k] = (int)(next() % (uint64_t)h);
                    fresh = true;
                    for (int q = 0; q < k; ++q) fresh = fresh && pick[q] != pick[k];
                } while (!fresh);
                rows[2 * k] = P[pick[k]].first;
                rows[2 * k + 1] = P[pick[k]].second;
            }
            for (int i = 2 * KICK - 1; i > 0; --i) std::swap(rows[i], rows[next() % (uint64_t)(i + 1)]);
            for (int k = 0; k < KICK; ++k) P[pick[k]] = {rows[2 * k], rows[2 * k + 1]};
            work.assign(pick, pick + KICK);
            improve_from(C, P, work);
            const int64_t c = pair_cost(C, P);
            if (c < best_cost) {
                best_cost = c;
                best = P;
            }
        }
    }
    groups.clear();
    for (auto& p : best) groups.push_back({p.first, p.second});
    return best_cost;
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
