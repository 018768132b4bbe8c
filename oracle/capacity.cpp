// Capacity stage of the MoE-FFN layer -- test infrastructure only.
//
//   capacity  C = floor( floor(k N / E) * alpha )          [P1] §3.1 formula (reading R2);
//             [P1] §5.3 works N=32, E=64, k=2, alpha=1.2 to C = 1
//   alpha     1 + 0.5 log2(N / 256)                         [P1] §3.1 (batch-dependent factor)
//   drop      each expert keeps its first C assignments in ascending token
//             order, whatever their slot; the rest are dropped  [P1] §4.2 code (reading R3)
//   reroute   overflow goes to the next-best unfilled expert [P1] §3.1 (reading R4):
//             in rounds, every pending slot proposes the best-ranked expert that
//             was not full when the round began and that its token neither
//             holds nor proposed earlier in the round (slots in order); each
//             expert accepts proposals in ascending (token, slot) order while it
//             has room; a slot with no such expert is dropped.  A rerouted slot
//             keeps its gate.  Inside an expert, primary assignments come first
//             (token order), then reroutes in (round, token, slot) order.
#include <cmath>
#include <vector>

#include "internal.hpp"

extern "C" {

double orc_alpha_for_batch(int64_t n_tokens) {
    return 1.0 + 0.5 * std::log2(static_cast<double>(n_tokens) / 256.0);
}

int64_t orc_capacity(int64_t n_tokens, int32_t E, int32_t k, double alpha) {
    const int64_t fair = (static_cast<int64_t>(k) * n_tokens) / E;
    return static_cast<int64_t>(std::floor(static_cast<double>(fair) * alpha));
}

int orc_dispatch(int32_t N, int32_t E, int32_t k, int32_t cap_mode, int64_t cap,
                 const int32_t* idx, const float* key, orc_dispatch_out* o) {
    if (cap_mode < 0 || cap_mode > 2 || (cap_mode == 2 && key == nullptr)) return -1;
    const bool limited = cap_mode != 0;
    int32_t* final_idx = o->final_idx;
    for (int64_t i = 0; i < static_cast<int64_t>(N) * k; ++i) final_idx[i] = idx[i];

    // primary assignments: the tokens of each expert in ascending order, the
    // first C kept
    std::vector<std::vector<int32_t>> members(E);
    int64_t n_dropped = 0;
    for (int32_t e = 0; e < E; ++e) {
        for (int32_t t = 0; t < N; ++t) {
            for (int32_t j = 0; j < k; ++j) {
                if (idx[static_cast<int64_t>(t) * k + j] != e) continue;
                if (!limited || static_cast<int64_t>(members[e].size()) < cap) {
                    members[e].push_back(t);
                } else {
                    final_idx[static_cast<int64_t>(t) * k + j] = -1;
                    ++n_dropped;
                }
            }
        }
    }

    int64_t n_rerouted = 0, rounds = 0;
    if (cap_mode == 2) {
        n_dropped = 0;        // counted below: slots that find no expert
        std::vector<int64_t> fill(E);
        for (int32_t e = 0; e < E; ++e) fill[e] = static_cast<int64_t>(members[e].size());
        std::vector<std::pair<int32_t, int32_t>> pending;        // (t, j) ascending
        for (int32_t t = 0; t < N; ++t)
            for (int32_t j = 0; j < k; ++j)
                if (final_idx[static_cast<int64_t>(t) * k + j] < 0) pending.push_back({t, j});
        while (!pending.empty()) {
            ++rounds;
            std::vector<char> full(E);
            for (int32_t e = 0; e < E; ++e) full[e] = fill[e] >= cap;    // start of the round
            std::vector<std::pair<std::pair<int32_t, int32_t>, int32_t>> proposals;
            std::vector<int32_t> proposed_here;         // experts proposed by the current token
            int32_t current = -1;
            for (const auto& tj : pending) {
                const int32_t t = tj.first;
                if (t != current) { current = t; proposed_here.clear(); }
                const float* kt = key + static_cast<int64_t>(t) * E;
                int32_t choice = -1;
                for (int32_t e = 0; e < E; ++e) {
                    if (full[e]) continue;
                    bool taken = false;
                    for (int32_t jj = 0; jj < k; ++jj)
                        if (final_idx[static_cast<int64_t>(t) * k + jj] == e) taken = true;
                    for (int32_t q : proposed_here)
                        if (q == e) taken = true;
                    if (taken) continue;
                    if (choice < 0 || kt[e] > kt[choice]) choice = e;   // ties: lower index
                }
                if (choice < 0) { ++n_dropped; continue; }               // stays dropped
                proposed_here.push_back(choice);
                proposals.push_back({tj, choice});
            }
            std::vector<std::pair<int32_t, int32_t>> still;
            for (const auto& pr : proposals) {                            // (t, j) order
                const int32_t e = pr.second;
                if (fill[e] < cap) {
                    final_idx[static_cast<int64_t>(pr.first.first) * k + pr.first.second] = e;
                    members[e].push_back(pr.first.first);
                    ++fill[e];
                    ++n_rerouted;
                } else {
                    still.push_back(pr.first);
                }
            }
            pending.swap(still);
        }
    }

    int32_t row = 0;
    for (int32_t e = 0; e < E; ++e) {
        o->member_start[e] = row;
        for (int32_t t : members[e]) o->members[row++] = t;
    }
    o->member_start[E] = row;
    o->n_dropped = n_dropped;
    o->n_rerouted = n_rerouted;
    o->rounds = rounds;
    return 0;
}

}  // extern "C"
