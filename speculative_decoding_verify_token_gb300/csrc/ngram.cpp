// Host-side n-gram drafter ("Speculative decoding on Apple Silicon" (mlx-optiq docs),
// section "N-gram lookup: any model"): when the last tokens of a sequence occurred earlier
// in it, draft the tokens that followed that earlier occurrence.
//
// The rule: for match lengths m from max_match down to min_match (at most n - 1), take the
// most recent earlier occurrence of the context's last m tokens -- the largest start
// s <= n - m - 1 with ctx[s, s + m) == ctx[n - m, n) -- and draft ctx[s + m, s + m + n_draft)
// (never empty, since s + m <= n - 1); no occurrence at any length drafts nothing.
//
// An index per match length maps each m-gram (its tokens, compared exactly) to its two most
// recent starts, updated as committed tokens are appended, so a draft costs one lookup per
// length instead of a scan of the context.  The suffix itself is always the most recent
// occurrence of its m-gram, so the answer is the second most recent.
#include <algorithm>
#include <array>
#include <cstdint>
#include <cmath>
#include <cstring>
#include <new>
#include <unordered_map>
#include <vector>

#include "host_util.h"
#include "specverify.h"

namespace sv {

constexpr int NG_MAX = SPEC_NGRAM_MAX_MATCH;

struct Gram {
    std::array<int32_t, NG_MAX> t{};
    bool operator==(const Gram& o) const { return t == o.t; }
};

struct GramHash {
    size_t operator()(const Gram& g) const {
        uint64_t h = 0x9e3779b97f4a7c15ull;
        for (int32_t x : g.t) {
            h ^= static_cast<uint32_t>(x);
            h *= 0xff51afd7ed558ccdull;
            h ^= h >> 32;
        }
        return static_cast<size_t>(h);
    }
};

struct Starts {
    int last = -1;   // most recent start
    int prev = -1;   // the one before it
};

}  // namespace sv

struct spec_ngram {
    int min_match = 3, max_match = 8;
    std::vector<int32_t> ctx;
    std::unordered_map<sv::Gram, sv::Starts, sv::GramHash> idx[sv::NG_MAX + 1];

    sv::Gram gram(int start, int m) const {
        sv::Gram g;
        std::memcpy(g.t.data(), ctx.data() + start, sizeof(int32_t) * m);
        return g;   // unused tail stays 0; the index is per length, so keys never mix lengths
    }

    void push(int32_t tok) {
        ctx.push_back(tok);
        const int n = static_cast<int>(ctx.size());
        for (int m = min_match; m <= max_match && m <= n; ++m) {
            sv::Starts& s = idx[m][gram(n - m, m)];
            s.prev = s.last;
            s.last = n - m;
        }
    }

    int draft(int n_draft, int32_t* out) const {
        const int n = static_cast<int>(ctx.size());
        for (int m = std::min(max_match, n - 1); m >= min_match; --m) {
            auto it = idx[m].find(gram(n - m, m));
            if (it == idx[m].end()) continue;
            const int s = it->second.last == n - m ? it->second.prev : it->second.last;
            if (s < 0) continue;
            int c = 0;
            for (int i = s + m; i < n && c < n_draft; ++i) out[c++] = ctx[i];
            return c;
        }
        return 0;
    }
};

using sv::set_error;

extern "C" int spec_ngram_create(int min_match, int max_match, spec_ngram** out) {
    sv::clear_error();
    if (out == nullptr) return set_error(SPEC_E_INVAL, "out is NULL");
    *out = nullptr;
    if (min_match < 1 || max_match < min_match || max_match > sv::NG_MAX)
        return set_error(SPEC_E_INVAL, "need 1 <= min_match (%d) <= max_match (%d) <= %d", min_match, max_match,
                         sv::NG_MAX);
    spec_ngram* g = new (std::nothrow) spec_ngram();
    if (g == nullptr) return set_error(SPEC_E_NOMEM, "spec_ngram allocation failed");
    g->min_match = min_match;
    g->max_match = max_match;
    *out = g;
    return SPEC_OK;
}

extern "C" int spec_ngram_append(spec_ngram* g, const int32_t* tokens, int n) {
    sv::clear_error();
    if (g == nullptr || (n > 0 && tokens == nullptr)) return set_error(SPEC_E_INVAL, "NULL argument");
    if (n < 0) return set_error(SPEC_E_INVAL, "n = %d < 0", n);
    try {
        g->ctx.reserve(g->ctx.size() + n);
        for (int i = 0; i < n; ++i) g->push(tokens[i]);
    } catch (const std::bad_alloc&) {
        return set_error(SPEC_E_NOMEM, "spec_ngram index allocation failed");
    }
    return SPEC_OK;
}

extern "C" int spec_ngram_draft(const spec_ngram* g, int n_draft, int32_t* out) {
    sv::clear_error();
    if (g == nullptr || (n_draft > 0 && out == nullptr)) return set_error(SPEC_E_INVAL, "NULL argument");
    if (n_draft < 0) return set_error(SPEC_E_INVAL, "n_draft = %d < 0", n_draft);
    return g->draft(n_draft, out);
}

extern "C" int spec_ngram_draft_batch(spec_ngram* const* g, int B, int K, int32_t* out_tokens, int32_t* out_len) {
    sv::clear_error();
    if (g == nullptr || out_tokens == nullptr || out_len == nullptr || B < 0 || K < 0)
        return set_error(SPEC_E_INVAL, "bad argument");
    for (int b = 0; b < B; ++b) {
        if (g[b] == nullptr) return set_error(SPEC_E_INVAL, "drafter %d is NULL", b);
        int32_t* row = out_tokens + static_cast<size_t>(b) * K;
        const int c = g[b]->draft(K, row);
        for (int i = c; i < K; ++i) row[i] = 0;
        out_len[b] = c;
    }
    return SPEC_OK;
}

extern "C" int spec_ngram_length(const spec_ngram* g) {
    return g == nullptr ? SPEC_E_INVAL : static_cast<int>(g->ctx.size());
}

extern "C" void spec_ngram_destroy(spec_ngram* g) { delete g; }

// ---- draft-length gate ------------------------------------------------------------------
//
// [OptiQ] "N-gram lookup: any model": the server times a verification pass per model, then
// picks how many tokens to draft each step from how often recent drafts were accepted,
// drafting long while text is copied and not at all during new prose.  Reading: the
// acceptance of a drafted token is alpha = (S + 1) / (S + F + 2), with S the accepted draft
// tokens and F the first rejections of recent rounds, both decayed by `decay` every round
// (so that after rounds without drafts alpha drifts back to 1/2 and drafting is tried
// again); a round with n drafts is expected to emit E(n) = 1 + alpha + ... + alpha^n tokens
// at the timed cost cost[n], and the gate drafts the n <= min(n_max, available) that
// maximises E(n) / cost[n] (the smaller n on ties).

struct spec_ngram_gate {
    int n_max = 0;
    std::vector<double> cost;
    double decay = 0.9;
    double S = 0.0, F = 0.0;

    double alpha() const { return (S + 1.0) / (S + F + 2.0); }

    int choose(int available) const {
        const int lim = std::max(0, std::min(n_max, available));
        const double a = alpha();
        double e = 1.0, pw = 1.0;
        int best = 0;
        double best_v = e / cost[0];
        for (int n = 1; n <= lim; ++n) {
            pw *= a;
            e += pw;
            const double v = e / cost[n];
            if (v > best_v) {
                best_v = v;
                best = n;
            }
        }
        return best;
    }

    void update(int drafted, int accepted) {
        S *= decay;
        F *= decay;
        if (drafted > 0) {
            S += accepted;
            if (accepted < drafted) F += 1.0;
        }
    }
};

extern "C" int spec_ngram_gate_create(int n_max, const double* cost, double decay, spec_ngram_gate** out) {
    sv::clear_error();
    if (out == nullptr || cost == nullptr) return set_error(SPEC_E_INVAL, "NULL argument");
    *out = nullptr;
    if (n_max < 0 || n_max > 1024) return set_error(SPEC_E_INVAL, "n_max = %d outside [0, 1024]", n_max);
    if (!(decay >= 0.0 && decay <= 1.0)) return set_error(SPEC_E_INVAL, "decay must be in [0, 1]");
    for (int n = 0; n <= n_max; ++n)
        if (!(cost[n] > 0.0) || std::isinf(cost[n])) return set_error(SPEC_E_INVAL, "cost[%d] must be finite and > 0", n);
    spec_ngram_gate* g = new (std::nothrow) spec_ngram_gate();
    if (g == nullptr) return set_error(SPEC_E_NOMEM, "spec_ngram_gate allocation failed");
    g->n_max = n_max;
    g->cost.assign(cost, cost + n_max + 1);
    g->decay = decay;
    *out = g;
    return SPEC_OK;
}

extern "C" int spec_ngram_gate_choose(const spec_ngram_gate* g, int available) {
    sv::clear_error();
    if (g == nullptr) return set_error(SPEC_E_INVAL, "gate is NULL");
    return g->choose(available);
}

extern "C" int spec_ngram_gate_update(spec_ngram_gate* g, int drafted, int accepted) {
    sv::clear_error();
    if (g == nullptr) return set_error(SPEC_E_INVAL, "gate is NULL");
    if (drafted < 0 || accepted < 0 || accepted > drafted)
        return set_error(SPEC_E_INVAL, "need 0 <= accepted (%d) <= drafted (%d)", accepted, drafted);
    g->update(drafted, accepted);
    return SPEC_OK;
}

extern "C" double spec_ngram_gate_acceptance(const spec_ngram_gate* g) { return g ? g->alpha() : -1.0; }

extern "C" void spec_ngram_gate_destroy(spec_ngram_gate* g) { delete g; }
