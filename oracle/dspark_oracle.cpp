// ORACLE - test infrastructure, not product code.
//
// Plain single-threaded CPU statement of what the DSpark sampling / verify /
// statistics path computes, in double precision, written for a reader to check
// against the pages by eye: no blocking, fusion or reordering beyond what the
// definitions state.  Only the test suite, the smoke check and the benchmark's
// CPU-baseline leg load this library.  It shares no code with the CUDA library.
//
// Sources (page title > section) are listed in dspark_oracle.h; each function
// below names the passage it follows and what pins it in the tests.
//
// Where the pages leave a step open, the reading taken is stated at the step.

#include "dspark_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <numeric>
#include <vector>

namespace {

// Width of the band inside which a floating-point decision (accept test,
// inverse-CDF boundary, top-p cut, near-tie of rounded logits) is reported as
// indeterminate instead of compared exactly.
const double kTol = 1e-5;

double bf16_to_double(uint16_t bits16) {
    uint32_t bits = static_cast<uint32_t>(bits16) << 16;
    float f;
    std::memcpy(&f, &bits, sizeof f);
    return static_cast<double>(f);
}

// Element i of a logit array stored as bf16 (dtype 0) or fp32 (dtype 1).
double load_value(const void* base, int32_t dtype, size_t i) {
    if (dtype == 0) return bf16_to_double(static_cast<const uint16_t*>(base)[i]);
    return static_cast<double>(static_cast<const float*>(base)[i]);
}

bool is_bad_logit(double z) {  // NaN or +inf; -inf is a legal "masked" logit
    return std::isnan(z) || z == std::numeric_limits<double>::infinity();
}

}  // namespace

// ---------------------------------------------------------------------------
// Philox-4x32-10 [SMDS, section 3.3 "Philox"].  The 128-bit counter is four
// 32-bit words; each of the ten rounds multiplies words 0 and 2 by the two
// round multipliers, xors the high halves of the products with the other two
// words and the two key words, and permutes; the key is advanced by the two
// Weyl increments between rounds.
// Pinned by: an independent implementation of the same published generator
// (triton.language.philox, run in triton's CPU interpreter) on many counters,
// plus uniformity and serial-correlation checks of the derived uniforms.
// ---------------------------------------------------------------------------
extern "C" void orc_philox4x32_10(uint32_t key0, uint32_t key1,
                                  const uint32_t ctr[4], uint32_t out[4]) {
    const uint32_t mult0 = 0xD2511F53u, mult1 = 0xCD9E8D57u;  // round multipliers
    const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;  // key increments
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key0, k1 = key1;
    for (int round = 0; round < 10; ++round) {
        uint64_t prod0 = static_cast<uint64_t>(mult0) * c0;
        uint64_t prod2 = static_cast<uint64_t>(mult1) * c2;
        uint32_t n0 = static_cast<uint32_t>(prod2 >> 32) ^ c1 ^ k0;
        uint32_t n1 = static_cast<uint32_t>(prod2);
        uint32_t n2 = static_cast<uint32_t>(prod0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = static_cast<uint32_t>(prod0);
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += weyl0;
        k1 += weyl1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// The per-decision uniform.  Keying by (seed, request, position, draw) is not
// on the pages; it is the reading that lets CPU and GPU draw identical
// uniforms.  draw 0 = proposal, 1 = accept test, 2 = residual / bonus.
extern "C" double orc_uniform(uint64_t seed, uint64_t request_id, int64_t pos,
                              uint32_t draw) {
    uint64_t upos = static_cast<uint64_t>(pos);
    uint32_t ctr[4] = {draw, static_cast<uint32_t>(upos),
                       static_cast<uint32_t>(upos >> 32),
                       static_cast<uint32_t>(request_id)};
    uint32_t out[4];
    orc_philox4x32_10(static_cast<uint32_t>(seed),
                      static_cast<uint32_t>(seed >> 32), ctr, out);
    return static_cast<double>(out[0] >> 8) * (1.0 / 16777216.0);
}

// ---------------------------------------------------------------------------
// Sampling policy [FT Exact decoding semantics > Probabilistic: p and q are
// "formed after applying the request's temperature, top-p, and top-k policy"].
// Readings (the pages fix no order or tie rule):
//   * greedy: one-hot at the argmax, lowest index on ties; truncation and
//     temperature are irrelevant to it.
//   * order pi: token indices by (logit descending, index ascending), taken
//     from the raw logits so temperature cannot create or merge ties.
//   * top-k (0 < k < V) keeps exactly the first k tokens of pi.
//   * weights s = exp((z - zmax) * (1/T)), 1/T rounded to fp32.
//   * top-p (p < 1) keeps the shortest prefix of pi (inside the top-k set)
//     whose cumulative share of the kept mass is >= p; at least one token.
//   * p = s / sum(s) over the final support, exactly 0 elsewhere.
// Pinned by: T=1 without truncation equals a float64 library softmax; top_k=1
// and top_p->0 give the argmax one-hot; top_k=V is a no-op; the support size
// equals k exactly on rows with forced ties; brute force over tiny V.
// ---------------------------------------------------------------------------
extern "C" int orc_policy_row(const double* z, int V, float temperature,
                              int32_t top_k, float top_p, int32_t greedy,
                              int32_t exact_logits, double* p,
                              int32_t* argmax_out, int32_t* support_size,
                              int32_t* indet) {
    *indet = 0;
    *argmax_out = -1;
    *support_size = 0;
    std::fill(p, p + V, 0.0);

    for (int v = 0; v < V; ++v)
        if (is_bad_logit(z[v])) return ORC_NONFINITE;

    double zmax = -std::numeric_limits<double>::infinity();
    int am = -1;
    for (int v = 0; v < V; ++v) {
        if (z[v] > zmax) { zmax = z[v]; am = v; }   // strict: lowest index wins
    }
    if (am < 0) return ORC_EMPTY;                    // every logit is -inf
    *argmax_out = am;

    if (greedy) {
        if (!exact_logits) {  // rounded logits: a near-tie may flip the argmax
            double second = -std::numeric_limits<double>::infinity();
            for (int v = 0; v < V; ++v)
                if (v != am && z[v] > second) second = z[v];
            if (zmax - second < kTol * std::max(1.0, std::fabs(zmax))) *indet = 1;
        }
        p[am] = 1.0;
        *support_size = 1;
        return ORC_OK;
    }

    if (!(temperature > 0.0f) || std::isinf(temperature) || top_k < 0 ||
        std::isnan(top_p))
        return ORC_BAD_POLICY;

    const bool use_k = top_k > 0 && top_k < V;
    const bool use_p = top_p < 1.0f;
    const double inv_t = static_cast<double>(1.0f / temperature);

    std::vector<int> order(V);
    std::iota(order.begin(), order.end(), 0);
    if (use_k || use_p) {
        std::sort(order.begin(), order.end(), [z](int a, int b) {
            return z[a] > z[b] || (z[a] == z[b] && a < b);
        });
    }
    const int kept = use_k ? top_k : V;

    std::vector<double> s(kept);
    double kept_mass = 0.0;
    for (int i = 0; i < kept; ++i) {
        s[i] = std::exp((z[order[i]] - zmax) * inv_t);
        kept_mass += s[i];
    }

    int m = kept;  // support = order[0 .. m)
    if (use_p) {
        double cum = 0.0;
        for (int i = 0; i < kept; ++i) {
            double before = cum;
            cum += s[i];
            if (cum / kept_mass >= static_cast<double>(top_p)) {
                m = i + 1;
                if (static_cast<double>(top_p) - before / kept_mass < kTol ||
                    cum / kept_mass - static_cast<double>(top_p) < kTol)
                    *indet = 1;
                break;
            }
        }
    }

    if (!exact_logits) {  // rounded logits: order near a cut may differ
        if (use_k) {
            double a = z[order[kept - 1]], b = z[order[kept]];
            if (a - b < kTol * std::max(1.0, std::fabs(a))) *indet = 1;
        }
        if (use_p && m < kept) {
            double a = z[order[m - 1]], b = z[order[m]];
            if (a - b < kTol * std::max(1.0, std::fabs(a))) *indet = 1;
        }
    }

    double mass = 0.0;
    for (int i = 0; i < m; ++i) mass += s[i];
    for (int i = 0; i < m; ++i) p[order[i]] = s[i] / mass;
    *support_size = m;
    return ORC_OK;
}

// ---------------------------------------------------------------------------
// Inverse-CDF draw in token-index order (the index order is a reading; the
// pages only say "sample").  Returns the smallest i with
// sum_{j<=i} w_j > u * S; if round-off leaves none, the last index with
// positive weight.
// Pinned by: brute-force frequency counts on tiny V and exact hand cases.
// ---------------------------------------------------------------------------
extern "C" int32_t orc_sample_index(const double* w, int V, double u,
                                    double* margin) {
    double total = 0.0;
    for (int v = 0; v < V; ++v) total += w[v];
    *margin = 0.0;
    if (!(total > 0.0)) return -1;
    const double target = u * total;
    double cum = 0.0;
    int last_positive = -1;
    for (int v = 0; v < V; ++v) {
        if (!(w[v] > 0.0)) continue;
        double before = cum;
        cum += w[v];
        last_positive = v;
        if (cum > target) {
            *margin = std::min(target - before, cum - target) / total;
            return v;
        }
    }
    return last_positive;
}

// ---------------------------------------------------------------------------
// (a) Markov-head draft sampling.
// [FT Checkpoint-faithful DSpark architecture]: the Markov head runs left to
// right, proposal k conditions on proposal k-1 and the first on the anchor;
// the full q and the confidences are kept.
// [MB Semi-autoregressive draft]: the Markov head is a low-rank
// token-conditioned additive logit bias; the confidence is
// c_k = sigmoid(w^T [h_k ; embed(x_{k-1})]).
// Readings: bias_k[v] = sum_j U[x_{k-1}, j] * Wm[j, v] with Wm stored as
// W[v, j]; the bias and backbone are summed in double and rounded to fp32
// once; "embed" is the draft token embedding E; w has length 2H, no bias term.
// Proposal k draws u at position pos0 + k, draw 0.  Greedy requests take the
// argmax and leave their q rows untouched, q_at_x = 1.
// Pinned by: r = 0 gives bias 0; a one-hot U row gives a W column; the bias
// equals a float64 library matmul; w = 0 gives confidence 1/2; a closed form
// for H = 2.
// ---------------------------------------------------------------------------
extern "C" void orc_markov_sample(
    const void* backbone, int32_t dtype, const int32_t* anchor,
    const uint16_t* U, const uint16_t* W, int32_t r, const void* h,
    int32_t h_dtype, const uint16_t* E, const float* w_conf, int32_t H,
    const float* temperature, const int32_t* top_k, const float* top_p,
    const int32_t* greedy, const uint64_t* seed, const uint64_t* request_id,
    const int64_t* pos0, int32_t B, int32_t gamma, int32_t V,
    int32_t* proposals, float* q, float* q_at_x, float* conf, int32_t* status,
    uint8_t* indet) {
    std::vector<double> z(V), p(V);
    for (int b = 0; b < B; ++b) {
        status[b] = ORC_OK;
        int x_prev = anchor[b];
        if (x_prev < 0 || x_prev >= V) status[b] = ORC_BAD_TOKEN;

        for (int k = 1; k <= gamma; ++k) {
            const size_t idx = static_cast<size_t>(b) * gamma + (k - 1);
            indet[idx] = 0;
            if (status[b] != ORC_OK) {
                proposals[idx] = -1;
                q_at_x[idx] = 0.0f;
                if (conf) conf[idx] = 0.0f;
                continue;
            }

            for (int v = 0; v < V; ++v) {
                double bias = 0.0;
                for (int j = 0; j < r; ++j)
                    bias += bf16_to_double(U[static_cast<size_t>(x_prev) * r + j]) *
                            bf16_to_double(W[static_cast<size_t>(v) * r + j]);
                double sum = load_value(backbone, dtype, idx * V + v) + bias;
                z[v] = static_cast<double>(static_cast<float>(sum));
            }

            if (h && conf) {
                double a = 0.0;
                for (int i = 0; i < H; ++i)
                    a += static_cast<double>(w_conf[i]) *
                         load_value(h, h_dtype, idx * H + i);
                for (int i = 0; i < H; ++i)
                    a += static_cast<double>(w_conf[H + i]) *
                         bf16_to_double(E[static_cast<size_t>(x_prev) * H + i]);
                conf[idx] = static_cast<float>(1.0 / (1.0 + std::exp(-a)));
            }

            int32_t am = -1, support = 0, pind = 0;
            int st = orc_policy_row(z.data(), V, temperature[b], top_k[b],
                                    top_p[b], greedy[b], r == 0 ? 1 : 0,
                                    p.data(), &am, &support, &pind);
            if (st != ORC_OK) {
                status[b] = st;
                proposals[idx] = -1;
                q_at_x[idx] = 0.0f;
                continue;
            }
            int x;
            if (greedy[b]) {
                x = am;
                q_at_x[idx] = 1.0f;
            } else {
                double u = orc_uniform(seed[b], request_id[b], pos0[b] + k, 0);
                double margin = 0.0;
                x = orc_sample_index(p.data(), V, u, &margin);
                if (margin < kTol) pind = 1;
                for (int v = 0; v < V; ++v)
                    q[idx * V + v] = static_cast<float>(p[v]);
                q_at_x[idx] = static_cast<float>(p[x]);
            }
            indet[idx] = static_cast<uint8_t>(pind);
            proposals[idx] = x;
            x_prev = x;
        }
    }
}

// ---------------------------------------------------------------------------
// (a') RNN-head draft sampling.
// [MB Semi-autoregressive draft]: besides the Markov head, DSpark offers an
// RNN head, a GRU-like recurrence that carries prefix state across the block
// and, like the Markov head, adds intra-block dependency on top of the
// parallel backbone logits; at inference it runs serially.  The pages give
// no equations, so every step below is a reading (parity of this function is
// pinned to the GRU's textbook definition and to the Markov / backbone-only
// sampler, not to the pages):
//   * the recurrence is a standard GRU cell (Cho et al., 2014) in the gate
//     layout r, z, n:  r = sigma(Wi_r e + bi_r + Wh_r s + bh_r),
//     z = sigma(Wi_z e + bi_z + Wh_z s + bh_z),
//     n = tanh(Wi_n e + bi_n + r * (Wh_n s + bh_n)),  s' = (1 - z) n + z s;
//   * its input is the rank-r embedding of the previous token, e_k =
//     U[x_{k-1}] (the Markov head's table), x_0 the anchor; its state starts
//     at s_0 = 0 for every block;
//   * its output is a logit bias of the same low-rank form as the Markov
//     head's, bias_k[v] = sum_j s_k[j] * Wm[j, v] with Wm stored as W[v, j],
//     added to the backbone logits; the state is not rounded (the sum is
//     rounded to fp32 once, as in the Markov sampler);
//   * the policy, the draw, q, q_at_x and the confidence are the Markov
//     sampler's.
// Pinned by: the states equal a float64 library GRU cell iterated over the
// proposals; log q against the bias of those states; an update gate held at
// one (the state stays 0) reproduces the backbone-only sampler; a state
// that carries nothing (update gate at zero, no hidden weights) makes the
// bias a function of x_{k-1} alone.
// ---------------------------------------------------------------------------
extern "C" void orc_rnn_sample(
    const void* backbone, int32_t dtype, const int32_t* anchor,
    const uint16_t* U, const uint16_t* W, int32_t r, const uint16_t* Wi,
    const uint16_t* Wh, const float* bi, const float* bh, const void* h,
    int32_t h_dtype, const uint16_t* E, const float* w_conf, int32_t H,
    const float* temperature, const int32_t* top_k, const float* top_p,
    const int32_t* greedy, const uint64_t* seed, const uint64_t* request_id,
    const int64_t* pos0, int32_t B, int32_t gamma, int32_t V,
    int32_t* proposals, float* q, float* q_at_x, float* conf, int32_t* status,
    uint8_t* indet, double* states) {
    std::vector<double> z(V), p(V), s(r), s_next(r), e(r), gi(3 * r), gh(3 * r);
    auto sigmoid = [](double a) { return 1.0 / (1.0 + std::exp(-a)); };
    for (int b = 0; b < B; ++b) {
        status[b] = ORC_OK;
        int x_prev = anchor[b];
        if (x_prev < 0 || x_prev >= V) status[b] = ORC_BAD_TOKEN;
        std::fill(s.begin(), s.end(), 0.0);

        for (int k = 1; k <= gamma; ++k) {
            const size_t idx = static_cast<size_t>(b) * gamma + (k - 1);
            indet[idx] = 0;
            if (status[b] != ORC_OK) {
                proposals[idx] = -1;
                q_at_x[idx] = 0.0f;
                if (conf) conf[idx] = 0.0f;
                if (states)
                    for (int j = 0; j < r; ++j) states[idx * r + j] = 0.0;
                continue;
            }

            // the GRU step on e_k = U[x_{k-1}]
            for (int j = 0; j < r; ++j) e[j] = bf16_to_double(U[static_cast<size_t>(x_prev) * r + j]);
            for (int g = 0; g < 3 * r; ++g) {
                double ai = bi[g], ah = bh[g];
                for (int j = 0; j < r; ++j) {
                    ai += bf16_to_double(Wi[static_cast<size_t>(g) * r + j]) * e[j];
                    ah += bf16_to_double(Wh[static_cast<size_t>(g) * r + j]) * s[j];
                }
                gi[g] = ai;
                gh[g] = ah;
            }
            for (int j = 0; j < r; ++j) {
                const double rg = sigmoid(gi[j] + gh[j]);
                const double ug = sigmoid(gi[r + j] + gh[r + j]);
                const double n = std::tanh(gi[2 * r + j] + rg * gh[2 * r + j]);
                s_next[j] = (1.0 - ug) * n + ug * s[j];
            }
            s.swap(s_next);
            if (states)
                for (int j = 0; j < r; ++j) states[idx * r + j] = s[j];

            for (int v = 0; v < V; ++v) {
                double bias = 0.0;
                for (int j = 0; j < r; ++j)
                    bias += s[j] * bf16_to_double(W[static_cast<size_t>(v) * r + j]);
                double sum = load_value(backbone, dtype, idx * V + v) + bias;
                z[v] = static_cast<double>(static_cast<float>(sum));
            }

            if (h && conf) {
                double a = 0.0;
                for (int i = 0; i < H; ++i)
                    a += static_cast<double>(w_conf[i]) * load_value(h, h_dtype, idx * H + i);
                for (int i = 0; i < H; ++i)
                    a += static_cast<double>(w_conf[H + i]) *
                         bf16_to_double(E[static_cast<size_t>(x_prev) * H + i]);
                conf[idx] = static_cast<float>(sigmoid(a));
            }

            int32_t am = -1, support = 0, pind = 0;
            int st = orc_policy_row(z.data(), V, temperature[b], top_k[b], top_p[b], greedy[b],
                                    r == 0 ? 1 : 0, p.data(), &am, &support, &pind);
            if (st != ORC_OK) {
                status[b] = st;
                proposals[idx] = -1;
                q_at_x[idx] = 0.0f;
                continue;
            }
            int x;
            if (greedy[b]) {
                x = am;
                q_at_x[idx] = 1.0f;
            } else {
                double u = orc_uniform(seed[b], request_id[b], pos0[b] + k, 0);
                double margin = 0.0;
                x = orc_sample_index(p.data(), V, u, &margin);
                if (margin < kTol) pind = 1;
                for (int v = 0; v < V; ++v) q[idx * V + v] = static_cast<float>(p[v]);
                q_at_x[idx] = static_cast<float>(p[x]);
            }
            indet[idx] = static_cast<uint8_t>(pind);
            proposals[idx] = x;
            x_prev = x;
        }
    }
}

// ---------------------------------------------------------------------------
// (b) Exact verify.
// [FT Exact decoding semantics > Greedy]: accept the contiguous prefix of
// proposals equal to the target argmax; at the first disagreement emit the
// target's token; a later match after a rejection is never accepted.
// [FT > Probabilistic]: accept x with probability min(1, p(x)/q(x)); at the
// first rejection sample from normalised max(p - q, 0); if every proposal
// survives, sample a bonus token from the target's next-position distribution.
// [PT Acceptance]: 1 .. gamma+1 emitted tokens per step.
// Readings: target row i scores proposal i+1, row gamma gives the bonus;
// accept iff p > 0 and u < p/q (q = 0 with p > 0 accepts), u drawn at
// pos0 + k, draw 1; the residual / bonus draw is at the emitted token's
// position, draw 2; a residual with zero mass falls back to p.
// Pinned by: identical rows accept all; a k=2 mismatch with a k=3 match
// emits 1 + 1 tokens; p == q accepts all; disjoint supports reject at k = 1
// and resample from p; a chi-square test of the emitted-token law against
// target-only sampling on agreeing, disagreeing and nearly disjoint rows.
// ---------------------------------------------------------------------------
// [FT Scope and limitations, and the review thread]: a later change lets the
// scheduler verify 0..gamma proposals per request, chosen from measured
// draft and verify costs; the choice has no formula on the pages, so the
// width is an input here.
// The verify of each request over its first width[b] proposals (width NULL:
// all gamma).  A request checks proposals 1..g and reads target rows 0..g
// (g = its width); every later row and proposal is ignored.  The bonus comes
// from row g, drawn at position pos0 + g + 1; g = 0 is one target-only draw
// from row 0.  A width outside [0, gamma] is reported as a bad token.
extern "C" void orc_verify_width(const void* target, int32_t dtype,
                                 const int32_t* proposals, const float* q,
                                 const float* q_at_x, const float* temperature,
                                 const int32_t* top_k, const float* top_p,
                                 const int32_t* greedy, const uint64_t* seed,
                                 const uint64_t* request_id, const int64_t* pos0,
                                 int32_t B, int32_t gamma, int32_t V,
                                 const int32_t* width, int32_t* out_tokens,
                                 int32_t* num_accepted, int32_t* status, uint8_t* indet,
                                 int32_t* det_tokens, uint8_t* det_nacc) {
    const int rows = gamma + 1;
    std::vector<double> z(V), w(V);
    std::vector<std::vector<double>> p(rows, std::vector<double>(V));
    std::vector<int32_t> am(rows), row_indet(rows);

    for (int b = 0; b < B; ++b) {
        int32_t* out = out_tokens + static_cast<size_t>(b) * rows;
        const int32_t* x = proposals + static_cast<size_t>(b) * gamma;
        for (int i = 0; i < rows; ++i) out[i] = -1;
        num_accepted[b] = -1;
        status[b] = ORC_OK;
        indet[b] = 0;
        // How much of the request stays exactly comparable: the leading
        // tokens emitted before its first indeterminate decision, and whether
        // num_accepted is decided before it (every output while indet is 0).
        if (det_tokens) det_tokens[b] = rows;
        if (det_nacc) det_nacc[b] = 1;
        auto first_indet = [&](int tokens, bool nacc) {
            if (indet[b]) return;  // only the first one counts
            indet[b] = 1;
            if (det_tokens) det_tokens[b] = tokens;
            if (det_nacc) det_nacc[b] = nacc ? 1 : 0;
        };
        const int g = width ? width[b] : gamma;  // proposals this request verifies
        if (g < 0 || g > gamma) {
            status[b] = ORC_BAD_TOKEN;
            continue;
        }

        for (int k = 0; k < g; ++k)
            if (x[k] < 0 || x[k] >= V) status[b] = ORC_BAD_TOKEN;
        if (status[b] != ORC_OK) continue;

        for (int i = 0; i <= g; ++i) {
            const size_t row = static_cast<size_t>(b) * rows + i;
            for (int v = 0; v < V; ++v) z[v] = load_value(target, dtype, row * V + v);
            int32_t support = 0;
            int st = orc_policy_row(z.data(), V, temperature[b], top_k[b],
                                    top_p[b], greedy[b], 1, p[i].data(), &am[i],
                                    &support, &row_indet[i]);
            if (st != ORC_OK) { status[b] = st; break; }
        }
        if (status[b] != ORC_OK) continue;

        if (greedy[b]) {
            int n = 0;
            while (n < g && x[n] == am[n]) ++n;
            for (int i = 0; i < n; ++i) out[i] = x[i];
            out[n] = am[n];
            num_accepted[b] = n;
            continue;
        }

        int rejected_at = 0;  // 1-based k of the first rejection, 0 = none
        for (int k = 1; k <= g; ++k) {
            const double pk = p[k - 1][x[k - 1]];
            const double qk = q_at_x[static_cast<size_t>(b) * gamma + (k - 1)];
            double ratio;
            if (qk > 0.0) ratio = pk / qk;
            else ratio = pk > 0.0 ? std::numeric_limits<double>::infinity() : 0.0;
            const double u = orc_uniform(seed[b], request_id[b], pos0[b] + k, 1);
            // decision k is indeterminate: x_1..x_{k-1} stay comparable
            if (row_indet[k - 1]) first_indet(k - 1, false);
            if (std::isfinite(ratio) && std::fabs(u - ratio) < kTol) first_indet(k - 1, false);
            const bool accept = pk > 0.0 && u < ratio;
            if (!accept) { rejected_at = k; break; }
        }

        double margin = 0.0;
        int token;
        if (rejected_at > 0) {
            const int j = rejected_at;
            const float* qrow = q + (static_cast<size_t>(b) * gamma + (j - 1)) * V;
            double mass = 0.0;
            for (int v = 0; v < V; ++v) {
                w[v] = std::max(p[j - 1][v] - static_cast<double>(qrow[v]), 0.0);
                mass += w[v];
            }
            if (!(mass > 0.0)) w = p[j - 1];
            const double u = orc_uniform(seed[b], request_id[b], pos0[b] + j, 2);
            token = orc_sample_index(w.data(), V, u, &margin);
            for (int i = 0; i < j - 1; ++i) out[i] = x[i];
            out[j - 1] = token;
            num_accepted[b] = j - 1;
            if (margin < kTol) first_indet(j - 1, true);  // only the drawn token
        } else {
            if (row_indet[g]) first_indet(g, true);
            const double u = orc_uniform(seed[b], request_id[b], pos0[b] + g + 1, 2);
            token = orc_sample_index(p[g].data(), V, u, &margin);
            for (int i = 0; i < g; ++i) out[i] = x[i];
            out[g] = token;
            num_accepted[b] = g;
            if (margin < kTol) first_indet(g, true);
        }
    }
}

extern "C" void orc_verify(const void* target, int32_t dtype,
                           const int32_t* proposals, const float* q,
                           const float* q_at_x, const float* temperature,
                           const int32_t* top_k, const float* top_p,
                           const int32_t* greedy, const uint64_t* seed,
                           const uint64_t* request_id, const int64_t* pos0,
                           int32_t B, int32_t gamma, int32_t V,
                           int32_t* out_tokens, int32_t* num_accepted,
                           int32_t* status, uint8_t* indet, int32_t* det_tokens, uint8_t* det_nacc) {
    orc_verify_width(target, dtype, proposals, q, q_at_x, temperature, top_k, top_p, greedy, seed,
                     request_id, pos0, B, gamma, V, nullptr, out_tokens, num_accepted, status, indet,
                     det_tokens, det_nacc);
}

// ---------------------------------------------------------------------------
// (c) Analytical acceptance statistics.
// [MB Training objective]: position weights exp(-k/gamma); L_ce (0.1) is the
// cross-entropy of the draft logits against the target's teacher-forced next
// tokens; L_l1 (0.9) is the raw ||p_draft - p_target||_1; L_conf (1.0) is the
// BCE of the confidence against the acceptance label.
// [MB Acceptance and confidence]: accept_rate = clamp(1 - 0.5 L1, 0, 1);
// tau = sum_k cumprod(accept_rate)_k + 1.
// [MB Loss return contract]: numerators and a token count, never ratios.
// Readings: k = 1..gamma; the teacher tokens are an explicit labels input;
// a block's status is the largest code of its positions (a label outside
// [0, V) outranks a non-finite logit);
// the confidence enters as a logit z and BCE = softplus(z) - accept * z in
// its stable form; the label is the clamped accept_rate; num_tokens counts
// mask = 1 positions; l1 / accept / tau are reported for every position.
// Pinned by: disjoint one-hot rows give L1 = 2, accept 0, tau 1; identical
// rows give L1 = 0, accept 1, tau = gamma + 1; two-point rows give
// L1 = 2|a - b|; a one-hot draft has CE 0; BCE closed forms at accept 0 / 1;
// the weights sum to a geometric series.
// ---------------------------------------------------------------------------
extern "C" void orc_accept_stats(const void* draft, const void* target,
                                 int32_t dtype, const int32_t* labels,
                                 const float* conf_logits, const uint8_t* mask,
                                 int32_t N, int32_t gamma, int32_t V, float* l1,
                                 float* accept, float* tau, double* loss_num,
                                 double* report, int64_t* num_tokens,
                                 int32_t* status) {
    std::vector<double> d(V), t(V);
    double ce_sum = 0.0, l1_sum = 0.0, bce_sum = 0.0, acc_sum = 0.0, tau_sum = 0.0;
    int64_t count = 0;
    const double nan = std::numeric_limits<double>::quiet_NaN();

    for (int n = 0; n < N; ++n) {
        int st = ORC_OK;
        double survive = 1.0, tau_n = 1.0;
        for (int k = 1; k <= gamma; ++k) {
            const size_t idx = static_cast<size_t>(n) * gamma + (k - 1);
            double dmax = -std::numeric_limits<double>::infinity(), tmax = dmax;
            for (int v = 0; v < V; ++v) {
                d[v] = load_value(draft, dtype, idx * V + v);
                t[v] = load_value(target, dtype, idx * V + v);
                if (is_bad_logit(d[v]) || is_bad_logit(t[v])) st = std::max(st, static_cast<int>(ORC_NONFINITE));
                dmax = std::max(dmax, d[v]);
                tmax = std::max(tmax, t[v]);
            }
            double dsum = 0.0, tsum = 0.0;
            for (int v = 0; v < V; ++v) {
                dsum += std::exp(d[v] - dmax);
                tsum += std::exp(t[v] - tmax);
            }
            double dist = 0.0;
            for (int v = 0; v < V; ++v)
                dist += std::fabs(std::exp(d[v] - dmax) / dsum -
                                  std::exp(t[v] - tmax) / tsum);
            const double acc = std::min(1.0, std::max(0.0, 1.0 - 0.5 * dist));

            const int y = labels[idx];
            double ce;
            if (y < 0 || y >= V) { st = std::max(st, static_cast<int>(ORC_BAD_TOKEN)); ce = nan; }
            else ce = dmax + std::log(dsum) - d[y];

            const double zc = conf_logits[idx];
            const double bce = std::max(zc, 0.0) - acc * zc + std::log1p(std::exp(-std::fabs(zc)));
            const double wk = std::exp(-static_cast<double>(k) / gamma);

            l1[idx] = static_cast<float>(dist);
            accept[idx] = static_cast<float>(acc);
            survive *= acc;
            tau_n += survive;

            const bool m = mask ? mask[idx] != 0 : true;
            if (m) {
                ce_sum += wk * ce;
                l1_sum += wk * dist;
                bce_sum += wk * bce;
                acc_sum += acc;
                ++count;
            }
        }
        tau[n] = static_cast<float>(tau_n);
        tau_sum += tau_n;
        if (status) status[n] = st;
    }
    loss_num[0] = ce_sum;
    loss_num[1] = l1_sum;
    loss_num[2] = bce_sum;
    loss_num[3] = 0.1 * ce_sum + 0.9 * l1_sum + 1.0 * bce_sum;
    report[0] = acc_sum;
    report[1] = tau_sum;
    *num_tokens = count;
}

// Gradient of the loss numerator's total J = sum m w_k (0.1 CE + 0.9 L1 +
// 1.0 BCE) [MB Training objective; Acceptance and confidence; Memory contract
// for the full-vocabulary terms], the target the frozen teacher and the BCE
// label accept detached, times scale:
//   dJ/dd_u = m w_k (0.1 (p_d,u - [u = y]) + 0.9 p_d,u (s_u - sum_v s_v p_d,v)),
//   s_v = sign(p_d,v - p_t,v) (0 at equality),
//   dJ/dz_c = m w_k (sigmoid(z_c) - accept).
// Masked positions get 0; a position with a NaN / +inf logit or a label
// outside [0, V) (and mask 1) gets NaN in its whole draft gradient row.
extern "C" void orc_accept_stats_backward(const void* draft, const void* target,
                                          int32_t dtype, const int32_t* labels,
                                          const float* conf_logits, const uint8_t* mask,
                                          int32_t N, int32_t gamma, int32_t V, double scale,
                                          float* grad_draft, float* grad_conf) {
    std::vector<double> d(V), t(V), pd(V), pt(V);
    const double nan = std::numeric_limits<double>::quiet_NaN();
    for (int n = 0; n < N; ++n) {
        for (int k = 1; k <= gamma; ++k) {
            const size_t idx = static_cast<size_t>(n) * gamma + (k - 1);
            float* g = grad_draft + idx * V;
            const bool m = mask ? mask[idx] != 0 : true;
            if (!m) {
                for (int v = 0; v < V; ++v) g[v] = 0.0f;
                grad_conf[idx] = 0.0f;
                continue;
            }
            bool bad = false;
            double dmax = -std::numeric_limits<double>::infinity(), tmax = dmax;
            for (int v = 0; v < V; ++v) {
                d[v] = load_value(draft, dtype, idx * V + v);
                t[v] = load_value(target, dtype, idx * V + v);
                if (is_bad_logit(d[v]) || is_bad_logit(t[v])) bad = true;
                dmax = std::max(dmax, d[v]);
                tmax = std::max(tmax, t[v]);
            }
            const int y = labels[idx];
            if (y < 0 || y >= V) bad = true;
            const double zc = conf_logits[idx];
            const double c = scale * std::exp(-static_cast<double>(k) / gamma);
            if (bad) {
                for (int v = 0; v < V; ++v) g[v] = static_cast<float>(nan);
                grad_conf[idx] = static_cast<float>(nan);
                continue;
            }
            double dsum = 0.0, tsum = 0.0;
            for (int v = 0; v < V; ++v) {
                dsum += std::exp(d[v] - dmax);
                tsum += std::exp(t[v] - tmax);
            }
            double dist = 0.0, S = 0.0;
            for (int v = 0; v < V; ++v) {
                pd[v] = std::exp(d[v] - dmax) / dsum;
                pt[v] = std::exp(t[v] - tmax) / tsum;
                const double diff = pd[v] - pt[v];
                dist += std::fabs(diff);
                S += (diff > 0.0 ? 1.0 : (diff < 0.0 ? -1.0 : 0.0)) * pd[v];
            }
            const double acc = std::min(1.0, std::max(0.0, 1.0 - 0.5 * dist));
            for (int v = 0; v < V; ++v) {
                const double diff = pd[v] - pt[v];
                const double sv = diff > 0.0 ? 1.0 : (diff < 0.0 ? -1.0 : 0.0);
                const double gce = pd[v] - (v == y ? 1.0 : 0.0);
                g[v] = static_cast<float>(c * (0.1 * gce + 0.9 * pd[v] * (sv - S)));
            }
            grad_conf[idx] = static_cast<float>(c * (1.0 / (1.0 + std::exp(-zc)) - acc));
        }
    }
}

// ---------------------------------------------------------------------------
// (d) Sequential Temperature Scaling of the confidence.
// [MB Acceptance and confidence]: the confidence head regresses to the
// accept rate, and a post-hoc Sequential Temperature Scaling calibrates it
// for serving.  The pages give no formula; the reading: temperature scaling
// (Guo et al., 2017) with one inverse temperature per block position k,
// beta_k >= 0, the calibrated confidence being sigmoid(beta_k * z); beta_k
// minimises the masked BCE of sigmoid(beta * z) against the accept labels
// a in [0, 1] over the logged pairs (z, a) of position k.  The objective is
// convex in beta, its derivative sum z (sigmoid(beta z) - a) non-decreasing,
// so the minimiser is its root, found here by plain bisection to the
// resolution of a double.  As beta grows the derivative tends to
// sum_{z>0} z (1 - a) + sum_{z<0} (-z) a >= 0, which is 0 exactly when every
// label agrees with the sign of its z (a = 1 for z > 0, a = 0 for z < 0):
// then no finite minimiser exists.  Per-position status: 0 fitted; 1 no
// information (no pair, or every z = 0): beta = 1; 2 labels separated by the
// sign of z, or a root beyond beta = 2^20: beta = 2^20; 3 a non-finite logit
// or a label outside [0, 1] in a counted pair: beta = NaN.  A derivative >= 0
// at beta = 0 gives beta = 0 (a constant confidence of 1/2).
// Pinned by: soft labels a = sigmoid(z / T) give back beta = 1 / T; a
// library scalar minimiser of the library BCE agrees; scaling every z by c
// divides beta by c; masked pairs do not count.
// ---------------------------------------------------------------------------
extern "C" void orc_sts_fit(const float* conf_logits, const float* labels, const uint8_t* mask,
                            int32_t N, int32_t gamma, double* beta, int32_t* status) {
    const double kBetaMax = 1048576.0;
    for (int k = 0; k < gamma; ++k) {
        // the derivative of the position's BCE in beta
        auto slope = [&](double bt) {
            double d = 0.0;
            for (int n = 0; n < N; ++n) {
                const size_t idx = static_cast<size_t>(n) * gamma + k;
                if (mask && !mask[idx]) continue;
                const double z = conf_logits[idx];
                d += z * (1.0 / (1.0 + std::exp(-bt * z)) - static_cast<double>(labels[idx]));
            }
            return d;
        };
        bool informative = false, separated = true, invalid = false;
        for (int n = 0; n < N; ++n) {
            const size_t idx = static_cast<size_t>(n) * gamma + k;
            if (mask && !mask[idx]) continue;
            const float z = conf_logits[idx], a = labels[idx];
            if (!std::isfinite(z) || !(a >= 0.0f && a <= 1.0f)) invalid = true;
            if (z != 0.0f) informative = true;
            if ((z > 0.0f && a < 1.0f) || (z < 0.0f && a > 0.0f)) separated = false;
        }
        if (invalid) {
            beta[k] = std::numeric_limits<double>::quiet_NaN();
            status[k] = 3;
            continue;
        }
        if (!informative) {
            beta[k] = 1.0;
            status[k] = 1;
            continue;
        }
        if (separated) {
            beta[k] = kBetaMax;
            status[k] = 2;
            continue;
        }
        status[k] = 0;
        if (slope(0.0) >= 0.0) {
            beta[k] = 0.0;
            continue;
        }
        double lo = 0.0, hi = 1.0;
        while (slope(hi) < 0.0 && hi < kBetaMax) {
            lo = hi;
            hi *= 2.0;
        }
        if (slope(hi) < 0.0) {
            beta[k] = kBetaMax;
            status[k] = 2;
            continue;
        }
        // slope(lo) < 0 <= slope(hi): halve the bracket until it stops shrinking
        for (int it = 0; it < 2000; ++it) {
            const double mid = 0.5 * (lo + hi);
            if (mid <= lo || mid >= hi) break;
            if (slope(mid) < 0.0) lo = mid;
            else hi = mid;
        }
        beta[k] = 0.5 * (lo + hi);
    }
}
