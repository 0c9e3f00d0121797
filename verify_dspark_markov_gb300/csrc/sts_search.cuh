// The per-position root search of the Sequential Temperature Scaling fit
// (sts.cu), host- and device-compilable so that the same code that runs in
// sts_update_kernel can be driven on the CPU.
//
// A position's state holds the sums of the pass just taken at its current
// beta: the BCE's slope s1 = sum z (sigmoid(beta z) - a), its curvature
// s2 = sum z^2 sigmoid (1 - sigmoid), and the pass's flags.  The slope does
// not decrease in beta, so its root is bracketed by [lo, hi] and approached
// by Newton steps that stay inside the bracket (doubling while hi is open,
// bisection when a step leaves it).
#pragma once

#include <cmath>
#include <limits>

#include "kernels.h"

namespace dspark {

constexpr double kStsBetaMax = 1048576.0;  // 2^20
constexpr unsigned kStsInformative = 1u, kStsViolated = 2u, kStsInvalid = 4u;

// Advance `s` by the sums of one pass; true when its search ends with this pass.
// Phase 0 (the pass at beta = 0) decides the degenerate cases: an invalid
// pair (status 3, beta NaN), no counted z != 0 (status 1, beta 1), every
// label agreeing with the sign of its z (no finite root: status 2, beta
// 2^20), a slope >= 0 at 0 (beta 0); else the search starts at beta = 1.
__host__ __device__ inline bool sts_search_step(StsState& s) {
    const double inf = std::numeric_limits<double>::infinity();
    if (s.phase == 2) return false;
    ++s.passes;  // this pass's sums are the position's
    if (s.phase == 0) {
        s.phase = 2;
        if (s.flags & kStsInvalid) {
            s.beta = std::numeric_limits<double>::quiet_NaN();
            s.status = 3;
        } else if (!(s.flags & kStsInformative)) {
            s.beta = 1.0;
            s.status = 1;
        } else if (!(s.flags & kStsViolated)) {
            s.beta = kStsBetaMax;
            s.status = 2;
        } else if (s.s1 >= 0.0) {
            s.beta = 0.0;
            s.status = 0;
        } else {
            s.lo = 0.0;
            s.hi = inf;
            s.beta = 1.0;
            s.status = 0;
            s.phase = 1;
        }
    } else {
        const double g = s.s1, h = s.s2, b = s.beta;
        if (g < 0.0) s.lo = b;
        else s.hi = b;
        if (g < 0.0 && b >= kStsBetaMax) {  // the root lies beyond the cap
            s.beta = kStsBetaMax;
            s.status = 2;
            s.phase = 2;
        } else if (g == 0.0) {
            s.phase = 2;
        } else {
            const double step = h > 0.0 ? b - g / h : b;
            double next;
            if (s.hi == inf) next = (step > b && step < inf) ? step : 2.0 * b;
            else next = (step > s.lo && step < s.hi) ? step : 0.5 * (s.lo + s.hi);
            next = fmin(next, kStsBetaMax);
            // stop at the accuracy the fp32 pair terms allow: nearer the
            // root their rounding decides the slope's sign
            const bool converged = fabs(next - b) <= 1e-7 * b || (s.hi != inf && s.hi - s.lo <= 1e-7 * s.hi);
            s.beta = next;
            if (converged) s.phase = 2;
        }
    }
    s.s1 = 0.0;
    s.s2 = 0.0;
    return s.phase == 2;
}

}  // namespace dspark
