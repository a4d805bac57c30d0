// schedule_model.cu -- the max-plus pipeline model of a warp-specialised
// GEMM main loop, as a host-side planning tool (no GPU involved).
//
// "Hopper and Blackwell GEMM", section "Maths": K slices are numbered
// g = t*K + k (tile t, slice k); with S ring stages and A accumulator buffers,
//   L_g = max(L_{g-1} + t_issue, D_{g-S})          a slot is free once its MMA is done
//   M_g = max(L_g + t_load, D_{g-1}, E_{t-A} if k = 0)   data in, tensor core free, buffer drained
//   D_g = M_g + t_mma
//   E_t = max(D_{tK+K-1}, E_{t-1}) + t_epi
// The run ends with the last epilogue; the tensor core is busy T*K*t_mma of it.
#include <algorithm>
#include <cmath>
#include <vector>

#include "gemm.h"

namespace {

struct Schedule {
    std::vector<double> L, M, D, E;
};

Schedule simulate(const gemm_sched_params_t& in) {
    const int T = in.tiles, K = in.k_slices, S = in.stages, A = in.accumulators;
    Schedule s;
    s.L.resize((size_t)T * K);
    s.M.resize((size_t)T * K);
    s.D.resize((size_t)T * K);
    s.E.resize((size_t)T);
    for (int t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            const int g = t * K + k;
            double l = g > 0 ? s.L[g - 1] + in.t_issue : 0.0;
            if (g >= S) l = std::max(l, s.D[g - S]);
            s.L[g] = l;
            double m = l + in.t_load;
            if (g > 0) m = std::max(m, s.D[g - 1]);
            if (k == 0 && t >= A) m = std::max(m, s.E[t - A]);
            s.M[g] = m;
            s.D[g] = m + in.t_mma;
        }
        double e = s.D[(size_t)t * K + K - 1];
        if (t > 0) e = std::max(e, s.E[t - 1]);
        s.E[t] = e + in.t_epi;
    }
    return s;
}

bool valid(const gemm_sched_params_t* in) {
    return in && in->tiles >= 1 && in->k_slices >= 1 && in->stages >= 1 && in->accumulators >= 1 &&
           in->tiles <= (1 << 20) && in->k_slices <= (1 << 20) && (int64_t)in->tiles * in->k_slices <= (1 << 24) &&
           in->t_issue >= 0 && in->t_load >= 0 && in->t_mma > 0 && in->t_epi >= 0;
}

}  // namespace

extern "C" {

gemm_status_t gemm_schedule_model(const gemm_sched_params_t* in, gemm_sched_result_t* out) {
    if (!valid(in) || !out) return GEMM_ERR_INVALID_ARG;
    const Schedule s = simulate(*in);
    const int T = in->tiles, K = in->k_slices, S = in->stages;
    out->run_length = s.E[T - 1];
    out->tensor_busy = (double)T * K * in->t_mma / out->run_length;
    // steady state inside the last tile: M_{g+S} - M_g for its last S slices
    const int last = T * K - 1;
    out->steady_period = (K > S) ? s.M[last] - s.M[last - S] : 0.0;
    out->stages_needed = (int32_t)std::ceil((in->t_load + in->t_mma) / in->t_mma - 1e-12);
    out->reserved = 0;
    return GEMM_OK;
}

gemm_status_t gemm_schedule_choose(const gemm_sched_params_t* in, int32_t max_stages, int32_t max_accumulators,
                                   double tolerance, int32_t* stages, int32_t* accumulators) {
    if (!valid(in) || max_stages < 1 || max_accumulators < 1 || tolerance < 0 || !stages || !accumulators)
        return GEMM_ERR_INVALID_ARG;
    gemm_sched_params_t p = *in;
    p.stages = max_stages;
    p.accumulators = max_accumulators;
    const double best = simulate(p).E[p.tiles - 1];
    // fewest accumulators, then fewest stages, whose run is within `tolerance` of the best
    for (int a = 1; a <= max_accumulators; ++a) {
        for (int s = 1; s <= max_stages; ++s) {
            p.stages = s;
            p.accumulators = a;
            if (simulate(p).E[p.tiles - 1] <= best * (1.0 + tolerance)) {
                *stages = s;
                *accumulators = a;
                return GEMM_OK;
            }
        }
    }
    *stages = max_stages;
    *accumulators = max_accumulators;
    return GEMM_OK;
}

}  // extern "C"
