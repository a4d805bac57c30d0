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
#include <cstdint>
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

// Unit costs measured on GB300 (SM clock cycles):
//  * 8,192 flop per cycle per SM for kind::f16 (a probe issuing M128 N256 K16
//    MMAs back to back: 128 cycles each);
//  * copy path 400 cycles per ring stage plus 128 bytes per cycle: a scratch
//    copy of the persistent kernel with its MMAs skipped streamed 8192^3's
//    operands at 657 cycles per 32 KB stage and 912 per 64 KB stage;
//  * tcgen05.ld 220 bytes per cycle per SM while the MMAs run (200-240 measured);
//  * load latency 1,400 cycles: the value whose model best matches a sweep of
//    the ring depth at 8192^3 (512-wide tiles: 2 stages 39 % slower than 4,
//    3 stages 1.6 % slower; 256-wide tiles of 128-deep stages: 2 stages 21 %
//    slower than 3);
//  * hand-back 600 cycles: an estimate (runs with two accumulators do not
//    depend on it).
constexpr gemm_machine_t kGb300 = {8192.0, 400.0, 128.0, 1400.0, 220.0, 600.0};

gemm_status_t gemm_machine_gb300(gemm_machine_t* out) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    *out = kGb300;
    return GEMM_OK;
}

gemm_status_t gemm_plan_schedule(const gemm_desc_t* desc, const gemm_plan_info_t* info,
                                 const gemm_device_props_t* props, const gemm_machine_t* machine,
                                 gemm_sched_params_t* params, gemm_sched_result_t* result,
                                 int32_t* model_stages, int32_t* model_accumulators) {
    if (!desc || !info || !props) return GEMM_ERR_INVALID_ARG;
    if (info->kernel != GEMM_KERNEL_PERSISTENT) return GEMM_ERR_UNSUPPORTED;
    const gemm_machine_t& mc = machine ? *machine : kGb300;
    if (!(mc.mma_flops_per_cycle > 0) || !(mc.ingest_bytes_per_cycle > 0) || !(mc.tmem_read_bytes_per_cycle > 0) ||
        mc.stage_fixed_cycles < 0 || mc.load_latency_cycles < 0 || mc.handback_cycles < 0)
        return GEMM_ERR_INVALID_ARG;
    if (info->cta_group < 1 || info->grid < info->cta_group || info->tile_n <= 0 || info->tile_k <= 0 ||
        info->stages < 1 || info->tmem_stages < 1 || info->num_tiles < 1 || info->stage_bytes <= 0 || desc->K <= 0)
        return GEMM_ERR_INVALID_ARG;
    const int64_t clusters = info->grid / info->cta_group;
    const int64_t k_slices = (desc->K + info->tile_k - 1) / info->tile_k;
    int64_t k_run = k_slices;   // K slices the model runs per tile
    int64_t tiles = (info->num_tiles + clusters - 1) / clusters;
    if (info->stream_k_tiles > 0) {
        // a cluster's share of all K slices, counted in whole tiles, or as
        // one shorter tile when it is less than a tile (fewer tiles than clusters)
        const int64_t slices = (info->num_tiles * k_slices + clusters - 1) / clusters;
        tiles = (slices + k_slices - 1) / k_slices;
        if (slices < k_slices) k_run = slices;
    }
    if (tiles > (1 << 20) || k_run > (1 << 20) || tiles * k_run > (1 << 24)) return GEMM_ERR_UNSUPPORTED;
    // tf32 multiplies at half the 16-bit rate (nominal 1.1 against 2.25 PFLOP/s)
    const double rate = mc.mma_flops_per_cycle * (desc->dtype_a == GEMM_TF32 ? 0.5 : 1.0);
    gemm_sched_params_t p{};
    p.tiles = (int32_t)tiles;
    p.k_slices = (int32_t)k_run;
    p.stages = info->stages;
    p.accumulators = info->tmem_stages;
    const double stage_bytes = (double)info->stage_bytes;   // per CTA, A and B
    p.t_mma = 2.0 * 128.0 * info->tile_n * info->tile_k / rate;
    p.t_issue = mc.stage_fixed_cycles + stage_bytes / mc.ingest_bytes_per_cycle;
    p.t_load = mc.load_latency_cycles + stage_bytes / mc.ingest_bytes_per_cycle;
    p.t_epi = 128.0 * info->tile_n * 4.0 / mc.tmem_read_bytes_per_cycle + mc.handback_cycles;
    if (params) *params = p;
    if (result) {
        gemm_status_t st = gemm_schedule_model(&p, result);
        if (st != GEMM_OK) return st;
    }
    if (model_stages || model_accumulators) {
        // the planner's limits: as many stages as the shared memory holds
        // (each costs its bytes and two 8-byte barriers), two accumulators up
        // to 256 columns and one for 512-wide tiles
        int64_t max_s = info->stages;
        if (props->smem_optin_bytes > 0)
            while (max_s < 16 && info->smem_bytes + (max_s + 1 - info->stages) * (info->stage_bytes + 16) <=
                                     props->smem_optin_bytes)
                ++max_s;
        const int32_t max_a = info->tile_n > 256 ? 1 : 2;
        int32_t s = 0, a = 0;
        gemm_status_t st = gemm_schedule_choose(&p, (int32_t)max_s, max_a, 0.005, &s, &a);
        if (st != GEMM_OK) return st;
        if (model_stages) *model_stages = s;
        if (model_accumulators) *model_accumulators = a;
    }
    return GEMM_OK;
}

}  // extern "C"
