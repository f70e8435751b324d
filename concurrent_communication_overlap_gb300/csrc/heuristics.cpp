// heuristics.cpp -- the pages' runtime heuristics for C3 (Section V-C of
// "Optimizing ML Concurrent Computation and Communication with GPU DMA
// Engines", as summarised on its pith.science page: "If this is right" and
// "Assumptions & free parameters").
//
// Schedule prioritisation: launch the kernel with the lower workgroup (CTA)
// count first.
//
// Resource partitioning: a one-time lookup table of how much each kernel
// slows down with a given number of SMs (the pages' Figure 5: a GEMM losing
// compute units, a collective given compute units) plus a roofline at 70%
// efficiency for the isolated times.  For every tabulated SM count k given to
// the collective, the concurrent time is predicted as
//     max(T_gemm_roofline * slowdown_gemm(k), T_comm_roofline * slowdown_comm(k))
// and the k with the smallest prediction is chosen.  The GEMM's table is
// picked by its class: compute-bound when its arithmetic intensity is at or
// above the ridge point of the roofline, memory-bound otherwise.
//
// The elastic variant models this library's partitions, which last only as
// long as both kernels run: a collective that outlasts the GEMM moves its
// remaining bytes on every SM once the GEMM is done.  With a = T_gemm *
// slowdown_gemm(k) and b = T_comm * slowdown_comm(k), by the time a the
// collective has moved a / b of its bytes; the rest takes (1 - a / b) * T_comm,
// so the prediction is T_comm + a * (1 - 1 / slowdown_comm(k)) where b > a,
// and a otherwise.
#include "../../include/c3_api.h"
#include "c3_internal.h"

namespace {

int rp_predict(const c3_rp_table* t, double gemm_flops, double gemm_bytes, double coll_bytes, double peak_flops,
               double peak_bytes_per_s, bool elastic, int* best_sms, double* t_pred_best, double* t_pred_each) {
    if (!t || !best_sms || !t_pred_best) return c3::set_error(C3_EINVAL, "NULL argument");
    if (t->n < 1 || t->n > C3_RP_MAX) return c3::set_error(C3_EINVAL, "table must hold 1..16 entries");
    if (!(gemm_flops >= 0) || !(gemm_bytes > 0) || !(coll_bytes >= 0) || !(peak_flops > 0) ||
        !(peak_bytes_per_s > 0))
        return c3::set_error(C3_EINVAL, "sizes and peaks must be positive");
    const double eff = 0.70;
    const double t_gemm = (gemm_flops / (eff * peak_flops) > gemm_bytes / (eff * peak_bytes_per_s))
                              ? gemm_flops / (eff * peak_flops)
                              : gemm_bytes / (eff * peak_bytes_per_s);
    const double t_comm = 2.0 * coll_bytes / (eff * peak_bytes_per_s);  // read + write
    const bool compute_bound = gemm_flops / gemm_bytes >= peak_flops / peak_bytes_per_s;
    int best = -1;
    double best_t = 0.0;
    for (int i = 0; i < t->n; ++i) {
        const double sg = compute_bound ? t->gemm_compute[i] : t->gemm_memory[i];
        const double sc = t->coll[i];
        if (!(sg > 0) || !(sc > 0) || t->sms[i] < 1) return c3::set_error(C3_EINVAL, "table entries must be > 0");
        const double a = t_gemm * sg, b = t_comm * sc;
        double tp = a > b ? a : b;
        if (elastic && b > a) tp = t_comm + a * (1.0 - 1.0 / sc);
        if (t_pred_each) t_pred_each[i] = tp;
        if (best < 0 || tp < best_t) {
            best = i;
            best_t = tp;
        }
    }
    *best_sms = t->sms[best];
    *t_pred_best = best_t;
    return C3_OK;
}

}  // namespace

extern "C" {

int c3_sp_predict(int gemm_ctas, int coll_ctas) {
    if (gemm_ctas < 0 || coll_ctas < 0) return c3::set_error(C3_EINVAL, "negative CTA count");
    return coll_ctas < gemm_ctas ? 1 : 0;
}

int c3_rp_predict(const c3_rp_table* t, double gemm_flops, double gemm_bytes, double coll_bytes,
                  double peak_flops, double peak_bytes_per_s, int* best_sms, double* t_pred_best,
                  double* t_pred_each) {
    return rp_predict(t, gemm_flops, gemm_bytes, coll_bytes, peak_flops, peak_bytes_per_s, false, best_sms,
                      t_pred_best, t_pred_each);
}

int c3_rp_predict_elastic(const c3_rp_table* t, double gemm_flops, double gemm_bytes, double coll_bytes,
                          double peak_flops, double peak_bytes_per_s, int* best_sms, double* t_pred_best,
                          double* t_pred_each) {
    return rp_predict(t, gemm_flops, gemm_bytes, coll_bytes, peak_flops, peak_bytes_per_s, true, best_sms,
                      t_pred_best, t_pred_each);
}

}  // extern "C"
