// latency.cpp -- the step-latency model (include/lora_latency.h): features, least-squares fit, prediction.
// Host code only.
#include <cmath>
#include <vector>

#include "lora_latency.h"
#include "plan.h"

namespace {

int32_t terms_of(int32_t model) {
    return model == LORA_LATENCY_EQ_I ? 5 : (model == LORA_LATENCY_EQ_II ? 3 : 0);
}

}  // namespace

extern "C" {

int32_t lora_latency_terms(int32_t model) { return terms_of(model); }

int lora_latency_features(int32_t model, const lora_segment_t* segs, int32_t n_segs, double kv_size,
                          double* feat_out) {
    const int32_t p = terms_of(model);
    if (p == 0 || feat_out == nullptr || n_segs < 0 || (n_segs > 0 && segs == nullptr)) {
        lora::set_last_error("lora_latency_features: unknown model, NULL pointer or negative count");
        return LORA_ERR_INVALID_ARG;
    }
    double b_d = 0.0, t_ft = 0.0;
    std::vector<double> prompts;
    for (int32_t i = 0; i < n_segs; ++i) {
        const lora_segment_t& s = segs[i];
        if (s.len <= 0) continue;
        if (s.is_train) t_ft += s.len;
        else if (s.len == 1) b_d += 1.0;
        else prompts.push_back(double(s.len));
    }
    if (model == LORA_LATENCY_EQ_I) {
        double sq = 0.0, t_in = 0.0;
        for (double n : prompts) {
            sq += (n + b_d) * (n + b_d);
            t_in += n;
        }
        feat_out[0] = sq;
        feat_out[1] = t_in + b_d;
        feat_out[2] = t_ft;
        feat_out[3] = kv_size;
        feat_out[4] = 1.0;
    } else {
        feat_out[0] = b_d;
        feat_out[1] = kv_size;
        feat_out[2] = 1.0;
    }
    return LORA_OK;
}

// Least squares by Householder QR on the kept columns, each scaled to unit maximum first (the features span
// many orders of magnitude: a squared prompt length next to the constant 1).
int lora_latency_fit(int32_t model, const double* feats, const double* times, int32_t n, double* coef_out) {
    const int32_t p = terms_of(model);
    if (p == 0 || feats == nullptr || times == nullptr || coef_out == nullptr || n <= 0) {
        lora::set_last_error("lora_latency_fit: unknown model, NULL pointer or no samples");
        return LORA_ERR_INVALID_ARG;
    }
    std::vector<int32_t> keep;
    std::vector<double> colscale;
    for (int32_t j = 0; j < p; ++j) {
        double m = 0.0;
        for (int32_t i = 0; i < n; ++i) m = std::fmax(m, std::fabs(feats[(size_t)i * p + j]));
        coef_out[j] = 0.0;
        if (m > 0.0) {
            keep.push_back(j);
            colscale.push_back(m);
        }
    }
    const int32_t q = int32_t(keep.size());
    if (n < q) {
        lora::set_last_error("lora_latency_fit: fewer samples than fitted terms");
        return LORA_ERR_INVALID_ARG;
    }
    // M = [scaled kept features | times], column-major n x (q+1)
    std::vector<double> M((size_t)n * (q + 1));
    for (int32_t c = 0; c < q; ++c)
        for (int32_t i = 0; i < n; ++i) M[(size_t)c * n + i] = feats[(size_t)i * p + keep[c]] / colscale[c];
    for (int32_t i = 0; i < n; ++i) M[(size_t)q * n + i] = times[i];
    double rmax = 0.0;
    std::vector<double> R((size_t)q * q, 0.0);
    for (int32_t c = 0; c < q; ++c) {
        double* v = &M[(size_t)c * n];
        double norm = 0.0;
        for (int32_t i = c; i < n; ++i) norm += v[i] * v[i];
        norm = std::sqrt(norm);
        if (c == 0) rmax = norm;
        if (norm <= 1e-12 * std::fmax(rmax, 1e-300)) {
            lora::set_last_error("lora_latency_fit: the sampled features are linearly dependent");
            return LORA_ERR_LIMIT;
        }
        const double alpha = (v[c] > 0.0) ? -norm : norm;   // R[c][c]
        // Householder vector u = v - alpha e_c (stored in v[c..n)), H = I - 2 u u^T / (u^T u)
        v[c] -= alpha;
        double uu = 0.0;
        for (int32_t i = c; i < n; ++i) uu += v[i] * v[i];
        for (int32_t d = c + 1; d <= q; ++d) {
            double* w = &M[(size_t)d * n];
            double dot = 0.0;
            for (int32_t i = c; i < n; ++i) dot += v[i] * w[i];
            const double f = 2.0 * dot / uu;
            for (int32_t i = c; i < n; ++i) w[i] -= f * v[i];
        }
        R[(size_t)c * q + c] = alpha;
        for (int32_t d = c + 1; d < q; ++d) R[(size_t)c * q + d] = M[(size_t)d * n + c];
    }
    // back substitution: R beta = (Q^T t)[0..q)
    std::vector<double> beta(q);
    for (int32_t c = q - 1; c >= 0; --c) {
        double s = M[(size_t)q * n + c];
        for (int32_t d = c + 1; d < q; ++d) s -= R[(size_t)c * q + d] * beta[d];
        beta[c] = s / R[(size_t)c * q + c];
    }
    for (int32_t c = 0; c < q; ++c) coef_out[keep[c]] = beta[c] / colscale[c];
    return LORA_OK;
}

double lora_latency_predict(int32_t model, const double* coef, const double* feat) {
    const int32_t p = terms_of(model);
    if (p == 0 || coef == nullptr || feat == nullptr) return NAN;
    double t = 0.0;
    for (int32_t j = 0; j < p; ++j) t += coef[j] * feat[j];
    return t;
}

}  // extern "C"
