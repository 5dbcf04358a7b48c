/*
 * lora_latency.h -- host-side step-latency model of a co-serving step (no GPU work).
 *
 * "DeltaServe: Host-Agnostic Co-Serving of Inference and Fine-Tuning for LLMs", section 3.3 (SLO Budgeting),
 * predicts the time of a forward step from its batch composition:
 *
 *   (I)  mixed steps:        T ~ alpha * sum_i (n_i + B_d)^2 + beta * (T_in + B_d) + gamma * T_ft + eps * K + c
 *   (II) decode-only steps:  T ~ beta' * B_d + eps' * K + c'
 *
 * with n_i the prompt lengths of the prefill requests, T_in their sum, B_d the number of decode requests,
 * T_ft the fine-tuning tokens and K the key-value cache size; the coefficients of each equation are fitted
 * (least squares) to measured step times.  This library fits and evaluates both forms; its benchmark fits
 * them to the timings of its own layer step.
 *
 * Reading of a segment table (lora_segment_t of lora_mixed.h): a fine-tuning segment contributes its length
 * to T_ft; any other segment of length 1 is one decode request (B_d); any other longer segment is one prefill
 * request of n_i = len.  The key-value cache size K is the caller's number (0 for a path without attention).
 *
 * Feature vectors, in coefficient order:
 *   model 1 (Eq. I):  {sum_i (n_i + B_d)^2, T_in + B_d, T_ft, K, 1}    coefficients {alpha, beta, gamma, eps, c}
 *   model 2 (Eq. II): {B_d, K, 1}                                        coefficients {beta', eps', c'}
 */
#ifndef LORA_LATENCY_H
#define LORA_LATENCY_H

#include <stdint.h>

#include "lora_mixed.h"

#ifdef __cplusplus
extern "C" {
#endif

#define LORA_LATENCY_EQ_I 1
#define LORA_LATENCY_EQ_II 2
#define LORA_LATENCY_MAX_TERMS 5

/* Number of features (and coefficients) of a model: 5 for Eq. I, 3 for Eq. II; 0 for an unknown model. */
int32_t lora_latency_terms(int32_t model);

/* Features of one step from its segment table (HOST) and key-value cache size, per the reading above.
 * feat_out: HOST [lora_latency_terms(model)].  Returns LORA_OK or LORA_ERR_INVALID_ARG. */
int lora_latency_features(int32_t model, const lora_segment_t* segs, int32_t n_segs, double kv_size,
                          double* feat_out);

/* Least-squares fit of a model to n measured steps: feats HOST [n, terms] row-major, times HOST [n].
 * A feature that is zero in every sample (e.g. K for a path without attention) gets coefficient 0 and is left
 * out of the solve.  coef_out HOST [terms].  Returns LORA_OK, LORA_ERR_INVALID_ARG (NULL pointers, unknown
 * model, fewer samples than fitted terms) or LORA_ERR_LIMIT (the kept features are linearly dependent). */
int lora_latency_fit(int32_t model, const double* feats, const double* times, int32_t n, double* coef_out);

/* Predicted time of one step: the dot product of its features with the coefficients. */
double lora_latency_predict(int32_t model, const double* coef, const double* feat);

#ifdef __cplusplus
}
#endif

#endif /* LORA_LATENCY_H */
