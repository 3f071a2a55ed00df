/*
 * AirCache oracle -- TEST INFRASTRUCTURE ONLY (see aircache_oracle.c).
 * This header belongs to the oracle alone; the CUDA library does not include it.
 */
#ifndef AIRCACHE_ORACLE_H
#define AIRCACHE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* A token-major tensor [tokens][heads][D]; strides in elements, D contiguous. */
typedef struct {
    const void* base;
    int32_t dtype;
    int32_t pad_;
    int64_t stride_tok;
    int64_t stride_head;
} oracle_view;

int oracle_elite(const oracle_view* q, const oracle_view* k, int h_q, int h_kv, int d,
                 int n_v, int n_t, int n_p, double alpha, double* p_out, int32_t* elite);
int oracle_score(const oracle_view* q, const oracle_view* k, int h_q, int h_kv, int d,
                 int n_v, int n_t, int n_p, const int32_t* elite, int n_tk,
                 double* iv, double* elite_mass, double* iv_heads);
int oracle_stats(const double* iv, int n_v, double* out);
int oracle_budget(const double* s_t, const double* s_k, int n_layers, int n_v, double r,
                  double* r_l, int32_t* keep);
int oracle_select(const double* iv, int n_v, int keep, int32_t* idx);
int64_t oracle_compact(const oracle_view* src, int h_kv, int d, int n_v, int n_t, int n_p,
                       const int32_t* idx, int keep, void* dst);
int oracle_decode(const oracle_view* q, const oracle_view* k, const oracle_view* v, int h_q, int h_kv,
                  int d, int64_t n_rows, double* out);
int oracle_quant_code(float x, float s);
int oracle_quantize_int8(const oracle_view* src, int64_t n_rows, int h_kv, int d, int8_t* codes,
                         float* scales);
int oracle_window(int n_t, int mode, int32_t* positions);
int oracle_budget_variant(const double* s_t, const double* s_k, int n_layers, int n_v, double r,
                          int mode, double* r_l, int32_t* keep);
int oracle_request_variant(const oracle_view* q, const oracle_view* k, int n_layers, int h_q,
                           int h_kv, int d, int n_v, int n_t, int n_p, double alpha, double r, int window_mode,
                           int budget_mode, double* iv, int32_t* elite, int32_t* n_tk, double* stats,
                           int32_t* keep, int32_t* idx, double* iv_heads, int32_t* idx_heads,
                           const oracle_view* qv);
int oracle_window_visual(int n_v, int32_t* positions);
int oracle_score_visual_window(const oracle_view* qv, const oracle_view* k, int h_q, int h_kv, int d, int n_v,
                               int n_p, const int32_t* pos, int n_w, double* iv);
int64_t oracle_compact_heads(const oracle_view* src, int h_kv, int d, int n_v, int n_t, int n_p,
                             const int32_t* idx_heads, int keep, void* dst);
int oracle_request(const oracle_view* q, const oracle_view* k, int n_layers, int h_q, int h_kv,
                   int d, int n_v, int n_t, double alpha, double r,
                   double* iv, int32_t* elite, int32_t* n_tk, double* stats,
                   int32_t* keep, int32_t* idx);

#ifdef __cplusplus
}
#endif

#endif
