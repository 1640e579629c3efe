/*
 * dgc_oracle.h -- interface of the oracle: a plain, slow, single-threaded CPU restatement of
 * the Deep Gradient Compression (DGC) per-worker compressor, its sparse codec and the
 * decode-and-sum aggregator.
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the benchmark's CPU-baseline
 * leg are the only callers. Nothing here is shared with the CUDA library: its own types, its
 * own constants, its own code, written from the same definitions.
 *
 * Parity pins for every function live in the CPU test suite (closed forms, brute force on
 * tiny inputs, published SplitMix64 outputs, hand-built codec streams).
 */
#ifndef DGC_ORACLE_H
#define DGC_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_OK = 0, ORC_EINVAL = -1, ORC_ECAPACITY = -2, ORC_ECORRUPT = -5, ORC_EUNSUPPORTED = -6,
       ORC_ENOMEM = -7 };
enum { ORC_EXACT = 0, ORC_SAMPLED = 1, ORC_ADACOMP = 2 };
enum { ORC_MASK_MOMENTUM = 1u };

typedef struct {
    uint32_t mode;          /* ORC_EXACT, ORC_SAMPLED or ORC_ADACOMP */
    uint32_t flags;         /* ORC_MASK_MOMENTUM: zero u where a value was sent */
    double sparsity;        /* fraction NOT sent, in [0,1] */
    float momentum;         /* m in u <- m*u + g */
    float clip_norm;        /* per-segment L2 bound on g; <= 0 or inf disables clipping */
    double sample_ratio;    /* sampled mode: fraction of a segment sampled */
    double reselect_factor; /* sampled mode: re-select exactly when |C| > factor * k */
    uint64_t seed;          /* sampled mode: seed of the sample positions */
    uint32_t bin_size;      /* AdaComp mode: entries per bin (>= 1) */
    float leak;             /* v <- leak*v + u, in [0, 1]; 0 means 1 (no filter) */
} orc_params;

typedef struct {
    uint64_t k;          /* target count for the segment (AdaComp: number of bins) */
    uint64_t candidates; /* sampled: |C|; exact and AdaComp: |S| */
    uint64_t sent;       /* |S| */
    uint32_t thresh_key; /* smallest |v| key among sent entries; 0xFFFFFFFF if none */
    uint32_t sample_key; /* sampled: the sampled threshold t; exact: 0 */
    uint32_t reselected; /* sampled: 1 if the exact re-selection ran */
    float clip_scale;    /* factor applied to g (1 when not clipped) */
    double clip_sumsq;   /* with clipping on: S = orc_sumsq of the segment's g; else 0 */
} orc_seg_stats;

/* building blocks, exported so the tests can pin each one on its own */
uint64_t orc_ppb(double fraction);
uint64_t orc_count(uint64_t n, uint64_t ppb);
uint64_t orc_mix64(uint64_t z);
uint64_t orc_sample_position(uint64_t seed, uint32_t segment, uint64_t j, uint64_t n_s);
double orc_sumsq(const float* g, int64_t n);
float orc_clip_scale(const float* g, int64_t n, float clip_norm, int* clipped);
void orc_accumulate_one(float g, float u, float v, float momentum, float scale, int clipped,
                        float* u_out, float* v_out);
void orc_accumulate_leak(float g, float u, float v, float momentum, float scale, int clipped,
                         float leak, float* u_out, float* v_out);
int orc_topk(const float* v, const uint32_t* cand, int64_t ncand, int64_t k, uint8_t* selected);
void orc_bin_select(const float* v, int64_t n, uint32_t bin_size, uint8_t* selected);

int orc_compress(const float* g, float* u, float* v, int64_t n, const int64_t* seg_off,
                 int32_t nseg, const orc_params* p, uint32_t* out_idx, float* out_val,
                 int64_t out_cap, int64_t* out_count, orc_seg_stats* stats);

uint64_t orc_encoded_size(const uint32_t* idx, int64_t count);
int orc_encode(const uint32_t* idx, const float* val, int64_t count, int64_t n, uint8_t* out,
               uint64_t out_cap, uint64_t* out_bytes);
int orc_decode_accumulate(const uint8_t* const* streams, const uint64_t* stream_bytes,
                          int32_t W, float* dense, int64_t n, int accumulate);
int orc_decode_apply(const uint8_t* const* streams, const uint64_t* stream_bytes, int32_t W,
                     float* w, int64_t n, float lr);

/* one index set shared by all learners */
int orc_compress_shared(const float* g, float* u, float* v, int64_t n, const int64_t* seg_off,
                        int32_t nseg, const orc_params* p, const uint32_t* idx, int64_t count,
                        float* out_val);
int orc_sum_shared(const float* const* vals, int32_t W, int64_t count, float* out);

/* integer-valued messages (version 2) */
int orc_encode_quant(const uint32_t* idx, const float* val, int64_t count, int64_t n, float alpha,
                     int bits, float* v, uint8_t* out, uint64_t out_cap, uint64_t* out_bytes);
int orc_decode_accumulate_quant(const uint8_t* const* streams, const uint64_t* stream_bytes,
                                int32_t W, int bits, float alpha, float* dense, int64_t n,
                                int accumulate);
int orc_decode_apply_quant(const uint8_t* const* streams, const uint64_t* stream_bytes, int32_t W,
                           int bits, float alpha, float* w, int64_t n, float lr);

#ifdef __cplusplus
}
#endif
#endif
