/*
 * tq_oracle.h -- plain CPU oracle for TurboQuant compressed-KV encode and
 * decode attention.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference arm may load, call or link this code. The product
 * library never includes this header and shares no code with it.
 *
 * Conventions: D = head_dim; b = index bits; matrices are row-major;
 * "fp64" functions compute in double. Codec modes: 0 = MSE, 1 = prod
 * (MSE with b-1 bits + 1-bit QJL sign of the residual), 2 = group.
 */
#ifndef TQ_ORACLE_H
#define TQ_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* SplitMix64 output number i (0-based) of the generator seeded with state s. */
uint64_t tqo_splitmix64_at(uint64_t s, uint64_t i);
/* n standard normals from stream (seed, stream) by Box-Muller. */
void tqo_normals(uint64_t seed, int stream, int64_t n, double *out);

/* Haar rotation R (D x D) from QR of a Gaussian matrix, fp64 and fp32. */
int tqo_rotation_f64(int D, uint64_t seed, double *R);
/* QJL matrix S (D x D), i.i.d. N(0,1), fp64. */
int tqo_qjl_f64(int D, uint64_t seed, double *S);
/* Lloyd-Max levels (2^b) and midpoints (2^b - 1) for the coordinate density
 * of a uniform unit vector in R^D, fp64. Returns iterations used. */
int tqo_lloyd_max(int D, int b, double *c, double *m);
/* Codec tables in the stored precision (fp32). R, S: D*D (S may be NULL
 * unless mode==prod); c: 2^ib; m: 2^ib - 1 where ib = index bits. */
int tqo_codec_tables(int D, int bits, int mode, uint64_t seed,
                     float *R, float *S, float *c, float *m);

int tqo_index_bits(int bits, int mode);
int tqo_packed_words(int D, int index_bits);
/* Key and value widths of a possibly fractional bit width. */
void tqo_bits_split(double b, int *key_bits, int *value_bits);
/* Bytes of one token's record for a codec. */
int tqo_record_bytes(int D, int bits, int mode, int group);

/* Bit packing (LSB-first, code i at bit i*b, codes may straddle words). */
void tqo_pack(const uint8_t *codes, int D, int b, uint32_t *words);
void tqo_unpack(const uint32_t *words, int D, int b, uint8_t *codes);

/* IEEE binary16 conversions (round to nearest even). */
uint16_t tqo_f32_to_f16(float x);
float tqo_f16_to_f32(uint16_t h);

/* Encoders over n vectors (x: n x D fp32). Outputs per vector:
 *  mse:  idx words [n][W], norm [n]
 *  prod: idx words [n][W] (b-1 bits), signs [n][D/32], norm [n], rnorm [n]
 *  group: data words [n][W], scale [n][D/g] (f16 bits), min [n][D/g] (f16 bits) */
void tqo_encode_mse(int64_t n, int D, const float *x, const float *R, const float *m,
                    int b, uint32_t *idx, float *norm);
void tqo_encode_prod(int64_t n, int D, const float *x, const float *R, const float *S,
                     const float *c, const float *m, int bits, uint32_t *idx,
                     uint32_t *sgn, float *norm, float *rnorm);
void tqo_encode_group(int64_t n, int D, const float *x, int bits, int g,
                      uint32_t *data, uint16_t *scale, uint16_t *mn);

/* Dequantisers to fp64 vectors [n][D]. */
void tqo_dequant_mse(int64_t n, int D, const uint32_t *idx, const float *norm,
                     const float *R, const float *c, int b, double *out);
void tqo_dequant_prod(int64_t n, int D, const uint32_t *idx, const uint32_t *sgn,
                      const float *norm, const float *rnorm, const float *R,
                      const float *S, const float *c, int bits, double *out);
void tqo_dequant_group(int64_t n, int D, const uint32_t *data, const uint16_t *scale,
                       const uint16_t *mn, int bits, int g, double *out);

/* Plain attention (fp64) of R = G*Lq query rows over N dequantised keys and
 * values. Row r = g*Lq + l may see keys t <= N - Lq + l. q: [G][Lq][D]. */
void tqo_attention_f64(int D, int64_t N, int G, int Lq, const double *q,
                       const double *K, const double *V, double scale, double *out);

/* Rotated-domain decode (O(N*D) per row) straight from the records, fp64.
 * Key mode 0/1, value mode 0/2; arguments as in the encoders. */
void tqo_decode_rotated(int D, int64_t N, int G, int Lq, const double *q,
                        int kmode, int kbits, const uint32_t *kidx, const uint32_t *ksgn,
                        const float *knorm, const float *krn, const float *kR,
                        const float *kS, const float *kc,
                        int vmode, int vbits, int vgroup, const uint32_t *vidx,
                        const float *vnorm, const uint16_t *vscale, const uint16_t *vmin,
                        const float *vR, const float *vc, double scale, double *out);

/* Sequence-sharded decode: the unnormalised softmax state (m, l, acc) of
 * each row over a shard of N local keys whose causal end is E (a local key t
 * is visible to query l when t <= E - Lq + l); acc in the rotated domain
 * (MSE values) or the value domain (group). Then the log-sum-exp merge of P
 * parts, each [rows] (m, l) and [rows][D] acc, into out [rows][D]. */
void tqo_decode_partial(int D, int64_t N, int64_t E, int G, int Lq, const double *q,
                        int kmode, int kbits, const uint32_t *kidx, const uint32_t *ksgn,
                        const float *knorm, const float *krn, const float *kR,
                        const float *kS, const float *kc,
                        int vmode, int vbits, int vgroup, const uint32_t *vidx,
                        const float *vnorm, const uint16_t *vscale, const uint16_t *vmin,
                        const float *vc, double scale, double *m_out, double *l_out,
                        double *acc_out);
void tqo_merge_partials(int D, int P, int64_t rows, const double *m, const double *l,
                        const double *acc, int vmode, const float *vR, double *out);

/* Paged-pool layout: byte offset of each stream inside one (block, head)
 * sub-block of BT tokens, in the stream order of the layout; returns the
 * sub-block size. off[] receives up to 4 key streams then up to 3 value
 * streams (unused = -1). */
int64_t tqo_subblock_layout(int D, int kmode, int kbits, int vmode, int vbits, int vgroup,
                            int BT, int64_t off[7]);
/* Write token records [t0, t0+n) of sequence `seq`, kv head h, into a layer pool. */
void tqo_pool_write(uint8_t *pool, int D, int Hkv, int BT, const int32_t *table,
                    int max_blocks, int seq, int h, int64_t t0, int64_t n,
                    int kmode, int kbits, int vmode, int vbits, int vgroup,
                    const uint32_t *kidx, const uint32_t *ksgn, const float *knorm,
                    const float *krn, const uint32_t *vidx, const float *vnorm,
                    const uint16_t *vscale, const uint16_t *vmin);

int tqo_num_threads(void);
void tqo_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
