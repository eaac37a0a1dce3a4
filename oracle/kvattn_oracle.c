/*
 * kvattn oracle -- plain, slow, fp64 CPU restatement of what the attention hot
 * path computes.  TEST INFRASTRUCTURE ONLY: it is loaded by tests/, by
 * __graft_entry__.smoke() and by bench.py's CPU-baseline leg, never by the
 * library.  It shares no code, header, table or constant with the CUDA path.
 *
 * Sources (web pages on hand-writing an LLM inference engine):
 *  - "Tokenizer, KV Cache and RoPE" page, section 4: rotary embedding rotates
 *    adjacent pairs (x0,x1),(x2,x3),... of a query/key vector by m*theta_i,
 *    theta_i = 10000^(-2i/d), m = token position; scale 1/sqrt(d_k) with d_k
 *    the head dimension.
 *  - "From-scratch AI inference engine" page, section 3.1: attention is
 *    softmax(Q K^T / sqrt(d_k)) V with the scale applied before the softmax;
 *    section 3.2: a new token's K/V are written at the cache index that equals
 *    its absolute position; section 3.3: causal mask -- a position sees itself
 *    and earlier positions; with a cache a new token sees all S cached keys.
 *  - "Nano-vLLM Part 2" page, section 05: paged cache addressed through a block
 *    table, physical block = table[t / block_size], offset = t % block_size.
 *
 * Everything is computed in double from the inputs' exact values.  The cache
 * here is slot-major, Kc[slot][kv_head][d] with slot = block*BS + offset: the
 * oracle's own layout, deliberately not the library's.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define KVO_OK 0
#define KVO_ERR_ARG 1
#define KVO_ERR_INDEX 2

/* ---- rounding to the stored element type --------------------------------- */

/* Round-to-nearest-even of a double straight to bfloat16 (8 significant bits,
 * exponent range of binary32), returned as a double.  Done in one step from
 * the double: no intermediate rounding to float, which could double-round. */
double kvo_round_bf16(double x)
{
    if (x != x || x == 0.0 || isinf(x)) return x;
    double ax = fabs(x);
    int e;
    (void)frexp(ax, &e);           /* ax = m * 2^e, m in [0.5, 1) */
    int q = e - 8;                 /* spacing of bf16 numbers in this binade */
    if (q < -133) q = -133;        /* subnormal spacing 2^-133 */
    double scaled = ldexp(ax, -q); /* exact: a power-of-two scaling */
    double r = nearbyint(scaled);  /* default mode: nearest, ties to even */
    double y = ldexp(r, q);
    if (y >= 0x1p128) y = INFINITY; /* rounded past the largest bf16, 0x1.fep127 */
    return x < 0 ? -y : y;
}

/* Round-to-nearest-even of a double to binary32 (C conversion, default mode). */
double kvo_round_f32(double x) { return (double)(float)x; }

void kvo_round_array(const double* x, int64_t n, int32_t dtype, double* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = dtype == 1 ? kvo_round_bf16(x[i]) : kvo_round_f32(x[i]);
}

/* ---- rotary position embedding ------------------------------------------- */

/* x, out: [T][H][D] (may alias); positions: [T].  Pair i of every head of
 * token t is rotated by angle positions[t] * base^(-2i/D):
 *   out[2i]   = x[2i] cos(a) - x[2i+1] sin(a)
 *   out[2i+1] = x[2i] sin(a) + x[2i+1] cos(a)                               */
int kvo_rope(const double* x, int64_t T, int32_t H, int32_t D,
             const int32_t* positions, double base, double* out)
{
    if (D <= 0 || (D & 1) || H <= 0 || T < 0) return KVO_ERR_ARG;
    for (int64_t t = 0; t < T; ++t) {
        double m = (double)positions[t];
        for (int32_t i = 0; i < D / 2; ++i) {
            double theta = pow(base, -2.0 * (double)i / (double)D);
            double a = m * theta;
            double c = cos(a), s = sin(a);
            for (int32_t h = 0; h < H; ++h) {
                int64_t o = (t * H + h) * (int64_t)D + 2 * i;
                double x0 = x[o], x1 = x[o + 1];
                out[o] = x0 * c - x1 * s;
                out[o + 1] = x0 * s + x1 * c;
            }
        }
    }
    return KVO_OK;
}

/* ---- KV-cache append ----------------------------------------------------- */

/* Physical slot of token position p of the sequence that owns block-table row
 * `row`: table[row][p / BS] * BS + p % BS.  Returns -1 when out of range. */
static int64_t slot_of(const int32_t* table, int32_t max_blocks, int32_t BS,
                       int64_t num_blocks, int32_t row, int32_t p)
{
    if (p < 0 || p / BS >= max_blocks) return -1;
    int32_t blk = table[(int64_t)row * max_blocks + p / BS];
    if (blk < 0 || blk >= num_blocks) return -1;
    return (int64_t)blk * BS + p % BS;
}

/* Writes k_rows[t] (already rotated and rounded by the caller) and v_rows[t]
 * into Kc/Vc at the slot of (seq_ids[t], positions[t]).
 * Kc, Vc: [num_blocks*BS][Hkv][D]; k_rows, v_rows: [T][Hkv][D]. */
int kvo_append(const double* k_rows, const double* v_rows, int64_t T,
               int32_t Hkv, int32_t D, const int32_t* positions,
               const int32_t* seq_ids, const int32_t* table, int32_t num_rows,
               int32_t max_blocks, int32_t BS, int64_t num_blocks, double* Kc,
               double* Vc)
{
    int64_t row_elems = (int64_t)Hkv * D;
    for (int64_t t = 0; t < T; ++t) {
        if (seq_ids[t] < 0 || seq_ids[t] >= num_rows) return KVO_ERR_INDEX;
        int64_t s = slot_of(table, max_blocks, BS, num_blocks, seq_ids[t], positions[t]);
        if (s < 0) return KVO_ERR_INDEX;
        memcpy(Kc + s * row_elems, k_rows + t * row_elems, sizeof(double) * row_elems);
        memcpy(Vc + s * row_elems, v_rows + t * row_elems, sizeof(double) * row_elems);
    }
    return KVO_OK;
}

/* ---- attention over the cache -------------------------------------------- */

typedef struct {
    const double *q, *Kc, *Vc;
    const int32_t *q_rows, *q_pos, *table;
    int64_t NQ, num_blocks;
    int32_t Hq, Hkv, D, max_blocks, BS;
    double scale;
    double* out;
    int64_t next;          /* work counter (query*Hq + head) */
    pthread_mutex_t lock;
    int status;
} attend_job;

/* One (query, head): out = sum_i softmax_i(q . K_i * scale) V_i over the keys
 * i = 0 .. q_pos (inclusive), K_i, V_i the cached rows of KV head
 * head / (Hq/Hkv).  Softmax is the two-pass max-subtracted definition. */
static int attend_one(attend_job* J, int64_t n, int32_t j, double* sbuf)
{
    const int32_t D = J->D, G = J->Hq / J->Hkv, h = j / G;
    const double* qv = J->q + (n * J->Hq + j) * (int64_t)D;
    double* o = J->out + (n * J->Hq + j) * (int64_t)D;
    int32_t L = J->q_pos[n] + 1; /* keys 0 .. q_pos */
    for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
    if (L <= 0) return KVO_OK;
    double mx = -INFINITY;
    for (int32_t i = 0; i < L; ++i) {
        int64_t s = slot_of(J->table, J->max_blocks, J->BS, J->num_blocks, J->q_rows[n], i);
        if (s < 0) return KVO_ERR_INDEX;
        const double* kv = J->Kc + (s * J->Hkv + h) * (int64_t)D;
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d) dot += qv[d] * kv[d];
        sbuf[i] = dot * J->scale;
        if (sbuf[i] > mx) mx = sbuf[i];
    }
    double den = 0.0;
    for (int32_t i = 0; i < L; ++i) {
        sbuf[i] = exp(sbuf[i] - mx);
        den += sbuf[i];
    }
    for (int32_t i = 0; i < L; ++i) {
        int64_t s = slot_of(J->table, J->max_blocks, J->BS, J->num_blocks, J->q_rows[n], i);
        const double* vv = J->Vc + (s * J->Hkv + h) * (int64_t)D;
        double w = sbuf[i] / den;
        for (int32_t d = 0; d < D; ++d) o[d] += w * vv[d];
    }
    return KVO_OK;
}

static void* attend_worker(void* arg)
{
    attend_job* J = (attend_job*)arg;
    int32_t maxL = 1;
    for (int64_t n = 0; n < J->NQ; ++n)
        if (J->q_pos[n] + 1 > maxL) maxL = J->q_pos[n] + 1;
    double* sbuf = (double*)malloc(sizeof(double) * (size_t)maxL);
    if (!sbuf) {
        pthread_mutex_lock(&J->lock);
        J->status = KVO_ERR_ARG;
        pthread_mutex_unlock(&J->lock);
        return NULL;
    }
    const int64_t total = J->NQ * J->Hq;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int64_t w = J->next;
        J->next += 16;
        pthread_mutex_unlock(&J->lock);
        if (w >= total) break;
        int64_t e = w + 16 < total ? w + 16 : total;
        for (int64_t u = w; u < e; ++u) {
            int rc = attend_one(J, u / J->Hq, (int32_t)(u % J->Hq), sbuf);
            if (rc != KVO_OK) {
                pthread_mutex_lock(&J->lock);
                J->status = rc;
                pthread_mutex_unlock(&J->lock);
            }
        }
    }
    free(sbuf);
    return NULL;
}

int kvo_num_cores(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }

/* Causal attention of NQ query tokens against the cache.
 * q: [NQ][Hq][D] (rotated and rounded like the stored keys);
 * q_rows[n]: block-table row of query n's sequence; q_pos[n]: its absolute
 * position -- it sees keys 0..q_pos[n].  A decode query has q_pos = L - 1;
 * prefill row r of a chunk with prefix P has q_pos = P + r.
 * out: [NQ][Hq][D].  nthreads <= 0 means all online cores. */
int kvo_attend(const double* q, int64_t NQ, int32_t Hq, int32_t Hkv, int32_t D,
               const int32_t* q_rows, const int32_t* q_pos, const double* Kc,
               const double* Vc, const int32_t* table, int32_t max_blocks,
               int32_t BS, int64_t num_blocks, double scale, double* out,
               int32_t nthreads)
{
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || BS <= 0) return KVO_ERR_ARG;
    attend_job J = {q, Kc, Vc, q_rows, q_pos, table, NQ, num_blocks, Hq, Hkv, D,
                    max_blocks, BS, scale, out, 0, PTHREAD_MUTEX_INITIALIZER, KVO_OK};
    int nt = nthreads > 0 ? nthreads : kvo_num_cores();
    if (nt < 1) nt = 1;
    if (nt > 256) nt = 256;
    pthread_t th[256];
    int started = 0;
    for (int i = 1; i < nt; ++i)
        if (pthread_create(&th[started], NULL, attend_worker, &J) == 0) ++started;
    attend_worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    return J.status;
}
