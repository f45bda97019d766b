/*
 * attn_oracle.c -- plain, slow fp64 CPU attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or constant with
 * the CUDA path.
 *
 * What it computes is the plain definition of scaled-dot-product attention,
 * written out one query row at a time with the probability row P materialised
 * (the same strategy as the unfused "attention_fwd_f32" / "attention_bwd_*"
 * kernels of forge src/kernels/attention.metal, which also keep P whole):
 *
 *   s_ij   = scale * sum_d Q[b,i,h,d] K[b,j,kv,d]        kv = h / (H/Hkv)
 *   st_ij  = softcap > 0 ? softcap * tanh(s_ij / softcap) : s_ij
 *   vis    = (!causal || j <= p) && (window == 0 || |p - j| < window)
 *            && (no mask || mask[b][j] > 0.5),          p = i + q_offset
 *   M_i    = max over visible j of st_ij,   L_i = sum over visible exp(st_ij - M_i)
 *   P_ij   = visible ? exp(st_ij - M_i) / L_i : 0
 *   O_i    = sum_j P_ij V_j,                LSE_i = M_i + ln L_i
 *
 * and, for the backward, with dO the upstream gradient of O:
 *
 *   D_i    = dO_i . O_i
 *   dP_ij  = dO_i . V_j
 *   dS_ij  = P_ij (dP_ij - D_i) * (softcap > 0 ? 1 - tanh^2(s_ij/softcap) : 1)
 *   dQ_i   = scale sum_j dS_ij K_j
 *   dK_j   = scale sum_{h in group} sum_i dS_ij Q_i
 *   dV_j   = sum_{h in group} sum_i P_ij dO_i
 *
 * Sources (page title, section):
 *  - scores, online/plain softmax, LSE: vision_rs flash_attn2.rs, "Forward"
 *    (score = q.k * softmax_scale; logsumexp saved as m + log l).
 *  - GQA head map h -> h / (H/Hkv): brotensor flash_attention.h,
 *    flash_attention_decode ("maps query head h to KV head h/(num_q_heads/
 *    num_kv_heads)"); forge attention.metal, attention_fwd_f32 (hkv = h / rep).
 *  - causal with offset and the window predicate |p - j| < window:
 *    ferrotensor engine/attention.rs, AttentionOptions doc comment.  With causal
 *    it gives keys [max(0, p-window+1), p], the set stated by brotensor
 *    flash_attention.h, flash_attention_decode "Gemma-2 extensions" and
 *    flash_attention_windowed_forward, and by forge attention.metal AttnParams
 *    ("keys kept, self incl.").  Without causal the pages disagree; this file
 *    takes the ferrotensor predicate (the only one written as a formula that
 *    reduces to the causal set).
 *  - softcap after the scale and before mask/max/exp, 0 = off: brotensor
 *    flash_attention.h, flash_attention_decode "Gemma-2 extensions".
 *  - key mask is a length-Tk fp32 array, a key kept iff mask > 0.5, combined
 *    multiplicatively: brotensor flash_attention.h, flash_attention_forward and
 *    flash_attention_backward contracts.
 *  - backward: vision_rs flash_attn2.rs, "Backward - dQ" and "Backward - dK / dV";
 *    forge attention.metal, attention_bwd_d_f32 (D = dO.O), attention_bwd_dq_f32
 *    and attention_bwd_dkv_f32 (softcap derivative, GQA group sum).
 *  - a row with no visible key: O = 0, LSE = -inf, no gradient (brotensor
 *    flash_attention.h: excluded positions "contribute nothing", a zero-length
 *    decode "writes zeros").  This is a reading; the pages do not define LSE there.
 *
 * The "_ex" entry points generalise two terms (every page's window, an additive mask):
 *
 *   vis    = (wl < 0 || j >= p - wl) && (wr < 0 || j <= p + wr) && (key mask)
 *   st_ij  = (softcap > 0 ? softcap * tanh(s_ij / softcap) : s_ij) + bias[b,h,i,j]
 *
 * A two-sided window [p - wl, p + wr] (negative = unbounded on that side) holds
 * every window the pages write: ferrotensor's |p - j| < w is (w-1, w-1), with
 * causal (w-1, 0); brotensor flash_attention_windowed_forward's bidirectional
 * window |r - j| <= w/2 is (w/2, w/2); forge attention.metal's one-sided window
 * (keys from i+1-window on) is (w-1, -1); causal alone is (-1, 0).  The bias is
 * ferrotensor's additive mask [batch, heads, seq_q, seq_k] with size-1
 * dimensions broadcast (stride 0; ferrotensor engine/attention.rs,
 * mask_strides), added to the scaled score; -inf entries drop the pair.  It
 * enters the backward only through P (dS has no bias term).
 *
 * Layouts: q, o, do, dq are [B][Tq][H*hd]; k, v, dk, dv are [B][Tk][Hkv*hd];
 * lse is [B][H][Tq]; key_mask (optional) is key_mask[b*mask_bstride + j].
 * All arrays are row-major fp64.  Functions return 0, or -1 on bad arguments.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int B, Tq, Tk, H, Hkv, hd;
    double scale;
    int causal, window;
    double softcap;
    long long q_offset;
    const double* key_mask;
    long long mask_bstride;
    int ext;             /* 1: the two-sided window and the bias below */
    long long wl, wr;    /* window [p - wl, p + wr]; negative = unbounded */
    const double* bias;  /* bias[b*bs[0] + h*bs[1] + i*bs[2] + j*bs[3]] or NULL */
    long long bs[4];
} attn_dims;

static int dims_ok(const attn_dims* d)
{
    if (d->B < 0 || d->Tq < 0 || d->Tk < 0 || d->H <= 0 || d->Hkv <= 0 || d->hd <= 0) return 0;
    if (d->H % d->Hkv != 0) return 0;
    if (d->window < 0 || d->softcap < 0 || d->q_offset < 0) return 0;
    return 1;
}

/* visibility of key j to the query at absolute position p (see header). */
static int visible(const attn_dims* d, int b, long long p, long long j)
{
    if (d->ext) {
        if (d->wl >= 0 && j < p - d->wl) return 0;
        if (d->wr >= 0 && j > p + d->wr) return 0;
    } else {
        if (d->causal && j > p) return 0;
        if (d->window > 0) {
            long long gap = p - j;
            if (gap < 0) gap = -gap;
            if (gap >= d->window) return 0;
        }
    }
    if (d->key_mask && !(d->key_mask[(long long)b * d->mask_bstride + j] > 0.5)) return 0;
    return 1;
}

static const double* q_row(const attn_dims* d, const double* q, int b, int i, int h)
{
    return q + ((long long)b * d->Tq + i) * (long long)d->H * d->hd + (long long)h * d->hd;
}

static const double* kv_row(const attn_dims* d, const double* k, int b, int j, int kvh)
{
    return k + ((long long)b * d->Tk + j) * (long long)d->Hkv * d->hd + (long long)kvh * d->hd;
}

/*
 * One query row (b, h, i): fills raw[j] = s_ij (uncapped, scaled), prob[j] = P_ij,
 * writes o_i (hd values) and returns LSE_i.  P is materialised over all Tk keys.
 */
static double attend_row(const attn_dims* d, const double* q, const double* k, const double* v,
                         int b, int h, int i, double* raw, double* prob, double* o_i)
{
    const int G = d->H / d->Hkv;
    const int kvh = h / G;
    const long long p = (long long)i + d->q_offset;
    const double* qi = q_row(d, q, b, i, h);
    double m = -INFINITY;
    for (int j = 0; j < d->Tk; ++j) {
        const double* kj = kv_row(d, k, b, j, kvh);
        double s = 0.0;
        for (int e = 0; e < d->hd; ++e) s += qi[e] * kj[e];
        s *= d->scale;
        raw[j] = s;
        if (visible(d, b, p, j)) {
            double st = d->softcap > 0 ? d->softcap * tanh(s / d->softcap) : s;
            if (d->bias)
                st += d->bias[(long long)b * d->bs[0] + (long long)h * d->bs[1] + (long long)i * d->bs[2] +
                              (long long)j * d->bs[3]];
            prob[j] = st;
            if (st > m) m = st;
        } else {
            prob[j] = -INFINITY;
        }
    }
    for (int e = 0; e < d->hd; ++e) o_i[e] = 0.0;
    if (m == -INFINITY) {
        for (int j = 0; j < d->Tk; ++j) prob[j] = 0.0;
        return -INFINITY;
    }
    double l = 0.0;
    for (int j = 0; j < d->Tk; ++j) {
        double e = prob[j] == -INFINITY ? 0.0 : exp(prob[j] - m);
        prob[j] = e;
        l += e;
    }
    for (int j = 0; j < d->Tk; ++j) prob[j] /= l;
    for (int j = 0; j < d->Tk; ++j) {
        if (prob[j] == 0.0) continue;
        const double* vj = kv_row(d, v, b, j, kvh);
        for (int e = 0; e < d->hd; ++e) o_i[e] += prob[j] * vj[e];
    }
    return m + log(l);
}

static attn_dims make_dims(int B, int Tq, int Tk, int H, int Hkv, int hd, double scale, int causal,
                           int window, double softcap, long long q_offset, const double* key_mask,
                           long long mask_bstride)
{
    attn_dims d;
    d.B = B; d.Tq = Tq; d.Tk = Tk; d.H = H; d.Hkv = Hkv; d.hd = hd;
    d.scale = scale; d.causal = causal; d.window = window; d.softcap = softcap;
    d.q_offset = q_offset; d.key_mask = key_mask; d.mask_bstride = mask_bstride;
    d.ext = 0; d.wl = d.wr = -1; d.bias = NULL;
    d.bs[0] = d.bs[1] = d.bs[2] = d.bs[3] = 0;
    return d;
}

static attn_dims make_dims_ex(int B, int Tq, int Tk, int H, int Hkv, int hd, double scale, long long wl,
                              long long wr, double softcap, long long q_offset, const double* key_mask,
                              long long mask_bstride, const double* bias, const long long* bs)
{
    attn_dims d = make_dims(B, Tq, Tk, H, Hkv, hd, scale, 0, 0, softcap, q_offset, key_mask, mask_bstride);
    d.ext = 1; d.wl = wl; d.wr = wr; d.bias = bias;
    for (int e = 0; e < 4; ++e) d.bs[e] = bias ? bs[e] : 0;
    return d;
}

static int fwd_dims(const attn_dims* dp, const double* q, const double* k, const double* v, double* o,
                    double* lse)
{
    const attn_dims d = *dp;
    const int B = d.B, Tq = d.Tq, Tk = d.Tk, H = d.H, hd = d.hd;
    if (!dims_ok(&d)) return -1;
    int failed = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h) {
            double* raw = (double*)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
            double* prob = (double*)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
            if (!raw || !prob) {
#pragma omp atomic write
                failed = 1;
                free(raw); free(prob);
                continue;
            }
            for (int i = 0; i < Tq; ++i) {
                double* oi = o + ((long long)b * Tq + i) * (long long)H * hd + (long long)h * hd;
                double l = attend_row(&d, q, k, v, b, h, i, raw, prob, oi);
                if (lse) lse[((long long)b * H + h) * Tq + i] = l;
            }
            free(raw);
            free(prob);
        }
    return failed ? -1 : 0;
}

/* Forward: o [B][Tq][H*hd], lse [B][H][Tq] (lse may be NULL). */
int oracle_attn_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                    int B, int Tq, int Tk, int H, int Hkv, int hd, double scale, int causal,
                    int window, double softcap, long long q_offset, const double* key_mask,
                    long long mask_bstride)
{
    attn_dims d = make_dims(B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset,
                            key_mask, mask_bstride);
    return fwd_dims(&d, q, k, v, o, lse);
}

/* The same with the two-sided window and the additive bias (see header). */
int oracle_attn_fwd_ex(const double* q, const double* k, const double* v, double* o, double* lse,
                       int B, int Tq, int Tk, int H, int Hkv, int hd, double scale, long long wl,
                       long long wr, double softcap, long long q_offset, const double* key_mask,
                       long long mask_bstride, const double* bias, const long long* bs)
{
    attn_dims d = make_dims_ex(B, Tq, Tk, H, Hkv, hd, scale, wl, wr, softcap, q_offset, key_mask,
                               mask_bstride, bias, bs);
    return fwd_dims(&d, q, k, v, o, lse);
}

static int probs_dims(const attn_dims* dp, const double* q, const double* k, const double* v, double* P,
                      int b, int h)
{
    const attn_dims d = *dp;
    const int B = d.B, Tq = d.Tq, Tk = d.Tk, H = d.H, hd = d.hd;
    if (!dims_ok(&d) || b < 0 || b >= B || h < 0 || h >= H) return -1;
    double* raw = (double*)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
    double* oi = (double*)malloc(sizeof(double) * (size_t)hd);
    if (!raw || !oi) { free(raw); free(oi); return -1; }
    for (int i = 0; i < Tq; ++i) attend_row(&d, q, k, v, b, h, i, raw, P + (long long)i * Tk, oi);
    free(raw);
    free(oi);
    return 0;
}

/* The probability matrix P [Tq][Tk] of one (b, h), for invariant checks. */
int oracle_attn_probs(const double* q, const double* k, const double* v, double* P, int b, int h,
                      int B, int Tq, int Tk, int H, int Hkv, int hd, double scale, int causal,
                      int window, double softcap, long long q_offset, const double* key_mask,
                      long long mask_bstride)
{
    attn_dims d = make_dims(B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset,
                            key_mask, mask_bstride);
    return probs_dims(&d, q, k, v, P, b, h);
}

int oracle_attn_probs_ex(const double* q, const double* k, const double* v, double* P, int b, int h,
                         int B, int Tq, int Tk, int H, int Hkv, int hd, double scale, long long wl,
                         long long wr, double softcap, long long q_offset, const double* key_mask,
                         long long mask_bstride, const double* bias, const long long* bs)
{
    attn_dims d = make_dims_ex(B, Tq, Tk, H, Hkv, hd, scale, wl, wr, softcap, q_offset, key_mask,
                               mask_bstride, bias, bs);
    return probs_dims(&d, q, k, v, P, b, h);
}

/*
 * Backward straight from the definition: P is rebuilt row by row from the
 * inputs (not from a saved LSE), O and D come from that P.  dq/dk/dv are
 * overwritten.  Parallel over (b, kv head) so that each thread owns its dK/dV
 * rows (the GQA group sum of forge attention.metal, attention_bwd_dkv_f32).
 */
static int bwd_dims(const attn_dims* dp, const double* q, const double* k, const double* v,
                    const double* dout, double* dq, double* dk, double* dv)
{
    const attn_dims d = *dp;
    const int B = d.B, Tq = d.Tq, Tk = d.Tk, H = d.H, Hkv = d.Hkv, hd = d.hd;
    const double scale = d.scale, softcap = d.softcap;
    if (!dims_ok(&d)) return -1;
    const int G = H / Hkv;
    int failed = 0;
#pragma omp parallel for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b)
        for (int kvh = 0; kvh < Hkv; ++kvh) {
            double* raw = (double*)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
            double* prob = (double*)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
            double* oi = (double*)malloc(sizeof(double) * (size_t)hd);
            if (!raw || !prob || !oi) {
#pragma omp atomic write
                failed = 1;
                free(raw); free(prob); free(oi);
                continue;
            }
            for (int j = 0; j < Tk; ++j) {
                double* dkj = dk + ((long long)b * Tk + j) * (long long)Hkv * hd + (long long)kvh * hd;
                double* dvj = dv + ((long long)b * Tk + j) * (long long)Hkv * hd + (long long)kvh * hd;
                memset(dkj, 0, sizeof(double) * (size_t)hd);
                memset(dvj, 0, sizeof(double) * (size_t)hd);
            }
            for (int h = kvh * G; h < (kvh + 1) * G; ++h) {
                for (int i = 0; i < Tq; ++i) {
                    const long long qoff = ((long long)b * Tq + i) * (long long)H * hd + (long long)h * hd;
                    const double* qi = q + qoff;
                    const double* doi = dout + qoff;
                    double* dqi = dq + qoff;
                    memset(dqi, 0, sizeof(double) * (size_t)hd);
                    attend_row(&d, q, k, v, b, h, i, raw, prob, oi);
                    double Di = 0.0;
                    for (int e = 0; e < hd; ++e) Di += doi[e] * oi[e];
                    for (int j = 0; j < Tk; ++j) {
                        const double pij = prob[j];
                        if (pij == 0.0) continue; /* invisible (or underflowed): no term */
                        const double* kj = kv_row(&d, k, b, j, kvh);
                        const double* vj = kv_row(&d, v, b, j, kvh);
                        double* dkj = dk + ((long long)b * Tk + j) * (long long)Hkv * hd + (long long)kvh * hd;
                        double* dvj = dv + ((long long)b * Tk + j) * (long long)Hkv * hd + (long long)kvh * hd;
                        double dpij = 0.0;
                        for (int e = 0; e < hd; ++e) dpij += doi[e] * vj[e];
                        double ds = pij * (dpij - Di);
                        if (softcap > 0) {
                            double t = tanh(raw[j] / softcap);
                            ds *= 1.0 - t * t;
                        }
                        for (int e = 0; e < hd; ++e) {
                            dqi[e] += scale * ds * kj[e];
                            dkj[e] += scale * ds * qi[e];
                            dvj[e] += pij * doi[e];
                        }
                    }
                }
            }
            free(raw);
            free(prob);
            free(oi);
        }
    return failed ? -1 : 0;
}

int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout,
                    double* dq, double* dk, double* dv, int B, int Tq, int Tk, int H, int Hkv,
                    int hd, double scale, int causal, int window, double softcap,
                    long long q_offset, const double* key_mask, long long mask_bstride)
{
    attn_dims d = make_dims(B, Tq, Tk, H, Hkv, hd, scale, causal, window, softcap, q_offset,
                            key_mask, mask_bstride);
    return bwd_dims(&d, q, k, v, dout, dq, dk, dv);
}

int oracle_attn_bwd_ex(const double* q, const double* k, const double* v, const double* dout,
                       double* dq, double* dk, double* dv, int B, int Tq, int Tk, int H, int Hkv,
                       int hd, double scale, long long wl, long long wr, double softcap,
                       long long q_offset, const double* key_mask, long long mask_bstride,
                       const double* bias, const long long* bs)
{
    attn_dims d = make_dims_ex(B, Tq, Tk, H, Hkv, hd, scale, wl, wr, softcap, q_offset, key_mask,
                               mask_bstride, bias, bs);
    return bwd_dims(&d, q, k, v, dout, dq, dk, dv);
}

/* Threads the OpenMP runtime will use (reported next to oracle timings). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
