/*
 * Plain CPU oracle for the Ulysses-style sequence-parallel attention step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file; it is used by the tests, by the smoke check and by the
 * benchmark's CPU-baseline leg.  It shares no code, header or table with the
 * CUDA library.
 *
 * Source: "LTX-2 序列并行拆解: token 切分、all2all 换头与 runner 接入全链路"
 * (LTX-2 sequence-parallel breakdown), sections 补齐 (pad), 切分 (partition),
 * 换头 (head exchange), 还原 (restore), the correctness paragraph that closes
 * 还原, and the kernel paragraphs on SM rotation and the barrier.
 *
 * Everything is a plain index loop.  Layout routines move raw bytes (so they
 * are exact for any element type); attention accumulates in fp64.
 *
 * Layout conventions (readings of the pages, see the design notes):
 *   activations are row-major [B, T, H, D];
 *   rank r owns tokens [r*Tl, (r+1)*Tl) and heads [r*Hl, (r+1)*Hl);
 *   masks are uint8 with 1 = may attend.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* 补齐 (pad): the sequence dim is padded up to a multiple of world_size. */
int oracle_padded_len(int T, int W) {
    if (T < 0 || W <= 0) return -1;
    int T_pad = T;
    while (T_pad % W != 0) T_pad++;
    return T_pad;
}

/* Zero rows are appended after the T real rows of every batch item. */
void oracle_pad(const uint8_t *x, uint8_t *x_pad, int B, int T, int T_pad, size_t row_bytes) {
    for (int b = 0; b < B; b++) {
        for (int t = 0; t < T_pad; t++) {
            uint8_t *dst = x_pad + ((size_t)b * T_pad + t) * row_bytes;
            if (t < T) {
                const uint8_t *src = x + ((size_t)b * T + t) * row_bytes;
                for (size_t i = 0; i < row_bytes; i++) dst[i] = src[i];
            } else {
                for (size_t i = 0; i < row_bytes; i++) dst[i] = 0;
            }
        }
    }
}

/* Key-only padding mask (1,1,T_pad): key k is visible iff it is a real token. */
void oracle_pad_mask_key(uint8_t *mask_out, int T, int T_pad) {
    for (int k = 0; k < T_pad; k++) mask_out[k] = (k < T) ? 1 : 0;
}

/* A user (B,T,T) mask grows pad rows and columns: real rows keep the user's
 * entries over real keys; a pad query row sees every real key (so no row is
 * fully masked and none yields NaN); no row sees a pad key. */
void oracle_pad_mask_user(const uint8_t *user, uint8_t *mask_out, int B, int T, int T_pad) {
    for (int b = 0; b < B; b++) {
        for (int q = 0; q < T_pad; q++) {
            for (int k = 0; k < T_pad; k++) {
                uint8_t m;
                if (k >= T) {
                    m = 0;
                } else if (q >= T) {
                    m = 1;
                } else {
                    m = user[((size_t)b * T + q) * T + k] ? 1 : 0;
                }
                mask_out[((size_t)b * T_pad + q) * T_pad + k] = m;
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* 切分 (partition): total_tokens must divide evenly by world_size. */
int oracle_partition(int total_tokens, int W, int *starts, int *lens) {
    if (W <= 0 || total_tokens < 0) return 2;
    if (total_tokens % W != 0) return 1;
    int Tl = total_tokens / W;
    for (int r = 0; r < W; r++) {
        starts[r] = r * Tl;
        lens[r] = Tl;
    }
    return 0;
}

/* tile_modality_for_rank: rank r's slice of the token dim. */
void oracle_tile(const uint8_t *x_pad, uint8_t **shards, int W, int B, int T_pad, size_t row_bytes) {
    int Tl = T_pad / W;
    for (int r = 0; r < W; r++)
        for (int b = 0; b < B; b++)
            for (int t = 0; t < Tl; t++)
                memcpy(shards[r] + ((size_t)b * Tl + t) * row_bytes,
                       x_pad + ((size_t)b * T_pad + (size_t)r * Tl + t) * row_bytes, row_bytes);
}

/* ------------------------------------------------------------------ */
/* 换头 (head exchange).  Before: rank s holds [B, Tl, H, D] (its tokens, all
 * heads).  After: rank r holds [B, W*Tl, Hl, D] (all tokens, its heads). */
void oracle_send_recv_heads(uint8_t **shards, uint8_t **heads, int W, int B, int Tl, int H, int D,
                            size_t elt) {
    int Hl = H / W;
    int T_all = W * Tl;
    for (int r = 0; r < W; r++)
        for (int s = 0; s < W; s++)
            for (int b = 0; b < B; b++)
                for (int t = 0; t < Tl; t++)
                    for (int hl = 0; hl < Hl; hl++)
                        for (int d = 0; d < D; d++) {
                            size_t src = (((size_t)b * Tl + t) * H + (size_t)r * Hl + hl) * D + d;
                            size_t dst = (((size_t)b * T_all + (size_t)s * Tl + t) * Hl + hl) * D + d;
                            memcpy(heads[r] + dst * elt, shards[s] + src * elt, elt);
                        }
}

/* gather_heads: the exact inverse of the exchange above. */
void oracle_gather_heads(uint8_t **heads, uint8_t **shards, int W, int B, int Tl, int H, int D,
                         size_t elt) {
    int Hl = H / W;
    int T_all = W * Tl;
    for (int s = 0; s < W; s++)
        for (int r = 0; r < W; r++)
            for (int b = 0; b < B; b++)
                for (int t = 0; t < Tl; t++)
                    for (int hl = 0; hl < Hl; hl++)
                        for (int d = 0; d < D; d++) {
                            size_t dst = (((size_t)b * Tl + t) * H + (size_t)r * Hl + hl) * D + d;
                            size_t src = (((size_t)b * T_all + (size_t)s * Tl + t) * Hl + hl) * D + d;
                            memcpy(shards[s] + dst * elt, heads[r] + src * elt, elt);
                        }
}

/* ------------------------------------------------------------------ */
/* 还原 (restore): every rank's local output is padded to the longest shard
 * (all shards are Tl long, so nothing changes), all shards are gathered, each
 * is cropped to its real token count n_r = clamp(T_out - r*Tl, 0, Tl), and the
 * pieces are concatenated.  With T_out = W*Tl this is a plain concatenation. */
void oracle_gather_output(uint8_t **shards, uint8_t *out, int W, int B, int Tl, int T_out,
                          size_t row_bytes) {
    for (int b = 0; b < B; b++) {
        int pos = 0;
        for (int r = 0; r < W; r++) {
            int n_r = T_out - r * Tl;
            if (n_r < 0) n_r = 0;
            if (n_r > Tl) n_r = Tl;
            for (int t = 0; t < n_r; t++) {
                memcpy(out + ((size_t)b * T_out + pos) * row_bytes,
                       shards[r] + ((size_t)b * Tl + t) * row_bytes, row_bytes);
                pos++;
            }
        }
    }
}

/* unpad back to the caller's original length. */
void oracle_unpad(const uint8_t *x_pad, uint8_t *out, int B, int T_pad, int T, size_t row_bytes) {
    for (int b = 0; b < B; b++)
        for (int t = 0; t < T; t++)
            memcpy(out + ((size_t)b * T + t) * row_bytes, x_pad + ((size_t)b * T_pad + t) * row_bytes,
                   row_bytes);
}

/* ------------------------------------------------------------------ */
/* 2-D spatial split (LongCat-Video context parallel, "智能张量拆分"): the
 * world size is factored as split_h x split_w, the factor pair closest to a
 * square (split_h <= split_w); every frame of the latent grid [F, Hg, Wg] is
 * cut into split_h bands of height and each band into split_w pieces of
 * width; rank r = ih * split_w + iw receives piece (ih, iw) of every frame,
 * tokens in (frame, row, column) order.  Block sizes are Hg / split_h and
 * Wg / split_w; a grid they do not divide is an error (return 1). */
int oracle_optimal_split(int W, int *split_h, int *split_w) {
    if (W < 1) return 2;
    int best_a = 1, best_gap = W - 1;
    for (int a = 1; a <= W; a++) {
        if (W % a != 0) continue;
        int b = W / a;
        if (a > b) continue;
        if (b - a < best_gap) {
            best_gap = b - a;
            best_a = a;
        }
    }
    *split_h = best_a;
    *split_w = W / best_a;
    return 0;
}

int oracle_tile_2d(const uint8_t *x, uint8_t **shards, int B, int F, int Hg, int Wg, int split_h,
                   int split_w, size_t row_bytes) {
    if (split_h < 1 || split_w < 1 || Hg % split_h != 0 || Wg % split_w != 0) return 1;
    int bh = Hg / split_h, bw = Wg / split_w;
    for (int ih = 0; ih < split_h; ih++)
        for (int iw = 0; iw < split_w; iw++) {
            uint8_t *dst = shards[ih * split_w + iw];
            for (int b = 0; b < B; b++)
                for (int f = 0; f < F; f++)
                    for (int h = 0; h < bh; h++)
                        for (int w = 0; w < bw; w++) {
                            size_t d = (((size_t)b * F + f) * bh + h) * bw + w;
                            size_t g = (((size_t)b * F + f) * Hg + (size_t)ih * bh + h) * Wg +
                                       (size_t)iw * bw + w;
                            memcpy(dst + d * row_bytes, x + g * row_bytes, row_bytes);
                        }
        }
    return 0;
}

/* The inverse: every rank's piece goes back to its place in the grid. */
int oracle_gather_2d(uint8_t **shards, uint8_t *out, int B, int F, int Hg, int Wg, int split_h,
                     int split_w, size_t row_bytes) {
    if (split_h < 1 || split_w < 1 || Hg % split_h != 0 || Wg % split_w != 0) return 1;
    int bh = Hg / split_h, bw = Wg / split_w;
    for (int ih = 0; ih < split_h; ih++)
        for (int iw = 0; iw < split_w; iw++) {
            const uint8_t *src = shards[ih * split_w + iw];
            for (int b = 0; b < B; b++)
                for (int f = 0; f < F; f++)
                    for (int h = 0; h < bh; h++)
                        for (int w = 0; w < bw; w++) {
                            size_t d = (((size_t)b * F + f) * bh + h) * bw + w;
                            size_t g = (((size_t)b * F + f) * Hg + (size_t)ih * bh + h) * Wg +
                                       (size_t)iw * bw + w;
                            memcpy(out + g * row_bytes, src + d * row_bytes, row_bytes);
                        }
        }
    return 0;
}

/* ------------------------------------------------------------------ */
/* SM rotation: SM i writes rank i % world_size.  counts[r] = #SMs on rank r. */
void oracle_sm_rotation_counts(int n_sm, int W, int *counts) {
    for (int r = 0; r < W; r++) counts[r] = 0;
    for (int i = 0; i < n_sm; i++) counts[i % W]++;
}

/* ------------------------------------------------------------------ */
/* Attention on the local heads (section 换头): plain softmax attention.
 *   s_k = scale * sum_d Q[b,q,h,d] K[b,k,h,d]  over the visible keys k,
 *   O[b,q,h,:] = sum_k exp(s_k - max s) V[b,k,h,:] / sum_k exp(s_k - max s).
 * A row with no visible key yields 0.
 * mask_kind: 0 = every key visible; 1 = key vector mask[k] (length Tk);
 *            2 = full mask[b, q, k] of shape (B, Tq, Tk).
 * q: [B,Tq,H,D], k/v: [B,Tk,H,D] fp32 values; o: [B,Tq,H,D] fp64. */
typedef struct {
    const float *q, *k, *v;
    double *o;
    int B, Tq, Tk, H, D, mask_kind;
    const uint8_t *mask;
    double scale;
    const int64_t *rows; /* optional list of (b,q,h) triples; NULL = all */
    int64_t n_rows;
    int64_t begin, end; /* row range handled by this worker */
} attn_job;

static int visible(const attn_job *J, int b, int q, int k) {
    if (J->mask_kind == 0) return 1;
    if (J->mask_kind == 1) return J->mask[k] != 0;
    return J->mask[((size_t)b * J->Tq + q) * J->Tk + k] != 0;
}

static void attn_one_row(const attn_job *J, int b, int q, int h, double *out, double *s) {
    const int D = J->D, H = J->H;
    const float *qrow = J->q + (((size_t)b * J->Tq + q) * H + h) * D;
    double m = -INFINITY;
    int any = 0;
    for (int k = 0; k < J->Tk; k++) {
        if (!visible(J, b, q, k)) continue;
        const float *krow = J->k + (((size_t)b * J->Tk + k) * H + h) * D;
        double dot = 0.0;
        for (int d = 0; d < D; d++) dot += (double)qrow[d] * (double)krow[d];
        s[k] = J->scale * dot;
        if (!any || s[k] > m) m = s[k];
        any = 1;
    }
    for (int d = 0; d < D; d++) out[d] = 0.0;
    if (!any) return;
    double denom = 0.0;
    for (int k = 0; k < J->Tk; k++) {
        if (!visible(J, b, q, k)) continue;
        double p = exp(s[k] - m);
        denom += p;
        const float *vrow = J->v + (((size_t)b * J->Tk + k) * H + h) * D;
        for (int d = 0; d < D; d++) out[d] += p * (double)vrow[d];
    }
    for (int d = 0; d < D; d++) out[d] /= denom;
}

static void *attn_worker(void *arg) {
    attn_job *J = (attn_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->Tk > 0 ? J->Tk : 1));
    if (!s) return (void *)1;
    for (int64_t i = J->begin; i < J->end; i++) {
        int b, q, h;
        double *out;
        if (J->rows) {
            b = (int)J->rows[3 * i + 0];
            q = (int)J->rows[3 * i + 1];
            h = (int)J->rows[3 * i + 2];
            out = J->o + (size_t)i * J->D;
        } else {
            /* i enumerates (b, q, h) in row-major order */
            h = (int)(i % J->H);
            q = (int)((i / J->H) % J->Tq);
            b = (int)(i / ((int64_t)J->H * J->Tq));
            out = J->o + (size_t)i * J->D;
        }
        attn_one_row(J, b, q, h, out, s);
    }
    free(s);
    return NULL;
}

static int run_attention(attn_job base, int64_t n_total, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if ((int64_t)nthreads > n_total) nthreads = (int)(n_total > 0 ? n_total : 1);
    pthread_t tid[512];
    attn_job jobs[512];
    int64_t per = (n_total + nthreads - 1) / nthreads;
    int started = 0, rc = 0;
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = base;
        jobs[t].begin = (int64_t)t * per;
        jobs[t].end = jobs[t].begin + per < n_total ? jobs[t].begin + per : n_total;
        if (jobs[t].begin >= jobs[t].end) break;
        if (pthread_create(&tid[t], NULL, attn_worker, &jobs[t]) != 0) {
            rc = 3;
            break;
        }
        started++;
    }
    for (int t = 0; t < started; t++) {
        void *ret = NULL;
        pthread_join(tid[t], &ret);
        if (ret) rc = 4;
    }
    return rc;
}

/* Full attention: o is [B,Tq,H,D] fp64. */
int oracle_attention(const float *q, const float *k, const float *v, double *o, int B, int Tq, int Tk,
                     int H, int D, int mask_kind, const uint8_t *mask, double scale, int nthreads) {
    attn_job J = {q, k, v, o, B, Tq, Tk, H, D, mask_kind, mask, scale, NULL, 0, 0, 0};
    return run_attention(J, (int64_t)B * Tq * H, nthreads);
}

/* Selected rows: rows is an int64 array of (b, q, h) triples; o is [n_rows, D]. */
int oracle_attention_rows(const float *q, const float *k, const float *v, double *o, int B, int Tq,
                          int Tk, int H, int D, int mask_kind, const uint8_t *mask, double scale,
                          const int64_t *rows, int64_t n_rows, int nthreads) {
    attn_job J = {q, k, v, o, B, Tq, Tk, H, D, mask_kind, mask, scale, rows, n_rows, 0, 0};
    return run_attention(J, n_rows, nthreads);
}
