/*
 * k6_oracle.c -- plain, slow fp64 CPU oracle for the joint-sequence attention
 * hot path of long-context video DiTs.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes, and where the pages say so:
 *   - Full non-causal multi-head attention softmax(Q K^T * scale) V over the
 *     joint sequence (video tokens followed by the text/audio "joint tensors"):
 *     xDiT PR #586 "KV-cache and joint tensors for USP", section "How?" and the
 *     USP dispatch listing (`_attention(query, key, value, is_causal=...)`);
 *     "Context Parallelism in vLLM Omni Neuron", section "Self-Attention with
 *     Context Parallelism" ("local Q x full K/V", `_nf_attend(q, k, v, scale)`).
 *     Scale = 1/sqrt(d) [reading: the page shows `self.scale` but not its value].
 *   - Rotary embeddings on Q and K only, from per-token cos/sin tables that can
 *     be sliced by sequence range: "Context Parallelism in vLLM Omni Neuron",
 *     sections "Self-Attention with Context Parallelism"
 *     (`apply_rotary_emb_wan`) and "Positional Embedding Handling"; vLLM-Omni
 *     recipe "Kandinsky 6 TI2VA -- H100", parallel features list ("visual
 *     tokens (and their RoPE) are sharded").  The exact rotation is a reading
 *     (the pages print no formula): each axis (t, h, w) owns a contiguous run of
 *     d_a head dims in that order; pair i of that run, i.e. dims (2i, 2i+1),
 *     turns by pos_a * theta^(-2i/d_a) as the complex product
 *     (x + i y) * exp(i angle); positions are 0-based grid indices; joint
 *     tokens are not rotated, or (joint_rope = 1) turn over the full head dim
 *     by their 0-based joint index.
 *   - Per-chunk partials (O_c, LSE_c) over a contiguous K/V range and their
 *     log-sum-exp merge, the arithmetic ring attention splits across ranks:
 *     "Context Parallelism in vLLM Omni Neuron", sections "Ring attention
 *     (current implementation)" and "Scaling Properties".  The merge formula
 *     is a reading: LSE = log sum_c exp(LSE_c), out = sum_c exp(LSE_c - LSE) O_c.
 *   - Cross-attention, queries of one stream over the keys/values of another
 *     (Sq != Sk, no rotary): vLLM-Omni recipe "Kandinsky 6 TI2VA -- H100",
 *     section "Notes" (in sequence parallelism the audio queries attend over
 *     every visual token); "Context Parallelism in vLLM Omni Neuron", "Forward
 *     Pass Flow" (cross-attention reads the encoder states unsharded).
 *   - The constant-max variant of ring attention ("Context Parallelism in vLLM
 *     Omni Neuron", "Related information": `ring_attention_const_max_fwd`
 *     takes the softmax max as a runtime bound instead of a running max).
 *     Read as the Cauchy-Schwarz bound M_i = |q~_i| * max_j |k~_j| / sqrt(d)
 *     >= max_j s_ij; the attention result does not depend on which bound is
 *     used, so the oracle supplies only the bound itself.
 *   - The backward pass of the attention (gradients of q, k, v and the joint
 *     keys/values for a given output gradient).  The pages describe inference
 *     only; this is the plain chain rule of softmax(Q K^T / sqrt(d)) V:
 *     D_i = sum_e dO_ie O_ie, dV = P^T dO, dS = P o (dO V^T - D),
 *     dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d), on the rotated q and k.
 *   - QK-norm before the rotary embedding: "Context Parallelism in vLLM Omni
 *     Neuron", "Self-Attention with Context Parallelism" (`norm_q(q)`,
 *     `norm_k(k)` on the projected rows before they are split into heads) and
 *     "Distributed Normalization" (an RMS statistic over the hidden dim).  Read
 *     as RMSNorm over each token's full hidden row of H*d values:
 *     y = x / sqrt(mean(x^2) + eps) * w.
 *   - The sequence-partitioned <-> head-partitioned relayout that Ulysses does
 *     with all-to-all: xDiT PR #586 USP listing (`_ft_c_input_all_to_all`,
 *     `_ft_c_output_all_to_all`); "Context Parallelism in vLLM Omni Neuron",
 *     section "Comparison with Other CP Strategies".  Index map (reading), with
 *     Sl = S/P and Hl = H/P:
 *       head[p][b][r*Sl + s][hh][e] = seq[r][b][s][p*Hl + hh][e].
 *
 * Layouts: q [B][Sq][H][d] with Sq = Nv + Nj (video rows first, joint rows at
 * the rear); k, v [B][Nv][H][d]; joint_k, joint_v [B][Nj][H][d].  The K/V
 * sequence is concat(k, joint_k) along the token axis.  Outputs are double.
 *
 * Everything is fp64.  bf16 and f32 inputs are widened exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { K6O_F32 = 0, K6O_BF16 = 1, K6O_F64 = 2 };

/* K6O_MUTANT plants one deliberate mistake, for the test that checks the pins
 * catch it (tests/test_oracle_mutants.py builds these variants separately).
 * 0 (the default) is the oracle itself. */
#ifndef K6O_MUTANT
#define K6O_MUTANT 0
#endif

typedef struct {
    int B, H, d;
    long Nv, Nj;              /* video tokens, joint tokens */
    int grid_t, grid_h, grid_w; /* Nv = grid_t * grid_h * grid_w */
    int axis_dim[3];          /* head dims owned by the t, h, w axes; sum = d */
    double theta;             /* rotary base */
    int joint_rope;           /* 0: joint tokens unrotated; 1: 1-D over full d */
} k6o_geom;

/* Exact widening of one element of a typed buffer to double. */
static double load_elem(const void *p, int type, size_t i) {
    if (type == K6O_F64) return ((const double *)p)[i];
    if (type == K6O_F32) return (double)((const float *)p)[i];
    /* bf16: the upper 16 bits of an IEEE binary32 */
    uint32_t bits = (uint32_t)((const uint16_t *)p)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

int k6o_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void k6o_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

static int geom_ok(const k6o_geom *g) {
    if (g->B < 1 || g->H < 1 || g->d < 2 || (g->d & 1)) return 0;
    if (g->Nv < 0 || g->Nj < 0) return 0;
    if ((long)g->grid_t * g->grid_h * g->grid_w != g->Nv) return 0;
    int sum = 0;
    for (int a = 0; a < 3; a++) {
        if (g->axis_dim[a] < 0 || (g->axis_dim[a] & 1)) return 0;
        sum += g->axis_dim[a];
    }
    return sum == g->d;
}

/* Rotate pair (x[2i], x[2i+1]) by `angle`: complex product (x + iy) e^{i angle}. */
static void rotate_pair(double *x, int i, double angle) {
    double c = cos(angle), s = sin(angle);
    double a = x[2 * i], b = x[2 * i + 1];
#if K6O_MUTANT == 1
    x[2 * i] = a * c + b * s; /* planted: wrong sign */
#else
    x[2 * i] = a * c - b * s;
#endif
    x[2 * i + 1] = a * s + b * c;
}

/* Rotary embedding of one head vector x[0..d) of token n (in place). */
void k6o_rope_vec(const k6o_geom *g, long n, double *x) {
    if (n < g->Nv) {
        long hw = (long)g->grid_h * g->grid_w;
        long pos[3];
#if K6O_MUTANT == 3
        pos[1] = n / hw;               /* planted: t and h swapped */
        pos[0] = (n / g->grid_w) % g->grid_h;
#else
        pos[0] = n / hw;               /* t */
        pos[1] = (n / g->grid_w) % g->grid_h; /* h */
#endif
        pos[2] = n % g->grid_w;        /* w */
        int off = 0;                   /* first dim owned by the axis */
        for (int a = 0; a < 3; a++) {
            int da = g->axis_dim[a];
            for (int i = 0; i < da / 2; i++) {
#if K6O_MUTANT == 2
                double omega = pow(g->theta, -1.0 * i / da); /* planted: dropped factor 2 */
#else
                double omega = pow(g->theta, -2.0 * i / da);
#endif
                rotate_pair(x + off, i, (double)pos[a] * omega);
            }
            off += da;
        }
    } else if (g->joint_rope == 1) {
        long j = n - g->Nv;
        for (int i = 0; i < g->d / 2; i++) {
            double omega = pow(g->theta, -2.0 * i / g->d);
            rotate_pair(x, i, (double)j * omega);
        }
    }
    /* joint_rope == 0: joint tokens keep their values */
}

/* Rotary embedding of a whole [B][S][H][d] tensor (S = Nv + Nj) into y. */
int k6o_rope(const k6o_geom *g, const void *x, int type, double *y) {
    if (!geom_ok(g)) return -1;
    long S = g->Nv + g->Nj;
    long rows = (long)g->B * S * g->H;
    int d = g->d;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; r++) {
        long n = (r / g->H) % S;
        double *out = y + (size_t)r * d;
        for (int e = 0; e < d; e++) out[e] = load_elem(x, type, (size_t)r * d + e);
        k6o_rope_vec(g, n, out);
    }
    return 0;
}

static const void *kv_ptr(const k6o_geom *g, long n, int b, int h, const void *video, const void *joint,
                          size_t *off);

/*
 * Row bounds of the constant-max softmax, from rotated (or unrotated when
 * rope = 0) q and keys: bound [B][H][Sq] = |q~_i| * max_j |k~_j| / sqrt(d),
 * the maximum over all Sk = Nv + Nj keys of the (b, h) pair.
 */
int k6o_row_bounds(const k6o_geom *g, int rope, const void *q, const void *k, const void *jk, int type,
                   double *bound) {
    if (!geom_ok(g)) return -1;
    const long S = g->Nv + g->Nj;
    const int d = g->d, H = g->H;
    for (int b = 0; b < g->B; b++)
        for (int h = 0; h < H; h++) {
            double kmax = 0.0;
#pragma omp parallel
            {
                double *x = (double *)malloc(sizeof(double) * d);
                double local = 0.0;
#pragma omp for schedule(static)
                for (long n = 0; n < S; n++) {
                    size_t off;
                    const void *src = kv_ptr(g, n, b, h, k, jk, &off);
                    for (int e = 0; e < d; e++) x[e] = load_elem(src, type, off + e);
                    if (rope) k6o_rope_vec(g, n, x);
                    double ss = 0.0;
                    for (int e = 0; e < d; e++) ss += x[e] * x[e];
                    if (sqrt(ss) > local) local = sqrt(ss);
                }
#pragma omp critical
                if (local > kmax) kmax = local;
                free(x);
            }
#pragma omp parallel
            {
                double *x = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(static)
                for (long i = 0; i < S; i++) {
                    const size_t off = (((size_t)b * S + i) * H + h) * d;
                    for (int e = 0; e < d; e++) x[e] = load_elem(q, type, off + e);
                    if (rope) k6o_rope_vec(g, i, x);
                    double ss = 0.0;
                    for (int e = 0; e < d; e++) ss += x[e] * x[e];
                    bound[((size_t)b * H + h) * S + i] = sqrt(ss) * kmax / sqrt((double)d);
                }
                free(x);
            }
        }
    return 0;
}

/* RMSNorm of `rows` rows of n values each: y = x / sqrt(mean(x^2) + eps) * w. */
int k6o_rms_norm(const void *x, int type, long rows, long n, const double *w, double eps, double *y) {
    if (rows < 0 || n < 1 || eps < 0) return -1;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; r++) {
        double ss = 0.0;
        for (long e = 0; e < n; e++) {
            double v = load_elem(x, type, (size_t)r * n + e);
            ss += v * v;
        }
        double inv = 1.0 / sqrt(ss / (double)n + eps);
        for (long e = 0; e < n; e++) y[(size_t)r * n + e] = load_elem(x, type, (size_t)r * n + e) * inv * w[e];
    }
    return 0;
}

/* Element offset of token n (of the concatenated K/V sequence), batch b,
 * head h, dim 0, and which buffer holds it. */
static const void *kv_ptr(const k6o_geom *g, long n, int b, int h, const void *video,
                          const void *joint, size_t *off) {
    if (n < g->Nv) {
        *off = (((size_t)b * g->Nv + n) * g->H + h) * g->d;
        return video;
    }
    *off = (((size_t)b * g->Nj + (n - g->Nv)) * g->H + h) * g->d;
#if K6O_MUTANT == 8
    return video; /* planted: joint rows read from the video tensor */
#else
    return joint;
#endif
}

/*
 * Attention of the given query rows over keys [kv_begin, kv_end) of the
 * concatenated K/V sequence.
 *   rope: 1 = rotate Q and K here (inputs are raw); 0 = inputs pre-rotated.
 *   rows[r] in [0, Sq); out [B][nrows][H][d]; lse [B][H][nrows] (natural log
 *   of the sum of exp of the scaled logits).
 * Per (b, h): rotate the K range once, then for each row
 *   s_j = q~ . k~_j / sqrt(d),  m = max_j s_j,
 *   LSE = m + log sum_j exp(s_j - m),  out = sum_j exp(s_j - LSE) v_j.
 */
int k6o_attention(const k6o_geom *g, int rope, const void *q, const void *k, const void *v,
                  const void *jk, const void *jv, int type, long kv_begin, long kv_end,
                  const long *rows, long nrows, double *out, double *lse) {
    if (!geom_ok(g)) return -1;
    long S = g->Nv + g->Nj;
    if (kv_begin < 0 || kv_end > S || kv_begin >= kv_end) return -2;
    for (long r = 0; r < nrows; r++)
        if (rows[r] < 0 || rows[r] >= S) return -3;
    int d = g->d, H = g->H;
    long L = kv_end - kv_begin;
#if K6O_MUTANT == 4
    double scale = 1.0 / (double)d; /* planted: 1/d */
#else
    double scale = 1.0 / sqrt((double)d);
#endif
    double *kr = (double *)malloc(sizeof(double) * (size_t)L * d);
    double *vr = (double *)malloc(sizeof(double) * (size_t)L * d);
    if (!kr || !vr) { free(kr); free(vr); return -4; }

    for (int b = 0; b < g->B; b++) {
        for (int h = 0; h < H; h++) {
            /* the key/value rows of this head, keys rotated at their own positions */
#pragma omp parallel for schedule(static)
            for (long j = 0; j < L; j++) {
                long n = kv_begin + j;
                size_t off;
                const void *kb = kv_ptr(g, n, b, h, k, jk, &off);
                const void *vb = kv_ptr(g, n, b, h, v, jv, &off);
                for (int e = 0; e < d; e++) {
                    kr[(size_t)j * d + e] = load_elem(kb, type, off + e);
                    vr[(size_t)j * d + e] = load_elem(vb, type, off + e);
                }
                if (rope) k6o_rope_vec(g, n, kr + (size_t)j * d);
            }
#pragma omp parallel
            {
                double *qv = (double *)malloc(sizeof(double) * d);
                double *s = (double *)malloc(sizeof(double) * (size_t)L);
#pragma omp for schedule(dynamic, 1)
                for (long r = 0; r < nrows; r++) {
                    long i = rows[r];
                    size_t qoff = (((size_t)b * S + i) * H + h) * d;
                    for (int e = 0; e < d; e++) qv[e] = load_elem(q, type, qoff + e);
                    if (rope) k6o_rope_vec(g, i, qv);
                    double m = -INFINITY;
                    for (long j = 0; j < L; j++) {
                        double acc = 0.0;
                        const double *kj = kr + (size_t)j * d;
                        for (int e = 0; e < d; e++) acc += qv[e] * kj[e];
                        s[j] = acc * scale;
                        if (s[j] > m) m = s[j];
                    }
                    double sum = 0.0;
                    for (long j = 0; j < L; j++) sum += exp(s[j] - m);
#if K6O_MUTANT == 7
                    double lse_i = log(sum); /* planted: dropped the max */
#else
                    double lse_i = m + log(sum);
#endif
                    double *o = out + (((size_t)b * nrows + r) * H + h) * d;
                    for (int e = 0; e < d; e++) o[e] = 0.0;
                    for (long j = 0; j < L; j++) {
                        double p = exp(s[j] - lse_i);
                        const double *vj = vr + (size_t)j * d;
                        for (int e = 0; e < d; e++) o[e] += p * vj[e];
                    }
                    lse[((size_t)b * H + h) * nrows + r] = lse_i;
                }
                free(qv);
                free(s);
            }
        }
    }
    free(kr);
    free(vr);
    return 0;
}

/*
 * Cross-attention: Sq query rows of q [B][Sq][H][d] over keys [kv_begin,
 * kv_end) of k, v [B][Sk][H][d]; no rotary.  out [B][Sq][H][d], lse
 * [B][H][Sq], the same definitions as k6o_attention.
 */
int k6o_cross_attention(int B, int H, int d, long Sq, long Sk, const void *q, const void *k, const void *v,
                        int type, long kv_begin, long kv_end, double *out, double *lse) {
    if (B < 1 || H < 1 || d < 1 || Sq < 0 || Sk < 1) return -1;
    if (kv_begin < 0 || kv_end > Sk || kv_begin >= kv_end) return -2;
    const long L = kv_end - kv_begin;
    const double scale = 1.0 / sqrt((double)d);
    const long tasks = (long)B * H * Sq;
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        if (!s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long t = 0; t < tasks; t++) {
            if (!s) continue;
            const long i = t % Sq;
            const int h = (int)((t / Sq) % H);
            const int b = (int)(t / ((long)Sq * H));
            const size_t qoff = (((size_t)b * Sq + i) * H + h) * d;
            double m = -INFINITY;
            for (long j = 0; j < L; j++) {
                const size_t koff = (((size_t)b * Sk + kv_begin + j) * H + h) * d;
                double acc = 0.0;
                for (int e = 0; e < d; e++) acc += load_elem(q, type, qoff + e) * load_elem(k, type, koff + e);
                s[j] = acc * scale;
                if (s[j] > m) m = s[j];
            }
            double sum = 0.0;
            for (long j = 0; j < L; j++) sum += exp(s[j] - m);
            const double lse_i = m + log(sum);
            double *o = out + qoff;
            for (int e = 0; e < d; e++) o[e] = 0.0;
            for (long j = 0; j < L; j++) {
                const double pj = exp(s[j] - lse_i);
                const size_t voff = (((size_t)b * Sk + kv_begin + j) * H + h) * d;
                for (int e = 0; e < d; e++) o[e] += pj * load_elem(v, type, voff + e);
            }
            lse[((size_t)b * H + h) * Sq + i] = lse_i;
        }
        free(s);
    }
    return bad ? -4 : 0;
}

/*
 * Backward of the attention over the full joint sequence, on rotated (or
 * unrotated, rope = 0) inputs in the layouts of k6o_attention, for the output
 * gradient dout [B][S][H][d].  Writes dq [B][S][H][d], dk/dv [B][Nv][H][d],
 * djk/djv [B][Nj][H][d] (double).  With rope = 1 the q/k gradients are with
 * respect to the rotated q~ and k~.
 */
int k6o_attention_backward(const k6o_geom *g, int rope, const void *q, const void *k, const void *v,
                           const void *jk, const void *jv, int type, const double *dout, double *dq, double *dk,
                           double *dv, double *djk, double *djv) {
    if (!geom_ok(g)) return -1;
    const long S = g->Nv + g->Nj;
    const int d = g->d, H = g->H;
    const double scale = 1.0 / sqrt((double)d);
    double *qr = (double *)malloc(sizeof(double) * (size_t)S * d);
    double *kr = (double *)malloc(sizeof(double) * (size_t)S * d);
    double *vr = (double *)malloc(sizeof(double) * (size_t)S * d);
    double *Pm = (double *)malloc(sizeof(double) * (size_t)S * S);
    double *dK = (double *)malloc(sizeof(double) * (size_t)S * d);
    double *dV = (double *)malloc(sizeof(double) * (size_t)S * d);
    double *Dr = (double *)malloc(sizeof(double) * (size_t)S);
    if (!qr || !kr || !vr || !Pm || !dK || !dV || !Dr) {
        free(qr); free(kr); free(vr); free(Pm); free(dK); free(dV); free(Dr);
        return -4;
    }
    for (int b = 0; b < g->B; b++)
        for (int h = 0; h < H; h++) {
            for (long n = 0; n < S; n++) {
                size_t off;
                const void *kb = kv_ptr(g, n, b, h, k, jk, &off);
                const void *vb = kv_ptr(g, n, b, h, v, jv, &off);
                const size_t qoff = (((size_t)b * S + n) * H + h) * d;
                for (int e = 0; e < d; e++) {
                    qr[(size_t)n * d + e] = load_elem(q, type, qoff + e);
                    kr[(size_t)n * d + e] = load_elem(kb, type, off + e);
                    vr[(size_t)n * d + e] = load_elem(vb, type, off + e);
                }
                if (rope) {
                    k6o_rope_vec(g, n, qr + (size_t)n * d);
                    k6o_rope_vec(g, n, kr + (size_t)n * d);
                }
            }
            /* P and the row terms, then dQ row by row */
#pragma omp parallel for schedule(dynamic, 4)
            for (long i = 0; i < S; i++) {
                double *p = Pm + (size_t)i * S;
                double m = -INFINITY;
                for (long j = 0; j < S; j++) {
                    double acc = 0.0;
                    for (int e = 0; e < d; e++) acc += qr[(size_t)i * d + e] * kr[(size_t)j * d + e];
                    p[j] = acc * scale;
                    if (p[j] > m) m = p[j];
                }
                double sum = 0.0;
                for (long j = 0; j < S; j++) sum += exp(p[j] - m);
                const double lse = m + log(sum);
                for (long j = 0; j < S; j++) p[j] = exp(p[j] - lse);
                const double *go = dout + (((size_t)b * S + i) * H + h) * d;
                /* D_i = dO_i . O_i with O_i = sum_j p_j v_j */
                double Di = 0.0;
                for (int e = 0; e < d; e++) {
                    double o = 0.0;
                    for (long j = 0; j < S; j++) o += p[j] * vr[(size_t)j * d + e];
                    Di += go[e] * o;
                }
#if K6O_MUTANT == 9
                Di = 0.0; /* planted: dropped the D_i term */
#endif
                Dr[i] = Di;
                /* dQ_i = sum_j dS_ij k_j / sqrt(d),  dS_ij = P_ij (dO_i . v_j - D_i) */
                double *gq = dq + (((size_t)b * S + i) * H + h) * d;
                for (int e = 0; e < d; e++) gq[e] = 0.0;
                for (long j = 0; j < S; j++) {
                    double dp = 0.0;
                    for (int e = 0; e < d; e++) dp += go[e] * vr[(size_t)j * d + e];
                    const double ds = p[j] * (dp - Di);
                    for (int e = 0; e < d; e++) gq[e] += ds * kr[(size_t)j * d + e] * scale;
                }
            }
            /* dK and dV key by key (P kept in Pm) */
#pragma omp parallel for schedule(dynamic, 4)
            for (long j = 0; j < S; j++) {
                double *gk = dK + (size_t)j * d, *gv = dV + (size_t)j * d;
                for (int e = 0; e < d; e++) gk[e] = gv[e] = 0.0;
                for (long i = 0; i < S; i++) {
                    const double pij = Pm[(size_t)i * S + j];
                    const double *go = dout + (((size_t)b * S + i) * H + h) * d;
                    double dp = 0.0;
                    for (int e = 0; e < d; e++) dp += go[e] * vr[(size_t)j * d + e];
                    const double ds = pij * (dp - Dr[i]);
                    for (int e = 0; e < d; e++) {
                        gv[e] += pij * go[e];
                        gk[e] += ds * qr[(size_t)i * d + e] * scale;
                    }
                }
            }
            for (long n = 0; n < S; n++) {
                double *tk, *tv;
                if (n < g->Nv) {
                    const size_t off = (((size_t)b * g->Nv + n) * H + h) * d;
                    tk = dk + off, tv = dv + off;
                } else {
                    const size_t off = (((size_t)b * g->Nj + (n - g->Nv)) * H + h) * d;
                    tk = djk + off, tv = djv + off;
                }
                for (int e = 0; e < d; e++) {
                    tk[e] = dK[(size_t)n * d + e];
                    tv[e] = dV[(size_t)n * d + e];
                }
            }
        }
    free(qr); free(kr); free(vr); free(Pm); free(dK); free(dV); free(Dr);
    return 0;
}

/*
 * Log-sum-exp merge of n per-chunk partials.
 *   part_o [n][B][Sq][H][d], part_lse [n][B][H][Sq] (typed: f32 or f64)
 *   out [B][Sq][H][d], lse [B][H][Sq] (double)
 *   LSE = M + log sum_c exp(LSE_c - M) with M = max_c LSE_c,
 *   out = sum_c exp(LSE_c - LSE) O_c.
 */
int k6o_lse_merge(int n, int B, long Sq, int H, int d, const void *part_o, const void *part_lse,
                  int type, double *out, double *lse) {
    if (n < 1 || B < 1 || Sq < 0 || H < 1 || d < 1) return -1;
    size_t o_stride = (size_t)B * Sq * H * d;   /* elements per chunk */
    size_t l_stride = (size_t)B * H * Sq;
    long rows = (long)B * Sq * H;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; r++) {
        int h = (int)(r % H);
        long s = (r / H) % Sq;
        int b = (int)(r / ((long)H * Sq));
        size_t li = ((size_t)b * H + h) * Sq + s;
        double M = -INFINITY;
        for (int c = 0; c < n; c++) {
            double x = load_elem(part_lse, type, c * l_stride + li);
            if (x > M) M = x;
        }
        double sum = 0.0;
        for (int c = 0; c < n; c++) sum += exp(load_elem(part_lse, type, c * l_stride + li) - M);
        double L = M + log(sum);
        double *o = out + (size_t)r * d;
        for (int e = 0; e < d; e++) o[e] = 0.0;
        for (int c = 0; c < n; c++) {
#if K6O_MUTANT == 5
            double w = exp(load_elem(part_lse, type, c * l_stride + li) - M); /* planted: max, not LSE */
#else
            double w = exp(load_elem(part_lse, type, c * l_stride + li) - L);
#endif
            for (int e = 0; e < d; e++)
                o[e] += w * load_elem(part_o, type, c * o_stride + (size_t)r * d + e);
        }
        lse[li] = L;
    }
    return 0;
}

/*
 * Sequence-partitioned <-> head-partitioned relayout, byte copy.
 *   seq  buffer: [P][B][S/P][H][d]   (rank r holds tokens [r*Sl, (r+1)*Sl))
 *   head buffer: [P][B][S][H/P][d]   (rank p holds heads  [p*Hl, (p+1)*Hl))
 *   direction 0: seq -> head, 1: head -> seq.
 */
int k6o_relayout(const void *src, void *dst, int B, long S, int H, int d, int elem_bytes, int P,
                 int direction) {
    if (P < 1 || S % P || H % P || elem_bytes < 1) return -1;
    long Sl = S / P;
    int Hl = H / P;
    const unsigned char *sp = (const unsigned char *)src;
    unsigned char *dp = (unsigned char *)dst;
    for (int r = 0; r < P; r++)
        for (int p = 0; p < P; p++)
            for (int b = 0; b < B; b++)
                for (long s = 0; s < Sl; s++)
                    for (int hh = 0; hh < Hl; hh++)
                        for (int e = 0; e < d; e++) {
#if K6O_MUTANT == 6
                            size_t seq_i = ((((size_t)p * B + b) * Sl + s) * H + (size_t)r * Hl + hh) * d + e; /* planted */
#else
                            size_t seq_i = ((((size_t)r * B + b) * Sl + s) * H + (size_t)p * Hl + hh) * d + e;
#endif
                            size_t head_i = ((((size_t)p * B + b) * S + (size_t)r * Sl + s) * Hl + hh) * d + e;
                            if (direction == 0)
                                memcpy(dp + head_i * elem_bytes, sp + seq_i * elem_bytes, elem_bytes);
                            else
                                memcpy(dp + seq_i * elem_bytes, sp + head_i * elem_bytes, elem_bytes);
                        }
    return 0;
}

/* Latent grid of a video: frames (F-1)//4 + 1, spatial (px//8)//2.
 * "Context Parallelism in vLLM Omni Neuron", section "Sequence Length
 * Constraints", worked example. */
void k6o_latent_grid(int height, int width, int frames, int *t, int *h, int *w) {
    *t = (frames - 1) / 4 + 1;
    *h = (height / 8) / 2;
    *w = (width / 8) / 2;
}
