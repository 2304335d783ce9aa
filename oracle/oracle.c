/*
 * oracle.c -- plain, slow, fp64 CPU definition of the small-batch decode hot path
 * described in "Hyper Optimizing Kimi K3 in vLLM: Moving Fast and Responsibly".
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library. The CUDA library neither links
 * nor includes it, and the two share no code, header, table or helper.
 *
 * Conventions (every function below follows them):
 *   - bf16 tensors arrive as their raw 16-bit patterns (uint16_t), row-major with
 *     the last dimension contiguous.
 *   - Every bf16 value is widened exactly to double. A product of two bf16 values
 *     is exact in double (8-bit x 8-bit significands), so the only rounding in a
 *     dot product is that of the running fp64 sum, taken with k ascending.
 *   - Results are rounded to bf16 only where the library stores bf16 (Y, latent,
 *     the gated intermediate A), directly from the fp64 value, round to nearest,
 *     ties to even.
 *   - OpenMP spreads independent output rows over threads; it never splits or
 *     reorders a single sum.
 *
 * Readings of the pages that this file fixes (the pages give prose only):
 *   - router: softmax over the raw router logits, no bias, no expert groups, no
 *     scaling; top-k chosen on the logits with ties to the lower expert index and
 *     the chosen experts listed by descending logit; weights renormalised over the
 *     chosen k.  The choice is taken on the logits rounded to fp32, the precision in
 *     which the GPU library takes it.
 *   - expert MLP: Wgu rows [0, I) are the gate, rows [I, 2I) are the up projection;
 *     a = bf16(silu(gate) * up), silu(t) = t / (1 + exp(-t)); y = a . Wd^T.
 *   - the shared expert is added with weight 1 before the single output rounding.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- bf16 ---- */

/* bf16 is the upper half of an IEEE binary32: 1 sign, 8 exponent, 7 fraction bits. */
double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round a double to the nearest bf16, ties to even, straight from fp64 (no
 * intermediate fp32 rounding). Written from the definition: find the spacing q of
 * bf16 values at |v| (2^(E-7) for a normal binade 2^E, 2^-133 for subnormals),
 * round |v|/q to the nearest integer with ties to even (rint under the default
 * rounding mode), scale back, and overflow to infinity at 2^128.
 */
uint16_t oracle_bf16_from_double(double v)
{
    if (isnan(v))
        return (uint16_t)(signbit(v) ? 0xFFC0u : 0x7FC0u);
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(sign | 0x7F80u);
    if (a == 0.0)
        return sign;
    int e;
    (void)frexp(a, &e);      /* a = m * 2^e, m in [0.5, 1) */
    int E = e - 1;           /* a in [2^E, 2^(E+1)) */
    int qexp = (E < -126) ? -133 : E - 7;
    double n = ldexp(a, -qexp);          /* exact: power-of-two scaling */
    double r = ldexp(rint(n), qexp);     /* rint: nearest, ties to even */
    if (r >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7F80u);
    float f = (float)r;                  /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

void oracle_bf16_decode_array(const uint16_t *h, double *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_to_double(h[i]);
}

void oracle_bf16_encode_array(const double *v, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_from_double(v[i]);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------- linear ---- */

/* sum_k x[k] * w[k], k ascending, in fp64 */
static double dot_bf16(const uint16_t *x, const uint16_t *w, int K)
{
    double s = 0.0;
    for (int k = 0; k < K; ++k)
        s += oracle_bf16_to_double(x[k]) * oracle_bf16_to_double(w[k]);
    return s;
}

/*
 * Decode projection, "Part 1 / 1. Tune shapes for the workload" (the attention input
 * projections), and the output projection followed by the attention-residual add,
 * "Part 1 / 2. Overlap computation and communication" (its single-GPU part):
 *
 *     y[b,n] = sum_k X[b,k] * W[n,k]  (+ R[b,n] when R is given)
 *     Y[b,n] = bf16(y[b,n])
 *
 * X [B,K], W [N,K], R [B,N] or NULL. y_exact [B,N] (fp64) and Y [B,N] (bf16 bits) are
 * each optional (NULL skips it).
 */
void oracle_linear(const uint16_t *X, const uint16_t *W, const uint16_t *R, int B, int N,
                   int K, double *y_exact, uint16_t *Y)
{
    #pragma omp parallel for schedule(static)
    for (int n = 0; n < N; ++n) {
        for (int b = 0; b < B; ++b) {
            double s = dot_bf16(X + (int64_t)b * K, W + (int64_t)n * K, K);
            if (R)
                s += oracle_bf16_to_double(R[(int64_t)b * N + n]);
            if (y_exact)
                y_exact[(int64_t)b * N + n] = s;
            if (Y)
                Y[(int64_t)b * N + n] = oracle_bf16_from_double(s);
        }
    }
}

/* ------------------------------------------------------------- router ---- */

/*
 * Routing of one decode batch, the step after the router scores of
 * "Part 1 / 3. Improve MoE scheduling and overlap" (the pages do not define it; the
 * readings are in the file header):
 *
 *     p_i   = exp(l_i - m) / sum_e exp(l_e - m),  m = max_e l_e
 *     idx   = the topk experts with the largest fp32(l_i), ties to the lower index,
 *             listed by descending fp32(l_i) then ascending index
 *     w_j   = exp(l_idx_j - m) / sum_{j'} exp(l_idx_j' - m)
 *
 * logits [B,E] fp64 in; idx [B,topk], w [B,topk], probs [B,E] (optional) out.
 */
void oracle_route(const double *logits, int B, int E, int topk, int32_t *idx, double *w,
                  double *probs)
{
    for (int b = 0; b < B; ++b) {
        const double *l = logits + (int64_t)b * E;
        double m = l[0];
        for (int e = 1; e < E; ++e)
            if (l[e] > m)
                m = l[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e)
            z += exp(l[e] - m);
        if (probs)
            for (int e = 0; e < E; ++e)
                probs[(int64_t)b * E + e] = exp(l[e] - m) / z;

        /* selection: repeatedly take the best remaining key (fp32 logit desc,
         * index asc); plain O(k*E) */
        unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
        for (int j = 0; j < topk; ++j) {
            int best = -1;
            float bestv = 0.0f;
            for (int e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                float v = (float)l[e];
                if (best < 0 || v > bestv) {   /* strict: equal keys keep the lower index */
                    best = e;
                    bestv = v;
                }
            }
            taken[best] = 1;
            idx[(int64_t)b * topk + j] = best;
        }
        free(taken);

        double zs = 0.0;
        for (int j = 0; j < topk; ++j)
            zs += exp(l[idx[(int64_t)b * topk + j]] - m);
        for (int j = 0; j < topk; ++j)
            w[(int64_t)b * topk + j] = exp(l[idx[(int64_t)b * topk + j]] - m) / zs;
    }
}

/*
 * MoE front end, "Part 1 / 3. Improve MoE scheduling and overlap": the router scores
 * and the latent input projection as ONE matrix product over the concatenated weight
 * Wcat [E+L, K] (router rows first), then routing.
 *
 *     z       = X . Wcat^T                       (fp64)
 *     logits  = z[:, 0:E]                        (kept in fp64, not rounded)
 *     latent  = bf16(z[:, E:E+L])
 *     idx, w, probs = oracle_route(logits)
 *
 * Outputs other than idx and w may be NULL.
 */
void oracle_moe_front(const uint16_t *X, const uint16_t *Wcat, int B, int K, int E, int L,
                      int topk, double *logits, uint16_t *latent, int32_t *idx, double *w,
                      double *probs)
{
    int N = E + L;
    double *z = (double *)malloc(sizeof(double) * (size_t)B * (size_t)N);
    oracle_linear(X, Wcat, NULL, B, N, K, z, NULL);
    double *lg = (double *)malloc(sizeof(double) * (size_t)B * (size_t)E);
    for (int b = 0; b < B; ++b) {
        for (int e = 0; e < E; ++e)
            lg[(int64_t)b * E + e] = z[(int64_t)b * N + e];
        if (latent)
            for (int i = 0; i < L; ++i)
                latent[(int64_t)b * L + i] = oracle_bf16_from_double(z[(int64_t)b * N + E + i]);
    }
    if (logits)
        memcpy(logits, lg, sizeof(double) * (size_t)B * (size_t)E);
    oracle_route(lg, B, E, topk, idx, w, probs);
    free(lg);
    free(z);
}

/*
 * Expert -> (token, slot) inverse of the routing, so that each used expert's weights
 * can be read once for all of its tokens ("Part 2 / 4. Check performance broadly":
 * expert selection decides which weights are read and how much work is reused).
 * A counting sort written out plainly:
 *
 *     counts[e]   = #{(b,j) : idx[b,j] == e}
 *     offsets[e]  = sum_{e' < e} counts[e'],  offsets[E] = B*topk
 *     pairs[...]  = the entries b*topk + j, ordered by (expert asc, b*topk + j asc)
 *     pos[b*topk+j] = the position of that entry in pairs
 *     used[0..U)  = the experts with counts > 0, ascending;  *num_used = U
 */
void oracle_route_map(const int32_t *idx, int B, int topk, int E, int32_t *counts,
                      int32_t *offsets, int32_t *pairs, int32_t *pos, int32_t *used,
                      int32_t *num_used)
{
    int P = B * topk;
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (int p = 0; p < P; ++p)
        counts[idx[p]] += 1;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int u = 0;
    for (int e = 0; e < E; ++e) {
        if (counts[e] > 0)
            used[u++] = e;
        int at = offsets[e];
        for (int p = 0; p < P; ++p) {
            if (idx[p] == e) {
                pairs[at] = p;
                pos[p] = at;
                at += 1;
            }
        }
    }
    *num_used = u;
}

/* ------------------------------------------------------------- experts --- */

double oracle_silu(double t)
{
    return t / (1.0 + exp(-t));
}

/*
 * One SiLU-gated expert MLP for one token, "Part 1 / 3. Improve MoE scheduling and
 * overlap" (routed experts and the shared expert have this form):
 *
 *     g[i] = x . Wgu[i]^T,  u[i] = x . Wgu[I+i]^T          i in [0, I)
 *     a[i] = bf16(silu(g[i]) * u[i])                        (stored intermediate)
 *     y[h] = sum_i a[i] * Wd[h,i]                           h in [0, H), fp64
 *
 * x [H], Wgu [2I, H], Wd [H, I]; a [I] (bf16 bits, optional), y [H] (fp64).
 */
void oracle_expert_mlp(const uint16_t *x, const uint16_t *Wgu, const uint16_t *Wd, int H, int I,
                       uint16_t *a_out, double *y)
{
    uint16_t *a = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)I);
    #pragma omp parallel for schedule(static)
    for (int i = 0; i < I; ++i) {
        double g = dot_bf16(x, Wgu + (int64_t)i * H, H);
        double u = dot_bf16(x, Wgu + (int64_t)(I + i) * H, H);
        a[i] = oracle_bf16_from_double(oracle_silu(g) * u);
    }
    #pragma omp parallel for schedule(static)
    for (int h = 0; h < H; ++h)
        y[h] = dot_bf16(a, Wd + (int64_t)h * I, I);
    if (a_out)
        memcpy(a_out, a, sizeof(uint16_t) * (size_t)I);
    free(a);
}

/*
 * Combine of the routed experts and the shared expert for a decode batch:
 *
 *     y[b,h] = sum_{j=0..topk-1} w[b,j] * yp[b,j,h]  (+ s[b,h] when s is given)
 *     Y[b,h] = bf16(y[b,h])
 *
 * w [B,topk], yp [B,topk,H], s [B,H] or NULL. y_exact and Y are each optional.
 */
void oracle_combine(int B, int H, int topk, const double *w, const double *yp, const double *s,
                    double *y_exact, uint16_t *Y)
{
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h) {
            double acc = 0.0;
            for (int j = 0; j < topk; ++j)
                acc += w[(int64_t)b * topk + j] * yp[((int64_t)b * topk + j) * H + h];
            if (s)
                acc += s[(int64_t)b * H + h];
            if (y_exact)
                y_exact[(int64_t)b * H + h] = acc;
            if (Y)
                Y[(int64_t)b * H + h] = oracle_bf16_from_double(acc);
        }
    }
}

/*
 * The routed experts plus the shared expert for a decode batch, with every weight in
 * host memory (small shapes):
 *
 *     yp[b,j] = expert_mlp(X[b], Wgu[idx[b,j]], Wd[idx[b,j]])
 *     s[b]    = expert_mlp(X[b], Wgu_s, Wd_s)      (when Wgu_s is given)
 *     Y       = combine(w, yp, s)
 *
 * X [B,H], idx [B,topk], w [B,topk], Wgu [E,2I,H], Wd [E,H,I], Wgu_s [2I,H], Wd_s [H,I].
 */
void oracle_moe_experts(const uint16_t *X, const int32_t *idx, const double *w,
                        const uint16_t *Wgu, const uint16_t *Wd, int E, const uint16_t *Wgu_s,
                        const uint16_t *Wd_s, int B, int H, int I, int topk, double *y_exact,
                        uint16_t *Y)
{
    (void)E;
    double *yp = (double *)malloc(sizeof(double) * (size_t)B * (size_t)topk * (size_t)H);
    double *s = Wgu_s ? (double *)malloc(sizeof(double) * (size_t)B * (size_t)H) : NULL;
    for (int b = 0; b < B; ++b) {
        const uint16_t *x = X + (int64_t)b * H;
        for (int j = 0; j < topk; ++j) {
            int e = idx[(int64_t)b * topk + j];
            oracle_expert_mlp(x, Wgu + (int64_t)e * 2 * I * H, Wd + (int64_t)e * H * I, H, I,
                              NULL, yp + ((int64_t)b * topk + j) * H);
        }
        if (s)
            oracle_expert_mlp(x, Wgu_s, Wd_s, H, I, NULL, s + (int64_t)b * H);
    }
    oracle_combine(B, H, topk, w, yp, s, y_exact, Y);
    free(s);
    free(yp);
}
