/*
 * hypic_oracle.c -- plain float64 CPU oracle for the linear-attention segment
 * transition cache.  TEST INFRASTRUCTURE ONLY: the product path never links,
 * loads or calls this file; only the tests, the smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header or constant
 * with the CUDA library.
 *
 * Source of every formula: the page "HYPIC: Accelerating Hybrid-Attention LLM
 * Serving with Position-Independent Caching -- reading notes" (HYPIC reading
 * notes below), which restates the paper's equations:
 *   - unified recurrence S_i = T_i S_{i-1} + u_i, o_i = q_i^T S_i
 *     (Motivation 2, paper Eq. (2));
 *   - per-variant T_i, u_i (Method 3, paper Table 1): RetNet/Lightning gamma*I,
 *     Mamba2 a_i*I, GLA diag(g_i) (all with u_i = k_i v_i^T), DeltaNet
 *     I - b k k^T, GDN g_i (I - b k k^T) and KDA (I - b k k^T) diag(g_i)
 *     (these three with u_i = b k_i v_i^T);
 *   - segment pair T_C = T_m...T_1, S_{C|0} = sum_t T_m...T_{t+1} u_t
 *     (Method 2, "segments as affine maps");
 *   - composition (T_B,B_B) o (T_A,B_A) = (T_B T_A, T_B B_A + B_B) and the
 *     n-segment form, paper Eq. (6) (Method 2);
 *   - two-pass build: S_0 = 0 with writes gives S_{C|0}; S_0 = I with all
 *     u_t = 0 gives T_C (Method 4, paper Sec. 5).
 *
 * Everything is written the plain way, token by token, with no blocking, no
 * chunking and no reordering beyond the definitions above.  All matrices are
 * row-major; the state S is d_k x d_v with the row index on the key channel.
 *
 * Transition storage by family (the "T_C families" table, paper Table 3):
 *   SCALAR_CONST, SCALAR : one number
 *   DIAG                 : d_k numbers (the diagonal)
 *   DELTA, GATED_DELTA, KDA : dense d_k x d_k
 *
 * Gate layout for one head over `len` tokens:
 *   SCALAR_CONST : alpha[0]            (gamma of the head, every token)
 *   SCALAR, GATED_DELTA : alpha[t]
 *   DIAG, KDA    : alpha[t*d_k + i]
 *   DELTA        : alpha unused (a = 1)
 *   beta[t] is read by DELTA, GATED_DELTA and KDA only.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { FAM_SCALAR_CONST = 0, FAM_SCALAR = 1, FAM_DIAG = 2, FAM_DELTA = 3, FAM_GATED_DELTA = 4, FAM_KDA = 5 };

int orc_t_size(int fam, int dk)
{
    if (fam == FAM_SCALAR_CONST || fam == FAM_SCALAR) return 1;
    if (fam == FAM_DIAG) return dk;
    return dk * dk;
}

/* The scalar gate a_t of token t for the scalar and gated-delta families. */
static double gate_scalar(int fam, const double *alpha, int64_t t)
{
    if (fam == FAM_SCALAR_CONST) return alpha[0];
    if (fam == FAM_DELTA) return 1.0;
    return alpha[t];
}

/*
 * One token of S <- T_t S + u_t (paper Eq. (2)) with T_t, u_t from Table 1.
 * For the delta families, (T_t S)_{ij} = a (S_ij - b k_i sum_l k_l S_lj);
 * with_write = 0 drops u_t (the second pass of the two-pass build).
 */
static void step(int fam, int dk, int dv, double *S, const double *k,
                 const double *v, const double *alpha, const double *beta,
                 int64_t t, int with_write, double *tmp)
{
    int i, j;
    if (fam == FAM_DIAG) {
        const double *g = alpha + t * dk;
        for (i = 0; i < dk; i++)
            for (j = 0; j < dv; j++)
                S[i * dv + j] = g[i] * S[i * dv + j] + (with_write ? k[i] * v[j] : 0.0);
        return;
    }
    if (fam == FAM_SCALAR_CONST || fam == FAM_SCALAR) {
        double a = gate_scalar(fam, alpha, t);
        for (i = 0; i < dk; i++)
            for (j = 0; j < dv; j++)
                S[i * dv + j] = a * S[i * dv + j] + (with_write ? k[i] * v[j] : 0.0);
        return;
    }
    if (fam == FAM_KDA) {
        /* T_t = (I - b k k^T) diag(g_t): first the per-channel gate, then the erase. */
        const double *g = alpha + t * dk;
        double b = beta[t];
        for (i = 0; i < dk; i++)
            for (j = 0; j < dv; j++) S[i * dv + j] *= g[i];
        for (j = 0; j < dv; j++) {
            double acc = 0.0;
            for (i = 0; i < dk; i++) acc += k[i] * S[i * dv + j];
            tmp[j] = acc; /* (k^T diag(g) S)_j */
        }
        for (i = 0; i < dk; i++)
            for (j = 0; j < dv; j++)
                S[i * dv + j] = S[i * dv + j] - b * k[i] * tmp[j] + (with_write ? b * k[i] * v[j] : 0.0);
        return;
    }
    /* DELTA / GATED_DELTA */
    {
        double a = gate_scalar(fam, alpha, t);
        double b = beta[t];
        for (j = 0; j < dv; j++) {
            double acc = 0.0;
            for (i = 0; i < dk; i++) acc += k[i] * S[i * dv + j];
            tmp[j] = acc; /* (k^T S)_j */
        }
        for (i = 0; i < dk; i++)
            for (j = 0; j < dv; j++) {
                double TS = a * (S[i * dv + j] - b * k[i] * tmp[j]);
                S[i * dv + j] = TS + (with_write ? b * k[i] * v[j] : 0.0);
            }
    }
}

/*
 * Run the recurrence over `len` tokens of one head from the state S (in/out).
 * k, q: [len][dk]; v: [len][dv].  If o != NULL, o[t][j] = (q_t^T S_t)_j with
 * the post-update state S_t (paper Eq. (2)).
 */
int orc_run(int fam, int dk, int dv, int64_t len, const double *k,
            const double *v, const double *q, const double *alpha,
            const double *beta, double *S, double *o)
{
    int64_t t;
    int i, j;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)(dv > 0 ? dv : 1));
    if (!tmp) return -1;
    for (t = 0; t < len; t++) {
        step(fam, dk, dv, S, k + t * dk, v + t * dv, alpha, beta, t, 1, tmp);
        if (o) {
            for (j = 0; j < dv; j++) {
                double acc = 0.0;
                for (i = 0; i < dk; i++) acc += q[t * dk + i] * S[i * dv + j];
                o[t * dv + j] = acc;
            }
        }
    }
    free(tmp);
    return 0;
}

/*
 * T_C = T_len ... T_1 of one head, in the family's storage form.
 * Scalar families: the product of the gates.  Diagonal: per-channel product.
 * Delta families: the recurrence run from S_0 = I with every u_t = 0 (the
 * second pass of the two-pass build), O(dk^2) per token.
 */
int orc_transition(int fam, int dk, int64_t len, const double *k,
                   const double *alpha, const double *beta, double *T)
{
    int64_t t;
    int i;
    if (fam == FAM_SCALAR_CONST || fam == FAM_SCALAR) {
        double p = 1.0;
        for (t = 0; t < len; t++) p *= gate_scalar(fam, alpha, t);
        T[0] = p;
        return 0;
    }
    if (fam == FAM_DIAG) {
        for (i = 0; i < dk; i++) T[i] = 1.0;
        for (t = 0; t < len; t++)
            for (i = 0; i < dk; i++) T[i] *= alpha[t * dk + i];
        return 0;
    }
    {
        double *tmp = (double *)malloc(sizeof(double) * (size_t)dk);
        if (!tmp) return -1;
        memset(T, 0, sizeof(double) * (size_t)dk * (size_t)dk);
        for (i = 0; i < dk; i++) T[i * dk + i] = 1.0;
        for (t = 0; t < len; t++)
            step(fam, dk, dk, T, k + t * dk, NULL, alpha, beta, t, 0, tmp);
        free(tmp);
    }
    return 0;
}

/* The cached pair of one segment body: T_C and S_{C|0} (from S_0 = 0). */
int orc_segment_pair(int fam, int dk, int dv, int64_t len, const double *k,
                     const double *v, const double *alpha, const double *beta,
                     double *T, double *S)
{
    memset(S, 0, sizeof(double) * (size_t)dk * (size_t)dv);
    if (orc_run(fam, dk, dv, len, k, v, NULL, alpha, beta, S, NULL)) return -1;
    return orc_transition(fam, dk, len, k, alpha, beta, T);
}

/* Y = T X for a transition T in storage form and X of dk x ncol. */
static void apply_T(int fam, int dk, int ncol, const double *T, const double *X, double *Y)
{
    int i, j, l;
    if (fam == FAM_SCALAR_CONST || fam == FAM_SCALAR) {
        for (i = 0; i < dk * ncol; i++) Y[i] = T[0] * X[i];
        return;
    }
    if (fam == FAM_DIAG) {
        for (i = 0; i < dk; i++)
            for (j = 0; j < ncol; j++) Y[i * ncol + j] = T[i] * X[i * ncol + j];
        return;
    }
    for (i = 0; i < dk; i++)
        for (j = 0; j < ncol; j++) {
            double acc = 0.0;
            for (l = 0; l < dk; l++) acc += T[i * dk + l] * X[l * ncol + j];
            Y[i * ncol + j] = acc;
        }
}

/* T3 = T2 T1 in storage form. */
static void mul_T(int fam, int dk, const double *T2, const double *T1, double *T3)
{
    int i;
    if (fam == FAM_SCALAR_CONST || fam == FAM_SCALAR) { T3[0] = T2[0] * T1[0]; return; }
    if (fam == FAM_DIAG) { for (i = 0; i < dk; i++) T3[i] = T2[i] * T1[i]; return; }
    apply_T(fam, dk, dk, T2, T1, T3);
}

/*
 * Composition of affine maps (Method 2): (T2,S2) o (T1,S1) = (T2 T1, T2 S1 + S2),
 * i.e. apply segment 1 first, then segment 2.  Outputs may not alias inputs.
 */
int orc_affine_combine(int fam, int dk, int dv, const double *T2, const double *S2,
                       const double *T1, const double *S1, double *T3, double *S3)
{
    int i;
    mul_T(fam, dk, T2, T1, T3);
    apply_T(fam, dk, dv, T2, S1, S3);
    for (i = 0; i < dk * dv; i++) S3[i] += S2[i];
    return 0;
}

/*
 * Compose n cached pairs onto S (in/out), in order j = 0..n-1:
 * S <- T_j S + S0_j.  This is paper Eq. (6) evaluated as n sequential
 * applications.  T: [n][t_size], S0: [n][dk*dv].
 */
int orc_compose(int fam, int dk, int dv, int n, const double *T, const double *S0, double *S)
{
    int j, i, ts = orc_t_size(fam, dk);
    double *Y = (double *)malloc(sizeof(double) * (size_t)dk * (size_t)dv);
    if (!Y) return -1;
    for (j = 0; j < n; j++) {
        apply_T(fam, dk, dv, T + (size_t)j * ts, S, Y);
        for (i = 0; i < dk * dv; i++) S[i] = Y[i] + S0[(size_t)j * dk * dv + i];
    }
    free(Y);
    return 0;
}

/*
 * Inclusive scan of affine maps: (Tp_0,Sp_0) = (T_0,S_0),
 * (Tp_i,Sp_i) = (T_i,S_i) o (Tp_{i-1},Sp_{i-1}).  Done sequentially.
 */
int orc_affine_scan(int fam, int dk, int dv, int n, const double *T, const double *S,
                    double *Tp, double *Sp)
{
    int i, ts = orc_t_size(fam, dk);
    size_t ss = (size_t)dk * dv;
    if (n <= 0) return 0;
    memcpy(Tp, T, sizeof(double) * ts);
    memcpy(Sp, S, sizeof(double) * ss);
    for (i = 1; i < n; i++)
        orc_affine_combine(fam, dk, dv, T + (size_t)i * ts, S + i * ss,
                           Tp + (size_t)(i - 1) * ts, Sp + (i - 1) * ss,
                           Tp + (size_t)i * ts, Sp + i * ss);
    return 0;
}
