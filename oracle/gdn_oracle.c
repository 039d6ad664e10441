/*
 * gdn_oracle.c -- plain fp64 CPU oracle for the gated delta rule (GDN), its
 * DeltaProduct generalisation and the camera-branch prep.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test-suite, the smoke check and the bench's CPU
 * baseline leg do.  It shares no code, header or constant with the CUDA path.
 *
 * Everything here is the plain definition written out, token by token, in
 * double precision, with no blocking, chunking or reordering:
 *
 *  - GDN (gated_deltaproduct test.py, the state-scan kernel
 *    `gated_chunk_delta_rule_fwd_kernel_h` and output kernel
 *    `gated_chunk_linear_attn_fwd_kernel_o`; fused_cam_gdn.py,
 *    `_cam_scan_kernel`, "decay, then predict, then correct"):
 *        S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
 *        o_t = scale * S_t^T q_t              (inclusive of token t)
 *    with S of shape Dk x Dv (rows = key dim, columns = value dim).
 *
 *  - DeltaProduct: per token the decay is applied once, then r Householder
 *    sub-steps j = 0..r-1, each with its own k_{t,j}, v_{t,j}, beta_{t,j};
 *    the output reads the state after the last sub-step.
 *
 *  - Block-masked DeltaProduct (gated_deltaproduct test.py: the mask_ij
 *    coupling of `gated_chunk_scaled_dot_kkt_fwd_kernel` and
 *    `gated_fwd_recompute_w_u_kernel`, the per-slice state update of
 *    `gated_chunk_delta_rule_fwd_kernel_h`, and the sum over r in
 *    `gated_chunk_fwd_o_fn`): the key dimension is cut into r slices of
 *    Dk/r; per token the decay is applied once, then every sub-row i < r
 *    predicts from that same state with the read key k_t (.) m_i (slice j of
 *    k_t times mask[i][j]) and corrects the state's slice-i rows with its
 *    write key, slice i of k_t; one value and one beta per token:
 *        S <- e^{g_t} S
 *        z_j = S_(j)^T k_t,(j)                 (slice j rows of S and k_t)
 *        d_i = beta_t (v_t - sum_j mask[i][j] z_j)
 *        S_(i) <- S_(i) + k_t,(i) d_i^T        (all i from the same z)
 *        o_t = scale * S^T q_t
 *
 *  - Frame-level camera scan (fused_cam_gdn.py, `_cam_scan_kernel`,
 *    `_torch_cam_scan_single_chunk` and `_torch_cam_scan_reference`): the
 *    tokens form F frames of S tokens; per frame the state is decayed once by
 *    the frame's factor, then every token of the frame predicts from that
 *    same decayed state and all S corrections are added at once,
 *        S <- d_f S ;  S <- S + K_f^T diag(beta_f) (V_f - K_f S)
 *    and every token of the frame reads the state after the frame's update,
 *        o_s = scale * S^T q_s.
 *    The reverse mode (the page's REVERSE=1, `flip_and_shift`) runs the frames
 *    from last to first, each frame's output reading the state built from
 *    the frames after it only (the last frame reads zero).
 *
 *  - Backward of the frame-level camera scan (fused_cam_gdn.py,
 *    `_cam_scan_bwd_kernel`, forward direction): the adjoint of the frame
 *    loop, frames from last to first, with the states recomputed forward.
 *
 *  - Backward of the camera prep (fused_cam_gdn.py, `_cam_prep_bwd_kernel`,
 *    continued through the full-C RMSNorm): the adjoint of the prep map from
 *    the raw rows to q_out, k_out, v_out, k_pre_sq and k_post_sq, written as
 *    the chain rule of the forward steps in reverse order.
 *
 *  - Camera prep (fused_cam_gdn.py, `_torch_cam_prep_reference` and
 *    `_cam_prep_kernel`): full-C RMSNorm (C = H*D) with per-channel weight on
 *    q and k, ReLU on q and k, K-scale on k, a 4x4 projection out = P*in on
 *    each group of 4 in the first D/2 dims (proj_q for q, proj_kv for k and
 *    v), interleaved-pair RoPE on the last D/2 dims, and ||k||^2 before and
 *    after the projection/RoPE.
 *
 * exp/sqrt/sin/cos/pow are the host libm double routines.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* x <- x / max(||x||_2, 1e-12); the zero vector stays zero. */
static void l2_normalise(double *x, int n) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += x[i] * x[i];
    double nrm = sqrt(s);
    if (nrm < 1e-12) nrm = 1e-12;
    for (int i = 0; i < n; ++i) x[i] /= nrm;
}

/* One delta-rule correction on S (Dk x Dv, row-major):
 *   p = S^T k ;  S += beta * k (v - p)^T
 * which equals S <- (I - beta k k^T) S + beta k v^T. */
static void delta_step(double *S, const double *k, const double *v, double beta,
                       int Dk, int Dv, double *p) {
    for (int j = 0; j < Dv; ++j) p[j] = 0.0;
    for (int i = 0; i < Dk; ++i) {
        const double ki = k[i];
        const double *row = S + (size_t)i * Dv;
        for (int j = 0; j < Dv; ++j) p[j] += row[j] * ki;
    }
    for (int i = 0; i < Dk; ++i) {
        const double c = beta * k[i];
        double *row = S + (size_t)i * Dv;
        for (int j = 0; j < Dv; ++j) row[j] += c * (v[j] - p[j]);
    }
}

/* o = scale * S^T q */
static void read_out(const double *S, const double *q, double scale, int Dk, int Dv,
                     double *o) {
    for (int j = 0; j < Dv; ++j) o[j] = 0.0;
    for (int i = 0; i < Dk; ++i) {
        const double qi = q[i];
        const double *row = S + (size_t)i * Dv;
        for (int j = 0; j < Dv; ++j) o[j] += row[j] * qi;
    }
    for (int j = 0; j < Dv; ++j) o[j] *= scale;
}

/*
 * GDN forward, token by token.
 *   q, k : [B,H,T,Dk]      v, o : [B,H,T,Dv]      beta, g : [B,H,T]
 *   s0 / s_final : [B,H,Dk,Dv] or NULL (NULL s0 = zero state).
 *   l2norm != 0 normalises q_t and k_t to unit length before use.
 * Returns 0, or -1 if scratch memory could not be allocated.
 */
int oracle_gdn_fwd(const double *q, const double *k, const double *v, const double *beta,
                   const double *g, const double *s0, double *o, double *s_final, int B,
                   int H, int T, int Dk, int Dv, double scale, int l2norm) {
    const int BH = B * H;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int bh = 0; bh < BH; ++bh) {
        double *S = (double *)malloc(sizeof(double) * (size_t)Dk * Dv);
        double *p = (double *)malloc(sizeof(double) * (size_t)Dv);
        double *kt = (double *)malloc(sizeof(double) * (size_t)Dk);
        double *qt = (double *)malloc(sizeof(double) * (size_t)Dk);
        if (!S || !p || !kt || !qt) {
            failed |= 1;
        } else {
            if (s0)
                memcpy(S, s0 + (size_t)bh * Dk * Dv, sizeof(double) * (size_t)Dk * Dv);
            else
                memset(S, 0, sizeof(double) * (size_t)Dk * Dv);
            for (int t = 0; t < T; ++t) {
                const size_t tok = (size_t)bh * T + t;
                memcpy(kt, k + tok * Dk, sizeof(double) * Dk);
                memcpy(qt, q + tok * Dk, sizeof(double) * Dk);
                if (l2norm) {
                    l2_normalise(kt, Dk);
                    l2_normalise(qt, Dk);
                }
                /* decay hits the old state only, before the correction */
                const double a = exp(g[tok]);
                for (size_t e = 0; e < (size_t)Dk * Dv; ++e) S[e] *= a;
                delta_step(S, kt, v + tok * Dv, beta[tok], Dk, Dv, p);
                read_out(S, qt, scale, Dk, Dv, o + tok * Dv);
            }
            if (s_final)
                memcpy(s_final + (size_t)bh * Dk * Dv, S, sizeof(double) * (size_t)Dk * Dv);
        }
        free(S);
        free(p);
        free(kt);
        free(qt);
    }
    return failed ? -1 : 0;
}

/*
 * DeltaProduct forward: decay once per token, then r sub-steps in index order.
 *   q : [B,H,T,Dk]   k : [B,H,T,r,Dk]   v : [B,H,T,r,Dv]   beta : [B,H,T,r]
 *   g : [B,H,T]      o : [B,H,T,Dv]     s0 / s_final : [B,H,Dk,Dv] or NULL.
 */
int oracle_deltaproduct_fwd(const double *q, const double *k, const double *v,
                            const double *beta, const double *g, const double *s0,
                            double *o, double *s_final, int B, int H, int T, int r, int Dk,
                            int Dv, double scale, int l2norm) {
    const int BH = B * H;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int bh = 0; bh < BH; ++bh) {
        double *S = (double *)malloc(sizeof(double) * (size_t)Dk * Dv);
        double *p = (double *)malloc(sizeof(double) * (size_t)Dv);
        double *kt = (double *)malloc(sizeof(double) * (size_t)Dk);
        double *qt = (double *)malloc(sizeof(double) * (size_t)Dk);
        if (!S || !p || !kt || !qt) {
            failed |= 1;
        } else {
            if (s0)
                memcpy(S, s0 + (size_t)bh * Dk * Dv, sizeof(double) * (size_t)Dk * Dv);
            else
                memset(S, 0, sizeof(double) * (size_t)Dk * Dv);
            for (int t = 0; t < T; ++t) {
                const size_t tok = (size_t)bh * T + t;
                const double a = exp(g[tok]);
                for (size_t e = 0; e < (size_t)Dk * Dv; ++e) S[e] *= a;
                for (int j = 0; j < r; ++j) {
                    const size_t sub = tok * r + j;
                    memcpy(kt, k + sub * Dk, sizeof(double) * Dk);
                    if (l2norm) l2_normalise(kt, Dk);
                    delta_step(S, kt, v + sub * Dv, beta[sub], Dk, Dv, p);
                }
                memcpy(qt, q + tok * Dk, sizeof(double) * Dk);
                if (l2norm) l2_normalise(qt, Dk);
                read_out(S, qt, scale, Dk, Dv, o + tok * Dv);
            }
            if (s_final)
                memcpy(s_final + (size_t)bh * Dk * Dv, S, sizeof(double) * (size_t)Dk * Dv);
        }
        free(S);
        free(p);
        free(kt);
        free(qt);
    }
    return failed ? -1 : 0;
}

/*
 * Block-masked DeltaProduct forward, token by token.
 *   q, k : [B,H,T,Dk]   v, o : [B,H,T,Dv]   beta, g : [B,H,T]
 *   mask : [r][r] row-major, shared by every head; r divides Dk
 *   s0 / s_final : [B,H,Dk,Dv] or NULL.
 */
int oracle_masked_deltaproduct_fwd(const double *q, const double *k, const double *v,
                                   const double *beta, const double *g, const double *mask,
                                   const double *s0, double *o, double *s_final, int B, int H,
                                   int T, int r, int Dk, int Dv, double scale, int l2norm) {
    if (r < 1 || Dk % r != 0) return -2;
    const int BH = B * H;
    const int dk = Dk / r;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int bh = 0; bh < BH; ++bh) {
        double *S = (double *)malloc(sizeof(double) * (size_t)Dk * Dv);
        double *z = (double *)malloc(sizeof(double) * (size_t)r * Dv);
        double *d = (double *)malloc(sizeof(double) * (size_t)r * Dv);
        double *kt = (double *)malloc(sizeof(double) * (size_t)Dk);
        double *qt = (double *)malloc(sizeof(double) * (size_t)Dk);
        if (!S || !z || !d || !kt || !qt) {
            failed |= 1;
        } else {
            if (s0)
                memcpy(S, s0 + (size_t)bh * Dk * Dv, sizeof(double) * (size_t)Dk * Dv);
            else
                memset(S, 0, sizeof(double) * (size_t)Dk * Dv);
            for (int t = 0; t < T; ++t) {
                const size_t tok = (size_t)bh * T + t;
                memcpy(kt, k + tok * Dk, sizeof(double) * Dk);
                memcpy(qt, q + tok * Dk, sizeof(double) * Dk);
                if (l2norm) {
                    l2_normalise(kt, Dk);
                    l2_normalise(qt, Dk);
                }
                const double a = exp(g[tok]);
                for (size_t e = 0; e < (size_t)Dk * Dv; ++e) S[e] *= a;
                /* per-slice predictions from the decayed state */
                for (int jj = 0; jj < r; ++jj) {
                    double *zj = z + (size_t)jj * Dv;
                    for (int c = 0; c < Dv; ++c) zj[c] = 0.0;
                    for (int i = jj * dk; i < (jj + 1) * dk; ++i) {
                        const double *row = S + (size_t)i * Dv;
                        for (int c = 0; c < Dv; ++c) zj[c] += row[c] * kt[i];
                    }
                }
                for (int ii = 0; ii < r; ++ii) {
                    double *di = d + (size_t)ii * Dv;
                    for (int c = 0; c < Dv; ++c) {
                        double pr = 0.0;
                        for (int jj = 0; jj < r; ++jj) pr += mask[ii * r + jj] * z[(size_t)jj * Dv + c];
                        di[c] = beta[tok] * (v[tok * Dv + c] - pr);
                    }
                }
                /* sub-row i writes the slice-i rows */
                for (int ii = 0; ii < r; ++ii)
                    for (int i = ii * dk; i < (ii + 1) * dk; ++i) {
                        double *row = S + (size_t)i * Dv;
                        for (int c = 0; c < Dv; ++c) row[c] += kt[i] * d[(size_t)ii * Dv + c];
                    }
                read_out(S, qt, scale, Dk, Dv, o + tok * Dv);
            }
            if (s_final)
                memcpy(s_final + (size_t)bh * Dk * Dv, S, sizeof(double) * (size_t)Dk * Dv);
        }
        free(S);
        free(z);
        free(d);
        free(kt);
        free(qt);
    }
    return failed ? -1 : 0;
}

/* One frame's joint update: P = K S with the state as it is on entry (every
 * row predicts from the same S), then S += sum_s beta_s k_s (v_s - p_s)^T. */
static void frame_update(double *S, const double *K, const double *V, const double *beta,
                         int S_len, int Dk, int Dv, double *P) {
    for (int s = 0; s < S_len; ++s) {
        double *p = P + (size_t)s * Dv;
        for (int j = 0; j < Dv; ++j) p[j] = 0.0;
        for (int i = 0; i < Dk; ++i) {
            const double ki = K[(size_t)s * Dk + i];
            const double *row = S + (size_t)i * Dv;
            for (int j = 0; j < Dv; ++j) p[j] += row[j] * ki;
        }
    }
    for (int s = 0; s < S_len; ++s) {
        const double *p = P + (size_t)s * Dv;
        const double *vs = V + (size_t)s * Dv;
        for (int i = 0; i < Dk; ++i) {
            const double c = beta[s] * K[(size_t)s * Dk + i];
            double *row = S + (size_t)i * Dv;
            for (int j = 0; j < Dv; ++j) row[j] += c * (vs[j] - p[j]);
        }
    }
}

/*
 * Frame-level camera scan, frame by frame.
 *   q, k : [B,H,F*S_len,Dk]     v, o : [B,H,F*S_len,Dv]     beta : [B,H,F*S_len]
 *   decay: [B,H,F] multiplicative factor of each frame (not its log)
 *   s0 / s_final : [B,H,Dk,Dv] or NULL (forward only; NULL s0 = zero state)
 *   reverse != 0: frames from last to first; the output of frame f reads the
 *   state built from frames f+1 .. F-1, and frame f's factor decays the state
 *   when frame f is taken in (the page's REVERSE=1).
 *   l2norm != 0 normalises q and k per token before use.
 * Returns 0, -1 if scratch memory could not be allocated, -2 if a state is
 * passed in reverse mode.
 */
int oracle_cam_scan_fwd(const double *q, const double *k, const double *v, const double *beta,
                        const double *decay, const double *s0, double *o, double *s_final,
                        int B, int H, int F, int S_len, int Dk, int Dv, double scale,
                        int reverse, int l2norm) {
    if (reverse && (s0 || s_final)) return -2;
    const int BH = B * H;
    const long N = (long)F * S_len;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int bh = 0; bh < BH; ++bh) {
        double *S = (double *)malloc(sizeof(double) * (size_t)Dk * Dv);
        double *P = (double *)malloc(sizeof(double) * (size_t)(S_len > 0 ? S_len : 1) * Dv);
        double *Kf = (double *)malloc(sizeof(double) * (size_t)(S_len > 0 ? S_len : 1) * Dk);
        double *qt = (double *)malloc(sizeof(double) * (size_t)Dk);
        if (!S || !P || !Kf || !qt) {
            failed |= 1;
        } else {
            if (s0)
                memcpy(S, s0 + (size_t)bh * Dk * Dv, sizeof(double) * (size_t)Dk * Dv);
            else
                memset(S, 0, sizeof(double) * (size_t)Dk * Dv);
            for (int it = 0; it < F; ++it) {
                /* frame whose keys / values enter now, and frame whose queries read */
                const int qf = reverse ? F - 1 - it : it;
                const int kf = reverse ? F - it : it; /* reverse: none at it = 0 */
                if (!reverse || it > 0) {
                    const double d = decay[(size_t)bh * F + kf];
                    for (size_t e = 0; e < (size_t)Dk * Dv; ++e) S[e] *= d;
                    const size_t t0 = (size_t)bh * N + (size_t)kf * S_len;
                    memcpy(Kf, k + t0 * Dk, sizeof(double) * (size_t)S_len * Dk);
                    if (l2norm)
                        for (int s = 0; s < S_len; ++s) l2_normalise(Kf + (size_t)s * Dk, Dk);
                    frame_update(S, Kf, v + t0 * Dv, beta + t0, S_len, Dk, Dv, P);
                }
                const size_t q0 = (size_t)bh * N + (size_t)qf * S_len;
                for (int s = 0; s < S_len; ++s) {
                    memcpy(qt, q + (q0 + s) * Dk, sizeof(double) * Dk);
                    if (l2norm) l2_normalise(qt, Dk);
                    read_out(S, qt, scale, Dk, Dv, o + (q0 + s) * Dv);
                }
            }
            if (s_final)
                memcpy(s_final + (size_t)bh * Dk * Dv, S, sizeof(double) * (size_t)Dk * Dv);
        }
        free(S);
        free(P);
        free(Kf);
        free(qt);
    }
    return failed ? -1 : 0;
}

/*
 * Camera-branch prep (fused_cam_gdn.py, `_torch_cam_prep_reference`).
 *   q_raw, k_raw, v_raw : [B,N,H,D]
 *   q_norm_w, k_norm_w  : [H*D] or NULL (NULL = all ones)
 *   proj_q, proj_kv     : [B,N,4,4] row-major, applied as out_i = sum_j P[i][j] in_j
 *   rope_cos, rope_sin  : [N, D/2] in the page's interleaved encoding
 *                         y[d] = x[d] cos[d] + x[d^1] sin[d], or both NULL, in
 *                         which case cos[2i]=cos[2i+1]=cos(th), sin[2i]=-sin(th),
 *                         sin[2i+1]=+sin(th), th = n * rope_base^(-2i/(D/2)).
 *   q_out, k_out, v_out : [B,H,N,D]
 *   k_pre_sq, k_post_sq : [B,H,N] or NULL
 */
int oracle_cam_prep_fwd(const double *q_raw, const double *k_raw, const double *v_raw,
                        const double *q_norm_w, const double *k_norm_w, const double *proj_q,
                        const double *proj_kv, const double *rope_cos, const double *rope_sin,
                        double rope_base, double *q_out, double *k_out, double *v_out,
                        double *k_pre_sq, double *k_post_sq, int B, int N, int H, int D,
                        double k_scale, double eps) {
    if (D % 2 != 0 || (D / 2) % 4 != 0) return -2;
    const int C = H * D;
    const int Dh = D / 2;
    const long BN = (long)B * N;
    int failed = 0;
#pragma omp parallel for schedule(static) reduction(| : failed)
    for (long bn = 0; bn < BN; ++bn) {
        const int b = (int)(bn / N);
        const int n = (int)(bn % N);
        double *xq = (double *)malloc(sizeof(double) * D);
        double *xk = (double *)malloc(sizeof(double) * D);
        double *xv = (double *)malloc(sizeof(double) * D);
        double *cs = (double *)malloc(sizeof(double) * Dh);
        double *sn = (double *)malloc(sizeof(double) * Dh);
        if (!xq || !xk || !xv || !cs || !sn) {
            failed |= 1;
        } else {
            const double *qr = q_raw + (size_t)bn * C;
            const double *kr = k_raw + (size_t)bn * C;
            const double *vr = v_raw + (size_t)bn * C;
            /* full-C RMSNorm statistics, shared by all heads of the token */
            double ssq = 0.0, ssk = 0.0;
            for (int c = 0; c < C; ++c) {
                ssq += qr[c] * qr[c];
                ssk += kr[c] * kr[c];
            }
            const double iq = 1.0 / sqrt(ssq / C + eps);
            const double ik = 1.0 / sqrt(ssk / C + eps);
            /* rotary tables for this position */
            for (int d = 0; d < Dh; ++d) {
                if (rope_cos && rope_sin) {
                    cs[d] = rope_cos[(size_t)n * Dh + d];
                    sn[d] = rope_sin[(size_t)n * Dh + d];
                } else {
                    const int i = d / 2;
                    const double th = (double)n * pow(rope_base, -2.0 * i / (double)Dh);
                    cs[d] = cos(th);
                    sn[d] = (d % 2 == 0) ? -sin(th) : sin(th);
                }
            }
            const double *Pq = proj_q + (size_t)bn * 16;
            const double *Pk = proj_kv + (size_t)bn * 16;
            for (int h = 0; h < H; ++h) {
                double pre = 0.0, post = 0.0;
                for (int d = 0; d < D; ++d) {
                    const int c = h * D + d;
                    const double wq = q_norm_w ? q_norm_w[c] : 1.0;
                    const double wk = k_norm_w ? k_norm_w[c] : 1.0;
                    double a = qr[c] * iq * wq;
                    double bk = kr[c] * ik * wk;
                    a = a > 0.0 ? a : 0.0;
                    bk = (bk > 0.0 ? bk : 0.0) * k_scale;
                    xq[d] = a;
                    xk[d] = bk;
                    xv[d] = vr[c];
                    pre += bk * bk;
                }
                const size_t ob = (((size_t)b * H + h) * N + n) * D;
                /* first half: out = P * in on each group of four */
                for (int g0 = 0; g0 < Dh; g0 += 4) {
                    for (int i = 0; i < 4; ++i) {
                        double sq = 0.0, sk = 0.0, sv = 0.0;
                        for (int j = 0; j < 4; ++j) {
                            sq += Pq[i * 4 + j] * xq[g0 + j];
                            sk += Pk[i * 4 + j] * xk[g0 + j];
                            sv += Pk[i * 4 + j] * xv[g0 + j];
                        }
                        q_out[ob + g0 + i] = sq;
                        k_out[ob + g0 + i] = sk;
                        v_out[ob + g0 + i] = sv;
                        post += sk * sk;
                    }
                }
                /* second half: interleaved-pair rotation */
                for (int d = 0; d < Dh; ++d) {
                    const int e = Dh + d;
                    const int pe = Dh + (d ^ 1);
                    const double yq = xq[e] * cs[d] + xq[pe] * sn[d];
                    const double yk = xk[e] * cs[d] + xk[pe] * sn[d];
                    const double yv = xv[e] * cs[d] + xv[pe] * sn[d];
                    q_out[ob + e] = yq;
                    k_out[ob + e] = yk;
                    v_out[ob + e] = yv;
                    post += yk * yk;
                }
                const size_t si = ((size_t)b * H + h) * N + n;
                if (k_pre_sq) k_pre_sq[si] = pre;
                if (k_post_sq) k_post_sq[si] = post;
            }
        }
        free(xq);
        free(xk);
        free(xv);
        free(cs);
        free(sn);
    }
    return failed ? -1 : 0;
}

/*
 * Backward of the camera prep: given the gradients of q_out, k_out, v_out
 * ([B,H,N,D]) and of k_pre_sq, k_post_sq ([B,H,N], each may be NULL = zero),
 * the gradients of q_raw, k_raw, v_raw ([B,N,H,D]).  Same arguments and
 * tables as oracle_cam_prep_fwd.  Per token, in reverse order of the forward:
 *   rotation:   dx[d] = dy[d] cos[d] + dy[d^1] sin[d^1]        (last D/2 dims)
 *   projection: dx_j = sum_i P[i][j] dy_i                       (first D/2 dims)
 *   k_post_sq:  dk_out += 2 k_out dpost;  k_pre_sq: da_k += 2 a_k dpre
 *   K-scale, ReLU: dxhat = k_scale [xhat > 0] da  (q: no K-scale)
 *   RMSNorm:    xhat_c = x_c r w_c, r = (sum x^2 / C + eps)^(-1/2):
 *               dx_j = r w_j dxhat_j - (r^3 / C) x_j sum_c w_c x_c dxhat_c
 *   v: the projection and rotation only.
 */
int oracle_cam_prep_bwd(const double *q_raw, const double *k_raw, const double *q_norm_w,
                        const double *k_norm_w, const double *proj_q, const double *proj_kv,
                        const double *rope_cos, const double *rope_sin, double rope_base,
                        const double *dq_out, const double *dk_out, const double *dv_out,
                        const double *dpre, const double *dpost, double *dq_raw, double *dk_raw,
                        double *dv_raw, int B, int N, int H, int D, double k_scale, double eps) {
    if (D % 2 != 0 || (D / 2) % 4 != 0) return -2;
    const int C = H * D, Dh = D / 2;
    const long BN = (long)B * N;
    int failed = 0;
#pragma omp parallel for schedule(static) reduction(| : failed)
    for (long bn = 0; bn < BN; ++bn) {
        const int b = (int)(bn / N), n = (int)(bn % N);
        double *cs = (double *)malloc(sizeof(double) * Dh);
        double *sn = (double *)malloc(sizeof(double) * Dh);
        double *dxq = (double *)malloc(sizeof(double) * C);  /* gradient of xhat_q (per channel) */
        double *dxk = (double *)malloc(sizeof(double) * C);
        double *ak = (double *)malloc(sizeof(double) * D);
        double *ko = (double *)malloc(sizeof(double) * D);
        double *gk = (double *)malloc(sizeof(double) * D);
        if (!cs || !sn || !dxq || !dxk || !ak || !ko || !gk) {
            failed |= 1;
        } else {
            const double *qr = q_raw + (size_t)bn * C, *kr = k_raw + (size_t)bn * C;
            double ssq = 0.0, ssk = 0.0;
            for (int c = 0; c < C; ++c) {
                ssq += qr[c] * qr[c];
                ssk += kr[c] * kr[c];
            }
            const double iq = 1.0 / sqrt(ssq / C + eps), ik = 1.0 / sqrt(ssk / C + eps);
            for (int d = 0; d < Dh; ++d) {
                if (rope_cos && rope_sin) {
                    cs[d] = rope_cos[(size_t)n * Dh + d];
                    sn[d] = rope_sin[(size_t)n * Dh + d];
                } else {
                    const int i = d / 2;
                    const double th = (double)n * pow(rope_base, -2.0 * i / (double)Dh);
                    cs[d] = cos(th);
                    sn[d] = (d % 2 == 0) ? -sin(th) : sin(th);
                }
            }
            const double *Pq = proj_q + (size_t)bn * 16, *Pk = proj_kv + (size_t)bn * 16;
            for (int h = 0; h < H; ++h) {
                const size_t ob = (((size_t)b * H + h) * N + n) * D;
                const size_t si = ((size_t)b * H + h) * N + n;
                const double gpre = dpre ? dpre[si] : 0.0, gpost = dpost ? dpost[si] : 0.0;
                /* forward values of k needed by the norm-square terms */
                for (int d = 0; d < D; ++d) {
                    const int c = h * D + d;
                    const double x = kr[c] * ik * (k_norm_w ? k_norm_w[c] : 1.0);
                    ak[d] = (x > 0.0 ? x : 0.0) * k_scale;
                }
                for (int g0 = 0; g0 < Dh; g0 += 4)
                    for (int i = 0; i < 4; ++i) {
                        double acc = 0.0;
                        for (int j = 0; j < 4; ++j) acc += Pk[i * 4 + j] * ak[g0 + j];
                        ko[g0 + i] = acc;
                    }
                for (int d = 0; d < Dh; ++d) {
                    const int e = Dh + d, pe = Dh + (d ^ 1);
                    ko[e] = ak[e] * cs[d] + ak[pe] * sn[d];
                }
                /* gradient reaching k_out, including ||k_out||^2 */
                for (int d = 0; d < D; ++d) gk[d] = dk_out[ob + d] + 2.0 * ko[d] * gpost;
                for (int t = 0; t < 3; ++t) {
                    const double *dy = t == 0 ? dq_out + ob : (t == 1 ? gk : dv_out + ob);
                    const double *P = t == 0 ? Pq : Pk;
                    double *out = t == 2 ? dv_raw + (size_t)bn * C + h * D : NULL;
                    double da[512];
                    for (int g0 = 0; g0 < Dh; g0 += 4)
                        for (int j = 0; j < 4; ++j) {
                            double acc = 0.0;
                            for (int i = 0; i < 4; ++i) acc += P[i * 4 + j] * dy[g0 + i];
                            da[g0 + j] = acc;
                        }
                    for (int d = 0; d < Dh; ++d) {
                        const int e = Dh + d, pe = Dh + (d ^ 1);
                        da[e] = dy[e] * cs[d] + dy[pe] * sn[d ^ 1];
                    }
                    if (t == 2) {
                        for (int d = 0; d < D; ++d) out[d] = da[d];
                    } else {
                        for (int d = 0; d < D; ++d) {
                            const int c = h * D + d;
                            if (t == 0) {
                                const double x = qr[c] * iq * (q_norm_w ? q_norm_w[c] : 1.0);
                                dxq[c] = x > 0.0 ? da[d] : 0.0;
                            } else {
                                const double x = kr[c] * ik * (k_norm_w ? k_norm_w[c] : 1.0);
                                const double dak = da[d] + 2.0 * ak[d] * gpre;
                                dxk[c] = x > 0.0 ? k_scale * dak : 0.0;
                            }
                        }
                    }
                }
            }
            /* RMSNorm over all C channels of the token */
            double sq = 0.0, sk = 0.0;
            for (int c = 0; c < C; ++c) {
                sq += (q_norm_w ? q_norm_w[c] : 1.0) * qr[c] * dxq[c];
                sk += (k_norm_w ? k_norm_w[c] : 1.0) * kr[c] * dxk[c];
            }
            for (int c = 0; c < C; ++c) {
                dq_raw[(size_t)bn * C + c] =
                    iq * (q_norm_w ? q_norm_w[c] : 1.0) * dxq[c] - iq * iq * iq / C * qr[c] * sq;
                dk_raw[(size_t)bn * C + c] =
                    ik * (k_norm_w ? k_norm_w[c] : 1.0) * dxk[c] - ik * ik * ik / C * kr[c] * sk;
            }
        }
        free(cs);
        free(sn);
        free(dxq);
        free(dxk);
        free(ak);
        free(ko);
        free(gk);
    }
    return failed ? -1 : 0;
}

/* y = x / max(||x||, 1e-12); given dy returns dx = (dy - y (y . dy)) / max(||x||, 1e-12)
 * (for ||x|| below the floor the map is x / 1e-12 and dx = dy / 1e-12). */
static void l2_normalise_bwd(const double *x, const double *dy, double *dx, int n) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += x[i] * x[i];
    const double nrm = sqrt(s);
    if (nrm < 1e-12) {
        for (int i = 0; i < n; ++i) dx[i] = dy[i] / 1e-12;
        return;
    }
    double yd = 0.0;
    for (int i = 0; i < n; ++i) yd += x[i] / nrm * dy[i];
    for (int i = 0; i < n; ++i) dx[i] = (dy[i] - x[i] / nrm * yd) / nrm;
}

/*
 * Backward of oracle_cam_scan_fwd (forward direction).  Given do [B,H,N,Dv]
 * and dsf [B,H,Dk,Dv] (or NULL), the gradients dq, dk [B,H,N,Dk], dv
 * [B,H,N,Dv], dbeta [B,H,N], ddecay [B,H,F] and ds0 [B,H,Dk,Dv] (or NULL).
 * With S' the state entering frame f and S_f the state after it,
 *   R = diag(beta) (V - d K S'),  S_f = d S' + K^T R,  O = scale Q S_f,
 * frames from last to first, dS the adjoint of S_f:
 *   dS += scale Q^T dO;  dq_t = scale S_f do_t
 *   dR = K dS;  dv_t = beta_t dR_t;  dbeta_t = dR_t . (v_t - d S'^T k_t)
 *   dk_t = dS r_t - d beta_t S' dR_t           (r_t = beta_t (v_t - d S'^T k_t))
 *   dd  = <dS, S'> - sum_t beta_t dR_t . (S'^T k_t)
 *   dS' = d (dS - K^T diag(beta) dR)
 * and with l2norm the unit-norm map's adjoint on each q_t and k_t.
 */
int oracle_cam_scan_bwd(const double *q, const double *k, const double *v, const double *beta,
                        const double *decay, const double *s0, const double *dout, const double *dsf,
                        double *dq, double *dk, double *dv, double *dbeta, double *ddecay, double *ds0,
                        int B, int H, int F, int S_len, int Dk, int Dv, double scale, int l2norm) {
    const int BH = B * H;
    const long N = (long)F * S_len;
    const size_t SD = (size_t)Dk * Dv;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int bh = 0; bh < BH; ++bh) {
        double *St = (double *)malloc(sizeof(double) * SD * (F + 1)); /* St[f] = state entering frame f */
        double *dS = (double *)malloc(sizeof(double) * SD);
        double *X = (double *)malloc(sizeof(double) * SD);
        double *P = (double *)malloc(sizeof(double) * (size_t)(S_len > 0 ? S_len : 1) * Dv);
        double *Kf = (double *)malloc(sizeof(double) * (size_t)(S_len > 0 ? S_len : 1) * Dk);
        double *vec = (double *)malloc(sizeof(double) * (size_t)(Dk + Dv) * 4);
        if (!St || !dS || !X || !P || !Kf || !vec) {
            failed |= 1;
        } else {
            double *dR = vec, *Pk = vec + Dv, *r = vec + 2 * Dv, *gk = vec + 3 * Dv, *tk = gk + Dk;
            double *qt = tk + Dk, *tq = qt + Dk;
            if (s0)
                memcpy(St, s0 + (size_t)bh * SD, sizeof(double) * SD);
            else
                memset(St, 0, sizeof(double) * SD);
            /* forward: the states entering each frame, and the last */
            for (int f = 0; f < F; ++f) {
                double *Sn = St + (size_t)(f + 1) * SD;
                memcpy(Sn, St + (size_t)f * SD, sizeof(double) * SD);
                const double d = decay[(size_t)bh * F + f];
                for (size_t e = 0; e < SD; ++e) Sn[e] *= d;
                const size_t t0 = (size_t)bh * N + (size_t)f * S_len;
                memcpy(Kf, k + t0 * Dk, sizeof(double) * (size_t)S_len * Dk);
                if (l2norm)
                    for (int s = 0; s < S_len; ++s) l2_normalise(Kf + (size_t)s * Dk, Dk);
                frame_update(Sn, Kf, v + t0 * Dv, beta + t0, S_len, Dk, Dv, P);
            }
            if (dsf)
                memcpy(dS, dsf + (size_t)bh * SD, sizeof(double) * SD);
            else
                memset(dS, 0, sizeof(double) * SD);
            for (int f = F - 1; f >= 0; --f) {
                const double *Sp = St + (size_t)f * SD, *Sf = St + (size_t)(f + 1) * SD;
                const double d = decay[(size_t)bh * F + f];
                const size_t t0 = (size_t)bh * N + (size_t)f * S_len;
                /* outputs of the frame */
                for (int s = 0; s < S_len; ++s) {
                    const size_t tok = t0 + s;
                    memcpy(qt, q + tok * Dk, sizeof(double) * Dk);
                    if (l2norm) l2_normalise(qt, Dk);
                    const double *go = dout + tok * Dv;
                    for (int i = 0; i < Dk; ++i) {
                        double acc = 0.0;
                        for (int c = 0; c < Dv; ++c) {
                            acc += Sf[(size_t)i * Dv + c] * go[c];
                            dS[(size_t)i * Dv + c] += scale * qt[i] * go[c];
                        }
                        tq[i] = scale * acc;
                    }
                    if (l2norm)
                        l2_normalise_bwd(q + tok * Dk, tq, dq + tok * Dk, Dk);
                    else
                        memcpy(dq + tok * Dk, tq, sizeof(double) * Dk);
                }
                /* the frame's update */
                double dd = 0.0;
                for (size_t e = 0; e < SD; ++e) dd += dS[e] * Sp[e];
                memset(X, 0, sizeof(double) * SD);
                for (int s = 0; s < S_len; ++s) {
                    const size_t tok = t0 + s;
                    memcpy(tk, k + tok * Dk, sizeof(double) * Dk);
                    if (l2norm) l2_normalise(tk, Dk);
                    const double bt = beta[tok];
                    for (int c = 0; c < Dv; ++c) {
                        double a = 0.0, b2 = 0.0;
                        for (int i = 0; i < Dk; ++i) {
                            a += tk[i] * dS[(size_t)i * Dv + c];
                            b2 += tk[i] * Sp[(size_t)i * Dv + c];
                        }
                        dR[c] = a;
                        Pk[c] = b2;
                        r[c] = bt * (v[tok * Dv + c] - d * b2);
                    }
                    double db = 0.0;
                    for (int c = 0; c < Dv; ++c) {
                        dv[tok * Dv + c] = bt * dR[c];
                        db += dR[c] * (v[tok * Dv + c] - d * Pk[c]);
                        dd -= bt * dR[c] * Pk[c];
                    }
                    dbeta[tok] = db;
                    for (int i = 0; i < Dk; ++i) {
                        double acc = 0.0;
                        for (int c = 0; c < Dv; ++c)
                            acc += dS[(size_t)i * Dv + c] * r[c] - d * bt * Sp[(size_t)i * Dv + c] * dR[c];
                        gk[i] = acc;
                        for (int c = 0; c < Dv; ++c) X[(size_t)i * Dv + c] += tk[i] * bt * dR[c];
                    }
                    if (l2norm)
                        l2_normalise_bwd(k + tok * Dk, gk, dk + tok * Dk, Dk);
                    else
                        memcpy(dk + tok * Dk, gk, sizeof(double) * Dk);
                }
                ddecay[(size_t)bh * F + f] = dd;
                for (size_t e = 0; e < SD; ++e) dS[e] = d * (dS[e] - X[e]);
            }
            if (ds0) memcpy(ds0 + (size_t)bh * SD, dS, sizeof(double) * SD);
        }
        free(St);
        free(dS);
        free(X);
        free(P);
        free(Kf);
        free(vec);
    }
    return failed ? -1 : 0;
}

/*
 * Backward of oracle_deltaproduct_fwd (r = 1 is oracle_gdn_fwd): the adjoint
 * of its token loop, tokens from last to first (gated_deltaproduct test.py
 * computes the same gradients chunk-wise: `gated_chunk_delta_rule_bwd_kernel_dhu`,
 * `gated_chunk_delta_rule_bwd_kernel_dqkw`, `gated_bwd_prepare_wy_repr_kernel`).
 * Given dout = dL/do [B,H,T,Dv] and dsf = dL/dS_final [B,H,Dk,Dv] (NULL = 0),
 * it writes dq [B,H,T,Dk], dk [B,H,T,r,Dk], dv [B,H,T,r,Dv], dbeta [B,H,T,r],
 * dg [B,H,T] and ds0 [B,H,Dk,Dv] (NULL = not wanted).  With G the adjoint of
 * the state after a step:
 *   output o = scale S^T q:             G += scale q do^T;  dq = scale S do
 *   sub-step X -> X + b k (v - X^T k)^T, e = v - X^T k, w = G^T k:
 *       dv = b w;  db = k . (G e);  dk = b (G e - X w);  G <- G - b k w^T
 *   decay D = e^{g} E (E the state entering the token, D = X before sub-step 0):
 *       dg = <G, D>;  G <- e^{g} G
 * and with l2norm the unit-norm map's adjoint on q and every k.  The states
 * entering the tokens are rebuilt from checkpoints every 64 tokens with the
 * forward's own arithmetic, so they are exactly the forward's.
 */
int oracle_deltaproduct_bwd(const double *q, const double *k, const double *v, const double *beta,
                            const double *g, const double *s0, const double *dout, const double *dsf,
                            double *dq, double *dk, double *dv, double *dbeta, double *dg, double *ds0,
                            int B, int H, int T, int r, int Dk, int Dv, double scale, int l2norm) {
    if (r < 1) return -2;
    const int BH = B * H;
    const int BLK = 64;
    const int nblk = (T + BLK - 1) / BLK;
    const size_t SD = (size_t)Dk * Dv;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int bh = 0; bh < BH; ++bh) {
        double *Cp = (double *)malloc(sizeof(double) * SD * (nblk > 0 ? nblk : 1)); /* entering token BLK*b */
        double *E = (double *)malloc(sizeof(double) * SD * BLK);                    /* entering each token */
        double *X = (double *)malloc(sizeof(double) * SD * (r + 1));                /* before each sub-step */
        double *G = (double *)malloc(sizeof(double) * SD);
        double *vec = (double *)malloc(sizeof(double) * (size_t)(4 * Dk + 3 * Dv));
        if (!Cp || !E || !X || !G || !vec) {
            failed |= 1;
        } else {
            double *kt = vec, *qt = vec + Dk, *gk = vec + 2 * Dk, *tq = vec + 3 * Dk;
            double *p = vec + 4 * Dk, *e = p + Dv, *w = e + Dv;
            double *S = X; /* scratch for the forward pass */
            if (s0)
                memcpy(S, s0 + (size_t)bh * SD, sizeof(double) * SD);
            else
                memset(S, 0, sizeof(double) * SD);
            /* forward: checkpoints of the state entering every BLK-th token */
            for (int t = 0; t < T; ++t) {
                if (t % BLK == 0) memcpy(Cp + (size_t)(t / BLK) * SD, S, sizeof(double) * SD);
                const size_t tok = (size_t)bh * T + t;
                const double a = exp(g[tok]);
                for (size_t x = 0; x < SD; ++x) S[x] *= a;
                for (int j = 0; j < r; ++j) {
                    const size_t sub = tok * r + j;
                    memcpy(kt, k + sub * Dk, sizeof(double) * Dk);
                    if (l2norm) l2_normalise(kt, Dk);
                    delta_step(S, kt, v + sub * Dv, beta[sub], Dk, Dv, p);
                }
            }
            if (dsf)
                memcpy(G, dsf + (size_t)bh * SD, sizeof(double) * SD);
            else
                memset(G, 0, sizeof(double) * SD);
            for (int b = nblk - 1; b >= 0; --b) {
                const int t0 = b * BLK, t1 = (t0 + BLK < T) ? t0 + BLK : T;
                /* rebuild the states entering the block's tokens */
                memcpy(E, Cp + (size_t)b * SD, sizeof(double) * SD);
                for (int t = t0; t + 1 < t1; ++t) {
                    const size_t tok = (size_t)bh * T + t;
                    double *Sn = E + (size_t)(t - t0 + 1) * SD;
                    memcpy(Sn, E + (size_t)(t - t0) * SD, sizeof(double) * SD);
                    const double a = exp(g[tok]);
                    for (size_t x = 0; x < SD; ++x) Sn[x] *= a;
                    for (int j = 0; j < r; ++j) {
                        const size_t sub = tok * r + j;
                        memcpy(kt, k + sub * Dk, sizeof(double) * Dk);
                        if (l2norm) l2_normalise(kt, Dk);
                        delta_step(Sn, kt, v + sub * Dv, beta[sub], Dk, Dv, p);
                    }
                }
                for (int t = t1 - 1; t >= t0; --t) {
                    const size_t tok = (size_t)bh * T + t;
                    const double a = exp(g[tok]);
                    /* the token's states: X[0] decayed, X[j+1] after sub-step j */
                    const double *Et = E + (size_t)(t - t0) * SD;
                    for (size_t x = 0; x < SD; ++x) X[x] = a * Et[x];
                    for (int j = 0; j < r; ++j) {
                        const size_t sub = tok * r + j;
                        memcpy(X + (size_t)(j + 1) * SD, X + (size_t)j * SD, sizeof(double) * SD);
                        memcpy(kt, k + sub * Dk, sizeof(double) * Dk);
                        if (l2norm) l2_normalise(kt, Dk);
                        delta_step(X + (size_t)(j + 1) * SD, kt, v + sub * Dv, beta[sub], Dk, Dv, p);
                    }
                    /* output */
                    const double *Sr = X + (size_t)r * SD;
                    const double *go = dout + tok * Dv;
                    memcpy(qt, q + tok * Dk, sizeof(double) * Dk);
                    if (l2norm) l2_normalise(qt, Dk);
                    for (int i = 0; i < Dk; ++i) {
                        double acc = 0.0;
                        for (int c = 0; c < Dv; ++c) {
                            acc += Sr[(size_t)i * Dv + c] * go[c];
                            G[(size_t)i * Dv + c] += scale * qt[i] * go[c];
                        }
                        tq[i] = scale * acc;
                    }
                    if (l2norm)
                        l2_normalise_bwd(q + tok * Dk, tq, dq + tok * Dk, Dk);
                    else
                        memcpy(dq + tok * Dk, tq, sizeof(double) * Dk);
                    /* sub-steps, last first */
                    for (int j = r - 1; j >= 0; --j) {
                        const size_t sub = tok * r + j;
                        const double *Xj = X + (size_t)j * SD;
                        const double bt = beta[sub];
                        const double *vt = v + sub * Dv;
                        memcpy(kt, k + sub * Dk, sizeof(double) * Dk);
                        if (l2norm) l2_normalise(kt, Dk);
                        for (int c = 0; c < Dv; ++c) {
                            double xk = 0.0, gk2 = 0.0;
                            for (int i = 0; i < Dk; ++i) {
                                xk += Xj[(size_t)i * Dv + c] * kt[i];
                                gk2 += G[(size_t)i * Dv + c] * kt[i];
                            }
                            e[c] = vt[c] - xk;
                            w[c] = gk2;
                            dv[sub * Dv + c] = bt * gk2;
                        }
                        double db = 0.0;
                        for (int i = 0; i < Dk; ++i) {
                            double ge = 0.0, xw = 0.0;
                            for (int c = 0; c < Dv; ++c) {
                                ge += G[(size_t)i * Dv + c] * e[c];
                                xw += Xj[(size_t)i * Dv + c] * w[c];
                            }
                            db += kt[i] * ge;
                            gk[i] = bt * (ge - xw);
                        }
                        dbeta[sub] = db;
                        if (l2norm)
                            l2_normalise_bwd(k + sub * Dk, gk, dk + sub * Dk, Dk);
                        else
                            memcpy(dk + sub * Dk, gk, sizeof(double) * Dk);
                        for (int i = 0; i < Dk; ++i)
                            for (int c = 0; c < Dv; ++c) G[(size_t)i * Dv + c] -= bt * kt[i] * w[c];
                    }
                    /* decay */
                    double dd = 0.0;
                    for (size_t x = 0; x < SD; ++x) dd += G[x] * X[x];
                    dg[tok] = dd;
                    for (size_t x = 0; x < SD; ++x) G[x] *= a;
                }
            }
            if (ds0) memcpy(ds0 + (size_t)bh * SD, G, sizeof(double) * SD);
        }
        free(Cp);
        free(E);
        free(X);
        free(G);
        free(vec);
    }
    return failed ? -1 : 0;
}

/* One token of oracle_masked_deltaproduct_fwd on S in place, in the same order
 * of operations: decay, the slice predictions z_j, d_i, the slice writes.  kt
 * receives the token's (unit, with l2norm) key; z, d are r x Dv scratch. */
static void masked_token_step(double *S, const double *k, const double *v, double beta, double g,
                              const double *mask, int r, int Dk, int Dv, int l2norm, double *kt,
                              double *z, double *d) {
    const int sl = Dk / r;
    memcpy(kt, k, sizeof(double) * Dk);
    if (l2norm) l2_normalise(kt, Dk);
    const double a = exp(g);
    for (size_t e = 0; e < (size_t)Dk * Dv; ++e) S[e] *= a;
    for (int jj = 0; jj < r; ++jj) {
        double *zj = z + (size_t)jj * Dv;
        for (int c = 0; c < Dv; ++c) zj[c] = 0.0;
        for (int i = jj * sl; i < (jj + 1) * sl; ++i) {
            const double *row = S + (size_t)i * Dv;
            for (int c = 0; c < Dv; ++c) zj[c] += row[c] * kt[i];
        }
    }
    for (int ii = 0; ii < r; ++ii) {
        double *di = d + (size_t)ii * Dv;
        for (int c = 0; c < Dv; ++c) {
            double pr = 0.0;
            for (int jj = 0; jj < r; ++jj) pr += mask[ii * r + jj] * z[(size_t)jj * Dv + c];
            di[c] = beta * (v[c] - pr);
        }
    }
    for (int ii = 0; ii < r; ++ii)
        for (int i = ii * sl; i < (ii + 1) * sl; ++i) {
            double *row = S + (size_t)i * Dv;
            for (int c = 0; c < Dv; ++c) row[c] += kt[i] * d[(size_t)ii * Dv + c];
        }
}

/*
 * Backward of oracle_masked_deltaproduct_fwd, tokens from last to first.  Per
 * token, with D the decayed state, sub-row i's read key kr_i (slice j of k
 * times mask[i][j]) and write key kw_i (slice i of k, zero elsewhere),
 * e_i = v - D^T kr_i and S = D + sum_i b kw_i e_i^T, the adjoint G of S gives
 *   w_i = G^T kw_i;  dv = b sum_i w_i;  db = sum_i kw_i . (G e_i)
 *   dkw_i = b G e_i;  dkr_i = -b D w_i;  dD = G - b sum_i kr_i w_i^T
 * then dk's slice j = slice j of (dkw_j + sum_i mask[i][j] dkr_i), dg = <dD, D>
 * and the state entering the token gets e^{g} dD.  Output, norms, shapes and
 * checkpoints (rebuilt with the forward's token step) as oracle_deltaproduct_bwd, with k, dk [B,H,T,Dk], v, dv
 * [B,H,T,Dv] and beta, dbeta [B,H,T].
 */
int oracle_masked_deltaproduct_bwd(const double *q, const double *k, const double *v,
                                   const double *beta, const double *g, const double *mask,
                                   const double *s0, const double *dout, const double *dsf, double *dq,
                                   double *dk, double *dv, double *dbeta, double *dg, double *ds0, int B,
                                   int H, int T, int r, int Dk, int Dv, double scale, int l2norm) {
    if (r < 1 || Dk % r != 0) return -2;
    const int BH = B * H;
    const int sl = Dk / r;
    const int BLK = 64;
    const int nblk = (T + BLK - 1) / BLK;
    const size_t SD = (size_t)Dk * Dv;
    int failed = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
    for (int bh = 0; bh < BH; ++bh) {
        double *Cp = (double *)malloc(sizeof(double) * SD * (nblk > 0 ? nblk : 1));
        double *E = (double *)malloc(sizeof(double) * SD * BLK);
        double *D = (double *)malloc(sizeof(double) * SD);
        double *S = (double *)malloc(sizeof(double) * SD);
        double *G = (double *)malloc(sizeof(double) * SD);
        double *kr = (double *)malloc(sizeof(double) * (size_t)r * Dk);
        double *ev = (double *)malloc(sizeof(double) * (size_t)r * Dv);
        double *wv = (double *)malloc(sizeof(double) * (size_t)r * Dv);
        double *z = (double *)malloc(sizeof(double) * (size_t)r * Dv);
        double *vec = (double *)malloc(sizeof(double) * (size_t)(4 * Dk));
        if (!Cp || !E || !D || !S || !G || !kr || !ev || !wv || !z || !vec) {
            failed |= 1;
        } else {
            double *kt = vec, *qt = vec + Dk, *gk = vec + 2 * Dk, *tq = vec + 3 * Dk;
            if (s0)
                memcpy(S, s0 + (size_t)bh * SD, sizeof(double) * SD);
            else
                memset(S, 0, sizeof(double) * SD);
            for (int t = 0; t < T; ++t) {
                if (t % BLK == 0) memcpy(Cp + (size_t)(t / BLK) * SD, S, sizeof(double) * SD);
                const size_t tok = (size_t)bh * T + t;
                masked_token_step(S, k + tok * Dk, v + tok * Dv, beta[tok], g[tok], mask, r, Dk, Dv, l2norm, kt, z, ev);
            }
            if (dsf)
                memcpy(G, dsf + (size_t)bh * SD, sizeof(double) * SD);
            else
                memset(G, 0, sizeof(double) * SD);
            for (int b = nblk - 1; b >= 0; --b) {
                const int t0 = b * BLK, t1 = (t0 + BLK < T) ? t0 + BLK : T;
                memcpy(E, Cp + (size_t)b * SD, sizeof(double) * SD);
                for (int t = t0; t + 1 < t1; ++t) {
                    const size_t tok = (size_t)bh * T + t;
                    double *Sn = E + (size_t)(t - t0 + 1) * SD;
                    memcpy(Sn, E + (size_t)(t - t0) * SD, sizeof(double) * SD);
                    masked_token_step(Sn, k + tok * Dk, v + tok * Dv, beta[tok], g[tok], mask, r, Dk, Dv, l2norm, kt, z,
                                      ev);
                }
                for (int t = t1 - 1; t >= t0; --t) {
                    const size_t tok = (size_t)bh * T + t;
                    const double a = exp(g[tok]);
                    memcpy(S, E + (size_t)(t - t0) * SD, sizeof(double) * SD);
                    masked_token_step(S, k + tok * Dk, v + tok * Dv, beta[tok], g[tok], mask, r, Dk, Dv, l2norm, kt, z,
                                      ev); /* S: the state after the token; kt: its (unit) key */
                    const double *Et = E + (size_t)(t - t0) * SD;
                    for (size_t x = 0; x < SD; ++x) D[x] = a * Et[x];
                    /* e_i = v - D^T kr_i, and the read keys */
                    for (int i = 0; i < r; ++i)
                        for (int m = 0; m < Dk; ++m) kr[(size_t)i * Dk + m] = mask[i * r + m / sl] * kt[m];
                    for (int i = 0; i < r; ++i)
                        for (int c = 0; c < Dv; ++c) {
                            double pr = 0.0;
                            for (int m = 0; m < Dk; ++m) pr += kr[(size_t)i * Dk + m] * D[(size_t)m * Dv + c];
                            ev[(size_t)i * Dv + c] = v[tok * Dv + c] - pr;
                        }
                    /* output */
                    const double *go = dout + tok * Dv;
                    memcpy(qt, q + tok * Dk, sizeof(double) * Dk);
                    if (l2norm) l2_normalise(qt, Dk);
                    for (int m = 0; m < Dk; ++m) {
                        double acc = 0.0;
                        for (int c = 0; c < Dv; ++c) {
                            acc += S[(size_t)m * Dv + c] * go[c];
                            G[(size_t)m * Dv + c] += scale * qt[m] * go[c];
                        }
                        tq[m] = scale * acc;
                    }
                    if (l2norm)
                        l2_normalise_bwd(q + tok * Dk, tq, dq + tok * Dk, Dk);
                    else
                        memcpy(dq + tok * Dk, tq, sizeof(double) * Dk);
                    /* w_i = G^T kw_i (slice i rows only) */
                    const double bt = beta[tok];
                    for (int i = 0; i < r; ++i)
                        for (int c = 0; c < Dv; ++c) {
                            double acc = 0.0;
                            for (int m = i * sl; m < (i + 1) * sl; ++m) acc += G[(size_t)m * Dv + c] * kt[m];
                            wv[(size_t)i * Dv + c] = acc;
                        }
                    double db = 0.0;
                    for (int c = 0; c < Dv; ++c) {
                        double acc = 0.0;
                        for (int i = 0; i < r; ++i) acc += wv[(size_t)i * Dv + c];
                        dv[tok * Dv + c] = bt * acc;
                    }
                    for (int m = 0; m < Dk; ++m) {
                        const int i = m / sl; /* the write key of sub-row i covers slice i */
                        double ge = 0.0;
                        for (int c = 0; c < Dv; ++c) ge += G[(size_t)m * Dv + c] * ev[(size_t)i * Dv + c];
                        db += kt[m] * ge;
                        double acc = bt * ge; /* dkw_i at row m */
                        for (int ii = 0; ii < r; ++ii) {
                            double dw = 0.0;
                            for (int c = 0; c < Dv; ++c) dw += D[(size_t)m * Dv + c] * wv[(size_t)ii * Dv + c];
                            acc += mask[ii * r + i] * (-bt * dw); /* mask[ii][j] dkr_ii, j = slice of m */
                        }
                        gk[m] = acc;
                    }
                    dbeta[tok] = db;
                    if (l2norm)
                        l2_normalise_bwd(k + tok * Dk, gk, dk + tok * Dk, Dk);
                    else
                        memcpy(dk + tok * Dk, gk, sizeof(double) * Dk);
                    /* dD = G - b sum_i kr_i w_i^T;  dg = <dD, D>;  G <- e^{g} dD */
                    for (int m = 0; m < Dk; ++m)
                        for (int c = 0; c < Dv; ++c) {
                            double acc = 0.0;
                            for (int i = 0; i < r; ++i) acc += kr[(size_t)i * Dk + m] * wv[(size_t)i * Dv + c];
                            G[(size_t)m * Dv + c] -= bt * acc;
                        }
                    double dd = 0.0;
                    for (size_t x = 0; x < SD; ++x) dd += G[x] * D[x];
                    dg[tok] = dd;
                    for (size_t x = 0; x < SD; ++x) G[x] *= a;
                }
            }
            if (ds0) memcpy(ds0 + (size_t)bh * SD, G, sizeof(double) * SD);
        }
        free(Cp);
        free(E);
        free(D);
        free(S);
        free(G);
        free(kr);
        free(ev);
        free(wv);
        free(z);
        free(vec);
    }
    return failed ? -1 : 0;
}
