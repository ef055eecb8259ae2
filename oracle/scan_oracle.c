/*
 * Selective state-space scan: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline use it. It shares no code, header or constant with the CUDA path.
 *
 * It evaluates the selective SSM (S6) exactly as the pages define it, one
 * (batch, channel) row at a time, sequentially in time, in double precision,
 * with the C library's exp/log1p, no vectorisation and no reassociation:
 *
 *   dt      = delta[l] (+ bias)                 -- bias of the dt projection
 *   dt      = softplus(dt)   if ORACLE_SOFTPLUS -- "Mamba 论文精读" (youngju.dev) §3.1,
 *                                                  Delta_t = softplus(Linear_Delta(x_t))
 *   dA[n]   = exp(dt * A[n])                     -- same page §2.2 (ZOH: A_bar = exp(Delta A))
 *   dBu[n]  = dt * B[l][n] * u[l]                -- same page §3.3 simplified scan: B_bar = Delta * B
 *   dBu[n]  = expm1(dt*A[n])/A[n] * B[l][n] * u[l]
 *                            if ORACLE_ZOH       -- same page §2.2, exact zero-order hold:
 *                                                  B_bar = (Delta A)^-1 (exp(Delta A) - I) Delta B, which
 *                                                  for a diagonal A is (exp(dt A[n]) - 1) / A[n] per state
 *                                                  (dt, its limit, where dt*A[n] = 0)
 *   h[n]    = dA[n] * h[n] + dBu[n],  h = 0 before the first step
 *                                                -- same page §2.2 recurrence h_t = A_bar h_{t-1} + B_bar x_t
 *   y[l]    = sum_n C[l][n] * h[n]               -- same page §2.2, y_t = C h_t (read after the update)
 *   y[l]   += D * u[l]        if D given         -- "Mamba的基础知识" (weblog-19d), 状态空间模型 section:
 *                                                  the D term is a skip connection
 *   y[l]   *= silu(z[l])      if z given         -- "Mamba 论文精读" §3.4 block: y = y * silu(z)
 *
 * The state update for decoding is one iteration of the same loop body applied
 * to a given state ("mamba->jamba" (blog.csdn.net) §2.2: constant-time recurrent
 * inference; "Mamba 论文精读" §6: O(1) per token, fixed state). Both entry points
 * call the same step function, so L successive updates from h = 0 reproduce the
 * scan bit for bit.
 *
 * softplus is written as max(x,0) + log1p(exp(-|x|)), which is the same
 * function as log(1 + exp(x)) for every x but does not overflow for large x.
 *
 * `flags` is a bit set: ORACLE_SOFTPLUS (1) applies softplus to dt,
 * ORACLE_ZOH (2) uses the exact zero-order-hold B_bar instead of Delta * B.
 */
#include <math.h>
#include <stdlib.h>
#include <stddef.h>
#include <stdint.h>

#define ORACLE_SOFTPLUS 1
#define ORACLE_ZOH 2

static double softplus_ref(double x)
{
    double ax = x < 0.0 ? -x : x;
    return (x > 0.0 ? x : 0.0) + log1p(exp(-ax));
}

static double silu_ref(double z)
{
    return z / (1.0 + exp(-z));
}

/* Exact zero-order-hold input gain of one diagonal state: (exp(dt a) - 1) / a,
 * written with expm1 so that small dt*a loses nothing to cancellation; its
 * value at dt*a = 0 is the limit dt. */
static double zoh_gain(double dt, double a)
{
    double x = dt * a;
    return x == 0.0 ? dt : expm1(x) / a;
}

/* Its derivative with respect to a: (dt e^{dt a} - gain) / a, which cancels
 * for small dt*a; there its series dt^2 (1/2 + x/3 + x^2/8 + x^3/30), x = dt a
 * (the next term, x^4/144, is below 1e-18 of the first for |x| < 1e-4). The
 * derivative with respect to dt is e^{dt a}. */
static double zoh_gain_da(double dt, double a)
{
    double x = dt * a;
    if (fabs(x) < 1e-4) return dt * dt * (0.5 + x * (1.0 / 3.0 + x * (1.0 / 8.0 + x / 30.0)));
    return (dt * exp(x) - expm1(x) / a) / a;
}

/* One time step of the selective SSM for one row.
 * h[dstate] in/out; A_row[dstate]; Bt, Ct: the step's B and C, read with
 * stride bc_stride (seqlen for the scan layout (batch, dstate, seqlen), 1 for
 * the decode layout (batch, dstate)). Returns y for the step. */
static double ssm_step(double* h, int64_t dstate, const double* A_row,
                       const double* Bt, const double* Ct, int64_t bc_stride,
                       double u, double delta, const double* zp,
                       const double* Dp, const double* biasp, int flags)
{
    double dt = delta;
    if (biasp) dt += *biasp;
    if (flags & ORACLE_SOFTPLUS) dt = softplus_ref(dt);
    double y = 0.0;
    for (int64_t n = 0; n < dstate; ++n) {
        double dA = exp(dt * A_row[n]);
        double dBu = (flags & ORACLE_ZOH) ? zoh_gain(dt, A_row[n]) * Bt[n * bc_stride] * u
                                          : dt * Bt[n * bc_stride] * u;
        h[n] = dA * h[n] + dBu;
        y += Ct[n * bc_stride] * h[n];
    }
    if (Dp) y += (*Dp) * u;
    if (zp) y *= silu_ref(*zp);
    return y;
}

/*
 * Scan of nrows independent rows over seqlen steps.
 *   u, delta, z : (nrows, seqlen)        z may be NULL
 *   A           : (nrows, dstate)        the A row of each row's channel
 *   Dskip, bias : (nrows)                either may be NULL
 *   B, C        : (nbatch, dstate, seqlen), row r uses batch bidx[r]
 *   h0          : (nrows, dstate) state before the first step, or NULL for
 *                 zero (a scan that continues an earlier one, "mamba->jamba"
 *                 §2.2: the recurrence carries h from one token to the next)
 *   y           : (nrows, seqlen) out
 *   hlast       : (nrows, dstate) out, may be NULL: state after the last step
 * Returns 0, or -1 if dstate is out of range.
 */
int oracle_scan(int64_t nrows, int64_t seqlen, int64_t dstate,
                const double* u, const double* delta, const double* z,
                const double* A, const double* Dskip, const double* bias,
                const double* B, const double* C, const int64_t* bidx,
                const double* h0, int flags, double* y, double* hlast)
{
    double h[1024];
    if (dstate < 1 || dstate > 1024) return -1;
    for (int64_t r = 0; r < nrows; ++r) {
        const double* Bb = B + bidx[r] * dstate * seqlen;
        const double* Cb = C + bidx[r] * dstate * seqlen;
        for (int64_t n = 0; n < dstate; ++n) h[n] = h0 ? h0[r * dstate + n] : 0.0;
        for (int64_t l = 0; l < seqlen; ++l) {
            int64_t i = r * seqlen + l;
            y[i] = ssm_step(h, dstate, A + r * dstate, Bb + l, Cb + l, seqlen,
                            u[i], delta[i], z ? z + i : NULL,
                            Dskip ? Dskip + r : NULL, bias ? bias + r : NULL,
                            flags);
        }
        if (hlast)
            for (int64_t n = 0; n < dstate; ++n) hlast[r * dstate + n] = h[n];
    }
    return 0;
}

/*
 * Single-token state update of nrows rows.
 *   state       : (nrows, dstate) in/out
 *   u, delta, z : (nrows)                z may be NULL
 *   A           : (nrows, dstate)
 *   Dskip, bias : (nrows)                either may be NULL
 *   B, C        : (nbatch, dstate), row r uses batch bidx[r]
 *   y           : (nrows) out
 */
int oracle_state_update(int64_t nrows, int64_t dstate, double* state,
                        const double* u, const double* delta, const double* z,
                        const double* A, const double* Dskip, const double* bias,
                        const double* B, const double* C, const int64_t* bidx,
                        int flags, double* y)
{
    if (dstate < 1 || dstate > 1024) return -1;
    for (int64_t r = 0; r < nrows; ++r) {
        y[r] = ssm_step(state + r * dstate, dstate, A + r * dstate,
                        B + bidx[r] * dstate, C + bidx[r] * dstate, 1,
                        u[r], delta[r], z ? z + r : NULL,
                        Dskip ? Dskip + r : NULL, bias ? bias + r : NULL,
                        flags);
    }
    return 0;
}

/*
 * Gradients of the scan (reverse-mode differentiation of the loop above, the
 * backward pass "mamba->jamba" §2.3 describes: A_bar and B_bar are recomputed
 * from the inputs, here by storing the forward states of the row).
 *
 * With the loss L = sum_l dy[l] * y[l], per row:
 *   gate      : y = p * silu(z), p = C.h + D u; dp = dy silu(z),
 *               dz = dy * p * silu'(z), silu'(z) = s (1 + z (1 - s)), s = sigmoid(z)
 *   readout   : dC[n][l] = dp h_l[n];  dD += dp u;  du += dp D;  gh[n] = g[n] + dp C[n]
 *   recurrence h_l = e h_{l-1} + dt u B, e = exp(dt A):
 *               dB[n][l] = gh[n] dt u;  d(dt u) += gh[n] B[n];
 *               de = gh[n] h_{l-1}[n]:  d(dt) += de e A[n],  dA[n] += de e dt;
 *               g[n] = gh[n] e          (the gradient reaching h_{l-1})
 *   dt u      : du += d(dt u) dt;  d(dt) += d(dt u) u
 *   dt        : ddelta = d(dt) * sigmoid(delta + bias) with softplus, else d(dt);
 *               dbias += ddelta
 *   dh0 = g after step 0.
 * With ORACLE_ZOH the input term is gain(dt, A[n]) u B[n] instead of dt u B[n]:
 *               dB[n][l] = gh[n] gain u;  du += gh[n] B[n] gain;
 *               d(dt) += gh[n] B[n] u e;  dA[n] += gh[n] B[n] u dgain/dA.
 * Outputs per row (the caller sums dA/dD/dbias over batch rows and dB/dC over
 * the channels of a batch row):
 *   du, ddelta, dz : (nrows, seqlen)          dz written only if z given
 *   dA             : (nrows, dstate)
 *   dD, dbias      : (nrows), either may be NULL
 *   dB, dC         : (nrows, dstate, seqlen)
 *   dh0            : (nrows, dstate), may be NULL
 * h0 and flags as in oracle_scan. Returns 0, -1 if dstate is out of range,
 * -2 if the work buffer cannot be allocated.
 */
int oracle_scan_bwd(int64_t nrows, int64_t seqlen, int64_t dstate,
                    const double* u, const double* delta, const double* z,
                    const double* A, const double* Dskip, const double* bias,
                    const double* B, const double* C, const int64_t* bidx,
                    const double* h0, int flags, const double* dy,
                    double* du, double* ddelta, double* dz, double* dA,
                    double* dD, double* dbias, double* dB, double* dC, double* dh0)
{
    const int softplus_flag = flags & ORACLE_SOFTPLUS;
    const int zoh = flags & ORACLE_ZOH;
    if (dstate < 1 || dstate > 1024) return -1;
    /* H[(l + 1) * dstate + n] = state after step l; H[n] = state before step 0 */
    double* H = (double*)malloc(sizeof(double) * (size_t)(seqlen + 1) * (size_t)dstate);
    if (!H) return -2;
    double g[1024];
    for (int64_t r = 0; r < nrows; ++r) {
        const double* Bb = B + bidx[r] * dstate * seqlen;
        const double* Cb = C + bidx[r] * dstate * seqlen;
        const double* Ar = A + r * dstate;
        const double Dr = Dskip ? Dskip[r] : 0.0;
        for (int64_t n = 0; n < dstate; ++n) H[n] = h0 ? h0[r * dstate + n] : 0.0;
        /* forward: states of every step */
        for (int64_t l = 0; l < seqlen; ++l) {
            const int64_t i = r * seqlen + l;
            double dt = delta[i] + (bias ? bias[r] : 0.0);
            if (softplus_flag) dt = softplus_ref(dt);
            for (int64_t n = 0; n < dstate; ++n) {
                const double gain = zoh ? zoh_gain(dt, Ar[n]) : dt;
                H[(l + 1) * dstate + n] = exp(dt * Ar[n]) * H[l * dstate + n] + gain * Bb[n * seqlen + l] * u[i];
            }
        }
        /* reverse */
        for (int64_t n = 0; n < dstate; ++n) { g[n] = 0.0; dA[r * dstate + n] = 0.0; }
        double dDr = 0.0, dbr = 0.0;
        for (int64_t l = seqlen - 1; l >= 0; --l) {
            const int64_t i = r * seqlen + l;
            const double x = delta[i] + (bias ? bias[r] : 0.0);
            const double dt = softplus_flag ? softplus_ref(x) : x;
            const double* hl = H + (l + 1) * dstate;
            const double* hp = H + l * dstate;
            double p = Dr * u[i];
            for (int64_t n = 0; n < dstate; ++n) p += Cb[n * seqlen + l] * hl[n];
            double dp = dy[i];
            if (z) {
                const double s = 1.0 / (1.0 + exp(-z[i]));
                dz[i] = dy[i] * p * s * (1.0 + z[i] * (1.0 - s));
                dp = dy[i] * z[i] * s;
            }
            dDr += dp * u[i];
            double dui = dp * Dr;
            double ddtu = 0.0, ddt = 0.0;
            for (int64_t n = 0; n < dstate; ++n) {
                const double e = exp(dt * Ar[n]);
                const double gh = g[n] + dp * Cb[n * seqlen + l];
                dC[(r * dstate + n) * seqlen + l] = dp * hl[n];
                if (zoh) {
                    const double gain = zoh_gain(dt, Ar[n]);
                    const double ghbu = gh * Bb[n * seqlen + l] * u[i];
                    dB[(r * dstate + n) * seqlen + l] = gh * gain * u[i];
                    dui += gh * Bb[n * seqlen + l] * gain;
                    ddt += ghbu * e;
                    dA[r * dstate + n] += ghbu * zoh_gain_da(dt, Ar[n]);
                } else {
                    dB[(r * dstate + n) * seqlen + l] = gh * dt * u[i];
                    ddtu += gh * Bb[n * seqlen + l];
                }
                const double de = gh * hp[n];
                ddt += de * e * Ar[n];
                dA[r * dstate + n] += de * e * dt;
                g[n] = gh * e;
            }
            dui += ddtu * dt;
            ddt += ddtu * u[i];
            const double dx = softplus_flag ? ddt / (1.0 + exp(-x)) : ddt;
            du[i] = dui;
            ddelta[i] = dx;
            dbr += dx;
        }
        if (dD) dD[r] = dDr;
        if (dbias) dbias[r] = dbr;
        if (dh0)
            for (int64_t n = 0; n < dstate; ++n) dh0[r * dstate + n] = g[n];
    }
    free(H);
    return 0;
}

/*
 * Causal depthwise convolution followed by SiLU, the step before the scan in
 * the Mamba block ("Mamba 论文精读" (youngju.dev) §3.4: a 1-D convolution over
 * the sequence, padded with width-1 zeros in front and cut back to the
 * sequence length so that step l sees only steps <= l, then SiLU):
 *   u[l] = silu( sum_{k=0}^{width-1} w[k] * x[l - (width-1) + k] + bias )
 * with x at negative steps taken from xprev (the last width-1 inputs of an
 * earlier piece of the sequence, oldest first) or zero when xprev is NULL.
 *   x, u   : (nrows, seqlen)
 *   w      : (nrows, width)    the weights of each row's channel
 *   bias   : (nrows) or NULL
 *   xprev  : (nrows, width-1) or NULL
 * Returns 0, or -1 if width is out of range.
 */
int oracle_causal_conv_silu(int64_t nrows, int64_t seqlen, int64_t width,
                            const double* x, const double* w, const double* bias,
                            const double* xprev, double* u)
{
    if (width < 1 || width > 64) return -1;
    for (int64_t r = 0; r < nrows; ++r) {
        for (int64_t l = 0; l < seqlen; ++l) {
            double acc = bias ? bias[r] : 0.0;
            for (int64_t k = 0; k < width; ++k) {
                const int64_t src = l - (width - 1) + k;
                double xv;
                if (src >= 0) xv = x[r * seqlen + src];
                else xv = xprev ? xprev[r * (width - 1) + (width - 1) + src] : 0.0;
                acc += w[r * width + k] * xv;
            }
            u[r * seqlen + l] = silu_ref(acc);
        }
    }
    return 0;
}

/*
 * State-space dual (SSD) layer of Mamba-2 ("Mamba 论文精读" (youngju.dev) §4.1:
 * the recurrence h_t = A_t h_{t-1} + B_t x_t, y_t = C_t h_t, whose matrix form
 * is Y = (T o M) X with T the causal mask and M semiseparable), read as the
 * Mamba-2 layer of the same page's §5.2 (multi-head, headdim channels a head,
 * a larger state): per batch row b and head h the state is a
 * (headdim x dstate) matrix, the decay is one scalar per head and step, and
 * B, C (one group) are shared by all heads:
 *
 *   dt      = delta[b,h,l] (+ bias[h]);  softplus(dt) if ORACLE_SOFTPLUS
 *   a       = exp(dt * A[h])
 *   H[p][n] = a * H[p][n] + dt * B[b,n,l] * x[b,h*P+p,l]
 *   y[b,h*P+p,l] = sum_n C[b,n,l] * H[p][n]  (+ D[h] * x[b,h*P+p,l])
 *
 *   x, y   : (batch, nheads * headdim, seqlen)   channel d = h * headdim + p
 *   delta  : (batch, nheads, seqlen)
 *   A, D, bias : (nheads)                        D and bias may be NULL
 *   B, C   : (batch, dstate, seqlen)
 *   h0, hlast : (batch, nheads, headdim, dstate) state before the first step
 *               (NULL: zero) and after the last (NULL: not returned)
 * Returns 0, -1 if a size is out of range, -2 if the state buffer cannot be
 * allocated, -3 if flags asks for the ZOH gain (not defined for this form).
 */
int oracle_ssd(int64_t batch, int64_t nheads, int64_t headdim, int64_t dstate, int64_t seqlen,
               const double* x, const double* delta, const double* A,
               const double* B, const double* C, const double* Dskip, const double* bias,
               const double* h0, int flags, double* y, double* hlast)
{
    if (batch < 0 || nheads < 0 || headdim < 1 || dstate < 1 || seqlen < 0) return -1;
    if (flags & ORACLE_ZOH) return -3;
    double* H = (double*)malloc(sizeof(double) * (size_t)headdim * (size_t)dstate);
    if (!H) return -2;
    const int64_t dim = nheads * headdim;
    for (int64_t b = 0; b < batch; ++b) {
        const double* Bb = B + b * dstate * seqlen;
        const double* Cb = C + b * dstate * seqlen;
        for (int64_t h = 0; h < nheads; ++h) {
            const int64_t s0 = ((b * nheads + h) * headdim) * dstate;
            for (int64_t i = 0; i < headdim * dstate; ++i) H[i] = h0 ? h0[s0 + i] : 0.0;
            for (int64_t l = 0; l < seqlen; ++l) {
                double dt = delta[(b * nheads + h) * seqlen + l];
                if (bias) dt += bias[h];
                if (flags & ORACLE_SOFTPLUS) dt = softplus_ref(dt);
                const double a = exp(dt * A[h]);
                for (int64_t p = 0; p < headdim; ++p) {
                    const int64_t i = (b * dim + h * headdim + p) * seqlen + l;
                    const double xv = x[i];
                    double acc = 0.0;
                    for (int64_t n = 0; n < dstate; ++n) {
                        double* hp = H + p * dstate + n;
                        *hp = a * (*hp) + dt * Bb[n * seqlen + l] * xv;
                        acc += Cb[n * seqlen + l] * (*hp);
                    }
                    if (Dskip) acc += Dskip[h] * xv;
                    y[i] = acc;
                }
            }
            if (hlast)
                for (int64_t i = 0; i < headdim * dstate; ++i) hlast[s0 + i] = H[i];
        }
    }
    free(H);
    return 0;
}
