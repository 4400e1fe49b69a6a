/*
 * TEST INFRASTRUCTURE ONLY -- slow, plain float64 CPU reference ("oracle") for
 * volumetric delay-and-sum (DAS) beamforming.  Only the tests, the package's
 * smoke check and the benchmark's CPU-baseline leg load it.  The product
 * library never includes, links or calls this file, and this file shares no
 * code, header, table or constant with the CUDA sources.
 *
 * What it computes -- the per-voxel accumulation that the ffdas paper
 * ("ffdas: volumetric ultrasound reconstruction at warp speed", Methods, the
 * accumulation it numbers Eq. (2); ffdas docs "How It Works", section "The
 * computational challenge") sums over every receiver and transmit event:
 *
 *   y[b,n] = sum_q sum_m  w_tx[q,n] * w_rx[m,n] * P_qmn * S_bqm(f_qmn)
 *
 *   tau_qmn = tau_tx[q,n] + |x_n - r_m| / c            (two-way delay, seconds)
 *   f_qmn   = (tau_qmn - t0) * fs                      (fractional sample index)
 *   S(f)    = (1 - a) * s[k0] + a * s[k0 + 1],  k0 = floor(f), a = f - k0
 *             with s[k] = 0 for every k outside [0, K-1]
 *   w_rx    = 1 if dz > 0 and (2 F#) * rho <= dz, else 0   (F-number aperture;
 *             rho = lateral distance, dz = depth of the voxel below the receiver;
 *             F# <= 0 switches the aperture off: w_rx = 1 for every receiver)
 *   P_qmn   = exp(+i 2 pi f_demod tau_qmn) for complex (IQ) data, 1 for real data
 *
 * Sources of each step:
 *  - transmit delay/weight given per (q, n); receive delay and weight derived
 *    from the receiver geometry (ffdas paper, Methods, first paragraph);
 *  - linear interpolation between the two neighbouring samples k and k + 1
 *    (ffdas paper, Methods, tensor-core paragraph);
 *  - the text of Eq. (2) itself did not survive on the pages, so four steps
 *    are readings of the plain formula: a sample outside the record counts as
 *    zero on its own (the pair is not dropped as a whole); t0 is the time of
 *    sample 0 in seconds; the aperture is a 0/1 cone about the +z array normal
 *    with half-width dz / (2 F#), boundary included; the IQ phase uses the full
 *    two-way delay tau (t0 excluded) with a + sign.
 *
 * Loops run voxel -> transmit -> receiver -> frame with no blocking, fusion or
 * reordering; OpenMP splits the voxel loop only.  All arithmetic is double.
 *
 * Aperture ties: a receiver whose aperture test |(2F#)^2 rho^2 - dz^2| is within
 * tie_rel * dz^2 of the boundary may legitimately flip in float32.  For those
 * pairs the oracle adds |contribution| to slack[b,n] (whether or not the pair is
 * counted), so a comparison can allow exactly that much extra difference.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL 1

static const double ORACLE_TWO_PI = 6.28318530717958647692528676655900577;

/* Voxel positions of a regular grid: n = ix + nx * (iy + ny * iz),
 * x = x0 + ix * dx (same for y, z).  Writes n_eval x 3 doubles. */
int das_oracle_voxel_positions(int nx, int ny, int nz,
                               double x0, double y0, double z0,
                               double dx, double dy, double dz,
                               const int64_t *idx, int64_t n_eval, double *xyz)
{
    if (nx <= 0 || ny <= 0 || nz <= 0 || (n_eval > 0 && (!idx || !xyz)))
        return ORACLE_EINVAL;
    const int64_t n_total = (int64_t)nx * ny * nz;
    for (int64_t e = 0; e < n_eval; ++e) {
        const int64_t n = idx[e];
        if (n < 0 || n >= n_total) return ORACLE_EINVAL;
        const int64_t ix = n % nx;
        const int64_t iy = (n / nx) % ny;
        const int64_t iz = n / ((int64_t)nx * ny);
        xyz[3 * e + 0] = x0 + (double)ix * dx;
        xyz[3 * e + 1] = y0 + (double)iy * dy;
        xyz[3 * e + 2] = z0 + (double)iz * dz;
    }
    return ORACLE_OK;
}

/* Sample k of receive line (b, q, m) in the B x Q x M x K record; zero outside
 * the record.  rf_type: 0 float32, 1 complex64, 2 float64, 3 complex128;
 * complex data are interleaved (re, im) pairs. */
static double element(const void *rf, int is_double, int64_t j)
{
    return is_double ? ((const double *)rf)[j] : (double)((const float *)rf)[j];
}

static void sample_at(const void *rf, int rf_type, int Q, int M, int K,
                      int b, int q, int m, int64_t k, double *re, double *im)
{
    const int is_double = rf_type >> 1;
    if (k < 0 || k > (int64_t)K - 1) {
        *re = 0.0;
        *im = 0.0;
        return;
    }
    const int64_t i = (((int64_t)b * Q + q) * M + m) * K + k;
    if (rf_type & 1) {
        *re = element(rf, is_double, 2 * i);
        *im = element(rf, is_double, 2 * i + 1);
    } else {
        *re = element(rf, is_double, i);
        *im = 0.0;
    }
}

/*
 * Evaluates y[:, n] for the n_eval voxels listed in vox_idx (positions in
 * vox_xyz, n_eval x 3).  tau_tx and w_tx are Q x N (float32, as the library
 * receives them); rf is B x Q x M x K of rf_type (0 float32, 1 complex64,
 * 2 float64, 3 complex128; complex interleaved).  out is B x n_eval (x 2
 * interleaved when complex); slack is B x n_eval or NULL.  Returns 0 on success.
 */
int das_oracle_beamform(int B, int Q, int M, int K, int64_t N,
                        const void *rf, int rf_type,
                        const float *tau_tx, const float *w_tx,
                        const double *rx_xyz,
                        const double *vox_xyz, const int64_t *vox_idx, int64_t n_eval,
                        double c, double fs, double t0, double fnum, double f_demod,
                        double tie_rel, double *out, double *slack, int nthreads)
{
    if (B < 0 || Q < 0 || M < 0 || K < 0 || N < 0 || n_eval < 0) return ORACLE_EINVAL;
    if (rf_type < 0 || rf_type > 3) return ORACLE_EINVAL;
    const int is_complex = rf_type & 1;
    if (!(c > 0.0) || !(fs > 0.0)) return ORACLE_EINVAL;
    if (n_eval > 0 && (!vox_xyz || !vox_idx || !out)) return ORACLE_EINVAL;
    if ((int64_t)B * Q * M * K > 0 && !rf) return ORACLE_EINVAL;
    if ((int64_t)Q * N > 0 && (!tau_tx || !w_tx)) return ORACLE_EINVAL;
    if (M > 0 && !rx_xyz) return ORACLE_EINVAL;
    for (int64_t e = 0; e < n_eval; ++e)
        if (vox_idx[e] < 0 || vox_idx[e] >= N) return ORACLE_EINVAL;

    const int ncomp = is_complex ? 2 : 1;
    memset(out, 0, sizeof(double) * (size_t)B * (size_t)n_eval * (size_t)ncomp);
    if (slack) memset(slack, 0, sizeof(double) * (size_t)B * (size_t)n_eval);
    const int rotate = is_complex && f_demod != 0.0;

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t e = 0; e < n_eval; ++e) {
        const int64_t n = vox_idx[e];
        const double px = vox_xyz[3 * e + 0];
        const double py = vox_xyz[3 * e + 1];
        const double pz = vox_xyz[3 * e + 2];
        for (int q = 0; q < Q; ++q) {
            const double tau_t = (double)tau_tx[(int64_t)q * N + n];
            const double wt = (double)w_tx[(int64_t)q * N + n];
            for (int m = 0; m < M; ++m) {
                const double ex = px - rx_xyz[3 * m + 0];
                const double ey = py - rx_xyz[3 * m + 1];
                const double ez = pz - rx_xyz[3 * m + 2];
                const double dist = sqrt(ex * ex + ey * ey + ez * ez);

                /* F-number receive aperture (0/1 weight) */
                int inside = 1, tie = 0;
                if (fnum > 0.0) {
                    const double lhs = (2.0 * fnum) * (2.0 * fnum) * (ex * ex + ey * ey);
                    const double rhs = ez * ez;
                    inside = (ez > 0.0) && (lhs <= rhs);
                    tie = (ez > 0.0) && (fabs(lhs - rhs) <= tie_rel * rhs);
                }
                if (!inside && !tie) continue;

                const double tau = tau_t + dist / c;
                const double f = (tau - t0) * fs;
                if (!isfinite(f)) continue;
                const double k0f = floor(f);
                if (k0f < -1.0 || k0f > (double)K - 1.0) continue; /* both samples outside */
                const double a = f - k0f;
                const int64_t k0 = (int64_t)k0f;

                double pr = 1.0, pim = 0.0;
                if (rotate) {
                    const double ph = ORACLE_TWO_PI * f_demod * tau;
                    pr = cos(ph);
                    pim = sin(ph);
                }
                for (int b = 0; b < B; ++b) {
                    double s0r, s0i, s1r, s1i;
                    sample_at(rf, rf_type, Q, M, K, b, q, m, k0, &s0r, &s0i);
                    sample_at(rf, rf_type, Q, M, K, b, q, m, k0 + 1, &s1r, &s1i);
                    const double vr = (1.0 - a) * s0r + a * s1r;
                    const double vi = (1.0 - a) * s0i + a * s1i;
                    const double cr = wt * (vr * pr - vi * pim);
                    const double ci = wt * (vr * pim + vi * pr);
                    const int64_t o = (int64_t)b * n_eval + e;
                    if (inside) {
                        out[ncomp * o] += cr;
                        if (is_complex) out[ncomp * o + 1] += ci;
                    }
                    if (tie && slack) slack[o] += sqrt(cr * cr + ci * ci);
                }
            }
        }
    }
    return ORACLE_OK;
}

/*
 * RF layout permute as a plain index map (ffdas paper, Methods, batch-inner
 * paragraph: B x Q x M x K with k contiguous -> K x Q x M x B with b
 * contiguous).  layout 0 writes K x Q x M x B; layout 1 writes Q x M x K x B
 * (same per-(q,m) transpose of the (b,k) plane, rows of one (q,m) adjacent).
 * Elements are copied as opaque bytes (elem_bytes each), so the result is
 * bit-exact by construction.
 */
int das_oracle_permute(const void *in, void *out, int elem_bytes,
                       int B, int Q, int M, int K, int layout)
{
    if (B < 0 || Q < 0 || M < 0 || K < 0 || elem_bytes <= 0) return ORACLE_EINVAL;
    if (layout != 0 && layout != 1) return ORACLE_EINVAL;
    if ((int64_t)B * Q * M * K > 0 && (!in || !out)) return ORACLE_EINVAL;
    const unsigned char *src = (const unsigned char *)in;
    unsigned char *dst = (unsigned char *)out;
    for (int b = 0; b < B; ++b)
        for (int q = 0; q < Q; ++q)
            for (int m = 0; m < M; ++m)
                for (int k = 0; k < K; ++k) {
                    const int64_t i = (((int64_t)b * Q + q) * M + m) * K + k;
                    const int64_t o = layout == 0
                        ? (((int64_t)k * Q + q) * M + m) * B + b
                        : (((int64_t)q * M + m) * K + k) * B + b;
                    memcpy(dst + o * elem_bytes, src + i * elem_bytes, (size_t)elem_bytes);
                }
    return ORACLE_OK;
}
