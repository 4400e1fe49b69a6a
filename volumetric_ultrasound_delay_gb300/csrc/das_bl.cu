// BL: the per-voxel baseline (ffdas paper, Methods, baseline paragraph and
// Algorithm 1; ffdas docs, ALG1).  One thread owns one voxel and a tile of
// B_TILE = 8 consecutive frames, loops over receivers and transmits, computes
// the receive delay and aperture weight on the fly, and reads the two samples
// it needs straight from the native B x Q x M x K record (k contiguous), so it
// needs no permute and works for any B and K.
//
// Loop order: receiver outer (one square root per voxel and receiver), transmit
// inner; tau_tx and w_tx are re-read per (q, m) through the L1 cache.  A
// float64 / complex128 variant runs the same loop in double.
#include "das_device.cuh"

namespace das {
namespace {

constexpr int B_TILE = 8;
constexpr int THREADS = 128;

template <bool CPLX>
__global__ void __launch_bounds__(THREADS)
das_bl_kernel(DasGeom g, const RxPos *__restrict__ rx, const float *__restrict__ rf,
              const float *__restrict__ tau, const float *__restrict__ wtx, float *__restrict__ out)
{
    using T = typename std::conditional<CPLX, float2, float>::type;
    const T *rfT = reinterpret_cast<const T *>(rf);
    T *outT = reinterpret_cast<T *>(out);
    const int s = blockIdx.x * THREADS + threadIdx.x;   // voxel slot
    const int b0 = blockIdx.y * B_TILE;
    if (s >= g.N) return;
    const int nb = min(B_TILE, g.B - b0);
    const float3 p = voxel_position(g, s);
    const int n = voxel_index(g, s);
    const long long b_stride = (long long)g.Q * g.M * g.K;

    T acc[B_TILE];
#pragma unroll
    for (int j = 0; j < B_TILE; ++j) acc[j] = T{};

    for (int m = 0; m < g.M; ++m) {
        float d;
        if (!receive_geometry(g, p, __ldg(rx + m), d)) continue;
        for (int q = 0; q < g.Q; ++q) {
            const float wq = __ldg(wtx + (long long)q * g.N + n);
            const float tq = fmaf(__ldg(tau + (long long)q * g.N + n), g.fs, -g.t0fs);
            const float f = tq + d;
            const float fl = floorf(f);
            if (!(fl >= -1.f && fl <= (float)(g.K - 1))) continue;
            const float a = f - fl;
            const int k0 = (int)fl;
            const float w1 = wq * a, w0 = wq - w1;
            const bool v0 = k0 >= 0, v1 = k0 + 1 <= g.K - 1;
            const T *line = rfT + ((long long)b0 * g.Q * g.M + (long long)q * g.M + m) * g.K;
            if constexpr (CPLX) {
                const float2 ph = demod_phase(g, f);
                const float2 W0 = make_float2(w0 * ph.x, w0 * ph.y);
                const float2 W1 = make_float2(w1 * ph.x, w1 * ph.y);
#pragma unroll
                for (int j = 0; j < B_TILE; ++j) {
                    if (j < nb) {
                        const T *l = line + j * b_stride;
                        const float2 s0 = v0 ? __ldg(l + k0) : make_float2(0.f, 0.f);
                        const float2 s1 = v1 ? __ldg(l + k0 + 1) : make_float2(0.f, 0.f);
                        cfma(acc[j], W0, s0);
                        cfma(acc[j], W1, s1);
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < B_TILE; ++j) {
                    if (j < nb) {
                        const T *l = line + j * b_stride;
                        const float s0 = v0 ? __ldg(l + k0) : 0.f;
                        const float s1 = v1 ? __ldg(l + k0 + 1) : 0.f;
                        acc[j] = fmaf(w0, s0, acc[j]);
                        acc[j] = fmaf(w1, s1, acc[j]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < B_TILE; ++j)
        if (j < nb) outT[(long long)(b0 + j) * g.N + n] = acc[j];
}

// float64 / complex128 records: the same loop with every step in double
// (ffdas docs, ALG1: the baseline supports float64 and complex128).
template <bool CPLX>
__global__ void __launch_bounds__(THREADS)
das_bl64_kernel(DasGeom64 g, const Pos64 *__restrict__ rx, const void *__restrict__ rf,
                const float *__restrict__ tau, const float *__restrict__ wtx, void *__restrict__ out)
{
    using T = typename std::conditional<CPLX, double2, double>::type;
    const T *rfT = static_cast<const T *>(rf);
    T *outT = static_cast<T *>(out);
    const int s = blockIdx.x * THREADS + threadIdx.x;   // voxel slot
    const int b0 = blockIdx.y * B_TILE;
    if (s >= g.N) return;
    const int nb = min(B_TILE, g.B - b0);
    const int n = g.order ? __ldg(g.order + s) : s;
    double px, py, pz;
    if (g.vox) {
        px = g.vox[s].x; py = g.vox[s].y; pz = g.vox[s].z;
    } else {
        const int ix = n % g.nx, iy = (n / g.nx) % g.ny, iz = n / (g.nx * g.ny);
        px = g.x0 + ix * g.dx; py = g.y0 + iy * g.dy; pz = g.z0 + iz * g.dz;
    }
    const long long b_stride = (long long)g.Q * g.M * g.K;

    T acc[B_TILE];
#pragma unroll
    for (int j = 0; j < B_TILE; ++j) acc[j] = T{};

    for (int m = 0; m < g.M; ++m) {
        const Pos64 r = rx[m];
        const double ex = px - r.x, ey = py - r.y, ez = pz - r.z;
        const double rho2 = ex * ex + ey * ey;
        if (g.aperture && !(ez > 0.0 && g.ap2 * rho2 <= ez * ez)) continue;
        const double d = sqrt(rho2 + ez * ez);
        for (int q = 0; q < g.Q; ++q) {
            const double wq = (double)__ldg(wtx + (long long)q * g.N + n);
            const double f = (double)__ldg(tau + (long long)q * g.N + n) * g.fs - g.t0fs + d;
            const double fl = floor(f);
            if (!(fl >= -1.0 && fl <= (double)(g.K - 1))) continue;
            const double a = f - fl;
            const int k0 = (int)fl;
            const double w1 = wq * a, w0 = wq - w1;
            const bool v0 = k0 >= 0, v1 = k0 + 1 <= g.K - 1;
            const T *line = rfT + ((long long)b0 * g.Q * g.M + (long long)q * g.M + m) * g.K;
            double2 ph = make_double2(1.0, 0.0);
            if constexpr (CPLX) {
                double cyc = (f + g.t0fs) * g.fd_over_fs;
                cyc -= rint(cyc);
                sincospi(2.0 * cyc, &ph.y, &ph.x);
            }
#pragma unroll
            for (int j = 0; j < B_TILE; ++j) {
                if (j < nb) {
                    const T *l = line + j * b_stride;
                    if constexpr (CPLX) {
                        const double2 s0 = v0 ? l[k0] : make_double2(0.0, 0.0);
                        const double2 s1 = v1 ? l[k0 + 1] : make_double2(0.0, 0.0);
                        const double vr = w0 * s0.x + w1 * s1.x, vi = w0 * s0.y + w1 * s1.y;
                        acc[j].x += vr * ph.x - vi * ph.y;
                        acc[j].y += vr * ph.y + vi * ph.x;
                    } else {
                        const double s0 = v0 ? l[k0] : 0.0;
                        const double s1 = v1 ? l[k0 + 1] : 0.0;
                        acc[j] = fma(w0, s0, fma(w1, s1, acc[j]));
                    }
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < B_TILE; ++j)
        if (j < nb) outT[(long long)(b0 + j) * g.N + n] = acc[j];
}

}  // namespace

cudaError_t launch_bl64(const DasGeom64 &g, const Pos64 *rx, const void *rf, const float *tau,
                        const float *w, void *out, bool cplx, cudaStream_t stream)
{
    dim3 grid((g.N + THREADS - 1) / THREADS, (g.B + B_TILE - 1) / B_TILE);
    if (cplx)
        das_bl64_kernel<true><<<grid, THREADS, 0, stream>>>(g, rx, rf, tau, w, out);
    else
        das_bl64_kernel<false><<<grid, THREADS, 0, stream>>>(g, rx, rf, tau, w, out);
    return cudaGetLastError();
}

cudaError_t launch_bl(const DasGeom &g, const RxPos *rx, const void *rf, const float *tau,
                      const float *w, void *out, bool cplx, cudaStream_t stream)
{
    dim3 grid((g.N + THREADS - 1) / THREADS, (g.B + B_TILE - 1) / B_TILE);
    if (cplx)
        das_bl_kernel<true><<<grid, THREADS, 0, stream>>>(g, rx, static_cast<const float *>(rf), tau,
                                                          w, static_cast<float *>(out));
    else
        das_bl_kernel<false><<<grid, THREADS, 0, stream>>>(g, rx, static_cast<const float *>(rf), tau,
                                                           w, static_cast<float *>(out));
    return cudaGetLastError();
}

}  // namespace das
