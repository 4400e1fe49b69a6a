// das_beamform_noalloc: the brick-kernel beamform for callers that must not
// allocate device memory.
//
// Some callers cannot call cudaMalloc once they are running: the real-time
// reconstruction loop of a scanner, where cudaMalloc's implicit device
// synchronisation would stall acquisition, or a host framework that hands out
// all device memory from its own pool at start-up and forbids other
// allocations.  A plan allocates its geometry copy and its permute scratch, so
// such callers use this entry point instead: it takes every input and output
// from the caller and keeps its scratch in the static array below.
//
// The scratch is a file-scope __device__ array of DAS_NOALLOC_SCRATCH_BYTES
// (64 MiB).  Every GPU on which libdas's kernels are loaded holds it until the
// process exits.  Host code may not use the array's name as an address (on the
// host it is only a stand-in), so each call looks up its device address with
// cudaGetSymbolAddress, with the caller's device current, and passes that
// pointer to the kernels.  The lookup allocates nothing and is repeated on
// every call rather than cached: after a cudaDeviceReset, or under another
// context of the same device, the array lives at a different address.
#include <cmath>
#include <cstdio>

#include "das_internal.cuh"

#define DAS_NOALLOC_SCRATCH_BYTES (64ull << 20)

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[DAS_NOALLOC_SCRATCH_BYTES];

das_status reject(das_status st, const char *msg)
{
    char text[320];
    snprintf(text, sizeof(text), "das_beamform_noalloc: %s", msg);
    das::record_error(text);
    return st;
}

// receiver positions (metres, M x 3) -> sample units in the scratch array,
// scaled in double and rounded once to float, as a plan scales them on the host
__global__ void scale_receivers(const float *__restrict__ rx_xyz, RxPos *__restrict__ dst, int M,
                                double s)
{
    const int m = blockIdx.x * blockDim.x + threadIdx.x;
    if (m < M)
        dst[m] = make_float4((float)((double)rx_xyz[3 * m] * s), (float)((double)rx_xyz[3 * m + 1] * s),
                             (float)((double)rx_xyz[3 * m + 2] * s), 0.f);
}

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

extern "C" das_status das_beamform_noalloc(const das_grid *grid, const float *rx_xyz, float c,
                                           float fs, float t0, float fnum, double f_demod,
                                           das_dtype dtype, int B, int Q, int M, int K,
                                           const void *rf, const float *tau_tx, const float *w_tx,
                                           void *out, cudaStream_t stream)
{
    das::record_error("");
    if (!grid || !rx_xyz || !rf || !tau_tx || !w_tx || !out)
        return reject(DAS_ERR_INVALID_ARG, "NULL argument");
    if (grid->nx < 1 || grid->ny < 1 || grid->nz < 1 || B < 1 || Q < 1 || M < 1 || K < 1)
        return reject(DAS_ERR_INVALID_ARG, "grid dimensions and B, Q, M, K must be >= 1");
    if (grid->xyz)
        return reject(DAS_ERR_UNSUPPORTED, "voxel lists need a plan (das_plan_create)");
    if (!(c > 0.f) || !(fs > 0.f) || !std::isfinite(c) || !std::isfinite(fs) ||
        !std::isfinite(t0) || !std::isfinite(fnum) || !std::isfinite(f_demod))
        return reject(DAS_ERR_INVALID_ARG, "c and fs must be > 0; t0, fnum, f_demod finite");
    const float gf[6] = {grid->x0, grid->y0, grid->z0, grid->dx, grid->dy, grid->dz};
    for (float v : gf)
        if (!std::isfinite(v)) return reject(DAS_ERR_INVALID_ARG, "grid origin/spacing not finite");
    if (dtype != DAS_F32 && dtype != DAS_C64) return reject(DAS_ERR_INVALID_ARG, "dtype must be DAS_F32 or DAS_C64");
    if (dtype == DAS_F32 && f_demod != 0.0)
        return reject(DAS_ERR_UNSUPPORTED, "demodulation needs DAS_C64 data");
    const bool cplx = dtype == DAS_C64;
    if (!das::brick_supported(B, cplx, K))
        return reject(DAS_ERR_UNSUPPORTED, "the brick kernel cannot serve this B / K");
    const long long N = (long long)grid->nx * grid->ny * grid->nz;
    if ((long long)Q * M * (K + 3) >= (1LL << 31) || N * B >= (1LL << 31) || K >= (1 << 22))
        return reject(DAS_ERR_INVALID_ARG, "sizes beyond the library's index limits");
    const size_t elem = cplx ? 8 : 4;
    const size_t rx_bytes = align256(sizeof(RxPos) * (size_t)M);
    const size_t perm_bytes = (size_t)B * Q * M * (size_t)(K + 3) * elem;
    if (rx_bytes + perm_bytes > DAS_NOALLOC_SCRATCH_BYTES) {
        char msg[200];
        snprintf(msg, sizeof(msg),
                 "needs %zu bytes of scratch (16*M + B*Q*M*(K+3)*element), the static "
                 "array holds %llu", rx_bytes + perm_bytes, DAS_NOALLOC_SCRATCH_BYTES);
        return reject(DAS_ERR_INVALID_ARG, msg);
    }
    const uintptr_t al = reinterpret_cast<uintptr_t>(rf) | reinterpret_cast<uintptr_t>(out);
    if ((al & 15u) || (reinterpret_cast<uintptr_t>(tau_tx) & 3u) ||
        (reinterpret_cast<uintptr_t>(w_tx) & 3u) || (reinterpret_cast<uintptr_t>(rx_xyz) & 3u))
        return reject(DAS_ERR_INVALID_ARG, "rf/out must be 16-byte and rx/tau/w 4-byte aligned");

    // ---- the scratch array's address on the current device (the first call on a
    // device also loads the library's kernels there)
    int dev = 0, sms = 1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return reject(DAS_ERR_CUDA, cudaGetErrorString(e));
    void *scratch = nullptr;
    e = cudaGetSymbolAddress(&scratch, g_noalloc_scratch);
    if (e != cudaSuccess || !scratch)
        return reject(DAS_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e) : "no scratch address");
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return reject(DAS_ERR_CUDA, cudaGetErrorString(e));

    // ---- geometry in sample units (metres * fs / c)
    const double s = (double)fs / (double)c;
    DasGeom g{};
    g.nx = grid->nx; g.ny = grid->ny; g.nz = grid->nz; g.N = (int)N;
    g.x0 = (float)(grid->x0 * s); g.y0 = (float)(grid->y0 * s); g.z0 = (float)(grid->z0 * s);
    g.dx = (float)(grid->dx * s); g.dy = (float)(grid->dy * s); g.dz = (float)(grid->dz * s);
    g.fs = fs;
    g.t0fs = (float)((double)t0 * fs);
    g.aperture = fnum > 0.f;
    g.ap2 = g.aperture ? (float)(4.0 * (double)fnum * fnum) : 0.f;
    g.fd_over_fs = (float)(f_demod / (double)fs);
    g.rotate = f_demod != 0.0;
    g.B = B; g.Q = Q; g.M = M; g.K = K;

    unsigned char *base = static_cast<unsigned char *>(scratch);
    RxPos *rx_dev = reinterpret_cast<RxPos *>(base);
    void *perm = base + rx_bytes;

    // the pad rows of the padded record copy must read as zero; earlier calls
    // leave other data behind, so clear the region this call uses
    e = cudaMemsetAsync(perm, 0, perm_bytes, stream);
    if (e != cudaSuccess) return reject(DAS_ERR_CUDA, cudaGetErrorString(e));
    scale_receivers<<<(M + 127) / 128, 128, 0, stream>>>(rx_xyz, rx_dev, M, s);
    e = cudaGetLastError();
    if (e == cudaSuccess) e = das::launch_permute(rf, perm, (int)elem, B, Q, M, K, 2, sms, stream);
    if (e == cudaSuccess) e = das::launch_brick(g, rx_dev, perm, tau_tx, w_tx, out, cplx, stream);
    if (e != cudaSuccess) return reject(DAS_ERR_CUDA, cudaGetErrorString(e));
    return DAS_OK;
}
